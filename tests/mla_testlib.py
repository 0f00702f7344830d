"""Shared helpers of the parity tests: move seeded inputs to the GPU, fill the
paged cache through the library, and compute oracle values for chosen
(sequence, head) pairs. Expected values come only from the oracle."""
from __future__ import annotations

import dataclasses
from typing import Optional, Sequence

import numpy as np
import torch

import mla_synth as S
from oracle import mla_oracle as O

# Tolerances. bf16 cache/queries with fp32 accumulation: the targets for the
# DeepSeek-V2-shaped decode. fp32 end to end (CUDA-core path): fp32 rounding
# of sums over <= 600 terms, ~1e-6 relative, with a wide margin.
TOL = {
    "bf16": dict(max_rel=1e-2, mean_rel=2e-3),
    "fp8_e4m3_b128": dict(max_rel=3e-2, mean_rel=2e-3 * 5),
    "fp32": dict(max_rel=1e-4, mean_rel=2e-5),
}


def err_stats(got: np.ndarray, ref: np.ndarray) -> dict:
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    diff = np.abs(got - ref)
    return dict(max_rel=float(diff.max() / max(np.abs(ref).max(), 1e-300)),
                mean_rel=float(diff.mean() / max(np.abs(ref).mean(), 1e-300)),
                max_abs=float(diff.max()))


def assert_close(got, ref, cache_dtype: str, what: str = ""):
    st = err_stats(got, ref)
    tol = TOL[cache_dtype]
    assert np.all(np.isfinite(got)), f"{what}: non-finite outputs"
    assert st["max_rel"] <= tol["max_rel"] and st["mean_rel"] <= tol["mean_rel"], f"{what}: {st} vs {tol}"
    return st


@dataclasses.dataclass
class DeviceCase:
    inp: S.MLAInputs
    cfg: object
    pool: torch.Tensor
    block_table: torch.Tensor
    seq_lens: torch.Tensor
    q_nope: torch.Tensor
    q_rope: torch.Tensor
    w_uk: torch.Tensor
    w_uv: torch.Tensor


def to_device(inp: S.MLAInputs, dev="cuda", pool_fill: Optional[int] = None) -> DeviceCase:
    import head_latent_attention_22_b300 as M
    cfg = M.MLAConfig.from_shape(inp.shape)
    pool = M.new_pool(cfg, inp.num_pages, dev, fill=pool_fill)
    return DeviceCase(inp, cfg, pool,
                      torch.from_numpy(inp.block_table).to(dev),
                      torch.from_numpy(inp.lengths.astype(np.int32)).to(dev),
                      inp.q_nope.to(dev), inp.q_rope.to(dev), inp.w_uk.to(dev), inp.w_uv.to(dev))


def fill_cache(dc: DeviceCase, chunk: int = 1 << 20):
    """Append every token of every sequence (positions 0..L_b-1) through mla_append."""
    import head_latent_attention_22_b300 as M
    inp = dc.inp
    pos = torch.from_numpy(inp.positions())
    seq = torch.from_numpy(inp.seq_index())
    T = pos.shape[0]
    for s in range(0, T, chunk):
        e = min(T, s + chunk)
        M.append(dc.cfg, inp.c_kv_raw[s:e].to("cuda"), inp.k_rope_raw[s:e].to("cuda"), pos[s:e].to("cuda"),
                 dc.pool, dc.block_table, seq_idx=seq[s:e].to("cuda"))
    torch.cuda.synchronize()


def run_decode(dc: DeviceCase, max_seq_len: Optional[int] = None) -> np.ndarray:
    import head_latent_attention_22_b300 as M
    L = int(dc.inp.lengths.max()) if max_seq_len is None else max_seq_len
    out = M.decode(dc.cfg, dc.q_nope, dc.q_rope, dc.w_uk, dc.w_uv, dc.pool, dc.block_table, dc.seq_lens, L)
    M.check_device_errors()
    return out.cpu().numpy()


def oracle_cache(inp: S.MLAInputs, b: int):
    """Oracle cache content (c, kR) of sequence b, in the cache's storage format."""
    s = inp.shape
    o0, o1 = int(inp.token_offsets[b]), int(inp.token_offsets[b + 1])
    c_raw = inp.c_kv_raw[o0:o1].double().numpy()
    k_raw = inp.k_rope_raw[o0:o1].double().numpy()
    c, kr, _ = O.append_rows(c_raw, k_raw, np.arange(o1 - o0), cache_dtype=s.cache_dtype, eps=s.eps,
                             theta=s.rope_theta, inv_freq=oracle_inv_freq(s))
    return c, kr


def oracle_inv_freq(s):
    """RoPE frequencies of a workload: plain, or YaRN-scaled when s.yarn_factor > 1."""
    return O.yarn_inv_freq(s.d_rope, s.rope_theta, s.yarn_factor, s.yarn_alpha, s.yarn_beta, s.yarn_orig_len)


def oracle_scale(s) -> float:
    """Softmax scale of a workload, with YaRN's logit factor when it is on."""
    return s.scale * O.yarn_logit_factor(s.yarn_factor, s.yarn_mscale)


def oracle_outputs(inp: S.MLAInputs, pairs: Sequence[tuple], form: str = "absorbed") -> np.ndarray:
    """Oracle out[b, i] for each (b, i) in pairs -> [len(pairs), d_h]."""
    s = inp.shape
    q_nope = inp.q_nope.double().numpy()
    q_rope = inp.q_rope.double().numpy()
    w_uk = inp.w_uk.double().numpy()
    w_uv = inp.w_uv.double().numpy()
    fn = O.head_absorbed if form == "absorbed" else O.head_explicit
    res = np.zeros((len(pairs), s.d_head))
    cache = {}
    for n, (b, i) in enumerate(pairs):
        if b not in cache:
            cache[b] = oracle_cache(inp, b)
        c, kr = cache[b]
        if len(c) == 0:
            continue
        res[n], _ = fn(q_nope[b, i], q_rope[b, i], w_uk[i], w_uv[i], c, kr, oracle_scale(s))
    return res
