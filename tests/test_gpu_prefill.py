"""GPU parity of mla_prefill (whole prompts and prompt chunks, non-absorbed form) against the
fp64 oracle's `prefill`. Expected values come only from the oracle."""
import numpy as np
import pytest
import torch

import mla_synth as S
from oracle import mla_oracle as O
from tests import mla_testlib as T

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from head_latent_attention_22_b300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def _device_prefill(inp, pf, max_seq_len=None, q_start=None):
    import head_latent_attention_22_b300 as M
    dc = T.to_device(inp)
    T.fill_cache(dc)
    qs = torch.from_numpy((pf.q_start if q_start is None else q_start).astype(np.int32)).cuda()
    L = int(inp.lengths.max()) if max_seq_len is None else max_seq_len
    out = M.prefill(dc.cfg, pf.q_nope.cuda(), pf.q_rope.cuda(), dc.w_uk, dc.w_uv, dc.pool, dc.block_table,
                    dc.seq_lens, qs, L)
    return out, M


def _oracle_prefill(inp, pf, heads=None, rows=None):
    cs, ks = zip(*[T.oracle_cache(inp, b) for b in range(inp.shape.batch)])
    return O.prefill(pf.q_nope.double().numpy(), pf.q_rope.double().numpy(), inp.w_uk.double().numpy(),
                     inp.w_uv.double().numpy(), cs, ks, pf.n_new, T.oracle_scale(inp.shape), heads=heads, rows=rows)


@pytest.mark.parametrize("lengths,n_new,yarn", [
    ((1, 130, 300), None, 1.0),              # whole prompts: one row, a ragged tile tail, three tiles
    ((200, 333, 64), (77, 333, 0), 1.0),     # a chunk after a 123-row prefix, a whole prompt, no new token
    ((260, 513), (260, 129), 40.0),          # the report's YaRN setting: scaled rope keys, logit factor
])
def test_prefill_all_outputs_small(lengths, n_new, yarn):
    shape = S.shape_with("prefill_b4", batch=len(lengths), lengths=lengths, yarn_factor=yarn)
    inp = S.make_inputs(shape)
    pf = S.draw_prefill(inp, None if n_new is None else np.array(n_new))
    out, M = _device_prefill(inp, pf)
    M.check_device_errors()
    want = _oracle_prefill(inp, pf)
    T.assert_close(out.cpu().numpy(), want, "bf16", f"prefill {lengths} {n_new}")


def test_prefill_full_size_sampled():
    shape = S.SHAPES["prefill_b4"]
    inp = S.make_inputs(shape)
    pf = S.draw_prefill(inp)
    out, M = _device_prefill(inp, pf)
    M.check_device_errors()
    got = out.cpu().numpy()
    assert np.isfinite(got).all()
    rng = np.random.default_rng(5)
    heads = sorted(set([0, shape.n_heads - 1] + list(rng.choice(np.arange(1, shape.n_heads - 1), 6, replace=False))))
    ks = [0, 1, 63, 64, 127, 128, 129, 1000, 2047, 2048, 3071, 4094, 4095]
    rows = [int(pf.q_start[b]) + k for b in range(shape.batch) for k in ks]
    want = _oracle_prefill(inp, pf, heads=heads, rows=rows)
    sel = np.ix_(rows, heads)
    T.assert_close(got[sel], want[sel], "bf16", "prefill_b4 sampled")


def test_prefill_flags_new_tokens_beyond_the_cache():
    import head_latent_attention_22_b300 as M
    shape = S.shape_with("prefill_b4", batch=2, lengths=(100, 150))
    inp = S.make_inputs(shape)
    pf = S.draw_prefill(inp)
    bad = pf.q_start.copy()
    bad[1] = 120   # sequence 0 claims 120 new tokens, but only 100 rows are cached
    out, M = _device_prefill(inp, pf, q_start=bad)
    with pytest.raises(M.MLAError) as e:
        M.check_device_errors()
    assert e.value.status == 5
    M.check_device_errors()   # the word was cleared


def test_prefill_refuses_unsupported_configs():
    import head_latent_attention_22_b300 as M
    cfg = M.MLAConfig.from_shape(S.SHAPES["fp8_b32"])
    assert M.prefill_workspace_size(cfg, 2, 128) == 0
    cfg32 = M.MLAConfig.from_shape(S.SHAPES["tiny_fp32"])
    assert M.prefill_workspace_size(cfg32, 2, 128) == 0
