"""fp64 CPU oracle for MLA decode over a compressed latent KV cache.

TEST INFRASTRUCTURE ONLY. Nothing in the product path imports this module:
only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg may.
It shares no code with the CUDA library (no kernels, headers, tables or
helpers); both sides are fed by the seeded generators in `mla_synth`.

What it computes, from the DeepSeek-V2 report (translated page), section 2.1:

  2.1.1  standard multi-head attention: per head i, softmax over the cached
         tokens of q_i . k_{j,i}, weighted sum of v_{j,i};
  2.1.2  low-rank joint KV compression: keys and values are up-projections of
         one cached latent c_j, k^C_{j,i} = W_UK_i c_j and v_{j,i} = W_UV_i c_j,
         with W_UK, W_UV in R^{(d_h n_h) x d_c}; head i owns rows
         [i d_h, (i+1) d_h), stored here as W[i] of shape [d_h, d_c];
  2.1.3  decoupled RoPE: a shared key k^R_j = RoPE(k_raw_j) of width d_h^R is
         cached beside c_j; the full key is [k^C_{j,i}; k^R_j] and the full
         query [q^C_i; q^R_i]; q^R arrives already rotated;
  3.1.2  an extra RMSNorm follows the compressed latent.

The pages lost every formula of these sections in extraction; the readings
taken here (softmax scale 1/sqrt(d_h + d_h^R), RMSNorm eps 1e-6 with unit
gain and no norm on k^R, RoPE base 10000 with RoFormer's interleaved pairs
(2m, 2m+1), 0-based positions, the cache modelled in its storage format) are
the plainest ones the surrounding prose supports.

Prefill (`prefill`) is the same attention with every new token of a prompt
as a query, causal over the rows up to its position, in the explicit form.

Two decode forms are given. `decode_explicit` materialises every per-head key
and value, exactly as 2.1.1 + 2.1.2 state attention. `decode_absorbed` uses
the absorption identity of 2.1.2 (W_UK folded into the query, W_UV applied
after the weighted sum), the form the GPU kernels compute. Tests pin both to
closed forms and to each other.
"""
from __future__ import annotations

import math
from typing import Optional, Sequence

import numpy as np

# ----------------------------------------------------------------------------
# storage formats


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round fp64 values to the nearest bfloat16 value, ties to even.

    bfloat16 keeps 8 significant bits and fp32's exponent range (normal
    numbers from 2^-126, subnormal spacing 2^-133). Values beyond the largest
    finite bf16 become inf. Returned as fp64 holding bf16 values.
    """
    x = np.asarray(x, dtype=np.float64)
    ax = np.abs(x)
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(ax > 0, ax, 1.0)))
    # log2 may misjudge the binade by one right at a power of two: fix it.
    e = np.where(np.ldexp(1.0, e.astype(np.int64)) > ax, e - 1, e)
    e = np.where(np.ldexp(1.0, (e + 1).astype(np.int64)) <= ax, e + 1, e)
    e = np.maximum(e, -126.0)
    quantum = np.ldexp(1.0, (e - 7).astype(np.int64))
    y = np.rint(x / quantum) * quantum          # np.rint rounds half to even
    max_bf16 = (2.0 - 2.0 ** -7) * 2.0 ** 127
    y = np.where(np.abs(y) > max_bf16, np.copysign(np.inf, x), y)
    return np.where(ax == 0, x, y)


E4M3_MAX = 448.0


def round_to_e4m3(x: np.ndarray) -> np.ndarray:
    """Round to the nearest OCP FP8 E4M3 value, ties to even, saturating at +-448.

    E4M3: 1 sign, 4 exponent bits (bias 7), 3 mantissa bits; normal values
    (1 + m/8) 2^(e-7) for e = 1..15 (the all-ones code is NaN, so the top
    finite value is 1.75 * 2^8 = 448); subnormals m/8 * 2^-6.
    """
    x = np.asarray(x, dtype=np.float64)
    ax = np.abs(x)
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(ax > 0, ax, 1.0)))
    e = np.where(np.ldexp(1.0, e.astype(np.int64)) > ax, e - 1, e)
    e = np.where(np.ldexp(1.0, (e + 1).astype(np.int64)) <= ax, e + 1, e)
    e = np.maximum(e, -6.0)
    quantum = np.ldexp(1.0, (e - 3).astype(np.int64))
    y = np.rint(x / quantum) * quantum
    y = np.clip(y, -E4M3_MAX, E4M3_MAX)
    return np.where(ax == 0, 0.0 * x, y)


def fp32(x) -> np.ndarray:
    """Round to IEEE binary32 (numpy's conversion is round-to-nearest-even)."""
    return np.asarray(x, dtype=np.float64).astype(np.float32)


def quantize_e4m3_blocks(c: np.ndarray, block: int = 128):
    """Block-scaled E4M3 storage of latent rows (one fp32 scale per `block` values).

    Per row and block: amax over the block, scale s = amax / 448 in fp32
    (s = 1 when amax = 0), code = E4M3(x / s) with x and the division in fp32
    (the precision the kernel decides codes in). Returns (codes as E4M3
    values in fp64, scales fp32 [rows, d_c / block], dequantised fp64 rows).
    The 6-bit serving quantisation of the DeepSeek-V2 report (section 3.2.3)
    gives no scheme; this block-scaled E4M3 form stands in for it.
    """
    rows, d_c = c.shape
    assert d_c % block == 0
    x32 = fp32(c).reshape(rows, d_c // block, block)
    amax = np.abs(x32).max(axis=2)                                    # fp32, exact
    s = (amax / np.float32(E4M3_MAX)).astype(np.float32)              # fp32 division
    s = np.where(amax == 0, np.float32(1.0), s).astype(np.float32)
    ratio = (x32 / s[:, :, None]).astype(np.float32)                  # fp32 division
    codes = round_to_e4m3(ratio.astype(np.float64))
    deq = codes * s[:, :, None].astype(np.float64)
    return codes.reshape(rows, d_c), s, deq.reshape(rows, d_c)


# ----------------------------------------------------------------------------
# the append step: RMSNorm'd latent + rotated shared key, in storage format


def rmsnorm(x: np.ndarray, eps: float, gamma: Optional[np.ndarray] = None) -> np.ndarray:
    """RMSNorm over the last axis: x / sqrt(mean(x^2) + eps) * gamma (gamma = 1 if None).

    The DeepSeek-V2 report (section 3.1.2) puts an extra RMSNorm after the
    compressed latent vector; it names neither eps nor a gain.
    """
    x = np.asarray(x, dtype=np.float64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    y = x / np.sqrt(ms + eps)
    if gamma is not None:
        y = y * np.asarray(gamma, dtype=np.float64)
    return y


def rope_inv_freq(d_rope: int, theta: float) -> np.ndarray:
    """Rotation frequencies theta^(-2m/d) for the pairs m = 0 .. d/2-1 (RoFormer)."""
    m = np.arange(d_rope // 2, dtype=np.float64)
    return np.power(float(theta), -2.0 * m / d_rope)


def yarn_ramp(r, alpha: float, beta: float):
    """YaRN's ramp gamma(r) (Peng et al. 2023, the method section 3.1.4 applies):
    0 below alpha, 1 above beta, linear in r between."""
    r = np.asarray(r, dtype=np.float64)
    return np.clip((r - alpha) / (beta - alpha), 0.0, 1.0)


def yarn_inv_freq(d_rope: int, theta: float, s: float, alpha: float, beta: float, orig_len: int) -> np.ndarray:
    """Rotation frequencies of the decoupled RoPE under YaRN (section 3.1.4: s = 40, alpha = 1,
    beta = 32, extending a 4K context).

    Pair m turns at theta_m = theta^(-2m/d), with wavelength 2 pi / theta_m; over the
    original context it makes r = orig_len / wavelength turns. YaRN's "NTK-by-parts" rule
    interpolates the slow pairs and keeps the fast ones:
        h(theta_m) = (1 - gamma(r)) theta_m / s + gamma(r) theta_m.
    s <= 1 leaves the frequencies as they are.
    """
    base = rope_inv_freq(d_rope, theta)
    if s <= 1.0:
        return base
    r = orig_len * base / (2.0 * math.pi)
    g = yarn_ramp(r, alpha, beta)
    return (1.0 - g) * base / s + g * base


def yarn_logit_factor(s: float, coeff: float = 0.0707) -> float:
    """Multiplier t of the attention logits under YaRN: sqrt(t) = coeff ln s + 1 (section 3.1.4),
    read as scaling both the query and the key by sqrt(t), as YaRN scales them; 1 for s <= 1."""
    if s <= 1.0:
        return 1.0
    return (coeff * math.log(s) + 1.0) ** 2


def rope(x: np.ndarray, pos: np.ndarray, theta: float, interleaved: bool = True,
         inv_freq: Optional[np.ndarray] = None) -> np.ndarray:
    """Rotary position embedding of the decoupled key (RoFormer, cited in section 2.1.3).

    Pair m of a d-vector at position p turns by the angle p * theta^(-2m/d):
    (a, b) -> (a cos - b sin, a sin + b cos). interleaved=True pairs
    components (2m, 2m+1) as in RoFormer's definition; False pairs (m, m + d/2).
    inv_freq replaces theta^(-2m/d) (YaRN: yarn_inv_freq).
    x: [..., d]; pos: broadcastable to x[..., 0].
    """
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    f = rope_inv_freq(d, theta) if inv_freq is None else np.asarray(inv_freq, dtype=np.float64)
    ang = np.asarray(pos, dtype=np.float64)[..., None] * f
    c, s = np.cos(ang), np.sin(ang)
    if interleaved:
        a, b = x[..., 0::2], x[..., 1::2]
    else:
        a, b = x[..., : d // 2], x[..., d // 2:]
    ra, rb = a * c - b * s, a * s + b * c
    out = np.empty_like(x)
    if interleaved:
        out[..., 0::2], out[..., 1::2] = ra, rb
    else:
        out[..., : d // 2], out[..., d // 2:] = ra, rb
    return out


def append_rows(c_kv_raw, k_rope_raw, positions, *, cache_dtype: str, eps: float,
                theta: float, interleaved: bool = True, gamma=None, block: int = 128, inv_freq=None):
    """What one cache row holds after the append step, as fp64 values.

    c = RMSNorm(c_kv_raw) (sections 2.1.2 + 3.1.2) and kR = RoPE(k_rope_raw, pos)
    (section 2.1.3), each then put in the cache's storage format:
    'fp32' -> rounded to binary32; 'bf16' -> RNE bf16;
    'fp8_e4m3_b128' -> latent block-scaled E4M3, rope part bf16.
    Returns (c_stored [T, d_c], kR_stored [T, d_r], extra) where extra holds the
    E4M3 codes and scales for the fp8 format (else None).
    """
    c = rmsnorm(np.asarray(c_kv_raw, dtype=np.float64), eps, gamma)
    kr = rope(np.asarray(k_rope_raw, dtype=np.float64), np.asarray(positions), theta, interleaved, inv_freq)
    if cache_dtype == "fp32":
        return fp32(c).astype(np.float64), fp32(kr).astype(np.float64), None
    if cache_dtype == "bf16":
        return round_to_bf16(c), round_to_bf16(kr), None
    if cache_dtype == "fp8_e4m3_b128":
        codes, scales, deq = quantize_e4m3_blocks(c, block)
        return deq, round_to_bf16(kr), {"codes": codes, "scales": scales}
    raise ValueError(cache_dtype)


def page_slot(block_table: np.ndarray, seq: int, pos: int, page_size: int) -> int:
    """Pool row of token `pos` of sequence `seq`: block_table[seq, pos // P] * P + pos % P."""
    return int(block_table[seq, pos // page_size]) * page_size + pos % page_size


# ----------------------------------------------------------------------------
# decode


def softmax_probs(logits: np.ndarray) -> np.ndarray:
    """Two-pass softmax over the last axis in fp64 (max subtracted first)."""
    z = np.asarray(logits, dtype=np.float64)
    z = z - z.max(axis=-1, keepdims=True)
    a = np.exp(z)
    return a / a.sum(axis=-1, keepdims=True)


def head_explicit(q_nope_i, q_rope_i, w_uk_i, w_uv_i, c, kr, scale):
    """One (sequence, head) of MLA decode with materialised per-head keys and values.

    k_{j,i} = [W_UK_i c_j ; kR_j], v_{j,i} = W_UV_i c_j, q_i = [q_nope_i ; q_rope_i]
    (sections 2.1.2-2.1.3); out = sum_j softmax_j(scale q_i . k_{j,i}) v_{j,i}
    (section 2.1.1). Returns (out [d_h], probs [L]).
    """
    c = np.asarray(c, dtype=np.float64)
    k_c = c @ np.asarray(w_uk_i, dtype=np.float64).T           # [L, d_h]
    v = c @ np.asarray(w_uv_i, dtype=np.float64).T             # [L, d_h]
    k = np.concatenate([k_c, np.asarray(kr, dtype=np.float64)], axis=1)
    q = np.concatenate([np.asarray(q_nope_i, np.float64), np.asarray(q_rope_i, np.float64)])
    p = softmax_probs(scale * (k @ q))
    return p @ v, p


def head_absorbed(q_nope_i, q_rope_i, w_uk_i, w_uv_i, c, kr, scale):
    """One (sequence, head) in the absorbed form of section 2.1.2.

    W_UK is folded into the query, q_lat = W_UK_i^T q_nope_i, so the latent
    score is q_lat . c_j; W_UV is applied once after the weighted sum of the
    latents, out = W_UV_i sum_j p_j c_j. Returns (out [d_h], probs [L]).
    """
    c = np.asarray(c, dtype=np.float64)
    w_uk_i = np.asarray(w_uk_i, dtype=np.float64)
    q_lat = w_uk_i.T @ np.asarray(q_nope_i, np.float64)                  # [d_c]
    logits = scale * (c @ q_lat + np.asarray(kr, np.float64) @ np.asarray(q_rope_i, np.float64))
    p = softmax_probs(logits)
    o_lat = p @ c                                                         # [d_c]
    return np.asarray(w_uv_i, dtype=np.float64) @ o_lat, p


def decode(q_nope, q_rope, w_uk, w_uv, c_seqs: Sequence[np.ndarray], kr_seqs: Sequence[np.ndarray],
           scale: float, form: str = "absorbed", heads: Optional[Sequence[int]] = None,
           batches: Optional[Sequence[int]] = None) -> np.ndarray:
    """MLA decode output [B, H, d_h] (only the requested batches/heads are filled).

    q_nope [B,H,d_h], q_rope [B,H,d_r], w_uk/w_uv [H,d_h,d_c]; c_seqs[b] [L_b, d_c]
    and kr_seqs[b] [L_b, d_r] are sequence b's cache content (storage format,
    as fp64). A sequence with L_b = 0 yields zeros. Unrequested entries are NaN.
    """
    q_nope = np.asarray(q_nope, np.float64)
    q_rope = np.asarray(q_rope, np.float64)
    w_uk = np.asarray(w_uk, np.float64)
    w_uv = np.asarray(w_uv, np.float64)
    B, H, d_h = q_nope.shape
    fn = {"explicit": head_explicit, "absorbed": head_absorbed}[form]
    out = np.full((B, H, d_h), np.nan)
    for b in (range(B) if batches is None else batches):
        for i in (range(H) if heads is None else heads):
            if len(c_seqs[b]) == 0:
                out[b, i] = 0.0
                continue
            out[b, i], _ = fn(q_nope[b, i], q_rope[b, i], w_uk[i], w_uv[i],
                              c_seqs[b], kr_seqs[b], scale)
    return out


def decode_multi(q_nope, q_rope, w_uk, w_uv, c_seqs: Sequence[np.ndarray], kr_seqs: Sequence[np.ndarray],
                 scale: float, form: str = "absorbed") -> np.ndarray:
    """Decode of q new tokens per sequence at once (multi-token prediction drafts, DeepSeek-V3
    summary; verified together as in speculative decoding): out [B, q, H, d_h].

    q_nope [B, q, H, d_h], q_rope [B, q, H, d_r]. The cache of sequence b already holds its q new
    tokens as its last q rows; new token k attends causally to every row up to and including
    its own: the first L_b - (q - 1 - k) rows.
    """
    q_nope = np.asarray(q_nope, np.float64)
    q_rope = np.asarray(q_rope, np.float64)
    B, q = q_nope.shape[:2]
    out = np.zeros(q_nope.shape)
    for k in range(q):
        drop = q - 1 - k
        cs = [c[:max(0, len(c) - drop)] for c in c_seqs]
        ks = [r[:max(0, len(r) - drop)] for r in kr_seqs]
        out[:, k] = decode(q_nope[:, k], q_rope[:, k], w_uk, w_uv, cs, ks, scale, form)
    return out


def prefill(q_nope, q_rope, w_uk, w_uv, c_seqs: Sequence[np.ndarray], kr_seqs: Sequence[np.ndarray],
            n_new: Sequence[int], scale: float, heads: Optional[Sequence[int]] = None,
            rows: Optional[Sequence[int]] = None) -> np.ndarray:
    """Prefill (or one chunk of a prompt) in the non-absorbed form of section 2.1.2: out [T, H, d_h].

    Sequence b caches L_b = len(c_seqs[b]) rows; its last n_b = n_new[b] rows are its new tokens,
    query rows q_start[b] .. q_start[b] + n_b - 1 of q_nope [T, H, d_h] and q_rope [T, H, d_r]
    (q_start = prefix sums of n_new). New token k sits at position p = L_b - n_b + k and attends
    causally (section 2.1.1) to rows 0 .. p, with the per-head keys [W_UK_i c_j ; kR_j] and values
    W_UV_i c_j materialised (sections 2.1.2-2.1.3). Only the requested heads and query rows are
    computed; the rest is NaN.
    """
    q_nope = np.asarray(q_nope, np.float64)
    q_rope = np.asarray(q_rope, np.float64)
    w_uk = np.asarray(w_uk, np.float64)
    w_uv = np.asarray(w_uv, np.float64)
    T, H, d_h = q_nope.shape
    n_new = [int(n) for n in n_new]
    q_start = np.concatenate([[0], np.cumsum(n_new)]).astype(np.int64)
    assert q_start[-1] == T
    want = np.zeros(T, dtype=bool)
    want[list(range(T)) if rows is None else list(rows)] = True
    out = np.full((T, H, d_h), np.nan)
    for b, n in enumerate(n_new):
        mine = [k for k in range(n) if want[q_start[b] + k]]
        if not mine:
            continue
        c = np.asarray(c_seqs[b], np.float64)
        kr = np.asarray(kr_seqs[b], np.float64)
        L = len(c)
        assert 0 <= n <= L
        for i in (range(H) if heads is None else heads):
            k_i = np.concatenate([c @ w_uk[i].T, kr], axis=1)     # [L, d_h + d_r]
            v_i = c @ w_uv[i].T                                    # [L, d_h]
            for k in mine:
                r = q_start[b] + k
                p = L - n + k
                q = np.concatenate([q_nope[r, i], q_rope[r, i]])
                a = softmax_probs(scale * (k_i[:p + 1] @ q))
                out[r, i] = a @ v_i[:p + 1]
    return out


def decode_hidden(q_nope, q_rope, w_uk, w_uv, w_o, c_seqs: Sequence[np.ndarray], kr_seqs: Sequence[np.ndarray],
                  scale: float, batches: Optional[Sequence[int]] = None, form: str = "explicit") -> np.ndarray:
    """Attention output projected to the hidden size: u[b] = W_O [o_{b,1}; ...; o_{b,H}] (section
    2.1.1: the per-head outputs are concatenated and multiplied by the output projection
    W_O in R^{hidden x (d_h n_h)}), with o_{b,i} the per-head outputs (explicit form by default; the
    absorbed form gives the same values). Returns [B, hidden] (rows of unrequested batches are NaN)."""
    w_o = np.asarray(w_o, np.float64)
    q_nope = np.asarray(q_nope, np.float64)
    B, H, d_h = q_nope.shape
    per_head = decode(q_nope, q_rope, w_uk, w_uv, c_seqs, kr_seqs, scale, form=form, batches=batches)
    out = np.full((B, w_o.shape[0]), np.nan)
    for b in (range(B) if batches is None else batches):
        out[b] = w_o @ per_head[b].reshape(H * d_h)
    return out


def fold_output_weight(w_uv, w_o) -> np.ndarray:
    """W_UV absorbed into W_O (section 2.1.2): W_OUV[:, i d_c:(i+1) d_c] = W_O[:, i d_h:(i+1) d_h] W_UV_i,
    so that W_O [W_UV_1 o_1; ...; W_UV_H o_H] = W_OUV [o_1; ...; o_H] for latent-space outputs o_i.
    Returns [hidden, H d_c]."""
    w_uv = np.asarray(w_uv, np.float64)
    w_o = np.asarray(w_o, np.float64)
    H, d_h, d_c = w_uv.shape
    return np.concatenate([w_o[:, i * d_h:(i + 1) * d_h] @ w_uv[i] for i in range(H)], axis=1)


# ----------------------------------------------------------------------------
# closed forms from the pages


def kv_elements_per_token(kind: str, *, n_h: int, d_h: int, l: int, n_g: int = 0,
                          d_c: int = 0, d_r: int = 0) -> int:
    """Per-token KV-cache element counts of section 2.1.4, Table 1.

    MHA caches keys and values of every head (2 n_h d_h l), GQA those of n_g
    groups (2 n_g d_h l), MQA one group (2 d_h l), MLA the latent and the
    shared rope key ((d_c + d_h^R) l).
    """
    return {"MHA": 2 * n_h * d_h * l, "GQA": 2 * n_g * d_h * l,
            "MQA": 2 * d_h * l, "MLA": (d_c + d_r) * l}[kind]


def yarn_mscale_sqrt_t(s: float) -> float:
    """Attention-entropy factor of section 3.1.4: sqrt(t) = 0.0707 ln s + 1."""
    return 0.0707 * math.log(s) + 1.0
