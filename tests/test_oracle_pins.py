"""Pins of the fp64 oracle to facts other than itself (CPU only).

Each test ties one part of the oracle to a closed form worked by hand, a
library routine, an invariant, a special case, brute force on tiny inputs or
a number the pages print. Together they are chosen so that a dropped term, a
sign error, a wrong index or a transposed operand anywhere in the oracle
fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

from oracle import mla_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# --------------------------------------------------------------- storage formats

def test_bf16_rounding_matches_torch_on_fp32_values():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(20000).astype(np.float32),
                        (rng.standard_normal(2000) * 1e-30).astype(np.float32),
                        (rng.standard_normal(2000) * 1e30).astype(np.float32),
                        np.array([1 + 2**-8, 1 + 3 * 2**-8, -(1 + 2**-8), 2**-130, 0.0],
                                 dtype=np.float32)])
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(O.round_to_bf16(x.astype(np.float64)), ref)


def test_bf16_ties_to_even_by_hand():
    # spacing of bf16 just above 1 is 2^-7; halfway points go to the even mantissa
    assert O.round_to_bf16(np.array([1 + 2**-8]))[0] == 1.0
    assert O.round_to_bf16(np.array([1 + 3 * 2**-8]))[0] == 1 + 2**-6
    assert O.round_to_bf16(np.array([1 + 2**-8 + 2**-20]))[0] == 1 + 2**-7


def test_e4m3_matches_torch_in_range():
    rng = np.random.default_rng(1)
    x = np.concatenate([rng.uniform(-448, 448, 20000), rng.standard_normal(20000),
                        rng.standard_normal(2000) * 2**-8]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    np.testing.assert_array_equal(O.round_to_e4m3(x.astype(np.float64)), ref)


def test_e4m3_by_hand():
    v = O.round_to_e4m3(np.array([448.0, 500.0, -1e6, 2.0**-9, 2.0**-10, 1.0625, 1.1875, 240.0, 232.0]))
    # max finite 448; saturation; smallest subnormal 2^-9; half of it ties to 0;
    # 1.0625 ties to 1.0 (even); 1.1875 ties to 1.25 (even); 240 exact; 232 ties to 224 (even)
    np.testing.assert_array_equal(v, [448.0, 448.0, -448.0, 2.0**-9, 0.0, 1.0, 1.25, 240.0, 224.0])


def test_e4m3_block_quantisation_properties():
    rng = np.random.default_rng(2)
    c = rng.standard_normal((7, 256))
    c[3, 128:] = 0.0                     # an all-zero block takes scale 1
    codes, scales, deq = O.quantize_e4m3_blocks(c, 128)
    assert scales.dtype == np.float32 and scales.shape == (7, 2)
    assert scales[3, 1] == 1.0 and np.all(codes[3, 128:] == 0)
    # every block's largest magnitude lands on (or within rounding of) +-448
    amax_codes = np.abs(codes).reshape(7, 2, 128).max(axis=2)
    assert np.all((amax_codes[[i for i in range(7)], 0] >= 416) & (amax_codes[:, 0] <= 448))
    # dequantised error stays within half an E4M3 step (relative 2^-4) of each value
    err = np.abs(deq - c)
    s = np.repeat(scales.astype(np.float64), 128, axis=1)
    assert np.all(err <= np.maximum(np.abs(c) * 2.0**-4, s * 2.0**-10) * 1.0001)


# --------------------------------------------------------------- RMSNorm, RoPE

def test_rmsnorm_by_hand_and_invariants():
    eps = 1e-6
    y = O.rmsnorm(np.array([3.0, 4.0]), eps)
    np.testing.assert_allclose(y, np.array([3.0, 4.0]) / math.sqrt(12.5 + eps), rtol=0, atol=1e-15)
    rng = np.random.default_rng(3)
    x = rng.standard_normal((5, 512))
    y = O.rmsnorm(x, eps)
    ms = np.mean(x * x, axis=1)
    np.testing.assert_allclose(np.sqrt(np.mean(y * y, axis=1)), 1 / np.sqrt(1 + eps / ms), rtol=1e-13)
    np.testing.assert_allclose(O.rmsnorm(7.5 * x, 0.0), O.rmsnorm(x, 0.0), rtol=1e-13)
    g = rng.standard_normal(512)
    np.testing.assert_allclose(O.rmsnorm(x, eps, g), O.rmsnorm(x, eps) * g, rtol=1e-14)


def test_rope_pairing_and_sign_by_hand():
    d, theta = 8, 10000.0
    for m in range(d // 2):
        for pos in (0, 1, 37, 131071):
            ang = pos * theta ** (-2.0 * m / d)
            e = np.zeros(d)
            e[2 * m] = 1.0
            want = np.zeros(d)
            want[2 * m], want[2 * m + 1] = math.cos(ang), math.sin(ang)
            np.testing.assert_allclose(O.rope(e, pos, theta), want, atol=1e-12)
            e = np.zeros(d)
            e[2 * m + 1] = 1.0
            want = np.zeros(d)
            want[2 * m], want[2 * m + 1] = -math.sin(ang), math.cos(ang)
            np.testing.assert_allclose(O.rope(e, pos, theta), want, atol=1e-12)
            # half-split pairing: (m, m + d/2)
            e = np.zeros(d)
            e[m] = 1.0
            want = np.zeros(d)
            want[m], want[m + d // 2] = math.cos(ang), math.sin(ang)
            np.testing.assert_allclose(O.rope(e, pos, theta, interleaved=False), want, atol=1e-12)


def test_rope_invariants():
    rng = np.random.default_rng(4)
    q, k = rng.standard_normal(64), rng.standard_normal(64)
    np.testing.assert_array_equal(O.rope(q, 0, 1e4), q)
    np.testing.assert_allclose(np.linalg.norm(O.rope(q, 12345, 1e4)), np.linalg.norm(q), rtol=1e-13)
    for m, n, s in ((3, 9, 100), (1000, 17, 4096), (0, 0, 65000)):
        a = O.rope(q, m, 1e4) @ O.rope(k, n, 1e4)
        b = O.rope(q, m + s, 1e4) @ O.rope(k, n + s, 1e4)
        assert abs(a - b) < 1e-9 * (1 + abs(a))


# --------------------------------------------------------------- softmax, decode

def test_softmax_matches_scipy_and_sums_to_one():
    rng = np.random.default_rng(5)
    z = rng.standard_normal((6, 300)) * 30
    p = O.softmax_probs(z)
    np.testing.assert_allclose(p, scipy.special.softmax(z, axis=1), rtol=1e-12, atol=1e-300)
    np.testing.assert_allclose(p.sum(axis=1), 1.0, rtol=0, atol=1e-14)
    assert np.all(p >= 0)


def _two_token_case():
    """A decode worked by hand: one head, d_h=2, d_c=3, d_r=2, two cached tokens."""
    eps, theta, scale = 1e-6, 10000.0, 0.7
    c_raw = np.array([[3.0, 4.0, 0.0], [1.0, -1.0, 2.0]])
    k_raw = np.array([[1.0, 0.0], [0.5, 2.0]])
    w_uk = np.array([[1.0, 2.0, 0.0], [0.0, 1.0, -1.0]])     # [d_h, d_c]
    w_uv = np.array([[1.0, 2.0, 3.0], [0.0, 1.0, -2.0]])     # [d_h, d_c]
    q_nope = np.array([1.0, -1.0])
    q_rope = np.array([0.3, -0.8])
    # by hand: c_j = c_raw_j / sqrt(mean(c_raw_j^2) + eps)
    n0, n1 = math.sqrt(25 / 3 + eps), math.sqrt(6 / 3 + eps)
    c0, c1 = np.array([3, 4, 0]) / n0, np.array([1, -1, 2]) / n1
    # d_r = 2: one pair at frequency 1, angle = position; token 0 unrotated
    kr0 = np.array([1.0, 0.0])
    a = 1.0
    kr1 = np.array([0.5 * math.cos(a) - 2.0 * math.sin(a), 0.5 * math.sin(a) + 2.0 * math.cos(a)])
    # k_{j} = [W_UK c_j ; kR_j]: W_UK c = (c[0] + 2 c[1], c[1] - c[2]); q_nope . that = c[0] + c[1] + c[2]
    s0 = scale * ((c0[0] + c0[1] + c0[2]) + 0.3 * kr0[0] - 0.8 * kr0[1])
    s1 = scale * ((c1[0] + c1[1] + c1[2]) + 0.3 * kr1[0] - 0.8 * kr1[1])
    p1 = 1.0 / (1.0 + math.exp(s0 - s1))
    p0 = 1.0 - p1
    mix = p0 * c0 + p1 * c1
    want = np.array([mix[0] + 2 * mix[1] + 3 * mix[2], mix[1] - 2 * mix[2]])
    return dict(eps=eps, theta=theta, scale=scale, c_raw=c_raw, k_raw=k_raw, w_uk=w_uk,
                w_uv=w_uv, q_nope=q_nope, q_rope=q_rope, want=want, p=np.array([p0, p1]))


@pytest.mark.parametrize("form", ["explicit", "absorbed"])
def test_two_token_decode_by_hand(form):
    t = _two_token_case()
    c = O.rmsnorm(t["c_raw"], t["eps"])
    kr = O.rope(t["k_raw"], np.array([0, 1]), t["theta"])
    fn = O.head_explicit if form == "explicit" else O.head_absorbed
    out, p = fn(t["q_nope"], t["q_rope"], t["w_uk"], t["w_uv"], c, kr, t["scale"])
    np.testing.assert_allclose(p, t["p"], rtol=1e-13)
    np.testing.assert_allclose(out, t["want"], rtol=1e-13)


def test_two_token_decode_catches_transposes_and_dropped_terms():
    t = _two_token_case()
    c = O.rmsnorm(t["c_raw"], t["eps"])
    kr = O.rope(t["k_raw"], np.array([0, 1]), t["theta"])
    base = t["want"]
    # each plausible mistake moves the answer well away from the hand value
    mistakes = [
        dict(kr=np.zeros_like(kr)),                       # rope term dropped
        dict(kr=O.rope(t["k_raw"], np.array([0, -1]), t["theta"])),   # rotation sign
        dict(kr=O.rope(t["k_raw"], np.array([1, 2]), t["theta"])),    # 1-based positions
        dict(scale=1.0),                                   # scale dropped
        dict(w_uv=np.concatenate([t["w_uv"][:, ::-1]], axis=1)),      # reversed latent index
    ]
    for m in mistakes:
        args = dict(q_nope=t["q_nope"], q_rope=t["q_rope"], w_uk=t["w_uk"], w_uv=t["w_uv"],
                    c=c, kr=kr, scale=t["scale"])
        args.update(m)
        out, _ = O.head_explicit(args["q_nope"], args["q_rope"], args["w_uk"], args["w_uv"],
                                 args["c"], args["kr"], args["scale"])
        assert np.max(np.abs(out - base)) > 1e-3


def _brute_force_mha(q_nope, q_rope, w_uk, w_uv, c, kr, scale):
    """Textbook multi-head attention with keys/values built element by element."""
    H, d_h, d_c = len(w_uk), len(w_uk[0]), len(w_uk[0][0])
    L, d_r = len(kr), len(kr[0])
    out = [[0.0] * d_h for _ in range(H)]
    for i in range(H):
        keys, vals = [], []
        for j in range(L):
            k = [sum(w_uk[i][r][s] * c[j][s] for s in range(d_c)) for r in range(d_h)]
            k += [kr[j][r] for r in range(d_r)]
            v = [sum(w_uv[i][r][s] * c[j][s] for s in range(d_c)) for r in range(d_h)]
            keys.append(k)
            vals.append(v)
        q = list(q_nope[i]) + list(q_rope[i])
        logits = [scale * sum(q[r] * keys[j][r] for r in range(d_h + d_r)) for j in range(L)]
        mx = max(logits)
        w = [math.exp(z - mx) for z in logits]
        tot = sum(w)
        for r in range(d_h):
            out[i][r] = sum(w[j] * vals[j][r] for j in range(L)) / tot
    return np.array(out)


def test_oracle_equals_brute_force_mha_tiny():
    rng = np.random.default_rng(6)
    H, d_h, d_c, d_r, L = 3, 4, 5, 2, 7
    q_nope, q_rope = rng.standard_normal((1, H, d_h)), rng.standard_normal((1, H, d_r))
    w_uk, w_uv = rng.standard_normal((H, d_h, d_c)), rng.standard_normal((H, d_h, d_c))
    c, kr = rng.standard_normal((L, d_c)), rng.standard_normal((L, d_r))
    want = _brute_force_mha(q_nope[0].tolist(), q_rope[0].tolist(), w_uk.tolist(), w_uv.tolist(),
                            c.tolist(), kr.tolist(), 0.37)
    for form in ("explicit", "absorbed"):
        got = O.decode(q_nope, q_rope, w_uk, w_uv, [c], [kr], 0.37, form=form)[0]
        np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-13)


def test_absorbed_equals_explicit_random_shapes():
    rng = np.random.default_rng(7)
    for (B, H, d_h, d_c, d_r) in ((2, 4, 16, 32, 8), (3, 5, 7, 11, 4), (1, 2, 128, 512, 64)):
        lens = rng.integers(1, 40, size=B)
        q_nope, q_rope = rng.standard_normal((B, H, d_h)), rng.standard_normal((B, H, d_r))
        w_uk, w_uv = rng.standard_normal((H, d_h, d_c)) * 0.2, rng.standard_normal((H, d_h, d_c)) * 0.2
        cs = [rng.standard_normal((n, d_c)) for n in lens]
        krs = [rng.standard_normal((n, d_r)) for n in lens]
        a = O.decode(q_nope, q_rope, w_uk, w_uv, cs, krs, 0.2, form="absorbed")
        e = O.decode(q_nope, q_rope, w_uk, w_uv, cs, krs, 0.2, form="explicit")
        assert np.max(np.abs(a - e)) <= 1e-10 * np.max(np.abs(e))


def test_special_cases():
    rng = np.random.default_rng(8)
    H, d_h, d_c, d_r = 3, 6, 10, 4
    q_nope, q_rope = rng.standard_normal((1, H, d_h)), rng.standard_normal((1, H, d_r))
    w_uk, w_uv = rng.standard_normal((H, d_h, d_c)), rng.standard_normal((H, d_h, d_c))
    # one cached token: attention returns its value exactly
    c1, kr1 = rng.standard_normal((1, d_c)), rng.standard_normal((1, d_r))
    out = O.decode(q_nope, q_rope, w_uk, w_uv, [c1], [kr1], 0.5)
    for i in range(H):
        np.testing.assert_allclose(out[0, i], w_uv[i] @ c1[0], rtol=1e-13)
    # identical rows: uniform weights, value of the row
    c, kr = np.repeat(c1, 9, axis=0), np.repeat(kr1, 9, axis=0)
    out = O.decode(q_nope, q_rope, w_uk, w_uv, [c], [kr], 0.5, form="explicit")
    for i in range(H):
        np.testing.assert_allclose(out[0, i], w_uv[i] @ c1[0], rtol=1e-12)
    # no key signal at all: plain mean of the values
    c, kr = rng.standard_normal((9, d_c)), rng.standard_normal((9, d_r))
    out = O.decode(q_nope, np.zeros_like(q_rope), np.zeros_like(w_uk), w_uv, [c], [kr], 0.5)
    for i in range(H):
        np.testing.assert_allclose(out[0, i], w_uv[i] @ c.mean(axis=0), rtol=1e-12)
    # empty cache gives zeros; a zeroed head gives zeros only for that head
    out = O.decode(q_nope, q_rope, w_uk, w_uv, [np.zeros((0, d_c))], [np.zeros((0, d_r))], 0.5)
    assert np.all(out == 0)
    w0 = w_uv.copy()
    w0[1] = 0
    out = O.decode(q_nope, q_rope, w_uk, w0, [c], [kr], 0.5)
    assert np.all(out[0, 1] == 0) and np.all(np.abs(out[0, 0]) > 0)


def test_probs_sum_to_one_on_long_sequence():
    rng = np.random.default_rng(9)
    c, kr = rng.standard_normal((5000, 32)), rng.standard_normal((5000, 8))
    _, p = O.head_absorbed(rng.standard_normal(16), rng.standard_normal(8),
                           rng.standard_normal((16, 32)), rng.standard_normal((16, 32)), c, kr, 0.2)
    assert abs(p.sum() - 1) < 1e-13 and np.all(p >= 0)


def test_append_rows_formats():
    rng = np.random.default_rng(10)
    c_raw, k_raw = rng.standard_normal((5, 256)), rng.standard_normal((5, 64))
    pos = np.array([0, 1, 2, 100, 131071])
    c, kr = O.rmsnorm(c_raw, 1e-6), O.rope(k_raw, pos, 1e4)
    c32, k32, _ = O.append_rows(c_raw, k_raw, pos, cache_dtype="fp32", eps=1e-6, theta=1e4)
    np.testing.assert_array_equal(c32, c.astype(np.float32))
    np.testing.assert_array_equal(k32, kr.astype(np.float32))
    cb, kb, _ = O.append_rows(c_raw, k_raw, pos, cache_dtype="bf16", eps=1e-6, theta=1e4)
    np.testing.assert_array_equal(cb, O.round_to_bf16(c))
    assert np.max(np.abs(cb - c) / np.abs(c)) <= 2.0**-8
    c8, k8, extra = O.append_rows(c_raw, k_raw, pos, cache_dtype="fp8_e4m3_b128", eps=1e-6, theta=1e4)
    np.testing.assert_array_equal(k8, kb)
    np.testing.assert_array_equal(c8, extra["codes"] * np.repeat(extra["scales"].astype(np.float64), 128, axis=1))


def test_page_slot_by_hand():
    bt = np.array([[5, 2, 9], [0, 7, 1]], dtype=np.int32)
    assert O.page_slot(bt, 0, 0, 64) == 5 * 64
    assert O.page_slot(bt, 0, 63, 64) == 5 * 64 + 63
    assert O.page_slot(bt, 0, 64, 64) == 2 * 64
    assert O.page_slot(bt, 1, 130, 64) == 1 * 64 + 2


# --------------------------------------------------------------- the pages' numbers

def test_table1_mla_equals_gqa_with_2_25_groups():
    f = json.load(open(os.path.join(GOLDEN, "pages_facts.json")))
    m, t = f["v2_mla"], f["table1"]
    assert m["d_c"] == t["d_c_over_d_h"] * m["d_h"] and m["d_h_R"] == t["d_h_R_over_d_h"] * m["d_h"]
    mla = O.kv_elements_per_token("MLA", n_h=m["n_h"], d_h=m["d_h"], l=1, d_c=m["d_c"], d_r=m["d_h_R"])
    gqa1 = O.kv_elements_per_token("GQA", n_h=m["n_h"], d_h=m["d_h"], l=1, n_g=1)
    assert mla / gqa1 == t["gqa_equivalent_groups"]
    assert O.kv_elements_per_token("MHA", n_h=128, d_h=128, l=60) / (mla * 60) == pytest.approx(2 * 128 / 4.5)


def test_kv_cache_reduction_93_3_percent():
    """93.3% follows from 60 layers x 576 elements x 6 bit against 95 layers x 8 groups x
    2 x 128 x 16 bit (the 67B head dim 128 and bf16 cache are assumptions)."""
    f = json.load(open(os.path.join(GOLDEN, "pages_facts.json")))
    m, s, g = f["v2_mla"], f["serving"], f["llm_67b"]
    v2 = O.kv_elements_per_token("MLA", n_h=m["n_h"], d_h=m["d_h"], l=m["layers"], d_c=m["d_c"],
                                 d_r=m["d_h_R"]) * s["kv_bits_per_element_v2"]
    ds67 = O.kv_elements_per_token("GQA", n_h=g["heads"], d_h=128, l=g["layers"], n_g=g["kv_groups"]) * 16
    assert round(100 * (1 - v2 / ds67), 1) == s["kv_cache_reduction_vs_67b_percent"]


def test_yarn_entropy_factor():
    f = json.load(open(os.path.join(GOLDEN, "pages_facts.json")))
    y = f["yarn"]
    assert O.yarn_mscale_sqrt_t(y["s"]) == pytest.approx(y["sqrt_t_coeff"] * math.log(40) + 1)
    assert O.yarn_mscale_sqrt_t(1.0) == 1.0


# ---------------------------------------------------------------------------- YaRN (section 3.1.4)

def _yarn_facts():
    y = json.load(open(os.path.join(GOLDEN, "pages_facts.json")))["yarn"]
    return y["s"], y["alpha"], y["beta"], y


def test_yarn_scale_factor_matches_the_pages_contexts():
    # the pages extend a 4K context with s = 40 to a 160K target
    s, _, _, y = _yarn_facts()
    assert int(y["orig_context"].rstrip("K")) * s == int(y["target_context"].rstrip("K"))


def test_yarn_ramp_endpoints_continuity_and_monotonicity():
    _, a, b, _ = _yarn_facts()
    r = np.linspace(0.0, 2 * b, 20001)
    g = O.yarn_ramp(r, a, b)
    assert np.all(g[r <= a] == 0.0) and np.all(g[r >= b] == 1.0)
    assert np.all(np.diff(g) >= 0.0)                        # never decreasing
    assert np.max(np.abs(np.diff(g))) <= (r[1] - r[0]) / (b - a) + 1e-12   # no jump anywhere
    assert O.yarn_ramp((a + b) / 2, a, b) == pytest.approx(0.5)


def test_yarn_frequencies_interpolate_slow_pairs_and_keep_fast_ones():
    s, a, b, _ = _yarn_facts()
    d, theta, L = 64, 10000.0, 4096
    base = O.rope_inv_freq(d, theta)
    f = O.yarn_inv_freq(d, theta, s, a, b, L)
    turns = L * base / (2 * math.pi)          # turns of each pair over the original context
    slow, fast = turns < a, turns > b
    assert slow.any() and fast.any() and (~slow & ~fast).any()   # the DeepSeek-V2 setting has all three regimes
    # fast pairs (many turns over the original context) are left as they are
    np.testing.assert_array_equal(f[fast], base[fast])
    # slow pairs are position-interpolated: over the extended context s L they turn exactly
    # as far as they used to over L
    np.testing.assert_allclose(s * L * f[slow], L * base[slow], rtol=1e-13)
    # in between, the slowdown factor lies strictly between 1/s and 1, and faster pairs are slowed less
    mid = ~slow & ~fast
    ratio = f / base
    assert np.all((ratio[mid] > 1 / s) & (ratio[mid] < 1))
    assert np.all(np.diff(ratio) <= 1e-15)    # pairs are ordered from fast (m = 0) to slow
    # s <= 1 is plain RoPE
    np.testing.assert_array_equal(O.yarn_inv_freq(d, theta, 1.0, a, b, L), base)


def test_yarn_rope_keeps_norm_and_relative_position_property():
    s, a, b, _ = _yarn_facts()
    rng = np.random.default_rng(5)
    f = O.yarn_inv_freq(64, 1e4, s, a, b, 4096)
    q, k = rng.standard_normal(64), rng.standard_normal(64)
    for m, n in [(100000, 99000), (5, 0), (131071, 130000)]:
        qm, kn = O.rope(q, m, 1e4, inv_freq=f), O.rope(k, n, 1e4, inv_freq=f)
        q2, k2 = O.rope(q, m + 777, 1e4, inv_freq=f), O.rope(k, n + 777, 1e4, inv_freq=f)
        assert qm @ kn == pytest.approx(q2 @ k2, rel=1e-9, abs=1e-9)
        assert np.linalg.norm(qm) == pytest.approx(np.linalg.norm(q))


def test_yarn_logit_factor_is_what_scaling_query_and_key_by_sqrt_t_does():
    # Section 3.1.4 gives sqrt(t) = 0.0707 ln s + 1 as a factor on the query and on the key (as in
    # YaRN). Scale a query and a key each by that factor, rotate both with the YaRN frequencies, and
    # their dot product must be the unscaled one times yarn_logit_factor(s): a factor that used
    # sqrt(t) instead of t, or squared it twice, fails here.
    s, a, b, y = _yarn_facts()
    rng = np.random.default_rng(11)
    f = O.yarn_inv_freq(64, 1e4, s, a, b, 4096)
    sq = O.yarn_mscale_sqrt_t(s)
    for m, n in [(130000, 1234), (77, 76), (4095, 0)]:
        q, k = rng.standard_normal(64), rng.standard_normal(64)
        plain = O.rope(q, m, 1e4, inv_freq=f) @ O.rope(k, n, 1e4, inv_freq=f)
        scaled = O.rope(sq * q, m, 1e4, inv_freq=f) @ O.rope(sq * k, n, 1e4, inv_freq=f)
        assert scaled == pytest.approx(O.yarn_logit_factor(s, y["sqrt_t_coeff"]) * plain, rel=1e-12)
    assert O.yarn_logit_factor(1.0) == 1.0


def test_yarn_logit_factor_on_the_scale_equals_scaled_explicit_queries_and_keys():
    # The decode applies t as a factor on the softmax scale of the absorbed form. The same result
    # must come from the explicit form of sections 2.1.2-2.1.3 whose whole query [q_C ; q_R] and
    # whole key [W_UK c ; k_R] are each multiplied by sqrt(t) (the values W_UV c are not).
    s, _, _, _ = _yarn_facts()
    rng = np.random.default_rng(12)
    d_h, d_c, d_r, L = 16, 32, 8, 37
    qn, qr = rng.standard_normal(d_h), rng.standard_normal(d_r)
    w_uk, w_uv = 0.3 * rng.standard_normal((d_h, d_c)), 0.3 * rng.standard_normal((d_h, d_c))
    c, kr = rng.standard_normal((L, d_c)), rng.standard_normal((L, d_r))
    scale = 1 / math.sqrt(d_h + d_r)
    sq = O.yarn_mscale_sqrt_t(s)
    want, p_want = O.head_explicit(sq * qn, sq * qr, sq * w_uk, w_uv, c, sq * kr, scale)
    got, p_got = O.head_absorbed(qn, qr, w_uk, w_uv, c, kr, scale * O.yarn_logit_factor(s))
    np.testing.assert_allclose(p_got, p_want, rtol=1e-11, atol=1e-14)
    np.testing.assert_allclose(got, want, rtol=1e-10, atol=1e-12)
    # and the factor is not a no-op here: without it the weights differ
    _, p_plain = O.head_absorbed(qn, qr, w_uk, w_uv, c, kr, scale)
    assert np.max(np.abs(p_plain - p_want)) > 1e-3


# ---------------------------------------------------------------------------- several new tokens per sequence

def _causal_brute_force(q_nope, q_rope, w_uk, w_uv, c, kr, scale, q):
    """Textbook causal attention of the last q positions over a cache of L rows: query k sits at
    position L - q + k and may attend to positions j <= L - q + k (a 0 / -inf mask on the logits)."""
    H, d_h, _ = len(w_uk), len(w_uk[0]), len(w_uk[0][0])
    L = len(c)
    out = np.zeros((q, H, d_h))
    for k in range(q):
        for i in range(H):
            keys = [np.concatenate([np.asarray(w_uk[i]) @ c[j], kr[j]]) for j in range(L)]
            vals = [np.asarray(w_uv[i]) @ c[j] for j in range(L)]
            qq = np.concatenate([q_nope[k][i], q_rope[k][i]])
            logits = [scale * float(qq @ keys[j]) if j <= L - q + k else -math.inf for j in range(L)]
            mx = max(logits)
            w = [math.exp(z - mx) for z in logits]
            out[k, i] = sum(wj * vj for wj, vj in zip(w, vals)) / sum(w)
    return out


def test_multi_token_decode_is_causal_attention():
    rng = np.random.default_rng(8)
    H, d_h, d_c, d_r, q = 2, 4, 6, 2, 3
    lens = [5, 9]
    w_uk, w_uv = rng.standard_normal((H, d_h, d_c)), rng.standard_normal((H, d_h, d_c))
    qn, qr = rng.standard_normal((2, q, H, d_h)), rng.standard_normal((2, q, H, d_r))
    cs = [rng.standard_normal((L, d_c)) for L in lens]
    ks = [rng.standard_normal((L, d_r)) for L in lens]
    got = O.decode_multi(qn, qr, w_uk, w_uv, cs, ks, 0.41)
    for b in range(2):
        want = _causal_brute_force(qn[b], qr[b], w_uk, w_uv, cs[b], ks[b], 0.41, q)
        np.testing.assert_allclose(got[b], want, rtol=1e-11, atol=1e-12)


def test_multi_token_decode_reduces_to_decode_and_ignores_the_future():
    rng = np.random.default_rng(9)
    H, d_h, d_c, d_r, q, L = 3, 4, 5, 2, 4, 12
    w_uk, w_uv = rng.standard_normal((H, d_h, d_c)), rng.standard_normal((H, d_h, d_c))
    qn, qr = rng.standard_normal((1, q, H, d_h)), rng.standard_normal((1, q, H, d_r))
    c, kr = rng.standard_normal((L, d_c)), rng.standard_normal((L, d_r))
    got = O.decode_multi(qn, qr, w_uk, w_uv, [c], [kr], 0.3)
    # the last new token sees the whole cache: plain decode
    np.testing.assert_allclose(got[0, -1], O.decode(qn[:, -1], qr[:, -1], w_uk, w_uv, [c], [kr], 0.3)[0],
                               rtol=1e-13, atol=1e-14)
    # changing the rows after new token k's position leaves its output unchanged
    c2, kr2 = c.copy(), kr.copy()
    c2[L - 2:] += 5.0
    kr2[L - 2:] -= 3.0
    got2 = O.decode_multi(qn, qr, w_uk, w_uv, [c2], [kr2], 0.3)
    np.testing.assert_array_equal(got2[0, :q - 2], got[0, :q - 2])
    assert np.abs(got2[0, q - 2] - got[0, q - 2]).max() > 1e-3


def test_prefill_is_the_multi_token_decode_over_every_position():
    # prefill (every prompt token a query, causal) is the multi-token decode with q = L; its
    # explicit form (per-head K and V materialised, as prefill kernels compute it) agrees with
    # the absorbed one
    rng = np.random.default_rng(10)
    H, d_h, d_c, d_r, L = 2, 4, 6, 2, 7
    w_uk, w_uv = rng.standard_normal((H, d_h, d_c)), rng.standard_normal((H, d_h, d_c))
    qn, qr = rng.standard_normal((1, L, H, d_h)), rng.standard_normal((1, L, H, d_r))
    c, kr = rng.standard_normal((L, d_c)), rng.standard_normal((L, d_r))
    a = O.decode_multi(qn, qr, w_uk, w_uv, [c], [kr], 0.5, form="absorbed")
    e = O.decode_multi(qn, qr, w_uk, w_uv, [c], [kr], 0.5, form="explicit")
    np.testing.assert_allclose(a, e, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(a[0], _causal_brute_force(qn[0], qr[0], w_uk, w_uv, c, kr, 0.5, L), rtol=1e-11,
                               atol=1e-12)
    # the first token attends only to itself: its value
    np.testing.assert_allclose(a[0, 0], np.einsum("hdk,k->hd", w_uv, c[0]), rtol=1e-12, atol=1e-13)


def _prefill_case(seed, lens, n_new, H=3, d_h=4, d_c=6, d_r=2):
    rng = np.random.default_rng(seed)
    w_uk, w_uv = rng.standard_normal((H, d_h, d_c)), rng.standard_normal((H, d_h, d_c))
    cs = [rng.standard_normal((L, d_c)) for L in lens]
    ks = [rng.standard_normal((L, d_r)) for L in lens]
    T = int(sum(n_new))
    qn, qr = rng.standard_normal((T, H, d_h)), rng.standard_normal((T, H, d_r))
    return qn, qr, w_uk, w_uv, cs, ks


def test_prefill_is_causal_attention_with_ragged_new_tokens():
    # whole prompts, a chunk after a cached prefix, a sequence with no new token
    lens, n_new = [7, 10, 4, 1], [7, 3, 0, 1]
    qn, qr, w_uk, w_uv, cs, ks = _prefill_case(11, lens, n_new)
    got = O.prefill(qn, qr, w_uk, w_uv, cs, ks, n_new, 0.37)
    r = 0
    for b, (L, n) in enumerate(zip(lens, n_new)):
        if n:
            want = _causal_brute_force(qn[r:r + n], qr[r:r + n], w_uk, w_uv, cs[b], ks[b], 0.37, n)
            np.testing.assert_allclose(got[r:r + n], want, rtol=1e-11, atol=1e-12)
        r += n
    assert r == len(got)


def test_prefill_chunks_compose_and_end_in_the_plain_decode():
    L, a = 11, 4
    qn, qr, w_uk, w_uv, cs, ks = _prefill_case(12, [L], [L])
    whole = O.prefill(qn, qr, w_uk, w_uv, cs, ks, [L], 0.29)
    # the first a tokens as a prompt of their own, then the rest as a chunk over the whole cache
    first = O.prefill(qn[:a], qr[:a], w_uk, w_uv, [cs[0][:a]], [ks[0][:a]], [a], 0.29)
    rest = O.prefill(qn[a:], qr[a:], w_uk, w_uv, cs, ks, [L - a], 0.29)
    np.testing.assert_allclose(np.concatenate([first, rest]), whole, rtol=1e-12, atol=1e-13)
    # the last prompt token sees every row: the absorbed single-token decode
    dec = O.decode(qn[-1:], qr[-1:], w_uk, w_uv, cs, ks, 0.29)
    np.testing.assert_allclose(whole[-1], dec[0], rtol=1e-10, atol=1e-12)
    # the first prompt token sees only itself: its value
    np.testing.assert_allclose(whole[0], np.einsum("hdk,k->hd", w_uv, cs[0][0]), rtol=1e-12, atol=1e-13)


def test_prefill_equals_the_absorbed_multi_token_decode():
    lens, q = [6, 9], 3
    qn, qr, w_uk, w_uv, cs, ks = _prefill_case(13, lens, [q, q])
    got = O.prefill(qn, qr, w_uk, w_uv, cs, ks, [q, q], 0.5)
    H, d_h = w_uk.shape[:2]
    multi = O.decode_multi(qn.reshape(2, q, H, d_h), qr.reshape(2, q, H, -1), w_uk, w_uv, cs, ks, 0.5,
                           form="absorbed")
    np.testing.assert_allclose(got, multi.reshape(2 * q, H, d_h), rtol=1e-10, atol=1e-12)


def test_prefill_subset_matches_the_full_result():
    lens, n_new = [8, 5], [8, 2]
    qn, qr, w_uk, w_uv, cs, ks = _prefill_case(14, lens, n_new)
    full = O.prefill(qn, qr, w_uk, w_uv, cs, ks, n_new, 0.4)
    part = O.prefill(qn, qr, w_uk, w_uv, cs, ks, n_new, 0.4, heads=[1], rows=[0, 7, 9])
    for r in range(len(full)):
        for i in range(full.shape[1]):
            if i == 1 and r in (0, 7, 9):
                np.testing.assert_array_equal(part[r, i], full[r, i])
            else:
                assert np.isnan(part[r, i]).all()


def test_hidden_output_is_the_folded_latent_output():
    # W_O [W_UV_i o_lat_i]_i computed from the explicit outputs equals the fold W_OUV o_lat of the
    # absorbed form (the output-side absorption of section 2.1.2)
    rng = np.random.default_rng(15)
    H, d_h, d_c, d_r, hidden = 3, 4, 6, 2, 7
    w_uk, w_uv = rng.standard_normal((H, d_h, d_c)), rng.standard_normal((H, d_h, d_c))
    w_o = rng.standard_normal((hidden, H * d_h))
    lens = [5, 1, 8]
    cs = [rng.standard_normal((L, d_c)) for L in lens]
    ks = [rng.standard_normal((L, d_r)) for L in lens]
    qn, qr = rng.standard_normal((3, H, d_h)), rng.standard_normal((3, H, d_r))
    got = O.decode_hidden(qn, qr, w_uk, w_uv, w_o, cs, ks, 0.45)
    w_ouv = O.fold_output_weight(w_uv, w_o)
    assert w_ouv.shape == (hidden, H * d_c)
    for b, L in enumerate(lens):
        o_lat = []
        for i in range(H):
            q_lat = w_uk[i].T @ qn[b, i]
            a = O.softmax_probs(0.45 * (cs[b] @ q_lat + ks[b] @ qr[b, i]))
            o_lat.append(a @ cs[b])
        np.testing.assert_allclose(got[b], w_ouv @ np.concatenate(o_lat), rtol=1e-10, atol=1e-12)


def test_hidden_output_with_identity_projection_is_the_head_concatenation():
    rng = np.random.default_rng(16)
    H, d_h, d_c, d_r = 2, 3, 5, 2
    w_uk, w_uv = rng.standard_normal((H, d_h, d_c)), rng.standard_normal((H, d_h, d_c))
    cs, ks = [rng.standard_normal((4, d_c))], [rng.standard_normal((4, d_r))]
    qn, qr = rng.standard_normal((1, H, d_h)), rng.standard_normal((1, H, d_r))
    got = O.decode_hidden(qn, qr, w_uk, w_uv, np.eye(H * d_h), cs, ks, 0.6)
    per_head = O.decode(qn, qr, w_uk, w_uv, cs, ks, 0.6, form="absorbed")
    np.testing.assert_allclose(got[0], per_head[0].reshape(-1), rtol=1e-11, atol=1e-13)
    # and a projection that keeps only head 1's first value picks it out
    w_o = np.zeros((1, H * d_h))
    w_o[0, d_h] = 1.0
    np.testing.assert_allclose(O.decode_hidden(qn, qr, w_uk, w_uv, w_o, cs, ks, 0.6)[0, 0], per_head[0, 1, 0],
                               rtol=1e-12)
