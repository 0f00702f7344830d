"""GPU parity of the C-ABI library against the fp64 oracle (needs a B300).

Append: every written cache row is compared with the oracle's row in the
storage format; placement through the page table is bit-exact (untouched
pool bytes keep a sentinel). Decode: all outputs at small sizes spanning
several pages and ragged tails, sampled (sequence, head) outputs at the full
workload sizes, plus the degenerate cases (empty and one-token sequences,
lengths at page boundaries).
"""
import numpy as np
import pytest
import torch

import mla_synth as S
from oracle import mla_oracle as O
from tests import mla_testlib as T

pytestmark = pytest.mark.gpu

SENTINEL = 0xAB


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from head_latent_attention_22_b300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def _ulp_bf16(x):
    x = np.abs(np.asarray(x, np.float64))
    e = np.floor(np.log2(np.maximum(x, 2.0**-126)))
    return np.ldexp(1.0, (e - 7).astype(np.int64))


def _rows_written(inp):
    slots = []
    for b, n in enumerate(inp.lengths):
        for p in range(int(n)):
            slots.append(O.page_slot(inp.block_table, b, p, inp.shape.page_size))
    return np.array(slots, dtype=np.int64)


def _check_near(got, want, ulp, max_frac, what):
    diff = np.abs(got - want)
    bad = diff > 0
    assert np.all(diff <= ulp * 1.0000001), f"{what}: off by more than one step, max {diff.max()}"
    assert bad.mean() <= max_frac, f"{what}: {bad.sum()} of {bad.size} differ by one step"


def c_want_unrounded(inp, shape):
    """The oracle's latent before any storage rounding (fp64)."""
    return O.rmsnorm(inp.c_kv_raw.double().numpy(), shape.eps)


APPEND_CASES = [
    ("tiny_fp32", None),
    ("dsv2_b16", dict(batch=3, lengths=(1, 64, 129))),
    ("fp8_b32", dict(batch=3, lengths=(1, 100, 257))),
]


@pytest.mark.parametrize("name,over", APPEND_CASES)
def test_append_rows_and_placement(name, over):
    shape = S.SHAPES[name] if over is None else S.shape_with(name, **over)
    inp = S.make_inputs(shape)
    dc = T.to_device(inp, pool_fill=SENTINEL)
    T.fill_cache(dc)
    import head_latent_attention_22_b300 as M
    M.check_device_errors()
    pool = dc.pool.cpu().numpy().reshape(-1, dc.pool.shape[-1])
    slots = _rows_written(inp)
    assert len(np.unique(slots)) == len(slots)
    untouched = np.ones(pool.shape[0], bool)
    untouched[slots] = False
    assert np.all(pool[untouched] == SENTINEL), "bytes outside the written rows changed"
    rows = pool[slots]
    pos = inp.positions()
    c_want, kr_want, extra = O.append_rows(inp.c_kv_raw.double().numpy(), inp.k_rope_raw.double().numpy(), pos,
                                           cache_dtype=shape.cache_dtype, eps=shape.eps, theta=shape.rope_theta)
    d_c, d_r = shape.d_c, shape.d_rope
    if shape.cache_dtype == "fp32":
        v = rows.view(np.float32).astype(np.float64)
        np.testing.assert_allclose(v[:, :d_c], c_want, rtol=4 * 2.0**-24, atol=1e-30)
        np.testing.assert_allclose(v[:, d_c:], kr_want, rtol=2 * 2.0**-24, atol=1e-30)
    elif shape.cache_dtype == "bf16":
        v = torch.from_numpy(rows.copy()).view(torch.bfloat16).double().numpy()
        _check_near(v[:, :d_c], c_want, _ulp_bf16(c_want), 1e-3, "latent")
        _check_near(v[:, d_c:], kr_want, _ulp_bf16(kr_want), 1e-4, "rope key")
    else:
        codes = torch.from_numpy(rows[:, :d_c].copy()).view(torch.float8_e4m3fn).double().numpy()
        scales = rows[:, d_c:d_c + 4 * (d_c // 128)].copy().view(np.float32)
        # the scale inherits the kernel's fp32 RMSNorm rounding (a few fp32 ulps from the oracle's)
        np.testing.assert_allclose(scales, extra["scales"], rtol=8 * 2.0**-24)
        # Codes must be equal, except where the exact ratio c / scale sits on a rounding tie
        # of E4M3 (common: bf16 inputs make 448 x / amax a short binary fraction); there the
        # last fp32 ulp picks the side, and either neighbour is a correct rounding.
        want_codes = extra["codes"]
        ratio = c_want_unrounded(inp, shape) / np.repeat(extra["scales"].astype(np.float64), 128, axis=1)
        diff = codes != want_codes
        mid = (codes + want_codes) / 2
        at_tie = np.abs(ratio - mid) <= 1e-6 * np.maximum(np.abs(mid), 2.0**-9)
        step = np.maximum(2.0 ** (np.floor(np.log2(np.maximum(np.abs(want_codes), 2.0**-6))) - 3), 2.0**-9)
        assert np.all(np.abs(codes - want_codes) <= step * 1.0000001), "e4m3 code off by more than one step"
        assert np.all(at_tie[diff]), f"{int((diff & ~at_tie).sum())} e4m3 codes differ away from a tie"
        kr = torch.from_numpy(rows[:, d_c + 4 * (d_c // 128):].copy()).view(torch.bfloat16).double().numpy()
        _check_near(kr, kr_want, _ulp_bf16(kr_want), 1e-4, "rope key")


DECODE_SMALL = [
    ("tiny_fp32", None),
    ("dsv2_b16", dict(batch=6, lengths=(1, 63, 64, 65, 700, 2049))),
    ("fp8_b32", dict(batch=3, lengths=(1, 130, 1000))),
]


@pytest.mark.parametrize("name,over", DECODE_SMALL)
def test_decode_all_outputs_small(name, over):
    shape = S.SHAPES[name] if over is None else S.shape_with(name, **over)
    inp = S.make_inputs(shape)
    dc = T.to_device(inp)
    T.fill_cache(dc)
    got = T.run_decode(dc)
    pairs = [(b, i) for b in range(shape.batch) for i in range(shape.n_heads)]
    want = T.oracle_outputs(inp, pairs).reshape(shape.batch, shape.n_heads, shape.d_head)
    T.assert_close(got, want, shape.cache_dtype, name)


@pytest.mark.parametrize("batch", [12, 4])
def test_merge_of_many_partials(batch):
    # one 40,000-token sequence beside 64-token ones: its tiles span most clusters' shares, so the
    # merge combines dozens of partials in several load groups. With 12 sequences the merge takes
    # four 4-element chunks per CTA and eight partials per group, with 4 one chunk and sixteen.
    shape = S.shape_with("dsv2_b16", batch=batch, lengths=(40000,) + (64,) * (batch - 1))
    inp = S.make_inputs(shape)
    dc = T.to_device(inp)
    T.fill_cache(dc)
    got = T.run_decode(dc)
    pairs = [(b, i) for b in (0, 1, batch - 1) for i in (0, 1, 63, 64, 127)]
    want = T.oracle_outputs(inp, pairs)
    T.assert_close(np.stack([got[b, i] for b, i in pairs]), want, shape.cache_dtype, f"merge b{batch}")


def test_decode_matches_explicit_form_too():
    shape = S.shape_with("dsv2_b16", batch=2, lengths=(77, 300))
    inp = S.make_inputs(shape)
    dc = T.to_device(inp)
    T.fill_cache(dc)
    got = T.run_decode(dc)
    pairs = [(0, 0), (0, 127), (1, 5), (1, 64)]
    want = T.oracle_outputs(inp, pairs, form="explicit")
    T.assert_close(np.stack([got[b, i] for b, i in pairs]), want, "bf16", "explicit")


def test_decode_empty_and_single_token_sequences():
    shape = S.shape_with("dsv2_b16", batch=3, lengths=(0, 1, 5))
    inp = S.make_inputs(shape)
    dc = T.to_device(inp)
    T.fill_cache(dc)
    got = T.run_decode(dc)
    assert np.all(got[0] == 0)
    w_uv = inp.w_uv.double().numpy()
    c, _ = T.oracle_cache(inp, 1)
    want = np.einsum("hdk,k->hd", w_uv, c[0])
    T.assert_close(got[1], want, "bf16", "one token")


def test_decode_is_deterministic():
    shape = S.shape_with("dsv2_b16", batch=2, lengths=(1000, 333))
    inp = S.make_inputs(shape)
    dc = T.to_device(inp)
    T.fill_cache(dc)
    a = T.run_decode(dc)
    b = T.run_decode(dc)
    np.testing.assert_array_equal(a, b)


def test_out_of_range_page_is_flagged_not_faulted():
    import head_latent_attention_22_b300 as M
    shape = S.shape_with("dsv2_b16", batch=2, lengths=(100, 100))
    inp = S.make_inputs(shape)
    dc = T.to_device(inp)
    T.fill_cache(dc)
    M.check_device_errors()
    bt = dc.block_table.clone()
    bt[1, 1] = inp.num_pages + 5           # outside the pool
    M.decode(dc.cfg, dc.q_nope, dc.q_rope, dc.w_uk, dc.w_uv, dc.pool, bt, dc.seq_lens, 100)
    with pytest.raises(M.MLAError) as e:
        M.check_device_errors()
    assert e.value.status == 5
    M.check_device_errors()               # the word was cleared
    pos = torch.tensor([70], dtype=torch.int32, device="cuda")
    M.append(dc.cfg, inp.c_kv_raw[:1].cuda(), inp.k_rope_raw[:1].cuda(), pos, dc.pool, bt,
             seq_idx=torch.tensor([1], dtype=torch.int32, device="cuda"))
    with pytest.raises(M.MLAError):
        M.check_device_errors()


FULL = ["dsv2_b16", "ragged_b64", "long_b4", "fp8_b32", "yarn_b4"]


# Outputs compared at full size: up to 16 sequences x 16 heads (first and last of each included),
# and for the ragged and 128K batches every sequence with 4 of those heads, so that every sequence
# whose tiles are cut between two clusters' shares is compared, whatever number of clusters fits.
FULL_SEQS = {"ragged_b64": None, "long_b4": None, "yarn_b4": None}


@pytest.mark.parametrize("name", FULL)
def test_decode_full_size_sampled(name):
    shape = S.SHAPES[name]
    inp = S.make_inputs(shape)
    dc = T.to_device(inp)
    T.fill_cache(dc)
    got = T.run_decode(dc)
    rng = np.random.default_rng(123)
    hs16 = sorted(set([0, shape.n_heads - 1] + list(rng.choice(np.arange(1, shape.n_heads - 1), 14, replace=False))))
    bs16 = sorted(set([0, shape.batch - 1] + list(rng.choice(shape.batch, min(shape.batch, 14), replace=False))))
    pairs = {(b, i) for b in bs16 for i in hs16}
    if name in FULL_SEQS:   # every sequence, with a few heads
        pairs |= {(b, i) for b in range(shape.batch) for i in hs16[::4]}
    pairs = sorted(pairs)
    want = T.oracle_outputs(inp, pairs)
    T.assert_close(np.stack([got[b, i] for b, i in pairs]), want, shape.cache_dtype, name)
