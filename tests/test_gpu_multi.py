"""Decode of several new tokens per sequence (mla_decode_multi) against the oracle (needs a B300).

The cache holds every sequence's q new tokens as its last rows; new token k
attends causally to the rows up to its own. Compared: all outputs at small
sizes (ragged lengths, a sequence shorter than q), and q = 1 against mla_decode.
"""
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


def _queries(shape, q, seed):
    gen = torch.Generator().manual_seed(seed)
    qn = torch.randn(shape.batch, q, shape.n_heads, shape.d_head, generator=gen).to(torch.bfloat16)
    qr = torch.randn(shape.batch, q, shape.n_heads, shape.d_rope, generator=gen).to(torch.bfloat16)
    return qn, qr


@pytest.mark.parametrize("name,lengths,q", [("dsv2_b16", (3, 64, 65, 700), 3),
                                            ("dsv2_b16", (1, 2, 200), 2),
                                            ("fp8_b32", (90, 1000), 4)])
def test_multi_token_decode_matches_oracle(name, lengths, q):
    import head_latent_attention_22_b300 as M
    shape = S.shape_with(name, batch=len(lengths), lengths=lengths)
    inp = S.make_inputs(shape)
    dc = T.to_device(inp)
    T.fill_cache(dc)
    qn, qr = _queries(shape, q, 21 + q)
    got = M.decode_multi(dc.cfg, qn.cuda(), qr.cuda(), dc.w_uk, dc.w_uv, dc.pool, dc.block_table, dc.seq_lens,
                         int(max(lengths))).cpu().numpy()
    M.check_device_errors()
    cache = [T.oracle_cache(inp, b) for b in range(shape.batch)]
    want = O.decode_multi(qn.double().numpy(), qr.double().numpy(), inp.w_uk.double().numpy(),
                          inp.w_uv.double().numpy(), [c for c, _ in cache], [k for _, k in cache],
                          T.oracle_scale(shape))
    T.assert_close(got, want, shape.cache_dtype, f"{name} q={q}")


def test_multi_with_one_new_token_is_decode():
    import head_latent_attention_22_b300 as M
    shape = S.shape_with("dsv2_b16", batch=2, lengths=(129, 640))
    inp = S.make_inputs(shape)
    dc = T.to_device(inp)
    T.fill_cache(dc)
    L = int(max(shape.lengths))
    one = M.decode(dc.cfg, dc.q_nope, dc.q_rope, dc.w_uk, dc.w_uv, dc.pool, dc.block_table, dc.seq_lens, L)
    multi = M.decode_multi(dc.cfg, dc.q_nope[:, None].contiguous(), dc.q_rope[:, None].contiguous(), dc.w_uk,
                           dc.w_uv, dc.pool, dc.block_table, dc.seq_lens, L)
    np.testing.assert_array_equal(multi[:, 0].cpu().numpy(), one.cpu().numpy())
