"""GPU parity of the W_UV-into-W_O fold: mla_fold_output_weight against the oracle's fold, and
mla_decode_hidden (the decode taken to the hidden size by one GEMM over the latent outputs) against
the oracle's W_O over the per-head outputs. Expected values come only from the oracle."""
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


def test_fold_matches_the_oracle_fold():
    import head_latent_attention_22_b300 as M
    shape = S.SHAPES["dsv2_b16"]
    inp = S.make_inputs(S.shape_with("dsv2_b16", batch=1, lengths=(64,)))
    w_o = S.draw_w_o(shape, 1024)
    cfg = M.MLAConfig.from_shape(shape)
    got = M.fold_output_weight(cfg, inp.w_uv.cuda(), w_o.cuda())
    torch.cuda.synchronize()
    got = got.float().cpu().numpy()
    want = O.fold_output_weight(inp.w_uv.double().numpy(), w_o.double().numpy())
    # fp32 sums of 128 products, then one rounding to fp16: within one fp16 step of the exact value
    # (relative 2^-10 for normal values, 2^-24 absolute below fp16's normal range)
    err = np.abs(got - want)
    assert (err <= np.abs(want) * 2.0 ** -10 + 2.0 ** -24).all(), err.max()


@pytest.mark.parametrize("lengths", [(1, 64, 700, 1500), (4096,) * 2 + (65, 130, 3, 0, 999, 2047)])
def test_decode_hidden_matches_the_oracle(lengths):
    import head_latent_attention_22_b300 as M
    shape = S.shape_with("dsv2_b16", batch=len(lengths), lengths=lengths)
    inp = S.make_inputs(shape)
    dc = T.to_device(inp)
    T.fill_cache(dc)
    w_o = S.draw_w_o(shape, 5120)
    w_ouv = M.fold_output_weight(dc.cfg, dc.w_uv, w_o.cuda())
    L = max(1, int(inp.lengths.max()))
    got = M.decode_hidden(dc.cfg, dc.q_nope, dc.q_rope, dc.w_uk, w_ouv, dc.pool, dc.block_table, dc.seq_lens, L)
    M.check_device_errors()
    got = got.cpu().numpy()
    cs, ks = zip(*[T.oracle_cache(inp, b) for b in range(shape.batch)])
    want = O.decode_hidden(inp.q_nope.double().numpy(), inp.q_rope.double().numpy(), inp.w_uk.double().numpy(),
                           inp.w_uv.double().numpy(), w_o.double().numpy(), cs, ks, T.oracle_scale(shape),
                           form="absorbed")
    T.assert_close(got, want, "bf16", f"decode_hidden {lengths}")


def test_decode_hidden_refuses_large_batches():
    import head_latent_attention_22_b300 as M
    cfg = M.MLAConfig.from_shape(S.SHAPES["dsv2_b16"])
    assert M.decode_hidden_workspace_size(cfg, 129, 4096, 5120) == 0
    assert M.decode_hidden_workspace_size(cfg, 128, 4096, 5120) > 0
    assert M.decode_hidden_workspace_size(cfg, 16, 4096, 5000) == 0
