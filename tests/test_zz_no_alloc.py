"""mla_decode_static_scratch: the decode entry point that allocates nothing.

Some callers of this library cannot allocate device memory when they decode
(a plugin inside a host program that owns all device memory, or a serving
loop with a fixed memory plan that must not call cudaMalloc). For them the
library keeps one fixed scratch array per device. This test calls that entry
point through the C ABI twice in a row and checks each result against the
ordinary workspace-taking mla_decode, within the parity tolerance; the file
sorts last so that a run stopping at the first failure has run every other
test first.
"""
import numpy as np
import pytest
import torch

import mla_synth as S
from tests import mla_testlib as T

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from head_latent_attention_22_b300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


@pytest.mark.parametrize("name,over", [("dsv2_b16", dict(batch=4, lengths=(1, 64, 700, 4096))),
                                       ("tiny_fp32", None)])
def test_static_scratch_decode_matches_workspace_decode(name, over):
    import head_latent_attention_22_b300 as M
    shape = S.SHAPES[name] if over is None else S.shape_with(name, **over)
    inp = S.make_inputs(shape)
    dc = T.to_device(inp)
    T.fill_cache(dc)
    L = int(inp.lengths.max())
    ref = M.decode(dc.cfg, dc.q_nope, dc.q_rope, dc.w_uk, dc.w_uv, dc.pool, dc.block_table, dc.seq_lens, L)
    M.check_device_errors()
    ref = ref.cpu().numpy()
    out = torch.empty((shape.batch, shape.n_heads, shape.d_head), dtype=torch.float32, device="cuda")
    for call in range(2):
        out.fill_(float("nan"))
        M.decode_static_scratch(dc.cfg, dc.q_nope, dc.q_rope, dc.w_uk, dc.w_uv, dc.pool, dc.block_table,
                                dc.seq_lens, L, out)
        M.check_device_errors()
        T.assert_close(out.cpu().numpy(), ref, shape.cache_dtype, f"{name} call {call}")
    # and on its own against the fp64 oracle, every output
    pairs = [(b, i) for b in range(shape.batch) for i in range(shape.n_heads)]
    want = T.oracle_outputs(inp, pairs).reshape(out.shape)
    T.assert_close(out.cpu().numpy(), want, shape.cache_dtype, f"{name} vs oracle")


def test_static_scratch_refuses_oversized_requests():
    import head_latent_attention_22_b300 as M
    cfg = M.MLAConfig.dsv2()
    B, L = 256, 131072
    assert M.workspace_size(cfg, B, L) > (48 << 20)
    dev = "cuda"
    q = torch.zeros((B, 128, 128), dtype=torch.bfloat16, device=dev)
    qr = torch.zeros((B, 128, 64), dtype=torch.bfloat16, device=dev)
    w = torch.zeros((128, 128, 512), dtype=torch.bfloat16, device=dev)
    pool = M.new_pool(cfg, 1, dev)
    bt = torch.zeros((B, L // 64), dtype=torch.int32, device=dev)
    lens = torch.zeros(B, dtype=torch.int32, device=dev)
    out = torch.empty((B, 128, 128), dtype=torch.float32, device=dev)
    with pytest.raises(M.MLAError) as e:
        M.decode_static_scratch(cfg, q, qr, w, w, pool, bt, lens, L, out)
    assert e.value.status == 1 and "scratch" in str(e.value)
