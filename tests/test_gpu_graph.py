"""The serving step captured as a CUDA graph (StepGraph) against eager calls (needs a B300).

Replaying the graph after writing a new step's inputs into its buffers must
give exactly the outputs of calling mla_append + mla_decode eagerly on the
same inputs (same kernels, same launch configuration, deterministic), and
those must match the oracle.
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


@pytest.mark.parametrize("name,over", [("dsv2_b16", dict(batch=3, lengths=(100, 64, 513))),
                                       ("fp8_b32", dict(batch=2, lengths=(7, 300)))])
def test_step_graph_replay_equals_eager(name, over):
    import head_latent_attention_22_b300 as M
    shape = S.shape_with(name, **over)
    inp = S.make_inputs(shape)
    dc = T.to_device(inp)
    T.fill_cache(dc)
    B = shape.batch
    L = int(inp.lengths.max())
    new_pos = torch.from_numpy((inp.lengths - 1).astype(np.int32)).cuda()
    new_seq = torch.arange(B, dtype=torch.int32, device="cuda")
    st0, st1 = S.draw_step(inp, 0), S.draw_step(inp, 1)
    ws = torch.empty(max(256, M.workspace_size(dc.cfg, B, L)), dtype=torch.uint8, device="cuda")

    # eager: step 1
    M.append(dc.cfg, st1.c_new.cuda(), st1.k_new.cuda(), new_pos, dc.pool, dc.block_table, seq_idx=new_seq)
    eager = M.decode(dc.cfg, st1.q_nope.cuda(), st1.q_rope.cuda(), dc.w_uk, dc.w_uv, dc.pool, dc.block_table,
                     dc.seq_lens, L, workspace=ws).clone()
    M.check_device_errors()

    # graph: captured on step 0's buffers, replayed after step 1's inputs are copied in
    bufs = [t.cuda() for t in (st0.q_nope, st0.q_rope, st0.c_new, st0.k_new)]
    out = torch.empty_like(eager)
    g = M.StepGraph(dc.cfg, c_new=bufs[2], k_new=bufs[3], positions=new_pos, seq_idx=new_seq, q_nope=bufs[0],
                    q_rope=bufs[1], w_uk=dc.w_uk, w_uv=dc.w_uv, pool=dc.pool, block_table=dc.block_table,
                    seq_lens=dc.seq_lens, max_seq_len=L, out=out, workspace=ws)
    for d, h in zip(bufs, (st1.q_nope, st1.q_rope, st1.c_new, st1.k_new)):
        d.copy_(h)
    got = g.replay()
    M.check_device_errors()
    np.testing.assert_array_equal(got.cpu().numpy(), eager.cpu().numpy())

    # and the oracle agrees with the step-1 state
    inp1 = S.with_step(inp, st1)
    pairs = [(b, i) for b in range(B) for i in (0, 37, 127)]
    want = T.oracle_outputs(inp1, pairs)
    gn = got.cpu().numpy()
    T.assert_close(np.stack([gn[b, i] for b, i in pairs]), want, shape.cache_dtype, "graph replay")
