"""YaRN-extended decoupled RoPE on the GPU against the oracle (needs a B300).

The report's 128K setting (section 3.1.4): s = 40, alpha = 1, beta = 32 over a
4K pre-training context, logits multiplied by (0.0707 ln s + 1)^2. Checked:
the rope keys mla_append writes at positions across the extended context, the
queries mla_rope_query rotates, and decode outputs with the logit factor.
"""
import dataclasses

import numpy as np
import pytest
import torch

import mla_synth as S
from oracle import mla_oracle as O
from tests import mla_testlib as T

pytestmark = pytest.mark.gpu

POSITIONS = [0, 1, 63, 4095, 4096, 65537, 100000, 131071]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from head_latent_attention_22_b300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def _cfg():
    import head_latent_attention_22_b300 as M
    return dataclasses.replace(M.MLAConfig.dsv2(), yarn_factor=40.0)


def _bf16_step(x):
    x = np.abs(np.asarray(x, np.float64))
    e = np.floor(np.log2(np.maximum(x, 2.0**-126)))
    return np.ldexp(1.0, (e - 7).astype(np.int64))


def _oracle_freq(cfg):
    return O.yarn_inv_freq(cfg.d_rope, cfg.rope_theta, cfg.yarn_factor, cfg.yarn_alpha, cfg.yarn_beta,
                           cfg.yarn_orig_len)


def test_append_rope_keys_across_the_extended_context():
    import head_latent_attention_22_b300 as M
    cfg = _cfg()
    gen = torch.Generator().manual_seed(11)
    n = len(POSITIONS)
    c_raw = torch.randn(n, 512, generator=gen).to(torch.bfloat16)
    k_raw = torch.randn(n, 64, generator=gen).to(torch.bfloat16)
    max_pages = 131072 // 64
    pool = M.new_pool(cfg, max_pages, "cuda", fill=0)
    pos = torch.tensor(POSITIONS, dtype=torch.int32)
    seq = torch.zeros(n, dtype=torch.int32)
    M.append(cfg, c_raw.cuda(), k_raw.cuda(), pos.cuda(), pool, None, seq_idx=seq.cuda(), batch=1,
             max_pages=max_pages)
    M.check_device_errors()
    rows = pool.view(-1, 1152)[pos.long().cuda()].cpu()
    kr = rows[:, 1024:].contiguous().view(torch.bfloat16).double().numpy()
    want = O.rope(k_raw.double().numpy(), np.array(POSITIONS), cfg.rope_theta, inv_freq=_oracle_freq(cfg))
    assert np.all(np.abs(kr - want) <= _bf16_step(want) * 1.0000001)
    # and it is not plain RoPE: at the far positions the slow pairs differ
    plain = O.rope(k_raw.double().numpy(), np.array(POSITIONS), cfg.rope_theta)
    assert np.abs(kr[-1] - plain[-1]).max() > 0.1


def test_rope_query_matches_the_keys_rotation():
    import head_latent_attention_22_b300 as M
    cfg = _cfg()
    gen = torch.Generator().manual_seed(12)
    B = 3
    q_raw = torch.randn(B, 128, 64, generator=gen).to(torch.bfloat16)
    pos = torch.tensor([5, 70000, 131071], dtype=torch.int32)
    got = M.rope_query(cfg, q_raw.cuda(), pos.cuda()).cpu().double().numpy()
    want = O.rope(q_raw.double().numpy(), pos.numpy()[:, None], cfg.rope_theta, inv_freq=_oracle_freq(cfg))
    assert np.all(np.abs(got - want) <= _bf16_step(want) * 1.0000001)
    # in place gives the same
    q_dev = q_raw.cuda()
    M.rope_query(cfg, q_dev, pos.cuda(), out=q_dev)
    np.testing.assert_array_equal(q_dev.cpu().double().numpy(), got)
    M.check_device_errors()


def test_decode_with_the_yarn_logit_factor():
    shape = S.shape_with("yarn_b4", batch=3, lengths=(1, 333, 2000))
    inp = S.make_inputs(shape)
    dc = T.to_device(inp)
    assert dc.cfg.yarn_factor == 40.0
    T.fill_cache(dc)
    got = T.run_decode(dc)
    pairs = [(b, i) for b in range(shape.batch) for i in range(shape.n_heads)]
    want = T.oracle_outputs(inp, pairs).reshape(shape.batch, shape.n_heads, shape.d_head)
    T.assert_close(got, want, "bf16", "yarn decode")
    # without the logit factor the 2000-token sequence's outputs would be visibly different
    last = [(2, i) for i in range(shape.n_heads)]
    plain = T.oracle_outputs(dataclasses.replace(inp, shape=dataclasses.replace(shape, yarn_mscale=0.0)), last)
    assert np.abs(plain - want[2]).max() > 10 * 1e-2 * np.abs(want[2]).max()
