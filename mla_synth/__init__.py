"""Seeded synthetic inputs for MLA decode over a paged latent KV cache.

This module only draws numbers and lays out page tables. It holds none of the
attention arithmetic: no normalisation, no rotation, no rounding beyond the
dtype cast of the drawn values. Both the fp64 oracle and the CUDA path are fed
from here, so that they see exactly the same values.

Shapes follow the MLA hyper-parameters of the DeepSeek-V2 report (translated
page, section 3.1.2 "Hyper-parameters": n_h = 128, d_h = 128, d_c = 512,
d_h^R = 64, init std 0.006, hidden 5120). The five workloads are:

  tiny_fp32   B=2,  H=4,   d_c=32,  d_r=8,  d_h=16,  L = {17, 64}, contiguous, fp32
  dsv2_b16    B=16, DSV2 shapes, L = 4096 each, 64-token pages shuffled, bf16
  ragged_b64  B=64, DSV2 shapes, old length U[1, 32768] + one appended token, bf16
  long_b4     B=4,  DSV2 shapes, L = 131072 each (128K context), bf16
  fp8_b32     B=32, DSV2 shapes, L = 8192 each, E4M3 cache with fp32 scale per 128

and, for prefill (every cached row of a prompt is also a query), prefill_b4: four
DSV2-shaped prompts of 4096 tokens (draw_prefill gives their queries).

Random streams use torch's CPU generator (bf16 values are drawn in fp32 and
cast by torch), seeded per workload; every array is returned on the CPU.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np
import torch

BF16 = "bf16"
FP32 = "fp32"
FP8 = "fp8_e4m3_b128"


@dataclasses.dataclass(frozen=True)
class MLAShape:
    """Static description of one workload."""

    name: str
    batch: int
    n_heads: int
    d_c: int
    d_rope: int
    d_head: int
    page_size: int
    io_dtype: str          # dtype of queries, weights and raw latent/rope inputs
    cache_dtype: str       # storage format of the paged latent cache
    w_std: float           # std of W_UK / W_UV entries
    scale: float           # softmax scale
    seed: int
    lengths: Optional[tuple] = None   # fixed lengths (None => drawn, see ragged)
    ragged_max: int = 0               # old lengths drawn U[1, ragged_max], +1 appended
    paged: bool = True                # False => contiguous [B, max_seq] layout
    eps: float = 1e-6
    rope_theta: float = 10000.0
    yarn_factor: float = 1.0          # YaRN scale s of the decoupled RoPE; <= 1: plain RoPE
    yarn_alpha: float = 1.0
    yarn_beta: float = 32.0
    yarn_mscale: float = 0.0707
    yarn_orig_len: int = 4096

    @property
    def row_elems(self) -> int:
        return self.d_c + self.d_rope


DSV2_W_STD = 0.006 * math.sqrt(5120 / 512)

SHAPES = {
    "tiny_fp32": MLAShape("tiny_fp32", 2, 4, 32, 8, 16, 64, FP32, FP32, 0.2,
                          1.0 / math.sqrt(16 + 8), 0, lengths=(17, 64), paged=False),
    "dsv2_b16": MLAShape("dsv2_b16", 16, 128, 512, 64, 128, 64, BF16, BF16, DSV2_W_STD,
                         1.0 / math.sqrt(192), 1, lengths=(4096,) * 16),
    "ragged_b64": MLAShape("ragged_b64", 64, 128, 512, 64, 128, 64, BF16, BF16, DSV2_W_STD,
                           1.0 / math.sqrt(192), 2, ragged_max=32768),
    "long_b4": MLAShape("long_b4", 4, 128, 512, 64, 128, 64, BF16, BF16, DSV2_W_STD,
                        1.0 / math.sqrt(192), 3, lengths=(131072,) * 4),
    "fp8_b32": MLAShape("fp8_b32", 32, 128, 512, 64, 128, 64, BF16, FP8, DSV2_W_STD,
                        1.0 / math.sqrt(192), 4, lengths=(8192,) * 32),
    # the 128K context with the report's YaRN setting (section 3.1.4): s = 40, alpha = 1,
    # beta = 32 over the 4K pre-training context, logit factor (0.0707 ln s + 1)^2
    "yarn_b4": MLAShape("yarn_b4", 4, 128, 512, 64, 128, 64, BF16, BF16, DSV2_W_STD,
                        1.0 / math.sqrt(192), 5, lengths=(131072,) * 4, yarn_factor=40.0),
    # prefill: 4 prompts of 4096 tokens, each token a query over its prefix
    "prefill_b4": MLAShape("prefill_b4", 4, 128, 512, 64, 128, 64, BF16, BF16, DSV2_W_STD,
                           1.0 / math.sqrt(192), 6, lengths=(4096,) * 4),
    # one such prompt (the size a profiler capture of the prefill kernels uses)
    "prefill_b1": MLAShape("prefill_b1", 1, 128, 512, 64, 128, 64, BF16, BF16, DSV2_W_STD,
                           1.0 / math.sqrt(192), 7, lengths=(4096,)),
}

PREFILL_SHAPES = ("prefill_b4", "prefill_b1")


def shape_with(base: str, **kw) -> MLAShape:
    """A copy of a named workload with some fields replaced (smaller parity cases)."""
    return dataclasses.replace(SHAPES[base], **kw)


def torch_dtype(name: str) -> torch.dtype:
    return {BF16: torch.bfloat16, FP32: torch.float32}[name]


@dataclasses.dataclass
class MLAInputs:
    """Every array a decode step needs, on the CPU.

    Token t of sequence b (0 <= t < lengths[b]) is stored at flat index
    token_offsets[b] + t of c_kv_raw / k_rope_raw; its position is t.
    """

    shape: MLAShape
    lengths: np.ndarray        # int64 [B]   cache length attended by the decode
    token_offsets: np.ndarray  # int64 [B+1] prefix sums of lengths
    c_kv_raw: torch.Tensor     # [sum L, d_c]   io dtype, before the latent RMSNorm
    k_rope_raw: torch.Tensor   # [sum L, d_rope] io dtype, before RoPE
    q_nope: torch.Tensor       # [B, H, d_h]    io dtype
    q_rope: torch.Tensor       # [B, H, d_rope] io dtype, already rotated
    w_uk: torch.Tensor         # [H, d_h, d_c]  io dtype
    w_uv: torch.Tensor         # [H, d_h, d_c]  io dtype
    block_table: np.ndarray    # int32 [B, max_pages] page ids into the pool
    num_pages: int             # pages in the pool

    @property
    def max_pages(self) -> int:
        return int(self.block_table.shape[1])

    def positions(self) -> np.ndarray:
        """int32 position of every stored token (0-based within its sequence)."""
        return np.concatenate([np.arange(int(n), dtype=np.int32) for n in self.lengths])

    def seq_index(self) -> np.ndarray:
        """int32 sequence id of every stored token."""
        return np.repeat(np.arange(len(self.lengths), dtype=np.int32), self.lengths)

    def last_token_index(self) -> np.ndarray:
        """Flat index of each sequence's newest token (the one a step appends)."""
        return self.token_offsets[1:] - 1


def _normal(gen: torch.Generator, shape, std: float, dtype: torch.dtype) -> torch.Tensor:
    x = torch.randn(*shape, generator=gen, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(dtype)


def draw_lengths(shape: MLAShape) -> np.ndarray:
    if shape.lengths is not None:
        return np.asarray(shape.lengths, dtype=np.int64)
    rng = np.random.Generator(np.random.PCG64(shape.seed))
    old = rng.integers(1, shape.ragged_max, size=shape.batch, endpoint=True)
    return old.astype(np.int64) + 1   # one appended token per sequence


def make_block_table(lengths: np.ndarray, page_size: int, paged: bool, seed: int,
                     spare_pages: int = 0):
    """Page table: sequence b's page p lives at pool page block_table[b, p].

    paged=False gives the contiguous layout (sequence b owns pool pages
    b*max_pages .. b*max_pages+max_pages-1 in order). paged=True shuffles
    every page of every sequence across one shared pool (a random
    permutation, seeded) with `spare_pages` unused pages mixed in.
    Unused table entries are -1.
    """
    pages = [(int(n) + page_size - 1) // page_size for n in lengths]
    max_pages = max(1, max(pages))
    bt = np.full((len(lengths), max_pages), -1, dtype=np.int32)
    if not paged:
        for b, n in enumerate(pages):
            bt[b, :n] = b * max_pages + np.arange(n)
        return bt, len(lengths) * max_pages
    total = sum(pages) + spare_pages
    rng = np.random.Generator(np.random.PCG64(10_000 + seed))
    perm = rng.permutation(total).astype(np.int32)
    k = 0
    for b, n in enumerate(pages):
        bt[b, :n] = perm[k:k + n]
        k += n
    return bt, total


def make_inputs(shape: MLAShape, lengths: Optional[np.ndarray] = None,
                spare_pages: int = 3) -> MLAInputs:
    """Draw a full seeded workload for `shape` (lengths may be overridden)."""
    if lengths is None:
        lengths = draw_lengths(shape)
    lengths = np.asarray(lengths, dtype=np.int64)
    assert lengths.shape == (shape.batch,)
    gen = torch.Generator().manual_seed(shape.seed)
    dt = torch_dtype(shape.io_dtype)
    B, H = shape.batch, shape.n_heads
    total = int(lengths.sum())
    # Draw order is fixed: weights, queries, then the cached tokens.
    w_uk = _normal(gen, (H, shape.d_head, shape.d_c), shape.w_std, dt)
    w_uv = _normal(gen, (H, shape.d_head, shape.d_c), shape.w_std, dt)
    q_nope = _normal(gen, (B, H, shape.d_head), 1.0, dt)
    q_rope = _normal(gen, (B, H, shape.d_rope), 1.0, dt)
    c_kv_raw = _normal(gen, (total, shape.d_c), 1.0, dt)
    k_rope_raw = _normal(gen, (total, shape.d_rope), 1.0, dt)
    offs = np.zeros(B + 1, dtype=np.int64)
    offs[1:] = np.cumsum(lengths)
    bt, num_pages = make_block_table(lengths, shape.page_size, shape.paged, shape.seed,
                                     spare_pages if shape.paged else 0)
    return MLAInputs(shape, lengths, offs, c_kv_raw, k_rope_raw, q_nope, q_rope,
                     w_uk, w_uv, bt, num_pages)


@dataclasses.dataclass
class StepInputs:
    """Per-step inputs: fresh queries and the newest token of every sequence."""

    q_nope: torch.Tensor   # [B, H, d_h]
    q_rope: torch.Tensor   # [B, H, d_rope]
    c_new: torch.Tensor    # [B, d_c]     raw latent of the token at position lengths[b]-1
    k_new: torch.Tensor    # [B, d_rope]  raw rope key of that token


def draw_step(inp: MLAInputs, step: int) -> StepInputs:
    """Seeded inputs of decode step `step` (weights, older tokens and pages are kept)."""
    s = inp.shape
    gen = torch.Generator().manual_seed(1_000_003 * (step + 1) + s.seed)
    dt = torch_dtype(s.io_dtype)
    B, H = s.batch, s.n_heads
    return StepInputs(_normal(gen, (B, H, s.d_head), 1.0, dt),
                      _normal(gen, (B, H, s.d_rope), 1.0, dt),
                      _normal(gen, (B, s.d_c), 1.0, dt),
                      _normal(gen, (B, s.d_rope), 1.0, dt))


def draw_step_multi(inp: MLAInputs, step: int, q_len: int) -> StepInputs:
    """Seeded inputs of a step that decodes q_len new tokens per sequence (drafted tokens verified
    together): queries [B, q_len, H, .] and the q_len newest rows [B * q_len, .] of each sequence,
    sequence-major."""
    s = inp.shape
    gen = torch.Generator().manual_seed(2_000_003 * (step + 1) + 7919 * q_len + s.seed)
    dt = torch_dtype(s.io_dtype)
    B, H = s.batch, s.n_heads
    return StepInputs(_normal(gen, (B, q_len, H, s.d_head), 1.0, dt),
                      _normal(gen, (B, q_len, H, s.d_rope), 1.0, dt),
                      _normal(gen, (B * q_len, s.d_c), 1.0, dt),
                      _normal(gen, (B * q_len, s.d_rope), 1.0, dt))


def with_step(inp: MLAInputs, st: StepInputs) -> MLAInputs:
    """A copy of `inp` whose queries and newest tokens are those of `st`."""
    last = inp.last_token_index()
    c_kv_raw = inp.c_kv_raw.clone()
    k_rope_raw = inp.k_rope_raw.clone()
    c_kv_raw[last] = st.c_new
    k_rope_raw[last] = st.k_new
    return dataclasses.replace(inp, q_nope=st.q_nope, q_rope=st.q_rope,
                               c_kv_raw=c_kv_raw, k_rope_raw=k_rope_raw)


@dataclasses.dataclass
class PrefillInputs:
    """Queries of a prefill: the last n_new[b] cached rows of sequence b are its new tokens, and
    new token k of sequence b is query row q_start[b] + k."""

    q_nope: torch.Tensor   # [T, H, d_h]
    q_rope: torch.Tensor   # [T, H, d_rope], already rotated
    n_new: np.ndarray      # int64 [B]
    q_start: np.ndarray    # int64 [B+1] prefix sums of n_new


def draw_prefill(inp: MLAInputs, n_new: Optional[np.ndarray] = None, step: int = 0) -> PrefillInputs:
    """Seeded queries of a prefill over `inp`'s cache; n_new defaults to whole prompts
    (every cached row of every sequence is a new token)."""
    s = inp.shape
    n = np.asarray(inp.lengths if n_new is None else n_new, dtype=np.int64)
    assert n.shape == (s.batch,) and (n >= 0).all() and (n <= inp.lengths).all()
    qs = np.zeros(s.batch + 1, dtype=np.int64)
    qs[1:] = np.cumsum(n)
    T = int(qs[-1])
    gen = torch.Generator().manual_seed(3_000_017 * (step + 1) + s.seed)
    dt = torch_dtype(s.io_dtype)
    return PrefillInputs(_normal(gen, (T, s.n_heads, s.d_head), 1.0, dt),
                         _normal(gen, (T, s.n_heads, s.d_rope), 1.0, dt), n, qs)


def draw_w_o(shape: MLAShape, hidden: int = 5120, seed: int = 0) -> torch.Tensor:
    """Output projection W_O [hidden, n_heads * d_head] in io dtype, N(0, 0.006^2) (the report's
    initialisation std, section 3.1.2)."""
    gen = torch.Generator().manual_seed(4_000_037 + 101 * seed + shape.seed)
    return _normal(gen, (hidden, shape.n_heads * shape.d_head), 0.006, torch_dtype(shape.io_dtype))
