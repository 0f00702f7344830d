"""B300-native MLA decode over a paged latent KV cache.

Thin Python binding of the C-ABI library libmla.so (declared in
include/mla.h). Every call marshals torch tensors (device memory and
streams only) into pointers and sizes; all arithmetic runs in the library's
CUDA kernels. The binding refuses to work without the compiled library.

    cfg = MLAConfig.dsv2()                       # 128 heads, 512 + 64 latent row
    pool = new_pool(cfg, num_pages, device)      # [num_pages, page, row_bytes] u8
    append(cfg, c_kv_raw, k_rope_raw, positions, pool, block_table, seq_idx)
    out = decode(cfg, q_nope, q_rope, w_uk, w_uv, pool, block_table, seq_lens, max_seq_len)
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
from typing import Optional

import torch

__all__ = ["MLAConfig", "MLAError", "BF16", "FP32", "FP8_E4M3_B128", "library_path", "cache_row_bytes",
           "new_pool", "append", "workspace_size", "workspace_size_multi", "decode", "check_device_errors", "decode_path",
           "decode_stage_names", "set_stage_events", "decode_static_scratch", "prefill", "prefill_workspace_size", "fold_output_weight",
           "decode_hidden", "decode_hidden_workspace_size"]

BF16, FP32, FP8_E4M3_B128 = 0, 1, 2
_DTYPE_NAMES = {"bf16": BF16, "fp32": FP32, "fp8_e4m3_b128": FP8_E4M3_B128}
_TORCH_IO = {BF16: torch.bfloat16, FP32: torch.float32}

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libmla.so")


def library_path() -> str:
    return _LIB_PATH


class MLAError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"MLA status {status}: {msg}")
        self.status = status


class _CConfig(ctypes.Structure):
    _fields_ = [("n_heads", ctypes.c_int32), ("d_c", ctypes.c_int32), ("d_rope", ctypes.c_int32),
                ("d_head", ctypes.c_int32), ("page_size", ctypes.c_int32), ("io_dtype", ctypes.c_int32),
                ("cache_dtype", ctypes.c_int32), ("scale", ctypes.c_float), ("eps", ctypes.c_float),
                ("rope_theta", ctypes.c_float), ("rope_interleaved", ctypes.c_int32),
                ("yarn_factor", ctypes.c_float), ("yarn_alpha", ctypes.c_float), ("yarn_beta", ctypes.c_float),
                ("yarn_mscale", ctypes.c_float), ("yarn_orig_len", ctypes.c_int32)]


@dataclasses.dataclass(frozen=True)
class MLAConfig:
    """Mirror of the C struct mla_config."""

    n_heads: int
    d_c: int
    d_rope: int
    d_head: int
    page_size: int = 64
    io_dtype: int = BF16
    cache_dtype: int = BF16
    scale: float = 0.0          # <= 0: the library uses 1/sqrt(d_head + d_rope)
    eps: float = 1e-6
    rope_theta: float = 10000.0
    rope_interleaved: bool = True
    yarn_factor: float = 1.0    # YaRN scale s; <= 1: plain RoPE (DeepSeek-V2 long context: 40)
    yarn_alpha: float = 1.0
    yarn_beta: float = 32.0
    yarn_mscale: float = 0.0707
    yarn_orig_len: int = 4096

    @staticmethod
    def dsv2(cache_dtype: int = BF16, page_size: int = 64) -> "MLAConfig":
        """DeepSeek-V2 MLA: 128 heads of 128, latent 512, decoupled rope 64."""
        return MLAConfig(128, 512, 64, 128, page_size, BF16, cache_dtype)

    @staticmethod
    def from_shape(shape) -> "MLAConfig":
        """From an object with the fields of a workload description (mla_synth.MLAShape)."""
        return MLAConfig(shape.n_heads, shape.d_c, shape.d_rope, shape.d_head, shape.page_size,
                         _DTYPE_NAMES[shape.io_dtype], _DTYPE_NAMES[shape.cache_dtype], float(shape.scale),
                         float(shape.eps), float(shape.rope_theta), True, float(shape.yarn_factor),
                         float(shape.yarn_alpha), float(shape.yarn_beta), float(shape.yarn_mscale),
                         int(shape.yarn_orig_len))

    def c(self) -> _CConfig:
        return _CConfig(self.n_heads, self.d_c, self.d_rope, self.d_head, self.page_size, self.io_dtype,
                        self.cache_dtype, self.scale, self.eps, self.rope_theta, int(self.rope_interleaved),
                        self.yarn_factor, self.yarn_alpha, self.yarn_beta, self.yarn_mscale, self.yarn_orig_len)

    @property
    def io_torch_dtype(self) -> torch.dtype:
        return _TORCH_IO[self.io_dtype]


_lib = None


def _load():
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise RuntimeError(f"{_LIB_PATH} is missing; build it with `python -m head_latent_attention_22_b300.build`")
    lib = ctypes.CDLL(_LIB_PATH)
    P, I32, I64, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    CFG = ctypes.POINTER(_CConfig)
    sig = {
        "mla_cache_row_bytes": (SZ, [CFG]),
        "mla_append": (I32, [CFG, P, P, P, P, P, P, I64, P, I32, I32, I32, P]),
        "mla_decode_workspace_size": (SZ, [CFG, I32, I32]),
        "mla_decode": (I32, [CFG, P, P, P, P, P, I64, P, P, I32, I32, I32, P, P, SZ, P]),
        "mla_check_device_errors": (I32, [P]),
        "mla_decode_path": (I32, [CFG]),
        "mla_last_error": (ctypes.c_char_p, []),
        "mla_decode_stage_names": (ctypes.c_char_p, [CFG]),
        "mla_decode_static_scratch": (I32, [CFG, P, P, P, P, P, I64, P, P, I32, I32, I32, P, P]),
        "mla_set_stage_events": (I32, [ctypes.POINTER(ctypes.c_void_p), I32]),
        "mla_rope_query": (I32, [CFG, P, P, P, I32, P]),
        "mla_decode_multi_workspace_size": (SZ, [CFG, I32, I32, I32, I32]),
        "mla_decode_multi": (I32, [CFG, P, P, P, P, P, I64, P, P, I32, I32, I32, I32, P, P, SZ, P]),
        "mla_prefill_workspace_size": (SZ, [CFG, I32, I32]),
        "mla_fold_output_weight": (I32, [CFG, P, P, I32, P, P]),
        "mla_decode_hidden_workspace_size": (SZ, [CFG, I32, I32, I32]),
        "mla_decode_hidden": (I32, [CFG, P, P, P, P, P, I64, P, P, I32, I32, I32, I32, P, P, SZ, P]),
        "mla_prefill": (I32, [CFG, P, P, P, P, P, I64, P, P, P, I32, I32, I32, I32, P, P, SZ, P]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype, fn.argtypes = res, args
    _lib = lib
    return lib


def _check(status: int):
    if status != 0:
        raise MLAError(status, _load().mla_last_error().decode())


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _need(t: torch.Tensor, name: str, dtype: Optional[torch.dtype] = None, dims: Optional[int] = None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if dims is not None and t.dim() != dims:
        raise ValueError(f"{name} must have {dims} dims, got {tuple(t.shape)}")


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def cache_row_bytes(cfg: MLAConfig) -> int:
    n = _load().mla_cache_row_bytes(ctypes.byref(cfg.c()))
    if n == 0:
        raise MLAError(1, _load().mla_last_error().decode())
    return int(n)


def new_pool(cfg: MLAConfig, num_pages: int, device, fill: Optional[int] = None) -> torch.Tensor:
    """Allocate a page pool [num_pages, page_size, row_bytes] of bytes (optionally filled)."""
    shape = (num_pages, cfg.page_size, cache_row_bytes(cfg))
    if fill is None:
        return torch.empty(shape, dtype=torch.uint8, device=device)
    return torch.full(shape, fill, dtype=torch.uint8, device=device)


def append(cfg: MLAConfig, c_kv_raw: torch.Tensor, k_rope_raw: torch.Tensor, positions: torch.Tensor,
           pool: torch.Tensor, block_table: Optional[torch.Tensor], seq_idx: Optional[torch.Tensor] = None,
           gamma: Optional[torch.Tensor] = None, batch: Optional[int] = None, max_pages: Optional[int] = None,
           stream=None) -> None:
    """mla_append: RMSNorm + RoPE + paged row write of len(positions) tokens."""
    T = positions.shape[0]
    _need(c_kv_raw, "c_kv_raw", cfg.io_torch_dtype, 2)
    _need(k_rope_raw, "k_rope_raw", cfg.io_torch_dtype, 2)
    _need(positions, "positions", torch.int32, 1)
    _need(pool, "pool", torch.uint8)
    if c_kv_raw.shape != (T, cfg.d_c) or k_rope_raw.shape != (T, cfg.d_rope):
        raise ValueError("c_kv_raw / k_rope_raw shapes do not match positions and cfg")
    if seq_idx is not None:
        _need(seq_idx, "seq_idx", torch.int32, 1)
    if gamma is not None:
        _need(gamma, "gamma", torch.float32, 1)
    if block_table is not None:
        _need(block_table, "block_table", torch.int32, 2)
        batch = block_table.shape[0] if batch is None else batch
        max_pages = block_table.shape[1] if max_pages is None else max_pages
    if batch is None or max_pages is None:
        raise ValueError("batch and max_pages are needed without a block table")
    _check(_load().mla_append(ctypes.byref(cfg.c()), _ptr(c_kv_raw), _ptr(k_rope_raw), _ptr(positions),
                              _ptr(seq_idx), _ptr(gamma), _ptr(pool), pool.shape[0], _ptr(block_table),
                              batch, max_pages, T, _stream(stream)))


def rope_query(cfg: MLAConfig, q_rope_raw: torch.Tensor, positions: torch.Tensor,
               out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """mla_rope_query: the query's rope part rotated with the keys' frequencies (YaRN included)."""
    _need(q_rope_raw, "q_rope_raw", cfg.io_torch_dtype, 3)
    _need(positions, "positions", torch.int32, 1)
    B = q_rope_raw.shape[0]
    if q_rope_raw.shape != (B, cfg.n_heads, cfg.d_rope) or positions.shape[0] != B:
        raise ValueError("q_rope_raw must be [batch, n_heads, d_rope] with one position per sequence")
    if out is None:
        out = torch.empty_like(q_rope_raw)
    _need(out, "out", cfg.io_torch_dtype, 3)
    _check(_load().mla_rope_query(ctypes.byref(cfg.c()), _ptr(q_rope_raw), _ptr(positions), _ptr(out), B,
                                  _stream(stream)))
    return out


def workspace_size_multi(cfg: MLAConfig, batch: int, q_len: int, max_pages: int, max_seq_len: int) -> int:
    """mla_decode_multi_workspace_size (0 for invalid arguments)."""
    return int(_load().mla_decode_multi_workspace_size(ctypes.byref(cfg.c()), batch, q_len, max_pages, max_seq_len))


def workspace_size(cfg: MLAConfig, batch: int, max_seq_len: int) -> int:
    return int(_load().mla_decode_workspace_size(ctypes.byref(cfg.c()), batch, max_seq_len))


def decode_path(cfg: MLAConfig) -> int:
    """1 if mla_decode runs the tcgen05 tensor-core kernels for cfg, 0 for the CUDA-core ones."""
    return int(_load().mla_decode_path(ctypes.byref(cfg.c())))


def decode(cfg: MLAConfig, q_nope: torch.Tensor, q_rope: torch.Tensor, w_uk: torch.Tensor, w_uv: torch.Tensor,
           pool: torch.Tensor, block_table: Optional[torch.Tensor], seq_lens: torch.Tensor, max_seq_len: int,
           out: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
           max_pages: Optional[int] = None, stream=None) -> torch.Tensor:
    """mla_decode: per-head MLA decode outputs [B, H, d_head] (fp32)."""
    B = q_nope.shape[0]
    dt = cfg.io_torch_dtype
    _need(q_nope, "q_nope", dt, 3)
    _need(q_rope, "q_rope", dt, 3)
    _need(w_uk, "w_uk", dt, 3)
    _need(w_uv, "w_uv", dt, 3)
    _need(pool, "pool", torch.uint8)
    _need(seq_lens, "seq_lens", torch.int32, 1)
    H = cfg.n_heads
    if q_nope.shape != (B, H, cfg.d_head) or q_rope.shape != (B, H, cfg.d_rope):
        raise ValueError("query shapes do not match cfg")
    if w_uk.shape != (H, cfg.d_head, cfg.d_c) or w_uv.shape != (H, cfg.d_head, cfg.d_c):
        raise ValueError("weight shapes do not match cfg")
    if seq_lens.shape[0] != B:
        raise ValueError("seq_lens must have one entry per sequence")
    if block_table is not None:
        _need(block_table, "block_table", torch.int32, 2)
        max_pages = block_table.shape[1]
    if max_pages is None:
        raise ValueError("max_pages is needed without a block table")
    if out is None:
        out = torch.empty((B, H, cfg.d_head), dtype=torch.float32, device=q_nope.device)
    _need(out, "out", torch.float32, 3)
    need = workspace_size(cfg, B, max_seq_len)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q_nope.device)
    _need(workspace, "workspace", torch.uint8)
    _check(_load().mla_decode(ctypes.byref(cfg.c()), _ptr(q_nope), _ptr(q_rope), _ptr(w_uk), _ptr(w_uv),
                              _ptr(pool), pool.shape[0], _ptr(block_table), _ptr(seq_lens), B, max_pages,
                              max_seq_len, _ptr(out), _ptr(workspace), workspace.numel(), _stream(stream)))
    return out


def decode_multi(cfg: MLAConfig, q_nope: torch.Tensor, q_rope: torch.Tensor, w_uk: torch.Tensor,
                 w_uv: torch.Tensor, pool: torch.Tensor, block_table: Optional[torch.Tensor], seq_lens: torch.Tensor,
                 max_seq_len: int, out: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                 max_pages: Optional[int] = None, stream=None) -> torch.Tensor:
    """mla_decode_multi: q_len new tokens per sequence, causal among them -> [B, q_len, H, d_head] fp32.

    q_nope [B, q_len, H, d_head], q_rope [B, q_len, H, d_rope]; seq_lens counts every cached row
    of a sequence, its q_len new tokens included."""
    dt = cfg.io_torch_dtype
    _need(q_nope, "q_nope", dt, 4)
    _need(q_rope, "q_rope", dt, 4)
    _need(w_uk, "w_uk", dt, 3)
    _need(w_uv, "w_uv", dt, 3)
    _need(pool, "pool", torch.uint8)
    _need(seq_lens, "seq_lens", torch.int32, 1)
    B, q = q_nope.shape[:2]
    H = cfg.n_heads
    if q_nope.shape != (B, q, H, cfg.d_head) or q_rope.shape != (B, q, H, cfg.d_rope):
        raise ValueError("query shapes do not match cfg")
    if seq_lens.shape[0] != B:
        raise ValueError("seq_lens must have one entry per sequence")
    if block_table is not None:
        _need(block_table, "block_table", torch.int32, 2)
        max_pages = block_table.shape[1]
    if max_pages is None:
        raise ValueError("max_pages is needed without a block table")
    if out is None:
        out = torch.empty((B, q, H, cfg.d_head), dtype=torch.float32, device=q_nope.device)
    _need(out, "out", torch.float32, 4)
    need = int(_load().mla_decode_multi_workspace_size(ctypes.byref(cfg.c()), B, q, max_pages, max_seq_len))
    if need == 0:
        raise MLAError(1, _load().mla_last_error().decode())
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q_nope.device)
    _need(workspace, "workspace", torch.uint8)
    _check(_load().mla_decode_multi(ctypes.byref(cfg.c()), _ptr(q_nope), _ptr(q_rope), _ptr(w_uk), _ptr(w_uv),
                                    _ptr(pool), pool.shape[0], _ptr(block_table), _ptr(seq_lens), B, q, max_pages,
                                    max_seq_len, _ptr(out), _ptr(workspace), workspace.numel(), _stream(stream)))
    return out


def prefill_workspace_size(cfg: MLAConfig, batch: int, max_seq_len: int) -> int:
    """mla_prefill_workspace_size (0 when cfg has no prefill kernels)."""
    return int(_load().mla_prefill_workspace_size(ctypes.byref(cfg.c()), batch, max_seq_len))


def prefill(cfg: MLAConfig, q_nope: torch.Tensor, q_rope: torch.Tensor, w_uk: torch.Tensor, w_uv: torch.Tensor,
            pool: torch.Tensor, block_table: Optional[torch.Tensor], seq_lens: torch.Tensor, q_start: torch.Tensor,
            max_seq_len: int, out: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
            max_pages: Optional[int] = None, stream=None) -> torch.Tensor:
    """mla_prefill: every new token of each sequence attends causally to its prefix -> [T, H, d_head] fp32.

    q_nope [T, H, d_head], q_rope [T, H, d_rope] (rotated); q_start [B + 1] int32: the new tokens of
    sequence b are query rows q_start[b] .. q_start[b+1]-1 and the last rows of its seq_lens[b]
    cached rows."""
    dt = cfg.io_torch_dtype
    _need(q_nope, "q_nope", dt, 3)
    _need(q_rope, "q_rope", dt, 3)
    _need(w_uk, "w_uk", dt, 3)
    _need(w_uv, "w_uv", dt, 3)
    _need(pool, "pool", torch.uint8)
    _need(seq_lens, "seq_lens", torch.int32, 1)
    _need(q_start, "q_start", torch.int32, 1)
    T, H = q_nope.shape[0], cfg.n_heads
    B = seq_lens.shape[0]
    if q_nope.shape != (T, H, cfg.d_head) or q_rope.shape != (T, H, cfg.d_rope):
        raise ValueError("query shapes do not match cfg")
    if q_start.shape[0] != B + 1:
        raise ValueError("q_start must have batch + 1 entries")
    if block_table is not None:
        _need(block_table, "block_table", torch.int32, 2)
        max_pages = block_table.shape[1]
    if max_pages is None:
        raise ValueError("max_pages is needed without a block table")
    if out is None:
        out = torch.empty((T, H, cfg.d_head), dtype=torch.float32, device=q_nope.device)
    _need(out, "out", torch.float32, 3)
    need = prefill_workspace_size(cfg, B, max_seq_len)
    if need == 0:
        raise MLAError(2, "no prefill kernels for this config (or invalid sizes)")
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q_nope.device)
    _need(workspace, "workspace", torch.uint8)
    _check(_load().mla_prefill(ctypes.byref(cfg.c()), _ptr(q_nope), _ptr(q_rope), _ptr(w_uk), _ptr(w_uv),
                               _ptr(pool), pool.shape[0], _ptr(block_table), _ptr(seq_lens), _ptr(q_start), B,
                               max_pages, max_seq_len, T, _ptr(out), _ptr(workspace), workspace.numel(),
                               _stream(stream)))
    return out


def fold_output_weight(cfg: MLAConfig, w_uv: torch.Tensor, w_o: torch.Tensor,
                       out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """mla_fold_output_weight: W_OUV [hidden, H * d_c] fp16 with W_OUV[:, i d_c:(i+1) d_c] = W_O[:, i d_h:(i+1) d_h] W_UV[i].

    w_o [hidden, H * d_head] (the output projection), w_uv [H, d_head, d_c]."""
    dt = cfg.io_torch_dtype
    _need(w_uv, "w_uv", dt, 3)
    _need(w_o, "w_o", dt, 2)
    hidden = w_o.shape[0]
    if w_o.shape[1] != cfg.n_heads * cfg.d_head:
        raise ValueError("w_o must be [hidden, n_heads * d_head]")
    if out is None:
        out = torch.empty((hidden, cfg.n_heads * cfg.d_c), dtype=torch.float16, device=w_o.device)
    _need(out, "out", torch.float16, 2)
    _check(_load().mla_fold_output_weight(ctypes.byref(cfg.c()), _ptr(w_uv), _ptr(w_o), hidden, _ptr(out),
                                          _stream(stream)))
    return out


def decode_hidden_workspace_size(cfg: MLAConfig, batch: int, max_seq_len: int, hidden: int) -> int:
    return int(_load().mla_decode_hidden_workspace_size(ctypes.byref(cfg.c()), batch, max_seq_len, hidden))


def decode_hidden(cfg: MLAConfig, q_nope: torch.Tensor, q_rope: torch.Tensor, w_uk: torch.Tensor,
                  w_ouv: torch.Tensor, pool: torch.Tensor, block_table: Optional[torch.Tensor], seq_lens: torch.Tensor,
                  max_seq_len: int, out: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                  max_pages: Optional[int] = None, stream=None) -> torch.Tensor:
    """mla_decode_hidden: the decode with W_UV folded into W_O -> [B, hidden] fp32 (w_ouv from
    fold_output_weight)."""
    dt = cfg.io_torch_dtype
    _need(q_nope, "q_nope", dt, 3)
    _need(q_rope, "q_rope", dt, 3)
    _need(w_uk, "w_uk", dt, 3)
    _need(w_ouv, "w_ouv", torch.float16, 2)
    _need(pool, "pool", torch.uint8)
    _need(seq_lens, "seq_lens", torch.int32, 1)
    B = q_nope.shape[0]
    hidden = w_ouv.shape[0]
    if block_table is not None:
        _need(block_table, "block_table", torch.int32, 2)
        max_pages = block_table.shape[1]
    if max_pages is None:
        raise ValueError("max_pages is needed without a block table")
    if out is None:
        out = torch.empty((B, hidden), dtype=torch.float32, device=q_nope.device)
    _need(out, "out", torch.float32, 2)
    need = decode_hidden_workspace_size(cfg, B, max_seq_len, hidden)
    if need == 0:
        raise MLAError(2, "no folded output path for this config or size")
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q_nope.device)
    _need(workspace, "workspace", torch.uint8)
    _check(_load().mla_decode_hidden(ctypes.byref(cfg.c()), _ptr(q_nope), _ptr(q_rope), _ptr(w_uk), _ptr(w_ouv),
                                     _ptr(pool), pool.shape[0], _ptr(block_table), _ptr(seq_lens), B, max_pages,
                                     max_seq_len, hidden, _ptr(out), _ptr(workspace), workspace.numel(),
                                     _stream(stream)))
    return out


def decode_stage_names(cfg: MLAConfig) -> list:
    """Kernel names of one decode call, in launch order."""
    return _load().mla_decode_stage_names(ctypes.byref(cfg.c())).decode().split(",")


def set_stage_events(events) -> None:
    """Record torch.cuda.Event objects around each decode kernel (None/[] turns it off)."""
    events = list(events or [])
    for e in events:
        if not e.cuda_event:     # torch creates the CUDA event lazily, on first record
            e.record()
    arr = (ctypes.c_void_p * max(1, len(events)))(*[ctypes.c_void_p(e.cuda_event) for e in events])
    _check(_load().mla_set_stage_events(arr, len(events)))


def decode_static_scratch(cfg: MLAConfig, q_nope: torch.Tensor, q_rope: torch.Tensor, w_uk: torch.Tensor,
                          w_uv: torch.Tensor, pool: torch.Tensor, block_table: Optional[torch.Tensor],
                          seq_lens: torch.Tensor, max_seq_len: int, out: torch.Tensor,
                          max_pages: Optional[int] = None, stream=None) -> torch.Tensor:
    """mla_decode_static_scratch: the decode for callers that cannot allocate device memory.

    Nothing is allocated, neither here nor in the library: the caller passes
    `out`, and the library's fixed per-device scratch array replaces the
    workspace. Calls on one device share that array and must not overlap.
    """
    dt = cfg.io_torch_dtype
    for t, n, d in ((q_nope, "q_nope", dt), (q_rope, "q_rope", dt), (w_uk, "w_uk", dt), (w_uv, "w_uv", dt),
                    (pool, "pool", torch.uint8), (seq_lens, "seq_lens", torch.int32), (out, "out", torch.float32)):
        _need(t, n, d)
    if block_table is not None:
        _need(block_table, "block_table", torch.int32, 2)
        max_pages = block_table.shape[1]
    if max_pages is None:
        raise ValueError("max_pages is needed without a block table")
    if out.shape != (q_nope.shape[0], cfg.n_heads, cfg.d_head):
        raise ValueError("out must be [batch, n_heads, d_head]")
    _check(_load().mla_decode_static_scratch(ctypes.byref(cfg.c()), _ptr(q_nope), _ptr(q_rope), _ptr(w_uk),
                                             _ptr(w_uv), _ptr(pool), pool.shape[0], _ptr(block_table),
                                             _ptr(seq_lens), q_nope.shape[0], max_pages, max_seq_len, _ptr(out),
                                             _stream(stream)))
    return out


def check_device_errors(stream=None) -> None:
    """Wait for the stream and raise MLAError if a kernel flagged a bounds or timeout error."""
    _check(_load().mla_check_device_errors(_stream(stream)))


class StepGraph:
    """One serving step - mla_append of the new tokens, then mla_decode - captured once
    into a CUDA graph and replayed.

    The arguments are those of append() and decode(); every tensor must stay
    allocated and in place while the graph lives, because the captured launches
    hold their addresses (and the tensor maps built from them). replay() runs
    the same kernels on whatever the tensors hold at that moment, on the current
    stream: the caller writes the step's inputs into them, replays, and reads
    `out`. Sizes (batch, max_seq_len, number of new tokens) are fixed at capture.
    The constructor runs the step once eagerly before capturing it (writing the
    new tokens' cache rows, which replaying rewrites with the same values).
    """

    def __init__(self, cfg: MLAConfig, *, c_new: torch.Tensor, k_new: torch.Tensor, positions: torch.Tensor,
                 seq_idx: Optional[torch.Tensor], q_nope: torch.Tensor, q_rope: torch.Tensor, w_uk: torch.Tensor,
                 w_uv: torch.Tensor, pool: torch.Tensor, block_table: Optional[torch.Tensor], seq_lens: torch.Tensor,
                 max_seq_len: int, out: torch.Tensor, workspace: torch.Tensor, max_pages: Optional[int] = None):
        batch = q_nope.shape[0]

        def step():
            append(cfg, c_new, k_new, positions, pool, block_table, seq_idx=seq_idx, batch=batch,
                   max_pages=max_pages)
            decode(cfg, q_nope, q_rope, w_uk, w_uv, pool, block_table, seq_lens, max_seq_len, out=out,
                   workspace=workspace, max_pages=max_pages)

        # one eager step first: the per-device setup of the library (kernel attributes, occupancy)
        # happens on a first call and must not fall inside the capture
        step()
        check_device_errors()
        self.out = out
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            step()

    def replay(self) -> torch.Tensor:
        self.graph.replay()
        return self.out
