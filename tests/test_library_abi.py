"""The C-ABI library without a GPU: it loads, exports what include/mla.h
declares, lays out the config struct as C does, and rejects bad arguments on
the host before touching CUDA."""
import ctypes
import os
import re
import subprocess
import tempfile

import pytest

import head_latent_attention_22_b300 as M
from head_latent_attention_22_b300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in os.listdir(os.path.join(ROOT, "include")) if f.endswith(".h")]


@pytest.fixture(scope="module")
def lib():
    B.build()
    return ctypes.CDLL(M.library_path())


def declared_functions():
    names = set()
    for h in HEADERS:
        text = open(h).read()
        names |= set(re.findall(r"MLA_API\s+[\w\s\*]+?\b(mla_\w+)\s*\(", text))
    return sorted(names)


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert {"mla_append", "mla_decode", "mla_decode_workspace_size", "mla_check_device_errors",
            "mla_cache_row_bytes", "mla_last_error", "mla_decode_path"} <= set(names)
    out = subprocess.run(["nm", "-D", "--defined-only", M.library_path()], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT\s+(mla_\w+)", out))
    missing = [n for n in names if n not in exported]
    assert not missing, missing
    for n in names:
        getattr(lib, n)


def test_config_struct_layout_matches_c():
    src = r'''
#include <stdio.h>
#include <stddef.h>
#include "mla.h"
int main(void) {
  printf("%zu %zu %zu %zu %zu %zu\n", sizeof(mla_config), offsetof(mla_config, scale),
         offsetof(mla_config, rope_theta), offsetof(mla_config, rope_interleaved),
         offsetof(mla_config, yarn_factor), offsetof(mla_config, yarn_orig_len));
  return 0;
}
'''
    with tempfile.TemporaryDirectory() as d:
        c = os.path.join(d, "t.c")
        open(c, "w").write(src)
        exe = os.path.join(d, "t")
        subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), c, "-o", exe], check=True)
        got = [int(x) for x in subprocess.run([exe], capture_output=True, text=True).stdout.split()]
    cc = M._CConfig
    assert got == [ctypes.sizeof(cc), cc.scale.offset, cc.rope_theta.offset, cc.rope_interleaved.offset,
                   cc.yarn_factor.offset, cc.yarn_orig_len.offset]


def test_row_bytes():
    assert M.cache_row_bytes(M.MLAConfig.dsv2()) == 1152
    assert M.cache_row_bytes(M.MLAConfig.dsv2(M.FP8_E4M3_B128)) == 512 + 16 + 128
    assert M.cache_row_bytes(M.MLAConfig(4, 32, 8, 16, 64, M.FP32, M.FP32)) == 160


def test_host_rejects_bad_config_and_arguments(lib):
    M._load()
    cfg = M.MLAConfig.dsv2().c()
    bad = M.MLAConfig(4, 32, 7, 16).c()        # odd rope width
    assert M._load().mla_cache_row_bytes(ctypes.byref(bad)) == 0
    assert M._load().mla_decode_workspace_size(ctypes.byref(bad), 4, 100) == 0
    fp8_bad = M.MLAConfig(4, 96, 8, 16, 64, M.BF16, M.FP8_E4M3_B128).c()   # d_c not a multiple of 128
    assert M._load().mla_cache_row_bytes(ctypes.byref(fp8_bad)) == 0
    # NULL pointers and misaligned pointers are refused before any CUDA call
    st = M._load().mla_append(ctypes.byref(cfg), None, None, None, None, None, None, 10, None, 4, 4, 4, None)
    assert st == 1 and b"non-NULL" in M._load().mla_last_error()
    st = M._load().mla_append(ctypes.byref(cfg), ctypes.c_void_p(8), ctypes.c_void_p(16), ctypes.c_void_p(16),
                              None, None, ctypes.c_void_p(16), 10, None, 4, 4, 4, None)
    assert st == 1 and b"aligned" in M._load().mla_last_error()
    st = M._load().mla_decode(ctypes.byref(cfg), None, None, None, None, None, 10, None, None, 4, 4, 100,
                              None, None, 0, None)
    assert st == 1
    # a length bound beyond the page table's reach
    st = M._load().mla_decode(ctypes.byref(cfg), *([ctypes.c_void_p(256)] * 5), 10, None, ctypes.c_void_p(256),
                              4, 2, 129, ctypes.c_void_p(256), ctypes.c_void_p(256), 1 << 30, None)
    assert st == 1 and b"max_seq_len" in M._load().mla_last_error()
    # YaRN on with an empty ramp (beta <= alpha) or no original context is refused
    import dataclasses
    for kw in (dict(yarn_beta=1.0), dict(yarn_orig_len=0)):
        y = dataclasses.replace(M.MLAConfig.dsv2(), yarn_factor=40.0, **kw).c()
        assert M._load().mla_cache_row_bytes(ctypes.byref(y)) == 0
        assert b"YaRN" in M._load().mla_last_error()
    # ... while yarn_factor <= 1 ignores the other YaRN fields
    off = dataclasses.replace(M.MLAConfig.dsv2(), yarn_factor=1.0, yarn_beta=0.0, yarn_orig_len=0).c()
    assert M._load().mla_cache_row_bytes(ctypes.byref(off)) == 1152
    st = M._load().mla_rope_query(ctypes.byref(cfg), None, None, None, 2, None)
    assert st == 1


def test_workspace_size_grows_with_batch_and_length():
    cfg = M.MLAConfig.dsv2()
    a = M.workspace_size(cfg, 4, 4096)
    assert a > 0 and M.workspace_size(cfg, 8, 4096) > a and M.workspace_size(cfg, 4, 131072) >= a


def test_host_rejects_bad_multi_token_and_rope_query_arguments(lib):
    L = M._load()
    cfg = M.MLAConfig.dsv2().c()
    P = ctypes.c_void_p
    # workspace size: invalid sizes give 0, valid ones grow with q_len
    assert L.mla_decode_multi_workspace_size(ctypes.byref(cfg), 4, 0, 64, 4096) == 0
    assert L.mla_decode_multi_workspace_size(ctypes.byref(cfg), 0, 2, 64, 4096) == 0
    w1 = L.mla_decode_multi_workspace_size(ctypes.byref(cfg), 4, 1, 64, 4096)
    w3 = L.mla_decode_multi_workspace_size(ctypes.byref(cfg), 4, 3, 64, 4096)
    assert 0 < w1 < w3
    # q_len 0, a missing workspace and a too-small workspace are refused before any launch
    st = L.mla_decode_multi(ctypes.byref(cfg), *([P(256)] * 5), 10, None, P(256), 4, 0, 64, 4096, P(256), P(256),
                            1 << 30, None)
    assert st == 1
    st = L.mla_decode_multi(ctypes.byref(cfg), *([P(256)] * 5), 10, None, P(256), 4, 2, 64, 4096, P(256), None,
                            1 << 30, None)
    assert st == 1 and b"non-NULL" in L.mla_last_error()
    st = L.mla_decode_multi(ctypes.byref(cfg), *([P(256)] * 5), 10, None, P(256), 4, 2, 64, 4096, P(256), P(256),
                            16, None)
    assert st == 1 and b"too small" in L.mla_last_error()
    # rope_query: negative batch and NULL pointers are refused; an empty batch is a no-op
    assert L.mla_rope_query(ctypes.byref(cfg), P(256), P(256), P(256), -1, None) == 1
    assert L.mla_rope_query(ctypes.byref(cfg), None, P(256), P(256), 2, None) == 1
    assert L.mla_rope_query(ctypes.byref(cfg), None, None, None, 0, None) == 0


def test_default_scale_is_left_to_the_library(lib):
    # scale <= 0 asks the library for 1/sqrt(d_head + d_rope); the binding passes it through untouched
    cfg = M.MLAConfig.dsv2()
    assert cfg.scale == 0.0 and cfg.c().scale == 0.0
    assert M.decode_path(cfg) == 1   # the tensor-core path accepts the default


def test_static_scratch_batch_limit_matches_the_header(lib):
    L = M._load()
    P = ctypes.c_void_p
    text = open(os.path.join(ROOT, "include", "mla.h")).read()
    limit = int(re.search(r"MLA_STATIC_SCRATCH_BYTES \(\(size_t\)(\d+) << 20\)", text).group(1)) << 20
    n_doc = int(re.search(r"batch of at most (\d+) sequences", text).group(1))
    cfg = M.MLAConfig.dsv2()
    assert M.workspace_size(cfg, n_doc, 131072) <= limit < M.workspace_size(cfg, n_doc + 1, 131072)
    c = cfg.c()
    # one past the limit: refused for its size, before anything is looked up or launched
    st = L.mla_decode_static_scratch(ctypes.byref(c), *([P(256)] * 5), 10, None, P(256), n_doc + 1, 2, 4096,
                                     P(256), None)
    assert st == 1 and b"bytes of scratch" in L.mla_last_error()
    # at the limit the size passes; the call then stops on the (deliberately) short page table
    st = L.mla_decode_static_scratch(ctypes.byref(c), *([P(256)] * 5), 10, None, P(256), n_doc, 2, 4096,
                                     P(256), None)
    assert st != 0 and b"bytes of scratch" not in L.mla_last_error()
