"""CPU checks of the C-ABI library: it loads, exports every declared symbol,
and its host-side validation rejects bad arguments before touching a GPU."""
import ctypes
import os
import re

import pytest

from fp4_kv_cache_06_b300 import csa2

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            names |= set(re.findall(r"CSA2_API[^;(]*?\b(csa2_[a-z0-9_]+)\s*\(", text))
    return names


def test_library_exports_every_declared_symbol():
    lib = csa2.lib()
    decl = declared_symbols()
    assert len(decl) >= 15
    for name in sorted(decl):
        assert hasattr(lib, name), name
    assert set(csa2.EXPORTS) <= decl


def test_status_strings_and_version():
    lib = csa2.lib()
    assert lib.csa2_status_string(0) == b"CSA2_OK"
    assert lib.csa2_status_string(6) == b"CSA2_ERR_DEVICE_BOUNDS"
    assert lib.csa2_status_string(99) == b"CSA2_ERR_UNKNOWN"
    assert csa2.version() >= 100


def test_workspace_sizes():
    ws = csa2.workspace_size
    assert ws(csa2.OP_TOPK, 0) >= 0
    assert ws(csa2.OP_INDEX_FULL, 32, 131072) >= 32 * 131072 * 4
    assert ws(csa2.OP_INDEX_FULL, 32, 131072) < ws(csa2.OP_INDEX_FULL, 32, 262144)
    assert ws(csa2.OP_LAYER_GROUP, 8, 1 << 20) >= ws(csa2.OP_FORM_POOL, 8, 1 << 20)
    assert ws(csa2.OP_LAYER_GROUP, 8, 1 << 20) >= ws(csa2.OP_INDEX_REINDEX, 8, 0)
    assert ws(99, 1, 1) == 0


def test_host_validation_rejects_bad_arguments():
    lib = csa2.lib()
    nul = None
    # unsupported head dim / null pointers: rejected before any CUDA call
    assert lib.csa2_quantize_kv_fp4(nul, 1, 1, 256, nul, nul, nul, 10, nul, nul) == 2
    assert lib.csa2_quantize_kv_fp4(nul, 1, 1, 512, nul, nul, nul, 10, nul, nul) == 1
    assert lib.csa2_quantize_kv_fp4(ctypes.c_void_p(8), 1, 1, 512, nul, ctypes.c_void_p(16), ctypes.c_void_p(32), 10, nul, nul) == 1  # misaligned x
    assert lib.csa2_quantize_kv_fp4(nul, 0, 5, 512, nul, nul, nul, 10, nul, nul) == 0   # empty: nothing to do
    assert lib.csa2_index_scores(nul, nul, nul, 0, nul, 1, 9, 128, 10, nul, 10, nul, nul) == 2   # H_I > 8
    assert lib.csa2_index_scores(nul, nul, nul, 0, nul, 1, 8, 96, 10, nul, 10, nul, nul) == 2    # d_I
    assert lib.csa2_topk(nul, nul, 10, nul, 1, 10, 4096, nul, nul, 0, nul) == 2                 # k too large
    assert lib.csa2_topk(ctypes.c_void_p(256), nul, 10, ctypes.c_void_p(256), 1, 10, 8, ctypes.c_void_p(256), nul, 0, nul) == 3  # no workspace
    assert lib.csa2_sparse_attn(nul, 1, 24, 512, nul, nul, 0, 0, nul, 512, nul, 128, 128, 0, nul, 0.1, nul, nul, 0, nul, nul) == 2  # H
    assert lib.csa2_sparse_attn(nul, 1, 64, 512, nul, nul, 0, 0, nul, 512, nul, 128, 129, 0, nul, 0.1, nul, nul, 0, nul, nul) == 2  # W
    assert lib.csa2_prefill_index_scores(nul, nul, 4, 4, 128, nul, 100, nul, 100, nul, nul) == 2  # H_I must be 8
    assert lib.csa2_prefill_group(None, nul) == 1
    assert lib.csa2_layer_group(None, nul) == 1
