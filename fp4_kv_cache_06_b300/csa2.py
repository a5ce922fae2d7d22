"""ctypes binding of libcsa2.so (argument marshalling only).

Every function takes torch CUDA tensors (PyTorch is used for device memory
and streams), checks dtype/shape/contiguity, and calls the C entry point of
the same name on the current CUDA stream. A non-zero status raises
:class:`Csa2Error`. Nothing here computes any part of the method.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libcsa2.so")

OK = 0
OP_TOPK, OP_INDEX_FULL, OP_INDEX_REINDEX, OP_FORM_POOL, OP_SPARSE_ATTN, OP_LAYER_GROUP = 1, 2, 3, 4, 5, 6
OP_PREFILL_GROUP = 7
OP_FORM_POOL_BLOCK_MAX = 8
POOL_NONE, POOL_MEAN_KEY, POOL_BLOCK_MAX = 0, 1, 2
MODE_FULL, MODE_REINDEX = 0, 1
TOPK_NOALLOC_MAX_ROWS = 64          # CSA2_TOPK_NOALLOC_MAX_ROWS

EXPORTS = (
    "csa2_status_string", "csa2_version", "csa2_launch_count", "csa2_workspace_size",
    "csa2_quantize_kv_fp4", "csa2_append_indexer_k", "csa2_block_means", "csa2_append_swa",
    "csa2_index_scores", "csa2_topk", "csa2_index_full", "csa2_form_pool", "csa2_form_pool_block_max",
    "csa2_index_reindex",
    "csa2_sparse_attn", "csa2_layer_group", "csa2_append_step", "csa2_append_step_ratio",
    "csa2_swa_export", "csa2_swa_restore",
    "csa2_prefill_index_scores",
    "csa2_prefill_group", "csa2_topk_noalloc", "csa2_debug_set_fault", "csa2_last_cuda_error",
)

_c_p, _c_i32, _c_i64, _c_sz, _c_f = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float


class Csa2Error(RuntimeError):
    pass


class GroupArgs(ctypes.Structure):
    """Mirror of ``csa2_group_args`` (include/csa2.h)."""
    _fields_ = [
        ("mode", _c_i32), ("n_reuse", _c_i32), ("form_pool", _c_i32),
        ("B", _c_i32), ("H", _c_i32), ("d", _c_i32), ("H_I", _c_i32), ("d_I", _c_i32),
        ("k", _c_i32), ("W", _c_i32), ("P", _c_i32),
        ("n_max", _c_i64), ("n_cap", _c_i64),
        ("n", _c_p), ("codes", _c_p), ("scales", _c_p), ("kI", _c_p), ("kbar", _c_p),
        ("qI", _c_p), ("w", _c_p), ("qI_pool", _c_p), ("w_pool", _c_p),
        ("pool", _c_p), ("idx", _c_p),
        ("q_layers", ctypes.POINTER(_c_p)), ("swa_layers", ctypes.POINTER(_c_p)),
        ("swa_len", _c_p), ("out_layers", ctypes.POINTER(_c_p)),
        ("softmax_scale", _c_f), ("ws", _c_p), ("ws_bytes", _c_sz), ("d_status", _c_p),
        ("events", ctypes.POINTER(_c_p)), ("n_events", _c_i32), ("rows_per_seq", _c_i32),
    ]


class PrefillArgs(ctypes.Structure):
    """Mirror of ``csa2_prefill_args`` (include/csa2.h)."""
    _fields_ = [
        ("Q", _c_i32), ("n_reuse", _c_i32), ("H", _c_i32), ("d", _c_i32), ("H_I", _c_i32), ("d_I", _c_i32),
        ("k", _c_i32), ("W", _c_i32), ("n_keys", _c_i64), ("n_vis", _c_p),
        ("codes", _c_p), ("scales", _c_p), ("kI", _c_p), ("qI", _c_p), ("w", _c_p), ("idx", _c_p),
        ("q_layers", ctypes.POINTER(_c_p)), ("swa_layers", ctypes.POINTER(_c_p)), ("swa_len", _c_p),
        ("out_layers", ctypes.POINTER(_c_p)), ("softmax_scale", _c_f), ("ws", _c_p), ("ws_bytes", _c_sz),
        ("d_status", _c_p), ("events", ctypes.POINTER(_c_p)), ("n_events", _c_i32),
    ]


_lib = None


def lib() -> ctypes.CDLL:
    """Load libcsa2.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise Csa2Error(f"{LIB_PATH} is missing: build it with `python -m fp4_kv_cache_06_b300.build`")
    L = ctypes.CDLL(LIB_PATH)
    L.csa2_status_string.restype = ctypes.c_char_p
    L.csa2_status_string.argtypes = [ctypes.c_int]
    L.csa2_version.restype = ctypes.c_int
    L.csa2_launch_count.restype = ctypes.c_uint64
    L.csa2_workspace_size.restype = _c_sz
    L.csa2_workspace_size.argtypes = [_c_i32, _c_i32, _c_i64, _c_i32, _c_i32, _c_i32]
    L.csa2_quantize_kv_fp4.argtypes = [_c_p, _c_i32, _c_i64, _c_i32, _c_p, _c_p, _c_p, _c_i64, _c_p, _c_p]
    L.csa2_append_indexer_k.argtypes = [_c_p, _c_i32, _c_i64, _c_i32, _c_p, _c_p, _c_p, _c_i64, _c_p, _c_p]
    L.csa2_block_means.argtypes = [_c_p, _c_i32, _c_i32, _c_p, _c_i64, _c_i64, _c_p, _c_p, _c_p]
    L.csa2_append_swa.argtypes = [_c_p, _c_i32, _c_i32, _c_p, _c_p, _c_i32, _c_p]
    L.csa2_index_scores.argtypes = [_c_p, _c_p, _c_p, _c_i64, _c_p, _c_i32, _c_i32, _c_i32, _c_i64, _c_p, _c_i64, _c_p, _c_p]
    L.csa2_topk.argtypes = [_c_p, _c_p, _c_i64, _c_p, _c_i32, _c_i64, _c_i32, _c_p, _c_p, _c_sz, _c_p]
    L.csa2_index_full.argtypes = [_c_p, _c_p, _c_p, _c_i64, _c_p, _c_i32, _c_i32, _c_i32, _c_i64, _c_i32, _c_p, _c_p, _c_p, _c_sz, _c_p, _c_p]
    L.csa2_form_pool.argtypes = [_c_p, _c_p, _c_p, _c_i64, _c_p, _c_i32, _c_i32, _c_i32, _c_i64, _c_i32, _c_p, _c_p, _c_sz, _c_p, _c_p]
    L.csa2_form_pool_block_max.argtypes = [_c_p, _c_i64, _c_p, _c_i32, _c_i64, _c_i32, _c_p, _c_p, _c_sz, _c_p]
    L.csa2_index_reindex.argtypes = [_c_p, _c_p, _c_p, _c_i64, _c_p, _c_p, _c_i32, _c_i32, _c_i32, _c_i32, _c_i32, _c_p, _c_p, _c_sz, _c_p, _c_p]
    L.csa2_sparse_attn.argtypes = [_c_p, _c_i32, _c_i32, _c_i32, _c_p, _c_p, _c_i64, _c_i64, _c_p, _c_i32, _c_p, _c_i64, _c_i32, _c_i32, _c_p, _c_f, _c_p, _c_p, _c_sz, _c_p, _c_p]
    L.csa2_layer_group.argtypes = [ctypes.POINTER(GroupArgs), _c_p]
    L.csa2_prefill_index_scores.argtypes = [_c_p, _c_p, _c_i32, _c_i32, _c_i32, _c_p, _c_i64, _c_p, _c_i64, _c_p, _c_p]
    L.csa2_prefill_group.argtypes = [ctypes.POINTER(PrefillArgs), _c_p]
    L.csa2_debug_set_fault.argtypes = [_c_i32, _c_i64]
    L.csa2_last_cuda_error.restype = ctypes.c_char_p
    L.csa2_append_step.argtypes = [_c_p, _c_p, ctypes.POINTER(_c_p), ctypes.POINTER(_c_p), _c_i32, _c_i32, _c_i32,
                                   _c_i32, _c_i32, _c_p, _c_p, _c_p, _c_p, _c_p, _c_i64, _c_p, _c_p]
    L.csa2_swa_export.argtypes = [ctypes.POINTER(_c_p), _c_i32, _c_i32, _c_i32, _c_i32, _c_p, ctypes.POINTER(_c_p), _c_p]
    L.csa2_swa_restore.argtypes = [ctypes.POINTER(_c_p), _c_i32, _c_i32, _c_i32, _c_i32, _c_p, ctypes.POINTER(_c_p),
                                   _c_p, _c_p]
    L.csa2_append_step_ratio.argtypes = [_c_p, _c_p, ctypes.POINTER(_c_p), ctypes.POINTER(_c_p), _c_i32, _c_i32,
                                         _c_i32, _c_i32, _c_i32, _c_p, _c_i32, _c_p, _c_p, _c_p, _c_p, _c_i64,
                                         _c_p, _c_p, _c_p, _c_p]
    for name in EXPORTS:
        if name not in ("csa2_status_string", "csa2_version", "csa2_launch_count", "csa2_workspace_size",
                        "csa2_last_cuda_error"):
            getattr(L, name).restype = ctypes.c_int
    _lib = L
    return L


# ---- marshalling helpers ------------------------------------------------------
def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check(rc: int, what: str):
    if rc != OK:
        msg = f"{what}: {lib().csa2_status_string(rc).decode()}"
        if rc == 4:                                   # CSA2_ERR_CUDA: add the CUDA error's text
            msg += f" ({lib().csa2_last_cuda_error().decode()})"
        raise Csa2Error(msg)


def _need(t: torch.Tensor, name: str, dtype, ndim=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {tuple(t.shape)}")


def _opt(t, name, dtype, ndim=None):
    if t is not None:
        _need(t, name, dtype, ndim)


def workspace_size(op: int, B: int, n_max: int = 0, k: int = 512, P: int = 2048, H: int = 64) -> int:
    return int(lib().csa2_workspace_size(op, B, n_max, k, P, H))


def alloc_workspace(nbytes: int, device="cuda") -> torch.Tensor:
    """A uint8 device buffer of at least nbytes (torch's allocator aligns to 512 B)."""
    t = torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)
    assert t.data_ptr() % 256 == 0
    return t


def launch_count() -> int:
    return int(lib().csa2_launch_count())


def version() -> int:
    return int(lib().csa2_version())


FAULT_NONE, FAULT_ATTN, FAULT_SCAN, FAULT_PREFILL = 0, 1, 2, 3


def debug_set_fault(fault: int, wait_ns: int = 0):
    """Test hook (csa2_debug_set_fault): make later launches of one kernel
    withhold a signal so that its bounded device waits run out, and set the
    bound of every device wait (0 = the 2 s default)."""
    _check(lib().csa2_debug_set_fault(int(fault), int(wait_ns)), "csa2_debug_set_fault")


# ---- entry points ---------------------------------------------------------------
def csa2_quantize_kv_fp4(x, codes, scales, pos=None, d_status=None, stream=None):
    """x [B][rows][512] bf16 -> codes [B][n_cap][256] u8, scales [B][n_cap][32] u8 at pos[b]+r."""
    _need(x, "x", torch.bfloat16, 3)
    _need(codes, "codes", torch.uint8, 3)
    _need(scales, "scales", torch.uint8, 3)
    _opt(pos, "pos", torch.int64, 1)
    _opt(d_status, "d_status", torch.int32)
    B, rows, d = x.shape
    rc = lib().csa2_quantize_kv_fp4(_ptr(x), B, rows, d, _ptr(pos), _ptr(codes), _ptr(scales),
                                    codes.shape[1], _ptr(d_status), _stream(stream))
    _check(rc, "csa2_quantize_kv_fp4")


def csa2_append_indexer_k(k_new, kI, kbar=None, pos=None, d_status=None, stream=None):
    """k_new [B][rows][d_I] u8 -> kI [B][n_cap][d_I] at pos[b]+r; refreshes kbar block means."""
    _need(k_new, "k_new", torch.uint8, 3)
    _need(kI, "kI", torch.uint8, 3)
    _opt(kbar, "kbar", torch.uint8, 3)
    _opt(pos, "pos", torch.int64, 1)
    B, rows, d_I = k_new.shape
    rc = lib().csa2_append_indexer_k(_ptr(k_new), B, rows, d_I, _ptr(pos), _ptr(kI), _ptr(kbar),
                                     kI.shape[1], _ptr(d_status), _stream(stream))
    _check(rc, "csa2_append_indexer_k")


def csa2_block_means(kI, n, kbar, n_max, d_status=None, stream=None):
    _need(kI, "kI", torch.uint8, 3)
    _need(n, "n", torch.int64, 1)
    _need(kbar, "kbar", torch.uint8, 3)
    B, n_cap, d_I = kI.shape
    rc = lib().csa2_block_means(_ptr(kI), B, d_I, _ptr(n), int(n_max), n_cap, _ptr(kbar),
                                _ptr(d_status), _stream(stream))
    _check(rc, "csa2_block_means")


def csa2_append_swa(x, pos, swa, stream=None):
    """x [B][512] bf16 -> swa [B][W][512] at slot pos[b] % W."""
    _need(x, "x", torch.bfloat16, 2)
    _need(pos, "pos", torch.int64, 1)
    _need(swa, "swa", torch.bfloat16, 3)
    B, d = x.shape
    rc = lib().csa2_append_swa(_ptr(x), B, d, _ptr(pos), _ptr(swa), swa.shape[1], _stream(stream))
    _check(rc, "csa2_append_swa")


def csa2_append_step(kv_new, kI_new, swa_new: Sequence[torch.Tensor], swa: Sequence[torch.Tensor], pos, codes,
                     scales, kI, kbar=None, d_status=None, stream=None):
    """One decode token into every cache in one launch: kv_new [B][512] bf16 (FP4 main KV),
    kI_new [B][d_I] u8 (indexer key + block mean), swa_new[l] [B][512] -> swa[l] [B][W][512]."""
    _need(kv_new, "kv_new", torch.bfloat16, 2)
    _need(kI_new, "kI_new", torch.uint8, 2)
    _need(pos, "pos", torch.int64, 1)
    _need(codes, "codes", torch.uint8, 3)
    _need(scales, "scales", torch.uint8, 3)
    _need(kI, "kI", torch.uint8, 3)
    _opt(kbar, "kbar", torch.uint8, 3)
    L = len(swa_new)
    if len(swa) != L:
        raise ValueError("swa_new and swa must have the same length")
    for i in range(L):
        _need(swa_new[i], f"swa_new[{i}]", torch.bfloat16, 2)
        _need(swa[i], f"swa[{i}]", torch.bfloat16, 3)
    B, d = kv_new.shape
    W = swa[0].shape[1] if L else 1
    sn = (_c_p * max(L, 1))(*[t.data_ptr() for t in swa_new])
    sw = (_c_p * max(L, 1))(*[t.data_ptr() for t in swa])
    rc = lib().csa2_append_step(_ptr(kv_new), _ptr(kI_new), sn, sw, L, W, B, d, kI_new.shape[1], _ptr(pos),
                                _ptr(codes), _ptr(scales), _ptr(kI), _ptr(kbar), codes.shape[1], _ptr(d_status),
                                _stream(stream))
    _check(rc, "csa2_append_step")


def csa2_append_step_ratio(kv_new, kI_new, swa_new: Sequence[torch.Tensor], swa: Sequence[torch.Tensor], pos, ratio,
                           codes, scales, kI, kbar=None, n_vis_out=None, swa_len_out=None, d_status=None,
                           stream=None):
    """One token at compression ratio `ratio`: every layer's SWA row at slot pos % W; the
    compressed entry (kv_new [B][512] bf16, kI_new [B][d_I]) only when it completes at this
    token, at entry index (pos + 1) / ratio - 1. Optionally writes the visible entry count
    n_vis_out [B] int64 and swa_len_out [B] int32."""
    _need(kv_new, "kv_new", torch.bfloat16, 2)
    _need(kI_new, "kI_new", torch.uint8, 2)
    _need(pos, "pos", torch.int64, 1)
    _need(codes, "codes", torch.uint8, 3)
    _need(scales, "scales", torch.uint8, 3)
    _need(kI, "kI", torch.uint8, 3)
    _opt(kbar, "kbar", torch.uint8, 3)
    _opt(n_vis_out, "n_vis_out", torch.int64, 1)
    _opt(swa_len_out, "swa_len_out", torch.int32, 1)
    L = len(swa_new)
    if len(swa) != L:
        raise ValueError("swa_new and swa must have the same length")
    for i in range(L):
        _need(swa_new[i], f"swa_new[{i}]", torch.bfloat16, 2)
        _need(swa[i], f"swa[{i}]", torch.bfloat16, 3)
    B, d = kv_new.shape
    W = swa[0].shape[1] if L else 128
    sn = (_c_p * max(L, 1))(*[t.data_ptr() for t in swa_new])
    sw = (_c_p * max(L, 1))(*[t.data_ptr() for t in swa])
    rc = lib().csa2_append_step_ratio(_ptr(kv_new), _ptr(kI_new), sn, sw, L, W, B, d, kI_new.shape[1], _ptr(pos),
                                      int(ratio), _ptr(codes), _ptr(scales), _ptr(kI), _ptr(kbar), codes.shape[1],
                                      _ptr(n_vis_out), _ptr(swa_len_out), _ptr(d_status), _stream(stream))
    _check(rc, "csa2_append_step_ratio")


def _swa_lists(a, b, n):
    _need(n, "n", torch.int64, 1)
    if len(a) != len(b) or not a:
        raise ValueError("one array per layer on both sides")
    for i in range(len(a)):
        _need(a[i], f"layer {i}", torch.bfloat16, 3)
        _need(b[i], f"layer {i}", torch.bfloat16, 3)
    L = len(a)
    B, W, d = a[0].shape
    return L, W, B, d, (_c_p * L)(*[t.data_ptr() for t in a]), (_c_p * L)(*[t.data_ptr() for t in b])


def csa2_swa_export(rings, n, rows_out, stream=None):
    """Each layer's window in token order: rows_out[l][b][i] = token n[b]-c+i (c = min(n[b], W))."""
    L, W, B, d, pa, pb = _swa_lists(rings, rows_out, n)
    _check(lib().csa2_swa_export(pa, L, W, B, d, _ptr(n), pb, _stream(stream)), "csa2_swa_export")


def csa2_swa_restore(rows, n, rings, swa_len_out=None, stream=None):
    """Write token-ordered window rows back into each layer's ring (token t at slot t % W)."""
    _opt(swa_len_out, "swa_len_out", torch.int32, 1)
    L, W, B, d, pa, pb = _swa_lists(rows, rings, n)
    _check(lib().csa2_swa_restore(pa, L, W, B, d, _ptr(n), pb, _ptr(swa_len_out), _stream(stream)),
           "csa2_swa_restore")


def csa2_index_scores(qI, w, kI, n, n_max, scores, kI_seq_stride=None, d_status=None, stream=None):
    """scores[b][t] = sum_h w[b][h] relu(qI[b][h] . kI[b][t]) for t < n[b]."""
    _need(qI, "qI", torch.uint8, 3)
    _need(w, "w", torch.float32, 2)
    _need(kI, "kI", torch.uint8)
    _need(n, "n", torch.int64, 1)
    _need(scores, "scores", torch.float32, 2)
    B, H_I, d_I = qI.shape
    stride = kI.shape[-2] if kI_seq_stride is None else int(kI_seq_stride)
    rc = lib().csa2_index_scores(_ptr(qI), _ptr(w), _ptr(kI), stride, _ptr(n), B, H_I, d_I, int(n_max),
                                 _ptr(scores), scores.shape[1], _ptr(d_status), _stream(stream))
    _check(rc, "csa2_index_scores")


def csa2_topk(scores, n, n_max, k, idx_out, ws, cand_pos=None, stream=None):
    _need(scores, "scores", torch.float32, 2)
    _opt(n, "n", torch.int64, 1)
    _need(idx_out, "idx_out", torch.int32, 2)
    _opt(cand_pos, "cand_pos", torch.int32, 2)
    _need(ws, "ws", torch.uint8)
    B = scores.shape[0]
    rc = lib().csa2_topk(_ptr(scores), _ptr(cand_pos), scores.shape[1], _ptr(n), B, int(n_max), int(k),
                         _ptr(idx_out), _ptr(ws), ws.numel(), _stream(stream))
    _check(rc, "csa2_topk")


def csa2_index_full(qI, w, kI, n, n_max, k, idx_out, ws, scores_out=None, kI_seq_stride=None,
                    d_status=None, stream=None):
    _need(qI, "qI", torch.uint8, 3)
    _need(w, "w", torch.float32, 2)
    _need(kI, "kI", torch.uint8)
    _need(n, "n", torch.int64, 1)
    _need(idx_out, "idx_out", torch.int32, 2)
    _opt(scores_out, "scores_out", torch.float32, 2)
    _need(ws, "ws", torch.uint8)
    B, H_I, d_I = qI.shape
    stride = kI.shape[-2] if kI_seq_stride is None else int(kI_seq_stride)
    rc = lib().csa2_index_full(_ptr(qI), _ptr(w), _ptr(kI), stride, _ptr(n), B, H_I, d_I, int(n_max), int(k),
                               _ptr(idx_out), _ptr(scores_out), _ptr(ws), ws.numel(), _ptr(d_status),
                               _stream(stream))
    _check(rc, "csa2_index_full")


def csa2_form_pool(qI, w, kbar, n, n_max, P, pool_out, ws, kbar_seq_stride=None, d_status=None, stream=None):
    _need(qI, "qI", torch.uint8, 3)
    _need(w, "w", torch.float32, 2)
    _need(kbar, "kbar", torch.uint8)
    _need(n, "n", torch.int64, 1)
    _need(pool_out, "pool_out", torch.int32, 2)
    _need(ws, "ws", torch.uint8)
    B, H_I, d_I = qI.shape
    stride = kbar.shape[-2] if kbar_seq_stride is None else int(kbar_seq_stride)
    rc = lib().csa2_form_pool(_ptr(qI), _ptr(w), _ptr(kbar), stride, _ptr(n), B, H_I, d_I, int(n_max), int(P),
                              _ptr(pool_out), _ptr(ws), ws.numel(), _ptr(d_status), _stream(stream))
    _check(rc, "csa2_form_pool")


def csa2_form_pool_block_max(scores, n, n_max, P, pool_out, ws, stream=None):
    """Pool by the max-of-token rule: scores [B][stride] fp32 from a Full scan."""
    _need(scores, "scores", torch.float32, 2)
    _need(pool_out, "pool_out", torch.int32, 2)
    _need(ws, "ws", torch.uint8)
    _opt(n, "n", torch.int64, 1)
    B = scores.shape[0]
    rc = lib().csa2_form_pool_block_max(_ptr(scores), scores.shape[1], _ptr(n), B, int(n_max), int(P),
                                        _ptr(pool_out), _ptr(ws), ws.numel(), _stream(stream))
    _check(rc, "csa2_form_pool_block_max")


def csa2_index_reindex(qI, w, kI, n, pool, k, idx_out, ws, kI_seq_stride=None, d_status=None, stream=None):
    _need(qI, "qI", torch.uint8, 3)
    _need(w, "w", torch.float32, 2)
    _need(kI, "kI", torch.uint8)
    _need(n, "n", torch.int64, 1)
    _need(pool, "pool", torch.int32, 2)
    _need(idx_out, "idx_out", torch.int32, 2)
    _need(ws, "ws", torch.uint8)
    B, H_I, d_I = qI.shape
    stride = kI.shape[-2] if kI_seq_stride is None else int(kI_seq_stride)
    rc = lib().csa2_index_reindex(_ptr(qI), _ptr(w), _ptr(kI), stride, _ptr(n), _ptr(pool), pool.shape[1], B,
                                  H_I, d_I, int(k), _ptr(idx_out), _ptr(ws), ws.numel(), _ptr(d_status),
                                  _stream(stream))
    _check(rc, "csa2_index_reindex")


def csa2_sparse_attn(q, codes, scales, idx, swa, swa_len, out, ws, softmax_scale=None, kv_seq_stride=None,
                     swa_seq_stride=None, W=None, swa_tail=False, d_status=None, stream=None):
    """q/out [B][H][512] bf16; codes/scales: [B or 1][n_cap][...]; idx [B][k] i32; swa rows bf16."""
    _need(q, "q", torch.bfloat16, 3)
    _need(codes, "codes", torch.uint8, 3)
    _need(scales, "scales", torch.uint8, 3)
    _need(idx, "idx", torch.int32, 2)
    _need(swa, "swa", torch.bfloat16)
    _need(swa_len, "swa_len", torch.int32, 1)
    _need(out, "out", torch.bfloat16, 3)
    _need(ws, "ws", torch.uint8)
    B, H, d = q.shape
    n_cap = codes.shape[1]
    kvs = n_cap if kv_seq_stride is None else int(kv_seq_stride)
    Wv = swa.shape[-2] if W is None else int(W)
    sws = Wv if swa_seq_stride is None else int(swa_seq_stride)
    scale = (1.0 / d ** 0.5) if softmax_scale is None else float(softmax_scale)
    rc = lib().csa2_sparse_attn(_ptr(q), B, H, d, _ptr(codes), _ptr(scales), kvs, n_cap, _ptr(idx), idx.shape[1],
                                _ptr(swa), sws, Wv, int(bool(swa_tail)), _ptr(swa_len), scale, _ptr(out), _ptr(ws), ws.numel(),
                                _ptr(d_status), _stream(stream))
    _check(rc, "csa2_sparse_attn")


def csa2_layer_group(mode, n, n_max, codes, scales, kI, qI, w, idx, q_layers: Sequence[torch.Tensor],
                     swa_layers: Sequence[torch.Tensor], swa_len, out_layers: Sequence[torch.Tensor], ws,
                     kbar=None, pool=None, form_pool=False, qI_pool=None, w_pool=None, P=2048,
                     softmax_scale=None, d_status=None, events=None, stream=None, rows_per_seq=1):
    """One layer group: Full or Reindex, then attention for it and each Reuse layer.

    rows_per_seq R > 1: multi-token decode. The per-row arrays have B rows
    (R per sequence), the caches B / R sequences, and each SWA array
    [B / R][W + R - 1][d] holds the linear window rows of each sequence."""
    _need(n, "n", torch.int64, 1)
    _need(codes, "codes", torch.uint8, 3)
    _need(scales, "scales", torch.uint8, 3)
    _need(kI, "kI", torch.uint8, 3)
    _need(qI, "qI", torch.uint8, 3)
    _need(w, "w", torch.float32, 2)
    _need(idx, "idx", torch.int32, 2)
    _need(swa_len, "swa_len", torch.int32, 1)
    _need(ws, "ws", torch.uint8)
    _opt(kbar, "kbar", torch.uint8, 3)
    _opt(pool, "pool", torch.int32, 2)
    L = len(q_layers)
    if L < 1 or len(swa_layers) != L or len(out_layers) != L:
        raise ValueError("q_layers, swa_layers and out_layers must have the same non-zero length")
    for i in range(L):
        _need(q_layers[i], f"q_layers[{i}]", torch.bfloat16, 3)
        _need(swa_layers[i], f"swa_layers[{i}]", torch.bfloat16, 3)
        _need(out_layers[i], f"out_layers[{i}]", torch.bfloat16, 3)
    B, H, d = q_layers[0].shape
    _, H_I, d_I = qI.shape
    a = GroupArgs()
    a.mode = int(mode)
    a.n_reuse = L - 1
    a.form_pool = int(form_pool)               # False/True -> none/mean-key; or a POOL_* rule
    a.B, a.H, a.d, a.H_I, a.d_I = B, H, d, H_I, d_I
    a.k = idx.shape[1]
    R = max(1, int(rows_per_seq))
    if B % R:
        raise ValueError("the row count must be a multiple of rows_per_seq")
    a.rows_per_seq = R
    a.W = swa_layers[0].shape[1] - (R - 1)
    a.P = int(P) if pool is None else pool.shape[1]
    a.n_max, a.n_cap = int(n_max), codes.shape[1]
    a.n, a.codes, a.scales, a.kI, a.kbar = n.data_ptr(), codes.data_ptr(), scales.data_ptr(), kI.data_ptr(), (kbar.data_ptr() if kbar is not None else None)
    a.qI, a.w = qI.data_ptr(), w.data_ptr()
    a.qI_pool = qI_pool.data_ptr() if qI_pool is not None else None
    a.w_pool = w_pool.data_ptr() if w_pool is not None else None
    a.pool = pool.data_ptr() if pool is not None else None
    a.idx = idx.data_ptr()
    qa = (_c_p * L)(*[t.data_ptr() for t in q_layers])
    sa = (_c_p * L)(*[t.data_ptr() for t in swa_layers])
    oa = (_c_p * L)(*[t.data_ptr() for t in out_layers])
    a.q_layers, a.swa_layers, a.out_layers = qa, sa, oa
    a.swa_len = swa_len.data_ptr()
    a.softmax_scale = (1.0 / d ** 0.5) if softmax_scale is None else float(softmax_scale)
    a.ws, a.ws_bytes = ws.data_ptr(), ws.numel()
    a.d_status = d_status.data_ptr() if d_status is not None else None
    if events:
        ea = (_c_p * len(events))(*[e.cuda_event for e in events])
        a.events, a.n_events = ea, len(events)
    else:
        a.events, a.n_events = None, 0
    rc = lib().csa2_layer_group(ctypes.byref(a), _stream(stream))
    _check(rc, "csa2_layer_group")


def csa2_prefill_index_scores(qI, w, kI, scores, d_status=None, stream=None):
    """scores[q][j] = sum_h w[q][h] relu(qI[q][h] . kI[j]) on the tensor cores (qI [Q][8][128], kI [n][128])."""
    _need(qI, "qI", torch.uint8, 3)
    _need(w, "w", torch.float32, 2)
    _need(kI, "kI", torch.uint8, 2)
    _need(scores, "scores", torch.float32, 2)
    Q, H_I, d_I = qI.shape
    rc = lib().csa2_prefill_index_scores(_ptr(qI), _ptr(w), Q, H_I, d_I, _ptr(kI), kI.shape[0], _ptr(scores),
                                         scores.shape[1], _ptr(d_status), _stream(stream))
    _check(rc, "csa2_prefill_index_scores")


def csa2_prefill_group(n_vis, codes, scales, kI, qI, w, idx, q_layers, swa_layers, swa_len, out_layers, ws,
                       softmax_scale=None, d_status=None, events=None, stream=None):
    """Encoder prefill group: indexer GEMM, per-query Top-K over n_vis[q] entries, attention per layer.
    codes/scales/kI: one shared cache [n_keys][...]; swa_layers[l]: [Q + W - 1][512] chunk rows."""
    _need(n_vis, "n_vis", torch.int64, 1)
    _need(codes, "codes", torch.uint8, 2)
    _need(scales, "scales", torch.uint8, 2)
    _need(kI, "kI", torch.uint8, 2)
    _need(qI, "qI", torch.uint8, 3)
    _need(w, "w", torch.float32, 2)
    _need(idx, "idx", torch.int32, 2)
    _need(swa_len, "swa_len", torch.int32, 1)
    _need(ws, "ws", torch.uint8)
    L = len(q_layers)
    for i in range(L):
        _need(q_layers[i], f"q_layers[{i}]", torch.bfloat16, 3)
        _need(swa_layers[i], f"swa_layers[{i}]", torch.bfloat16, 2)
        _need(out_layers[i], f"out_layers[{i}]", torch.bfloat16, 3)
    Q, H, d = q_layers[0].shape
    a = PrefillArgs()
    a.Q, a.n_reuse, a.H, a.d, a.H_I, a.d_I = Q, L - 1, H, d, qI.shape[1], qI.shape[2]
    a.k, a.W = idx.shape[1], swa_layers[0].shape[0] - Q + 1
    a.n_keys = codes.shape[0]
    a.n_vis, a.codes, a.scales, a.kI = n_vis.data_ptr(), codes.data_ptr(), scales.data_ptr(), kI.data_ptr()
    a.qI, a.w, a.idx = qI.data_ptr(), w.data_ptr(), idx.data_ptr()
    qa = (_c_p * L)(*[t.data_ptr() for t in q_layers])
    sa = (_c_p * L)(*[t.data_ptr() for t in swa_layers])
    oa = (_c_p * L)(*[t.data_ptr() for t in out_layers])
    a.q_layers, a.swa_layers, a.out_layers = qa, sa, oa
    a.swa_len = swa_len.data_ptr()
    a.softmax_scale = (1.0 / d ** 0.5) if softmax_scale is None else float(softmax_scale)
    a.ws, a.ws_bytes = ws.data_ptr(), ws.numel()
    a.d_status = d_status.data_ptr() if d_status is not None else None
    if events:
        ea = (_c_p * len(events))(*[e.cuda_event for e in events])
        a.events, a.n_events = ea, len(events)
    else:
        a.events, a.n_events = None, 0
    rc = lib().csa2_prefill_group(ctypes.byref(a), _stream(stream))
    _check(rc, "csa2_prefill_group")


def csa2_topk_noalloc(scores, n, n_max, k, idx_out, cand_pos=None, stream=None):
    """Top-K like csa2_topk but with no workspace argument.

    For callers that cannot allocate device memory: the library keeps the
    scratch in a fixed per-GPU device array (at most 64 rows per call).
    Calls that overlap on the GPU share that array and race; keep them
    ordered on one stream. The first call on a device does a one-time
    lookup of the array's address, so make it before any stream capture.
    """
    L = lib()
    f = L.csa2_topk_noalloc
    f.restype = ctypes.c_int
    f.argtypes = [_c_p, _c_p, _c_i64, _c_p, _c_i32, _c_i64, _c_i32, _c_p, _c_p]
    _need(scores, "scores", torch.float32, 2)
    _opt(n, "n", torch.int64, 1)
    _need(idx_out, "idx_out", torch.int32, 2)
    _opt(cand_pos, "cand_pos", torch.int32, 2)
    rc = f(_ptr(scores), _ptr(cand_pos), scores.shape[1], _ptr(n), scores.shape[0], int(n_max), int(k),
           _ptr(idx_out), _stream(stream))
    _check(rc, "csa2_topk_noalloc")
