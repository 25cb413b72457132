"""Python binding of libmsa: ctypes declarations of include/msa.h and thin
wrappers with the same names that only marshal torch tensors into pointers.

Every step of the path runs in the CUDA library.  There is no CPU or PyTorch
fallback: if libmsa.so is missing or fails to load, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

from . import build as _build

MSA_OK, MSA_ERR_NULL, MSA_ERR_SHAPE, MSA_ERR_DTYPE, MSA_ERR_UNSUPPORTED, MSA_ERR_WORKSPACE, \
    MSA_ERR_CUDA = range(7)
MSA_KV_BF16, MSA_KV_FP8_E4M3 = 0, 1
MSA_SCALE_NONE, MSA_SCALE_SCALAR, MSA_SCALE_PER_TOKEN_HEAD = 0, 1, 2
MSA_DEV_BAD_PAGE, MSA_DEV_BAD_LEN, MSA_DEV_MALFORMED, MSA_DEV_BAD_TABLE, MSA_DEV_TIMEOUT = \
    1, 2, 4, 8, 16

EXPORTED = ("msa_index_score", "msa_topk_build_table", "msa_sparse_paged_attn", "msa_decode",
            "msa_kv_insert", "msa_sparse_mla_decode", "msa_sparse_mla_workspace_size",
            "msa_workspace_size", "msa_status_string", "msa_check_bounded_wait")
MSA_CHECK_WAIT_TMEM, MSA_CHECK_WAIT_COPY = 1, 2


class MsaError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn}: {status_string(code)} (status {code})")
        self.code = code


class msa_batch(ctypes.Structure):
    _fields_ = [("cu_seqlens_q", ctypes.c_void_p), ("cu_seqlens_k", ctypes.c_void_p),
                ("context_lens", ctypes.c_void_p), ("block_table", ctypes.c_void_p),
                ("bt_stride", ctypes.c_int32), ("num_reqs", ctypes.c_int32),
                ("num_rows", ctypes.c_int32), ("num_pages", ctypes.c_int32),
                ("max_q_len", ctypes.c_int32),
                ("min_q_len", ctypes.c_int32)]


class msa_attn_args(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("num_rows", ctypes.c_int32),
                ("num_heads", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("k_cache", ctypes.c_void_p),
                ("v_cache", ctypes.c_void_p), ("kv_dtype", ctypes.c_int32),
                ("num_pages", ctypes.c_int32), ("scale_mode", ctypes.c_int32),
                ("k_scale", ctypes.c_void_p), ("v_scale", ctypes.c_void_p),
                ("sinks", ctypes.c_void_p), ("softmax_scale", ctypes.c_float),
                ("out", ctypes.c_void_p), ("lse", ctypes.c_void_p)]


class msa_index_cache(ctypes.Structure):
    _fields_ = [("k_cache", ctypes.c_void_p), ("k_scale", ctypes.c_void_p),
                ("dtype", ctypes.c_int32), ("heads", ctypes.c_int32), ("dim", ctypes.c_int32)]


class msa_mla_args(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("num_rows", ctypes.c_int32),
                ("num_heads", ctypes.c_int32), ("dqk", ctypes.c_int32), ("dv", ctypes.c_int32),
                ("kv_cache", ctypes.c_void_p), ("num_tokens", ctypes.c_int64),
                ("kv_indptr", ctypes.c_void_p), ("kv_indices", ctypes.c_void_p),
                ("max_tokens", ctypes.c_int32), ("sinks", ctypes.c_void_p),
                ("softmax_scale", ctypes.c_float), ("out", ctypes.c_void_p),
                ("lse", ctypes.c_void_p), ("q_dtype", ctypes.c_int32),
                ("kv_dtype", ctypes.c_int32), ("q_scale", ctypes.c_void_p),
                ("kv_scale", ctypes.c_void_p)]


class msa_trace(ctypes.Structure):
    _fields_ = [("after_score", ctypes.c_void_p), ("after_topk", ctypes.c_void_p),
                ("after_attn", ctypes.c_void_p), ("kernels", ctypes.c_int32)]


_lock = threading.Lock()
_lib: Optional[ctypes.CDLL] = None


def library_path() -> str:
    return _build.LIB


def lib(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load libmsa.so (building it first if asked and needed)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.LIB
            if build_if_missing and not _build.up_to_date():
                _build.build()
            if not os.path.exists(path):
                raise RuntimeError(f"libmsa.so not built ({path}); run "
                                   "python -m block_sparse_paged_02_gb300.build")
            L = ctypes.CDLL(path)
            P, i32 = ctypes.c_void_p, ctypes.c_int32
            L.msa_index_score.restype = ctypes.c_int
            L.msa_index_score.argtypes = [P, P, P, P, i32, P, P]
            L.msa_topk_build_table.restype = ctypes.c_int
            L.msa_topk_build_table.argtypes = [P, P, i32, i32, P, P, i32, P, P, P]
            L.msa_sparse_paged_attn.restype = ctypes.c_int
            L.msa_sparse_paged_attn.argtypes = [P, P, i32, P, P, ctypes.c_size_t, P, P]
            L.msa_decode.restype = ctypes.c_int
            L.msa_decode.argtypes = [P, P, P, i32, P, P, P, i32, P, P, ctypes.c_size_t, P, P, P]
            L.msa_kv_insert.restype = ctypes.c_int
            L.msa_kv_insert.argtypes = [P, P, P, i32, i32, P, P, i32, i32, P, P, P, P, i32, P,
                                        P]
            L.msa_sparse_mla_workspace_size.restype = ctypes.c_size_t
            L.msa_sparse_mla_workspace_size.argtypes = [i32, i32, i32]
            L.msa_sparse_mla_decode.restype = ctypes.c_int
            L.msa_sparse_mla_decode.argtypes = [P, P, ctypes.c_size_t, P, P]
            L.msa_workspace_size.restype = ctypes.c_size_t
            L.msa_workspace_size.argtypes = [i32, i32, i32, i32, i32, i32]
            L.msa_check_bounded_wait.restype = ctypes.c_int
            L.msa_check_bounded_wait.argtypes = [P, ctypes.c_uint32, i32, P, P]
            L.msa_status_string.restype = ctypes.c_char_p
            L.msa_status_string.argtypes = [ctypes.c_int]
            _lib = L
    return _lib


def msa_status_string(code: int) -> str:
    return lib().msa_status_string(int(code)).decode()


status_string = msa_status_string


def _p(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("libmsa takes device tensors")
    if not t.is_contiguous():
        raise ValueError("libmsa takes contiguous tensors")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _check(fn: str, code: int):
    if code != MSA_OK:
        raise MsaError(fn, code)


def make_batch(cu_seqlens_q, cu_seqlens_k, context_lens, block_table, num_pages: int,
               num_rows: Optional[int] = None, max_q_len: int = 0,
               min_q_len: int = 0) -> msa_batch:
    for t in (cu_seqlens_q, cu_seqlens_k, context_lens, block_table):
        if t.dtype != torch.int32:
            raise ValueError("batch geometry arrays are int32")
    b = msa_batch(_p(cu_seqlens_q), _p(cu_seqlens_k), _p(context_lens), _p(block_table),
                  int(block_table.shape[1]), int(context_lens.shape[0]),
                  int(num_rows if num_rows is not None else 0), int(num_pages), int(max_q_len),
                  int(min_q_len))
    b._keep = (cu_seqlens_q, cu_seqlens_k, context_lens, block_table)
    return b


def check_sinks(sinks: Optional[torch.Tensor], num_heads: int):
    """Sink contract of the sparse-MLA sink PR: fp32, 1-D, num_heads long,
    contiguous -- a C ABI cannot see dtypes, so it is checked here."""
    if sinks is None:
        return
    if sinks.dtype != torch.float32:
        raise ValueError(f"sinks must be float32, got {sinks.dtype}")
    if sinks.ndim != 1 or sinks.numel() != num_heads:
        raise ValueError(f"sinks must have shape ({num_heads},), got {tuple(sinks.shape)}")
    if not sinks.is_contiguous():
        raise ValueError("sinks must be contiguous")


def make_index_cache(k_cache, dtype: int = MSA_KV_BF16, k_scale=None) -> msa_index_cache:
    """The paged index-K cache [P, 128, heads, dim] (bf16, or e4m3 codes with
    optional fp32 per-token scales [P, 128, heads])."""
    x = msa_index_cache(_p(k_cache), _p(k_scale), int(dtype), int(k_cache.shape[2]),
                        int(k_cache.shape[3]))
    x._keep = (k_cache, k_scale)
    return x


def make_attn_args(q, k_cache, v_cache, kv_dtype: int, num_pages: int, out, lse, *,
                   scale_mode: int = MSA_SCALE_NONE, k_scale=None, v_scale=None, sinks=None,
                   softmax_scale: float) -> msa_attn_args:
    check_sinks(sinks, int(q.shape[1]))
    a = msa_attn_args(_p(q), int(q.shape[0]), int(q.shape[1]), int(k_cache.shape[-2]),
                      int(q.shape[2]), _p(k_cache), _p(v_cache), int(kv_dtype), int(num_pages),
                      int(scale_mode), _p(k_scale), _p(v_scale), _p(sinks),
                      float(softmax_scale), _p(out), _p(lse))
    a._keep = (q, k_cache, v_cache, out, lse, k_scale, v_scale, sinks)
    return a


# ------------------------------------------------------------- entry points

def msa_workspace_size(num_rows, bt_stride, topk, num_heads, head_dim, tbl_stride) -> int:
    return int(lib().msa_workspace_size(int(num_rows), int(bt_stride), int(topk),
                                        int(num_heads), int(head_dim), int(tbl_stride)))


def msa_index_score(batch: msa_batch, idx_q, index: msa_index_cache, scores, score_stride,
                    dev_status, stream=None):
    _check("msa_index_score", lib().msa_index_score(
        ctypes.byref(batch), _p(idx_q), ctypes.byref(index), _p(scores), int(score_stride),
        _p(dev_status), _stream(stream)))


def msa_topk_build_table(batch: msa_batch, scores, score_stride, topk, topk_idx, sparse_tbl,
                         tbl_stride, sparse_len, dev_status, stream=None):
    _check("msa_topk_build_table", lib().msa_topk_build_table(
        ctypes.byref(batch), _p(scores), int(score_stride), int(topk), _p(topk_idx),
        _p(sparse_tbl), int(tbl_stride), _p(sparse_len), _p(dev_status), _stream(stream)))


def msa_sparse_paged_attn(attn: msa_attn_args, sparse_tbl, tbl_stride, sparse_len, workspace,
                          dev_status, stream=None):
    _check("msa_sparse_paged_attn", lib().msa_sparse_paged_attn(
        ctypes.byref(attn), _p(sparse_tbl), int(tbl_stride), _p(sparse_len), _p(workspace),
        int(workspace.numel() * workspace.element_size()) if workspace is not None else 0,
        _p(dev_status), _stream(stream)))


def msa_decode(batch: msa_batch, idx_q, index: msa_index_cache, topk, attn: msa_attn_args,
               topk_idx, sparse_tbl, tbl_stride, sparse_len, workspace, dev_status,
               trace: Optional[msa_trace] = None, stream=None):
    _check("msa_decode", lib().msa_decode(
        ctypes.byref(batch), _p(idx_q), ctypes.byref(index), int(topk), ctypes.byref(attn),
        _p(topk_idx), _p(sparse_tbl), int(tbl_stride), _p(sparse_len), _p(workspace),
        int(workspace.numel() * workspace.element_size()) if workspace is not None else 0,
        _p(dev_status), ctypes.byref(trace) if trace is not None else None, _stream(stream)))


def msa_kv_insert(batch: msa_batch, k_new, v_new, num_kv_heads, head_dim, k_cache, v_cache,
                  kv_dtype, scale_mode, k_scale, v_scale, idx_new,
                  index: Optional[msa_index_cache], skip_index, dev_status, stream=None):
    _check("msa_kv_insert", lib().msa_kv_insert(
        ctypes.byref(batch), _p(k_new), _p(v_new), int(num_kv_heads), int(head_dim),
        _p(k_cache), _p(v_cache), int(kv_dtype), int(scale_mode), _p(k_scale), _p(v_scale),
        _p(idx_new), ctypes.byref(index) if index is not None else None,
        int(bool(skip_index)), _p(dev_status), _stream(stream)))


def make_mla_args(q, kv_cache, kv_indptr, kv_indices, out, lse, *, max_tokens: int,
                  sinks=None, softmax_scale: float, q_scale=None,
                  kv_scale=None) -> msa_mla_args:
    """Sparse MLA operands: q [N, H, 576] bf16 (or uint8 e4m3 codes with
    q_scale), kv_cache [T, 576] bf16 (or uint8 e4m3 codes with kv_scale),
    int32 kv_indptr [N+1] / kv_indices, out [N, H, 512] bf16, lse [N, H]
    fp32; scales are device fp32 [1]."""
    check_sinks(sinks, int(q.shape[1]))
    for t in (kv_indptr, kv_indices):
        if t.dtype != torch.int32:
            raise ValueError("kv_indptr / kv_indices are int32")
    q8 = q.dtype == torch.uint8
    kv8 = kv_cache.dtype == torch.uint8
    a = msa_mla_args(_p(q), int(q.shape[0]), int(q.shape[1]), int(q.shape[2]),
                     int(out.shape[2]), _p(kv_cache), int(kv_cache.shape[0]), _p(kv_indptr),
                     _p(kv_indices), int(max_tokens), _p(sinks), float(softmax_scale), _p(out),
                     _p(lse), MSA_KV_FP8_E4M3 if q8 else MSA_KV_BF16,
                     MSA_KV_FP8_E4M3 if kv8 else MSA_KV_BF16, _p(q_scale), _p(kv_scale))
    a._keep = (q, kv_cache, kv_indptr, kv_indices, out, lse, sinks, q_scale, kv_scale)
    return a


def msa_sparse_mla_workspace_size(num_rows, num_heads, max_tokens) -> int:
    return int(lib().msa_sparse_mla_workspace_size(int(num_rows), int(num_heads),
                                                   int(max_tokens)))


def msa_sparse_mla_decode(mla: msa_mla_args, workspace, dev_status, stream=None):
    _check("msa_sparse_mla_decode", lib().msa_sparse_mla_decode(
        ctypes.byref(mla), _p(workspace),
        int(workspace.numel() * workspace.element_size()) if workspace is not None else 0,
        _p(dev_status), _stream(stream)))


def msa_check_bounded_wait(dev_status, limit_us: int, flags: int = 0, copy_src=None,
                           stream=None):
    """Run the bounded-wait check (see msa.h): a wait that nothing satisfies
    gives up after limit_us and sets MSA_DEV_TIMEOUT in dev_status."""
    _check("msa_check_bounded_wait", lib().msa_check_bounded_wait(
        _p(dev_status), int(limit_us), int(flags), _p(copy_src), _stream(stream)))


def make_trace(after_score=None, after_topk=None, after_attn=None) -> msa_trace:
    """Events (torch.cuda.Event, created with enable_timing) that msa_decode
    records after each stage.  torch creates an event lazily on its first
    record, so each is recorded once here to obtain its handle."""
    for e in (after_score, after_topk, after_attn):
        if e is not None and not e.cuda_event:
            e.record()
    h = lambda e: ctypes.c_void_p(e.cuda_event) if e is not None else None
    t = msa_trace(h(after_score), h(after_topk), h(after_attn), 0)
    t._keep = (after_score, after_topk, after_attn)
    return t
