"""CPU oracle for the block-sparse paged decode path -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product package never does: it
has no CPU fallback.

The arithmetic lives in ``msa_oracle.c`` (plain C, fp64, one sequential
loop per row, rows shared across pthreads); this module only compiles it
with gcc and marshals numpy arrays into it.  It shares no code with the
CUDA library.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "msa_oracle.c")
_HDR = os.path.join(_HERE, "msa_oracle.h")
_LIB = os.path.join(_HERE, "libmsa_oracle.so")
_lock = threading.Lock()
_lib = None

BAD_PAGE, BAD_LEN, MALFORMED, BAD_TABLE = 1, 2, 4, 8


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (IEEE arithmetic: no fast-math)."""
    newest = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < newest:
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                               "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


class _Batch(ctypes.Structure):
    _fields_ = [("num_reqs", ctypes.c_int32), ("num_rows", ctypes.c_int32),
                ("cu_seqlens_q", ctypes.c_void_p), ("cu_seqlens_k", ctypes.c_void_p),
                ("context_lens", ctypes.c_void_p), ("block_table", ctypes.c_void_p),
                ("bt_stride", ctypes.c_int32), ("num_pages", ctypes.c_int32)]


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i32 = ctypes.c_int32
            lib.orc_fp8_e4m3_value.restype = ctypes.c_double
            lib.orc_fp8_e4m3_value.argtypes = [ctypes.c_uint8]
            lib.orc_bf16_value.restype = ctypes.c_double
            lib.orc_bf16_value.argtypes = [ctypes.c_uint16]
            lib.orc_row_geometry.restype = ctypes.c_uint32
            lib.orc_row_geometry.argtypes = [P, P, P, P, P]
            lib.orc_index_score.restype = ctypes.c_uint32
            lib.orc_index_score.argtypes = [P, P, P, i32, i32, P, i32, i32]
            lib.orc_sparse_mla.restype = ctypes.c_uint32
            lib.orc_sparse_mla.argtypes = [i32, i32, i32, i32, P, P, ctypes.c_int64, P, P, P,
                                           ctypes.c_double, P, P, i32]
            lib.orc_sparse_mla_ex.restype = ctypes.c_uint32
            lib.orc_sparse_mla_ex.argtypes = [i32, i32, i32, i32, P, i32, ctypes.c_double, P,
                                              i32, ctypes.c_double, ctypes.c_int64, P, P, P,
                                              ctypes.c_double, P, P, i32]
            lib.orc_index_score_fp8.restype = ctypes.c_uint32
            lib.orc_index_score_fp8.argtypes = [P, P, P, P, i32, i32, P, i32, i32]
            lib.orc_topk_build_table.restype = ctypes.c_uint32
            lib.orc_topk_build_table.argtypes = [P, P, i32, i32, P, P, i32, P, i32]
            lib.orc_sparse_attn.restype = ctypes.c_uint32
            lib.orc_sparse_attn.argtypes = [i32, i32, i32, i32, P, P, P, i32, i32, i32, P, P, P,
                                            i32, P, P, ctypes.c_double, P, P, i32]
            lib.orc_fp8_e4m3_encode.restype = ctypes.c_uint8
            lib.orc_fp8_e4m3_encode.argtypes = [ctypes.c_float]
            lib.orc_kv_insert.restype = ctypes.c_uint32
            lib.orc_kv_insert.argtypes = [P, i32, i32, P, P, i32, i32, P, P, P, P, i32, i32, P, P,
                                          i32, i32, P]
            lib.orc_dense_attn.restype = ctypes.c_uint32
            lib.orc_dense_attn.argtypes = [P, i32, i32, i32, P, P, P, i32, i32, P, P, P,
                                           ctypes.c_double, P, P, i32]
            _lib = lib
    return _lib


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


class Batch:
    """Holds contiguous copies of the batch geometry and the ctypes struct."""

    def __init__(self, cu_seqlens_q, cu_seqlens_k, context_lens, block_table, num_pages):
        self.cu_q = _c(cu_seqlens_q, np.int32)
        self.cu_k = _c(cu_seqlens_k, np.int32)
        self.ctx = _c(context_lens, np.int32)
        self.bt = _c(block_table, np.int32)
        if self.bt.ndim != 2:
            raise ValueError("block_table must be 2-D")
        self.num_reqs = int(self.ctx.shape[0])
        self.num_rows = int(self.cu_q[-1]) if self.cu_q.size else 0
        self.s = _Batch(self.num_reqs, self.num_rows, _ptr(self.cu_q), _ptr(self.cu_k),
                        _ptr(self.ctx), _ptr(self.bt), int(self.bt.shape[1]), int(num_pages))

    @classmethod
    def of(cls, w, num_rows: Optional[int] = None):
        b = cls(w.cu_seqlens_q, w.cu_seqlens_k, w.context_lens, w.block_table, w.num_pages)
        if num_rows is not None:
            b.num_rows = int(num_rows)
            b.s.num_rows = int(num_rows)
        return b


def fp8_e4m3_value(code: int) -> float:
    return _load().orc_fp8_e4m3_value(int(code))


def bf16_value(bits: int) -> float:
    return _load().orc_bf16_value(int(bits))


def row_geometry(batch: Batch):
    n = max(batch.num_rows, 1)
    req, pos, nb, ok = (np.zeros(n, np.int32) for _ in range(4))
    st = _load().orc_row_geometry(ctypes.byref(batch.s), _ptr(req), _ptr(pos), _ptr(nb), _ptr(ok))
    k = batch.num_rows
    return dict(req=req[:k], pos=pos[:k], nb=nb[:k], ok=ok[:k], status=int(st))


def index_score(batch: Batch, idx_q, idx_k, score_stride: Optional[int] = None,
                nthreads: Optional[int] = None, *, fp8: bool = False, k_scale=None):
    """Block scores; idx_k holds bf16 bits, or e4m3 codes when fp8 (with
    optional per-token scales k_scale [P,128,Hi])."""
    idx_q = _c(idx_q, np.uint16)
    hi, di = int(idx_q.shape[1]), int(idx_q.shape[2])
    stride = int(score_stride or batch.s.bt_stride)
    scores = np.empty((max(batch.num_rows, 1), stride), np.float32)
    n = nthreads or default_threads()
    if fp8:
        idx_k = _c(idx_k, np.uint8)
        ks = None if k_scale is None else _c(k_scale, np.float32)
        st = _load().orc_index_score_fp8(ctypes.byref(batch.s), _ptr(idx_q), _ptr(idx_k),
                                         _ptr(ks), hi, di, _ptr(scores), stride, n)
    else:
        idx_k = _c(idx_k, np.uint16)
        st = _load().orc_index_score(ctypes.byref(batch.s), _ptr(idx_q), _ptr(idx_k), hi, di,
                                     _ptr(scores), stride, n)
    return scores[: batch.num_rows], int(st)


def topk_build_table(batch: Batch, scores, topk: int, tbl_stride: Optional[int] = None,
                     nthreads: Optional[int] = None):
    scores = _c(scores, np.float32)
    stride = int(tbl_stride or 8 * topk)
    n = max(batch.num_rows, 1)
    topk_idx = np.empty((n, topk), np.int32)
    tbl = np.empty((n, stride), np.int32)
    slen = np.empty(n, np.int32)
    st = _load().orc_topk_build_table(ctypes.byref(batch.s), _ptr(scores), int(scores.shape[1]),
                                      int(topk), _ptr(topk_idx), _ptr(tbl), stride, _ptr(slen),
                                      nthreads or default_threads())
    k = batch.num_rows
    return topk_idx[:k], tbl[:k], slen[:k], int(st)


def sparse_attn(q, k_cache, v_cache, kv_dtype: int, sparse_tbl, sparse_len, *, scale_mode=0,
                k_scale=None, v_scale=None, sinks=None, softmax_scale: float,
                num_pages16: Optional[int] = None, nthreads: Optional[int] = None):
    q = _c(q, np.uint16)
    kdt = np.uint8 if kv_dtype == 1 else np.uint16
    k_cache = _c(k_cache, kdt)
    v_cache = _c(v_cache, kdt)
    tbl = _c(sparse_tbl, np.int32)
    slen = _c(sparse_len, np.int32)
    N, hq, d = (int(x) for x in q.shape)
    hkv = int(k_cache.shape[-2])
    if num_pages16 is None:
        num_pages16 = int(k_cache.size // (16 * hkv * d))
    out = np.empty((max(N, 1), hq, d), np.float64)
    lse = np.empty((max(N, 1), hq), np.float64)
    st = _load().orc_sparse_attn(N, hq, hkv, d, _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                 int(kv_dtype), int(num_pages16), int(scale_mode),
                                 _ptr(_c(k_scale, np.float32)), _ptr(_c(v_scale, np.float32)),
                                 _ptr(tbl), int(tbl.shape[1]), _ptr(slen),
                                 _ptr(_c(sinks, np.float32)), float(softmax_scale), _ptr(out),
                                 _ptr(lse), nthreads or default_threads())
    return out[:N], lse[:N], int(st)


def dense_attn(batch: Batch, q, k_cache, v_cache, kv_dtype: int, *, scale_mode=0, k_scale=None,
               v_scale=None, sinks=None, softmax_scale: float, nthreads: Optional[int] = None):
    q = _c(q, np.uint16)
    kdt = np.uint8 if kv_dtype == 1 else np.uint16
    k_cache = _c(k_cache, kdt)
    v_cache = _c(v_cache, kdt)
    N, hq, d = (int(x) for x in q.shape)
    hkv = int(k_cache.shape[-2])
    out = np.empty((max(N, 1), hq, d), np.float64)
    lse = np.empty((max(N, 1), hq), np.float64)
    st = _load().orc_dense_attn(ctypes.byref(batch.s), hq, hkv, d, _ptr(q), _ptr(k_cache),
                                _ptr(v_cache), int(kv_dtype), int(scale_mode),
                                _ptr(_c(k_scale, np.float32)), _ptr(_c(v_scale, np.float32)),
                                _ptr(_c(sinks, np.float32)), float(softmax_scale), _ptr(out),
                                _ptr(lse), nthreads or default_threads())
    return out[:N], lse[:N], int(st)


def decode(w, nthreads: Optional[int] = None, topk: Optional[int] = None):
    """The whole path on a workload: scores -> top-k/table -> sparse attention."""
    b = Batch.of(w)
    k = int(topk or w.topk)
    scores, st1 = index_score(b, w.idx_q, w.idx_k, nthreads=nthreads,
                              fp8=w.index_dtype == 1, k_scale=w.idx_k_scale)
    topk_idx, tbl, slen, st2 = topk_build_table(b, scores, k, nthreads=nthreads)
    out, lse, st3 = sparse_attn(w.q, w.k_cache, w.v_cache, w.kv_dtype, tbl, slen,
                                scale_mode=w.scale_mode, k_scale=w.k_scale, v_scale=w.v_scale,
                                sinks=w.sinks, softmax_scale=w.softmax_scale,
                                num_pages16=8 * w.num_pages, nthreads=nthreads)
    return dict(scores=scores, topk_idx=topk_idx, tbl=tbl, sparse_len=slen, out=out, lse=lse,
                status=st1 | st2 | st3)


def dense(w, nthreads: Optional[int] = None):
    b = Batch.of(w)
    return dense_attn(b, w.q, w.k_cache, w.v_cache, w.kv_dtype, scale_mode=w.scale_mode,
                      k_scale=w.k_scale, v_scale=w.v_scale, sinks=w.sinks,
                      softmax_scale=w.softmax_scale, nthreads=nthreads)


def fp8_e4m3_encode(x: float) -> int:
    return int(_load().orc_fp8_e4m3_encode(float(x)))


def kv_insert(w, k_new, v_new, idx_new, skip_index: bool = False):
    """Insert the rows' new K/V/index-K into copies of the workload's pools;
    returns (k_cache, v_cache, idx_k, k_scale, v_scale, status), plus the
    index scales as a 7th item when the index cache is FP8."""
    b = Batch.of(w)
    kdt = np.uint8 if w.kv_dtype == 1 else np.uint16
    k_cache = np.array(w.k_cache, dtype=kdt, copy=True)
    v_cache = np.array(w.v_cache, dtype=kdt, copy=True)
    idt = np.uint8 if w.index_dtype == 1 else np.uint16
    idx_k = np.array(w.idx_k, dtype=idt, copy=True)
    idx_scale = None if w.idx_k_scale is None else np.array(w.idx_k_scale, np.float32, copy=True)
    k_scale = None if w.k_scale is None else np.array(w.k_scale, np.float32, copy=True)
    v_scale = None if w.v_scale is None else np.array(w.v_scale, np.float32, copy=True)
    k_new = _c(k_new, np.uint16)
    v_new = _c(v_new, np.uint16)
    idx_new = _c(idx_new, np.uint16)
    st = _load().orc_kv_insert(ctypes.byref(b.s), int(w.hkv), int(w.head_dim), _ptr(k_new),
                               _ptr(v_new), int(w.index_heads), int(w.index_dim), _ptr(idx_new),
                               _ptr(k_cache), _ptr(v_cache), _ptr(idx_k), int(w.kv_dtype),
                               int(w.scale_mode), _ptr(k_scale), _ptr(v_scale),
                               int(bool(skip_index)), int(w.index_dtype), _ptr(idx_scale))
    if w.index_dtype == 1:
        return k_cache, v_cache, idx_k, k_scale, v_scale, int(st), idx_scale
    return k_cache, v_cache, idx_k, k_scale, v_scale, int(st)


def sparse_mla(q, kv_cache, kv_indptr, kv_indices, dv: int, *, sinks=None,
               softmax_scale: float, nthreads: Optional[int] = None, q_scale=None,
               kv_scale=None):
    """Sparse MLA decode: q [N, H, Dqk] bf16 bits (or e4m3 codes, uint8, with
    q_scale), kv_cache [T, Dqk] bf16 bits (or e4m3 codes, uint8, with
    kv_scale; value = first dv columns), per-row token ids through kv_indptr
    [N+1] / kv_indices; returns (out [N, H, dv] fp64, lse [N, H] fp64, status)."""
    q = np.ascontiguousarray(q)
    kv = np.ascontiguousarray(kv_cache)
    q_fp8 = q.dtype == np.uint8
    kv_fp8 = kv.dtype == np.uint8
    q = _c(q, np.uint8 if q_fp8 else np.uint16)
    kv = _c(kv, np.uint8 if kv_fp8 else np.uint16)
    ip = _c(kv_indptr, np.int32)
    ix = _c(kv_indices if len(kv_indices) else np.zeros(1, np.int32), np.int32)
    N, H, dqk = (int(x) for x in q.shape)
    out = np.empty((max(N, 1), H, dv), np.float64)
    lse = np.empty((max(N, 1), H), np.float64)
    sk = None if sinks is None else _c(sinks, np.float32)
    qs = 1.0 if q_scale is None else float(np.asarray(q_scale, np.float32).reshape(-1)[0])
    ks = 1.0 if kv_scale is None else float(np.asarray(kv_scale, np.float32).reshape(-1)[0])
    st = _load().orc_sparse_mla_ex(N, H, dqk, int(dv), _ptr(q), int(q_fp8), qs, _ptr(kv),
                                   int(kv_fp8), ks, int(kv.shape[0]), _ptr(ip), _ptr(ix), _ptr(sk),
                                   float(softmax_scale), _ptr(out), _ptr(lse),
                                   nthreads or default_threads())
    return out[:N], lse[:N], int(st)
