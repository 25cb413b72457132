"""Seeded synthetic inputs for the block-sparse paged decode path.

This module only draws random numbers and lays them out in the cache
formats the path reads; it holds none of the method's arithmetic (no
scoring, selection, table expansion or attention).  Both the CPU oracle
tests and the CUDA path take their inputs from here.

Formats (all host numpy arrays, little-endian):
  * bf16 tensors are ``uint16`` arrays of bf16 bit patterns;
  * fp8 tensors are ``uint8`` arrays of OCP e4m3fn codes (encoded with
    torch's round-to-nearest-even cast after clamping to +-448);
  * ``idx_k`` is the paged index-K cache ``[P, 128, Hi, Di]``;
  * ``k_cache`` / ``v_cache`` are ``[P, 128, Hkv, D]``; the page-16 view
    ``[8P, 16, Hkv, D]`` is the same bytes;
  * per-token-head scales are fp32 ``[P, 128, Hkv]``; scalar scales are
    fp32 ``[1]``.

The five named workloads follow the problem statement of the MiniMax-M3
sparse-attention pages (vLLM PR 47287 "AITER sparse paged attention",
PR 54682 "gfx950 decode index + top-k", PR 54404 "sparse MLA sinks + LSE",
PR 56170 "cu_seqlens_k device zeroing"): one KV head, head_dim 128, one
index head, 128-token blocks, page-16 attention view.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np
import torch

BLOCK = 128  # tokens per index block == tokens per KV page
PAGE16 = 16  # tokens per page of the attention view

KV_BF16 = 0
KV_FP8 = 1
SCALE_NONE = 0
SCALE_SCALAR = 1
SCALE_PER_TOKEN_HEAD = 2


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """float array -> bf16 bit patterns (round to nearest even, via torch)."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()


def _int_bf16(x: np.ndarray) -> np.ndarray:
    """small integers (int8) -> their (exact) bf16 bit patterns"""
    t = torch.from_numpy(np.ascontiguousarray(x)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def fp8_codes(x: np.ndarray) -> np.ndarray:
    """float array -> OCP e4m3fn codes (saturating RNE, via torch)."""
    x = np.clip(np.asarray(x, dtype=np.float32), -448.0, 448.0)
    t = torch.from_numpy(np.ascontiguousarray(x))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy().copy()


@dataclasses.dataclass
class Workload:
    name: str
    # batch geometry
    cu_seqlens_q: np.ndarray  # int32 [R+1]
    cu_seqlens_k: np.ndarray  # int32 [R+1], [0] == 0
    context_lens: np.ndarray  # int32 [R]
    block_table: np.ndarray   # int32 [R, bt_stride]; unused entries -1
    num_pages: int            # P (page-128 pages in the pool)
    # index path
    idx_q: np.ndarray         # bf16 bits [N, Hi, Di]
    idx_k: np.ndarray         # bf16 bits [P, 128, Hi, Di]
    topk: int
    # attention path
    q: np.ndarray             # bf16 bits [N, Hq, D]
    k_cache: np.ndarray       # [P, 128, Hkv, D] (uint16 bf16 bits or uint8 fp8)
    v_cache: np.ndarray
    kv_dtype: int
    scale_mode: int
    k_scale: Optional[np.ndarray]  # fp32 [1] or [P,128,Hkv]
    v_scale: Optional[np.ndarray]
    sinks: Optional[np.ndarray]    # fp32 [Hq]
    softmax_scale: float
    seed: int = 0
    # index-K cache format: KV_BF16 (idx_k holds bf16 bits) or KV_FP8 (idx_k
    # holds OCP e4m3 codes, idx_k_scale optional fp32 [P, 128, Hi])
    index_dtype: int = 0
    idx_k_scale: Optional[np.ndarray] = None

    @property
    def num_reqs(self) -> int:
        return int(self.context_lens.shape[0])

    @property
    def num_rows(self) -> int:
        return int(self.q.shape[0])

    @property
    def hq(self) -> int:
        return int(self.q.shape[1])

    @property
    def hkv(self) -> int:
        return int(self.k_cache.shape[2])

    @property
    def head_dim(self) -> int:
        return int(self.q.shape[2])

    @property
    def index_heads(self) -> int:
        return int(self.idx_q.shape[1])

    @property
    def index_dim(self) -> int:
        return int(self.idx_q.shape[2])

    @property
    def bt_stride(self) -> int:
        return int(self.block_table.shape[1])

    @property
    def seq_lens(self) -> np.ndarray:
        return np.diff(self.cu_seqlens_k).astype(np.int64)

    @property
    def q_lens(self) -> np.ndarray:
        return np.diff(self.cu_seqlens_q).astype(np.int64)

    @property
    def tbl_stride(self) -> int:
        return 8 * self.topk


def _build(name: str, seed: int, rng: np.random.Generator, *, q_lens, seq_lens,
           hq: int, di: int, idx_range: int, topk: int, kv_dtype: int,
           scale_mode: int, with_sink: bool, pool_pages: Optional[int] = None,
           pool_factor: float = 1.25, hkv: int = 1, hi: int = 1, d: int = 128,
           fill_unused_nan: bool = False) -> Workload:
    q_lens = np.asarray(q_lens, dtype=np.int64)
    seq_lens = np.asarray(seq_lens, dtype=np.int64)
    R = len(seq_lens)
    assert np.all(seq_lens >= q_lens)
    nb = (seq_lens + BLOCK - 1) // BLOCK
    total_pages = int(nb.sum())
    P = int(pool_pages) if pool_pages is not None else max(
        total_pages, int(math.ceil(total_pages * pool_factor)))
    assert P >= total_pages
    bt_stride = max(1, int(nb.max()) if R else 1)
    perm = rng.permutation(P).astype(np.int32)
    block_table = np.full((R, bt_stride), -1, dtype=np.int32)
    off = 0
    for r in range(R):
        block_table[r, : nb[r]] = perm[off: off + nb[r]]
        off += nb[r]
    cu_q = np.zeros(R + 1, dtype=np.int32)
    cu_q[1:] = np.cumsum(q_lens)
    cu_k = np.zeros(R + 1, dtype=np.int32)
    cu_k[1:] = np.cumsum(seq_lens)
    context = (seq_lens - q_lens).astype(np.int32)
    N = int(cu_q[-1])

    # integer-valued index vectors, uniform in {-idx_range..idx_range}
    idx_q = _int_bf16(rng.integers(-idx_range, idx_range + 1, size=(N, hi, di), dtype=np.int8))
    idx_k = _int_bf16(rng.integers(-idx_range, idx_range + 1, size=(P, BLOCK, hi, di),
                                   dtype=np.int8))
    # N(0,1) activations: torch's seeded CPU generator (much faster than numpy's)
    tg = torch.Generator().manual_seed(int(seed) * 7919 + 17)
    q = torch.empty((N, hq, d)).normal_(generator=tg).to(torch.bfloat16).view(torch.int16)
    q = q.numpy().view(np.uint16)
    caches = []
    for _ in range(2):
        x = torch.empty((P, BLOCK, hkv, d)).normal_(generator=tg)
        if kv_dtype == KV_FP8:
            caches.append(x.clamp_(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8).numpy())
        else:
            caches.append(x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16))
        del x
    k_cache, v_cache = caches
    if fill_unused_nan:
        # slots past each request's last token hold garbage the path must never use
        nan_bf16 = np.uint16(0x7FC0)
        nan_fp8 = np.uint8(0x7F)
        for r in range(R):
            if nb[r] == 0:
                continue
            last = block_table[r, nb[r] - 1]
            tail = int(seq_lens[r] - (nb[r] - 1) * BLOCK)
            idx_k[last, tail:] = nan_bf16
            fill = nan_fp8 if kv_dtype == KV_FP8 else nan_bf16
            k_cache[last, tail:] = fill
            v_cache[last, tail:] = fill
        used = np.zeros(P, dtype=bool)
        used[block_table[block_table >= 0]] = True
        idx_k[~used] = nan_bf16

    k_scale = v_scale = None
    if scale_mode == SCALE_SCALAR:
        k_scale = np.array([rng.lognormal(0.0, 0.5)], dtype=np.float32)
        v_scale = np.array([rng.lognormal(0.0, 0.5)], dtype=np.float32)
    elif scale_mode == SCALE_PER_TOKEN_HEAD:
        k_scale = rng.lognormal(0.0, 0.5, size=(P, BLOCK, hkv)).astype(np.float32)
        v_scale = rng.lognormal(0.0, 0.5, size=(P, BLOCK, hkv)).astype(np.float32)
    sinks = rng.standard_normal(hq).astype(np.float32) if with_sink else None
    return Workload(name=name, cu_seqlens_q=cu_q, cu_seqlens_k=cu_k, context_lens=context,
                    block_table=block_table, num_pages=P, idx_q=idx_q, idx_k=idx_k, topk=topk,
                    q=q, k_cache=k_cache, v_cache=v_cache, kv_dtype=kv_dtype,
                    scale_mode=scale_mode, k_scale=k_scale, v_scale=v_scale, sinks=sinks,
                    softmax_scale=float(np.float32(1.0 / math.sqrt(d))), seed=seed)


# --- the five named workloads -------------------------------------------------

def tiny(seed: int = 1) -> Workload:
    """1 request x 1 row, 8 heads / 1 KV head, Di 64 ints in {-2..2},
    context 1000 tokens in 8 shuffled pages (last one partial), top-k 4, bf16."""
    rng = np.random.default_rng(seed)
    return _build("tiny_decode", seed, rng, q_lens=[1], seq_lens=[1000], hq=8, di=64,
                  idx_range=2, topk=4, kv_dtype=KV_BF16, scale_mode=SCALE_NONE,
                  with_sink=False, pool_pages=8)


def batched(seed: int = 2) -> Workload:
    """8 requests x 1 row, 16/1 heads, Di 128 ints in {-3..3}, contexts U[8K,32K],
    top-k 16, bf16 K/V, 4096-page pool, no sink."""
    rng = np.random.default_rng(seed)
    lens = rng.integers(8192, 32768 + 1, size=8)
    return _build("batched_decode", seed, rng, q_lens=[1] * 8, seq_lens=lens, hq=16, di=128,
                  idx_range=3, topk=16, kv_dtype=KV_BF16, scale_mode=SCALE_NONE,
                  with_sink=False, pool_pages=4096)


def speculative(seed: int = 3) -> Workload:
    """4 requests x 4 speculative rows (row i at position L-4+i), contexts U[64K,128K],
    top-k 32, FP8 K/V with per-token-head scales lognormal(0,0.5), sinks N(0,1)."""
    rng = np.random.default_rng(seed)
    lens = rng.integers(65536, 131072 + 1, size=4)
    return _build("speculative_decode", seed, rng, q_lens=[4] * 4, seq_lens=lens, hq=16,
                  di=128, idx_range=3, topk=32, kv_dtype=KV_FP8,
                  scale_mode=SCALE_PER_TOKEN_HEAD, with_sink=True)


def large_batch_lengths(rng: np.random.Generator, n: int = 64) -> np.ndarray:
    """Context lengths lognormal around a 16384 median (sigma 1.0 on ln L),
    clipped to [512, 131072] and rounded to integers."""
    lens = np.exp(rng.normal(math.log(16384.0), 1.0, size=n))
    return np.clip(np.rint(lens), 512, 131072).astype(np.int64)


def large_batch(seed: int = 4) -> Workload:
    """64 requests x 1 row, lognormal contexts (median 16K), top-k 16, FP8 K/V with
    scalar k/v scales (one lognormal(0,0.5) draw each), sinks N(0,1)."""
    rng = np.random.default_rng(seed)
    lens = large_batch_lengths(rng, 64)
    return _build("large_batch_decode", seed, rng, q_lens=[1] * 64, seq_lens=lens, hq=16,
                  di=128, idx_range=3, topk=16, kv_dtype=KV_FP8, scale_mode=SCALE_SCALAR,
                  with_sink=True)


def chunked_prefill(seed: int = 5, context: int = 30720, new_tokens: int = 2048,
                    reqs: int = 2) -> Workload:
    """2 requests, each appending 2048 query tokens to a 30720-token cached context
    (seq_len 32768), per-token causal top-k 16, bf16 Q/K/V, no sink."""
    rng = np.random.default_rng(seed)
    return _build("chunked_prefill", seed, rng, q_lens=[new_tokens] * reqs,
                  seq_lens=[context + new_tokens] * reqs, hq=16, di=128, idx_range=3,
                  topk=16, kv_dtype=KV_BF16, scale_mode=SCALE_NONE, with_sink=False)


def custom(seed: int, q_lens, seq_lens, *, hq=16, di=128, idx_range=3, topk=16,
           kv_dtype=KV_BF16, scale_mode=SCALE_NONE, with_sink=False, hi=1,
           pool_pages=None, fill_unused_nan=False, name="custom") -> Workload:
    """A smaller workload with the same recipe (used for edge cases and quick parity)."""
    rng = np.random.default_rng(seed)
    return _build(name, seed, rng, q_lens=q_lens, seq_lens=seq_lens, hq=hq, di=di,
                  idx_range=idx_range, topk=topk, kv_dtype=kv_dtype, scale_mode=scale_mode,
                  with_sink=with_sink, hi=hi, pool_pages=pool_pages,
                  fill_unused_nan=fill_unused_nan)


def row_subset(w: Workload, rows) -> Workload:
    """A batch holding only the given rows, each as its own one-row request at
    the same position over the same pages and caches.  A row's result depends
    only on its own position, query and its request's pages, so the oracle on
    this batch reproduces those rows of the full batch."""
    req_of = np.searchsorted(w.cu_seqlens_q, np.arange(w.num_rows), side="right") - 1
    rows = np.asarray(rows)
    pos = np.array([w.context_lens[req_of[r]] + (r - w.cu_seqlens_q[req_of[r]]) for r in rows])
    seq = pos + 1
    n = len(rows)
    cu = np.arange(n + 1, dtype=np.int32)
    cu_k = np.concatenate([[0], np.cumsum(seq)]).astype(np.int32)
    return Workload(name=w.name + "_rows", cu_seqlens_q=cu, cu_seqlens_k=cu_k,
                    context_lens=pos.astype(np.int32),
                    block_table=w.block_table[req_of[rows]].copy(), num_pages=w.num_pages,
                    idx_q=w.idx_q[rows], idx_k=w.idx_k, topk=w.topk, q=w.q[rows],
                    k_cache=w.k_cache, v_cache=w.v_cache, kv_dtype=w.kv_dtype,
                    scale_mode=w.scale_mode, k_scale=w.k_scale, v_scale=w.v_scale,
                    sinks=w.sinks, softmax_scale=w.softmax_scale, seed=w.seed,
                    index_dtype=w.index_dtype, idx_k_scale=w.idx_k_scale)


def fp8_index(w: Workload, seed: int, scaled: bool = True) -> Workload:
    """The same workload with its index-K cache stored as OCP e4m3 codes (the
    integer index values are exact in e4m3; NaN fill stays NaN) and, when
    scaled, per-token scales drawn from {1/2, 1, 2} (powers of two keep every
    score exact)."""
    rng = np.random.default_rng(seed)
    vals = (np.asarray(w.idx_k, np.uint16).astype(np.uint32) << 16).view(np.float32)
    codes = fp8_codes(vals)
    scale = None
    if scaled:
        shape = (w.num_pages, BLOCK, w.index_heads)
        scale = rng.choice(np.array([0.5, 1.0, 2.0], np.float32), size=shape).astype(np.float32)
    return dataclasses.replace(w, name=w.name + "_fp8_index", idx_k=codes, index_dtype=KV_FP8,
                               idx_k_scale=scale)


def large_batch_fp8_index(seed: int = 6) -> Workload:
    """The 64-request decode recipe with an FP8 (e4m3, per-token scaled)
    index-K cache."""
    return fp8_index(large_batch(seed), seed + 100)


NAMED = {
    "tiny_decode": tiny,
    "batched_decode": batched,
    "speculative_decode": speculative,
    "large_batch_decode": large_batch,
    "chunked_prefill": chunked_prefill,
    "large_batch_decode_fp8_index": large_batch_fp8_index,
}


# ------------------------------------------------------------ sparse MLA decode

@dataclasses.dataclass
class MlaWorkload:
    """Sparse MLA decode inputs: one latent KV head, one row of dqk values per
    cached token (the first dv of them are the value), and per query row the
    list of selected token ids (kv_indptr / kv_indices)."""
    name: str
    q: np.ndarray            # bf16 bits [N, H, dqk]
    kv_cache: np.ndarray     # bf16 bits [T, dqk]
    kv_indptr: np.ndarray    # int32 [N + 1]
    kv_indices: np.ndarray   # int32 [nnz] token ids (< 0 or >= T marks a bad row)
    dv: int
    sinks: Optional[np.ndarray]  # fp32 [H]
    softmax_scale: float
    seed: int = 0
    # FP8 operands: q / kv_cache hold OCP e4m3 codes (uint8) and the element
    # is scale * code; None for bf16 operands
    q_scale: Optional[np.ndarray] = None   # fp32 [1]
    kv_scale: Optional[np.ndarray] = None  # fp32 [1]

    @property
    def num_rows(self) -> int:
        return int(self.q.shape[0])

    @property
    def heads(self) -> int:
        return int(self.q.shape[1])

    @property
    def dqk(self) -> int:
        return int(self.q.shape[2])

    @property
    def num_tokens(self) -> int:
        return int(self.kv_cache.shape[0])


def sparse_mla_custom(seed: int, counts, *, heads=16, ctx=4096, dqk=576, dv=512,
                      with_sink=True, duplicates=False, name="sparse_mla_custom") -> MlaWorkload:
    """Row r selects counts[r] token ids from its own context of ctx tokens
    (ascending and distinct unless duplicates); q and the latent cache are
    N(0,1) in bf16; the scale is 1/sqrt(192) (a 128 + 64 query-key head)."""
    rng = np.random.default_rng(seed)
    N = len(counts)
    T = max(1, N * ctx)
    tg = torch.Generator().manual_seed(int(seed) * 7919 + 29)
    q = torch.empty((N, heads, dqk)).normal_(generator=tg).to(torch.bfloat16)
    kv = torch.empty((T, dqk)).normal_(generator=tg).to(torch.bfloat16)
    idx = []
    for r, n in enumerate(counts):
        if duplicates:
            sel = rng.integers(0, ctx, size=n)
        else:
            sel = np.sort(rng.choice(ctx, size=min(n, ctx), replace=False))
        idx.append((r * ctx + sel).astype(np.int32))
    indptr = np.concatenate([[0], np.cumsum([len(x) for x in idx])]).astype(np.int32)
    indices = np.concatenate(idx).astype(np.int32) if idx else np.zeros(0, np.int32)
    sinks = rng.standard_normal(heads).astype(np.float32) if with_sink else None
    return MlaWorkload(name=name, q=q.view(torch.int16).numpy().view(np.uint16).copy(),
                       kv_cache=kv.view(torch.int16).numpy().view(np.uint16).copy(),
                       kv_indptr=indptr, kv_indices=indices, dv=dv, sinks=sinks,
                       softmax_scale=float(np.float32(1.0 / np.sqrt(192.0))), seed=seed)


def sparse_mla_decode(seed: int = 7) -> MlaWorkload:
    """64 decode rows, 16 heads, 2048 selected tokens each out of an 8192-token
    context per row: the sparse-MLA decode recipe."""
    return sparse_mla_custom(seed, [2048] * 64, heads=16, ctx=8192, name="sparse_mla_decode")


def mla_fp8(w: MlaWorkload, seed: int, fp8_q: bool = True) -> MlaWorkload:
    """The same recipe with an FP8 latent cache (and query, if fp8_q): the
    N(0,1) values encoded as e4m3 (RNE, saturating) with unit scale, then one
    scale per tensor drawn from lognormal(0, 0.5) -- the element is scale *
    code, as in the decode op's q_scale / kv_scale."""
    rng = np.random.default_rng(seed)
    as_f32 = lambda bits: (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)
    kv = fp8_codes(as_f32(w.kv_cache))
    kv_scale = np.array([rng.lognormal(0.0, 0.5)], np.float32)
    q, q_scale = w.q, None
    if fp8_q:
        q = fp8_codes(as_f32(w.q))
        q_scale = np.array([rng.lognormal(0.0, 0.5)], np.float32)
    return dataclasses.replace(w, name=w.name + "_fp8", q=q, kv_cache=kv, q_scale=q_scale,
                               kv_scale=kv_scale)


def sparse_mla_decode_fp8(seed: int = 8) -> MlaWorkload:
    """The sparse-MLA decode recipe with e4m3 query and latent cache, scalar
    q_scale / kv_scale."""
    return mla_fp8(sparse_mla_decode(seed), seed + 100)

