"""Device-resident copy of one batch (host arrays -> torch CUDA tensors) with
the output buffers and workspace the C ABI needs.  Marshalling only."""
from __future__ import annotations

from typing import Optional

import numpy as np
import torch

from . import binding as B


def _dev(a: np.ndarray, device, dtype=None) -> torch.Tensor:
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:  # bf16 bit patterns
        t = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(a)
    if dtype is not None:
        t = t.to(dtype)
    return t.to(device)


class DeviceCase:
    """Inputs of one decode call resident on the GPU, plus outputs.

    `w` is any object with the fields of `workloads.Workload` (host numpy
    arrays).  The KV and index-K pools stay resident; after
    `pack_step_inputs()` what changes per step (queries and batch geometry)
    sits in one device buffer, `step_inputs`, that one copy refreshes, and
    O / LSE in another, `step_outputs`.  The batch carries the request
    length bounds as host hints (max_q_len, and min_q_len unless
    `min_q_len_hint` is False; an int overrides it)."""

    def __init__(self, w, device: str = "cuda", topk: Optional[int] = None,
                 tbl_stride: Optional[int] = None, min_q_len_hint=True):
        self.w = w
        self.device = device
        self.topk = int(topk or w.topk)
        self.tbl_stride = int(tbl_stride or 8 * self.topk)
        self.cu_q = _dev(w.cu_seqlens_q, device)
        self.cu_k = _dev(w.cu_seqlens_k, device)
        self.ctx = _dev(w.context_lens, device)
        self.bt = _dev(w.block_table, device)
        self.idx_q = _dev(w.idx_q, device)
        self.idx_k = _dev(w.idx_k, device)
        idx_scale = getattr(w, "idx_k_scale", None)
        self.idx_k_scale = None if idx_scale is None else _dev(idx_scale, device)
        self.index = B.make_index_cache(self.idx_k, getattr(w, "index_dtype", B.MSA_KV_BF16),
                                        self.idx_k_scale)
        self.q = _dev(w.q, device)
        self.k = _dev(w.k_cache, device)
        self.v = _dev(w.v_cache, device)
        self.k_scale = None if w.k_scale is None else _dev(w.k_scale, device)
        self.v_scale = None if w.v_scale is None else _dev(w.v_scale, device)
        self.sinks = None if w.sinks is None else _dev(w.sinks, device)
        N, hq, d = (int(x) for x in w.q.shape)
        self.num_rows = N
        self.out = torch.empty((N, hq, d), dtype=torch.bfloat16, device=device)
        self.lse = torch.empty((N, hq), dtype=torch.float32, device=device)
        self.scores = torch.empty((max(N, 1), w.bt_stride), dtype=torch.float32, device=device)
        self.topk_idx = torch.empty((max(N, 1), self.topk), dtype=torch.int32, device=device)
        self.tbl = torch.empty((max(N, 1), self.tbl_stride), dtype=torch.int32, device=device)
        self.sparse_len = torch.empty((max(N, 1),), dtype=torch.int32, device=device)
        self.status = torch.zeros((1,), dtype=torch.int32, device=device)
        q_lens = np.diff(np.asarray(w.cu_seqlens_q, np.int64))
        self.max_q_len = int(q_lens.max()) if q_lens.size else 0
        if min_q_len_hint is True:
            self.min_q_len = int(q_lens.min()) if q_lens.size else 0
        else:
            self.min_q_len = int(min_q_len_hint or 0)
        ws = B.msa_workspace_size(N, w.bt_stride, self.topk, hq, d, self.tbl_stride)
        self.workspace = torch.zeros((ws,), dtype=torch.uint8, device=device)
        ws_a = B.msa_workspace_size(N, 0, 0, hq, d, self.tbl_stride)
        self.attn_workspace = torch.zeros((ws_a,), dtype=torch.uint8, device=device)
        self.step_inputs = None
        self.step_outputs = None
        self._args()

    def _args(self):
        w = self.w
        self.batch = B.make_batch(self.cu_q, self.cu_k, self.ctx, self.bt, w.num_pages,
                                  self.num_rows, max_q_len=self.max_q_len,
                                  min_q_len=self.min_q_len)
        self.attn = B.make_attn_args(self.q, self.k, self.v, w.kv_dtype, w.num_pages, self.out,
                                     self.lse, scale_mode=w.scale_mode, k_scale=self.k_scale,
                                     v_scale=self.v_scale, sinks=self.sinks,
                                     softmax_scale=w.softmax_scale)

    @staticmethod
    def _pack(tensors, device):
        """One byte buffer holding the tensors (256-byte aligned each) and
        views of it with their shapes and dtypes, contents copied."""
        offs, total = [], 0
        for t in tensors:
            offs.append(total)
            total += (t.numel() * t.element_size() + 255) // 256 * 256
        buf = torch.empty((max(total, 256),), dtype=torch.uint8, device=device)
        views = []
        for t, o in zip(tensors, offs):
            n = t.numel() * t.element_size()
            v = buf[o:o + n].view(t.dtype).view(t.shape)
            v.copy_(t)
            views.append(v)
        return buf, views

    _STEP_FIELDS = ("q", "idx_q", "cu_q", "cu_k", "ctx", "bt", "out", "lse", "batch", "attn",
                    "step_inputs", "step_outputs")

    def pack_step_inputs(self, sets: int = 1):
        """Move the per-step inputs into one device buffer and O / LSE into
        another (the argument structs are rebuilt on the new addresses).
        With sets > 1, that many independent buffer pairs with their own
        argument structs (same pools and workspace), for a pipeline that
        copies one step's inputs in while another step runs;
        `use_step_set(i)` selects set i (the first is selected)."""
        src_in = [self.q, self.idx_q, self.cu_q, self.cu_k, self.ctx, self.bt]
        src_out = [self.out, self.lse]
        self._sets = []
        for _ in range(sets):
            buf, (self.q, self.idx_q, self.cu_q, self.cu_k, self.ctx, self.bt) = self._pack(
                src_in, self.device)
            self.step_inputs = buf
            obuf, (self.out, self.lse) = self._pack(src_out, self.device)
            self.step_outputs = obuf
            self._args()
            self._sets.append({k: getattr(self, k) for k in self._STEP_FIELDS})
        self.use_step_set(0)

    def use_step_set(self, i: int):
        for k, v in self._sets[i].items():
            setattr(self, k, v)

    # -- the four entry points on this batch
    def index_score(self, stream=None):
        B.msa_index_score(self.batch, self.idx_q, self.index, self.scores, self.w.bt_stride,
                          self.status, stream)

    def topk_build_table(self, stream=None):
        B.msa_topk_build_table(self.batch, self.scores, self.w.bt_stride, self.topk,
                               self.topk_idx, self.tbl, self.tbl_stride, self.sparse_len,
                               self.status, stream)

    def sparse_paged_attn(self, stream=None):
        B.msa_sparse_paged_attn(self.attn, self.tbl, self.tbl_stride, self.sparse_len,
                                self.attn_workspace, self.status, stream)

    def decode(self, keep_tables: bool = True, trace=None, stream=None):
        B.msa_decode(self.batch, self.idx_q, self.index, self.topk, self.attn,
                     self.topk_idx if keep_tables else None,
                     self.tbl if keep_tables else None, self.tbl_stride,
                     self.sparse_len if keep_tables else None, self.workspace, self.status,
                     trace, stream)

    def kv_insert(self, k_new, v_new, idx_new, skip_index: bool = False, stream=None):
        """Write the rows' new K/V/index-K (device bf16 tensors) into the pools."""
        B.msa_kv_insert(self.batch, k_new, v_new, self.w.hkv, self.w.head_dim, self.k, self.v,
                        self.w.kv_dtype, self.w.scale_mode, self.k_scale, self.v_scale,
                        idx_new, self.index, skip_index, self.status, stream)

    def fetch(self):
        torch.cuda.synchronize()
        n = self.num_rows
        return dict(scores=self.scores[:n].cpu().numpy(), topk_idx=self.topk_idx[:n].cpu().numpy(),
                    tbl=self.tbl[:n].cpu().numpy(), sparse_len=self.sparse_len[:n].cpu().numpy(),
                    out=self.out.float().cpu().numpy().astype(np.float64),
                    lse=self.lse.cpu().numpy().astype(np.float64),
                    status=int(self.status.item()))


class MlaCase:
    """A sparse-MLA workload (`workloads.MlaWorkload` fields) resident on the
    GPU, with outputs and workspace."""

    def __init__(self, w, device: str = "cuda", max_tokens: Optional[int] = None):
        self.w = w
        counts = np.diff(np.asarray(w.kv_indptr, np.int64))
        self.max_tokens = int(max_tokens or max(1, int(counts.max()) if counts.size else 1))
        self.q = _dev(w.q, device)
        self.kv = _dev(w.kv_cache, device)
        self.indptr = _dev(w.kv_indptr, device)
        self.indices = _dev(w.kv_indices if len(w.kv_indices) else np.zeros(1, np.int32), device)
        self.sinks = None if w.sinks is None else _dev(w.sinks, device)
        q_scale = getattr(w, "q_scale", None)
        kv_scale = getattr(w, "kv_scale", None)
        self.q_scale = None if q_scale is None else _dev(q_scale, device)
        self.kv_scale = None if kv_scale is None else _dev(kv_scale, device)
        N, H = int(w.q.shape[0]), int(w.q.shape[1])
        self.out = torch.empty((max(N, 1), H, w.dv), dtype=torch.bfloat16, device=device)
        self.lse = torch.empty((max(N, 1), H), dtype=torch.float32, device=device)
        self.status = torch.zeros((1,), dtype=torch.int32, device=device)
        self.args = B.make_mla_args(self.q, self.kv, self.indptr, self.indices, self.out,
                                    self.lse, max_tokens=self.max_tokens, sinks=self.sinks,
                                    softmax_scale=w.softmax_scale, q_scale=self.q_scale,
                                    kv_scale=self.kv_scale)
        ws = B.msa_sparse_mla_workspace_size(N, H, self.max_tokens)
        self.workspace = torch.zeros((max(ws, 1),), dtype=torch.uint8, device=device)

    def decode(self, stream=None):
        B.msa_sparse_mla_decode(self.args, self.workspace, self.status, stream)

    def fetch(self):
        torch.cuda.synchronize()
        n = int(self.w.q.shape[0])
        return dict(out=self.out[:n].float().cpu().numpy().astype(np.float64),
                    lse=self.lse[:n].cpu().numpy().astype(np.float64),
                    status=int(self.status.item()))
