"""block_sparse_paged_02_gb300 -- block-sparse paged decode (MiniMax-M3-style
index top-k + sparse paged attention) for one GB300 (sm_103a).

The compute runs in libmsa.so (CUDA kernels behind the C ABI of
include/msa.h); this package builds it and marshals torch tensors into it.
"""
from .binding import (MSA_DEV_BAD_LEN, MSA_DEV_BAD_PAGE, MSA_DEV_BAD_TABLE, MSA_DEV_MALFORMED,
                      MSA_DEV_TIMEOUT, MSA_KV_BF16, MSA_KV_FP8_E4M3, MSA_SCALE_NONE,
                      MSA_SCALE_PER_TOKEN_HEAD, MSA_SCALE_SCALAR, MsaError, lib, make_attn_args,
                      make_batch, make_index_cache, make_trace, msa_decode, msa_index_score, msa_kv_insert,
                      msa_sparse_paged_attn, msa_status_string, msa_topk_build_table,
                      msa_workspace_size)
from .binding import make_mla_args, msa_sparse_mla_decode, msa_sparse_mla_workspace_size
from .binding import MSA_CHECK_WAIT_COPY, MSA_CHECK_WAIT_TMEM, msa_check_bounded_wait
from .case import DeviceCase, MlaCase

__all__ = [
    "lib", "make_batch", "make_attn_args", "make_index_cache", "make_trace", "msa_index_score",
    "msa_topk_build_table", "msa_sparse_paged_attn", "msa_decode", "msa_kv_insert",
    "msa_workspace_size",
    "msa_status_string", "MsaError", "DeviceCase", "MlaCase", "make_mla_args",
    "msa_sparse_mla_decode", "msa_sparse_mla_workspace_size", "MSA_KV_BF16", "MSA_KV_FP8_E4M3",
    "MSA_SCALE_NONE", "MSA_SCALE_SCALAR", "MSA_SCALE_PER_TOKEN_HEAD", "MSA_DEV_BAD_PAGE",
    "MSA_DEV_BAD_LEN", "MSA_DEV_MALFORMED", "MSA_DEV_BAD_TABLE", "MSA_DEV_TIMEOUT",
    "msa_check_bounded_wait", "MSA_CHECK_WAIT_TMEM", "MSA_CHECK_WAIT_COPY",
]
