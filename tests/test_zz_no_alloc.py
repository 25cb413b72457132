"""msa_sparse_paged_attn_static: the attention entry point for callers that
cannot allocate device memory (its scratch lives in a static device array
inside the library).  Checked through the C ABI against the workspace entry
point on two calls in a row; this file is collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

import workloads as W
from tests.helpers import assert_attn_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def msa():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import block_sparse_paged_02_gb300 as m
    L = m.lib()
    P, i32 = ctypes.c_void_p, ctypes.c_int32
    L.msa_sparse_paged_attn_static.restype = ctypes.c_int
    L.msa_sparse_paged_attn_static.argtypes = [P, P, i32, P, P, P]
    return m


def _static_call(msa, c, stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return msa.lib().msa_sparse_paged_attn_static(
        ctypes.byref(c.attn), ctypes.c_void_p(c.tbl.data_ptr()), int(c.tbl_stride),
        ctypes.c_void_p(c.sparse_len.data_ptr()), ctypes.c_void_p(c.status.data_ptr()),
        ctypes.c_void_p(s.cuda_stream))


@pytest.mark.parametrize("kv,scale,sink", [(W.KV_FP8, W.SCALE_SCALAR, True),
                                           (W.KV_BF16, W.SCALE_NONE, False),
                                           (W.KV_FP8, W.SCALE_PER_TOKEN_HEAD, True)])
def test_static_scratch_matches_workspace_entry_point(msa, kv, scale, sink):
    w = W.custom(70, q_lens=[1, 4, 1, 2], seq_lens=[9000, 3000, 600, 20000], hq=16, di=128,
                 topk=16, kv_dtype=kv, scale_mode=scale, with_sink=sink)
    c = msa.DeviceCase(w)
    c.index_score()
    c.topk_build_table()
    c.sparse_paged_attn()            # the existing entry point, with a workspace
    ref = c.fetch()
    for _ in range(2):               # two calls in a row share the static array
        c.out.fill_(7.0)
        c.lse.fill_(7.0)
        assert _static_call(msa, c) == 0
        got = c.fetch()
        assert got["status"] == 0
        assert_attn_close(got["out"], got["lse"], ref["out"], ref["lse"])
        assert np.all(np.isfinite(got["out"]))


def test_static_scratch_rejects_oversized_calls(msa):
    # 2048 rows run one split each; their split records need ~17 MB of scratch,
    # more than the static array holds, so the call is refused before launch
    w = W.custom(71, q_lens=[2048], seq_lens=[2100], hq=16, di=128, topk=2)
    c = msa.DeviceCase(w)
    need = msa.msa_workspace_size(w.num_rows, 0, 0, 16, 128, c.tbl_stride)
    assert need > (8 << 20)
    c.status.zero_()
    assert _static_call(msa, c) == 5  # MSA_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert int(c.status.item()) == 0
