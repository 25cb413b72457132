"""msa_sparse_paged_attn_static: the attention entry point for callers that
cannot allocate device memory (its scratch lives in a static device array
inside the library).  Checked through the C ABI against the fp64 oracle and
against the workspace entry point, on calls in a row; this file is
collected last on purpose, so a failure here comes after every other test."""
import ctypes

import numpy as np
import pytest
import torch

import workloads as W
from tests.helpers import assert_attn_close

pytestmark = pytest.mark.gpu

MSA_ERR_NULL, MSA_ERR_DTYPE, MSA_ERR_WORKSPACE = 1, 3, 5
STATIC_BYTES = 8 << 20


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


def _static_call(msa, c, stream=None, attn=None, tbl=True, length=True):
    s = torch.cuda.current_stream() if stream is None else stream
    return msa.lib().msa_sparse_paged_attn_static(
        ctypes.byref(c.attn if attn is None else attn),
        ctypes.c_void_p(c.tbl.data_ptr()) if tbl else None, int(c.tbl_stride),
        ctypes.c_void_p(c.sparse_len.data_ptr()) if length else None,
        ctypes.c_void_p(c.status.data_ptr()), ctypes.c_void_p(s.cuda_stream))


def _tables_from_gpu_path(c, orc, w):
    """Scores, top-k and table on the GPU, checked bit for bit against the
    oracle's own (the oracle never takes a table from the GPU)."""
    ref = orc.decode(w)
    assert ref["status"] == 0
    c.index_score()
    c.topk_build_table()
    got = c.fetch()
    assert np.array_equal(got["tbl"][:, : 8 * w.topk], ref["tbl"][:, : 8 * w.topk])
    assert np.array_equal(got["sparse_len"], ref["sparse_len"])
    return ref


def _check_static_calls(msa, c, ref, want_ws, calls=2):
    for _ in range(calls):  # calls in a row share the static array
        c.out.fill_(7.0)
        c.lse.fill_(7.0)
        assert _static_call(msa, c) == 0
        got = c.fetch()
        assert got["status"] == 0
        assert_attn_close(got["out"], got["lse"], ref["out"], ref["lse"])  # the oracle
        assert_attn_close(got["out"], got["lse"], want_ws["out"], want_ws["lse"])
        assert np.all(np.isfinite(got["out"]))


@pytest.mark.parametrize("kv,scale,sink", [(W.KV_FP8, W.SCALE_SCALAR, True),
                                           (W.KV_BF16, W.SCALE_NONE, False),
                                           (W.KV_FP8, W.SCALE_PER_TOKEN_HEAD, True)])
def test_static_scratch_matches_oracle_and_workspace_entry_point(msa, orc, kv, scale, sink):
    w = W.custom(70, q_lens=[1, 4, 1, 2], seq_lens=[9000, 3000, 600, 20000], hq=16, di=128,
                 topk=16, kv_dtype=kv, scale_mode=scale, with_sink=sink)
    c = msa.DeviceCase(w)
    ref = _tables_from_gpu_path(c, orc, w)
    c.sparse_paged_attn()            # the existing entry point, with a workspace
    want_ws = c.fetch()
    _check_static_calls(msa, c, ref, want_ws)


def test_static_scratch_more_splits_than_a_cluster(msa, orc):
    # top-k 160 blocks = 1280 page-16 entries per row = 10 splits of 128, so
    # the rows merge through the array's counters and partials; a call of
    # cluster-merged rows in between must not disturb the next one
    w = W.custom(72, q_lens=[1, 2, 1], seq_lens=[24000, 30000, 21000], hq=16, di=128,
                 topk=160, kv_dtype=W.KV_FP8, scale_mode=W.SCALE_SCALAR, with_sink=True)
    c = msa.DeviceCase(w)
    ref = _tables_from_gpu_path(c, orc, w)
    c.sparse_paged_attn()
    want_ws = c.fetch()
    _check_static_calls(msa, c, ref, want_ws, calls=2)
    small = W.custom(73, q_lens=[1, 3], seq_lens=[5000, 7000], hq=16, di=128, topk=16,
                     kv_dtype=W.KV_BF16, scale_mode=W.SCALE_NONE, with_sink=False)
    cs = msa.DeviceCase(small)
    ref_s = _tables_from_gpu_path(cs, orc, small)
    cs.sparse_paged_attn()
    _check_static_calls(msa, cs, ref_s, cs.fetch(), calls=1)
    _check_static_calls(msa, c, ref, want_ws, calls=1)


def test_static_scratch_takes_many_single_split_rows(msa, orc):
    # 2048 rows of one split each: no merge, so only 4 bytes per row of the
    # array are in play and the call is accepted, although the workspace
    # entry point would ask for ~17 MB
    w = W.custom(71, q_lens=[2048], seq_lens=[2100], hq=16, di=128, topk=2)
    c = msa.DeviceCase(w)
    assert msa.msa_workspace_size(w.num_rows, 0, 0, 16, 128, c.tbl_stride) > STATIC_BYTES
    c.index_score()
    c.topk_build_table()
    c.sparse_paged_attn()
    want_ws = c.fetch()
    c.out.fill_(7.0)
    c.lse.fill_(7.0)
    assert _static_call(msa, c) == 0
    got = c.fetch()
    assert got["status"] == 0
    assert np.array_equal(got["out"], want_ws["out"])  # the same kernel and split
    assert np.array_equal(got["lse"], want_ws["lse"])
    rows = np.arange(0, w.num_rows, 97)  # sampled rows against the oracle
    from tests.helpers import sub_workload
    sub = sub_workload(w, rows)
    ref = orc.decode(sub)
    assert_attn_close(got["out"][rows], got["lse"][rows], ref["out"], ref["lse"])


def test_static_scratch_rejects_oversized_and_bad_calls(msa):
    # 128 rows of 10 splits each need 128 x 10 x 8320 bytes of partials,
    # more than the array holds: refused before anything is launched
    w = W.custom(74, q_lens=[128], seq_lens=[21000], hq=16, di=128, topk=160)
    c = msa.DeviceCase(w)
    c.status.zero_()
    c.out.fill_(7.0)
    assert _static_call(msa, c) == MSA_ERR_WORKSPACE
    # argument errors come back as they do from the workspace entry point
    assert _static_call(msa, c, tbl=False) == MSA_ERR_NULL
    assert _static_call(msa, c, length=False) == MSA_ERR_NULL
    bad = msa.make_attn_args(c.q, c.k, c.v, 7, w.num_pages, c.out, c.lse,
                             softmax_scale=w.softmax_scale)
    assert _static_call(msa, c, attn=bad) == MSA_ERR_DTYPE
    torch.cuda.synchronize()
    assert int(c.status.item()) == 0
    assert bool((c.out.float() == 7.0).all())  # nothing ran
