"""Sparse MLA decode (msa_sparse_mla_decode) against the fp64 oracle."""
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
    m.lib()
    return m


def run(msa, orc, w, **kw):
    c = msa.MlaCase(w, **kw)
    c.decode()
    got = c.fetch()
    out, lse, st = orc.sparse_mla(w.q, w.kv_cache, w.kv_indptr, w.kv_indices, w.dv,
                                  sinks=w.sinks, softmax_scale=w.softmax_scale,
                                  q_scale=w.q_scale, kv_scale=w.kv_scale)
    return c, got, out, lse, st


@pytest.mark.parametrize("heads,sink,dup", [(16, True, False), (16, False, False),
                                            (20, True, True), (128, True, False)])
def test_sparse_mla_matches_oracle(msa, orc, heads, sink, dup):
    counts = [0, 1, 15, 16, 17, 300, 2048, 33]
    w = W.sparse_mla_custom(70 + heads, counts, heads=heads, ctx=4096, with_sink=sink,
                            duplicates=dup)
    _, got, out, lse, st = run(msa, orc, w)
    assert st == 0 and got["status"] == 0
    assert_attn_close(got["out"], got["lse"], out, lse)


def test_sparse_mla_named_workload(msa, orc):
    w = W.sparse_mla_decode()
    c, got, out, lse, st = run(msa, orc, w)
    assert st == 0 and got["status"] == 0
    assert_attn_close(got["out"], got["lse"], out, lse)
    # repeated calls (split counters back at zero) give identical outputs
    first = c.out.clone()
    c.decode()
    torch.cuda.synchronize()
    assert torch.equal(first, c.out)


def test_sparse_mla_poisoned_rows(msa, orc):
    w = W.sparse_mla_custom(75, [40, 500, 7], heads=16, ctx=1024)
    w.kv_indices = w.kv_indices.copy()
    w.kv_indices[45] = w.num_tokens  # an id past the cache in row 1
    _, got, out, lse, st = run(msa, orc, w)
    assert st == 8 and got["status"] & 8
    assert_attn_close(got["out"], got["lse"], out, lse)  # row 1 empty on both sides
    assert np.all(got["out"][1] == 0)


def test_sparse_mla_rows_longer_than_the_bound_are_refused(msa, orc):
    w = W.sparse_mla_custom(76, [100, 64], heads=16, ctx=1024)
    c = msa.MlaCase(w, max_tokens=64)
    c.decode()
    got = c.fetch()
    assert got["status"] & 8
    assert np.all(got["out"][0] == 0)
    out, lse, _ = orc.sparse_mla(w.q, w.kv_cache, w.kv_indptr, w.kv_indices, w.dv,
                                 sinks=w.sinks, softmax_scale=w.softmax_scale)
    assert_attn_close(got["out"][1:], got["lse"][1:], out[1:], lse[1:])


def test_sparse_mla_more_splits_than_a_cluster(msa, orc):
    # 20000 ids in one row need more than 8 splits of <= 2048 ids: those
    # splits merge through the workspace (last-arriving CTA), and an id past
    # the cache in that row still empties it
    w = W.sparse_mla_custom(77, [20000, 3, 700], heads=16, ctx=24000)
    _, got, out, lse, st = run(msa, orc, w)
    assert st == 0 and got["status"] == 0
    assert_attn_close(got["out"], got["lse"], out, lse)
    w.kv_indices = w.kv_indices.copy()
    w.kv_indices[12345] = w.num_tokens
    _, got, out, lse, st = run(msa, orc, w)
    assert st == 8 and got["status"] & 8
    assert np.all(got["out"][0] == 0)
    assert_attn_close(got["out"], got["lse"], out, lse)


# ------------------------------------------------------ FP8 latent cache / query

@pytest.mark.parametrize("fp8_q,heads,sink,dup", [(True, 16, True, False), (False, 16, True, False),
                                                  (True, 20, False, True), (True, 128, True, False)])
def test_fp8_sparse_mla_matches_oracle(msa, orc, fp8_q, heads, sink, dup):
    # e4m3 cache (and query) with scalar scales; lengths that leave the
    # last step ragged, an empty row, a row of one token, 2048 tokens
    counts = [0, 1, 15, 16, 17, 300, 2048, 33]
    w = W.mla_fp8(W.sparse_mla_custom(90 + heads, counts, heads=heads, ctx=4096,
                                      with_sink=sink, duplicates=dup), seed=91, fp8_q=fp8_q)
    _, got, out, lse, st = run(msa, orc, w)
    assert st == 0 and got["status"] == 0
    assert_attn_close(got["out"], got["lse"], out, lse)


def test_fp8_sparse_mla_more_splits_than_a_cluster(msa, orc):
    # 20000 tokens per row: more splits than one cluster holds, merged through
    # the workspace partials (and the kv_scale applied there too)
    w = W.mla_fp8(W.sparse_mla_custom(93, [20000, 5000, 3], heads=16, ctx=32768), seed=94)
    c, got, out, lse, st = run(msa, orc, w)
    assert st == 0 and got["status"] == 0
    assert_attn_close(got["out"], got["lse"], out, lse)
    first = c.out.clone()
    c.decode()
    torch.cuda.synchronize()
    assert torch.equal(first, c.out)


def test_fp8_sparse_mla_named_workload_sampled(msa, orc):
    w = W.sparse_mla_decode_fp8()
    c = msa.MlaCase(w)
    c.decode()
    got = c.fetch()
    assert got["status"] == 0
    rows = [0, 17, 40, 63]
    ip = w.kv_indptr
    sub = np.concatenate([w.kv_indices[ip[r]:ip[r + 1]] for r in rows])
    sub_ip = np.concatenate([[0], np.cumsum([ip[r + 1] - ip[r] for r in rows])]).astype(np.int32)
    out, lse, st = orc.sparse_mla(w.q[rows], w.kv_cache, sub_ip, sub, w.dv, sinks=w.sinks,
                                  softmax_scale=w.softmax_scale, q_scale=w.q_scale,
                                  kv_scale=w.kv_scale)
    assert st == 0
    assert_attn_close(got["out"][rows], got["lse"][rows], out, lse)


def test_fp8_query_with_bf16_cache_is_refused(msa):
    w = W.sparse_mla_custom(95, [10], heads=16, ctx=64)
    c = msa.MlaCase(w)
    q8 = torch.zeros(c.q.shape, dtype=torch.uint8, device="cuda")
    scale = torch.ones(1, dtype=torch.float32, device="cuda")
    args = msa.make_mla_args(q8, c.kv, c.indptr, c.indices, c.out, c.lse,
                             max_tokens=c.max_tokens, softmax_scale=w.softmax_scale,
                             q_scale=scale)
    with pytest.raises(msa.MsaError):
        msa.msa_sparse_mla_decode(args, c.workspace, c.status)

