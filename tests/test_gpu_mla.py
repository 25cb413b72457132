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
                                  sinks=w.sinks, softmax_scale=w.softmax_scale)
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
