"""Index-top-k reuse across layers: a later layer skips scoring and
selection and runs attention over the page-16 table an earlier layer's
msa_decode produced (vLLM PR 47287 page, "Features and motivation" and
"Related work": index-topk reuse).

The oracle computes layer 1's whole path itself; the GPU's layer-1 table
must equal the oracle's bit for bit, and every reuse layer's attention is
checked against the oracle's attention over the oracle's own table."""
import dataclasses

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


def _layer(seed, like, kv, scale, sink):
    """Another layer over the same requests and pages: its own queries, K/V,
    scales and sinks (and index cache, which a reuse layer never reads)."""
    w = W.custom(seed, q_lens=list(like.q_lens), seq_lens=list(like.seq_lens), hq=16, di=128,
                 topk=like.topk, kv_dtype=kv, scale_mode=scale, with_sink=sink,
                 pool_pages=like.num_pages)
    return dataclasses.replace(w, block_table=like.block_table)


@pytest.mark.parametrize("kv,scale,sink", [(W.KV_FP8, W.SCALE_PER_TOKEN_HEAD, True),
                                           (W.KV_BF16, W.SCALE_NONE, False),
                                           (W.KV_FP8, W.SCALE_SCALAR, True)])
def test_later_layers_reuse_the_sparse_table(msa, orc, kv, scale, sink):
    w1 = W.custom(80, q_lens=[1, 4, 1, 3], seq_lens=[12000, 5000, 900, 40000], hq=16, di=128,
                  topk=16, kv_dtype=kv, scale_mode=scale, with_sink=sink)
    ref1 = orc.decode(w1)  # the oracle's own layer-1 path
    assert ref1["status"] == 0
    c1 = msa.DeviceCase(w1)
    c1.decode()  # layer 1: score, select, table, attention
    first = c1.fetch()
    assert first["status"] == 0
    for key in ("topk_idx", "tbl", "sparse_len"):
        assert np.array_equal(first[key], ref1[key]), key
    assert_attn_close(first["out"], first["lse"], ref1["out"], ref1["lse"])
    # layers 2 and 3 reuse layer 1's selection: attention only, on the table
    # layer 1's decode left on the device
    for seed in (81, 82):
        wl = _layer(seed, w1, kv, scale, sink)
        cl = msa.DeviceCase(wl)
        cl.tbl.copy_(c1.tbl)
        cl.sparse_len.copy_(c1.sparse_len)
        cl.sparse_paged_attn()
        got = cl.fetch()
        ref_o, ref_l, st = orc.sparse_attn(wl.q, wl.k_cache, wl.v_cache, wl.kv_dtype,
                                           ref1["tbl"], ref1["sparse_len"],
                                           scale_mode=wl.scale_mode, k_scale=wl.k_scale,
                                           v_scale=wl.v_scale, sinks=wl.sinks,
                                           softmax_scale=wl.softmax_scale,
                                           num_pages16=8 * wl.num_pages)
        assert st == 0 and got["status"] == 0
        assert_attn_close(got["out"], got["lse"], ref_o, ref_l)
