"""Index-top-k reuse across layers: a later layer skips scoring and
selection and runs attention over the page-16 table an earlier layer's
msa_decode produced (vLLM PR 47287 page, "Features and motivation" and
"Related work": index-topk reuse).  Checked against the oracle's attention
on the same table."""
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


def test_later_layer_reuses_the_sparse_table(msa, orc):
    w1 = W.custom(80, q_lens=[1, 4, 1], seq_lens=[12000, 5000, 900], hq=16, di=128, topk=16,
                  kv_dtype=W.KV_FP8, scale_mode=W.SCALE_PER_TOKEN_HEAD, with_sink=True)
    # layer 2: the same requests and pages, its own queries, K/V, scales and sinks
    w2 = W.custom(81, q_lens=[1, 4, 1], seq_lens=[12000, 5000, 900], hq=16, di=128, topk=16,
                  kv_dtype=W.KV_FP8, scale_mode=W.SCALE_PER_TOKEN_HEAD, with_sink=True,
                  pool_pages=w1.num_pages)
    w2.block_table = w1.block_table
    c1 = msa.DeviceCase(w1)
    c1.decode()  # layer 1: score, select, table, attention
    first = c1.fetch()
    c2 = msa.DeviceCase(w2)
    c2.tbl.copy_(c1.tbl)  # layer 2: reuse the table, attention only
    c2.sparse_len.copy_(c1.sparse_len)
    c2.sparse_paged_attn()
    got = c2.fetch()
    ref_o, ref_l, st = orc.sparse_attn(w2.q, w2.k_cache, w2.v_cache, w2.kv_dtype, first["tbl"],
                                       first["sparse_len"], scale_mode=w2.scale_mode,
                                       k_scale=w2.k_scale, v_scale=w2.v_scale, sinks=w2.sinks,
                                       softmax_scale=w2.softmax_scale,
                                       num_pages16=8 * w2.num_pages)
    assert st == 0 and got["status"] == 0
    assert_attn_close(got["out"], got["lse"], ref_o, ref_l)
