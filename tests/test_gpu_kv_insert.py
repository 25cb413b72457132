"""msa_kv_insert (the step before the path) against the oracle, byte for byte,
then a decode over the updated pools against the oracle."""
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


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()


@pytest.mark.parametrize("kv,scale", [(W.KV_BF16, W.SCALE_NONE), (W.KV_FP8, W.SCALE_SCALAR),
                                      (W.KV_FP8, W.SCALE_PER_TOKEN_HEAD),
                                      (W.KV_FP8, W.SCALE_NONE)])
@pytest.mark.parametrize("skip_index", [False, True])
def test_kv_insert_matches_oracle_then_decode(msa, orc, kv, scale, skip_index):
    w = W.custom(92, q_lens=[1, 4, 2, 1], seq_lens=[3000, 700, 129, 9000], hq=16, di=128,
                 topk=8, kv_dtype=kv, scale_mode=scale, with_sink=True)
    rng = np.random.default_rng(5)
    k_new = W.bf16_bits(rng.standard_normal((w.num_rows, 1, 128)) * 2)
    v_new = W.bf16_bits(rng.standard_normal((w.num_rows, 1, 128)) * 2)
    idx_new = W.bf16_bits(rng.integers(-3, 4, (w.num_rows, 1, 128)).astype(np.float32))
    c = msa.DeviceCase(w)
    c.kv_insert(_dev(k_new), _dev(v_new), _dev(idx_new), skip_index=skip_index)
    torch.cuda.synchronize()
    assert int(c.status.item()) == 0
    k, v, ik, ks, vs, st = orc.kv_insert(w, k_new, v_new, idx_new, skip_index=skip_index)
    assert st == 0
    view = (lambda t: t.view(torch.int16).cpu().numpy().view(np.uint16)) if kv == W.KV_BF16 \
        else (lambda t: t.cpu().numpy())
    assert np.array_equal(view(c.k), k)
    assert np.array_equal(view(c.v), v)
    assert np.array_equal(c.idx_k.view(torch.int16).cpu().numpy().view(np.uint16), ik)
    if scale == W.SCALE_PER_TOKEN_HEAD:
        assert np.array_equal(c.k_scale.cpu().numpy(), ks)
        assert np.array_equal(c.v_scale.cpu().numpy(), vs)
    # decode over the updated pools
    c.decode()
    got = c.fetch()
    w.k_cache, w.v_cache, w.idx_k = k, v, ik
    if ks is not None:
        w.k_scale, w.v_scale = ks, vs
    ref = orc.decode(w)
    for key in ("topk_idx", "tbl", "sparse_len"):
        assert np.array_equal(got[key], ref[key])
    assert_attn_close(got["out"], got["lse"], ref["out"], ref["lse"])


def test_kv_insert_skips_invalid_requests(msa, orc):
    w = W.custom(93, q_lens=[1, 1], seq_lens=[300, 300], hq=16, di=128, topk=2)
    bt = w.block_table.copy()
    bt[1, 0] = w.num_pages + 3
    w.block_table = bt
    rng = np.random.default_rng(6)
    k_new = W.bf16_bits(rng.standard_normal((2, 1, 128)))
    idx_new = W.bf16_bits(rng.integers(-3, 4, (2, 1, 128)).astype(np.float32))
    c = msa.DeviceCase(w)
    before = c.k.clone()
    c.kv_insert(_dev(k_new), _dev(k_new), _dev(idx_new))
    torch.cuda.synchronize()
    assert int(c.status.item()) == msa.MSA_DEV_BAD_PAGE
    k, _, _, _, _, st = orc.kv_insert(w, k_new, k_new, idx_new)
    assert st == orc.BAD_PAGE
    assert np.array_equal(c.k.view(torch.int16).cpu().numpy().view(np.uint16), k)
    assert (c.k != before).any()  # request 0 was written


@pytest.mark.parametrize("hi,di", [(1, 64), (2, 64), (1, 128)])
@pytest.mark.parametrize("scaled", [True, False])
def test_kv_insert_fp8_index_cache(msa, orc, hi, di, scaled):
    # e4m3 index keys (+ per-token scales) written byte for byte as the oracle
    # writes them, then a decode that scores the new keys
    base = W.custom(94, q_lens=[1, 3, 1], seq_lens=[2000, 300, 129], hq=8, di=di, hi=hi, topk=4)
    w = W.fp8_index(base, seed=95, scaled=scaled)
    rng = np.random.default_rng(6)
    k_new = W.bf16_bits(rng.standard_normal((w.num_rows, 1, 128)))
    v_new = W.bf16_bits(rng.standard_normal((w.num_rows, 1, 128)))
    idx_new = W.bf16_bits(rng.integers(-3, 4, (w.num_rows, hi, di)).astype(np.float32))
    c = msa.DeviceCase(w)
    c.kv_insert(_dev(k_new), _dev(v_new), _dev(idx_new))
    torch.cuda.synchronize()
    assert int(c.status.item()) == 0
    res = orc.kv_insert(w, k_new, v_new, idx_new)
    ik, st, iscale = res[2], res[5], res[6]
    assert st == 0
    assert np.array_equal(c.idx_k.cpu().numpy(), ik)
    if scaled:
        assert np.array_equal(c.idx_k_scale.cpu().numpy(), iscale)
    c.decode()
    got = c.fetch()
    w.k_cache, w.v_cache, w.idx_k = res[0], res[1], ik
    w.idx_k_scale = iscale
    ref = orc.decode(w)
    for key in ("topk_idx", "tbl", "sparse_len"):
        assert np.array_equal(got[key], ref[key])
    assert_attn_close(got["out"], got["lse"], ref["out"], ref["lse"])
