"""GPU parity: the CUDA path through the C ABI against the fp64 CPU oracle.

Block scores, top-k indices, page-16 tables and sparse lengths must be
bit-exact (integer-valued index vectors make every fp32 score exact);
attention must satisfy |O - O_ref| <= 1e-2 (1 + |O_ref|) and
|LSE - LSE_ref| <= 2e-3.
"""
import numpy as np
import pytest
import torch

import workloads as W
from tests.helpers import assert_attn_close, prefill_rows, sub_workload, valid_score_mask

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def msa():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import block_sparse_paged_02_gb300 as m
    m.lib()
    return m


def run_steps(msa, w, **kw):
    """Run the three entry points separately, then the fused call, and return
    the separate results plus the fused ones."""
    c = msa.DeviceCase(w, **kw)
    c.index_score()
    c.topk_build_table()
    c.sparse_paged_attn()
    sep = c.fetch()
    # fused path into fresh outputs
    c.out.zero_()
    c.lse.zero_()
    c.topk_idx.fill_(123)
    c.tbl.fill_(123)
    c.sparse_len.fill_(123)
    c.decode()
    fused = c.fetch()
    return c, sep, fused


def check_against_oracle(orc, w, sep, fused, topk=None):
    k = int(topk or w.topk)
    b = orc.Batch.of(w)
    geom = orc.row_geometry(b)
    ref = orc.decode(w, topk=k)
    mask = valid_score_mask(geom, w.bt_stride)
    assert np.array_equal(sep["scores"][mask], ref["scores"][mask]), "block scores differ"
    assert np.array_equal(sep["topk_idx"], ref["topk_idx"]), "top-k indices differ"
    assert np.array_equal(sep["sparse_len"], ref["sparse_len"]), "sparse lengths differ"
    assert np.array_equal(sep["tbl"][:, : 8 * k], ref["tbl"][:, : 8 * k]), "sparse tables differ"
    assert np.all(sep["tbl"][:, 8 * k:] == 0)
    assert sep["status"] == ref["status"]
    assert_attn_close(sep["out"], sep["lse"], ref["out"], ref["lse"])
    check_fused(w, sep, fused, ref, topk=k)
    return ref


def check_fused(w, sep, fused, ref, topk=None):
    """The fused call's tables equal the separate calls' bit for bit; so do
    its outputs on rows of the split-K decode attention, while rows of the
    prefill path are held to the oracle (ref: the oracle's decode, or None
    to skip that check)."""
    for key in ("topk_idx", "tbl", "sparse_len"):
        assert np.array_equal(fused[key], sep[key]), f"fused {key} differs"
    pre = prefill_rows(w, topk)
    dec = ~pre
    for key in ("out", "lse"):
        assert np.array_equal(fused[key][dec], sep[key][dec], equal_nan=True), f"fused {key} differs"
    if ref is not None and pre.any():
        assert fused["status"] == ref["status"]
        assert_attn_close(fused["out"][pre], fused["lse"][pre], ref["out"][pre], ref["lse"][pre])


@pytest.mark.parametrize("name", ["tiny_decode", "batched_decode", "speculative_decode",
                                  "large_batch_decode", "large_batch_decode_fp8_index"])
def test_named_workload_full_size(msa, orc, name):
    w = W.NAMED[name]()
    _, sep, fused = run_steps(msa, w)
    check_against_oracle(orc, w, sep, fused)


def test_chunked_prefill_full_size_sampled_rows(msa, orc):
    w = W.chunked_prefill()
    _, sep, fused = run_steps(msa, w)
    check_fused(w, sep, fused, None)
    assert prefill_rows(w).all()  # every row takes the prefill path in the fused call
    rng = np.random.default_rng(0)
    # first/last rows of each request, rows around block boundaries, random rows
    rows = {0, 1, 127, 128, 2047, 2048, 2049, 4095}
    rows |= set(int(x) for x in rng.choice(w.num_rows, 40, replace=False))
    rows = np.array(sorted(rows))
    sub = sub_workload(w, rows)
    ref = orc.decode(sub)
    assert ref["status"] == 0 and sep["status"] == 0
    assert np.array_equal(sep["topk_idx"][rows], ref["topk_idx"])
    assert np.array_equal(sep["tbl"][rows], ref["tbl"])
    assert np.array_equal(sep["sparse_len"][rows], ref["sparse_len"])
    nb = ref["tbl"].shape[1]
    assert_attn_close(sep["out"][rows], sep["lse"][rows], ref["out"], ref["lse"])
    assert_attn_close(fused["out"][rows], fused["lse"][rows], ref["out"], ref["lse"])
    assert fused["status"] == 0
    assert np.all(np.isfinite(fused["out"])) and np.all(np.isfinite(fused["lse"]))
    # every row: the length is the clamp of the selected blocks, the table has
    # exactly ceil(len/16) leading non-empty slots per selected block pattern
    L = (w.context_lens[0] + np.arange(2048) + 1)
    assert np.all(sep["sparse_len"][:2048] <= np.minimum(L, 16 * 128))


def test_chunked_prefill_small_elementwise(msa, orc):
    w = W.chunked_prefill(seed=15, context=1000, new_tokens=300, reqs=2)
    _, sep, fused = run_steps(msa, w)
    check_against_oracle(orc, w, sep, fused)


@pytest.mark.parametrize("kv", [W.KV_BF16, W.KV_FP8])
@pytest.mark.parametrize("scale", [W.SCALE_NONE, W.SCALE_SCALAR, W.SCALE_PER_TOKEN_HEAD])
@pytest.mark.parametrize("sink", [False, True])
def test_dtype_scale_sink_matrix(msa, orc, kv, scale, sink):
    w = W.custom(40 + 3 * kv + scale, q_lens=[1, 4, 2, 1, 3],
                 seq_lens=[5000, 2100, 700, 130, 9000], hq=16, di=128, topk=8, kv_dtype=kv,
                 scale_mode=scale, with_sink=sink)
    _, sep, fused = run_steps(msa, w)
    check_against_oracle(orc, w, sep, fused)


def test_edge_lengths_and_empty_requests(msa, orc):
    seq = [1, 15, 16, 17, 127, 128, 129, 255, 256, 257, 2000, 3, 640]
    ql = [1, 1, 1, 2, 1, 0, 4, 1, 0, 3, 1, 2, 1]
    w = W.custom(50, q_lens=ql, seq_lens=seq, hq=8, di=64, topk=3, kv_dtype=W.KV_FP8,
                 scale_mode=W.SCALE_PER_TOKEN_HEAD, with_sink=True)
    _, sep, fused = run_steps(msa, w)
    check_against_oracle(orc, w, sep, fused)


@pytest.mark.parametrize("topk", [1, 2, 40])
def test_topk_extremes(msa, orc, topk):
    # k = 1, small k, and k larger than every row's block count (select all)
    w = W.custom(51, q_lens=[1, 2, 1], seq_lens=[4000, 1100, 130], hq=16, di=128, topk=topk,
                 with_sink=True)
    _, sep, fused = run_steps(msa, w)
    check_against_oracle(orc, w, sep, fused)


def test_more_attention_splits_than_a_cluster(msa, orc):
    # k = 160 blocks = 1280 page-16 entries per row: more than 8 splits of
    # <= 128 entries, so the splits merge through the workspace instead of a
    # thread-block cluster
    w = W.custom(59, q_lens=[1, 2], seq_lens=[30000, 24000], hq=16, di=128, topk=160,
                 kv_dtype=W.KV_FP8, scale_mode=W.SCALE_SCALAR, with_sink=True)
    _, sep, fused = run_steps(msa, w)
    check_against_oracle(orc, w, sep, fused)


def test_largest_block_table_and_topk(msa, orc):
    # the largest sizes the ABI accepts: a row with bt_stride = 16384 blocks
    # (2^21 tokens) selecting topk = 2048 blocks (16384 page-16 entries, 128
    # attention splits merged through the workspace), beside a row whose
    # blocks are fewer than k (all selected)
    w = W.custom(71, q_lens=[1, 1], seq_lens=[16384 * 128, 5000], hq=8, di=64, topk=2048,
                 kv_dtype=W.KV_FP8, scale_mode=W.SCALE_SCALAR, with_sink=True)
    assert w.bt_stride == 16384
    _, sep, fused = run_steps(msa, w)
    check_against_oracle(orc, w, sep, fused)


def test_largest_request_count(msa, orc):
    # num_reqs = 4096 (the most a batch may hold): one-row requests and a few
    # empty ones, contexts of 1..400 tokens; thousands of rows take the
    # one-warp-per-row top-k
    rng = np.random.default_rng(72)
    ql = [0 if i % 97 == 5 else 1 for i in range(4096)]
    seq = [int(x) for x in rng.integers(1, 401, size=4096)]
    w = W.custom(72, q_lens=ql, seq_lens=seq, hq=8, di=64, topk=3, kv_dtype=W.KV_FP8,
                 scale_mode=W.SCALE_PER_TOKEN_HEAD, with_sink=True)
    assert len(w.cu_seqlens_q) - 1 == 4096
    _, sep, fused = run_steps(msa, w)
    check_against_oracle(orc, w, sep, fused)


@pytest.mark.parametrize("rows,kv", [(152, W.KV_FP8), (101, W.KV_FP8), (60, W.KV_FP8),
                                     (50, W.KV_FP8), (43, W.KV_FP8), (101, W.KV_BF16),
                                     (43, W.KV_BF16)])
def test_cluster_merge_split_counts(msa, orc, rows, kv):
    # k = 16 blocks = 128 entries per row; on 152 SMs x 2 CTAs these row
    # counts give 2, 3, 5, 6 and 7 splits per row, so the cluster merge runs
    # with every owner layout (two chunks per CTA at 2 and 3 splits, one at
    # 5..7, CTAs that own nothing at 5..7); bf16 slabs take the pull merge
    rng = np.random.default_rng(rows)
    seq = [int(x) for x in rng.integers(2100, 2600, size=rows)]
    w = W.custom(80 + rows, q_lens=[1] * rows, seq_lens=seq, hq=16, di=128, topk=16,
                 kv_dtype=kv, scale_mode=W.SCALE_SCALAR if kv == W.KV_FP8 else W.SCALE_NONE,
                 with_sink=True)
    _, sep, fused = run_steps(msa, w)
    check_against_oracle(orc, w, sep, fused)


@pytest.mark.parametrize("idx_range", [1, 3])
def test_radix_select_few_long_rows(msa, orc, idx_range):
    # few rows whose block tables exceed 512 entries take the radix-select
    # top-k; idx_range 1 makes many blocks tie at the threshold
    w = W.custom(90 + idx_range, q_lens=[1, 2, 1], seq_lens=[70000, 90000, 3000], hq=16,
                 di=128, topk=16, idx_range=idx_range, kv_dtype=W.KV_FP8,
                 scale_mode=W.SCALE_SCALAR, with_sink=True)
    assert w.bt_stride > 512
    _, sep, fused = run_steps(msa, w)
    check_against_oracle(orc, w, sep, fused)


def test_heavy_ties(msa, orc):
    # index values in {-1, 0, 1} with Di 64: many blocks tie at the same score
    w = W.custom(52, q_lens=[1, 4], seq_lens=[30000, 20000], hq=16, di=64, idx_range=1,
                 topk=16)
    _, sep, fused = run_steps(msa, w)
    check_against_oracle(orc, w, sep, fused)


@pytest.mark.parametrize("seq,idx_range", [(200_000, 3), (200_000, 1), (1_000_000, 3)])
def test_long_rows_wide_block_tables(msa, orc, seq, idx_range):
    # rows with more than 1024 candidate blocks take the several-keys-per-thread
    # top-k (bt_stride up to 16384); k = 64 and, with idx_range 1, many ties
    w = W.custom(53, q_lens=[1, 2], seq_lens=[seq, seq // 3], hq=16, di=64, topk=64,
                 idx_range=idx_range)
    assert w.bt_stride > 1024
    _, sep, fused = run_steps(msa, w)
    check_against_oracle(orc, w, sep, fused)


@pytest.mark.parametrize("hi,di", [(1, 64), (2, 64), (1, 128)])
@pytest.mark.parametrize("scaled", [True, False])
def test_fp8_index_cache(msa, orc, hi, di, scaled):
    # e4m3 index keys (+ per-token scales): scores and tables bit-exact
    w = W.fp8_index(W.custom(60 + hi + di, q_lens=[1, 4, 9, 2], seq_lens=[5000, 2100, 700, 9000],
                             hq=16, di=di, hi=hi, topk=8, kv_dtype=W.KV_FP8,
                             scale_mode=W.SCALE_SCALAR, with_sink=True),
                    seed=61, scaled=scaled)
    _, sep, fused = run_steps(msa, w)
    check_against_oracle(orc, w, sep, fused)  # scores included, bit for bit


@pytest.mark.parametrize("reqs", [64, 1200])
def test_fp8_index_ring_sizes(msa, orc, reqs):
    # e4m3 pages of 128 dims: the 12-stage ring while the batch's request
    # prefix fits beside it (64 requests), the 10-stage ring beyond that
    # (1200 requests); scores, selection and attention against the oracle
    rng = np.random.default_rng(reqs)
    seq = [int(x) for x in rng.integers(100, 1400, size=reqs)]
    w = W.fp8_index(W.custom(90, q_lens=[1] * reqs, seq_lens=seq, hq=8, di=128, topk=2,
                             kv_dtype=W.KV_FP8, scale_mode=W.SCALE_SCALAR), seed=91)
    _, sep, fused = run_steps(msa, w)
    check_against_oracle(orc, w, sep, fused)


def test_fp8_index_many_rows_and_garbage(msa, orc):
    # a request with >= 64 rows (no tensor-core scorer for e4m3 keys) and NaN
    # codes in every slot no row may see
    w = W.fp8_index(W.custom(62, q_lens=[70, 1], seq_lens=[3000, 300], hq=8, di=64, topk=4,
                             fill_unused_nan=True), seed=63)
    _, sep, fused = run_steps(msa, w)
    check_against_oracle(orc, w, sep, fused)


def test_garbage_past_the_end_is_ignored(msa, orc):
    for kv in (W.KV_BF16, W.KV_FP8):
        w = W.custom(53, q_lens=[1, 3, 1], seq_lens=[1000, 517, 129], hq=16, di=128, topk=4,
                     kv_dtype=kv, with_sink=True, fill_unused_nan=True)
        _, sep, fused = run_steps(msa, w)
        check_against_oracle(orc, w, sep, fused)
        assert np.all(np.isfinite(sep["out"])) and np.all(np.isfinite(sep["lse"]))


@pytest.mark.parametrize("hi,di", [(1, 64), (2, 64), (1, 128)])
def test_index_head_variants(msa, orc, hi, di):
    w = W.custom(54, q_lens=[1, 4, 2], seq_lens=[3000, 1500, 260], hq=16, di=di, hi=hi, topk=4)
    _, sep, fused = run_steps(msa, w)
    check_against_oracle(orc, w, sep, fused)


@pytest.mark.parametrize("hq", [1, 8, 12, 16])
def test_query_head_counts(msa, orc, hq):
    w = W.custom(55, q_lens=[1, 2], seq_lens=[2500, 900], hq=hq, di=128, topk=4, with_sink=True,
                 kv_dtype=W.KV_FP8, scale_mode=W.SCALE_SCALAR)
    _, sep, fused = run_steps(msa, w)
    check_against_oracle(orc, w, sep, fused)


def test_many_rows_single_split(msa, orc):
    # enough rows that each row runs as a single split (no cross-CTA merge)
    w = W.custom(56, q_lens=[300, 200], seq_lens=[2500, 1200], hq=16, di=128, topk=8)
    _, sep, fused = run_steps(msa, w)
    check_against_oracle(orc, w, sep, fused)


@pytest.mark.parametrize("long_seq,topk", [(20_000, 8), (60_000, 8), (120_000, 8),
                                           (20_000, 32), (20_000, 48)])
def test_many_rows_warp_topk(msa, orc, long_seq, topk):
    # >= 512 rows take the warp-per-row top-k; the longest request sets the
    # block-table width (157 / 469 / 938 blocks: 8, 16 or 32 keys per lane).
    # With 8 keys a lane, k <= 32 is found by extraction and k = 48 by the
    # bit search.  Index values in {-1, 0, 1} make many blocks tie at the
    # threshold; an empty request, a request with a page outside the pool
    # and rows that see fewer blocks than k are in the same batch.
    q_lens = [400, 0, 100, 6, 10, 3]
    seq = [2600, 50, 1500, long_seq, 9000, 300]
    w = W.custom(61, q_lens=q_lens, seq_lens=seq, hq=8, di=64, idx_range=1, topk=topk,
                 kv_dtype=W.KV_BF16, with_sink=True)
    bt = w.block_table.copy()
    bt[2, 3] = w.num_pages + 1
    w.block_table = bt
    c, sep, fused = run_steps(msa, w)
    ref = orc.decode(w)
    assert sep["status"] == ref["status"] == msa.MSA_DEV_BAD_PAGE
    for key in ("topk_idx", "tbl", "sparse_len"):
        assert np.array_equal(sep[key], ref[key]), key
    assert_attn_close(sep["out"], sep["lse"], ref["out"], ref["lse"])
    check_fused(w, sep, fused, ref)


@pytest.mark.parametrize("topk", [4, 16, 32, 48])
def test_warp_topk_crafted_scores(msa, orc, topk):
    # the warp-per-row top-k (>= 512 rows) on scores written directly: NaN,
    # -inf, +inf and a few repeated values, so the k-th largest key sits in
    # a run of ties or among NaNs (NaN ranks below -inf); rows of the second
    # request see fewer blocks than k.  k <= 32 takes the extraction, 48 the
    # bit search; the selection, the table and the length equal the
    # oracle's bit for bit.
    w = W.custom(66, q_lens=[600, 20], seq_lens=[20000, 300], hq=8, di=64, topk=topk,
                 kv_dtype=W.KV_BF16)
    c = msa.DeviceCase(w)
    rng = np.random.default_rng(topk)
    vals = np.array([np.nan, -np.inf, np.inf, 0.0, 1.0, 2.0, -1.0, 3.5], np.float32)
    sc = vals[rng.integers(0, len(vals), size=tuple(c.scores.shape))]
    sc[::7] = np.nan  # rows that are mostly NaN: the k-th key is a NaN's
    sc[::7, :5] = 1.0
    c.scores.copy_(torch.from_numpy(sc))
    c.topk_build_table()
    res = c.fetch()
    ref_idx, ref_tbl, ref_len, st = orc.topk_build_table(orc.Batch.of(w), sc, topk,
                                                         tbl_stride=c.tbl_stride)
    assert st == 0 and res["status"] == 0
    assert np.array_equal(res["topk_idx"], ref_idx)
    assert np.array_equal(res["tbl"], ref_tbl)
    assert np.array_equal(res["sparse_len"], ref_len)


# ------------------------------------------------ block-major prefill path

@pytest.mark.parametrize("hq,scale,sink", [(16, W.SCALE_NONE, False), (16, W.SCALE_SCALAR, True),
                                           (8, W.SCALE_NONE, True), (12, W.SCALE_SCALAR, False)])
def test_prefill_path_mixed_batch(msa, orc, hq, scale, sink):
    # requests of 100 and 64 rows take the prefill attention in the fused
    # call, those of 1, 3 and 63 rows the split-K decode attention; contexts
    # end inside a block (partial last blocks) and on a block boundary
    q_lens = [100, 1, 3, 64, 63, 130]
    seq = [5000, 3000, 700, 64 + 256, 2000, 9000 + 77]
    w = W.custom(63 + hq, q_lens=q_lens, seq_lens=seq, hq=hq, di=128, topk=8,
                 kv_dtype=W.KV_BF16, scale_mode=scale, with_sink=sink)
    assert prefill_rows(w).sum() == 100 + 64 + 130
    _, sep, fused = run_steps(msa, w)
    check_against_oracle(orc, w, sep, fused)


def test_prefill_path_all_blocks_and_garbage(msa, orc):
    # top-k covering every block (short contexts), a request of a single
    # partial block, NaN in every slot past each request's end
    w = W.custom(70, q_lens=[90, 70, 65], seq_lens=[700, 70, 1000], hq=16, di=128, topk=16,
                 kv_dtype=W.KV_BF16, with_sink=True, fill_unused_nan=True)
    _, sep, fused = run_steps(msa, w)
    check_against_oracle(orc, w, sep, fused)
    assert np.all(np.isfinite(fused["out"])) and np.all(np.isfinite(fused["lse"]))


def test_prefill_path_poisoned_request(msa, orc):
    # a request of the prefill path with a page outside the pool: its rows
    # are empty rows (O = 0, LSE = sink); the other requests are unaffected
    w = W.custom(71, q_lens=[80, 120, 2], seq_lens=[3000, 4000, 900], hq=16, di=128, topk=8,
                 kv_dtype=W.KV_BF16, with_sink=True)
    bt = w.block_table.copy()
    bt[0, 5] = w.num_pages + 3
    w.block_table = bt
    _, sep, fused = run_steps(msa, w)
    ref = check_against_oracle(orc, w, sep, fused)
    assert ref["status"] == msa.MSA_DEV_BAD_PAGE
    assert np.all(fused["out"][:80] == 0)
    np.testing.assert_allclose(fused["lse"][:80], np.tile(w.sinks, (80, 1)), atol=1e-6)


def test_prefill_path_repeated_calls(msa):
    # the list counters and plan are rebuilt on every call: the same inputs
    # give bit-identical results call after call (and across a call with
    # another batch shape on the same workspace in between)
    w = W.chunked_prefill(seed=16, context=3000, new_tokens=500, reqs=3)
    c = msa.DeviceCase(w)
    c.decode()
    a = c.fetch()
    other = W.custom(72, q_lens=[200, 1], seq_lens=[900, 400], hq=16, di=128, topk=16)
    c2 = msa.DeviceCase(other)
    c2.workspace = c.workspace[: c2.workspace.numel()] if c.workspace.numel() >= c2.workspace.numel() \
        else c2.workspace
    c2.decode()
    for _ in range(2):
        c.decode()
        b = c.fetch()
        for key in ("topk_idx", "tbl", "sparse_len", "out", "lse"):
            assert np.array_equal(a[key], b[key], equal_nan=True), key
        assert b["status"] == 0


def test_prefill_only_batch_skips_decode_attention(msa, orc):
    # every request brings >= 64 rows and the batch says so (min_q_len):
    # msa_decode launches neither the CUDA-core scorer nor the split-K decode
    # attention, and its results equal those of the call without the hint
    # bit for bit, and the oracle's
    w = W.chunked_prefill(seed=17, context=1500, new_tokens=200, reqs=2)
    runs = {}
    for hint in (True, False):
        c = msa.DeviceCase(w, min_q_len_hint=hint)
        tr = msa.make_trace()
        c.decode(trace=tr)
        runs[hint] = (c.fetch(), tr.kernels)
    (got, k_hint), (plain, k_plain) = runs[True], runs[False]
    assert k_hint == k_plain - 2
    for key in ("topk_idx", "tbl", "sparse_len", "out", "lse"):
        assert np.array_equal(got[key], plain[key], equal_nan=True), key
    ref = orc.decode(w)
    assert got["status"] == ref["status"] == 0
    for key in ("topk_idx", "tbl", "sparse_len"):
        assert np.array_equal(got[key], ref[key]), key
    assert_attn_close(got["out"], got["lse"], ref["out"], ref["lse"])


def test_min_q_len_hint_with_fp8_kv(msa, orc):
    # every request has >= 64 rows (hint given) but the KV is FP8, which the
    # block-major path does not take: the tensor-core scorer alone scores
    # (the CUDA-core one is not launched) and the split-K decode attention
    # still serves every row
    w = W.custom(75, q_lens=[96, 70], seq_lens=[2500, 1800], hq=16, di=128, topk=8,
                 kv_dtype=W.KV_FP8, scale_mode=W.SCALE_PER_TOKEN_HEAD, with_sink=True)
    c = msa.DeviceCase(w)
    assert c.min_q_len == 70
    tr = msa.make_trace()
    c.decode(trace=tr)
    got = c.fetch()
    assert tr.kernels == 3  # tensor-core scorer, top-k, decode attention
    ref = orc.decode(w)
    assert got["status"] == ref["status"] == 0
    for key in ("topk_idx", "tbl", "sparse_len"):
        assert np.array_equal(got[key], ref[key]), key
    assert_attn_close(got["out"], got["lse"], ref["out"], ref["lse"])


def test_min_q_len_hint_violated(msa, orc):
    # a bound of 64 rows per request on a batch that also holds a 3-row and a
    # 0-row request: both are poisoned (MSA_DEV_MALFORMED; the 3 rows are
    # empty rows, written by the prefill merge since no decode attention
    # runs); the prefill request is unaffected
    w = W.custom(73, q_lens=[100, 3, 0], seq_lens=[3000, 900, 500], hq=16, di=128, topk=8,
                 kv_dtype=W.KV_BF16, with_sink=True)
    c = msa.DeviceCase(w, min_q_len_hint=64)
    c.decode()
    got = c.fetch()
    ref = orc.decode(w)
    assert ref["status"] == 0 and got["status"] == msa.MSA_DEV_MALFORMED
    pre = slice(0, 100)
    for key in ("topk_idx", "tbl", "sparse_len"):
        assert np.array_equal(got[key][pre], ref[key][pre]), key
    assert_attn_close(got["out"][pre], got["lse"][pre], ref["out"][pre], ref["lse"][pre])
    assert np.all(got["topk_idx"][100:] == -1) and np.all(got["sparse_len"][100:] == 0)
    assert np.all(got["out"][100:] == 0)
    np.testing.assert_allclose(got["lse"][100:], np.tile(w.sinks, (3, 1)), atol=1e-6)


def test_prefill_only_batch_poisoned_request(msa, orc):
    # the prefill-only launch (min_q_len hint) with a page outside the pool
    # in request 0: its rows are empty rows, the status bit is reported
    # without the CUDA-core scorer, request 1 is unaffected
    w = W.custom(74, q_lens=[80, 120], seq_lens=[3000, 4000], hq=16, di=128, topk=8,
                 kv_dtype=W.KV_BF16, with_sink=True)
    bt = w.block_table.copy()
    bt[0, 5] = w.num_pages + 3
    w.block_table = bt
    c = msa.DeviceCase(w)
    assert c.min_q_len == 80
    c.decode()
    got = c.fetch()
    ref = orc.decode(w)
    assert got["status"] == ref["status"] == msa.MSA_DEV_BAD_PAGE
    for key in ("topk_idx", "tbl", "sparse_len"):
        assert np.array_equal(got[key], ref[key]), key
    assert_attn_close(got["out"], got["lse"], ref["out"], ref["lse"])
    assert np.all(got["out"][:80] == 0)
    np.testing.assert_allclose(got["lse"][:80], np.tile(w.sinks, (80, 1)), atol=1e-6)


def test_poisoned_requests_match_oracle(msa, orc):
    w = W.custom(57, q_lens=[1, 2, 1, 1], seq_lens=[900, 700, 400, 300], hq=16, di=128, topk=2,
                 with_sink=True)
    bt = w.block_table.copy()
    bt[1, 2] = w.num_pages + 5  # request 1 addresses a page outside the pool
    w.block_table = bt
    ctx = w.context_lens.copy()
    ctx[2] -= 1                 # request 2: context + q_len != seq_len
    w.context_lens = ctx
    _, sep, fused = run_steps(msa, w)
    ref = orc.decode(w)
    assert sep["status"] == ref["status"] == (msa.MSA_DEV_BAD_PAGE | msa.MSA_DEV_BAD_LEN)
    for key in ("topk_idx", "tbl", "sparse_len"):
        assert np.array_equal(sep[key], ref[key])
    assert_attn_close(sep["out"], sep["lse"], ref["out"], ref["lse"])
    for r in (1, 2, 3):  # poisoned rows are empty rows: O = 0, LSE = sink
        assert np.all(sep["out"][r] == 0)
        np.testing.assert_allclose(sep["lse"][r], w.sinks, atol=1e-6)


def test_malformed_batch_sets_status(msa):
    w = W.custom(58, q_lens=[1, 1], seq_lens=[300, 200], hq=16, di=128, topk=2)
    cu = w.cu_seqlens_q.copy()
    cu[2] = 1  # rows are not tiled: cu_seqlens_q decreases and stops short of num_rows
    w.cu_seqlens_q = cu
    c = msa.DeviceCase(w)
    c.decode()
    res = c.fetch()
    assert res["status"] & msa.MSA_DEV_MALFORMED
    assert np.all(res["sparse_len"] == 0) and np.all(res["out"] == 0)


def test_standalone_attention_bad_table(msa, orc):
    w = W.custom(59, q_lens=[1, 1, 1], seq_lens=[600, 600, 600], hq=16, di=128, topk=4,
                 with_sink=True)
    c = msa.DeviceCase(w)
    c.index_score()
    c.topk_build_table()
    c.tbl[1, 3] = 8 * w.num_pages  # first id past the page-16 pool
    c.sparse_len[2] = 16 * c.tbl_stride + 1
    c.sparse_paged_attn()
    res = c.fetch()
    assert res["status"] == msa.MSA_DEV_BAD_TABLE
    ref_o, ref_l, st = orc.sparse_attn(w.q, w.k_cache, w.v_cache, w.kv_dtype, res["tbl"],
                                       res["sparse_len"], sinks=w.sinks,
                                       softmax_scale=w.softmax_scale, num_pages16=8 * w.num_pages)
    assert st == orc.BAD_TABLE
    assert_attn_close(res["out"], res["lse"], ref_o, ref_l)
    assert np.all(res["out"][1:] == 0)


def test_page_permutation_invariance(msa):
    w = W.custom(60, q_lens=[1, 4, 1], seq_lens=[6000, 3000, 900], hq=16, di=128, topk=8,
                 kv_dtype=W.KV_FP8, scale_mode=W.SCALE_PER_TOKEN_HEAD, with_sink=True)
    _, a, _ = run_steps(msa, w)
    perm = np.random.default_rng(1).permutation(w.num_pages)
    inv = np.argsort(perm)
    w.idx_k, w.k_cache, w.v_cache = w.idx_k[perm], w.k_cache[perm], w.v_cache[perm]
    w.k_scale, w.v_scale = w.k_scale[perm], w.v_scale[perm]
    bt = w.block_table.copy()
    bt[bt >= 0] = inv[bt[bt >= 0]]
    w.block_table = bt
    _, b, _ = run_steps(msa, w)
    for key in ("topk_idx", "sparse_len", "out", "lse"):
        assert np.array_equal(a[key], b[key]), key


def test_graph_capture_and_replay(msa):
    w = W.custom(61, q_lens=[1, 4, 1, 1], seq_lens=[7000, 3000, 1200, 260], hq=16, di=128,
                 topk=8, kv_dtype=W.KV_FP8, scale_mode=W.SCALE_SCALAR, with_sink=True)
    c = msa.DeviceCase(w)
    c.decode()
    eager = c.fetch()
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        c.decode(stream=s)  # capture fails if the call syncs or copies to/from the host
    for _ in range(3):
        c.out.zero_()
        c.lse.zero_()
        g.replay()
        rep = c.fetch()
        for key in ("topk_idx", "tbl", "sparse_len", "out", "lse"):
            assert np.array_equal(rep[key], eager[key]), key


def test_repeated_calls_are_identical(msa):
    w = W.custom(62, q_lens=[1, 1], seq_lens=[20000, 9000], hq=16, di=128, topk=16,
                 kv_dtype=W.KV_FP8, scale_mode=W.SCALE_PER_TOKEN_HEAD, with_sink=True)
    c = msa.DeviceCase(w)
    c.decode()
    a = c.fetch()
    for _ in range(3):
        c.sparse_paged_attn()  # separate workspace, counters must be back at 0
        c.decode()
    b = c.fetch()
    for key in ("out", "lse", "tbl"):
        assert np.array_equal(a[key], b[key])


def test_packed_step_inputs(msa):
    # per-step inputs and outputs moved into one buffer each (one copy per
    # step each way): the same results, and a refreshed input buffer is used
    w = W.custom(63, q_lens=[1, 3, 2], seq_lens=[7000, 3000, 900], hq=16, di=128, topk=8,
                 kv_dtype=W.KV_FP8, scale_mode=W.SCALE_SCALAR, with_sink=True)
    c = msa.DeviceCase(w)
    c.decode()
    a = c.fetch()
    assert c.step_inputs is None
    c.pack_step_inputs()
    host = c.step_inputs.cpu()
    c.step_inputs.zero_()
    c.step_inputs.copy_(host)
    c.decode()
    b = c.fetch()
    for key in ("out", "lse", "tbl", "topk_idx", "sparse_len"):
        assert np.array_equal(a[key], b[key]), key
    assert b["status"] == 0


def test_two_step_buffer_sets(msa):
    # two sets of step buffers with their own argument structs over the same
    # pools and workspace (the pipelined end-to-end loop): each set gives the
    # results of the plain call, and steps alternating sets on two streams'
    # copies stay intact
    w = W.custom(64, q_lens=[1, 3, 2], seq_lens=[7000, 3000, 900], hq=16, di=128, topk=8,
                 kv_dtype=W.KV_FP8, scale_mode=W.SCALE_SCALAR, with_sink=True)
    c = msa.DeviceCase(w)
    c.decode()
    a = c.fetch()
    c.pack_step_inputs(sets=2)
    for b in (1, 0, 1):
        c.use_step_set(b)
        c.step_outputs.zero_()
        c.decode()
        got = c.fetch()
        for key in ("out", "lse", "tbl", "topk_idx", "sparse_len"):
            assert np.array_equal(a[key], got[key]), (b, key)
    assert c._sets[0]["step_inputs"].data_ptr() != c._sets[1]["step_inputs"].data_ptr()


def test_every_call_rescores_every_block(msa, orc):
    # New queries on later calls must change every block score of the fused
    # path (stale workspace scores from the first call would show up as wrong
    # selections), on 20 requests of different lengths.
    import dataclasses
    w = W.custom(63, q_lens=[1] * 20, seq_lens=[3000 + 700 * i for i in range(20)], hq=16,
                 di=128, topk=8, kv_dtype=W.KV_FP8, scale_mode=W.SCALE_SCALAR, with_sink=True)
    c = msa.DeviceCase(w)
    c.decode()
    ref = orc.decode(w, topk=w.topk)
    assert np.array_equal(c.fetch()["topk_idx"], ref["topk_idx"])
    rng = np.random.default_rng(64)
    w2 = dataclasses.replace(w, idx_q=W._int_bf16(rng.integers(-3, 4, size=w.idx_q.shape,
                                                               dtype=np.int8)))
    c.idx_q.copy_(torch.from_numpy(w2.idx_q.view(np.int16)).to(c.idx_q.device).view(c.idx_q.dtype))
    for _ in range(2):
        c.decode()
        got = c.fetch()
        ref2 = orc.decode(w2, topk=w.topk)
        assert np.array_equal(got["topk_idx"], ref2["topk_idx"])
        assert np.array_equal(got["tbl"], ref2["tbl"])
        assert_attn_close(got["out"], got["lse"], ref2["out"], ref2["lse"])


def test_outputs_stay_inside_their_rows(msa):
    """Sentinel guard regions around every output stay untouched."""
    w = W.custom(63, q_lens=[1, 3], seq_lens=[3000, 700], hq=16, di=128, topk=4, with_sink=True)
    c = msa.DeviceCase(w)
    G = 4096
    N, k, ts = w.num_rows, c.topk, c.tbl_stride

    def guarded(n, dtype, fill):
        buf = torch.full((2 * G + n,), fill, dtype=dtype, device="cuda")
        return buf, buf[G:G + n]

    tb, tbl = guarded(N * ts, torch.int32, -7)
    kb, kidx = guarded(N * k, torch.int32, -7)
    lb, slen = guarded(N, torch.int32, -7)
    ob, out = guarded(N * 16 * 128, torch.bfloat16, 3.0)
    eb, lse = guarded(N * 16, torch.float32, 3.0)
    c.attn = msa.make_attn_args(c.q, c.k, c.v, w.kv_dtype, w.num_pages, out.view(N, 16, 128),
                                lse.view(N, 16), sinks=c.sinks, softmax_scale=w.softmax_scale)
    msa.msa_decode(c.batch, c.idx_q, c.index, k, c.attn, kidx, tbl, ts, slen, c.workspace,
                   c.status)
    torch.cuda.synchronize()
    for buf, n, fill in ((tb, N * ts, -7), (kb, N * k, -7), (lb, N, -7), (ob, N * 2048, 3.0),
                         (eb, N * 16, 3.0)):
        assert torch.all(buf[:G] == fill) and torch.all(buf[G + n:] == fill)
    assert int(c.status.item()) == 0


def test_empty_batch_is_a_no_op(msa):
    dev = "cuda"
    z = torch.zeros(1, dtype=torch.int32, device=dev)
    bt = torch.zeros((0, 1), dtype=torch.int32, device=dev)
    b = msa.make_batch(z, z, torch.zeros(0, dtype=torch.int32, device=dev), bt, 0, 0)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    scores = torch.zeros((1, 1), dtype=torch.float32, device=dev)
    q = torch.zeros((1, 1, 64), dtype=torch.bfloat16, device=dev)
    kc = torch.zeros((1, 128, 1, 64), dtype=torch.bfloat16, device=dev)
    msa.msa_index_score(b, q, msa.make_index_cache(kc), scores, 1, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
