"""Pins for the CPU oracle: checks against facts that do not come from the
oracle itself -- the FP8 format definition, hand-worked examples, closed
forms, brute force on tiny inputs, library routines (numpy matmul, torch
SDPA in float64) and invariances.  A plausible slip anywhere in the oracle
(a dropped sink term, a wrong causal bound, a transposed operand, a wrong
tie rule) fails at least one of these.

Definitions cited (MiniMax-M3 sparse-attention pages): vLLM PR 47287 page
"Implementation breakdown" items 2-3 (page-16 table, FP8 scales); PR 54682
page "Implementation breakdown" item 1 (top-k fused with the page-16 table
and context length); PR 54404 page "Features and motivation" / "Key source
snippets" (sinks, natural-log LSE); PR 56170 page "Key source snippets"
(128-token blocks, cu_seqlens).
"""
import dataclasses
import itertools
import math
import os

import numpy as np
import pytest
import torch

import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
NEG_INF = -np.inf


# ---------------------------------------------------------------- formats

def test_fp8_golden_values(orc):
    with open(os.path.join(GOLDEN, "fp8_e4m3_values.txt")) as f:
        rows = [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]
    assert len(rows) >= 20
    for code, val in rows:
        got = orc.fp8_e4m3_value(int(code, 16))
        if val == "nan":
            assert math.isnan(got), code
        else:
            assert got == float(val) and math.copysign(1, got) == math.copysign(1, float(val)), code


def test_fp8_all_codes_match_torch(orc):
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([orc.fp8_e4m3_value(c) for c in range(256)])
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert np.array_equal(ref[~nan], got[~nan])


def test_bf16_values_match_torch(orc):
    rng = np.random.default_rng(0)
    bits = rng.integers(0, 1 << 16, size=2000, dtype=np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([orc.bf16_value(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert np.array_equal(ref[~nan], got[~nan])


# --------------------------------------------------------------- geometry

def _batch(orc, q_lens, seq_lens, bt, num_pages, context=None):
    q_lens = np.asarray(q_lens)
    seq_lens = np.asarray(seq_lens)
    cu_q = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    cu_k = np.concatenate([[0], np.cumsum(seq_lens)]).astype(np.int32)
    ctx = (seq_lens - q_lens) if context is None else np.asarray(context)
    return orc.Batch(cu_q, cu_k, ctx, np.asarray(bt, np.int32), num_pages)


def test_geometry_speculative_rows(orc):
    # 4 speculative rows of a request of length L sit at L-4 .. L-1
    b = _batch(orc, [4, 1], [258, 128], [[0, 1, 2], [3, -1, -1]], 4)
    g = orc.row_geometry(b)
    assert g["status"] == 0
    assert list(g["req"]) == [0, 0, 0, 0, 1]
    assert list(g["pos"]) == [254, 255, 256, 257, 127]
    assert list(g["nb"]) == [2, 2, 3, 3, 1]
    assert list(g["ok"]) == [1, 1, 1, 1, 1]


def test_geometry_errors(orc):
    # length mismatch (context + q_len != seq_len)
    b = _batch(orc, [1], [200], [[0, 1]], 2, context=[150])
    g = orc.row_geometry(b)
    assert g["status"] == orc.BAD_LEN and list(g["ok"]) == [0]
    # page id out of range in a block the request covers
    b = _batch(orc, [1], [200], [[0, 9]], 2)
    g = orc.row_geometry(b)
    assert g["status"] == orc.BAD_PAGE and list(g["ok"]) == [2]
    # an out-of-range id beyond the request's blocks is never looked at
    b = _batch(orc, [1], [100], [[0, 9]], 2)
    assert orc.row_geometry(b)["status"] == 0
    # sequence longer than the block table can address
    b = _batch(orc, [1], [300], [[0, 1]], 4)
    assert orc.row_geometry(b)["status"] == orc.MALFORMED
    # cu_seqlens_q that does not tile the rows
    b = orc.Batch(np.array([0, 2], np.int32), np.array([0, 10], np.int32),
                  np.array([8], np.int32), np.zeros((1, 1), np.int32), 1)
    b.s.num_rows = 3
    b.num_rows = 3
    assert orc.row_geometry(b)["status"] == orc.MALFORMED


# ------------------------------------------------------------ index score

def _planted_index_case():
    """One request, L = 1000 (8 blocks, last 104 tokens), Di = 64, q = e_0.
    Every index-K vector is 0 except dim 0 of a few planted tokens, so block
    b's score is max(0, planted values of b that sit at t <= 999)."""
    L, di = 1000, 64
    perm = np.array([5, 2, 7, 0, 6, 1, 3, 4], np.int32)
    kf = np.zeros((8, 128, 1, di), np.float32)
    planted = {0: [(3, 4.0)], 1: [(127, 9.0), (5, 2.0)], 2: [(0, -5.0)],  # block 2: all <= 0 -> 0
               3: [(64, 1.0)], 4: [], 5: [(100, 7.0)], 6: [(1, 3.0)],
               7: [(103, 6.0), (104, 50.0), (127, 60.0)]}  # 104+ lie past the last token
    for blk, items in planted.items():
        for tl, v in items:
            kf[perm[blk], tl, 0, 0] = v
    expected = np.array([4, 9, 0, 1, 0, 7, 3, 6], np.float32)
    qf = np.zeros((1, 1, di), np.float32)
    qf[0, 0, 0] = 1.0
    return L, perm, W.bf16_bits(qf), W.bf16_bits(kf), expected


def test_index_score_planted(orc):
    L, perm, q, k, expected = _planted_index_case()
    b = _batch(orc, [1], [L], perm[None, :], 8)
    scores, st = orc.index_score(b, q, k, score_stride=10)
    assert st == 0
    assert np.array_equal(scores[0, :8], expected)
    assert np.all(scores[0, 8:] == NEG_INF)


def test_index_score_planted_causal_rows(orc):
    # three rows at positions 997..999: the token at 999 (block 7, slot 103)
    # is visible only to the last row
    L, perm, q, k, _ = _planted_index_case()
    b = _batch(orc, [3], [L], perm[None, :], 8)
    scores, _ = orc.index_score(b, np.repeat(q, 3, axis=0), k)
    assert list(scores[:, 7]) == [0.0, 0.0, 6.0]


def _dense_index_scores(w, k_values=None):
    """numpy reference: gather each request's index-K through the block table,
    matmul in float64, mask future tokens, max within each 128-token block.
    k_values: the keys as floats (default: w.idx_k as bf16 bits)."""
    to_f = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).double().numpy()
    qf = to_f(w.idx_q)
    kf = to_f(w.idx_k) if k_values is None else k_values
    out = np.full((w.num_rows, w.bt_stride), NEG_INF)
    for r in range(w.num_reqs):
        L = int(w.seq_lens[r])
        nb = -(-L // 128)
        pages = w.block_table[r, :nb]
        K = kf[pages].reshape(nb * 128, w.index_heads, w.index_dim)
        for j in range(int(w.q_lens[r])):
            row = int(w.cu_seqlens_q[r]) + j
            pos = int(w.context_lens[r]) + j
            s = np.einsum("hd,thd->th", qf[row], K).max(axis=1)  # max over index heads
            s[pos + 1:] = NEG_INF
            out[row, : -(-(pos + 1) // 128)] = s.reshape(nb, 128).max(axis=1)[: -(-(pos + 1) // 128)]
    return out


@pytest.mark.parametrize("hi,di", [(1, 64), (2, 64), (1, 128)])
def test_index_score_matches_matmul(orc, hi, di):
    w = W.custom(11, q_lens=[1, 4, 3], seq_lens=[700, 1029, 130], hq=4, di=di, hi=hi, topk=3)
    b = orc.Batch.of(w)
    scores, st = orc.index_score(b, w.idx_q, w.idx_k)
    assert st == 0
    ref = _dense_index_scores(w)
    assert np.array_equal(scores.astype(np.float64), ref)


def _fp8_float(codes):
    # an e4m3 decoder independent of the oracle's: torch's float8_e4m3fn
    t = torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn)
    return t.to(torch.float64).numpy()


@pytest.mark.parametrize("hi,di", [(1, 64), (2, 64), (1, 128)])
def test_fp8_index_score_matches_matmul(orc, hi, di):
    # e4m3 index-K with per-token scales: s_t * (q . k_t), max over the block's
    # visible tokens and heads, checked against a matmul over torch-decoded keys
    w = W.fp8_index(W.custom(13, q_lens=[1, 4, 3], seq_lens=[700, 1029, 130], hq=4, di=di,
                             hi=hi, topk=3), seed=14)
    scores, st = orc.index_score(orc.Batch.of(w), w.idx_q, w.idx_k, fp8=True,
                                 k_scale=w.idx_k_scale)
    assert st == 0
    deq = _fp8_float(w.idx_k) * w.idx_k_scale[..., None].astype(np.float64)
    ref = _dense_index_scores(w, k_values=deq)
    assert np.array_equal(scores.astype(np.float64), ref)


def test_fp8_index_without_scales_equals_bf16_index(orc):
    # the integer index values are exact in e4m3, so unscaled FP8 keys score
    # exactly as the bf16 keys they were encoded from
    w = W.custom(15, q_lens=[2, 1], seq_lens=[2000, 333], hq=4, di=128, topk=4)
    w8 = W.fp8_index(w, seed=16, scaled=False)
    b = orc.Batch.of(w)
    s16, _ = orc.index_score(b, w.idx_q, w.idx_k)
    s8, _ = orc.index_score(b, w8.idx_q, w8.idx_k, fp8=True, k_scale=None)
    assert np.array_equal(s16, s8, equal_nan=True)
    # doubling every scale doubles every finite score
    w8s = W.fp8_index(w, seed=17)
    a, _ = orc.index_score(b, w8s.idx_q, w8s.idx_k, fp8=True, k_scale=w8s.idx_k_scale)
    d, _ = orc.index_score(b, w8s.idx_q, w8s.idx_k, fp8=True, k_scale=2 * w8s.idx_k_scale)
    fin = np.isfinite(a)
    assert np.array_equal(2 * a[fin], d[fin]) and np.array_equal(np.isfinite(d), fin)


def test_index_score_ignores_garbage(orc):
    # NaN in unused slots and pages must not reach any score
    w = W.custom(12, q_lens=[1, 2], seq_lens=[300, 513], hq=4, di=64, topk=2, fill_unused_nan=True)
    scores, st = orc.index_score(orc.Batch.of(w), w.idx_q, w.idx_k)
    g = orc.row_geometry(orc.Batch.of(w))
    for r in range(w.num_rows):
        assert np.all(np.isfinite(scores[r, : g["nb"][r]]))


# ------------------------------------------------------------------ top-k

def _one_row_batch(orc, L, nblocks, num_pages=None):
    bt = np.arange(nblocks, dtype=np.int32)[None, :]
    return _batch(orc, [1], [L], bt, num_pages or nblocks)


def test_topk_brute_force_with_ties(orc):
    """For tiny rows, enumerate every subset of size min(k, n) and keep the
    ones where each selected block beats each unselected block under
    (higher score, then lower index).  Exactly one subset qualifies; the
    oracle must return it in ascending order."""
    rng = np.random.default_rng(5)
    for trial in range(150):
        n = int(rng.integers(1, 9))
        k = int(rng.integers(1, 7))
        L = 128 * (n - 1) + int(rng.integers(1, 129))
        sc = rng.integers(0, 3, size=n).astype(np.float32)  # heavy ties
        b = _one_row_batch(orc, L, n)
        sel, tbl, slen, st = orc.topk_build_table(b, sc[None, :], k)
        m = min(k, n)
        beats = lambda a, c: sc[a] > sc[c] or (sc[a] == sc[c] and a < c)
        good = [S for S in itertools.combinations(range(n), m)
                if all(beats(a, c) for a in S for c in set(range(n)) - set(S))]
        assert len(good) == 1
        assert list(sel[0, :m]) == list(good[0])
        assert np.all(sel[0, m:] == -1)


def test_topk_nan_ranks_last(orc):
    sc = np.array([[np.nan, 1.0, np.nan, -np.inf, 0.5]], np.float32)
    b = _one_row_batch(orc, 5 * 128, 5)
    sel, *_ = orc.topk_build_table(b, sc, 3)
    assert list(sel[0]) == [1, 3, 4]
    sel, *_ = orc.topk_build_table(b, sc, 4)
    assert list(sel[0]) == [0, 1, 3, 4]


def test_table_golden_example(orc):
    with open(os.path.join(GOLDEN, "table_example.txt")) as f:
        kv = {ln.split()[0]: [int(x) for x in ln.split()[1:]]
              for ln in f if ln.strip() and not ln.startswith("#")}
    L = kv["L"][0]
    bt = np.array(kv["block_table"], np.int32)[None, :]
    b = _batch(orc, [1], [L], bt, 8)
    sc = np.array([[5, 7, 3, 3, 3, 7, 5, 7]], np.float32)  # ties: 5 at blocks 0 and 6 -> 0 wins
    sel, tbl, slen, st = orc.topk_build_table(b, sc, 4, tbl_stride=40)
    assert st == 0
    assert list(sel[0]) == kv["selected"]
    assert list(tbl[0]) == kv["table"]
    assert int(slen[0]) == kv["sparse_len"][0]


def test_table_all_blocks_closed_form(orc):
    # k >= number of blocks: every block is selected, the length is the whole
    # visible length and the table is the block table expanded in order
    w = W.custom(13, q_lens=[1, 4], seq_lens=[1000, 385], hq=4, di=64, topk=8)
    b = orc.Batch.of(w)
    scores, _ = orc.index_score(b, w.idx_q, w.idx_k)
    sel, tbl, slen, st = orc.topk_build_table(b, scores, 8, tbl_stride=70)
    g = orc.row_geometry(b)
    for r in range(w.num_rows):
        L = g["pos"][r] + 1
        assert slen[r] == L
        pages = w.block_table[g["req"][r]]
        exp = []
        for blk in range(-(-L // 128)):
            sub = -(-min(128, L - 128 * blk) // 16)
            exp += [8 * int(pages[blk]) + j for j in range(sub)] + [0] * (8 - sub)
        exp += [0] * (70 - len(exp))
        assert list(tbl[r]) == exp


def test_poisoned_rows_get_empty_tables(orc):
    bt = np.array([[0, 7]], np.int32)  # page 7 is outside a 2-page pool
    b = _batch(orc, [1], [200], bt, 2)
    sc = np.zeros((1, 2), np.float32)
    sel, tbl, slen, st = orc.topk_build_table(b, sc, 2)
    assert st == orc.BAD_PAGE
    assert np.all(sel == -1) and np.all(tbl == 0) and slen[0] == 0


# -------------------------------------------------------------- attention

def _f64(a, kv_dtype):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if kv_dtype == W.KV_FP8:
        return t.view(torch.float8_e4m3fn).double().numpy()
    return t.view(torch.int16).view(torch.bfloat16).double().numpy()


def _sdpa_reference(w):
    """torch SDPA (float64) over the dense visible tokens of each row, with the
    dequant scales applied to K and V and the sink as one extra key whose
    logit is the sink and whose value is zero.  LSE via torch.logsumexp."""
    qf = _f64(w.q, W.KV_BF16)
    kf = _f64(w.k_cache, w.kv_dtype)
    vf = _f64(w.v_cache, w.kv_dtype)
    P = w.num_pages
    if w.scale_mode == W.SCALE_SCALAR:
        kf = kf * float(w.k_scale[0])
        vf = vf * float(w.v_scale[0])
    elif w.scale_mode == W.SCALE_PER_TOKEN_HEAD:
        kf = kf * w.k_scale.reshape(P, 128, w.hkv, 1)
        vf = vf * w.v_scale.reshape(P, 128, w.hkv, 1)
    out = np.zeros((w.num_rows, w.hq, w.head_dim))
    lse = np.zeros((w.num_rows, w.hq))
    group = w.hq // w.hkv
    for r in range(w.num_reqs):
        for j in range(int(w.q_lens[r])):
            row = int(w.cu_seqlens_q[r]) + j
            L = int(w.context_lens[r]) + j + 1
            pages = w.block_table[r, : -(-L // 128)]
            K = torch.from_numpy(kf[pages].reshape(-1, w.hkv, w.head_dim)[:L])
            V = torch.from_numpy(vf[pages].reshape(-1, w.hkv, w.head_dim)[:L])
            for h in range(w.hq):
                kvh = h // group
                qv = torch.from_numpy(qf[row, h])
                Kh, Vh = K[:, kvh], V[:, kvh]
                logits = (Kh @ qv) * w.softmax_scale
                if w.sinks is not None:
                    # a key whose logit is exactly the sink, carrying a zero value
                    sink = float(w.sinks[h])
                    ks = qv * (sink / (w.softmax_scale * float(qv @ qv)))
                    Kh = torch.cat([Kh, ks[None]])
                    Vh = torch.cat([Vh, torch.zeros(1, w.head_dim, dtype=torch.float64)])
                    logits = torch.cat([logits, torch.tensor([sink], dtype=torch.float64)])
                o = torch.nn.functional.scaled_dot_product_attention(
                    qv[None, None, None], Kh[None, None], Vh[None, None], scale=w.softmax_scale)
                out[row, h] = o[0, 0, 0].numpy()
                lse[row, h] = float(torch.logsumexp(logits, 0))
    return out, lse


@pytest.mark.parametrize("kv_dtype,scale_mode,sink", [
    (W.KV_BF16, W.SCALE_NONE, False), (W.KV_BF16, W.SCALE_NONE, True),
    (W.KV_FP8, W.SCALE_SCALAR, True), (W.KV_FP8, W.SCALE_PER_TOKEN_HEAD, False)])
def test_dense_attention_matches_sdpa(orc, kv_dtype, scale_mode, sink):
    w = W.custom(21, q_lens=[1, 2], seq_lens=[300, 170], hq=4, di=64, topk=2,
                 kv_dtype=kv_dtype, scale_mode=scale_mode, with_sink=sink)
    out, lse, st = orc.dense(w)
    ref_o, ref_l = _sdpa_reference(w)
    assert st == 0
    np.testing.assert_allclose(out, ref_o, rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(lse, ref_l, rtol=1e-11, atol=1e-11)


def test_dense_attention_gqa_heads(orc):
    # two KV heads, four query heads: head h reads KV head h // 2
    w = W.custom(22, q_lens=[1], seq_lens=[200], hq=4, di=64, topk=2)
    rng = np.random.default_rng(3)
    w.k_cache = W.bf16_bits(rng.standard_normal((w.num_pages, 128, 2, 128)))
    w.v_cache = W.bf16_bits(rng.standard_normal((w.num_pages, 128, 2, 128)))
    out, lse, _ = orc.dense(w)
    ref_o, ref_l = _sdpa_reference(w)
    np.testing.assert_allclose(out, ref_o, rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(lse, ref_l, rtol=1e-11)


def test_sparse_equals_dense_when_k_covers_all(orc):
    # spec identity: with k >= number of blocks the sparse path is dense attention
    for kv, sm, sink in [(W.KV_BF16, W.SCALE_NONE, False), (W.KV_FP8, W.SCALE_PER_TOKEN_HEAD, True)]:
        w = W.custom(23, q_lens=[1, 4, 2], seq_lens=[900, 385, 129], hq=8, di=64, topk=8,
                     kv_dtype=kv, scale_mode=sm, with_sink=sink)
        r = orc.decode(w)
        out, lse, _ = orc.dense(w)
        np.testing.assert_allclose(r["out"], out, rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(r["lse"], lse, rtol=1e-12, atol=1e-13)


def test_sink_to_minus_infinity_is_no_sink(orc):
    w = W.custom(24, q_lens=[1, 1], seq_lens=[700, 1500], hq=8, di=64, topk=3, with_sink=True)
    w.sinks = np.full(8, -1e30, np.float32)
    r1 = orc.decode(w)
    w.sinks = None
    r0 = orc.decode(w)
    np.testing.assert_array_equal(r1["out"], r0["out"])
    np.testing.assert_array_equal(r1["lse"], r0["lse"])


def test_page_permutation_invariance(orc):
    w = W.custom(25, q_lens=[1, 3], seq_lens=[1200, 650], hq=8, di=64, topk=4,
                 kv_dtype=W.KV_FP8, scale_mode=W.SCALE_PER_TOKEN_HEAD, with_sink=True)
    r0 = orc.decode(w)
    perm = np.random.default_rng(9).permutation(w.num_pages)
    inv = np.argsort(perm)  # new page p holds old page perm[p]
    w.idx_k, w.k_cache, w.v_cache = w.idx_k[perm], w.k_cache[perm], w.v_cache[perm]
    w.k_scale, w.v_scale = w.k_scale[perm], w.v_scale[perm]
    bt = w.block_table.copy()
    bt[bt >= 0] = inv[bt[bt >= 0]]
    w.block_table = bt
    r1 = orc.decode(w)
    for key in ("topk_idx", "sparse_len", "out", "lse", "scores"):
        np.testing.assert_array_equal(r0[key], r1[key])


def _single_token_case(orc, sink):
    """One row, one visible token: O = v * e^s / (e^s + e^sink)."""
    w = W.custom(26, q_lens=[1], seq_lens=[1], hq=4, di=64, topk=1, with_sink=sink is not None)
    if sink is not None:
        w.sinks = np.array(sink, np.float32)
    r = orc.decode(w)
    qf = _f64(w.q, W.KV_BF16)[0]
    page = w.block_table[0, 0]
    k = _f64(w.k_cache, W.KV_BF16)[page, 0, 0]
    v = _f64(w.v_cache, W.KV_BF16)[page, 0, 0]
    return w, r, qf, k, v


def test_single_token_closed_form(orc):
    w, r, qf, k, v = _single_token_case(orc, [0.3, -1.0, 2.0, -4.0])
    sinks = [float(x) for x in w.sinks]  # the fp32 values the oracle sees
    for h in range(4):
        s = float(w.softmax_scale) * float(qf[h] @ k)
        sig = 1.0 / (1.0 + math.exp(sinks[h] - s))
        np.testing.assert_allclose(r["out"][0, h], v * sig, rtol=1e-12, atol=1e-15)
        assert abs(r["lse"][0, h] - math.log(math.exp(s) + math.exp(sinks[h]))) < 1e-12
    w, r, qf, k, v = _single_token_case(orc, None)
    np.testing.assert_allclose(r["out"][0], np.tile(v, (4, 1)), rtol=0, atol=0)


def test_equal_scores_and_constant_values(orc):
    # K = 0 -> every logit is 0: LSE = ln(n) (+ sink term), O = mean of V.
    # V = c everywhere -> O = c * (1 - e^(sink - LSE)).
    w = W.custom(27, q_lens=[1], seq_lens=[777], hq=4, di=64, topk=8, with_sink=True)
    w.k_cache = np.zeros_like(w.k_cache)
    r = orc.decode(w)
    n = 777
    vf = _f64(w.v_cache, W.KV_BF16)[w.block_table[0, :7]].reshape(-1, 128)[:n]
    for h in range(4):
        sink = float(w.sinks[h])
        den = n + math.exp(sink)
        assert abs(r["lse"][0, h] - math.log(den)) < 1e-12
        np.testing.assert_allclose(r["out"][0, h], vf.sum(0) / den, rtol=1e-10, atol=1e-13)
    w2 = W.custom(28, q_lens=[2], seq_lens=[500], hq=4, di=64, topk=2, with_sink=True)
    w2.v_cache = np.full_like(w2.v_cache, W.bf16_bits(np.array([1.5], np.float32))[0])
    r2 = orc.decode(w2)
    for row in range(2):
        for h in range(4):
            c = 1.5 * (1 - math.exp(float(w2.sinks[h]) - r2["lse"][row, h]))
            np.testing.assert_allclose(r2["out"][row, h], c, rtol=1e-12)


def test_scalar_and_uniform_per_token_scales_agree(orc):
    # per-token-head scales that are all equal to c behave like scalar c, and
    # scalar (a, b) equals unscaled attention with softmax scale x a, times b
    w = W.custom(29, q_lens=[1, 2], seq_lens=[640, 333], hq=8, di=64, topk=3,
                 kv_dtype=W.KV_FP8, scale_mode=W.SCALE_SCALAR, with_sink=True)
    a, bsc = 0.75, 1.25
    w.k_scale = np.array([a], np.float32)
    w.v_scale = np.array([bsc], np.float32)
    r_scalar = orc.decode(w)
    w.scale_mode = W.SCALE_PER_TOKEN_HEAD
    w.k_scale = np.full((w.num_pages, 128, 1), a, np.float32)
    w.v_scale = np.full((w.num_pages, 128, 1), bsc, np.float32)
    r_tok = orc.decode(w)
    np.testing.assert_allclose(r_tok["out"], r_scalar["out"], rtol=1e-13, atol=1e-15)
    w.scale_mode = W.SCALE_NONE
    w.k_scale = w.v_scale = None
    w.softmax_scale = w.softmax_scale * a
    r_none = orc.decode(w)
    np.testing.assert_allclose(r_scalar["out"], bsc * r_none["out"], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(r_scalar["lse"], r_none["lse"], rtol=1e-13)


def test_empty_and_poisoned_rows(orc):
    w = W.custom(30, q_lens=[1], seq_lens=[300], hq=4, di=64, topk=2, with_sink=True)
    tbl = np.zeros((3, 16), np.int32)
    slen = np.array([0, 20, 16 * 16 + 1], np.int32)  # empty; bad id below; too long
    tbl[1, 1] = 10 ** 6
    q = np.repeat(w.q, 3, axis=0)
    out, lse, st = orc.sparse_attn(q, w.k_cache, w.v_cache, w.kv_dtype, tbl, slen,
                                   sinks=w.sinks, softmax_scale=w.softmax_scale)
    assert st == orc.BAD_TABLE
    assert np.all(out == 0)
    np.testing.assert_array_equal(lse, np.tile(w.sinks.astype(np.float64), (3, 1)))
    out, lse, st = orc.sparse_attn(q[:1], w.k_cache, w.v_cache, w.kv_dtype, tbl[:1], slen[:1],
                                   softmax_scale=w.softmax_scale)
    assert st == 0 and np.all(out == 0) and np.all(lse == NEG_INF)


def test_threads_do_not_change_results(orc):
    w = W.custom(31, q_lens=[2, 1, 3], seq_lens=[900, 1300, 260], hq=8, di=64, topk=3,
                 kv_dtype=W.KV_FP8, scale_mode=W.SCALE_PER_TOKEN_HEAD, with_sink=True)
    r1 = orc.decode(w, nthreads=1)
    r4 = orc.decode(w, nthreads=4)
    for key in ("scores", "topk_idx", "tbl", "sparse_len", "out", "lse"):
        np.testing.assert_array_equal(r1[key], r4[key])


# ------------------------------------------------------------- KV insert

def test_fp8_encode_matches_torch_in_range(orc):
    # torch's float -> float8_e4m3fn cast is round-to-nearest-even; inside the
    # finite range the two must agree code for code
    rng = np.random.default_rng(4)
    xs = np.concatenate([rng.standard_normal(3000) * s for s in (0.01, 1.0, 30.0, 150.0)])
    xs = np.clip(xs, -448, 448).astype(np.float32)
    ref = torch.from_numpy(xs).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([orc.fp8_e4m3_encode(x) for x in xs], np.uint8)
    assert np.array_equal(ref, got)


def test_fp8_encode_roundtrip_ties_and_saturation(orc):
    for code in range(256):
        if code & 0x7F == 0x7F:
            continue
        v = orc.fp8_e4m3_value(code)
        assert orc.fp8_e4m3_encode(np.float32(v)) == code  # every value encodes to itself
    # halfway cases go to the even code
    assert orc.fp8_e4m3_encode(1.0625) == 0x38      # between 1.0 (0x38) and 1.125 (0x39)
    assert orc.fp8_e4m3_encode(1.1875) == 0x3A      # between 1.125 (0x39) and 1.25 (0x3a)
    assert orc.fp8_e4m3_encode(2.0 ** -10) == 0x00  # between 0 and the smallest subnormal
    assert orc.fp8_e4m3_encode(1.5 * 2.0 ** -9) == 0x02
    # beyond the largest finite value: saturate, keeping the sign
    for x in (449.0, 480.0, 1e30, float("inf")):
        assert orc.fp8_e4m3_encode(x) == 0x7E and orc.fp8_e4m3_encode(-x) == 0xFE
    assert orc.fp8_e4m3_encode(float("nan")) == 0x7F


def _new_rows(w, seed):
    rng = np.random.default_rng(seed)
    k_new = W.bf16_bits(rng.standard_normal((w.num_rows, w.hkv, w.head_dim)) * 3)
    v_new = W.bf16_bits(rng.standard_normal((w.num_rows, w.hkv, w.head_dim)) * 3)
    idx_new = W.bf16_bits(rng.integers(-3, 4, (w.num_rows, w.index_heads, w.index_dim)))
    return k_new, v_new, idx_new


def test_kv_insert_writes_each_row_at_its_slot(orc):
    w = W.custom(90, q_lens=[1, 3, 2], seq_lens=[300, 129, 1000], hq=4, di=64, topk=2)
    k_new, v_new, idx_new = _new_rows(w, 1)
    k, v, ik, _, _, st = orc.kv_insert(w, k_new, v_new, idx_new)
    assert st == 0
    r = 0
    for q in range(w.num_reqs):
        for j in range(int(w.q_lens[q])):
            pos = int(w.context_lens[q]) + j
            page = w.block_table[q, pos // 128]
            assert np.array_equal(k[page, pos % 128], k_new[r])
            assert np.array_equal(v[page, pos % 128], v_new[r])
            assert np.array_equal(ik[page, pos % 128], idx_new[r])
            r += 1
    # nothing else changed
    changed = (k != w.k_cache).any(axis=(2, 3))
    assert changed.sum() <= w.num_rows
    _, _, ik2, _, _, _ = orc.kv_insert(w, k_new, v_new, idx_new, skip_index=True)
    assert np.array_equal(ik2, w.idx_k)  # index-reuse layers leave the index cache alone


def test_kv_insert_fp8_per_token_scale_definition(orc):
    w = W.custom(91, q_lens=[2, 1], seq_lens=[500, 77], hq=4, di=64, topk=2,
                 kv_dtype=W.KV_FP8, scale_mode=W.SCALE_PER_TOKEN_HEAD)
    k_new, v_new, idx_new = _new_rows(w, 2)
    k, v, _, ks, vs, st = orc.kv_insert(w, k_new, v_new, idx_new)
    assert st == 0
    to_f = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).float().numpy()
    r = 0
    for q in range(w.num_reqs):
        for j in range(int(w.q_lens[q])):
            pos = int(w.context_lens[q]) + j
            page, slot = w.block_table[q, pos // 128], pos % 128
            x = to_f(k_new[r, 0])
            s = np.float32(np.abs(x).max()) / np.float32(448)
            assert ks[page, slot, 0] == s
            codes = k[page, slot, 0]
            vals = np.array([orc.fp8_e4m3_value(c) for c in codes])
            assert np.abs(vals).max() == 448.0  # the largest element lands on the top code
            np.testing.assert_allclose(vals * s, x, rtol=2 ** -4, atol=s * 2 ** -9)
            r += 1


# Hand-worked codes of the SCALAR and NONE insert rules (code = e4m3 of x / s):
# (x, s, code) from the OCP e4m3fn definition -- bias 7, 3 mantissa bits,
# value = 2^(e-7) * (1 + m/8), largest finite 448 = 0x7E.  Each pair is chosen
# so that a plausible slip changes the code: x * s instead of x / s, no
# saturation, round-half-up instead of half-to-even, a dropped sign.
_SCALAR_INSERT_CASES = [
    (1.0, 0.5, 0x40),       # 1 / 0.5 = 2 = 2^1 -> e = 8, m = 0   (x * s = 0.5 would give 0x30)
    (-3.0, 2.0, 0xBC),      # -1.5 -> e = 7, m = 4, sign bit
    (2.125, 2.0, 0x38),     # 1.0625: halfway 1.0 (0x38) / 1.125 (0x39) -> even 0x38
    (2.375, 2.0, 0x3A),     # 1.1875: halfway 1.125 (0x39) / 1.25 (0x3A) -> even 0x3A
    (300.0, 0.5, 0x7E),     # 600 is beyond 448: saturate
    (-300.0, 0.5, 0xFE),    # ... keeping the sign
    (0.0, 4.0, 0x00),
    (0.0078125, 4.0, 0x01),  # 2^-7 / 4 = 2^-9, the smallest subnormal
    (96.0, 0.25, 0x7C),     # 384 = 2^8 * 1.5 -> e = 15, m = 4
]
_NONE_INSERT_CASES = [      # s = 1: the codes of x itself
    (1.0, 0x38), (-0.5, 0xB0), (1000.0, 0x7E), (1.0625, 0x38), (0.001953125, 0x01),
    (240.0, 0x77),          # 240 = 2^7 * 1.875 -> e = 14, m = 7
]


def _fp8_insert_workload(scale_mode, k_s, v_s, seed):
    w = W.custom(seed, q_lens=[2, 1], seq_lens=[500, 77], hq=4, di=64, topk=2,
                 kv_dtype=W.KV_FP8, scale_mode=scale_mode)
    if scale_mode == W.SCALE_SCALAR:
        w = dataclasses.replace(w, k_scale=np.array([k_s], np.float32),
                                v_scale=np.array([v_s], np.float32))
    return w


def _slot(w, r):
    q = int(np.searchsorted(w.cu_seqlens_q, r, side="right") - 1)
    pos = int(w.context_lens[q]) + r - int(w.cu_seqlens_q[q])
    return w.block_table[q, pos // 128], pos % 128


@pytest.mark.parametrize("mode", ["scalar", "none"])
def test_kv_insert_fp8_fixed_scale_hand_worked_codes(orc, mode):
    # one hand-worked element at dim i of row 0's K and dim 5 + i of row 1's V,
    # the rest zero; every case brings its own scale, so one workload each
    cases = (_SCALAR_INSERT_CASES if mode == "scalar"
             else [(x, 1.0, c) for x, c in _NONE_INSERT_CASES])
    for i, (x, s, code) in enumerate(cases):
        w = _fp8_insert_workload(W.SCALE_SCALAR if mode == "scalar" else W.SCALE_NONE, s, s,
                                 seed=94)
        k_new = np.zeros((w.num_rows, w.hkv, w.head_dim), np.float32)
        v_new = np.zeros_like(k_new)
        k_new[0, 0, i] = x
        v_new[1, 0, 5 + i] = x
        idx_new = W.bf16_bits(np.zeros((w.num_rows, w.index_heads, w.index_dim)))
        k, v, _, ks, vs, st = orc.kv_insert(w, W.bf16_bits(k_new), W.bf16_bits(v_new), idx_new)
        assert st == 0
        pk, sk = _slot(w, 0)
        pv, sv = _slot(w, 1)
        assert k[pk, sk, 0, i] == code, (x, s, hex(int(k[pk, sk, 0, i])), hex(code))
        assert v[pv, sv, 0, 5 + i] == code, (x, s)
        assert np.count_nonzero(k[pk, sk, 0]) == (code & 0x7F != 0)
        if mode == "scalar":  # the given scales are inputs, never rewritten
            assert ks[0] == np.float32(s) and vs[0] == np.float32(s)


@pytest.mark.parametrize("mode", [W.SCALE_SCALAR, W.SCALE_NONE])
def test_kv_insert_fp8_fixed_scale_matches_torch_cast(orc, mode):
    # a sweep over normal, large and tiny values: code = torch's float8_e4m3fn
    # cast (round to nearest even) of the fp32 quotient x / s, saturated
    w = _fp8_insert_workload(mode, 0.37109375, 2.75, seed=95)
    rng = np.random.default_rng(96)
    mag = np.exp(rng.uniform(np.log(1e-4), np.log(2e3), (w.num_rows, w.hkv, w.head_dim)))
    sign = rng.choice([-1.0, 1.0], size=mag.shape)
    k_new = W.bf16_bits(mag * sign)
    v_new = W.bf16_bits(-mag[::-1] * sign)
    idx_new = W.bf16_bits(rng.integers(-3, 4, (w.num_rows, w.index_heads, w.index_dim)))
    k, v, _, _, _, st = orc.kv_insert(w, k_new, v_new, idx_new)
    assert st == 0
    to_f = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).float().numpy()
    sk_ = np.float32(w.k_scale[0]) if mode == W.SCALE_SCALAR else np.float32(1)
    sv_ = np.float32(w.v_scale[0]) if mode == W.SCALE_SCALAR else np.float32(1)
    for r in range(w.num_rows):
        page, slot = _slot(w, r)
        want_k = W.fp8_codes(to_f(k_new[r, 0]) / sk_)
        want_v = W.fp8_codes(to_f(v_new[r, 0]) / sv_)
        assert np.array_equal(k[page, slot, 0], want_k)
        assert np.array_equal(v[page, slot, 0], want_v)
    # the sweep reaches both the saturating and the subnormal range
    assert (np.abs(to_f(k_new)) / sk_ > 448).any() and (np.abs(to_f(k_new)) / sk_ < 2 ** -6).any()


@pytest.mark.parametrize("scaled", [True, False])
def test_kv_insert_fp8_index_cache(orc, scaled):
    # e4m3 index keys per token and index head: with scales kept, the
    # per-token-head rule (s = max|x| / 448, codes of x / s, torch's float8
    # cast as the independent encoder); without, the codes of x itself
    w = W.fp8_index(W.custom(92, q_lens=[2, 1], seq_lens=[500, 77], hq=4, di=64, hi=2, topk=2),
                    seed=93, scaled=scaled)
    k_new, v_new, idx_new = _new_rows(w, 2)
    *_, st, iscale = orc.kv_insert(w, k_new, v_new, idx_new)
    assert st == 0
    codes = orc.kv_insert(w, k_new, v_new, idx_new)[2]
    to_f = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).float().numpy()
    r = 0
    for q in range(w.num_reqs):
        for j in range(int(w.q_lens[q])):
            pos = int(w.context_lens[q]) + j
            page, slot = w.block_table[q, pos // 128], pos % 128
            for h in range(w.index_heads):
                x = to_f(idx_new[r, h])
                s = np.float32(np.abs(x).max()) / np.float32(448) if scaled else np.float32(1)
                if scaled:
                    assert iscale[page, slot, h] == s
                want = W.fp8_codes(x / s)
                assert np.array_equal(codes[page, slot, h], want)
            r += 1


# ----------------------------------------------------------- sparse MLA decode

def _mla_reference(w):
    """float64 torch reference: gather each row's latent rows, softmax over the
    scaled logits with the sink as one more logit, value = first dv columns."""
    to_f = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).double()
    q, kv = to_f(w.q), to_f(w.kv_cache)
    out = np.zeros((w.num_rows, w.heads, w.dv))
    lse = np.full((w.num_rows, w.heads), NEG_INF)
    for r in range(w.num_rows):
        ids = torch.from_numpy(w.kv_indices[w.kv_indptr[r]:w.kv_indptr[r + 1]].astype(np.int64))
        K = kv[ids]                                   # [n, dqk]
        logits = w.softmax_scale * (q[r] @ K.T)       # [H, n]
        if w.sinks is not None:
            logits = torch.cat([logits, torch.from_numpy(w.sinks).double()[:, None]], dim=1)
        if logits.shape[1] == 0:
            continue
        p = torch.softmax(logits, dim=1)[:, : len(ids)]
        out[r] = (p @ K[:, : w.dv]).numpy()
        lse[r] = torch.logsumexp(logits, dim=1).numpy()
    return out, lse


@pytest.mark.parametrize("sink,dup", [(True, False), (False, False), (True, True)])
def test_sparse_mla_matches_softmax_reference(orc, sink, dup):
    w = W.sparse_mla_custom(31, [37, 16, 1, 200, 0], heads=8, ctx=512, dqk=96, dv=64,
                            with_sink=sink, duplicates=dup)
    out, lse, st = orc.sparse_mla(w.q, w.kv_cache, w.kv_indptr, w.kv_indices, w.dv,
                                  sinks=w.sinks, softmax_scale=w.softmax_scale)
    assert st == 0
    ref_o, ref_l = _mla_reference(w)
    np.testing.assert_allclose(out, ref_o, rtol=1e-10, atol=1e-12)
    fin = np.isfinite(ref_l)
    assert np.array_equal(np.isfinite(lse), fin)
    np.testing.assert_allclose(lse[fin], ref_l[fin], rtol=1e-12, atol=1e-12)
    # the empty row: O = 0 and LSE = the sink (or -inf)
    assert np.all(out[4] == 0)
    assert np.array_equal(lse[4], w.sinks.astype(np.float64) if sink else np.full(8, NEG_INF))


def test_sparse_mla_order_invariance_and_bad_ids(orc):
    w = W.sparse_mla_custom(32, [50, 9], heads=4, ctx=256, dqk=96, dv=64)
    a = orc.sparse_mla(w.q, w.kv_cache, w.kv_indptr, w.kv_indices, w.dv, sinks=w.sinks,
                       softmax_scale=w.softmax_scale)
    perm = w.kv_indices.copy()
    perm[:50] = perm[:50][::-1]
    b = orc.sparse_mla(w.q, w.kv_cache, w.kv_indptr, perm, w.dv, sinks=w.sinks,
                       softmax_scale=w.softmax_scale)
    np.testing.assert_allclose(a[0], b[0], rtol=1e-12, atol=1e-14)
    # an id outside the cache poisons its row only: empty row + status bit
    bad = w.kv_indices.copy()
    bad[52] = w.num_tokens
    o, l, st = orc.sparse_mla(w.q, w.kv_cache, w.kv_indptr, bad, w.dv, sinks=w.sinks,
                              softmax_scale=w.softmax_scale)
    assert st == 8
    assert np.all(o[1] == 0) and np.array_equal(l[1], w.sinks.astype(np.float64))
    np.testing.assert_array_equal(o[0], a[0][0])


# ------------------------------------------------------------ FP8 sparse MLA

def _mla_fp8_reference(w):
    """float64 torch reference for FP8 operands: e4m3 codes decoded by
    torch's float8_e4m3fn (an independent decoder), times the per-tensor
    scale (q_scale for the query, kv_scale for the key and the value), then
    the same softmax with the sink as one more logit."""
    def dec(a, scale):
        if a.dtype == np.uint8:
            return torch.from_numpy(a).view(torch.float8_e4m3fn).double() * float(scale[0])
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).double()
    q, kv = dec(w.q, w.q_scale), dec(w.kv_cache, w.kv_scale)
    out = np.zeros((w.num_rows, w.heads, w.dv))
    lse = np.full((w.num_rows, w.heads), NEG_INF)
    for r in range(w.num_rows):
        ids = torch.from_numpy(w.kv_indices[w.kv_indptr[r]:w.kv_indptr[r + 1]].astype(np.int64))
        K = kv[ids]
        logits = w.softmax_scale * (q[r] @ K.T)
        if w.sinks is not None:
            logits = torch.cat([logits, torch.from_numpy(w.sinks).double()[:, None]], dim=1)
        if logits.shape[1] == 0:
            continue
        p = torch.softmax(logits, dim=1)[:, : len(ids)]
        out[r] = (p @ K[:, : w.dv]).numpy()
        lse[r] = torch.logsumexp(logits, dim=1).numpy()
    return out, lse


@pytest.mark.parametrize("fp8_q,sink", [(True, True), (False, True), (True, False)])
def test_fp8_sparse_mla_matches_torch_reference(orc, fp8_q, sink):
    w = W.mla_fp8(W.sparse_mla_custom(33, [37, 16, 1, 200, 0], heads=8, ctx=512, dqk=96, dv=64,
                                      with_sink=sink), seed=34, fp8_q=fp8_q)
    out, lse, st = orc.sparse_mla(w.q, w.kv_cache, w.kv_indptr, w.kv_indices, w.dv,
                                  sinks=w.sinks, softmax_scale=w.softmax_scale,
                                  q_scale=w.q_scale, kv_scale=w.kv_scale)
    assert st == 0
    ref_o, ref_l = _mla_fp8_reference(w)
    np.testing.assert_allclose(out, ref_o, rtol=1e-10, atol=1e-12)
    fin = np.isfinite(ref_l)
    assert np.array_equal(np.isfinite(lse), fin)
    np.testing.assert_allclose(lse[fin], ref_l[fin], rtol=1e-12, atol=1e-12)


def test_fp8_sparse_mla_unit_scales_equal_bf16(orc):
    # e4m3 values are exact in bf16: with unit scales the FP8 oracle must
    # equal the bf16 oracle on the decoded values bit for bit
    w8 = W.mla_fp8(W.sparse_mla_custom(35, [20, 3, 64], heads=4, ctx=256, dqk=96, dv=64), 36)
    w8 = dataclasses.replace(w8, q_scale=np.ones(1, np.float32), kv_scale=np.ones(1, np.float32))
    to_bf16 = lambda codes: W.bf16_bits(torch.from_numpy(codes).view(torch.float8_e4m3fn)
                                        .float().numpy())
    a = orc.sparse_mla(w8.q, w8.kv_cache, w8.kv_indptr, w8.kv_indices, w8.dv, sinks=w8.sinks,
                       softmax_scale=w8.softmax_scale, q_scale=w8.q_scale,
                       kv_scale=w8.kv_scale)
    b = orc.sparse_mla(to_bf16(w8.q), to_bf16(w8.kv_cache), w8.kv_indptr, w8.kv_indices, w8.dv,
                       sinks=w8.sinks, softmax_scale=w8.softmax_scale)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1]) and a[2] == b[2] == 0


def test_fp8_sparse_mla_scale_placement(orc):
    # kv_scale multiplies keys and values, q_scale the query: doubling
    # kv_scale doubles every logit (so halving softmax_scale undoes it for
    # the weights) and doubles every output value
    w = W.mla_fp8(W.sparse_mla_custom(37, [40, 9], heads=4, ctx=256, dqk=96, dv=64,
                                      with_sink=False), 38)
    o1, l1, _ = orc.sparse_mla(w.q, w.kv_cache, w.kv_indptr, w.kv_indices, w.dv,
                               softmax_scale=w.softmax_scale, q_scale=w.q_scale,
                               kv_scale=w.kv_scale)
    o2, l2, _ = orc.sparse_mla(w.q, w.kv_cache, w.kv_indptr, w.kv_indices, w.dv,
                               softmax_scale=w.softmax_scale / 2, q_scale=w.q_scale,
                               kv_scale=w.kv_scale * 2)
    np.testing.assert_allclose(o2, 2 * o1, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(l2, l1, rtol=1e-12, atol=1e-12)
    o3, l3, _ = orc.sparse_mla(w.q, w.kv_cache, w.kv_indptr, w.kv_indices, w.dv,
                               softmax_scale=w.softmax_scale * 2, q_scale=w.q_scale / 2,
                               kv_scale=w.kv_scale)
    np.testing.assert_allclose(o3, o1, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(l3, l1, rtol=1e-12, atol=1e-12)

