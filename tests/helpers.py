"""Shared test helpers: tolerances, comparisons and sampled-row sub-batches."""
import numpy as np

import workloads as W

# Attention tolerance for bf16/FP8 KV against the fp64 oracle:
# |O - O_ref| <= 1e-2 * (1 + |O_ref|), |LSE - LSE_ref| <= 2e-3.
O_RTOL = 1e-2
LSE_ATOL = 2e-3


def assert_attn_close(out, lse, ref_out, ref_lse, rows=None):
    out = np.asarray(out, np.float64)
    ref_out = np.asarray(ref_out, np.float64)
    if rows is not None:
        out, lse = out[rows], np.asarray(lse)[rows]
    err = np.abs(out - ref_out)
    bound = O_RTOL * (1.0 + np.abs(ref_out))
    bad = ~(err <= bound)
    assert not bad.any(), (f"O mismatch at {np.argwhere(bad)[:5].tolist()}: "
                           f"max err/bound {float(np.max(err / bound)):.3f}")
    lse = np.asarray(lse, np.float64)
    ref_lse = np.asarray(ref_lse, np.float64)
    both_inf = np.isneginf(lse) & np.isneginf(ref_lse)
    with np.errstate(invalid="ignore"):  # -inf - -inf where both rows are empty
        lerr = np.where(both_inf, 0.0, np.abs(lse - ref_lse))
    assert np.all(lerr <= LSE_ATOL), f"LSE max err {float(np.nanmax(lerr))}"


def valid_score_mask(geom, score_stride):
    """Entries the score kernel defines: rows that are scored, b < nb_r."""
    n = len(geom["nb"])
    mask = np.zeros((n, score_stride), bool)
    for r in range(n):
        if geom["ok"][r] != 0:
            mask[r, : geom["nb"][r]] = True
    return mask


# A batch holding only the given rows (each its own one-row request at the
# same position over the same pages); see workloads.row_subset.
sub_workload = W.row_subset


# Rows msa_decode sends through the block-major prefill attention (requests
# of >= 64 rows, bf16 KV without per-token scales, top-k <= 128): the fused
# call's attention there differs from the stand-alone attention entry point
# in rounding only, so those rows are checked against the oracle instead of
# bit for bit against the separate calls.
PREFILL_MIN_ROWS = 64
PREFILL_MAX_TOPK = 128


def prefill_rows(w, topk=None):
    k = int(topk or w.topk)
    mask = np.zeros(w.num_rows, bool)
    if w.kv_dtype != W.KV_BF16 or w.scale_mode == W.SCALE_PER_TOKEN_HEAD or k > PREFILL_MAX_TOPK:
        return mask
    q_lens = np.diff(np.asarray(w.cu_seqlens_q, np.int64))
    if q_lens.size == 0 or q_lens.max() < PREFILL_MIN_ROWS:
        return mask
    for q, ql in enumerate(q_lens):
        if ql >= PREFILL_MIN_ROWS:
            mask[int(w.cu_seqlens_q[q]): int(w.cu_seqlens_q[q + 1])] = True
    return mask

