"""Comparison helpers shared by the GPU parity tests (tolerances in one place).

Acceptance bars for one DSA decode step:
  scores   |gpu - oracle| <= 1e-3 * max(|oracle|, 1e-3 * max_s |oracle[r, s]|)
  top-k    bit-exact sets when the GPU select is fed the oracle's scores
           (rounded to fp32); with GPU scores, equal sets outside near-ties,
           a near-tie being |oracle_s - oracle_kth| < 1e-3 * |oracle_kth|
  output   bf16 attention output within 2e-2 max-abs of the float64 oracle
"""
import numpy as np

SCORE_RTOL = 1e-3
NEAR_TIE_RTOL = 1e-3
OUT_ATOL = 2e-2


def assert_scores_close(gpu, ora, row_len):
    for r, L in enumerate(row_len):
        if L == 0:
            continue
        g = np.asarray(gpu[r, :L], np.float64)
        o = np.asarray(ora[r, :L], np.float64)
        assert np.isfinite(g).all(), f"row {r}: {np.count_nonzero(~np.isfinite(g))} non-finite scores"
        assert np.isfinite(o).all(), f"row {r}: the oracle left scores unwritten"
        floor = 1e-3 * np.abs(o).max()
        tol = SCORE_RTOL * np.maximum(np.abs(o), floor)
        bad = np.abs(g - o) > tol
        assert not bad.any(), (f"row {r}: {bad.sum()} scores off, worst "
                               f"{np.max(np.abs(g - o) / np.maximum(tol, 1e-300)):.3g}x tol")


def selected(idx_row):
    idx_row = np.asarray(idx_row)
    return set(int(x) for x in idx_row[idx_row >= 0])


def assert_topk_equal_outside_near_ties(gpu_idx, ora_idx, ora_scores, row_len, k):
    for r, L in enumerate(row_len):
        g, o = selected(gpu_idx[r]), selected(ora_idx[r])
        assert len(g) == min(k, L), f"row {r}: {len(g)} selected, expected {min(k, L)}"
        if g == o:
            continue
        s = np.asarray(ora_scores[r, :L], np.float64)
        kth = np.sort(s)[::-1][min(k, L) - 1]
        near = set(np.nonzero(np.abs(s - kth) < NEAR_TIE_RTOL * abs(kth))[0].tolist())
        assert g - near == o - near, (f"row {r}: selections differ outside near-ties: "
                                      f"{sorted((g ^ o) - near)[:10]}")


def assert_out_close(gpu_out, ora_out):
    err = np.abs(np.asarray(gpu_out, np.float64) - ora_out)
    assert np.isfinite(err).all(), "non-finite attention output"
    assert err.max() <= OUT_ATOL, f"max |out - oracle| = {err.max():.3g} > {OUT_ATOL}"
    return float(err.max())


def e4m3_midpoints(oracle_mod):
    """Midpoints between consecutive non-negative finite E4M3 values."""
    vals = sorted({oracle_mod.e4m3_decode(c) for c in range(0x7F)})
    return np.array([(a + b) / 2 for a, b in zip(vals[:-1], vals[1:])])


def near_midpoint(v, mids, rel=1e-5):
    """True where |v| lies within rel * |v| of an E4M3 rounding midpoint: there
    fp32 and float64 arithmetic may round to neighbouring codes."""
    a = np.abs(np.asarray(v, np.float64))
    j = np.clip(np.searchsorted(mids, a), 1, len(mids) - 1)
    d = np.minimum(np.abs(a - mids[j - 1]), np.abs(a - mids[j]))
    return d <= rel * np.maximum(a, 1e-30)
