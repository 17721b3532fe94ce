"""Acceptance rules shared by the GPU parity tests.

Scores.  A GPU score g matches the oracle's o when
    |g - o| <= rtol * max(|o|, 0.1 * rms(row))
with rtol = 1e-5 for fp32 inputs, 2e-2 for bf16 and 6e-2 for fp8.  The
floor (10% of the row's RMS score) keeps the relative rule meaningful for
scores near zero.  The rounding error of an fp32 dot product is a fraction
of the magnitude of its *terms*, sum_k |q~_k c_k|, not of the (cancelled)
result: for the workloads' distributions a score's terms add up to about
ten times the row RMS, so a typical fp32 error is ~1e-7 x RMS, and a score
at 1% of the RMS can miss a pure 1e-5 relative bound while being exact to
working precision.  Scores under 10% of the RMS lie far below any row's
k-th score (the 75th percentile or higher here) and never decide a
selection.

Index sets.  Let tau be the oracle's k-th largest valid score of the row and
Band = {t : |o_t - tau| <= rtol * max(|tau|, floor)}.  The GPU set must have
min(k, V) distinct valid positions (padded with -1) and agree with the
oracle's set outside the band; inside the band any choice is a correct
top-k up to the score tolerance.
"""
from __future__ import annotations

import numpy as np

RTOL = {"f32": 1e-5, "bf16": 2e-2, "fp8": 6e-2}
FLOOR_FRAC = 0.1

# One entry per assert_scores_close call: (what, scores compared, outside the
# floored rule, outside the pure relative rule |g - o| <= rtol |o|).  The
# session summary prints the totals, so the floor's effect stays visible.
REPORT: list[tuple[str, int, int, int]] = []


def _floor(o_row: np.ndarray) -> float:
    v = o_row[np.isfinite(o_row)]
    return FLOOR_FRAC * float(np.sqrt(np.mean(v * v))) if v.size else 0.0


def score_errors(g, o, rtol: float):
    """Per-element allowed error and the violation mask for rows along the last axis."""
    g = np.asarray(g, dtype=np.float64)
    o = np.asarray(o, dtype=np.float64)
    o2 = o.reshape(-1, o.shape[-1])
    floors = np.array([_floor(r) for r in o2]).reshape(o.shape[:-1] + (1,))
    allowed = rtol * np.maximum(np.abs(o), floors)
    bad = ~(np.abs(g - o) <= allowed)
    return allowed, bad


def assert_scores_close(g, o, rtol: float, what: str = "scores"):
    g = np.asarray(g, dtype=np.float64)
    o = np.asarray(o, dtype=np.float64)
    assert g.shape == o.shape, (g.shape, o.shape)
    _, bad = score_errors(g, o, rtol)
    pure = int(np.count_nonzero(~(np.abs(g - o) <= rtol * np.abs(o))))
    REPORT.append((what, int(bad.size), int(bad.sum()), pure))
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {bad.size} outside rtol={rtol} "
            f"({pure} outside the pure relative rule); first at {tuple(i)}: "
            f"gpu={g[tuple(i)]!r} oracle={o[tuple(i)]!r}")


def max_rel_err(g, o) -> float:
    g = np.asarray(g, dtype=np.float64)
    o = np.asarray(o, dtype=np.float64)
    o2 = o.reshape(-1, o.shape[-1])
    floors = np.array([_floor(r) for r in o2]).reshape(o.shape[:-1] + (1,))
    return float(np.max(np.abs(g - o) / np.maximum(np.abs(o), np.maximum(floors, 1e-300))))


def assert_topk_row(gpu_idx, o_row, k: int, V: int, rtol: float, what: str = "topk",
                    allowed=None):
    """Band rule for one row.  `allowed`: optional set the selection must lie in (HS)."""
    gpu_idx = np.asarray(gpu_idx)
    n = min(k, V)
    sel = gpu_idx[:n]
    assert (gpu_idx[n:] == -1).all(), f"{what}: padding slots not -1"
    assert len(set(sel.tolist())) == n, f"{what}: duplicate or missing indices"
    assert sel.min(initial=0) >= 0 and sel.max(initial=-1) < max(V, 1), f"{what}: index out of range"
    if n == 0:
        return
    o_row = np.asarray(o_row, dtype=np.float64)
    pool = np.arange(V) if allowed is None else np.array(sorted(allowed))
    assert set(sel.tolist()) <= set(pool.tolist()), f"{what}: selection outside the candidate set"
    vals = o_row[pool]
    order = np.lexsort((pool, -vals))
    orc = set(pool[order[:n]].tolist())
    tau = vals[order[n - 1]]
    fl = _floor(o_row[:V])
    band = set(pool[np.abs(vals - tau) <= rtol * max(abs(tau), fl)].tolist())
    g_out, o_out = set(sel.tolist()) - band, orc - band
    if g_out != o_out:
        raise AssertionError(
            f"{what}: sets differ outside the band: gpu-only {sorted(g_out - o_out)[:8]}, "
            f"oracle-only {sorted(o_out - g_out)[:8]} (tau={tau}, |band|={len(band)})")


def exact_sets_equal(gpu_idx, orc_idx):
    a = np.sort(np.asarray(gpu_idx), axis=-1)
    b = np.sort(np.asarray(orc_idx), axis=-1)
    np.testing.assert_array_equal(a, b)
