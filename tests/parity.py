"""Acceptance rule for GPU-vs-oracle parity of the indexer.

* Scores: |I_gpu - I_ref| <= 1e-3 * max_s |I_ref[t, s]| (per query t), for
  every returned top-k score and, when requested, every entry of the full
  score row.
* Top-k sets: identical, except entries whose oracle score lies within that
  tolerance of the oracle's k-th score (any of those may fill the last
  places). The GPU list must hold no duplicate, be ordered by score
  descending with the lower index first on equal GPU scores, and be padded
  with -1 / -inf exactly where fewer than k keys are valid.
"""

import numpy as np

REL_TOL = 1e-3


def check_query(I_ref, gi, gs, k, rel_tol=REL_TOL, where=""):
    """I_ref: oracle scores of one query (float64, -inf = not a candidate);
    gi / gs: the GPU's k indices / scores."""
    gi = np.asarray(gi, dtype=np.int64)
    gs = np.asarray(gs, dtype=np.float64)
    assert gi.shape == (k,) and gs.shape == (k,), where
    if I_ref is None:
        assert np.all(gi == -1) and np.all(np.isneginf(gs)), f"{where}: expected all padding"
        return
    cand = np.nonzero(~np.isneginf(I_ref))[0]
    n = min(k, cand.size)
    assert np.all(gi[n:] == -1), f"{where}: padding indices"
    assert np.all(np.isneginf(gs[n:])), f"{where}: padding scores"
    sel = gi[:n]
    assert np.all(sel >= 0) and np.all(sel < I_ref.shape[0]), f"{where}: index out of range"
    assert np.unique(sel).size == n, f"{where}: duplicate indices"
    assert np.all(~np.isneginf(I_ref[sel])), f"{where}: returned a non-candidate key"
    if n == 0:
        return
    tol = rel_tol * float(np.max(np.abs(I_ref[cand])))
    err = np.abs(gs[:n] - I_ref[sel])
    assert np.all(err <= tol), f"{where}: score error {err.max():.3e} > tol {tol:.3e}"
    d = np.diff(gs[:n])
    assert np.all(d <= 0), f"{where}: scores not descending"
    eq = d == 0
    assert np.all(np.diff(sel)[eq] > 0), f"{where}: equal scores not in ascending index order"
    ref_sorted = np.sort(I_ref[cand])[::-1]
    kth = ref_sorted[n - 1]
    must = cand[I_ref[cand] > kth + tol]
    allowed = cand[I_ref[cand] >= kth - tol]
    s = set(sel.tolist())
    missing = [m for m in must.tolist() if m not in s]
    assert not missing, f"{where}: {len(missing)} keys above the k-th score + tol missing"
    extra = s - set(allowed.tolist())
    assert not extra, f"{where}: {len(extra)} keys below the k-th score - tol returned"


def check_scores_row(I_ref, row, rel_tol=REL_TOL, where=""):
    """Full score row (scores_out) against the oracle: -inf where the oracle
    has -inf, otherwise within the tolerance."""
    row = np.asarray(row, dtype=np.float64)[: I_ref.shape[0]]
    neg = np.isneginf(I_ref)
    assert np.array_equal(np.isneginf(row), neg), f"{where}: -inf pattern differs"
    if (~neg).any():
        tol = rel_tol * float(np.max(np.abs(I_ref[~neg])))
        err = np.abs(row[~neg] - I_ref[~neg])
        assert np.all(err <= tol), f"{where}: score error {err.max():.3e} > tol {tol:.3e}"
