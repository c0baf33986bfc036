"""Threshold calibration from the kernels' per-tile margins.

BLASST talk notes, "threshold calibration" (Algorithm 2): one pass over calibration
data sweeps many candidate thresholds at once, the observed sparsity is recorded per
(threshold, sequence length), the model lambda * L = a * exp(b * S) is fitted, and
any target sparsity S then gives lambda = a * exp(b * S) / L (the inverse length
law, Eq. 3).

The one pass is a lambda = 0 launch with margins requested: a tile is skipped at
threshold lambda iff its margin is below ln(lambda), and for lambda <= 1 the margins
do not depend on lambda, so the sparsity of every candidate is read off one set of
margins.  The fit is ordinary least squares of ln(lambda * L) on S over the points
whose sparsity is strictly between 0 and 1.
"""
from __future__ import annotations

import math

import numpy as np


def sparsity_at(margins, lam: float) -> float:
    """Fraction of visited tiles (non-NaN margins) that threshold lam skips."""
    g = np.asarray(margins, dtype=np.float64)
    g = g[~np.isnan(g)]
    if g.size == 0 or lam <= 0:
        return 0.0
    return float(np.count_nonzero(g < math.log(lam))) / g.size


def lambda_for_sparsity(margins, target: float) -> float:
    """Smallest threshold in (0, 1] whose sparsity reaches `target` (1.0 if none)."""
    g = np.asarray(margins, dtype=np.float64)
    g = np.sort(g[~np.isnan(g)])
    if g.size == 0:
        return 1.0
    k = int(math.ceil(target * g.size))
    if k <= 0:
        return 0.0
    if k > g.size:
        return 1.0
    # skipped iff margin < ln(lambda): lambda just above exp(g[k-1]) skips k tiles
    lam = math.exp(g[k - 1]) * (1.0 + 1e-6)
    return min(lam, 1.0)


def sweep(margins_by_len: dict, candidates) -> list:
    """[(lambda, L, S)] for every candidate threshold and sequence length."""
    return [(float(lam), int(L), sparsity_at(g, lam)) for L, g in margins_by_len.items() for lam in candidates]


def fit(points):
    """(a, b) of lambda * L = a * exp(b * S) by least squares; None if fewer than two
    points have 0 < S < 1 with distinct S."""
    xs, ys = [], []
    for lam, L, S in points:
        if lam > 0 and 0.0 < S < 1.0:
            xs.append(S)
            ys.append(math.log(lam * L))
    if len(xs) < 2 or max(xs) == min(xs):
        return None
    A = np.stack([np.ones(len(xs)), np.asarray(xs)], axis=1)
    coef, *_ = np.linalg.lstsq(A, np.asarray(ys), rcond=None)
    return float(math.exp(coef[0])), float(coef[1])
