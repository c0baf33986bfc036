"""Oracle for the threshold calibration (test infrastructure only).

BLASST talk notes, "threshold calibration" (Algorithm 2), in its four steps:
  (1) sweep many candidate thresholds in one pass over a calibration set,
  (2) record the observed sparsity for each (threshold, sequence length),
  (3) fit the exponential model  lambda * L = a * exp(b * S),
  (4) for a chosen target sparsity S, lambda = a * exp(b * S) / L.

Step (1)-(2) read the sparsity of every candidate lambda off the per-tile margins
of one lambda = 0 pass: a tile is skipped at lambda iff its margin < ln(lambda),
and the margins do not depend on lambda (for lambda <= 1 a skip never moves the
running max).  Step (3) is an ordinary least-squares line through
(S, ln(lambda * L)); points at S = 0 or S = 1 carry no information about lambda and
are dropped.
"""
from __future__ import annotations

import math

import numpy as np

from .oracle import sparsity_from_margins


def sweep(margins_by_L: dict, lambdas) -> list:
    """[(lambda, L, S)] for every candidate lambda and every length L."""
    pts = []
    for L, g in margins_by_L.items():
        for lam in lambdas:
            pts.append((float(lam), int(L), sparsity_from_margins(g, lam)))
    return pts


def fit(points) -> tuple:
    """Least-squares fit of ln(lambda*L) = ln(a) + b*S; returns (a, b)."""
    xs, ys = [], []
    for lam, L, S in points:
        if lam <= 0 or S <= 0.0 or S >= 1.0:
            continue
        xs.append(S)
        ys.append(math.log(lam * L))
    if len(xs) < 2 or np.ptp(xs) == 0:
        raise ValueError("calibration: fewer than two informative points")
    A = np.stack([np.ones(len(xs)), np.asarray(xs)], axis=1)
    coef, *_ = np.linalg.lstsq(A, np.asarray(ys), rcond=None)
    return float(math.exp(coef[0])), float(coef[1])


def lambda_for(a: float, b: float, S: float, L: int) -> float:
    return a * math.exp(b * S) / L
