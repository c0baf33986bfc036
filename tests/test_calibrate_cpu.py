"""The calibration harness (skip_softmax_flashattention_gb300/calibrate.py) against
the oracle's calibration (BLASST talk notes, "threshold calibration", Algorithm 2
and Eq. 3).  The harness turns per-tile margins into the sparsity of every
candidate threshold, fits lambda * L = a * exp(b * S), and picks the threshold that
reaches a target sparsity; the bench derives its 70 % thresholds and the long-context
fit from it.  Every function must agree with the oracle's on the same margins."""
from __future__ import annotations

import math

import numpy as np
import pytest

from oracle import calibration as ocal
from oracle import oracle as orc
from skip_softmax_flashattention_gb300 import calibrate


def _margins(seed, n=4000, visited=0.8):
    """Synthetic per-tile margins: non-positive values like a real pass (m~ - m <= 0),
    some exact zeros (the tile that sets the running max), some +inf (a row with no
    visible key yet) and NaN for tiles that were not visited."""
    rng = np.random.default_rng(seed)
    g = -np.abs(rng.normal(0.0, 3.0, n))
    g[rng.random(n) < 0.05] = 0.0
    g[rng.random(n) < 0.01] = math.inf
    g[rng.random(n) > visited] = math.nan
    return g.reshape(8, -1)


LAMBDAS = [0.0, 1e-9, 1e-4, 1e-3, 1e-2, 0.05, 0.3, 0.9, 1.0]


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_sparsity_matches_the_oracle(seed):
    g = _margins(seed)
    for lam in LAMBDAS:
        assert calibrate.sparsity_at(g, lam) == orc.sparsity_from_margins(g, lam)


def test_sweep_matches_the_oracle():
    by_len = {8192: _margins(3), 32768: _margins(4, n=8000), 65536: _margins(5, n=16000)}
    cands = [float(x) for x in np.logspace(-6, 0, 25)]
    assert calibrate.sweep(by_len, cands) == ocal.sweep(by_len, cands)


def test_fit_matches_the_oracle():
    by_len = {8192: _margins(6), 32768: _margins(7, n=8000), 65536: _margins(8, n=16000)}
    pts = calibrate.sweep(by_len, [float(x) for x in np.logspace(-6, 0, 25)])
    a, b = calibrate.fit(pts)
    ao, bo = ocal.fit(pts)
    assert a == pytest.approx(ao, rel=1e-12)
    assert b == pytest.approx(bo, rel=1e-12)


def test_fit_without_informative_points():
    # every point at S = 0 (or 1): the harness returns None where the oracle refuses
    pts = [(1e-3, 8192, 0.0), (1e-2, 8192, 0.0), (0.5, 32768, 1.0)]
    assert calibrate.fit(pts) is None
    with pytest.raises(ValueError):
        ocal.fit(pts)


def test_fit_recovers_a_known_curve():
    a0, b0 = 1234.5, 4.25
    pts = [(a0 * math.exp(b0 * s) / L, L, s) for L in (8192, 32768) for s in (0.1, 0.3, 0.55, 0.8)]
    a, b = calibrate.fit(pts)
    assert a == pytest.approx(a0, rel=1e-9) and b == pytest.approx(b0, rel=1e-9)


@pytest.mark.parametrize("seed", [0, 1, 2, 3])
@pytest.mark.parametrize("target", [0.0, 0.01, 0.25, 0.5, 0.7, 0.85])
def test_lambda_for_sparsity_is_the_smallest_that_reaches_the_target(seed, target):
    g = _margins(seed)
    lam = calibrate.lambda_for_sparsity(g, target)
    s = orc.sparsity_from_margins(g, lam)
    vis = np.sort(g[~np.isnan(g)])
    if target == 0.0:
        assert lam == 0.0
        return
    k = math.ceil(target * vis.size)
    if vis[k - 1] >= 0.0:
        # no threshold <= 1 skips a tile whose margin is >= 0 = ln 1
        assert lam == 1.0 and s < target
        return
    assert 0.0 < lam <= 1.0
    assert s >= target
    # just below the k-th smallest margin the target is missed
    lam_lo = math.exp(vis[k - 1]) * (1.0 - 1e-9)
    assert orc.sparsity_from_margins(g, lam_lo) < target


def test_lambda_for_sparsity_unreachable_target():
    g = np.array([[-5.0, -1.0, 0.0, 0.0, math.inf, math.nan]])
    # 2 of the 5 visited tiles can be skipped at lambda <= 1
    assert calibrate.lambda_for_sparsity(g, 0.4) == pytest.approx(math.exp(-1.0), rel=1e-5)
    assert calibrate.lambda_for_sparsity(g, 0.6) == 1.0
    assert orc.sparsity_from_margins(g, 1.0) == pytest.approx(0.4)


def test_harness_on_oracle_margins_of_a_planted_workload():
    # margins from the oracle's own tiled pass: the threshold the harness picks for
    # 50 % reproduces, through the oracle's skip test, exactly the planted half
    from skip_softmax_flashattention_gb300 import workloads as W

    a = W.tiny(seed=0, planted=True)
    r0 = orc.prefill_tiled(a.q.float(), a.k.float(), a.v.float(), a.causal, a.scale, 0.0, precision="f32")
    lam = calibrate.lambda_for_sparsity(r0["margin"], 0.5)
    r = orc.prefill_tiled(a.q.float(), a.k.float(), a.v.float(), a.causal, a.scale, lam, precision="f32")
    assert r["skipped"] == int(np.count_nonzero(r0["margin"] < math.log(lam)))
    assert r["skipped"] / np.count_nonzero(~np.isnan(r0["margin"])) >= 0.5
