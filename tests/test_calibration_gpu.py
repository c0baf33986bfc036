"""Threshold calibration on the GPU (BLASST talk notes, "threshold calibration",
Algorithm 2, Table 6): per-tile margins from one lambda = 0 launch decide the
sparsity of every threshold, a threshold picked from them for a target sparsity
skips exactly the tiles the margins say, and one fixed threshold skips more at
longer contexts."""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

from skip_softmax_flashattention_gb300 import blasst as K
from skip_softmax_flashattention_gb300 import calibrate
from skip_softmax_flashattention_gb300 import workloads as W
from tests import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _status_clean():
    K.blasst_device_status(1)
    yield
    assert K.blasst_device_status(1) == K.BLASST_OK, "a kernel wait timed out"
    torch.cuda.empty_cache()


def _margins(L, seed=1):
    a = W.llm(seed=seed, L=L, device="cuda")
    r = K.prefill(a.q, a.k, a.v, True, a.scale, 0.0, want_margins=True)
    torch.cuda.synchronize()
    return a, r["margins"].cpu().numpy()


def test_threshold_from_gpu_margins_reaches_its_target():
    """Causal GQA prefill, L = 16384: the threshold the harness reads off the GPU
    margins for 5 % sparsity skips, in the kernel, exactly the tiles whose margins
    are below its logarithm (up to the 1e-3 band)."""
    a, g = _margins(16384)
    lam = calibrate.lambda_for_sparsity(g, 0.05)
    assert 0.0 < lam <= 1.0
    res = K.prefill(a.q, a.k, a.v, True, a.scale, lam, want_map=True)
    torch.cuda.synchronize()
    gmap = res["map"].cpu().numpy()
    pred = parity.oracle_map_at(g, lam)
    vis = pred != 2
    assert np.array_equal(gmap == 2, ~vis)
    diff = vis & (gmap != pred)
    band = np.abs(g.astype(np.float64) - math.log(lam)) < parity.BAND
    assert not (diff & ~band).any()
    n = int(res["skipped"].item())
    assert n == int((gmap == 1).sum())
    n_pred = int((pred == 1).sum())
    assert n_pred >= 0.05 * int(vis.sum())
    assert abs(n - n_pred) <= int(diff.sum())


def test_fixed_threshold_skips_more_at_longer_contexts():
    """The trend of Table 6 on the long-context workload's calibration seed: at each
    fixed threshold that skips anything, the sparsity does not fall as the context
    grows from 8192 to 32768 keys (and grows overall)."""
    by_len = {}
    for L in (8192, 16384, 32768):
        _, g = _margins(L)
        by_len[L] = g
    for lam in (0.1, 0.3, 1.0):
        s = [calibrate.sparsity_at(by_len[L], lam) for L in sorted(by_len)]
        if s[-1] == 0:
            continue
        assert all(b >= a for a, b in zip(s, s[1:])), (lam, s)
    s1 = [calibrate.sparsity_at(by_len[L], 1.0) for L in sorted(by_len)]
    assert s1[-1] > s1[0], s1
