"""The whole-problem parity checks decide every threshold from one lambda = 0 oracle
pass (tests.parity.oracle_map_at).  That shortcut must give exactly the map of the
oracle run at each threshold, on prefill (causal, GQA, ragged) and split decode."""
from __future__ import annotations

import numpy as np
import pytest

from oracle import oracle as orc
from skip_softmax_flashattention_gb300 import workloads as W
from tests import parity

LAMS = [0.0, 1e-4, 1e-3, 1e-2, 0.05, 0.3, 1.0]


@pytest.mark.parametrize("shape", [(1, 4, 2, 300, 300, 64, True), (1, 2, 2, 129, 513, 64, False),
                                   (1, 2, 1, 500, 200, 64, True)])
def test_prefill_map_from_margins_equals_oracle_runs(shape):
    B, Hq, Hkv, Lq, Lkv, d, causal = shape
    a = W.small_random(21, B, Hq, Hkv, Lq, Lkv, d, causal, logit_mult=3.0)
    q, k, v = a.q.float(), a.k.float(), a.v.float()
    own0 = orc.prefill_tiled(q, k, v, causal, a.scale, 0.0, Br=32, Bc=32)
    for lam in LAMS:
        r = orc.prefill_tiled(q, k, v, causal, a.scale, lam, Br=32, Bc=32)
        assert np.array_equal(parity.oracle_map_at(own0["margin"], lam), r["map"]), lam
        assert int((r["map"] == 1).sum()) == r["skipped"]


def test_planted_tiny_map_from_margins():
    a = W.tiny(seed=0, planted=True)
    q, k, v = a.q.float(), a.k.float(), a.v.float()
    own0 = orc.prefill_tiled(q, k, v, a.causal, a.scale, 0.0)
    for lam in LAMS:
        r = orc.prefill_tiled(q, k, v, a.causal, a.scale, lam)
        assert np.array_equal(parity.oracle_map_at(own0["margin"], lam), r["map"]), lam


@pytest.mark.parametrize("S", [1, 3])
def test_decode_map_from_margins_equals_oracle_runs(S):
    a = W.decode(seed=3, B=3, Hq=8, Hkv=2, Lkv=1000, device="cpu")
    q, k, v = a.q.float(), a.k.float(), a.v.float()
    own0 = orc.decode_tiled(q, k, v, a.scale, 0.0, num_splits=S, Bc=32)
    for lam in LAMS:
        r = orc.decode_tiled(q, k, v, a.scale, lam, num_splits=S, Bc=32)
        assert np.array_equal(parity.oracle_map_at(own0["margin"], lam), r["map"]), lam
