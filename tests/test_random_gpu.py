"""Randomized parity on the GPU: seeded random small problems (shapes, GQA ratio,
head size, mask, window, lambda, kernel variant, split count, page layout) against
the CPU oracle, to catch interactions the hand-picked edge cases miss.  Every case
is reproducible from its index."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from skip_softmax_flashattention_gb300 import blasst as K
from skip_softmax_flashattention_gb300 import workloads as W
from tests import parity

pytestmark = pytest.mark.gpu

PREFILL_FLAGS = [0, K.BLASST_PREFILL_ELIDE_V, K.BLASST_PREFILL_WIDE, K.BLASST_PREFILL_ONE_QTILE,
                 K.BLASST_PREFILL_P_VIA_SMEM]
LAMS = [0.0, 0.01, 0.1, 0.5, 1.0]


@pytest.fixture(autouse=True)
def _status_clean():
    K.blasst_device_status(1)
    yield
    assert K.blasst_device_status(1) == K.BLASST_OK, "a kernel wait timed out"


def _prefill_case(case):
    rng = np.random.default_rng(1000 + case)
    d = int(rng.choice([64, 128]))
    G = int(rng.choice([1, 2, 4]))
    Hkv = int(rng.integers(1, 3))
    B = int(rng.integers(1, 3))
    Lq = int(rng.integers(1, 700))
    Lkv = int(rng.integers(1, 900))
    causal = bool(rng.random() < 0.6)
    window = int(rng.choice([0, 0, 1, 37, 128, 300])) if causal else 0
    flags = int(rng.choice(PREFILL_FLAGS[:2] if window else PREFILL_FLAGS))
    lam = float(rng.choice(LAMS))
    return B, G * Hkv, Hkv, Lq, Lkv, d, causal, window, flags, lam


@pytest.mark.parametrize("case", range(40))
def test_random_prefill(case):
    B, Hq, Hkv, Lq, Lkv, d, causal, window, flags, lam = _prefill_case(case)
    a = parity.to_gpu(W.small_random(2000 + case, B, Hq, Hkv, Lq, Lkv, d, causal))
    res = K.prefill(a.q, a.k, a.v, causal, a.scale, lam, want_map=True, flags=flags, window=window)
    torch.cuda.synchronize()
    parity.prefill_full_check(a, res, lam, window=window)


@pytest.mark.parametrize("case", range(25))
def test_random_paged_decode(case):
    rng = np.random.default_rng(3000 + case)
    G = int(rng.choice([1, 2, 4, 8, 16]))
    Hkv = int(rng.integers(1, 3))
    B = int(rng.integers(1, 5))
    max_len = int(rng.integers(1, 2000))
    page_size = int(rng.choice([8, 16, 32, 64, 128, 256]))
    token_major = bool(rng.random() < 0.5)
    lens = [int(x) for x in rng.integers(0, max_len + 1, size=B)]
    window = int(rng.choice([0, 0, 1, 50, 200]))
    nT = -(-max_len // 128)
    S = int(rng.integers(1, min(4, nT) + 1))
    lam = float(rng.choice(LAMS))
    a = W.paged_decode(seed=4000 + case, B=B, Hq=G * Hkv, Hkv=Hkv, max_len=max_len, page_size=page_size,
                       token_major=token_major, lens=lens, device="cuda")
    e = a.extra
    res = K.decode_paged(a.q, e["k_pages"], e["v_pages"], e["page_table"], e["seq_lens"], max_len, page_size,
                         token_major, a.scale, lam, S, want_map=True, window=window)
    torch.cuda.synchronize()
    parity.decode_paged_check(a, res, lam, S, window=window)
