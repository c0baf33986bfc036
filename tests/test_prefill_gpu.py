"""Prefill parity on the GPU: the CUDA kernel against the CPU oracle.

Small problems are compared whole (every tile decision, the exact skipped count,
every output row); the full-size LLM-prefill, video-DiT and planted-70 workloads
are compared on sampled query tiles (first, last and random ones), in the same
launch configuration the benchmark times."""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

from skip_softmax_flashattention_gb300 import blasst as K
from skip_softmax_flashattention_gb300 import workloads as W
from tests import parity

pytestmark = pytest.mark.gpu

VARIANTS = [0, K.BLASST_PREFILL_ELIDE_V, K.BLASST_PREFILL_WIDE, K.BLASST_PREFILL_ONE_QTILE,
            K.BLASST_PREFILL_P_VIA_SMEM]
VARIANT_IDS = ["two-qtiles", "two-qtiles-elide-V", "two-qtiles-wide", "one-qtile-P-in-TMEM", "one-qtile-P-in-SMEM"]


@pytest.fixture(autouse=True)
def _status_clean():
    K.blasst_device_status(1)
    yield
    assert K.blasst_device_status(1) == K.BLASST_OK, "a kernel wait timed out"


@pytest.mark.parametrize("flags", VARIANTS, ids=VARIANT_IDS)
@pytest.mark.parametrize("planted", [False, True])
@pytest.mark.parametrize("lam", [0.0, 1e-3, 1e-2])
def test_tiny_workload(flags, planted, lam):
    a = parity.to_gpu(W.tiny(seed=0, planted=planted))
    res = K.prefill(a.q, a.k, a.v, a.causal, a.scale, lam, want_map=True, flags=flags)
    torch.cuda.synchronize()
    band, mx, mean, n = parity.prefill_full_check(a, res, lam)
    if lam == 0.0:
        assert n == 0
    if planted and lam == 1e-2:
        assert n == 16  # keys 256..511 = tiles 2,3 of every query tile: 2 heads x 4 q-tiles x 2


SHAPES = [
    # B, Hq, Hkv, Lq, Lkv, d, causal
    (1, 2, 1, 1, 1, 128, False),
    (1, 2, 2, 120, 120, 64, True),
    (2, 4, 2, 300, 300, 128, True),
    (1, 4, 1, 257, 1000, 128, True),   # Lq < Lkv: bottom-right diagonal
    (1, 2, 1, 500, 200, 128, True),    # Lq > Lkv: the first 300 rows see no key
    (1, 2, 2, 129, 513, 64, False),
    (1, 8, 2, 640, 640, 128, False),
]


@pytest.mark.parametrize("flags", VARIANTS, ids=VARIANT_IDS)
@pytest.mark.parametrize("shape", SHAPES, ids=[str(s) for s in SHAPES])
@pytest.mark.parametrize("lam", [0.0, 0.05, 0.5])
def test_ragged_and_edge_shapes(shape, lam, flags):
    B, Hq, Hkv, Lq, Lkv, d, causal = shape
    a = parity.to_gpu(W.small_random(11, B, Hq, Hkv, Lq, Lkv, d, causal, logit_mult=3.0))
    res = K.prefill(a.q, a.k, a.v, a.causal, a.scale, lam, want_map=True, flags=flags)
    torch.cuda.synchronize()
    parity.prefill_full_check(a, res, lam)


def test_margins_output_matches_oracle():
    a = parity.to_gpu(W.small_random(12, 1, 4, 2, 384, 640, 128, True, logit_mult=3.0))
    res = K.prefill(a.q, a.k, a.v, True, a.scale, 0.0, want_map=True, want_margins=True)
    torch.cuda.synchronize()
    from oracle import oracle as orc

    own = orc.prefill_tiled(a.q.float().cpu(), a.k.float().cpu(), a.v.float().cpu(), True, a.scale, 0.0)
    g = res["margins"].cpu().numpy()
    ref = own["margin"]
    assert np.array_equal(np.isnan(g), np.isnan(ref))
    fin = np.isfinite(ref)
    assert np.array_equal(np.isinf(g), np.isinf(ref))
    assert np.abs(g[fin] - ref[fin]).max() < 1e-3


def test_llm_prefill_full_size():
    L = 16384
    a = parity.to_gpu(W.llm(seed=0, L=L, device="cuda"))
    rng = np.random.default_rng(0)
    nQ = L // 128
    units = parity.sample_units(rng, 1, a.Hq, nQ, 6, always=[(0, 0, 0), (0, 31, nQ - 1), (0, 17, nQ // 2)])
    for A in (0, 4, 40):
        lam = A / L
        res = K.prefill(a.q, a.k, a.v, True, a.scale, lam, want_map=True)
        torch.cuda.synchronize()
        n = int(res["skipped"].item())
        assert n == int((res["map"] == 1).sum().item())
        if A == 0:
            assert n == 0
        parity.prefill_units_check(a, res, lam, units)


@pytest.mark.parametrize("L", [32768, 65536])
def test_llm_prefill_long_context_sampled(L):
    """The calibration lengths: causal LLM prefill at 32k and 64k keys (seed 1, as the
    calibration fit uses), at lambda = 0 and at lambda = 1 where 20-40 % of the tiles
    are skipped; the first, last and random query tiles checked against the oracle."""
    a = parity.to_gpu(W.llm(seed=1, L=L, device="cuda"))
    rng = np.random.default_rng(L)
    nQ = L // 128
    units = parity.sample_units(rng, 1, a.Hq, nQ, 3, always=[(0, 0, 0), (0, a.Hq - 1, nQ - 1)])
    for lam in (0.0, 1.0):
        res = K.prefill(a.q, a.k, a.v, True, a.scale, lam, want_map=True)
        torch.cuda.synchronize()
        n = int(res["skipped"].item())
        assert n == int((res["map"] == 1).sum().item())
        if lam == 0.0:
            assert n == 0
        else:
            assert n > 0
        parity.prefill_units_check(a, res, lam, units)
    del a, res
    torch.cuda.empty_cache()


@pytest.mark.parametrize("L,B,Hq,Hkv", [(16384, 3, 4, 1), (8192, 3, 8, 2)], ids=["L16384-B3-H4", "L8192-B3-H8"])
def test_causal_prefill_bands_with_a_partial_last_band(L, B, Hq, Hkv):
    """Causal CTAs run in bands of (sequence, head) pairs whose K/V fit an eighth of L2,
    longest-first within each band (two KV-head groups per band at L = 16384 and d = 128,
    four at 8192 on this part).  With an odd number of KV heads in all, the last band is
    partial.  The first, middle and last query tiles of every (sequence, head) pair are
    checked against the oracle, at lambda = 0 and at lambda = 1."""
    a = parity.to_gpu(W.llm(seed=5, L=L, B=B, Hq=Hq, Hkv=Hkv, device="cuda"))
    nQ = L // 128
    units = [(b, h, qt) for b in range(B) for h in range(Hq) for qt in (0, nQ // 2, nQ - 1)]
    for lam in (0.0, 1.0):
        res = K.prefill(a.q, a.k, a.v, True, a.scale, lam, want_map=True)
        torch.cuda.synchronize()
        n = int(res["skipped"].item())
        assert n == int((res["map"] == 1).sum().item())
        # every visited tile has a decision in the map (0 or 1), none is left unvisited
        visited = int((res["map"] != 2).sum().item())
        assert visited == B * Hq * (nQ * (nQ + 1) // 2)
        if lam == 0.0:
            assert n == 0
        parity.prefill_units_check(a, res, lam, units)
    del a, res
    torch.cuda.empty_cache()


def test_dit_full_size():
    a = parity.to_gpu(W.dit(seed=0, device="cuda"))
    rng = np.random.default_rng(1)
    nQ = -(-a.Lq // 128)
    units = parity.sample_units(rng, 1, a.Hq, nQ, 4, always=[(0, 0, 0), (0, a.Hq - 1, nQ - 1)])
    for lam in (0.0, 1e-4, 1e-3, 1e-2):
        res = K.prefill(a.q, a.k, a.v, False, a.scale, lam, want_map=True)
        torch.cuda.synchronize()
        n = int(res["skipped"].item())
        assert n == int((res["map"] == 1).sum().item())
        if lam == 0:
            assert n == 0
        parity.prefill_units_check(a, res, lam, units)


def test_planted70_skip_set_and_parity():
    L = 16384
    a = parity.to_gpu(W.planted70(seed=0, L=L, device="cuda"))
    first = a.extra["first_zero_tile"]
    res = K.prefill(a.q, a.k, a.v, False, a.scale, 1e-2, want_map=True)
    torch.cuda.synchronize()
    mp = res["map"].cpu().numpy()
    assert (mp[..., first:] == 1).all()
    assert (mp[..., :first] == 0).mean() > 0.99
    rng = np.random.default_rng(2)
    units = parity.sample_units(rng, 1, a.Hq, L // 128, 3, always=[(0, 0, 0)])
    parity.prefill_units_check(a, res, 1e-2, units)


@pytest.mark.parametrize("workload", ["planted70", "dit", "llm"])
def test_elide_v_is_bitwise_identical_at_full_size(workload):
    """Eliding V changes which V tiles are loaded, never what is computed: outputs,
    lse, skip map and count equal the default kernel's bit for bit, with skips
    (planted-70 at 70 %, DiT at 51 %) and without (LLM prefill)."""
    if workload == "planted70":
        a, causal, lam = W.planted70(seed=0, L=16384, device="cuda"), False, 1e-2
    elif workload == "dit":
        a, causal, lam = W.dit(seed=0, device="cuda"), False, 1e-2
    else:
        a, causal, lam = W.llm(seed=0, L=16384, device="cuda"), True, 40 / 16384
    a = parity.to_gpu(a)
    ref = K.prefill(a.q, a.k, a.v, causal, a.scale, lam, want_map=True)
    got = K.prefill(a.q, a.k, a.v, causal, a.scale, lam, want_map=True, flags=K.BLASST_PREFILL_ELIDE_V)
    torch.cuda.synchronize()
    assert torch.equal(got["map"], ref["map"])
    assert int(got["skipped"].item()) == int(ref["skipped"].item())
    assert torch.equal(got["o"], ref["o"])
    assert torch.equal(got["lse"], ref["lse"])
    if workload != "llm":
        assert int(ref["skipped"].item()) > 0


WINDOW_SHAPES = [(1, 4, 2, 1000, 1000, 128), (1, 4, 1, 257, 1000, 128), (2, 2, 2, 300, 300, 64),
                 (1, 2, 2, 1000, 700, 128)]


@pytest.mark.parametrize("shape", WINDOW_SHAPES, ids=[str(s) for s in WINDOW_SHAPES])
@pytest.mark.parametrize("window", [1, 64, 128, 129, 300, 5000])
@pytest.mark.parametrize("flags", [0, K.BLASST_PREFILL_ELIDE_V], ids=["two-qtiles", "two-qtiles-elide-V"])
def test_sliding_window_matches_oracle(shape, window, flags):
    B, Hq, Hkv, Lq, Lkv, d = shape
    a = parity.to_gpu(W.small_random(31 + window, B, Hq, Hkv, Lq, Lkv, d, True))
    for lam in (0.0, 0.05, 0.5):
        res = K.prefill(a.q, a.k, a.v, True, a.scale, lam, want_map=True, flags=flags, window=window)
        torch.cuda.synchronize()
        parity.prefill_full_check(a, res, lam, window=window)


def test_sliding_window_covering_all_keys_equals_causal_bitwise():
    a = parity.to_gpu(W.small_random(77, 1, 4, 2, 900, 1100, 128, True))
    for lam in (0.0, 0.3):
        ref = K.prefill(a.q, a.k, a.v, True, a.scale, lam, want_map=True)
        got = K.prefill(a.q, a.k, a.v, True, a.scale, lam, want_map=True, window=1100)
        torch.cuda.synchronize()
        assert torch.equal(got["map"], ref["map"]) and torch.equal(got["o"], ref["o"])
        assert torch.equal(got["lse"], ref["lse"])


def test_sliding_window_llm_full_size_sampled():
    """LLM prefill at 16k keys with a 4096-key window: sampled query tiles."""
    L, Wn = 16384, 4096
    a = parity.to_gpu(W.llm(seed=0, L=L, device="cuda"))
    rng = np.random.default_rng(5)
    nQ = L // 128
    units = parity.sample_units(rng, 1, a.Hq, nQ, 4, always=[(0, 0, 0), (0, 31, nQ - 1), (0, 3, 40)])
    for lam in (0.0, 40 / Wn, 0.3):
        res = K.prefill(a.q, a.k, a.v, True, a.scale, lam, want_map=True, window=Wn)
        torch.cuda.synchronize()
        mp = res["map"]
        assert int(res["skipped"].item()) == int((mp == 1).sum().item())
        # a query tile visits at most ceil(W/128) + 1 key tiles
        assert int((mp != 2).sum(dim=-1).max().item()) <= Wn // 128 + 1
        parity.prefill_units_check(a, res, lam, units, window=Wn)


def test_short_watchdog_reports_timeout_and_context_survives():
    """Waits with a ~1 us limit give up; the kernel records a timeout, drains its
    copies, frees its tensor memory and exits; the next normal call is correct."""
    a = parity.to_gpu(W.small_random(13, 1, 4, 2, 1024, 4096, 128, True))
    K.blasst_device_status(1)
    K.prefill(a.q, a.k, a.v, True, a.scale, 0.0, flags=K.BLASST_FLAG_TEST_SHORT_WATCHDOG)
    assert K.blasst_device_status(1) == K.BLASST_ERR_TIMEOUT
    res = K.prefill(a.q, a.k, a.v, True, a.scale, 0.0, want_map=True)
    torch.cuda.synchronize()
    assert K.blasst_device_status(0) == K.BLASST_OK
    parity.prefill_full_check(a, res, 0.0)


@pytest.mark.parametrize("flags", [0, K.BLASST_PREFILL_ELIDE_V], ids=["two-qtiles", "two-qtiles-elide-V"])
@pytest.mark.parametrize("causal", [False, True])
def test_long_runs_of_skipped_tiles(flags, causal):
    """The last 90 % of the keys hold K = 0, so at lambda = 0.1 almost every key tile
    after the first few is skipped by both query tiles of a CTA: long runs in which the
    MMA issuers wait for no V tile and run ahead of the V producer by as much as the
    kernel allows.  Every decision, the exact count, O and lse against the oracle."""
    a = W.planted70(seed=5, L=4096, Hq=4, Hkv=2, device="cuda", frac=0.9)
    a.causal = causal
    res = K.prefill(a.q, a.k, a.v, a.causal, a.scale, 0.1, want_map=True, flags=flags)
    torch.cuda.synchronize()
    band, mx, mean, n = parity.prefill_full_check(a, res, 0.1)
    visited = int((res["map"] != 2).sum().item())
    assert n > 0.75 * visited, (n, visited)


def test_long_skip_runs_in_a_window():
    """The same with a causal sliding window of 1000 keys (windowed CTAs start their key
    walk past tile 0)."""
    a = W.planted70(seed=6, L=4096, Hq=4, Hkv=2, device="cuda", frac=0.9)
    a.causal = True
    for flags in (0, K.BLASST_PREFILL_ELIDE_V):
        res = K.prefill(a.q, a.k, a.v, True, a.scale, 0.1, want_map=True, flags=flags, window=1000)
        torch.cuda.synchronize()
        parity.prefill_full_check(a, res, 0.1, window=1000)
