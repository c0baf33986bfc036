"""Pins for the CPU oracle: checks against things other than the oracle itself.

Each test ties the oracle to a closed form, a textbook definition computed a
different way (numpy matmul / pure-Python loops), an invariant the method fixes,
or a worked example printed on the pages.  None of these tests needs a GPU.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import calibration, lambda_resolution
from oracle import oracle as orc
from skip_softmax_flashattention_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- helpers ---
def np_dense(q, k, v, causal, scale, rows=None, window=0):
    """Textbook attention with a library matmul (float64): softmax(scale*QK^T)V.

    q [B,Hq,Lq,d], k/v [B,Hkv,Lkv,d].  ``rows`` optionally restricts to a list of
    (b, h, r) query rows.  Returns dict (b,h,r) -> (o row, lse) or full arrays."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    B, Hq, Lq, d = q.shape
    Hkv, Lkv = k.shape[1], k.shape[2]
    G = Hq // Hkv
    if rows is None:
        o = np.zeros_like(q)
        lse = np.zeros((B, Hq, Lq))
        for b in range(B):
            for h in range(Hq):
                s = scale * q[b, h] @ k[b, h // G].T
                if causal:
                    r = np.arange(Lq)[:, None]
                    c = np.arange(Lkv)[None, :]
                    s = np.where(band(r, c, Lq, Lkv, window), s, -np.inf)
                M = s.max(axis=1, keepdims=True)
                Mf = np.where(np.isfinite(M), M, 0.0)
                p = np.exp(s - Mf)
                z = p.sum(axis=1, keepdims=True)
                with np.errstate(invalid="ignore", divide="ignore"):
                    o[b, h] = np.where(z > 0, (p @ v[b, h // G]) / np.where(z > 0, z, 1), 0)
                    lse[b, h] = np.where(z[:, 0] > 0, Mf[:, 0] + np.log(np.where(z[:, 0] > 0, z[:, 0], 1)), -np.inf)
        return o, lse
    out = {}
    for (b, h, r) in rows:
        s = scale * k[b, h // G] @ q[b, h, r]
        if causal:
            s = np.where(np.arange(Lkv) <= r + (Lkv - Lq), s, -np.inf)
        M = s.max()
        p = np.exp(s - M)
        out[(b, h, r)] = (p @ v[b, h // G] / p.sum(), M + math.log(p.sum()))
    return out


def band(r, c, Lq, Lkv, window):
    """Causal visibility as a band of the score matrix: the key may not lie past the
    row's own position r' = r + Lkv - Lq, and with a window W > 0 not W or more
    keys before it."""
    rr = r + (Lkv - Lq)
    ok = c <= rr
    if window > 0:
        ok = ok & (rr - c < window)
    return ok


def closed_form_skip(q, k, causal, scale, lam, Br, Bc, Lq_rows=None, window=0):
    """Skip map from the dense score matrix, without the online loop.

    For query tile i and key tile j: the running max of row r after tile j is the
    max of its visible scores over key tiles 0..j; the tile's max m~ is the max over
    tile j.  Tile skipped iff every row has m~ - runmax < ln(lambda).  Returns
    (map [B,Hq,nQ,nK] with 0/1/2, margin)."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    B, Hq, Lq, d = q.shape
    Hkv, Lkv = k.shape[1], k.shape[2]
    G = Hq // Hkv
    nQ, nK = -(-Lq // Br), -(-Lkv // Bc)
    ln = -math.inf if lam <= 0 else math.log(lam)
    mp = np.zeros((B, Hq, nQ, nK), np.uint8)
    mg = np.full((B, Hq, nQ, nK), np.nan)
    for b in range(B):
        for h in range(Hq):
            s = scale * q[b, h] @ k[b, h // G].T
            r = np.arange(Lq)[:, None]
            c = np.arange(Lkv)[None, :]
            vis = np.ones_like(s, bool) if not causal else band(r, c, Lq, Lkv, window)
            s = np.where(vis, s, -np.inf)
            for i in range(nQ):
                rows = slice(i * Br, min(Lq, (i + 1) * Br))
                run = np.full(rows.stop - rows.start, -np.inf)
                for j in range(nK):
                    cols = slice(j * Bc, min(Lkv, (j + 1) * Bc))
                    if not vis[rows, cols].any():
                        mp[b, h, i, j] = 2
                        continue
                    mt = s[rows, cols].max(axis=1)
                    run = np.maximum(run, mt)
                    with np.errstate(invalid="ignore"):
                        diff = mt - run
                    votes = diff < ln
                    mp[b, h, i, j] = 1 if votes.all() else 0
                    both_inf = np.isneginf(mt) & np.isneginf(run)
                    mg[b, h, i, j] = np.max(np.where(both_inf, np.inf, diff))
    return mp, mg


def rnd(seed, *shape):
    g = np.random.default_rng(seed)
    return g.standard_normal(shape)


# ------------------------------------------------------------ dense pins ---
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", [(1, 2, 2, 37, 37, 8), (2, 4, 2, 20, 29, 16), (1, 3, 1, 33, 17, 8)])
def test_dense_matches_textbook_matmul(causal, shape):
    B, Hq, Hkv, Lq, Lkv, d = shape
    q, k, v = rnd(1, B, Hq, Lq, d), rnd(2, B, Hkv, Lkv, d), rnd(3, B, Hkv, Lkv, d)
    o, lse = orc.dense(q, k, v, causal, 0.7, precision="f64")
    o2, lse2 = np_dense(q, k, v, causal, 0.7)
    np.testing.assert_allclose(o, o2, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse, lse2, rtol=1e-12, atol=1e-12)


def test_dense_closed_forms():
    B, H, L, d = 1, 2, 50, 8
    q = rnd(4, B, H, L, d)
    v = rnd(5, B, H, L, d)
    # identical keys -> uniform weights: O = mean of V, lse = s + ln(L)
    k = np.repeat(rnd(6, B, H, 1, d), L, axis=2)
    o, lse = orc.dense(q, k, v, False, 0.5, precision="f64")
    np.testing.assert_allclose(o, np.broadcast_to(v.mean(axis=2, keepdims=True), o.shape), atol=1e-12)
    s = 0.5 * np.einsum("bhld,bhd->bhl", q, k[:, :, 0])
    np.testing.assert_allclose(lse, s + math.log(L), atol=1e-12)
    # causal with zero keys: row r sees r+1 keys -> lse = ln(r+1), O = mean of V[0..r]
    k0 = np.zeros((B, H, L, d))
    o, lse = orc.dense(q, k0, v, True, 1.0, precision="f64")
    np.testing.assert_allclose(lse[0, 0], np.log(np.arange(1, L + 1)), atol=1e-12)
    np.testing.assert_allclose(o[0, 1], np.cumsum(v[0, 1], axis=0) / np.arange(1, L + 1)[:, None], atol=1e-12)
    # constant V rows -> O is that constant whatever the weights
    vc = np.broadcast_to(rnd(7, B, H, 1, d), v.shape).copy()
    o, _ = orc.dense(q, rnd(8, B, H, L, d), vc, True, 2.0, precision="f64")
    np.testing.assert_allclose(o, vc, atol=1e-12)


def test_dense_fully_masked_rows():
    # causal with Lq > Lkv: the first Lq-Lkv rows see no key -> O = 0, lse = -inf
    q, k, v = rnd(9, 1, 1, 10, 4), rnd(10, 1, 1, 6, 4), rnd(11, 1, 1, 6, 4)
    o, lse = orc.dense(q, k, v, True, 1.0, precision="f64")
    assert np.all(o[0, 0, :4] == 0) and np.all(np.isneginf(lse[0, 0, :4]))
    assert np.all(np.isfinite(lse[0, 0, 4:]))


# ------------------------------------------------- online recurrence pins ---
def brute_force_tiled(q, k, v, causal, scale, lam, Br, Bc):
    """Pure-Python (float) version of the tiled pass for tiny inputs: the same
    recurrence written with explicit loops, used to pin the C oracle's indexing."""
    B, Hq, Lq, d = q.shape
    Hkv, Lkv = k.shape[1], k.shape[2]
    G = Hq // Hkv
    nQ, nK = -(-Lq // Br), -(-Lkv // Bc)
    ln = -math.inf if lam <= 0 else math.log(lam)
    O = np.zeros(q.shape)
    LSE = np.zeros((B, Hq, Lq))
    MAP = np.zeros((B, Hq, nQ, nK), np.uint8)
    for b in range(B):
        for h in range(Hq):
            for i in range(nQ):
                rows = list(range(i * Br, min(Lq, (i + 1) * Br)))
                m = {r: -math.inf for r in rows}
                l = {r: 0.0 for r in rows}
                acc = {r: [0.0] * d for r in rows}
                for j in range(nK):
                    cols = list(range(j * Bc, min(Lkv, (j + 1) * Bc)))
                    vis = lambda r, c: (not causal) or c <= r + (Lkv - Lq)
                    if not any(vis(r, c) for r in rows for c in cols):
                        MAP[b, h, i, j] = 2
                        continue
                    S = {}
                    for r in rows:
                        for c in cols:
                            S[r, c] = (scale * sum(q[b, h, r, x] * k[b, h // G, c, x] for x in range(d))
                                       if vis(r, c) else -math.inf)
                    mt = {r: max(S[r, c] for c in cols) for r in rows}
                    mn = {r: max(m[r], mt[r]) for r in rows}
                    skip = True
                    for r in rows:
                        if mt[r] == -math.inf and mn[r] == -math.inf:
                            skip = False
                        elif not (mt[r] - mn[r] < ln):
                            skip = False
                    MAP[b, h, i, j] = 1 if skip else 0
                    if skip:
                        continue
                    for r in rows:
                        if mn[r] == -math.inf:
                            continue
                        alpha = 0.0 if m[r] == -math.inf else math.exp(m[r] - mn[r])
                        ps = [math.exp(S[r, c] - mn[r]) if S[r, c] > -math.inf else 0.0 for c in cols]
                        l[r] = alpha * l[r] + sum(ps)
                        acc[r] = [alpha * acc[r][x] + sum(p * v[b, h // G, c, x] for p, c in zip(ps, cols))
                                  for x in range(d)]
                        m[r] = mn[r]
                for r in rows:
                    if l[r] > 0:
                        O[b, h, r] = [a / l[r] for a in acc[r]]
                        LSE[b, h, r] = m[r] + math.log(l[r])
                    else:
                        LSE[b, h, r] = -math.inf
    return O, LSE, MAP


@pytest.mark.parametrize("tiles", [(1, 1), (2, 2), (4, 4), (2, 4), (4, 1)])
@pytest.mark.parametrize("causal", [False, True])
def test_tiled_matches_brute_force_tiny(tiles, causal):
    Br, Bc = tiles
    B, Hq, Hkv, Lq, Lkv, d = 1, 2, 1, 7, 11, 3
    q, k, v = rnd(12, B, Hq, Lq, d), rnd(13, B, Hkv, Lkv, d), rnd(14, B, Hkv, Lkv, d)
    for lam in (0.0, 0.2, 0.6):
        res = orc.prefill_tiled(q, k, v, causal, 1.3, lam, Br, Bc, precision="f64")
        O, LSE, MAP = brute_force_tiled(q, k, v, causal, 1.3, lam, Br, Bc)
        np.testing.assert_array_equal(res["map"], MAP)
        np.testing.assert_allclose(res["o"], O, atol=1e-12)
        np.testing.assert_allclose(res["lse"], LSE, atol=1e-12)


@pytest.mark.parametrize("Br,Bc", [(1, 1), (2, 4), (16, 8)])
def test_tiled_lambda0_equals_dense_small(Br, Bc):
    for causal in (False, True):
        q, k, v = rnd(15, 2, 4, 40, 8), rnd(16, 2, 2, 45, 8), rnd(17, 2, 2, 45, 8)
        res = orc.prefill_tiled(q, k, v, causal, 0.9, 0.0, Br, Bc, precision="f64")
        o, lse = np_dense(q, k, v, causal, 0.9)
        assert res["skipped"] == 0
        np.testing.assert_allclose(res["o"], o, atol=1e-12)
        np.testing.assert_allclose(res["lse"], lse, atol=1e-12)


def test_tiny_config_lambda0_equals_dense_fp32():
    """Tiny workload, fp32 copy: the fp32 tiled pass at lambda=0 equals dense
    attention to 1e-5 relative, and no tile is skipped."""
    a = W.tiny(seed=0, fp32=True)
    res = orc.prefill_tiled(a.q, a.k, a.v, a.causal, a.scale, 0.0, precision="f32")
    o, lse = np_dense(a.q.numpy(), a.k.numpy(), a.v.numpy(), a.causal, a.scale)
    assert res["skipped"] == 0
    rel = np.abs(res["o"] - o).max() / np.abs(o).max()
    assert rel < 1e-5, rel
    assert np.abs(res["lse"] - lse).max() / np.abs(lse).max() < 1e-5
    od, lsed = orc.dense(a.q, a.k, a.v, a.causal, a.scale, precision="f32")
    assert np.abs(od - o).max() / np.abs(o).max() < 1e-5


@pytest.mark.slow
def test_sampled_slices_of_llm_and_dit_lambda0():
    """Full-size LLM-prefill and video-DiT shapes: sampled query tiles of the
    tiled pass at lambda=0 equal the textbook rows; nothing is skipped."""
    for a, units in ((W.llm(seed=0, L=16384), [(0, 0, 0), (0, 13, 64), (0, 31, 127)]),
                     (W.dit(seed=0, H=2), [(0, 0, 0), (0, 1, 255)])):
        res = orc.prefill_tiled(a.q, a.k, a.v, a.causal, a.scale, 0.0, units=units, precision="f32")
        assert res["skipped"] == 0
        rows = [(b, h, t * 128 + r) for (b, h, t) in units for r in (0, 57, 127) if t * 128 + r < a.Lq]
        ref = np_dense(a.q.float().numpy(), a.k.float().numpy(), a.v.float().numpy(), a.causal, a.scale, rows=rows)
        for (b, h, r), (orow, l) in ref.items():
            assert np.abs(res["o"][b, h, r] - orow).max() <= 1e-5 * max(1.0, np.abs(orow).max())
            assert abs(res["lse"][b, h, r] - l) <= 1e-5 * abs(l)


# --------------------------------------------------------- skip-set pins ---
@pytest.mark.parametrize("causal", [False, True])
def test_skip_set_equals_closed_form(causal):
    a = W.tiny(seed=3, fp32=True)
    q, k = a.q.numpy().astype(np.float64), a.k.numpy().astype(np.float64)
    for lam in (0.0, 1e-3, 1e-2, 0.1, 0.5, 1.0):
        res = orc.prefill_tiled(a.q, a.k, a.v, causal, a.scale, lam, 128, 128, precision="f64")
        mp, mg = closed_form_skip(q, k, causal, a.scale, lam, 128, 128)
        np.testing.assert_array_equal(res["map"], mp)
        np.testing.assert_allclose(res["margin"], mg, atol=1e-12)
        assert res["skipped"] == int((mp == 1).sum())


def test_skip_set_closed_form_small_tiles_gqa():
    q, k, v = rnd(20, 2, 4, 64, 8), rnd(21, 2, 2, 72, 8), rnd(22, 2, 2, 72, 8)
    for causal in (False, True):
        for lam in (0.05, 0.3, 0.9):
            res = orc.prefill_tiled(q, k, v, causal, 1.5, lam, 16, 8, precision="f64")
            mp, mg = closed_form_skip(q, k, causal, 1.5, lam, 16, 8)
            np.testing.assert_array_equal(res["map"], mp)


def test_margins_are_lambda_independent_and_nested():
    a = W.tiny(seed=5, fp32=True)
    maps = []
    lams = [1e-4, 1e-3, 1e-2, 0.05, 0.2, 0.7, 1.0]
    g0 = orc.prefill_tiled(a.q, a.k, a.v, True, a.scale, 0.0, precision="f64")["margin"]
    for lam in lams:
        r = orc.prefill_tiled(a.q, a.k, a.v, True, a.scale, lam, precision="f64")
        np.testing.assert_array_equal(np.isnan(r["margin"]), np.isnan(g0))
        np.testing.assert_allclose(r["margin"][~np.isnan(g0)], g0[~np.isnan(g0)], atol=0)
        maps.append(r["map"] == 1)
        assert r["skipped"] == int(round(orc.sparsity_from_margins(g0, lam) * (~np.isnan(g0)).sum()))
    for lo, hi in zip(maps, maps[1:]):
        assert np.all(hi | ~lo)  # a tile skipped at a smaller lambda stays skipped


def test_planted_gap_30():
    """Planted keys scoring >= 30 below the row max are skipped at every lambda in
    [1e-13, 1], and the whole map equals the closed-form prediction."""
    g = np.random.default_rng(30)
    d, L = 64, 512
    u = np.zeros(d)
    u[0] = math.sqrt(d)
    q = g.standard_normal((1, 1, L, d)) + u
    k = g.standard_normal((1, 1, L, d))
    k[0, 0, 256:512] = -8 * u
    v = g.standard_normal((1, 1, L, d))
    scale = 1 / math.sqrt(d)
    s = scale * q[0, 0] @ k[0, 0].T
    gap = s[:, :256].max(axis=1)[:, None] - s[:, 256:]
    assert gap.min() >= 30
    for lam in (1e-13, 1e-9, 1e-6, 1e-3, 0.5, 1.0):
        res = orc.prefill_tiled(q, k, v, False, scale, lam, precision="f64")
        assert np.all(res["map"][0, 0, :, 2:] == 1)
        mp, _ = closed_form_skip(q, k, False, scale, lam, 128, 128)
        np.testing.assert_array_equal(res["map"], mp)
    res = orc.prefill_tiled(q, k, v, False, scale, 1e-3, precision="f64")
    assert np.all(res["map"][0, 0, :, :2] == 0)


def test_planted_tiny_workload_skip_counts():
    """The tiny workload's planted variant (keys 256..511 = -2 mean(Q)): its
    skip set equals the closed form at the thresholds the workload names."""
    a = W.tiny(seed=0, planted=True)
    q, k = a.q.float().numpy(), a.k.float().numpy()
    for lam in (0.0, 1e-3, 1e-2):
        res = orc.prefill_tiled(a.q, a.k, a.v, False, a.scale, lam, precision="f64")
        mp, _ = closed_form_skip(q, k, False, a.scale, lam, 128, 128)
        np.testing.assert_array_equal(res["map"], mp)
        if lam == 0.0:
            assert res["skipped"] == 0


# --------------------------------------------- skipped-contribution pins ---
@pytest.mark.parametrize("lam", [1e-3, 1e-2, 0.1, 0.5])
def test_skipped_contribution_closed_form(lam):
    a = W.tiny(seed=7, fp32=True)
    q = a.q.numpy().astype(np.float64)
    k = a.k.numpy().astype(np.float64)
    v = a.v.numpy().astype(np.float64)
    res = orc.prefill_tiled(q, k, v, True, a.scale, lam, precision="f64")
    o_d, lse_d = np_dense(q, k, v, True, a.scale)
    B, H, L, d = q.shape
    vmax = np.abs(v).max()
    for h in range(H):
        s = a.scale * q[0, h] @ k[0, h].T
        s = np.where(np.arange(L)[None, :] <= np.arange(L)[:, None], s, -np.inf)
        M = s.max(axis=1)
        w = np.exp(s - M[:, None])
        Z = w.sum(axis=1)
        skipped_keys = np.zeros_like(s, bool)
        for i in range(res["map"].shape[2]):
            for j in range(res["map"].shape[3]):
                if res["map"][0, h, i, j] == 1:
                    skipped_keys[i * 128:(i + 1) * 128, j * 128:(j + 1) * 128] = True
        bsk = np.where(skipped_keys, w, 0).sum(axis=1)
        err = np.abs(res["o"][0, h] - o_d[0, h]).max(axis=1)
        assert np.all(err <= 2 * vmax * bsk / Z + 1e-12)
        np.testing.assert_allclose(lse_d[0, h] - res["lse"][0, h], -np.log1p(-bsk / Z), atol=1e-10)
        nsk = (skipped_keys & np.isfinite(s)).sum(axis=1)
        assert np.all(bsk <= lam * nsk + 1e-300)


def test_masked_dense_identity():
    """O with skips = dense attention with every skipped block masked out."""
    q, k, v = rnd(40, 1, 2, 96, 8), rnd(41, 1, 2, 96, 8), rnd(42, 1, 2, 96, 8)
    for causal in (False, True):
        Br, Bc = 4, 8
        res = orc.prefill_tiled(q, k, v, causal, 4.0, 0.3, Br, Bc, precision="f64")
        assert res["skipped"] >= 10
        B, H, L, d = q.shape
        o = np.zeros_like(q)
        lse = np.zeros((B, H, L))
        for h in range(H):
            s = 4.0 * q[0, h] @ k[0, h].T
            if causal:
                s = np.where(np.arange(L)[None, :] <= np.arange(L)[:, None], s, -np.inf)
            for i in range(L // Br):
                for j in range(L // Bc):
                    if res["map"][0, h, i, j] == 1:
                        s[i * Br:(i + 1) * Br, j * Bc:(j + 1) * Bc] = -np.inf
            M = s.max(axis=1, keepdims=True)
            p = np.exp(s - M)
            o[0, h] = p @ v[0, h] / p.sum(axis=1, keepdims=True)
            lse[0, h] = M[:, 0] + np.log(p.sum(axis=1))
        np.testing.assert_allclose(res["o"], o, atol=1e-12)
        np.testing.assert_allclose(res["lse"], lse, atol=1e-12)


def test_forced_map_replaces_the_test():
    q, k, v = rnd(43, 1, 2, 64, 8), rnd(44, 1, 2, 64, 8), rnd(45, 1, 2, 64, 8)
    ref = orc.prefill_tiled(q, k, v, False, 2.0, 0.3, 16, 16, precision="f64")
    forced = orc.prefill_tiled(q, k, v, False, 2.0, 0.0, 16, 16, forced=ref["map"], precision="f64")
    np.testing.assert_array_equal(forced["map"], ref["map"])
    np.testing.assert_allclose(forced["o"], ref["o"], atol=0)
    assert forced["skipped"] == ref["skipped"]


def test_units_subset_matches_full_run():
    a = W.small_random(50, 1, 4, 2, 300, 300, 16, True)
    full = orc.prefill_tiled(a.q, a.k, a.v, True, a.scale, 0.05)
    units = [(0, 3, 2), (0, 0, 0), (0, 1, 1)]
    part = orc.prefill_tiled(a.q, a.k, a.v, True, a.scale, 0.05, units=units)
    for (b, h, t) in units:
        rows = slice(t * 128, min(300, (t + 1) * 128))
        np.testing.assert_array_equal(part["o"][b, h, rows], full["o"][b, h, rows])
        np.testing.assert_array_equal(part["map"][b, h, t], full["map"][b, h, t])


# ------------------------------------------------------------ decode pins ---
def test_decode_lambda0_equals_dense_any_split():
    q, k, v = rnd(60, 3, 8, 1, 16), rnd(61, 3, 2, 1000, 16), rnd(62, 3, 2, 1000, 16)
    o_d, lse_d = np_dense(q, k, v, False, 0.4)
    for S in (1, 2, 3, 8):
        res = orc.decode_tiled(q, k, v, 0.4, 0.0, num_splits=S, precision="f64")
        assert res["skipped"] == 0
        np.testing.assert_allclose(res["o"], o_d[:, :, 0], atol=1e-12)
        np.testing.assert_allclose(res["lse"], lse_d[:, :, 0], atol=1e-12)


def test_decode_skip_set_closed_form_and_split_merge():
    """Decode: the tile unit is the G heads of one KV head x 128 keys; each split
    restarts the running max; the merged output equals the masked dense result."""
    B, Hq, Hkv, L, d = 2, 8, 2, 1500, 16
    G = Hq // Hkv
    q, k, v = rnd(63, B, Hq, 1, d), rnd(64, B, Hkv, L, d), rnd(65, B, Hkv, L, d)
    scale, lam = 3.0, 0.6
    nK = -(-L // 128)
    for S in (1, 2, 5):
        res = orc.decode_tiled(q, k, v, scale, lam, num_splits=S, precision="f64")
        assert res["skipped"] >= 5
        for b in range(B):
            for hk in range(Hkv):
                s = scale * np.stack([k[b, hk] @ q[b, hk * G + g, 0] for g in range(G)])  # [G, L]
                keep = np.ones(L, bool)
                for sp in range(S):
                    t0, t1 = sp * nK // S, (sp + 1) * nK // S
                    run = np.full(G, -np.inf)
                    for t in range(t0, t1):
                        mt = s[:, t * 128:(t + 1) * 128].max(axis=1)
                        run = np.maximum(run, mt)
                        sk = bool(np.all(mt - run < math.log(lam)))
                        assert res["map"][b, hk, t] == (1 if sk else 0)
                        if sk:
                            keep[t * 128:(t + 1) * 128] = False
                sm = np.where(keep[None, :], s, -np.inf)
                M = sm.max(axis=1, keepdims=True)
                p = np.exp(sm - M)
                o = p @ v[b, hk] / p.sum(axis=1, keepdims=True)
                np.testing.assert_allclose(res["o"][b, hk * G:(hk + 1) * G], o, atol=1e-12)
                np.testing.assert_allclose(res["lse"][b, hk * G:(hk + 1) * G],
                                           M[:, 0] + np.log(p.sum(axis=1)), atol=1e-12)


def test_decode_partials_merge_by_lse():
    q, k, v = rnd(66, 1, 4, 1, 8), rnd(67, 1, 1, 700, 8), rnd(68, 1, 1, 700, 8)
    res = orc.decode_tiled(q, k, v, 1.0, 0.0, num_splits=3, precision="f64")
    lp, op = res["lse_part"], res["o_part"]
    lse = np.log(np.exp(lp).sum(axis=0))
    o = (np.exp(lp - lse)[..., None] * op).sum(axis=0)
    np.testing.assert_allclose(res["lse"], lse, atol=1e-12)
    np.testing.assert_allclose(res["o"], o, atol=1e-12)
    one = orc.decode_tiled(q, k, v, 1.0, 0.0, num_splits=1, precision="f64")
    np.testing.assert_allclose(one["o_part"][0], one["o"], atol=0)


# --------------------------------------------------------- MLA decode ---
def np_latent_attention(q, kv, dv, scale, seq_lens=None, keep=None):
    """Textbook attention over a latent cache with library matmuls (float64): for
    head h of sequence b, softmax(scale * kv[:Lb] q_h) kv[:Lb, :dv].  ``keep``
    optionally masks keys ([B, Lmax] bool).  Returns (o [B,Hq,dv], lse [B,Hq])."""
    q = np.asarray(q, np.float64)
    kv = np.asarray(kv, np.float64)
    B, Hq, dk = q.shape
    Lmax = kv.shape[1]
    o = np.zeros((B, Hq, dv))
    lse = np.full((B, Hq), -np.inf)
    for b in range(B):
        Lb = Lmax if seq_lens is None else min(max(int(seq_lens[b]), 0), Lmax)
        if Lb == 0:
            continue
        s = scale * q[b] @ kv[b, :Lb].T  # [Hq, Lb]
        if keep is not None:
            s = np.where(keep[b, :Lb][None, :], s, -np.inf)
        M = s.max(axis=1, keepdims=True)
        p = np.exp(s - M)
        o[b] = p @ kv[b, :Lb, :dv] / p.sum(axis=1, keepdims=True)
        lse[b] = M[:, 0] + np.log(p.sum(axis=1))
    return o, lse


@pytest.mark.parametrize("S", [1, 2, 5])
def test_mla_lambda0_equals_textbook_latent_attention(S):
    """lambda = 0 skips nothing, and the latent form is plain attention whose keys
    are the cached rows and whose values are their leading dv entries."""
    B, Hq, L, dk, dv = 3, 4, 700, 24, 16
    q, kv = rnd(90, B, Hq, dk), rnd(91, B, L, dk)
    lens = [700, 333, 129]
    res = orc.mla_decode_tiled(q, kv, dv, 0.5, 0.0, num_splits=S, seq_lens=lens, precision="f64")
    assert res["skipped"] == 0
    o, lse = np_latent_attention(q, kv, dv, 0.5, lens)
    np.testing.assert_allclose(res["o"], o, atol=1e-12)
    np.testing.assert_allclose(res["lse"], lse, atol=1e-12)


def test_mla_skip_set_closed_form_and_masked_dense():
    """One decision covers every query head x 128 keys; each split restarts the
    running max; the merged result equals latent attention with the skipped key
    tiles masked out."""
    B, Hq, L, dk, dv = 2, 8, 1500, 24, 16
    u = rnd(98, dk)
    u /= np.linalg.norm(u)
    q, kv = rnd(92, B, Hq, dk) + 3.0 * u, rnd(93, B, L, dk)
    kv[:, :4] = 20.0 * u  # sink keys every head attends to
    scale, lam = 0.3, 0.05
    lens = [1500, 900]
    for S in (1, 3):
        res = orc.mla_decode_tiled(q, kv, dv, scale, lam, num_splits=S, seq_lens=lens, precision="f64")
        assert res["skipped"] >= 3
        keep = np.ones((B, L), bool)
        for b in range(B):
            nT = -(-lens[b] // 128)
            s = scale * q[b] @ kv[b, :lens[b]].T
            for sp in range(S):
                t0, t1 = sp * nT // S, (sp + 1) * nT // S
                run = np.full(Hq, -np.inf)
                for t in range(t0, t1):
                    mt = s[:, t * 128:(t + 1) * 128].max(axis=1)
                    run = np.maximum(run, mt)
                    sk = bool(np.all(mt - run < math.log(lam)))
                    assert res["map"][b, t] == (1 if sk else 0)
                    assert res["margin"][b, t] == pytest.approx(np.max(mt - run), abs=1e-12)
                    if sk:
                        keep[b, t * 128:(t + 1) * 128] = False
            assert (res["map"][b, nT:] == 2).all() and np.isnan(res["margin"][b, nT:]).all()
        o, lse = np_latent_attention(q, kv, dv, scale, lens, keep)
        np.testing.assert_allclose(res["o"], o, atol=1e-12)
        np.testing.assert_allclose(res["lse"], lse, atol=1e-12)


def test_mla_equals_gqa_decode_with_one_kv_head_and_the_value_prefix():
    """The latent form is GQA decode with one KV head holding the rows as keys and
    their first dv entries (zero-padded) as values: same map, margins and output."""
    B, Hq, L, dk, dv = 2, 4, 600, 16, 12
    q, kv = rnd(94, B, Hq, dk), rnd(95, B, L, dk)
    v = np.concatenate([kv[..., :dv], np.zeros((B, L, dk - dv))], axis=-1)
    for lam in (0.0, 0.3):
        a = orc.mla_decode_tiled(q, kv, dv, 1.1, lam, num_splits=2, precision="f64")
        g = orc.decode_tiled(q, kv[:, None], v[:, None], 1.1, lam, num_splits=2, precision="f64")
        assert a["skipped"] == g["skipped"]
        np.testing.assert_array_equal(a["map"], g["map"][:, 0])
        np.testing.assert_allclose(a["o"], g["o"][..., :dv], atol=1e-12)
        assert np.all(g["o"][..., dv:] == 0)
        np.testing.assert_allclose(a["lse"], g["lse"], atol=1e-12)


def test_mla_sequence_lengths_truncate_the_cache():
    """A sequence of length Lb gives what a cache of exactly Lb rows gives; a
    sequence of length 0 gives O = 0 and lse = -inf; splits beyond a short
    sequence's tiles are empty and change nothing."""
    B, Hq, L, dk, dv = 3, 2, 520, 16, 8
    q, kv = rnd(96, B, Hq, dk), rnd(97, B, L, dk)
    lens = [520, 200, 0]
    res = orc.mla_decode_tiled(q, kv, dv, 0.7, 0.2, num_splits=4, seq_lens=lens, precision="f64")
    for b in range(2):
        Lb = lens[b]
        nT = -(-Lb // 128)
        one = orc.mla_decode_tiled(q[b:b + 1], kv[b:b + 1, :Lb], dv, 0.7, 0.2, num_splits=min(4, nT),
                                   precision="f64")
        if nT >= 4:
            np.testing.assert_array_equal(res["map"][b, :nT], one["map"][0])
            np.testing.assert_allclose(res["o"][b], one["o"][0], atol=1e-12)
        assert (res["map"][b, nT:] == 2).all()
    assert np.all(res["o"][2] == 0) and np.all(np.isneginf(res["lse"][2]))
    # two tiles over four splits: two splits are empty and the merge ignores them
    short = orc.mla_decode_tiled(q, kv, dv, 0.7, 0.0, num_splits=4, seq_lens=[200, 200, 200], precision="f64")
    ref, lref = np_latent_attention(q, kv, dv, 0.7, [200, 200, 200])
    np.testing.assert_allclose(short["o"], ref, atol=1e-12)
    np.testing.assert_allclose(short["lse"], lref, atol=1e-12)
    assert np.all(np.isneginf(short["lse_part"][0])) and np.all(short["o_part"][0] == 0)


# ---------------------------------------------------- lambda resolution ---
def test_lambda_threshold_is_length_independent():
    for t in (0.0, 1e-4, 0.3, 0.99):
        for L in (1, 128, 32760, 65536, 1 << 20):
            assert lambda_resolution.lambda_threshold(t, L) == pytest.approx(t, rel=1e-15, abs=0)


def test_lambda_curve_worked_example():
    gold = json.load(open(os.path.join(GOLDEN, "wan22_calibration.json")))
    a, b = gold["a"], gold["b"]
    for e in gold["expected"]:
        assert lambda_resolution.factor_from_curve(a, b, e["s"]) == pytest.approx(e["factor"], rel=1e-12)
        assert lambda_resolution.lambda_curve(a, b, e["s"], e["L"]) == pytest.approx(e["lambda"], rel=1e-12)
    # the curve mode scales as 1/L (the inverse length law)
    l1 = lambda_resolution.lambda_curve(a, b, 0.5, 8192)
    l2 = lambda_resolution.lambda_curve(a, b, 0.5, 16384)
    assert l1 == pytest.approx(2 * l2, rel=1e-14)
    with pytest.raises(lambda_resolution.NoCalibration):
        lambda_resolution.lambda_curve(float("nan"), b, 0.5, 100)


# ----------------------------------------------------------- calibration ---
def test_calibration_fit_recovers_known_curve():
    a0, b0 = 123.4, 5.6
    pts = []
    for L in (8192, 32768, 65536):
        for S in (0.1, 0.3, 0.5, 0.8):
            pts.append((a0 * math.exp(b0 * S) / L, L, S))
    a, b = calibration.fit(pts)
    assert a == pytest.approx(a0, rel=1e-10) and b == pytest.approx(b0, rel=1e-10)
    assert calibration.lambda_for(a, b, 0.5, 8192) == pytest.approx(a0 * math.exp(b0 * 0.5) / 8192, rel=1e-10)


def test_calibration_sweep_reads_sparsity_off_margins():
    a = W.tiny(seed=0, planted=True)
    r0 = orc.prefill_tiled(a.q, a.k, a.v, False, a.scale, 0.0, precision="f64")
    pts = calibration.sweep({512: r0["margin"]}, [1e-4, 1e-2, 0.3])
    for lam, L, S in pts:
        r = orc.prefill_tiled(a.q, a.k, a.v, False, a.scale, lam, precision="f64")
        visited = int((r["map"] != 2).sum())
        assert S == pytest.approx(r["skipped"] / visited)


# ------------------------------------------------------- sliding window ---
# A window of W keys keeps, for query row r with r' = r + Lkv - Lq, the keys
# r' - W < c <= r' (the causal mask cut to the last W keys).

@pytest.mark.parametrize("Lq,Lkv", [(37, 37), (20, 29), (29, 20)])
def test_window_of_one_key_returns_that_keys_value(Lq, Lkv):
    """W = 1: every row attends to key r' alone, so O = V[r'] and lse = s(r, r');
    a row with r' < 0 sees nothing (O = 0, lse = -inf)."""
    q, k, v = rnd(1, 1, 2, Lq, 8), rnd(2, 1, 1, Lkv, 8), rnd(3, 1, 1, Lkv, 8)
    o, lse = orc.dense(q, k, v, True, 0.5, precision="f64", window=1)
    t = orc.prefill_tiled(q, k, v, True, 0.5, 0.0, Br=4, Bc=8, precision="f64", window=1)
    for h in range(2):
        for r in range(Lq):
            rr = r + Lkv - Lq
            for oo, ll in ((o, lse), (t["o"], t["lse"])):
                if rr < 0:
                    assert (oo[0, h, r] == 0).all() and ll[0, h, r] == -np.inf
                    continue
                np.testing.assert_allclose(oo[0, h, r], v[0, 0, rr], rtol=0, atol=1e-12)
                assert ll[0, h, r] == pytest.approx(0.5 * float(q[0, h, r] @ k[0, 0, rr]), abs=1e-12)


def test_window_of_two_keys_is_a_logistic_mix():
    """W = 2: O = sigma(s1 - s0) V[r'] + sigma(s0 - s1) V[r'-1] with s1, s0 the
    scores of keys r' and r'-1, and lse = s0 + ln(1 + e^(s1 - s0))."""
    Lq = Lkv = 23
    q, k, v = rnd(4, 1, 1, Lq, 8), rnd(5, 1, 1, Lkv, 8), rnd(6, 1, 1, Lkv, 8)
    t = orc.prefill_tiled(q, k, v, True, 0.7, 0.0, Br=4, Bc=4, precision="f64", window=2)
    for r in range(1, Lq):
        s1 = 0.7 * float(q[0, 0, r] @ k[0, 0, r])
        s0 = 0.7 * float(q[0, 0, r] @ k[0, 0, r - 1])
        w1 = 1.0 / (1.0 + math.exp(s0 - s1))
        np.testing.assert_allclose(t["o"][0, 0, r], w1 * v[0, 0, r] + (1 - w1) * v[0, 0, r - 1], rtol=0, atol=1e-12)
        assert t["lse"][0, 0, r] == pytest.approx(s0 + math.log1p(math.exp(s1 - s0)), abs=1e-12)
    np.testing.assert_allclose(t["o"][0, 0, 0], v[0, 0, 0], rtol=0, atol=1e-12)


@pytest.mark.parametrize("W", [29, 40, 10 ** 6])
def test_window_covering_every_key_is_plain_causal(W):
    q, k, v = rnd(7, 1, 2, 20, 8), rnd(8, 1, 1, 29, 8), rnd(9, 1, 1, 29, 8)
    a = orc.prefill_tiled(q, k, v, True, 0.4, 0.2, Br=4, Bc=8, precision="f64")
    b = orc.prefill_tiled(q, k, v, True, 0.4, 0.2, Br=4, Bc=8, precision="f64", window=W)
    for key in ("o", "lse", "map"):
        assert np.array_equal(a[key], b[key], equal_nan=True), key


@pytest.mark.parametrize("W", [3, 8, 13])
@pytest.mark.parametrize("Lq,Lkv", [(37, 37), (20, 45)])
def test_window_tiled_lambda0_equals_textbook(W, Lq, Lkv):
    q, k, v = rnd(10 + W, 1, 4, Lq, 16), rnd(20 + W, 1, 2, Lkv, 16), rnd(30 + W, 1, 2, Lkv, 16)
    o_ref, lse_ref = np_dense(q, k, v, True, 0.3, window=W)
    t = orc.prefill_tiled(q, k, v, True, 0.3, 0.0, Br=4, Bc=8, precision="f64", window=W)
    o, lse = orc.dense(q, k, v, True, 0.3, precision="f64", window=W)
    np.testing.assert_allclose(t["o"], o_ref, rtol=0, atol=1e-10)
    np.testing.assert_allclose(t["lse"], lse_ref, rtol=0, atol=1e-10)
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-10)
    assert t["skipped"] == 0


@pytest.mark.parametrize("lam", [0.05, 0.3])
def test_window_skip_set_equals_closed_form(lam):
    q, k = rnd(41, 1, 4, 40, 8) * 2, rnd(42, 1, 2, 48, 8) * 2
    v = rnd(43, 1, 2, 48, 8)
    for W in (5, 12, 30):
        t = orc.prefill_tiled(q, k, v, True, 0.6, lam, Br=4, Bc=8, precision="f64", window=W)
        mp, mg = closed_form_skip(q, k, True, 0.6, lam, 4, 8, window=W)
        assert np.array_equal(t["map"], mp), W
        fin = np.isfinite(mg)
        np.testing.assert_allclose(t["margin"][fin], mg[fin], rtol=0, atol=1e-12)
        assert (t["map"] == 1).any() or lam < 0.1


def test_decode_window_splits_cover_the_window():
    """Decode with a window: tiles before the window are not visited, the splits
    share the visited tiles (each non-empty when S <= their count), and at lambda = 0
    the result is attention over the last W keys."""
    B, Hq, Hkv, Lkv, d, W = 2, 4, 2, 1000, 16, 300
    q, k, v = rnd(51, B, Hq, 1, d), rnd(52, B, Hkv, Lkv, d), rnd(53, B, Hkv, Lkv, d)
    lo = (Lkv - W) // 128
    for S in (1, 2, 3):
        r = orc.decode_tiled(q, k, v, 0.4, 0.0, num_splits=S, precision="f64", window=W)
        assert (r["map"][:, :, :lo] == 2).all() and (r["map"][:, :, lo:] == 0).all()
        assert np.isfinite(r["lse_part"]).all(), S
        o_ref, lse_ref = np_dense(q, k[:, :, Lkv - W:], v[:, :, Lkv - W:], False, 0.4)
        np.testing.assert_allclose(r["o"], o_ref[:, :, 0], rtol=0, atol=1e-10)
        np.testing.assert_allclose(r["lse"], lse_ref[:, :, 0], rtol=0, atol=1e-10)
    with pytest.raises(ValueError):
        orc.decode_tiled(q, k, v, 0.4, 0.0, num_splits=4, precision="f64", window=W)  # 3 visited tiles
