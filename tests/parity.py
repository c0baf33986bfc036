"""GPU-vs-oracle comparison rules shared by the GPU tests and the smoke check.

Acceptance (per tile and per element):
  * every visited tile's skip decision equals the oracle's, except tiles whose
    oracle margin lies within 1e-3 of ln(lambda) -- those are logged, not failed;
  * the skipped-tile count the kernel reports equals the number of skipped tiles
    in its map, and (where the oracle covers the whole problem) the oracle's count
    up to the logged band tiles;
  * O (bf16) is within max-abs 2e-2 and mean-abs 2e-3 of the fp32 oracle run with
    the GPU's skip map forced; lse is within 1e-3 (both -inf for rows with no key).
"""
from __future__ import annotations

import math

import numpy as np
import torch

from oracle import oracle as orc

BAND = 1e-3
O_MAX_ABS = 2e-2
O_MEAN_ABS = 2e-3
LSE_ABS = 1e-3
TILE = 128


def _lnlam(lam):
    return -math.inf if lam <= 0 else math.log(lam)


def _check_rows(o_gpu, lse_gpu, o_ref, lse_ref, what):
    o_gpu = np.asarray(o_gpu, np.float64)
    o_ref = np.asarray(o_ref, np.float64)
    err = np.abs(o_gpu - o_ref)
    assert np.isfinite(o_gpu).all(), f"{what}: non-finite O"
    mx, mean = float(err.max()), float(err.mean())
    assert mx <= O_MAX_ABS, f"{what}: O max-abs {mx:.3e} > {O_MAX_ABS}"
    assert mean <= O_MEAN_ABS, f"{what}: O mean-abs {mean:.3e} > {O_MEAN_ABS}"
    lse_gpu = np.asarray(lse_gpu, np.float64)
    lse_ref = np.asarray(lse_ref, np.float64)
    inf_g, inf_r = np.isneginf(lse_gpu), np.isneginf(lse_ref)
    assert np.array_equal(inf_g, inf_r), f"{what}: -inf lse rows differ"
    fin = ~inf_r
    if fin.any():
        le = float(np.abs(lse_gpu[fin] - lse_ref[fin]).max())
        assert le <= LSE_ABS, f"{what}: lse abs err {le:.3e} > {LSE_ABS}"
    return mx, mean


def _decisions(gpu_map, ora_map, ora_margin, lam, what):
    gpu_map = np.asarray(gpu_map)
    ora_map = np.asarray(ora_map)
    assert np.array_equal(gpu_map == 2, ora_map == 2), f"{what}: visited tiles differ"
    vis = ora_map != 2
    diff = vis & (gpu_map != ora_map)
    band = np.abs(np.asarray(ora_margin, np.float64) - _lnlam(lam)) < BAND
    bad = diff & ~band
    assert not bad.any(), (f"{what}: {int(bad.sum())} tile decisions differ outside the 1e-3 band "
                           f"(first at {np.argwhere(bad)[0].tolist()})")
    return int(diff.sum())


def prefill_units_check(a, res, lam, units, log=None, window=0):
    """Compare the GPU prefill result on the given (b, h, qtile) units.

    a: workloads.Attn on the GPU; res: dict from blasst.prefill(..., want_map=True).
    Returns (#band tiles, max abs O err, mean abs O err)."""
    G = a.Hq // a.Hkv
    gmap = res["map"].cpu().numpy()
    o_gpu = res["o"]
    lse_gpu = res["lse"]
    by_head = {}
    for (b, h, t) in units:
        by_head.setdefault((b, h), []).append(t)
    band_total, errs = 0, []
    for (b, h), tiles in sorted(by_head.items()):
        hk = h // G
        q = a.q[b:b + 1, h:h + 1].float().cpu()
        k = a.k[b:b + 1, hk:hk + 1].float().cpu()
        v = a.v[b:b + 1, hk:hk + 1].float().cpu()
        uu = [(0, 0, t) for t in tiles]
        own = orc.prefill_tiled(q, k, v, a.causal, a.scale, lam, units=uu, precision="f32", window=window)
        forced_map = np.full(own["map"].shape, 0, np.uint8)
        forced_map[0, 0] = gmap[b, h]
        ref = orc.prefill_tiled(q, k, v, a.causal, a.scale, lam, units=uu, forced=forced_map, precision="f32",
                                window=window)
        for t in tiles:
            what = f"{a.name} lam={lam:g} b={b} h={h} qtile={t}"
            band_total += _decisions(gmap[b, h, t], own["map"][0, 0, t], own["margin"][0, 0, t], lam, what)
            rows = slice(t * TILE, min(a.Lq, (t + 1) * TILE))
            og = o_gpu[b, h, rows].float().cpu().numpy()
            lg = lse_gpu[b, h, rows].cpu().numpy()
            errs.append(_check_rows(og, lg, ref["o"][0, 0, rows], ref["lse"][0, 0, rows], what))
    if log is not None and band_total:
        log.append(f"{a.name} lam={lam:g}: {band_total} tiles inside the 1e-3 margin band")
    return band_total, max(e[0] for e in errs), float(np.mean([e[1] for e in errs]))


def prefill_full_check(a, res, lam, log=None, window=0):
    """Whole-problem comparison (small problems): decisions, exact count, O, lse."""
    own = orc.prefill_tiled(a.q.float().cpu(), a.k.float().cpu(), a.v.float().cpu(), a.causal, a.scale, lam,
                            precision="f32", window=window)
    gmap = res["map"].cpu().numpy()
    band = _decisions(gmap, own["map"], own["margin"], lam, f"{a.name} lam={lam:g}")
    n_gpu = int(res["skipped"].item())
    assert n_gpu == int((gmap == 1).sum()), "reported count differs from the map"
    assert abs(n_gpu - own["skipped"]) <= band, f"count {n_gpu} vs oracle {own['skipped']} (band {band})"
    if band == 0:
        assert n_gpu == own["skipped"]
    ref = orc.prefill_tiled(a.q.float().cpu(), a.k.float().cpu(), a.v.float().cpu(), a.causal, a.scale, lam,
                            forced=gmap, precision="f32", window=window)
    mx, mean = _check_rows(res["o"].float().cpu().numpy(), res["lse"].cpu().numpy(), ref["o"], ref["lse"],
                           f"{a.name} lam={lam:g}")
    if log is not None and band:
        log.append(f"{a.name} lam={lam:g}: {band} tiles inside the 1e-3 margin band")
    return band, mx, mean, n_gpu


def decode_units_check(a, res, lam, S, units, log=None):
    """Compare a GPU decode result on (b, hkv) units (q is [B,Hq,1,d])."""
    G = a.Hq // a.Hkv
    gmap = res["map"].cpu().numpy()
    band_total, errs = 0, []
    for (b, hk) in units:
        q = a.q[b:b + 1, hk * G:(hk + 1) * G].float().cpu()
        k = a.k[b:b + 1, hk:hk + 1].float().cpu()
        v = a.v[b:b + 1, hk:hk + 1].float().cpu()
        own = orc.decode_tiled(q, k, v, a.scale, lam, num_splits=S, precision="f32")
        ref = orc.decode_tiled(q, k, v, a.scale, lam, num_splits=S, forced=gmap[b:b + 1, hk:hk + 1],
                               precision="f32")
        what = f"{a.name} lam={lam:g} S={S} b={b} hkv={hk}"
        band_total += _decisions(gmap[b, hk], own["map"][0, 0], own["margin"][0, 0], lam, what)
        og = res["o"][b, hk * G:(hk + 1) * G].float().cpu().numpy()
        lg = res["lse"][b, hk * G:(hk + 1) * G].cpu().numpy()
        errs.append(_check_rows(og, lg, ref["o"][0], ref["lse"][0], what))
    if log is not None and band_total:
        log.append(f"{a.name} lam={lam:g} S={S}: {band_total} tiles inside the 1e-3 margin band")
    return band_total, max(e[0] for e in errs), float(np.mean([e[1] for e in errs]))


def decode_full_check(a, res, lam, S, log=None):
    own = orc.decode_tiled(a.q.float().cpu(), a.k.float().cpu(), a.v.float().cpu(), a.scale, lam, num_splits=S,
                           precision="f32")
    gmap = res["map"].cpu().numpy()
    band = _decisions(gmap, own["map"], own["margin"], lam, f"{a.name} lam={lam:g} S={S}")
    n_gpu = int(res["skipped"].item())
    assert n_gpu == int((gmap == 1).sum())
    assert abs(n_gpu - own["skipped"]) <= band
    if band == 0:
        assert n_gpu == own["skipped"]
    ref = orc.decode_tiled(a.q.float().cpu(), a.k.float().cpu(), a.v.float().cpu(), a.scale, lam, num_splits=S,
                           forced=gmap, precision="f32")
    mx, mean = _check_rows(res["o"].float().cpu().numpy(), res["lse"].cpu().numpy(), ref["o"], ref["lse"],
                           f"{a.name} lam={lam:g} S={S}")
    if log is not None and band:
        log.append(f"{a.name} lam={lam:g} S={S}: {band} tiles inside the 1e-3 margin band")
    return band, mx, mean, n_gpu


def decode_paged_check(a, res, lam, S, seqs=None, log=None, window=0):
    """A paged decode (workloads.paged_decode) against the oracle run on each
    sequence alone: its own key count, the call's lambda and split count.  Tiles
    past a sequence's end must stay "not visited"."""
    lens = a.extra["seq_lens"].cpu().tolist()
    gmap = res["map"].cpu().numpy()
    o_gpu = res["o"].float().cpu().numpy()
    lse_gpu = res["lse"].cpu().numpy()
    B = len(lens)
    assert int(res["skipped"].item()) == int((gmap == 1).sum())
    band_total, oracle_skipped = 0, 0
    for b in (range(B) if seqs is None else seqs):
        L = lens[b]
        nt = -(-L // 128)
        lo = (L - window) // 128 if 0 < window < L else 0  # first tile holding a key in the window
        what = f"{a.name} seq {b} (L={L}) lam={lam:g} S={S} window={window}"
        assert (gmap[b, :, nt:] == 2).all(), f"{what}: tiles past the end visited"
        assert (gmap[b, :, :lo] == 2).all(), f"{what}: tiles before the window visited"
        if L == 0:
            assert (o_gpu[b] == 0).all() and np.isneginf(lse_gpu[b]).all(), what
            continue
        q = a.q[b:b + 1].float().cpu()
        k = a.k[b:b + 1, :, :L].float().cpu()
        v = a.v[b:b + 1, :, :L].float().cpu()
        # With more splits than tiles, split s = [floor(s*nt/S), floor((s+1)*nt/S)) puts
        # every tile in a split of its own and leaves the rest empty (no contribution):
        # the same partition as nt splits.
        Sb = min(S, nt - lo)
        own = orc.decode_tiled(q, k, v, a.scale, lam, num_splits=Sb, precision="f32", window=window)
        band = _decisions(gmap[b:b + 1, :, :nt], own["map"], own["margin"], lam, what)
        band_total += band
        oracle_skipped += int(own["skipped"])
        ref = orc.decode_tiled(q, k, v, a.scale, lam, num_splits=Sb, forced=gmap[b:b + 1, :, :nt], precision="f32",
                               window=window)
        _check_rows(o_gpu[b:b + 1], lse_gpu[b:b + 1], ref["o"], ref["lse"], what)
        if log is not None and band:
            log.append(f"{what}: {band} tiles inside the 1e-3 margin band")
    return band_total, oracle_skipped


def mla_check(a, res, lam, S, seqs=None, log=None, counts=False):
    """An MLA decode (workloads.mla_decode) against the oracle run on each checked
    sequence with its own key count, the call's lambda and split count: every tile
    decision (outside the 1e-3 margin band), then O and lse with the GPU's decisions
    forced.  Tiles past a sequence's end must stay "not visited".  Returns the number
    of decisions that differ inside the band (and, with counts, the oracle's skipped
    count over the checked sequences)."""
    kv = a.extra["kv"]
    dv = a.extra["dv"]
    Lmax = kv.shape[1]
    sl = a.extra.get("seq_lens")
    lens = [Lmax] * a.B if sl is None else sl.cpu().tolist()
    gmap = res["map"].cpu().numpy()
    o_gpu = res["o"].float().cpu().numpy()
    lse_gpu = res["lse"].cpu().numpy()
    assert int(res["skipped"].item()) == int((gmap == 1).sum())
    band_total, oracle_skipped = 0, 0
    for b in (range(a.B) if seqs is None else seqs):
        L = min(max(lens[b], 0), Lmax)
        nt = -(-L // 128)
        what = f"{a.name} seq {b} (L={L}) lam={lam:g} S={S}"
        assert (gmap[b, nt:] == 2).all(), f"{what}: tiles past the end visited"
        if L == 0:
            assert (o_gpu[b] == 0).all() and np.isneginf(lse_gpu[b]).all(), what
            continue
        q = a.q[b:b + 1].float().cpu()
        kvb = kv[b:b + 1].float().cpu()
        own = orc.mla_decode_tiled(q, kvb, dv, a.scale, lam, num_splits=S, seq_lens=[L], precision="f32")
        band = _decisions(gmap[b:b + 1], own["map"], own["margin"], lam, what)
        ref = orc.mla_decode_tiled(q, kvb, dv, a.scale, lam, num_splits=S, seq_lens=[L], forced=gmap[b:b + 1],
                                   precision="f32")
        _check_rows(o_gpu[b:b + 1], lse_gpu[b:b + 1], ref["o"], ref["lse"], what)
        band_total += band
        oracle_skipped += int(own["skipped"])
        if log is not None and band:
            log.append(f"{what}: {band} tiles inside the 1e-3 margin band")
    return (band_total, oracle_skipped) if counts else band_total


def oracle_map_at(margin, lam):
    """The oracle's own decisions at threshold lam, read off the margins of its fp32
    pass: a visited tile is skipped iff its margin (max over the voting rows of
    m~ - m) is below ln(lam) rounded to fp32 -- the very comparison of the oracle's
    test, row by row, since max_r x_r < t iff x_r < t for every r.  The margins do
    not depend on lam <= 1 (a skip never moves the running max), so one lam = 0
    pass decides every threshold.  Not visited: 2."""
    g = np.asarray(margin, np.float32)
    lnl = np.float32(-np.inf) if lam <= 0 else np.float32(math.log(lam))
    out = np.full(g.shape, 2, np.uint8)
    vis = ~np.isnan(g)
    out[vis] = (g[vis] < lnl).astype(np.uint8)
    return out


def margins_check(g_gpu, g_ref, what, tol=BAND):
    """GPU margins against the oracle's: the same not-visited (NaN) and +inf tiles,
    finite values within tol."""
    g_gpu = np.asarray(g_gpu, np.float64)
    g_ref = np.asarray(g_ref, np.float64)
    assert np.array_equal(np.isnan(g_gpu), np.isnan(g_ref)), f"{what}: visited tiles differ"
    assert np.array_equal(np.isposinf(g_gpu), np.isposinf(g_ref)), f"{what}: +inf margins differ"
    fin = np.isfinite(g_ref)
    assert np.array_equal(fin, np.isfinite(g_gpu)), f"{what}: finite margins differ"
    if fin.any():
        err = float(np.abs(g_gpu[fin] - g_ref[fin]).max())
        assert err < tol, f"{what}: margin abs err {err:.3e} >= {tol}"


def whole_check(what, lam, res, own0, forced_run, log=None):
    """Whole-problem acceptance for one threshold from one lam = 0 oracle pass.

    res: the GPU result (map, skipped, o, lse); own0: the oracle's lam = 0 pass over
    the same problem (margins, and O/lse with every tile computed); forced_run(map):
    the oracle with the GPU's map forced, run only when the GPU skipped a tile.
    Checks every decision outside the 1e-3 band, the exact skipped count, O and lse.
    Returns (#band tiles, GPU count)."""
    gmap = res["map"].cpu().numpy()
    omap = oracle_map_at(own0["margin"], lam)
    band = _decisions(gmap, omap, own0["margin"], lam, what)
    n_gpu = int(res["skipped"].item())
    assert n_gpu == int((gmap == 1).sum()), f"{what}: reported count differs from the map"
    n_ora = int((omap == 1).sum())
    assert abs(n_gpu - n_ora) <= band, f"{what}: count {n_gpu} vs oracle {n_ora} (band {band})"
    if band == 0:
        assert n_gpu == n_ora, f"{what}: count {n_gpu} vs oracle {n_ora}"
    ref = forced_run(gmap) if (gmap == 1).any() else own0
    _check_rows(res["o"].float().cpu().numpy(), res["lse"].cpu().numpy(), ref["o"], ref["lse"], what)
    if log is not None and band:
        log.append(f"{what}: {band} tiles inside the 1e-3 margin band")
    return band, n_gpu


def sample_units(rng, B, H, nQ, k, always=()):
    """k random (b, h, qtile) units plus the listed ones (first/last tiles)."""
    units = set(always)
    while len(units) < k + len(always):
        units.add((int(rng.integers(B)), int(rng.integers(H)), int(rng.integers(nQ))))
    return sorted(units)


def to_gpu(a, device="cuda"):
    a.q, a.k, a.v = a.q.to(device), a.k.to(device), a.v.to(device)
    return a
