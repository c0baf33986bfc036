"""Host-side logic of bench.py that feeds its JSON line: the DRAM traffic figure of a
kernel is reported only while the kernel's sources are the ones it was captured on,
and the causal FLOP / tile counts match brute force."""
from __future__ import annotations

import bench


def test_traffic_is_reported_only_for_the_captured_sources(monkeypatch):
    for kernel in ("prefill", "decode"):
        t = bench.TRAFFIC[kernel]
        got, note = bench.traffic_for(kernel)
        if t["bytes"] is None:
            assert got is None
            continue
        if t["sources_sha256"] != bench.sources_sha256(kernel):
            # recorded for another version of the sources: the line must not report it
            assert got is None and "changed" in note
            continue
        assert got == t["bytes"] and note == t["capture"]
        # any edit of a source file makes the figure belong to another kernel
        monkeypatch.setitem(bench.TRAFFIC, kernel, dict(t, sources_sha256="0" * 64))
        got2, note2 = bench.traffic_for(kernel)
        assert got2 is None and "changed" in note2


def test_causal_counts_match_brute_force():
    for Lq, Lkv in ((1, 1), (300, 300), (257, 1000), (500, 200), (1024, 1024)):
        off = Lkv - Lq
        pairs = sum(max(0, min(Lkv, r + off + 1)) for r in range(Lq))
        assert bench.causal_pairs(Lq, Lkv) == pairs
        T = 128
        nK = -(-Lkv // T)
        tiles = 0
        for qt in range(-(-Lq // T)):
            rows = range(qt * T, min(Lq, (qt + 1) * T))
            vis = {c // T for r in rows for c in range(0, max(0, min(Lkv, r + off + 1)))}
            tiles += len(vis)
        assert bench.visited_tiles_causal(Lq, Lkv) == tiles
        assert tiles <= -(-Lq // T) * nK
