"""Host-side logic of bench.py that feeds its JSON line: the DRAM traffic figure of a
kernel is reported only while the kernel's code (comments aside) is the code it was
captured on, and the causal FLOP / tile counts match brute force."""
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


def test_source_hash_ignores_comments_but_not_code():
    src = (
        "// header comment\n"
        "__global__ void k(int* p) {  // trailing comment\n"
        "    p[0] = 1;\n"
        "\n"
        "    asm volatile(\"mov.u32 %0, 1;\" : \"=r\"(p[1]));\n"
        "}\n"
    )
    recommented = (
        "// another header\n"
        "// and a second line\n"
        "__global__ void k(int* p) {\n"
        "    p[0] = 1;    // the store\n"
        "\n"
        "    asm volatile(\"mov.u32 %0, 1;\" : \"=r\"(p[1]));\n"
        "}\n"
    )
    changed = src.replace("p[0] = 1;", "p[0] = 2;")
    assert bench._code_only(src) == bench._code_only(recommented)
    assert bench._code_only(src) != bench._code_only(changed)
    # the line-based stripping relies on the kernels' sources holding no block comments
    # and no "//" inside a string literal
    import os
    import re

    for kernel in ("prefill", "decode"):
        for rel in bench.KERNEL_SOURCES[kernel]:
            path = os.path.join(bench.ROOT, "skip_softmax_flashattention_gb300", rel)
            with open(path, encoding="utf-8") as f:
                text = f.read()
            assert "/*" not in text
            assert not re.search(r'"[^"\n]*//[^"\n]*"', text)


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
