"""The oracle's pins must catch plausible mistakes.

Each case plants one mistake in a copy of the oracle's C source (on the CPU, in
a temporary directory), builds it, points the oracle front end at the mutant
and runs the pins; at least one pin must fail for every mutant.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import pytest

from oracle import oracle as orc
from oracle import build as obuild
from tests import test_oracle_pins as pins

MUTANTS = {
    "test-uses-previous-max": ("real diff = mt[i] - mnew[i];", "real diff = mt[i] - m[i];"),
    "margin-sign-flipped": ("real diff = mt[i] - mnew[i];", "real diff = mnew[i] - mt[i];"),
    "no-rescale-of-O": ("for (int x = 0; x < d; ++x) Oi[x] *= alpha;", ""),
    "no-rescale-of-l": ("l[i] = alpha * l[i] + rowsum;", "l[i] = l[i] + rowsum;"),
    "causal-top-left": ("const long rr = r + (Lkv - Lq);", "const long rr = r;"),
    "window-edge-off-by-one": ("return window <= 0 || c > rr - window;", "return window <= 0 || c >= rr - window;"),
    "decode-window-splits-from-zero": ("const int lo = (int)(first_key / Bc);", "const int lo = 0;"),
    "gqa-head-modulo": ("long hk = h / G;\n            for (int i = 0; i < n; ++i) {",
                        "long hk = h % Hkv;\n            for (int i = 0; i < n; ++i) {"),
    "any-row-instead-of-all": ("if (!vote) skip = 0;", "if (vote && i == 0) skip = 1; else if (!vote && i == 0) skip = 0;"),
    "skip-keeps-contribution": ("if (skip) {\n            ++skipped;", "if (0) {\n            ++skipped;"),
    "lse-missing-max": ("m[i] = m[i] + R_LOG(l[i]);", "m[i] = R_LOG(l[i]);"),
    "split-bounds-truncated": ("int t0 = lo + (int)(((long)s * (nK - lo)) / S), t1 = lo + (int)(((long)(s + 1) * (nK - lo)) / S);",
                               "int t0 = lo + s * ((nK - lo) / S), t1 = (s == S - 1) ? nK : lo + (s + 1) * ((nK - lo) / S);"),
    "transposed-score-index": ("sv = score(a->qrow[i], a->kb + c * a->kstride, a->d, a->scale);",
                               "sv = score(a->qrow[i], a->kb + (c0 + (Bc - 1 - cc < a->Lkv - c0 ? Bc - 1 - cc : cc)) * a->kstride, a->d, a->scale);"),
    "mla-value-from-the-row-tail": ("a.vb = a.kb; /* the value is", "a.vb = a.kb + (dk - dv); /* the value is"),
    "mla-score-over-value-width": ("a.d = dk;\n            a.dv = dv;", "a.d = dv;\n            a.dv = dv;"),
    "mla-sequence-length-ignored": ("if (Lb > Lmax) Lb = Lmax;\n            }", "if (Lb > Lmax) Lb = Lmax;\n                Lb = Lmax;\n            }"),
    "mla-splits-over-the-whole-cache": ("int t0 = (int)(((long)s * nT) / S), t1 = (int)(((long)(s + 1) * nT) / S);",
                                        "int t0 = (int)(((long)s * nK) / S), t1 = (int)(((long)(s + 1) * nK) / S);"),
}

PINS = [
    lambda: pins.test_dense_matches_textbook_matmul(True, (2, 4, 2, 20, 29, 16)),
    lambda: pins.test_tiled_matches_brute_force_tiny((2, 4), True),
    lambda: pins.test_tiled_lambda0_equals_dense_small(2, 4),
    lambda: pins.test_skip_set_equals_closed_form(True),
    lambda: pins.test_skip_set_closed_form_small_tiles_gqa(),
    lambda: pins.test_masked_dense_identity(),
    lambda: pins.test_decode_skip_set_closed_form_and_split_merge(),
    lambda: pins.test_skipped_contribution_closed_form(0.1),
    lambda: pins.test_window_of_one_key_returns_that_keys_value(20, 29),
    lambda: pins.test_decode_window_splits_cover_the_window(),
    lambda: pins.test_mla_lambda0_equals_textbook_latent_attention(2),
    lambda: pins.test_mla_skip_set_closed_form_and_masked_dense(),
    lambda: pins.test_mla_sequence_lengths_truncate_the_cache(),
]


def _build_mutant(tmp, name, old, new):
    src = open(obuild.SRC).read()
    assert old in src, f"mutation anchor for {name} not found"
    path_c = os.path.join(tmp, f"{name}.c")
    open(path_c, "w").write(src.replace(old, new, 1))
    objs = []
    for real, suf in (("float", "_f32"), ("double", "_f64")):
        o = os.path.join(tmp, f"{name}{suf}.o")
        subprocess.run(["gcc", "-O1", "-fPIC", "-fopenmp", "-std=c11", "-ffp-contract=off",
                        f"-DREAL={real}", f"-DSUFFIX={suf}", "-c", path_c, "-o", o], check=True)
        objs.append(o)
    so = os.path.join(tmp, f"lib{name}.so")
    subprocess.run(["gcc", "-shared", "-fopenmp", "-o", so, *objs, "-lm"], check=True)
    return so


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    old, new = MUTANTS[name]
    so = _build_mutant(str(tmp_path), name, old, new)
    saved = orc._lib
    orc._lib = orc._configure(ctypes.CDLL(so))
    caught = []
    try:
        for pin in PINS:
            try:
                pin()
            except (AssertionError, ValueError, IndexError):
                caught.append(pin)
    finally:
        orc._lib = saved
    assert caught, f"no pin caught the planted mistake '{name}'"
