"""CPU-side checks of the C ABI: the library loads, exports every declared entry
point, and its host logic (threshold resolution, validation, split plan,
workspace sizing, status strings) behaves as documented.  No call here reaches a
GPU: every compute call below is rejected by validation before any CUDA work."""
from __future__ import annotations

import ctypes
import json
import math
import os
import re

import pytest

from skip_softmax_flashattention_gb300 import blasst as K

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "blasst.h")


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(blasst_[a-z_0-9]+)\s*\(", src)))


def test_library_exports_every_declared_symbol():
    lib = K.load()
    names = declared_functions()
    assert len(names) >= 8
    for n in names:
        assert hasattr(lib, n), n
    raw = ctypes.CDLL(K.library_path())
    for n in names:
        getattr(raw, n)


def test_status_strings():
    for code in (0, 1, -1, -2, -3, -4, -5, -6):
        s = K.blasst_status_string(code)
        assert s and s != "unknown status"
    assert K.blasst_status_string(1234) == "unknown status"
    assert "threshold" in K.blasst_status_string(K.BLASST_ERR_NO_CALIBRATION)


def test_lambda_threshold_mode():
    for t in (0.0, 1e-4, 0.5, 1.0):
        for L in (1, 4096, 32760, 1 << 20):
            rc, lam = K.blasst_lambda(0, threshold=t, Lkv=L)
            assert rc == K.BLASST_OK and lam == t
    rc, lam = K.blasst_lambda(0, threshold=1.5, Lkv=10)
    assert rc == K.BLASST_WARN_LAMBDA_GE_1 and lam == 1.5
    for bad in (-1e-3, math.nan, math.inf):
        assert K.blasst_lambda(0, threshold=bad, Lkv=10)[0] == K.BLASST_ERR_INVALID_ARG
    assert K.blasst_lambda(0, threshold=0.1, Lkv=0)[0] == K.BLASST_ERR_INVALID_ARG
    assert K.blasst_lambda(7, threshold=0.1, Lkv=5)[0] == K.BLASST_ERR_INVALID_ARG


def test_lambda_curve_mode_worked_example():
    gold = json.load(open(os.path.join(ROOT, "tests", "golden", "wan22_calibration.json")))
    for e in gold["expected"]:
        rc, lam = K.blasst_lambda(1, a=gold["a"], b=gold["b"], target_sparsity=e["s"], Lkv=e["L"])
        assert lam == pytest.approx(e["lambda"], rel=1e-12)
        assert rc == (K.BLASST_WARN_LAMBDA_GE_1 if e["lambda"] > 1 else K.BLASST_OK)
    assert K.blasst_lambda(1, a=math.nan, b=1.0, target_sparsity=0.5, Lkv=8)[0] == K.BLASST_ERR_NO_CALIBRATION
    assert K.blasst_lambda(1, a=1.0, b=math.inf, target_sparsity=0.5, Lkv=8)[0] == K.BLASST_ERR_NO_CALIBRATION
    assert K.blasst_lambda(1, a=1.0, b=1.0, target_sparsity=1.5, Lkv=8)[0] == K.BLASST_ERR_INVALID_ARG


def test_split_plan_and_workspace_host_logic():
    assert K.blasst_decode_num_splits(64, 32, 8, 32768, 128, 3) == (0, 3)
    assert K.blasst_decode_num_splits(1, 4, 1, 1000, 128, 8) == (0, 8)
    assert K.blasst_decode_num_splits(1, 4, 1, 1000, 128, 9)[0] == K.BLASST_ERR_INVALID_ARG
    assert K.blasst_decode_num_splits(1, 5, 2, 1000, 128, 1)[0] == K.BLASST_ERR_INVALID_ARG
    assert K.blasst_decode_workspace_size(64, 32, 8, 32768, 128, 1) == 0
    ws = K.blasst_decode_workspace_size(2, 8, 2, 1000, 128, 3)
    assert ws >= 3 * 2 * 8 * 128 * 4 + 3 * 2 * 8 * 4


FAKE = 1 << 20  # never dereferenced: every call below fails validation first


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), K.BLASST_ERR_INVALID_ARG),
    (dict(Hq=6, Hkv=4), K.BLASST_ERR_INVALID_ARG),
    (dict(Lq=0), K.BLASST_ERR_INVALID_ARG),
    (dict(lam=1.01), K.BLASST_ERR_INVALID_ARG),
    (dict(lam=-0.1), K.BLASST_ERR_INVALID_ARG),
    (dict(lam=math.nan), K.BLASST_ERR_INVALID_ARG),
    (dict(scale=0.0), K.BLASST_ERR_INVALID_ARG),
    (dict(scale=math.inf), K.BLASST_ERR_INVALID_ARG),
    (dict(causal=2), K.BLASST_ERR_INVALID_ARG),
    (dict(flags=0x100), K.BLASST_ERR_INVALID_ARG),
    (dict(d=96), K.BLASST_ERR_UNSUPPORTED),
    (dict(flags=K.BLASST_PREFILL_ELIDE_V | K.BLASST_PREFILL_WIDE), K.BLASST_ERR_UNSUPPORTED),
    (dict(flags=K.BLASST_PREFILL_ELIDE_V | K.BLASST_PREFILL_ONE_QTILE), K.BLASST_ERR_UNSUPPORTED),
    (dict(flags=K.BLASST_PREFILL_ELIDE_V | K.BLASST_PREFILL_P_VIA_SMEM), K.BLASST_ERR_UNSUPPORTED),
    (dict(q=FAKE + 8), K.BLASST_ERR_UNSUPPORTED),
])
def test_prefill_validation(kw, code):
    a = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=None, B=1, Hq=4, Hkv=2, Lq=100, Lkv=100, d=128, causal=1,
             scale=0.1, lam=0.01, flags=0)
    a.update(kw)
    rc = K.blasst_prefill_ex(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["Hq"], a["Hkv"], a["Lq"],
                             a["Lkv"], a["d"], a["causal"], a["scale"], a["lam"], None, None, None, a["flags"],
                             stream=0)
    assert rc == code


@pytest.mark.parametrize("kw,code", [
    (dict(o=None), K.BLASST_ERR_INVALID_ARG),
    (dict(S=0), K.BLASST_ERR_INVALID_ARG),
    (dict(S=9), K.BLASST_ERR_INVALID_ARG),
    (dict(lam=2.0), K.BLASST_ERR_INVALID_ARG),
    (dict(d=96), K.BLASST_ERR_UNSUPPORTED),
    (dict(Hq=24, Hkv=8), K.BLASST_ERR_UNSUPPORTED),
    (dict(Hq=96, Hkv=2), K.BLASST_ERR_UNSUPPORTED),   # G = 48
    (dict(Hq=512, Hkv=2), K.BLASST_ERR_UNSUPPORTED),  # G = 256
    (dict(S=2, ws=None, wsb=0), K.BLASST_ERR_INVALID_ARG),
    (dict(S=2, wsb=16), K.BLASST_ERR_WORKSPACE_TOO_SMALL),
])
def test_decode_validation(kw, code):
    a = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, B=2, Hq=8, Hkv=2, Lkv=1000, d=128, scale=0.1, lam=0.01, S=1,
             ws=FAKE, wsb=1 << 30)
    a.update(kw)
    rc = K.blasst_decode(a["q"], a["k"], a["v"], a["o"], None, a["B"], a["Hq"], a["Hkv"], a["Lkv"], a["d"],
                         a["scale"], a["lam"], a["S"], a["ws"], a["wsb"], None, None, None, stream=0)
    assert rc == code


@pytest.mark.parametrize("kw,code", [
    (dict(table=None), K.BLASST_ERR_INVALID_ARG),
    (dict(mp=1), K.BLASST_ERR_INVALID_ARG),          # 1 page of 16 keys cannot hold 1000 keys
    (dict(tm=2), K.BLASST_ERR_INVALID_ARG),
    (dict(npg=0), K.BLASST_ERR_INVALID_ARG),
    (dict(S=9), K.BLASST_ERR_INVALID_ARG),
    (dict(ps=24, mp=42), K.BLASST_ERR_UNSUPPORTED),  # neither a divisor nor a multiple of 128
    (dict(ps=200, mp=5), K.BLASST_ERR_UNSUPPORTED),
    (dict(d=96), K.BLASST_ERR_UNSUPPORTED),
    (dict(Hq=64, Hkv=2), K.BLASST_ERR_UNSUPPORTED),  # G = 32: the paged form holds up to 16
    (dict(table=FAKE + 2), K.BLASST_ERR_UNSUPPORTED),
    (dict(S=2, wsb=16), K.BLASST_ERR_WORKSPACE_TOO_SMALL),
    (dict(win=-1), K.BLASST_ERR_INVALID_ARG),
])
def test_decode_paged_validation(kw, code):
    a = dict(q=FAKE, kp=FAKE, vp=FAKE, table=FAKE, lens=None, o=FAKE, B=2, Hq=8, Hkv=2, L=1000, d=128, npg=200,
             ps=16, mp=63, tm=1, scale=0.1, lam=0.01, S=1, ws=FAKE, wsb=1 << 30, win=0)
    a.update(kw)
    rc = K.blasst_decode_paged(a["q"], a["kp"], a["vp"], a["table"], a["lens"], a["o"], None, a["B"], a["Hq"],
                               a["Hkv"], a["L"], a["win"], a["d"], a["npg"], a["ps"], a["mp"], a["tm"], a["scale"],
                               a["lam"], a["S"], a["ws"], a["wsb"], None, None, None, stream=0)
    assert rc == code


@pytest.mark.parametrize("kw,code", [
    (dict(window=0), K.BLASST_ERR_INVALID_ARG),
    (dict(window=-5), K.BLASST_ERR_INVALID_ARG),
    (dict(flags=K.BLASST_PREFILL_WIDE), K.BLASST_ERR_UNSUPPORTED),
    (dict(flags=K.BLASST_PREFILL_ONE_QTILE), K.BLASST_ERR_UNSUPPORTED),
    (dict(q=None), K.BLASST_ERR_INVALID_ARG),
    (dict(lam=2.0), K.BLASST_ERR_INVALID_ARG),
])
def test_prefill_window_validation(kw, code):
    a = dict(q=FAKE, window=64, flags=0, lam=0.01)
    a.update(kw)
    rc = K.blasst_prefill_window(a["q"], FAKE, FAKE, FAKE, None, 1, 4, 2, 100, 100, 128, a["window"], 0.1, a["lam"],
                                 None, None, None, a["flags"], stream=0)
    assert rc == code


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), K.BLASST_ERR_INVALID_ARG),
    (dict(kv=None), K.BLASST_ERR_INVALID_ARG),
    (dict(Hq=256), K.BLASST_ERR_UNSUPPORTED),
    (dict(Hq=48), K.BLASST_ERR_UNSUPPORTED),
    (dict(Hq=3), K.BLASST_ERR_UNSUPPORTED),
    (dict(dk=512), K.BLASST_ERR_UNSUPPORTED),
    (dict(dv=256), K.BLASST_ERR_UNSUPPORTED),
    (dict(S=0), K.BLASST_ERR_INVALID_ARG),
    (dict(S=9), K.BLASST_ERR_INVALID_ARG),             # 1000 keys are 8 tiles
    (dict(lam=2.0), K.BLASST_ERR_INVALID_ARG),
    (dict(scale=0.0), K.BLASST_ERR_INVALID_ARG),
    (dict(table=FAKE, mp=1), K.BLASST_ERR_INVALID_ARG),   # one 64-row page cannot hold 1000 rows
    (dict(table=FAKE, npg=0), K.BLASST_ERR_INVALID_ARG),
    (dict(table=FAKE, ps=24, mp=42), K.BLASST_ERR_UNSUPPORTED),
    # the pool's rows plus the row an out-of-range page reads must fit a 32-bit row index
    (dict(table=FAKE, ps=128, npg=(2 ** 31 - 128) // 128 - 1, mp=8), K.BLASST_ERR_UNSUPPORTED),
    (dict(table=FAKE + 2), K.BLASST_ERR_UNSUPPORTED),
    (dict(kv=FAKE + 2), K.BLASST_ERR_UNSUPPORTED),
    (dict(S=2, ws=None), K.BLASST_ERR_INVALID_ARG),
    (dict(S=2, wsb=16), K.BLASST_ERR_WORKSPACE_TOO_SMALL),
])
def test_mla_decode_validation(kw, code):
    a = dict(q=FAKE, kv=FAKE, table=None, lens=None, B=2, Hq=16, L=1000, dk=576, dv=512, npg=40, ps=64, mp=16,
             scale=0.1, lam=0.01, S=1, ws=FAKE, wsb=1 << 30)
    a.update(kw)
    rc = K.blasst_mla_decode(a["q"], a["kv"], a["table"], a["lens"], FAKE, None, a["B"], a["Hq"], a["L"], a["dk"],
                             a["dv"], a["npg"], a["ps"], a["mp"], a["scale"], a["lam"], a["S"], a["ws"], a["wsb"],
                             None, None, None, stream=0)
    assert rc == code


def test_mla_split_request_and_workspace_host_logic():
    assert K.blasst_mla_decode_num_splits(4, 16, 1000, 8) == (K.BLASST_OK, 8)
    assert K.blasst_mla_decode_num_splits(4, 16, 1000, 9)[0] == K.BLASST_ERR_INVALID_ARG
    assert K.blasst_mla_decode_workspace_size(4, 16, 1000, 1) == 0
    o_bytes = 3 * 4 * 16 * 512 * 4
    assert K.blasst_mla_decode_workspace_size(4, 16, 1000, 3) == ((o_bytes + 255) & ~255) + 3 * 4 * 16 * 4


# The cluster paths (MLA decode above 64 heads, GQA decode with 128 heads per KV
# head) multicast their key loads inside a cluster; they accept only device memory
# of the current GPU.  A host address (here one that is never dereferenced) is
# refused after argument validation and before any work is enqueued.
def test_cluster_paths_refuse_memory_not_on_this_gpu():
    rc = K.blasst_mla_decode(FAKE, FAKE, None, None, FAKE, None, 2, 128, 1000, 576, 512, 0, 0, 0, 0.1, 0.01, 1,
                             None, 0, None, None, None, stream=0)
    assert rc == K.BLASST_ERR_UNSUPPORTED
    rc = K.blasst_mla_decode(FAKE, FAKE, FAKE, None, FAKE, None, 2, 128, 1000, 576, 512, 40, 64, 16, 0.1, 0.01, 1,
                             None, 0, None, None, None, stream=0)
    assert rc == K.BLASST_ERR_UNSUPPORTED
    rc = K.blasst_decode(FAKE, FAKE, FAKE, FAKE, None, 2, 128, 1, 1000, 128, 0.1, 0.01, 1, None, 0, None, None, None,
                         stream=0)
    assert rc == K.BLASST_ERR_UNSUPPORTED
    # validation still comes first: a bad argument is reported as such
    rc = K.blasst_mla_decode(FAKE, FAKE, None, None, FAKE, None, 2, 128, 1000, 576, 512, 0, 0, 0, 0.1, 2.0, 1,
                             None, 0, None, None, None, stream=0)
    assert rc == K.BLASST_ERR_INVALID_ARG


@pytest.mark.parametrize("kw,code", [
    (dict(S=300), K.BLASST_ERR_INVALID_ARG),           # more splits than the 256 key tiles
    (dict(Hq=96, Hkv=2), K.BLASST_ERR_UNSUPPORTED),    # G = 48
    (dict(d=96), K.BLASST_ERR_UNSUPPORTED),
    (dict(lam=1.5), K.BLASST_ERR_INVALID_ARG),
    (dict(q=None), K.BLASST_ERR_INVALID_ARG),
    (dict(S=64), K.BLASST_ERR_SCRATCH_LIMIT),          # valid, but the partials exceed the scratch
])
def test_noalloc_validates_before_the_scratch_limit(kw, code):
    # every case but the last is also far beyond the scratch size, so the argument
    # error must win over BLASST_ERR_SCRATCH_LIMIT
    a = dict(q=FAKE, B=64, Hq=32, Hkv=8, Lkv=32768, d=128, lam=0.0, S=200)
    a.update(kw)
    rc = K.blasst_decode_noalloc(a["q"], FAKE, FAKE, FAKE, None, a["B"], a["Hq"], a["Hkv"], a["Lkv"], a["d"], 0.1,
                                 a["lam"], a["S"], None, None, None, stream=0)
    assert rc == code
