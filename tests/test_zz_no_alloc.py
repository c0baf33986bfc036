"""blasst_decode_noalloc: the decode entry point for callers that cannot allocate
device memory (their memory belongs to another allocator, or they must not
allocate between serving steps).  It must give the results of blasst_decode with
a caller workspace, call after call, although every call reuses the library's one
static scratch array.  Collected last on purpose (file name), so a failure here
cannot hide any other test's result."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from skip_softmax_flashattention_gb300 import blasst as K
from skip_softmax_flashattention_gb300 import workloads as W
from tests import parity

pytestmark = pytest.mark.gpu

O_MAX_ABS = 2e-2
LSE_ABS = 1e-3


def _run_noalloc(a, lam, S):
    q3 = a.q.reshape(a.B, a.Hq, a.d)
    o = torch.empty(a.B, a.Hq, a.d, device="cuda", dtype=torch.bfloat16)
    lse = torch.empty(a.B, a.Hq, device="cuda", dtype=torch.float32)
    skipped = torch.zeros(1, device="cuda", dtype=torch.int64)
    nK = -(-a.Lkv // 128)
    mp = torch.empty(a.B, a.Hkv, nK, device="cuda", dtype=torch.uint8)
    rc = K.blasst_decode_noalloc(q3, a.k, a.v, o, lse, a.B, a.Hq, a.Hkv, a.Lkv, a.d, a.scale, lam, S, skipped, mp,
                                 None)
    assert rc == K.BLASST_OK, K.blasst_status_string(rc)
    torch.cuda.synchronize()
    return o, lse, skipped, mp


def _compare_oracle(a, lam, S, got):
    """The no-alloc result against the CPU oracle: every tile decision (outside the
    1e-3 margin band), the exact skipped count, O and lse."""
    o, lse, skipped, mp = got
    parity.decode_full_check(a, {"o": o, "lse": lse, "skipped": skipped, "map": mp}, lam, S)


def _compare(ref, got):
    o, lse, skipped, mp = got
    assert torch.equal(ref["map"], mp)
    assert int(ref["skipped"].item()) == int(skipped.item())
    err = (o.float() - ref["o"].float()).abs()
    assert float(err.max()) <= O_MAX_ABS
    assert float((lse - ref["lse"]).abs().max()) <= LSE_ABS


def test_noalloc_matches_workspace_decode_on_consecutive_calls():
    torch.cuda.set_device(0)
    K.blasst_device_status(1)
    S, lam = 3, 0.05
    first = W.decode(seed=31, B=4, Hq=32, Hkv=8, Lkv=3000, device="cuda")
    second = W.decode(seed=32, B=4, Hq=32, Hkv=8, Lkv=3000, device="cuda")
    ref1 = K.decode(first.q, first.k, first.v, first.scale, lam, num_splits=S, want_map=True)
    ref2 = K.decode(second.q, second.k, second.v, second.scale, lam, num_splits=S, want_map=True)
    torch.cuda.synchronize()
    # two calls in a row on different inputs: the second must not see the first's partials
    _compare(ref1, _run_noalloc(first, lam, S))
    _compare(ref2, _run_noalloc(second, lam, S))
    # and once more on the first input
    _compare(ref1, _run_noalloc(first, lam, S))
    assert K.blasst_device_status(1) == K.BLASST_OK


def test_noalloc_matches_the_oracle():
    torch.cuda.set_device(0)
    K.blasst_device_status(1)
    a = W.decode(seed=33, B=3, Hq=16, Hkv=4, Lkv=1500, device="cuda")
    for lam, S in ((0.0, 3), (0.3, 3), (0.3, 1)):
        _compare_oracle(a, lam, S, _run_noalloc(a, lam, S))
    assert K.blasst_device_status(1) == K.BLASST_OK


def test_noalloc_wide_group_head_dim_64():
    """32 query heads per KV head (the wide-group kernel, which also writes its split
    partials to the scratch) at head dim 64."""
    torch.cuda.set_device(0)
    K.blasst_device_status(1)
    a = W.decode(seed=34, B=2, Hq=64, Hkv=2, Lkv=1000, d=64, device="cuda")
    for lam in (0.0, 0.3):
        got = _run_noalloc(a, lam, 3)
        ref = K.decode(a.q, a.k, a.v, a.scale, lam, num_splits=3, want_map=True)
        torch.cuda.synchronize()
        _compare(ref, got)
        _compare_oracle(a, lam, 3, got)
    assert K.blasst_device_status(1) == K.BLASST_OK


def test_noalloc_large_call_then_smaller_call():
    """A call that fills much of the scratch (8 splits) followed by a smaller one (2
    splits, other inputs, other shape): the smaller call must read only its own
    partials, not what the larger one left behind."""
    torch.cuda.set_device(0)
    K.blasst_device_status(1)
    big = W.decode(seed=35, B=8, Hq=32, Hkv=8, Lkv=4096, device="cuda")
    small = W.decode(seed=36, B=5, Hq=16, Hkv=4, Lkv=2000, device="cuda")
    lam = 0.2
    assert K.blasst_decode_workspace_size(big.B, big.Hq, big.Hkv, big.Lkv, big.d, 8) > \
        K.blasst_decode_workspace_size(small.B, small.Hq, small.Hkv, small.Lkv, small.d, 2)
    _compare_oracle(big, lam, 8, _run_noalloc(big, lam, 8))
    got = _run_noalloc(small, lam, 2)
    _compare_oracle(small, lam, 2, got)
    ref = K.decode(small.q, small.k, small.v, small.scale, lam, num_splits=2, want_map=True)
    torch.cuda.synchronize()
    _compare(ref, got)
    assert K.blasst_device_status(1) == K.BLASST_OK


def test_noalloc_rejects_partials_beyond_the_scratch():
    cap = K.blasst_decode_noalloc_scratch_bytes()
    assert cap == 4 << 20
    B, Hq, Hkv, Lkv, d = 64, 32, 8, 32768, 128
    S = 64  # 64 * 64 * 32 * 129 * 4 bytes >> 4 MiB
    assert K.blasst_decode_workspace_size(B, Hq, Hkv, Lkv, d, S) > cap
    fake = 1 << 20  # never dereferenced: the size check comes first
    rc = K.blasst_decode_noalloc(fake, fake, fake, fake, None, B, Hq, Hkv, Lkv, d, 0.1, 0.0, S, None, None, None,
                                 None)
    assert rc == K.BLASST_ERR_SCRATCH_LIMIT
