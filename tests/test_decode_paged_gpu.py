"""Paged, variable-length decode on the GPU (blasst_decode_paged) against the CPU
oracle run on each sequence alone, plus bit-for-bit agreement with the contiguous
decode when every sequence is full length."""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

from skip_softmax_flashattention_gb300 import blasst as K
from skip_softmax_flashattention_gb300 import workloads as W
from tests import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _status_clean():
    K.blasst_device_status(1)
    yield
    assert K.blasst_device_status(1) == K.BLASST_OK, "a kernel wait timed out or read a bad page index"


def _run(a, lam, S, **kw):
    e = a.extra
    res = K.decode_paged(a.q, e["k_pages"], e["v_pages"], e["page_table"], e["seq_lens"], e["max_len"],
                         e["page_size"], e["token_major"], a.scale, lam, S, want_map=True, **kw)
    torch.cuda.synchronize()
    return res


# lengths: full, one key, a ragged middle, an exact tile multiple, below one tile
LENS = [1000, 1, 517, 768, 100]


@pytest.mark.parametrize("page_size", [8, 16, 32, 64, 128, 256])
@pytest.mark.parametrize("token_major", [True, False], ids=["key-major", "head-major"])
@pytest.mark.parametrize("S", [1, 3])
@pytest.mark.parametrize("lam", [0.0, 0.3])
def test_paged_matches_oracle_per_sequence(page_size, token_major, S, lam):
    a = W.paged_decode(seed=3, B=len(LENS), Hq=8, Hkv=2, max_len=1000, page_size=page_size,
                       token_major=token_major, lens=LENS, device="cuda")
    res = _run(a, lam, S)
    assert res["num_splits"] == S
    parity.decode_paged_check(a, res, lam, S)


@pytest.mark.parametrize("G", [1, 4, 16])
def test_paged_group_sizes(G):
    Hkv = 2
    a = W.paged_decode(seed=4, B=3, Hq=G * Hkv, Hkv=Hkv, max_len=700, page_size=32, lens=[700, 300, 129],
                       device="cuda")
    for lam in (0.0, 0.3):
        parity.decode_paged_check(a, _run(a, lam, 2), lam, 2)


@pytest.mark.parametrize("page_size,token_major", [(16, True), (128, False), (512, True)])
def test_paged_full_length_equals_contiguous_bitwise(page_size, token_major):
    """With every sequence at full length the paged kernel computes exactly what the
    contiguous one does; only the addresses of the loads differ."""
    L = 2048
    a = W.paged_decode(seed=5, B=4, Hq=16, Hkv=4, max_len=L, page_size=page_size, token_major=token_major,
                       lens=[L] * 4, device="cuda")
    q3 = a.q.reshape(a.B, a.Hq, a.d)
    for lam, S in ((0.0, 1), (0.3, 2)):
        ref = K.decode(q3, a.k, a.v, a.scale, lam, S, want_map=True, want_margins=True)
        got = _run(a, lam, S, want_margins=True)
        torch.cuda.synchronize()
        assert torch.equal(got["map"], ref["map"])
        assert torch.equal(got["o"], ref["o"])
        assert torch.equal(got["lse"], ref["lse"])
        assert torch.equal(got["margins"], ref["margins"])
        assert int(got["skipped"].item()) == int(ref["skipped"].item())


@pytest.mark.parametrize("window", [1, 100, 128, 300, 2000])
@pytest.mark.parametrize("page_size", [16, 128])
def test_paged_sliding_window(window, page_size):
    a = W.paged_decode(seed=9, B=len(LENS), Hq=8, Hkv=2, max_len=1000, page_size=page_size, lens=LENS, device="cuda")
    for lam, S in ((0.0, 1), (0.3, 2), (0.0, 3)):
        res = _run(a, lam, S, window=window)
        parity.decode_paged_check(a, res, lam, S, window=window)


def test_paged_zero_length_sequence():
    a = W.paged_decode(seed=6, B=3, Hq=8, Hkv=2, max_len=600, page_size=64, lens=[600, 0, 5], device="cuda")
    for S in (1, 2):
        parity.decode_paged_check(a, _run(a, 0.0, S), 0.0, S)


def test_paged_bad_page_index_reads_zeros_and_is_reported():
    """An out-of-range page index is never dereferenced: the box reads as zeros, the
    device status says so, and the next call is normal."""
    a = W.paged_decode(seed=7, B=2, Hq=8, Hkv=2, max_len=512, page_size=64, lens=[512, 300], device="cuda")
    table = a.extra["page_table"].clone()
    bad = table.clone()
    bad[0, 1] = a.extra["k_pages"].shape[0] + 1000
    a.extra["page_table"] = bad
    res = _run(a, 0.0, 1)
    assert K.blasst_device_status(1) == K.BLASST_ERR_PAGE_TABLE
    assert torch.isfinite(res["o"].float()).all()
    a.extra["page_table"] = table
    parity.decode_paged_check(a, _run(a, 0.0, 1), 0.0, 1)


def test_paged_serving_batch_sampled():
    """B=64 sequences of 16k-32k keys in 16-key pages, split as the library chooses;
    six sequences checked against the oracle."""
    a = W.paged_decode(seed=8, B=64, Hq=32, Hkv=8, max_len=32768, page_size=16, min_len=16384, device="cuda")
    for lam in (0.0, 0.3):
        res = _run(a, lam, 0)
        parity.decode_paged_check(a, res, lam, res["num_splits"], seqs=[0, 1, 17, 40, 62, 63])


@pytest.mark.parametrize("page_size,token_major", [(16, True), (128, False)])
def test_paged_head_dim_64(page_size, token_major):
    a = W.paged_decode(seed=12, B=4, Hq=8, Hkv=2, max_len=1000, d=64, page_size=page_size,
                       token_major=token_major, lens=[1000, 1, 517, 300], device="cuda")
    for lam, S in ((0.0, 1), (0.3, 3)):
        res = _run(a, lam, S)
        parity.decode_paged_check(a, res, lam, S)
