"""MLA decode parity on the GPU: the CUDA kernel against the CPU oracle.

The latent cache holds one 576-value row per token (keys of every head; values =
the first 512 values).  Small problems are compared sequence by sequence in full
(every tile decision, the exact skipped count, O and lse); the full-size problem
(64 sequences x 32k rows, 16 heads) on sampled sequences in the launch
configuration the benchmark times."""
from __future__ import annotations

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


def _run(a, lam, S, page=False):
    ex = a.extra
    if page:
        return K.mla_decode(a.q, ex["kv_pages"], a.scale, lam, S, seq_lens=ex["seq_lens"],
                            page_table=ex["page_table"], page_size=ex["page_size"], max_kv_len=ex["kv"].shape[1],
                            want_map=True, want_margins=True)
    return K.mla_decode(a.q, ex["kv"], a.scale, lam, S, seq_lens=ex["seq_lens"], want_map=True, want_margins=True)


@pytest.mark.parametrize("Hq", [1, 8, 16])
@pytest.mark.parametrize("L", [1, 127, 129, 700, 1500])
@pytest.mark.parametrize("lam", [0.0, 0.03, 0.1])
def test_contiguous_cache(Hq, L, lam):
    a = W.mla_decode(seed=L + Hq, B=3, Hq=Hq, L=L, device="cuda")
    nT = -(-L // 128)
    for S in sorted({1, min(2, nT), min(5, nT)}):
        res = _run(a, lam, S)
        torch.cuda.synchronize()
        parity.mla_check(a, res, lam, S)
        if lam == 0.0:
            assert int(res["skipped"].item()) == 0


@pytest.mark.parametrize("Hq", [2, 4])
def test_other_head_counts(Hq):
    a = W.mla_decode(seed=3, B=2, Hq=Hq, L=1000, device="cuda")
    for lam in (0.0, 0.05):
        res = _run(a, lam, 3)
        torch.cuda.synchronize()
        parity.mla_check(a, res, lam, 3)


def test_sequence_lengths_including_empty_and_tile_edges():
    lens = [0, 1, 127, 128, 129, 1000, 2048, 2049]
    a = W.mla_decode(seed=5, B=len(lens), Hq=16, L=2049, lens=lens, device="cuda")
    for lam, S in ((0.0, 1), (0.03, 4), (0.1, 17)):
        res = _run(a, lam, S)
        torch.cuda.synchronize()
        parity.mla_check(a, res, lam, S)


@pytest.mark.parametrize("page_size", [8, 16, 32, 64, 128, 256])
def test_paged_cache_matches_contiguous_bitwise_and_oracle(page_size):
    """The paged form reads the same rows through a page table: its map, O and lse
    equal the contiguous form's bit for bit, and the oracle's."""
    a = W.mla_decode(seed=page_size, B=6, Hq=16, L=1500, min_len=0, page_size=page_size, device="cuda")
    for lam, S in ((0.0, 1), (0.05, 3)):
        ref = _run(a, lam, S)
        got = _run(a, lam, S, page=True)
        torch.cuda.synchronize()
        assert torch.equal(got["map"], ref["map"])
        assert torch.equal(got["o"], ref["o"]) and torch.equal(got["lse"], ref["lse"])
        assert int(got["skipped"].item()) == int(ref["skipped"].item())
        parity.mla_check(a, got, lam, S)


def test_margins_match_oracle():
    from oracle import oracle as orc
    import numpy as np

    a = W.mla_decode(seed=9, B=2, Hq=16, L=2000, device="cuda")
    res = _run(a, 0.0, 2)
    torch.cuda.synchronize()
    g = res["margins"].cpu().numpy()
    for b in range(2):
        own = orc.mla_decode_tiled(a.q[b:b + 1].float().cpu(), a.extra["kv"][b:b + 1].float().cpu(), 512, a.scale,
                                   0.0, num_splits=2)
        ref = own["margin"][0]
        fin = np.isfinite(ref)
        assert np.array_equal(np.isnan(g[b]), np.isnan(ref))
        assert np.abs(g[b][fin] - ref[fin]).max() < 1e-3


def test_full_size_sampled_sequences():
    """64 sequences x 32768 rows x 16 heads, the split count the planner picks, at
    lambda = 0 and at a threshold that skips part of the tiles: the first, the
    last and two random sequences against the oracle."""
    a = W.mla_decode(seed=0, B=64, Hq=16, L=32768, device="cuda")
    for lam in (0.0, 0.03):
        res = _run(a, lam, 0)
        torch.cuda.synchronize()
        S = res["num_splits"]
        n = int(res["skipped"].item())
        if lam == 0.0:
            assert n == 0
        else:
            assert n > 0
        parity.mla_check(a, res, lam, S, seqs=[0, 17, 40, 63])
    del a, res
    torch.cuda.empty_cache()


# Above 16 heads the heads are spread over a cluster of Hq / 16 CTAs that share every
# load and exchange their votes.  The workload gives every head a shared query
# component and matching sinks, so that tiles skipped by all heads exist.
CLUSTER_KW = dict(q_shared=6.0, sink_norm=32.0)


@pytest.mark.parametrize("Hq", [32, 64, 128])
@pytest.mark.parametrize("L", [129, 1500])
def test_cluster_head_counts(Hq, L):
    a = W.mla_decode(seed=Hq + L, B=3, Hq=Hq, L=L, device="cuda", **CLUSTER_KW)
    nT = -(-L // 128)
    skipped = 0
    for lam in (0.0, 0.03, 0.1):
        for S in sorted({1, min(3, nT)}):
            res = _run(a, lam, S)
            torch.cuda.synchronize()
            parity.mla_check(a, res, lam, S)
            skipped += int(res["skipped"].item())
    if L > 129:
        assert skipped > 0


def test_cluster_lengths_and_pages():
    lens = [0, 1, 128, 129, 1000, 2049]
    a = W.mla_decode(seed=7, B=len(lens), Hq=64, L=2049, lens=lens, page_size=64, device="cuda", **CLUSTER_KW)
    for lam, S in ((0.0, 1), (0.1, 4)):
        ref = _run(a, lam, S)
        got = _run(a, lam, S, page=True)
        torch.cuda.synchronize()
        assert torch.equal(got["map"], ref["map"])
        assert torch.equal(got["o"], ref["o"]) and torch.equal(got["lse"], ref["lse"])
        parity.mla_check(a, got, lam, S)


def test_cluster_full_size_sampled():
    """64 sequences x 32768 rows x 128 heads (clusters of 8 CTAs), planner's splits."""
    a = W.mla_decode(seed=0, B=64, Hq=128, L=32768, device="cuda", **CLUSTER_KW)
    for lam in (0.0, 0.1):
        res = _run(a, lam, 0)
        torch.cuda.synchronize()
        n = int(res["skipped"].item())
        assert (n == 0) if lam == 0.0 else (n > 0)
        parity.mla_check(a, res, lam, res["num_splits"], seqs=[0, 63])
    del a, res
    torch.cuda.empty_cache()


@pytest.mark.parametrize("Hq", [16, 64])
def test_bad_page_index_and_length_are_contained_and_reported(Hq):
    """Out-of-range page indices (too large, negative) are never dereferenced: those
    rows read as zeros and the device status says so; a length above max_kv_len is
    clamped and reported.  The next normal call is exact."""
    kw = CLUSTER_KW if Hq > 16 else {}
    a = W.mla_decode(seed=11, B=3, Hq=Hq, L=640, lens=[640, 300, 500], page_size=64, device="cuda", **kw)
    ex = a.extra
    table, lens = ex["page_table"].clone(), ex["seq_lens"].clone()
    bad = table.clone()
    bad[0, 1] = ex["kv_pages"].shape[0] + 1000
    bad[1, 2] = -5
    ex["page_table"] = bad
    res = _run(a, 0.0, 2, page=True)
    torch.cuda.synchronize()
    assert K.blasst_device_status(1) == K.BLASST_ERR_PAGE_TABLE
    assert torch.isfinite(res["o"].float()).all() and not torch.isnan(res["lse"]).any()
    ex["page_table"] = table
    long_lens = lens.clone()
    long_lens[2] = 10 ** 6  # clamped to max_kv_len
    ex["seq_lens"] = long_lens
    res = _run(a, 0.0, 2, page=True)
    torch.cuda.synchronize()
    assert K.blasst_device_status(1) == K.BLASST_ERR_PAGE_TABLE
    assert int((res["map"][2] != 2).sum().item()) == 5  # 640 rows = 5 tiles
    ex["seq_lens"] = lens
    res = _run(a, 0.03, 2, page=True)
    torch.cuda.synchronize()
    parity.mla_check(a, res, 0.03, 2)


def test_cluster_paths_refuse_host_and_managed_memory():
    """The cluster kernels multicast key loads and accept only device memory of the
    current GPU: pinned host memory is refused before any work is enqueued, while
    the same data in device memory runs."""
    K.blasst_device_status(1)
    a = W.mla_decode(seed=5, B=1, Hq=128, L=300, device="cuda", q_shared=6.0, sink_norm=32.0)
    kv = a.extra["kv"]
    kv_host = kv.cpu().pin_memory()
    o = torch.empty(1, 128, 512, device="cuda", dtype=torch.bfloat16)
    rc = K.blasst_mla_decode(a.q, kv_host, None, None, o, None, 1, 128, 300, 576, 512, 0, 0, 0, a.scale, 0.1, 1,
                             None, 0, None, None, None)
    assert rc == K.BLASST_ERR_UNSUPPORTED
    rc = K.blasst_mla_decode(a.q, kv, None, None, o, None, 1, 128, 300, 576, 512, 0, 0, 0, a.scale, 0.1, 1,
                             None, 0, None, None, None)
    assert rc == K.BLASST_OK
    d = W.decode(seed=6, B=1, Hq=128, Hkv=1, Lkv=300, device="cuda")
    q3 = d.q.reshape(1, 128, 128)
    od = torch.empty(1, 128, 128, device="cuda", dtype=torch.bfloat16)
    rc = K.blasst_decode(q3, d.k.cpu().pin_memory(), d.v, od, None, 1, 128, 1, 300, 128, d.scale, 0.1, 1, None, 0,
                         None, None, None)
    assert rc == K.BLASST_ERR_UNSUPPORTED
    rc = K.blasst_decode(q3, d.k, d.v, od, None, 1, 128, 1, 300, 128, d.scale, 0.1, 1, None, 0, None, None, None)
    assert rc == K.BLASST_OK
    torch.cuda.synchronize()
    assert K.blasst_device_status(1) == K.BLASST_OK
