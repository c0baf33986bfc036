"""Split-KV decode parity on the GPU: the CUDA kernels (split pass + merge)
against the CPU oracle, whole on small problems and on sampled (batch, KV head)
pairs at the full decode workload size."""
from __future__ import annotations

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
    assert K.blasst_device_status(1) == K.BLASST_OK, "a kernel wait timed out"


SHAPES = [
    # B, Hq, Hkv, Lkv
    (2, 8, 2, 1000),
    (3, 4, 4, 129),
    (1, 16, 1, 5000),
    (2, 32, 2, 777),
    (1, 2, 1, 128),
    (4, 32, 8, 2048),
]


@pytest.mark.parametrize("shape", SHAPES, ids=[str(s) for s in SHAPES])
@pytest.mark.parametrize("S", [1, 2, 5])
@pytest.mark.parametrize("lam", [0.0, 0.05, 0.3])
def test_decode_small(shape, S, lam):
    B, Hq, Hkv, L = shape
    if S > -(-L // 128):
        pytest.skip("more splits than key tiles")
    a = parity.to_gpu(W.decode(seed=21, B=B, Hq=Hq, Hkv=Hkv, Lkv=L))
    res = K.decode(a.q, a.k, a.v, a.scale, lam, num_splits=S, want_map=True)
    torch.cuda.synchronize()
    band, mx, mean, n = parity.decode_full_check(a, res, lam, S)
    if lam == 0.0:
        assert n == 0


def test_decode_full_size():
    a = parity.to_gpu(W.decode(seed=0, device="cuda"))
    rc, S = K.blasst_decode_num_splits(a.B, a.Hq, a.Hkv, a.Lkv, a.d, 0)
    assert rc == 0
    rng = np.random.default_rng(3)
    units = sorted({(0, 0), (a.B - 1, a.Hkv - 1)} | {(int(rng.integers(a.B)), int(rng.integers(a.Hkv)))
                                                       for _ in range(6)})
    for lam in (0.0, 4 / a.Lkv, 40 / a.Lkv, 0.3):
        res = K.decode(a.q, a.k, a.v, a.scale, lam, num_splits=S, want_map=True)
        torch.cuda.synchronize()
        n = int(res["skipped"].item())
        assert n == int((res["map"] == 1).sum().item())
        if lam == 0.0:
            assert n == 0
        parity.decode_units_check(a, res, lam, S, units)


@pytest.mark.parametrize("shape", [(2, 8, 2, 1000), (1, 16, 1, 777), (3, 4, 4, 129)], ids=str)
@pytest.mark.parametrize("lam", [0.0, 0.3])
def test_decode_head_dim_64(shape, lam):
    """d = 64 runs the width-128 kernel with the upper 64 columns read as zeros."""
    B, Hq, Hkv, L = shape
    a = parity.to_gpu(W.decode(seed=23, B=B, Hq=Hq, Hkv=Hkv, Lkv=L, d=64))
    for S in sorted({1, min(3, -(-L // 128))}):
        res = K.decode(a.q, a.k, a.v, a.scale, lam, num_splits=S, want_map=True)
        torch.cuda.synchronize()
        assert res["o"].shape[-1] == 64
        parity.decode_full_check(a, res, lam, S)


# More than 16 query heads per KV head (MQA and wide GQA): the wide-group kernel,
# 32 / 64 heads in one CTA, 128 in a cluster of two.
WIDE = [
    # B, Hq, Hkv, Lkv, d
    (2, 32, 1, 1000, 128),
    (1, 64, 1, 777, 64),
    (2, 64, 2, 1500, 128),
    (1, 128, 1, 600, 128),
    (2, 128, 2, 300, 64),
]


@pytest.mark.parametrize("shape", WIDE, ids=[str(s) for s in WIDE])
@pytest.mark.parametrize("lam", [0.0, 0.3])
def test_decode_wide_groups(shape, lam):
    B, Hq, Hkv, L, d = shape
    a = parity.to_gpu(W.decode(seed=29, B=B, Hq=Hq, Hkv=Hkv, Lkv=L, d=d))
    for S in sorted({1, min(3, -(-L // 128))}):
        res = K.decode(a.q, a.k, a.v, a.scale, lam, num_splits=S, want_map=True)
        torch.cuda.synchronize()
        assert res["o"].shape == (B, Hq, d)
        parity.decode_full_check(a, res, lam, S)


def test_decode_wide_group_full_size_sampled():
    """64 sequences x 32768 keys, one KV head read by 64 query heads (MQA), the
    library's split plan: two sequences against the oracle."""
    a = parity.to_gpu(W.decode(seed=30, B=64, Hq=64, Hkv=1, Lkv=32768, d=128))
    for lam in (0.0, 0.3):
        res = K.decode(a.q, a.k, a.v, a.scale, lam, want_map=True)
        torch.cuda.synchronize()
        parity.decode_units_check(a, res, lam, res["num_splits"], [(0, 0), (63, 0)])
    del a, res
    torch.cuda.empty_cache()


MARGIN_SHAPES = [
    # B, Hq, Hkv, Lkv, d, S
    (2, 8, 2, 1000, 128, 3),
    (3, 4, 4, 129, 128, 1),
    (1, 16, 1, 5000, 128, 5),
    (2, 8, 2, 777, 64, 2),
    (2, 32, 1, 1000, 128, 2),    # wide group, one CTA
    (1, 128, 1, 600, 128, 2),    # wide group, cluster of two
]


@pytest.mark.parametrize("shape", MARGIN_SHAPES, ids=[str(s) for s in MARGIN_SHAPES])
def test_decode_margins_match_oracle(shape):
    """The decode margins (what threshold calibration reads) against the oracle's, tile
    by tile; at lambda = 0 the margins are the same for every threshold."""
    from oracle import oracle as orc

    B, Hq, Hkv, L, d, S = shape
    a = parity.to_gpu(W.decode(seed=41, B=B, Hq=Hq, Hkv=Hkv, Lkv=L, d=d))
    res = K.decode(a.q, a.k, a.v, a.scale, 0.0, num_splits=S, want_map=True, want_margins=True)
    torch.cuda.synchronize()
    own = orc.decode_tiled(a.q.float().cpu(), a.k.float().cpu(), a.v.float().cpu(), a.scale, 0.0, num_splits=S,
                           precision="f32")
    parity.margins_check(res["margins"].cpu().numpy(), own["margin"], f"decode margins {shape}")
    # and a threshold taken from them skips exactly the oracle's tiles (outside the band)
    from skip_softmax_flashattention_gb300 import calibrate

    lam = calibrate.lambda_for_sparsity(own["margin"], 0.5)
    r2 = K.decode(a.q, a.k, a.v, a.scale, lam, num_splits=S, want_map=True)
    torch.cuda.synchronize()
    parity.decode_full_check(a, r2, lam, S)


def test_decode_margins_full_size_sampled():
    """The bench's decode workload: margins of sampled (sequence, KV head) units against
    the oracle (the 70 % threshold of the bench is read off these margins)."""
    from oracle import oracle as orc

    a = parity.to_gpu(W.decode(seed=0, device="cuda"))
    res = K.decode(a.q, a.k, a.v, a.scale, 0.0, want_map=True, want_margins=True)
    torch.cuda.synchronize()
    S = res["num_splits"]
    g = res["margins"].cpu().numpy()
    G = a.Hq // a.Hkv
    for (b, hk) in [(0, 0), (17, 3), (63, 7)]:
        own = orc.decode_tiled(a.q[b:b + 1, hk * G:(hk + 1) * G].float().cpu(), a.k[b:b + 1, hk:hk + 1].float().cpu(),
                               a.v[b:b + 1, hk:hk + 1].float().cpu(), a.scale, 0.0, num_splits=S, precision="f32")
        parity.margins_check(g[b:b + 1, hk:hk + 1], own["margin"], f"decode margins b={b} hkv={hk}")
    del a, res
    torch.cuda.empty_cache()
