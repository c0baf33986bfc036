"""Full-size parity with exact skipped-tile counts: the GPU kernels against the CPU
oracle on whole problems of the benchmark's workloads.

Each problem is run once through the oracle at lambda = 0.  That pass gives the
lambda-independent per-tile margins, hence the oracle's own decision at every
threshold (tests.parity.oracle_map_at), and O / lse with every tile computed.  Every
GPU threshold is then checked on every visited tile:
  * each decision equals the oracle's outside the 1e-3 margin band;
  * the skipped count equals the oracle's (exactly, when no tile is in the band);
  * O and lse match the oracle run with the GPU's skip map forced (re-run only
    when the GPU skipped a tile, otherwise the lambda = 0 pass is that run).

Workloads: causal GQA LLM prefill at 16384 (whole), split-KV decode of 64 x 32768
(whole), video DiT (two whole heads: every query tile of each), the long-context
prefill at 8192 on the evaluation seed (whole), planted-70 (two whole heads), paged
decode of a 64-sequence serving batch (whole), MLA decode with 16 heads (whole).  These are slow (minutes of CPU
oracle time in total)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from oracle import oracle as orc
from skip_softmax_flashattention_gb300 import blasst as K
from skip_softmax_flashattention_gb300 import workloads as W
from tests import parity

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(autouse=True)
def _status_clean():
    K.blasst_device_status(1)
    yield
    assert K.blasst_device_status(1) == K.BLASST_OK, "a kernel wait timed out"
    torch.cuda.empty_cache()


def _prefill_whole(a, lams, heads=None, expect_zero=(0.0,)):
    """Every threshold of `lams` on the whole problem (or on every query tile of the
    listed heads, each with its own exact count)."""
    G = a.Hq // a.Hkv
    if heads is None:
        hq = list(range(a.Hq))
    else:
        hq = list(heads)
    hk = sorted({h // G for h in hq})
    q = a.q[:, hq].float().cpu()
    k = a.k[:, hk].float().cpu()
    v = a.v[:, hk].float().cpu()
    own0 = orc.prefill_tiled(q, k, v, a.causal, a.scale, 0.0, precision="f32")
    assert own0["skipped"] == 0
    counts = {}
    for lam in lams:
        res = K.prefill(a.q, a.k, a.v, a.causal, a.scale, lam, want_map=True, want_margins=(lam == 0.0))
        torch.cuda.synchronize()
        n_all = int(res["skipped"].item())
        assert n_all == int((res["map"] == 1).sum().item()), "reported count differs from the map"
        sub = {"map": res["map"][:, hq], "o": res["o"][:, hq], "lse": res["lse"][:, hq]}
        sub["skipped"] = torch.tensor(int((sub["map"] == 1).sum().item()))
        if lam == 0.0:
            parity.margins_check(res["margins"][:, hq].cpu().numpy(), own0["margin"], f"{a.name} margins")

        def forced(gmap, lam=lam):
            return orc.prefill_tiled(q, k, v, a.causal, a.scale, lam, forced=gmap, precision="f32")

        band, n = parity.whole_check(f"{a.name} lam={lam:g} heads={'all' if heads is None else hq}", lam, sub,
                                     own0, forced)
        if lam in expect_zero:
            assert n == 0
        counts[lam] = (n, band)
        del res, sub
    return counts


def test_llm_prefill_whole_problem_exact_counts():
    """LLM prefill, causal GQA, L = 16384, at lambda = a / L for a in {0, 4, 40} and at
    lambda = 1 (about 8 % of the tiles skipped)."""
    L = 16384
    a = W.llm(seed=0, L=L, device="cuda")
    counts = _prefill_whole(a, [0.0, 4 / L, 40 / L, 1.0])
    assert counts[1.0][0] > 0


def test_long_context_prefill_L8192_whole_problem():
    """The long-context sweep's shortest length, whole, on the evaluation seed (2): at
    lambda = 0 and at lambda = 1 (the fitted curve asks for lambda > 1 there, so the
    sweep runs lambda = 1)."""
    a = W.llm(seed=2, L=8192, device="cuda")
    counts = _prefill_whole(a, [0.0, 1.0])
    assert counts[1.0][0] > 0


@pytest.mark.parametrize("heads", [(0, 23), (11, 39)])
def test_dit_two_whole_heads_exact_counts(heads):
    """Video DiT, non-causal, H = 40, L = 32760: every query tile of two heads at each
    of the workload's thresholds, with the exact count per pair of heads."""
    a = W.dit(seed=0, device="cuda")
    counts = _prefill_whole(a, [0.0, 1e-4, 1e-3, 1e-2], heads=heads)
    for lam in (1e-4, 1e-3, 1e-2):
        assert counts[lam][0] > 0


def test_decode_whole_problem_exact_counts():
    """Split-KV decode, B = 64, Hq = 32, Hkv = 8, Lkv = 32768, with the bench's split
    plan, at lambda = a / Lkv for a in {0, 4, 40} and at lambda = 0.3: all 512
    (sequence, KV head) units, every tile decision, the exact count, every O / lse row
    and the margins."""
    a = W.decode(seed=0, device="cuda")
    q3 = a.q.reshape(a.B, a.Hq, a.d)
    lams = [0.0, 4 / a.Lkv, 40 / a.Lkv, 0.3]
    results = {}
    S = None
    for lam in lams:
        r = K.decode(q3, a.k, a.v, a.scale, lam, num_splits=0 if S is None else S, want_map=True,
                     want_margins=(lam == 0.0))
        torch.cuda.synchronize()
        S = r["num_splits"]
        results[lam] = r
    # the oracle in chunks of sequences (the fp32 copy of the whole cache is 17 GB)
    chunk = 8
    parts = []
    for b0 in range(0, a.B, chunk):
        sl = slice(b0, b0 + chunk)
        parts.append(orc.decode_tiled(a.q[sl].float().cpu(), a.k[sl].float().cpu(), a.v[sl].float().cpu(), a.scale,
                                      0.0, num_splits=S, precision="f32"))
    own0 = {key: np.concatenate([p[key] for p in parts], axis=0) for key in ("o", "lse", "map", "margin")}
    own0["skipped"] = sum(p["skipped"] for p in parts)
    assert own0["skipped"] == 0
    parity.margins_check(results[0.0]["margins"].cpu().numpy(), own0["margin"], "decode margins")

    def forced(gmap, lam):
        o, lse = [], []
        for b0 in range(0, a.B, chunk):
            sl = slice(b0, b0 + chunk)
            r = orc.decode_tiled(a.q[sl].float().cpu(), a.k[sl].float().cpu(), a.v[sl].float().cpu(), a.scale,
                                 lam, num_splits=S, forced=gmap[sl], precision="f32")
            o.append(r["o"])
            lse.append(r["lse"])
        return {"o": np.concatenate(o), "lse": np.concatenate(lse)}

    for lam in lams:
        band, n = parity.whole_check(f"decode lam={lam:g} S={S}", lam, results[lam], own0,
                                     lambda gmap, lam=lam: forced(gmap, lam))
        if lam == 0.0:
            assert n == 0
    assert int(results[0.3]["skipped"].item()) > 0


def test_planted70_two_whole_heads_exact_counts():
    """The bench's skip point: planted-70 (the LLM prefill shapes, non-causal, the last
    70 % of key tiles hold K = 0) at lambda = 1e-2, every query tile of two heads of one
    K/V group, with the exact count; 70.3 % of their tiles are skipped."""
    a = W.planted70(seed=0, L=16384, device="cuda")
    counts = _prefill_whole(a, [0.0, 1e-2], heads=(4, 7))
    n, band = counts[1e-2]
    assert band == 0
    assert n == 2 * 128 * 90  # key tiles 38..127 of every query tile of the two heads


def test_paged_decode_whole_serving_batch_exact_counts():
    """Paged decode of a serving batch: 64 sequences of 16k-32k keys in 16-key pages
    (key-major pool), the library's split plan, at lambda = 0 and 0.3.  Every sequence
    against the oracle run on it alone (decisions outside the 1e-3 band, O, lse), and
    the batch's skipped count equal to the oracle's up to the decisions that differ
    inside the band (exactly, when none do)."""
    a = W.paged_decode(seed=8, B=64, Hq=32, Hkv=8, max_len=32768, page_size=16, min_len=16384, device="cuda")
    e = a.extra
    for lam in (0.0, 0.3):
        res = K.decode_paged(a.q, e["k_pages"], e["v_pages"], e["page_table"], e["seq_lens"], e["max_len"],
                             e["page_size"], e["token_major"], a.scale, lam, 0, want_map=True)
        torch.cuda.synchronize()
        n = int(res["skipped"].item())
        differ, n_oracle = parity.decode_paged_check(a, res, lam, res["num_splits"])
        assert abs(n - n_oracle) <= differ
        if differ == 0:
            assert n == n_oracle
        if lam == 0.0:
            assert n == 0
        else:
            assert n > 0
        del res
    del a
    torch.cuda.empty_cache()


def test_mla_decode_whole_problem_exact_counts():
    """MLA decode, 64 sequences x 32768 latent rows, 16 query heads, the planner's
    splits, at lambda = 0 and 0.03: every sequence against the oracle (decisions
    outside the 1e-3 band, O, lse), and the skipped count equal to the oracle's up to
    the decisions that differ inside the band (exactly, when none do)."""
    a = W.mla_decode(seed=0, B=64, Hq=16, L=32768, device="cuda")
    for lam in (0.0, 0.03):
        res = K.mla_decode(a.q, a.extra["kv"], a.scale, lam, 0, want_map=True)
        torch.cuda.synchronize()
        n = int(res["skipped"].item())
        differ, n_oracle = parity.mla_check(a, res, lam, res["num_splits"], counts=True)
        assert abs(n - n_oracle) <= differ
        if differ == 0:
            assert n == n_oracle
        assert (n == 0) if lam == 0.0 else (n > 0)
        del res
    del a
    torch.cuda.empty_cache()
