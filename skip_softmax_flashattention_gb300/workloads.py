"""Seeded synthetic inputs for the skip-softmax attention path.

This module only draws random numbers and arranges them into the shapes of the
workloads; it holds none of the attention arithmetic.  Both the CUDA path and the
CPU oracle take their inputs from here (the oracle receives the same bf16 values
widened to fp32/fp64), so the two can be compared element by element.

Workloads (shapes and distributions follow the kinds of rows the pages talk
about: long-context LLM prefill/decode with GQA, and video-DiT self-attention
with tens of thousands of keys per row -- Skip-Softmax design doc, "Motivation";
BLASST talk notes, "Results"):

* ``tiny``       B=1, H=2, L=512, d=64, iid N(0,1), logits x3 (scale 3/sqrt(64));
                 optional planted variant: keys 256..511 of each head are set to
                 -2 * (mean over the 512 query rows of that head).
* ``llm``        causal GQA prefill, B=1, Hq=32, Hkv=8, L=16384, d=128, iid N(0,1),
                 four sink keys at positions 0..3 of every KV head set to
                 3 * unit(mean of all query vectors that read that KV head),
                 logits x2 (scale 2/sqrt(128)).
* ``decode``     B=64, Hq=32, Hkv=8, one query token, Lkv=32768, d=128, same
                 generation and sink keys as ``llm``.
* ``dit``        non-causal MHA, B=1, H=40, L=32760 = 21x30x52 latent grid
                 (t-major, w fastest), Q and K = N(0,1) + 1.5 * (vector shared by
                 the 4x6x8 neighbourhood the token falls in; edge neighbourhoods
                 truncated), V iid N(0,1), scale 1/sqrt(128).
* ``planted70``  the ``llm`` shapes, non-causal, with K = 0 on the last 70% of the
                 key tiles: those tiles score 0 against a row max of several units,
                 so a threshold of 1e-2 skips exactly them.
* ``paged_decode`` a ``decode`` problem whose cache is cut into pages of
                 ``page_size`` keys and scattered over a page pool in a seeded
                 random order (the paged-KV indirection of The Hitchhiker's Guide,
                 Phase 08, Section 3), with a key count per sequence drawn
                 uniformly from [min_len, max_len] unless given.  Unused pool rows
                 hold N(0,1) values.

All tensors are drawn with a ``torch.Generator`` seeded by ``seed`` on the device
the tensors are made on; the values therefore depend on that device, and every
comparison uses one set of tensors for both sides.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

TILE = 128  # key/query tile edge used by the kernels (B_r = B_c = 128)


@dataclass
class Attn:
    """One attention problem: q [B,Hq,Lq,d], k/v [B,Hkv,Lkv,d] (bf16, contiguous)."""

    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    causal: bool
    scale: float
    name: str = ""
    extra: dict = field(default_factory=dict)

    @property
    def B(self):
        return self.q.shape[0]

    @property
    def Hq(self):
        return self.q.shape[1]

    @property
    def Hkv(self):
        return self.k.shape[1]

    @property
    def Lq(self):
        return self.q.shape[2]

    @property
    def Lkv(self):
        return self.k.shape[2]

    @property
    def d(self):
        return self.q.shape[3]


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _randn(shape, g, device, dtype=torch.float32):
    return torch.randn(*shape, generator=g, device=device, dtype=dtype)


def _fill_randn_bf16(t: torch.Tensor, g: torch.Generator, chunk_dim0: bool = True):
    """Fill a bf16 tensor with N(0,1) draws, one leading index at a time (bounds
    the fp32 temporary to one slice)."""
    for i in range(t.shape[0]):
        t[i].copy_(torch.randn(*t.shape[1:], generator=g, device=t.device, dtype=torch.float32))
    return t


def _sink_direction(q: torch.Tensor, Hkv: int) -> torch.Tensor:
    """unit(mean of every query vector that reads each KV head), per batch element.

    q: [B, Hq, Lq, d] -> [B, Hkv, d] (fp32)."""
    B, Hq, Lq, d = q.shape
    G = Hq // Hkv
    out = torch.empty(B, Hkv, d, device=q.device, dtype=torch.float32)
    for b in range(B):
        for h in range(Hkv):
            mu = q[b, h * G:(h + 1) * G].float().reshape(-1, d).mean(dim=0)
            out[b, h] = mu / mu.norm().clamp_min(1e-30)
    return out


def tiny(seed: int = 0, planted: bool = False, device="cpu", fp32: bool = False) -> Attn:
    """B=1, H=2, L=512, d=64 non-causal; logits multiplied by 3.

    With ``fp32=True`` the fp32 draws are returned (the fp32 copy); otherwise the
    bf16 copy (the fp32 draws rounded to bf16)."""
    g = _gen(seed, device)
    B, H, L, d = 1, 2, 512, 64
    q = _randn((B, H, L, d), g, device)
    k = _randn((B, H, L, d), g, device)
    v = _randn((B, H, L, d), g, device)
    if planted:
        k[:, :, 256:512, :] = -2.0 * q.mean(dim=2, keepdim=True)
    dt = torch.float32 if fp32 else torch.bfloat16
    return Attn(q.to(dt).contiguous(), k.to(dt).contiguous(), v.to(dt).contiguous(),
                causal=False, scale=3.0 / math.sqrt(d), name="tiny" + ("-planted" if planted else ""))


def llm(seed: int = 0, L: int = 16384, B: int = 1, Hq: int = 32, Hkv: int = 8, d: int = 128,
        device="cpu", causal: bool = True, sinks: int = 4) -> Attn:
    """Causal GQA prefill; iid N(0,1) with sink keys at positions 0..sinks-1."""
    g = _gen(seed, device)
    q = torch.empty(B, Hq, L, d, device=device, dtype=torch.bfloat16)
    k = torch.empty(B, Hkv, L, d, device=device, dtype=torch.bfloat16)
    v = torch.empty(B, Hkv, L, d, device=device, dtype=torch.bfloat16)
    _fill_randn_bf16(q.view(B * Hq, L, d), g)
    _fill_randn_bf16(k.view(B * Hkv, L, d), g)
    _fill_randn_bf16(v.view(B * Hkv, L, d), g)
    if sinks:
        u = _sink_direction(q, Hkv)  # [B,Hkv,d]
        k[:, :, :sinks, :] = (3.0 * u).unsqueeze(2).to(torch.bfloat16)
    return Attn(q, k, v, causal=causal, scale=2.0 / math.sqrt(d), name=f"llm-L{L}")


def decode(seed: int = 0, B: int = 64, Hq: int = 32, Hkv: int = 8, Lkv: int = 32768, d: int = 128,
           device="cpu", sinks: int = 4) -> Attn:
    """Split-KV decode problem: one query token per sequence (q is [B,Hq,1,d])."""
    g = _gen(seed, device)
    q = torch.empty(B, Hq, 1, d, device=device, dtype=torch.bfloat16)
    k = torch.empty(B, Hkv, Lkv, d, device=device, dtype=torch.bfloat16)
    v = torch.empty(B, Hkv, Lkv, d, device=device, dtype=torch.bfloat16)
    q.copy_(_randn((B, Hq, 1, d), g, device))
    _fill_randn_bf16(k.view(B * Hkv, Lkv, d), g)
    _fill_randn_bf16(v.view(B * Hkv, Lkv, d), g)
    if sinks:
        u = _sink_direction(q, Hkv)
        k[:, :, :sinks, :] = (3.0 * u).unsqueeze(2).to(torch.bfloat16)
    return Attn(q, k, v, causal=False, scale=2.0 / math.sqrt(d), name=f"decode-B{B}-L{Lkv}")


DIT_GRID = (21, 30, 52)
DIT_NBHD = (4, 6, 8)


def dit(seed: int = 0, H: int = 40, grid=DIT_GRID, nbhd=DIT_NBHD, d: int = 128, device="cpu",
        strength: float = 1.5) -> Attn:
    """Video-DiT self-attention over a t x h x w latent grid (t-major, w fastest).

    Each token's Q and K are N(0,1) plus ``strength`` times a vector shared by all
    tokens of its neighbourhood (the same vectors for Q and K); V is iid N(0,1)."""
    g = _gen(seed, device)
    T, Hh, W = grid
    nt, nh, nw = nbhd
    L = T * Hh * W
    tt = torch.arange(T, device=device).view(T, 1, 1) // nt
    hh = torch.arange(Hh, device=device).view(1, Hh, 1) // nh
    ww = torch.arange(W, device=device).view(1, 1, W) // nw
    NH, NW = -(-Hh // nh), -(-W // nw)
    nb_index = ((tt * NH + hh) * NW + ww).reshape(L)  # neighbourhood id of each token
    n_nb = int(nb_index.max().item()) + 1
    q = torch.empty(1, H, L, d, device=device, dtype=torch.bfloat16)
    k = torch.empty(1, H, L, d, device=device, dtype=torch.bfloat16)
    v = torch.empty(1, H, L, d, device=device, dtype=torch.bfloat16)
    for h in range(H):
        shared = _randn((n_nb, d), g, device)[nb_index]  # [L, d]
        q[0, h].copy_(_randn((L, d), g, device) + strength * shared)
        k[0, h].copy_(_randn((L, d), g, device) + strength * shared)
        v[0, h].copy_(_randn((L, d), g, device))
    return Attn(q, k, v, causal=False, scale=1.0 / math.sqrt(d), name=f"dit-H{H}-L{L}",
                extra={"grid": grid, "nbhd": nbhd})


def planted70(seed: int = 0, L: int = 16384, B: int = 1, Hq: int = 32, Hkv: int = 8, d: int = 128,
              device="cpu", frac: float = 0.7) -> Attn:
    """Non-causal GQA prefill whose last ``frac`` of key tiles hold K = 0."""
    a = llm(seed=seed, L=L, B=B, Hq=Hq, Hkv=Hkv, d=d, device=device, causal=False, sinks=0)
    nT = -(-L // TILE)
    first = nT - int(round(frac * nT))
    a.k[:, :, first * TILE:, :] = 0
    a.name = f"planted70-L{L}"
    a.extra["first_zero_tile"] = first
    return a


def small_random(seed: int, B: int, Hq: int, Hkv: int, Lq: int, Lkv: int, d: int, causal: bool,
                 scale: float | None = None, device="cpu", logit_mult: float = 1.0) -> Attn:
    """Generic iid N(0,1) problem of any shape (edge-case and ragged-size tests)."""
    g = _gen(seed, device)
    q = _randn((B, Hq, Lq, d), g, device).to(torch.bfloat16)
    k = _randn((B, Hkv, Lkv, d), g, device).to(torch.bfloat16)
    v = _randn((B, Hkv, Lkv, d), g, device).to(torch.bfloat16)
    if scale is None:
        scale = logit_mult / math.sqrt(d)
    return Attn(q, k, v, causal=causal, scale=scale, name=f"rand-{B}x{Hq}/{Hkv}x{Lq}x{Lkv}x{d}")


def paged_decode(seed: int = 0, B: int = 8, Hq: int = 32, Hkv: int = 8, max_len: int = 4096, d: int = 128,
                 page_size: int = 16, token_major: bool = True, lens=None, min_len: int = 1, spare_pages: int = 7,
                 device="cpu", sinks: int = 4) -> Attn:
    """``decode(seed, B, Hq, Hkv, max_len)`` plus a paged copy of its K and V.

    extra: k_pages/v_pages [P, page_size, Hkv, d] (token_major) or [P, Hkv,
    page_size, d]; page_table int32 [B, ceil(max_len/page_size)] (-1 past each
    sequence's last page); seq_lens int32 [B]; page_size; token_major.  The
    contiguous q/k/v stay in the object: key i of sequence b is k[b, :, i] for
    i < seq_lens[b] (what the oracle reads)."""
    a = decode(seed, B, Hq, Hkv, max_len, d, device, sinks)
    g = torch.Generator(device="cpu")
    g.manual_seed(seed * 7919 + 11)
    if lens is None:
        lens = torch.randint(min_len, max_len + 1, (B,), generator=g)
    lens = torch.as_tensor(lens, dtype=torch.int64).cpu()
    npg_max = -(-max_len // page_size)
    npg = (lens + page_size - 1) // page_size  # pages used by each sequence
    used = int(npg.sum().item())
    P = used + spare_pages
    perm = torch.randperm(P, generator=g)  # pool slot of each used page, in (b, page) order
    table = torch.full((B, npg_max), -1, dtype=torch.int32)
    valid = torch.arange(npg_max).unsqueeze(0) < npg.unsqueeze(1)  # [B, npg_max]
    table[valid] = perm[:used].to(torch.int32)
    # pages of the contiguous cache: [B, npg_max, page_size, Hkv, d] (token-major view)
    pad = npg_max * page_size - max_len
    def pages_of(x):
        x = x.permute(0, 2, 1, 3)  # [B, L, Hkv, d]
        if pad:
            x = torch.cat([x, torch.zeros(B, pad, Hkv, d, dtype=x.dtype, device=x.device)], dim=1)
        x = x.reshape(B, npg_max, page_size, Hkv, d)
        return x if token_major else x.permute(0, 1, 3, 2, 4)
    shape = (P, page_size, Hkv, d) if token_major else (P, Hkv, page_size, d)
    gd = _gen(seed + 101, device)
    out = {}
    sel = valid.to(device)
    dst = table[valid].to(torch.int64).to(device)
    for name, x in (("k_pages", a.k), ("v_pages", a.v)):
        pool = torch.empty(shape, dtype=torch.bfloat16, device=device)
        _fill_randn_bf16(pool.view(P, -1), gd)
        src = pages_of(x)[sel]  # [used, ...] in (b, page) order
        pool[dst] = src.contiguous()
        out[name] = pool
    a.extra.update(out)
    a.extra.update(page_table=table.to(device), seq_lens=lens.to(torch.int32).to(device), page_size=page_size,
                   token_major=token_major, max_len=max_len)
    a.name = f"paged-decode-B{B}-L{max_len}-ps{page_size}-{'nhd' if token_major else 'hnd'}"
    return a


def mla_decode(seed: int = 0, B: int = 64, Hq: int = 16, L: int = 32768, dk: int = 576, dv: int = 512,
               device="cpu", sinks: int = 4, lens=None, min_len: int = 1, page_size: int = 0,
               spare_pages: int = 7, q_shared: float = 0.0, sink_norm: float = 0.0) -> Attn:
    """MLA decode in absorbed form: q [B,Hq,1,dk]; one latent cache kv [B,L,dk]
    whose rows are the keys of every head and whose first dv columns are the
    values.  The decode recipe applied to the latent rows: q and kv N(0,1), scores
    scaled by 2/sqrt(dk), and the first ``sinks`` rows of each sequence sink keys
    along unit(mean of its queries), here with an ordinary row's norm sqrt(dk) (one
    decision covers all Hq heads, so the weaker 3 * unit(...) sinks of the GQA recipe
    would leave every tile computed).  With q_shared > 0 every query also gets
    q_shared * u for one random unit vector u per sequence and the sinks point along
    u with norm sink_norm (default sqrt(dk)): many heads then share strong sinks, as
    the 64- and 128-head cases need for any tile to be skipped by all heads.

    extra: kv, dv, seq_lens (int32 [B], or None when ``lens`` is None and no pages
    are asked for); with page_size > 0 also kv_pages [P, page_size, dk] and
    page_table int32 [B, ceil(L/page_size)] (-1 past each sequence's last page),
    the contiguous cache staying in ``kv`` (what the oracle reads).  k/v of the
    returned object are views of the cache ([B,1,L,dk] and [B,1,L,dv])."""
    g = _gen(seed, device)
    q = torch.empty(B, Hq, 1, dk, device=device, dtype=torch.bfloat16)
    kv = torch.empty(B, L, dk, device=device, dtype=torch.bfloat16)
    q.copy_(_randn((B, Hq, 1, dk), g, device))
    _fill_randn_bf16(kv, g)
    norm = sink_norm if sink_norm > 0 else math.sqrt(dk)
    if q_shared > 0:
        u = _randn((B, 1, dk), g, device)
        u = u / u.norm(dim=-1, keepdim=True)
        q.copy_((q.float() + q_shared * u.unsqueeze(2)).to(torch.bfloat16))
    if sinks:
        if q_shared <= 0:
            u = _sink_direction(q, 1)  # [B, 1, dk]
        kv[:, :sinks, :] = (norm * u).to(torch.bfloat16)
    extra = {"kv": kv, "dv": dv, "seq_lens": None}
    gl = torch.Generator(device="cpu")
    gl.manual_seed(seed * 7919 + 13)
    if lens is not None or page_size > 0:
        if lens is None:
            lens = torch.randint(min_len, L + 1, (B,), generator=gl)
        lens = torch.as_tensor(lens, dtype=torch.int64).cpu()
        extra["seq_lens"] = lens.to(torch.int32).to(device)
    if page_size > 0:
        npg_max = -(-L // page_size)
        npg = (lens + page_size - 1) // page_size
        used = int(npg.sum().item())
        P = used + spare_pages
        perm = torch.randperm(P, generator=gl)
        table = torch.full((B, npg_max), -1, dtype=torch.int32)
        valid = torch.arange(npg_max).unsqueeze(0) < npg.unsqueeze(1)
        table[valid] = perm[:used].to(torch.int32)
        pad = npg_max * page_size - L
        x = kv if not pad else torch.cat([kv, torch.zeros(B, pad, dk, dtype=kv.dtype, device=device)], dim=1)
        pool = torch.empty(P, page_size, dk, dtype=torch.bfloat16, device=device)
        _fill_randn_bf16(pool, _gen(seed + 103, device))
        pool[table[valid].to(torch.int64).to(device)] = x.reshape(B, npg_max, page_size, dk)[valid.to(device)]
        extra.update(kv_pages=pool, page_table=table.to(device), page_size=page_size)
    return Attn(q, kv.unsqueeze(1), kv[:, :, :dv].unsqueeze(1), causal=False, scale=2.0 / math.sqrt(dk),
                name=f"mla-decode-B{B}-H{Hq}-L{L}" + (f"-ps{page_size}" if page_size else ""), extra=extra)


def l2_flush_buffer(device, nbytes: int = 512 << 20) -> torch.Tensor:
    """A buffer larger than the 126 MB L2, written between timed iterations."""
    return torch.empty(nbytes // 4, dtype=torch.float32, device=device)
