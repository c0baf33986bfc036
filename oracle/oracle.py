"""Python front end of the CPU oracle (ctypes over oracle/_build/liboracle.so).

TEST INFRASTRUCTURE ONLY: imported by the tests, the smoke check and the CPU
baseline of the benchmark, never by the CUDA product path.

Inputs may be numpy arrays or CPU torch tensors of any float dtype; they are
widened to the oracle's precision ("f32" -- the fp32 oracle the parity tests
use -- or "f64" for self-checks).  bf16 values widen exactly.
"""
from __future__ import annotations

import ctypes
import math
import os

import numpy as np

from . import build as _build

_lib = None


def _load():
    global _lib
    if _lib is None:
        _lib = _configure(ctypes.CDLL(_build.build()))
    return _lib


def _configure(lib):
    """Declare the C signatures on a loaded oracle library."""
    for suf, ct in (("_f32", ctypes.c_float), ("_f64", ctypes.c_double)):
        P = ctypes.POINTER(ct)
        f = getattr(lib, "oracle_dense" + suf)
        f.restype = ctypes.c_int
        f.argtypes = [P, P, P, P, P] + [ctypes.c_int] * 7 + [ctypes.c_double, ctypes.c_int]
        f = getattr(lib, "oracle_prefill_tiled" + suf)
        f.restype = ctypes.c_longlong
        f.argtypes = ([P, P, P, P, P] + [ctypes.c_int] * 7 + [ctypes.c_double, ctypes.c_double,
                      ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_int,
                      ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int])
        f = getattr(lib, "oracle_decode_tiled" + suf)
        f.restype = ctypes.c_longlong
        f.argtypes = ([P, P, P, P, P] + [ctypes.c_int] * 5 + [ctypes.c_double, ctypes.c_double,
                      ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_int,
                      ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                      ctypes.c_void_p, ctypes.c_int])
        f = getattr(lib, "oracle_mla_decode_tiled" + suf)
        f.restype = ctypes.c_longlong
        f.argtypes = ([P, P, ctypes.c_void_p, P, P] + [ctypes.c_int] * 5 +
                      [ctypes.c_double, ctypes.c_double, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                       ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                       ctypes.c_void_p, ctypes.c_void_p])
    return lib


def _np(x, dt):
    try:
        import torch

        if isinstance(x, torch.Tensor):
            x = x.detach().to("cpu", torch.float64 if dt == np.float64 else torch.float32).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(x, dtype=dt))


def _ptr(a, ct):
    return a.ctypes.data_as(ctypes.POINTER(ct))


def _vp(a):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _types(precision):
    if precision == "f32":
        return np.float32, ctypes.c_float, "_f32"
    if precision == "f64":
        return np.float64, ctypes.c_double, "_f64"
    raise ValueError(precision)


def dense(q, k, v, causal: bool, scale: float, precision: str = "f32", window: int = 0):
    """softmax(scale*QK^T + mask) V and lse for q [B,Hq,Lq,d], k/v [B,Hkv,Lkv,d].
    window > 0 (with causal): only the last `window` keys up to the row's position."""
    dt, ct, suf = _types(precision)
    q, k, v = _np(q, dt), _np(k, dt), _np(v, dt)
    B, Hq, Lq, d = q.shape
    _, Hkv, Lkv, _ = k.shape
    o = np.zeros_like(q)
    lse = np.zeros((B, Hq, Lq), dt)
    rc = getattr(_load(), "oracle_dense" + suf)(
        _ptr(q, ct), _ptr(k, ct), _ptr(v, ct), _ptr(o, ct), _ptr(lse, ct),
        B, Hq, Hkv, Lq, Lkv, d, int(causal), float(scale), int(window))
    if rc != 0:
        raise ValueError("oracle_dense: bad arguments")
    return o, lse


def prefill_tiled(q, k, v, causal: bool, scale: float, lam: float, Br: int = 128, Bc: int = 128,
                  units=None, forced=None, precision: str = "f32", out=None, window: int = 0):
    """Tiled skip-softmax pass for prefill.

    window: > 0 (with causal) keeps only the last `window` keys up to each row.

    units:  optional iterable of (b, h, qtile); only those query tiles are run
    forced: optional uint8 map [B,Hq,nQ,nK] (1 = skip) replacing the test
    Returns dict(o, lse, map, margin, skipped); rows/tiles of units not run stay
    at o=0, lse=nan, map=255, margin=nan.
    """
    dt, ct, suf = _types(precision)
    q, k, v = _np(q, dt), _np(k, dt), _np(v, dt)
    B, Hq, Lq, d = q.shape
    _, Hkv, Lkv, _ = k.shape
    nQ, nK = -(-Lq // Br), -(-Lkv // Bc)
    o = np.zeros_like(q)
    lse = np.full((B, Hq, Lq), np.nan, dt)
    m = np.full((B, Hq, nQ, nK), 255, np.uint8)
    g = np.full((B, Hq, nQ, nK), np.nan, dt)
    u = None
    nu = 0
    if units is not None:
        u = np.ascontiguousarray(np.asarray(list(units), dtype=np.int32).reshape(-1, 3))
        nu = u.shape[0]
    f = None
    if forced is not None:
        f = np.ascontiguousarray(np.asarray(forced, dtype=np.uint8).reshape(B, Hq, nQ, nK))
    sk = getattr(_load(), "oracle_prefill_tiled" + suf)(
        _ptr(q, ct), _ptr(k, ct), _ptr(v, ct), _ptr(o, ct), _ptr(lse, ct),
        B, Hq, Hkv, Lq, Lkv, d, int(causal), float(scale), float(lam), Br, Bc,
        _vp(u), nu, _vp(f), _vp(m), _vp(g), int(window))
    if sk < 0:
        raise ValueError("oracle_prefill_tiled: bad arguments")
    return {"o": o, "lse": lse, "map": m, "margin": g, "skipped": int(sk)}


def decode_tiled(q, k, v, scale: float, lam: float, num_splits: int = 1, Bc: int = 128,
                 units=None, forced=None, precision: str = "f32", window: int = 0):
    """Tiled skip-softmax pass for decode (one query token; G heads per KV head).

    q [B,Hq,d] (or [B,Hq,1,d]), k/v [B,Hkv,Lkv,d].
    window > 0: only the last `window` keys; the splits cover the visited tiles.
    units: optional iterable of (b, hkv); forced: optional uint8 [B,Hkv,nK].
    Returns dict(o [B,Hq,d], lse [B,Hq], map, margin, skipped, o_part, lse_part).
    """
    dt, ct, suf = _types(precision)
    q = _np(q, dt)
    if q.ndim == 4:
        q = np.ascontiguousarray(q[:, :, 0, :])
    k, v = _np(k, dt), _np(v, dt)
    B, Hq, d = q.shape
    _, Hkv, Lkv, _ = k.shape
    nK = -(-Lkv // Bc)
    S = int(num_splits)
    o = np.zeros((B, Hq, d), dt)
    lse = np.full((B, Hq), np.nan, dt)
    m = np.full((B, Hkv, nK), 255, np.uint8)
    g = np.full((B, Hkv, nK), np.nan, dt)
    op = np.zeros((S, B, Hq, d), dt)
    lp = np.full((S, B, Hq), np.nan, dt)
    u = None
    nu = 0
    if units is not None:
        u = np.ascontiguousarray(np.asarray(list(units), dtype=np.int32).reshape(-1, 2))
        nu = u.shape[0]
    f = None
    if forced is not None:
        f = np.ascontiguousarray(np.asarray(forced, dtype=np.uint8).reshape(B, Hkv, nK))
    sk = getattr(_load(), "oracle_decode_tiled" + suf)(
        _ptr(q, ct), _ptr(k, ct), _ptr(v, ct), _ptr(o, ct), _ptr(lse, ct),
        B, Hq, Hkv, Lkv, d, float(scale), float(lam), Bc, S, _vp(u), nu, _vp(f), _vp(m), _vp(g),
        _vp(op), _vp(lp), int(window))
    if sk < 0:
        raise ValueError("oracle_decode_tiled: bad arguments")
    return {"o": o, "lse": lse, "map": m, "margin": g, "skipped": int(sk), "o_part": op,
            "lse_part": lp}


def mla_decode_tiled(q, kv, dv: int, scale: float, lam: float, num_splits: int = 1, seq_lens=None,
                     Bc: int = 128, units=None, forced=None, precision: str = "f32"):
    """Tiled skip-softmax pass for MLA decode in its absorbed form.

    q [B,Hq,dk]; kv [B,Lmax,dk], one latent row per cached token shared by every
    query head; the value of a token is the first `dv` entries of its row.  One
    decision covers all Hq heads x Bc keys.  seq_lens: optional [B] key counts.
    units: optional iterable of batch indices; forced: optional uint8 [B,nK].
    Returns dict(o [B,Hq,dv], lse [B,Hq], map [B,nK], margin [B,nK], skipped,
    o_part [S,B,Hq,dv], lse_part [S,B,Hq]).
    """
    dt, ct, suf = _types(precision)
    q = _np(q, dt)
    if q.ndim == 4:
        q = np.ascontiguousarray(q[:, :, 0, :])
    kv = _np(kv, dt)
    B, Hq, dk = q.shape
    Lmax = kv.shape[1]
    if kv.shape != (B, Lmax, dk):
        raise ValueError("kv must be [B, Lmax, dk]")
    nK = -(-Lmax // Bc)
    S = int(num_splits)
    o = np.zeros((B, Hq, dv), dt)
    lse = np.full((B, Hq), np.nan, dt)
    m = np.full((B, nK), 255, np.uint8)
    g = np.full((B, nK), np.nan, dt)
    op = np.zeros((S, B, Hq, dv), dt)
    lp = np.full((S, B, Hq), np.nan, dt)
    sl = None
    if seq_lens is not None:
        sl = np.ascontiguousarray(np.asarray(seq_lens, dtype=np.int32).reshape(B))
    u = None
    nu = 0
    if units is not None:
        u = np.ascontiguousarray(np.asarray(list(units), dtype=np.int32).reshape(-1))
        nu = u.shape[0]
    f = None
    if forced is not None:
        f = np.ascontiguousarray(np.asarray(forced, dtype=np.uint8).reshape(B, nK))
    sk = getattr(_load(), "oracle_mla_decode_tiled" + suf)(
        _ptr(q, ct), _ptr(kv, ct), _vp(sl), _ptr(o, ct), _ptr(lse, ct),
        B, Hq, Lmax, dk, int(dv), float(scale), float(lam), Bc, S, _vp(u), nu, _vp(f), _vp(m), _vp(g),
        _vp(op), _vp(lp))
    if sk < 0:
        raise ValueError("oracle_mla_decode_tiled: bad arguments")
    return {"o": o, "lse": lse, "map": m, "margin": g, "skipped": int(sk), "o_part": op,
            "lse_part": lp}


def sparsity_from_margins(margin, lam: float) -> float:
    """Fraction of visited tiles that a threshold lambda skips, read off the
    lambda-independent margins (tile skipped iff margin < ln lambda)."""
    g = np.asarray(margin, dtype=np.float64)
    g = g[~np.isnan(g)]  # tiles that were not visited carry NaN
    if g.size == 0:
        return 0.0
    ln = -math.inf if lam <= 0 else math.log(lam)
    return float(np.count_nonzero(g < ln)) / g.size


def num_threads() -> int:
    """Threads the OpenMP runtime of the oracle will use."""
    n = os.environ.get("OMP_NUM_THREADS")
    if n:
        return int(n)
    return os.cpu_count() or 1
