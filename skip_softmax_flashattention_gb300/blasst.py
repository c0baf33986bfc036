"""Python binding of the C ABI in include/blasst.h (ctypes; argument marshalling only).

The functions named ``blasst_*`` mirror the C entry points one to one and take
device pointers as ints or torch tensors.  ``prefill`` and ``decode`` are small
conveniences that allocate the outputs with torch and raise ``BlasstError`` on a
non-zero status.  Every step of the computation runs in the CUDA library; if the
library cannot be built or loaded, the import of the functions fails loudly.
"""
from __future__ import annotations

import ctypes
import math
import os

from . import build as _build

TILE = 128

BLASST_OK = 0
BLASST_WARN_LAMBDA_GE_1 = 1
BLASST_ERR_INVALID_ARG = -1
BLASST_ERR_UNSUPPORTED = -2
BLASST_ERR_WORKSPACE_TOO_SMALL = -3
BLASST_ERR_CUDA = -4
BLASST_ERR_TIMEOUT = -5
BLASST_ERR_NO_CALIBRATION = -6
BLASST_ERR_SCRATCH_LIMIT = -7
BLASST_ERR_PAGE_TABLE = -8

BLASST_PREFILL_ELIDE_V = 0x1
BLASST_PREFILL_P_VIA_SMEM = 0x2
BLASST_PREFILL_ONE_QTILE = 0x4
BLASST_PREFILL_WIDE = 0x8
BLASST_FLAG_TEST_SHORT_WATCHDOG = 0x80000000

_lib = None


class BlasstError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {blasst_status_string(status)} ({status})")


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True):
    """Load libblasst.so (building it first when it is missing or stale)."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.build() if build_if_missing else _build.LIB
    if not os.path.exists(path):
        raise ImportError(f"CUDA library not found at {path}")
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    I = ctypes.c_int
    F = ctypes.c_float
    lib.blasst_prefill.restype = I
    lib.blasst_prefill.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, F, F, P, P]
    lib.blasst_prefill_ex.restype = I
    lib.blasst_prefill_ex.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, F, F, P, P, P, ctypes.c_uint, P]
    lib.blasst_decode_num_splits.restype = I
    lib.blasst_decode_num_splits.argtypes = [I, I, I, I, I, I, ctypes.POINTER(I)]
    lib.blasst_decode_workspace_size.restype = ctypes.c_size_t
    lib.blasst_decode_workspace_size.argtypes = [I, I, I, I, I, I]
    lib.blasst_decode.restype = I
    lib.blasst_decode.argtypes = [P, P, P, P, P, I, I, I, I, I, F, F, I, P, ctypes.c_size_t, P, P, P, P]
    lib.blasst_decode_paged.restype = I
    lib.blasst_decode_paged.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, I, I, I, I, I, F, F, I, P,
                                        ctypes.c_size_t, P, P, P, P]
    lib.blasst_prefill_window.restype = I
    lib.blasst_prefill_window.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, F, F, P, P, P, ctypes.c_uint, P]
    lib.blasst_decode_noalloc.restype = I
    lib.blasst_decode_noalloc.argtypes = [P, P, P, P, P, I, I, I, I, I, F, F, I, P, P, P, P]
    lib.blasst_decode_noalloc_scratch_bytes.restype = ctypes.c_size_t
    lib.blasst_decode_noalloc_scratch_bytes.argtypes = []
    lib.blasst_mla_decode.restype = I
    lib.blasst_mla_decode.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, I, I, F, F, I, P, ctypes.c_size_t,
                                      P, P, P, P]
    lib.blasst_mla_decode_num_splits.restype = I
    lib.blasst_mla_decode_num_splits.argtypes = [I, I, I, I, ctypes.POINTER(I)]
    lib.blasst_mla_decode_workspace_size.restype = ctypes.c_size_t
    lib.blasst_mla_decode_workspace_size.argtypes = [I, I, I, I]
    lib.blasst_lambda.restype = I
    lib.blasst_lambda.argtypes = [I, ctypes.c_double, ctypes.c_double, ctypes.c_double, ctypes.c_double,
                                  ctypes.c_longlong, ctypes.POINTER(ctypes.c_double)]
    lib.blasst_device_status.restype = I
    lib.blasst_device_status.argtypes = [I]
    lib.blasst_status_string.restype = ctypes.c_char_p
    lib.blasst_status_string.argtypes = [I]
    _lib = lib
    return lib


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()  # torch tensor


def _stream(stream):
    if stream is None:
        import torch

        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


# ------------------------------------------------------------------ raw ABI
def blasst_prefill(q, k, v, o, lse, B, Hq, Hkv, Lq, Lkv, d, causal, scale, lambda_, skipped_tiles_out=None,
                   stream=None) -> int:
    return load().blasst_prefill(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, Lq, Lkv, d,
                                 int(causal), float(scale), float(lambda_), _ptr(skipped_tiles_out),
                                 _stream(stream))


def blasst_prefill_ex(q, k, v, o, lse, B, Hq, Hkv, Lq, Lkv, d, causal, scale, lambda_, skipped_tiles_out=None,
                      skip_map=None, margins=None, flags=0, stream=None) -> int:
    return load().blasst_prefill_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, Lq, Lkv, d,
                                    int(causal), float(scale), float(lambda_), _ptr(skipped_tiles_out),
                                    _ptr(skip_map), _ptr(margins), int(flags), _stream(stream))


def blasst_decode_num_splits(B, Hq, Hkv, Lkv, d, requested=0) -> tuple:
    out = ctypes.c_int(0)
    rc = load().blasst_decode_num_splits(B, Hq, Hkv, Lkv, d, requested, ctypes.byref(out))
    return rc, out.value


def blasst_decode_workspace_size(B, Hq, Hkv, Lkv, d, num_splits) -> int:
    return int(load().blasst_decode_workspace_size(B, Hq, Hkv, Lkv, d, num_splits))


def blasst_decode(q, k_cache, v_cache, o, lse, B, Hq, Hkv, Lkv, d, scale, lambda_, num_splits, workspace,
                  workspace_bytes, skipped_tiles_out=None, skip_map=None, margins=None, stream=None) -> int:
    return load().blasst_decode(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(o), _ptr(lse), B, Hq, Hkv, Lkv, d,
                                float(scale), float(lambda_), int(num_splits), _ptr(workspace),
                                int(workspace_bytes), _ptr(skipped_tiles_out), _ptr(skip_map), _ptr(margins),
                                _stream(stream))


def blasst_prefill_window(q, k, v, o, lse, B, Hq, Hkv, Lq, Lkv, d, window, scale, lambda_, skipped_tiles_out=None,
                          skip_map=None, margins=None, flags=0, stream=None) -> int:
    return load().blasst_prefill_window(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, Lq, Lkv, d,
                                        int(window), float(scale), float(lambda_), _ptr(skipped_tiles_out),
                                        _ptr(skip_map), _ptr(margins), int(flags), _stream(stream))


def blasst_decode_paged(q, k_pages, v_pages, page_table, seq_lens, o, lse, B, Hq, Hkv, max_kv_len, window, d,
                        num_pages, page_size, max_pages_per_seq, token_major, scale, lambda_, num_splits, workspace,
                        workspace_bytes, skipped_tiles_out=None, skip_map=None, margins=None, stream=None) -> int:
    return load().blasst_decode_paged(_ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(page_table), _ptr(seq_lens),
                                      _ptr(o), _ptr(lse), B, Hq, Hkv, max_kv_len, int(window), d, num_pages, page_size,
                                      max_pages_per_seq, int(token_major), float(scale), float(lambda_),
                                      int(num_splits), _ptr(workspace), int(workspace_bytes),
                                      _ptr(skipped_tiles_out), _ptr(skip_map), _ptr(margins), _stream(stream))


def blasst_decode_noalloc(q, k_cache, v_cache, o, lse, B, Hq, Hkv, Lkv, d, scale, lambda_, num_splits,
                          skipped_tiles_out=None, skip_map=None, margins=None, stream=None) -> int:
    """blasst_decode for callers that cannot allocate: the per-split partials live in
    the library's static device scratch (shared by every call on the device)."""
    return load().blasst_decode_noalloc(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(o), _ptr(lse), B, Hq, Hkv,
                                        Lkv, d, float(scale), float(lambda_), int(num_splits),
                                        _ptr(skipped_tiles_out), _ptr(skip_map), _ptr(margins), _stream(stream))


def blasst_decode_noalloc_scratch_bytes() -> int:
    return int(load().blasst_decode_noalloc_scratch_bytes())


def blasst_mla_decode(q, kv, page_table, seq_lens, o, lse, B, Hq, max_kv_len, dk, dv, num_pages, page_size,
                      max_pages_per_seq, scale, lambda_, num_splits, workspace, workspace_bytes,
                      skipped_tiles_out=None, skip_map=None, margins=None, stream=None) -> int:
    return load().blasst_mla_decode(_ptr(q), _ptr(kv), _ptr(page_table), _ptr(seq_lens), _ptr(o), _ptr(lse), B, Hq,
                                    max_kv_len, dk, dv, num_pages, page_size, max_pages_per_seq, float(scale),
                                    float(lambda_), int(num_splits), _ptr(workspace), int(workspace_bytes),
                                    _ptr(skipped_tiles_out), _ptr(skip_map), _ptr(margins), _stream(stream))


def blasst_mla_decode_num_splits(B, Hq, max_kv_len, requested=0) -> tuple:
    out = ctypes.c_int(0)
    rc = load().blasst_mla_decode_num_splits(B, Hq, max_kv_len, requested, ctypes.byref(out))
    return rc, out.value


def blasst_mla_decode_workspace_size(B, Hq, max_kv_len, num_splits) -> int:
    return int(load().blasst_mla_decode_workspace_size(B, Hq, max_kv_len, num_splits))


def blasst_lambda(mode, threshold=0.0, a=math.nan, b=math.nan, target_sparsity=0.0, Lkv=1) -> tuple:
    out = ctypes.c_double(math.nan)
    rc = load().blasst_lambda(int(mode), float(threshold), float(a), float(b), float(target_sparsity), int(Lkv),
                              ctypes.byref(out))
    return rc, out.value


def blasst_device_status(clear: int = 1) -> int:
    return load().blasst_device_status(int(clear))


def blasst_status_string(status: int) -> str:
    return load().blasst_status_string(int(status)).decode()


# ------------------------------------------------------------------ conveniences
def _check(rc, what):
    if rc < 0:
        raise BlasstError(rc, what)
    return rc


def prefill(q, k, v, causal: bool, scale: float, lam: float, *, want_map=False, want_margins=False,
            flags=0, out=None, stream=None, window=0):
    """Run blasst_prefill_ex (blasst_prefill_window when window > 0, causal implied) on
    torch tensors; returns dict(o, lse, skipped, map, margins)."""
    import torch

    B, Hq, Lq, d = q.shape
    Hkv, Lkv = k.shape[1], k.shape[2]
    nQ, nK = -(-Lq // TILE), -(-Lkv // TILE)
    dev = q.device
    o = out if out is not None else torch.empty_like(q)
    lse = torch.empty(B, Hq, Lq, device=dev, dtype=torch.float32)
    skipped = torch.zeros(1, device=dev, dtype=torch.int64)
    mp = torch.empty(B, Hq, nQ, nK, device=dev, dtype=torch.uint8) if want_map else None
    mg = torch.empty(B, Hq, nQ, nK, device=dev, dtype=torch.float32) if want_margins else None
    if window > 0:
        rc = blasst_prefill_window(q, k, v, o, lse, B, Hq, Hkv, Lq, Lkv, d, window, scale, lam, skipped, mp, mg,
                                   flags, stream)
        _check(rc, "blasst_prefill_window")
    else:
        rc = blasst_prefill_ex(q, k, v, o, lse, B, Hq, Hkv, Lq, Lkv, d, causal, scale, lam, skipped, mp, mg, flags,
                               stream)
        _check(rc, "blasst_prefill_ex")
    return {"o": o, "lse": lse, "skipped": skipped, "map": mp, "margins": mg}


def decode(q, k, v, scale: float, lam: float, num_splits: int = 0, *, want_map=False, want_margins=False,
           stream=None):
    """Run blasst_decode on torch tensors (q [B,Hq,d] or [B,Hq,1,d]); returns dict(o, lse, skipped, map,
    margins, num_splits)."""
    import torch

    q3 = q.reshape(q.shape[0], q.shape[1], q.shape[-1])
    B, Hq, d = q3.shape
    Hkv, Lkv = k.shape[1], k.shape[2]
    nK = -(-Lkv // TILE)
    rc, S = blasst_decode_num_splits(B, Hq, Hkv, Lkv, d, num_splits)
    _check(rc, "blasst_decode_num_splits")
    dev = q.device
    ws_bytes = blasst_decode_workspace_size(B, Hq, Hkv, Lkv, d, S)
    ws = torch.empty(max(ws_bytes, 16), device=dev, dtype=torch.uint8) if ws_bytes else None
    o = torch.empty(B, Hq, d, device=dev, dtype=q.dtype)
    lse = torch.empty(B, Hq, device=dev, dtype=torch.float32)
    skipped = torch.zeros(1, device=dev, dtype=torch.int64)
    mp = torch.empty(B, Hkv, nK, device=dev, dtype=torch.uint8) if want_map else None
    mg = torch.empty(B, Hkv, nK, device=dev, dtype=torch.float32) if want_margins else None
    rc = blasst_decode(q3, k, v, o, lse, B, Hq, Hkv, Lkv, d, scale, lam, S, ws, ws_bytes, skipped, mp, mg, stream)
    _check(rc, "blasst_decode")
    return {"o": o, "lse": lse, "skipped": skipped, "map": mp, "margins": mg, "num_splits": S}


def decode_paged(q, k_pages, v_pages, page_table, seq_lens, max_kv_len: int, page_size: int, token_major: bool,
                 scale: float, lam: float, num_splits: int = 0, *, want_map=False, want_margins=False, stream=None,
                 window: int = 0):
    """Run blasst_decode_paged on torch tensors.  k_pages/v_pages: [P, page_size, Hkv, d] (token_major)
    or [P, Hkv, page_size, d]; page_table int32 [B, max_pages]; seq_lens int32 [B] or None.
    Returns dict(o, lse, skipped, map, margins, num_splits)."""
    import torch

    q3 = q.reshape(q.shape[0], q.shape[1], q.shape[-1])
    B, Hq, d = q3.shape
    num_pages = k_pages.shape[0]
    Hkv = k_pages.shape[2] if token_major else k_pages.shape[1]
    nK = -(-max_kv_len // TILE)
    # an automatic split count is planned on the keys one sequence reads
    plan_len = min(max_kv_len, window + TILE - 1) if (window > 0 and num_splits == 0) else max_kv_len
    rc, S = blasst_decode_num_splits(B, Hq, Hkv, plan_len, d, num_splits)
    _check(rc, "blasst_decode_num_splits")
    dev = q.device
    ws_bytes = blasst_decode_workspace_size(B, Hq, Hkv, max_kv_len, d, S)
    ws = torch.empty(max(ws_bytes, 16), device=dev, dtype=torch.uint8) if ws_bytes else None
    o = torch.empty(B, Hq, d, device=dev, dtype=q.dtype)
    lse = torch.empty(B, Hq, device=dev, dtype=torch.float32)
    skipped = torch.zeros(1, device=dev, dtype=torch.int64)
    mp = torch.empty(B, Hkv, nK, device=dev, dtype=torch.uint8) if want_map else None
    mg = torch.empty(B, Hkv, nK, device=dev, dtype=torch.float32) if want_margins else None
    rc = blasst_decode_paged(q3, k_pages, v_pages, page_table, seq_lens, o, lse, B, Hq, Hkv, max_kv_len, window, d,
                             num_pages, page_size, page_table.shape[1], token_major, scale, lam, S, ws, ws_bytes,
                             skipped, mp, mg, stream)
    _check(rc, "blasst_decode_paged")
    return {"o": o, "lse": lse, "skipped": skipped, "map": mp, "margins": mg, "num_splits": S}


MLA_DK, MLA_DV = 576, 512


def mla_decode(q, kv, scale: float, lam: float, num_splits: int = 0, *, seq_lens=None, page_table=None,
               page_size: int = 0, max_kv_len: int = 0, dv: int = MLA_DV, want_map=False, want_margins=False,
               stream=None):
    """Run blasst_mla_decode on torch tensors.  q [B,Hq,576] (or [B,Hq,1,576]); kv the
    latent cache: [B, L, 576] without a page table, else a page pool [P, page_size, 576]
    with page_table int32 [B, max_pages] (max_kv_len then required).  seq_lens int32 [B]
    or None.  Returns dict(o [B,Hq,512], lse, skipped, map [B,nK], margins, num_splits)."""
    import torch

    q3 = q.reshape(q.shape[0], q.shape[1], q.shape[-1])
    B, Hq, dk = q3.shape
    if page_table is None:
        max_kv_len = kv.shape[1]
        num_pages = mpp = 0
    else:
        if max_kv_len < 1:
            raise ValueError("max_kv_len is required with a page table")
        num_pages, mpp = kv.shape[0], page_table.shape[1]
    nK = -(-max_kv_len // TILE)
    rc, S = blasst_mla_decode_num_splits(B, Hq, max_kv_len, num_splits)
    _check(rc, "blasst_mla_decode_num_splits")
    dev = q.device
    ws_bytes = blasst_mla_decode_workspace_size(B, Hq, max_kv_len, S)
    ws = torch.empty(max(ws_bytes, 16), device=dev, dtype=torch.uint8) if ws_bytes else None
    o = torch.empty(B, Hq, dv, device=dev, dtype=q.dtype)
    lse = torch.empty(B, Hq, device=dev, dtype=torch.float32)
    skipped = torch.zeros(1, device=dev, dtype=torch.int64)
    mp = torch.empty(B, nK, device=dev, dtype=torch.uint8) if want_map else None
    mg = torch.empty(B, nK, device=dev, dtype=torch.float32) if want_margins else None
    rc = blasst_mla_decode(q3, kv, page_table, seq_lens, o, lse, B, Hq, max_kv_len, dk, dv, num_pages, page_size,
                           mpp, scale, lam, S, ws, ws_bytes, skipped, mp, mg, stream)
    _check(rc, "blasst_mla_decode")
    return {"o": o, "lse": lse, "skipped": skipped, "map": mp, "margins": mg, "num_splits": S}
