"""Exact IO-aware attention on GB300: the Python binding of libfa.so.

Thin argument marshalling over the C ABI declared in ``include/fa.h``: every
step of the computation runs in the library's CUDA kernels; PyTorch only
supplies device memory and the current stream. There is no fallback: when
the library is missing or the device is not a CC 10.3 GPU, the calls raise.

The functions carry the C entry points' names:

    fa_fwd(q, k, v, causal=False, scale=None)        -> (o, lse)
    fa_bwd(q, k, v, o, lse, do, causal=False, scale=None) -> (dq, dk, dv)
    fa_bwd_workspace_bytes(B, H, N, d)
    fa_fwd_ex(q, k, v, causal=False, window=0, scale=None) -> (o, lse)
    fa_decode_splitkv(q, k, v, causal=False, window=0, scale=None, n_splits=0) -> (o, lse)
    fa_strerror(code), fa_get_last_device_status(), fa_version()

fa_fwd_ex and fa_decode_splitkv take Nq queries [B, H, Nq, d] over Nk keys
[B, H, Nk, d] (causal queries are the last Nq positions) and an optional
sliding window.

q, k, v, o, do: bfloat16 CUDA tensors [B, H, N, d], contiguous; lse: float32
[B, H, N]. ``scale`` defaults to 1/sqrt(d) as in the dense attention block of
"FlashAttention -- the same attention, made memory-aware", section 00.
"""

from __future__ import annotations

import ctypes
import math
import os

from .accounting import (flops_fwd, flops_bwd, bytes_fwd, bytes_bwd,  # noqa: F401
                         transfer_ledger)

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libfa.so")

FA_OK = 0
FA_ERR_INVALID = -1
FA_ERR_UNSUPPORTED = -2
FA_ERR_LAUNCH = -3
FA_ERR_TIMEOUT = -4
FA_ERR_WORKSPACE = -5

# Every symbol include/fa.h declares, with (restype, argtypes).
_P = ctypes.c_void_p
_I = ctypes.c_int
_F = ctypes.c_float
_S = ctypes.c_size_t
_U64 = ctypes.c_ulonglong
SIGNATURES = {
    "fa_fwd": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F]),
    "fa_fwd_stream": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _P]),
    "fa_bwd": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F]),
    "fa_bwd_stream": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _P, _S, _P]),
    "fa_bwd_preprocess_stream": (_I, [_P, _P, _P, _I, _I, _I, _I, _P, _S, _P]),
    "fa_bwd_main_stream": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _P, _S, _P]),
    "fa_bwd_finish_stream": (_I, [_P, _I, _I, _I, _I, _P, _S, _P]),
    "fa_bwd_noalloc": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _P]),
    "fa_bwd_workspace_bytes": (_S, [_I, _I, _I, _I]),
    "fa_bwd_ex": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _P, _S, _P]),
    "fa_fwd_ex": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _F, _P]),
    "fa_decode_splitkv": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _F, _I, _P, _S, _P]),
    "fa_decode_num_splits": (_I, [_I, _I, _I, _I, _I]),
    "fa_decode_workspace_bytes": (_S, [_I, _I, _I, _I, _I, _I]),
    "fa_fwd_dropout": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _F, _U64, _U64, _P]),
    "fa_bwd_dropout": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _F, _U64, _U64,
                            _P, _S, _P]),
    "fa_strerror": (ctypes.c_char_p, [_I]),
    "fa_get_last_device_status": (_I, []),
    "fa_version": (_I, []),
}


class FAError(RuntimeError):
    """A libfa call returned a non-zero code."""

    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {fa_strerror(code)} (code {code})")


_lib = None


def load_library(path: str | None = None) -> ctypes.CDLL:
    """Load libfa.so (once) and declare its signatures. Raises if missing."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise ImportError(
            f"libfa.so is not built ({p}); run `python -m exact_io_aware_33_gb300.build` "
            "or __graft_entry__.build() first")
    lib = ctypes.CDLL(p)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if path is None:
        _lib = lib
    return lib


def fa_version() -> int:
    return load_library().fa_version()


def fa_strerror(code: int) -> str:
    try:
        return load_library().fa_strerror(int(code)).decode()
    except ImportError:
        return f"code {code}"


def fa_get_last_device_status() -> int:
    return load_library().fa_get_last_device_status()


def fa_bwd_workspace_bytes(B: int, H: int, N: int, d: int) -> int:
    return load_library().fa_bwd_workspace_bytes(B, H, N, d)


def _check(code: int, what: str):
    if code != FA_OK:
        raise FAError(code, what)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None and t.numel() > 0 else ctypes.c_void_p(0)


def _stream_handle(stream, device):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return ctypes.c_void_p(s.cuda_stream)


def _check_tensor(t, name, shape, dtype):
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor (no CPU path exists)")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def fa_fwd(q, k, v, causal: bool = False, scale: float | None = None, out=None, lse=None,
           stream=None):
    """Exact attention forward; returns (o bf16 [B,H,N,d], lse fp32 [B,H,N])."""
    import torch
    if q.dim() != 4:
        raise ValueError("q must be [B, H, N, d]")
    B, H, N, d = q.shape
    for name, t in (("q", q), ("k", k), ("v", v)):
        _check_tensor(t, name, (B, H, N, d), torch.bfloat16)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    _check_tensor(out, "out", (B, H, N, d), torch.bfloat16)
    _check_tensor(lse, "lse", (B, H, N), torch.float32)
    lib = load_library()
    with torch.cuda.device(q.device):
        rc = lib.fa_fwd_stream(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, N, d,
                               int(bool(causal)), float(scale), _stream_handle(stream, q.device))
    _check(rc, "fa_fwd")
    return out, lse


def fa_bwd(q, k, v, o, lse, do, causal: bool = False, scale: float | None = None, dq=None,
           dk=None, dv=None, workspace=None, stream=None):
    """Exact attention backward by recomputation; returns (dq, dk, dv) bf16."""
    import torch
    if q.dim() != 4:
        raise ValueError("q must be [B, H, N, d]")
    B, H, N, d = q.shape
    for name, t in (("q", q), ("k", k), ("v", v), ("o", o), ("do", do)):
        _check_tensor(t, name, (B, H, N, d), torch.bfloat16)
    _check_tensor(lse, "lse", (B, H, N), torch.float32)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    for name, t in (("dq", dq), ("dk", dk), ("dv", dv)):
        _check_tensor(t, name, (B, H, N, d), torch.bfloat16)
    lib = load_library()
    need = lib.fa_bwd_workspace_bytes(B, H, N, d)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    if workspace.numel() < need:
        raise ValueError(f"workspace needs {need} bytes")
    with torch.cuda.device(q.device):
        rc = lib.fa_bwd_stream(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(do), _ptr(dq),
                               _ptr(dk), _ptr(dv), B, H, N, d, int(bool(causal)), float(scale),
                               _ptr(workspace), ctypes.c_size_t(workspace.numel()),
                               _stream_handle(stream, q.device))
    _check(rc, "fa_bwd")
    return dq, dk, dv


# Size of the scratch array built into the library for fa_bwd_noalloc.
FA_BWD_NOALLOC_MAX_SCRATCH_BYTES = 64 << 20


def fa_bwd_noalloc(q, k, v, o, lse, do, causal: bool = False, scale: float | None = None,
                   dq=None, dk=None, dv=None, stream=None):
    """fa_bwd using the library's built-in scratch array instead of a workspace.

    For callers that may not allocate device memory on this path (the C entry
    point allocates nothing; passing dq/dk/dv keeps this wrapper allocation
    free too). Problems needing more than FA_BWD_NOALLOC_MAX_SCRATCH_BYTES of
    workspace raise FAError(FA_ERR_WORKSPACE). Calls that overlap on the GPU
    share the scratch and race: keep them on one stream.
    """
    import torch
    if q.dim() != 4:
        raise ValueError("q must be [B, H, N, d]")
    B, H, N, d = q.shape
    for name, t in (("q", q), ("k", k), ("v", v), ("o", o), ("do", do)):
        _check_tensor(t, name, (B, H, N, d), torch.bfloat16)
    _check_tensor(lse, "lse", (B, H, N), torch.float32)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    for name, t in (("dq", dq), ("dk", dk), ("dv", dv)):
        _check_tensor(t, name, (B, H, N, d), torch.bfloat16)
    lib = load_library()
    with torch.cuda.device(q.device):
        rc = lib.fa_bwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(do), _ptr(dq),
                                _ptr(dk), _ptr(dv), B, H, N, d, int(bool(causal)), float(scale),
                                _stream_handle(stream, q.device))
    _check(rc, "fa_bwd_noalloc")
    return dq, dk, dv


def _fwd_ex_args(q, k, v, causal, window, scale):
    import torch
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise ValueError("q, k, v must be [B, H, N, d]")
    B, H, Nq, d = q.shape
    Nk, dv = k.shape[2], v.shape[3]
    _check_tensor(q, "q", (B, H, Nq, d), torch.bfloat16)
    _check_tensor(k, "k", (B, H, Nk, d), torch.bfloat16)
    _check_tensor(v, "v", (B, H, Nk, dv), torch.bfloat16)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    return B, H, Nq, Nk, d, dv, int(bool(causal)), int(window), float(scale)


def fa_fwd_ex(q, k, v, causal: bool = False, window: int = 0, scale: float | None = None,
              out=None, lse=None, stream=None):
    """Forward with Nq queries over Nk keys and an optional window; (o, lse)."""
    import torch
    B, H, Nq, Nk, d, dv, c, w, sc = _fwd_ex_args(q, k, v, causal, window, scale)
    out = torch.empty((B, H, Nq, dv), dtype=torch.bfloat16, device=q.device) if out is None else out
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device) if lse is None else lse
    _check_tensor(out, "out", (B, H, Nq, dv), torch.bfloat16)
    _check_tensor(lse, "lse", (B, H, Nq), torch.float32)
    lib = load_library()
    with torch.cuda.device(q.device):
        rc = lib.fa_fwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, Nq, Nk, d, dv, c,
                           w, sc, _stream_handle(stream, q.device))
    _check(rc, "fa_fwd_ex")
    return out, lse


def fa_decode_num_splits(B: int, H: int, Nq: int, Nk: int, n_splits: int = 0) -> int:
    return load_library().fa_decode_num_splits(B, H, Nq, Nk, n_splits)


def fa_decode_workspace_bytes(B: int, H: int, Nq: int, Nk: int, dv: int, n_splits: int = 0) -> int:
    return load_library().fa_decode_workspace_bytes(B, H, Nq, Nk, dv, n_splits)


def fa_decode_splitkv(q, k, v, causal: bool = False, window: int = 0, scale: float | None = None,
                      n_splits: int = 0, out=None, lse=None, workspace=None, stream=None):
    """Split-key-range forward (decode over a long key/value cache); (o, lse)."""
    import torch
    B, H, Nq, Nk, d, dv, c, w, sc = _fwd_ex_args(q, k, v, causal, window, scale)
    out = torch.empty((B, H, Nq, dv), dtype=torch.bfloat16, device=q.device) if out is None else out
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device) if lse is None else lse
    _check_tensor(out, "out", (B, H, Nq, dv), torch.bfloat16)
    _check_tensor(lse, "lse", (B, H, Nq), torch.float32)
    lib = load_library()
    need = lib.fa_decode_workspace_bytes(B, H, Nq, Nk, dv, n_splits)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    with torch.cuda.device(q.device):
        rc = lib.fa_decode_splitkv(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, Nq, Nk,
                                   d, dv, c, w, sc, int(n_splits), _ptr(workspace),
                                   ctypes.c_size_t(workspace.numel()), _stream_handle(stream, q.device))
    _check(rc, "fa_decode_splitkv")
    return out, lse


def fa_bwd_ex(q, k, v, o, lse, do, causal: bool = False, window: int = 0,
              scale: float | None = None, dq=None, dk=None, dv=None, workspace=None, stream=None):
    """Backward with an optional causal sliding window; returns (dq, dk, dv)."""
    import torch
    if q.dim() != 4:
        raise ValueError("q must be [B, H, N, d]")
    B, H, N, d = q.shape
    d_v = v.shape[3]
    for name, t in (("q", q), ("k", k)):
        _check_tensor(t, name, (B, H, N, d), torch.bfloat16)
    for name, t in (("v", v), ("o", o), ("do", do)):
        _check_tensor(t, name, (B, H, N, d_v), torch.bfloat16)
    _check_tensor(lse, "lse", (B, H, N), torch.float32)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    lib = load_library()
    need = lib.fa_bwd_workspace_bytes(B, H, N, d)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    with torch.cuda.device(q.device):
        rc = lib.fa_bwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(do), _ptr(dq),
                           _ptr(dk), _ptr(dv), B, H, N, d, d_v, int(bool(causal)), int(window),
                           float(scale), _ptr(workspace), ctypes.c_size_t(workspace.numel()),
                           _stream_handle(stream, q.device))
    _check(rc, "fa_bwd_ex")
    return dq, dk, dv


def fa_fwd_dropout(q, k, v, dropout_p: float, seed: int, offset: int = 0, causal: bool = False,
                   scale: float | None = None, out=None, lse=None, stream=None):
    """Forward with dropout on the probabilities; returns (o, lse). The mask
    is a function of (seed, offset, batch-head, query, key) only."""
    import torch
    if q.dim() != 4:
        raise ValueError("q must be [B, H, N, d]")
    B, H, N, d = q.shape
    for name, t in (("q", q), ("k", k), ("v", v)):
        _check_tensor(t, name, (B, H, N, d), torch.bfloat16)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    out = torch.empty_like(q) if out is None else out
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    _check_tensor(out, "out", (B, H, N, d), torch.bfloat16)
    _check_tensor(lse, "lse", (B, H, N), torch.float32)
    lib = load_library()
    with torch.cuda.device(q.device):
        rc = lib.fa_fwd_dropout(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, N, d,
                                int(bool(causal)), float(scale), float(dropout_p), int(seed),
                                int(offset), _stream_handle(stream, q.device))
    _check(rc, "fa_fwd_dropout")
    return out, lse


def fa_bwd_dropout(q, k, v, o, lse, do, dropout_p: float, seed: int, offset: int = 0,
                   causal: bool = False, scale: float | None = None, dq=None, dk=None, dv=None,
                   workspace=None, stream=None):
    """Backward of fa_fwd_dropout for the same (dropout_p, seed, offset); returns (dq, dk, dv)."""
    import torch
    if q.dim() != 4:
        raise ValueError("q must be [B, H, N, d]")
    B, H, N, d = q.shape
    for name, t in (("q", q), ("k", k), ("v", v), ("o", o), ("do", do)):
        _check_tensor(t, name, (B, H, N, d), torch.bfloat16)
    _check_tensor(lse, "lse", (B, H, N), torch.float32)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    for name, t in (("dq", dq), ("dk", dk), ("dv", dv)):
        _check_tensor(t, name, (B, H, N, d), torch.bfloat16)
    lib = load_library()
    need = lib.fa_bwd_workspace_bytes(B, H, N, d)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    if workspace.numel() < need:
        raise ValueError(f"workspace needs {need} bytes")
    with torch.cuda.device(q.device):
        rc = lib.fa_bwd_dropout(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(do), _ptr(dq),
                                _ptr(dk), _ptr(dv), B, H, N, d, int(bool(causal)), float(scale),
                                float(dropout_p), int(seed), int(offset), _ptr(workspace),
                                ctypes.c_size_t(workspace.numel()), _stream_handle(stream, q.device))
    _check(rc, "fa_bwd_dropout")
    return dq, dk, dv
