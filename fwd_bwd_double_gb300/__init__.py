"""Python binding of libfbd: exact attention (causal by default) forward, backward (GProj) and
backward-over-backward on GB300.

Argument marshalling only.  Every computation runs in the CUDA kernels of
``libfbd.so`` behind the C ABI declared in ``include/fbd.h``; PyTorch is used for
device memory and streams.  Importing the package loads the library and raises
if it is missing: there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os

from . import _lib
from ._lib import (ATTN_BF16, ATTN_COL_PASS, ATTN_F32, ATTN_ROW_PASS, AttnDesc, FbdError, lib,  # noqa: F401
                   status_name)

__all__ = [
    "attn_fwd", "attn_bwd", "attn_bob", "attn_bwd_passes", "attn_bob_passes", "ATTN_ROW_PASS", "ATTN_COL_PASS", "attn_bwd_workspace_bytes", "attn_bob_workspace_bytes",
    "attn_bob_static", "attn_bwd_projected_dS", "attn_segment_bounds", "attn_device_status", "attn_check_wait_timeout",
    "attn_status_string", "attn_version", "make_desc",
    "FbdError", "AttnDesc", "ATTN_F32", "ATTN_BF16", "lib",
]

LIB_PATH = _lib.LIB_PATH


def _torch():
    import torch
    return torch


def _dtype_code(t) -> int:
    torch = _torch()
    if t.dtype == torch.float32:
        return ATTN_F32
    if t.dtype == torch.bfloat16:
        return ATTN_BF16
    raise FbdError(2, f"unsupported tensor dtype {t.dtype} (float32 or bfloat16)")


def make_desc(Q, scale: float = 0.0, causal: int = 1, K=None, window: int = 0, bounds=None) -> AttnDesc:
    """Descriptor from a [B, H, N, d] query tensor and, for grouped key/value heads,
    the [B, H / g, N, d] key tensor (g query heads per key/value head); window W > 0
    (with causal) limits query i to the keys i - W < j <= i; bounds = (seg_lo, seg_hi)
    from attn_segment_bounds sets the document mask (the descriptor keeps their device
    addresses: keep the tensors alive while it is used)."""
    if Q.dim() != 4 or (K is not None and K.dim() != 4):
        raise FbdError(1, "tensors must be [B, H, N, d]")
    B, H, N, d = Q.shape
    Hkv = H if K is None else K.shape[1]
    if (Hkv == 0) != (H == 0) or (Hkv and H % Hkv):
        raise FbdError(1, f"key/value heads ({Hkv}) must divide query heads ({H})")
    lo, hi = (None, None) if bounds is None else (_ptr(bounds[0]), _ptr(bounds[1]))
    return AttnDesc(B, H, N, d, float(scale), int(causal), _dtype_code(Q), H // Hkv if Hkv else 1, int(window),
                    lo, hi)


def _ptr(t):
    if t is None:
        return None
    if not t.is_contiguous():
        raise FbdError(1, "tensors must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    torch = _torch()
    if stream is None:
        if torch.cuda.is_available():
            stream = torch.cuda.current_stream()
        else:
            return None
    return ctypes.c_void_p(int(getattr(stream, "cuda_stream", stream)))


def _check(status: int):
    if status != 0:
        raise FbdError(status, lib.attn_last_error().decode())


def attn_fwd(Q, K, V, O=None, lse=None, scale: float = 0.0, stream=None, desc=None, causal: bool = True, window: int = 0,
             bounds=None):
    """O, lse = attention forward (allocates O and lse with torch when not given)."""
    torch = _torch()
    desc = desc or make_desc(Q, scale, int(causal), K, window, bounds)
    if O is None:
        O = torch.empty_like(Q)
    if lse is None:
        lse = torch.empty(Q.shape[:3], dtype=torch.float32, device=Q.device)
    _check(lib.attn_fwd(ctypes.byref(desc), _ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(lse), _stream(stream)))
    return O, lse


def attn_bwd_workspace_bytes(desc: AttnDesc, gproj: int = 0) -> int:
    return int(lib.attn_bwd_workspace_bytes(ctypes.byref(desc), int(gproj)))


def attn_bob_workspace_bytes(desc: AttnDesc, gproj: int = 0) -> int:
    return int(lib.attn_bob_workspace_bytes(ctypes.byref(desc), int(gproj)))


def _workspace(nbytes, like, workspace):
    torch = _torch()
    if workspace is None:
        workspace = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=like.device)
    return workspace


def attn_bwd(Q, K, V, O, dO, lse, gproj: int = 0, dQ=None, dK=None, dV=None, workspace=None,
             scale: float = 0.0, stream=None, desc=None, causal: bool = True, window: int = 0, bounds=None):
    """dQ, dK, dV = recompute backward (GProj when gproj != 0, bf16 only)."""
    return attn_bwd_passes(Q, K, V, O, dO, lse, ATTN_ROW_PASS | ATTN_COL_PASS, gproj, dQ, dK, dV, workspace,
                           scale, stream, desc, causal, window, bounds)


def attn_bwd_passes(Q, K, V, O, dO, lse, passes, gproj: int = 0, dQ=None, dK=None, dV=None, workspace=None,
                    scale: float = 0.0, stream=None, desc=None, causal: bool = True, window: int = 0, bounds=None):
    """The backward's row pass (dQ) and/or column pass (dK, dV); see attn_bwd_passes in fbd.h."""
    torch = _torch()
    desc = desc or make_desc(Q, scale, int(causal), K, window, bounds)
    dQ = torch.empty_like(Q) if dQ is None else dQ
    dK = torch.empty_like(K) if dK is None else dK
    dV = torch.empty_like(V) if dV is None else dV
    need = attn_bwd_workspace_bytes(desc, gproj)
    workspace = _workspace(need, Q, workspace)
    _check(lib.attn_bwd_passes(ctypes.byref(desc), _ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(dO), _ptr(lse),
                               _ptr(dQ), _ptr(dK), _ptr(dV), int(gproj), _ptr(workspace),
                               ctypes.c_size_t(workspace.numel() * workspace.element_size()), int(passes),
                               _stream(stream)))
    return dQ, dK, dV


def attn_bob(Q, K, V, O, dO, lse, gdQ, gdK, gdV, gQ=None, gK=None, gV=None, gdO=None, workspace=None,
             scale: float = 0.0, stream=None, desc=None, causal: bool = True, window: int = 0, gproj: int = 0,
             bounds=None):
    """gQ, gK, gV, gdO = backward over backward against cotangents (gdQ, gdK, gdV)
    (GProj on the rounded dS of its dS b and dS^T a products when gproj != 0, bf16 only)."""
    return attn_bob_passes(Q, K, V, O, dO, lse, gdQ, gdK, gdV, ATTN_ROW_PASS | ATTN_COL_PASS, gQ, gK, gV, gdO,
                           workspace, scale, stream, desc, causal, window, gproj, bounds)


def attn_bob_passes(Q, K, V, O, dO, lse, gdQ, gdK, gdV, passes, gQ=None, gK=None, gV=None, gdO=None,
                    workspace=None, scale: float = 0.0, stream=None, desc=None, causal: bool = True, window: int = 0,
                    gproj: int = 0, bounds=None):
    """BoB's row pass (gQ, gdO, row states) and/or column pass (gK, gV); see fbd.h."""
    torch = _torch()
    desc = desc or make_desc(Q, scale, int(causal), K, window, bounds)
    gQ = torch.empty_like(Q) if gQ is None else gQ
    gK = torch.empty_like(K) if gK is None else gK
    gV = torch.empty_like(V) if gV is None else gV
    gdO = torch.empty_like(dO) if gdO is None else gdO
    workspace = _workspace(attn_bob_workspace_bytes(desc, gproj), Q, workspace)
    _check(lib.attn_bob_passes(ctypes.byref(desc), _ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(dO), _ptr(lse),
                               _ptr(gdQ), _ptr(gdK), _ptr(gdV), _ptr(gQ), _ptr(gK), _ptr(gV), _ptr(gdO), int(gproj),
                               _ptr(workspace), ctypes.c_size_t(workspace.numel() * workspace.element_size()),
                               int(passes), _stream(stream)))
    return gQ, gK, gV, gdO


def attn_bob_static(Q, K, V, O, dO, lse, gdQ, gdK, gdV, gQ=None, gK=None, gV=None, gdO=None,
                    scale: float = 0.0, stream=None, desc=None, causal: bool = True, window: int = 0, bounds=None):
    """attn_bob without a workspace argument: the library's static scratch array is used
    (for callers that cannot allocate device memory; B*H*Np <= 1,048,576 with Np = N
    rounded up to an even count)."""
    torch = _torch()
    desc = desc or make_desc(Q, scale, int(causal), K, window, bounds)
    gQ = torch.empty_like(Q) if gQ is None else gQ
    gK = torch.empty_like(K) if gK is None else gK
    gV = torch.empty_like(V) if gV is None else gV
    gdO = torch.empty_like(dO) if gdO is None else gdO
    _check(lib.attn_bob_static(ctypes.byref(desc), _ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(dO), _ptr(lse),
                               _ptr(gdQ), _ptr(gdK), _ptr(gdV), _ptr(gQ), _ptr(gK), _ptr(gV), _ptr(gdO),
                               _stream(stream)))
    return gQ, gK, gV, gdO


def attn_bwd_projected_dS(Q, K, V, O, dO, lse, dS=None, scale: float = 0.0, stream=None, desc=None, causal: bool = True,
                          window: int = 0, bounds=None):
    """Diagnostic: the GProj-projected dS [B, H, N, N] float32 (small N only)."""
    torch = _torch()
    desc = desc or make_desc(Q, scale, int(causal), K, window, bounds)
    B, H, N, _ = Q.shape
    dS = torch.empty((B, H, N, N), dtype=torch.float32, device=Q.device) if dS is None else dS
    _check(lib.attn_bwd_projected_dS(ctypes.byref(desc), _ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(dO),
                                     _ptr(lse), _ptr(dS), _stream(stream)))
    return dS


def attn_segment_bounds(seg, seg_lo=None, seg_hi=None, stream=None):
    """(seg_lo, seg_hi) int32 [B, N] of the document mask from segment ids seg [B, N]
    (int32, non-decreasing along N); pass them as `bounds` to the attention calls."""
    torch = _torch()
    if seg.dim() != 2 or seg.dtype != torch.int32:
        raise FbdError(1, "seg must be an int32 [B, N] tensor")
    B, N = seg.shape
    seg_lo = torch.empty_like(seg) if seg_lo is None else seg_lo
    seg_hi = torch.empty_like(seg) if seg_hi is None else seg_hi
    _check(lib.attn_segment_bounds(int(B), int(N), _ptr(seg), _ptr(seg_lo), _ptr(seg_hi), _stream(stream)))
    return seg_lo, seg_hi


def attn_device_status(stream=None) -> int:
    """Synchronise the stream; raise FbdError if a device-side wait timed out."""
    _check(lib.attn_device_status(_stream(stream)))
    return 0


def attn_check_wait_timeout(stream=None) -> int:
    """Run the library's failure-detection check (a bounded device wait that is made to
    give up); returns the status code, ATTN_ERR_TIMEOUT (6) when the path works."""
    return int(lib.attn_check_wait_timeout(_stream(stream)))


def attn_status_string(status: int) -> str:
    return lib.attn_status_string(int(status)).decode()


def attn_version() -> str:
    return lib.attn_version().decode()
