"""Host-side checks of the C ABI that need no GPU: the library loads, exports every
function include/fbd.h declares, and rejects bad arguments synchronously (before
any CUDA call, so fake non-NULL pointers are never dereferenced)."""
import ctypes
import os
import re

import pytest

import __graft_entry__

__graft_entry__.build()
import fwd_bwd_double_gb300 as fbd  # noqa: E402
from fwd_bwd_double_gb300 import AttnDesc, lib  # noqa: E402

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "fbd.h")

OK, INVALID, UNSUP, ALIGN, WS = 0, 1, 2, 3, 4
FAKE = 1 << 40  # a 16-byte aligned address that is never dereferenced


def declared_functions():
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    return sorted(set(re.findall(r"\b(attn_\w+)\s*\(", text)))


def test_library_exports_every_declared_function():
    names = declared_functions()
    assert "attn_fwd" in names and "attn_bwd" in names and "attn_bob" in names
    for n in names:
        assert hasattr(lib, n), n
        assert n in fbd._lib.PROTOTYPES, f"binding lacks a prototype for {n}"


def desc(B=1, H=2, N=64, d=64, scale=0.0, causal=1, dtype=1, group=0, window=0):
    return AttnDesc(B, H, N, d, scale, causal, dtype, group, window)


def ptrs(n, base=FAKE, stride=1 << 30):
    return [ctypes.c_void_p(base + i * stride) for i in range(n)]


def fwd(dsc, p=None):
    p = p or ptrs(5)
    return lib.attn_fwd(ctypes.byref(dsc), *p, None)


def bwd(dsc, p=None, gproj=0, ws_bytes=None):
    p = p or ptrs(10)
    wsb = lib.attn_bwd_workspace_bytes(ctypes.byref(dsc), gproj) if ws_bytes is None else ws_bytes
    return lib.attn_bwd(ctypes.byref(dsc), *p[:9], gproj, p[9], wsb, None)


def bob(dsc, p=None, ws_bytes=None, gproj=0):
    p = p or ptrs(14)
    wsb = lib.attn_bob_workspace_bytes(ctypes.byref(dsc), gproj) if ws_bytes is None else ws_bytes
    return lib.attn_bob(ctypes.byref(dsc), *p[:13], gproj, p[13], wsb, None)


@pytest.mark.parametrize("kw,code", [
    (dict(causal=2), UNSUP), (dict(causal=-1), UNSUP), (dict(d=16), UNSUP), (dict(d=48), UNSUP), (dict(d=512), UNSUP), (dict(dtype=7), UNSUP),
    (dict(B=-1), INVALID), (dict(N=-5), INVALID), (dict(d=0), INVALID),
    (dict(scale=float("nan")), INVALID), (dict(scale=float("inf")), INVALID), (dict(scale=-1.0), INVALID),
    (dict(N=1 << 31), INVALID),
    (dict(group=-1), INVALID), (dict(H=2, group=3), INVALID), (dict(H=6, group=4), INVALID),
    (dict(window=-1), INVALID), (dict(window=8, causal=0), UNSUP),
])
def test_rejects_bad_descriptors(kw, code):
    d = desc(**kw)
    assert fwd(d) == code
    assert bwd(d) == code
    assert bob(d) == code
    assert lib.attn_last_error()  # a detail message is recorded


@pytest.mark.parametrize("d", [32, 64, 96, 128, 256])
@pytest.mark.parametrize("dtype", [0, 1])
def test_every_supported_head_dim_passes_the_descriptor_check(d, dtype):
    # each (d, dtype) passes the descriptor check and fails on the NULL workspace instead
    p = ptrs(14)
    p[13] = ctypes.c_void_p(0)
    assert bob(desc(d=d, dtype=dtype), p) == WS
    p = ptrs(10)
    p[9] = ctypes.c_void_p(0)
    assert bwd(desc(d=d, dtype=dtype), p) == WS


def test_null_misaligned_and_overlapping_pointers():
    d = desc()
    p = ptrs(5)
    p[2] = ctypes.c_void_p(0)
    assert fwd(d, p) == INVALID
    p = ptrs(5)
    p[1] = ctypes.c_void_p(FAKE + (1 << 30) + 8)
    assert fwd(d, p) == ALIGN
    p = ptrs(5)
    p[3] = ctypes.c_void_p(FAKE + 1024)  # O inside Q
    assert fwd(d, p) == INVALID
    p = ptrs(10)
    p[7] = p[6]                           # dK == dQ
    assert bwd(d, p) == INVALID


def test_workspace_checks():
    d = desc(B=2, H=3, N=100)
    # The single-pass bf16 backward (d <= 64, no GProj): the statistics and then the fp32
    # dQ accumulator (64 floats per row); with GProj, at d > 64 or in float32 the
    # statistics alone.
    assert lib.attn_bwd_workspace_bytes(ctypes.byref(d), 0) == 2 * 3 * 100 * (16 + 256)
    assert lib.attn_bwd_workspace_bytes(ctypes.byref(d), 1) == 2 * 3 * 100 * 16
    assert lib.attn_bwd_workspace_bytes(ctypes.byref(desc(B=2, H=3, N=100, d=128)), 0) == 2 * 3 * 100 * 16
    assert lib.attn_bwd_workspace_bytes(ctypes.byref(desc(B=2, H=3, N=100, dtype=0)), 0) == 2 * 3 * 100 * 16
    assert lib.attn_bwd_workspace_bytes(ctypes.byref(desc(B=1, H=1, N=7, d=32)), 0) == 8 * 16 + 7 * 256
    # From N = 2^21 on the backward takes its two passes: the statistics alone.
    n1 = (1 << 21) - 1
    assert lib.attn_bwd_workspace_bytes(ctypes.byref(desc(B=1, H=2, N=n1)), 0) == 2 * (n1 + 1) * 16 + 2 * n1 * 256
    assert lib.attn_bwd_workspace_bytes(ctypes.byref(desc(B=1, H=2, N=1 << 21)), 0) == 2 * (1 << 21) * 16
    assert lib.attn_bob_workspace_bytes(ctypes.byref(d), 0) == 2 * 3 * 100 * 16
    assert bwd(d, ws_bytes=2 * 3 * 100 * (16 + 256) - 1) == WS
    assert bob(d, ws_bytes=0) == WS
    p = ptrs(14)
    p[13] = ctypes.c_void_p(0)
    assert bob(d, p) == WS
    # BoB with GProj (bf16): the coefficients (16 B per row) and, on the tensor-core
    # path, P^ b in fp32 (64 per row at d <= 64, 128 at d <= 128); float32 ignores it.
    rows = 2 * 3 * 100
    assert lib.attn_bob_workspace_bytes(ctypes.byref(d), 1) == rows * 32 + rows * 64 * 4
    d128 = desc(B=2, H=3, N=100, d=96)
    assert lib.attn_bob_workspace_bytes(ctypes.byref(d128), 1) == rows * 32 + rows * 128 * 4
    d256 = desc(B=2, H=3, N=100, d=256)
    assert lib.attn_bob_workspace_bytes(ctypes.byref(d256), 1) == rows * 32
    f32 = desc(B=2, H=3, N=100, dtype=0)
    assert lib.attn_bob_workspace_bytes(ctypes.byref(f32), 1) == rows * 16
    odd = desc(B=1, H=1, N=7)  # rows of a slice rounded up to an even count for the states only
    assert lib.attn_bob_workspace_bytes(ctypes.byref(odd), 1) == 8 * 32 + 7 * 64 * 4
    assert bob(d, gproj=1, ws_bytes=lib.attn_bob_workspace_bytes(ctypes.byref(d), 1) - 1) == WS
    assert bob(f32, gproj=1, ws_bytes=rows * 16 - 1) == WS


def test_empty_problems_are_ok_without_touching_memory():
    for kw in (dict(N=0), dict(B=0), dict(H=0)):
        d = desc(**kw)
        nulls = [ctypes.c_void_p(0)] * 14
        assert fwd(d, nulls[:5]) == OK
        assert bwd(d, nulls[:10]) == OK
        assert bob(d, nulls) == OK


def test_status_strings_and_version():
    for code in range(8):
        assert fbd.attn_status_string(code)
    assert fbd.attn_status_string(99) == "unknown status"
    assert "sm_103a" in fbd.attn_version()


def test_python_binding_raises_on_error():
    torch = pytest.importorskip("torch")
    q = torch.zeros(1, 1, 4, 48)  # d = 48 is unsupported: rejected before any device use
    with pytest.raises(fbd.FbdError) as e:
        fbd.attn_fwd(q, q, q, O=torch.zeros_like(q), lse=torch.zeros(1, 1, 4))
    assert e.value.status == UNSUP


def test_pass_masks_are_validated():
    d = desc()
    p = ptrs(10)
    wsb = lib.attn_bwd_workspace_bytes(ctypes.byref(d), 0)
    for bad in (0, 4, -1):
        assert lib.attn_bwd_passes(ctypes.byref(d), *p[:9], 0, p[9], wsb, bad, None) == INVALID
    q = ptrs(14)
    wsb = lib.attn_bob_workspace_bytes(ctypes.byref(d), 0)
    for bad in (0, 7):
        assert lib.attn_bob_passes(ctypes.byref(d), *q[:13], 0, q[13], wsb, bad, None) == INVALID
    assert fbd.ATTN_ROW_PASS == 1 and fbd.ATTN_COL_PASS == 2


def test_grouped_heads_size_the_key_side_tensors():
    """With g query heads per key/value head, K and V span B * H/g * N * d elements: an
    output starting one byte before the end of that span overlaps K, and the span of an
    ungrouped K (four times longer here) covers the same address."""
    nb = 1 * 1 * 64 * 64 * 2  # bytes of K for B=1, H=4, g=4, N=64, d=64, bf16
    for group, off in ((4, nb - 16), (1, nb), (1, 3 * nb)):
        p = ptrs(5)
        p[3] = ctypes.c_void_p(p[1].value + off)  # O placed inside K
        assert fwd(desc(H=4, group=group), p) == INVALID, (group, off)


def test_binding_derives_the_group_from_the_key_heads():
    torch = pytest.importorskip("torch")
    q, k = torch.zeros(2, 6, 8, 64), torch.zeros(2, 3, 8, 64)
    dsc = fbd.make_desc(q, K=k)
    assert (dsc.H, dsc.group) == (6, 2)
    assert fbd.make_desc(q).group == 1
    with pytest.raises(fbd.FbdError):
        fbd.make_desc(q, K=torch.zeros(2, 4, 8, 64))  # 4 key/value heads do not divide 6


def test_document_mask_descriptor_checks():
    """seg_lo / seg_hi: both or neither, only with the causal mask, 16-byte aligned, and
    never overlapping an output."""
    lo, hi = ctypes.c_void_p(FAKE + (9 << 30)), ctypes.c_void_p(FAKE + (10 << 30))
    d = desc()
    d.seg_lo = lo
    assert fwd(d) == INVALID                    # only one of the two
    d.seg_hi = hi
    d.causal = 0
    assert fwd(d) == UNSUP                      # a document mask needs causal = 1
    d.causal = 1
    d.seg_hi = ctypes.c_void_p(FAKE + (10 << 30) + 4)
    assert fwd(d) == ALIGN
    d.seg_hi = hi
    p = ptrs(5)
    p[3] = ctypes.c_void_p(lo.value)              # O placed on seg_lo
    assert fwd(d, p) == INVALID
    assert "seg_lo" in lib.attn_last_error().decode() or "overlaps" in lib.attn_last_error().decode()


def test_segment_bounds_argument_checks():
    f = lib.attn_segment_bounds
    a, b, c = ptrs(3)
    assert f(-1, 4, a, b, c, None) == INVALID
    assert f(2, -4, a, b, c, None) == INVALID
    assert f(0, 5, None, None, None, None) == OK       # empty: nothing launched
    assert f(2, 8, None, b, c, None) == INVALID
    assert f(2, 8, a, b, b, None) == INVALID           # the two outputs overlap
    assert f(2, 8, a, a, c, None) == INVALID           # an output overlaps the ids
    assert f(2, 8, ctypes.c_void_p(FAKE + 8), b, c, None) == ALIGN
