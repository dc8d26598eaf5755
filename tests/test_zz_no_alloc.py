"""attn_bob_static: backward-over-backward for callers that cannot allocate device
memory (for example a plugin whose host application owns all device memory, or a
deployment whose memory plan forbids allocation after start-up).  It uses the
library's file-scope scratch array instead of a caller workspace.

The GPU test calls it through the C ABI several times in a row -- a larger problem
first, then smaller ones with an odd N (a padding row in the statistics), head dim
128 (the two-CTA BoB kernels) and 256 (the tf32 tensor-core engine), and again the first
one -- and checks each result against attn_bob run with a caller workspace that
is filled with NaN beforehand.  The bf16 parity tolerance of the other tests is the
bound the task sets; since the two entry points run the same kernels on the same
inputs, the outputs are also required to be bit for bit identical.  This file is
collected last so that a stop-at-first-failure run has already run every other
test."""
import ctypes

import numpy as np
import pytest

import __graft_entry__

__graft_entry__.build()
import fwd_bwd_double_gb300 as fbd  # noqa: E402
from fwd_bwd_double_gb300 import AttnDesc, lib  # noqa: E402

TOL = 2e-2
LIMIT_ROWS = 1 << 20  # 16 MiB of 16-byte row records


def _cabi_static(desc, t, outs, stream):
    args = [t["Q"], t["K"], t["V"], t["O"], t["dO"], t["lse"], t["gdQ"], t["gdK"], t["gdV"],
            outs["gQ"], outs["gK"], outs["gV"], outs["gdO"]]
    return lib.attn_bob_static(ctypes.byref(desc), *[ctypes.c_void_p(a.data_ptr()) for a in args],
                               ctypes.c_void_p(stream))


def test_static_limit_and_error_order_without_a_gpu():
    fake = [ctypes.c_void_p((1 << 40) + i * (1 << 32)) for i in range(13)]
    # Rows are counted with N rounded up to even: 3 * 349525 = 1,048,575 queries, but
    # 3 * 349526 = 1,048,578 stored rows, one record too many.
    over = AttnDesc(1, 3, 349525, 64, 0.0, 1, 1)
    assert lib.attn_bob_static(ctypes.byref(over), *fake, None) == 4  # ATTN_ERR_WORKSPACE
    assert b"static limit" in lib.attn_last_error() and b"rounded up to even" in lib.attn_last_error()
    assert 3 * 349526 > LIMIT_ROWS >= 3 * 349525
    big = AttnDesc(8, 16, 8193, 64, 0.0, 1, 1)  # 8 * 16 * 8194 rows
    assert lib.attn_bob_static(ctypes.byref(big), *fake, None) == 4
    # The descriptor is checked before the size, as attn_bob checks it.
    bad_d = AttnDesc(8, 16, 8193, 48, 0.0, 1, 1)
    assert lib.attn_bob_static(ctypes.byref(bad_d), *fake, None) == 2  # ATTN_ERR_UNSUPPORTED
    neg = AttnDesc(-1, 16, 8193, 64, 0.0, 1, 1)
    assert lib.attn_bob_static(ctypes.byref(neg), *fake, None) == 1  # ATTN_ERR_INVALID_ARG
    assert lib.attn_bob_static(None, *fake, None) == 1


def test_empty_problem_is_the_set_up_call():
    """An empty problem launches nothing; it looks the scratch array up on the current
    device (the start-up call), which needs a device: ATTN_OK with one, else
    ATTN_ERR_DEVICE."""
    import torch
    empty = AttnDesc(1, 1, 0, 64, 0.0, 1, 1)
    st = lib.attn_bob_static(ctypes.byref(empty), *([ctypes.c_void_p(0)] * 13), None)
    assert st == (0 if torch.cuda.is_available() else 7), lib.attn_last_error()


def _problem(name, B, H, N, d, seed):
    import torch

    import workloads as W
    w = W.Workload(name, B, H, N, d, "bf16", seed=seed)
    t = {k: torch.from_numpy(v).to("cuda").to(torch.bfloat16).contiguous() for k, v in W.inputs(w).items()}
    t["O"], t["lse"] = fbd.attn_fwd(t["Q"], t["K"], t["V"])
    return t


@pytest.mark.gpu
def test_static_scratch_matches_attn_bob_on_calls_in_a_row():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    stream = torch.cuda.current_stream().cuda_stream
    cases = [("noalloc_B2H3N300d64", 2, 3, 300, 64, 0),     # the largest first
             ("noalloc_B1H2N301d128", 1, 2, 301, 128, 1),   # odd N: a padding row per slice
             ("noalloc_B1H2N129d256", 1, 2, 129, 256, 2),   # the tf32 engine
             ("noalloc_B2H3N300d64", 2, 3, 300, 64, 0)]     # the first one again
    for call, (name, B, H, N, d, seed) in enumerate(cases):
        t = _problem(name, B, H, N, d, seed)
        desc = fbd.make_desc(t["Q"])
        ws = torch.full((fbd.attn_bob_workspace_bytes(desc, 0) // 4,), float("nan"), dtype=torch.float32,
                        device="cuda")
        ref = fbd.attn_bob(t["Q"], t["K"], t["V"], t["O"], t["dO"], t["lse"], t["gdQ"], t["gdK"], t["gdV"],
                           workspace=ws)
        outs = {k: torch.full_like(t["Q"], float("nan")) for k in ("gQ", "gK", "gV", "gdO")}
        assert _cabi_static(desc, t, outs, stream) == 0, lib.attn_last_error()
        assert lib.attn_device_status(ctypes.c_void_p(stream)) == 0
        for k, r in zip(("gQ", "gK", "gV", "gdO"), ref):
            got = outs[k].float().cpu().numpy().astype(np.float64)
            want = r.float().cpu().numpy().astype(np.float64)
            err = np.linalg.norm(got - want) / max(np.linalg.norm(want), 1e-30)
            assert err <= TOL, (call, name, k, err)
            assert torch.equal(outs[k], r), (call, name, k)
