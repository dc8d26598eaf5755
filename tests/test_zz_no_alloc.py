"""attn_bob_static: backward-over-backward for callers that cannot allocate device
memory (for example a plugin whose host application owns all device memory, or a
deployment whose memory plan forbids allocation after start-up).  It uses the
library's file-scope scratch array instead of a caller workspace.

The GPU test calls it through the C ABI twice in a row and checks each result
against attn_bob with a caller workspace, within the bf16 parity tolerance (the
two run the same kernels, so the outputs are expected to be identical).  This
file is collected last so that a stop-at-first-failure run has already run every
other test."""
import ctypes

import numpy as np
import pytest

import __graft_entry__

__graft_entry__.build()
import fwd_bwd_double_gb300 as fbd  # noqa: E402
from fwd_bwd_double_gb300 import AttnDesc, lib  # noqa: E402

TOL = 2e-2


def _cabi_static(desc, t, outs, stream):
    args = [t["Q"], t["K"], t["V"], t["O"], t["dO"], t["lse"], t["gdQ"], t["gdK"], t["gdV"],
            outs["gQ"], outs["gK"], outs["gV"], outs["gdO"]]
    return lib.attn_bob_static(ctypes.byref(desc), *[ctypes.c_void_p(a.data_ptr()) for a in args],
                               ctypes.c_void_p(stream))


def test_rejects_problems_beyond_the_static_limit_without_a_gpu():
    big = AttnDesc(8, 16, 8193, 64, 0.0, 1, 1)  # 1,048,704 rows > 1,048,576
    fake = [ctypes.c_void_p((1 << 40) + i * (1 << 32)) for i in range(13)]
    assert lib.attn_bob_static(ctypes.byref(big), *fake, None) == 4  # ATTN_ERR_WORKSPACE
    assert b"static limit" in lib.attn_last_error()
    empty = AttnDesc(1, 1, 0, 64, 0.0, 1, 1)
    assert lib.attn_bob_static(ctypes.byref(empty), *([ctypes.c_void_p(0)] * 13), None) == 0


@pytest.mark.gpu
def test_static_scratch_matches_attn_bob_on_two_calls():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import workloads as W
    w = W.Workload("noalloc_B2H3N300d64", 2, 3, 300, 64, "bf16")
    x = W.inputs(w)
    t = {k: torch.from_numpy(v).to("cuda").to(torch.bfloat16).contiguous() for k, v in x.items()}
    t["O"], t["lse"] = fbd.attn_fwd(t["Q"], t["K"], t["V"])
    ref = fbd.attn_bob(t["Q"], t["K"], t["V"], t["O"], t["dO"], t["lse"], t["gdQ"], t["gdK"], t["gdV"])
    desc = fbd.make_desc(t["Q"])
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        outs = {k: torch.full_like(t["Q"], float("nan")) for k in ("gQ", "gK", "gV", "gdO")}
        assert _cabi_static(desc, t, outs, stream) == 0, lib.attn_last_error()
        assert lib.attn_device_status(ctypes.c_void_p(stream)) == 0
        for k, r in zip(("gQ", "gK", "gV", "gdO"), ref):
            got = outs[k].float().cpu().numpy().astype(np.float64)
            want = r.float().cpu().numpy().astype(np.float64)
            err = np.linalg.norm(got - want) / np.linalg.norm(want)
            assert err <= TOL, (call, k, err)
