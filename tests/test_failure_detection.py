"""Failure detection on the GPU without a fault: a bounded device wait is made to run
out (a barrier that nothing completes), and the host must read ATTN_ERR_TIMEOUT from
the status word while the context stays usable for the next call."""
import pytest

import workloads as W
from gpu_util import check_tol_fwd, host, inputs, to_device

pytestmark = pytest.mark.gpu

TIMEOUT = 6


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()


def test_bounded_wait_gives_up_and_the_context_stays_usable():
    import fwd_bwd_double_gb300 as fbd
    assert fbd.attn_check_wait_timeout() == TIMEOUT
    assert fbd.attn_device_status() == 0  # the status word was read and cleared
    # the next call runs normally on the same context
    w = W.Workload("after_timeout_B1H2N300d64_bf16", 1, 2, 300, 64, "bf16")
    x = to_device(inputs(w), w)
    O, lse = fbd.attn_fwd(x["Q"], x["K"], x["V"])
    fbd.attn_device_status()
    check_tol_fwd(w, host(O), host(lse))
    assert fbd.attn_check_wait_timeout() == TIMEOUT  # and the check repeats
