"""Document (segment) mask on the GPU: packed documents, query i sees key j iff j <= i and
both tokens carry the same segment id ("FlashBoB: second-order attention", "When FlashBoB
changes the engineering plan", flexible masks).  attn_segment_bounds turns the ids into
per-token bounds (the first key of each row's document, the last query of each key's
document); every operation is checked against the oracle under the same mask."""
import numpy as np
import pytest

import oracle
import workloads as W
from gpu_util import host, rel_fro, to_device

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-5, "bf16": 2e-2}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()


def _bounds(seg):
    import torch

    import fwd_bwd_double_gb300 as fbd
    t = torch.from_numpy(np.ascontiguousarray(seg, dtype=np.int32)).cuda()
    lo, hi = fbd.attn_segment_bounds(t)
    return t, lo, hi


def _np_bounds(seg):
    B, N = seg.shape
    lo, hi = np.empty_like(seg), np.empty_like(seg)
    for b in range(B):
        for i in range(N):
            j = i
            while j > 0 and seg[b, j - 1] == seg[b, i]:
                j -= 1
            lo[b, i] = j
            j = i
            while j < N - 1 and seg[b, j + 1] == seg[b, i]:
                j += 1
            hi[b, i] = j
    return lo, hi


@pytest.mark.parametrize("N,mean", [(1, 1), (7, 1), (300, 1), (300, 17), (1000, 400), (333, 5000)])
def test_segment_bounds_match_runs(N, mean):
    seg = W.segment_ids(3, N, mean, seed=N)
    _, lo, hi = _bounds(seg)
    wlo, whi = _np_bounds(seg)
    assert np.array_equal(lo.cpu().numpy(), wlo) and np.array_equal(hi.cpu().numpy(), whi)


def run_all(w, x, bounds, gproj=0, window=0, ops=("bwd", "bob")):
    import fwd_bwd_double_gb300 as fbd
    out = {}
    O, lse = fbd.attn_fwd(x["Q"], x["K"], x["V"], window=window, bounds=bounds)
    out["O"], out["L"] = O, lse
    if "bwd" in ops:
        out["dQ"], out["dK"], out["dV"] = fbd.attn_bwd(x["Q"], x["K"], x["V"], O, x["dO"], lse, gproj=gproj,
                                                       window=window, bounds=bounds)
    if "bob" in ops:
        out["gQ"], out["gK"], out["gV"], out["gdO"] = fbd.attn_bob(
            x["Q"], x["K"], x["V"], O, x["dO"], lse, x["gdQ"], x["gdK"], x["gdV"], window=window, gproj=gproj,
            bounds=bounds)
    fbd.attn_device_status()
    return out


def check(w, got, seg, window=0, ops=("bwd", "bob")):
    x = W.inputs(w)
    mask = oracle.SegmentsBatch(seg, window)
    ref = dict(zip(("O", "L"), (None, None)))
    f = oracle.forward_all(x["Q"], x["K"], x["V"], causal=mask, groups=w.group)
    ref = {"O": f["O"], "L": f["L"]}
    if "bwd" in ops:
        ref.update(oracle.backward_all(x["Q"], x["K"], x["V"], x["dO"], causal=mask, groups=w.group))
    if "bob" in ops:
        ref.update(oracle.bob_all(x["Q"], x["K"], x["V"], x["dO"], x["gdQ"], x["gdK"], x["gdV"], causal=mask,
                                  groups=w.group))
    errs = {k: rel_fro(host(got[k]), ref[k]) for k in got}
    tol = TOL[w.dtype]
    bad = {k: v for k, v in errs.items() if not v <= tol}
    assert not bad, f"{w.name}: {bad} (all {errs})"
    return errs


@pytest.mark.parametrize("mean", [17, 100, 300])
@pytest.mark.parametrize("d,dtype", [(64, "bf16"), (128, "bf16"), (64, "f32")])
def test_documents_all_ops(mean, d, dtype):
    w = W.Workload(f"docs_B2H3N1000d{d}_{dtype}", 2, 3, 1000, d, dtype)
    seg = W.segment_ids(w.B, w.N, mean, seed=mean)
    _, lo, hi = _bounds(seg)
    got = run_all(w, to_device(W.inputs(w), w), (lo, hi))
    errs = check(w, got, seg)
    print(w.name, mean, {k: f"{v:.2e}" for k, v in errs.items()})


@pytest.mark.parametrize("d", [64, 128])
def test_documents_gproj_window_and_grouped_heads(d):
    w = W.Workload(f"docs_gqa_B2H6g3N700d{d}_bf16", 2, 6, 700, d, "bf16", group=3)
    seg = W.segment_ids(w.B, w.N, 150, seed=d)
    _, lo, hi = _bounds(seg)
    x = to_device(W.inputs(w), w)
    for gp in (0, 1):
        for win in (0, 90):
            got = run_all(w, x, (lo, hi), gproj=gp, window=win)
            errs = check(w, got, seg, window=win)
            print(w.name, gp, win, {k: f"{v:.2e}" for k, v in errs.items()})


@pytest.mark.parametrize("d", [32, 96, 256])
def test_documents_other_head_dims(d):
    w = W.Workload(f"docs_B1H2N600d{d}_bf16", 1, 2, 600, d, "bf16")
    seg = W.segment_ids(w.B, w.N, 120, seed=d)
    _, lo, hi = _bounds(seg)
    x = to_device(W.inputs(w), w)
    for gp in (0, 1):
        check(w, run_all(w, x, (lo, hi), gproj=gp), seg)


def test_documents_limits():
    """One document is the causal mask (the same bits as no document mask, on the same
    kernels with the band on); a document per token leaves each row its own key only."""
    import torch

    import fwd_bwd_double_gb300 as fbd
    w = W.Workload("docs_limits_B1H2N300d64_bf16", 1, 2, 300, 64, "bf16")
    x = to_device(W.inputs(w), w)
    one = np.zeros((1, 300), np.int32)
    _, lo, hi = _bounds(one)
    a = run_all(w, x, (lo, hi))
    check(w, a, one)
    each = np.arange(300, dtype=np.int32)[None]
    _, lo1, hi1 = _bounds(each)
    b = run_all(w, x, (lo1, hi1))
    xi = W.inputs(w)
    assert rel_fro(host(b["O"]), xi["V"]) <= 2e-2 and rel_fro(host(b["dV"]), xi["dO"]) <= 2e-2
    assert rel_fro(host(b["gdO"]), xi["gdV"]) <= 2e-2
    scale = float(np.abs(xi["dO"]).max())
    for k in ("dQ", "dK", "gQ", "gK", "gV"):
        assert float(np.abs(host(b[k])).max()) <= 2e-2 * scale, k
    assert torch.isfinite(b["L"]).all()
    fbd.attn_device_status()


@pytest.mark.parametrize("d", [64, 128])
def test_documents_passes_compose_on_nan_workspace(d):
    import torch

    import fwd_bwd_double_gb300 as fbd
    from gpu_util import assert_same_up_to_sum_order
    w = W.Workload(f"docs_passes_B2H3N300d{d}_bf16", 2, 3, 300, d, "bf16")
    seg = W.segment_ids(w.B, w.N, 60, seed=7)
    _, lo, hi = _bounds(seg)
    x = to_device(W.inputs(w), w)
    O, lse = fbd.attn_fwd(x["Q"], x["K"], x["V"], bounds=(lo, hi))
    for gp in (0, 1):
        ref_b = fbd.attn_bwd(x["Q"], x["K"], x["V"], O, x["dO"], lse, gproj=gp, bounds=(lo, hi))
        ref_g = fbd.attn_bob(x["Q"], x["K"], x["V"], O, x["dO"], lse, x["gdQ"], x["gdK"], x["gdV"], gproj=gp,
                             bounds=(lo, hi))
        desc = fbd.make_desc(x["Q"], bounds=(lo, hi))
        nbytes = max(fbd.attn_bwd_workspace_bytes(desc, gp), fbd.attn_bob_workspace_bytes(desc, gp))
        ws = torch.full((nbytes // 4,), float("nan"), device="cuda")
        b = [torch.full_like(x["Q"], float("nan")) for _ in range(3)]
        g = [torch.full_like(x["Q"], float("nan")) for _ in range(4)]
        for ps in (fbd.ATTN_ROW_PASS, fbd.ATTN_COL_PASS):
            fbd.attn_bwd_passes(x["Q"], x["K"], x["V"], O, x["dO"], lse, ps, gproj=gp, dQ=b[0], dK=b[1], dV=b[2],
                                workspace=ws, desc=desc)
        for ps in (fbd.ATTN_ROW_PASS, fbd.ATTN_COL_PASS):
            fbd.attn_bob_passes(x["Q"], x["K"], x["V"], O, x["dO"], lse, x["gdQ"], x["gdK"], x["gdV"], ps,
                                gQ=g[0], gK=g[1], gV=g[2], gdO=g[3], workspace=ws, desc=desc, gproj=gp)
        fbd.attn_device_status()
        for n, (a, r) in enumerate(zip(b + g, list(ref_b) + list(ref_g))):
            if n < 3 and gp == 0 and d <= 64:  # the separate passes vs the single-pass form
                assert_same_up_to_sum_order(a, r, ("dQ", "dK", "dV")[n])
            else:
                assert torch.equal(a, r)


def test_documents_long_sampled():
    """B1 H2 N8192 d64 bf16 with documents of mean length 1000: sampled rows and late
    columns of every output against the oracle under the same mask."""
    from test_gpu_parity import sample_rows_cols, sampled_check
    w = W.Workload("docs_long_B1H2N8192d64_bf16", 1, 2, 8192, 64, "bf16")
    seg = W.segment_ids(1, w.N, 1000, seed=8192)
    _, lo, hi = _bounds(seg)
    got = run_all(w, to_device(W.inputs(w), w), (lo, hi))
    rows, cols = sample_rows_cols(w.N, np.random.default_rng(5))
    errs = sampled_check(w, got, ("bwd", "bob"), heads=[0, 1], rows=rows, cols=cols,
                         causal=oracle.Segments(seg[0]))
    print(w.name, {k: f"{v:.2e}" for k, v in errs.items()})


def test_document_mask_arguments():
    """Only one bound given, or a document mask without the causal mask, is refused
    before any launch."""
    import torch

    import fwd_bwd_double_gb300 as fbd
    from fwd_bwd_double_gb300 import FbdError
    w = W.Workload("docs_args_B1H1N64d64_bf16", 1, 1, 64, 64, "bf16")
    x = to_device(W.inputs(w), w)
    _, lo, hi = _bounds(np.zeros((1, 64), np.int32))
    d = fbd.make_desc(x["Q"], bounds=(lo, hi))
    d.seg_hi = None
    with pytest.raises(FbdError) as e:
        fbd.attn_fwd(x["Q"], x["K"], x["V"], desc=d)
    assert e.value.status == 1
    with pytest.raises(FbdError) as e:
        fbd.attn_fwd(x["Q"], x["K"], x["V"], causal=False, bounds=(lo, hi))
    assert e.value.status == 2
    torch.cuda.synchronize()
