"""GPU parity: the CUDA path (through the C ABI) against the CPU fp64 oracle on the
same seeded inputs.

Tolerances (relative Frobenius error per output tensor over all slices checked):
1e-5 for float32 inputs, 2e-2 for bf16 inputs with fp32 accumulation.  At long
sequence lengths the oracle checks sampled rows (row-pass outputs) and late
columns (column-pass outputs, which need only the rows after them)."""
import numpy as np
import pytest

import oracle
import workloads as W
from gpu_util import (assert_same_up_to_sum_order, host, inputs, oracle_full, rel_fro, row_rel_errors, run_ops,
                      to_device)

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-5, "bf16": 2e-2}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()


def err_vs(got, ref, scale):
    """Relative Frobenius error; for a reference that is exactly zero, the error norm over
    `scale`.  Such outputs vanish by cancellation (at N = 1, P = 1 makes dS = dP - D = 0,
    and with it dQ, dK, gQ, gK, gV), and an fp32 computation that does not evaluate the
    two cancelling dot products dP = dO.V and D = dO.O in the same order leaves about
    2^-24 sqrt(d) |dO| |V| of each: relative to zero that is no error measure, so those
    outputs are held to the tolerance times the scale of the terms that cancel (the norm
    of dO), as the closed forms of the one-key window are held to the scale of dO."""
    if not np.any(np.asarray(ref)):
        return float(np.linalg.norm(np.asarray(got, np.float64)) / scale)
    return rel_fro(got, ref)


def check_full(w, got, ops, causal=True, window=0):
    tol = TOL[w.dtype]
    causal = oracle.Window(window) if window else causal
    scale = float(np.linalg.norm(inputs(w)["dO"].astype(np.float64))) or 1.0
    errs = {}
    f = oracle_full(w, "fwd", causal)
    errs["O"], errs["L"] = rel_fro(host(got["O"]), f["O"]), rel_fro(host(got["L"]), f["L"])
    if "bwd" in ops:
        b = oracle_full(w, "bwd", causal)
        for k in ("dQ", "dK", "dV"):
            errs[k] = err_vs(host(got[k]), b[k], scale)
    if "bob" in ops:
        b = oracle_full(w, "bob", causal)
        for k in ("gQ", "gK", "gV", "gdO"):
            errs[k] = err_vs(host(got[k]), b[k], scale)
    bad = {k: v for k, v in errs.items() if not v <= tol}
    assert not bad, f"{w.name}: errors above {tol}: {bad} (all: {errs})"
    return errs


def test_tiny_f32_all_ops():
    w = W.TINY_F32
    got = run_ops(w, to_device(inputs(w), w))
    errs = check_full(w, got, ("bwd", "bob"))
    print(w.name, {k: f"{v:.2e}" for k, v in errs.items()})


@pytest.mark.parametrize("gproj", [0, 1])
def test_gpt2_layer_bf16(gproj):
    w = W.GPT2_LAYER
    got = run_ops(w, to_device(inputs(w), w), ops=("bwd", "bob"), gproj=gproj)
    errs = check_full(w, got, ("bwd", "bob"))
    print(w.name, gproj, {k: f"{v:.2e}" for k, v in errs.items()})


def test_long_sweep_n4096_all_heads():
    w = W.LONG_SWEEP[0]
    got = run_ops(w, to_device(inputs(w), w))
    errs = check_full(w, got, ("bwd", "bob"))
    print(w.name, {k: f"{v:.2e}" for k, v in errs.items()})


def sampled_check(w, got, ops, heads, rows, cols, batch=0, causal=True):
    """Oracle on sampled rows (row outputs) and columns (column outputs) of given heads
    of one batch entry (causal: True, False or an oracle.Window)."""
    tol = TOL[w.dtype]
    errs = {}
    x = W.inputs(w, heads=heads, batches=[batch])
    acc = {k: ([], []) for k in ("O", "L", "dQ", "dK", "dV", "gQ", "gK", "gV", "gdO")}
    b = batch
    for hi, h in enumerate(heads):
        s = {k: v[0, hi].astype(np.float64) for k, v in x.items()}
        O, L = oracle.forward_rows(s["Q"], s["K"], s["V"], rows, scale=w.scale, causal=causal)
        acc["O"][0].append(host(got["O"][b, h])[rows]); acc["O"][1].append(O)
        acc["L"][0].append(host(got["L"][b, h])[rows]); acc["L"][1].append(L)
        if "bwd" in ops:
            acc["dQ"][0].append(host(got["dQ"][b, h])[rows])
            acc["dQ"][1].append(oracle.backward_rows(s["Q"], s["K"], s["V"], s["dO"], rows, scale=w.scale, causal=causal))
            dK, dV = oracle.backward_cols(s["Q"], s["K"], s["V"], s["dO"], cols, scale=w.scale, causal=causal)
            acc["dK"][0].append(host(got["dK"][b, h])[cols]); acc["dK"][1].append(dK)
            acc["dV"][0].append(host(got["dV"][b, h])[cols]); acc["dV"][1].append(dV)
        if "bob" in ops:
            r = oracle.bob_rows(s["Q"], s["K"], s["V"], s["dO"], s["gdQ"], s["gdK"], s["gdV"], rows, scale=w.scale, causal=causal)
            acc["gQ"][0].append(host(got["gQ"][b, h])[rows]); acc["gQ"][1].append(r["gQ"])
            acc["gdO"][0].append(host(got["gdO"][b, h])[rows]); acc["gdO"][1].append(r["gdO"])
            gK, gV = oracle.bob_cols(s["Q"], s["K"], s["V"], s["dO"], s["gdQ"], s["gdK"], s["gdV"], cols,
                                     scale=w.scale, causal=causal)
            acc["gK"][0].append(host(got["gK"][b, h])[cols]); acc["gK"][1].append(gK)
            acc["gV"][0].append(host(got["gV"][b, h])[cols]); acc["gV"][1].append(gV)
    for k, (g, r) in acc.items():
        if g:
            errs[k] = rel_fro(np.concatenate(g), np.concatenate(r))
    bad = {k: v for k, v in errs.items() if not v <= tol}
    assert not bad, f"{w.name}: sampled errors above {tol}: {bad} (all: {errs})"
    return errs


def sample_rows_cols(N, rng, n_rows=48, n_tail_cols=96):
    """Rows anywhere (row outputs need only keys <= row); columns late in the sequence
    (column outputs need every row after them)."""
    rows = np.unique(np.concatenate([[0, 1, 127, 128, N - 1], rng.integers(0, N, n_rows), np.arange(N - 40, N)]))
    cols = np.unique(np.concatenate([np.arange(N - n_tail_cols, N), rng.integers(max(0, N - 1024), N, 16)]))
    return rows[(rows >= 0) & (rows < N)], cols[(cols >= 0) & (cols < N)]


@pytest.mark.parametrize("N", [16384, 65536, 262144])
def test_long_sweep_sampled(N):
    w = W.LONG_SWEEP[0].with_n(N)
    x = to_device(W.inputs(w), w)
    got = run_ops(w, x)
    rows, cols = sample_rows_cols(N, np.random.default_rng(N))
    errs = sampled_check(w, got, ("bwd", "bob"), heads=[0, 11], rows=rows, cols=cols)
    print(w.name, {k: f"{v:.2e}" for k, v in errs.items()})


def test_backward_two_passes_from_n_2_21():
    """At N = 2^21 the bf16 backward at d = 64 takes its two passes (the single-pass form
    only runs below that length): sampled rows of dQ and late columns of dK, dV of both
    heads against the oracle, and the workspace it asks for is the statistics alone."""
    import fwd_bwd_double_gb300 as fbd
    N = 1 << 21
    w = W.Workload(f"longbwd_B1H2N{N}d64_bf16", 1, 2, N, 64, "bf16")
    x = to_device(W.inputs(w, names=("Q", "K", "V", "dO")), w)
    assert fbd.attn_bwd_workspace_bytes(fbd.make_desc(x["Q"]), 0) == 2 * N * 16
    got = run_ops(w, x, ops=("fwd", "bwd"))
    rng = np.random.default_rng(21)
    rows = np.unique(np.concatenate([[0, 1, 127, 128, N // 2, N - 2, N - 1], rng.integers(0, N, 16)]))
    cols = np.arange(N - 48, N)  # the last keys: each needs only the queries after it
    errs = sampled_check(w, got, ("bwd",), heads=[0, 1], rows=rows, cols=cols)
    print(w.name, {k: f"{v:.2e}" for k, v in errs.items()})


@pytest.mark.parametrize("d", [64, 256])
def test_f32_long_sampled(d):
    """float32 on the tf32 engine over many key blocks with a ragged tail (N = 5000:
    39 blocks of 128 rows, 79 of 64 keys), sampled rows and late columns of two heads."""
    w = W.Workload(f"f32long_B1H2N5000d{d}_f32", 1, 2, 5000, d, "f32")
    got = run_ops(w, to_device(W.inputs(w), w))
    rows, cols = sample_rows_cols(w.N, np.random.default_rng(d))
    errs = sampled_check(w, got, ("bwd", "bob"), heads=[0, 1], rows=rows, cols=cols)
    print(w.name, {k: f"{v:.2e}" for k, v in errs.items()})


@pytest.mark.parametrize("gproj", [0, 1])
def test_bench_workload_sampled(gproj):
    """The throughput workload itself (B4 H12 N8192 d64 bf16, the kernels and grids the
    bench times), sampled rows and late columns of the first and the last batch entry."""
    w = W.GPT2_N8192
    x = to_device(W.inputs(w), w)
    ops = ("bwd", "bob")
    got = run_ops(w, x, ops=ops, gproj=gproj)
    rows, cols = sample_rows_cols(w.N, np.random.default_rng(8192))
    for b in (0, w.B - 1):
        errs = sampled_check(w, got, ops, heads=[0, 11], rows=rows, cols=cols, batch=b)
        print(w.name, gproj, b, {k: f"{v:.2e}" for k, v in errs.items()})


def test_full_day_ragged_tail():
    """B2 H12 N23400 (N = 182 * 128 + 104): sampled rows (the whole ragged last tile of 104
    rows among them) and late columns of four heads in each batch entry (every slice has
    its own offset in the tensor maps)."""
    w = W.FULL_DAY
    x = to_device(W.inputs(w), w)
    got = run_ops(w, x, ops=("bwd",))
    rows, cols = sample_rows_cols(w.N, np.random.default_rng(3))
    rows = np.unique(np.concatenate([rows, np.arange(w.N - 104, w.N)]))
    for b, heads in ((0, [0, 3, 7, 11]), (1, [1, 5, 8, 11])):
        errs = sampled_check(w, got, ("bwd",), heads=heads, rows=rows, cols=cols, batch=b)
        print(w.name, b, heads, {k: f"{v:.2e}" for k, v in errs.items()})
    for k in ("O", "dQ", "dK", "dV"):
        assert not np.isnan(host(got[k])).any(), k


def test_large_key_gproj_reduces_dQ_error():
    """GProj page, "How the zero sum turns into a false gradient": large shared key
    mean + near-copy queries.  Reports the median per-row relative dQ error with and
    without GProj on batches 0-1 (16 slices) against the exact fp64 dQ, and beside
    them the cheaper fix the page compares against: subtracting the mean key of each
    slice before attention (softmax does not change when every key moves by the same
    vector, so the exact dQ is the same; the caller centres K and rounds it to bf16)."""
    import fwd_bwd_double_gb300 as fbd
    w = W.LARGE_KEY
    x = W.inputs(w)
    xd = to_device(x, w)
    O, lse = fbd.attn_fwd(xd["Q"], xd["K"], xd["V"], scale=w.scale)
    dQ0, dK0, dV0 = fbd.attn_bwd(xd["Q"], xd["K"], xd["V"], O, xd["dO"], lse, gproj=0, scale=w.scale)
    dQ1, dK1, dV1 = fbd.attn_bwd(xd["Q"], xd["K"], xd["V"], O, xd["dO"], lse, gproj=1, scale=w.scale)
    outs = {0: [host(t) for t in (dQ0, dK0, dV0)], 1: [host(t) for t in (dQ1, dK1, dV1)]}
    Kc = W.round_to_bf16((x["K"] - x["K"].astype(np.float64).mean(axis=2, keepdims=True)).astype(np.float32))
    xc = to_device({"K": Kc}, w)
    Oc, lsec = fbd.attn_fwd(xd["Q"], xc["K"], xd["V"], scale=w.scale)
    dQc, _, _ = fbd.attn_bwd(xd["Q"], xc["K"], xd["V"], Oc, xd["dO"], lsec, gproj=0, scale=w.scale)
    fbd.attn_device_status()
    dQc = host(dQc)
    e0, e1, ec, k0, k1, maxp = [], [], [], [], [], []
    acc = {(gp, k): ([], []) for gp in (0, 1) for k in ("dQ", "dK", "dV")}
    for b in range(2):
        for h in range(w.H):
            s = {k: x[k][b, h].astype(np.float64) for k in ("Q", "K", "V", "dO")}
            ref = oracle.backward(s["Q"], s["K"], s["V"], s["dO"], scale=w.scale)
            for gp in (0, 1):
                for k, o in zip(("dQ", "dK", "dV"), outs[gp]):
                    acc[gp, k][0].append(o[b, h])
                    acc[gp, k][1].append(ref[k])
            e0.append(row_rel_errors(outs[0][0][b, h], ref["dQ"]))
            e1.append(row_rel_errors(outs[1][0][b, h], ref["dQ"]))
            ec.append(row_rel_errors(dQc[b, h], ref["dQ"]))
            k0.append(row_rel_errors(outs[0][1][b, h], ref["dK"]))
            k1.append(row_rel_errors(outs[1][1][b, h], ref["dK"]))
            P, _ = oracle.softmax_rows(oracle.scores(s["Q"], s["K"], np.arange(256, 2048, 64), w.scale))
            maxp.append(P.max(axis=1))
    # Parity of every output, with and without GProj, against the exact fp64 backward.
    fro = {f"{k} gproj={gp}": rel_fro(np.stack(g), np.stack(r)) for (gp, k), (g, r) in acc.items()}
    m0, m1, mc, mk0, mk1 = (float(np.median(np.concatenate(e))) for e in (e0, e1, ec, k0, k1))
    print(f"{w.name}: median row dQ rel err no-GProj {m0:.4e}, GProj {m1:.4e}, mean-key subtraction {mc:.4e}; "
          f"median row dK rel err no-GProj {mk0:.4e}, GProj {mk1:.4e}; "
          f"median row max P {float(np.median(np.concatenate(maxp))):.3f}; rel-Frobenius "
          + ", ".join(f"{k} {v:.2e}" for k, v in fro.items()))
    assert all(v <= TOL["bf16"] for v in fro.values()), fro
    assert m1 < m0
    assert mc < m0


@pytest.mark.parametrize("d", [64, 128])
def test_bob_gproj_large_mean_b(d):
    """GProj page, "How the zero sum turns into a false gradient", carried to BoB.  A
    cotangent b = gdK with a large common mean (norm 40 per head, the size of the
    large-key workload's key mean) meets the bf16 row residual of dS in gQ's dS b
    product, and puts the per-row constant s q_i.mean(b) into G.  The exact BoB sees
    neither (every output is unchanged when one vector is added to every row of b).
    Median per-row errors against the exact fp64 result, with and without GProj, next
    to the same inputs without the mean."""
    import fwd_bwd_double_gb300 as fbd
    w = W.Workload(f"bob_meanb_B1H4N1024d{d}_bf16", 1, 4, 1024, d, "bf16")
    x = dict(W.inputs(w))
    g = np.random.default_rng(40).standard_normal((w.H, w.d))
    m = 40.0 * g / np.linalg.norm(g, axis=1, keepdims=True)
    bm = W.round_to_bf16((x["gdK"].astype(np.float64) + m[None, :, None, :]).astype(np.float32))
    xd = to_device(x, w)
    bmd = to_device({"gdK": bm}, w)["gdK"]
    O, lse = fbd.attn_fwd(xd["Q"], xd["K"], xd["V"])
    got = {}
    for gp in (0, 1):
        for name, bb in (("b", xd["gdK"]), ("b+m", bmd)):
            got[gp, name] = [host(t) for t in fbd.attn_bob(xd["Q"], xd["K"], xd["V"], O, xd["dO"], lse,
                                                           xd["gdQ"], bb, xd["gdV"], gproj=gp)]
    fbd.attn_device_status()
    ref = {"b": oracle.bob_all(x["Q"], x["K"], x["V"], x["dO"], x["gdQ"], x["gdK"], x["gdV"]),
           "b+m": oracle.bob_all(x["Q"], x["K"], x["V"], x["dO"], x["gdQ"], bm, x["gdV"])}
    med = {}
    for (gp, name), outs in got.items():
        for k, o in zip(("gQ", "gK", "gV", "gdO"), outs):
            med[gp, name, k] = float(np.median(row_rel_errors(o, ref[name][k])))
            assert rel_fro(o, ref[name][k]) <= TOL["bf16"], (gp, name, k)
    print(w.name, {f"{k[2]} gproj={k[0]} {k[1]}": f"{v:.2e}" for k, v in sorted(med.items())})
    # GProj removes most of what the mean adds to the gQ error ...
    assert med[1, "b+m", "gQ"] < 0.8 * med[0, "b+m", "gQ"]
    assert med[1, "b+m", "gQ"] < 1.5 * med[1, "b", "gQ"]
    # ... and the row pass's per-row shift of G keeps gdO at its level without the mean.
    for gp in (0, 1):
        assert med[gp, "b+m", "gdO"] < 1.5 * med[gp, "b", "gdO"]


def test_large_key_projected_rows_sum_to_zero():
    """The projected dS rows fed to the products sum to zero within 1e-6 of their L1 norm."""
    import fwd_bwd_double_gb300 as fbd
    w = W.LARGE_KEY
    x = W.inputs(w, batches=[0], heads=[0, 5])
    xd = to_device(x, w)
    O, lse = fbd.attn_fwd(xd["Q"], xd["K"], xd["V"], scale=w.scale)
    dS = host(fbd.attn_bwd_projected_dS(xd["Q"], xd["K"], xd["V"], O, xd["dO"], lse, scale=w.scale))
    rs = np.abs(dS.sum(axis=-1))
    l1 = np.abs(dS).sum(axis=-1)
    keep = l1 > 0
    worst = float(np.max(rs[keep] / l1[keep]))
    print(f"{w.name}: max |row sum| / L1 of projected dS = {worst:.3e}")
    assert worst <= 1e-6
    assert np.all(np.triu(dS[0, 0], 1) == 0)


def test_projected_dS_with_window():
    """The diagnostic under a sliding window: keys outside i - W < j <= i are 0 and the
    projected rows still sum to zero."""
    import fwd_bwd_double_gb300 as fbd
    w = W.Workload("projected_window_B1H2N300d64", 1, 2, 300, 64, "bf16")
    xd = to_device(inputs(w), w)
    O, lse = fbd.attn_fwd(xd["Q"], xd["K"], xd["V"], window=40)
    dS = host(fbd.attn_bwd_projected_dS(xd["Q"], xd["K"], xd["V"], O, xd["dO"], lse, window=40))
    i, j = np.meshgrid(np.arange(300), np.arange(300), indexing="ij")
    assert np.all(dS[:, :, (j > i) | (j <= i - 40)] == 0)
    l1 = np.abs(dS).sum(axis=-1)
    keep = l1 > 0
    assert float(np.max(np.abs(dS.sum(axis=-1))[keep] / l1[keep])) <= 1e-6


EDGE_N = [1, 2, 15, 17, 127, 128, 129, 255, 300]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N", EDGE_N)
def test_edge_sizes(N, d, dtype):
    w = W.Workload(f"edge_B1H2N{N}d{d}_{dtype}", 1, 2, N, d, dtype)
    got = run_ops(w, to_device(inputs(w), w), ops=("bwd", "bob"))
    check_full(w, got, ("bwd", "bob"))


# Head dims 32, 96 and 256 (every op, both dtypes, causal or not, grouped heads, a
# ragged N spanning several tiles) and bf16 BoB at d = 128.
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("d", [32, 96, 256])
@pytest.mark.parametrize("N", [1, 17, 300])
def test_other_head_dims(N, d, dtype, causal):
    w = W.Workload(f"headdim_B1H2N{N}d{d}_{dtype}", 1, 2, N, d, dtype)
    got = run_ops(w, to_device(inputs(w), w), ops=("bwd", "bob"), causal=causal)
    check_full(w, got, ("bwd", "bob"), causal=causal)
    if dtype == "bf16":
        got1 = run_ops(w, to_device(inputs(w), w), ops=("bwd", "bob"), gproj=1, causal=causal)
        check_full(w, got1, ("bwd", "bob"), causal=causal)


@pytest.mark.parametrize("d", [96, 128, 256])
def test_f32_wide_heads(d):
    """float32 past d = 64 on the tf32 tensor-core kernels: the head dim in chunks of 64
    (the last 32 wide at d = 96), the output columns split over CTAs in parts of 64;
    several row blocks, a ragged tail, grouped heads, causal and not, and a window."""
    w = W.Workload(f"f32wide_B1H4g2N700d{d}_f32", 1, 4, 700, d, "f32", group=2)
    x = to_device(inputs(w), w)
    for causal, win in ((True, 0), (False, 0), (True, 90)):
        got = run_ops(w, x, ops=("bwd", "bob"), causal=causal, window=win)
        errs = check_full(w, got, ("bwd", "bob"), causal=causal, window=win)
        print(w.name, causal, win, {k: f"{v:.2e}" for k, v in errs.items()})


@pytest.mark.parametrize("gproj", [0, 1])
@pytest.mark.parametrize("d", [32, 96, 128, 256])
def test_other_head_dims_grouped_bf16(d, gproj):
    w = W.Workload(f"headdim_gqa_B2H4g2N200d{d}_bf16", 2, 4, 200, d, "bf16", group=2)
    got = run_ops(w, to_device(inputs(w), w), ops=("bwd", "bob"), gproj=gproj)
    check_full(w, got, ("bwd", "bob"))


@pytest.mark.parametrize("d,win", [(64, 0), (64, 70), (128, 0), (128, 70)])
def test_outputs_written_once_and_nothing_outside(d, win):
    """Outputs live inside NaN-filled guard buffers: every output element is written
    (no NaN left) and no guard element is touched (with and without a window)."""
    import torch

    import fwd_bwd_double_gb300 as fbd
    w = W.Workload(f"guard_B1H3N200d{d}", 1, 3, 200, d, "bf16")
    xd = to_device(inputs(w), w)
    n = xd["Q"].numel()
    pad = 4096

    def guarded():
        buf = torch.full((n + 2 * pad,), float("nan"), dtype=torch.bfloat16, device="cuda")
        return buf, buf[pad:pad + n].view_as(xd["Q"])

    def lse_guarded():
        buf = torch.full((3 * 200 + 2 * pad,), float("nan"), dtype=torch.float32, device="cuda")
        return buf, buf[pad:pad + 600].view(1, 3, 200)

    bufs = {k: guarded() for k in ("O", "dQ", "dK", "dV", "gQ", "gK", "gV", "gdO")}
    lb, lse = lse_guarded()
    O = bufs["O"][1]
    fbd.attn_fwd(xd["Q"], xd["K"], xd["V"], O=O, lse=lse, window=win)
    fbd.attn_bwd(xd["Q"], xd["K"], xd["V"], O, xd["dO"], lse, gproj=1, dQ=bufs["dQ"][1], dK=bufs["dK"][1],
                 dV=bufs["dV"][1], window=win)
    fbd.attn_bob(xd["Q"], xd["K"], xd["V"], O, xd["dO"], lse, xd["gdQ"], xd["gdK"], xd["gdV"], gQ=bufs["gQ"][1],
                 gK=bufs["gK"][1], gV=bufs["gV"][1], gdO=bufs["gdO"][1], window=win, gproj=1)
    fbd.attn_device_status()
    for k, (buf, view) in list(bufs.items()) + [("lse", (lb, lse))]:
        b = buf.float().cpu().numpy()
        assert np.isnan(b[:pad]).all() and np.isnan(b[-pad:]).all(), f"{k}: guard touched"
        assert not np.isnan(view.float().cpu().numpy()).any(), f"{k}: element not written"


@pytest.mark.parametrize("gproj", [0, 1])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_separate_passes_equal_the_fused_call(dtype, gproj):
    """attn_*_passes(ROW) then attn_*_passes(COL) is exactly attn_bwd / attn_bob."""
    import fwd_bwd_double_gb300 as fbd
    w = W.Workload(f"passes_B2H3N300d64_{dtype}", 2, 3, 300, 64, dtype)
    x = to_device(inputs(w), w)
    O, lse = fbd.attn_fwd(x["Q"], x["K"], x["V"])
    ref_b = fbd.attn_bwd(x["Q"], x["K"], x["V"], O, x["dO"], lse, gproj=1)
    ref_g = fbd.attn_bob(x["Q"], x["K"], x["V"], O, x["dO"], lse, x["gdQ"], x["gdK"], x["gdV"], gproj=gproj)
    import torch
    outs = [torch.empty_like(x["Q"]) for _ in range(3)]
    desc = fbd.make_desc(x["Q"])
    nbytes = max(fbd.attn_bwd_workspace_bytes(desc, 1), fbd.attn_bob_workspace_bytes(desc, gproj))
    ws = torch.full((nbytes // 4,), float("nan"), dtype=torch.float32, device="cuda")
    for ps in (fbd.ATTN_ROW_PASS, fbd.ATTN_COL_PASS):
        fbd.attn_bwd_passes(x["Q"], x["K"], x["V"], O, x["dO"], lse, ps, gproj=1, dQ=outs[0], dK=outs[1],
                            dV=outs[2], workspace=ws)
    gouts = [torch.empty_like(x["Q"]) for _ in range(4)]
    for ps in (fbd.ATTN_ROW_PASS, fbd.ATTN_COL_PASS):
        fbd.attn_bob_passes(x["Q"], x["K"], x["V"], O, x["dO"], lse, x["gdQ"], x["gdK"], x["gdV"], ps,
                            gQ=gouts[0], gK=gouts[1], gV=gouts[2], gdO=gouts[3], workspace=ws, gproj=gproj)
    fbd.attn_device_status()
    for a, b in zip(outs + gouts, list(ref_b) + list(ref_g)):
        assert torch.equal(a, b)


def test_deterministic():
    """Every output is the same bits on every run, except the dQ of the single-pass bf16
    backward (d <= 64, no GProj), whose fp32 accumulator adds the key blocks' partial
    sums in the order they arrive: that one is the same up to that order.  With GProj
    (two passes) dQ is the same bits too."""
    w = W.GPT2_LAYER.with_n(512)
    xd = to_device(inputs(w), w)
    a = run_ops(w, xd)
    b = run_ops(w, xd)
    for k in a:
        if k == "dQ":
            assert_same_up_to_sum_order(a[k], b[k], k)
        else:
            assert np.array_equal(host(a[k]), host(b[k])), k
    a1 = run_ops(w, xd, ops=("bwd",), gproj=1)
    b1 = run_ops(w, xd, ops=("bwd",), gproj=1)
    for k in ("dQ", "dK", "dV"):
        assert np.array_equal(host(a1[k]), host(b1[k])), k


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("N", [17, 129, 255])
def test_result_does_not_depend_on_workspace_content(N, dtype):
    """An odd N leaves one padding row in each slice of the row-state workspace; the
    column pass reads it (with P = 0 there).  A workspace full of NaN must give the
    same bits as a zeroed one, for the backward with and without GProj and for BoB."""
    import torch

    import fwd_bwd_double_gb300 as fbd
    w = W.Workload(f"wsfill_B2H3N{N}d64_{dtype}", 2, 3, N, 64, dtype)
    x = to_device(inputs(w), w)
    O, lse = fbd.attn_fwd(x["Q"], x["K"], x["V"])
    nbytes = max(fbd.attn_bwd_workspace_bytes(fbd.make_desc(x["Q"]), 0), fbd.attn_bwd_workspace_bytes(fbd.make_desc(x["Q"]), 1),
                 fbd.attn_bob_workspace_bytes(fbd.make_desc(x["Q"])))

    def run(fill):
        ws = torch.full((nbytes // 4,), fill, dtype=torch.float32, device="cuda").view(torch.uint8)
        outs = list(fbd.attn_bwd(x["Q"], x["K"], x["V"], O, x["dO"], lse, gproj=0, workspace=ws))
        outs += list(fbd.attn_bwd(x["Q"], x["K"], x["V"], O, x["dO"], lse, gproj=1, workspace=ws))
        outs += list(fbd.attn_bob(x["Q"], x["K"], x["V"], O, x["dO"], lse, x["gdQ"], x["gdK"], x["gdV"], workspace=ws))
        fbd.attn_device_status()
        return outs

    for n, (a, b) in enumerate(zip(run(0.0), run(float("nan")))):
        assert not torch.isnan(b).any()
        if n == 0 and dtype == "bf16":  # single-pass dQ: the same up to its summation order
            assert_same_up_to_sum_order(a, b, "dQ")
        else:
            assert torch.equal(a, b)



# ---------------------------------------------------------------- non-causal
# Every key visible to every query: the same kernels with the causal mask off (only
# keys past N masked), against the oracle's non-causal mode.

def test_noncausal_tiny_f32_all_ops():
    w = W.Workload("noncausal_tiny_f32_B1H1N256d64", 1, 1, 256, 64, "f32")
    got = run_ops(w, to_device(inputs(w), w), causal=False)
    errs = check_full(w, got, ("bwd", "bob"), causal=False)
    print(w.name, {k: f"{v:.2e}" for k, v in errs.items()})


@pytest.mark.parametrize("gproj", [0, 1])
def test_noncausal_gpt2_layer_bf16(gproj):
    w = W.Workload("noncausal_gpt2small_B4H12N1024d64", 4, 12, 1024, 64, "bf16")
    ops = ("bwd", "bob")
    got = run_ops(w, to_device(inputs(w), w), ops=ops, gproj=gproj, causal=False)
    errs = check_full(w, got, ops, causal=False)
    print(w.name, gproj, {k: f"{v:.2e}" for k, v in errs.items()})


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N", [1, 17, 129, 300])
def test_noncausal_edge_sizes(N, d, dtype):
    w = W.Workload(f"noncausal_edge_B1H2N{N}d{d}_{dtype}", 1, 2, N, d, dtype)
    ops = ("bwd", "bob")
    got = run_ops(w, to_device(inputs(w), w), ops=ops, causal=False)
    check_full(w, got, ops, causal=False)
    if dtype == "bf16":
        got1 = run_ops(w, to_device(inputs(w), w), ops=("bwd",), gproj=1, causal=False)
        check_full(w, got1, ("bwd",), causal=False)


def test_noncausal_differs_from_causal_and_passes_compose():
    """The mask flag reaches the kernels (the outputs differ), and the separate row and
    column passes give the one-call results without the causal mask too (dQ up to the
    summation order of the single-pass backward)."""
    import torch

    import fwd_bwd_double_gb300 as fbd
    w = W.Workload("noncausal_passes_B2H3N300d64_bf16", 2, 3, 300, 64, "bf16")
    x = to_device(inputs(w), w)
    O, lse = fbd.attn_fwd(x["Q"], x["K"], x["V"], causal=False)
    Oc, _ = fbd.attn_fwd(x["Q"], x["K"], x["V"], causal=True)
    assert not torch.equal(O[:, :, :-1], Oc[:, :, :-1])
    ref_b = fbd.attn_bwd(x["Q"], x["K"], x["V"], O, x["dO"], lse, causal=False)
    ref_g = fbd.attn_bob(x["Q"], x["K"], x["V"], O, x["dO"], lse, x["gdQ"], x["gdK"], x["gdV"], causal=False)
    outs = [torch.empty_like(x["Q"]) for _ in range(3)]
    ws = torch.full((fbd.attn_bwd_workspace_bytes(fbd.make_desc(x["Q"]), 0) // 4,), float("nan"),
                    dtype=torch.float32, device="cuda").view(torch.uint8)
    for ps in (fbd.ATTN_ROW_PASS, fbd.ATTN_COL_PASS):
        fbd.attn_bwd_passes(x["Q"], x["K"], x["V"], O, x["dO"], lse, ps, dQ=outs[0], dK=outs[1], dV=outs[2],
                            workspace=ws, causal=False)
    gouts = [torch.empty_like(x["Q"]) for _ in range(4)]
    for ps in (fbd.ATTN_ROW_PASS, fbd.ATTN_COL_PASS):
        fbd.attn_bob_passes(x["Q"], x["K"], x["V"], O, x["dO"], lse, x["gdQ"], x["gdK"], x["gdV"], ps,
                            gQ=gouts[0], gK=gouts[1], gV=gouts[2], gdO=gouts[3], workspace=ws, causal=False)
    fbd.attn_device_status()
    # The backward's two separate passes against the single-pass form of attn_bwd: dQ is
    # summed in another order and dK's product reads dS from shared memory instead of TMEM,
    # so they agree up to the order of the fp32 roundings; the BoB outputs are the same bits.
    for n, k in enumerate(("dQ", "dK", "dV")):
        assert_same_up_to_sum_order(outs[n], ref_b[n], k)
    for a, b in zip(gouts, list(ref_g)):
        assert torch.equal(a, b)


# ------------------------------------------------------ grouped key/value heads
# g query heads share one key/value head: K, V, gdK, gdV (and dK, dV, gK, gV) have
# H / g heads.  Checked against the oracle's grouped mode, and bit for bit against
# plain multi-head attention on repeated K, V where the arithmetic is the same.

@pytest.mark.parametrize("causal", [True, False])
def test_gqa_tiny_f32_all_ops(causal):
    w = W.Workload("gqa_tiny_f32_B1H4g2N256d64", 1, 4, 256, 64, "f32", group=2)
    got = run_ops(w, to_device(inputs(w), w), causal=causal)
    errs = check_full(w, got, ("bwd", "bob"), causal=causal)
    print(w.name, causal, {k: f"{v:.2e}" for k, v in errs.items()})


@pytest.mark.parametrize("group,gproj", [(3, 0), (3, 1), (12, 0)])
def test_gqa_gpt2_layer_bf16(group, gproj):
    """GPT-2 small layer shape with 4 key/value heads (g = 3) and multi-query (g = 12)."""
    w = W.Workload(f"gqa_gpt2small_B2H12g{group}N1024d64", 2, 12, 1024, 64, "bf16", group=group)
    ops = ("bwd", "bob")
    got = run_ops(w, to_device(inputs(w), w), ops=ops, gproj=gproj)
    errs = check_full(w, got, ops)
    print(w.name, gproj, {k: f"{v:.2e}" for k, v in errs.items()})


@pytest.mark.parametrize("N", [1, 17, 129, 300])
@pytest.mark.parametrize("d,dtype", [(64, "bf16"), (128, "bf16"), (64, "f32")])
@pytest.mark.parametrize("causal", [True, False])
def test_gqa_edge_sizes(N, d, dtype, causal):
    w = W.Workload(f"gqa_edge_B2H4g2N{N}d{d}_{dtype}", 2, 4, N, d, dtype, group=2)
    ops = ("bwd", "bob")
    got = run_ops(w, to_device(inputs(w), w), ops=ops, causal=causal)
    check_full(w, got, ops, causal=causal)
    if dtype == "bf16":
        got1 = run_ops(w, to_device(inputs(w), w), ops=("bwd", "bob"), gproj=1, causal=causal)
        check_full(w, got1, ("bwd", "bob"), causal=causal)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_gqa_row_outputs_equal_repeated_heads_bitwise(dtype):
    """O, lse, dQ, gQ and gdO of a query head depend on its own key/value head only, and
    the kernels do the same arithmetic whether that head is shared or repeated: the bits
    must match.  dK, dV, gK, gV are sums over the group (checked against the oracle)."""
    import torch
    import fwd_bwd_double_gb300 as fbd
    w = W.Workload(f"gqa_bits_B2H6g3N300d64_{dtype}", 2, 6, 300, 64, dtype, group=3)
    x = to_device(inputs(w), w)
    rep = {k: (v.repeat_interleave(3, dim=1).contiguous() if k in W.KV_TENSORS else v) for k, v in x.items()}
    for causal in (True, False):
        O, lse = fbd.attn_fwd(x["Q"], x["K"], x["V"], causal=causal)
        Or, lser = fbd.attn_fwd(rep["Q"], rep["K"], rep["V"], causal=causal)
        assert torch.equal(O, Or) and torch.equal(lse, lser)
        dQ, dK, dV = fbd.attn_bwd(x["Q"], x["K"], x["V"], O, x["dO"], lse, causal=causal)
        dQr, dKr, dVr = fbd.attn_bwd(rep["Q"], rep["K"], rep["V"], O, x["dO"], lse, causal=causal)
        if dtype == "bf16":  # the single-pass accumulator: the same up to its summation order
            assert_same_up_to_sum_order(dQ, dQr, "dQ")
        else:
            assert torch.equal(dQ, dQr)
        assert dK.shape == x["K"].shape
        g = fbd.attn_bob(x["Q"], x["K"], x["V"], O, x["dO"], lse, x["gdQ"], x["gdK"], x["gdV"], causal=causal)
        gr = fbd.attn_bob(rep["Q"], rep["K"], rep["V"], O, x["dO"], lse, x["gdQ"], rep["gdK"], rep["gdV"],
                          causal=causal)
        assert torch.equal(g[0], gr[0]) and torch.equal(g[3], gr[3])
        # The group sum of the repeated heads' key-side gradients is the same quantity.
        tol = TOL[dtype] if dtype == "bf16" else 1e-5
        for a, b in ((dK, dKr), (dV, dVr), (g[1], gr[1]), (g[2], gr[2])):
            s = host(b).reshape(2, 2, 3, 300, 64).sum(axis=2)
            assert rel_fro(host(a), s) <= tol
    fbd.attn_device_status()


# ------------------------------------------------------- BoB at head dim 128
# The tensor-core BoB at d = 128 runs each block of rows (keys) as two CTAs, one per
# output half; both halves and the row states written by half 0 are checked here.

@pytest.mark.parametrize("gproj", [0, 1])
@pytest.mark.parametrize("causal", [True, False])
def test_bob_head_dim_128_bf16(causal, gproj):
    w = W.Workload("bob_d128_B2H4N1000d128_bf16", 2, 4, 1000, 128, "bf16")
    got = run_ops(w, to_device(inputs(w), w), ops=("bob",), causal=causal, gproj=gproj)
    errs = check_full(w, got, ("bob",), causal=causal)
    print(w.name, causal, gproj, {k: f"{v:.2e}" for k, v in errs.items()})


@pytest.mark.parametrize("gproj", [0, 1])
def test_bob_head_dim_128_passes_compose_on_nan_workspace(gproj):
    import torch
    import fwd_bwd_double_gb300 as fbd
    w = W.Workload("bob_d128_passes_B1H3N300d128_bf16", 1, 3, 300, 128, "bf16")
    x = to_device(inputs(w), w)
    O, lse = fbd.attn_fwd(x["Q"], x["K"], x["V"])
    ref = fbd.attn_bob(x["Q"], x["K"], x["V"], O, x["dO"], lse, x["gdQ"], x["gdK"], x["gdV"], gproj=gproj)
    nbytes = fbd.attn_bob_workspace_bytes(fbd.make_desc(x["Q"]), gproj)
    ws = torch.full((nbytes // 4,), float("nan"), device="cuda")
    outs = [torch.full_like(x["Q"], float("nan")) for _ in range(4)]
    for ps in (fbd.ATTN_ROW_PASS, fbd.ATTN_COL_PASS):
        fbd.attn_bob_passes(x["Q"], x["K"], x["V"], O, x["dO"], lse, x["gdQ"], x["gdK"], x["gdV"], ps,
                            gQ=outs[0], gK=outs[1], gV=outs[2], gdO=outs[3], workspace=ws, gproj=gproj)
    fbd.attn_device_status()
    for a, b in zip(outs, ref):
        assert torch.equal(a, b)


# Head dims 32 and 96 on the tensor-core kernels of d = 64 and 128, the head dim
# zero-padded in shared memory: several row and key blocks and a ragged tail.
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("d", [32, 96])
def test_padded_head_dims_bf16(d, causal):
    w = W.Workload(f"padded_B2H4N1000d{d}_bf16", 2, 4, 1000, d, "bf16")
    got = run_ops(w, to_device(inputs(w), w), ops=("bwd", "bob"), causal=causal)
    errs = check_full(w, got, ("bwd", "bob"), causal=causal)
    got1 = run_ops(w, to_device(inputs(w), w), ops=("bwd", "bob"), gproj=1, causal=causal)
    errs1 = check_full(w, got1, ("bwd", "bob"), causal=causal)
    print(w.name, causal, {k: f"{v:.2e}" for k, v in errs.items()}, "gproj", {k: f"{v:.2e}" for k, v in errs1.items()})


# --------------------------------------------------------- causal sliding window ----
# Key j visible to query i iff i - win < j <= i (desc->window).  The windows cover less
# than one 64-key block (1, 17), one block (64, 128), between blocks (100, 200) and past
# N (the causal mask); N = 1000 spans several row and key blocks and a ragged tail.

@pytest.mark.parametrize("win", [1, 17, 64, 100, 128, 200, 5000])
@pytest.mark.parametrize("d,dtype", [(64, "bf16"), (128, "bf16"), (64, "f32")])
def test_window_all_ops(win, d, dtype):
    w = W.Workload(f"window_B1H3N1000d{d}_{dtype}", 1, 3, 1000, d, dtype)
    got = run_ops(w, to_device(inputs(w), w), ops=("bwd", "bob"), window=win)
    if win == 1:
        # Each row sees only its own key: P = I, so dQ, dK, gQ, gK, gV are exactly 0 and
        # O = V, dV = dO, gdO = gdV (the oracle's pinned closed forms).  The zeros are
        # checked against the scale of the outputs that are not zero.
        x = inputs(w)
        for k, want in (("O", x["V"]), ("dV", x["dO"]), ("gdO", x["gdV"])):
            assert rel_fro(host(got[k]), want) <= TOL[w.dtype], k
        scale = float(np.abs(x["dO"]).max())
        for k in ("dQ", "dK", "gQ", "gK", "gV"):
            assert float(np.abs(host(got[k])).max()) <= TOL[w.dtype] * scale, k
        return
    errs = check_full(w, got, ("bwd", "bob"), window=win)
    print(w.name, win, {k: f"{v:.2e}" for k, v in errs.items()})


@pytest.mark.parametrize("win", [33, 130])
@pytest.mark.parametrize("d", [32, 96, 256])
def test_window_other_head_dims_bf16(d, win):
    w = W.Workload(f"window_B1H2N600d{d}_bf16", 1, 2, 600, d, "bf16")
    for gp in (0, 1):
        got = run_ops(w, to_device(inputs(w), w), ops=("bwd", "bob"), gproj=gp, window=win)
        check_full(w, got, ("bwd", "bob"), window=win)


@pytest.mark.parametrize("d", [64, 128])
def test_window_gproj_and_grouped_heads(d):
    w = W.Workload(f"window_gqa_B2H6g3N700d{d}_bf16", 2, 6, 700, d, "bf16", group=3)
    for gp in (0, 1):
        got = run_ops(w, to_device(inputs(w), w), ops=("bwd", "bob"), gproj=gp, window=150)
        errs = check_full(w, got, ("bwd", "bob"), window=150)
        print(w.name, gp, {k: f"{v:.2e}" for k, v in errs.items()})


@pytest.mark.parametrize("d", [64, 128])
def test_window_passes_compose_on_nan_workspace(d):
    import torch
    import fwd_bwd_double_gb300 as fbd
    w = W.Workload(f"window_passes_B1H3N300d{d}_bf16", 1, 3, 300, d, "bf16")
    x = to_device(inputs(w), w)
    O, lse = fbd.attn_fwd(x["Q"], x["K"], x["V"], window=70)
    for gp in (0, 1):
        ref_b = fbd.attn_bwd(x["Q"], x["K"], x["V"], O, x["dO"], lse, gproj=gp, window=70)
        ref_g = fbd.attn_bob(x["Q"], x["K"], x["V"], O, x["dO"], lse, x["gdQ"], x["gdK"], x["gdV"], window=70,
                             gproj=gp)
        desc = fbd.make_desc(x["Q"], window=70)
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


# The forward at d = 256 runs on tensor cores with 64-key blocks: several row blocks, the
# two-block diagonal of a 128-row block, ragged tails, causal and not, a window.
@pytest.mark.parametrize("N,causal,win", [(1000, True, 0), (2500, True, 0), (1000, False, 0), (1000, True, 200)])
def test_forward_head_dim_256_bf16(N, causal, win):
    import fwd_bwd_double_gb300 as fbd
    w = W.Workload(f"fwd256_B1H3N{N}d256_bf16", 1, 3, N, 256, "bf16")
    xd = to_device(inputs(w), w)
    O, lse = fbd.attn_fwd(xd["Q"], xd["K"], xd["V"], causal=causal, window=win)
    fbd.attn_device_status()
    mask = oracle.Window(win) if win else causal
    x = inputs(w)
    ref = oracle.forward_all(x["Q"], x["K"], x["V"], causal=mask)
    assert rel_fro(host(O), ref["O"]) <= TOL["bf16"] and rel_fro(host(lse), ref["L"]) <= 1e-5


@pytest.mark.parametrize("win", [1024, 4000])
def test_window_long_sampled(win):
    """A window at the bench's sequence length (B1 H2 N8192 d64 bf16), sampled rows and
    late columns of every output against the oracle under the same window."""
    w = W.Workload(f"window_long_B1H2N8192d64_bf16", 1, 2, 8192, 64, "bf16")
    got = run_ops(w, to_device(W.inputs(w), w), ops=("bwd", "bob"), window=win)
    rows, cols = sample_rows_cols(w.N, np.random.default_rng(win))
    errs = sampled_check(w, got, ("bwd", "bob"), heads=[0, 1], rows=rows, cols=cols, causal=oracle.Window(win))
    print(w.name, win, {k: f"{v:.2e}" for k, v in errs.items()})


# The backward at d = 256 on tensor cores (without GProj): a row pass with one stage of
# 64-key tiles, a column pass split over two CTAs by output half.  Several row and key
# blocks, a ragged tail, causal and not, grouped heads, a window.
@pytest.mark.parametrize("causal,win,group", [(True, 0, 1), (False, 0, 1), (True, 300, 1), (True, 0, 3)])
def test_backward_head_dim_256_tensor_cores(causal, win, group):
    w = W.Workload(f"bwd256_B1H3N1000d256_g{group}_bf16", 1, 3, 1000, 256, "bf16", group=group)
    got = run_ops(w, to_device(inputs(w), w), ops=("bwd",), causal=causal, window=win)
    errs = check_full(w, got, ("bwd",), causal=causal, window=win)
    print(w.name, causal, win, {k: f"{v:.2e}" for k, v in errs.items()})
