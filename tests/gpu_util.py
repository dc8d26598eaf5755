"""Helpers shared by the GPU parity tests: device tensors from the seeded workloads,
oracle results per slice (cached), and the error measures the tolerances use."""
from __future__ import annotations

import functools

import numpy as np

import oracle
import workloads as W


def torch_dtype(w):
    import torch
    return torch.float32 if w.dtype == "f32" else torch.bfloat16


def to_device(x: dict, w, names=None):
    import torch
    names = names or list(x)
    return {k: torch.from_numpy(np.ascontiguousarray(x[k])).to("cuda").to(torch_dtype(w)).contiguous()
            for k in names}


def host(t) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def rel_fro(got, ref) -> float:
    got, ref = np.asarray(got, np.float64), np.asarray(ref, np.float64)
    n = np.linalg.norm(ref)
    return float(np.linalg.norm(got - ref) / (n if n > 0 else 1.0))


def row_rel_errors(got, ref):
    """Per-row relative errors ||got_i - ref_i|| / ||ref_i|| over rows with ||ref_i|| > 0."""
    got = np.asarray(got, np.float64).reshape(-1, got.shape[-1])
    ref = np.asarray(ref, np.float64).reshape(-1, ref.shape[-1])
    nr = np.linalg.norm(ref, axis=1)
    keep = nr > 0
    return np.linalg.norm(got - ref, axis=1)[keep] / nr[keep]


@functools.lru_cache(maxsize=8)
def inputs(w):
    return W.inputs(w)


@functools.lru_cache(maxsize=8)
def oracle_full(w, op, causal=True):
    """Oracle outputs [B, H, ...] for every slice of workload w (op: fwd, bwd, bob)."""
    x = inputs(w)
    g = w.group
    if op == "fwd":
        return oracle.forward_all(x["Q"], x["K"], x["V"], scale=w.scale, causal=causal, groups=g)
    if op == "bwd":
        return oracle.backward_all(x["Q"], x["K"], x["V"], x["dO"], scale=w.scale, causal=causal, groups=g)
    return oracle.bob_all(x["Q"], x["K"], x["V"], x["dO"], x["gdQ"], x["gdK"], x["gdV"], scale=w.scale,
                          causal=causal, groups=g)


def run_ops(w, x_dev, ops=("fwd", "bwd", "bob"), gproj=0, causal=True, window=0):
    """Run the requested ops through the binding (gproj for the backward and the BoB;
    window: the causal sliding window, 0 for none)."""
    import fwd_bwd_double_gb300 as fbd
    out = {}
    O, lse = fbd.attn_fwd(x_dev["Q"], x_dev["K"], x_dev["V"], scale=w.scale, causal=causal, window=window)
    out["O"], out["L"] = O, lse
    if "bwd" in ops:
        out["dQ"], out["dK"], out["dV"] = fbd.attn_bwd(x_dev["Q"], x_dev["K"], x_dev["V"], O, x_dev["dO"], lse,
                                                       gproj=gproj, scale=w.scale, causal=causal, window=window)
    if "bob" in ops:
        out["gQ"], out["gK"], out["gV"], out["gdO"] = fbd.attn_bob(
            x_dev["Q"], x_dev["K"], x_dev["V"], O, x_dev["dO"], lse, x_dev["gdQ"], x_dev["gdK"], x_dev["gdV"],
            scale=w.scale, causal=causal, window=window, gproj=gproj)
    fbd.attn_device_status()
    return out


def check_tol_fwd(w, O, L, causal=True, tol=2e-2):
    """Forward outputs against the oracle within the bf16 tolerance."""
    f = oracle_full(w, "fwd", causal)
    assert rel_fro(O, f["O"]) <= tol and rel_fro(L, f["L"]) <= tol


def assert_same_up_to_sum_order(a, b, what=""):
    """Two bf16 results that differ only in the order of their fp32 roundings (the
    single-pass backward's dQ accumulator adds the key blocks' partial sums in the order
    they arrive; its dK product reads dS from shared memory where the two-pass column pass
    reads it from TMEM): elementwise within two bf16 steps of the larger magnitude (plus a
    floor of 1e-6 of the largest element) and within 1e-3 in relative Frobenius norm."""
    a, b = host(a) if not isinstance(a, np.ndarray) else a, host(b) if not isinstance(b, np.ndarray) else b
    scale = max(float(np.abs(b).max()), 1e-30)
    bound = 2.0 ** -7 * np.maximum(np.abs(a), np.abs(b)) + 1e-6 * scale
    assert np.all(np.abs(a - b) <= bound), what
    assert rel_fro(a, b) <= 1e-3, what
