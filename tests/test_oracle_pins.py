"""Pins for the CPU fp64 oracle, against facts that do not come from the oracle itself.

Each pin names the page passage (or the mathematical fact) it rests on:
  * brute-force loops over the definition (Flash attention page, "Why attention is
    memory-bound": softmax(QK^T/sqrt(d)) V);
  * online softmax = two-pass softmax in exact arithmetic (same page, "Online softmax
    recurrence");
  * probability rows sum to one; a per-row constant in S changes nothing;
  * exact dS rows sum to zero and dQ ignores a common shift of all keys (GProj page,
    "How the zero sum turns into a false gradient"); every BoB output ignores a
    common shift of the keys and of the cotangent b; the GProj projection of BoB's
    rounded dS sums to zero and makes gQ ignore a shift of b, which the unprojected
    residual turns into exactly s r_i v;
  * central finite differences of the forward (first backward) and of the first
    backward (second backward, a Hessian-vector product), and of O along the
    cotangent direction (gdO is that directional derivative);
  * symbolic differentiation (sympy) and fp64 autograd on tiny cases, both of
    which know nothing of the hand-derived closed form;
  * closed-form special cases (N = 1; Q = 0 gives uniform causal attention);
  * the non-causal mode (every key visible) against the same kinds of pins:
    brute force, online = two-pass, finite differences, the Hessian-vector
    product, the forward JVP, the streaming passes and fp64 autograd;
  * the streaming row/column-pass form of BoB (FlashBoB page, "Two scalar states
    replace quadratic tensors") equals the closed form.
A final group plants mistakes in the oracle and checks that these pins catch them.
"""
import math

import numpy as np
import pytest

import oracle
from oracle import attention as A


def rel(x, y):
    x, y = np.asarray(x, np.float64), np.asarray(y, np.float64)
    n = np.linalg.norm(y)
    return np.linalg.norm(x - y) / (n if n > 0 else 1.0)


def rnd(seed, *shape):
    return np.random.default_rng(seed).standard_normal(shape)


def slice_set(N, d, seed=0):
    r = np.random.default_rng(seed)
    return [r.standard_normal((N, d)) for _ in range(7)]  # Q K V dO a b c


# ---------------------------------------------------------------- forward ----

def brute_forward(Q, K, V, scale, causal=True):
    """Pure-Python loops over the definition: no NumPy linear algebra."""
    N, d = len(Q), len(Q[0])
    O = [[0.0] * d for _ in range(N)]
    L = [0.0] * N
    for i in range(N):
        n = i + 1 if causal else N
        s = [scale * sum(Q[i][t] * K[j][t] for t in range(d)) for j in range(n)]
        m = max(s)
        e = [math.exp(x - m) for x in s]
        tot = sum(e)
        L[i] = m + math.log(tot)
        for t in range(d):
            O[i][t] = sum(e[j] / tot * V[j][t] for j in range(n))
    return O, L


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("N,d", [(1, 4), (2, 3), (7, 5), (16, 8)])
def test_forward_brute_force(N, d, causal):
    Q, K, V = rnd(1, N, d), rnd(2, N, d), rnd(3, N, d)
    s = 0.37
    Ob, Lb = brute_forward(Q.tolist(), K.tolist(), V.tolist(), s, causal)
    O, L = oracle.forward(Q, K, V, scale=s, causal=causal)
    assert rel(O, Ob) <= 1e-13
    assert rel(L, Lb) <= 1e-13


@pytest.mark.parametrize("Br,Bc", [(1, 1), (3, 3), (16, 16), (37, 37), (16, 3), (3, 16), (5, 37)])
def test_online_softmax_equals_two_pass(Br, Bc):
    N, d = 37, 8
    Q, K, V = rnd(4, N, d) * 2, rnd(5, N, d) * 2, rnd(6, N, d)
    O2, L2 = oracle.forward(Q, K, V)
    O1, L1 = oracle.forward_online(Q, K, V, Br, Bc)
    assert rel(O1, O2) <= 1e-13
    assert rel(L1, L2) <= 1e-13


def test_probability_rows_sum_to_one_and_are_causal():
    N, d = 50, 16
    Q, K = rnd(7, N, d) * 3, rnd(8, N, d) * 3
    P, L = oracle.softmax_rows(oracle.scores(Q, K, np.arange(N), 0.25))
    assert np.max(np.abs(P.sum(axis=1) - 1.0)) <= 1e-14
    assert np.all(P[np.triu_indices(N, 1)] == 0.0)
    assert np.all(P[np.tril_indices(N)] > 0.0)


def test_forward_invariant_to_common_key_shift():
    N, d = 40, 8
    Q, K, V = rnd(9, N, d), rnd(10, N, d), rnd(11, N, d)
    v = rnd(12, d) * 5
    O0, L0 = oracle.forward(Q, K, V)
    O1, L1 = oracle.forward(Q, K + v[None, :], V)
    assert rel(O1, O0) <= 1e-12
    # L moves by exactly s q_i . v
    assert np.allclose(L1 - L0, oracle.default_scale(d) * Q @ v, rtol=0, atol=1e-12)


def test_forward_uniform_attention_closed_form():
    """Q = 0: every allowed score is 0, so P_ij = 1/(i+1) for j <= i, O_i is the running
    mean of V and L_i = log(i+1)."""
    N, d = 33, 6
    K, V = rnd(13, N, d), rnd(14, N, d)
    O, L = oracle.forward(np.zeros((N, d)), K, V)
    cum = np.cumsum(V, axis=0) / np.arange(1, N + 1)[:, None]
    assert rel(O, cum) <= 1e-14
    assert np.allclose(L, np.log(np.arange(1, N + 1)), rtol=0, atol=1e-14)


def test_forward_row_blocking_and_sampling_agree():
    N, d = 70, 8
    Q, K, V = rnd(15, N, d), rnd(16, N, d), rnd(17, N, d)
    O, L = oracle.forward(Q, K, V)
    Ob, Lb = oracle.forward(Q, K, V, block=9)
    assert rel(Ob, O) <= 1e-15 and rel(Lb, L) <= 1e-15
    rows = np.array([69, 0, 33, 5])
    Or, Lr = oracle.forward_rows(Q, K, V, rows)
    assert rel(Or, O[rows]) <= 1e-15 and rel(Lr, L[rows]) <= 1e-15


# --------------------------------------------------------------- backward ----

def loss(Q, K, V, dO, s):
    O, _ = oracle.forward(Q, K, V, scale=s)
    return float((O * dO).sum())


def fd_grad(f, X, h=1e-5):
    g = np.zeros_like(X)
    for idx in np.ndindex(X.shape):
        e = np.zeros_like(X)
        e[idx] = h
        g[idx] = (f(X + e) - f(X - e)) / (2 * h)
    return g


@pytest.mark.parametrize("N,d", [(1, 3), (6, 3), (11, 4)])
def test_backward_matches_finite_differences(N, d):
    Q, K, V, dO = (x * 0.8 for x in slice_set(N, d, 20)[:4])
    s = 0.6
    g = oracle.backward(Q, K, V, dO, scale=s)
    gQ = fd_grad(lambda X: loss(X, K, V, dO, s), Q)
    gK = fd_grad(lambda X: loss(Q, X, V, dO, s), K)
    gV = fd_grad(lambda X: loss(Q, K, X, dO, s), V)
    top = max(np.abs(gQ).max(), np.abs(gK).max(), np.abs(gV).max(), 1e-3)
    assert np.abs(g["dQ"] - gQ).max() <= 1e-8 * top
    assert np.abs(g["dK"] - gK).max() <= 1e-8 * top
    assert np.abs(g["dV"] - gV).max() <= 1e-8 * top


def test_dS_rows_sum_to_zero():
    N, d = 60, 16
    Q, K, V, dO = slice_set(N, d, 21)[:4]
    t = A._row_terms(Q * 2, K * 2, V, dO, np.arange(N), 0.25)
    l1 = np.abs(t["dS"]).sum(axis=1)
    assert np.all(np.abs(t["dS"].sum(axis=1)) <= 1e-13 * np.maximum(l1, 1e-300))


def test_backward_invariant_to_common_key_shift():
    N, d = 45, 8
    Q, K, V, dO = slice_set(N, d, 22)[:4]
    v = rnd(23, d) * 7
    g0 = oracle.backward(Q, K, V, dO)
    g1 = oracle.backward(Q, K + v[None, :], V, dO)
    for k in ("dQ", "dK", "dV"):
        assert rel(g1[k], g0[k]) <= 1e-12, k


def test_backward_single_token_closed_form():
    """N = 1: P = 1, O = V, dV = dO and dS = 0, so dQ = dK = 0."""
    q, k, v, do = (rnd(i, 1, 5) for i in range(30, 34))
    g = oracle.backward(q, k, v, do)
    assert np.all(g["dQ"] == 0) and np.all(g["dK"] == 0)
    assert np.allclose(g["dV"], do, rtol=0, atol=1e-15)


def test_backward_uniform_attention_dV_closed_form():
    """Q = 0: dV_j = sum_{i >= j} dO_i / (i + 1) and dK = s dS^T Q = 0."""
    N, d = 29, 5
    K, V, dO = rnd(34, N, d), rnd(35, N, d), rnd(36, N, d)
    g = oracle.backward(np.zeros((N, d)), K, V, dO)
    w = dO / np.arange(1, N + 1)[:, None]
    want = np.cumsum(w[::-1], axis=0)[::-1]
    assert rel(g["dV"], want) <= 1e-14
    assert np.abs(g["dK"]).max() == 0.0


def test_backward_sampling_agrees():
    N, d = 64, 8
    Q, K, V, dO = slice_set(N, d, 37)[:4]
    g = oracle.backward(Q, K, V, dO)
    rows, cols = np.array([63, 3, 40]), np.array([50, 63, 7])
    assert rel(oracle.backward_rows(Q, K, V, dO, rows), g["dQ"][rows]) <= 1e-14
    dK, dV = oracle.backward_cols(Q, K, V, dO, cols)
    assert rel(dK, g["dK"][cols]) <= 1e-14 and rel(dV, g["dV"][cols]) <= 1e-14


# ----------------------------------------------------------------- GProj ----

def test_gproj_projected_rows_sum_to_zero_and_rounding_leaves_residual():
    N, d = 96, 16
    Q, K, V, dO = slice_set(N, d, 40)[:4]
    K = K + 10.0  # large common key: the residual then shows up in dQ
    plain = oracle.backward_bf16_dS(Q, K, V, dO, gproj=False)
    proj = oracle.backward_bf16_dS(Q, K, V, dO, gproj=True)
    exact = oracle.backward(Q, K, V, dO)
    assert proj["dS_proj_rowsum_rel"] <= 1e-13
    assert plain["dS_proj_rowsum_rel"] > 1e-5          # bf16 rounding leaves a row mass
    assert rel(proj["dQ"], exact["dQ"]) < rel(plain["dQ"], exact["dQ"])


def test_gproj_row_coefficients_brute_force():
    """The per-row quantities the emulation reports (r_i, rho_i = r_i / sum P^_i and the
    L1 norm of the projected row) against pure-Python loops over the definitions of P,
    dP, D and dS, rounded with the pinned bf16 rounding."""
    N, d = 12, 4
    Q, K, V, dO = slice_set(N, d, 41)[:4]
    K = K + 3.0
    s = 1.0 / math.sqrt(d)
    proj = oracle.backward_bf16_dS(Q, K, V, dO, gproj=True)
    plain = oracle.backward_bf16_dS(Q, K, V, dO, gproj=False)
    for i in range(N):
        sc = [s * sum(Q[i][t] * K[j][t] for t in range(d)) for j in range(i + 1)]
        m = max(sc)
        e = [math.exp(x - m) for x in sc]
        P = [x / sum(e) for x in e]
        dP = [sum(dO[i][t] * V[j][t] for t in range(d)) for j in range(i + 1)]
        D = sum(P[j] * dP[j] for j in range(i + 1))
        dS = [P[j] * (dP[j] - D) for j in range(i + 1)]
        dSh = [float(x) for x in A.bf16_round(np.array(dS))]
        Ph = [float(x) for x in A.bf16_round(np.array(P))]
        r = sum(dSh)
        rho = r / sum(Ph)
        l1 = sum(abs(dSh[j] - rho * Ph[j]) for j in range(i + 1))
        assert abs(proj["r"][i] - r) <= 1e-12 * sum(abs(x) for x in dSh)
        assert abs(proj["rho"][i] - rho) <= 1e-12 * (abs(rho) + 1e-300) + 1e-15
        assert abs(proj["l1"][i] - l1) <= 1e-12 * l1
        assert abs(plain["l1"][i] - sum(abs(x) for x in dSh)) <= 1e-12 * l1
        assert plain["rho"][i] == 0.0


def test_bf16_round_is_round_to_nearest_even():
    # 1 + 2^-8 is halfway between 1 and 1 + 2^-7: ties to even gives 1.
    x = np.array([1.0, 1 + 2 ** -8, 1 + 3 * 2 ** -8, -2.5 + 2 ** -9, 3.0e-39])
    y = A.bf16_round(x)
    assert y[0] == 1.0 and y[1] == 1.0 and y[2] == 1 + 2 ** -6
    assert abs(y[3] - x[3]) <= 2 ** -8 * 2.5
    import torch
    t = torch.tensor(x, dtype=torch.float32).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(t, y)


# -------------------------------------------------------------------- BoB ----

def grads(Q, K, V, dO, s):
    g = oracle.backward(Q, K, V, dO, scale=s)
    return g["dQ"], g["dK"], g["dV"]


@pytest.mark.parametrize("N,d", [(1, 3), (5, 3), (12, 4), (16, 2)])
def test_bob_is_hessian_vector_product(N, d):
    """(gQ, gK, gV) = d/dh grad l(X + h U) at h = 0, U = (a, b, c): central differences."""
    Q, K, V, dO, a, b, c = slice_set(N, d, 50)
    s, h = 0.55, 1e-5
    out = oracle.bob(Q, K, V, dO, a, b, c, scale=s)
    gp = grads(Q + h * a, K + h * b, V + h * c, dO, s)
    gm = grads(Q - h * a, K - h * b, V - h * c, dO, s)
    fd = [(p - m) / (2 * h) for p, m in zip(gp, gm)]
    top = max(np.abs(x).max() for x in fd)
    for name, want in zip(("gQ", "gK", "gV"), fd):
        assert np.abs(out[name] - want).max() <= 1e-8 * max(top, 1e-3), name


@pytest.mark.parametrize("N,d", [(1, 3), (9, 4), (16, 8)])
def test_bob_gdO_is_forward_jvp(N, d):
    Q, K, V, dO, a, b, c = slice_set(N, d, 51)
    s, h = 0.4, 1e-5
    out = oracle.bob(Q, K, V, dO, a, b, c, scale=s)
    Op, _ = oracle.forward(Q + h * a, K + h * b, V + h * c, scale=s)
    Om, _ = oracle.forward(Q - h * a, K - h * b, V - h * c, scale=s)
    fd = (Op - Om) / (2 * h)
    assert np.abs(out["gdO"] - fd).max() <= 1e-8 * max(np.abs(fd).max(), 1e-3)


def test_bob_gdO_independent_of_dO():
    Q, K, V, dO, a, b, c = slice_set(20, 6, 52)
    g1 = oracle.bob(Q, K, V, dO, a, b, c)["gdO"]
    g2 = oracle.bob(Q, K, V, 3 * dO + 1, a, b, c)["gdO"]
    assert rel(g2, g1) <= 1e-13


def test_bob_hvp_symmetry():
    """<U', H U> = <U, H U'> for the Hessian of l = <O, dO> in (Q, K, V)."""
    Q, K, V, dO, a, b, c = slice_set(24, 6, 53)
    a2, b2, c2 = slice_set(24, 6, 54)[:3]
    h1 = oracle.bob(Q, K, V, dO, a, b, c)
    h2 = oracle.bob(Q, K, V, dO, a2, b2, c2)
    lhs = (a2 * h1["gQ"]).sum() + (b2 * h1["gK"]).sum() + (c2 * h1["gV"]).sum()
    rhs = (a * h2["gQ"]).sum() + (b * h2["gK"]).sum() + (c * h2["gV"]).sum()
    assert abs(lhs - rhs) <= 1e-12 * max(abs(lhs), 1.0)


def test_bob_row_sums_of_sbar_and_dpbar_vanish():
    N, d = 40, 8
    Q, K, V, dO, a, b, c = slice_set(N, d, 55)
    t = A._row_terms(Q, K, V, dO, np.arange(N), 0.3, a, b, c)
    for k in ("Sbar", "dPbar"):
        l1 = np.abs(t[k]).sum(axis=1)
        assert np.all(np.abs(t[k].sum(axis=1)) <= 1e-13 * np.maximum(l1, 1e-300)), k


def test_bob_invariant_to_common_key_shift():
    Q, K, V, dO, a, b, c = slice_set(30, 8, 56)
    v = rnd(57, 8) * 6
    o0 = oracle.bob(Q, K, V, dO, a, b, c)
    o1 = oracle.bob(Q, K + v[None, :], V, dO, a, b, c)
    for k in ("gQ", "gK", "gV", "gdO"):
        assert rel(o1[k], o0[k]) <= 1e-11, k


def test_bob_invariant_to_common_shift_of_b():
    # b = gdK enters only through G = s(a K^T + Q b^T) and the product dS b.  One vector
    # v added to every row of b adds the per-row constant s q_i.v to G, which
    # dPbar = P(G - E) and Sbar = P(Pbar - F) do not see (E and F move with it), and
    # adds s (sum_j dS_ij) v = 0 to dS b (exact dS rows sum to zero).
    Q, K, V, dO, a, b, c = slice_set(30, 8, 58)
    v = rnd(59, 8) * 6
    o0 = oracle.bob(Q, K, V, dO, a, b, c)
    o1 = oracle.bob(Q, K, V, dO, a, b + v[None, :], c)
    for k in ("gQ", "gK", "gV", "gdO"):
        assert rel(o1[k], o0[k]) <= 1e-11, k


@pytest.mark.parametrize("causal", [True, False])
def test_bob_bf16_dS_projection(causal):
    # GProj page, "How the zero sum turns into a false gradient", applied to the dS
    # of BoB's dS b and dS^T a products.
    N, d = 96, 16
    Q, K, V, dO, a, b, c = slice_set(N, d, 60)
    b = b + 10.0  # a large common b: the rounding residual then shows up in gQ
    s = 1.0 / math.sqrt(d)
    exact = oracle.bob(Q, K, V, dO, a, b, c, causal=causal)
    # No rounding: nothing to project (exact rows sum to zero), every output exact.
    ident = oracle.bob_bf16_dS(Q, K, V, dO, a, b, c, True, causal=causal, rnd=lambda x: x)
    for k in ("gQ", "gK", "gV", "gdO"):
        assert rel(ident[k], exact[k]) <= 1e-12, k
    plain = oracle.bob_bf16_dS(Q, K, V, dO, a, b, c, False, causal=causal)
    proj = oracle.bob_bf16_dS(Q, K, V, dO, a, b, c, True, causal=causal)
    assert proj["dS_rowsum_rel"] <= 1e-13
    assert plain["dS_rowsum_rel"] > 1e-5  # bf16 rounding leaves a row mass
    for k in ("gV", "gdO"):  # they never see dS
        assert rel(plain[k], exact[k]) <= 1e-13 and rel(proj[k], exact[k]) <= 1e-13, k
    # A common shift v of b: unprojected, gQ moves by exactly s r_i v (the residual
    # times the shift); projected, it does not move at all.
    v = rnd(61, d) * 3
    plain_v = oracle.bob_bf16_dS(Q, K, V, dO, a, b + v[None, :], c, False, causal=causal)
    proj_v = oracle.bob_bf16_dS(Q, K, V, dO, a, b + v[None, :], c, True, causal=causal)
    assert rel(plain_v["gQ"] - plain["gQ"], s * np.outer(plain["r"], v)) <= 1e-8
    assert rel(proj_v["gQ"], proj["gQ"]) <= 1e-11
    assert rel(proj["gQ"], exact["gQ"]) < rel(plain["gQ"], exact["gQ"])


def test_bob_single_token_closed_form():
    """N = 1: gQ = gK = gV = 0 and gdO = c (gdO = P c + dPbar V with P = 1, dPbar = 0)."""
    Q, K, V, dO, a, b, c = slice_set(1, 5, 58)
    o = oracle.bob(Q, K, V, dO, a, b, c)
    for k in ("gQ", "gK", "gV"):
        assert np.abs(o[k]).max() <= 1e-15, k
    assert np.allclose(o["gdO"], c, rtol=0, atol=1e-15)


@pytest.mark.parametrize("Bc,Br", [(1, 1), (4, 7), (16, 16), (64, 64)])
def test_bob_streaming_passes_equal_closed_form(Bc, Br):
    N, d = 53, 8
    Q, K, V, dO, a, b, c = slice_set(N, d, 59)
    ref = oracle.bob(Q, K, V, dO, a, b, c)
    O, L = oracle.forward(Q, K, V)
    rp = oracle.bob_row_pass(Q, K, V, dO, a, b, c, O, L, Bc)
    for k in ("gQ", "gdO", "E", "F"):
        assert rel(rp[k], ref[k]) <= 1e-12, k
    gK, gV = oracle.bob_col_pass(Q, K, V, dO, a, b, c, L, rp["D"], rp["E"], rp["F"], Br)
    assert rel(gK, ref["gK"]) <= 1e-12 and rel(gV, ref["gV"]) <= 1e-12


def test_bob_sampling_agrees():
    N, d = 64, 8
    Q, K, V, dO, a, b, c = slice_set(N, d, 60)
    ref = oracle.bob(Q, K, V, dO, a, b, c, block=11)
    rows, cols = np.array([0, 63, 17]), np.array([60, 2, 63])
    r = oracle.bob_rows(Q, K, V, dO, a, b, c, rows)
    assert rel(r["gQ"], ref["gQ"][rows]) <= 1e-13 and rel(r["gdO"], ref["gdO"][rows]) <= 1e-13
    gK, gV = oracle.bob_cols(Q, K, V, dO, a, b, c, cols)
    assert rel(gK, ref["gK"][cols]) <= 1e-13 and rel(gV, ref["gV"][cols]) <= 1e-13


def test_bob_against_fp64_autograd():
    """Independent check: PyTorch's fp64 CPU double backward of the same loss."""
    torch = pytest.importorskip("torch")
    N, d = 13, 8
    arrs = slice_set(N, d, 61)
    s = 1 / math.sqrt(d)
    Q, K, V, dO, a, b, c = (torch.tensor(x, dtype=torch.float64, requires_grad=i < 4)
                            for i, x in enumerate(arrs))
    S = (Q @ K.T) * s
    S = S.masked_fill(torch.triu(torch.ones(N, N, dtype=torch.bool), 1), float("-inf"))
    O = torch.softmax(S, dim=-1) @ V
    dQ, dK, dV = torch.autograd.grad((O * dO).sum(), (Q, K, V), create_graph=True)
    psi = (a * dQ).sum() + (b * dK).sum() + (c * dV).sum()
    gQ, gK, gV, gdO = torch.autograd.grad(psi, (Q, K, V, dO))
    ref = oracle.bob(*arrs)
    for k, t in zip(("gQ", "gK", "gV", "gdO"), (gQ, gK, gV, gdO)):
        assert rel(ref[k], t.numpy()) <= 1e-13, k
    fb = oracle.backward(*arrs[:4])
    assert rel(fb["dQ"], dQ.detach().numpy()) <= 1e-13


def test_bob_against_symbolic_second_derivative():
    """Independent check: sympy differentiates the causal attention loss twice."""
    sp = pytest.importorskip("sympy")
    N, d = 3, 2
    vals = slice_set(N, d, 62)
    s = sp.Rational(7, 10)
    sym = {n: sp.Matrix(N, d, lambda i, j, n=n: sp.Symbol(f"{n}{i}{j}")) for n in ("q", "k", "v", "o")}
    q, k, v, o = (sym[n] for n in ("q", "k", "v", "o"))
    loss_expr = 0
    for i in range(N):
        w = [sp.exp(s * (q.row(i).dot(k.row(j)))) for j in range(i + 1)]
        z = sum(w)
        for t in range(d):
            loss_expr += o[i, t] * sum(w[j] * v[j, t] for j in range(i + 1)) / z
    a_, b_, c_ = (sp.Matrix(vals[4 + i]) for i in range(3))
    psi = 0
    for i in range(N):
        for t in range(d):
            psi += a_[i, t] * sp.diff(loss_expr, q[i, t]) + b_[i, t] * sp.diff(loss_expr, k[i, t]) \
                + c_[i, t] * sp.diff(loss_expr, v[i, t])
    point = {}
    for n, arr in zip(("q", "k", "v", "o"), vals[:4]):
        for i in range(N):
            for t in range(d):
                point[sym[n][i, t]] = float(arr[i, t])
    syms = [sym[n][i, t] for n in ("q", "k", "v", "o") for i in range(N) for t in range(d)]
    f = sp.lambdify(syms, [sp.diff(psi, x) for x in syms], "math")
    g = np.array(f(*[point[x] for x in syms])).reshape(4, N, d)
    ref = oracle.bob(*vals, scale=0.7)
    for idx, key in enumerate(("gQ", "gK", "gV", "gdO")):
        assert rel(ref[key], g[idx]) <= 1e-12, key


# ------------------------------------------------------ planted mistakes ----

MUTATIONS = {
    "drop_H": lambda t: t.update(Hm=t["Hm"] * 0),
    "sign_E": lambda t: t.update(dPbar=t["P"] * (t["G"] + t["E"][:, None])),
    "drop_F": lambda t: t.update(Sbar=t["P"] * t["Pbar"]),
    "transpose_b": lambda t: None,  # handled below: b and a swapped in G
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistakes_are_caught(name, monkeypatch):
    """Plant a plausible mistake in the oracle's BoB and check the FD pin fails."""
    orig = A._row_terms

    def mutated(Q, K, V, dO, rows, scale, a=None, b=None, c=None, causal=True):
        if name == "transpose_b" and a is not None:
            return orig(Q, K, V, dO, rows, scale, b, a, c, causal=causal)
        t = orig(Q, K, V, dO, rows, scale, a, b, c, causal=causal)
        if a is not None:
            MUTATIONS[name](t)
            # re-derive the dependants of the mutated tile as the real code would
            if name == "drop_H":
                t["Pbar"] = t["G"] * (t["dP"] - t["D"][:, None]) - t["E"][:, None] * t["dP"]
                t["F"] = (t["P"] * t["Pbar"]).sum(axis=1)
                t["Sbar"] = t["P"] * (t["Pbar"] - t["F"][:, None])
        return t

    N, d = 8, 3
    Q, K, V, dO, a, b, c = slice_set(N, d, 70)
    s, h = 0.5, 1e-5
    gp = grads(Q + h * a, K + h * b, V + h * c, dO, s)
    gm = grads(Q - h * a, K - h * b, V - h * c, dO, s)
    fd = [(p - m) / (2 * h) for p, m in zip(gp, gm)]
    Op, _ = oracle.forward(Q + h * a, K + h * b, V + h * c, scale=s)
    Om, _ = oracle.forward(Q - h * a, K - h * b, V - h * c, scale=s)
    fd.append((Op - Om) / (2 * h))
    monkeypatch.setattr(A, "_row_terms", mutated)
    out = A.bob(Q, K, V, dO, a, b, c, scale=s)
    errs = [rel(out[k], w) for k, w in zip(("gQ", "gK", "gV", "gdO"), fd)]
    assert max(errs) > 1e-4, (name, errs)


# ------------------------------------------------------------- non-causal ----
# The same method with every key visible to every query (the "causal=False" mode):
# pinned the same ways as the causal default.

def loss_nc(Q, K, V, dO, s):
    O, _ = oracle.forward(Q, K, V, scale=s, causal=False)
    return float((O * dO).sum())


@pytest.mark.parametrize("Br,Bc", [(1, 1), (16, 3), (5, 37), (37, 37)])
def test_noncausal_online_softmax_equals_two_pass(Br, Bc):
    N, d = 37, 8
    Q, K, V = rnd(80, N, d) * 2, rnd(81, N, d) * 2, rnd(82, N, d)
    O2, L2 = oracle.forward(Q, K, V, causal=False)
    O1, L1 = oracle.forward_online(Q, K, V, Br, Bc, causal=False)
    assert rel(O1, O2) <= 1e-13 and rel(L1, L2) <= 1e-13


def test_noncausal_uniform_attention_closed_form():
    """Q = 0: P_ij = 1/N for every pair, O_i = the mean of V, L_i = log N."""
    N, d = 29, 5
    K, V = rnd(83, N, d), rnd(84, N, d)
    O, L = oracle.forward(np.zeros((N, d)), K, V, causal=False)
    assert rel(O, np.broadcast_to(V.mean(axis=0), (N, d))) <= 1e-14
    assert np.allclose(L, np.log(N), rtol=0, atol=1e-14)


def test_noncausal_probabilities_have_full_support_and_differ_from_causal():
    N, d = 30, 8
    Q, K, V = rnd(85, N, d), rnd(86, N, d), rnd(87, N, d)
    P, _ = oracle.softmax_rows(oracle.scores(Q, K, np.arange(N), 0.3, causal=False))
    assert P.shape == (N, N) and np.all(P > 0) and np.max(np.abs(P.sum(axis=1) - 1.0)) <= 1e-14
    Oc, _ = oracle.forward(Q, K, V, causal=True)
    On, _ = oracle.forward(Q, K, V, causal=False)
    assert rel(On[-1], Oc[-1]) <= 1e-15       # the last row sees every key either way
    assert rel(On[:-1], Oc[:-1]) > 1e-3


@pytest.mark.parametrize("N,d", [(1, 3), (6, 3), (11, 4)])
def test_noncausal_backward_matches_finite_differences(N, d):
    Q, K, V, dO = (x * 0.8 for x in slice_set(N, d, 88)[:4])
    s = 0.6
    g = oracle.backward(Q, K, V, dO, scale=s, causal=False)
    gQ = fd_grad(lambda X: loss_nc(X, K, V, dO, s), Q)
    gK = fd_grad(lambda X: loss_nc(Q, X, V, dO, s), K)
    gV = fd_grad(lambda X: loss_nc(Q, K, X, dO, s), V)
    top = max(np.abs(gQ).max(), np.abs(gK).max(), np.abs(gV).max(), 1e-3)
    assert np.abs(g["dQ"] - gQ).max() <= 1e-8 * top
    assert np.abs(g["dK"] - gK).max() <= 1e-8 * top
    assert np.abs(g["dV"] - gV).max() <= 1e-8 * top


def test_noncausal_backward_sampling_agrees():
    N, d = 45, 6
    Q, K, V, dO = slice_set(N, d, 89)[:4]
    ref = oracle.backward(Q, K, V, dO, block=7, causal=False)
    rows, cols = np.array([0, 44, 13]), np.array([0, 30, 44])
    assert rel(oracle.backward_rows(Q, K, V, dO, rows, causal=False), ref["dQ"][rows]) <= 1e-13
    dK, dV = oracle.backward_cols(Q, K, V, dO, cols, causal=False)
    assert rel(dK, ref["dK"][cols]) <= 1e-13 and rel(dV, ref["dV"][cols]) <= 1e-13


def grads_nc(Q, K, V, dO, s):
    g = oracle.backward(Q, K, V, dO, scale=s, causal=False)
    return g["dQ"], g["dK"], g["dV"]


@pytest.mark.parametrize("N,d", [(1, 3), (5, 3), (12, 4)])
def test_noncausal_bob_is_hessian_vector_product(N, d):
    Q, K, V, dO, a, b, c = slice_set(N, d, 90)
    s, h = 0.55, 1e-5
    out = oracle.bob(Q, K, V, dO, a, b, c, scale=s, causal=False)
    gp = grads_nc(Q + h * a, K + h * b, V + h * c, dO, s)
    gm = grads_nc(Q - h * a, K - h * b, V - h * c, dO, s)
    fd = [(p - m) / (2 * h) for p, m in zip(gp, gm)]
    top = max(np.abs(x).max() for x in fd)
    for name, want in zip(("gQ", "gK", "gV"), fd):
        assert np.abs(out[name] - want).max() <= 1e-8 * max(top, 1e-3), name


def test_noncausal_bob_gdO_is_forward_jvp():
    Q, K, V, dO, a, b, c = slice_set(9, 4, 91)
    s, h = 0.4, 1e-5
    out = oracle.bob(Q, K, V, dO, a, b, c, scale=s, causal=False)
    Op, _ = oracle.forward(Q + h * a, K + h * b, V + h * c, scale=s, causal=False)
    Om, _ = oracle.forward(Q - h * a, K - h * b, V - h * c, scale=s, causal=False)
    fd = (Op - Om) / (2 * h)
    assert np.abs(out["gdO"] - fd).max() <= 1e-8 * max(np.abs(fd).max(), 1e-3)


@pytest.mark.parametrize("Bc,Br", [(1, 1), (4, 7), (16, 16)])
def test_noncausal_bob_streaming_passes_equal_closed_form(Bc, Br):
    N, d = 41, 8
    Q, K, V, dO, a, b, c = slice_set(N, d, 92)
    ref = oracle.bob(Q, K, V, dO, a, b, c, causal=False)
    O, L = oracle.forward(Q, K, V, causal=False)
    rp = oracle.bob_row_pass(Q, K, V, dO, a, b, c, O, L, Bc, causal=False)
    for k in ("gQ", "gdO", "E", "F"):
        assert rel(rp[k], ref[k]) <= 1e-12, k
    gK, gV = oracle.bob_col_pass(Q, K, V, dO, a, b, c, L, rp["D"], rp["E"], rp["F"], Br, causal=False)
    assert rel(gK, ref["gK"]) <= 1e-12 and rel(gV, ref["gV"]) <= 1e-12
    rows, cols = np.array([40, 3]), np.array([0, 40])
    r = oracle.bob_rows(Q, K, V, dO, a, b, c, rows, causal=False)
    assert rel(r["gQ"], ref["gQ"][rows]) <= 1e-13 and rel(r["gdO"], ref["gdO"][rows]) <= 1e-13
    gKc, gVc = oracle.bob_cols(Q, K, V, dO, a, b, c, cols, causal=False)
    assert rel(gKc, ref["gK"][cols]) <= 1e-13 and rel(gVc, ref["gV"][cols]) <= 1e-13


def test_noncausal_bob_against_fp64_autograd():
    torch = pytest.importorskip("torch")
    N, d = 11, 6
    arrs = slice_set(N, d, 93)
    s = 1 / math.sqrt(d)
    Q, K, V, dO, a, b, c = (torch.tensor(x, dtype=torch.float64, requires_grad=i < 4)
                            for i, x in enumerate(arrs))
    O = torch.softmax((Q @ K.T) * s, dim=-1) @ V
    dQ, dK, dV = torch.autograd.grad((O * dO).sum(), (Q, K, V), create_graph=True)
    psi = (a * dQ).sum() + (b * dK).sum() + (c * dV).sum()
    gQ, gK, gV, gdO = torch.autograd.grad(psi, (Q, K, V, dO))
    ref = oracle.bob(*arrs, causal=False)
    for k, t in zip(("gQ", "gK", "gV", "gdO"), (gQ, gK, gV, gdO)):
        assert rel(ref[k], t.numpy()) <= 1e-13, k
    fb = oracle.backward(*arrs[:4], causal=False)
    assert rel(fb["dQ"], dQ.detach().numpy()) <= 1e-13


# ----------------------------------------------------- grouped key/value heads ----
# H query heads share H / g key/value heads: query head h reads key/value head h // g.
# Pinned by finite differences of the loss summed over the heads (so the gradient of a
# shared head is whatever the chain rule makes it, not the oracle's group sum).

def _gqa_loss(Q, K, V, dO, s, g, causal):
    O = oracle.forward_all(Q, K, V, scale=s, causal=causal, groups=g)["O"]
    return float((O * dO).sum())


@pytest.mark.parametrize("causal", [True, False])
def test_gqa_backward_matches_finite_differences(causal):
    r = np.random.default_rng(94)
    B, H, g, N, d = 1, 4, 2, 5, 3
    Q, dO = r.standard_normal((B, H, N, d)), r.standard_normal((B, H, N, d))
    K, V = r.standard_normal((B, H // g, N, d)), r.standard_normal((B, H // g, N, d))
    s = 0.6
    out = oracle.backward_all(Q, K, V, dO, scale=s, causal=causal, groups=g)
    assert out["dK"].shape == K.shape and out["dQ"].shape == Q.shape
    gK = fd_grad(lambda X: _gqa_loss(Q, X, V, dO, s, g, causal), K)
    gV = fd_grad(lambda X: _gqa_loss(Q, K, X, dO, s, g, causal), V)
    gQ = fd_grad(lambda X: _gqa_loss(X, K, V, dO, s, g, causal), Q)
    top = max(np.abs(gK).max(), np.abs(gV).max(), np.abs(gQ).max())
    assert np.abs(out["dK"] - gK).max() <= 1e-8 * top
    assert np.abs(out["dV"] - gV).max() <= 1e-8 * top
    assert np.abs(out["dQ"] - gQ).max() <= 1e-8 * top


@pytest.mark.parametrize("causal", [True, False])
def test_gqa_bob_is_hessian_vector_product(causal):
    """BoB with shared heads: the directional derivative of the grouped first backward
    (dQ per query head, dK and dV per shared head) along (a, b, c), by central differences."""
    r = np.random.default_rng(95)
    B, H, g, N, d = 1, 4, 2, 5, 3
    Q, dO, a = (r.standard_normal((B, H, N, d)) for _ in range(3))
    K, V, b, c = (r.standard_normal((B, H // g, N, d)) for _ in range(4))
    s, h = 0.55, 1e-5
    out = oracle.bob_all(Q, K, V, dO, a, b, c, scale=s, causal=causal, groups=g)
    gp = oracle.backward_all(Q + h * a, K + h * b, V + h * c, dO, scale=s, causal=causal, groups=g)
    gm = oracle.backward_all(Q - h * a, K - h * b, V - h * c, dO, scale=s, causal=causal, groups=g)
    for name, key in (("gQ", "dQ"), ("gK", "dK"), ("gV", "dV")):
        fd = (gp[key] - gm[key]) / (2 * h)
        assert out[name].shape == fd.shape
        assert np.abs(out[name] - fd).max() <= 1e-8 * max(np.abs(fd).max(), 1e-3), name
    Op = oracle.forward_all(Q + h * a, K + h * b, V + h * c, scale=s, causal=causal, groups=g)["O"]
    Om = oracle.forward_all(Q - h * a, K - h * b, V - h * c, scale=s, causal=causal, groups=g)["O"]
    fd = (Op - Om) / (2 * h)
    assert np.abs(out["gdO"] - fd).max() <= 1e-8 * max(np.abs(fd).max(), 1e-3)


def test_gqa_with_one_group_is_plain_attention():
    r = np.random.default_rng(96)
    X = [r.standard_normal((2, 3, 7, 4)) for _ in range(7)]
    a = oracle.bob_all(*X, groups=1)
    b = oracle.bob_all(*X)
    for k in ("gQ", "gK", "gV", "gdO"):
        assert np.array_equal(a[k], b[k])


# ------------------------------------------------------ causal sliding window ----
# A flexible mask (FlashBoB page, "When FlashBoB changes the engineering plan", names
# flexible masks as a next extension): key j visible to query i iff i - W < j <= i.

def brute_forward_window(Q, K, V, scale, W):
    """Pure-Python loops over the definition with the banded mask."""
    N, d = len(Q), len(Q[0])
    O = [[0.0] * d for _ in range(N)]
    L = [0.0] * N
    for i in range(N):
        js = [j for j in range(N) if i - W < j <= i]
        s = [scale * sum(Q[i][t] * K[j][t] for t in range(d)) for j in js]
        m = max(s)
        e = [math.exp(x - m) for x in s]
        tot = sum(e)
        L[i] = m + math.log(tot)
        for t in range(d):
            O[i][t] = sum(e[n] / tot * V[js[n]][t] for n in range(len(js)))
    return O, L


@pytest.mark.parametrize("N,d,W", [(1, 3, 1), (7, 5, 2), (16, 8, 5), (16, 4, 40)])
def test_window_forward_brute_force(N, d, W):
    Q, K, V = (rnd(100 + k, N, d) for k in range(3))
    O, L = oracle.forward(Q, K, V, scale=0.7, causal=oracle.Window(W))
    Ob, Lb = brute_forward_window(Q.tolist(), K.tolist(), V.tolist(), 0.7, W)
    assert rel(O, np.array(Ob)) <= 1e-13 and rel(L, np.array(Lb)) <= 1e-13


@pytest.mark.parametrize("Br,Bc", [(1, 1), (16, 3), (5, 37), (37, 37)])
def test_window_online_softmax_equals_two_pass(Br, Bc):
    N, d = 37, 8
    Q, K, V = rnd(103, N, d) * 2, rnd(104, N, d) * 2, rnd(105, N, d)
    w = oracle.Window(9)
    O2, L2 = oracle.forward(Q, K, V, causal=w)
    O1, L1 = oracle.forward_online(Q, K, V, Br, Bc, causal=w)
    assert rel(O1, O2) <= 1e-13 and rel(L1, L2) <= 1e-13


def test_window_limits_reduce_to_causal_and_to_one_key():
    """W >= N is the causal mask.  W = 1: every row sees only its own key, so P = I:
    O = V, L_i = s q_i.k_i; dS = 0 (dQ = dK = 0), dV = dO; BoB: G - E = 0 and Sbar = 0,
    so gQ = gK = gV = 0 and gdO = c."""
    N, d = 12, 4
    Q, K, V, dO, a, b, c = slice_set(N, d, 106)
    s = 0.45
    for fn in (oracle.forward, ):
        assert all(np.array_equal(x, y) for x, y in zip(fn(Q, K, V, scale=s, causal=oracle.Window(N)),
                                                        fn(Q, K, V, scale=s, causal=True)))
    full = oracle.bob(Q, K, V, dO, a, b, c, scale=s, causal=oracle.Window(N + 5))
    ref = oracle.bob(Q, K, V, dO, a, b, c, scale=s, causal=True)
    for k in ("gQ", "gK", "gV", "gdO"):
        assert np.array_equal(full[k], ref[k]), k
    one = oracle.Window(1)
    O, L = oracle.forward(Q, K, V, scale=s, causal=one)
    assert rel(O, V) <= 1e-15 and np.allclose(L, s * (Q * K).sum(axis=1), rtol=0, atol=1e-14)
    g = oracle.backward(Q, K, V, dO, scale=s, causal=one)
    assert np.abs(g["dQ"]).max() <= 1e-14 and np.abs(g["dK"]).max() <= 1e-14 and rel(g["dV"], dO) <= 1e-15
    bb = oracle.bob(Q, K, V, dO, a, b, c, scale=s, causal=one)
    for k in ("gQ", "gK", "gV"):
        assert np.abs(bb[k]).max() <= 1e-13, k
    assert rel(bb["gdO"], c) <= 1e-15


def loss_w(Q, K, V, dO, s, w):
    O, _ = oracle.forward(Q, K, V, scale=s, causal=w)
    return float((O * dO).sum())


@pytest.mark.parametrize("N,d,W", [(6, 3, 2), (11, 4, 4)])
def test_window_backward_matches_finite_differences(N, d, W):
    Q, K, V, dO = (x * 0.8 for x in slice_set(N, d, 107)[:4])
    s, w = 0.6, oracle.Window(W)
    g = oracle.backward(Q, K, V, dO, scale=s, causal=w)
    gQ = fd_grad(lambda X: loss_w(X, K, V, dO, s, w), Q)
    gK = fd_grad(lambda X: loss_w(Q, X, V, dO, s, w), K)
    gV = fd_grad(lambda X: loss_w(Q, K, X, dO, s, w), V)
    top = max(np.abs(gQ).max(), np.abs(gK).max(), np.abs(gV).max(), 1e-3)
    for got, want in ((g["dQ"], gQ), (g["dK"], gK), (g["dV"], gV)):
        assert np.abs(got - want).max() <= 1e-8 * top


@pytest.mark.parametrize("N,d,W", [(5, 3, 2), (12, 4, 5)])
def test_window_bob_is_hessian_vector_product_and_jvp(N, d, W):
    Q, K, V, dO, a, b, c = slice_set(N, d, 108)
    s, h, w = 0.55, 1e-5, oracle.Window(W)
    out = oracle.bob(Q, K, V, dO, a, b, c, scale=s, causal=w)

    def grads_w(Q, K, V):
        g = oracle.backward(Q, K, V, dO, scale=s, causal=w)
        return g["dQ"], g["dK"], g["dV"]
    gp = grads_w(Q + h * a, K + h * b, V + h * c)
    gm = grads_w(Q - h * a, K - h * b, V - h * c)
    fd = [(p - m) / (2 * h) for p, m in zip(gp, gm)]
    top = max(np.abs(x).max() for x in fd)
    for name, want in zip(("gQ", "gK", "gV"), fd):
        assert np.abs(out[name] - want).max() <= 1e-8 * max(top, 1e-3), name
    Op, _ = oracle.forward(Q + h * a, K + h * b, V + h * c, scale=s, causal=w)
    Om, _ = oracle.forward(Q - h * a, K - h * b, V - h * c, scale=s, causal=w)
    jvp = (Op - Om) / (2 * h)
    assert np.abs(out["gdO"] - jvp).max() <= 1e-8 * max(np.abs(jvp).max(), 1e-3)


@pytest.mark.parametrize("Bc,Br", [(1, 1), (4, 7), (16, 16)])
def test_window_bob_streaming_passes_equal_closed_form(Bc, Br):
    N, d = 33, 5
    Q, K, V, dO, a, b, c = slice_set(N, d, 109)
    w = oracle.Window(6)
    ref = oracle.bob(Q, K, V, dO, a, b, c, causal=w)
    O, L = oracle.forward(Q, K, V, causal=w)
    row = oracle.bob_row_pass(Q, K, V, dO, a, b, c, O, L, Bc, causal=w)
    gK, gV = oracle.bob_col_pass(Q, K, V, dO, a, b, c, L, row["D"], row["E"], row["F"], Br, causal=w)
    for got, want in ((row["gQ"], ref["gQ"]), (row["gdO"], ref["gdO"]), (gK, ref["gK"]), (gV, ref["gV"])):
        assert rel(got, want) <= 1e-12


def test_window_sampling_agrees():
    N, d = 45, 6
    Q, K, V, dO, a, b, c = slice_set(N, d, 110)
    w = oracle.Window(8)
    ref = oracle.bob(Q, K, V, dO, a, b, c, block=7, causal=w)
    rows, cols = np.array([0, 44, 13]), np.array([0, 30, 44])
    r = oracle.bob_rows(Q, K, V, dO, a, b, c, rows, causal=w)
    assert rel(r["gQ"], ref["gQ"][rows]) <= 1e-13 and rel(r["gdO"], ref["gdO"][rows]) <= 1e-13
    gK, gV = oracle.bob_cols(Q, K, V, dO, a, b, c, cols, causal=w)
    assert rel(gK, ref["gK"][cols]) <= 1e-13 and rel(gV, ref["gV"][cols]) <= 1e-13


def test_window_bob_gproj_projection():
    """GProj inside BoB under a sliding window: the projected rows (over each row's
    visible keys) sum to zero, and a common shift of b leaves the projected gQ alone."""
    N, d = 80, 8
    Q, K, V, dO, a, b, c = slice_set(N, d, 111)
    w = oracle.Window(13)
    proj = oracle.bob_bf16_dS(Q, K, V, dO, a, b + 7.0, c, True, causal=w)
    assert proj["dS_rowsum_rel"] <= 1e-13
    v = rnd(112, d) * 3
    proj_v = oracle.bob_bf16_dS(Q, K, V, dO, a, b + 7.0 + v[None, :], c, True, causal=w)
    assert rel(proj_v["gQ"], proj["gQ"]) <= 1e-11
    exact = oracle.bob(Q, K, V, dO, a, b + 7.0, c, causal=w)
    plain = oracle.bob_bf16_dS(Q, K, V, dO, a, b + 7.0, c, False, causal=w)
    assert rel(proj["gQ"], exact["gQ"]) < rel(plain["gQ"], exact["gQ"])


# ------------------------------------------------------ document (segment) mask ----
# Query i sees key j iff j <= i and seg[j] == seg[i] (packed documents), optionally also
# inside a window.  The strongest pin: the mask is block diagonal over the documents, so
# every output restricted to one document equals plain causal attention run on that
# document alone -- a different code path (sub-arrays, no segment logic at all).

def brute_forward_segments(Q, K, V, scale, seg, W=0):
    """Pure-Python loops over the definition with the document mask."""
    N, d = len(Q), len(Q[0])
    O = [[0.0] * d for _ in range(N)]
    L = [0.0] * N
    for i in range(N):
        js = [j for j in range(N) if j <= i and seg[j] == seg[i] and (W == 0 or j > i - W)]
        s = [scale * sum(Q[i][t] * K[j][t] for t in range(d)) for j in js]
        m = max(s)
        e = [math.exp(x - m) for x in s]
        tot = sum(e)
        L[i] = m + math.log(tot)
        for t in range(d):
            O[i][t] = sum(e[u] / tot * V[js[u]][t] for u in range(len(js)))
    return O, L


SEGS = [np.array([0, 0, 0, 1, 1, 2, 2, 2, 2, 3, 4, 4, 4, 4, 4, 4, 5]),
        np.array([7] * 5 + [9] * 11 + [12])]


@pytest.mark.parametrize("seg", SEGS)
@pytest.mark.parametrize("W", [0, 3])
def test_segments_forward_brute_force(seg, W):
    N, d = len(seg), 5
    Q, K, V = rnd(201, N, d), rnd(202, N, d), rnd(203, N, d)
    Ob, Lb = brute_forward_segments(Q.tolist(), K.tolist(), V.tolist(), 0.41, seg.tolist(), W)
    O, L = oracle.forward(Q, K, V, scale=0.41, causal=oracle.Segments(seg, W))
    assert rel(O, Ob) <= 1e-13 and rel(L, Lb) <= 1e-13


def _runs(seg):
    cut = np.flatnonzero(np.diff(seg)) + 1
    return np.split(np.arange(len(seg)), cut)


@pytest.mark.parametrize("W", [0, 4])
def test_segments_are_block_diagonal(W):
    seg = np.repeat(np.arange(6), [1, 9, 4, 13, 2, 8])  # 37 tokens, runs of 1 .. 13
    N, d = len(seg), 6
    Q, K, V, dO, a, b, c = slice_set(N, d, 204)
    m = oracle.Segments(seg, W)
    f = oracle.forward(Q, K, V, causal=m)
    g = oracle.backward(Q, K, V, dO, causal=m)
    h = oracle.bob(Q, K, V, dO, a, b, c, causal=m)
    for r in _runs(seg):
        sub = lambda X: X[r]
        cm = oracle.Window(W) if W else True
        fr = oracle.forward(sub(Q), sub(K), sub(V), causal=cm)
        gr = oracle.backward(sub(Q), sub(K), sub(V), sub(dO), causal=cm)
        hr = oracle.bob(sub(Q), sub(K), sub(V), sub(dO), sub(a), sub(b), sub(c), causal=cm)
        assert rel(f[0][r], fr[0]) <= 1e-13 and rel(f[1][r], fr[1]) <= 1e-13
        for k in ("dQ", "dK", "dV"):
            assert rel(g[k][r], gr[k]) <= 1e-12, k
        for k in ("gQ", "gK", "gV", "gdO"):
            assert rel(h[k][r], hr[k]) <= 1e-12, k


def test_segments_limits():
    """One segment is the causal mask (bit for bit); one token per segment leaves each row
    its own key only: O = V, lse = s q.k, dQ = dK = 0, dV = dO, gQ = gK = gV = 0, gdO = c."""
    N, d = 21, 4
    Q, K, V, dO, a, b, c = slice_set(N, d, 205)
    one = oracle.Segments(np.zeros(N, int))
    for f in (lambda m: oracle.forward(Q, K, V, causal=m)[0], lambda m: oracle.backward(Q, K, V, dO, causal=m)["dK"],
              lambda m: oracle.bob(Q, K, V, dO, a, b, c, causal=m)["gK"]):
        assert np.array_equal(f(one), f(True))
    each = oracle.Segments(np.arange(N))
    O, L = oracle.forward(Q, K, V, scale=0.5, causal=each)
    assert rel(O, V) <= 1e-15 and rel(L, 0.5 * (Q * K).sum(axis=1)) <= 1e-15
    g = oracle.backward(Q, K, V, dO, causal=each)
    assert np.abs(g["dQ"]).max() == 0 and np.abs(g["dK"]).max() == 0 and rel(g["dV"], dO) <= 1e-15
    h = oracle.bob(Q, K, V, dO, a, b, c, causal=each)
    assert max(np.abs(h[k]).max() for k in ("gQ", "gK", "gV")) <= 1e-14 and rel(h["gdO"], c) <= 1e-15


@pytest.mark.parametrize("Br,Bc", [(1, 1), (3, 5), (16, 16), (7, 33)])
def test_segments_online_softmax_equals_two_pass(Br, Bc):
    seg = np.repeat(np.arange(5), [6, 1, 12, 3, 11])
    N, d = len(seg), 5
    Q, K, V = rnd(206, N, d), rnd(207, N, d), rnd(208, N, d)
    m = oracle.Segments(seg, 5)
    O1, L1 = oracle.forward_online(Q, K, V, Br, Bc, causal=m)
    O2, L2 = oracle.forward(Q, K, V, causal=m)
    assert rel(O1, O2) <= 1e-13 and rel(L1, L2) <= 1e-13


def test_segments_backward_fd_and_bob_hvp_jvp():
    seg = np.array([0, 0, 0, 1, 1, 1, 1, 2, 3, 3, 3])
    N, d = len(seg), 4
    Q, K, V, dO, a, b, c = (x * 0.8 for x in slice_set(N, d, 209))
    s, h, m = 0.6, 1e-5, oracle.Segments(seg)
    g = oracle.backward(Q, K, V, dO, scale=s, causal=m)
    top = 0.0
    fds = []
    for k, X in (("dQ", 0), ("dK", 1), ("dV", 2)):
        def f(Y, X=X):
            args = [Q, K, V]
            args[X] = Y
            O, _ = oracle.forward(*args, scale=s, causal=m)
            return float((O * dO).sum())
        fd = fd_grad(f, (Q, K, V)[X])
        fds.append((k, fd))
        top = max(top, np.abs(fd).max())
    for k, fd in fds:
        assert np.abs(g[k] - fd).max() <= 1e-8 * max(top, 1e-3), k
    out = oracle.bob(Q, K, V, dO, a, b, c, scale=s, causal=m)

    def gr(Q, K, V):
        x = oracle.backward(Q, K, V, dO, scale=s, causal=m)
        return x["dQ"], x["dK"], x["dV"]
    gp, gm = gr(Q + h * a, K + h * b, V + h * c), gr(Q - h * a, K - h * b, V - h * c)
    fd = [(p_ - m_) / (2 * h) for p_, m_ in zip(gp, gm)]
    top = max(np.abs(x).max() for x in fd)
    for name, want in zip(("gQ", "gK", "gV"), fd):
        assert np.abs(out[name] - want).max() <= 1e-8 * max(top, 1e-3), name
    Op, _ = oracle.forward(Q + h * a, K + h * b, V + h * c, scale=s, causal=m)
    Om, _ = oracle.forward(Q - h * a, K - h * b, V - h * c, scale=s, causal=m)
    jvp = (Op - Om) / (2 * h)
    assert np.abs(out["gdO"] - jvp).max() <= 1e-8 * max(np.abs(jvp).max(), 1e-3)


def test_segments_streaming_passes_and_sampling():
    seg = np.repeat(np.arange(4), [10, 3, 15, 7])
    N, d = len(seg), 5
    Q, K, V, dO, a, b, c = slice_set(N, d, 210)
    m = oracle.Segments(seg, 9)
    ref = oracle.bob(Q, K, V, dO, a, b, c, causal=m)
    O, L = oracle.forward(Q, K, V, causal=m)
    row = oracle.bob_row_pass(Q, K, V, dO, a, b, c, O, L, 6, causal=m)
    gK, gV = oracle.bob_col_pass(Q, K, V, dO, a, b, c, L, row["D"], row["E"], row["F"], 5, causal=m)
    for got, want in ((row["gQ"], ref["gQ"]), (row["gdO"], ref["gdO"]), (gK, ref["gK"]), (gV, ref["gV"])):
        assert rel(got, want) <= 1e-12
    rows, cols = np.array([0, 34, 12, 13]), np.array([0, 20, 34])
    r = oracle.bob_rows(Q, K, V, dO, a, b, c, rows, causal=m)
    assert rel(r["gQ"], ref["gQ"][rows]) <= 1e-13 and rel(r["gdO"], ref["gdO"][rows]) <= 1e-13
    gKc, gVc = oracle.bob_cols(Q, K, V, dO, a, b, c, cols, causal=m)
    assert rel(gKc, ref["gK"][cols]) <= 1e-13 and rel(gVc, ref["gV"][cols]) <= 1e-13


def test_segments_batched_helpers_use_each_rows_ids():
    seg = np.array([np.repeat([0, 1], [5, 9]), np.repeat([3, 4, 5], [2, 2, 10])])
    B, H, N, d = 2, 2, 14, 4
    r = np.random.default_rng(211)
    X = [r.standard_normal((B, H, N, d)) for _ in range(4)]
    out = oracle.backward_all(*X, causal=oracle.SegmentsBatch(seg))
    for bb in range(B):
        for hh in range(H):
            g = oracle.backward(*(x[bb, hh] for x in X), causal=oracle.Segments(seg[bb]))
            assert np.array_equal(out["dQ"][bb, hh], g["dQ"]) and np.array_equal(out["dK"][bb, hh], g["dK"])


def test_planted_mistake_segments_ignored_in_backward_is_caught(monkeypatch):
    """A backward that drops the segment test (but keeps it in the forward) breaks the
    block-diagonal pin."""
    seg = np.repeat(np.arange(3), [4, 6, 5])
    N, d = len(seg), 4
    Q, K, V, dO = slice_set(N, d, 212)[:4]
    real = A.hidden
    monkeypatch.setattr(A, "hidden", lambda rows, keys, causal: real(rows, keys, True if isinstance(causal, A.Segments) else causal))
    g = oracle.backward(Q, K, V, dO, causal=oracle.Segments(seg))
    monkeypatch.setattr(A, "hidden", real)
    r = _runs(seg)[1]
    gr = oracle.backward(Q[r], K[r], V[r], dO[r])
    assert rel(g["dQ"][r], gr["dQ"]) > 1e-3
