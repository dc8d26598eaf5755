"""CPU fp64 oracle for softmax attention (causal by default), its backward and its backward-over-backward.

TEST INFRASTRUCTURE ONLY.  Nothing in the library's product path may import this
module: only the tests, the smoke check and the benchmark's CPU-baseline leg use it.
It shares no code with the CUDA path.

Everything here is the plain definition written out in float64 with S and P
materialised, one block of query rows at a time (with the causal mask the rows of
a block see keys 0..max(row); without it, every key).  Row blocking changes nothing
in the arithmetic: every output row or column is the same sum of the same terms.

Notation (one (batch, head) slice; Q, K, V, dO, a, b, c are [N, d]):
  s = 1/sqrt(d) unless given;  S = s Q K^T with S_ij = -inf for j > i when causal
  (the default; causal=False keeps every key);
  L_i = log sum_j exp(S_ij);   P = exp(S - L);   O = P V.
Sources:
  * forward and stored statistics: "Flash attention for trading models", sections
    "Why attention is memory-bound" (S = QK^T/sqrt(d_k), softmax, PV) and
    "Backward pass: recompute instead of store" (only O and the softmax statistics
    are kept; we keep their single-number form, the log-sum-exp);
  * causal masking: same page, section "Causal masking is where trading gets a discount";
    the causal sliding window (``Window``), one of the flexible masks the FlashBoB page
    names as a next extension, is accepted wherever `causal` is;
  * first backward: the vector-Jacobian product of O with respect to Q, K, V given dO.
    The pages describe it only as a recompute from Q, K and the statistics, so the
    oracle writes out the standard derivative (dP = dO V^T, D_i = sum_k dO_ik O_ik,
    dS = P*(dP - D), dQ = s dS K, dK = s dS^T Q, dV = P^T dO);
  * GProj: "FlashAttention bf16 gradient and GProj" page, sections "How the zero sum
    turns into a false gradient" (exact dS rows sum to zero; bf16 rounding of dS
    leaves a residual that multiplies the mean key; GProj measures the remaining row
    mass of the rounded dS and subtracts the matching share of the probabilities);
    the same projection applied to the dS that BoB's dS b and dS^T a products see
    is emulated by ``bob_bf16_dS``;
  * backward-over-backward (BoB): "FlashBoB: second-order attention" page, section
    "Why go backward through an already computed gradient": the gradient of the first
    backward's outputs (dQ, dK, dV) with respect to Q, K, V and the incoming dO,
    contracted with cotangents a = gdQ, b = gdK, c = gdV.  The closed form below is
    derived by hand from that definition (see ``bob``); the two per-row scalars E_i
    and F_i are the "two scalar states" of the section "Two scalar states replace
    quadratic tensors".
"""
from __future__ import annotations

import numpy as np

NEG_INF = -np.inf


class Window:
    """Causal sliding-window mask: key j is visible to query i iff i - W < j <= i.

    The FlashBoB page ("When FlashBoB changes the engineering plan") names flexible
    masks among the next extensions without fixing one; this is the banded causal
    mask.  Every function's `causal` argument accepts it in place of True (which is
    the window without a lower limit); each row keeps its own key, so no row is empty.
    """

    def __init__(self, W: int):
        if int(W) < 1:
            raise ValueError("window must be >= 1")
        self.W = int(W)

    def __repr__(self):
        return f"Window({self.W})"

    def __eq__(self, other):
        return isinstance(other, Window) and other.W == self.W

    def __hash__(self):
        return hash(("Window", self.W))


class Segments:
    """Document (segment) mask over one sequence: key j is visible to query i iff j <= i
    and the two tokens carry the same segment id, seg[j] == seg[i] (packed documents
    attend only within their own document); with W > 0 the causal window i - W < j
    applies as well.

    A second flexible mask beside the window (the FlashBoB page, "When FlashBoB changes
    the engineering plan", names flexible masks among the next extensions): the ids of
    a packed batch row are non-decreasing, each document one run, so every row keeps
    its own key and its visible keys form one contiguous range.  Accepted wherever
    `causal` is, for one (batch, head) slice; ``SegmentsBatch`` carries the ids of
    every batch row for the batched helpers."""

    def __init__(self, seg, W: int = 0):
        self.seg = np.asarray(seg, dtype=np.int64).reshape(-1)
        if int(W) < 0:
            raise ValueError("window must be >= 0")
        self.W = int(W)

    def __repr__(self):
        return f"Segments(n={len(self.seg)}, W={self.W})"


class SegmentsBatch:
    """Segment ids [B, N] of a batch: slice (b, h) uses ``Segments(seg[b], W)``."""

    def __init__(self, seg, W: int = 0):
        self.seg = np.asarray(seg, dtype=np.int64)
        self.W = int(W)

    def for_batch(self, b):
        return Segments(self.seg[b], self.W)


def hidden(rows, keys, causal):
    """Boolean [len(rows), len(keys)]: True where the key is masked for the row
    (causal: j > i; a Window also masks j <= i - W; Segments also masks keys of another
    segment; causal=False masks nothing)."""
    r = np.asarray(rows)[:, None]
    k = np.asarray(keys)[None, :]
    if not causal:
        return np.zeros((r.shape[0], k.shape[1]), bool)
    m = k > r
    if isinstance(causal, Window):
        m |= k <= r - causal.W
    if isinstance(causal, Segments):
        m |= causal.seg[k] != causal.seg[r]
        if causal.W:
            m |= k <= r - causal.W
    return m


def _f64(x):
    return np.asarray(x, dtype=np.float64)


def default_scale(d: int) -> float:
    return 1.0 / np.sqrt(d)


def _blocks(rows: np.ndarray, block: int):
    for s0 in range(0, len(rows), block):
        yield rows[s0:s0 + block]


def _panel_budget(n_keys: int, mats: int = 8) -> int:
    """Rows per block so that `mats` fp64 matrices of [rows, n_keys] stay near 1 GiB."""
    return max(1, min(4096, int((1 << 30) // (8 * mats * max(n_keys, 1)))))


# ---------------------------------------------------------------------------
# Forward (two-pass softmax, materialised)
# ---------------------------------------------------------------------------

def scores(Q, K, rows, scale, causal=True):
    """S[rows, keys] = scale * Q[rows] K^T: with the causal mask the keys are
    0..max(rows) and S = -inf for j > i; without it, all keys."""
    rows = np.asarray(rows)
    if not causal:
        return scale * (Q[rows] @ K.T)
    kmax = int(rows.max()) + 1
    S = scale * (Q[rows] @ K[:kmax].T)
    S[hidden(rows, np.arange(kmax), causal)] = NEG_INF
    return S


def softmax_rows(S):
    """Two-pass softmax of each row: max first, then exponentials and their sum.

    Returns (P, L) with L_i = m_i + log sum_j exp(S_ij - m_i) the natural-log
    log-sum-exp."""
    m = S.max(axis=1)
    E = np.exp(S - m[:, None])
    l = E.sum(axis=1)
    L = m + np.log(l)
    return E / l[:, None], L


def forward(Q, K, V, scale=None, block=None, causal=True):
    """Attention forward for one slice: returns (O [N,d], L [N])."""
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    N, d = Q.shape
    scale = default_scale(d) if scale is None else scale
    O = np.empty_like(Q)
    L = np.empty(N)
    block = block or _panel_budget(N, 3)
    for r in _blocks(np.arange(N), block):
        P, Lr = softmax_rows(scores(Q, K, r, scale, causal))
        O[r] = P @ V[:P.shape[1]]
        L[r] = Lr
    return O, L


def forward_rows(Q, K, V, rows, scale=None, causal=True):
    """O[rows], L[rows] only (a causal row needs keys 0..row): for sampled checks at large N."""
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    scale = default_scale(Q.shape[1]) if scale is None else scale
    rows = np.asarray(rows)
    O = np.empty((len(rows), Q.shape[1]))
    L = np.empty(len(rows))
    order = np.argsort(rows)
    for blk in _blocks(order, _panel_budget(int(rows.max()) + 1 if causal else len(K), 3)):
        P, Lr = softmax_rows(scores(Q, K, rows[blk], scale, causal))
        O[blk] = P @ V[:P.shape[1]]
        L[blk] = Lr
    return O, L


def forward_online(Q, K, V, Br, Bc, scale=None, causal=True):
    """The tiled forward with the online softmax recurrence, in the pages' order.

    "Flash attention for trading models", sections "The Flash Attention algorithm"
    and "Online softmax recurrence": Q is cut into blocks of Br rows and K, V into
    blocks of Bc rows.  For each query block the running max m, running sum l and
    the output O start at (-inf, 0, 0); every key/value block contributes its local
    max, its exponentials and local sum, and the running state is rescaled so that
    it is as if the new max had been known from the start.  Key blocks entirely in
    the future of a query block are skipped when causal (section on causal masking).  Exact
    arithmetic gives the two-pass result; this is used only to pin that fact.
    Returns (O, L) with L = m + log l.
    """
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    N, d = Q.shape
    scale = default_scale(d) if scale is None else scale
    O = np.zeros((N, d))
    L = np.empty(N)
    for q0 in range(0, N, Br):
        qi = np.arange(q0, min(q0 + Br, N))
        Oi = np.zeros((len(qi), d))
        mi = np.full(len(qi), NEG_INF)
        li = np.zeros(len(qi))
        for k0 in range(0, N, Bc):
            kj = np.arange(k0, min(k0 + Bc, N))
            if causal and kj[0] > qi[-1]:
                break  # the whole block is in the future of every query: never loaded
            Sij = scale * (Q[qi] @ K[kj].T)
            if causal:
                Sij[hidden(qi, kj, causal)] = NEG_INF
            mij = Sij.max(axis=1)
            # a row whose keys in this block are all masked contributes nothing
            live = np.isfinite(mij)
            Pij = np.zeros_like(Sij)
            Pij[live] = np.exp(Sij[live] - mij[live, None])
            lij = Pij.sum(axis=1)
            m_new = np.maximum(mi, mij)
            fin = np.isfinite(m_new)  # (the others have seen nothing: both factors 0)
            a_old = np.where(np.isfinite(mi), np.exp(np.where(np.isfinite(mi), mi, 0.0) - np.where(fin, m_new, 0.0)), 0.0)
            a_new = np.where(live, np.exp(np.where(live, mij, 0.0) - np.where(fin, m_new, 0.0)), 0.0)
            l_new = li * a_old + lij * a_new
            # rows that have seen no visible key yet (possible under a window) keep
            # their starting state (-inf, 0, 0)
            seen = l_new > 0
            l_div = np.where(seen, l_new, 1.0)
            Oi = np.where(seen[:, None],
                          Oi * (li * a_old / l_div)[:, None] + (Pij @ V[kj]) * (a_new / l_div)[:, None], Oi)
            mi, li = m_new, l_new
        O[qi] = Oi
        L[qi] = mi + np.log(li)
    return O, L


# ---------------------------------------------------------------------------
# Row-block quantities shared by the first and second backward
# ---------------------------------------------------------------------------

def _row_terms(Q, K, V, dO, rows, scale, a=None, b=None, c=None, causal=True):
    """All per-row-block tiles of the first backward (and of BoB if a, b, c given).

    Keys are 0..max(rows) when causal, else all keys.  Returns a dict of
    [len(rows), n_keys] matrices and per-row vectors.  Everything is computed from
    Q, K, V, dO alone (the statistics are recomputed, as the oracle has no stored
    ones to trust)."""
    S = scores(Q, K, rows, scale, causal)
    P, L = softmax_rows(S)
    nk = P.shape[1]
    dP = dO[rows] @ V[:nk].T
    D = (P * dP).sum(axis=1)              # = sum_k dO_ik O_ik
    dS = P * (dP - D[:, None])
    t = dict(P=P, L=L, dP=dP, D=D, dS=dS, nk=nk)
    if a is not None:
        G = scale * (a[rows] @ K[:nk].T + Q[rows] @ b[:nk].T)
        Hm = dO[rows] @ c[:nk].T
        if causal:
            mask = hidden(rows, np.arange(nk), causal)
            G[mask] = 0.0
            Hm[mask] = 0.0
        E = (P * G).sum(axis=1)
        dPbar = P * (G - E[:, None])
        Pbar = G * (dP - D[:, None]) - E[:, None] * dP + Hm
        F = (P * Pbar).sum(axis=1)
        Sbar = P * (Pbar - F[:, None])
        t.update(G=G, Hm=Hm, E=E, dPbar=dPbar, Pbar=Pbar, F=F, Sbar=Sbar)
    return t


# ---------------------------------------------------------------------------
# First backward
# ---------------------------------------------------------------------------

def backward(Q, K, V, dO, scale=None, block=None, causal=True):
    """Vector-Jacobian product of O = attn(Q, K, V) against dO, for one slice.

    Returns dict(dQ, dK, dV, D, L)."""
    Q, K, V, dO = map(_f64, (Q, K, V, dO))
    N, d = Q.shape
    scale = default_scale(d) if scale is None else scale
    dQ, dK, dV = np.zeros((N, d)), np.zeros((N, d)), np.zeros((N, d))
    D, L = np.empty(N), np.empty(N)
    for r in _blocks(np.arange(N), block or _panel_budget(N, 4)):
        t = _row_terms(Q, K, V, dO, r, scale, causal=causal)
        nk = t["nk"]
        dQ[r] = scale * (t["dS"] @ K[:nk])
        dK[:nk] += scale * (t["dS"].T @ Q[r])
        dV[:nk] += t["P"].T @ dO[r]
        D[r], L[r] = t["D"], t["L"]
    return dict(dQ=dQ, dK=dK, dV=dV, D=D, L=L)


def backward_rows(Q, K, V, dO, rows, scale=None, causal=True):
    """dQ[rows] only."""
    Q, K, V, dO = map(_f64, (Q, K, V, dO))
    scale = default_scale(Q.shape[1]) if scale is None else scale
    rows = np.asarray(rows)
    out = np.empty((len(rows), Q.shape[1]))
    order = np.argsort(rows)
    for blk in _blocks(order, _panel_budget(int(rows.max()) + 1 if causal else len(K), 4)):
        t = _row_terms(Q, K, V, dO, rows[blk], scale, causal=causal)
        out[blk] = scale * (t["dS"] @ K[:t["nk"]])
    return out


def backward_cols(Q, K, V, dO, cols, scale=None, causal=True):
    """dK[cols], dV[cols] only.  Causal: needs every row i >= min(cols), cheap for late
    columns; otherwise every row."""
    Q, K, V, dO = map(_f64, (Q, K, V, dO))
    N, d = Q.shape
    scale = default_scale(d) if scale is None else scale
    cols = np.asarray(cols)
    dK, dV = np.zeros((len(cols), d)), np.zeros((len(cols), d))
    for r in _blocks(np.arange(int(cols.min()) if causal else 0, N), _panel_budget(N, 4)):
        t = _row_terms(Q, K, V, dO, r, scale, causal=causal)
        ok = cols < t["nk"]
        cc = cols[ok]
        dK[ok] += scale * (t["dS"][:, cc].T @ Q[r])
        dV[ok] += t["P"][:, cc].T @ dO[r]
    return dK, dV


def bf16_round(x):
    """Round float64 values to the nearest bfloat16 (ties to even), returned as float64.

    Goes through float32 first (as a kernel holding fp32 values would)."""
    f = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    u = f.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32).astype(np.float64)


def backward_bf16_dS(Q, K, V, dO, gproj, scale=None, block=None, causal=True):
    """Emulate a backward that rounds dS to bf16 before the dS K and dS^T Q products.

    Without GProj: dQ = s bf16(dS) K, dK = s bf16(dS)^T Q.  With GProj (GProj page,
    "How the zero sum turns into a false gradient"): each rounded row
    dS^_i = bf16(dS_i) has remaining mass r_i = sum_j dS^_ij; the projection
    subtracts r_i times the row's share of the probabilities actually fed to the
    product, P^_ij / sum_k P^_ik with P^ = bf16(P), so that the projected row sums to
    zero exactly.  Everything except the two roundings is fp64.  Used only to show
    what the rounding does; the reference for errors is always ``backward``.
    Returns dict(dQ, dK, r, rho, l1, dS_proj_rowsum_rel): r_i and rho_i = r_i / sum_k P^_ik
    per row (both 0 without GProj), l1_i = sum_j |dS~_ij| (the L1 norm of the row the
    products see: dS~ with GProj, dS^ without), and the worst row's
    |sum_j dS~_ij| / sum_j |dS~_ij| over rows with nonzero L1.
    """
    Q, K, V, dO = map(_f64, (Q, K, V, dO))
    N, d = Q.shape
    scale = default_scale(d) if scale is None else scale
    dQ, dK = np.zeros((N, d)), np.zeros((N, d))
    r_all, rho_all, l1_all = np.zeros(N), np.zeros(N), np.zeros(N)
    worst = 0.0
    for r in _blocks(np.arange(N), block or _panel_budget(N, 4)):
        t = _row_terms(Q, K, V, dO, r, scale, causal=causal)
        nk = t["nk"]
        dSh = bf16_round(t["dS"])
        if gproj:
            res = dSh.sum(axis=1)
            Ph = bf16_round(t["P"])
            rho = res / Ph.sum(axis=1)
            dSt = dSh - rho[:, None] * Ph
            r_all[r], rho_all[r] = res, rho
        else:
            dSt = dSh
        l1 = np.abs(dSt).sum(axis=1)
        l1_all[r] = l1
        nz = l1 > 0
        if nz.any():
            worst = max(worst, float(np.max(np.abs(dSt.sum(axis=1))[nz] / l1[nz])))
        dQ[r] = scale * (dSt @ K[:nk])
        dK[:nk] += scale * (dSt.T @ Q[r])
    return dict(dQ=dQ, dK=dK, r=r_all, rho=rho_all, l1=l1_all, dS_proj_rowsum_rel=worst)


# ---------------------------------------------------------------------------
# Backward over backward (FlashBoB)
# ---------------------------------------------------------------------------

def bob(Q, K, V, dO, a, b, c, scale=None, block=None, keep=False, causal=True):
    """Backward-over-backward for one slice, closed form.

    Let Phi(Q, K, V, dO) = (dQ, dK, dV) be the first backward and
    psi = <a, dQ> + <b, dK> + <c, dV>.  Writing G = s(a K^T + Q b^T) and
    H = dO c^T, psi = sum_ij dS_ij G_ij + sum_ij P_ij H_ij.  Differentiating with
    dS = P*(dP - D), D_i = sum_j P_ij dP_ij, dP = dO V^T and the softmax Jacobian:
        E_i   = sum_j P_ij G_ij                     (first scalar state)
        dPbar = P*(G - E)                           (d psi / d dP)
        Pbar  = G*(dP - D) - E*dP + H               (d psi / d P)
        F_i   = sum_j P_ij Pbar_ij                  (second scalar state)
        Sbar  = P*(Pbar - F)                        (d psi / d S)
        gQ  = s (dS b + Sbar K)      gK  = s (dS^T a + Sbar^T Q)
        gV  = dPbar^T dO             gdO = P c + dPbar V
    Returns dict(gQ, gK, gV, gdO, E, F, D, L) (and the tiles if keep=True and the
    slice is done in one block).
    """
    Q, K, V, dO, a, b, c = map(_f64, (Q, K, V, dO, a, b, c))
    N, d = Q.shape
    scale = default_scale(d) if scale is None else scale
    gQ, gK, gV, gdO = (np.zeros((N, d)) for _ in range(4))
    E, F, D, L = (np.empty(N) for _ in range(4))
    kept = None
    for r in _blocks(np.arange(N), block or _panel_budget(N, 12)):
        t = _row_terms(Q, K, V, dO, r, scale, a, b, c, causal=causal)
        nk = t["nk"]
        gQ[r] = scale * (t["dS"] @ b[:nk] + t["Sbar"] @ K[:nk])
        gK[:nk] += scale * (t["dS"].T @ a[r] + t["Sbar"].T @ Q[r])
        gV[:nk] += t["dPbar"].T @ dO[r]
        gdO[r] = t["P"] @ c[:nk] + t["dPbar"] @ V[:nk]
        E[r], F[r], D[r], L[r] = t["E"], t["F"], t["D"], t["L"]
        kept = t
    out = dict(gQ=gQ, gK=gK, gV=gV, gdO=gdO, E=E, F=F, D=D, L=L)
    if keep:
        out["tiles"] = kept
    return out


def bob_bf16_dS(Q, K, V, dO, a, b, c, gproj, scale=None, block=None, causal=True, rnd=None):
    """Emulate a BoB whose dS b and dS^T a products see bf16(dS), with or without GProj.

    The products of the closed form (``bob``) that contract dS, gQ's dS b and gK's
    dS^T a, get the rounded row dS^ = rnd(dS) (rnd defaults to ``bf16_round``).
    Without GProj that is all.  With GProj the rounded row is projected back to zero
    sum as the GProj page describes for the first backward ("FlashAttention bf16
    gradient and GProj", "How the zero sum turns into a false gradient": measure the
    remaining row mass r_i = sum_j dS^_ij and subtract the matching share of the
    probabilities actually fed to the products, P^ = rnd(P)):
        dS~ = dS^ - (r_i / sum_k P^_ik) P^,
        gQ = s (dS~ b + Sbar K),   gK = s (dS~^T a + Sbar^T Q);
    gV, gdO and everything else are the exact fp64 values.  Used only to show what
    the rounding and the projection do; the reference for errors is always ``bob``.
    Returns dict(gQ, gK, gV, gdO, r, rho, l1_dS, l1_Sbar, dS_rowsum_rel): per row the
    residual r_i, the coefficient rho_i (0 without GProj), the L1 norms of the row of
    dS~ (dS^ without GProj) and of Sbar, and the worst row's
    |sum_j dS~_ij| / sum_j |dS~_ij| over rows with nonzero L1.
    """
    rnd = bf16_round if rnd is None else rnd
    Q, K, V, dO, a, b, c = map(_f64, (Q, K, V, dO, a, b, c))
    N, d = Q.shape
    scale = default_scale(d) if scale is None else scale
    gQ, gK, gV, gdO = (np.zeros((N, d)) for _ in range(4))
    r_all, rho_all, l1_all, l1s_all = np.zeros(N), np.zeros(N), np.zeros(N), np.zeros(N)
    worst = 0.0
    for r in _blocks(np.arange(N), block or _panel_budget(N, 12)):
        t = _row_terms(Q, K, V, dO, r, scale, a, b, c, causal=causal)
        nk = t["nk"]
        dSh = rnd(t["dS"])
        if gproj:
            res = dSh.sum(axis=1)
            Ph = rnd(t["P"])
            rho = res / Ph.sum(axis=1)
            dSt = dSh - rho[:, None] * Ph
            r_all[r], rho_all[r] = res, rho
        else:
            dSt = dSh
            r_all[r] = dSh.sum(axis=1)
        l1 = np.abs(dSt).sum(axis=1)
        l1_all[r], l1s_all[r] = l1, np.abs(t["Sbar"]).sum(axis=1)
        nz = l1 > 0
        if nz.any():
            worst = max(worst, float(np.max(np.abs(dSt.sum(axis=1))[nz] / l1[nz])))
        gQ[r] = scale * (dSt @ b[:nk] + t["Sbar"] @ K[:nk])
        gK[:nk] += scale * (dSt.T @ a[r] + t["Sbar"].T @ Q[r])
        gV[:nk] += t["dPbar"].T @ dO[r]
        gdO[r] = t["P"] @ c[:nk] + t["dPbar"] @ V[:nk]
    return dict(gQ=gQ, gK=gK, gV=gV, gdO=gdO, r=r_all, rho=rho_all, l1_dS=l1_all, l1_Sbar=l1s_all,
                dS_rowsum_rel=worst)


def bob_rows(Q, K, V, dO, a, b, c, rows, scale=None, causal=True):
    """gQ[rows], gdO[rows] and the row states (E, F) only."""
    Q, K, V, dO, a, b, c = map(_f64, (Q, K, V, dO, a, b, c))
    d = Q.shape[1]
    scale = default_scale(d) if scale is None else scale
    rows = np.asarray(rows)
    gQ, gdO = np.empty((len(rows), d)), np.empty((len(rows), d))
    E, F = np.empty(len(rows)), np.empty(len(rows))
    order = np.argsort(rows)
    for blk in _blocks(order, _panel_budget(int(rows.max()) + 1 if causal else len(K), 12)):
        t = _row_terms(Q, K, V, dO, rows[blk], scale, a, b, c, causal=causal)
        nk = t["nk"]
        gQ[blk] = scale * (t["dS"] @ b[:nk] + t["Sbar"] @ K[:nk])
        gdO[blk] = t["P"] @ c[:nk] + t["dPbar"] @ V[:nk]
        E[blk], F[blk] = t["E"], t["F"]
    return dict(gQ=gQ, gdO=gdO, E=E, F=F)


def bob_cols(Q, K, V, dO, a, b, c, cols, scale=None, causal=True):
    """gK[cols], gV[cols] only.  Causal: needs every row i >= min(cols), cheap for late
    columns; otherwise every row."""
    Q, K, V, dO, a, b, c = map(_f64, (Q, K, V, dO, a, b, c))
    N, d = Q.shape
    scale = default_scale(d) if scale is None else scale
    cols = np.asarray(cols)
    gK, gV = np.zeros((len(cols), d)), np.zeros((len(cols), d))
    for r in _blocks(np.arange(int(cols.min()) if causal else 0, N), _panel_budget(N, 12)):
        t = _row_terms(Q, K, V, dO, r, scale, a, b, c, causal=causal)
        ok = cols < t["nk"]
        cc = cols[ok]
        gK[ok] += scale * (t["dS"][:, cc].T @ a[r] + t["Sbar"][:, cc].T @ Q[r])
        gV[ok] += t["dPbar"][:, cc].T @ dO[r]
    return gK, gV


def bob_row_pass(Q, K, V, dO, a, b, c, O, L, Bc, scale=None, causal=True):
    """The BoB row pass in its streaming form, for one slice.

    FlashBoB page, section "Two scalar states replace quadratic tensors": a block of
    query rows stays on chip while key/value blocks stream past; probabilities are
    recomputed from the stored normaliser L; row sums are accumulated, and the
    corrections that need the finished row are applied once the row is complete.
    Per row i, over key blocks (keys <= i when causal, else all keys):
        P = exp(S - L), dP = dO V^T, dS = P*(dP - D) with D_i = dO_i . O_i,
        G = s(a K^T + Q b^T), H = dO c^T, W = G*dS + P*H,
        E_i += sum P*G,  F'_i += sum W,
        X_i += P c + (P*G) V,  Y_i += dS b + W K,  Z_i += dS K,  U_i += P K.
    After the last block:
        gdO_i = X_i - E_i O_i,  gQ_i = s (Y_i - E_i Z_i - F'_i U_i),  F_i = F'_i - E_i D_i.
    These follow from the closed form in ``bob`` by linearity in E and F (shown in
    the docstring of ``bob`` and checked against it in the tests).
    Returns dict(gQ, gdO, E, F, D).
    """
    Q, K, V, dO, a, b, c, O, L = map(_f64, (Q, K, V, dO, a, b, c, O, L))
    N, d = Q.shape
    scale = default_scale(d) if scale is None else scale
    D = (dO * O).sum(axis=1)
    E, Fp = np.zeros(N), np.zeros(N)
    X, Y, Z, U = (np.zeros((N, d)) for _ in range(4))
    rows = np.arange(N)
    for k0 in range(0, N, Bc):
        kj = np.arange(k0, min(k0 + Bc, N))
        live = rows >= k0 if causal else rows >= 0  # rows that see at least one key here
        r = rows[live]
        S = scale * (Q[r] @ K[kj].T)
        mask = hidden(r, kj, causal)
        P = np.exp(np.where(mask, NEG_INF, S) - L[r, None])
        dP = dO[r] @ V[kj].T
        dS = P * (dP - D[r, None])
        G = np.where(mask, 0.0, scale * (a[r] @ K[kj].T + Q[r] @ b[kj].T))
        Hm = np.where(mask, 0.0, dO[r] @ c[kj].T)
        W = G * dS + P * Hm
        E[r] += (P * G).sum(axis=1)
        Fp[r] += W.sum(axis=1)
        X[r] += P @ c[kj] + (P * G) @ V[kj]
        Y[r] += dS @ b[kj] + W @ K[kj]
        Z[r] += dS @ K[kj]
        U[r] += P @ K[kj]
    gdO = X - E[:, None] * O
    gQ = scale * (Y - E[:, None] * Z - Fp[:, None] * U)
    return dict(gQ=gQ, gdO=gdO, E=E, F=Fp - E * D, D=D)


def bob_col_pass(Q, K, V, dO, a, b, c, L, D, E, F, Br, scale=None, causal=True):
    """The BoB column pass in its streaming form, for one slice.

    FlashBoB page, same section: a block of keys stays on chip while query rows
    stream past; the probabilities are recomputed and the stored row states (L, D,
    E, F) of each streamed row are read back.  Per key j, over query rows i >= j
    (all rows when not causal):
        dPbar = P*(G - E),  Sbar = P*(G*(dP - D) - E*dP + H - F),
        gV_j += dPbar^T dO,  gK_j += s (dS^T a + Sbar^T Q).
    Returns (gK, gV)."""
    Q, K, V, dO, a, b, c, L, D, E, F = map(_f64, (Q, K, V, dO, a, b, c, L, D, E, F))
    N, d = Q.shape
    scale = default_scale(d) if scale is None else scale
    gK, gV = np.zeros((N, d)), np.zeros((N, d))
    for q0 in range(0, N, Br):
        qi = np.arange(q0, min(q0 + Br, N))
        kj = np.arange(0, qi[-1] + 1) if causal else np.arange(N)
        mask = hidden(qi, kj, causal)
        S = scale * (Q[qi] @ K[kj].T)
        P = np.exp(np.where(mask, NEG_INF, S) - L[qi, None])
        dP = dO[qi] @ V[kj].T
        dS = P * (dP - D[qi, None])
        G = np.where(mask, 0.0, scale * (a[qi] @ K[kj].T + Q[qi] @ b[kj].T))
        Hm = np.where(mask, 0.0, dO[qi] @ c[kj].T)
        dPbar = P * (G - E[qi, None])
        Sbar = P * (G * (dP - D[qi, None]) - E[qi, None] * dP + Hm - F[qi, None])
        gV[kj] += dPbar.T @ dO[qi]
        gK[kj] += scale * (dS.T @ a[qi] + Sbar.T @ Q[qi])
    return gK, gV


# ---------------------------------------------------------------------------
# Batched helpers over [B, H, N, d]
# ---------------------------------------------------------------------------

def _each_slice(fn, *tensors, **kw):
    B, H = tensors[0].shape[:2]
    outs = None
    for bb in range(B):
        kb = dict(kw)
        if hasattr(kw.get("causal"), "for_batch"):  # per-batch segment ids
            kb["causal"] = kw["causal"].for_batch(bb)
        for hh in range(H):
            r = fn(*(t[bb, hh] for t in tensors), **kb)
            if outs is None:
                outs = {k: np.empty((B, H) + np.shape(v)) for k, v in r.items()
                        if isinstance(v, np.ndarray)}
            for k in outs:
                outs[k][bb, hh] = r[k]
    return outs


def _expand_kv(X, groups):
    """Grouped key/value heads: query head h of a [B, H, ...] problem reads key/value
    head h // groups of the [B, H / groups, ...] tensors."""
    return X if groups == 1 else np.repeat(X, groups, axis=1)


def _sum_groups(X, groups):
    """Gradient of a shared key/value head: the sum over the query heads that read it
    (chain rule through the repetition)."""
    if groups == 1:
        return X
    B, H = X.shape[:2]
    return X.reshape((B, H // groups, groups) + X.shape[2:]).sum(axis=2)


def forward_all(Q, K, V, scale=None, causal=True, groups=1):
    K, V = _expand_kv(K, groups), _expand_kv(V, groups)
    return _each_slice(lambda q, k, v, **kw: dict(zip(("O", "L"), forward(q, k, v, **kw))),
                       Q, K, V, scale=scale, causal=causal)


def backward_all(Q, K, V, dO, scale=None, causal=True, groups=1):
    out = _each_slice(backward, Q, _expand_kv(K, groups), _expand_kv(V, groups), dO, scale=scale, causal=causal)
    out["dK"], out["dV"] = _sum_groups(out["dK"], groups), _sum_groups(out["dV"], groups)
    return out


def bob_all(Q, K, V, dO, a, b, c, scale=None, causal=True, groups=1):
    """With grouped heads the first backward's dK, dV are sums over each group, so their
    cotangents b, c are per key/value head and enter every query head of the group; the
    per-head second derivatives of K and V are summed over the group the same way."""
    e = lambda X: _expand_kv(X, groups)
    out = _each_slice(bob, Q, e(K), e(V), dO, a, e(b), e(c), scale=scale, causal=causal)
    out["gK"], out["gV"] = _sum_groups(out["gK"], groups), _sum_groups(out["gV"], groups)
    return out


def bob_bf16_dS_all(Q, K, V, dO, a, b, c, gproj, scale=None, causal=True, groups=1):
    """``bob_bf16_dS`` over every (batch, head) slice, grouped heads as in ``bob_all``."""
    e = lambda X: _expand_kv(X, groups)
    out = _each_slice(lambda *x, **kw: bob_bf16_dS(*x, gproj, **kw), Q, e(K), e(V), dO, a, e(b), e(c),
                      scale=scale, causal=causal)
    out["gK"], out["gV"] = _sum_groups(out["gK"], groups), _sum_groups(out["gV"], groups)
    return out
