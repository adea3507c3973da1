"""Pins for the float64 oracle: checks against what the mathematics fixes.

Nothing here compares the oracle with itself.  The checks use exact rational
arithmetic, hand-written Gauss-Jordan inverses, closed forms, the Woodbury
identity through a library solve, a Cholesky factorisation, invariants and a
hand-worked example (tests/golden/).  ``test_mutants_are_caught`` then plants
plausible mistakes in a copy of the oracle's source (a dropped term, a wrong
sign or index, a transposed operand) and requires every mutant to fail at least
one check.

Formulas: "Mathematical Primitives" §2-§5 (Sherman-Morrison tracking, guard,
nudge, Woodbury, alpha = A s, state update and renormalisation); README "VLA v3"
items 1-5 (phi = ELU+1, normalised u, nudging, calibrated readout).
"""
from __future__ import annotations

import math
import os
import types
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from oracle import vla_ref
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------------------------
# independent helpers
# ----------------------------------------------------------------------------

def gj_inverse(M):
    """Gauss-Jordan inverse with partial pivoting; works on floats or Fractions."""
    n = len(M)
    aug = [list(M[i]) + [type(M[i][0])(1 if i == j else 0) for j in range(n)] for i in range(n)]
    for c in range(n):
        p = max(range(c, n), key=lambda r: abs(aug[r][c]))
        if aug[p][c] == 0:
            raise ZeroDivisionError("singular")
        aug[c], aug[p] = aug[p], aug[c]
        piv = aug[c][c]
        aug[c] = [x / piv for x in aug[c]]
        for r in range(n):
            if r != c and aug[r][c] != 0:
                f = aug[r][c]
                aug[r] = [x - f * y for x, y in zip(aug[r], aug[c])]
    return [row[n:] for row in aug]


def gj_inv_np(M):
    return np.array(gj_inverse([[float(x) for x in row] for row in np.asarray(M)]))


def phi_torch(x):
    """1 + ELU(x) through torch's own ELU, float64 (independent of the oracle's phi)."""
    t = torch.as_tensor(np.asarray(x, dtype=np.float64))
    return (torch.nn.functional.elu(t, alpha=1.0) + 1.0).numpy()


def rng(seed):
    return np.random.default_rng([seed, 99])


def unit_rows(x):
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def run(mod, q, k, v, u, A0, S0, n0, **kw):
    return mod.scan(q, k, v, u, A0, S0, n0, **kw)


def rand_case(seed, N, T, d, dv, r, *, spd_A0=False):
    g = rng(seed)
    q = g.normal(size=(N, T, d))
    k = g.normal(size=(N, T, d))
    v = g.normal(size=(N, T, dv))
    u = unit_rows(g.normal(size=(N, T, r, d)))
    if spd_A0:
        B = g.normal(size=(N, d, d))
        M0 = np.eye(d) + np.matmul(B, B.transpose(0, 2, 1)) / d
        A0 = np.stack([gj_inv_np(m) for m in M0])
    else:
        M0 = np.broadcast_to(np.eye(d), (N, d, d)).copy()
        A0 = M0.copy()
    S0 = np.zeros((N, dv, d))
    n0 = np.zeros((N, d))
    return q, k, v, u, A0, M0, S0, n0


def rel(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300))


# ----------------------------------------------------------------------------
# checks (each takes the oracle module, so mutants can be run through them)
# ----------------------------------------------------------------------------

def load_golden():
    rows = []
    with open(os.path.join(GOLDEN, "sm_d2_worked.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            rows.append([Fraction(x) for x in line.split()])
    return rows


def check_golden_worked(mod):
    rows = load_golden()
    T = len(rows)
    u = np.array([[float(r[1]), float(r[2])] for r in rows])[None, :, None, :]
    q = np.zeros((1, T, 2)); k = np.zeros((1, T, 2)); v = np.zeros((1, T, 1))
    _, _, _, _, tr = run(mod, q, k, v, u, np.eye(2)[None], np.zeros((1, 1, 2)), np.zeros((1, 2)),
                         P=0, eps_n=0.0, tau=1e30, trace=True, keep_A=True)
    for t, r in enumerate(rows):
        assert abs(tr["delta"][0, t, 0] - float(r[3])) < 1e-15
        want = np.array([float(x) for x in r[4:8]]).reshape(2, 2)
        assert np.max(np.abs(tr["A"][0, t] - want)) < 1e-15


def check_exact_rational(mod):
    g = rng(1)
    for d, A0diag in ((3, [1, 1, 1]), (4, [Fraction(1, 2), Fraction(1, 4), 1, 2])):
        T = 6
        u_fr = [[Fraction(int(x), 8) for x in g.integers(-8, 9, size=d)] for _ in range(T)]
        for row in u_fr:
            if all(x == 0 for x in row):
                row[0] = Fraction(1, 2)
        M = [[(Fraction(1) / Fraction(A0diag[i]) if i == j else Fraction(0)) for j in range(d)] for i in range(d)]
        u = np.array([[float(x) for x in row] for row in u_fr])[None, :, None, :]
        A0 = np.diag([float(x) for x in A0diag])[None]
        _, _, _, _, tr = run(mod, np.zeros((1, T, d)), np.zeros((1, T, d)), np.zeros((1, T, 1)), u, A0,
                             np.zeros((1, 1, d)), np.zeros((1, d)), P=0, eps_n=0.0, tau=1e30,
                             trace=True, keep_A=True)
        for t in range(T):
            M = [[M[i][j] + u_fr[t][i] * u_fr[t][j] for j in range(d)] for i in range(d)]
            exact = np.array([[float(x) for x in row] for row in gj_inverse(M)])
            assert rel(tr["A"][0, t], exact) < 1e-12


def check_gauss_jordan(mod):
    for seed, d, T, r, spd in ((2, 3, 64, 1, False), (3, 8, 128, 2, True), (4, 16, 256, 1, True)):
        q, k, v, u, A0, M0, S0, n0 = rand_case(seed, 2, T, d, 2, r, spd_A0=spd)
        _, _, _, _, tr = run(mod, q, k, v, u, A0, S0, n0, P=0, eps_n=0.0, tau=1e30,
                             trace=True, keep_A=True)
        M = M0.copy()
        for t in range(T):
            for i in range(r):
                M = M + u[:, t, i, :, None] * u[:, t, i, None, :]
            if t % 16 == 15 or t == T - 1:
                for p in range(2):
                    assert rel(tr["A"][p, t], gj_inv_np(M[p])) < 1e-10


def check_d1_closed_form(mod):
    g = rng(5)
    T, dv = 40, 3
    u = np.where(g.random(size=(1, T, 1, 1)) < 0.5, -1.0, 1.0)
    q = g.normal(size=(1, T, 1)); k = g.normal(size=(1, T, 1)); v = g.normal(size=(1, T, dv))
    o, A, S, n = run(mod, q, k, v, u, np.ones((1, 1, 1)), np.zeros((1, dv, 1)), np.zeros((1, 1)),
                     P=0, eps_n=0.0, tau=1e30)
    Sx = np.zeros(dv); nx = 0.0
    for t in range(T):
        a_t = 1.0 / (2.0 + t)                  # M_t = 1 + (t+1)  (t is 0-based here)
        fk = phi_torch(k[0, t, 0]); fq = phi_torch(q[0, t, 0])
        alpha = a_t * fk                       # s_t = phi(k)/sqrt(1)
        Sx = Sx + v[0, t] * alpha
        nx = nx + fk
        want = Sx * fq / (nx * fq + 1e-6)
        assert rel(o[0, t], want) < 1e-12
    assert abs(A[0, 0, 0] - 1.0 / (1.0 + T)) < 1e-15
    assert rel(S[0, :, 0], Sx) < 1e-12 and abs(n[0, 0] - nx) < 1e-12


def check_basis_cycling(mod):
    """u_t = e_{t mod d}: A stays diagonal, a_i <- a_i / (1 + a_i) on a hit,
    a <- a + eps on a nudge (global step g = t0 + t with g % P == 0)."""
    d, dv, T, P, eps, t0 = 4, 2, 23, 3, 1e-2, 1
    g = rng(6)
    u = np.zeros((1, T, 1, d))
    for t in range(T):
        u[0, t, 0, t % d] = 1.0
    q = g.normal(size=(1, T, d)); k = g.normal(size=(1, T, d)); v = g.normal(size=(1, T, dv))
    o, A, S, n, tr = run(mod, q, k, v, u, np.eye(d)[None], np.zeros((1, dv, d)), np.zeros((1, d)),
                         P=P, eps_n=eps, tau=1e30, t0=t0, trace=True, keep_A=True)
    a = np.ones(d)
    Sx = np.zeros((dv, d)); nx = np.zeros(d)
    for t in range(T):
        i = t % d
        a[i] = a[i] / (1.0 + a[i])
        if (t0 + t + 1) % P == 0:
            a = a + eps
        assert np.max(np.abs(tr["A"][0, t] - np.diag(a))) < 1e-15
        fk = phi_torch(k[0, t]); fq = phi_torch(q[0, t])
        alpha = a * fk / math.sqrt(d)
        Sx = Sx + np.outer(v[0, t], alpha)
        nx = nx + fk
        assert rel(o[0, t], Sx @ fq / (nx @ fq + 1e-6)) < 1e-12


def check_woodbury_rank_r(mod):
    for seed, d, r in ((7, 6, 4), (8, 5, 2)):
        q, k, v, u, A0, M0, S0, n0 = rand_case(seed, 3, 3, d, 2, r, spd_A0=True)
        _, A, _, _, tr = run(mod, q, k, v, u, A0, S0, n0, P=0, eps_n=0.0, tau=1e30,
                             trace=True, keep_A=True)
        for p in range(3):
            Ap = A0[p]
            for t in range(3):
                U = u[p, t].T                                   # d x r
                G = np.eye(r) + U.T @ Ap @ U
                Ap = Ap - Ap @ U @ np.linalg.solve(G, U.T @ Ap)
                assert rel(tr["A"][p, t], Ap) < 1e-12


def check_ldl_pivots(mod):
    """The sequential deltas are the pivots of G = I + U^T A_0 U (Cholesky: D_jj = R_jj^2)."""
    q, k, v, u, A0, M0, S0, n0 = rand_case(9, 2, 10, 6, 2, 2, spd_A0=True)
    _, _, _, _, tr = run(mod, q, k, v, u, A0, S0, n0, P=0, eps_n=0.0, tau=1e30, trace=True)
    for p in range(2):
        U = u[p].reshape(-1, 6).T                               # d x (T r), step-major columns
        G = np.eye(U.shape[1]) + U.T @ A0[p] @ U
        R = np.linalg.cholesky(G)
        assert rel(tr["delta"][p].reshape(-1), np.diag(R) ** 2) < 1e-10


def check_alpha_least_squares(mod):
    """alpha_t = M_t^{-1} s_t: the minimiser of 1/2 a^T M_t a - s_t^T a (v = 1, d_v = 1)."""
    d, T = 5, 20
    q, k, v, u, A0, M0, S0, n0 = rand_case(10, 1, T, d, 1, 1, spd_A0=True)
    v = np.ones_like(v)
    A, S, n = A0.copy(), S0.copy(), n0.copy()
    M = M0.copy()
    for t in range(T):
        S_prev = S.copy()
        _, A, S, n = run(mod, q[:, t:t + 1], k[:, t:t + 1], v[:, t:t + 1], u[:, t:t + 1], A, S, n,
                         P=0, eps_n=0.0, tau=1e30, t0=t)
        M = M + u[:, t, 0, :, None] * u[:, t, 0, None, :]
        s = phi_torch(k[0, t]) / math.sqrt(d)
        alpha = (S - S_prev)[0, 0]
        assert rel(alpha, np.linalg.solve(M[0], s)) < 1e-10


def check_invariants(mod):
    x = workloads.make_inputs(0, T=160)
    P, eps = 16, 1e-3
    o, A, S, n, tr = run(mod, x["q"], x["k"], x["v"], x["u"], x["A0"], x["S0"], x["n0"],
                         P=P, eps_n=eps, tau=1e30, trace=True, keep_A=True)
    At = tr["A"][0]
    assert np.max(np.abs(At - At.transpose(0, 2, 1))) < 1e-13
    assert tr["delta"].min() >= 1 - 1e-12
    for t in range(0, 160, 7):
        ev = np.linalg.eigvalsh(At[t])
        assert ev.min() > 0 and ev.max() <= 1 + ((t + 1) // P) * eps + 1e-12


def check_guard(mod):
    d = 3
    g = rng(11)
    u = unit_rows(g.normal(size=(1, 2, 1, d)))
    z3 = np.zeros((1, 2, d))
    # delta = 1 + u^T(-I)u = 0 -> guard replaces the update with A += 1e-6 I
    _, _, _, _, tr = run(mod, z3, z3, np.zeros((1, 2, 1)), u, -np.eye(d)[None], np.zeros((1, 1, d)),
                         np.zeros((1, d)), P=0, eps_n=0.0, tau=1e30, trace=True, keep_A=True)
    assert tr["guard"][0, 0, 0] and abs(tr["delta"][0, 0, 0]) < 1e-15
    assert np.max(np.abs(tr["A"][0, 0] - (-1 + 1e-6) * np.eye(d))) < 1e-18
    # delta = 1 - 2 = -1: |delta| is large, so the rank-1 update applies: A = -2I + 4 u u^T
    _, _, _, _, tr = run(mod, z3[:, :1], z3[:, :1], np.zeros((1, 1, 1)), u[:, :1], -2 * np.eye(d)[None],
                         np.zeros((1, 1, d)), np.zeros((1, d)), P=0, eps_n=0.0, tau=1e30,
                         trace=True, keep_A=True)
    assert not tr["guard"][0, 0, 0]
    uu = u[0, 0, 0]
    assert np.max(np.abs(tr["A"][0, 0] - (-2 * np.eye(d) + 4 * np.outer(uu, uu)))) < 1e-14


def check_renorm(mod):
    x = workloads.make_inputs(0, T=64)
    tau = 4.0        # many steps land with tau < ||S|| <= 1.5 tau
    A, S, n = x["A0"], x["S0"], x["n0"]
    fired = 0
    for t in range(64):
        sl = slice(t, t + 1)
        _, A, S, n, tr = run(mod, x["q"][:, sl], x["k"][:, sl], x["v"][:, sl], x["u"][:, sl], A, S, n,
                             P=64, eps_n=1e-6, tau=tau, t0=t, trace=True)
        nrm = np.linalg.norm(S[0])
        if tr["renorm"][0, 0]:
            fired += 1
            assert tr["snorm_pre"][0, 0] > tau and abs(nrm - tau) < 1e-12 * tau
        else:
            assert nrm <= tau and abs(nrm - tr["snorm_pre"][0, 0]) < 1e-14
    assert fired > 32
    # S from one 64-step call equals the step-by-step result
    _, A1, S1, n1 = run(mod, x["q"], x["k"], x["v"], x["u"], x["A0"], x["S0"], x["n0"],
                        P=64, eps_n=1e-6, tau=tau)
    assert rel(S1, S) < 1e-13


def check_split_calls(mod):
    q, k, v, u, A0, M0, S0, n0 = rand_case(12, 2, 20, 4, 3, 2)
    kw = dict(P=5, eps_n=1e-3, tau=2.0)
    o, A, S, n = run(mod, q, k, v, u, A0, S0, n0, **kw)
    o1, A1, S1, n1 = run(mod, q[:, :7], k[:, :7], v[:, :7], u[:, :7], A0, S0, n0, **kw)
    o2, A2, S2, n2 = run(mod, q[:, 7:], k[:, 7:], v[:, 7:], u[:, 7:], A1, S1, n1, t0=7, **kw)
    assert np.array_equal(np.concatenate([o1, o2], axis=1), o)
    assert np.array_equal(A2, A) and np.array_equal(S2, S) and np.array_equal(n2, n)


def check_readout_bruteforce(mod):
    """alpha_t from a Gauss-Jordan solve of M_t, S_t and n_t summed directly, d != d_v."""
    d, dv, T = 5, 3, 30
    q, k, v, u, A0, M0, S0, n0 = rand_case(13, 2, T, d, dv, 1, spd_A0=True)
    g = rng(14)
    S0 = g.normal(size=(2, dv, d)); n0 = g.random(size=(2, d))
    o, A, S, n = run(mod, q, k, v, u, A0, S0, n0, P=0, eps_n=0.0, tau=1e30)
    for p in range(2):
        M = M0[p].copy(); Sx = S0[p].copy(); nx = n0[p].copy()
        for t in range(T):
            M = M + np.outer(u[p, t, 0], u[p, t, 0])
            fk = phi_torch(k[p, t]); fq = phi_torch(q[p, t])
            Minv = gj_inv_np(M)
            alpha = Minv @ (fk / math.sqrt(d))
            Sx = Sx + np.outer(v[p, t], alpha)
            nx = nx + fk
            assert rel(o[p, t], Sx @ fq / (nx @ fq + 1e-6)) < 1e-10
        assert rel(S[p], Sx) < 1e-10 and rel(n[p], nx) < 1e-12 and rel(A[p], Minv) < 1e-10


def check_phi(mod):
    x = np.concatenate([np.linspace(-30, 30, 1201), [0.0, -0.0, 1e-300, -1e-300, 700.0, -745.0]])
    # 1 + ELU(x) = 1 + expm1(x) cancels for x << 0, so compare absolutely there
    # (one rounding of a number near 1), and check the x <= 0 branch is exp(x).
    got, want = mod.phi(x), phi_torch(x)
    assert np.max(np.abs(got - want) / np.maximum(np.abs(want), 1.0)) < 2.3e-16
    neg = x <= 0
    assert np.max(np.abs(got[neg] - np.exp(x[neg])) / np.exp(x[neg]).clip(1e-300)) < 1e-15
    assert mod.phi(np.array([0.0]))[0] == 1.0


# ---- the delta-rule variant (gist.science summary §2.3)

def check_delta_d1_overwrite(mod):
    """d = 1: k_hat = 1 and alpha_hat = 1 (A > 0), so S_t = v_t exactly; the readout
    is the additive path's ratio with that S."""
    g = rng(31)
    T, dv = 30, 3
    q = g.normal(size=(1, T, 1)); k = g.normal(size=(1, T, 1)); v = g.normal(size=(1, T, dv))
    u = 0.5 * np.where(g.random(size=(1, T, 1, 1)) < 0.5, -1.0, 1.0)
    S0 = g.normal(size=(1, dv, 1))
    o, A, S, n = run(mod, q, k, v, u, np.ones((1, 1, 1)), S0, np.zeros((1, 1)), P=0, eps_n=0.0,
                     tau=1e30, rule="delta")
    nx = 0.0
    for t in range(T):
        fk = phi_torch(k[0, t, 0]); fq = phi_torch(q[0, t, 0])
        nx = nx + fk
        assert rel(o[0, t], v[0, t] * fq / (nx * fq + 1e-6)) < 1e-12
    assert rel(S[0, :, 0], v[0, T - 1]) < 1e-14


def _delta_steps(mod, seed, d=6, dv=4, N=3, T=10):
    """Run the delta rule one step per call; yields (t, S_prev, S_next, A_next, k_hat, v_t)."""
    q, k, v, u, A0, M0, S0, n0 = rand_case(seed, N, T, d, dv, 1, spd_A0=True)
    S0 = rng(seed + 1).normal(size=(N, dv, d))
    A, S, n = A0, S0, n0
    for t in range(T):
        _, A1, S1, n1 = run(mod, q[:, t:t + 1], k[:, t:t + 1], v[:, t:t + 1], u[:, t:t + 1], A, S, n,
                            P=0, eps_n=0.0, tau=1e30, t0=t, rule="delta")
        fk = phi_torch(k[:, t])
        kh = fk / np.linalg.norm(fk, axis=1, keepdims=True)
        yield t, S, S1, A1, kh, v[:, t]
        A, S, n = A1, S1, n1


def check_delta_residual_contraction(mod):
    """The residual at the written key shrinks by exactly (1 - alpha_hat . k_hat):
    v - S_t k_hat = (1 - c)(v - S_{t-1} k_hat), c = (A_t k_hat / |A_t k_hat|) . k_hat."""
    for t, S0, S1, A1, kh, vt in _delta_steps(mod, 41):
        ak = np.einsum("pij,pj->pi", A1, kh)
        c = np.sum(ak * kh, axis=1) / np.linalg.norm(ak, axis=1)
        r0 = vt - np.einsum("pij,pj->pi", S0, kh)
        r1 = vt - np.einsum("pij,pj->pi", S1, kh)
        assert rel(r1, (1.0 - c)[:, None] * r0) < 1e-10


def check_delta_orthogonal_untouched(mod):
    """Directions orthogonal to alpha_hat = A_t k_hat / |A_t k_hat| keep their image:
    S_t w = S_{t-1} w for w . alpha_hat = 0."""
    g = rng(43)
    for t, S0, S1, A1, kh, vt in _delta_steps(mod, 42):
        ah = np.einsum("pij,pj->pi", A1, kh)
        ah = ah / np.linalg.norm(ah, axis=1, keepdims=True)
        w = g.normal(size=kh.shape)
        w = w - np.sum(w * ah, axis=1, keepdims=True) * ah
        assert rel(np.einsum("pij,pj->pi", S1, w), np.einsum("pij,pj->pi", S0, w)) < 1e-10


def check_delta_tracks_the_same_A(mod):
    """The variant changes the state write only: A, n and the guard are the additive path's."""
    q, k, v, u, A0, M0, S0, n0 = rand_case(44, 2, 25, 5, 3, 2, spd_A0=True)
    kw = dict(P=7, eps_n=1e-3, tau=3.0)
    _, Aa, _, na = run(mod, q, k, v, u, A0, S0, n0, **kw)
    _, Ad, _, nd = run(mod, q, k, v, u, A0, S0, n0, rule="delta", **kw)
    assert np.array_equal(Aa, Ad) and np.array_equal(na, nd)


# ---- the direction projection u = normalize(W_u k_raw) (README "VLA v3" item 2)

def check_project_u_closed_forms(mod):
    g = rng(51)
    d, N = 7, 9
    k = g.normal(size=(N, d))
    # identity: the keys' own directions
    u = mod.project_u(k, np.eye(d)[None])
    assert rel(u[:, 0], k / np.linalg.norm(k, axis=1, keepdims=True)) < 1e-15
    # a permutation permutes the unit vector; a positive scale changes nothing
    perm = g.permutation(d)
    Pm = np.eye(d)[perm]
    u2 = mod.project_u(k, np.stack([Pm, 3.5 * Pm]))
    want = (k / np.linalg.norm(k, axis=1, keepdims=True))[:, perm]
    assert rel(u2[:, 0], want) < 1e-15 and rel(u2[:, 1], want) < 1e-15
    # a zero key gives a zero direction (the 1e-12 floor), not NaN
    z = mod.project_u(np.zeros((1, d)), np.eye(d)[None])
    assert np.array_equal(z, np.zeros((1, 1, d)))
    # rank-one W: every output is +-w / |w| according to the sign of a.k
    a, w = g.normal(size=d), g.normal(size=d)
    u3 = mod.project_u(k, np.outer(w, a)[None])[:, 0]
    sgn = np.sign(k @ a)[:, None]
    assert rel(u3, sgn * w / np.linalg.norm(w)) < 1e-14


# ---- the parity metric (the reading adopted for the workloads' "max relative error")

def check_errors_metric(mod):
    """errors() on constructed discrepancies whose value is known exactly (dyadic numbers,
    so every expected value below is exact in float64).

    State X in {A, S, n}: per pair max|X - X_ref| / max|X_ref|, then the max over pairs.
    Outputs: per row ||o_t - o_ref_t||_inf / ||o_ref_t||_inf, then the max over (pair, t)."""
    d, dv, T = 3, 2, 3
    A_ref = np.zeros((2, d, d))
    A_ref[0] = [[2.0, -1.0, 0.0], [-1.0, 2.0, 0.5], [0.0, 0.5, 1.0]]   # max |.| = 2
    A_ref[1] = 64.0 * np.eye(d)                                         # max |.| = 64
    S_ref = np.zeros((2, dv, d))
    S_ref[0] = [[4.0, -2.0, 1.0], [0.5, 0.25, -4.0]]                    # max |.| = 4
    S_ref[1] = [[64.0, 8.0, -16.0], [2.0, 1.0, 0.5]]                    # max |.| = 64
    n_ref = np.array([[1.0, 2.0, 8.0], [0.5, 0.25, 0.125]])             # max 8 and 0.5
    o_ref = np.zeros((2, T, dv))
    o_ref[0] = [[1024.0, -512.0], [0.25, -0.125], [2.0, 1.0]]           # rows of very different scale
    o_ref[1] = [[1.0, 1.0], [-8.0, 4.0], [0.5, 0.5]]

    # identical inputs: every error is exactly zero
    e = mod.errors(o_ref, A_ref, S_ref, n_ref, o_ref, A_ref, S_ref, n_ref)
    assert e == dict(o=0.0, A=0.0, S=0.0, n=0.0), e

    A, S, n, o = A_ref.copy(), S_ref.copy(), n_ref.copy(), o_ref.copy()
    # A: a zero-crossing off-diagonal entry of the small pair moves by 2^-6 -> 2^-6 / 2 = 2^-7;
    # the large pair's diagonal moves by 2^-2 -> 2^-2 / 64 = 2^-8 (smaller: the max is pair 0's)
    A[0, 0, 2] = 2.0 ** -6
    A[1, 1, 1] += 0.25
    # S: the largest entry of pair 0 moves down by 1 -> 1/4 (normalising by the moved side would
    # give 1/4 too, so a second entry of pair 1 rises above its reference max: 72 vs 64 -> 8/64)
    S[0, 0, 0] = 3.0
    S[1, 0, 0] = 72.0
    # n: the largest entry of pair 1 moves by 2^-4 on a max of 0.5 -> 2^-3
    n[1, 0] += 2.0 ** -4
    # o: row 1 of pair 0 (scale 0.25) moves by 2^-5 -> 2^-3; row 0 (scale 1024) by 8 -> 2^-7
    o[0, 1, 1] -= 2.0 ** -5
    o[0, 0, 0] += 8.0
    e = mod.errors(o, A, S, n, o_ref, A_ref, S_ref, n_ref)
    assert e["A"] == 2.0 ** -7, e        # per-pair scale, max over pairs
    assert e["S"] == 0.25, e             # pair 0: 1/4; pair 1: 8/64 = 1/8
    assert e["n"] == 2.0 ** -3, e
    assert e["o"] == 2.0 ** -3, e        # per row: pair-wide scaling would give 2^-5 / 1024
    # the sides are not interchangeable: the reference side (the last four) sets the scale
    e2 = mod.errors(o_ref, A_ref, S_ref, n_ref, o, A, S, n)
    assert e2["n"] == 2.0 ** -4 / (0.5 + 2.0 ** -4), e2
    two = mod.errors(2 * o_ref, 2 * A_ref, 2 * S_ref, 2 * n_ref, o_ref, A_ref, S_ref, n_ref)
    half = mod.errors(o_ref, A_ref, S_ref, n_ref, 2 * o_ref, 2 * A_ref, 2 * S_ref, 2 * n_ref)
    assert two == dict(o=1.0, A=1.0, S=1.0, n=1.0), two
    assert half == dict(o=0.5, A=0.5, S=0.5, n=0.5), half
    # the sign of a discrepancy does not matter
    e3 = mod.errors(2 * o_ref - o, 2 * A_ref - A, 2 * S_ref - S, 2 * n_ref - n, o_ref, A_ref, S_ref, n_ref)
    assert e3 == e, (e3, e)
    # a single pair of several: the error of one bad pair is not averaged away
    N = 8
    big = np.broadcast_to(A_ref[1], (N, d, d)).copy()
    bad = big.copy()
    bad[5, 2, 0] = 16.0
    assert mod.errors(np.zeros((N, 0, dv)), bad, big[:, :dv], big[:, 0], np.zeros((N, 0, dv)), big,
                      big[:, :dv], big[:, 0])["A"] == 0.25


CHECKS = [check_golden_worked, check_exact_rational, check_gauss_jordan, check_d1_closed_form,
          check_basis_cycling, check_woodbury_rank_r, check_ldl_pivots, check_alpha_least_squares,
          check_invariants, check_guard, check_renorm, check_split_calls,
          check_readout_bruteforce, check_phi, check_delta_d1_overwrite, check_delta_residual_contraction,
          check_delta_orthogonal_untouched, check_delta_tracks_the_same_A, check_project_u_closed_forms,
          check_errors_metric]


@pytest.mark.parametrize("check", CHECKS, ids=lambda c: c.__name__)
def test_oracle_pin(check):
    check(vla_ref)


# ----------------------------------------------------------------------------
# checks of the fixtures and formulas themselves (no oracle involved)
# ----------------------------------------------------------------------------

def test_golden_fixture_is_the_exact_inverse():
    rows = load_golden()
    M = [[Fraction(1), Fraction(0)], [Fraction(0), Fraction(1)]]
    A = [[Fraction(1), Fraction(0)], [Fraction(0), Fraction(1)]]
    for r in rows:
        uu = [r[1], r[2]]
        M = [[M[i][j] + uu[i] * uu[j] for j in range(2)] for i in range(2)]
        z = [sum(A[i][j] * uu[j] for j in range(2)) for i in range(2)]
        delta = 1 + sum(uu[i] * z[i] for i in range(2))
        A = [[A[i][j] - z[i] * z[j] / delta for j in range(2)] for i in range(2)]
        assert delta == r[3]
        assert [A[0][0], A[0][1], A[1][0], A[1][1]] == list(r[4:8])
        assert gj_inverse(M) == A


def test_sherman_morrison_exact_in_rationals():
    """Exact arithmetic: the rank-1 recurrence equals the inverse of M_0 + sum u u^T."""
    g = rng(15)
    d, T = 4, 8
    M = [[Fraction(int(i == j) * 2) for j in range(d)] for i in range(d)]
    A = gj_inverse(M)
    for t in range(T):
        uu = [Fraction(int(x), int(y)) for x, y in zip(g.integers(-5, 6, size=d), g.integers(1, 7, size=d))]
        M = [[M[i][j] + uu[i] * uu[j] for j in range(d)] for i in range(d)]
        z = [sum(A[i][j] * uu[j] for j in range(d)) for i in range(d)]
        delta = 1 + sum(uu[i] * z[i] for i in range(d))
        A = [[A[i][j] - z[i] * z[j] / delta for j in range(d)] for i in range(d)]
        assert gj_inverse(M) == A


def test_chunked_form_matches_sequential():
    for seed, N, T, d, dv, r, P, tau, t0, C in ((16, 2, 50, 8, 5, 1, 7, 1e4, 3, 8),
                                                (17, 3, 64, 6, 6, 4, 16, 1e4, 0, 16),
                                                (18, 2, 40, 5, 4, 2, 0, 0.7, 0, 6)):
        q, k, v, u, A0, M0, S0, n0 = rand_case(seed, N, T, d, dv, r, spd_A0=True)
        kw = dict(P=P, eps_n=1e-3, tau=tau, t0=t0)
        ref = oracle.scan(q, k, v, u, A0, S0, n0, **kw)
        got = oracle.scan_chunked(q, k, v, u, A0, S0, n0, C=C, **kw)
        e = oracle.errors(*got, *ref)
        assert max(e.values()) < 1e-10, e


def test_ldl_unit_reconstructs():
    g = rng(19)
    B = g.normal(size=(3, 9, 9))
    G = np.eye(9) + B @ B.transpose(0, 2, 1)
    L, D = oracle.ldl_unit(G)
    assert np.allclose(np.triu(L, 1), 0) and np.allclose(np.diagonal(L, axis1=1, axis2=2), 1)
    assert rel(L @ (D[:, :, None] * L.transpose(0, 2, 1)), G) < 1e-13


def test_workload_generators_are_subset_stable():
    w = workloads.get(2).with_(T=2048)
    full = workloads.make_inputs(w, pairs=[0, 5, 9])
    sub = workloads.make_inputs(w, pairs=[5])
    for key in ("q", "k", "v", "u"):
        assert torch.equal(full[key][1], sub[key][0])
    # u rows are unit before rounding (bf16 rounding moves the norm by < 1%)
    nr = torch.linalg.vector_norm(full["u"].float(), dim=-1)
    assert float((nr - 1).abs().max()) < 1e-2


# ----------------------------------------------------------------------------
# planted mistakes
# ----------------------------------------------------------------------------

MUTATIONS = {
    "update_sign": ("A - z[:, :, None] * z[:, None, :] / dsafe", "A + z[:, :, None] * z[:, None, :] / dsafe"),
    "delta_drops_one": ("delta = 1.0 + np.sum(ui * z, axis=1)", "delta = np.sum(ui * z, axis=1)"),
    "nudge_sign": ("A = A + eps_n * eye", "A = A - eps_n * eye"),
    "nudge_phase": ("g = t0 + t + 1", "g = t0 + t"),
    "state_transposed": ("S = S + v[:, t, :, None] * alpha[:, None, :]",
                         "S = S + (alpha[:, :, None] * v[:, t, None, :]).reshape(S.shape)"),
    "phi_drops_one": ("x + 1.0, np.exp", "x, np.exp"),
    "renorm_threshold": ("fire = nrm > tau", "fire = nrm > 1.5 * tau"),
    "s_unscaled": ("s = phk * inv_sqrt_d", "s = phk"),
    "rank_index": ("ui = u[:, t, i, :]", "ui = u[:, t, 0, :]"),
    "guard_also_updates": ("A + GUARD_EPS * eye, updated", "updated + GUARD_EPS * eye, updated"),
    "guard_no_abs": ("guard = np.abs(delta) < GUARD_EPS", "guard = delta < GUARD_EPS"),
    "readout_no_eps": ("den = np.sum(n * phq, axis=1) + READOUT_EPS", "den = np.sum(n * phq, axis=1)"),
    "readout_uses_k": ("num = np.matmul(S, phq[:, :, None])", "num = np.matmul(S, phk[:, :, None])"),
    "normaliser_scaled": ("n = n + phk", "n = n + phk * inv_sqrt_d"),
    "renorm_to_one": ("tau / np.where(fire, nrm, 1.0)", "1.0 / np.where(fire, nrm, 1.0)"),
    "alpha_before_nudge": ("            if P > 0 and g % P == 0:\n                A = A + eps_n * eye\n",
                           ""),
    "readout_before_renorm": ("            S = S * scale[:, None, None]\n", ""),
    # delta-rule variant
    "delta_gate_unnormalised": ("gate = ak / np.maximum(np.linalg.norm(ak, axis=1, keepdims=True), NORM_EPS)",
                                "gate = ak"),
    "delta_key_unnormalised": ("kh = phk / np.maximum(np.linalg.norm(phk, axis=1, keepdims=True), NORM_EPS)",
                               "kh = phk"),
    "delta_residual_sign": ("resid = v[:, t, :] - np.matmul(S, kh[:, :, None])[:, :, 0]",
                            "resid = v[:, t, :] + np.matmul(S, kh[:, :, None])[:, :, 0]"),
    "delta_no_residual": ("resid = v[:, t, :] - np.matmul(S, kh[:, :, None])[:, :, 0]", "resid = v[:, t, :]"),
    "delta_gate_from_raw_key": ("ak = np.matmul(A, kh[:, :, None])[:, :, 0]",
                                "ak = np.matmul(A, k[:, t, :, None])[:, :, 0]"),
    "delta_outer_transposed": ("S = S + resid[:, :, None] * gate[:, None, :]",
                               "S = S + (gate[:, :, None] * resid[:, None, :]).reshape(S.shape)"),
    # direction projection
    "project_transposed_W": ('x = np.einsum("ijm,nm->nij", W_u, k_raw)', 'x = np.einsum("imj,nm->nij", W_u, k_raw)'),
    "project_no_normalise": ("return x / np.maximum(np.linalg.norm(x, axis=-1, keepdims=True), NORM_EPS)",
                             "return x"),
    # the parity metric
    "errors_scale_from_tested_side": ("den = np.abs(xr).reshape(xr.shape[0], -1).max(axis=1)",
                                      "den = np.abs(x).reshape(x.shape[0], -1).max(axis=1)"),
    "errors_mean_over_pairs": ("return float(np.max(num / np.maximum(den, 1e-300))) if x.size else 0.0",
                               "return float(np.mean(num / np.maximum(den, 1e-300))) if x.size else 0.0"),
    "errors_global_scale": ("den = np.abs(xr).reshape(xr.shape[0], -1).max(axis=1)",
                            "den = np.abs(xr).max()"),
    "errors_o_scaled_per_pair": ("den = np.abs(o_ref).max(axis=2)",
                                 "den = np.abs(o_ref).max(axis=(1, 2))[:, None]"),
    "errors_o_signed": ("num = np.abs(o - o_ref).max(axis=2)", "num = (o - o_ref).max(axis=2)"),
}


def _mutant(name):
    old, new = MUTATIONS[name]
    src = open(vla_ref.__file__).read()
    assert src.count(old) == 1, name
    mod = types.ModuleType("vla_ref_mutant_" + name)
    exec(compile(src.replace(old, new), mod.__name__, "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_mutants_are_caught(name):
    mod = _mutant(name)
    caught = []
    for check in CHECKS:
        try:
            with np.errstate(all="ignore"):
                check(mod)
        except Exception:  # noqa: BLE001  (assertion or shape error: the mistake is visible)
            caught.append(check.__name__)
    assert caught, f"mutant {name} passed every pin"
