"""Chunked float64 form of the VLA scan: exact Woodbury / LDL^T over C steps.

TEST INFRASTRUCTURE ONLY (see the package docstring).

"Mathematical Primitives" §3 names the Woodbury identity as the closed form of
r sequential Sherman-Morrison updates; the gist.science summary (Technical
Summary §2.4) says the recurrence has a parallel (scan) formulation.  Neither page
writes the chunked algebra out, so this module states it and the tests check it
against the sequential oracle (``vla_ref.scan``) to 1e-10.

For a chunk of c steps with directions U = [u_1 .. u_m] (m = r c columns, ordered
step-major), starting inverse A_0:

    W = A_0 U,   G = I + U^T W = L D L^T      (L unit lower triangular)
    Z = W L^{-T}  gives the sequential z_j,   D_jj = delta_j
    A after column j  = A_0 - Z_{<=j} D_{<=j}^{-1} Z_{<=j}^T
    alpha_t = A_0 s_t - Z [ (D^{-1} Z^T s_t) masked to the columns of steps <= t ]
    S_t     = S_0 + sum_{j<=t} v_j alpha_j^T
    o_t     = (S_0 phi(q_t) + sum_{j<=t} (alpha_j . phi(q_t)) v_j)
              / (n_0 . phi(q_t) + sum_{j<=t} phi(k_j) . phi(q_t) + 1e-6)

Chunks end at nudge steps (the nudge A += eps_n I is not a rank-1 update).  A
chunk whose pivots hit the singularity guard, or in which the renormalisation of
S would fire, is taken step by step instead (that is what the chunked GPU kernel
does too).
"""
from __future__ import annotations

import numpy as np

from .vla_ref import GUARD_EPS, READOUT_EPS, phi, scan as _scan_seq


def ldl_unit(G):
    """LDL^T of a batch of symmetric matrices without pivoting.

    G [N, m, m] -> (L [N, m, m] unit lower triangular, D [N, m]).
    Column by column: D_j = G_jj - sum_{k<j} L_jk^2 D_k and, for i > j,
    L_ij = (G_ij - sum_{k<j} L_ik L_jk D_k) / D_j.
    """
    G = np.asarray(G, dtype=np.float64)
    N, m, _ = G.shape
    L = np.zeros_like(G)
    D = np.zeros((N, m))
    for j in range(m):
        L[:, j, j] = 1.0
        D[:, j] = G[:, j, j] - np.sum(L[:, j, :j] ** 2 * D[:, :j], axis=1)
        if j + 1 < m:
            rest = G[:, j + 1:, j] - np.einsum("nik,nk,nk->ni", L[:, j + 1:, :j], L[:, j, :j], D[:, :j])
            with np.errstate(divide="ignore", invalid="ignore"):
                L[:, j + 1:, j] = rest / D[:, j, None]
    return L, D


def _chunk_bounds(T: int, t0: int, P: int, C: int):
    """Split local steps [0, T) into chunks of at most C steps that end at nudges."""
    out = []
    a = 0
    while a < T:
        b = min(a + C, T)
        if P > 0:
            # first nudge step (global g = t0 + t + 1, g % P == 0) inside [a, b)
            g_a = t0 + a + 1
            first = g_a + ((-g_a) % P)      # smallest g >= g_a with g % P == 0
            t_n = first - t0 - 1
            if t_n < b:
                b = t_n + 1
        out.append((a, b))
        a = b
    return out


def scan_chunked(q, k, v, u, A0, S0, n0, *, P: int, eps_n: float, tau: float, t0: int = 0,
                 C: int = 64, stats: dict | None = None):
    """Same contract as ``vla_ref.scan`` (without traces), chunk by chunk."""
    f = lambda x: np.array(x.detach().double().numpy() if hasattr(x, "detach") else x,
                           dtype=np.float64, copy=True)
    q, k, v, u, A, S, n = map(f, (q, k, v, u, A0, S0, n0))
    N, T, d = q.shape
    dv = v.shape[2]
    r = u.shape[2]
    eye = np.eye(d)
    o = np.zeros((N, T, dv))
    if stats is not None:
        stats.setdefault("chunks", 0)
        stats.setdefault("seq_fallback", 0)
    for a, b in _chunk_bounds(T, t0, P, C):
        c = b - a
        m = c * r
        nudge = P > 0 and (t0 + b) % P == 0
        U = u[:, a:b].reshape(N, m, d)                         # rows = directions
        W = np.matmul(A, U.transpose(0, 2, 1))                  # [N, d, m]
        G = np.eye(m) + np.matmul(U, W)                         # [N, m, m]
        L, D = ldl_unit(G)
        phk = phi(k[:, a:b])                                    # [N, c, d]
        Sig = phk / np.sqrt(d)
        phq = phi(q[:, a:b])
        V = v[:, a:b]                                           # [N, c, dv]
        if np.any(np.abs(D) < GUARD_EPS) or not np.all(np.isfinite(D)):
            o[:, a:b], A, S, n = _scan_seq(q[:, a:b], k[:, a:b], v[:, a:b], u[:, a:b], A, S, n,
                                           P=P, eps_n=eps_n, tau=tau, t0=t0 + a)
            if stats is not None:
                stats["seq_fallback"] += 1
            continue
        # Z^T = L^{-1} W^T (forward substitution with a unit lower triangle)
        Zt = np.zeros((N, m, d))
        Wt = W.transpose(0, 2, 1)
        for j in range(m):
            Zt[:, j] = Wt[:, j] - np.einsum("nl,nld->nd", L[:, j, :j], Zt[:, :j])
        Z = Zt.transpose(0, 2, 1)                               # [N, d, m]
        coef = np.matmul(Zt, Sig.transpose(0, 2, 1)) / D[:, :, None]   # [N, m, c]
        col_step = np.arange(m) // r
        mask = (col_step[:, None] <= np.arange(c)[None, :]).astype(np.float64)
        alpha = (np.matmul(A, Sig.transpose(0, 2, 1)) - np.matmul(Z, coef * mask)).transpose(0, 2, 1)
        A = A - np.matmul(Z / D[:, None, :], Zt)
        if nudge:
            A = A + eps_n * eye
            alpha[:, -1] += eps_n * Sig[:, -1]
        # --- state side: norms of S_t for every t of the chunk (Gram form)
        S0v = np.einsum("nad,ntd->nta", S, alpha)              # S_0 alpha_t   [N, c, dv]
        cross = np.einsum("nta,nta->nt", V, S0v)                # v_t . S_0 alpha_t
        VV = np.matmul(V, V.transpose(0, 2, 1))                 # [N, c, c]
        AA = np.matmul(alpha, alpha.transpose(0, 2, 1))
        tri = np.tril(np.ones((c, c)))
        gram = VV * AA
        pref = np.einsum("ntj,njl,ntl->nt", tri[None].repeat(N, 0), gram, tri[None].repeat(N, 0))
        nrm2 = np.sum(S * S, axis=(1, 2))[:, None] + 2.0 * np.cumsum(cross, axis=1) + pref
        if np.any(np.sqrt(np.maximum(nrm2, 0.0)) > tau * (1 - 1e-9)):
            # renormalisation may fire: take the state side step by step
            for t in range(c):
                S = S + V[:, t, :, None] * alpha[:, t, None, :]
                n = n + phk[:, t]
                nrm = np.sqrt(np.sum(S * S, axis=(1, 2)))
                fire = nrm > tau
                S = S * np.where(fire, tau / np.where(fire, nrm, 1.0), 1.0)[:, None, None]
                num = np.matmul(S, phq[:, t, :, None])[:, :, 0]
                o[:, a + t] = num / (np.sum(n * phq[:, t], axis=1) + READOUT_EPS)[:, None]
            if stats is not None:
                stats["seq_fallback"] += 1
            continue
        qa = np.matmul(phq, alpha.transpose(0, 2, 1)) * tri      # [N, c(t), c(j)]  (alpha_j . phq_t), j <= t
        num = np.matmul(phq, S.transpose(0, 2, 1)) + np.matmul(qa, V)
        qk = np.matmul(phq, phk.transpose(0, 2, 1)) * tri
        den = np.matmul(phq, n[:, :, None])[:, :, 0] + qk.sum(axis=2) + READOUT_EPS
        o[:, a:b] = num / den[:, :, None]
        S = S + np.matmul(V.transpose(0, 2, 1), alpha)
        n = n + phk.sum(axis=1)
        if stats is not None:
            stats["chunks"] += 1
    return o, A, S, n
