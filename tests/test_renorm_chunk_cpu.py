"""The chunked kernel's exact renormalisation path, restated on the host in float64.

"Mathematical Primitives" §5 (dynamic renormalisation) rescales S to tau whenever its
Frobenius norm passes tau after a step.  The chunked kernel takes a chunk's steps without
forming S step by step: it keeps S_t = sigma_t S_reg,t with
S_reg,t = S_0 + sum_{t'<=t} v_t' alpha_t'^T / sigma_{t'-1}, and decides from

    ||S_t||^2 (before the rescale) = ||S_{t-1}||^2 + 2 sigma_{t-1} (XS_t + R_t) + PP[t][t],
    XS_t = v_t^T S_0 alpha_t,  PP[t][t'] = (v_t . v_t') (alpha_t . alpha_t'),
    R_t = sum_{t'<t} PP[t][t'] / sigma_{t'-1}.

One warp takes the decisions in order.  It keeps R_t for the steps not yet decided as if no
further step renormalised (R_t = Q[t][t], Q the exclusive row prefix sums of PP) and, when
step u renormalises, adds d (Q[t][t] - Q[t][u + 1]) to every later R_t (d: the change of
1 / sigma).  These tests check both forms against the recurrence as the pages define it, S
formed step by step, on random chunks where renormalisation fires at many steps, at none,
and at every one.
"""
from __future__ import annotations

import numpy as np
import pytest


def explicit(S0, V, AL, tau):
    """S += v_t alpha_t^T, then S *= tau / ||S||_F when ||S||_F > tau, step by step."""
    S = S0.copy()
    fired = []
    for t in range(V.shape[0]):
        S = S + np.outer(V[t], AL[t])
        n = np.linalg.norm(S)
        fired.append(n > tau)
        if n > tau:
            S *= tau / n
    return S, np.array(fired)


def chunk_terms(S0, V, AL):
    XS = np.einsum("ti,ij,tj->t", V, S0, AL)
    PP = (V @ V.T) * (AL @ AL.T)
    return XS, PP


def direct(S0, V, AL, tau):
    """The decisions from the norm recurrence, each R_t summed in full."""
    XS, PP = chunk_terms(S0, V, AL)
    c = V.shape[0]
    n2, sg = float(np.sum(S0 * S0)), 1.0
    IS = np.zeros(c)
    fired, SG = [], []
    for t in range(c):
        IS[t] = 1.0 / sg
        R = sum(PP[t, tp] * IS[tp] for tp in range(t))
        npre2 = n2 + 2.0 * sg * (XS[t] + R) + PP[t, t]
        fired.append(npre2 > tau * tau)
        if npre2 > tau * tau:
            sg *= tau / np.sqrt(npre2)
            n2 = tau * tau
        else:
            n2 = npre2
        SG.append(sg)
    return np.array(fired), np.array(SG), IS


def warp_scheme(S0, V, AL, tau):
    """The kernel's form: R_t from row prefix sums, corrected at each renormalisation."""
    XS, PP = chunk_terms(S0, V, AL)
    c = V.shape[0]
    Q = np.zeros((c, c + 1))   # Q[t][m] = sum_{t'<m} PP[t][t'], t' < t only
    for t in range(c):
        q = 0.0
        for m in range(c + 1):
            Q[t, m] = q
            if m < t:
                q += PP[t, m]
    x = np.array([XS[t] + Q[t, t] for t in range(c)])
    n2, sg, isg = float(np.sum(S0 * S0)), 1.0, 1.0
    fired, SG = [], []
    for t in range(c):
        npre2 = n2 + 2.0 * sg * x[t] + PP[t, t]
        fired.append(npre2 > tau * tau)
        if npre2 > tau * tau:
            sgn = sg * (tau / np.sqrt(npre2))
            isn = 1.0 / sgn
            for tq in range(t + 2, c):
                x[tq] += (isn - isg) * (Q[tq, tq] - Q[tq, t + 1])
            sg, isg, n2 = sgn, isn, tau * tau
        else:
            n2 = npre2
        SG.append(sg)
    return np.array(fired), np.array(SG)


def s_from_scales(S0, V, AL, SG):
    """S_c = sigma_c (S_0 + sum_t v_t alpha_t^T / sigma_{t-1}), the kernel's fold of the scales."""
    prev = np.concatenate([[1.0], SG[:-1]])
    Sreg = S0 + sum(np.outer(V[t], AL[t]) / prev[t] for t in range(V.shape[0]))
    return SG[-1] * Sreg


def _chunk(seed, c, d, s0_scale, a_scale):
    rng = np.random.default_rng(seed)
    S0 = rng.normal(size=(d, d)) * s0_scale
    V = rng.normal(size=(c, d))
    AL = rng.normal(size=(c, d)) * a_scale
    return S0, V, AL


@pytest.mark.parametrize("seed", range(12))
@pytest.mark.parametrize("c", [1, 16, 37, 64])
def test_decisions_match_the_step_by_step_recurrence(seed, c):
    d = 16
    S0, V, AL = _chunk(seed, c, d, 0.3, 0.2)
    tau = float(np.linalg.norm(S0)) * (0.8 + 0.1 * (seed % 5))   # some chunks fire often, some rarely
    S_ref, fired_ref = explicit(S0, V, AL, tau)
    fired_d, SG_d, _ = direct(S0, V, AL, tau)
    fired_w, SG_w = warp_scheme(S0, V, AL, tau)
    assert np.array_equal(fired_d, fired_ref)
    assert np.array_equal(fired_w, fired_ref)
    np.testing.assert_allclose(SG_w, SG_d, rtol=1e-12)
    np.testing.assert_allclose(s_from_scales(S0, V, AL, SG_w), S_ref, rtol=1e-10, atol=1e-12)


def test_every_step_renormalises():
    S0, V, AL = _chunk(99, 64, 16, 1.0, 1.0)
    tau = 0.5 * float(np.linalg.norm(S0))
    S_ref, fired_ref = explicit(S0, V, AL, tau)
    assert fired_ref.all()
    fired_w, SG_w = warp_scheme(S0, V, AL, tau)
    assert fired_w.all()
    np.testing.assert_allclose(s_from_scales(S0, V, AL, SG_w), S_ref, rtol=1e-10, atol=1e-12)


def test_no_step_renormalises():
    S0, V, AL = _chunk(7, 64, 16, 0.1, 0.05)
    tau = 1e6
    S_ref, fired_ref = explicit(S0, V, AL, tau)
    assert not fired_ref.any()
    fired_w, SG_w = warp_scheme(S0, V, AL, tau)
    assert not fired_w.any() and np.all(SG_w == 1.0)
    np.testing.assert_allclose(s_from_scales(S0, V, AL, SG_w), S_ref, rtol=1e-12, atol=1e-12)


def test_a_wrong_correction_is_caught():
    """The correction runs over t'' in (u, t) only: applying it from t'' = u (one step early)
    changes the decisions on a chunk that renormalises often."""
    S0, V, AL = _chunk(3, 64, 16, 0.3, 0.3)
    tau = 0.9 * float(np.linalg.norm(S0))
    _, fired_ref = explicit(S0, V, AL, tau)
    XS, PP = chunk_terms(S0, V, AL)
    c = 64
    Q = np.zeros((c, c + 1))
    for t in range(c):
        q = 0.0
        for m in range(c + 1):
            Q[t, m] = q
            if m < t:
                q += PP[t, m]
    x = np.array([XS[t] + Q[t, t] for t in range(c)])
    n2, sg, isg = float(np.sum(S0 * S0)), 1.0, 1.0
    fired, SG = [], []
    for t in range(c):
        npre2 = n2 + 2.0 * sg * x[t] + PP[t, t]
        fired.append(npre2 > tau * tau)
        if npre2 > tau * tau:
            sgn = sg * (tau / np.sqrt(npre2))
            isn = 1.0 / sgn
            for tq in range(t + 1, c):
                x[tq] += (isn - isg) * (Q[tq, tq] - Q[tq, t])   # wrong: from t'' = t
            sg, isg, n2 = sgn, isn, tau * tau
        else:
            n2 = npre2
        SG.append(sg)
    S_ref, _ = explicit(S0, V, AL, tau)
    assert not np.allclose(s_from_scales(S0, V, AL, np.array(SG)), S_ref, rtol=1e-6)
