"""Sequential float64 oracle of the VLA forward scan (test infrastructure only).

Sources (three web pages on Variational Linear Attention):

* "Mathematical Primitives" (variational-linear-attention.vercel.app/maths.html):
  §1 scaled inner-product scoring and finite-state enforcement, §2 Sherman-Morrison
  rank-1 inverse tracking with its execution pipeline (z = A u, delta = 1 + u.z,
  singularity guard, A -= z z^T / delta, periodic diagonal nudging), §3 Woodbury
  generalisation as r sequential rank-1 updates, §4 alpha_t = A_t s_t, §5 state
  update and dynamic renormalisation of S.
* "Variational Linear Attention (VLA)" project README, section "VLA v3 (Research
  Implementation Notes)": phi = ELU + 1 on q and k (item 1), u_t = normalize(W_u
  k_raw) (item 2), periodic diagonal nudging (item 3), calibrated readout with a
  normaliser dot product (item 5).
* "Variational Linear Attention: Stable Associative Memory for Long-Context
  Transformers" (gist.science summary), Technical Summary §2.2-2.3 (A_t = M_t^{-1}
  maintained by Sherman-Morrison; output as a ratio of recurrences with ELU+1).

Reading adopted where the pages are loose (each is listed in the design notes):

* s_t is the vector phi(k_t)/sqrt(d) (the first page writes a scalar k.q/sqrt(d)
  but then uses s_t as a vector in alpha_t = A_t s_t).
* The state update is S_t = S_{t-1} + v_t alpha_t^T (the first page's
  "alpha (x) (v k^T)" is not well-typed); S is d_v x d and alpha is not
  normalised.
* Guard: if |delta| < 1e-6 the rank-1 update of that direction is REPLACED by
  A += 1e-6 I (strict '<').
* Rank r: the r directions of a step are applied one after another (§3).
* Nudge: at global 1-indexed steps g = t0 + t with g % P == 0 (P > 0), after the
  step's r updates and before alpha; A += eps_n I.  P = 0 disables it.
* Renormalisation: after the state update, if ||S||_F > tau (strict) then
  S <- S * tau / ||S||_F; the readout uses the renormalised S.
* Readout: o_t = S_t phi(q_t) / (n_t . phi(q_t) + 1e-6) with n_t = n_{t-1} + phi(k_t).
* phi(x) = x + 1 for x > 0, exp(x) otherwise (ELU with alpha = 1, plus one).

The delta-rule variant (``rule="delta"``) follows the gist.science summary
§2.3 ("Recursive Update Rule"): the same tracking of A, then
alpha_hat_t = A_t k_hat_t / |A_t k_hat_t| and S_t = S_{t-1} + (v_t - S_{t-1} k_hat_t)
alpha_hat_t^T, with both vectors of unit length.  Readings: k_hat_t is the
feature-mapped key phi(k_t) normalised (the summary calls it "the normalized
key" and uses the ELU+1 features for the output); unit length is x / max(|x|,
1e-12), the convention of u's normalisation; the normaliser n, the
renormalisation and the readout are the additive path's.

The loop runs over t; independent (batch, head) pairs are stacked on a leading
axis and advanced together with numpy (no reordering of any step).
"""
from __future__ import annotations

import numpy as np

GUARD_EPS = 1e-6     # singularity threshold and injected diagonal (Mathematical Primitives §2)
NORM_EPS = 1e-12     # floor of the norms in unit-length vectors (delta-rule variant)
READOUT_EPS = 1e-6   # readout denominator offset (the reading adopted for the README's calibrated readout)


def phi(x):
    """ELU(x) + 1 with ELU's alpha = 1 (README "VLA v3" item 1)."""
    x = np.asarray(x, dtype=np.float64)
    return np.where(x > 0, x + 1.0, np.exp(np.minimum(x, 0.0)))


def _f64(x):
    if hasattr(x, "detach"):  # torch tensor (CPU)
        x = x.detach().to("cpu").double().numpy()
    return np.array(x, dtype=np.float64, copy=True)


def scan(q, k, v, u, A0, S0, n0, *, P: int, eps_n: float, tau: float, t0: int = 0,
         trace: bool = False, keep_A: bool = False, rule: str = "additive"):
    """Run the recurrence over T steps for N independent (batch, head) pairs.

    Shapes: q, k [N, T, d]; v [N, T, dv]; u [N, T, r, d]; A0 [N, d, d];
    S0 [N, dv, d]; n0 [N, d].  Any leading dims before N are not supported:
    flatten (batch, head) first.  Inputs are upcast to float64 exactly.

    Returns ``(o, A, S, n)`` with o [N, T, dv] and the final state, plus a trace
    dict when ``trace``: delta [N, T, r], guard [N, T, r] (bool), renorm [N, T]
    (bool), snorm_pre [N, T] (||S_t||_F before renormalisation), and A_t [N, T, d, d]
    when ``keep_A``.  ``rule`` = "additive" (S += v alpha^T) or "delta" (the
    delta-rule variant in the module docstring).
    """
    assert rule in ("additive", "delta")
    q, k, v, u = _f64(q), _f64(k), _f64(v), _f64(u)
    A, S, n = _f64(A0), _f64(S0), _f64(n0)
    N, T, d = q.shape
    dv = v.shape[2]
    r = u.shape[2]
    assert k.shape == (N, T, d) and v.shape == (N, T, dv) and u.shape == (N, T, r, d)
    assert A.shape == (N, d, d) and S.shape == (N, dv, d) and n.shape == (N, d)
    eye = np.eye(d)
    o = np.zeros((N, T, dv))
    tr = None
    if trace:
        tr = dict(delta=np.zeros((N, T, r)), guard=np.zeros((N, T, r), bool),
                  renorm=np.zeros((N, T), bool), snorm_pre=np.zeros((N, T)))
        if keep_A:
            tr["A"] = np.zeros((N, T, d, d))
    inv_sqrt_d = 1.0 / np.sqrt(d)
    with np.errstate(divide="ignore", invalid="ignore"):
        for t in range(T):
            g = t0 + t + 1                                # global 1-indexed step
            # --- Sherman-Morrison, r directions in sequence (Primitives §2, §3)
            for i in range(r):
                ui = u[:, t, i, :]
                z = np.matmul(A, ui[:, :, None])[:, :, 0]           # z = A u
                delta = 1.0 + np.sum(ui * z, axis=1)                # delta = 1 + u.z
                guard = np.abs(delta) < GUARD_EPS
                dsafe = np.where(guard, 1.0, delta)
                updated = A - z[:, :, None] * z[:, None, :] / dsafe[:, None, None]
                A = np.where(guard[:, None, None], A + GUARD_EPS * eye, updated)
                if trace:
                    tr["delta"][:, t, i] = delta
                    tr["guard"][:, t, i] = guard
            # --- periodic spectrum stabilisation (Primitives §2, last item)
            if P > 0 and g % P == 0:
                A = A + eps_n * eye
            phk = phi(k[:, t, :])
            if rule == "delta":
                # --- unit key, unit gate alpha_hat = A k_hat / |A k_hat|, residual write
                #     (gist.science summary §2.3)
                kh = phk / np.maximum(np.linalg.norm(phk, axis=1, keepdims=True), NORM_EPS)
                ak = np.matmul(A, kh[:, :, None])[:, :, 0]
                gate = ak / np.maximum(np.linalg.norm(ak, axis=1, keepdims=True), NORM_EPS)
                resid = v[:, t, :] - np.matmul(S, kh[:, :, None])[:, :, 0]
                S = S + resid[:, :, None] * gate[:, None, :]
            else:
                # --- coefficient alpha_t = A_t s_t (Primitives §4)
                s = phk * inv_sqrt_d
                alpha = np.matmul(A, s[:, :, None])[:, :, 0]
                # --- state update (Primitives §5)
                S = S + v[:, t, :, None] * alpha[:, None, :]
            # --- normaliser (README v3 item 5)
            n = n + phk
            # --- dynamic renormalisation (Primitives §5)
            nrm = np.sqrt(np.sum(S * S, axis=(1, 2)))
            fire = nrm > tau
            scale = np.where(fire, tau / np.where(fire, nrm, 1.0), 1.0)
            S = S * scale[:, None, None]
            # --- readout (README v3 item 5)
            phq = phi(q[:, t, :])
            num = np.matmul(S, phq[:, :, None])[:, :, 0]
            den = np.sum(n * phq, axis=1) + READOUT_EPS
            o[:, t, :] = num / den[:, None]
            if trace:
                tr["renorm"][:, t] = fire
                tr["snorm_pre"][:, t] = nrm
                if keep_A:
                    tr["A"][:, t] = A
    if trace:
        return o, A, S, n, tr
    return o, A, S, n


def project_u(k_raw, W_u):
    """u_{t,i} = W_u[i] k_t / max(|W_u[i] k_t|_2, 1e-12): the learned penalty directions
    "u_t = normalize(W_u k_t^raw)" (README "VLA v3" item 2).

    k_raw [N, d] (any leading dims flattened by the caller), W_u [r, d, d] with
    W_u[i][j][m] the weight of input m in output j; returns u [N, r, d] in float64.
    """
    k_raw, W_u = _f64(k_raw), _f64(W_u)
    x = np.einsum("ijm,nm->nij", W_u, k_raw)
    return x / np.maximum(np.linalg.norm(x, axis=-1, keepdims=True), NORM_EPS)


def errors(o, A, S, n, o_ref, A_ref, S_ref, n_ref):
    """Scale-aware errors used by the parity gates.

    For the final state X in {A, S, n}: max over pairs of max|X - X_ref| / max|X_ref|.
    For the outputs: max over (pair, t) of ||o_t - o_ref_t||_inf / ||o_ref_t||_inf
    (rows are compared separately because o_t shrinks like 1/t).  Elementwise
    relative error is not used: off-diagonal entries of A cross zero.
    """
    def _state(x, xr):
        x, xr = _f64(x), _f64(xr)
        num = np.abs(x - xr).reshape(x.shape[0], -1).max(axis=1)
        den = np.abs(xr).reshape(xr.shape[0], -1).max(axis=1)
        return float(np.max(num / np.maximum(den, 1e-300))) if x.size else 0.0

    o, o_ref = _f64(o), _f64(o_ref)
    if o.size:
        num = np.abs(o - o_ref).max(axis=2)
        den = np.abs(o_ref).max(axis=2)
        eo = float(np.max(num / np.maximum(den, 1e-300)))
    else:
        eo = 0.0
    return dict(o=eo, A=_state(A, A_ref), S=_state(S, S_ref), n=_state(n, n_ref))
