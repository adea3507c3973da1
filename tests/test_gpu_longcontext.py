"""GPU checks of the long-context workload (b2h8_t65536_d128_f32) at its full length.

The workload asks for stability over T = 65536 steps at d = 128:

* the scan of all 16 pairs is compared with the float64 oracle on two pairs at the
  workload's gate (1e-3, relative to the largest entry of each final state and
  row-wise on the outputs);
* the tracked inverse is compared with the definition it tracks.  Without nudges
  A_t = M_t^{-1} exactly, with M_t = A_0^{-1} + sum_{t' <= t} u u^T ("Mathematical
  Primitives" §2, "Theoretical Derivation"); M is accumulated on the host in float64
  and max|A_t M_t - I| is read every 4096 steps through calls that carry t0.  With
  nudges on, A differs from M^{-1} by about eps_n ||M|| per nudge; that run is
  printed (a report, as the workload asks), not gated.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import workloads
from _util import ensure_built, errs, gpu_scan, oracle_scan

pytestmark = pytest.mark.gpu

SEG = 4096
# float32 drift of A M - I without nudges: measured 9.7e-4 after 65536 steps on this
# workload (the condition number of A reaches about 2000); the gate leaves a factor 5
DRIFT_GATE = 5e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    ensure_built()
    import sherman_morrison_inverse_gb300 as vla
    vla.load_library()


@pytest.fixture(scope="module")
def inputs():
    w = workloads.get(3)
    return w, workloads.make_inputs(w)


def test_long_context_full_length_against_the_oracle(inputs):
    w, x = inputs
    kw = dict(P=w.P, eps_n=w.eps_n, tau=w.tau)
    got = gpu_scan(x, w.B, w.H, **kw)
    sample = [0, 15]
    ref = oracle_scan(x, idx=sample, **kw)
    e = errs(got, ref, idx=sample)
    print("long context, pairs", sample, {k: f"{v:.2e}" for k, v in e.items()})
    assert max(e.values()) <= 1e-3, e
    assert got[4]["flags"] == 0


def _drift(w, x, P):
    import sherman_morrison_inverse_gb300 as vla
    dev = torch.device("cuda")
    B, H, T, d = w.B, w.H, w.T, w.d
    N = B * H
    g = {k: x[k].reshape(B, H, *x[k].shape[1:]).to(dev).contiguous() for k in ("q", "k", "v", "u")}
    A = x["A0"].reshape(B, H, d, d).to(dev).contiguous()
    S = x["S0"].reshape(B, H, d, d).to(dev).contiguous()
    n = x["n0"].reshape(B, H, d).to(dev).contiguous()
    M = np.linalg.inv(x["A0"].double().numpy())
    h = vla.default_handle()
    h.status()
    rows = []
    for a0 in range(0, T, SEG):
        sl = lambda t: t[:, :, a0:a0 + SEG].contiguous()
        vla.scan_fwd(sl(g["q"]), sl(g["k"]), sl(g["v"]), sl(g["u"]), A, S, n, t0=a0, P=P, eps_n=w.eps_n, tau=w.tau)
        Ud = x["u"][:, a0:a0 + SEG].double().numpy().reshape(N, -1, d)
        M += np.matmul(Ud.transpose(0, 2, 1), Ud)
        Ah = A.reshape(N, d, d).double().cpu().numpy()
        rows.append((a0 + SEG, float(np.abs(np.matmul(Ah, M) - np.eye(d)).max()),
                     float(torch.linalg.norm(S.reshape(N, -1).double(), dim=1).max())))
    return rows, h.status()


def test_long_context_inverse_tracks_M_inverse_without_nudges(inputs):
    w, x = inputs
    rows, st = _drift(w, x, P=0)
    for t, drift, sf in rows:
        print(f"P=0  t={t:6d}  max|A M - I| = {drift:.3e}  max ||S||_F = {sf:.1f}")
    assert st["flags"] == 0
    assert all(np.isfinite(sf) for _, _, sf in rows)
    assert max(dr for _, dr, _ in rows) <= DRIFT_GATE, rows


def test_long_context_drift_report_with_nudges(inputs):
    w, x = inputs
    rows, st = _drift(w, x, P=w.P)
    for t, drift, sf in rows:
        print(f"P={w.P}  t={t:6d}  max|A M - I| = {drift:.3e}  max ||S||_F = {sf:.1f}")
    assert st["flags"] == 0
    # eps_n = 1e-6 per nudge against ||M|| of a few hundred: the departure stays far below 1
    assert max(dr for _, dr, _ in rows) < 0.1


def test_long_context_with_renormalisation_firing_against_the_oracle(inputs):
    """The labelled companion run of the long-context workload with tau = 500, where
    dynamic renormalisation ("Mathematical Primitives" §5) fires from about t = 2000 on
    (at the workload's tau = 1e3 the norm of S stays below tau from a fresh state).

    All 16 pairs run at full length on the kernel the workload uses (the two-CTA cluster
    at d = 128); two pairs are compared with the oracle at the 1e-3 gate.  The number of
    renormalisations of those two pairs, counted by the kernel, equals the oracle's up to
    steps where ||S||_F lands within float32 rounding of tau (a decision that float32 and
    float64 may take differently); none is expected and few are allowed."""
    w, x = inputs
    kw = dict(P=w.P, eps_n=w.eps_n, tau=500.0)
    got = gpu_scan(x, w.B, w.H, **kw)
    assert got[4]["flags"] == 0 and got[4]["renorm_count"] > 0
    sample = [0, 15]
    ref = oracle_scan(x, idx=sample, trace=True, **kw)
    e = errs(got, ref, idx=sample)
    n_ref = int(ref[4]["renorm"].sum())
    sub = {k: v[sample] for k, v in x.items() if k in ("q", "k", "v", "u", "A0", "S0", "n0")}
    got2 = gpu_scan(sub, 1, len(sample), **kw)
    n_gpu = int(got2[4]["renorm_count"])
    print("long context, tau = 500, pairs", sample, {k: f"{v:.2e}" for k, v in e.items()},
          f"renormalisations: kernel {n_gpu}, oracle {n_ref} (all 16 pairs: {got[4]['renorm_count']})")
    assert n_ref > 1000, n_ref                       # it does fire, over most of the sequence
    assert max(e.values()) <= 1e-3, e
    assert abs(n_gpu - n_ref) <= max(2, n_ref // 1000), (n_gpu, n_ref)

