"""GPU parity of the delta-rule variant (mode "delta") against the float64 oracle.

The variant (gist.science summary §2.3) keeps the exact tracking of A and writes
the state with a residual and unit vectors: alpha_hat = A k_hat / |A k_hat|,
k_hat = phi(k) / |phi(k)|, S += (v - S k_hat) alpha_hat^T.  The oracle's
``scan(..., rule="delta")`` is pinned by its own checks (tests/test_oracle_pins.py);
here the CUDA kernel (the blocked scan kernel's delta-rule variant: rounds of
several steps, the residuals solved within the round, renormalisation decided on
one reduction of Gram scalars) is compared with it element by element on seeded
inputs:
full-length workloads (all pairs of the f32 one, sampled pairs of the bf16 one)
and edge cases (ragged tiles, nudges with a t0 phase, renormalisation that
fires, the singularity guard, split calls, every built head width and rank).
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import workloads
from _util import ensure_built, errs, gpu_scan, oracle_scan

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-4, "bf16": 2e-2}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    ensure_built()
    import sherman_morrison_inverse_gb300 as vla
    vla.load_library()


def _check(e, tol, label):
    print(label, {k: f"{v:.2e}" for k, v in e.items()})
    assert max(e.values()) <= tol, (label, e)


CASES = [
    # (N, T, d, r, io, P, tau, t0)
    (3, 300, 16, 1, "f32", 64, 1e4, 0),
    (2, 211, 16, 4, "bf16", 50, 1e4, 5),
    (4, 517, 64, 1, "f32", 100, 1e4, 17),
    (3, 333, 64, 1, "bf16", 1024, 1e4, 0),
    (3, 129, 64, 4, "f32", 40, 1e4, 3),
    (2, 300, 64, 1, "f32", 64, 1.5, 0),        # renormalisation fires
    (3, 333, 64, 4, "bf16", 30, 2.0, 7),       # r = 4: renormalisation, nudges, ragged tail
    (2, 261, 64, 1, "bf16", 1024, 0.7, 0),     # renormalisation at nearly every step
    (2, 150, 128, 1, "f32", 64, 1e3, 0),
    (2, 77, 128, 4, "bf16", 16, 1e4, 1),
]


@pytest.mark.parametrize("N,T,d,r,io,P,tau,t0", CASES)
def test_delta_matches_oracle(N, T, d, r, io, P, tau, t0):
    x = workloads.gaussian_inputs(N, T, d, d, r, io, seed=1300 + d + r + T)
    x["S0"] = torch.from_numpy(np.random.default_rng([d, T]).normal(size=(N, d, d)) * 0.1).float()
    kw = dict(P=P, eps_n=1e-3, tau=tau, t0=t0)
    got = gpu_scan(x, 1, N, mode="delta", **kw)
    ref = oracle_scan(x, rule="delta", trace=True, **kw)
    _check(errs(got, ref), TOL[io], f"delta N{N} T{T} d{d} r{r} {io} tau{tau}")
    assert got[4]["renorm_count"] == int(ref[4]["renorm"].sum())
    assert got[4]["flags"] == 0


def test_delta_workload_f32_all_pairs():
    w = workloads.get(1)   # b4h8_t4096_d64_f32
    x = workloads.make_inputs(w)
    kw = dict(P=w.P, eps_n=w.eps_n, tau=w.tau)
    got = gpu_scan(x, w.B, w.H, mode="delta", **kw)
    _check(errs(got, oracle_scan(x, rule="delta", **kw)), TOL["f32"], f"delta {w.name}")


def test_delta_recall_workload_sampled():
    w = workloads.get(2)   # b8h16_t16384_d64_bf16_recall
    x = workloads.make_inputs(w)
    kw = dict(P=w.P, eps_n=w.eps_n, tau=w.tau)
    got = gpu_scan(x, w.B, w.H, mode="delta", **kw)
    sample = [5, 90]
    _check(errs(got, oracle_scan(x, idx=sample, rule="delta", **kw), idx=sample), TOL["bf16"],
           f"delta {w.name} pairs {sample}")


def test_delta_guard():
    d = 64
    x = workloads.gaussian_inputs(2, 40, d, d, 1, "f32", seed=66)
    x["A0"] = -torch.eye(d).expand(2, d, d).contiguous()
    x["u"][:, 0] = 0.0
    x["u"][:, 0, 0, 9] = 1.0
    x["u"][:, 1:] *= 0.5
    kw = dict(P=0, eps_n=0.0, tau=1e30)
    got = gpu_scan(x, 1, 2, mode="delta", **kw)
    ref = oracle_scan(x, rule="delta", trace=True, **kw)
    assert got[4]["guard_count"] == int(ref[4]["guard"].sum()) > 0
    _check(errs(got, ref), TOL["f32"], "delta guard")


@pytest.mark.parametrize("T1", [160, 150])
def test_delta_split_calls_continue_the_state(T1):
    """Two calls with t0 continue the state of one.  The blocked kernel takes rounds of up to
    4 steps inside tiles of 32 counted from each call's start, so a split at a tile boundary
    (160) gives the same rounds and the same bits; elsewhere (150) the rounds differ and the
    results agree to float32 rounding."""
    import sherman_morrison_inverse_gb300 as vla
    import oracle
    N, T2, d = 3, 247 - T1, 64
    x = workloads.gaussian_inputs(N, T1 + T2, d, d, 1, "f32", seed=88)
    kw = dict(P=50, eps_n=1e-3, tau=1e4)
    whole = gpu_scan(x, 1, N, mode="delta", **kw)
    dev = torch.device("cuda")
    A = x["A0"].reshape(1, N, d, d).to(dev).contiguous()
    S = x["S0"].reshape(1, N, d, d).to(dev).contiguous()
    n = x["n0"].reshape(1, N, d).to(dev).contiguous()
    outs = []
    for a, b in ((0, T1), (T1, T1 + T2)):
        g = [x[k][:, a:b].reshape(1, N, b - a, *x[k].shape[2:]).to(dev).contiguous() for k in ("q", "k", "v", "u")]
        outs.append(vla.scan_fwd(*g, A, S, n, t0=a, mode="delta", **kw))
    o = torch.cat(outs, dim=2).reshape(N, T1 + T2, d).double().cpu().numpy()
    got = (o, A.reshape(N, d, d).double().cpu().numpy(), S.reshape(N, d, d).double().cpu().numpy(),
           n.reshape(N, d).double().cpu().numpy())
    if T1 % 32 == 0:
        for x1, x2 in zip(got, whole[:4]):
            assert np.array_equal(x1, x2)
    else:
        e = oracle.errors(*got, *whole[:4])
        assert max(e.values()) <= 1e-5, e


def test_delta_rejects_a_chunk_size():
    import sherman_morrison_inverse_gb300 as vla
    x = workloads.gaussian_inputs(1, 8, 64, 64, 1, "f32", seed=3)
    with pytest.raises(vla.VlaError, match="UNSUPPORTED"):
        gpu_scan(x, 1, 1, mode="delta", chunk=4, P=0, eps_n=0.0, tau=1e4)
