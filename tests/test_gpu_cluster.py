"""GPU tests of the sequential scan on a two-CTA cluster per pair.

With `chunk` = 2 in sequential mode each (batch, head) pair runs on a cluster of
two CTAs: one tracks A, the other S, and alpha crosses between their shared
memories.  Where both variants take the same steps per reduction round (d <= 64,
and r = 4) it is the same arithmetic as the one-CTA kernel (`chunk` = 1), so every
output and state element must agree bit for bit.  At d = 128, r = 1 the cluster
takes 4-step rounds and the single CTA 2-step ones: the two then agree to the
float32 gate.  The cluster path is also checked against the float64 oracle on the
long-context d = 128 workload and on the edge cases (ragged tiles, nudges with a
t0 phase, renormalisation that fires, the singularity guard and its replay, split
calls).
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import workloads
from _util import ensure_built, errs, gpu_scan, oracle_scan

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    ensure_built()
    import sherman_morrison_inverse_gb300 as vla
    vla.load_library()


def _same(a, b, label):
    for name, x, y in zip(("o", "A", "S", "n"), a[:4], b[:4]):
        assert np.array_equal(x, y), (label, name, float(np.abs(x - y).max()))
    for key in ("flags", "guard_count", "renorm_count", "chunk_fallbacks"):
        assert a[4][key] == b[4][key], (label, key, a[4][key], b[4][key])


CASES = [
    # (N, T, d, r, io, P, tau, t0)
    (3, 300, 16, 1, "f32", 64, 1e4, 0),
    (2, 250, 16, 4, "bf16", 50, 2.0, 5),
    (5, 333, 64, 1, "f32", 100, 1e4, 17),
    (4, 517, 64, 1, "bf16", 1024, 8.0, 0),     # renormalisation fires
    (3, 129, 64, 4, "f32", 40, 1e4, 3),
    (2, 300, 128, 1, "f32", 64, 1e3, 0),
    (2, 301, 128, 1, "bf16", 60, 6.0, 9),      # 4-step rounds: ragged tail, nudges, renormalisation
    (2, 77, 128, 4, "bf16", 16, 3.0, 1),
]


def _same_rounds(d, r):
    """True where the cluster and the single CTA take the same steps per round."""
    return not (d == 128 and r == 1)


def _close(a, b, tol, label):
    import oracle
    e = oracle.errors(*a[:4], *b[:4])
    assert max(e.values()) <= tol, (label, e)
    assert a[4]["flags"] == b[4]["flags"] == 0, (label, a[4], b[4])


@pytest.mark.parametrize("N,T,d,r,io,P,tau,t0", CASES)
def test_cluster_matches_one_cta(N, T, d, r, io, P, tau, t0):
    x = workloads.gaussian_inputs(N, T, d, d, r, io, seed=900 + d + r + T)
    kw = dict(P=P, eps_n=1e-3, tau=tau, t0=t0)
    one = gpu_scan(x, 1, N, chunk=1, **kw)
    two = gpu_scan(x, 1, N, chunk=2, **kw)
    tol = 1e-4 if io == "f32" else 2e-2
    if _same_rounds(d, r):
        _same(one, two, f"N{N} T{T} d{d} r{r} {io}")
    else:
        _close(one, two, tol, f"N{N} T{T} d{d} r{r} {io}")
    ref = oracle_scan(x, **kw)
    e = errs(two, ref)
    assert max(e.values()) <= tol, e


def test_cluster_guard_and_replay():
    d = 64
    x = workloads.gaussian_inputs(2, 40, d, d, 1, "f32", seed=55)
    x["A0"] = -torch.eye(d).expand(2, d, d).contiguous()
    x["u"][:, 0] = 0.0
    x["u"][:, 0, 0, 3] = 1.0
    x["u"][:, 1:] *= 0.5
    kw = dict(P=0, eps_n=0.0, tau=1e30)
    one = gpu_scan(x, 1, 2, chunk=1, **kw)
    two = gpu_scan(x, 1, 2, chunk=2, **kw)
    _same(one, two, "guard")
    ref = oracle_scan(x, **kw, trace=True)
    assert two[4]["guard_count"] == int(ref[4]["guard"].sum()) > 0
    assert max(errs(two, ref).values()) <= 1e-4


def test_cluster_long_context_workload_sampled():
    """b2h8_t65536_d128_f32 (B H = 16 pairs) on clusters, two pairs against the oracle."""
    w = workloads.get(3)
    T = 8192
    x = workloads.make_inputs(w, T=T)
    kw = dict(P=w.P, eps_n=w.eps_n, tau=w.tau)
    got = gpu_scan(x, w.B, w.H, chunk=2, **kw)
    ref = oracle_scan(x, idx=[0, 11], **kw)
    e = errs(got, ref, idx=[0, 11])
    assert max(e.values()) <= 1e-3, e
    one = gpu_scan(x, w.B, w.H, chunk=1, **kw)
    _close(one, got, 1e-3, "workload 3 prefix")     # 2-step against 4-step rounds


def test_cluster_split_calls_continue_the_state():
    import sherman_morrison_inverse_gb300 as vla
    N, T1, T2, d = 3, 200, 131, 64
    x = workloads.gaussian_inputs(N, T1 + T2, d, d, 1, "f32", seed=77)
    kw = dict(P=64, eps_n=1e-3, tau=1e4)
    whole = gpu_scan(x, 1, N, chunk=2, **kw)
    dev = torch.device("cuda")
    A = x["A0"].reshape(1, N, d, d).to(dev).contiguous()
    S = x["S0"].reshape(1, N, d, d).to(dev).contiguous()
    n = x["n0"].reshape(1, N, d).to(dev).contiguous()
    outs = []
    for a, b in ((0, T1), (T1, T1 + T2)):
        g = [x[k][:, a:b].reshape(1, N, b - a, *x[k].shape[2:]).to(dev).contiguous() for k in ("q", "k", "v", "u")]
        outs.append(vla.scan_fwd(*g, A, S, n, t0=a, chunk=2, **kw))
    o = torch.cat(outs, dim=2).reshape(N, T1 + T2, d).double().cpu().numpy()
    assert np.array_equal(o, whole[0])
    assert np.array_equal(A.reshape(N, d, d).double().cpu().numpy(), whole[1])


def test_sequential_chunk_values_other_than_1_2_are_refused():
    import sherman_morrison_inverse_gb300 as vla
    x = workloads.gaussian_inputs(1, 8, 64, 64, 1, "f32", seed=3)
    with pytest.raises(vla.VlaError, match="UNSUPPORTED"):
        gpu_scan(x, 1, 1, chunk=3, P=0, eps_n=0.0, tau=1e4)
