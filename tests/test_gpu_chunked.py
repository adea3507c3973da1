"""GPU parity of the chunked (exact Woodbury / LDL^T, tcgen05) scan.

The chunked mode takes 64 directions per chunk (64 steps at r = 1, 16 at r = 4)
with the dense contractions on tensor cores in tf32, for d = d_v = 64, bfloat16
and float32 I/O (float32: 3xTF32 on every product).  It is checked against the
float64 oracle and against the sequential kernel at the gate of its I/O type
(bfloat16 2e-2, float32 1e-4 at T <= 4096), on full-length workloads and on edge
cases: ragged lengths, nudges that split chunks (t0 phase), renormalisation
firing (the exact per-step path) and the singularity guard (the step-by-step
fallback).

While two CTAs per pair fit on the SMs, each pair runs on a cluster of two (the A
side and the S side of every chunk on two SMs, alpha handed over through
distributed shared memory); with more pairs, on one CTA.  Both forms compute the
same values in the same order, so they must agree bit for bit wherever the guard
does not fire; the edge cases (few pairs) run the cluster form, the full
workloads of 128 and 256 pairs the one-CTA form.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import workloads
from _util import ensure_built, errs, gpu_scan, oracle_scan

pytestmark = pytest.mark.gpu

TOL = 2e-2
TOL_F32 = 1e-4


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    ensure_built()
    import sherman_morrison_inverse_gb300 as vla
    vla.load_library()


def _check(e, tol, label):
    print(label, {k: f"{v:.2e}" for k, v in e.items()})
    assert max(e.values()) <= tol, (label, e)


@pytest.mark.parametrize("idx,T,sample", [(2, 16384, [0, 77]), (4, 8192, [3, 200])])
def test_chunked_workload_parity(idx, T, sample):
    w = workloads.get(idx)
    x = workloads.make_inputs(w, T=T)
    kw = dict(P=w.P, eps_n=w.eps_n, tau=w.tau)
    got = gpu_scan(x, w.B, w.H, mode="chunked", chunk=0, **kw)
    ref = oracle_scan(x, idx=sample, **kw)
    _check(errs(got, ref, idx=sample), TOL, f"chunked {w.name} vs oracle")
    seq = gpu_scan(x, w.B, w.H, **kw)
    import oracle
    _check(oracle.errors(*got[:4], *seq[:4]), TOL, f"chunked vs sequential {w.name}")
    assert got[4]["flags"] == 0 and got[4]["chunk_fallbacks"] == 0


EDGE = [
    # (N, T, r, P, tau, t0)
    (2, 1, 1, 64, 1e4, 0),
    (3, 100, 1, 1024, 1e4, 0),        # ragged: one full chunk and a partial one
    (2, 300, 1, 50, 1e4, 7),          # nudges split chunks, t0 phase
    (2, 130, 4, 20, 1e4, 3),
    (1, 200, 1, 1024, 5.0, 0),        # renormalisation fires: exact per-step path
    (2, 90, 4, 1024, 3.0, 0),
    (1, 200, 1, 1024, 0.05, 0),       # scales of a chunk fall below 2^-64: S step by step
]


@pytest.mark.parametrize("io", ["bf16", "f32"])
@pytest.mark.parametrize("N,T,r,P,tau,t0", EDGE)
def test_chunked_edges(N, T, r, P, tau, t0, io):
    x = workloads.gaussian_inputs(N, T, 64, 64, r, io, seed=500 + T + r)
    kw = dict(P=P, eps_n=1e-3, tau=tau, t0=t0)
    got = gpu_scan(x, 1, N, mode="chunked", chunk=0, **kw)
    ref = oracle_scan(x, **kw, trace=True)
    _check(errs(got, ref), TOL if io == "bf16" else TOL_F32, f"chunked edge {io} N{N} T{T} r{r} P{P} tau{tau}")
    assert got[4]["renorm_count"] == int(ref[4]["renorm"].sum())


def test_chunked_f32_workload_parity():
    """b4h8_t4096_d64_f32 (float32 I/O, 32 pairs) in chunked mode: every pair against the
    oracle at the float32 gate, and against the sequential kernel."""
    w = workloads.get(1)
    x = workloads.make_inputs(w)
    kw = dict(P=w.P, eps_n=w.eps_n, tau=w.tau)
    got = gpu_scan(x, w.B, w.H, mode="chunked", chunk=0, **kw)
    assert got[4]["flags"] == 0 and got[4]["chunk_fallbacks"] == 0
    ref = oracle_scan(x, **kw)
    _check(errs(got, ref), TOL_F32, f"chunked {w.name} vs oracle")
    seq = gpu_scan(x, w.B, w.H, **kw)
    import oracle
    _check(oracle.errors(*got[:4], *seq[:4]), TOL_F32, f"chunked vs sequential {w.name}")


def _one_cta_pairs():
    """The smallest pair count that no longer fits two CTAs per pair on the SMs."""
    return torch.cuda.get_device_properties(0).multi_processor_count // 2 + 1


@pytest.mark.parametrize("io", ["bf16", "f32"])
@pytest.mark.parametrize("r,T,P,tau,t0", [(1, 300, 50, 12.0, 7), (4, 130, 20, 6.0, 3)])
def test_chunked_one_cta_and_cluster_agree(io, r, T, P, tau, t0):
    """The first three pairs alone (a cluster of two CTAs each) and inside a launch of
    SMs / 2 + 1 pairs (one CTA each): the same bits in o, A, S and n, with nudges that
    split chunks, a t0 phase, a ragged last chunk and renormalisation firing."""
    N = _one_cta_pairs()
    x = workloads.gaussian_inputs(N, T, 64, 64, r, io, seed=900 + r)
    kw = dict(P=P, eps_n=1e-3, tau=tau, t0=t0)
    one = gpu_scan(x, 1, N, mode="chunked", chunk=0, **kw)
    few = {k: v[:3].contiguous() for k, v in x.items()}
    clu = gpu_scan(few, 1, 3, mode="chunked", chunk=0, **kw)
    assert clu[4]["renorm_count"] > 0
    for i, name in enumerate("oASn"):
        assert np.array_equal(one[i][:3], clu[i]), name
    assert one[4]["flags"] == 0 and clu[4]["flags"] == 0


@pytest.mark.parametrize("form", ["cluster", "one_cta"])
@pytest.mark.parametrize("io", ["bf16", "f32"])
def test_chunked_guard_falls_back_step_by_step(io, form):
    N, T = (2 if form == "cluster" else _one_cta_pairs()), 40
    x = workloads.gaussian_inputs(N, T, 64, 64, 1, io, seed=77)
    x["A0"] = -torch.eye(64).expand(N, 64, 64).contiguous()
    x["u"][:, 0] = 0.0
    x["u"][:, 0, 0, 5] = 1.0          # exactly unit: delta = 1 - 1 = 0 at step 1
    x["u"][:, 1:] = (x["u"][:, 1:].float() * 0.5).to(x["u"].dtype)
    kw = dict(P=0, eps_n=0.0, tau=1e30)
    got = gpu_scan(x, 1, N, mode="chunked", chunk=0, **kw)
    ref = oracle_scan(x, **kw, trace=True)
    assert ref[4]["guard"][:, 0, 0].all()
    assert got[4]["chunk_fallbacks"] >= N
    assert got[4]["guard_count"] == int(ref[4]["guard"].sum())
    _check(errs(got, ref), TOL if io == "bf16" else TOL_F32, f"chunked guard fallback {io} {form}")


def test_chunked_rejects_shapes_it_does_not_build():
    import sherman_morrison_inverse_gb300 as vla
    x = workloads.gaussian_inputs(1, 8, 64, 64, 2, "f32", seed=3)   # r = 2
    with pytest.raises(vla.VlaError, match="UNSUPPORTED"):
        gpu_scan(x, 1, 1, mode="chunked", P=0, eps_n=0.0, tau=1e4)
    x = workloads.gaussian_inputs(1, 8, 16, 16, 1, "bf16", seed=3)
    with pytest.raises(vla.VlaError, match="UNSUPPORTED"):
        gpu_scan(x, 1, 1, mode="chunked", P=0, eps_n=0.0, tau=1e4)


def test_chunked_needs_aligned_o():
    import sherman_morrison_inverse_gb300 as vla
    x = workloads.gaussian_inputs(1, 8, 64, 64, 1, "bf16", seed=4)
    q, k, v = (x[n].reshape(1, 1, 8, 64).cuda() for n in ("q", "k", "v"))
    u = x["u"].reshape(1, 1, 8, 1, 64).cuda()
    A, S, n = x["A0"].reshape(1, 1, 64, 64).cuda(), x["S0"].reshape(1, 1, 64, 64).cuda(), x["n0"].reshape(1, 1, 64).cuda()
    buf = torch.empty(8 * 64 + 8, dtype=torch.bfloat16, device="cuda")
    o = buf[1:1 + 8 * 64].view(1, 1, 8, 64)   # 2-byte offset
    with pytest.raises(vla.VlaError, match="INVALID_ARG"):
        vla.scan_fwd(q, k, v, u, A, S, n, o, P=0, eps_n=0.0, tau=1e4, mode="chunked")
