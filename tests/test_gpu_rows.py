"""GPU tests of the row-split sequential scan (`chunk` = 4 or 8 CTAs per pair).

Each (batch, head) pair runs on a cluster of 4 or 8 CTAs; CTA c holds rows
[c d/NC, (c+1) d/NC) of A and the same columns of S, and the CTAs exchange the slices
of z and the partial sums of every step through distributed shared memory
("Mathematical Primitives" §2-§5, README "VLA v3" items 1-5).  The step is the
oracle's step by step, so the float32 gate (1e-4) holds at these lengths, and the
singularity guard, the nudges (with a t0 phase) and the renormalisation must fire
exactly where the oracle's do.  A call carries no state besides A, S and n, so a
sequence split into calls at any step gives the same bits as one call.
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


CASES = [
    # (N, T, d, ctas, io, P, tau, t0)
    (3, 300, 64, 4, "f32", 64, 1e4, 0),
    (2, 301, 64, 8, "bf16", 60, 6.0, 9),       # renormalisation fires; ragged last tile
    (4, 517, 64, 4, "bf16", 1024, 8.0, 0),     # renormalisation fires
    (2, 300, 128, 4, "f32", 64, 1e3, 0),
    (2, 301, 128, 4, "bf16", 60, 6.0, 9),
    (2, 77, 128, 8, "f32", 16, 3.0, 1),        # nudges with a t0 phase, renormalisation
    (1, 1, 64, 4, "f32", 1, 1e4, 0),           # one step, nudged
    (2, 33, 128, 8, "f32", 0, 1e4, 0),         # no nudges, just past one 16-step tile
]


@pytest.mark.parametrize("N,T,d,ctas,io,P,tau,t0", CASES)
def test_row_split_matches_oracle(N, T, d, ctas, io, P, tau, t0):
    x = workloads.gaussian_inputs(N, T, d, d, 1, io, seed=1300 + d + ctas + T)
    kw = dict(P=P, eps_n=1e-3, tau=tau, t0=t0)
    got = gpu_scan(x, 1, N, chunk=ctas, **kw)
    ref = oracle_scan(x, **kw, trace=True)
    e = errs(got, ref)
    tol = 1e-4 if io == "f32" else 2e-2
    assert max(e.values()) <= tol, e
    assert got[4]["flags"] == 0, got[4]
    if io == "f32":   # the same decisions as the oracle (bf16 I/O rounds the inputs the same way,
        # but a norm within rounding of tau may decide either way there)
        assert got[4]["renorm_count"] == int(ref[4]["renorm"].sum()), (got[4], int(ref[4]["renorm"].sum()))
    assert got[4]["guard_count"] == int(ref[4]["guard"].sum())


@pytest.mark.parametrize("d,ctas", [(64, 4), (128, 8)])
def test_row_split_guard(d, ctas):
    """u_0 = e_3 with A_0 = -I gives delta = 0: the guard (A += 1e-6 I, no update) fires in
    every CTA at once, and the later steps continue from there."""
    x = workloads.gaussian_inputs(2, 40, d, d, 1, "f32", seed=55)
    x["A0"] = -torch.eye(d).expand(2, d, d).contiguous()
    x["u"][:, 0] = 0.0
    x["u"][:, 0, 0, 3] = 1.0
    x["u"][:, 1:] *= 0.5
    kw = dict(P=0, eps_n=0.0, tau=1e30)
    got = gpu_scan(x, 1, 2, chunk=ctas, **kw)
    ref = oracle_scan(x, **kw, trace=True)
    assert got[4]["guard_count"] == int(ref[4]["guard"].sum()) > 0
    assert max(errs(got, ref).values()) <= 1e-4


@pytest.mark.parametrize("d,ctas", [(64, 4), (128, 4)])
def test_row_split_split_calls_give_the_same_bits(d, ctas):
    import sherman_morrison_inverse_gb300 as vla
    N, T1, T2 = 3, 200, 131
    x = workloads.gaussian_inputs(N, T1 + T2, d, d, 1, "f32", seed=77)
    kw = dict(P=64, eps_n=1e-3, tau=5.0)
    whole = gpu_scan(x, 1, N, chunk=ctas, **kw)
    assert whole[4]["renorm_count"] > 0
    dev = torch.device("cuda")
    A = x["A0"].reshape(1, N, d, d).to(dev).contiguous()
    S = x["S0"].reshape(1, N, d, d).to(dev).contiguous()
    n = x["n0"].reshape(1, N, d).to(dev).contiguous()
    outs = []
    for a, b in ((0, T1), (T1, T1 + T2)):
        g = [x[k][:, a:b].reshape(1, N, b - a, *x[k].shape[2:]).to(dev).contiguous() for k in ("q", "k", "v", "u")]
        outs.append(vla.scan_fwd(*g, A, S, n, t0=a, chunk=ctas, **kw))
    o = torch.cat(outs, dim=2).reshape(N, T1 + T2, d).double().cpu().numpy()
    assert np.array_equal(o, whole[0])
    assert np.array_equal(A.reshape(N, d, d).double().cpu().numpy(), whole[1])
    assert np.array_equal(S.reshape(N, d, d).double().cpu().numpy(), whole[2])
    assert np.array_equal(n.reshape(N, d).double().cpu().numpy(), whole[3])


@pytest.mark.parametrize("ctas", [4, 8])
def test_row_split_long_context_workload_prefix(ctas):
    """b2h8_t65536_d128_f32 (B H = 16 pairs, 16 clusters), the first 8192 steps, two pairs
    against the oracle at the long-context gate."""
    w = workloads.get(3)
    T = 8192
    x = workloads.make_inputs(w, T=T)
    kw = dict(P=w.P, eps_n=w.eps_n, tau=w.tau)
    got = gpu_scan(x, w.B, w.H, chunk=ctas, **kw)
    assert got[4]["flags"] == 0
    ref = oracle_scan(x, idx=[0, 11], **kw)
    e = errs(got, ref, idx=[0, 11])
    assert max(e.values()) <= 1e-3, e


@pytest.mark.parametrize("d,r,ctas", [(16, 1, 4), (64, 4, 4), (128, 4, 8)])
def test_row_split_unbuilt_shapes_are_refused(d, r, ctas):
    import sherman_morrison_inverse_gb300 as vla
    x = workloads.gaussian_inputs(1, 8, d, d, r, "f32", seed=3)
    with pytest.raises(vla.VlaError, match="UNSUPPORTED"):
        gpu_scan(x, 1, 1, chunk=ctas, P=0, eps_n=0.0, tau=1e4)
