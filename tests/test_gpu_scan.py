"""GPU parity of the sequential scan kernel against the float64 oracle.

Every call goes through the C ABI (ctypes binding).  Gates (max error as
defined by ``oracle.errors``): 1e-4 for float32 I/O at T <= 4096, 1e-3 for the
T = 65536 float32 workload, 2e-2 for bfloat16 I/O with float32 state.  At the
full workload sizes the GPU runs every pair and the oracle a sample of pairs
(pairs are independent, so the sample is checked exactly).
"""
from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

import workloads
from _util import ensure_built, errs, gpu_scan, oracle_scan, to_gpu

pytestmark = pytest.mark.gpu

TOL_F32 = 1e-4
TOL_F32_LONG = 1e-3
TOL_BF16 = 2e-2


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    ensure_built()
    import sherman_morrison_inverse_gb300 as vla
    vla.load_library()


def _params(w):
    return dict(P=w.P, eps_n=w.eps_n, tau=w.tau)


def _check(e, tol, label):
    print(label, {k: f"{v:.2e}" for k, v in e.items()})
    assert max(e.values()) <= tol, (label, e)


@pytest.mark.parametrize("idx", [0, 1])
def test_workload_full_parity(idx):
    w = workloads.get(idx)
    x = workloads.make_inputs(w)
    got = gpu_scan(x, w.B, w.H, **_params(w))
    ref = oracle_scan(x, **_params(w), trace=True)
    _check(errs(got, ref), TOL_F32, w.name)
    assert got[4]["guard_count"] == int(ref[4]["guard"].sum())
    assert got[4]["renorm_count"] == int(ref[4]["renorm"].sum())
    assert got[4]["flags"] == 0


@pytest.mark.parametrize("idx,sample,tol", [(2, [0, 37, 127], TOL_BF16),
                                            (3, [0, 15], TOL_F32_LONG),
                                            (4, [0, 131, 255], TOL_BF16)])
def test_workload_sampled_parity(idx, sample, tol):
    w = workloads.get(idx)
    x = workloads.make_inputs(w)
    got = gpu_scan(x, w.B, w.H, **_params(w))
    ref = oracle_scan(x, idx=sample, **_params(w), trace=True)
    _check(errs(got, ref, idx=sample), tol, w.name)
    assert got[4]["flags"] == 0
    # properties that hold for every pair, not only the sampled ones
    o, A, S, n = got[:4]
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(A))
    assert np.max(np.abs(A - A.transpose(0, 2, 1))) <= 1e-3 * np.max(np.abs(A))
    assert np.all(np.linalg.norm(S.reshape(S.shape[0], -1), axis=1) <= w.tau * (1 + 1e-5))


EDGE = [
    # (N, T, d, r, io, P, tau, t0)
    (1, 1, 16, 1, "f32", 64, 1e4, 0),
    (3, 7, 16, 4, "f32", 3, 1e4, 5),
    (2, 100, 64, 1, "f32", 16, 1e4, 0),
    (2, 33, 64, 4, "bf16", 8, 1e4, 1),
    (1, 200, 64, 1, "f32", 50, 4.0, 0),      # renormalisation fires most steps
    (2, 37, 128, 1, "f32", 10, 1e4, 3),
    (1, 20, 128, 4, "bf16", 7, 2.0, 0),
    (5, 65, 16, 1, "bf16", 0, 1e4, 0),       # P = 0: no nudge
]


@pytest.mark.parametrize("N,T,d,r,io,P,tau,t0", EDGE)
def test_edge_shapes(N, T, d, r, io, P, tau, t0):
    x = workloads.gaussian_inputs(N, T, d, d, r, io, seed=1000 + T + d + r)
    kw = dict(P=P, eps_n=1e-3, tau=tau, t0=t0)
    got = gpu_scan(x, 1, N, **kw)
    ref = oracle_scan(x, **kw, trace=True)
    _check(errs(got, ref), TOL_F32 if io == "f32" else TOL_BF16, f"edge N{N} T{T} d{d} r{r} {io}")
    assert got[4]["renorm_count"] == int(ref[4]["renorm"].sum())


def test_split_calls_match_one_call():
    w = workloads.get(1).with_(B=1, H=4, T=600)
    x = workloads.make_inputs(w.with_(T=4096), pairs=range(4), T=600)
    kw = dict(P=64, eps_n=1e-3, tau=30.0)
    whole = gpu_scan(x, 1, 4, **kw)
    import sherman_morrison_inverse_gb300 as vla
    g = to_gpu(x, 1, 4)
    A, S, n = g["A0"].clone(), g["S0"].clone(), g["n0"].clone()
    outs = []
    for a, b in ((0, 250), (250, 251), (251, 600)):
        outs.append(vla.scan_fwd(g["q"][:, :, a:b].contiguous(), g["k"][:, :, a:b].contiguous(),
                                 g["v"][:, :, a:b].contiguous(), g["u"][:, :, a:b].contiguous(),
                                 A, S, n, t0=a, **kw))
    o = torch.cat(outs, dim=2).reshape(4, 600, -1).double().cpu().numpy()
    import oracle
    e = oracle.errors(o, A.reshape(4, 64, 64).cpu(), S.reshape(4, 64, 64).cpu(), n.reshape(4, 64).cpu(),
                      *whole[:4])
    _check(e, 1e-5, "split vs whole")
    ref = oracle_scan(x, **kw)
    _check(errs((o, A.reshape(4, 64, 64).cpu().double().numpy(), S.reshape(4, 64, 64).cpu().double().numpy(),
                 n.reshape(4, 64).cpu().double().numpy()), ref), TOL_F32, "split vs oracle")


def test_guard_through_the_abi():
    """A0 = -I and a unit u give delta = 0 at step 1: the guard replaces the update
    with A += 1e-6 I.  Later directions are scaled by 1/2 so that their deltas
    (about 3/4) sit far from the threshold in both precisions."""
    d = 16
    x = workloads.gaussian_inputs(2, 6, d, d, 1, "f32", seed=5)
    x["A0"] = -torch.eye(d).expand(2, d, d).contiguous()
    x["u"][:, 1:] *= 0.5
    got = gpu_scan(x, 1, 2, P=0, eps_n=0.0, tau=1e30)
    ref = oracle_scan(x, P=0, eps_n=0.0, tau=1e30, trace=True)
    assert ref[4]["guard"][:, 0, 0].all()
    assert got[4]["guard_count"] == int(ref[4]["guard"].sum())
    _check(errs(got, ref), TOL_F32, "guard")


def test_nonfinite_input_is_reported():
    x = workloads.gaussian_inputs(2, 40, 64, 64, 1, "f32", seed=6)
    x["q"][1, 5, 3] = float("nan")
    got = gpu_scan(x, 1, 2, P=16, eps_n=1e-6, tau=1e4)
    assert got[4]["nonfinite"]
    ref = oracle_scan(x, idx=[0], P=16, eps_n=1e-6, tau=1e4)
    _check(errs(got, ref, idx=[0]), TOL_F32, "clean pair next to a NaN pair")


def _raw_call(h, t, **over):
    """Call vla_scan_fwd with explicit pointers (for the error paths)."""
    lib = h.lib
    args = dict(q=t["q"].data_ptr(), k=t["k"].data_ptr(), v=t["v"].data_ptr(), u=t["u"].data_ptr(),
                A=t["A"].data_ptr(), S=t["S"].data_ptr(), n=t["n"].data_ptr(), o=t["o"].data_ptr(),
                B=1, H=2, T=8, d=64, dv=64, r=1, P=4, eps=1e-6, tau=1e4, t0=0, dtype=0, mode=0, chunk=0)
    args.update(over)
    return lib.vla_scan_fwd(h.ptr, args["q"], args["k"], args["v"], args["u"], args["A"], args["S"],
                            args["n"], args["o"], args["B"], args["H"], args["T"], args["d"], args["dv"],
                            args["r"], args["P"], args["eps"], args["tau"], args["t0"], args["dtype"],
                            args["mode"], args["chunk"], None)


def _raw_tensors(N=2, T=8, d=64):
    dev = torch.device("cuda")
    return dict(q=torch.randn(N, T, d, device=dev), k=torch.randn(N, T, d, device=dev),
                v=torch.randn(N, T, d, device=dev), u=torch.randn(N, T, 1, d, device=dev),
                A=torch.eye(d, device=dev).repeat(N, 1, 1), S=torch.zeros(N, d, d, device=dev),
                n=torch.zeros(N, d, device=dev), o=torch.zeros(N, T, d, device=dev))


def test_argument_errors_launch_nothing():
    import sherman_morrison_inverse_gb300 as vla
    h = vla.Handle()
    t = _raw_tensors()
    before = {k: v.clone() for k, v in t.items()}
    assert _raw_call(h, t, u=t["u"].data_ptr() + 4) == 1          # misaligned
    assert _raw_call(h, t, A=t["A"].data_ptr() + 8) == 1
    assert _raw_call(h, t, q=0) == 1                              # NULL
    assert _raw_call(h, t, P=-1) == 1
    assert _raw_call(h, t, tau=0.0) == 1
    assert _raw_call(h, t, tau=float("nan")) == 1
    assert _raw_call(h, t, t0=-3) == 1
    assert _raw_call(h, t, T=-1) == 1
    assert _raw_call(h, t, d=32, dv=32) == 2                      # not built
    assert _raw_call(h, t, d=64, dv=16) == 2
    assert _raw_call(h, t, r=2) == 2
    assert _raw_call(h, t, dtype=7) == 1
    assert _raw_call(h, t, T=0) == 0                              # no-op
    assert _raw_call(h, t, B=0) == 0
    torch.cuda.synchronize()
    for k in t:
        assert torch.equal(t[k], before[k]), k
    assert h.status()["flags"] == 0
    h.close()


def test_outputs_stay_inside_their_buffers():
    """Poisoned guard bands around o, A, S and n must come back untouched."""
    import sherman_morrison_inverse_gb300 as vla
    h = vla.Handle()
    N, T, d, pad = 3, 45, 64, 4096
    t = _raw_tensors(N, T, d)
    poison = -7.25e13
    big = {}
    for key in ("A", "S", "n", "o"):
        flat = torch.full((t[key].numel() + 2 * pad,), poison, device="cuda")
        flat[pad:pad + t[key].numel()] = t[key].reshape(-1)
        big[key] = flat
        t[key] = flat[pad:pad + t[key].numel()].view_as(t[key])
    t["u"] = torch.nn.functional.normalize(t["u"], dim=-1)
    assert _raw_call(h, t, B=1, H=N, T=T) == 0
    torch.cuda.synchronize()
    for key, flat in big.items():
        assert torch.all(flat[:pad] == poison) and torch.all(flat[-pad:] == poison), key
    assert h.status()["flags"] == 0
    h.close()


def test_a_wait_that_runs_out_reports_a_timeout_and_leaves_the_context_usable():
    """The bounded-wait path of every kernel: a wait on an mbarrier that nothing completes
    gives up after its limit and sets the timeout flag; the next scan runs normally."""
    import time
    import sherman_morrison_inverse_gb300 as vla
    h = vla.default_handle()
    h.status()
    t0 = time.perf_counter()
    h.selftest_wait(200)
    st = h.status()   # synchronises
    waited = time.perf_counter() - t0
    assert st["timeout"] and st["flags"] == vla.STATUS_TIMEOUT
    assert 0.19 <= waited < 5.0
    x = workloads.gaussian_inputs(2, 50, 16, 16, 1, "f32", seed=9)
    got = gpu_scan(x, 1, 2, P=16, eps_n=1e-3, tau=1e4)
    assert got[4]["flags"] == 0
    assert max(errs(got, oracle_scan(x, P=16, eps_n=1e-3, tau=1e4)).values()) <= 1e-4
    with pytest.raises(vla.VlaError, match="INVALID_ARG"):
        h.selftest_wait(0)
