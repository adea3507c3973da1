"""GPU parity of the host-buffer entry point (vla_scan_fwd_host).

The host path cuts the sequence into windows, copies each window of q, k, v, u
in, scans it with the same kernels as the device path and copies its o out,
with the state kept on the device between windows and t0 advanced window by
window.  So its results must equal, bit for bit, the device path called once
per window on the same inputs.  They are also checked against the float64
oracle at the mode's gate.  Both copy-in paths are covered: the SM gather
through the mapping of page-locked inputs, and the copy engines for pageable or
misaligned ones.  Edge cases: ragged last window, one window (default segment
on a short sequence), t0 phase, views into a larger page-locked buffer, a
workspace that grows between calls, and argument errors.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import workloads
from _util import ensure_built, errs, oracle_scan

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    ensure_built()
    import sherman_morrison_inverse_gb300 as vla
    vla.load_library()


def _host(x, B, H, pin=True):
    f = lambda t: t.reshape(B, H, *t.shape[1:]).contiguous()
    out = {k: f(x[k]) for k in ("q", "k", "v", "u", "A0", "S0", "n0")}
    if pin:
        out = {k: t.pin_memory() for k, t in out.items()}
    return out


def _device_windows(h, x, B, H, seg, **kw):
    """Reference: the device entry point called once per window of `seg` steps."""
    dev = torch.device("cuda")
    f = lambda t: t.reshape(B, H, *t.shape[1:]).to(dev).contiguous()
    g = {k: f(x[k]) for k in ("q", "k", "v", "u")}
    A, S, n = f(x["A0"]), f(x["S0"]), f(x["n0"])
    T = g["q"].shape[2]
    t0 = kw.pop("t0", 0)
    outs = []
    for off in range(0, T, seg):
        sl = lambda t: t[:, :, off:off + seg].contiguous()
        outs.append(h.scan_fwd(sl(g["q"]), sl(g["k"]), sl(g["v"]), sl(g["u"]), A, S, n, t0=t0 + off, **kw))
    o = torch.cat(outs, dim=2) if outs else torch.empty(0)
    st = h.status()
    return o.cpu(), A.cpu(), S.cpu(), n.cpu(), st


def _run_host(h, x, B, H, seg, pin=True, **kw):
    hx = _host(x, B, H, pin)
    A, S, n = hx["A0"].clone(), hx["S0"].clone(), hx["n0"].clone()
    if pin:
        A, S, n = A.pin_memory(), S.pin_memory(), n.pin_memory()
    o = h.scan_fwd_host(hx["q"], hx["k"], hx["v"], hx["u"], A, S, n, seg=seg, **kw)
    st = h.status()
    return o, A, S, n, st


def _same(a, b, label):
    for name, p, q in zip(("o", "A", "S", "n"), a[:4], b[:4]):
        assert torch.equal(p, q), (label, name, (p.float() - q.float()).abs().max().item())


CASES = [
    # (mode, N, T, d, r, io, seg, P, tau, t0, tol)
    ("sequential", 1, 256, 16, 1, "f32", 100, 64, 1e4, 0, 1e-4),    # ragged: 100, 100, 56
    ("sequential", 3, 700, 64, 4, "bf16", 256, 50, 1e4, 5, 2e-2),
    ("chunked", 4, 1000, 64, 1, "bf16", 256, 300, 1e4, 7, 2e-2),     # windows of whole chunks
    ("chunked", 2, 333, 64, 4, "bf16", 100, 1024, 3.0, 0, 2e-2),     # ragged chunks, renorm fires
    ("delta", 2, 300, 64, 1, "bf16", 128, 64, 1e4, 0, 2e-2),
    ("sequential", 2, 90, 128, 1, "f32", 0, 32, 1e4, 0, 1e-4),       # default: one window
]


@pytest.mark.parametrize("mode,N,T,d,r,io,seg,P,tau,t0,tol", CASES)
def test_host_path_equals_device_windows(mode, N, T, d, r, io, seg, P, tau, t0, tol):
    import sherman_morrison_inverse_gb300 as vla
    h = vla.default_handle()
    x = workloads.gaussian_inputs(N, T, d, d, r, io, seed=900 + T + d + r)
    kw = dict(P=P, eps_n=1e-3, tau=tau, t0=t0, mode=mode)
    got = _run_host(h, x, 1, N, seg, **kw)
    info = h.host_path_info()
    assert info["gathered"] == 1, info          # page-locked inputs: the SM gather
    assert info["seg"] == (seg if seg else T)
    ref_dev = _device_windows(h, x, 1, N, seg if seg else T, **kw)
    _same(got, ref_dev, f"host vs device windows {mode}")
    assert got[4] == ref_dev[4]
    assert got[4]["flags"] == 0
    ref = oracle_scan(x, P=P, eps_n=1e-3, tau=tau, t0=t0, rule="delta" if mode == "delta" else "additive")
    f = lambda t: t.reshape(N, *t.shape[2:]).double().numpy()
    e = errs(tuple(f(t) for t in got[:4]), ref)
    print(mode, {k: f"{v:.2e}" for k, v in e.items()})
    assert max(e.values()) <= tol, e


def test_host_path_full_length_recall_workload():
    """The recall workload's full length with the default windows, on a few pairs."""
    import sherman_morrison_inverse_gb300 as vla
    h = vla.default_handle()
    w = workloads.get(2)
    x = workloads.make_inputs(w, pairs=[0, 1, 2, 77])
    kw = dict(P=w.P, eps_n=w.eps_n, tau=w.tau, mode="chunked")
    got = _run_host(h, x, 1, 4, 0, **kw)
    assert h.host_path_info() == {"gathered": 1, "seg": 512}   # the default window at T = 16384
    ref_dev = _device_windows(h, x, 1, 4, 512, **kw)
    _same(got, ref_dev, "host vs device windows, recall workload")
    ref = oracle_scan(x, idx=[0, 3], P=w.P, eps_n=w.eps_n, tau=w.tau)
    f = lambda t: t.reshape(4, *t.shape[2:]).double().numpy()
    e = errs(tuple(f(t) for t in got[:4]), ref, idx=[0, 3])
    print({k: f"{v:.2e}" for k, v in e.items()})
    assert max(e.values()) <= 2e-2, e


def test_host_path_pageable_memory_and_growing_workspace():
    import sherman_morrison_inverse_gb300 as vla
    h = vla.Handle(0)
    try:
        for N, T, seg in ((1, 64, 32), (2, 500, 200), (3, 1500, 0)):   # the workspace grows twice
            x = workloads.gaussian_inputs(N, T, 64, 64, 1, "bf16", seed=40 + N)
            kw = dict(P=128, eps_n=1e-3, tau=1e4, mode="sequential")
            got = _run_host(h, x, 1, N, seg, pin=False, **kw)
            assert h.host_path_info()["gathered"] == 0      # pageable: the copy engines
            ref_dev = _device_windows(h, x, 1, N, seg if seg else T, **kw)
            _same(got, ref_dev, f"pageable N{N} T{T}")
    finally:
        h.close()


@pytest.mark.parametrize("shift,gathered", [(8, 0), (32, 1)])
def test_host_path_inputs_inside_a_larger_pinned_buffer(shift, gathered):
    """q is a view `shift` bytes into a larger page-locked buffer: 16-byte aligned views
    are gathered through the mapping, others go through the copy engines; same results."""
    import sherman_morrison_inverse_gb300 as vla
    h = vla.default_handle()
    N, T = 2, 700
    x = workloads.gaussian_inputs(N, T, 64, 64, 1, "bf16", seed=71)
    kw = dict(P=100, eps_n=1e-3, tau=1e4, mode="chunked")
    hx = _host(x, 1, N)
    nq = hx["q"].numel()
    big = torch.zeros(nq + 64, dtype=torch.bfloat16).pin_memory()
    qv = big[shift // 2: shift // 2 + nq].view(hx["q"].shape)
    qv.copy_(hx["q"])
    assert qv.data_ptr() % 16 == shift % 16
    A, S, n = (hx[k].clone().pin_memory() for k in ("A0", "S0", "n0"))
    o = h.scan_fwd_host(qv, hx["k"], hx["v"], hx["u"], A, S, n, seg=256, **kw)
    assert h.host_path_info()["gathered"] == gathered
    h.status()
    ref_dev = _device_windows(h, x, 1, N, 256, **kw)
    _same((o, A, S, n), ref_dev, f"view at +{shift} B")


def test_host_path_async_on_a_side_stream():
    """wait=False on a user stream: results are final once that stream is synchronised."""
    import sherman_morrison_inverse_gb300 as vla
    h = vla.default_handle()
    x = workloads.gaussian_inputs(2, 600, 64, 64, 1, "bf16", seed=61)
    kw = dict(P=100, eps_n=1e-3, tau=1e4, mode="chunked")
    hx = _host(x, 1, 2)
    A, S, n = (hx[k].clone().pin_memory() for k in ("A0", "S0", "n0"))
    s = torch.cuda.Stream()
    o = h.scan_fwd_host(hx["q"], hx["k"], hx["v"], hx["u"], A, S, n, seg=128, stream=s, wait=False, **kw)
    s.synchronize()
    h.status()
    ref_dev = _device_windows(h, x, 1, 2, 128, **kw)
    _same((o, A, S, n), ref_dev, "side stream")


def test_host_path_zero_sizes_and_errors():
    import sherman_morrison_inverse_gb300 as vla
    h = vla.default_handle()
    x = workloads.gaussian_inputs(1, 8, 64, 64, 1, "bf16", seed=5)
    hx = _host(x, 1, 1)
    A, S, n = hx["A0"].clone(), hx["S0"].clone(), hx["n0"].clone()
    kw = dict(P=0, eps_n=0.0, tau=1e4)
    with pytest.raises(vla.VlaError, match="INVALID_ARG"):
        h.scan_fwd_host(hx["q"], hx["k"], hx["v"], hx["u"], A, S, n, seg=-1, **kw)
    with pytest.raises(vla.VlaError, match="UNSUPPORTED"):   # chunked mode is built for d = 64 only
        xf = workloads.gaussian_inputs(1, 8, 16, 16, 1, "bf16", seed=5)
        hf = _host(xf, 1, 1)
        h.scan_fwd_host(hf["q"], hf["k"], hf["v"], hf["u"], hf["A0"], hf["S0"], hf["n0"], mode="chunked", **kw)
    with pytest.raises(ValueError, match="expected cpu"):
        h.scan_fwd_host(hx["q"].cuda(), hx["k"], hx["v"], hx["u"], A, S, n, **kw)
    # T == 0 leaves the state untouched
    e = {k: t[:, :, :0].contiguous() for k, t in hx.items() if k in ("q", "k", "v", "u")}
    A0 = A.clone()
    o = h.scan_fwd_host(e["q"], e["k"], e["v"], e["u"], A, S, n, **kw)
    assert o.shape[2] == 0 and torch.equal(A, A0)
    assert h.status()["flags"] == 0


def test_host_path_chunked_float32_matches_the_device_windows():
    """Float32 I/O in chunked mode (3xTF32, inputs read from global memory) through the host
    path: bit for bit the device entry point called once per window, and within the float32
    gate of the oracle."""
    import sherman_morrison_inverse_gb300 as vla
    h = vla.default_handle()
    N, T = 3, 640
    x = workloads.gaussian_inputs(N, T, 64, 64, 1, "f32", seed=83)
    kw = dict(P=100, eps_n=1e-3, tau=1e4, mode="chunked")
    hx = _host(x, 1, N)
    A, S, n = (hx[k].clone().pin_memory() for k in ("A0", "S0", "n0"))
    o = h.scan_fwd_host(hx["q"], hx["k"], hx["v"], hx["u"], A, S, n, seg=256, **kw)
    assert h.status()["flags"] == 0
    ref_dev = _device_windows(h, x, 1, N, 256, **kw)
    _same((o, A, S, n), ref_dev, "float32 chunked")
    import oracle
    ref = oracle_scan(x, P=100, eps_n=1e-3, tau=1e4)
    e = oracle.errors(o.reshape(N, T, 64).double().numpy(), A.reshape(N, 64, 64).double().numpy(),
                      S.reshape(N, 64, 64).double().numpy(), n.reshape(N, 64).double().numpy(), *ref[:4])
    assert max(e.values()) <= 1e-4, e
