"""The entry point that allocates nothing (vla_scan_fwd_noalloc).

Some callers may not allocate device memory: code running under a framework or
server whose allocator owns the GPU's memory, and callers that keep no handle
between calls.  vla_scan_fwd_noalloc serves them with the same scan as
vla_scan_fwd; its scratch (one status record per (batch, head) pair) is a
static array inside the library.  These tests call it through the C ABI and
check, on two calls in a row, that it gives the existing entry point's results
bit for bit,
that each call starts its status records from zero, and that sizes beyond the
static scratch are refused.  This file is collected last so that a failure here
stops a run only after every other test has run; it passes on its own as well.
"""
from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

import workloads
from _util import ensure_built

pytestmark = pytest.mark.gpu

@pytest.fixture(scope="module")
def vla():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    ensure_built()
    import sherman_morrison_inverse_gb300 as mod
    mod.load_library()
    return mod


def _gpu(x, key, a, b):
    t = x[key][:, a:b]
    return t.reshape(1, t.shape[0], *t.shape[1:]).cuda().contiguous()


def _noalloc_call(vla, q, k, v, u, A, S, n, o, *, P, eps_n, tau, t0, pair_status=None):
    lib = vla.load_library()
    B, H, T, d = q.shape
    r = u.shape[3]
    io = vla.F32 if q.dtype == torch.float32 else vla.BF16
    ps = ctypes.cast(pair_status, ctypes.c_void_p) if pair_status is not None else None
    return lib.vla_scan_fwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), u.data_ptr(), A.data_ptr(),
                                    S.data_ptr(), n.data_ptr(), o.data_ptr(), B, H, T, d, d, r, P, eps_n,
                                    tau, t0, io, ps, torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("io,r", [("f32", 1), ("bf16", 4)])
def test_two_calls_match_the_handle_entry_point(vla, io, r):
    N, T1, T2 = 5, 300, 157           # ragged lengths, the second call continues the first
    x = workloads.gaussian_inputs(N, T1 + T2, 64, 64, r, io, seed=4242 + r)
    kw = dict(P=64, eps_n=1e-3, tau=40.0)
    A0 = x["A0"].reshape(1, N, 64, 64).cuda()
    S0 = x["S0"].reshape(1, N, 64, 64).cuda()
    n0 = x["n0"].reshape(1, N, 64).cuda()
    ref_state = [A0.clone(), S0.clone(), n0.clone()]
    new_state = [A0.clone(), S0.clone(), n0.clone()]
    h = vla.Handle()
    for a, b in ((0, T1), (T1, T1 + T2)):
        g = [_gpu(x, key, a, b) for key in ("q", "k", "v", "u")]
        o_ref = h.scan_fwd(*g, *ref_state, t0=a, **kw)
        o_new = torch.empty_like(o_ref)
        recs = (vla.VlaPairStatus * N)()
        assert _noalloc_call(vla, *g, *new_state, o_new, t0=a, pair_status=recs, **kw) == 0, \
            vla.load_library().vla_last_error(None)
        torch.cuda.synchronize()
        # both entry points run the same sequential kernel on the same inputs (they differ only
        # in where the status records go), so the results agree bit for bit
        assert torch.equal(o_new, o_ref), "o differs from vla_scan_fwd"
        for got, want, name in zip(new_state, ref_state, "ASn"):
            assert torch.equal(got, want), f"{name} differs from vla_scan_fwd"
        st = h.status()
        assert st["flags"] == 0 and all(rec.flags == 0 for rec in recs)
        assert sum(rec.renorm_count for rec in recs) == st["renorm_count"]
    h.close()


def test_status_records_start_from_zero_on_every_call(vla):
    N, T = 4, 96
    x = workloads.gaussian_inputs(N, T, 64, 64, 1, "f32", seed=9)
    bad = {k: v.clone() for k, v in x.items()}
    bad["q"][2, 10, 5] = float("nan")
    for inputs, want_bad in ((bad, True), (x, False)):
        g = [_gpu(inputs, key, 0, T) for key in ("q", "k", "v", "u")]
        A = inputs["A0"].reshape(1, N, 64, 64).cuda()
        S = inputs["S0"].reshape(1, N, 64, 64).cuda()
        n = inputs["n0"].reshape(1, N, 64).cuda()
        o = torch.empty(1, N, T, 64, device="cuda")
        recs = (vla.VlaPairStatus * N)()
        assert _noalloc_call(vla, *g, A, S, n, o, P=32, eps_n=1e-6, tau=1e4, t0=0, pair_status=recs) == 0
        torch.cuda.synchronize()
        flags = [rec.flags for rec in recs]
        if want_bad:
            assert flags[2] & vla.STATUS_NONFINITE and flags[0] == flags[1] == flags[3] == 0, flags
        else:
            assert flags == [0] * N, flags
            assert np.isfinite(o.cpu().numpy()).all()


def test_sizes_beyond_the_static_scratch_are_refused(vla):
    lib = vla.load_library()
    x = torch.zeros(16, device="cuda")
    p = x.data_ptr()
    code = lib.vla_scan_fwd_noalloc(p, p, p, p, p, p, p, p, 16385, 1, 8, 64, 64, 1, 0, 0.0, 1.0, 0,
                                    vla.F32, None, None)
    assert code == 1
    assert b"VLA_NOALLOC_MAX_PAIRS" in lib.vla_last_error(None)
    assert lib.vla_scan_fwd_noalloc(p, p, p, p, p, p, p, p, 1, 1, 8, 32, 32, 1, 0, 0.0, 1.0, 0,
                                    vla.F32, None, None) == 2
