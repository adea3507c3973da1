"""Helpers shared by the tests: build/load the library, run both sides."""
from __future__ import annotations

import os
import re

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "vla.h")


def ensure_built():
    """Build libvla.so if it is missing or older than any source or the header."""
    from sherman_morrison_inverse_gb300 import build as b
    lib = b.LIB
    deps = b.sources() + [os.path.join(b.CSRC, f) for f in os.listdir(b.CSRC) if f.endswith(".cuh")]
    deps.append(HEADER)
    if not os.path.exists(lib) or os.path.getmtime(lib) < max(os.path.getmtime(p) for p in deps):
        b.build()
    return lib


def header_functions() -> list[str]:
    """Names of the functions that include/vla.h declares."""
    txt = open(HEADER).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\**\s+\**(vla_\w+)\s*\(", txt, flags=re.M)))


def to_gpu(x: dict, B: int, H: int):
    """Workload inputs [N, ...] (N = B*H) -> CUDA tensors [B, H, ...]."""
    dev = torch.device("cuda")
    out = {}
    for key in ("q", "k", "v", "u", "A0", "S0", "n0"):
        t = x[key]
        out[key] = t.reshape(B, H, *t.shape[1:]).to(dev).contiguous()
    return out


def gpu_scan(x: dict, B: int, H: int, *, P, eps_n, tau, t0=0, mode="sequential", chunk=0, handle=None):
    """Run the CUDA scan on workload inputs; returns CPU float64 arrays [N, ...] and the status."""
    import sherman_morrison_inverse_gb300 as vla
    g = to_gpu(x, B, H)
    A, S, n = g["A0"].clone(), g["S0"].clone(), g["n0"].clone()
    h = handle or vla.default_handle()
    h.status()  # reset
    o = h.scan_fwd(g["q"], g["k"], g["v"], g["u"], A, S, n, P=P, eps_n=eps_n, tau=tau, t0=t0,
                   mode=mode, chunk=chunk)
    st = h.status()
    N = B * H
    f = lambda t: t.reshape(N, *t.shape[2:]).double().cpu().numpy()
    return f(o), f(A), f(S), f(n), st


def oracle_scan(x: dict, idx=None, **kw):
    import oracle
    sel = (lambda t: t) if idx is None else (lambda t: t[idx])
    return oracle.scan(sel(x["q"]), sel(x["k"]), sel(x["v"]), sel(x["u"]), sel(x["A0"]), sel(x["S0"]),
                       sel(x["n0"]), **kw)


def errs(gpu, ref, idx=None):
    import oracle
    o, A, S, n = gpu[:4]
    if idx is not None:
        o, A, S, n = o[idx], A[idx], S[idx], n[idx]
    return oracle.errors(o, A, S, n, *ref[:4])


def bf16_round(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.asarray(x, np.float64)).to(torch.bfloat16).double().numpy()
