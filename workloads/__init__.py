"""Seeded synthetic workloads for the VLA forward scan.

This module only draws random numbers and lays them out; it holds none of the
scan's arithmetic.  Both the CUDA path (through the tests and the bench) and the
float64 oracle receive the *same* arrays from here, already rounded to the I/O
precision of the workload, so the two sides never disagree about their inputs.

What each workload draws (Variational Linear Attention, "VLA v3 (Research
Implementation Notes)" items 1-2 on the project README page; the five sizes are
the scan's benchmark configurations):

* q_raw, v ~ N(0, 1) i.i.d.  (the feature map phi = ELU+1 is applied by the scan,
  not here).
* k_raw ~ N(0, 1) i.i.d., except for the associative-recall workload (see
  ``_recall_keys``).
* u_{t,i} = W_u^{(i)} k_raw_t / max(||W_u^{(i)} k_raw_t||_2, 1e-12): the pages'
  learned penalty direction "normalize(W_u k_raw)", with W_u^{(i)} ~ N(0, 1/d)
  (second argument = variance).  It is formed here in float64 and then rounded,
  because the scan takes u as an input; the scan does not renormalise it.
* A0 = I, S0 = 0, n0 = 0, t0 = 0.

Randomness is reproducible per (batch, head) pair: pair p of workload c draws
from ``numpy.random.default_rng([seed_c, 1, p])``, shared matrices (W_u, the
recall directions) from ``default_rng([seed_c, 0])``.  Any subset of pairs can
therefore be generated on its own and equals the same rows of the full batch.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace
from typing import Iterable, Sequence

import numpy as np
import torch

__all__ = ["Workload", "WORKLOADS", "get", "make_inputs", "round_to_io"]


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    T: int
    d: int
    dv: int
    r: int
    io: str            # "f32" or "bf16": dtype of q, k, v, u and o; state is always f32
    P: int             # nudge period (A += eps_n I at global steps g with g % P == 0)
    eps_n: float
    tau: float         # renormalisation threshold on ||S||_F
    keys: str = "gauss"  # "gauss" or "recall"
    seed: int = 0
    notes: str = ""

    @property
    def pairs(self) -> int:
        return self.B * self.H

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


def _w(idx: int, **kw) -> Workload:
    return Workload(seed=20260000 + idx, **kw)


#: The five benchmark configurations of the scan (index = position).
WORKLOADS: tuple[Workload, ...] = (
    _w(0, name="tiny_d16_f32", B=1, H=1, T=256, d=16, dv=16, r=1, io="f32",
       P=64, eps_n=1e-6, tau=1e4),
    _w(1, name="b4h8_t4096_d64_f32", B=4, H=8, T=4096, d=64, dv=64, r=1, io="f32",
       P=1024, eps_n=1e-6, tau=1e4),
    _w(2, name="b8h16_t16384_d64_bf16_recall", B=8, H=16, T=16384, d=64, dv=64, r=1,
       io="bf16", P=1024, eps_n=1e-6, tau=1e4, keys="recall"),
    _w(3, name="b2h8_t65536_d128_f32", B=2, H=8, T=65536, d=128, dv=128, r=1, io="f32",
       P=4096, eps_n=1e-6, tau=1e3),
    _w(4, name="b16h16_t8192_d64_bf16_r4", B=16, H=16, T=8192, d=64, dv=64, r=4,
       io="bf16", P=1024, eps_n=1e-6, tau=1e4),
)


def get(idx_or_name) -> Workload:
    if isinstance(idx_or_name, Workload):
        return idx_or_name
    if isinstance(idx_or_name, int):
        return WORKLOADS[idx_or_name]
    for w in WORKLOADS:
        if w.name == idx_or_name:
            return w
    raise KeyError(idx_or_name)


# ----------------------------------------------------------------------------
# rounding to the I/O precision
# ----------------------------------------------------------------------------

def round_to_io(x: np.ndarray, io: str) -> torch.Tensor:
    """float64 array -> CPU tensor in the I/O dtype (torch's round-to-nearest).

    Whatever rounding torch applies, both sides of a comparison receive the
    resulting values, so the choice does not affect parity.
    """
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float64))
    if io == "f32":
        return t.to(torch.float32)
    if io == "bf16":
        return t.to(torch.bfloat16)
    raise ValueError(io)


# ----------------------------------------------------------------------------
# generators
# ----------------------------------------------------------------------------

def _shared(w: Workload):
    g = np.random.default_rng([w.seed, 0])
    Wu = g.normal(0.0, np.sqrt(1.0 / w.d), size=(w.r, w.d, w.d))
    dirs = g.normal(0.0, 1.0, size=(256, w.d)) if w.keys == "recall" else None
    return Wu, dirs


def _recall_keys(g: np.random.Generator, T: int, d: int, dirs: np.ndarray) -> np.ndarray:
    """Associative-recall-shaped keys for one (b, h) pair.

    Each of the shared directions gets a repeat count c ~ U{1..8}; its c
    occurrences sit at distinct uniformly random positions and are the direction
    plus N(0, 0.05) noise.  Every other position holds a filler key ~ N(0, 1).
    """
    k = g.normal(0.0, 1.0, size=(T, d))
    counts = g.integers(1, 9, size=dirs.shape[0])
    total = int(counts.sum())
    if total > T:
        raise ValueError("sequence too short for the recall keys")
    pos = g.permutation(T)[:total]
    owner = np.repeat(np.arange(dirs.shape[0]), counts)
    noise = g.normal(0.0, np.sqrt(0.05), size=(total, d))
    k[pos] = dirs[owner] + noise
    return k


def _pair_arrays(w: Workload, p: int, Wu: np.ndarray, dirs, T: int):
    g = np.random.default_rng([w.seed, 1, p])
    q = g.normal(0.0, 1.0, size=(T, w.d))
    if w.keys == "recall":
        k = _recall_keys(g, T, w.d, dirs)
    else:
        k = g.normal(0.0, 1.0, size=(T, w.d))
    v = g.normal(0.0, 1.0, size=(T, w.dv))
    # u_{t,i} = normalize(W_u^{(i)} k_t): a projection followed by a unit scaling.
    proj = np.einsum("iab,tb->tia", Wu, k)                   # [T, r, d]
    nrm = np.maximum(np.linalg.norm(proj, axis=-1, keepdims=True), 1e-12)
    u = proj / nrm
    return q, k, v, u


def make_inputs(w: Workload | int | str, pairs: Sequence[int] | None = None,
                T: int | None = None) -> dict:
    """Inputs of workload ``w`` as CPU tensors.

    Returns a dict with q, k [N, T, d], v [N, T, dv], u [N, T, r, d] in the I/O
    dtype (N = number of selected pairs, in the order given) and A0 [N, d, d],
    S0 [N, dv, d], n0 [N, d] in float32, Wu [r, d, d] (the shared projection
    weights, float32), plus ``pairs`` and ``workload``.
    ``T`` truncates the sequence (the first T steps; identical prefix values).
    """
    w = get(w)
    if pairs is None:
        pairs = range(w.pairs)
    pairs = list(pairs)
    T_full = w.T
    T_use = T_full if T is None else int(T)
    Wu, dirs = _shared(w)
    io_t = torch.float32 if w.io == "f32" else torch.bfloat16
    N = len(pairs)
    q = torch.empty((N, T_use, w.d), dtype=io_t)
    k = torch.empty((N, T_use, w.d), dtype=io_t)
    v = torch.empty((N, T_use, w.dv), dtype=io_t)
    u = torch.empty((N, T_use, w.r, w.d), dtype=io_t)
    for j, p in enumerate(pairs):
        if not (0 <= p < w.pairs):
            raise IndexError(p)
        qa, ka, va, ua = _pair_arrays(w, p, Wu, dirs, T_full)
        q[j] = round_to_io(qa[:T_use], w.io)
        k[j] = round_to_io(ka[:T_use], w.io)
        v[j] = round_to_io(va[:T_use], w.io)
        u[j] = round_to_io(ua[:T_use], w.io)
    A0 = torch.eye(w.d, dtype=torch.float32).expand(N, w.d, w.d).contiguous()
    S0 = torch.zeros((N, w.dv, w.d), dtype=torch.float32)
    n0 = torch.zeros((N, w.d), dtype=torch.float32)
    Wu_f32 = torch.from_numpy(np.ascontiguousarray(Wu)).float()   # [r, d, d], the shared projection weights
    return dict(q=q, k=k, v=v, u=u, A0=A0, S0=S0, n0=n0, Wu=Wu_f32, pairs=pairs, workload=w)


def gaussian_inputs(N: int, T: int, d: int, dv: int, r: int, io: str, seed: int,
                    u_scale: float = 1.0) -> dict:
    """Free-form i.i.d. inputs for edge-case tests (any sizes).

    q, k, v ~ N(0, 1); u = normalize(g) * u_scale with g ~ N(0, I).  Same layout
    and dtypes as ``make_inputs``.
    """
    g = np.random.default_rng([seed, 7])
    q = g.normal(size=(N, T, d))
    k = g.normal(size=(N, T, d))
    v = g.normal(size=(N, T, dv))
    uu = g.normal(size=(N, T, r, d))
    uu = uu / np.maximum(np.linalg.norm(uu, axis=-1, keepdims=True), 1e-12) * u_scale
    A0 = torch.eye(d, dtype=torch.float32).expand(N, d, d).contiguous()
    return dict(q=round_to_io(q, io), k=round_to_io(k, io), v=round_to_io(v, io),
                u=round_to_io(uu, io), A0=A0,
                S0=torch.zeros((N, dv, d), dtype=torch.float32),
                n0=torch.zeros((N, d), dtype=torch.float32))
