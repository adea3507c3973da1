"""Variational Linear Attention forward scan on GB300 (sm_103a).

Thin Python binding over the C ABI in ``include/vla.h`` (``libvla.so``, built
in-tree by ``sherman_morrison_inverse_gb300.build``).  It only marshals
arguments: shapes, dtypes and devices are checked, pointers and the current
CUDA stream are passed, and every step of the scan runs in the library's CUDA
kernels.  There is no fallback: without the built library every call raises.

    o = scan_fwd(q, k, v, u, A, S, n, P=1024, eps_n=1e-6, tau=1e4)

q, k [B, H, T, d] and v [B, H, T, d_v] and u [B, H, T, r, d] are CUDA tensors of
one dtype (float32 or bfloat16); A [B, H, d, d], S [B, H, d_v, d], n [B, H, d]
are float32 CUDA tensors updated in place; o [B, H, T, d_v] is returned.

    o = scan_fwd_host(q, k, v, u, A, S, n, P=1024, eps_n=1e-6, tau=1e4)

takes the same tensors in (page-locked) host memory and pipelines the copies in
and out with the scan, window by window of the sequence.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

__all__ = ["scan_fwd", "scan_fwd_host", "project_u", "Handle", "VlaError", "library_path", "load_library",
           "STATUS_NONFINITE", "STATUS_TIMEOUT", "SEQUENTIAL", "CHUNKED", "DELTA"]

_PKG = os.path.dirname(os.path.abspath(__file__))
SEQUENTIAL, CHUNKED, DELTA = 0, 1, 2
F32, BF16 = 0, 1
STATUS_NONFINITE, STATUS_TIMEOUT = 1, 2
ERR_NAMES = {0: "VLA_OK", 1: "VLA_ERR_INVALID_ARG", 2: "VLA_ERR_UNSUPPORTED", 3: "VLA_ERR_CUDA",
             4: "VLA_ERR_NOMEM"}


class VlaStatus(ctypes.Structure):
    _fields_ = [("flags", ctypes.c_uint), ("reserved", ctypes.c_uint),
                ("guard_count", ctypes.c_ulonglong), ("renorm_count", ctypes.c_ulonglong),
                ("chunk_fallbacks", ctypes.c_ulonglong)]


class VlaPairStatus(ctypes.Structure):
    _fields_ = [("flags", ctypes.c_uint), ("guard_count", ctypes.c_uint),
                ("renorm_count", ctypes.c_uint), ("chunk_fallbacks", ctypes.c_uint)]


class VlaError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{ERR_NAMES.get(code, code)}: {msg}")
        self.code = code


def library_path() -> str:
    return os.path.join(_PKG, "libvla.so")


_lib = None
_lib_lock = threading.Lock()


def load_library():
    """Load libvla.so and declare its C signatures (raises if it is not built)."""
    global _lib
    with _lib_lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is not built; run `python -m sherman_morrison_inverse_gb300.build`")
        lib = ctypes.CDLL(path)
        vp, ci, cll, cf = ctypes.c_void_p, ctypes.c_int, ctypes.c_longlong, ctypes.c_float
        lib.vla_create.argtypes = [ctypes.POINTER(vp), ci]
        lib.vla_create.restype = ci
        lib.vla_scan_fwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, ci, ci, cll, ci, ci, ci,
                                     ci, cf, cf, cll, ci, ci, ci, vp]
        lib.vla_scan_fwd.restype = ci
        lib.vla_status.argtypes = [vp, vp, ctypes.POINTER(VlaStatus)]
        lib.vla_status.restype = ci
        lib.vla_last_error.argtypes = [vp]
        lib.vla_last_error.restype = ctypes.c_char_p
        lib.vla_destroy.argtypes = [vp]
        lib.vla_destroy.restype = ci
        lib.vla_scan_fwd_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, ci, ci, cll, ci, ci, ci,
                                             ci, cf, cf, cll, ci, vp, vp]
        lib.vla_scan_fwd_noalloc.restype = ci
        lib.vla_scan_fwd_host.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, ci, ci, cll, ci, ci, ci,
                                          ci, cf, cf, cll, ci, ci, ci, cll, vp]
        lib.vla_scan_fwd_host.restype = ci
        lib.vla_selftest_wait.argtypes = [vp, ctypes.c_uint, vp]
        lib.vla_selftest_wait.restype = ci
        lib.vla_ffma_probe.argtypes = [vp, cll, ctypes.POINTER(ctypes.c_double), vp]
        lib.vla_ffma_probe.restype = ci
        lib.vla_host_path_info.argtypes = [vp, ctypes.POINTER(ci), ctypes.POINTER(cll)]
        lib.vla_host_path_info.restype = ci
        lib.vla_project_u.argtypes = [vp, vp, vp, vp, cll, ci, ci, ci, vp]
        lib.vla_project_u.restype = ci
        _lib = lib
        return lib


def _check(lib, h, code):
    if code != 0:
        msg = lib.vla_last_error(h)
        raise VlaError(code, msg.decode() if msg else "")


def _stream_ptr(stream, device) -> int:
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return int(stream.cuda_stream)


class Handle:
    """A library handle bound to one CUDA device (owns the device status block)."""

    def __init__(self, device: int | torch.device | None = None):
        self.lib = load_library()
        if device is None:
            device = torch.cuda.current_device()
        self.device = torch.device("cuda", device if isinstance(device, int) else device.index or 0)
        h = ctypes.c_void_p()
        _check(self.lib, None, self.lib.vla_create(ctypes.byref(h), self.device.index))
        self._h = h

    @property
    def ptr(self):
        return self._h

    def close(self):
        if self._h:
            _check(self.lib, None, self.lib.vla_destroy(self._h))
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:  # noqa: BLE001 - interpreter shutdown
            pass

    def status(self, stream=None) -> dict:
        """Synchronise the stream and return (then reset) the accumulated status."""
        st = VlaStatus()
        _check(self.lib, self._h, self.lib.vla_status(self._h, _stream_ptr(stream, self.device),
                                                      ctypes.byref(st)))
        return dict(flags=st.flags, nonfinite=bool(st.flags & STATUS_NONFINITE),
                    timeout=bool(st.flags & STATUS_TIMEOUT), guard_count=st.guard_count,
                    renorm_count=st.renorm_count, chunk_fallbacks=st.chunk_fallbacks)

    def project_u(self, k_raw, W_u, u=None, stream=None):
        """u[..., i, :] = normalize(W_u[i] k_raw[...]) (README "VLA v3" item 2); k_raw [..., d]
        float32 or bfloat16, W_u [r, d, d] float32; returns u [..., r, d] in k_raw's dtype."""
        d = k_raw.shape[-1]
        if W_u.dim() != 3 or tuple(W_u.shape[1:]) != (d, d) or W_u.dtype != torch.float32:
            raise ValueError("W_u must be float32 [r, d, d]")
        if k_raw.dtype not in (torch.float32, torch.bfloat16):
            raise ValueError("k_raw must be float32 or bfloat16")
        r = W_u.shape[0]
        if u is None:
            u = torch.empty((*k_raw.shape[:-1], r, d), dtype=k_raw.dtype, device=k_raw.device)
        for name, t in (("k_raw", k_raw), ("W_u", W_u), ("u", u)):
            if t.device != self.device:
                raise ValueError(f"{name} is on {t.device}, the handle is on {self.device}")
            if not t.is_contiguous():
                raise ValueError(f"{name} must be contiguous")
        if tuple(u.shape) != (*k_raw.shape[:-1], r, d) or u.dtype != k_raw.dtype:
            raise ValueError("u must be [..., r, d] in k_raw's dtype")
        n = k_raw.numel() // d
        code = self.lib.vla_project_u(self._h, k_raw.data_ptr(), W_u.data_ptr(), u.data_ptr(), n, d, r,
                                      F32 if k_raw.dtype == torch.float32 else BF16,
                                      _stream_ptr(stream, self.device))
        _check(self.lib, self._h, code)
        return u

    @staticmethod
    def _scan_shapes(q, k, v, u, A, S, n, o, device, pin: bool):
        """Check the scan's tensors against the C layouts; allocate o (on `device`) if None."""
        if q.dim() != 4:
            raise ValueError("q must be [B, H, T, d]")
        B, H, T, d = q.shape
        dv = v.shape[-1]
        r = u.shape[3] if u.dim() == 5 else -1
        io = q.dtype
        if io not in (torch.float32, torch.bfloat16):
            raise ValueError("q, k, v, u must be float32 or bfloat16")
        want = {"q": (q, (B, H, T, d), io), "k": (k, (B, H, T, d), io), "v": (v, (B, H, T, dv), io),
                "u": (u, (B, H, T, r, d), io), "A": (A, (B, H, d, d), torch.float32),
                "S": (S, (B, H, dv, d), torch.float32), "n": (n, (B, H, d), torch.float32)}
        if o is None:
            o = torch.empty((B, H, T, dv), dtype=io, device=device, pin_memory=pin)
        want["o"] = (o, (B, H, T, dv), io)
        for name, (t, shape, dt) in want.items():
            if tuple(t.shape) != tuple(shape):
                raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
            if t.dtype != dt:
                raise ValueError(f"{name} has dtype {t.dtype}, expected {dt}")
            if t.device != device:
                raise ValueError(f"{name} is on {t.device}, expected {device}")
            if not t.is_contiguous():
                raise ValueError(f"{name} must be contiguous")
        return (B, H, T, d, dv, r, F32 if io == torch.float32 else BF16), o

    def scan_fwd(self, q, k, v, u, A, S, n, o=None, *, P: int, eps_n: float, tau: float, t0: int = 0,
                 mode: str = "sequential", chunk: int = 0, stream=None):
        """The scan on device tensors (asynchronous on `stream`); A, S, n are updated in place."""
        (B, H, T, d, dv, r, io), o = self._scan_shapes(q, k, v, u, A, S, n, o, self.device, False)
        mode_i = {"sequential": SEQUENTIAL, "chunked": CHUNKED, "delta": DELTA}[mode]
        code = self.lib.vla_scan_fwd(
            self._h, q.data_ptr(), k.data_ptr(), v.data_ptr(), u.data_ptr(),
            A.data_ptr(), S.data_ptr(), n.data_ptr(), o.data_ptr(),
            B, H, T, d, dv, r, int(P), float(eps_n), float(tau), int(t0),
            io, mode_i, int(chunk), _stream_ptr(stream, self.device))
        _check(self.lib, self._h, code)
        return o

    def ffma_probe(self, iters: int, stream=None) -> float:
        """Launch the FP32 throughput probe (packed FMAs on every SM) on `stream`; returns
        the launch's flop count.  Time the launch on the same stream to get FLOP/s."""
        flops = ctypes.c_double(0.0)
        _check(self.lib, self._h, self.lib.vla_ffma_probe(self._h, int(iters), ctypes.byref(flops),
                                                          _stream_ptr(stream, self.device)))
        return float(flops.value)

    def selftest_wait(self, limit_ms: int = 200, stream=None):
        """Launch a wait that nothing completes; it gives up after limit_ms and sets the
        timeout flag in status() (the bounded-wait path of the scan kernels)."""
        _check(self.lib, self._h, self.lib.vla_selftest_wait(self._h, int(limit_ms), _stream_ptr(stream, self.device)))

    def host_path_info(self) -> dict:
        """How the last scan_fwd_host call moved its inputs: {"gathered": 1 (SM gather),
        0 (copy engines) or -1 (no call yet), "seg": window in steps}."""
        g, sg = ctypes.c_int(), ctypes.c_longlong()
        _check(self.lib, self._h, self.lib.vla_host_path_info(self._h, ctypes.byref(g), ctypes.byref(sg)))
        return {"gathered": g.value, "seg": sg.value}

    def scan_fwd_host(self, q, k, v, u, A, S, n, o=None, *, P: int, eps_n: float, tau: float, t0: int = 0,
                      mode: str = "sequential", chunk: int = 0, seg: int = 0, stream=None, wait: bool = True):
        """The scan on CPU tensors (page-locked ones let the copies overlap the scan): windows
        of `seg` steps are copied in, scanned and copied out in a pipeline on the handle's
        device.  A, S, n are updated in place; o (page-locked if allocated here) is returned.
        With wait=False the call returns once the work is enqueued on `stream`, and the
        results are final after that stream is synchronised."""
        cpu = torch.device("cpu")
        (B, H, T, d, dv, r, io), o = self._scan_shapes(q, k, v, u, A, S, n, o, cpu, True)
        mode_i = {"sequential": SEQUENTIAL, "chunked": CHUNKED, "delta": DELTA}[mode]
        st = _stream_ptr(stream, self.device)
        code = self.lib.vla_scan_fwd_host(
            self._h, q.data_ptr(), k.data_ptr(), v.data_ptr(), u.data_ptr(),
            A.data_ptr(), S.data_ptr(), n.data_ptr(), o.data_ptr(),
            B, H, T, d, dv, r, int(P), float(eps_n), float(tau), int(t0),
            io, mode_i, int(chunk), int(seg), st)
        _check(self.lib, self._h, code)
        if wait:
            (stream or torch.cuda.current_stream(self.device)).synchronize()
        return o


_default_handles: dict[int, Handle] = {}


def default_handle(device=None) -> Handle:
    if device is None:
        device = torch.cuda.current_device()
    idx = device if isinstance(device, int) else (device.index or 0)
    h = _default_handles.get(idx)
    if h is None:
        h = _default_handles[idx] = Handle(idx)
    return h


def project_u(k_raw, W_u, u=None, *, stream=None, handle: Handle | None = None):
    """u = normalize(W_u k_raw) on k_raw's device (see Handle.project_u)."""
    h = handle if handle is not None else default_handle(k_raw.device)
    return h.project_u(k_raw, W_u, u, stream=stream)


def scan_fwd(q, k, v, u, A, S, n, o=None, *, P: int, eps_n: float, tau: float, t0: int = 0,
             mode: str = "sequential", chunk: int = 0, stream=None, handle: Handle | None = None):
    """Run the scan on q's device (see the module docstring); returns o."""
    h = handle if handle is not None else default_handle(q.device)
    return h.scan_fwd(q, k, v, u, A, S, n, o, P=P, eps_n=eps_n, tau=tau, t0=t0, mode=mode, chunk=chunk,
                      stream=stream)


def scan_fwd_host(q, k, v, u, A, S, n, o=None, *, P: int, eps_n: float, tau: float, t0: int = 0,
                  mode: str = "sequential", chunk: int = 0, seg: int = 0, stream=None, wait: bool = True,
                  device=None, handle: Handle | None = None):
    """Run the scan on host tensors through the device `device` (see Handle.scan_fwd_host)."""
    h = handle if handle is not None else default_handle(device)
    return h.scan_fwd_host(q, k, v, u, A, S, n, o, P=P, eps_n=eps_n, tau=tau, t0=t0, mode=mode,
                           chunk=chunk, seg=seg, stream=stream, wait=wait)
