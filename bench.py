#!/usr/bin/env python3
"""Benchmark of the VLA forward scan on GB300.

One "step" is one pass of the whole scan (every row of the hot path: the
Sherman-Morrison tracking of A, alpha, the state update, renormalisation and
the readout) over one batch of the workload below.  The headline workload is
d = d_v = 64, T = 16384 with B = 8, H = 16 (bfloat16 q/k/v/u/o, float32 state,
associative-recall-shaped keys); its inputs (1.07 GB) exceed the 129 MB L2, so
no flush is needed between steps.  Successive steps continue the same streams
(t0 advances by T), so every step does identical work on resident inputs.

The scan runs in the chunked tensor-core kernel where it is built (d = d_v =
64, bfloat16 I/O, r = 1 or 4; ``--mode auto``, the default) and in the
sequential CUDA-core kernel otherwise; ``--mode`` picks one explicitly.  Both
pass the same parity tests against the oracle.

Prints one JSON line (rank 0).  ``--impl reference`` times the float64 CPU
oracle instead (the only reference this method has), on a bounded sample.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads  # noqa: E402

METRIC = "VLA scan tokens*heads/s (d=64, T=16384)"
UNIT = "tokens*heads/s"
SM_COUNT_NOMINAL = 152
FP32_LANES_PER_SM = 128
SM_MAX_MHZ_NOMINAL = 2070.0


def flops_per_token_head(d: int, dv: int, r: int, mode: str = "sequential") -> int:
    """Algorithmic flops of one step of one pair (FMA = 2): r (A u: 2d^2, u.z: 2d,
    rank-1 update: 2d^2) + alpha = A s (2d^2) + S += v alpha^T (2 d dv) + S phi(q) (2 d dv);
    the delta-rule variant adds S k_hat (2 d dv)."""
    return r * (4 * d * d + 2 * d) + 2 * d * d + (6 if mode == "delta" else 4) * d * dv


def flops_per_token_head_short(d: int, dv: int, r: int) -> int:
    """The shorter count 4 r d^2 + 2 d d_v (omits alpha = A s and the readout)."""
    return 4 * r * d * d + 2 * d * dv


def streamed_bytes_per_token_head(w) -> int:
    es = 4 if w.io == "f32" else 2
    return (2 * w.d + w.r * w.d + 2 * w.dv) * es


# DRAM traffic per launch (dram__bytes_read.sum + dram__bytes_write.sum) of the
# timed kernel, from the ncu captures summarised under profiles/ (scaled from the
# captured T to the full launch; traffic grows with T).  None when the kernel has
# changed since its capture.
TRAFFIC = {
    ("b16h16_t8192_d64_bf16_r4", "chunked"):
        (274.16e6 * 8, "bytes per launch: profiles/chunk_scan_kernel_r4_b16h16_d64_bf16.md, 274.2 MB at "
                       "T = 1024 scaled by 8 to T = 8192"),
    ("b4h8_t4096_d64_f32", "sequential"):
        (154.31e6, "bytes per launch: profiles/seq_block_kernel_b4h8_d64_f32.md (the full T = 4096)"),
    ("b2h8_t65536_d128_f32", "sequential"):
        (156.39e6 * 16, "bytes per launch: profiles/seq_block_kernel_cluster_b2h8_d128_f32.md, 156.4 MB at "
                        "T = 4096 scaled by 16 to T = 65536"),
    ("b8h16_t16384_d64_bf16_recall", "sequential"):
        (325.31e6 * 4, "bytes per launch: profiles/seq_block_kernel_b8h16_d64_bf16.md, 325.3 MB at "
                       "T = 4096 scaled by 4 to T = 16384"),
    ("b8h16_t16384_d64_bf16_recall", "delta"):
        (325.57e6 * 4, "bytes per launch: profiles/seq_block_kernel_delta_b8h16_d64_bf16.md, 325.6 MB at "
                       "T = 4096 scaled by 4 to T = 16384"),
    ("b8h16_t16384_d64_bf16_recall", "chunked"):
        (156.69e6 * 8, "bytes per launch: profiles/chunk_scan_kernel_b8h16_d64_bf16.md, 156.7 MB at "
                       "T = 2048 scaled by 8 to T = 16384"),
}

# arithmetic type of each mode's path
MODE_DTYPE = {"sequential": "f32", "chunked": "tf32", "delta": "f32"}


def fp32_peak_tflops(peaks: dict) -> tuple[float, str]:
    """FP32 CUDA-core peak: SMs x 128 FMA lanes x 2 flops x max SM clock."""
    mhz = float(peaks.get("sm_max_mhz", SM_MAX_MHZ_NOMINAL))
    return SM_COUNT_NOMINAL * FP32_LANES_PER_SM * 2 * mhz * 1e6 / 1e12, (
        f"{SM_COUNT_NOMINAL} SMs x {FP32_LANES_PER_SM} FP32 lanes x 2 flop x {mhz:.0f} MHz")


def load_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        d["_source"] = "measured"
        return d
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "sm_max_mhz": SM_MAX_MHZ_NOMINAL, "_source": "fallback"}


class ClockSampler:
    """nvidia-smi sampled during the timed region (clocks and throttle reasons)."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int, period_ms: int = 100):
        self.proc = None
        self.lines: list[str] = []
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(device_index), "-lms", str(period_ms)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0])); smax.append(float(parts[1]))
                power.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[4:8]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None,
                "samples": len(sm), "reasons": sorted(reasons)}


def dist_setup(n_gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
        return rank, local, world, dist
    return 0, 0, 1, None


def max_over_ranks(x: float, dist, dev) -> float:
    if dist is None:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(dist):
    if dist is not None:
        dist.barrier()


def job_value(units_per_rank: int, world: int, ms_max: float) -> float:
    """Whole-job throughput: the units every rank processed over the slowest rank's time."""
    return units_per_rank * world / (ms_max / 1e3)


class OracleLeg:
    """The float64 oracle, as it stands, timed on the host cores on a bounded
    sample of the workload: every pair, the first `steps` steps."""

    def __init__(self, w, T_max: int = 8192):
        import oracle
        self.oracle = oracle
        self.w = w
        self.T_max = min(w.T, T_max)
        self.x = workloads.make_inputs(w, T=self.T_max)

    def run(self, steps: int):
        x, w = self.x, self.w
        c0, t0 = time.process_time(), time.perf_counter()
        self.oracle.scan(x["q"][:, :steps], x["k"][:, :steps], x["v"][:, :steps], x["u"][:, :steps],
                         x["A0"], x["S0"], x["n0"], P=w.P, eps_n=w.eps_n, tau=w.tau)
        wall = time.perf_counter() - t0
        cpu = time.process_time() - c0
        return self.w.pairs * steps / wall, wall, max(1, round(cpu / wall))

    def calibrate(self, budget_s: float) -> int:
        steps = 16
        while True:
            _, wall, _ = self.run(steps)
            if wall * 2 >= budget_s or steps >= self.T_max:
                return min(self.T_max, max(1, int(steps * budget_s / max(wall, 1e-6))))
            steps = min(self.T_max, steps * 4)

    def sample_text(self, steps: int, wall: float) -> str:
        return f"all {self.w.pairs} pairs x first {steps} of {self.w.T} steps of {self.w.name} ({wall:.1f} s wall)"


def host_cpu_info() -> dict:
    """The host the oracle ran on: logical CPUs, CPU model, BLAS threads (when threadpoolctl
    is importable)."""
    info = {"host_cpus": os.cpu_count()}
    model = None
    try:
        with open("/proc/cpuinfo") as f:
            for ln in f:
                key = ln.split(":")[0].strip().lower()
                if key in ("model name", "cpu part", "hardware") and ":" in ln:
                    model = ln.split(":", 1)[1].strip()
                    if key == "model name":
                        break
    except OSError:
        pass
    import platform
    arm_parts = {"0xd4f": "Arm Neoverse V2", "0xd40": "Arm Neoverse V1", "0xd0c": "Arm Neoverse N1"}
    if model in arm_parts:
        model = f"{arm_parts[model]} (cpu part {model})"
    info["cpu_model"] = model or platform.processor() or platform.machine()
    try:
        from threadpoolctl import threadpool_info
        info["blas_threads"] = max((p.get("num_threads", 1) for p in threadpool_info()), default=1)
    except Exception:  # noqa: BLE001 - not installed on every host
        info["blas_threads"] = None
    return info


def oracle_leg(w, budget_s: float = 15.0):
    leg = OracleLeg(w)
    steps = leg.calibrate(budget_s)
    value, wall, cores = leg.run(steps)
    return value, cores, leg.sample_text(steps, wall)


def run_reference(args, w):
    if int(os.environ.get("RANK", "0")) != 0:      # torchrun: rank 0 alone times the oracle
        return
    leg = OracleLeg(w)
    per_step = max(1.0, 150.0 / (args.warmup + args.steps))
    steps = leg.calibrate(per_step)
    for _ in range(args.warmup):
        leg.run(steps)
    vals, walls, cores = [], [], 1
    for _ in range(args.steps):
        v, wall, cores = leg.run(steps)
        vals.append(v)
        walls.append(wall)
    value = len(vals) * w.pairs * steps / sum(walls)
    sample = leg.sample_text(steps, statistics.median(walls)) + " per step"
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * statistics.mean(walls), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": {"workload": w.name, "B": w.B, "H": w.H, "T": w.T, "d": w.d, "dv": w.dv, "r": w.r,
                       "io": w.io},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": sample, **host_cpu_info()},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_project_u(args, w):
    """Time vla_project_u (u = normalize(W_u k_raw)) over the workload's B H T keys."""
    import sherman_morrison_inverse_gb300 as vla
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    x = workloads.make_inputs(w, pairs=[0], T=w.T)
    n = w.B * w.H * w.T
    k = x["k"][0].to(dev).repeat(w.B * w.H, 1).contiguous()          # [B H T, d] keys (pair 0's, repeated)
    W = x["Wu"].to(dev)
    u = torch.empty((n, w.r, w.d), dtype=k.dtype, device=dev)
    h = vla.Handle(0)
    for _ in range(args.warmup):
        h.project_u(k, W, u)
    torch.cuda.synchronize(dev)
    clocks = ClockSampler(0)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        h.project_u(k, W, u)
    e1.record()
    torch.cuda.synchronize(dev)
    clk = clocks.stop()
    ms = e0.elapsed_time(e1) / args.steps
    peaks = load_peaks()
    flops = 2 * w.r * w.d * w.d * n
    nbytes = n * (w.d + w.r * w.d) * k.element_size()   # keys in, directions out (W: a few KB)
    # the tensor-core form (tcgen05 kind::tf32, W as hi + lo) serves every shape but d = 128 with
    # float32 keys; it is bound by HBM: a few flops per byte, far below the tensor ridge
    tc = not (w.d == 128 and w.io == "f32")
    gbs = nbytes / (ms / 1e3) / 1e9
    line = {"metric": "u projection tokens/s (normalize(W_u k_raw))", "value": n / (ms / 1e3), "unit": "tokens/s",
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "tf32" if tc else "f32", "data": "synthetic",
            "config": {"workload": w.name, "tokens": n, "d": w.d, "r": w.r, "io": w.io, "op": "project_u",
                       "l2": "keys and directions 2 x %.0f MB > 129 MB L2 (no flush)" % (n * w.d * k.element_size() / 1e6)},
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": float(peaks["hbm_gbs"]), "unit": "GB/s",
                         "frac": gbs / float(peaks["hbm_gbs"]), "traffic": None,
                         "peak_how": "%s HBM copy bandwidth" % peaks["_source"],
                         "algorithmic_bytes": nbytes, "tflops": flops / (ms / 1e3) / 1e12,
                         "form": "tcgen05 kind::tf32, 2 passes (W hi + lo)" if tc else "CUDA cores, float32"},
            "clocks": clk, "gpu_launches": args.steps}
    print(json.dumps(line), flush=True)
    h.close()


def drift_trace(h, w, x, g, kw, seg, dev):
    """max|A_t M_t - I| and the largest ||S_t||_F after every `seg` steps of one pass over
    the sequence, with t0 carried from call to call.  M_t = A_0^{-1} + sum_{t' <= t} u u^T is
    accumulated on the host in float64.  Nudges (A += eps_n I every P steps) make A differ
    from M^{-1} by about eps_n ||M|| per nudge: with nudges on this is a report, not a gate."""
    B, H, T, d = w.B, w.H, w.T, w.d
    N = B * H
    A = x["A0"].reshape(B, H, d, d).to(dev).contiguous()
    S = x["S0"].reshape(B, H, w.dv, d).to(dev).contiguous()
    n = x["n0"].reshape(B, H, d).to(dev).contiguous()
    M = np.linalg.inv(x["A0"].double().numpy())
    eye = np.eye(d)
    rows = []
    for a0 in range(0, T, seg):
        b0 = min(T, a0 + seg)
        sl = lambda t: t[:, :, a0:b0].contiguous()
        h.scan_fwd(sl(g["q"]), sl(g["k"]), sl(g["v"]), sl(g["u"]), A, S, n, t0=a0, **kw)
        Ud = x["u"][:, a0:b0].double().numpy().reshape(N, -1, d)   # the r directions of each step, in order
        M += np.matmul(Ud.transpose(0, 2, 1), Ud)
        Ah = A.reshape(N, d, d).double().cpu().numpy()
        drift = float(np.abs(np.matmul(Ah, M) - eye).max())
        sfn = float(torch.linalg.norm(S.reshape(N, -1).double(), dim=1).max().item())
        rows.append({"t": b0, "max_abs_AM_minus_I": drift, "max_S_F": sfn})
    return rows


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=40)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="2", help="index or name of the workload")
    ap.add_argument("--mode", choices=["auto", "sequential", "chunked", "delta"], default="auto",
                    help="auto: the chunked tensor-core kernel where it is built (d = d_v = 64, bf16 I/O, "
                         "r = 1 or 4), else the sequential one; delta: the delta-rule variant")
    ap.add_argument("--chunk", type=int, default=0)
    ap.add_argument("--op", choices=["scan", "project_u"], default="scan",
                    help="project_u: time the direction projection u = normalize(W_u k_raw) instead")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--trace", type=int, default=0,
                    help="untimed, after the timed legs: run the sequence again in calls of this many steps "
                         "(t0 carried) and report max|A M - I| (M = A_0^-1 + sum u u^T in float64 on the host) "
                         "and the largest ||S||_F after each call")
    ap.add_argument("--trace-P", type=int, default=None,
                    help="nudge period for the trace run (default: the workload's; 0 turns nudges off, so "
                         "that A tracks M^-1 exactly in exact arithmetic)")
    ap.add_argument("--e2e-steps", type=int, default=None)
    ap.add_argument("--seg", type=int, default=0,
                    help="steps per window of the host-buffer (e2e) path; 0 = the library's choice")
    ap.add_argument("--T", type=int, default=None,
                    help="truncate the sequence (profiling a smaller case; not a bench number)")
    args = ap.parse_args()
    w = workloads.get(int(args.workload) if args.workload.isdigit() else args.workload)
    T_full = w.T
    if args.T is not None:
        w = w.with_(T=args.T)

    if args.mode == "auto":
        args.mode = "chunked" if (w.d == 64 and w.dv == 64 and w.io == "bf16" and w.r in (1, 4)) else "sequential"
    if args.impl == "reference":
        run_reference(args, w)
        return
    if args.op == "project_u":
        run_project_u(args, w)
        return

    import sherman_morrison_inverse_gb300 as vla

    rank, local, world, dist = dist_setup(args.gpus)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    h = vla.Handle(local)

    x = workloads.make_inputs(w.with_(T=T_full), T=w.T)
    B, H, T = w.B, w.H, w.T
    g = {k: x[k].reshape(B, H, *x[k].shape[1:]).to(dev).contiguous() for k in ("q", "k", "v", "u")}
    A = x["A0"].reshape(B, H, w.d, w.d).to(dev).contiguous()
    S = x["S0"].reshape(B, H, w.dv, w.d).to(dev).contiguous()
    n = x["n0"].reshape(B, H, w.d).to(dev).contiguous()
    o = torch.empty((B, H, T, w.dv), dtype=g["q"].dtype, device=dev)
    kw = dict(P=w.P, eps_n=w.eps_n, tau=w.tau, mode=args.mode, chunk=args.chunk)

    t0 = 0
    for _ in range(args.warmup):
        h.scan_fwd(g["q"], g["k"], g["v"], g["u"], A, S, n, o, t0=t0, **kw)
        t0 += T
    torch.cuda.synchronize(dev)
    st_warm = h.status()

    # ---- device-resident timing (inputs already in HBM)
    barrier(dist)
    torch.cuda.synchronize(dev)
    clocks = ClockSampler(local)
    time.sleep(0.3)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(args.steps):
        h.scan_fwd(g["q"], g["k"], g["v"], g["u"], A, S, n, o, t0=t0, **kw)
        t0 += T
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    clk = clocks.stop()
    barrier(dist)
    ms = ev0.elapsed_time(ev1)
    ms_max = max_over_ranks(ms, dist, dev)
    st = h.status()
    value = job_value(B * H * T * args.steps, world, ms_max)
    ms_per_step = ms_max / args.steps

    # ---- end to end through the host-buffer entry point: every step copies q, k, v, u and
    # the state in from page-locked host memory and o and the state back, pipelined with
    # the scan window by window inside the library
    e2e_steps = args.e2e_steps or max(3, args.steps // 4)
    host = {k: x[k].reshape(B, H, *x[k].shape[1:]).contiguous().pin_memory() for k in ("q", "k", "v", "u")}
    host_state = {"A": x["A0"].reshape(B, H, w.d, w.d).contiguous().pin_memory(),
                  "S": x["S0"].reshape(B, H, w.dv, w.d).contiguous().pin_memory(),
                  "n": x["n0"].reshape(B, H, w.d).contiguous().pin_memory()}
    host_o = torch.empty_like(o, device="cpu").pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in list(host.values()) + list(host_state.values()))
    d2h = host_o.numel() * host_o.element_size() + sum(t.numel() * t.element_size()
                                                       for t in host_state.values())
    hkw = dict(kw, seg=args.seg, stream=stream, wait=False)
    h.scan_fwd_host(host["q"], host["k"], host["v"], host["u"], host_state["A"], host_state["S"],
                    host_state["n"], host_o, t0=0, **hkw)   # warm-up: allocates the workspace
    torch.cuda.synchronize(dev)
    h.status()
    barrier(dist)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    te = T
    for _ in range(e2e_steps):
        h.scan_fwd_host(host["q"], host["k"], host["v"], host["u"], host_state["A"], host_state["S"],
                        host_state["n"], host_o, t0=te, **hkw)
        te += T
    e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(dist)
    host_info = h.host_path_info()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), dist, dev)
    e2e_value = job_value(B * H * T * e2e_steps, world, e2e_ms)
    st_e2e = h.status()

    # ---- roofline of the (only) kernel: FP32 CUDA-core arithmetic binds
    peaks = load_peaks()
    peak_tf, peak_how = fp32_peak_tflops(peaks)
    F = flops_per_token_head(w.d, w.dv, w.r, args.mode)
    achieved_tf = B * H * T * F / (ms_per_step / 1e3) / 1e12
    bytes_step = B * H * T * streamed_bytes_per_token_head(w)
    traffic = TRAFFIC.get((w.name, args.mode), (None, "no capture for this workload"))
    if w.T != T_full:
        traffic = (None, "not the full-length workload")

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": MODE_DTYPE[args.mode], "data": "synthetic",
        "config": {"workload": w.name, "B": B, "H": H, "T": T, "d": w.d, "dv": w.dv, "r": w.r,
                   "io": w.io, "state": "f32", "mode": args.mode,
                   "precision": ("tcgen05 kind::tf32, 3xTF32 on the products that carry A; fp32 state"
                                 if args.mode == "chunked" else "fp32 CUDA-core arithmetic"),
                   "rule": "delta (gist.science summary §2.3)" if args.mode == "delta" else "additive",
                   "l2": f"inputs {bytes_step / 1e9:.2f} GB per step > 129 MB L2 (no flush)",
                   "parallelism": f"replicas x{world}, one CTA per (b,h) pair"},
        "roofline": {"bound": "alu", "achieved": achieved_tf, "peak": peak_tf, "unit": "TFLOP/s",
                     "frac": achieved_tf / peak_tf, "traffic": traffic[0], "traffic_source": traffic[1],
                     "peak_how": peak_how + " (derived; FP32 is not in the measured-peaks file)",
                     "flops_per_token_head": F,
                     "frac_short_count": (B * H * T * flops_per_token_head_short(w.d, w.dv, w.r)
                                          / (ms_per_step / 1e3) / 1e12) / peak_tf,
                     "hbm_gbs": bytes_step / (ms_per_step / 1e3) / 1e9,
                     "hbm_frac": bytes_step / (ms_per_step / 1e3) / 1e9 / float(peaks["hbm_gbs"]),
                     "sm_ceiling": min(1.0, B * H / SM_COUNT_NOMINAL)},
        "clocks": clk,
        "gpu_launches": args.steps,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "steps": e2e_steps, "ms_per_step": e2e_ms / e2e_steps,
                "api": "scan_fwd_host: windows of the sequence copied in, scanned and copied out "
                       "in a pipeline", "seg": host_info["seg"],
                "copy_in": "SM gather from mapped page-locked memory" if host_info["gathered"] == 1
                           else "copy engines (cudaMemcpy2DAsync)"},
        "status": {"warmup": st_warm, "timed": st, "e2e": st_e2e},
    }
    if args.trace > 0 and rank == 0:
        tkw = dict(kw, P=w.P if args.trace_P is None else args.trace_P)
        rows = drift_trace(h, w, x, g, tkw, args.trace, dev)
        line["trace"] = {"seg": args.trace, "P": tkw["P"], "tau": w.tau, "rows": rows, "status": h.status(),
                         "note": "untimed; M = A_0^-1 + sum u u^T in float64 on the host"}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, cores, sample = oracle_leg(w)
        line["cpu_baseline"] = {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample,
                                **host_cpu_info()}
    if rank == 0:
        print(json.dumps(line), flush=True)
    h.close()
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
