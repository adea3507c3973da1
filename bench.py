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
FP32_LANES_PER_SM = 128
SM_MAX_MHZ_NOMINAL = 2070.0
CSRC = os.path.join(ROOT, "sherman_morrison_inverse_gb300", "csrc")


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


def chunk_tensor_flops_per_token_head(r: int, f32: bool = False) -> float:
    """Tensor-core flops the chunked kernel executes per step of a pair (d = d_v = 64, 64
    directions a chunk, C = 64 / r steps): the 128 x 64 x 64 products G1 (2 passes), G2 (1),
    G3 (3), G4 (3), G5 (128 x 128 x 64) and G6 (2 x 128 x 64 x C), each pass counted.  With
    float32 I/O every product takes 3 passes (3xTF32)."""
    C = 64 // r
    base = 2.0 * 128 * 64 * 64
    if f32:
        per_chunk = (3 + 3 + 3 + 3) * base + 3 * 2.0 * 128 * 128 * 64 + 3 * 2 * (2.0 * 128 * 64 * C)
    else:
        per_chunk = (2 + 1 + 3 + 3) * base + 2.0 * 128 * 128 * 64 + 2 * (2.0 * 128 * 64 * C)
    return per_chunk / C


# Source files of each timed kernel; a traffic record holds the hash of these files at the
# time of its ncu capture and is reported only while the hash still matches.
KERNEL_SOURCES = {
    "sequential": ["vla_seqk.cuh", "vla_internal.cuh", "vla_seqk_d16.cu", "vla_seqk_d64.cu", "vla_seqk_d128.cu"],
    "delta": ["vla_seqk.cuh", "vla_internal.cuh", "vla_seqk_delta_d16.cu", "vla_seqk_delta_d64.cu",
              "vla_seqk_delta_d128.cu", "vla_delta.cu"],
    "chunked": ["vla_chunk.cuh", "vla_tc.cuh", "vla_internal.cuh", "vla_chunked.cu"],
    "project_u": ["vla_proj_tma.cu", "vla_tc.cuh", "vla_internal.cuh"],
}


def kernel_source_hash(mode: str) -> str:
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[mode]:
        with open(os.path.join(CSRC, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


# DRAM traffic per launch (dram__bytes_read.sum + dram__bytes_write.sum) of the timed kernel
# from ncu captures: (bytes per full-length launch, captured T, kernel source hash).  Captures
# at a truncated T are scaled by the units processed (traffic grows with T).
TRAFFIC = {
    ("b4h8_t4096_d64_f32", "sequential"): (154.42e6, 4096, "09b46c6b7e90fb86"),
    ("b2h8_t65536_d128_f32", "sequential"): (155.86e6 * 16, 4096, "09b46c6b7e90fb86"),
    ("b8h16_t16384_d64_bf16_recall", "sequential"): (324.69e6 * 4, 4096, "09b46c6b7e90fb86"),
    ("b8h16_t16384_d64_bf16_recall", "delta"): (324.66e6 * 4, 4096, "a1a90440234bd2e5"),
    ("b8h16_t16384_d64_bf16_recall", "chunked"): (156.03e6 * 8, 2048, "d7624e73d18c2b23"),
    ("b16h16_t8192_d64_bf16_r4", "chunked"): (274.33e6 * 8, 1024, "d7624e73d18c2b23"),
    ("b4h8_t4096_d64_f32", "chunked"): (153.79e6, 4096, "d7624e73d18c2b23"),
    # the u projection's TMA form (whole workload captured)
    ("b8h16_t16384_d64_bf16_recall", "project_u"): (482.59e6, 16384, "bad2b2f554b35e74"),
    ("b16h16_t8192_d64_bf16_r4", "project_u"): (1280.58e6, 8192, "bad2b2f554b35e74"),
}


def traffic_record(workload: str, mode: str, T: int, T_full: int):
    """(bytes per launch or None, how it was obtained)."""
    rec = TRAFFIC.get((workload, mode))
    if rec is None:
        return None, "no ncu capture of this kernel on this workload"
    if T != T_full:
        return None, "not the full-length workload"
    nbytes, t_cap, src = rec
    if src != kernel_source_hash(mode):
        return None, "the kernel source changed since its last ncu capture (source hash %s, now %s)" % (
            src, kernel_source_hash(mode))
    how = "ncu dram__bytes_read.sum + dram__bytes_write.sum"
    if t_cap != T_full:
        how += f", captured at T = {t_cap} and scaled by {T_full // t_cap} to T = {T_full}"
    return nbytes, how


# arithmetic type of each mode's path
MODE_DTYPE = {"sequential": "f32", "chunked": "tf32", "delta": "f32"}


def sm_count(dev) -> int:
    return int(torch.cuda.get_device_properties(dev).multi_processor_count)


def fp32_peak_derived(peaks: dict, sms: int) -> tuple[float, str]:
    """FP32 CUDA-core peak from the unit count: SMs x 128 FMA lanes x 2 flops x max SM clock."""
    mhz = float(peaks.get("sm_max_mhz", SM_MAX_MHZ_NOMINAL))
    return sms * FP32_LANES_PER_SM * 2 * mhz * 1e6 / 1e12, (
        f"{sms} SMs x {FP32_LANES_PER_SM} FP32 lanes x 2 flop x {mhz:.0f} MHz")


def measure_fp32_peak(h, dev, stream, target_ms: float = 10.0, launches: int = 3) -> dict:
    """The FP32 CUDA-core throughput of this GPU, measured: the library's packed-FMA probe
    (every SM busy) timed with CUDA events on the launching stream, clocks sampled beside it."""
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    iters = 1 << 12
    for _ in range(8):   # calibrate to about target_ms a launch
        e0.record(stream)
        h.ffma_probe(iters, stream=stream)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        ms = e0.elapsed_time(e1)
        if ms >= 0.5 * target_ms:
            break
        iters = min(1 << 30, int(iters * max(2.0, target_ms / max(ms, 1e-3))))
    clocks = ClockSampler(dev.index)
    time.sleep(0.2)
    best = 0.0
    for _ in range(launches):
        e0.record(stream)
        flops = h.ffma_probe(iters, stream=stream)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        best = max(best, flops / (e0.elapsed_time(e1) / 1e3) / 1e12)
    clk = clocks.stop()
    st = h.status()
    return {"tflops": best, "iters": iters, "launches": launches, "clocks": clk, "status_flags": st["flags"]}


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


def _oracle_worker(conn, job):
    """Worker process: generate the inputs of its pairs (the seeded generators are
    subset-stable, so each pair's inputs are the same as in the full workload), then, for
    every `steps` received, run the oracle over its pairs and the first `steps` steps and
    send back its wall time; None ends it."""
    import oracle
    w, T_max, pairs = job
    x = workloads.make_inputs(w, pairs=list(pairs), T=T_max)
    conn.send(len(pairs))
    while True:
        steps = conn.recv()
        if steps is None:
            break
        t0 = time.perf_counter()
        oracle.scan(x["q"][:, :steps], x["k"][:, :steps], x["v"][:, :steps], x["u"][:, :steps],
                    x["A0"], x["S0"], x["n0"], P=w.P, eps_n=w.eps_n, tau=w.tau)
        conn.send(time.perf_counter() - t0)
    conn.close()


class OracleLeg:
    """The float64 oracle, as it stands, timed on the host cores on a bounded sample of the
    workload: every pair, the first `steps` steps.  The pairs are independent, so they are
    shared out over one single-threaded process per host CPU (spawned, so no process is
    forked from one that has used the GPU), each holding one fixed group of pairs; the wall
    time of all of them together is timed."""

    def __init__(self, w, T_full: int, T_max: int = 8192, procs: int | None = None):
        import multiprocessing as mp
        for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
            os.environ.setdefault(var, "1")   # one BLAS thread per worker process
        self.w = w
        self.T_max = min(w.T, T_max)
        self.procs = max(1, min(procs or (os.cpu_count() or 1), w.pairs))
        groups = np.array_split(np.arange(w.pairs), self.procs)
        ctx = mp.get_context("spawn")
        self.workers = []
        for g in groups:
            parent, child = ctx.Pipe()
            p = ctx.Process(target=_oracle_worker, args=(child, (w.with_(T=T_full), self.T_max,
                                                                 tuple(int(i) for i in g))), daemon=True)
            p.start()
            child.close()
            self.workers.append((p, parent))
        done = sum(conn.recv() for _, conn in self.workers)   # every worker holds its inputs
        assert done == w.pairs, (done, w.pairs)

    def run(self, steps: int):
        t0 = time.perf_counter()
        for _, conn in self.workers:
            conn.send(steps)
        for _, conn in self.workers:
            conn.recv()
        wall = time.perf_counter() - t0
        return self.w.pairs * steps / wall, wall, self.procs

    def calibrate(self, budget_s: float) -> int:
        steps = 16
        while True:
            _, wall, _ = self.run(steps)
            if wall * 2 >= budget_s or steps >= self.T_max:
                return min(self.T_max, max(1, int(steps * budget_s / max(wall, 1e-6))))
            steps = min(self.T_max, steps * 4)

    def sample_text(self, steps: int, wall: float) -> str:
        return (f"all {self.w.pairs} pairs x first {steps} of {self.w.T} steps of {self.w.name}, "
                f"pairs shared out over {self.procs} single-threaded processes ({wall:.1f} s wall)")

    def close(self):
        for p, conn in self.workers:
            try:
                conn.send(None)
                conn.close()
            except OSError:
                pass
        for p, _ in self.workers:
            p.join(timeout=30)
            if p.is_alive():
                p.terminate()


def host_cpu_info() -> dict:
    """The host the oracle ran on: logical CPUs, CPU model, BLAS threads per process."""
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
    info["blas_threads_per_process"] = int(os.environ.get("OMP_NUM_THREADS", "1"))
    return info


def oracle_leg(w, T_full: int, budget_s: float = 15.0):
    leg = OracleLeg(w, T_full)
    try:
        steps = leg.calibrate(budget_s)
        value, wall, cores = leg.run(steps)
    finally:
        leg.close()
    return value, cores, leg.sample_text(steps, wall)


def sampled_pair_errors(h, w, T_full: int, modes, dev, pairs=(0, 1)) -> dict:
    """Errors of each mode against the oracle on a sample of pairs over the whole sequence,
    from the workload's initial state (part of the CPU-baseline leg: the oracle runs here)."""
    import oracle
    x = workloads.make_inputs(w.with_(T=T_full), pairs=list(pairs), T=w.T)
    N = len(pairs)
    ref = oracle.scan(x["q"], x["k"], x["v"], x["u"], x["A0"], x["S0"], x["n0"], P=w.P, eps_n=w.eps_n, tau=w.tau)
    out = {"pairs": list(pairs), "T": w.T, "metric": "oracle.errors (state: per pair max|X - X_ref| / max|X_ref|; "
                                                     "o: per row)"}
    for mode in modes:
        g = {k: x[k].reshape(1, N, *x[k].shape[1:]).to(dev).contiguous() for k in ("q", "k", "v", "u")}
        A = x["A0"].reshape(1, N, w.d, w.d).to(dev).contiguous()
        S = x["S0"].reshape(1, N, w.dv, w.d).to(dev).contiguous()
        n = x["n0"].reshape(1, N, w.d).to(dev).contiguous()
        o = h.scan_fwd(g["q"], g["k"], g["v"], g["u"], A, S, n, P=w.P, eps_n=w.eps_n, tau=w.tau, mode=mode)
        st = h.status()
        f = lambda t: t.reshape(N, *t.shape[2:]).double().cpu().numpy()
        e = oracle.errors(f(o), f(A), f(S), f(n), *ref)
        out[mode] = {k: float(v) for k, v in e.items()}
        out[mode]["status_flags"] = st["flags"]
    return out


def run_reference(args, w):
    if int(os.environ.get("RANK", "0")) != 0:      # torchrun: rank 0 alone times the oracle
        return
    leg = OracleLeg(w, args.T_full)
    per_step = max(1.0, 150.0 / (args.warmup + args.steps))
    steps = leg.calibrate(per_step)
    for _ in range(args.warmup):
        leg.run(steps)
    vals, walls, cores = [], [], 1
    for _ in range(args.steps):
        v, wall, cores = leg.run(steps)
        vals.append(v)
        walls.append(wall)
    leg.close()
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


def measure_host_link(dev, nbytes: int = 256 << 20, reps: int = 3) -> dict:
    """The host <-> device link of this GPU: page-locked buffers of `nbytes` copied with
    cudaMemcpyAsync host to device, device to host, and both at once on two streams (best of
    `reps`).  The end-to-end leg's bytes over these rates bound its time from below."""
    h_src = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    h_dst = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    d_src = torch.zeros(nbytes, dtype=torch.uint8, device=dev)
    d_dst = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    s1, s2 = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def run(h2d: bool, d2h: bool) -> float:
        best = float("inf")
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize(dev)
            e0.record(s1)
            s2.wait_event(e0)
            if h2d:
                with torch.cuda.stream(s1):
                    d_dst.copy_(h_src, non_blocking=True)
            if d2h:
                with torch.cuda.stream(s2):
                    h_dst.copy_(d_src, non_blocking=True)
            s1.wait_stream(s2)
            e1.record(s1)
            torch.cuda.synchronize(dev)
            best = min(best, e0.elapsed_time(e1))
        return best

    t_in, t_out, t_both = run(True, False), run(False, True), run(True, True)
    gb = nbytes / 1e9
    return {"h2d_gbs": gb / (t_in / 1e3), "d2h_gbs": gb / (t_out / 1e3), "both_gbs": 2 * gb / (t_both / 1e3),
            "bytes": nbytes, "how": "cudaMemcpyAsync of page-locked buffers: host to device, device to host, "
                                    "and both at once on two streams (best of %d)" % reps}


def link_bound_ms(h2d: int, d2h: int, link: dict) -> float:
    """Least time the link allows for moving h2d bytes in and d2h bytes out."""
    return 1e3 * max((h2d + d2h) / (link["both_gbs"] * 1e9), h2d / (link["h2d_gbs"] * 1e9),
                     d2h / (link["d2h_gbs"] * 1e9))


def ctas_per_pair(mode: str, d: int, chunk: int, pairs: int, sms: int) -> int:
    """CTAs the library gives one (b, h) pair: the sequential mode takes `chunk` (0: the
    default), the sequential and delta defaults are a two-CTA cluster at d = 128 while 2 B H
    CTAs fit on the SMs, the chunked mode a two-CTA cluster at any d while they fit."""
    if mode == "chunked":
        return 2 if 2 * pairs <= sms else 1
    return chunk if (mode == "sequential" and chunk) else (2 if d == 128 and 2 * pairs <= sms else 1)


def ctas_label(mode: str, d: int, chunk: int, pairs: int, sms: int) -> str:
    """How the library places one (b, h) pair (ctas_per_pair)."""
    ctas = ctas_per_pair(mode, d, chunk, pairs, sms)
    if ctas == 1:
        return "one CTA per (b,h) pair"
    if ctas == 2:
        what = "the A side and the S side of each chunk" if mode == "chunked" else "A and S"
        return f"a two-CTA cluster per (b,h) pair ({what} on separate SMs)"
    return f"a cluster of {ctas} CTAs per (b,h) pair (rows of A and columns of S split)"


def proj_tma_fits(d: int, r: int) -> bool:
    """Whether vla_project_u takes its TMA-fed bf16 form: a key ring of at least two stages,
    the staging tiles and W's three bf16 terms for all r ranks fit in one CTA's 227 KB of
    shared memory."""
    bx = min(d, 64)
    slab = 128 * bx * 2
    ks = 2
    nbytes = ks * (d // bx) * slab + 4 * slab + 3 * r * d * d * 2
    return (nbytes + 15) // 16 * 16 + 8 * (2 * ks + 5) + 16 <= 227 * 1024


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
    # A call takes a fraction of a millisecond: the clock sampler needs a few hundred ms to
    # start, so warm-up calls continue until it is up, and the timed region repeats blocks of
    # `steps` calls until it spans at least a second (every call timed, none skipped).
    clocks = ClockSampler(0)
    t_start = time.perf_counter()
    while time.perf_counter() - t_start < 0.5:
        for _ in range(args.steps):
            h.project_u(k, W, u)
        torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    calls = 0
    e0.record()
    t_start = time.perf_counter()
    while calls == 0 or time.perf_counter() - t_start < 1.0:
        for _ in range(args.steps):
            h.project_u(k, W, u)
        calls += args.steps   # the launch queue bounds how far the host runs ahead
    e1.record()
    torch.cuda.synchronize(dev)
    clk = clocks.stop()
    ms = e0.elapsed_time(e1) / calls
    peaks = load_peaks()
    flops = 2 * w.r * w.d * w.d * n
    nbytes = n * (w.d + w.r * w.d) * k.element_size()   # keys in, directions out (W: a few KB)
    # the tensor-core forms serve every shape but d = 128 with float32 keys; the projection is
    # bound by HBM: a few flops per byte, far below the tensor ridge
    tc = not (w.d == 128 and w.io == "f32")
    if w.io == "bf16" and proj_tma_fits(w.d, w.r):
        form, dt = ("tcgen05 kind::f16: bf16 key tiles by TMA tensor loads (swizzled), the r weight sets "
                    "stacked into one N = r d product, outputs by TMA tensor stores; W as three bf16 terms "
                    "(3 passes), fp32 accumulation"), "bf16"
    elif w.io == "bf16":
        form, dt = ("tcgen05 kind::f16: bf16 keys through registers, one rank at a time; W as three bf16 "
                    "terms (3 passes), fp32 accumulation"), "bf16"
    elif tc:
        form, dt = "tcgen05 kind::tf32: keys and W as tf32 hi + lo (3 passes), fp32 accumulation", "tf32"
    else:
        form, dt = "CUDA cores, float32", "f32"
    gbs = nbytes / (ms / 1e3) / 1e9
    if w.io == "bf16" and proj_tma_fits(w.d, w.r):
        traffic, traffic_how = traffic_record(w.name, "project_u", w.T, w.T)
    else:
        traffic, traffic_how = None, "no ncu capture of this form on this workload"
    line = {"metric": "u projection tokens/s (normalize(W_u k_raw))", "value": n / (ms / 1e3), "unit": "tokens/s",
            "n_gpus": 1, "steps": calls, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": dt, "data": "synthetic",
            "config": {"workload": w.name, "tokens": n, "d": w.d, "r": w.r, "io": w.io, "op": "project_u",
                       "l2": "keys and directions 2 x %.0f MB > 129 MB L2 (no flush)" % (n * w.d * k.element_size() / 1e6)},
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": float(peaks["hbm_gbs"]), "unit": "GB/s",
                         "frac": gbs / float(peaks["hbm_gbs"]), "traffic": traffic, "traffic_how": traffic_how,
                         "peak_how": "%s HBM copy bandwidth" % peaks["_source"],
                         "algorithmic_bytes": nbytes, "tflops": flops / (ms / 1e3) / 1e12,
                         "form": form},
            "clocks": clk, "gpu_launches": calls}
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
    ap.add_argument("--tau", type=float, default=None,
                    help="renormalisation threshold in place of the workload's (a labelled companion run, "
                         "e.g. 500 on the long-context workload so that renormalisation fires)")
    args = ap.parse_args()
    w = workloads.get(int(args.workload) if args.workload.isdigit() else args.workload)
    T_full = w.T
    if args.T is not None:
        w = w.with_(T=args.T)
    if args.tau is not None:
        w = w.with_(tau=args.tau)

    args.T_full = T_full
    if args.mode == "auto":
        args.mode = "chunked" if (w.d == 64 and w.dv == 64 and w.r in (1, 4)) else "sequential"
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
    link = measure_host_link(dev)
    link_ms = link_bound_ms(h2d, d2h, link)

    # ---- the other kernel on the same workload: the sequential fp32 CUDA-core scan beside
    # the chunked tensor-core one (timed the same way, after the headline legs)
    other = "sequential" if args.mode == "chunked" else None
    modes = {args.mode: {"ms_per_step": ms_per_step, "value": value}}
    if other is not None:
        okw = dict(kw, mode=other, chunk=0)
        A2, S2, n2 = A.clone(), S.clone(), n.clone()
        for _ in range(2):
            h.scan_fwd(g["q"], g["k"], g["v"], g["u"], A2, S2, n2, o, t0=t0, **okw)
            t0 += T
        o_steps = max(3, args.steps // 4)
        barrier(dist)
        torch.cuda.synchronize(dev)
        f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        f0.record(stream)
        for _ in range(o_steps):
            h.scan_fwd(g["q"], g["k"], g["v"], g["u"], A2, S2, n2, o, t0=t0, **okw)
            t0 += T
        f1.record(stream)
        torch.cuda.synchronize(dev)
        barrier(dist)
        o_ms = max_over_ranks(f0.elapsed_time(f1), dist, dev) / o_steps
        modes[other] = {"ms_per_step": o_ms, "value": job_value(B * H * T, world, o_ms), "steps": o_steps,
                        "status": h.status()}

    # ---- roofline: FP32 CUDA-core arithmetic binds (both kernels quoted on this one scale);
    # the peak is measured here, on this GPU, by the library's packed-FMA probe
    peaks = load_peaks()
    sms = sm_count(dev)
    probe = measure_fp32_peak(h, dev, stream)
    peak_tf = probe["tflops"]
    derived_tf, derived_how = fp32_peak_derived(peaks, sms)
    F = flops_per_token_head(w.d, w.dv, w.r, args.mode)
    achieved_tf = B * H * T * F / (ms_per_step / 1e3) / 1e12
    bytes_step = B * H * T * streamed_bytes_per_token_head(w)
    traffic, traffic_how = traffic_record(w.name, args.mode, T, T_full)
    for m, rec in modes.items():
        rec["frac"] = B * H * T * flops_per_token_head(w.d, w.dv, w.r, m) / (rec["ms_per_step"] / 1e3) / 1e12 / peak_tf
        rec["dtype"] = MODE_DTYPE[m]
    roofline = {"bound": "alu", "achieved": achieved_tf, "peak": peak_tf, "unit": "TFLOP/s",
                "frac": achieved_tf / peak_tf, "traffic": traffic, "traffic_how": traffic_how,
                "peak_how": (f"measured: the library's packed-FMA probe on all {sms} SMs, best of "
                             f"{probe['launches']} launches of {probe['iters']} rounds, median SM clock "
                             f"{probe['clocks'].get('sm_mhz')} MHz; derived {derived_tf:.1f} TFLOP/s = {derived_how}"),
                "peak_derived": derived_tf, "flops_per_token_head": F,
                "frac_short_count": (B * H * T * flops_per_token_head_short(w.d, w.dv, w.r)
                                     / (ms_per_step / 1e3) / 1e12) / peak_tf,
                "hbm_gbs": bytes_step / (ms_per_step / 1e3) / 1e9,
                "hbm_frac": bytes_step / (ms_per_step / 1e3) / 1e9 / float(peaks["hbm_gbs"]),
                "sm_count": sms,
                "sm_ceiling": min(1.0, B * H * ctas_per_pair(args.mode, w.d, args.chunk, B * H, sms) / sms)}
    if args.mode == "chunked":
        tf32_peak = float(peaks["bf16_tflops"]) / 2.0
        tfl = B * H * T * chunk_tensor_flops_per_token_head(w.r, w.io == "f32") / (ms_per_step / 1e3) / 1e12
        roofline["tensor"] = {
            "bound": "tensor", "achieved": tfl, "peak": tf32_peak, "unit": "TFLOP/s", "frac": tfl / tf32_peak,
            "flops_per_token_head": chunk_tensor_flops_per_token_head(w.r, w.io == "f32"),
            "counts": "every tcgen05 pass the kernel executes (a 3xTF32 product counts three times)",
            "peak_how": "%s bf16 burst (%.0f TFLOP/s) x 1/2, the nominal tf32:bf16 dense ratio" % (
                peaks["_source"], float(peaks["bf16_tflops"]))}

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": MODE_DTYPE[args.mode], "data": "synthetic",
        "config": {"workload": w.name, "B": B, "H": H, "T": T, "d": w.d, "dv": w.dv, "r": w.r,
                   "io": w.io, "state": "f32", "mode": args.mode, "P": w.P, "eps_n": w.eps_n, "tau": w.tau,
                   "tau_override": args.tau is not None,
                   "precision": (("tcgen05 kind::tf32, 3xTF32 on every product; fp32 state" if w.io == "f32" else
                                  "tcgen05 kind::tf32, 3xTF32 on the products that carry A; fp32 state")
                                 if args.mode == "chunked" else "fp32 CUDA-core arithmetic"),
                   "rule": "delta (gist.science summary §2.3)" if args.mode == "delta" else "additive",
                   "l2": f"inputs {bytes_step / 1e9:.2f} GB per step > 129 MB L2 (no flush)",
                   "parallelism": f"replicas x{world}, {ctas_label(args.mode, w.d, args.chunk, B * H, sm_count(dev))}"},
        "roofline": roofline,
        "modes": modes,
        "fp32_probe": probe,
        "clocks": clk,
        "gpu_launches": args.steps,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "steps": e2e_steps, "ms_per_step": e2e_ms / e2e_steps,
                "api": "scan_fwd_host: windows of the sequence copied in, scanned and copied out "
                       "in a pipeline", "seg": host_info["seg"],
                "copy_in": "SM gather from mapped page-locked memory" if host_info["gathered"] == 1
                           else "copy engines (cudaMemcpy2DAsync)",
                "link": link, "link_bound_ms": link_ms, "link_frac": link_ms / (e2e_ms / e2e_steps)},
        "status": {"warmup": st_warm, "timed": st, "e2e": st_e2e},
    }
    if args.trace > 0 and rank == 0:
        tkw = dict(kw, P=w.P if args.trace_P is None else args.trace_P)
        rows = drift_trace(h, w, x, g, tkw, args.trace, dev)
        line["trace"] = {"seg": args.trace, "P": tkw["P"], "tau": w.tau, "rows": rows, "status": h.status(),
                         "note": "untimed; M = A_0^-1 + sum u u^T in float64 on the host"}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, cores, sample = oracle_leg(w, T_full)
        line["cpu_baseline"] = {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample,
                                **host_cpu_info()}
        errs = sampled_pair_errors(h, w, T_full, list(modes), dev, pairs=(0, 1) if w.pairs > 1 else (0,))
        for m in modes:
            modes[m]["errors"] = {"pairs": errs["pairs"], "T": errs["T"], **errs[m]}
    if rank == 0:
        print(json.dumps(line), flush=True)
    h.close()
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
