"""bench.py's host-side pieces that need no GPU: the work and byte counts behind its
roofline figures, and the reference arm (the float64 oracle timed on the host),
whose JSON line follows the same contract as the GPU arm's."""
from __future__ import annotations

import io
import json
import os
import sys
from contextlib import redirect_stdout

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import workloads  # noqa: E402


def test_flop_counts_per_token_head():
    # r (A u: 2 d^2, u.z: 2 d, rank-1 update: 2 d^2) + A s (2 d^2) + S += v alpha^T and S phi(q) (2 d dv each)
    assert bench.flops_per_token_head(64, 64, 1) == 41_088
    assert bench.flops_per_token_head(64, 64, 4) == 90_624
    assert bench.flops_per_token_head(128, 128, 1) == 4 * 128 * 128 + 2 * 128 + 2 * 128 * 128 + 4 * 128 * 128
    assert bench.flops_per_token_head(64, 64, 1, "delta") == 41_088 + 2 * 64 * 64   # plus S k_hat
    assert bench.flops_per_token_head_short(64, 64, 1) == 24_576                     # 4 d^2 + 2 d dv


@pytest.mark.parametrize("idx,nbytes", [(0, 320), (1, 1280), (2, 640), (3, 2560), (4, 1024)])
def test_streamed_bytes_per_token_head(idx, nbytes):
    # q, k, u and v in, o out: (2 d + r d + 2 dv) times the I/O element size
    assert bench.streamed_bytes_per_token_head(workloads.get(idx)) == nbytes


def test_reference_arm_prints_one_contract_line():
    class Args:
        gpus, steps, warmup = 1, 1, 0
        T_full = workloads.get(0).T

    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.run_reference(Args, workloads.get(0))
    lines = [ln for ln in buf.getvalue().splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == bench.UNIT
    assert d["value"] > 0 and d["higher_is_better"] is True and d["vs_baseline"] is None
    assert d["config"]["workload"] == "tiny_d16_f32"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and "pairs" in cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_traffic_records_are_tied_to_their_kernel_source():
    for (name, mode), (traffic, t_cap, src) in bench.TRAFFIC.items():
        w = workloads.get(name)
        assert w.name == name and mode in bench.KERNEL_SOURCES
        assert len(src) == 16 and int(src, 16) >= 0 and w.T % t_cap == 0
        # a capture's DRAM traffic is close to the bytes the launch must stream at least (the
        # last writes may still be in L2 when the kernel ends)
        if mode == "project_u":   # keys in, r directions out, bf16
            assert bench.proj_tma_fits(w.d, w.r)
            assert traffic >= 0.85 * w.pairs * w.T * (w.d + w.r * w.d) * 2
        else:
            assert mode in bench.MODE_DTYPE
            assert traffic >= 0.9 * w.pairs * w.T * bench.streamed_bytes_per_token_head(w)
        got, how = bench.traffic_record(name, mode, w.T, w.T)
        if src == bench.kernel_source_hash(mode):
            assert got == traffic and "ncu" in how
        else:   # the kernel changed since the capture: no traffic figure
            assert got is None and "changed" in how
    # a truncated run reports none
    assert bench.traffic_record("b4h8_t4096_d64_f32", "sequential", 1024, 4096)[0] is None


def test_kernel_source_hash_follows_the_files(tmp_path, monkeypatch):
    h = bench.kernel_source_hash("chunked")
    assert h == bench.kernel_source_hash("chunked") and len(h) == 16
    for f in bench.KERNEL_SOURCES["chunked"]:
        (tmp_path / f).write_bytes(open(os.path.join(bench.CSRC, f), "rb").read())
    monkeypatch.setattr(bench, "CSRC", str(tmp_path))
    assert bench.kernel_source_hash("chunked") == h
    (tmp_path / "vla_chunk.cuh").write_bytes(b"// changed\n" + (tmp_path / "vla_chunk.cuh").read_bytes())
    assert bench.kernel_source_hash("chunked") != h


def test_tensor_flops_of_the_chunked_kernel():
    base = 2 * 128 * 64 * 64   # one pass of a 128 x 64 x 64 product
    # r = 1, 64 steps a chunk: G1 2 + G2 1 + G3 3 + G4 3 passes, G5 128 x 128 x 64, G6 2 x 128 x 64 x 64
    assert bench.chunk_tensor_flops_per_token_head(1) == 13 * base / 64
    # r = 4, 16 steps a chunk: G6 has K = 16
    assert bench.chunk_tensor_flops_per_token_head(4) == (9 * base + 2 * base + 2 * base / 4) / 16
    # float32 I/O: 3 passes everywhere
    assert bench.chunk_tensor_flops_per_token_head(1, True) == (12 * base + 6 * base + 6 * base) / 64


def test_oracle_leg_shares_the_pairs_over_processes():
    w = workloads.get(0).with_(B=1, H=4, T=64)
    leg = bench.OracleLeg(w, T_full=64, procs=2)
    try:
        value, wall, procs = leg.run(16)
    finally:
        leg.close()
    assert procs == 2 and value > 0 and wall > 0
    assert "2 single-threaded processes" in leg.sample_text(16, wall)


def test_oracle_leg_runs_every_group_in_its_own_process_each_time():
    """Each worker holds one fixed group of pairs and runs it on every call (a pool that may
    hand two calls to one worker would leave a group unrun, or run a worker with no inputs)."""
    w = workloads.get(0).with_(B=1, H=4, T=32)
    leg = bench.OracleLeg(w, T_full=32, procs=4)
    try:
        for steps in (4, 8, 16):
            value, wall, procs = leg.run(steps)
            assert procs == 4 and value > 0
    finally:
        leg.close()
    assert all(not p.is_alive() for p, _ in leg.workers)


def test_no_function_shadows_a_module_function_it_calls():
    """bench.py's GPU legs run only on a GPU; this static check catches a local variable
    that hides a module-level function the same body calls (an error the CPU suite would
    not reach otherwise)."""
    import ast
    tree = ast.parse(open(os.path.join(ROOT, "bench.py")).read())
    module_funcs = {n.name for n in tree.body if isinstance(n, ast.FunctionDef)}
    for fn in ast.walk(tree):
        if not isinstance(fn, ast.FunctionDef):
            continue
        stored = {n.id for n in ast.walk(fn) if isinstance(n, ast.Name) and isinstance(n.ctx, ast.Store)}
        called = {n.func.id for n in ast.walk(fn) if isinstance(n, ast.Call) and isinstance(n.func, ast.Name)}
        clash = stored & called & module_funcs
        assert not clash, (fn.name, clash)


def test_ctas_label_names_the_placement_the_library_takes():
    assert bench.ctas_label("chunked", 64, 0, 128, 152) == "one CTA per (b,h) pair"   # 256 > 152 SMs
    assert "A side and the S side" in bench.ctas_label("chunked", 64, 0, 32, 152)
    assert bench.ctas_per_pair("chunked", 64, 0, 76, 152) == 2 and bench.ctas_per_pair("chunked", 64, 0, 77, 152) == 1
    assert bench.ctas_label("sequential", 64, 0, 32, 152) == "one CTA per (b,h) pair"
    assert "two-CTA cluster" in bench.ctas_label("sequential", 128, 0, 16, 152)
    assert bench.ctas_label("sequential", 128, 0, 128, 152) == "one CTA per (b,h) pair"   # 256 > 152 SMs
    assert "two-CTA cluster" in bench.ctas_label("delta", 128, 0, 16, 152)
    assert "cluster of 4 CTAs" in bench.ctas_label("sequential", 128, 4, 16, 152)


def test_link_bound_takes_the_tightest_of_the_three_rates():
    # a link shared by both directions: the sum of the bytes over the shared rate binds
    shared = {"h2d_gbs": 200.0, "d2h_gbs": 200.0, "both_gbs": 200.0}
    assert bench.link_bound_ms(2e9, 1e9, shared) == 1e3 * 3e9 / 200e9
    # independent directions: the larger direction binds
    duplex = {"h2d_gbs": 200.0, "d2h_gbs": 100.0, "both_gbs": 300.0}
    assert bench.link_bound_ms(2e9, 1e9, duplex) == 1e3 * max(3e9 / 300e9, 2e9 / 200e9, 1e9 / 100e9)
