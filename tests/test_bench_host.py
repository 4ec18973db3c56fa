"""Host-side logic of bench.py that needs no GPU: the cross-rank max used for timing (run as a
world-size-2 gloo job on CPU), per-rank seeds, algorithmic byte counts, the kernel-source hash
and the reference arm's JSON line."""
import json
import os
import subprocess
import sys

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        vals = [1.0 + rank, 10.0 - rank, 5.0 * rank]
        q.put((rank, bench.max_over_ranks(vals, torch.device("cpu")), bench.rank_seed_shift(rank)))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_world_2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + (os.getpid() % 2000)
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res[0][1] == res[1][1] == [2.0, 10.0, 5.0]
    assert res[0][2] != res[1][2]  # independent batches per rank


def test_max_over_ranks_single_process_is_identity():
    assert bench.max_over_ranks([3.0, 1.5], torch.device("cpu")) == [3.0, 1.5]


def test_algorithmic_bytes_llada_r05():
    # W once + gathered rows once + bf16 logits once + int32 indices
    assert bench.algorithmic_bytes(2048, 126464, 4096, 2) == (
        2 * 126464 * 4096 + 2 * 2048 * 4096 + 2 * 2048 * 126464 + 4 * 2048)


def test_kernel_source_hash_is_stable():
    assert bench.kernel_source_hash() == bench.kernel_source_hash()
    assert len(bench.kernel_source_hash()) == 16


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "tiny", "--steps", "2", "--warmup", "1", "--ref-step-s", "0.2"],
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    j = json.loads(lines[0])
    assert j["impl"] == "reference" and j["unit"] == "TFLOP/s" and j["higher_is_better"]
    assert j["cpu_baseline"]["kind"] == "oracle" and j["cpu_baseline"]["cores"] >= 1
    assert j["e2e"]["h2d_bytes_per_step"] == 0 and j["e2e"]["value"] == j["value"]


def test_reference_arm_non_zero_rank_exits_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "tiny", "--steps", "1", "--warmup", "1"],
                       capture_output=True, text=True, timeout=120, env=env)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_clock_sampler_keeps_only_the_timed_region():
    clk = bench.ClockSampler(0)
    # (arrival time, "sm MHz, max MHz, power, hw_slowdown, hw_thermal, sw_thermal, sw_power_cap")
    clk.lines = [
        (0.9, "2070, 2070, 300.0, Not Active, Not Active, Not Active, Not Active"),  # before
        (1.1, "1600, 2070, 1360.0, Not Active, Not Active, Not Active, Active"),
        (1.2, "1500, 2070, 1370.0, Not Active, Not Active, Not Active, Active"),
        (1.3, "1550, 2070, 1365.0, Not Active, Not Active, Not Active, Active"),
        (1.6, "2070, 2070, 250.0, Active, Not Active, Not Active, Not Active"),       # after
        (1.25, "garbled line"),
    ]
    clk.t0, clk.t1 = 1.0, 1.5
    s = clk.summary()
    assert s["samples"] == 3 and s["sm_mhz"] == 1550 and s["sm_max_mhz"] == 2070
    assert s["reasons"] == ["sw_power_cap"]  # hw_slowdown was seen only outside the region
    clk.t0, clk.t1 = 5.0, 6.0
    s = clk.summary()
    assert s["samples"] == 0 and s["sm_mhz"] is None and "note" in s


def test_launch_rows_follow_the_chunking_rule():
    assert bench.launch_rows(0, 4096) == []
    assert bench.launch_rows(100, 0) == [100]
    assert bench.launch_rows(100, 100) == [100]
    assert bench.launch_rows(172201, 8192) == [8192] * 21 + [169]


def test_roofline_uses_the_burst_peak_and_reports_the_sustained_fraction():
    peaks = (6784.8, 1898.6, 1685.2, "measured")
    flops, nbytes = 2 * 2048 * 126464 * 4096, bench.algorithmic_bytes(2048, 126464, 4096, 2)
    r = bench.roofline_entry(flops, nbytes, 1.2e-3, peaks, "logits")
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s" and r["peak"] == 1898.6
    assert abs(r["achieved"] - flops / 1.2e-3 / 1e12) < 1e-9
    assert abs(r["frac"] - r["achieved"] / 1898.6) < 1e-12
    assert abs(r["frac_of_sustained_peak"] - r["achieved"] / 1685.2) < 1e-12
    r8 = bench.roofline_entry(flops, nbytes, 1.2e-3, peaks, "fp8")
    assert r8["peak"] == 2 * 1898.6 and "E4M3" in r8["peak_source"]
    # far below the ridge the HBM roof binds and the fraction is of bandwidth
    small = bench.roofline_entry(2 * 16 * 126464 * 4096, bench.algorithmic_bytes(16, 126464, 4096, 2),
                                 1.8e-4, peaks, "logits")
    assert small["bound"] == "hbm" and small["unit"] == "GB/s" and small["peak"] == 6784.8


def test_small_m_workloads_have_exactly_m_rows():
    for m in (1, 16, 320, 410, 4096):
        (w,) = bench.workload_set(f"llada8b_M{m}")
        assert w.mask().M == m and (w.d, w.V, w.L) == (4096, 126464, 4096)
