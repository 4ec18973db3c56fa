"""Benchmark of mask-only logits on GB300 (one JSON line on rank 0).

Default workload: the Dream-7B-shaped ragged batch, the largest configuration that runs on one GPU:
8 sequences of L = 32,768 tokens (L_tot = 262,144 hidden rows), d = 3584, V = 152,064, bf16; each
sequence masks a fraction r_b ~ U(0, 1) of its positions (seeded: M = 172,201 rows in all),
addressed through per-sequence CSR offsets, and the logits are computed lazily in chunks of 8192
rows into one reused bf16 output buffer [8192, V] (21 launches per step). One step is one whole
call. Inputs are seeded synthetic data resident in HBM; W alone (1.09 GB) and every chunk's output
(2.49 GB) are larger than the 129 MB L2, so no L2 flush is needed between steps. The call is
captured once into a CUDA graph and the timed steps replay it (``--no-graph``: direct calls).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]
                  [--mode logits|sample|fp8] [--oracle-timing]

Other workloads (--workload): llada8b (the LLaDA-8B LM head, r_m = 0.1, 0.5, 0.9 back to back),
decode (16 x 2048 block decode), long (L = 131,072, four mask ratios), tiny, dream_chunk (one
Dream-shaped chunk launch, for profiling), llada8b_M<m> (the LLaDA-8B head with m masked rows),
or one member by name.

Under torchrun (N > 1) every rank computes its own batch (different seeds) with no collective
on the data path; timing is the max over ranks ("weak" scaling).
``--impl reference`` times the CPU oracle on this host's cores on a bounded sample of the same
workload (the comparison arm; rank 0 only). ``--oracle-timing`` times the oracle on the full
small configurations and extrapolates it on the large ones (one JSON line per configuration).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "masked-logits TFLOP/s (and GB/s) at 1 GB300, % of roofline"
UNIT = "TFLOP/s"
DEFAULT_WORKLOAD = "dream"


def workload_set(name):
    import re

    from masked_token_lm_gb300 import workloads as wl

    m = re.fullmatch(r"llada8b_M(\d+)", name)
    if m:  # the LLaDA-8B LM head with exactly M masked rows (small-M sweeps)
        M = int(m.group(1))
        if not 1 <= M <= 4096:
            raise SystemExit("llada8b_M<m> needs 1 <= m <= 4096")
        return [wl.Workload(name=name, B=1, L=4096, d=4096, V=126464, out_dtype="bf16",
                            chunk_rows=0, mask_kind="flat", r_m=M / 4096, seed=1001)]
    table = {
        "llada8b": wl.LLADA,
        "tiny": [wl.TINY],
        "decode": [wl.DECODE],
        "dream": [wl.DREAM],
        "long": wl.LONG,
        "dream_chunk": [wl.DREAM_CHUNK],
    }
    for w in wl.LONG + wl.LLADA:
        table[w.name] = [w]
    return table[name]


def describe(name, ws):
    w0 = ws[0]
    return {
        "workload": w0.name if len(ws) == 1 else name,
        "members": [w.name for w in ws],
        "B": w0.B, "L": w0.L, "d": w0.d, "V": w0.V,
        "out_dtype": w0.out_dtype,
        "chunk_rows": w0.chunk_rows,
        "mask": w0.mask_kind,
        "l2": "inputs larger than L2 (W alone exceeds the 129 MB L2); no flush",
    }


def algorithmic_bytes(M, V, d, out_elt):
    """W once + the gathered hidden rows once + the output once (+ 4 B per index)."""
    return 2 * V * d + 2 * M * d + out_elt * M * V + 4 * M


def launch_rows(M, chunk_rows):
    """Rows of every gather-GEMM launch of one call (one launch per chunk)."""
    if M == 0:
        return []
    if chunk_rows <= 0 or M <= chunk_rows:
        return [M]
    return [min(chunk_rows, M - b) for b in range(0, M, chunk_rows)]


# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) per gather-GEMM launch, from an ncu
# capture of the kernel sources with the given hash; reported only while the sources still match.
# Entries: source hash -> {workload: bytes per launch (average over the workload's launches)}.
MEASURED_TRAFFIC = {
    # ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum,gpu__time_duration.sum,
    #     lts__t_sector_hit_rate.pct --clock-control none -k regex:gather_gemm -s 9 -c 3
    #     python bench.py --workload llada8b --no-graph --steps 1 --warmup 3 --no-e2e --no-cpu-baseline
    # r_m 0.1 / 0.5 / 0.9 launches: 1.137 / 1.859 / 2.763 GB (mean per launch below)
    "efb394bd87f06b2b": {"llada8b": 1919696469},
    # ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum --clock-control none
    #     -k regex:gather_gemm -s 66 -c 22 python bench.py --workload dream --no-graph --steps 1
    #     --warmup 3 --no-e2e --no-cpu-baseline --no-cublas-context
    # (one pass: the step's 22 launches at full size; mean 5.702 GB read + 2.359 GB written)
    # and the same metrics plus time and L2 hit rate, -s 3 -c 1, on --workload dream_chunk.
    "d725342dfd59cc0b": {"dream": 8061049961, "dream_chunk": 8523418112},
    # the same two captures on the 16-warp build with the register split
    # (mean 5.752 GB read + 2.357 GB written per launch of the step)
    "1d50d76c612cf313": {"dream": 8108922030, "dream_chunk": 8849310464},
    # and on the build whose sampling epilogue takes the split too (logits code unchanged)
    "fb96857a8e98c3e5": {"dream": 7805993356, "dream_chunk": 8155889664},
    # and on the same code with the epilogue's slot wait factored into one helper
    "9ba26e04727a3cfd": {"dream": 8092198633, "dream_chunk": 8610032896},
    # and after an error-message change in capi.cu (the schedule and device code unchanged)
    "1202b6c212626a55": {"dream": 8340067025, "dream_chunk": 8525994240},
    # and after the sampling epilogues' shared fold/merge helpers (the logits code unchanged)
    "bfab402e17a4fe41": {"dream": 9608324201, "dream_chunk": 9778002432},
}


# The device code, and the host code that sets its schedule (raster groups, grid).
KERNEL_SOURCES = ("gather_gemm.cu", "gather_gemm.h", "ptx.cuh", "capi.cu")


def kernel_source_hash():
    """sha256 over the code of the gather-GEMM kernel's sources (the device code whose DRAM
    traffic the capture measured, and the host code that picks its schedule): `//` comments and
    blank lines are left out, so editing a comment keeps the hash."""
    import hashlib
    import re

    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "masked_token_lm_gb300", "csrc")
    for name in KERNEL_SOURCES:
        h.update(name.encode())
        for line in open(os.path.join(csrc, name), encoding="utf-8"):
            code = re.sub(r"//.*$", "", line).rstrip()
            if code:
                h.update(code.encode() + b"\n")
    return h.hexdigest()[:16]


def max_over_ranks(values, device):
    """Element-wise max of a list of floats over all ranks (identity with one process)."""
    import torch

    if not (torch.distributed.is_available() and torch.distributed.is_initialized()):
        return list(values)
    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return t.tolist()


def rank_seed_shift(rank):
    """Each rank draws an independent batch."""
    return 100000 * rank


def sample_bytes(M, V, d, ws_bytes):
    """Fused sampling: W once + gathered rows once + the partials written and read back once +
    token and confidence (the [M, V] logits are never written)."""
    return 2 * V * d + 2 * M * d + 2 * ws_bytes + 8 * M + 4 * M


def load_peaks():
    """(HBM GB/s, bf16 burst TFLOP/s, bf16 sustained TFLOP/s, source)."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        j = json.load(open(p))
        return j["hbm_gbs"], j["bf16_tflops"], j.get("bf16_tflops_sustained"), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


def roofline_entry(tot_flops, tot_bytes, kernel_s, peaks, mode):
    """The roofline object of the JSON line. The step is timed as a loop of kernel launches of
    milliseconds each, so the denominator is the burst figure (a kernel timed by itself); the
    fraction of the sustained figure (cuBLAS looped for seconds under the power cap) is given
    beside it. E4M3 contractions run at twice the bf16 rate (nominal 4.5 vs 2.25 PFLOP/s)."""
    hbm, bf16, bf16_sus, src = peaks
    mult = 2 if mode == "fp8" else 1
    tensor_peak = mult * bf16
    sus_peak = mult * bf16_sus if bf16_sus else None
    achieved = tot_flops / kernel_s / 1e12
    bound = "tensor" if tot_flops / (tensor_peak * 1e12) >= tot_bytes / (hbm * 1e9) else "hbm"
    src_txt = (f"{src} bf16 dense burst ({'MEASURED_PEAKS.json' if src == 'measured' else 'profiling recipe fallback'})"
               + (" x 2 (nominal E4M3/bf16 ratio)" if mult == 2 else ""))
    if bound == "tensor":
        ach, peak, unit = achieved, tensor_peak, "TFLOP/s"
    else:
        ach, peak, unit = tot_bytes / kernel_s / 1e9, hbm, "GB/s"
    return {
        "bound": bound, "achieved": ach, "peak": peak, "unit": unit, "frac": ach / peak,
        "peak_source": src_txt,
        "sustained_peak": sus_peak,
        "frac_of_sustained_peak": (achieved / sus_peak) if (sus_peak and bound == "tensor") else None,
        "achieved_tflops": achieved,
        "achieved_gbs": tot_bytes / kernel_s / 1e9,
        "hbm_peak_gbs": hbm,
        "roof_s": max(tot_flops / (tensor_peak * 1e12), tot_bytes / (hbm * 1e9)),
    }


class ClockSampler:
    """nvidia-smi samples (every 50 ms, each stamped on arrival) of SM clock and throttle
    reasons; the summary keeps the samples taken between region_start() and region_end()."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []  # (monotonic seconds on arrival, csv line)
        self.t0 = self.t1 = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None
        deadline = time.monotonic() + 3.0  # until the sampler is running (first line)
        while self.proc and not self.lines and time.monotonic() < deadline:
            time.sleep(0.01)
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.monotonic(), line.strip()))

    def region_start(self):
        self.t0 = time.monotonic()

    def region_end(self):
        self.t1 = time.monotonic()

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, pw, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ts, ln in self.lines:
            if self.t0 is not None and not (self.t0 <= ts <= (self.t1 or ts)):
                continue  # outside the timed region
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            try:
                pw.append(float(parts[2]))
            except ValueError:
                pass
            for n, v in zip(names, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "note": "no nvidia-smi sample fell inside the timed region"}
        out = {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
               "reasons": sorted(reasons), "samples": len(sm)}
        if pw:
            out["power_w"] = statistics.median(pw)
        return out


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


class CpuOracleTimer:
    """Times the CPU oracle, as it stands, on a bounded sample of a workload: n masked rows of
    the middle member (its rows in order, repeated cyclically when n exceeds them; repeated
    indices are valid input) against all V columns, or against the first cols rows of W when
    even the smallest row sample would take longer than the target. Inputs are generated once.

    A call costs a fixed part (the oracle decodes all of W on every call) plus a part per row;
    calibrate() measures both, which also gives the time of a whole step by linear
    extrapolation in the number of masked rows."""

    def __init__(self, ws):
        import numpy as np
        import torch

        from oracle import mask_only_logits as orc

        self.orc = orc
        self.cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
        self.ws = ws
        self.w = w = ws[len(ws) // 2]
        mask = w.mask()
        self.Hb = w.hidden("cpu").view(torch.int16).numpy().view(np.uint16)
        self.Wb = w.weight("cpu").view(torch.int16).numpy().view(np.uint16)
        so = None if mask.seq_offsets is None else mask.seq_offsets.numpy()
        mo = None if mask.mask_offsets is None else mask.mask_offsets.numpy()
        self.rows = orc.resolve_rows(mask.idx.numpy(), w.L_tot, so, mo).astype(np.int32)
        self.n = None
        self.cols = w.V
        self.fixed = self.per_row = None

    def _secs(self, n):
        import numpy as np

        rows = np.resize(self.rows, n)
        t0 = time.perf_counter()
        self.orc.masked_logits(self.Hb, rows, self.Wb)
        return time.perf_counter() - t0

    def calibrate(self, target_s, lo=256, hi=1024):
        """Rows per call so that one call takes about target_s (measured at lo and hi rows:
        enough rows that the fp64 matmul, not the W stream, sets the per-row cost)."""
        self._secs(lo)  # first call: pays the one-time costs (allocation, page faults)
        t_lo, t_hi = self._secs(lo), self._secs(hi)
        self.per_row = max((t_hi - t_lo) / (hi - lo), 1e-7)
        self.fixed = max(t_lo - lo * self.per_row, 0.0)
        self.n = int(min(8 * len(self.rows), max(lo, (target_s - self.fixed) / self.per_row)))
        # both parts scale with the columns: fewer of them when lo rows exceed the target
        t_lo_est = self.fixed + lo * self.per_row
        self.cols = self.w.V
        if target_s < t_lo_est:
            self.cols = max(1024, int(self.w.V * target_s / t_lo_est) // 8 * 8)
        return self.n

    def sample_rows(self):
        import numpy as np

        return np.resize(self.rows, self.n)

    def run(self):
        rows = self.sample_rows()
        t0 = time.perf_counter()
        self.orc.masked_logits(self.Hb, rows, self.Wb[:self.cols])
        dt = time.perf_counter() - t0
        flops = 2 * self.n * self.cols * self.w.d
        return flops / dt / 1e12, dt

    def step_seconds(self, Ms):
        """Whole-step oracle time, extrapolated linearly in the masked rows: one call per member
        (the fixed W decode each time) plus the per-row cost of every row."""
        return sum(self.fixed + self.per_row * M for M in Ms)

    def sample(self):
        cols = (f"all V={self.w.V} columns" if self.cols == self.w.V
                else f"the first {self.cols} of V={self.w.V} columns")
        return (f"oracle (bf16 decode + fp64 gather and matmul, numpy/OpenBLAS) on {self.n} masked "
                f"rows of {self.w.name} (its {len(self.rows)} rows in order, repeated cyclically), "
                f"{cols}; per call")

    @staticmethod
    def cpu():
        """The host CPU: architecture, model (or ARM part number) and logical cores."""
        import platform

        model = ""
        try:
            with open("/proc/cpuinfo", encoding="utf-8") as f:
                info = f.read()
            for key in ("model name", "CPU part"):
                for line in info.splitlines():
                    if line.startswith(key):
                        model = f"{key} {line.split(':', 1)[1].strip()}"
                        break
                if model:
                    break
        except OSError:
            pass
        return f"{platform.machine()}, {model or 'model unknown'}, {os.cpu_count()} logical cores"


def oracle_probe(workload, target_s):
    """Child-process entry of the single-thread oracle figure: the process was started with one
    BLAS / OpenMP thread; prints {tflops, seconds, n, cols, fixed_s, per_row_s} as JSON."""
    ws = workload_set(workload)
    t = CpuOracleTimer(ws)
    t.calibrate(target_s, lo=16, hi=64)
    v, secs = t.run()
    print(json.dumps({"tflops": v, "seconds": secs, "n": t.n, "cols": t.cols,
                      "fixed_s": t.fixed, "per_row_s": t.per_row, "sample": t.sample()}))


def single_thread_oracle(workload, target_s, Ms):
    """The oracle on one host core (a child process with one BLAS thread): its rate on a sample
    and the whole step's time extrapolated from it. None if the child fails."""
    env = dict(os.environ, OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1", MKL_NUM_THREADS="1")
    env.pop("RANK", None), env.pop("WORLD_SIZE", None), env.pop("LOCAL_RANK", None)
    try:
        r = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-probe",
                            "--workload", workload, "--ref-step-s", str(target_s)],
                           capture_output=True, text=True, timeout=600, env=env)
        j = json.loads(r.stdout.strip().splitlines()[-1])
    except (subprocess.SubprocessError, ValueError, IndexError):
        return None
    step = sum(j["fixed_s"] + j["per_row_s"] * M for M in Ms)
    return {"value": j["tflops"], "unit": UNIT, "cores": 1, "seconds": j["seconds"],
            "sample": j["sample"],
            "step_s_extrapolated": step}


def bench_reference(args):
    world, rank, _ = dist_setup()
    if rank != 0:
        return 0
    ws = workload_set(args.workload)
    timer = CpuOracleTimer(ws)
    per_step = min(args.ref_step_s, 150.0 / max(1, args.steps + args.warmup))
    timer.calibrate(per_step)
    for _ in range(args.warmup):
        timer.run()
    vals, secs = [], 0.0
    for _ in range(args.steps):
        v, s = timer.run()
        vals.append(v)
        secs += s
    value = secs and (2 * timer.n * timer.cols * timer.w.d * args.steps) / secs / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000 * secs / max(1, args.steps), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": describe(args.workload, ws),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": timer.cores, "kind": "oracle",
                         "sample": timer.sample(), "cpu": timer.cpu()},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def oracle_timing(args):
    """The oracle's time for whole configurations on this host's cores: measured on the ones it
    finishes in seconds (Tiny, the LLaDA-8B ratios, block decode), extrapolated linearly in the
    masked rows (fixed W decode per call plus a per-row cost, both measured) on the long-context
    and Dream-shaped ones. One JSON line per configuration."""
    import numpy as np

    from masked_token_lm_gb300 import workloads as wl
    from oracle import mask_only_logits as orc

    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    for w in [wl.TINY] + wl.LLADA + [wl.DECODE] + wl.LONG + [wl.DREAM]:
        import torch

        mask = w.mask()
        flops = w.flops(mask.M)
        if w in wl.LONG or w is wl.DREAM:
            t = CpuOracleTimer([w])
            t.calibrate(args.ref_step_s)
            secs, how = t.step_seconds([mask.M]), "extrapolated"
        else:
            Hb = w.hidden("cpu").view(torch.int16).numpy().view(np.uint16)
            Wb = w.weight("cpu").view(torch.int16).numpy().view(np.uint16)
            so = None if mask.seq_offsets is None else mask.seq_offsets.numpy()
            mo = None if mask.mask_offsets is None else mask.mask_offsets.numpy()
            rows = orc.resolve_rows(mask.idx.numpy(), w.L_tot, so, mo)
            orc.masked_logits(Hb, rows[:8], Wb)  # warm-up: one-time allocation and page faults
            t0 = time.perf_counter()
            orc.masked_logits(Hb, mask.idx.numpy(), Wb, so, mo)
            secs, how = time.perf_counter() - t0, "measured"
        print(json.dumps({"workload": w.name, "M": mask.M, "flop": flops, "oracle_s": secs,
                          "tflops": flops / secs / 1e12, "how": how, "cores": cores,
                          "cpu": CpuOracleTimer.cpu()}), flush=True)
    return 0


def bench_e2e(args, mo, mz, calls, tot_flops, world, dev, stream):
    """The same step end to end through the public call: every step copies its inputs (H, idx,
    CSR offsets and W) from pinned host memory to the device and reads all logits back to pinned
    host memory. Uploads and read-backs run on their own streams and overlap compute and each
    other (within and across steps); W and H have two device buffers each, used by alternate
    steps, so one step's uploads do not wait for the previous step's compute. Unchunked members
    read their [M, V] logits back into a pinned [M, V] host buffer. Chunked members read every
    chunk back into one reused pinned [chunk_rows, V] host buffer: the chunk callback (the
    consumer) copies the chunk out of the library's buffer into one of two device staging
    buffers on the compute stream, so the next chunk can start while the read-back runs. The
    timed region spans all of it."""
    import torch

    host_in, host_out = [], []
    h2d = d2h = 0
    for c in calls:
        hi = {"H": c["H"].cpu().pin_memory(), "idx": c["mask"].idx.cpu().pin_memory()}
        if c is calls[0] or c["W"] is not calls[0]["W"]:
            hi["W"] = c["W"].cpu().pin_memory()
        for k2 in ("so", "mo"):
            t = c["mask"].seq_offsets if k2 == "so" else c["mask"].mask_offsets
            if t is not None:
                hi[k2] = t.cpu().pin_memory()
        host_in.append(hi)
        h2d += sum(t.numel() * t.element_size() for t in hi.values())
        rows_host = c["w"].chunk_rows if c["chunked"] else c["mask"].M
        ho = torch.empty((rows_host, c["w"].V), dtype=c["odt"], pin_memory=True)
        host_out.append(ho)
        d2h += c["mask"].M * c["w"].V * ho.element_size()
    # two sets of device inputs, used by alternate steps
    dev_in = [[{k2: torch.empty_like(v, device=dev) for k2, v in hi.items()} for hi in host_in]
              for _ in range(2)]
    dev_out = [torch.empty_like(c["out"]) for c in calls]
    staging = [[torch.empty_like(c["out"]) for _ in range(2)] if c["chunked"] else None
               for c in calls]
    s_in = torch.cuda.Stream(device=dev)
    s_out = torch.cuda.Stream(device=dev)

    consumed = [[None] * len(calls) for _ in range(2)]  # last use of each input set per member
    read_back = [None] * len(calls)                     # read-back of each member's output done
    stage_free = [[None, None] for _ in calls]          # read-back of each staging buffer done
    parity = [0]

    def e2e_step():
        par = parity[0]
        Wd = None
        for j, (c, hi, ho, do) in enumerate(zip(calls, host_in, host_out, dev_out)):
            di = dev_in[par][j]
            with torch.cuda.stream(s_in):
                if consumed[par][j] is not None:
                    s_in.wait_event(consumed[par][j])
                if j == 0 and consumed[par][-1] is not None:
                    # member 0's W buffer serves every member of the step: wait for the last one
                    s_in.wait_event(consumed[par][-1])
                for k2, v in hi.items():
                    di[k2].copy_(v, non_blocking=True)
                ready = torch.cuda.Event()
                ready.record(s_in)
            stream.wait_event(ready)
            if read_back[j] is not None and not c["chunked"]:
                stream.wait_event(read_back[j])
            Wd = di["W"] if "W" in di else dev_in[par][0]["W"]

            def on_chunk(ci, rb, rows, out, j=j, ho=ho, c=c):
                if not c["chunked"]:
                    done = torch.cuda.Event()
                    done.record(stream)
                    s_out.wait_event(done)
                    with torch.cuda.stream(s_out):
                        ho.copy_(out, non_blocking=True)
                    return
                k = ci % 2
                st = staging[j][k]
                with torch.cuda.stream(stream):
                    if stage_free[j][k] is not None:
                        stream.wait_event(stage_free[j][k])
                    st[:rows].copy_(out[:rows], non_blocking=True)
                    done = torch.cuda.Event()
                    done.record(stream)
                s_out.wait_event(done)
                with torch.cuda.stream(s_out):
                    ho[:rows].copy_(st[:rows], non_blocking=True)
                    ev = torch.cuda.Event()
                    ev.record(s_out)
                stage_free[j][k] = ev

            mo.masked_logits(di["H"], di["idx"], Wd, di.get("so"), di.get("mo"), out=do,
                             chunk_rows=c["w"].chunk_rows, on_chunk=on_chunk, stream=stream)
            ev_c = torch.cuda.Event()
            ev_c.record(stream)
            consumed[par][j] = ev_c
            read_back[j] = torch.cuda.Event()
            read_back[j].record(s_out)
        parity[0] ^= 1

    for _ in range(max(1, args.warmup)):
        e2e_step()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    n_e2e = max(1, min(args.steps, args.e2e_steps))
    e0.record(stream)
    s_in.wait_event(e0)
    for _ in range(n_e2e):
        e2e_step()
    for ev in read_back:  # the timed region ends when the last logits are on the host
        stream.wait_event(ev)
    e1.record(stream)
    torch.cuda.synchronize()
    e_ms = e0.elapsed_time(e1) / n_e2e
    (e_ms,) = max_over_ranks([e_ms], dev)
    if mo.check() != mz.MOSAIC_OK:
        raise SystemExit(f"kernel status in the e2e leg: {mz.mosaic_last_error_string()}")
    # What reached the host is the device-timed leg's result bit for bit: each member's pinned
    # buffer holds its last chunk (or all rows), the device-timed leg's output buffer the same.
    for c, ho in zip(calls, host_out):
        n = launch_rows(c["mask"].M, c["w"].chunk_rows)[-1]
        if not torch.equal(ho[:n].view(torch.int16) if ho.dtype == torch.bfloat16 else ho[:n],
                           c["out"][:n].cpu().view(torch.int16) if ho.dtype == torch.bfloat16
                           else c["out"][:n].cpu()):
            raise SystemExit(f"e2e leg: logits read back for {c['w'].name} differ from the device result")
    return {"value": world * tot_flops / (e_ms * 1e-3) / 1e12, "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e_ms,
            "steps": n_e2e, "verified": "last chunk on the host equals the device result bitwise",
            "path": "pinned host -> Mosaic.masked_logits (C ABI) -> pinned host; chunks read back "
                    "through two device staging buffers into one reused pinned chunk buffer"}


def cublas_context(args, calls, replay_step, tot_flops, stream, local):
    """Context only (not a target, not this library): the same step done unfused by torch --
    index_select of the masked rows into a gathered buffer, then a cuBLAS bf16 matmul with W^T
    into the same output buffer, chunk by chunk as the library's call is chunked (CSR members use
    their resolved rows). It runs interleaved step by step with this library's step (A/B/A/B,
    the same step count, after the same warm-up) inside one clock-sampled region, so both see the
    same clocks; per-step CUDA events time each side."""
    import torch

    prepared = []
    for c in calls:
        m = c["mask"]
        if m.seq_offsets is None:
            rows = m.idx.long()
        else:  # resolve the CSR batch once, outside the timed region
            counts = (m.mask_offsets[1:] - m.mask_offsets[:-1]).long()
            seq = torch.repeat_interleave(torch.arange(counts.numel(), device=counts.device), counts)
            rows = m.seq_offsets.long()[seq] + m.idx.long()
        cr = c["out"].shape[0]
        gbuf = torch.empty((cr, c["w"].d), dtype=torch.bfloat16, device=c["H"].device)
        out = torch.empty_like(c["out"])
        prepared.append((c, rows, gbuf, out, launch_rows(m.M, c["w"].chunk_rows)))

    def cublas_step():
        for c, rows, gbuf, out, chunks in prepared:
            rb = 0
            for n in chunks:
                torch.index_select(c["H"], 0, rows[rb:rb + n], out=gbuf[:n])
                torch.matmul(gbuf[:n], c["W"].t(), out=out[:n])
                rb += n

    for _ in range(args.warmup):
        cublas_step()
        replay_step()
    torch.cuda.synchronize()
    n = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(n)]
    with ClockSampler(local) as clk:
        clk.region_start()
        for s in range(n):
            ev[s][0].record(stream)
            replay_step()
            ev[s][1].record(stream)
            ev[s][2].record(stream)
            cublas_step()
            ev[s][3].record(stream)
        torch.cuda.synchronize()
        clk.region_end()
    fused_ms = sum(e[0].elapsed_time(e[1]) for e in ev) / n
    cub_ms = sum(e[2].elapsed_time(e[3]) for e in ev) / n
    return {"value": tot_flops / (cub_ms * 1e-3) / 1e12, "unit": UNIT, "ms_per_step": cub_ms,
            "fused_ms_per_step_same_region": fused_ms,
            "fused_over_cublas_speed": cub_ms / fused_ms,
            "steps": n, "clocks": clk.summary(),
            "what": "torch index_select + cuBLAS bf16 matmul per chunk (unfused, writes the "
                    "gathered rows), interleaved A/B with this library's step"}


def bench_cuda(args):
    import torch

    from masked_token_lm_gb300 import mosaic as mz
    from masked_token_lm_gb300 import workloads as wl

    world, rank, local = dist_setup()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (no CPU fallback)")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)
    ws = workload_set(args.workload)
    mo = mz.Mosaic(local)
    stream = torch.cuda.current_stream()

    # ---- inputs resident in HBM (per-rank seeds: each rank owns an independent batch)
    seed_shift = rank_seed_shift(rank)
    calls = []
    tot_flops = tot_bytes = 0
    n_launch_units = 0  # gather-GEMM launches per step
    for w in ws:
        mask = w.mask().to(dev)
        H = wl.make_hidden(w.L_tot, w.d, w.seed + 1 + seed_shift, dev)
        W = wl.make_weight(w.V, w.d, w.seed + 2 + seed_shift, dev)
        odt = torch.float32 if w.out_dtype == "f32" else torch.bfloat16
        chunked = 0 < w.chunk_rows < mask.M
        out = torch.empty((w.chunk_rows if chunked else mask.M, w.V), dtype=odt, device=dev)
        call = dict(w=w, mask=mask, H=H, W=W, out=out, odt=odt, chunked=chunked)
        if args.mode == "sample":
            ws_bytes = mz.mosaic_masked_sample_workspace_bytes(mask.M, w.V, w.chunk_rows)
            call["workspace"] = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
            tot_bytes += sample_bytes(mask.M, w.V, w.d, ws_bytes)
        elif args.mode == "fp8":
            # E4M3 W and gathered rows (1 byte), logits, indices, and the step's quantization of
            # the masked hidden rows (bf16 read, codes and scales written)
            tot_bytes += (w.V * w.d + mask.M * w.d + mask.M * w.V * out.element_size() + 4 * mask.M
                          + mask.M * w.d * 3 + 4 * mask.M)
        else:
            tot_bytes += algorithmic_bytes(mask.M, w.V, w.d, out.element_size())
        calls.append(call)
        tot_flops += w.flops(mask.M)
        n_launch_units += len(launch_rows(mask.M, w.chunk_rows))
    # identical W across members of one workload set: share it
    for c in calls[1:]:
        if c["w"].V == calls[0]["w"].V and c["w"].d == calls[0]["w"].d:
            c["W"] = calls[0]["W"]
    if args.mode == "fp8":
        # W is quantized once (model load); each step quantizes the hidden rows it reads
        for c in calls:
            if c is calls[0] or c["W"] is not calls[0]["W"]:
                c["Wq"], c["sW"] = mz.quantize_rows_e4m3(c["W"])
            else:
                c["Wq"], c["sW"] = calls[0]["Wq"], calls[0]["sW"]
            c["Hq"] = torch.empty(c["H"].shape, dtype=torch.uint8, device=dev)
            c["sH"] = torch.empty(c["H"].shape[0], dtype=torch.float32, device=dev)
        torch.cuda.synchronize()

    noop = (lambda *a: None)

    def one_call(c, st=None):
        st = stream if st is None else st
        m = c["mask"]
        if args.mode == "fp8":
            # this step's hidden rows that the logits read, quantized in place
            mz.quantize_masked_rows_e4m3(c["H"], m.idx, c["Hq"], c["sH"], m.seq_offsets,
                                         m.mask_offsets, stream=st)
            mo.masked_logits_fp8(c["Hq"], c["sH"], m.idx, c["Wq"], c["sW"], m.seq_offsets,
                                 m.mask_offsets, out=c["out"], chunk_rows=c["w"].chunk_rows,
                                 on_chunk=noop if c["chunked"] else None, stream=st)
            return
        if args.mode == "sample":
            mo.masked_sample(c["H"], m.idx, c["W"], m.seq_offsets, m.mask_offsets,
                             chunk_rows=c["w"].chunk_rows, workspace=c["workspace"], stream=st)
            return
        mo.masked_logits(c["H"], m.idx, c["W"], m.seq_offsets, m.mask_offsets, out=c["out"],
                         chunk_rows=c["w"].chunk_rows, on_chunk=noop if c["chunked"] else None,
                         stream=st)

    def step():
        for c in calls:
            one_call(c)

    for _ in range(args.warmup):
        step()
    st = mo.check()
    if st != mz.MOSAIC_OK:
        raise SystemExit(f"kernel status {st}: {mz.mosaic_last_error_string()}")

    # Each member's call (every launch of it: quantization, gather-GEMM chunks, reduction) is
    # captured once into a CUDA graph and replayed per step, so the host's per-call argument
    # checks and enqueue time do not leave the GPU idle between launches; the kernels and their
    # work are exactly those of the direct calls (--no-graph times the direct calls instead).
    graphs = []
    captured_launches = 0
    if not args.no_graph:
        cap = torch.cuda.Stream(device=dev)
        cap.wait_stream(stream)
        for c in calls:
            g = torch.cuda.CUDAGraph()
            l0 = mo.launches
            with torch.cuda.graph(g, stream=cap, capture_error_mode="relaxed"):
                one_call(c, cap)
            captured_launches += mo.launches - l0
            graphs.append(g)
        stream.wait_stream(cap)
        torch.cuda.synchronize()
        for g in graphs:  # one untimed replay each
            g.replay()
        torch.cuda.synchronize()

    def replay_member(j):
        if graphs:
            graphs[j].replay()
        else:
            one_call(calls[j])

    def replay_step():
        for j in range(len(calls)):
            replay_member(j)

    # ---- device-timed region: per-call events on the launching stream
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    launches0 = mo.launches
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps * len(calls))]
    with ClockSampler(local) as clk:
        t_start = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        clk.region_start()
        t_start.record(stream)
        k = 0
        for _ in range(args.steps):
            for j in range(len(calls)):
                evs[k][0].record(stream)
                replay_member(j)
                evs[k][1].record(stream)
                k += 1
        t_end.record(stream)
        torch.cuda.synchronize()
        clk.region_end()
    launches = mo.launches - launches0 + (args.steps * captured_launches if graphs else 0)
    if args.mode == "fp8":
        launches += args.steps * len(calls)  # one hidden-state quantization per call
    st = mo.check()
    if st != mz.MOSAIC_OK:
        raise SystemExit(f"kernel status {st}: {mz.mosaic_last_error_string()}")
    total_ms = t_start.elapsed_time(t_end)
    member_ms = [0.0] * len(calls)
    for k, (a, b) in enumerate(evs):
        member_ms[k % len(calls)] += a.elapsed_time(b) / args.steps
    kernel_ms = sum(member_ms) * args.steps
    total_ms, kernel_ms, *member_ms = max_over_ranks([total_ms, kernel_ms, *member_ms], dev)
    ms_per_step = total_ms / args.steps
    value = world * tot_flops / (ms_per_step * 1e-3) / 1e12
    gbs = world * tot_bytes / (ms_per_step * 1e-3) / 1e9

    # ---- end to end through the public call: pinned host inputs -> device -> logits -> host
    e2e = None
    if not args.no_e2e and args.mode == "logits":
        e2e = bench_e2e(args, mo, mz, calls, tot_flops, world, dev, stream)

    cublas = None
    if not args.no_cublas_context and args.mode == "logits":
        cublas = cublas_context(args, calls, replay_step, tot_flops, stream, local)

    peaks = load_peaks()
    clocks = clk.summary()
    roof = roofline_entry(tot_flops * args.steps, tot_bytes * args.steps, kernel_ms * 1e-3,
                          peaks, args.mode)
    traffic = None
    if args.traffic is not None:
        traffic = args.traffic
    elif args.mode == "logits":
        traffic = MEASURED_TRAFFIC.get(kernel_source_hash(), {}).get(args.workload)
    roof.update({
        "traffic": traffic,
        "traffic_per": "launch (mean over the step's gather-GEMM launches)",
        "launches_per_step": n_launch_units,
        "algorithmic_bytes_per_launch": tot_bytes / max(1, n_launch_units),
        "kernel": ("gather_gemm_kernel<fp8> + per-step masked-row quantization"
                   if args.mode == "fp8" else
                   "gather_gemm_kernel<sample> + sample_reduce_kernel" if args.mode == "sample"
                   else "gather_gemm_kernel<bf16 out, CTA pair>"),
        "timing": "CUDA events around every member call on the launching stream, summed",
    })
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "e4m3" if args.mode == "fp8" else "bf16", "data": "synthetic",
        "config": {**describe(args.workload, ws),
                   "M": [c["mask"].M for c in calls],
                   "flop_per_step": tot_flops,
                   "algorithmic_bytes_per_step": tot_bytes,
                   "parallelism": f"replicas x{world} (independent batches, no collective)",
                   "launch": "direct calls" if args.no_graph else
                             "one CUDA-graph replay per member call (captured from the public calls)"},
        "gbs": gbs,
        "member_ms": dict(zip([c["w"].name for c in calls], member_ms)),
        "mode": args.mode,
        "kernel_source_hash": kernel_source_hash(),
        "roofline": roof,
        "gpu_launches": launches,
        "cublas_context": cublas,
        "clocks": clocks,
        "e2e": e2e,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        timer = CpuOracleTimer(ws)
        timer.calibrate(args.ref_step_s)
        v, secs = timer.run()
        Ms = [c["mask"].M for c in calls]
        line["cpu_baseline"] = {
            "value": v, "unit": UNIT, "cores": timer.cores, "kind": "oracle",
            "sample": timer.sample(), "seconds": secs, "cpu": timer.cpu(),
            "step_s_extrapolated": timer.step_seconds(Ms),
            "step_extrapolation": "whole step, linear in the masked rows: one W decode per call "
                                  "plus the measured per-row cost",
            "single_thread": single_thread_oracle(args.workload, args.ref_step_s_single, Ms),
        }
    if rank == 0:
        print(json.dumps(line), flush=True)
    mo.close()
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--impl", default="cuda", choices=["cuda", "reference"])
    ap.add_argument("--mode", default="logits", choices=["logits", "sample", "fp8"],
                    help="logits: [M, V] mask-only logits (the metric); sample: fused greedy "
                         "sampling (token + confidence per masked row); fp8: the E4M3 variant "
                         "(W quantized once, the masked hidden rows every step)")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-cublas-context", action="store_true")
    ap.add_argument("--no-graph", action="store_true",
                    help="time direct calls instead of one CUDA-graph replay per member call")
    ap.add_argument("--ref-step-s", type=float, default=15.0)
    ap.add_argument("--ref-step-s-single", type=float, default=8.0,
                    help="target seconds of the single-thread oracle sample")
    ap.add_argument("--traffic", type=float, default=None,
                    help="dram bytes per launch from an ncu capture of the current kernel")
    ap.add_argument("--oracle-timing", action="store_true",
                    help="time the oracle on whole configurations (no GPU)")
    ap.add_argument("--oracle-probe", action="store_true", help=argparse.SUPPRESS)
    args = ap.parse_args()
    if args.oracle_probe:
        oracle_probe(args.workload, args.ref_step_s)
        return 0
    if args.oracle_timing:
        return oracle_timing(args)
    if args.warmup < 3 and args.impl == "cuda":
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        return bench_reference(args)
    return bench_cuda(args)


if __name__ == "__main__":
    sys.exit(main())
