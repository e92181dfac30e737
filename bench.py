"""Benchmark: BF16-in / FP32-accumulate GEMM, M = N = K = 8192, row-major.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl {gb300,reference}]
                    [--suite [--suite-out PATH]]

One step is one call of gemm_bf16f32 on the M = N = K = 8192 workload (A and
B drawn from normal(0, 1/sqrt(K)) and rounded to BF16, C in FP32).  A and B
(256 MiB together) exceed the 129 MB L2, so no flush is needed between steps.
Prints one JSON line (rank 0): TFLOP/s over the whole job, the dominant
kernel's roofline fraction (against the measured cuBLAS BF16 burst rate and
against the clock-limited tensor-core peak, SMs x 8192 FLOP/clk x the sampled
SM clock), a sustained reading (at least 2 s back to back, binned by the SM
clock seen), every workload configuration timed with its own roofline, the
oracle timed on the host cores (a bounded sample of rows) and used to check
the GPU's timed output and each configuration's output on samples, an
end-to-end figure through host buffers, the clocks seen while timing and the
number of kernel launches.

--impl reference times the CPU oracle instead (there is no other reference
implementation), on the same workload and metric, each step a bounded sample
of output rows.

--suite additionally times the extended operations (alpha/beta, transposed
storage, TF32, FP8, 16-bit C; not part of the JSON line) and writes them with
the workload configurations as JSON to --suite-out (default bench_suite.json
in the working directory).

With torchrun (N > 1) every rank runs its own replica of the workload on its
own GPU; nothing is exchanged between ranks (the product's rows are
independent), and the value is the total over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

M = N = K = 8192
FLOP = 2.0 * M * N * K
WORKLOAD = ("gemm_bf16f32 M=N=K=8192 row-major; A,B ~ normal(0, 1/sqrt(K)) rounded to BF16, "
            "C FP32, FP32 accumulate")
METRIC = "GEMM TFLOP/s (FP16-in/FP32-acc, M=N=K=8192) and % of GB300 dense peak"
SEED = 1238
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "tc_gemm_bf16_8192_traffic.json")
KERNEL_SOURCES = [os.path.join(ROOT, "dense_gemm_tensor_tcgen05_gb300", "csrc", f)
                  for f in ("tc_gemm.cu", "ptx.cuh", "cstore.cuh")]


# The workload configurations: (name, dtype, distribution, M, N, K, sigma,
# seed).  Seeds are 1234 + the configuration's index; the headline is index 4.
CONFIGS = [
    ("f16_1024_uniform", "f16", "uniform", 1024, 1024, 1024, 1.0, 1234),
    ("sgemm_1024_uniform", "f32", "uniform", 1024, 1024, 1024, 1.0, 1235),
    ("sgemm_4096_uniform", "f32", "uniform", 4096, 4096, 4096, 1.0, 1236),
    ("f16_2048_normal", "f16", "normal", 2048, 2048, 2048, 1.0, 1237),
    ("bf16_8192_normal", "bf16", "normal", 8192, 8192, 8192, 1 / math.sqrt(8192), 1238),
    ("f16_4000x3000x1000_uniform", "f16", "uniform", 4000, 3000, 1000, 1.0, 1239),
    ("f16_16384x128x4096_uniform", "f16", "uniform", 16384, 128, 4096, 1.0, 1240),
    ("f16_8x8192x8192_uniform", "f16", "uniform", 8, 8192, 8192, 1.0, 1241),
]
TC_FLOP_PER_CLK_SM = 8192      # dense 16-bit tensor-core FLOP per clock per SM
FP32_FLOP_PER_CLK_SM = 256     # 128 FP32 FMA lanes per SM


def clock_limited_tflops(sms: int, flop_per_clk: int, mhz: float) -> float:
    """Peak FLOP rate of `sms` SMs doing flop_per_clk FLOP per clock at mhz."""
    return sms * flop_per_clk * mhz * 1e6 / 1e12


def config_roofline(dtype: str, M: int, N: int, K: int, us: float, peaks: dict, sms: int,
                    mhz: float) -> dict:
    """Roofline of one configuration: the bound (tensor, alu or hbm: whichever
    of FLOP/peak and bytes/bandwidth takes longer), the achieved rate and the
    fraction of that bound's peak.  Bytes: A and B read once, C written once."""
    flop = 2.0 * M * N * K
    eb = 4 if dtype == "f32" else 2
    byts = (M * K + K * N) * eb + M * N * 4
    tflops = flop / us / 1e6
    gbs = byts / us / 1e3
    if dtype == "f32":
        bound, peak, unit, achieved = "alu", clock_limited_tflops(sms, FP32_FLOP_PER_CLK_SM, mhz), \
            "TFLOP/s", tflops
        source = f"{sms} SMs x {FP32_FLOP_PER_CLK_SM} FLOP/clk x {mhz:.0f} MHz (sampled)"
    else:
        t_tensor = flop / (peaks["bf16_tflops"] * 1e12)
        t_hbm = byts / (peaks["hbm_gbs"] * 1e9)
        if t_hbm > t_tensor:
            bound, peak, unit, achieved = "hbm", peaks["hbm_gbs"], "GB/s", gbs
            source = f"hbm_gbs of {peaks['source']}"
        else:
            bound, peak, unit, achieved = "tensor", peaks["bf16_tflops"], "TFLOP/s", tflops
            source = f"bf16_tflops (burst) of {peaks['source']}"
    return {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
            "frac": achieved / peak, "peak_source": source, "tflops": tflops, "gbs": gbs,
            "algorithmic_bytes": byts, "flop": flop}


def bin_by_clock(chunks):
    """chunks: [(tflops, [sm_mhz samples])] in time order.  Returns bins
    [{sm_mhz, tflops, chunks}] (one per distinct median clock, ascending)."""
    bins = {}
    for tf, mhz in chunks:
        if not mhz:
            continue
        key = float(statistics.median(mhz))
        bins.setdefault(key, []).append(tf)
    return [{"sm_mhz": k, "tflops": statistics.mean(v), "chunks": len(v)}
            for k, v in sorted(bins.items())]


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for p in KERNEL_SOURCES:
        with open(p, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "hbm_gbs": float(p["hbm_gbs"]), "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0,
                "source": "fallback"}


def load_traffic(plan: str):
    """DRAM bytes per launch from the committed ncu capture, if it was taken
    on the current kernel sources with the same plan; else None."""
    try:
        with open(PROFILE_TRAFFIC) as f:
            t = json.load(f)
    except (OSError, ValueError):
        return None
    if t.get("source_hash") != kernel_source_hash() or t.get("plan") != plan:
        return None
    return t.get("dram_bytes_per_launch")


def kernel_name(plan: str) -> str:
    if "pair=1" in plan:
        tail = ", the tiles after the last whole wave cut into K pieces" if "tail_split" in plan else ""
        return f"tc_gemm_pair_kernel<256, 0> (CTA pairs, 256x256 tiles, 3 stages of 2 K atoms{tail})"
    return "tc_gemm_kernel<256, false, 0> (one CTA, 128x256 tiles)"


# ---- multi-rank aggregation ------------------------------------------------------

def max_over_ranks(ms: float, dist=None, device="cpu") -> float:
    """The slowest rank's timed-region length (every rank gets it)."""
    if dist is None:
        return ms
    import torch
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(world: int, flop_per_step: float, steps: int, max_ms: float) -> float:
    """Whole-job throughput: every rank runs its own replica of the step, so
    the job did world x steps steps in the slowest rank's time."""
    return world * flop_per_step * steps / (max_ms / 1e3) / 1e12


# ---- clocks ---------------------------------------------------------------

class ClockSampler:
    """nvidia-smi samples (every 50 ms) while the benchmark runs."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 7:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)

    def sm_mhz_between(self, t0: float, t1: float):
        """SM clocks (MHz) of the samples taken between wall times t0 and t1."""
        out = []
        for t, s in self.samples:
            if t0 <= t <= t1:
                try:
                    out.append(float(s[0]))
                except ValueError:
                    pass
        return out

    def summary(self, t0: float, t1: float):
        win = [s for (t, s) in self.samples if t0 - 0.15 <= t <= t1 + 0.15]
        window = "timed"
        if not win:
            win = [s for (_, s) in self.samples]
            window = "run"
        if not win:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(s[0]) for s in win if num(s[0]) is not None]
        mx = [num(s[1]) for s in win if num(s[1]) is not None]
        pw = [num(s[2]) for s in win if num(s[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for s in win for i in range(4) if s[3 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": max(pw) if pw else None,
                "reasons": reasons, "samples": len(win), "window": window}


# ---- CPU oracle timing ------------------------------------------------------

def oracle_rows_timing(A, B, target_s: float, max_rows: int):
    """Time the oracle on a band of output rows sized to take about target_s.
    Returns (seconds, rows, threads, the band's values)."""
    import oracle
    threads = os.cpu_count() or 1
    rows = 1 if target_s < 1.0 else 8
    t = None
    while True:
        rows = min(rows, max_rows)
        t0 = time.perf_counter()
        band = oracle.gemm_rows("bf16", A, B, 0, rows, M=M, N=N, K=K, nthreads=threads)
        t = time.perf_counter() - t0
        if t >= target_s * 0.5 or rows >= max_rows:
            return t, rows, threads, band
        rows = int(rows * min(8.0, max(2.0, target_s / max(t, 1e-3))))


def make_inputs():
    from dense_gemm_tensor_tcgen05_gb300 import inputs
    A = inputs.make("normal", "bf16", M, K, SEED, 0, sigma=1 / math.sqrt(K))
    B = inputs.make("normal", "bf16", K, N, SEED, 1, sigma=1 / math.sqrt(K))
    return A, B


# ---- the reference arm: the oracle ------------------------------------------

def run_reference(args, rank, world):
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    A, B = make_inputs()
    threads = os.cpu_count() or 1
    # size one step so the whole run stays within a few minutes (a step is at
    # least one output row, plus the oracle's decode of B)
    target = max(0.05, min(2.0, 150.0 / (args.steps + args.warmup)))
    _, rows, _, _ = oracle_rows_timing(A, B, target_s=target, max_rows=M)
    for _ in range(args.warmup):
        oracle.gemm_rows("bf16", A, B, 0, rows, M=M, N=N, K=K, nthreads=threads)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.gemm_rows("bf16", A, B, 0, rows, M=M, N=N, K=K, nthreads=threads)
    dt = time.perf_counter() - t0
    flop = 2.0 * rows * N * K * args.steps
    value = flop / dt / 1e12
    sample = (f"{rows} of {M} output rows per step (2*{rows}*N*K FLOP), oracle in double, "
              f"{threads} threads")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "M": M, "N": N, "K": K, "sample": sample},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---- our arm -------------------------------------------------------------------

def to_device(bits, dt):
    """Element bits (numpy) -> a CUDA tensor holding the same bytes."""
    import numpy as np
    import torch
    if dt in ("f32", "tf32"):
        return torch.from_numpy(np.ascontiguousarray(bits)).cuda()
    if dt in ("e4m3", "e5m2"):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.uint8)).cuda()
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda()


def sustained_run(call, stream, sampler, launch_ms: float, min_s: float, sms: int):
    """Back-to-back launches for at least min_s seconds, timed in chunks of
    about 100 ms with CUDA events on the launching stream; each chunk is
    matched with the nvidia-smi samples taken while it ran."""
    import torch
    per_chunk = max(1, int(round(100.0 / max(launch_ms, 1e-3))))
    n_chunks = max(3, int(math.ceil(min_s * 1000.0 / (per_chunk * launch_ms))))
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(n_chunks + 1)]
    stream.synchronize()
    t_wall0 = time.time()
    with torch.cuda.stream(stream):
        evs[0].record(stream)
        for c in range(n_chunks):
            for _ in range(per_chunk):
                call()
            evs[c + 1].record(stream)
    stream.synchronize()
    t_wall1 = time.time()
    offs = [evs[0].elapsed_time(e) / 1e3 for e in evs]          # seconds from the first event
    chunks, all_mhz = [], []
    for c in range(n_chunks):
        dt = offs[c + 1] - offs[c]
        tf = FLOP * per_chunk / dt / 1e12
        mhz = sampler.sm_mhz_between(t_wall0 + offs[c], t_wall0 + offs[c + 1])
        chunks.append((tf, mhz))
        all_mhz += mhz
    total_s = offs[-1]
    tflops = FLOP * per_chunk * n_chunks / total_s / 1e12
    med = statistics.median(all_mhz) if all_mhz else None
    tenth = max(1, n_chunks // 10)
    out = {"seconds": total_s, "launches": per_chunk * n_chunks, "tflops": tflops,
           "tflops_first_tenth": statistics.mean(c[0] for c in chunks[:tenth]),
           "tflops_last_tenth": statistics.mean(c[0] for c in chunks[-tenth:]),
           "sm_mhz_median": med, "clock_bins": bin_by_clock(chunks),
           "clocks": sampler.summary(t_wall0, t_wall1)}
    if med:
        # work per clock, independent of the clock the power cap allowed
        out["flop_per_clk_per_sm"] = tflops * 1e12 / (med * 1e6) / sms
        out["tflops_per_ghz"] = tflops / (med / 1e3)
        peak = clock_limited_tflops(sms, TC_FLOP_PER_CLK_SM, med)
        out["clock_limited_peak"] = peak
        out["frac_of_clock_limited"] = tflops / peak
    return out


def time_config(g, torch, fn, stream, flush, min_ms=100.0):
    """(warm_us, cold_us) of one call: warm = back-to-back for at least min_ms;
    cold = median of 10 single launches, each after a 256 MiB write that
    flushes the L2."""
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for _ in range(5):
        fn()
    stream.synchronize()
    iters = 20
    while True:
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(iters):
                fn()
            e1.record(stream)
        stream.synchronize()
        ms = e0.elapsed_time(e1)
        if ms >= min_ms or iters >= 20000:
            break
        iters = int(iters * max(2.0, 1.1 * min_ms / max(ms, 1e-3)))
    warm_us = ms / iters * 1e3
    cold = []
    for _ in range(10):
        with torch.cuda.stream(stream):
            flush.zero_()
            e0.record(stream)
            fn()
            e1.record(stream)
        stream.synchronize()
        cold.append(e0.elapsed_time(e1) * 1e3)
    return warm_us, statistics.median(cold)


def output_samples(C_host, M, N, seed, band=8, n_entries=256):
    """Rows and entries of a product kept for the oracle check: the first,
    a middle and the last band of rows, and random single entries (some in
    the last columns)."""
    import numpy as np
    bands = []
    for r0 in (0, M // 2, max(0, M - band)):
        r1 = min(M, r0 + band)
        if bands and r0 < bands[-1][1]:          # overlapping bands merge
            bands[-1] = (bands[-1][0], max(bands[-1][1], r1))
        else:
            bands.append((r0, r1))
    rows = [r for (r0, r1) in bands for r in range(r0, r1)]
    rng = np.random.default_rng(seed)
    er = rng.integers(0, M, size=n_entries)
    ec = rng.integers(0, N, size=n_entries)
    ec[: n_entries // 4] = N - 1 - (np.arange(n_entries // 4) % min(N, 16))
    return {"bands": bands, "rows": rows, "row_values": C_host[rows].copy(), "entry_rows": er,
            "entry_cols": ec, "entry_values": C_host[er, ec].copy()}


def run_configs(g, torch, np, peaks, stream, sms, sampler, headline):
    """Every workload configuration through its fixed entry point's default
    plan, timed warm and cold, with samples of its output kept for the
    oracle.  `headline` = (A bits, B bits, C on the device, A and B device
    addresses) reuses the headline's inputs for the BF16 8192^3
    configuration.  The clock for the FP32 roofline is the median SM clock
    sampled while the configuration ran."""
    from dense_gemm_tensor_tcgen05_gb300 import inputs
    fns = {"f16": g.gemm_f16f32, "bf16": g.gemm_bf16f32, "f32": g.sgemm_f32}
    codes = {"f16": 0, "bf16": 1, "f32": 2}
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    sh = stream.cuda_stream
    out, keep = [], []
    for name, dt, dist, m, n, k, sigma, seed in CONFIGS:
        if name == "bf16_8192_normal":
            A, B, Cd = headline[0], headline[1], headline[2]
            Ad, Bd = None, None
            args = (headline[3], headline[4], Cd.data_ptr(), m, n, k, k, n, n)
        else:
            A = inputs.make(dist, dt, m, k, seed, 0, sigma)
            B = inputs.make(dist, dt, k, n, seed, 1, sigma)
            Ad, Bd = to_device(A, dt), to_device(B, dt)
            Cd = torch.empty((m, n), dtype=torch.float32, device="cuda")
            args = (Ad.data_ptr(), Bd.data_ptr(), Cd.data_ptr(), m, n, k, k, n, n)
        fn = lambda args=args, f=fns[dt]: f(*args, stream=sh)
        plan = g.gemm_plan_describe(codes[dt], *args)
        t0 = time.time()
        warm_us, cold_us = time_config(g, torch, fn, stream, flush)
        clk = sampler.sm_mhz_between(t0 - 0.05, time.time() + 0.05)
        mhz = statistics.median(clk) if clk else 2070.0
        g.gemm_device_error(sh)
        C_host = Cd.cpu().numpy()
        r_warm = config_roofline(dt, m, n, k, warm_us, peaks, sms, mhz)
        r_cold = config_roofline(dt, m, n, k, cold_us, peaks, sms, mhz)
        out.append({"name": name, "dtype": dt, "M": m, "N": n, "K": k, "dist": dist,
                    "sigma": sigma, "seed": seed, "plan": plan,
                    "us_warm": warm_us, "us_cold": cold_us,
                    "tflops_warm": r_warm["tflops"], "tflops_cold": r_cold["tflops"],
                    "gbs_warm": r_warm["gbs"], "gbs_cold": r_cold["gbs"],
                    "roofline": {"bound": r_warm["bound"], "peak": r_warm["peak"],
                                 "unit": r_warm["unit"], "peak_source": r_warm["peak_source"],
                                 "achieved_warm": r_warm["achieved"],
                                 "frac_warm": r_warm["frac"],
                                 "achieved_cold": r_cold["achieved"],
                                 "frac_cold": r_cold["frac"],
                                 "algorithmic_bytes": r_warm["algorithmic_bytes"],
                                 "sm_mhz_median": mhz if clk else None},
                    "timing": "warm: back to back for >= 100 ms (small inputs may stay in "
                              "L2); cold: median of 10 launches, each after a 256 MiB write"})
        keep.append((dt, A, B, m, n, k, output_samples(C_host, m, n, seed)))
        del Ad, Bd, C_host
        if name != "bf16_8192_normal":
            del Cd
        torch.cuda.empty_cache()
    del flush
    torch.cuda.empty_cache()
    return out, keep


def oracle_leg(A, B, C_host, configs, kept, target_s=12.0):
    """The CPU side, run after every GPU timing: the oracle, as it stands,
    timed on a band of rows of the headline product (the cpu_baseline), and
    the same rows -- with the last band and random entries -- compared with
    the GPU's output of the timed steps; then each configuration's output
    samples compared with the oracle's values at the same places."""
    import numpy as np
    import oracle
    from dense_gemm_tensor_tcgen05_gb300 import inputs
    oracle.build()
    t, rows, threads, R = oracle_rows_timing(A, B, target_s=target_s, max_rows=M)
    cpu = {"value": 2.0 * rows * N * K / t / 1e12, "unit": "TFLOP/s", "cores": threads,
           "kind": "oracle",
           "sample": f"rows 0..{rows - 1} of the {M}x{N}x{K} product ({t:.1f} s, double "
                     f"accumulation, {threads} threads)"}
    amax, bmax = inputs.bits_abs_max(A, "bf16"), inputs.bits_abs_max(B, "bf16")
    tail = oracle.gemm_rows("bf16", A, B, M - 16, M, M=M, N=N, K=K, nthreads=threads)
    rng = np.random.default_rng(7)
    er, ec = rng.integers(0, M, 2048), rng.integers(0, N, 2048)
    ent = oracle.gemm_entries("bf16", A, B, er, ec, M=M, N=N, K=K)
    got = np.concatenate([C_host[:rows].ravel(), C_host[M - 16:].ravel(), C_host[er, ec]])
    want = np.concatenate([R.ravel(), tail.ravel(), ent])
    cmp = oracle.compare(got, want, K, amax, bmax)
    parity = {"ok": bool(cmp.ok), "checked": f"rows 0..{rows - 1} and {M - 16}..{M - 1} "
              f"({(rows + 16) * N} elements) and 2048 random entries of the last timed step's C",
              "max_abs": cmp.max_abs, "abs_bound": cmp.abs_bound, "rel_frob": cmp.rel_frob,
              "rel_bound": cmp.rel_bound}
    for cfg, (dt, Ac, Bc, m, n, k, smp) in zip(configs, kept):
        Rr = np.concatenate([oracle.gemm_rows(dt, Ac, Bc, r0, r1, M=m, N=n, K=k, nthreads=threads)
                             for (r0, r1) in smp["bands"]])
        Re = oracle.gemm_entries(dt, Ac, Bc, smp["entry_rows"], smp["entry_cols"], M=m, N=n, K=k)
        c = oracle.compare(np.concatenate([smp["row_values"].ravel(), smp["entry_values"]]),
                           np.concatenate([Rr.ravel(), Re]), k, inputs.bits_abs_max(Ac, dt),
                           inputs.bits_abs_max(Bc, dt))
        cfg["parity"] = {"ok": bool(c.ok), "max_abs": c.max_abs, "abs_bound": c.abs_bound,
                         "rel_frob": c.rel_frob, "checked": f"{len(smp['rows'])} rows + "
                         f"{len(smp['entry_rows'])} entries"}
    return cpu, parity


def run_gb300(args, rank, world, local_rank):
    import numpy as np
    import torch
    import dense_gemm_tensor_tcgen05_gb300 as g
    from dense_gemm_tensor_tcgen05_gb300 import build

    dist = None
    if world > 1:
        import torch.distributed as dist_mod
        dist = dist_mod
    torch.cuda.set_device(local_rank)
    if rank == 0 or world == 1:
        build.build()
    if dist:
        dist.barrier()
    g.lib()
    sms = torch.cuda.get_device_properties(local_rank).multi_processor_count

    A, B = make_inputs()
    Ad = torch.from_numpy(A.view(np.int16)).view(torch.bfloat16).cuda()
    Bd = torch.from_numpy(B.view(np.int16)).view(torch.bfloat16).cuda()
    Cd = torch.empty((M, N), dtype=torch.float32, device="cuda")
    stream = torch.cuda.Stream()
    sh = stream.cuda_stream
    call = lambda: g.gemm_bf16f32(Ad.data_ptr(), Bd.data_ptr(), Cd.data_ptr(), M, N, K, K, N, N, sh)

    # one run first: the plan, the device error word; the output of the timed
    # steps is checked against the oracle after all GPU timing
    torch.cuda.synchronize()
    call()
    g.gemm_device_error(sh)
    plan = g.gemm_plan_describe(1, Ad.data_ptr(), Bd.data_ptr(), Cd.data_ptr(), M, N, K, K, N, N)

    sampler = ClockSampler(local_rank)
    sampler.start()
    time.sleep(0.3)
    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    launches0 = g.gemm_launch_count()
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    t_wall0 = time.time()
    with torch.cuda.stream(stream):
        evs[0].record(stream)
        for i in range(args.steps):
            call()
            evs[i + 1].record(stream)
    stream.synchronize()
    t_wall1 = time.time()
    launches = g.gemm_launch_count() - launches0
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    g.gemm_device_error(sh)
    C_host = Cd.cpu().numpy()          # the last timed step's output, for the oracle

    per = [evs[i].elapsed_time(evs[i + 1]) for i in range(args.steps)]
    total_ms = max_over_ranks(evs[0].elapsed_time(evs[-1]), dist, device="cuda")
    value = job_tflops(world, FLOP, args.steps, total_ms)
    kernel_ms = statistics.mean(per)
    peaks = load_peaks()
    achieved = FLOP / (kernel_ms / 1e3) / 1e12
    time.sleep(0.2)
    clocks = sampler.summary(t_wall0, t_wall1)
    mhz = clocks.get("sm_mhz") or clocks.get("sm_max_mhz") or 2070.0
    clock_peak = clock_limited_tflops(sms, TC_FLOP_PER_CLK_SM, mhz)
    roofline = {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s", "frac": achieved / peaks["bf16_tflops"],
                "traffic": load_traffic(plan),
                "peak_source": f"bf16_tflops (burst) of {peaks['source']}",
                "kernel": kernel_name(plan), "kernel_ms_mean": kernel_ms,
                "kernel_ms_median": statistics.median(per),
                "kernel_ms_first_tenth": statistics.mean(per[: max(1, len(per) // 10)]),
                "kernel_ms_last_tenth": statistics.mean(per[-max(1, len(per) // 10):]),
                "clock_limited_peak": clock_peak,
                "clock_limited_peak_source": f"{sms} SMs x {TC_FLOP_PER_CLK_SM} FLOP/clk x "
                                             f"{mhz:.0f} MHz (median SM clock sampled while timing)",
                "frac_of_clock_limited": achieved / clock_peak,
                "frac_of_sustained": achieved / peaks["bf16_tflops_sustained"]}

    # sustained: the same call back to back for at least --sustained-s seconds
    sustained = None
    if args.sustained_s > 0:
        if dist:
            dist.barrier()
        sustained = sustained_run(call, stream, sampler, kernel_ms, args.sustained_s, sms)
        sustained["frac_of_measured_sustained"] = (sustained["tflops"] /
                                                   peaks["bf16_tflops_sustained"])
        sustained["measured_sustained_source"] = f"bf16_tflops_sustained of {peaks['source']}"
        g.gemm_device_error(sh)

    # end to end through the C ABI with host buffers (gemm_ex_host): every
    # step copies A and B in from page-locked host memory, multiplies, and
    # copies C back; the library pipelines the copies with the product
    Ah = torch.from_numpy(A.view(np.int16)).pin_memory()
    Bh = torch.from_numpy(B.view(np.int16)).pin_memory()
    Ch = torch.empty((M, N), dtype=torch.float32).pin_memory()
    e2e_steps = max(3, min(args.steps, 20))
    host_call = lambda: g.gemm_ex_host(Ah.data_ptr(), Bh.data_ptr(), Ch.data_ptr(), M, N, K, K, N, N,
                                       dtype=1, stream=sh)
    host_call()
    stream.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    launches_e2e0 = g.gemm_launch_count()
    e0.record(stream)
    for _ in range(e2e_steps):
        host_call()
    e1.record(stream)
    stream.synchronize()
    g.gemm_device_error(sh)
    e2e_launches = g.gemm_launch_count() - launches_e2e0
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), dist, device="cuda")
    e2e_value = job_tflops(world, FLOP, e2e_steps, e2e_ms)
    e2e = {"value": e2e_value, "unit": "TFLOP/s",
           "h2d_bytes_per_step": int(Ah.numel() * 2 + Bh.numel() * 2),
           "d2h_bytes_per_step": int(Ch.numel() * 4), "steps": e2e_steps,
           "api": "gemm_ex_host (C ABI, page-locked host buffers, copies pipelined over row panels)",
           "gpu_launches": e2e_launches}
    del Ah, Bh, Ch

    configs, kept = None, None
    if rank == 0 and not args.no_configs:
        configs, kept = run_configs(g, torch, np, peaks, stream, sms, sampler,
                                    (A, B, Cd, Ad.data_ptr(), Bd.data_ptr()))
        for c in configs:
            if c["name"] == "bf16_8192_normal":
                c["note"] = "the headline workload; its timed steps are `value`"
    sampler.stop()

    if args.suite and rank == 0:
        run_suite(g, torch, np, peaks, args.suite_out, configs or [])

    cpu, parity = None, None
    if rank == 0 and not args.no_cpu_baseline:
        cpu, parity = oracle_leg(A, B, C_host, configs or [], kept or [])

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_ms / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic",
            "config": {"workload": WORKLOAD, "M": M, "N": N, "K": K, "plan": plan,
                       "l2": "inputs exceed L2 (A+B = 256 MiB > 129 MB); no flush",
                       "parallelism": "replicas" if world > 1 else "single-gpu"},
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": launches, "clocks": clocks,
            "pct_of_peak": 100.0 * achieved / peaks["bf16_tflops"],
            "pct_of_clock_limited_peak": 100.0 * achieved / clock_peak,
            "parity": parity, "sustained": sustained, "configs": configs,
        }
        print(json.dumps(line), flush=True)
        bad = (parity is not None and not parity["ok"]) or \
            any(c.get("parity") and not c["parity"]["ok"] for c in (configs or []))
        if bad:
            sys.stderr.write("parity check against the oracle FAILED\n")
            return 3
    return 0


def run_suite(g, torch, np, peaks, suite_out, base):
    """The headline shape under the extended operations, timed (not part of
    the JSON line); written to suite_out after the configurations in `base`."""
    from dense_gemm_tensor_tcgen05_gb300 import inputs
    sig = 1 / math.sqrt(8192)
    # (dtype, dist, M, N, K, sigma, options): alpha/beta epilogue, transposed
    # storage of A and/or B, TF32, FP8, 16-bit C
    cfgs = [("bf16", "normal", 8192, 8192, 8192, sig, dict(alpha=0.5, beta=1.0)),
            ("bf16", "normal", 8192, 8192, 8192, sig, dict(trans_a=1)),
            ("bf16", "normal", 8192, 8192, 8192, sig, dict(trans_b=1)),
            ("bf16", "normal", 8192, 8192, 8192, sig, dict(trans_a=1, trans_b=1)),
            ("tf32", "normal", 8192, 8192, 8192, sig, dict(trans_b=1)),
            ("e4m3", "normal", 8192, 8192, 8192, sig, dict(trans_b=1)),
            ("e5m2", "normal", 8192, 8192, 8192, sig, dict(trans_b=1)),
            ("e4m3", "normal", 16384, 16384, 16384, 1 / 128, dict(trans_b=1)),
            ("bf16", "normal", 8192, 8192, 8192, sig, dict(c_dtype=2)),
            ("f16", "normal", 8192, 8192, 8192, sig, dict(c_dtype=1)),
            ("e4m3", "normal", 8192, 8192, 8192, sig, dict(trans_b=1, c_dtype=2))]
    fns = {"f16": g.gemm_f16f32, "bf16": g.gemm_bf16f32, "f32": g.sgemm_f32,
           "tf32": g.gemm_tf32f32_bt, "e4m3": g.gemm_e4m3f32_bt, "e5m2": g.gemm_e5m2f32_bt}
    codes = {"f16": 0, "bf16": 1, "f32": 2, "tf32": 3, "e4m3": 4, "e5m2": 5}
    ebytes = {"f16": 2, "bf16": 2, "f32": 4, "tf32": 4, "e4m3": 1, "e5m2": 1}
    # tensor-core peak per input type: the measured BF16 figure times the
    # nominal dense ratio (TF32 1.1, FP8 4.5 against BF16 2.25 PFLOP/s)
    tc_ratio = {"f16": 1.0, "bf16": 1.0, "tf32": 1.1 / 2.25, "e4m3": 2.0, "e5m2": 2.0}
    # FP32 on the CUDA cores: 152 SMs x 128 FMA lanes x 2 flops at 2.07 GHz
    fp32_peak = 152 * 128 * 2 * 2.07e9 / 1e12

    out = []
    stream = torch.cuda.Stream()
    sh = stream.cuda_stream
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    for dt, dist, m, n, k, sigma, opts in cfgs:
        A = inputs.make(dist, dt, m, k, 1, 0, sigma)
        B = inputs.make(dist, dt, k, n, 1, 1, sigma)
        ta, tb = opts.get("trans_a", 0), opts.get("trans_b", 0)
        if ta:
            A = np.ascontiguousarray(A.T)     # stored K x M
        if tb:
            B = np.ascontiguousarray(B.T)     # stored N x K
        Ad, Bd = to_device(A, dt), to_device(B, dt)
        del A, B
        Cd = torch.zeros((m, n), dtype=torch.float32, device="cuda")
        code = codes[dt]
        lda, ldb = (m if ta else k), (k if tb else n)
        args = (Ad.data_ptr(), Bd.data_ptr(), Cd.data_ptr(), m, n, k, lda, ldb, n)
        if code >= 3 and opts == {"trans_b": 1}:
            call = lambda: fns[dt](*args, sh)     # the _bt entry point
        elif opts:
            call = lambda: g.gemm_ex(*args, dtype=code, stream=sh, **opts)
        else:
            call = lambda: fns[dt](*args, sh)
        plan = g.gemm_plan_describe(code, *args, **opts)
        for _ in range(5):
            call()
        torch.cuda.synchronize()
        # warm: back to back, at least 100 ms
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        iters = 20
        while True:
            with torch.cuda.stream(stream):
                e0.record(stream)
                for _ in range(iters):
                    call()
                e1.record(stream)
            stream.synchronize()
            ms = e0.elapsed_time(e1)
            if ms >= 100 or iters >= 20000:
                break
            iters = int(iters * max(2.0, 110.0 / max(ms, 1e-3)))
        warm_ms = ms / iters
        # cold: L2 flushed (256 MiB write) before each timed launch
        cold = []
        for _ in range(10):
            with torch.cuda.stream(stream):
                flush.zero_()
                e0.record(stream)
                call()
                e1.record(stream)
            stream.synchronize()
            cold.append(e0.elapsed_time(e1))
        cold_ms = statistics.median(cold)
        g.gemm_device_error(sh)
        flop = 2.0 * m * n * k
        peak = fp32_peak if dt == "f32" else peaks["bf16_tflops"] * tc_ratio[dt]
        byts = (m * k + k * n) * ebytes[dt] + m * n * (2 if opts.get("c_dtype") else 4)
        if opts.get("beta"):
            byts += m * n * 4            # C is read as well
        out.append({"dtype": dt, "M": m, "N": n, "K": k, "options": opts, "plan": plan,
                    "warm_ms": warm_ms, "cold_ms": cold_ms,
                    "tflops_warm": flop / warm_ms / 1e9, "tflops_cold": flop / cold_ms / 1e9,
                    "gbs_warm": byts / warm_ms / 1e6, "gbs_cold": byts / cold_ms / 1e6,
                    "peak_tflops": peak,
                    "frac_peak_warm": flop / warm_ms / 1e9 / peak})
        del Ad, Bd, Cd
        torch.cuda.empty_cache()
    out_dir = os.path.dirname(os.path.abspath(suite_out))
    os.makedirs(out_dir, exist_ok=True)
    with open(suite_out, "w") as f:
        json.dump({"configs": base, "extended": out}, f, indent=1)
    for r in out:
        sys.stderr.write(json.dumps(r) + "\n")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--suite", action="store_true")
    ap.add_argument("--suite-out", default="bench_suite.json")
    ap.add_argument("--no-cpu-baseline", action="store_true",
                    help="skip the oracle leg (the CPU baseline and the parity checks)")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip timing the other workload configurations")
    ap.add_argument("--sustained-s", type=float, default=3.0,
                    help="length of the sustained back-to-back run (0: skip)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        return run_reference(args, rank, world)
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    try:
        return run_gb300(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
