"""Benchmark of the quantized-weight GEMM on one GB300 (or N replicas).

Workload (one step): the dense W4A16 asymmetric-INT4 sweep -- uint4 codes with uint4 zero
points and BF16 scales per group of 128, shapes N x K = 28672 x 8192 and 8192 x 28672,
M = 1, 2, 4, ..., 8192 -- 28 GEMM calls, each timed alone with CUDA events after an L2
flush (a 256 MiB device write, outside the events) and a ~0.1 ms device-side spin that
keeps host launch latency out of the events, mirroring the protocol of "Humming
wird angekündigt" (vLLM blog, German edition), section "Leistung".

value   = sum of 2*M*N*K over the step / sum of the event-timed call durations (TFLOP/s)
e2e     = the same calls through the public host-buffer entry point (qgemm_w4a16_host): X
          copied in from pinned host memory and Y copied back to pinned host memory inside the
          timed region, the copies overlapped with the GEMM chunk by chunk (mean over steps;
          the per-step times and each call's median sit beside it)
roofline: the dominant launch (the call with the largest share of the step time, a
          tensor-bound M = 8192 call): 2*M*N*K / its event time against the measured bf16
          peak; the HBM-bound small-M calls (M <= 16: weight + X + Y bytes / time against
          the measured copy bandwidth) are reported beside it
other_workloads: the MXFP4 W4A16, MXFP4 W4A8 (both packings: weights widened to e4m3 in
          registers, and e2m1 weights as FP4 tensor-core operands), W4A4, MXINT4 W4A16 and
          NVFP4 W4A16 sweeps and the MoE sweep (grouped, and the indexed gate_up), measured
          once after the timed region (--no-extra skips them)
cpu_baseline: the float64 numpy oracle on every host core (one single-threaded worker
          process per core) on a bounded sample of the workload

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the same CPU oracle on a bounded sample of the same workload.  Multi-GPU runs (torchrun) execute independent replicas (weak scaling);
the GEMM has no exchange step.
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "quantized GEMM TFLOP/s + weight GB/s vs M=1..8192, % of roofline (1 GB300)"
SHAPES = ((28672, 8192), (8192, 28672))
M_SWEEP = tuple(2 ** i for i in range(14))
GROUP = 128
WORKLOAD = ("dense W4A16 asymmetric INT4 (uint4 codes + uint4 zero points, BF16 scales, "
            "group 128), N x K in {28672 x 8192, 8192 x 28672}, M = 1..8192 (powers of two)")
FLUSH_BYTES = 256 * 1024 * 1024
HOLD_CYCLES = 200000            # ~0.1 ms device-side spin before each timed call
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def weight_bytes(N, K, g=GROUP):
    return N * K // 2 + N * (K // g) * 2 + N * (K // g) // 2


def alg_bytes(M, N, K):
    return weight_bytes(N, K) + M * K * 2 + M * N * 2


# DRAM bytes (read + write) per launch from one ncu capture of the same call, keyed by
# (N, K, M), with the digest of the kernel sources they were taken on; a changed kernel
# reports null until it is captured again.
CAPTURED_TRAFFIC = {
    # profiles/qgemm_tc_kernel_tile256_w4a16_28672x8192_m8192.md (ncu --set full, one launch of
    # the GEMM kernel; dram__bytes_read.sum + dram__bytes_write.sum)
    "csrc_sha256": "bea8d7d08313fc7b8e03235c2c9a5faf2484849ad4f6bcf0ff7639619a7dfecb",
    "launches": {"28672,8192,8192": 2359230000 + 462686464},
}


# Sources that define the GEMM kernel, its activation pre-pass and its launch plan (not the
# no-alloc or host-buffer wrappers).
GEMM_SOURCES = ("api.cu", "dequant.cuh", "gemm_a16_any.cu", "gemm_a16_mxfp4.cu",
                "gemm_a16_mxfp4f16.cu", "gemm_a16_mxint4.cu", "gemm_a16_nvfp4.cu",
                "gemm_a16_nvfp4f16.cu",
                "gemm_a16_sym_g1.cu",
                "gemm_a16_zp_g1.cu", "gemm_a4.cu", "gemm_a8.cu", "gemm_a8n.cu",
                "gemm_kernel.cuh", "kernels.h", "kernels_aux.cu", "ptx.cuh", "qgemm_internal.h")


def _code_only(text):
    """Source text without comments and blank space, so that comment edits keep the digest."""
    import re
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def csrc_digest():
    """sha256 over the code (comments and white space dropped) of the GEMM sources and the
    public header."""
    import hashlib
    h = hashlib.sha256()
    d = os.path.join(ROOT, "quantized_weight_gemm_gb300", "csrc")
    for f in sorted(os.listdir(d)):
        if f in GEMM_SOURCES:
            with open(os.path.join(d, f), encoding="utf-8") as fh:
                h.update(f.encode() + b"\0" + _code_only(fh.read()).encode())
    with open(os.path.join(ROOT, "include", "qgemm.h"), encoding="utf-8") as fh:
        h.update(_code_only(fh.read()).encode())
    return h.hexdigest()


def captured_traffic(N, K, M):
    if CAPTURED_TRAFFIC["csrc_sha256"] != csrc_digest():
        return None
    return CAPTURED_TRAFFIC["launches"].get(f"{N},{K},{M}")


def job_times(local, dist=None, device="cpu"):
    """The job's times: each entry of `local` as its slowest rank saw it (one MAX all_reduce;
    a job ends when its last rank does), or `local` itself on one rank."""
    if dist is None:
        return [float(v) for v in local]
    import torch
    t = torch.tensor([float(v) for v in local], device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t]


def job_value(ws, flops_step, ms):
    """Whole-job TFLOP/s: each of the ws ranks does flops_step per step (weak scaling) in the
    slowest rank's ms."""
    return ws * flops_step / (ms * 1e-3) / 1e12


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


# --------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples (every PERIOD_MS) of SM clock and throttle reasons during the
    timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    PERIOD_MS = 20

    def __init__(self, index):
        self.index = index
        self.proc = None

    def start(self):
        """Start sampling (before the warm-up, so the sampler is running when timing starts);
        each line read is stamped with the host clock by a reader thread."""
        import threading
        self.lines = []
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", str(self.PERIOD_MS)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return

        def reader():
            for line in self.proc.stdout:
                self.lines.append((time.perf_counter(), line))
        self.thread = threading.Thread(target=reader, daemon=True)
        self.thread.start()

    def stop(self, t0, t1):
        """Samples taken within the host-time window [t0, t1] of the timed region."""
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=5)
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ts, line in self.lines:
            if not (t0 <= ts <= t1):
                continue
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax = float(f[2])
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "samples": len(sm), "period_ms": self.PERIOD_MS, "reasons": sorted(reasons)}


# --------------------------------------------------------------------------- ours
def build_inputs(device):
    import numpy as np
    import torch
    import workloads as WL
    import quantized_weight_gemm_gb300 as qg

    cases = []
    for (N, K) in SHAPES:
        x, w = WL.int4_asym_shape(N, K, max(M_SWEEP), seed=0)
        d = qg.WeightDesc("uint4_zp", N, K, GROUP)
        packed = qg.repack(d, torch.from_numpy(w.codes).to(device),
                           torch.from_numpy(w.scales.view(np.int16)).to(device),
                           torch.from_numpy(w.zeros).to(device))
        X = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).to(device)
        Y = torch.empty(max(M_SWEEP), N, dtype=torch.bfloat16, device=device)
        ws = qg.workspace(d, max(M_SWEEP), device)
        staging = qg.host_staging(d, max(M_SWEEP), device)
        cases.append({"N": N, "K": K, "desc": d, "packed": packed, "X": X, "Y": Y, "ws": ws,
                      "staging": staging,
                      "x_host": torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).pin_memory(),
                      "y_host": torch.empty(max(M_SWEEP), N, dtype=torch.bfloat16).pin_memory()})
        del x, w
    torch.cuda.synchronize()
    if qg.device_status(clear=True) != 0:
        raise RuntimeError("repack reported a device error")
    return cases


def run_step(cases, flush, e2e=False):
    """One pass over the sweep; returns [(N, K, M, ms)] from CUDA events per call."""
    import torch
    import quantized_weight_gemm_gb300 as qg
    out = []
    st = torch.cuda.current_stream()
    for c in cases:
        for M in M_SWEEP:
            flush.zero_()
            if not e2e:
                # keep the GPU busy while the host enqueues the call, so that host-side
                # launch latency does not show up between the events of the kernel-only
                # timing; the end-to-end timing keeps it
                torch.cuda._sleep(HOLD_CYCLES)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(st)
            if e2e:
                # the public host-buffer call: X in from pinned host memory, Y back out, the
                # copies overlapped with the GEMM chunk by chunk
                qg.w4a16_host(c["desc"], c["packed"], c["x_host"][:M], out=c["y_host"][:M],
                              staging=c["staging"], ws=c["ws"])
            else:
                qg.w4a16(c["desc"], c["packed"], c["X"][:M], out=c["Y"][:M], ws=c["ws"])
            e1.record(st)
            out.append((c["N"], c["K"], M, e0, e1))
    torch.cuda.synchronize()
    return [(N, K, M, e0.elapsed_time(e1)) for (N, K, M, e0, e1) in out]


def host_copy_rates(device, nbytes=256 << 20, reps=3):
    """Pinned host <-> device copy rates of this machine in GB/s (best of `reps`), each direction
    alone and both at once on two streams: the ceiling that the e2e leg's copies work under."""
    import torch
    h = [torch.empty(nbytes, dtype=torch.uint8).pin_memory() for _ in range(2)]
    d = [torch.empty(nbytes, dtype=torch.uint8, device=device) for _ in range(2)]
    s = [torch.cuda.Stream(device=device) for _ in range(2)]

    def timed(fn):
        best = float("inf")
        for _ in range(reps):
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            fn()
            torch.cuda.synchronize()
            best = min(best, time.perf_counter() - t0)
        return best

    def both():
        with torch.cuda.stream(s[0]):
            d[0].copy_(h[0], non_blocking=True)
        with torch.cuda.stream(s[1]):
            h[1].copy_(d[1], non_blocking=True)

    t_h2d = timed(lambda: d[0].copy_(h[0], non_blocking=True))
    t_d2h = timed(lambda: h[1].copy_(d[1], non_blocking=True))
    t_both = timed(both)
    return {"h2d": round(nbytes / t_h2d / 1e9, 1), "d2h": round(nbytes / t_d2h / 1e9, 1),
            "both": round(2 * nbytes / t_both / 1e9, 1), "bytes_per_copy": nbytes}


_SLAB = None


def _oracle_worker(args):
    """One worker of the CPU baseline: draw two seeded 512-row slabs of the INT4 sweep's
    format and shape (K, M, group, distributions) once per process, then run the oracle on
    512-row chunks, cycling over them, for `seconds`; return (rows, seconds)."""
    global _SLAB
    wid, seconds = args
    import oracle
    import workloads as WL
    chunk, K, M = 512, 8192, 16
    if _SLAB is None:
        _SLAB = WL.int4_asym_shape(2 * chunk, K, M, seed=wid)
    x, w = _SLAB
    rows, t0, a = 0, time.perf_counter(), 0
    while time.perf_counter() - t0 < seconds:
        oracle.w4a16(x, w.wfmt, w.group, w.codes[a:a + chunk], w.scales[a:a + chunk],
                     w.zeros[a:a + chunk])
        rows += chunk
        a = chunk - a
    return rows, time.perf_counter() - t0


def _oracle_pool(seconds, workers):
    """Run _oracle_worker on `workers` spawned processes; print rows and wall time."""
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    with ctx.Pool(workers) as pool:
        pool.map(_oracle_worker, [(i, 0.5) for i in range(workers)])     # imports and inputs
        t0 = time.perf_counter()
        res = pool.map(_oracle_worker, [(i, seconds) for i in range(workers)])
        wall = time.perf_counter() - t0
    rows = sum(r for r, _ in res)
    print(json.dumps({"flops": 2.0 * 16 * rows * 8192, "seconds": wall, "rows": rows}))


def cpu_sample(seconds=12.0, workers=None):
    """Time the oracle, as it stands, on a bounded sample in a fresh process that runs one
    single-threaded worker process per host core; the rate is all workers' flops over the
    wall time."""
    if workers is None:
        workers = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    env = dict(os.environ)
    for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[v] = "1"
    code = (f"import sys; sys.path.insert(0, {ROOT!r}); import bench; "
            f"bench._oracle_pool({seconds}, {workers})")
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env,
                       timeout=900)
    if r.returncode != 0:
        raise RuntimeError("oracle sample failed: " + r.stderr[-2000:])
    d = json.loads(r.stdout.strip().splitlines()[-1])
    return {"value": d["flops"] / d["seconds"] / 1e12, "unit": "TFLOP/s", "cores": workers,
            "kind": "oracle",
            "sample": (f"float64 numpy oracle on the INT4 sweep's K = 8192, M = 16 (uint4 + "
                       f"zero points, group 128): {d['rows']} weight rows dequantized and "
                       f"multiplied in 512-row chunks by {workers} single-threaded worker "
                       f"processes (one per host core, each cycling over two seeded 512-row "
                       f"slabs), {d['seconds']:.1f} s of wall time")}


# --------------------------------------------------------------------------- other workloads
MX_SHAPES = ((4096, 7168), (7168, 2048))


def mx_weight_bytes(N, K):
    return N * K // 2 + N * K // 32


def time_one(fn, flush, reps=5, warm=3):
    """Median CUDA-event time (ms) of fn() after an L2 flush and a device spin."""
    import torch
    st = torch.cuda.current_stream()
    ts = []
    for i in range(warm + reps):
        flush.zero_()
        torch.cuda._sleep(HOLD_CYCLES)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(st)
        fn()
        e1.record(st)
        torch.cuda.synchronize()
        if i >= warm:
            ts.append(e0.elapsed_time(e1))
    return statistics.median(ts)


# Datasheet figures of one GB300, for the second roofline fraction of every row (the first
# is against the measured copy bandwidth and cuBLAS BF16 rate): HBM3e 7.9 TB/s, dense BF16
# 2.25 PFLOP/s (FP8 twice, FP4 six times that).
SPEC_HBM, SPEC_BF16 = 7.9e12, 2.25e15


def _spec_frac(ms, abytes, flops, factor=1.0):
    return round(max(abytes / SPEC_HBM, flops / (SPEC_BF16 * factor)) / (ms * 1e-3), 3)


def _row(N, K, M, ms, wbytes, abytes, flops, bw, tc, factor=1.0):
    rt = max(abytes / bw, flops / tc)
    return {"N": N, "K": K, "M": M, "us": round(ms * 1e3, 2),
            "tflops": round(flops / (ms * 1e-3) / 1e12, 2),
            "weight_gbs": round(wbytes / (ms * 1e-3) / 1e9, 1),
            "roofline_frac": round(rt / (ms * 1e-3), 3),
            "roofline_frac_spec": _spec_frac(ms, abytes, flops, factor),
            "bound": "hbm" if abytes / bw > flops / tc else "tensor"}


def sweep_mxfp4(device, flush, peaks, afmt):
    """The MXFP4 dense sweep: W4A16 (afmt "bf16": BF16 X) or W4A8 (per-token FP8 X with 1%
    outliers; afmt "fp8": weights widened to e4m3 in registers, "fp8n": weights as FP4
    tensor-core operands), N x K in {4096 x 7168, 7168 x 2048}, M = 1..8192."""
    fp8 = afmt != "bf16"
    import numpy as np
    import torch
    import workloads as WL
    import quantized_weight_gemm_gb300 as qg
    bw = peaks["hbm_gbs"] * 1e9
    tc = peaks["bf16_tflops"] * 1e12 * (2.0 if fp8 else 1.0)   # fp8 dense = 2x bf16 nominal
    rows = []
    Mmax = max(M_SWEEP)
    for (N, K) in MX_SHAPES:
        x, w = WL.mxfp4_shape(N, K, Mmax, seed=0, outliers=fp8)
        d = qg.WeightDesc("mxfp4", N, K, 32, afmt)
        packed = qg.repack(d, torch.from_numpy(w.codes).to(device),
                           torch.from_numpy(w.scales).to(device))
        X = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).to(device)
        Y = torch.empty(Mmax, N, dtype=torch.bfloat16, device=device)
        ws = qg.workspace(d, Mmax, device)
        if fp8:
            Xq, ts = qg.quant_act_fp8(X)
            Xq2, ts2 = torch.empty_like(Xq), torch.empty_like(ts)
        wb = mx_weight_bytes(N, K)
        for M in M_SWEEP:
            if fp8:
                ms = time_one(lambda: qg.w4a8(d, packed, Xq[:M], ts[:M], out=Y[:M], ws=ws), flush)
                ab = wb + M * K + 4 * M + M * N * 2
            else:
                ms = time_one(lambda: qg.w4a16(d, packed, X[:M], out=Y[:M], ws=ws), flush)
                ab = wb + M * K * 2 + M * N * 2
            r = _row(N, K, M, ms, wb, ab, 2.0 * M * N * K, bw, tc, 2.0 if fp8 else 1.0)
            if fp8:
                qms = time_one(lambda: qg.quant_act_fp8(X[:M], out=Xq2[:M], scale=ts2[:M]), flush)
                r["quant_act_us"] = round(qms * 1e3, 2)
            rows.append(r)
        del packed, X, Y, ws
    torch.cuda.synchronize()
    if qg.device_status(clear=True) != 0:
        raise RuntimeError("an MXFP4 GEMM reported a device error")
    return rows


def sweep_w4a4(device, flush, peaks):
    """Dense W4A4 (MXFP4 x MXFP4 on the block-scaled FP4 MMA), the MXFP4 shapes, M in
    M_SWEEP.  The activation quantization is a separate call, timed beside each GEMM as
    quant_act_us.  Tensor peak: the measured BF16 peak times 6, the nominal dense FP4 / BF16
    ratio of a GB300 (13.5 / 2.25 PFLOP/s)."""
    import numpy as np
    import torch
    import workloads as WL
    import quantized_weight_gemm_gb300 as qg
    bw = peaks["hbm_gbs"] * 1e9
    tc = peaks["bf16_tflops"] * 1e12 * 6.0
    rows = []
    Mmax = max(M_SWEEP)
    for (N, K) in MX_SHAPES:
        x, w = WL.mxfp4_shape(N, K, Mmax, seed=0, outliers=True)
        d = qg.WeightDesc("mxfp4", N, K, 32, "mxfp4")
        packed = qg.repack(d, torch.from_numpy(w.codes).to(device),
                           torch.from_numpy(w.scales).to(device))
        X = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).to(device)
        Xq, E = qg.quant_act_mxfp4(X)
        Xq2, E2 = torch.empty_like(Xq), torch.empty_like(E)
        Y = torch.empty(Mmax, N, dtype=torch.bfloat16, device=device)
        ws = qg.workspace(d, Mmax, device)
        wb = mx_weight_bytes(N, K)
        for M in M_SWEEP:
            ms = time_one(lambda: qg.w4a4(d, packed, Xq[:M], E[:M], out=Y[:M], ws=ws), flush)
            ab = wb + M * K // 2 + M * K // 32 + M * N * 2
            r = _row(N, K, M, ms, wb, ab, 2.0 * M * N * K, bw, tc, 6.0)
            qms = time_one(lambda: qg.quant_act_mxfp4(X[:M], out=Xq2[:M], exps=E2[:M]), flush)
            r["quant_act_us"] = round(qms * 1e3, 2)
            rows.append(r)
        del packed, X, Xq, E, Y, ws
    torch.cuda.synchronize()
    if qg.device_status(clear=True) != 0:
        raise RuntimeError("a W4A4 GEMM reported a device error")
    return rows


FMT_M = (1, 16, 128, 1024, 8192)


def sweep_w4a16_fmt(device, flush, peaks, wfmt):
    """Dense W4A16 on the MXINT4 (E8M0 per 32) or NVFP4 (E4M3 per 16 and a per-tensor
    scale) weight formats, N x K in {4096 x 7168, 7168 x 2048}, M in FMT_M."""
    import numpy as np
    import torch
    import workloads as WL
    import quantized_weight_gemm_gb300 as qg
    bw = peaks["hbm_gbs"] * 1e9
    tc = peaks["bf16_tflops"] * 1e12
    rows = []
    Mmax = max(FMT_M)
    for (N, K) in MX_SHAPES:
        r = WL.rng(0)
        x = WL.gen_x(r, Mmax, K)
        w = WL.gen_weights(r, wfmt, N, K)
        d = qg.WeightDesc(wfmt, N, K, w.group)
        packed = qg.repack(d, torch.from_numpy(w.codes).to(device),
                           torch.from_numpy(w.scales).to(device), global_scale=w.global_scale)
        X = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).to(device)
        Y = torch.empty(Mmax, N, dtype=torch.bfloat16, device=device)
        ws = qg.workspace(d, Mmax, device)
        wb = N * K // 2 + N * (K // w.group)
        for M in FMT_M:
            ms = time_one(lambda: qg.w4a16(d, packed, X[:M], out=Y[:M], ws=ws), flush)
            rows.append(_row(N, K, M, ms, wb, wb + M * K * 2 + M * N * 2, 2.0 * M * N * K, bw, tc))
        del packed, X, Y, ws
    torch.cuda.synchronize()
    if qg.device_status(clear=True) != 0:
        raise RuntimeError(f"a {wfmt} GEMM reported a device error")
    return rows


def sweep_moe(device, flush, peaks):
    """The MoE layer (E = 256 MXFP4 experts, top-8, hidden 7168, intermediate 2048):
    gate_up [4096 x 7168] and down [7168 x 2048] grouped GEMMs over expert-sorted rows,
    T in {1, 16, 128, 1024, 8192}, uniform and skewed routing; each GEMM timed alone.  The
    gate_up GEMM is also timed on the indexed path (token-order X gathered by index, with
    the indexed workspace: from 256 rows on the call gathers into it and runs the grouped
    kernel), reported as gate_up_indexed_us beside the grouped time."""
    import numpy as np
    import torch
    import workloads as WL
    import quantized_weight_gemm_gb300 as qg
    E, H, I = WL.MOE_E, WL.MOE_HIDDEN, WL.MOE_INTER
    shapes = {"gate_up": (2 * I, H, 0), "down": (H, I, 1)}
    descs, packs = {}, {}
    for name, (N, K, seed) in shapes.items():
        d = qg.WeightDesc("mxfp4", N, K, 32)
        nb = qg.packed_bytes(d)
        p = torch.empty(nb * E, dtype=torch.uint8, device=device)
        for e, w in enumerate(WL.iter_moe_weights(E, N, K, seed=seed)):
            qg.repack(d, torch.from_numpy(w.codes).to(device), torch.from_numpy(w.scales).to(device),
                      None, out=p[e * nb:(e + 1) * nb])
        descs[name], packs[name] = d, p
    bw = peaks["hbm_gbs"] * 1e9
    tc = peaks["bf16_tflops"] * 1e12
    rows = []
    for skewed in (False, True):
        for T in WL.MOE_T:
            case = WL.moe_case(T, seed=0, skewed=skewed)
            off = torch.from_numpy(np.asarray(case.offsets, dtype=np.int32)).to(device)
            R = len(case.valid)
            valid = int(case.valid.sum())
            active = int((np.asarray(case.counts) > 0).sum())
            ins = {"gate_up": case.x_bits, "down": case.down_bits}
            r = {"T": T, "skewed": skewed, "rows": R, "active_experts": active}
            tot_ms, tot_flops, tot_w, tot_b = 0.0, 0.0, 0, 0
            for name, (N, K, _) in shapes.items():
                X = torch.from_numpy(ins[name].view(np.int16)).view(torch.bfloat16).to(device)
                Y = torch.empty(R, N, dtype=torch.bfloat16, device=device)
                d, p = descs[name], packs[name]
                wsp = qg.moe_workspace(d, E, R, device=device)
                ms = time_one(lambda: qg.moe_grouped(d, p, E, X, off, out=Y, ws=wsp), flush)
                wb = active * mx_weight_bytes(N, K)
                r[name + "_us"] = round(ms * 1e3, 2)
                tot_ms += ms
                tot_flops += 2.0 * valid * N * K
                tot_w += wb
                tot_b += wb + valid * K * 2 + valid * N * 2
            # the same gate_up GEMM on the indexed path: X in token order [T, hidden], rows
            # gathered by index (padding positions -1), no sorted copy of X from the caller
            N, K, _ = shapes["gate_up"]
            Xt = torch.from_numpy(case.x_tok_bits.view(np.int16)).view(torch.bfloat16).to(device)
            idx = torch.from_numpy(case.token_of_row.astype(np.int32)).to(device)
            Y = torch.empty(R, N, dtype=torch.bfloat16, device=device)
            d, p = descs["gate_up"], packs["gate_up"]
            wsp = qg.moe_indexed_workspace(d, E, T, R, device=device)
            ms = time_one(lambda: qg.moe_indexed(d, p, E, Xt, off, idx, out=Y, ws=wsp), flush)
            r["gate_up_indexed_us"] = round(ms * 1e3, 2)
            del wsp
            r.update({"us": round(tot_ms * 1e3, 2),
                      "tflops": round(tot_flops / (tot_ms * 1e-3) / 1e12, 2),
                      "weight_gbs": round(tot_w / (tot_ms * 1e-3) / 1e9, 1),
                      "roofline_frac": round(max(tot_b / bw, tot_flops / tc) / (tot_ms * 1e-3), 3),
                      "roofline_frac_spec": _spec_frac(tot_ms, tot_b, tot_flops)})
            rows.append(r)
    torch.cuda.synchronize()
    if qg.device_status(clear=True) != 0:
        raise RuntimeError("an MoE GEMM reported a device error")
    return rows


def bench_ours(args):
    import torch
    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    dist = None
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    import __graft_entry__ as ge
    ge.build()
    import quantized_weight_gemm_gb300 as qg
    peaks, peak_kind = load_peaks()
    device = torch.device("cuda", local)
    cases = build_inputs(device)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=device)

    sampler = ClockSampler(local)
    sampler.start()
    for _ in range(args.warmup):
        run_step(cases, flush)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    steps = [run_step(cases, flush) for _ in range(args.steps)]
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    t1 = time.perf_counter()
    wall = t1 - t0
    clocks = sampler.stop(t0, t1)
    # end-to-end leg: the same warm-up as the kernel-only leg, then the timed steps.  The
    # host enqueues every call while the GPU runs, so a pause of this Python harness lands
    # inside a call's events; the garbage collector is held off while the warm-up and the
    # timed steps run (as timeit does), its pauses of about 0.2 ms being the harness's, not
    # the library's, and the one collection before them lies outside both.
    import gc
    gc.collect()
    gc.disable()
    try:
        for _ in range(args.warmup):
            run_step(cases, flush, e2e=True)
        e2e_steps = [run_step(cases, flush, e2e=True) for _ in range(max(1, args.steps))]
        torch.cuda.synchronize()
    finally:
        gc.enable()
    copy_gbs = host_copy_rates(device)
    extra = None
    if not args.no_extra:
        del cases
        torch.cuda.empty_cache()
        extra = {"mxfp4_a16": sweep_mxfp4(device, flush, peaks, "bf16"),
                 "mxfp4_a8": sweep_mxfp4(device, flush, peaks, "fp8"),
                 "mxfp4_a8n": sweep_mxfp4(device, flush, peaks, "fp8n"),
                 "w4a4": sweep_w4a4(device, flush, peaks),
                 "mxint4_a16": sweep_w4a16_fmt(device, flush, peaks, "mxint4"),
                 "nvfp4_a16": sweep_w4a16_fmt(device, flush, peaks, "nvfp4"),
                 "moe": sweep_moe(device, flush, peaks)}
    if qg.device_status(clear=True) != 0:
        raise RuntimeError("a GEMM reported a device error")

    flops_step = sum(2.0 * M * N * K for (N, K) in SHAPES for M in M_SWEEP)
    step_ms = [sum(r[3] for r in s) for s in steps]
    e2e_ms = [sum(r[3] for r in s) for s in e2e_steps]
    local_ms = statistics.mean(step_ms)
    local_e2e = statistics.mean(e2e_ms)
    local_ms, local_e2e = job_times([local_ms, local_e2e], dist, device)
    value = job_value(ws, flops_step, local_ms)
    e2e_value = job_value(ws, flops_step, local_e2e)

    # per-call table (median over steps), with each call's end-to-end time beside it
    per, per_e2e = {}, {}
    for s in steps:
        for (N, K, M, ms) in s:
            per.setdefault((N, K, M), []).append(ms)
    for s in e2e_steps:
        for (N, K, M, ms) in s:
            per_e2e.setdefault((N, K, M), []).append(ms)
    bw = peaks["hbm_gbs"] * 1e9
    tc = peaks["bf16_tflops"] * 1e12
    sweep = []
    for (N, K, M), v in sorted(per.items(), key=lambda kv: (kv[0][0], kv[0][2])):
        ms = statistics.median(v)
        rt = max(alg_bytes(M, N, K) / bw, 2.0 * M * N * K / tc)
        sweep.append({"N": N, "K": K, "M": M, "us": round(ms * 1e3, 2),
                      "tflops": round(2.0 * M * N * K / (ms * 1e-3) / 1e12, 2),
                      "weight_gbs": round(weight_bytes(N, K) / (ms * 1e-3) / 1e9, 1),
                      "roofline_frac": round(rt / (ms * 1e-3), 3),
                      "roofline_frac_spec": _spec_frac(ms, alg_bytes(M, N, K), 2.0 * M * N * K),
                      "bound": "hbm" if alg_bytes(M, N, K) / bw > 2.0 * M * N * K / tc else "tensor",
                      "e2e_us": round(statistics.median(per_e2e[(N, K, M)]) * 1e3, 2)})
    # dominant launch: the call with the largest share of the step's time
    dom = max(sweep, key=lambda r: r["us"])
    dom_flops = 2.0 * dom["M"] * dom["N"] * dom["K"]
    achieved_tc = dom_flops / (dom["us"] * 1e-6) / 1e12
    small = [r for r in sweep if r["M"] <= 16]
    small_time = sum(r["us"] for r in small) * 1e-6
    small_bytes = sum(alg_bytes(r["M"], r["N"], r["K"]) for r in small)
    achieved_bw = small_bytes / small_time / 1e9
    traffic = captured_traffic(dom["N"], dom["K"], dom["M"])
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(local_ms, 3),
        "wall_ms_per_step": round(wall * 1e3 / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded: X ~ N(0,1) bf16, uint4 codes U[0,15], zero points U[6,9], "
                "scales U[0.005,0.02] bf16)",
        "config": {"workload": WORKLOAD, "shapes": [list(s) for s in SHAPES], "M": list(M_SWEEP),
                   "l2": "flushed before every timed call (256 MiB device write outside the events)",
                   "launch": "0.1 ms device spin before each call so host latency is not timed",
                   "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU"},
        "impl": "ours",
        "roofline": {"bound": dom["bound"], "achieved": round(achieved_tc, 1),
                     "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                     "frac": round(achieved_tc / peaks["bf16_tflops"], 3), "traffic": traffic,
                     "frac_spec": round(achieved_tc * 1e12 / SPEC_BF16, 3),
                     "kernel": (f"qgemm_tc_kernel, 256-token tile, uint4+zp on FP16 operands "
                                f"(the call's time includes its FP16 activation pre-pass): the "
                                f"N={dom['N']} K={dom['K']} M={dom['M']} call, "
                                f"{dom['us'] / sum(r['us'] for r in sweep):.0%} of the step"),
                     "algorithmic": "2*M*N*K flops per launch",
                     "peak_source": f"bf16_tflops (burst; each call is timed alone) of {peak_kind}"},
        "roofline_small_m": {"bound": "hbm", "achieved": round(achieved_bw, 1),
                             "peak": peaks["hbm_gbs"], "unit": "GB/s",
                             "frac": round(achieved_bw / peaks["hbm_gbs"], 3),
                             "frac_spec": round(achieved_bw * 1e9 / SPEC_HBM, 3),
                             "kernel": "qgemm_tc_kernel<16, bf16> (M <= 16 calls, split-K)",
                             "peak_source": f"hbm_gbs of {peak_kind}"},
        "sweep": sweep,
        "e2e": {"value": round(e2e_value, 2), "unit": "TFLOP/s",
                "h2d_bytes_per_step": sum(M * K * 2 for (N, K) in SHAPES for M in M_SWEEP),
                "d2h_bytes_per_step": sum(M * N * 2 for (N, K) in SHAPES for M in M_SWEEP),
                "host_copy_gbs": copy_gbs,
                # value is the mean over steps; the steps themselves show any outliers
                "step_ms": [round(v, 3) for v in e2e_ms],
                "median_step_ms": round(statistics.median(e2e_ms), 3)},
        # each call: the FP16 activation pre-pass and the GEMM
        "gpu_launches": 2 * len(SHAPES) * len(M_SWEEP) * args.steps,
        "clocks": clocks,
    }
    if extra is not None:
        line["other_workloads"] = {
            "note": ("measured once after the timed region, each call alone with a cold L2 "
                     "(median of 5); not part of value"),
            "mxfp4_a16": {"workload": "dense W4A16 MXFP4, N x K in {4096 x 7168, 7168 x 2048}",
                          "sweep": extra["mxfp4_a16"]},
            "w4a4": {"workload": ("dense W4A4 MXFP4 x MXFP4 (E8M0 per 32 on both operands; "
                                  "activations with 1% outliers x20, quantized by a separate "
                                  "call timed as quant_act_us), N x K in {4096 x 7168, "
                                  "7168 x 2048}"),
                     "tensor_peak": "measured BF16 x 6 (nominal dense FP4 / BF16)",
                     "sweep": extra["w4a4"]},
            "mxfp4_a8": {"workload": ("dense W4A8 MXFP4 x per-token FP8 e4m3 (1% outliers x20), "
                                      "same shapes; quant_act_us = the separate quantization call; "
                                      "roofline tensor peak = 2 x measured bf16"),
                         "sweep": extra["mxfp4_a8"]},
            "mxfp4_a8n": {"workload": ("dense W4A8 as mxfp4_a8, the e2m1 weights fed to the "
                                       "tensor core as FP4 operands of the block-scaled "
                                       "FP8/FP6/FP4 MMA (no register decode)"),
                          "sweep": extra["mxfp4_a8n"]},
            "mxint4_a16": {"workload": ("dense W4A16 MXINT4 (two's-complement nibbles, E8M0 per "
                                        "32), same shapes"),
                           "sweep": extra["mxint4_a16"]},
            "nvfp4_a16": {"workload": ("dense W4A16 NVFP4 (e2m1, E4M3 per 16, float32 "
                                       "per-tensor scale), same shapes"),
                          "sweep": extra["nvfp4_a16"]},
            "moe": {"workload": ("MoE grouped W4A16 MXFP4, E=256 top-8, gate_up 4096 x 7168 + "
                                 "down 7168 x 2048, expert-sorted rows padded to 8; flops and "
                                 "bytes on routed (unpadded) rows and active experts"),
                    "sweep": extra["moe"]}}
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_sample()
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def bench_case(args):
    """One GEMM shape, timed alone (profiling aid): --case N,K,M[,wfmt[,afmt]]."""
    import numpy as np
    import torch
    import workloads as WL
    import __graft_entry__ as ge
    ge.build()
    import quantized_weight_gemm_gb300 as qg
    parts = args.case.split(",")
    N, K, M = int(parts[0]), int(parts[1]), int(parts[2])
    wfmt = parts[3] if len(parts) > 3 else "uint4_zp"
    afmt = parts[4] if len(parts) > 4 else "bf16"
    r = WL.rng(0)
    x = WL.gen_x(r, M, K, outliers=afmt != "bf16")
    w = WL.gen_weights(r, wfmt, N, K)
    d = qg.WeightDesc(wfmt, N, K, w.group, afmt)
    scales = torch.from_numpy(w.scales.view(np.int16) if w.scales.dtype == np.uint16 else w.scales)
    packed = qg.repack(d, torch.from_numpy(w.codes).cuda(), scales.cuda(),
                       None if w.zeros is None else torch.from_numpy(w.zeros).cuda())
    X = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).cuda()
    if afmt in ("fp8", "fp8n"):
        Xq, ts = qg.quant_act_fp8(X)
    elif afmt == "mxfp4":
        Xq, xe = qg.quant_act_mxfp4(X)
    ws = qg.workspace(d, M)
    Y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    times = []
    for i in range(args.warmup + args.steps):
        flush.zero_()
        torch.cuda._sleep(HOLD_CYCLES)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        if afmt in ("fp8", "fp8n"):
            qg.w4a8(d, packed, Xq, ts, out=Y, ws=ws)
        elif afmt == "mxfp4":
            qg.w4a4(d, packed, Xq, xe, out=Y, ws=ws)
        else:
            qg.w4a16(d, packed, X, out=Y, ws=ws)
        e1.record()
        torch.cuda.synchronize()
        if i >= args.warmup:
            times.append(e0.elapsed_time(e1))
    st = qg.device_status(clear=True)
    if st != 0:
        raise RuntimeError(f"device status {st}")
    ms = statistics.median(times)
    wb = qg.packed_bytes(d)
    print(json.dumps({"case": args.case, "us": round(ms * 1e3, 2),
                      "tflops": round(2.0 * M * N * K / (ms * 1e-3) / 1e12, 1),
                      "weight_gbs": round(wb / (ms * 1e-3) / 1e9, 1)}), flush=True)


def bench_moe_case(args):
    """One MoE GEMM of the 256-expert layer, timed alone (profiling aid):
    --moe T,gate_up|down[,skewed][,indexed][,E<experts>][,top<k>] -- fewer experts (and a
    smaller top-k) keep the rows per expert, and so the kernel's tiles, of the full layer
    with a fraction of its weights on the device."""
    import numpy as np
    import torch
    import workloads as WL
    import __graft_entry__ as ge
    ge.build()
    import quantized_weight_gemm_gb300 as qg
    parts = args.moe.split(",")
    T, gemm = int(parts[0]), parts[1]
    skewed, indexed = "skewed" in parts[2:], "indexed" in parts[2:]
    E_opt = [int(p[1:]) for p in parts[2:] if p.startswith("E")]
    k_opt = [int(p[3:]) for p in parts[2:] if p.startswith("top")]
    case = WL.moe_case(T, seed=0, skewed=skewed, E=E_opt[0] if E_opt else WL.MOE_E,
                       topk=k_opt[0] if k_opt else WL.MOE_TOPK)
    N, K = (2 * WL.MOE_INTER, WL.MOE_HIDDEN) if gemm == "gate_up" else (WL.MOE_HIDDEN, WL.MOE_INTER)
    E, R = case.E, len(case.token_of_row)
    d = qg.WeightDesc("mxfp4", N, K, 32, "bf16")
    nb = qg.packed_bytes(d)
    packed = torch.empty(nb * E, dtype=torch.uint8, device="cuda")
    for e, w in enumerate(WL.iter_moe_weights(E, N, K, seed=0)):
        qg.repack(d, torch.from_numpy(w.codes).cuda(), torch.from_numpy(w.scales).cuda(), None,
                  out=packed[e * nb:(e + 1) * nb])
    off = torch.tensor(case.offsets, device="cuda")
    if indexed:
        X = torch.from_numpy(case.x_tok_bits.view(np.int16)).view(torch.bfloat16).cuda()
        idx = torch.tensor(case.token_of_row.astype(np.int32), device="cuda")
        call = lambda: qg.moe_indexed(d, packed, E, X, off, idx, out=Y, ws=wsp)
    else:
        xb = case.x_bits if gemm == "gate_up" else case.down_bits
        X = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).cuda()
        call = lambda: qg.moe_grouped(d, packed, E, X, off, out=Y, ws=wsp)
    wsp = qg.moe_indexed_workspace(d, E, case.T, R) if indexed else qg.moe_workspace(d, E, R)
    Y = torch.empty(R, N, dtype=torch.bfloat16, device="cuda")
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    times = []
    for i in range(args.warmup + args.steps):
        flush.zero_()
        torch.cuda._sleep(HOLD_CYCLES)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        call()
        e1.record()
        torch.cuda.synchronize()
        if i >= args.warmup:
            times.append(e0.elapsed_time(e1))
    st = qg.device_status(clear=True)
    if st != 0:
        raise RuntimeError(f"device status {st}")
    ms = statistics.median(times)
    active = int(np.count_nonzero(case.counts))
    print(json.dumps({"moe": args.moe, "us": round(ms * 1e3, 2), "active_experts": active,
                      "weight_gbs": round(active * nb / (ms * 1e-3) / 1e9, 1)}), flush=True)


def bench_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    for _ in range(args.warmup):
        cpu_sample(seconds=2.0)
    t0 = time.perf_counter()
    samples = [cpu_sample(seconds=8.0) for _ in range(args.steps)]
    wall = time.perf_counter() - t0
    v = statistics.mean(s["value"] for s in samples)
    cb = dict(samples[-1])
    cb["value"] = round(v, 6)
    line = {
        "metric": METRIC, "value": round(v, 6), "unit": "TFLOP/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(wall * 1e3 / args.steps, 1), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "shapes": [list(s) for s in SHAPES], "M": list(M_SWEEP),
                   "l2": "n/a (CPU)", "parallelism": "single process"},
        "impl": "reference", "cpu_baseline": cb,
        "e2e": {"value": round(v, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the MXFP4, W4A8 and MoE sweeps reported beside the main line")
    ap.add_argument("--case", default=None, help="N,K,M[,wfmt[,afmt]]: time one GEMM shape")
    ap.add_argument("--moe", default=None,
                    help="T,gate_up|down[,skewed][,indexed][,E<experts>][,top<k>]: time one MoE GEMM of the layer")
    args = ap.parse_args()
    if args.case:
        bench_case(args)
    elif args.moe:
        bench_moe_case(args)
    elif args.impl == "reference":
        bench_reference(args)
    else:
        bench_ours(args)


if __name__ == "__main__":
    main()
