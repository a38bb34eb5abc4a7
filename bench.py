#!/usr/bin/env python
"""IQ4_XS x Q8_1 batched-matmul benchmark on GB300.

Workload (default): the 4096 x 4096 square projection swept over the decode /
verify batch sizes M = 1, 2, 4, 8, 12, 16, 32, 64, 96.  One step is one pass
of the hot path over that sweep: for every M, Q8_1-quantize a fresh resident
activation batch x [M, 4096] and run the batched matmul (path chosen by the
library's dispatcher) against one of 45 resident copies of W, rotating so the
streamed weights (401 MB) exceed the 129 MB L2 several times over.  Each
step is one CUDA-graph replay of those 18 launches.

Metric: whole-job GB/s = algorithmic bytes of the step / step time, where a
matmul moves 0.53125*N*K (IQ4_XS W) + 1.125*M*K (Q8_1 x) + 4*M*N (y) bytes and
a quantization 4*M*K in + 1.125*M*K out.  TOPS (2*M*N*K per matmul) and a
per-M breakdown come alongside.  ``e2e`` repeats the step through the public
Python/C-ABI calls on pinned host buffers (the kernels read x from and write
y to host memory every step; the explicit-copy form is reported beside it).  ``--impl reference`` times the CPU oracle on a bounded sample of the
same workload instead.

Under torchrun (N > 1) every rank runs its own replica (the path shards into
independent problems; no collective is on the data path) and rank 0 prints
the aggregate.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "IQ4_XS×Q8_1 matmul GB/s and TOPS vs GB300 roofline, M=1..96"
UNIT = "GB/s"
N_COPIES = 45
FALLBACK_HBM_GBS = 6800.0
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "matmul_square4096_traffic.txt")
# Sources of the kernels whose DRAM traffic is recorded, per kernel path
# (2 = tcgen05, 4 = warp-level MMA).
KERNEL_SOURCES = {
    2: ("iq4_xs_quantized_gb300/csrc/matmul_tc.cu", "iq4_xs_quantized_gb300/csrc/internal.cuh"),
    4: ("iq4_xs_quantized_gb300/csrc/matmul_mma.cu", "iq4_xs_quantized_gb300/csrc/internal.cuh"),
}
TRAFFIC_PREFIX = {2: "", 4: "mma."}  # key prefix of each kernel's entries in TRAFFIC_FILE
PATH_NAMES = {1: "dp4a", 2: "tc (prepared operand)", 4: "mma (warp-level tensor cores)"}
KERNEL_NAMES = {1: "matmul_dp4a_kernel (CUDA cores)", 2: "matmul_tc_kernel (tcgen05, prepared-operand form)",
                4: "matmul_mma_kernel (warp-level mma.sync, decode into registers)"}


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ms", default=None,
                    help="comma-separated subset of the M sweep (profiling runs only)")
    ap.add_argument("--shape", default=None,
                    help="N,K: another weight shape instead of the square 4096 one (profiling runs "
                         "only; the weights and activations come from the same seeded generators)")
    ap.add_argument("--no-pdl", action="store_true",
                    help="launch without programmatic dependent launch (for serialised profilers)")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the dequantize+GEMM baseline and the decode-stream workload")
    ap.add_argument("--formats-only", action="store_true",
                    help="profiling runs only: time the Q4_0 / IQ4_NL matmuls (square, or --shape; --ms), "
                         "print their line and stop")
    ap.add_argument("--moe-tokens", type=int, default=None,
                    help="profiling runs only: time the grouped MoE layer at this many tokens, "
                         "print its line and stop")
    return ap.parse_args()


# --------------------------------------------------------------------------- bytes
def matmul_bytes(M, N, K):
    return N * (K // 256) * 136 + M * K + M * (K // 32) * 4 + 4 * M * N


def quantize_bytes(M, K):
    return 4 * M * K + M * K + M * (K // 32) * 4


def step_bytes(ms, N, K):
    return sum(matmul_bytes(M, N, K) + quantize_bytes(M, K) for M in ms)


def step_ops(ms, N, K):
    return sum(2 * M * N * K for M in ms)


def hbm_peak_gbs():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


FALLBACK_BF16_TFLOPS = 1900.0


def tensor_peak_tflops():
    """Dense fp16/bf16 tensor peak (TFLOP/s), burst: the tcgen05 kernel runs
    kind::f16 MMAs on fp16 operands, whose dense rate is the bf16 rate."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["bf16_tflops"]), "measured (bf16 burst = fp16 dense rate)"
    except Exception:
        return FALLBACK_BF16_TFLOPS, "fallback"


def tc_executed_flops(M, N, K):
    """Floating-point work the tensor cores execute for one tcgen05 launch:
    128-row tiles x activation tiles padded to 16 rows (at most 128), two
    128 x MT x 16 MMAs per 32-weight sub-block (exact fp16 integers)."""
    mt = min(128, (M + 15) // 16 * 16)
    mtiles = -(-M // mt)
    return 2 * (-(-N // 128) * 128) * (mtiles * mt) * K


def mma_executed_flops(M, N, K):
    """Floating-point work of one warp-MMA launch: m16n8k16 MMAs over the
    weight rows (16-row fragments) x activation tiles of 8, 16, 24 or 32
    rows (M above 32 in tiles of 32)."""
    mt = min(32, -(-M // 8) * 8)
    mtiles = -(-M // mt)
    return 2 * (-(-N // 16) * 16) * (mtiles * mt) * K


def executed_flops(path, M, N, K):
    return mma_executed_flops(M, N, K) if path == 4 else tc_executed_flops(M, N, K)


ROOFLINE_SLACK = 1.10


def roofline_gate(items, peak_gbs, slack=ROOFLINE_SLACK):
    """items: (name, algorithmic bytes, seconds).  A call reported faster
    than its bytes allow (more than `slack` x the measured HBM rate) did not
    do its work; every such call is listed."""
    bad = []
    for name, nbytes, sec in items:
        gbs = nbytes / sec / 1e9 if sec > 0 else float("inf")
        if gbs > slack * peak_gbs:
            bad.append({"call": name, "GBps": round(gbs, 1)})
    return {"slack": slack, "peak_gbs": peak_gbs, "checked": len(items), "violations": bad,
            "ok": not bad}


def kernel_source_hash(path=2):
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES[path]:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_counters(path=2):
    """Per matmul launch of the kernel on `path` (mean over the sweep's M on
    that path) from the committed ncu summary: DRAM bytes and warp
    instructions executed.  Empty if absent or taken on different kernel
    sources."""
    try:
        pre = TRAFFIC_PREFIX[path]
        vals = {}
        with open(TRAFFIC_FILE) as f:
            for line in f:
                if ":" in line and not line.startswith("#"):
                    k, v = line.split(":", 1)
                    vals[k.strip()] = v.strip()
        if vals.get(pre + "kernel_source_sha256_16") != kernel_source_hash(path):
            return {}
        out = {"dram_bytes": float(vals[pre + "dram_bytes_per_tc_launch_mean"])}
        if pre + "inst_executed_per_tc_launch_mean" in vals:
            out["inst"] = float(vals[pre + "inst_executed_per_tc_launch_mean"])
        return out
    except Exception:
        return {}


def recorded_traffic(path=2):
    return recorded_counters(path).get("dram_bytes")


# ------------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for name, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(name)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ distributed
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(value: float, world: int) -> float:
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------- CPU oracle leg
def oracle_sample(rows: int, threads: int, min_seconds: float = 0.0):
    """Time the CPU oracle (as it stands) on the square workload restricted to
    the first `rows` weight rows, every M of the sweep, repeating the sweep
    until `min_seconds` have passed.  Returns (GB/s, seconds, description)."""
    import oracle
    from iq4_xs_quantized_gb300 import synth
    W = synth.SQUARE
    N, K = W.shapes[0]
    w, x = W.inputs(0)
    wr = np.ascontiguousarray(w[:rows])
    orc = oracle.get()
    passes = 0
    t0 = time.perf_counter()
    while True:
        for M in W.ms:
            qs, d_h, _ = orc.quantize_q8_1(x[:M])
            orc.matmul(wr, rows, K, qs, d_h, nthreads=threads)
        passes += 1
        dt = time.perf_counter() - t0
        if dt >= min_seconds:
            break
    nbytes = passes * step_bytes(W.ms, rows, K)
    desc = (f"weight rows 0..{rows - 1} of 4096 (K=4096), all M in {list(W.ms)}, "
            f"quantize + matmul, {passes} pass(es), {threads} threads")
    return nbytes / dt / 1e9, dt, desc


def oracle_per_config(min_seconds: float = 2.0):
    """The oracle single-threaded on the tiny configuration (all of it: 256 x
    1024, M = 1, 4, 8) and on a 64-row sample of the square one (every M),
    as GB/s of each workload's algorithmic bytes."""
    import oracle
    from iq4_xs_quantized_gb300 import synth
    orc = oracle.get()
    out = []
    for W, rows in ((synth.TINY, None), (synth.SQUARE, 64)):
        N, K = W.shapes[0]
        w, x = W.inputs(0)
        n = N if rows is None else rows
        wr = np.ascontiguousarray(w[:n])
        passes, t0 = 0, time.perf_counter()
        while True:
            for M in W.ms:
                qs, d_h, _ = orc.quantize_q8_1(x[:M])
                orc.matmul(wr, n, K, qs, d_h, nthreads=1)
            passes += 1
            dt = time.perf_counter() - t0
            if dt >= min_seconds:
                break
        out.append({"workload": W.name, "rows": n, "of_rows": N, "ms": list(W.ms), "threads": 1,
                    "GBps": round(passes * step_bytes(W.ms, n, K) / dt / 1e9, 4),
                    "seconds": round(dt, 2)})
    return out


def run_reference(args, world, rank):
    if rank != 0:
        return
    import oracle
    threads = oracle.threads_available()
    rows = 256
    oracle_sample(16, threads)  # build, page in
    for _ in range(min(args.warmup, 1)):
        oracle_sample(rows, threads)
    vals, secs = [], 0.0
    for _ in range(args.steps):
        v, dt, desc = oracle_sample(rows, threads)
        vals.append(v)
        secs += dt
        if secs > 120:
            break
    value = len(vals) * step_bytes((1, 2, 4, 8, 12, 16, 32, 64, 96), rows, 4096) / secs / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": len(vals), "warmup": args.warmup,
        "ms_per_step": secs / len(vals) * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "int32 dot / f64 accumulate (CPU oracle)",
        "data": "synthetic",
        "config": {"workload": "square_4096x4096, M=1..96 sweep (quantize + matmul per M)",
                   "N": 4096, "K": 4096, "ms": [1, 2, 4, 8, 12, 16, 32, 64, 96],
                   "sample_rows": rows},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "same_config": ("the square 4096 x 4096 sweep on a 256-row sample of W (the oracle's "
                        "rate per byte; the GPU arm runs all 4096 rows)"),
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------- our GPU leg
def run_ours(args, world, rank, local):
    import torch

    from iq4_xs_quantized_gb300 import binding as B
    from iq4_xs_quantized_gb300 import build, synth

    build.build()
    B.load()
    B.iq4xs_set_pdl(not args.no_pdl)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if args.moe_tokens:
        res = moe_grouped(torch, B, dev, layers=2, reps=2, tokens=(args.moe_tokens,))
        if rank == 0:
            print(json.dumps({"moe_grouped": res}), flush=True)
        return
    if args.formats_only:
        fN, fK = (int(v) for v in args.shape.split(",")) if args.shape else (4096, 4096)
        fms = tuple(int(v) for v in args.ms.split(",")) if args.ms else (1, 4, 8, 16, 64, 96)
        res = weight_formats(torch, B, dev, torch.cuda.Stream(device=dev), {}, N=fN, K=fK, ms=fms)
        if rank == 0:
            print(json.dumps({"weight_formats": res}), flush=True)
        return
    W = synth.SQUARE
    N, K = W.shapes[0]
    ms = list(W.ms) if not args.ms else [int(v) for v in args.ms.split(",")]
    w_np, x_np = W.inputs(0, M=max(W.ms))  # W and x [96, K]; smaller M use prefixes
    workload = "square_4096x4096, M=1..96 sweep (quantize + matmul per M)"
    if args.shape:
        N, K = (int(v) for v in args.shape.split(","))
        rng = np.random.default_rng([W.seed, N, K])
        w_np = synth.iq4xs_weights(rng, N, K, W.d_scale)
        x_np = synth.activations(rng, max(max(ms), max(W.ms)), K)
        workload = f"shape_{N}x{K}, M sweep (quantize + matmul per M)"
    wd0 = torch.from_numpy(w_np).to(dev)
    wcopies = [wd0] + [wd0.clone() for _ in range(N_COPIES - 1)]
    xs = {M: torch.from_numpy(np.ascontiguousarray(x_np[:M])).to(dev) for M in ms}
    acts = {M: B.alloc_activations(M, K, dev) for M in ms}
    ops = {M: B.alloc_tc_operand(M, K, dev) for M in ms}
    ys = {M: torch.empty((M, N), dtype=torch.float32, device=dev) for M in ms}
    paths = {M: kernel_path(B, M, N, K) for M in ms}
    variants = N_COPIES // len(ms)
    stream = torch.cuda.Stream(device=dev)

    def launch_step(v):
        for i, M in enumerate(ms):
            qs, ds = acts[M]
            w = wcopies[v * len(ms) + i]
            if paths[M] == B.PATH_TC:  # the faster, prepared form (as iq4xs_linear takes it)
                B.iq4xs_quantize_q8_1_tc(xs[M], qs, ds, ops[M], stream)
                B.iq4xs_matmul_tc_operand(w, N, K, ops[M], M, ys[M], stream=stream)
            else:
                B.iq4xs_quantize_q8_1(xs[M], qs, ds, stream)
                B.iq4xs_matmul(w, N, K, qs, ds, M, ys[M], paths[M], stream)

    # Eager warm-up (also performs the library's one-time device set-up).
    with torch.cuda.stream(stream):
        for v in range(variants):
            launch_step(v)
    torch.cuda.synchronize(dev)

    # One graph per weight-copy variant.  No event nodes inside the graphs:
    # an event-record node between two kernels costs microseconds and breaks
    # programmatic dependent launch.
    graphs = []
    for v in range(variants):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            launch_step(v)
        graphs.append(g)
    torch.cuda.synchronize(dev)

    with torch.cuda.stream(stream):
        for s in range(max(3, args.warmup)):
            graphs[s % variants].replay()
    torch.cuda.synchronize(dev)

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.2)
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize(dev)
    with torch.cuda.stream(stream):
        start.record(stream)
        for s in range(args.steps):
            graphs[s % variants].replay()
        stop.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    clk = clocks.stop()
    ms_local = start.elapsed_time(stop)
    ms_total = max_over_ranks(ms_local, world)

    # Per-matmul device time: graphs of back-to-back matmul launches over the
    # rotating weight copies, CUDA events on the launching stream.
    per_m = []
    mm_us = matmul_only_times(torch, B, stream, ms, N, K, wcopies, acts, ys, paths, ops)
    q8_us = matmul_only_times(torch, B, stream, [M for M in ms if paths[M] == B.PATH_TC], N, K,
                              wcopies, acts, ys, paths)
    mm_timing = ("CUDA events around graph replays of 45 back-to-back matmul launches "
                 "(rotating weight copies) on the launching stream, per M")
    peak, peak_kind = hbm_peak_gbs()
    for M in ms:
        us = mm_us[M]
        gbs = matmul_bytes(M, N, K) / (us * 1e-6) / 1e9
        row = {"M": M, "path": PATH_NAMES[paths[M]],
               "matmul_us": round(us, 3), "GBps": round(gbs, 1),
               "TOPS": round(2 * M * N * K / (us * 1e-6) / 1e12, 3), "hbm_frac": round(gbs / peak, 4)}
        if M in q8_us:
            row["q8_form_us"] = round(q8_us[M], 3)
            row["q8_form_GBps"] = round(matmul_bytes(M, N, K) / (q8_us[M] * 1e-6) / 1e9, 1)
        per_m.append(row)
    # Dominant kernel: the path with the largest share of the sweep's matmul time.
    share = {}
    for M in ms:
        share[paths[M]] = share.get(paths[M], 0.0) + mm_us[M]
    dom = max(share, key=share.get)
    tc_ms = [M for M in ms if paths[M] == dom]
    tc_bytes = sum(matmul_bytes(M, N, K) for M in tc_ms)
    tc_us = sum(mm_us[M] for M in tc_ms)
    achieved = tc_bytes / (tc_us * 1e-6) / 1e9
    traffic = recorded_traffic(dom) if (not args.shape and dom in KERNEL_SOURCES) else None
    mm_bytes = sum(matmul_bytes(M, N, K) for M in ms)
    mm_us_total = sum(mm_us.values())

    # Tensor roofline of the same kernel: the method's 2*M*N*K and the fp16
    # MMA work the tensor cores execute (padded tiles), against the dense
    # fp16 peak.  Issue roofline: warp instructions per launch (ncu, same
    # sources) against 4 per SM and cycle at the sampled SM clock.
    tpeak, tpeak_kind = tensor_peak_tflops()
    tc_method = sum(2 * M * N * K for M in tc_ms) / (tc_us * 1e-6) / 1e12
    tc_exec = (sum(executed_flops(dom, M, N, K) for M in tc_ms) / (tc_us * 1e-6) / 1e12
               if dom in KERNEL_SOURCES else 0.0)
    counts = {2: "achieved = executed fp16 MMA flops (128 x MT x 16 MMAs on padded tiles: two per "
                 "sub-block from the Q8_1 codes, four from the prepared operand, counted as two); "
                 "method_tops = 2*M*N*K",
              4: "achieved = executed fp16 MMA flops (m16n8k16 on 8/16/24/32-row activation tiles); "
                 "method_tops = 2*M*N*K; peak = the dense fp16/bf16 rate of the 5th-generation "
                 "tensor cores (warp-level MMA issues at a fraction of it)"}.get(dom, "no tensor work")
    tensor = {"achieved": tc_exec, "peak": tpeak, "unit": "TFLOP/s", "frac": tc_exec / tpeak,
              "method_tops": tc_method, "method_frac": tc_method / tpeak,
              "peak_kind": tpeak_kind, "counts": counts}
    nsm = torch.cuda.get_device_properties(dev).multi_processor_count
    inst = recorded_counters(dom).get("inst") if (not args.shape and dom in KERNEL_SOURCES) else None
    issue = None
    if inst and clk.get("sm_mhz"):
        ipeak = nsm * 4 * clk["sm_mhz"] * 1e6 / 1e12  # T warp-instructions / s
        ach = inst / (tc_us / len(tc_ms) * 1e-6) / 1e12
        issue = {"achieved": ach, "peak": ipeak, "unit": "Twarp-inst/s", "frac": ach / ipeak,
                 "inst_per_launch": inst,
                 "peak_kind": f"{nsm} SMs x 4 issue slots x sampled SM clock"}
    fracs = {"hbm": achieved / peak, "tensor": tensor["frac"]}
    if issue:
        fracs["alu"] = issue["frac"]
    binding = max(fracs, key=fracs.get)
    gate_items = [(f"matmul M={M} {N}x{K}", matmul_bytes(M, N, K), mm_us[M] * 1e-6) for M in ms]

    sbytes = step_bytes(ms, N, K)
    ms_per_step = ms_total / args.steps
    value = world * sbytes / (ms_per_step * 1e-3) / 1e9
    tops = world * step_ops(ms, N, K) / (ms_per_step * 1e-3) / 1e12

    e2e = run_e2e(args, dev, w_np, x_np, ms, N, K, world, wcopies, paths)
    extras = {}
    if not args.no_extras and not args.ms:
        extras["baseline_dequant_gemm"] = baseline_times(torch, B, stream, ms, N, K, wcopies,
                                                         xs, mm_us)
        del wcopies, acts, ys, graphs
        torch.cuda.empty_cache()
        extras["decode_stream"] = decode_stream(torch, B, dev)
        extras["moe_grouped"] = moe_grouped(torch, B, dev)
        extras["moe_grouped_q4_0"] = moe_grouped(torch, B, dev, tokens=(4, 16, 64), wtype=B.WTYPE_Q4_0)
        extras["weight_formats"] = weight_formats(torch, B, dev, stream, mm_us)
        extras["decoder_shapes"] = decoder_shapes(torch, B, dev, stream)
        extras["prefill_sweep"] = prefill_sweep(torch, B, dev, stream)
        for r in extras["decoder_shapes"]:
            gate_items.append((f"matmul M={r['M']} {r['N']}x{r['K']}", matmul_bytes(r["M"], r["N"], r["K"]),
                               r["us"] * 1e-6))
        for r in extras["weight_formats"]:
            gate_items.append((f"{r['format']} M={r['M']}", r["GBps"] * 1e9 * r["us"] * 1e-6,
                               r["us"] * 1e-6))

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        import oracle
        threads = oracle.threads_available()
        v, dt, desc = oracle_sample(4096, threads, min_seconds=10.0)
        cpu = {"value": v, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": desc,
               "seconds": round(dt, 2), "single_thread": oracle_per_config()}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "int8/fp16-exact integer dots, f32 scale-in",
            "data": "synthetic",
            "config": {"workload": workload,
                       "N": N, "K": K, "ms": ms, "weight_copies": N_COPIES,
                       "l2": f"inputs larger than L2: {N_COPIES} rotating weight copies "
                             f"({N_COPIES * N * K * 17 // 32 / 1e6:.0f} MB)",
                       "graph": "one CUDA graph replay per step",
                       "pdl": not args.no_pdl,
                       "parallelism": f"replicas x{world}"},
            "tops": tops,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": traffic,
                         "traffic_algorithmic": tc_bytes / len(tc_ms),
                         "kernel": f"{KERNEL_NAMES[dom]}, M in {tc_ms}: "
                                   "algorithmic bytes per launch / mean launch time",
                         "time_share": {PATH_NAMES[p]: round(v / mm_us_total, 3) for p, v in share.items()},
                         "peak_kind": peak_kind, "timing": mm_timing,
                         "tensor": tensor, "alu": issue, "binding": binding,
                         "binding_rule": "the roofline with the largest fraction"},
            "roofline_gate": roofline_gate(gate_items, peak),
            "matmul_all": {"achieved_gbs": mm_bytes / (mm_us_total * 1e-6) / 1e9,
                           "frac": mm_bytes / (mm_us_total * 1e-6) / 1e9 / peak,
                           "kernels": "the dispatcher's path per M (dp4a, warp MMA, tcgen05), whole sweep"},
            "per_m": per_m,
            "e2e": e2e,
            **extras,
            "gpu_launches": args.steps * 2 * len(ms),
            "clocks": clk,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)


def projection(B, w, N, K, x, qs, ds, op, M, y, path, stream):
    """quantize + matmul as iq4xs_linear runs them with its full workspace:
    the prepared tensor-core operand on the TC path, the Q8_1 arrays on dp4a."""
    if path == B.PATH_TC:
        B.iq4xs_quantize_q8_1_tc(x, qs, ds, op, stream)
        B.iq4xs_matmul_tc_operand(w, N, K, op, M, y, stream=stream)
    else:
        B.iq4xs_quantize_q8_1(x, qs, ds, stream)
        B.iq4xs_matmul(w, N, K, qs, ds, M, y, path, stream)


def kernel_path(B, M, N, K):
    """The library kernel the dispatcher's choice runs on: its BASELINE advice
    (dequantize + a dense GEMM in the caller's BLAS) maps to the tcgen05
    kernel, which this benchmark measures; the baseline route is timed
    separately (baseline_dequant_gemm)."""
    p = B.iq4xs_select_path(M, N, K)
    return B.PATH_TC if p == B.PATH_BASELINE else p


def matmul_only_times(torch, B, stream, ms, N, K, wcopies, acts, ys, paths, ops=None, reps=20):
    """Average device time per matmul launch (us) from graphs of back-to-back
    matmuls over the rotating weight copies (tensor-core M from the prepared
    operands `ops` when given, else from the Q8_1 arrays)."""
    out = {}
    for M in ms:
        qs, ds = acts[M]
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for w in wcopies:
                if ops is not None and paths[M] == B.PATH_TC:
                    B.iq4xs_matmul_tc_operand(w, N, K, ops[M], M, ys[M], stream=stream)
                else:
                    B.iq4xs_matmul(w, N, K, qs, ds, M, ys[M], paths[M], stream)
        with torch.cuda.stream(stream):
            g.replay()
            t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            t0.record(stream)
            for _ in range(reps):
                g.replay()
            t1.record(stream)
        torch.cuda.synchronize()
        out[M] = t0.elapsed_time(t1) * 1e3 / (reps * len(wcopies))
    return out


def baseline_times(torch, B, stream, ms, N, K, wcopies, xs, mm_us, reps=10):
    """The path the batched kernel replaces (engine page, kernel table at M=64):
    dequantize the whole weight to bf16 (this library's kernel), then a dense
    bf16 GEMM (torch/cuBLAS) on bf16 activations.  Same rotating weight
    copies, per-call device time from graph replays."""
    wbf = torch.empty((N, K), dtype=torch.bfloat16, device=wcopies[0].device)
    out = []
    for M in ms:
        xb = xs[M].to(torch.bfloat16)
        with torch.cuda.stream(stream):  # eager first: cuBLAS sets up outside capture
            B.iq4xs_dequantize(wcopies[0], N, K, wbf, stream)
            torch.matmul(xb, wbf.t())
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for w in wcopies:
                B.iq4xs_dequantize(w, N, K, wbf, stream)
                torch.matmul(xb, wbf.t())
        with torch.cuda.stream(stream):
            g.replay()
            t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            t0.record(stream)
            for _ in range(reps):
                g.replay()
            t1.record(stream)
        torch.cuda.synchronize()
        us = t0.elapsed_time(t1) * 1e3 / (reps * len(wcopies))
        out.append({"M": M, "us": round(us, 3), "speedup_of_iq4xs_matmul": round(us / mm_us[M], 2)})
        del g
    return out


def decode_stream(torch, B, dev, reps=5):
    """Decode-step weight streaming: 64 decoder layers x 4 projections
    (12288x5120, 5120x6144, 34816x5120, 5120x17408; 12.3 GB of IQ4_XS resident),
    a fresh activation batch per call, each call = quantize + matmul, all 256
    calls of a step captured in one CUDA graph.  One layer's matrices are drawn
    from the seeded generator and replicated to 64 distinct device copies."""
    from iq4_xs_quantized_gb300 import synth
    W = synth.DECODE_STREAM
    layer0 = [torch.from_numpy(W.weights(i, 0)).to(dev) for i in range(len(W.shapes))]
    layers = [layer0] + [[w.clone() for w in layer0] for _ in range(W.layers - 1)]
    wbytes = sum(w.numel() for w in layer0) * W.layers
    stream = torch.cuda.Stream(device=dev)
    res = []
    for M in W.ms:
        g = torch.Generator(device=dev)
        g.manual_seed(W.seed * 1000 + M)
        calls = []
        for l in range(W.layers):
            for i, (N, K) in enumerate(W.shapes):
                x = torch.randn((M, K), device=dev, generator=g)
                qs, ds = B.alloc_activations(M, K, dev)
                y = torch.empty((M, N), dtype=torch.float32, device=dev)
                path = kernel_path(B, M, N, K)
                op = B.alloc_tc_operand(M, K, dev) if path == B.PATH_TC else None
                calls.append((layers[l][i], N, K, x, qs, ds, op, y, path))

        def step():
            for (w, N, K, x, qs, ds, op, y, path) in calls:
                projection(B, w, N, K, x, qs, ds, op, M, y, path, stream)
        with torch.cuda.stream(stream):
            step()
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            step()
        with torch.cuda.stream(stream):
            graph.replay()
            t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            t0.record(stream)
            for _ in range(reps):
                graph.replay()
            t1.record(stream)
        torch.cuda.synchronize()
        ms_step = t0.elapsed_time(t1) / reps
        nbytes = sum(matmul_bytes(M, N, K) + quantize_bytes(M, K) for (_, N, K, *_r) in calls)
        res.append({"M": M, "ms_per_step": round(ms_step, 4), "GBps": round(nbytes / (ms_step * 1e-3) / 1e9, 1),
                    "weight_GB": round(wbytes / 1e9, 2), "calls": len(calls)})
        del graph, calls
        torch.cuda.empty_cache()
    return res


def moe_grouped(torch, B, dev, layers=12, reps=5, tokens=(1, 4, 16, 64, 256), wtype=0):
    """Routed-expert layer (128 experts of 1536 x 2048, top-8; IQ4_XS experts,
    or Q4_0 / IQ4_NL ones with ``wtype``, which have no tcgen05 form): per token
    count T, one layer call = quantize the T*8 routed rows + the grouped
    matmul in one launch (the dispatcher's form, and the CUDA-core,
    warp-MMA and tcgen05 forms forced), against the same layer with one launch per
    routed expert (each on the dispatcher's path for its rows).  `layers`
    copies of the expert set (2.6 GB) rotate so the touched experts' bytes
    exceed L2.  GB/s counts the touched experts' weights plus activations
    and outputs."""
    from iq4_xs_quantized_gb300 import synth
    W = synth.MOE_DECODE
    if wtype == B.WTYPE_IQ4_XS:
        w0 = torch.from_numpy(W.weights().reshape(W.G, -1)).to(dev)
    else:
        w0 = torch.from_numpy(np.stack([synth.block32_weights(np.random.default_rng([W.seed, wtype, g]), W.N, W.K,
                                                              W.d_scale) for g in range(W.G)]).reshape(W.G, -1)).to(dev)
    stride = w0.shape[1]
    ws = [w0] + [w0.clone() for _ in range(layers - 1)]
    stream = torch.cuda.Stream(device=dev)
    res = []
    for T in tokens:
        _, rows, offsets = W.inputs(T)
        M = rows.shape[0]
        xr = torch.from_numpy(rows).to(dev)
        off = torch.from_numpy(offsets).to(dev)
        qs, ds = B.alloc_activations(M, W.K, dev)
        y = torch.empty((M, W.N), dtype=torch.float32, device=dev)
        touched = [g for g in range(W.G) if offsets[g + 1] > offsets[g]]

        def grouped(path):
            def fn(s):
                for w in ws:
                    B.iq4xs_quantize_q8_1(xr, qs, ds, s)
                    B.iq4xs_matmul_grouped(w, stride, W.G, W.N, W.K, qs, ds, off, y, s, path=path, wtype=wtype)
            return fn

        def per_expert(s):
            for w in ws:
                B.iq4xs_quantize_q8_1(xr, qs, ds, s)
                for g in touched:
                    r0, r1 = int(offsets[g]), int(offsets[g + 1])
                    B.iq4xs_matmul_wt(w[g], wtype, W.N, W.K, qs[r0:r1], ds[r0:r1], r1 - r0, y[r0:r1],
                                      B.PATH_AUTO, s)

        times = {}
        forms = [("grouped", grouped("auto")), ("grouped_dp4a", grouped("dp4a")), ("grouped_mma", grouped("mma"))]
        if wtype == B.WTYPE_IQ4_XS:
            forms.append(("grouped_tc", grouped("tc")))
        for name, fn in forms + [("per_expert", per_expert)]:
            with torch.cuda.stream(stream):
                fn(stream)
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                fn(stream)
            with torch.cuda.stream(stream):
                g.replay()
                t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                t0.record(stream)
                for _ in range(reps):
                    g.replay()
                t1.record(stream)
            torch.cuda.synchronize()
            times[name] = t0.elapsed_time(t1) * 1e3 / (reps * layers)
            del g
        nbytes = (len(touched) * B.iq4xs_weight_bytes(wtype, W.N, W.K) + M * W.K + M * (W.K // 32) * 4
                  + 4 * M * W.N + quantize_bytes(M, W.K))
        auto = {B.PATH_DP4A: "dp4a", B.PATH_MMA: "mma", B.PATH_TC: "tc"}[
            B.iq4xs_select_grouped_path(W.G, W.N, W.K, M, wtype)]
        res.append({"tokens": T, "rows": M, "experts_touched": len(touched), "auto_form": auto,
                    "grouped_us_per_layer": round(times["grouped"], 3),
                    "grouped_dp4a_us": round(times["grouped_dp4a"], 3),
                    "grouped_mma_us": round(times["grouped_mma"], 3),
                    "grouped_tc_us": round(times["grouped_tc"], 3) if "grouped_tc" in times else None,
                    "per_expert_launches_us_per_layer": round(times["per_expert"], 3),
                    "grouped_GBps": round(nbytes / (times["grouped"] * 1e-6) / 1e9, 1)})
    del ws
    torch.cuda.empty_cache()
    return res


def weight_formats(torch, B, dev, stream, iq4xs_us, N=4096, K=4096, copies=None, reps=10,
                   ms=(1, 4, 8, 16, 64, 96)):
    """The same square 4096 x 4096 matmul (or N x K) with Q4_0 and IQ4_NL
    weights (18-byte blocks of 32, 0.5625 B/weight) on the dispatcher's
    path: device time per launch from graphs of back-to-back launches over
    rotating weight copies (three times L2 unless `copies` is given),
    beside the IQ4_XS time of the main sweep; `path` names the kernel (dp4a, mma,
    tc).  Where the path is the tcgen05 kernel, `us` is its
    prepared-operand form (as in the main sweep) and `q8_form_us` the Q8_1
    form.  GB/s counts the format's weight bytes plus the Q8_1 activations
    and fp32 outputs."""
    from iq4_xs_quantized_gb300 import synth
    res = []
    for name in ("q4_0", "iq4_nl"):
        wt = B.WTYPES[name]
        w0 = torch.from_numpy(synth.block32_weights(np.random.default_rng([7, wt]), N, K,
                                                    1e-3)).to(dev)
        wbytes = B.iq4xs_weight_bytes(wt, N, K)
        ncopy = copies if copies else max(2, -(-3 * 129 * 2**20 // wbytes))  # three times L2
        ws = [w0] + [w0.clone() for _ in range(ncopy - 1)]
        rng = np.random.default_rng(8)
        for M in ms:
            x = torch.from_numpy(synth.activations(rng, M, K)).to(dev)
            qs, ds = B.alloc_activations(M, K, dev)
            B.iq4xs_quantize_q8_1(x, qs, ds, stream)
            y = torch.empty((M, N), dtype=torch.float32, device=dev)
            # the 32-weight formats take the dispatcher's path for the shape
            path = B.iq4xs_select_path(M, N, K)
            tc = path in (B.PATH_TC, B.PATH_BASELINE)
            op = None
            if tc:
                op = B.alloc_tc_operand(M, K, dev)
                B.iq4xs_quantize_q8_1_tc(x, qs, ds, op, stream)

            def timed(fn):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    for w in ws:
                        fn(w)
                with torch.cuda.stream(stream):
                    g.replay()
                    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    t0.record(stream)
                    for _ in range(reps):
                        g.replay()
                    t1.record(stream)
                torch.cuda.synchronize()
                return t0.elapsed_time(t1) * 1e3 / (reps * ncopy)

            q8_us = timed(lambda w: B.iq4xs_matmul_wt(w, wt, N, K, qs, ds, M, y, B.PATH_AUTO, stream))
            us = timed(lambda w: B.iq4xs_matmul_tc_operand(w, N, K, op, M, y, wt, stream=stream)) if tc else q8_us
            nbytes = wbytes + M * K + M * (K // 32) * 4 + 4 * M * N
            row = {"format": name, "M": M, "path": "tc" if tc else ("mma" if path == B.PATH_MMA else "dp4a"),
                   "us": round(us, 3),
                   "GBps": round(nbytes / (us * 1e-6) / 1e9, 1),
                   "iq4_xs_us": round(iq4xs_us[M], 3) if M in iq4xs_us else None}
            if tc:
                row["q8_form_us"] = round(q8_us, 3)
            res.append(row)
        del ws, w0
        torch.cuda.empty_cache()
    return res


def _graph_us(torch, stream, fn, calls, reps):
    """Device time per call of `fn` (which issues `calls` launches) from
    graph replays timed with CUDA events on the launching stream."""
    with torch.cuda.stream(stream):
        fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        fn()
    with torch.cuda.stream(stream):
        g.replay()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for _ in range(reps):
            g.replay()
        t1.record(stream)
    torch.cuda.synchronize()
    del g
    return t0.elapsed_time(t1) * 1e3 / (reps * calls)


def _copies_over_l2(torch, w0, target=4 * 129 * 2**20):
    n = max(4, -(-target // w0.numel()))
    return [w0] + [w0.clone() for _ in range(n - 1)]


def decoder_shapes(torch, B, dev, stream, reps=10):
    """The nine projection shapes of a ~27B-class decoder layer (1% of the
    activation channels x20), M = 1, 4, 8, 16, 64: the matmul on the
    dispatcher's kernel path, device time per launch from graphs of
    back-to-back launches over rotating weight copies (more than 4x L2 per
    shape); GB/s counts W, the Q8_1 activations and y."""
    from iq4_xs_quantized_gb300 import synth
    W = synth.DECODER_27B
    res = []
    for si, (N, K) in enumerate(W.shapes):
        w_np, x_np = W.inputs(si, M=max(W.ms))
        ws = _copies_over_l2(torch, torch.from_numpy(w_np).to(dev))
        y = torch.empty((max(W.ms), N), dtype=torch.float32, device=dev)
        for M in W.ms:
            path = kernel_path(B, M, N, K)
            x = torch.from_numpy(np.ascontiguousarray(x_np[:M])).to(dev)
            qs, ds = B.alloc_activations(M, K, dev)
            op = B.alloc_tc_operand(M, K, dev)
            B.iq4xs_quantize_q8_1_tc(x, qs, ds, op, stream)

            def mm():
                for w in ws:
                    if path == B.PATH_TC:
                        B.iq4xs_matmul_tc_operand(w, N, K, op, M, y, stream=stream)
                    else:
                        B.iq4xs_matmul(w, N, K, qs, ds, M, y, path, stream)

            def mm_path(p):
                def f():
                    for w in ws:
                        if p == "tcp":
                            B.iq4xs_matmul_tc_operand(w, N, K, op, M, y, stream=stream)
                        else:
                            B.iq4xs_matmul(w, N, K, qs, ds, M, y, p, stream)
                return f
            us = _graph_us(torch, stream, mm, len(ws), reps)
            gbs = matmul_bytes(M, N, K) / (us * 1e-6) / 1e9
            row = {"N": N, "K": K, "M": M, "path": PATH_NAMES[path],
                   "us": round(us, 3), "GBps": round(gbs, 1),
                   "TOPS": round(2 * M * N * K / (us * 1e-6) / 1e12, 2)}
            # every other kernel path beside the dispatcher's choice
            alts = {"tc_us": "tcp", "q8_form_us": B.PATH_TC, "mma_us": B.PATH_MMA}
            if M <= 16:
                alts["dp4a_us"] = B.PATH_DP4A
            for key, p in alts.items():
                row[key] = round(_graph_us(torch, stream, mm_path(p), len(ws), reps), 3)
            res.append(row)
        del ws
        torch.cuda.empty_cache()
    return res


def prefill_sweep(torch, B, dev, stream, reps=3):
    """Prefill range: (17408, 5120) and (5120, 17408), M = 96..512, x rounded
    to bf16.  The tcgen05 matmul (quantize included) against the dequantize to
    bf16 + dense bf16 GEMM route, same rotating weight copies, device time
    per call; `advised` is the route iq4xs_select_path names."""
    from iq4_xs_quantized_gb300 import synth
    W = synth.PREFILL
    res = []
    for si, (N, K) in enumerate(W.shapes):
        w_np, x_np = W.inputs(si, M=max(W.ms))
        ws = _copies_over_l2(torch, torch.from_numpy(w_np).to(dev))
        wbf = torch.empty((N, K), dtype=torch.bfloat16, device=dev)
        for M in W.ms:
            x = torch.from_numpy(np.ascontiguousarray(x_np[:M])).to(dev)
            xb = x.to(torch.bfloat16)
            qs, ds = B.alloc_activations(M, K, dev)
            op = B.alloc_tc_operand(M, K, dev)
            y = torch.empty((M, N), dtype=torch.float32, device=dev)

            def tc():
                for w in ws:
                    projection(B, w, N, K, x, qs, ds, op, M, y, B.PATH_TC, stream)

            def base():
                for w in ws:
                    B.iq4xs_dequantize(w, N, K, wbf, stream)
                    torch.matmul(xb, wbf.t())
            t_tc = _graph_us(torch, stream, tc, len(ws), reps)
            t_b = _graph_us(torch, stream, base, len(ws), reps)
            adv = B.iq4xs_select_path(M, N, K)
            res.append({"N": N, "K": K, "M": M, "tc_us": round(t_tc, 2), "dequant_gemm_us": round(t_b, 2),
                        "advised": "baseline" if adv == B.PATH_BASELINE else "tc"})
        del ws, wbf
        torch.cuda.empty_cache()
    return res


def run_e2e(args, dev, w_np, x_np, ms, N, K, world, wcopies, paths):
    """Same step through the public API with HOST buffers, as a serving
    caller on a Grace-Blackwell node runs it: the step's activations (every
    M's rows, packed) sit in pinned host memory and the library's one-call
    projection iq4xs_linear (quantize + matmul on the dispatcher's path) per
    M reads its rows from there and writes its outputs into pinned host
    memory -- the quantizer loads x and the matmul stores y over the
    host-device link, no staging copy.  The calls are captured once in a
    CUDA graph (one per weight-copy variant), replayed and synchronised
    every step, so the host-device traffic and every kernel are inside the
    timed region.  The same step with one explicit pinned H2D copy of x and
    one D2H copy of y around device buffers is timed alongside
    (``with_copies``)."""
    import torch

    from iq4_xs_quantized_gb300 import binding as B
    stream = torch.cuda.Stream(device=dev)
    offs = np.concatenate([[0], np.cumsum(ms)]).astype(int)
    rows = int(offs[-1])
    hx = torch.from_numpy(np.concatenate([x_np[:M] for M in ms])).pin_memory()
    hy = torch.empty((rows, N), dtype=torch.float32).pin_memory()
    dx = torch.empty((rows, K), dtype=torch.float32, device=dev)
    dy = torch.empty((rows, N), dtype=torch.float32, device=dev)
    ws = {M: torch.empty(B.iq4xs_linear_workspace_bytes(M, N, K), dtype=torch.uint8, device=dev)
          for M in ms}
    h2d = rows * K * 4
    d2h = rows * N * 4
    variants = len(wcopies) // len(ms)

    def host_calls(v):
        for i, M in enumerate(ms):
            o = int(offs[i])
            B.iq4xs_linear(wcopies[v * len(ms) + i], N, K, hx[o:o + M], hy[o:o + M], ws[M], stream)

    def copy_calls(v):
        dx.copy_(hx, non_blocking=True)
        for i, M in enumerate(ms):
            o = int(offs[i])
            B.iq4xs_linear(wcopies[v * len(ms) + i], N, K, dx[o:o + M], dy[o:o + M], ws[M], stream)
        hy.copy_(dy, non_blocking=True)

    def timed(calls):
        with torch.cuda.stream(stream):
            for v in range(variants):  # eager first: one-time set-up outside capture
                calls(v)
        stream.synchronize()
        graphs = []
        for v in range(variants):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                calls(v)
            graphs.append(g)

        def step(s):
            with torch.cuda.stream(stream):
                graphs[s % variants].replay()
            stream.synchronize()

        for s in range(5):
            step(s)
        barrier(world)
        t0 = time.perf_counter()
        for s in range(args.e2e_steps):
            step(s)
        dt = max_over_ranks(time.perf_counter() - t0, world)
        del graphs
        return dt

    dt = timed(host_calls)
    dt_copy = timed(copy_calls)
    value = world * args.e2e_steps * step_bytes(ms, N, K) / dt / 1e9
    value_copy = world * args.e2e_steps * step_bytes(ms, N, K) / dt_copy / 1e9
    return {"value": value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "steps": args.e2e_steps, "ms_per_step": dt / args.e2e_steps * 1e3,
            "calls": "iq4xs_linear per M on pinned host x and y (the kernels read x and write y "
                     "over the host-device link); captured in a CUDA graph, replayed and "
                     "synchronised every step",
            "with_copies": {"value": value_copy, "unit": UNIT,
                            "ms_per_step": dt_copy / args.e2e_steps * 1e3,
                            "calls": "one pinned H2D copy of x, iq4xs_linear per M on device "
                                     "buffers, one pinned D2H copy of y; same graph and sync"}}


def main():
    args = parse_args()
    world, rank, local = dist_setup()
    try:
        if args.impl == "reference":
            run_reference(args, world, rank)
        else:
            run_ours(args, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
