"""Measure the dp4a <-> tcgen05 crossover and store it for the dispatcher.

The engine page's dispatcher hard-coded its mmvq -> dequantize threshold at
M=8 while the measured crossover sat near M=15 (V100TPS engine page, mmvq vs
dequantize table).  Here the crossover is measured: for every M in 1..16 and
every calibration shape, both kernel paths are timed from CUDA-graph replays
over rotating weight copies (inputs larger than L2); the dispatcher's
threshold becomes the largest M at which the dp4a path costs less summed over
the shapes, each shape's times taken relative to the faster path there (so
that every shape counts alike, not the one with the most bytes).  The result is written to ``dispatch_table.json`` beside this file
and installed with ``iq4xs_set_crossover`` whenever the binding loads.

Run on the GPU:  python -m iq4_xs_quantized_gb300.calibrate
"""
from __future__ import annotations

import json
import os
import sys

import numpy as np

TABLE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "dispatch_table.json")
SHAPES = ((4096, 4096), (5120, 5120), (12288, 5120), (5120, 17408), (34816, 5120))
MS = tuple(range(1, 17))
# Upper threshold: the tcgen05 route (quantize + matmul) against dequantize
# to bf16 + a dense bf16 GEMM, on the square and the two prefill shapes.
BASE_SHAPES = ((4096, 4096), (17408, 5120), (5120, 17408))
BASE_MS = (32, 48, 64, 80, 96, 128, 192, 256, 512)
L2_MULTIPLE = 3
L2_BYTES = 129 * 2**20


def time_path(B, torch, wcopies, N, K, M, path, reps=20):
    """us per matmul on `path`; the tensor-core path in its prepared-operand
    form (the one iq4xs_linear takes with its full workspace)."""
    qs, ds = B.alloc_activations(M, K, "cuda")
    op = B.alloc_tc_operand(M, K, "cuda")
    x = torch.randn(M, K, device="cuda")
    y = torch.empty(M, N, device="cuda")
    B.iq4xs_quantize_q8_1_tc(x, qs, ds, op)
    s = torch.cuda.Stream()

    def run():
        for w in wcopies:
            if path == B.PATH_TC:
                B.iq4xs_matmul_tc_operand(w, N, K, op, M, y, stream=s)
            else:
                B.iq4xs_matmul(w, N, K, qs, ds, M, y, path, s)
    with torch.cuda.stream(s):
        run()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        run()
    with torch.cuda.stream(s):
        g.replay()
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(s):
        t0.record(s)
        for _ in range(reps):
            g.replay()
        t1.record(s)
    torch.cuda.synchronize()
    return t0.elapsed_time(t1) * 1e3 / (reps * len(wcopies))  # us per call


def calibrate(shapes=SHAPES, ms=MS, verbose=True):
    import torch

    from . import binding as B
    from . import synth
    rng = np.random.default_rng(123)
    per_shape = {}
    for N, K in shapes:
        w = torch.from_numpy(synth.iq4xs_weights(rng, N, K, 1e-3)).cuda()
        ncopy = max(2, int(np.ceil(L2_MULTIPLE * L2_BYTES / w.numel())))
        wcopies = [w] + [w.clone() for _ in range(ncopy - 1)]
        rows = {}
        for M in ms:
            t_dp = time_path(B, torch, wcopies, N, K, M, B.PATH_DP4A)
            t_tc = time_path(B, torch, wcopies, N, K, M, B.PATH_TC)
            rows[M] = {"dp4a_us": round(t_dp, 3), "tc_us": round(t_tc, 3)}
            if verbose:
                print(f"N={N} K={K} M={M}: dp4a {t_dp:.2f} us  tc {t_tc:.2f} us", flush=True)
        per_shape[f"{N}x{K}"] = rows
        del wcopies, w
        torch.cuda.empty_cache()
    table = {"crossover_m_max_dp4a": crossover_from(per_shape, ms), "gpu": torch.cuda.get_device_name(),
             "crossover_classes": class_crossovers(per_shape, ms),
             "shapes": per_shape, "rule": CROSSOVER_RULE, "class_rule": CLASS_RULE}
    return table


CROSSOVER_RULE = ("largest M (scanning up from 1) at which the dp4a path costs less than the "
                  "tcgen05 path summed over the calibration shapes, each shape's time relative "
                  "to the faster path at that shape and M")


def crossover_from(per_shape, ms):
    """The dispatcher threshold from per-shape timings {shape: {M: {"dp4a_us", "tc_us"}}}."""
    crossover = 0
    for M in ms:
        rel = {"dp4a": 0.0, "tc": 0.0}
        for rows in per_shape.values():
            r = rows.get(M, rows.get(str(M)))
            best = min(r["dp4a_us"], r["tc_us"])
            rel["dp4a"] += r["dp4a_us"] / best
            rel["tc"] += r["tc_us"] / best
        if rel["dp4a"] < rel["tc"]:
            crossover = M
        else:
            break
    return crossover


CLASS_RULE = ("per weight-size class: each calibration shape's own crossover (largest M, "
              "scanning up from 1, at which dp4a is faster on that shape); a shape's class "
              "starts at the geometric mean of its weight count and the next smaller shape's")


def shape_crossover(rows, ms):
    """Largest M (scanning up from 1) at which dp4a beats tcgen05 on one shape."""
    crossover = 0
    for M in ms:
        r = rows.get(M, rows.get(str(M)))
        if r["dp4a_us"] < r["tc_us"]:
            crossover = M
        else:
            break
    return crossover


def class_crossovers(per_shape, ms):
    """[[min_weights, m_max_dp4a], ...] ascending, one class per calibration
    shape above the smallest (the smallest shape's crossover is the default
    for everything below the first class)."""
    sizes = sorted((int(k.split("x")[0]) * int(k.split("x")[1]), k) for k in per_shape)
    out = []
    for i in range(1, len(sizes)):
        lo = int(round((sizes[i - 1][0] * sizes[i][0]) ** 0.5))
        out.append([lo, shape_crossover(per_shape[sizes[i][1]], ms)])
    return out


def _graph_time(torch, fn, reps=10):
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        fn(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        fn(s)
    with torch.cuda.stream(s):
        g.replay()
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(s):
        t0.record(s)
        for _ in range(reps):
            g.replay()
        t1.record(s)
    torch.cuda.synchronize()
    return t0.elapsed_time(t1) * 1e3 / reps


def calibrate_baseline(shapes=BASE_SHAPES, ms=BASE_MS, verbose=True):
    """Smallest M from which dequantize + bf16 GEMM beats quantize + tcgen05
    matmul at that M and every larger one (summed over the shapes); 0 if
    never.  Returns (threshold, per-shape times)."""
    import torch

    from . import binding as B
    from . import synth
    rng = np.random.default_rng(321)
    per_shape, total = {}, {M: [0.0, 0.0] for M in ms}
    for N, K in shapes:
        w = torch.from_numpy(synth.iq4xs_weights(rng, N, K, 1e-3)).cuda()
        ncopy = max(2, int(np.ceil(L2_MULTIPLE * L2_BYTES / w.numel())))
        wcopies = [w] + [w.clone() for _ in range(ncopy - 1)]
        wbf = torch.empty((N, K), dtype=torch.bfloat16, device="cuda")
        rows = {}
        for M in ms:
            x = torch.randn(M, K, device="cuda")
            qs, ds = B.alloc_activations(M, K, "cuda")
            op = B.alloc_tc_operand(M, K, "cuda")
            y = torch.empty(M, N, device="cuda")

            def tc(s):
                for ww in wcopies:
                    B.iq4xs_quantize_q8_1_tc(x, qs, ds, op, s)
                    B.iq4xs_matmul_tc_operand(ww, N, K, op, M, y, stream=s)

            def base(s):
                for ww in wcopies:
                    B.iq4xs_dequantize(ww, N, K, wbf, s)
                    torch.matmul(x.to(torch.bfloat16), wbf.t())

            t_tc = _graph_time(torch, tc) / len(wcopies)
            t_b = _graph_time(torch, base) / len(wcopies)
            rows[M] = {"tc_us": round(t_tc, 3), "dequant_gemm_us": round(t_b, 3)}
            total[M][0] += t_tc
            total[M][1] += t_b
            if verbose:
                print(f"N={N} K={K} M={M}: tc {t_tc:.2f} us  dequant+gemm {t_b:.2f} us", flush=True)
        per_shape[f"{N}x{K}"] = rows
        del wcopies, w, wbf
        torch.cuda.empty_cache()
    threshold = 0
    for M in sorted(ms, reverse=True):
        if total[M][1] < total[M][0]:
            threshold = M
        else:
            break
    return threshold, per_shape


def load_table():
    try:
        with open(TABLE) as f:
            return json.load(f)
    except (OSError, ValueError):
        return None


def main():
    table = calibrate()
    thr, per_shape = calibrate_baseline()
    table["baseline_m_min"] = thr
    table["baseline_shapes"] = per_shape
    table["baseline_rule"] = ("smallest M from which dequantize to bf16 + a dense bf16 GEMM beats "
                              "quantize + tcgen05 matmul at that M and every larger one, summed "
                              "over the shapes (0 = never)")
    with open(TABLE, "w") as f:
        json.dump(table, f, indent=1)
    print(json.dumps({"crossover_m_max_dp4a": table["crossover_m_max_dp4a"],
                      "baseline_m_min": table["baseline_m_min"]}))


if __name__ == "__main__":
    sys.exit(main())
