"""Measure the path crossovers (dp4a -> warp MMA -> tcgen05) and store them
for the dispatcher.

The engine page's dispatcher hard-coded its mmvq -> dequantize threshold at
M=8 while the measured crossover sat near M=15 (V100TPS engine page, mmvq vs
dequantize table).  Here every crossover is measured: for each calibration
shape and M, the three kernel paths are timed from CUDA-graph replays over
rotating weight copies (inputs larger than L2), the tensor-core path in the
prepared form iq4xs_linear runs.  Per shape, the DP4A range ends at the
first M at which another path is faster, the MMA range at the first M above
it at which tcgen05 is faster; each shape's thresholds apply to its
weight-size class (from the geometric mean of its weight count and the next
smaller shape's), the smallest shape's to everything below.  The result is
written to ``dispatch_table.json`` beside this file and installed whenever
the binding loads.

Before the crossovers, the warp-MMA launches are tuned: on the shapes the
benchmark runs (the square 4096 projection and the nine projections of a
~27B decoder layer), for each activation-tile height (8, 16, 24, 32 rows),
every launch configuration the kernel holds (rows per CTA, K split, CTAs
per SM) is timed and the fastest goes into the table's ``mma_launch``
entries; other shapes use the kernel's launch model.

Run on the GPU:  python -m iq4_xs_quantized_gb300.calibrate
"""
from __future__ import annotations

import json
import os
import sys

import numpy as np

TABLE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "dispatch_table.json")
# Crossover shapes, one per weight-size class (classes are keyed by N*K
# alone, so no two shapes share a weight count).
SHAPES = ((1024, 5120), (4096, 4096), (5120, 5120), (6144, 5120), (12288, 5120), (5120, 17408), (34816, 5120))
MS = tuple(range(1, 17)) + (20, 24, 28, 32, 40, 48, 64)
DP4A_MS = tuple(range(1, 17))  # dp4a is timed up to here (its cost grows with M)
# Upper threshold: the tcgen05 route (quantize + matmul) against dequantize
# to bf16 + a dense bf16 GEMM, on the square and the two prefill shapes.
BASE_SHAPES = ((4096, 4096), (17408, 5120), (5120, 17408))
BASE_MS = (32, 48, 64, 80, 96, 128, 192, 256, 512)
L2_MULTIPLE = 3
L2_BYTES = 129 * 2**20
# Shapes whose warp-MMA launches are tuned, and the activation-tile heights.
LAUNCH_SHAPES = ((4096, 4096), (5120, 5120), (6144, 5120), (1024, 5120), (10240, 5120), (12288, 5120),
                 (5120, 6144), (17408, 5120), (34816, 5120), (5120, 17408))
LAUNCH_TILES = (8, 16, 24, 32)


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
            r = {}
            if M in DP4A_MS:
                r["dp4a_us"] = round(time_path(B, torch, wcopies, N, K, M, B.PATH_DP4A), 3)
            r["mma_us"] = round(time_path(B, torch, wcopies, N, K, M, B.PATH_MMA), 3)
            r["tc_us"] = round(time_path(B, torch, wcopies, N, K, M, B.PATH_TC), 3)
            rows[M] = r
            if verbose:
                print(f"N={N} K={K} M={M}: " + "  ".join(f"{k[:-3]} {v:.2f} us" for k, v in r.items()),
                      flush=True)
        per_shape[f"{N}x{K}"] = rows
        del wcopies, w
        torch.cuda.empty_cache()
    dp4a_cls, mma_cls, dflt = class_crossovers(per_shape, ms)
    table = {"crossover_m_max_dp4a": dflt[0], "mma_m_max": dflt[1], "gpu": torch.cuda.get_device_name(),
             "crossover_classes": dp4a_cls, "mma_classes": mma_cls,
             "shapes": per_shape, "rule": CROSSOVER_RULE, "class_rule": CLASS_RULE}
    return table


CROSSOVER_RULE = ("per shape: DP4A up to the last M (scanning up from 1) at which it is the fastest of "
                  "the three paths; MMA from there up to the last M at which it is faster than the "
                  "tcgen05 path (prepared form); tcgen05 above")
CLASS_RULE = ("a calibration shape's thresholds apply from the geometric mean of its weight count "
              "and the next smaller shape's; the smallest shape's thresholds are the defaults")


def _row(rows, M):
    return rows.get(M, rows.get(str(M)))


def shape_thresholds(rows, ms):
    """(m_max_dp4a, m_max_mma) of one shape from {M: {"dp4a_us", "mma_us", "tc_us"}}."""
    m_dp4a = 0
    for M in ms:
        r = _row(rows, M)
        if "dp4a_us" in r and r["dp4a_us"] < min(r["mma_us"], r["tc_us"]):
            m_dp4a = M
        else:
            break
    m_mma = m_dp4a
    for M in ms:
        if M <= m_dp4a:
            continue
        r = _row(rows, M)
        if r["mma_us"] < r["tc_us"]:
            m_mma = M
        else:
            break
    return m_dp4a, m_mma


def class_crossovers(per_shape, ms):
    """([[min_weights, m_max_dp4a], ...], [[min_weights, m_max_mma], ...],
    (default dp4a, default mma)): one class per calibration shape above the
    smallest, whose thresholds are the defaults."""
    sizes = sorted((int(k.split("x")[0]) * int(k.split("x")[1]), k) for k in per_shape)
    th = [shape_thresholds(per_shape[k], ms) for _, k in sizes]
    dp4a, mma = [], []
    for i in range(1, len(sizes)):
        lo = int(round((sizes[i - 1][0] * sizes[i][0]) ** 0.5))
        dp4a.append([lo, th[i][0]])
        mma.append([lo, th[i][1]])
    return dp4a, mma, th[0]


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


def launch_candidates(K, tile_rows):
    """Every (rows per CTA, K split, CTAs per SM) the warp-MMA kernel may hold
    for this tile height (the kernel reports which it does)."""
    pairs = K // 512
    rmax = 256 if tile_rows <= 16 else 128
    out = [(r, s, 1) for r in range(32, rmax + 1, 32) for s in range(1, 9) if s <= pairs]
    out += [(r, s, 2) for r in (32, 64) for s in (1, 2, 3, 4) if s <= pairs]
    return out


def calibrate_launches(shapes=LAUNCH_SHAPES, tiles=LAUNCH_TILES, verbose=True):
    """[[N, K, tile_rows, rows, splits, ctas_per_sm], ...] of the fastest
    warp-MMA launch per shape and tile height, and the timings behind them
    (the launch model's own choice beside the best)."""
    import torch

    from . import binding as B
    from . import synth
    B.iq4xs_set_mma_launch_table([])  # time the model's choices, not an older table's
    rng = np.random.default_rng(77)
    entries, detail = [], {}
    for N, K in shapes:
        w = torch.from_numpy(synth.iq4xs_weights(rng, N, K, 1e-3)).cuda()
        ncopy = max(2, int(np.ceil(L2_MULTIPLE * L2_BYTES / w.numel())))
        wcopies = [w] + [w.clone() for _ in range(ncopy - 1)]
        for mt in tiles:
            M = mt
            qs, ds = B.alloc_activations(M, K, "cuda")
            B.iq4xs_quantize_q8_1(torch.randn(M, K, device="cuda"), qs, ds)
            y = torch.empty(M, N, device="cuda")

            def run(s):
                for ww in wcopies:
                    B.iq4xs_matmul(ww, N, K, qs, ds, M, y, B.PATH_MMA, s)

            model = B.iq4xs_mma_launch_config(M, N, K)
            times = {}
            try:
                for c in launch_candidates(K, mt):
                    B.iq4xs_test_mma_config(*c)
                    if B.iq4xs_mma_launch_config(M, N, K) != c:
                        continue  # not one the kernel holds
                    times[c] = _graph_time(torch, run, reps=5) / len(wcopies)
            finally:
                B.iq4xs_test_mma_config(0, 0, 0)
            best = min(times, key=times.get)
            entries.append([N, K, mt, *best])
            detail[f"{N}x{K}/{mt}"] = {"best": list(best), "best_us": round(times[best], 3),
                                       "model": list(model), "model_us": round(times.get(model, -1.0), 3)}
            if verbose:
                print(f"N={N} K={K} tile {mt}: best {best} {times[best]:.2f} us, model {model} "
                      f"{times.get(model, float('nan')):.2f} us", flush=True)
        del wcopies, w
        torch.cuda.empty_cache()
    return entries, detail


def load_table():
    try:
        with open(TABLE) as f:
            return json.load(f)
    except (OSError, ValueError):
        return None


def main():
    from . import binding as B
    launches, launch_detail = calibrate_launches()
    B.iq4xs_set_mma_launch_table(launches)  # the crossovers below see the tuned launches
    table = calibrate()
    table["mma_launch"] = launches
    table["mma_launch_detail"] = launch_detail
    thr, per_shape = calibrate_baseline()
    table["baseline_m_min"] = thr
    table["baseline_shapes"] = per_shape
    table["baseline_rule"] = ("smallest M from which dequantize to bf16 + a dense bf16 GEMM beats "
                              "quantize + tcgen05 matmul at that M and every larger one, summed "
                              "over the shapes (0 = never)")
    with open(TABLE, "w") as f:
        json.dump(table, f, indent=1)
    print(json.dumps({"crossover_m_max_dp4a": table["crossover_m_max_dp4a"], "mma_m_max": table["mma_m_max"],
                      "crossover_classes": table["crossover_classes"], "mma_classes": table["mma_classes"],
                      "baseline_m_min": table["baseline_m_min"]}))


if __name__ == "__main__":
    sys.exit(main())
