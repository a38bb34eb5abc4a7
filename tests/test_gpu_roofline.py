"""Roofline gate (V100TPS engine page, the passage on the broken batched
route: besides a zero error against an independent path, a kernel that skipped
its work shows up as a call faster than its bytes allow).  Every path is timed
the way the benchmark times it -- CUDA events around graph replays of
back-to-back launches over rotating weight copies larger than L2 -- and its
algorithmic bytes per call divided by that time must stay within 1.1x the
measured HBM copy bandwidth."""
import json
import os

import numpy as np
import pytest
import torch

from _gates import gate_roofline
from iq4_xs_quantized_gb300 import binding as B
from iq4_xs_quantized_gb300 import synth

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
L2_BYTES = 129 * 2**20


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from iq4_xs_quantized_gb300 import build
    build.build()
    B.load()
    yield
    assert B.iq4xs_last_device_error() == 0


def hbm_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]) * 1e9
    except (OSError, KeyError, ValueError):
        return 6800.0e9  # one earlier measurement of a GB300 copy


def copies_of(w: torch.Tensor):
    n = max(2, int(np.ceil(3 * L2_BYTES / (w.numel() * w.element_size()))))
    return [w] + [w.clone() for _ in range(n - 1)]


def time_calls(launch, count, reps=10):
    """Mean device time (s) per call: graph of `count` launches, replayed."""
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        launch(s)  # eager first: one-time set-up outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        launch(s)
    with torch.cuda.stream(s):
        g.replay()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(s)
        for _ in range(reps):
            g.replay()
        t1.record(s)
    torch.cuda.synchronize()
    return t0.elapsed_time(t1) * 1e-3 / (reps * count)


def matmul_bytes(wbytes, M, N, K):
    return wbytes + M * K + M * (K // 32) * 4 + 4 * M * N


@pytest.mark.parametrize("N,K", [(4096, 4096), (12288, 5120)])
@pytest.mark.parametrize("path,M", [("dp4a", 1), ("dp4a", 4), ("tc", 8), ("tc", 16), ("tc", 64),
                                    ("tc", 96), ("mma", 1), ("mma", 8), ("mma", 16), ("mma", 32)])
def test_matmul_within_hbm_roofline(N, K, path, M):
    rng = np.random.default_rng([N, K, M])
    w = torch.from_numpy(synth.iq4xs_weights(rng, N, K, 1e-3)).cuda()
    x = torch.from_numpy(synth.activations(rng, M, K)).cuda()
    qs, ds = B.alloc_activations(M, K, "cuda")
    B.iq4xs_quantize_q8_1(x, qs, ds)
    y = torch.empty((M, N), device="cuda")
    ws = copies_of(w)

    def launch(s):
        for wc in ws:
            B.iq4xs_matmul(wc, N, K, qs, ds, M, y, path, s)

    t = time_calls(launch, len(ws))
    r = gate_roofline(matmul_bytes(w.numel(), M, N, K), t, hbm_peak())
    assert r is None, f"{path} M={M} {N}x{K}: {r}"


@pytest.mark.parametrize("wtype", ["q4_0", "iq4_nl"])
@pytest.mark.parametrize("M", (1, 16))
def test_weight_formats_within_hbm_roofline(wtype, M):
    N, K = 4096, 4096
    rng = np.random.default_rng([7, M])
    w = torch.from_numpy(synth.block32_weights(rng, N, K, 1e-3)).cuda()
    x = torch.from_numpy(synth.activations(rng, M, K)).cuda()
    qs, ds = B.alloc_activations(M, K, "cuda")
    B.iq4xs_quantize_q8_1(x, qs, ds)
    y = torch.empty((M, N), device="cuda")
    ws = copies_of(w)

    def launch(s):
        for wc in ws:
            B.iq4xs_matmul_wt(wc, wtype, N, K, qs, ds, M, y, B.PATH_AUTO, s)

    t = time_calls(launch, len(ws))
    r = gate_roofline(matmul_bytes(w.numel(), M, N, K), t, hbm_peak())
    assert r is None, f"{wtype} M={M}: {r}"


@pytest.mark.parametrize("T,path", [(1, "auto"), (16, "auto"), (64, "mma"), (128, "mma")])
def test_grouped_within_hbm_roofline(T, path):
    W = synth.MOE_DECODE
    _, rows, offsets = W.inputs(T)
    M = rows.shape[0]
    w_np = W.weights()
    stride = w_np.shape[1] * w_np.shape[2]
    wg = torch.from_numpy(w_np.reshape(W.G, -1)).cuda()
    qs, ds = B.alloc_activations(M, W.K, "cuda")
    B.iq4xs_quantize_q8_1(torch.from_numpy(rows).cuda(), qs, ds)
    off = torch.from_numpy(offsets).cuda()
    y = torch.empty((M, W.N), device="cuda")
    ws = copies_of(wg)
    touched = sum(1 for g in range(W.G) if offsets[g + 1] > offsets[g])

    def launch(s):
        for wc in ws:
            B.iq4xs_matmul_grouped(wc, stride, W.G, W.N, W.K, qs, ds, off, y, s, path=path)

    t = time_calls(launch, len(ws))
    # only the experts that have rows are read
    r = gate_roofline(matmul_bytes(touched * W.N * (W.K // 256) * 136, M, W.N, W.K), t, hbm_peak())
    assert r is None, f"grouped T={T} {path}: {r}"
