"""iq4xs_linear (quantize + matmul through a caller workspace) on the GPU:
same result as the two separate calls of the form it takes (the prepared
tensor-core operand when the workspace holds it, else the Q8_1 arrays),
within 1e-5 per row of the oracle, and the workspace holds the Q8_1 codes
and {d, s}, bit-exact."""
import numpy as np
import pytest
import torch

from _gates import gate_parity, gate_written
from _gpu import dev, matmul_gpu, oracle_matmul, oracle_q8, prepare_gpu, quantize_gpu, sample_rows
from iq4_xs_quantized_gb300 import binding as B
from iq4_xs_quantized_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from iq4_xs_quantized_gb300 import build
    build.build()
    B.load()
    yield
    assert B.iq4xs_last_device_error() == 0


@pytest.fixture(autouse=True)
def _fixed_dispatch():
    """DP4A to M = 4, warp MMA to M = 8, tcgen05 above, whatever the
    calibrated table says; the table is restored afterwards."""
    B.iq4xs_set_crossover_classes([])
    B.iq4xs_set_mma_crossover_classes([])
    B.iq4xs_set_mma_crossover(8)
    yield
    B.reset_dispatch()


NAMES = {B.PATH_DP4A: "dp4a", B.PATH_MMA: "mma", B.PATH_TC: "tc", B.PATH_BASELINE: "tc"}  # linear runs TC on the advice


@pytest.mark.parametrize("M", (1, 3, 6, 8, 33, 96, 200))
def test_linear_matches_two_calls_and_oracle(M):
    W = synth.SQUARE
    N, K = W.shapes[0]
    w, x = W.inputs(0, M=M)
    wd, xd = dev(w), dev(x)
    ws = torch.full((B.iq4xs_linear_workspace_bytes(M, N, K),), 0xFF, dtype=torch.uint8,
                    device="cuda")
    y = torch.full((M, N), float("nan"), device="cuda")
    B.iq4xs_linear(wd, N, K, xd, y, ws)
    torch.cuda.synchronize()
    yl = y.cpu().numpy()
    assert gate_written(yl) is None
    path = NAMES[B.iq4xs_select_path(M, N, K)]
    qs, ds = quantize_gpu(x)
    # the full workspace: the prepared operand on the tensor-core path
    y2 = matmul_gpu(wd, N, K, qs, ds, M, "tcp" if path == "tc" else path,
                    op=prepare_gpu(x, qs, ds) if path == "tc" else None)
    assert np.array_equal(yl, y2)
    qs_o, d_o, _ = oracle_q8(x)
    rows = sample_rows(N, 40, seed=M)
    r = gate_parity(yl[:, rows], oracle_matmul(w, N, K, qs_o, d_o, rows))
    assert r is None, r
    # the least workspace: the Q8_1 form, the same bits as iq4xs_matmul
    least = B.iq4xs_linear_workspace_min_bytes(M, N, K)
    ws2 = torch.full((least,), 0xFF, dtype=torch.uint8, device="cuda")
    y3 = torch.full((M, N), float("nan"), device="cuda")
    B.iq4xs_linear(wd, N, K, xd, y3, ws2)
    torch.cuda.synchronize()
    assert np.array_equal(y3.cpu().numpy(), matmul_gpu(wd, N, K, qs, ds, M, path))
    r = gate_parity(y3.cpu().numpy()[:, rows], oracle_matmul(w, N, K, qs_o, d_o, rows))
    assert r is None, r


@pytest.mark.parametrize("M,N,K", [(1, 5120, 5120), (2, 12288, 5120), (3, 300, 1536),
                                   (4, 1024, 17408), (4, 256, 25600), (1, 34816, 5120)])
def test_linear_small_m_bitwise_and_workspace_q8(M, N, K):
    """The dispatcher's small-M path (the CUDA-core kernel across its launch
    shapes, or the warp-MMA kernel where the calibration measured it
    faster), a ragged N and a long K: bitwise the two separate calls, and
    the workspace holds the Q8_1 arrays."""
    rng = np.random.default_rng([51, M, N, K])
    w = synth.iq4xs_weights(rng, N, K, 1e-3)
    x = synth.activations(rng, M, K, outlier_frac=0.01)
    wd, xd = dev(w), dev(x)
    ws = torch.full((B.iq4xs_linear_workspace_bytes(M, N, K),), 0xFF, dtype=torch.uint8,
                    device="cuda")
    y = torch.full((M, N), float("nan"), device="cuda")
    B.iq4xs_linear(wd, N, K, xd, y, ws)
    torch.cuda.synchronize()
    yl = y.cpu().numpy()
    assert gate_written(yl) is None
    qs, ds = quantize_gpu(x)
    path = NAMES[B.iq4xs_select_path(M, N, K)]
    assert path in ("dp4a", "mma"), path
    assert np.array_equal(yl, matmul_gpu(wd, N, K, qs, ds, M, path))
    qs_o, d_o, s_o = oracle_q8(x)
    wsh = ws.cpu().numpy()
    assert np.array_equal(wsh[:M * K].view(np.int8).reshape(M, K), qs_o)
    off = (M * K + 15) // 16 * 16
    dsw = wsh[off:off + M * (K // 32) * 4].view(np.uint16).reshape(M, K // 32, 2)
    assert np.array_equal(dsw[:, :, 0], d_o) and np.array_equal(dsw[:, :, 1], s_o)
    rows = sample_rows(N, 24, seed=M)
    assert gate_parity(yl[:, rows], oracle_matmul(w, N, K, qs_o, d_o, rows)) is None


def test_linear_rejects_small_workspace():
    N, K, M = 256, 1024, 4
    w, x = synth.TINY.inputs(0, M=M)
    need = B.iq4xs_linear_workspace_bytes(M, N, K)
    ws = torch.empty((need - 16,), dtype=torch.uint8, device="cuda")
    y = torch.empty((M, N), device="cuda")
    with pytest.raises(B.IQ4XSError) as e:
        B.iq4xs_linear(dev(w), N, K, dev(x), y, ws)
    assert e.value.status == B.ERR_ARG


def test_linear_baseline_route_only_when_asked():
    """Above the advised threshold, linear(allow_baseline=True) takes the
    dequantize + bf16 GEMM route (bf16 precision: within a few 1e-2 of the
    oracle's row maximum, which also carries the Q8_1 rounding the route
    skips); without the opt-in the exact tensor-core path runs."""
    N, K, M = 256, 1024, 128
    w, x = synth.TINY.inputs(0, M=M)
    wd, xd = dev(w), dev(x)
    qs_o, d_o, _ = oracle_q8(x)
    rows = sample_rows(N, 32, seed=5)
    ref = oracle_matmul(w, N, K, qs_o, d_o, rows)
    B.iq4xs_set_baseline_threshold(64)
    try:
        assert B.iq4xs_select_path(M, N, K) == B.PATH_BASELINE
        yb = B.linear(wd, N, K, xd, allow_baseline=True)
        ye = B.linear(wd, N, K, xd)
        torch.cuda.synchronize()
    finally:
        B.iq4xs_set_baseline_threshold(0)
    yb, ye = yb.cpu().numpy(), ye.cpu().numpy()
    assert gate_written(yb) is None and gate_written(ye) is None
    assert gate_parity(ye[:, rows], ref) is None
    scale = np.abs(ref).max(axis=1, keepdims=True)
    err = np.abs(yb[:, rows] - ref) / scale
    assert 0 < err.max() < 5e-2, err.max()


@pytest.mark.parametrize("M", (1, 4, 16, 96))
def test_linear_on_pinned_host_buffers_is_bitwise_device(M):
    """x read from and y written to page-locked host memory by the kernels
    (the e2e form of the benchmark): bit-identical to device buffers, on
    both paths, with a ragged N tail and split K."""
    N, K = 1000, 4096
    rng = np.random.default_rng([77, M])
    w = dev(synth.iq4xs_weights(rng, N, K, 1e-3))
    x = synth.activations(rng, M, K, outlier_frac=0.01)
    ws = torch.empty((B.iq4xs_linear_workspace_bytes(M, N, K),), dtype=torch.uint8, device="cuda")
    yd = torch.full((M, N), float("nan"), device="cuda")
    B.iq4xs_linear(w, N, K, dev(x), yd, ws)
    hx = torch.from_numpy(x).pin_memory()
    hy = torch.full((M, N), float("nan")).pin_memory()
    B.iq4xs_linear(w, N, K, hx, hy, ws)
    torch.cuda.synchronize()
    assert gate_written(hy.numpy()) is None
    assert np.array_equal(hy.numpy().view(np.uint32), yd.cpu().numpy().view(np.uint32))
