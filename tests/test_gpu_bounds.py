"""The bounds-checked debug build on the GPU (libiq4xs_bounds.so: the same
sources compiled with IQ4XS_BOUNDS_CHECK, standing in for a memory checker).

Every kernel, on every path and launch configuration, runs small shapes that
span several tiles and end in ragged tails; each result must match the
oracle as in the parity suite, and the device error word must stay clean:
no checked global access, TMA box origin or computed shared-memory range
left its buffer.  Negative control: with a test margin that treats the last
bytes of every global buffer as outside it (no access ever leaves a buffer),
each kernel must report a bounds code from its own site range."""
import numpy as np
import pytest
import torch

import oracle
from _gates import gate_parity, gate_written
from _gpu import check_q8, dev, oracle_matmul, oracle_q8, prepare_gpu, quantize_gpu, run_and_gate
from iq4_xs_quantized_gb300 import binding as B
from iq4_xs_quantized_gb300 import synth

pytestmark = pytest.mark.gpu

# site ranges of the kernels (code = 0x200 + site)
SITES = {"quantize": (0x01, 0x05), "dequantize": (0x10, 0x11), "dp4a": (0x20, 0x25),
         "mma": (0x30, 0x39), "tc": (0x40, 0x4A)}


@pytest.fixture(scope="module", autouse=True)
def _bounds_lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from iq4_xs_quantized_gb300 import build
    build.build()
    build.build(bounds_check=True)
    B.use(B.BOUNDS_LIB_PATH)
    try:
        assert B.iq4xs_bounds_checked()
        B.iq4xs_test_bounds_margin(0)
        B.iq4xs_last_device_error()
        yield
        assert B.iq4xs_last_device_error() == 0
    finally:
        B.iq4xs_test_bounds_margin(0)
        B.iq4xs_test_mma_config(0, 0, 0)
        B.use(None)
    assert not B.iq4xs_bounds_checked()


def _clean():
    code = B.iq4xs_last_device_error()
    assert code == 0, f"bounds code {code:#x}"


# ------------------------------------------------------------- clean runs
@pytest.mark.parametrize("M,K", [(1, 1024), (5, 4352), (33, 2560), (130, 1536)])
def test_quantize_both_forms_clean(M, K):
    x = synth.activations(np.random.default_rng([M, K]), M, K, outlier_frac=0.01)
    qs, ds = quantize_gpu(x)
    check_q8(x, qs, ds)
    prepare_gpu(x, qs, ds)
    _clean()


def test_dequantize_every_format_clean():
    rng = np.random.default_rng(5)
    N, K = 37, 1280
    orc = oracle.get()
    for wt in (B.WTYPE_IQ4_XS, B.WTYPE_Q4_0, B.WTYPE_IQ4_NL):
        w = synth.iq4xs_weights(rng, N, K, 2e-3) if wt == B.WTYPE_IQ4_XS else synth.block32_weights(rng, N, K, 2e-3)
        out = torch.full((N, K), float("nan"), dtype=torch.float32, device="cuda")
        B.iq4xs_dequantize_wt(dev(w), wt, N, K, out)
        outb = torch.full((N, K), float("nan"), dtype=torch.bfloat16, device="cuda")
        B.iq4xs_dequantize_wt(dev(w), wt, N, K, outb)
        torch.cuda.synchronize()
        f32, b16 = (orc.dequantize(w, N, K, bf16=True) if wt == B.WTYPE_IQ4_XS
                    else orc.dequantize_wt(wt, w, N, K, bf16=True))
        assert np.array_equal(out.cpu().numpy().view(np.uint32), f32.view(np.uint32))
        assert np.array_equal(outb.view(torch.int16).cpu().numpy().view(np.uint16), b16)
        _clean()


@pytest.mark.parametrize("path,Ms", [("dp4a", (1, 2, 3, 5, 8, 9)), ("mma", (1, 7, 12, 20, 32)),
                                     ("tc", (3, 17, 48, 130)), ("tcp", (3, 17, 48, 130))])
@pytest.mark.parametrize("N,K", [(300, 4608), (129, 512)])
def test_matmul_paths_clean(path, Ms, N, K):
    rng = np.random.default_rng([N, K])
    w = synth.iq4xs_weights(rng, N, K, 2e-3)
    for M in Ms:
        x = synth.activations(rng, M, K, outlier_frac=0.01)
        run_and_gate(w, N, K, x, path, independent=False)
        _clean()


@pytest.mark.parametrize("rows,splits,occ", [(32, 1, 0), (64, 3, 0), (128, 8, 0), (256, 2, 0), (96, 5, 0),
                                             (32, 4, 2), (64, 1, 2)])
def test_mma_launch_configs_clean(rows, splits, occ):
    rng = np.random.default_rng([rows, splits])
    N, K = 300, 4608
    w = synth.iq4xs_weights(rng, N, K, 2e-3)
    B.iq4xs_test_mma_config(rows, splits, occ)
    try:
        for M in (8, 16, 24):
            x = synth.activations(rng, M, K)
            run_and_gate(w, N, K, x, "mma", independent=False)
            _clean()
    finally:
        B.iq4xs_test_mma_config(0, 0, 0)


@pytest.mark.parametrize("K", (1536, 3584, 7168))
def test_tc_split_k_clean(K):
    """Clusters of 3, 7 and 7 ranks along K: the split-K slices move between
    the ranks' shared memory by bulk copies."""
    rng = np.random.default_rng(K)
    w = synth.iq4xs_weights(rng, 384, K, 1e-3)
    for path in ("tc", "tcp"):
        for M in (3, 40):
            run_and_gate(w, 384, K, synth.activations(rng, M, K), path, independent=False)
            _clean()


@pytest.mark.parametrize("wt", (B.WTYPE_Q4_0, B.WTYPE_IQ4_NL))
def test_block32_formats_clean(wt):
    rng = np.random.default_rng([wt, 7])
    N, K = 200, 1024
    w = synth.block32_weights(rng, N, K, 2e-3)
    for M in (1, 5, 40):
        x = synth.activations(rng, M, K)
        qs, ds = quantize_gpu(x)
        qs_o, d_o, _ = oracle_q8(x)
        ref = oracle.get().matmul_wt(wt, w, N, K, qs_o, d_o)
        for path in (B.PATH_DP4A, B.PATH_TC, B.PATH_MMA):
            y = torch.full((M, N), float("nan"), device="cuda")
            B.iq4xs_matmul_wt(dev(w), wt, N, K, qs, ds, M, y, path)
            torch.cuda.synchronize()
            assert gate_parity(y.cpu().numpy(), ref) is None
            _clean()


@pytest.mark.parametrize("path", ("dp4a", "mma", "tc"))
@pytest.mark.parametrize("T,topk,G", [(20, 4, 8), (3, 2, 70), (64, 8, 8)])
def test_grouped_clean(path, T, topk, G):
    W = synth.MoEWorkload("moe_bounds", seed=19, G=G, N=136, K=1024, topk=topk, tokens=(T,), d_scale=2e-3)
    _, rows_x, offsets = W.inputs(T)
    w = W.weights()
    qs, ds = quantize_gpu(rows_x)
    y = torch.full((rows_x.shape[0], W.N), float("nan"), device="cuda")
    B.iq4xs_matmul_grouped(dev(w.reshape(G, -1)), w.shape[1] * w.shape[2], G, W.N, W.K, qs, ds,
                           dev(offsets.astype(np.int32)), y, path=path)
    torch.cuda.synchronize()
    yn = y.cpu().numpy()
    assert gate_written(yn) is None
    qs_o, d_o, _ = oracle_q8(rows_x)
    for g in range(G):
        r0, r1 = int(offsets[g]), int(offsets[g + 1])
        if r1 > r0:
            assert gate_parity(yn[r0:r1], oracle_matmul(w[g], W.N, W.K, qs_o[r0:r1], d_o[r0:r1])) is None
    _clean()


@pytest.mark.parametrize("path", ("dp4a", "mma"))
@pytest.mark.parametrize("wt", (B.WTYPE_Q4_0, B.WTYPE_IQ4_NL))
def test_grouped_formats_clean(path, wt):
    G, T, topk = 8, 20, 4
    W = synth.MoEWorkload("moe_bounds_b18", seed=37, G=G, N=136, K=1024, topk=topk, tokens=(T,), d_scale=2e-3)
    _, rows_x, offsets = W.inputs(T)
    w = np.stack([synth.block32_weights(np.random.default_rng([37, wt, g]), W.N, W.K, 2e-3) for g in range(G)])
    qs, ds = quantize_gpu(rows_x)
    y = torch.full((rows_x.shape[0], W.N), float("nan"), device="cuda")
    B.iq4xs_matmul_grouped(dev(w.reshape(G, -1)), w.shape[1] * w.shape[2], G, W.N, W.K, qs, ds,
                           dev(offsets.astype(np.int32)), y, path=path, wtype=wt)
    torch.cuda.synchronize()
    yn = y.cpu().numpy()
    assert gate_written(yn) is None
    qs_o, d_o, _ = oracle_q8(rows_x)
    for g in range(G):
        r0, r1 = int(offsets[g]), int(offsets[g + 1])
        if r1 > r0:
            assert gate_parity(yn[r0:r1], oracle.get().matmul_wt(wt, w[g], W.N, W.K, qs_o[r0:r1], d_o[r0:r1])) is None
    _clean()


@pytest.mark.parametrize("M", (2, 40))
def test_linear_entry_points_clean(M):
    N, K = 256, 1024
    w, x = synth.TINY.inputs(0, M=M)
    wd, xd = dev(w), dev(x)
    ws = torch.empty((B.iq4xs_linear_workspace_bytes(M, N, K),), dtype=torch.uint8, device="cuda")
    y1 = torch.full((M, N), float("nan"), device="cuda")
    y2 = torch.full((M, N), float("nan"), device="cuda")
    B.iq4xs_linear(wd, N, K, xd, y1, ws)
    B.iq4xs_linear_static(wd, N, K, xd, y2)
    torch.cuda.synchronize()
    qs_o, d_o, _ = oracle_q8(x)
    ref = oracle_matmul(w, N, K, qs_o, d_o)
    for y in (y1, y2):
        assert gate_parity(y.cpu().numpy(), ref) is None
    _clean()


# ------------------------------------------------------- negative control
def _under_margin(run, kernel):
    """run() launches one kernel; with a 16-byte margin it must report a code
    of that kernel's site range (its inputs were made beforehand)."""
    _clean()
    B.iq4xs_test_bounds_margin(16)
    try:
        run()
        torch.cuda.synchronize()
    finally:
        B.iq4xs_test_bounds_margin(0)
    code = B.iq4xs_last_device_error()
    lo, hi = SITES[kernel]
    assert 0x200 + lo <= code <= 0x200 + hi, f"{kernel}: code {code:#x}"


def test_margin_reports_every_kernel():
    rng = np.random.default_rng(3)
    N, K, M = 300, 4608, 12
    w = synth.iq4xs_weights(rng, N, K, 2e-3)
    wd = dev(w)
    x = synth.activations(rng, M, K)
    xd = dev(x)
    qs, ds = B.alloc_activations(M, K, "cuda")
    B.iq4xs_quantize_q8_1(xd, qs, ds)
    op = B.alloc_tc_operand(M, K, "cuda")
    B.iq4xs_quantize_q8_1_tc(xd, qs, ds, op)
    y = torch.empty((M, N), device="cuda")
    out = torch.empty((N, K), device="cuda")
    torch.cuda.synchronize()
    _under_margin(lambda: B.iq4xs_quantize_q8_1(xd, qs, ds), "quantize")
    _under_margin(lambda: B.iq4xs_quantize_q8_1_tc(xd, qs, ds, op), "quantize")
    B.iq4xs_quantize_q8_1_tc(xd, qs, ds, op)  # restore the inputs
    _under_margin(lambda: B.iq4xs_dequantize(wd, N, K, out), "dequantize")
    for path, kernel in (("dp4a", "dp4a"), ("mma", "mma"), ("tc", "tc")):
        _under_margin(lambda: B.iq4xs_matmul(wd, N, K, qs, ds, M, y, path), kernel)
    _under_margin(lambda: B.iq4xs_matmul_tc_operand(wd, N, K, op, M, y), "tc")
    offsets = dev(np.array([0, 5, 5, M], dtype=np.int32))
    stride = N * (K // 256) * 136
    wg = dev(np.concatenate([w] * 3))
    for path in ("dp4a", "mma", "tc"):
        _under_margin(lambda: B.iq4xs_matmul_grouped(wg, stride, 3, N, K, qs, ds, offsets, y, path=path), path)
    w18 = dev(synth.block32_weights(rng, N, K, 2e-3))
    for path, kernel in ((B.PATH_DP4A, "dp4a"), (B.PATH_MMA, "mma"), (B.PATH_TC, "tc")):
        _under_margin(lambda: B.iq4xs_matmul_wt(w18, B.WTYPE_Q4_0, N, K, qs, ds, M, y, path), kernel)
    _clean()
