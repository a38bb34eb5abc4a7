"""Q4_0 and IQ4_NL weights (32-weight blocks of 18 bytes) on the GPU through
the C ABI, against the oracle: every path (DP4A, warp MMA, tcgen05 in both
forms), ragged N tails, several M tiles, split K, every warp-MMA launch
configuration, full-size sampled rows; dequantization bit-exact; and the
IQ4_NL / IQ4_XS identity (uniform sub-block scale) bit for bit."""
import numpy as np
import pytest
import torch

import oracle
from _gates import gate_independent, gate_parity, gate_written
from _gpu import dev, matmul_gpu, oracle_q8, prepare_gpu, quantize_gpu, sample_rows
from iq4_xs_quantized_gb300 import binding as B
from iq4_xs_quantized_gb300 import synth

pytestmark = pytest.mark.gpu

FORMATS = [("q4_0", B.WTYPE_Q4_0), ("iq4_nl", B.WTYPE_IQ4_NL)]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from iq4_xs_quantized_gb300 import build
    build.build()
    B.load()
    yield
    assert B.iq4xs_last_device_error() == 0


def _oracle_wt(wt, w, N, K, qs, d_h, rows=None):
    orc = oracle.get()
    nt = max(1, min(16, oracle.threads_available()))
    if rows is not None:
        w = np.ascontiguousarray(w.reshape(N, -1)[rows])
        N = len(rows)
    return orc.matmul_wt(wt, w, N, K, qs, d_h, nthreads=nt)


def _matmul_wt(wd, wt, N, K, qs, ds, M, path):
    y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    B.iq4xs_matmul_wt(wd, wt, N, K, qs, ds, M, y, path)
    torch.cuda.synchronize()
    return y.cpu().numpy()


def _independent(wt, w, N, K, qs, d_h):
    W = oracle.get().dequantize_wt(wt, w, N, K)
    xhat = qs.astype(np.float32) * np.repeat(d_h.view(np.float16).astype(np.float32), 32, axis=1)
    prev = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = False
    try:
        return (dev(xhat) @ dev(W).T).cpu().numpy()
    finally:
        torch.backends.cuda.matmul.allow_tf32 = prev


@pytest.mark.parametrize("name,wt", FORMATS)
@pytest.mark.parametrize("N,K", [(300, 2048), (128, 1024), (200, 768)])
def test_formats_match_oracle_on_every_path(name, wt, N, K):
    rng = np.random.default_rng([41, wt, N, K])
    w = synth.block32_weights(rng, N, K, 2e-3)
    wd = dev(w)
    Ms = (1, 2, 3, 4, 5, 8, 16, 33, 96, 130)
    x = synth.activations(rng, max(Ms), K, outlier_frac=0.01)
    for M in Ms:
        qs, ds = quantize_gpu(x[:M])
        qs_o, d_o, _ = oracle_q8(x[:M])
        ref = _oracle_wt(wt, w, N, K, qs_o, d_o)
        paths = [B.PATH_AUTO, B.PATH_DP4A] + ([B.PATH_TC, "tcp", B.PATH_MMA] if K % 512 == 0 else [])
        for path in paths:
            if path == "tcp":
                y = matmul_gpu(wd, N, K, None, None, M, "tcp", op=prepare_gpu(x[:M]), wtype=wt)
            else:
                y = _matmul_wt(wd, wt, N, K, qs, ds, M, path)
            assert gate_written(y) is None, (name, M, path)
            r = gate_parity(y, ref)
            assert r is None, (name, N, K, M, path, r)
        assert gate_independent(y, _independent(wt, w, N, K, qs_o, d_o)) is None


@pytest.mark.parametrize("name,wt", FORMATS)
@pytest.mark.parametrize("N,K", [(4096, 4096), (5120, 5120), (12288, 5120)])
def test_formats_full_size_sampled_rows(name, wt, N, K):
    rng = np.random.default_rng([42, wt, N])
    w = synth.block32_weights(rng, N, K, 1e-3)
    wd = dev(w)
    rows = sample_rows(N, 48, seed=wt)
    for M in ((1, 2, 4, 16, 64, 96) if N == 4096 else (1, 2, 16)):
        x = synth.activations(rng, M, K)
        qs, ds = quantize_gpu(x)
        qs_o, d_o, _ = oracle_q8(x)
        ref = _oracle_wt(wt, w, N, K, qs_o, d_o, rows)
        for path in (B.PATH_AUTO, B.PATH_MMA) if M <= 32 else (B.PATH_AUTO,):
            y = _matmul_wt(wd, wt, N, K, qs, ds, M, path)
            assert gate_written(y) is None
            assert gate_parity(y[:, rows], ref) is None, (name, M, path)


@pytest.mark.parametrize("name,wt", FORMATS)
@pytest.mark.parametrize("rows,splits,occ", [(32, 1, 0), (64, 3, 0), (96, 5, 0), (128, 8, 0), (192, 1, 0),
                                             (256, 2, 0), (32, 4, 2), (64, 1, 2)])
def test_formats_mma_launch_configs(name, wt, rows, splits, occ):
    """Every warp-MMA launch the 18-byte formats can take (rows per CTA,
    K split over a cluster, one or two CTAs per SM), with ragged row tiles
    and activation tiles of 8 to 32 rows."""
    rng = np.random.default_rng([45, wt, rows, splits])
    N, K = 300, 4608
    w = synth.block32_weights(rng, N, K, 2e-3)
    wd = dev(w)
    B.iq4xs_test_mma_config(rows, splits, occ)
    try:
        for M in (1, 8, 13, 24, 40):
            x = synth.activations(rng, M, K, outlier_frac=0.01)
            qs, ds = quantize_gpu(x)
            qs_o, d_o, _ = oracle_q8(x)
            y = _matmul_wt(wd, wt, N, K, qs, ds, M, B.PATH_MMA)
            assert gate_written(y) is None
            assert gate_parity(y, _oracle_wt(wt, w, N, K, qs_o, d_o)) is None, (name, rows, splits, occ, M)
    finally:
        B.iq4xs_test_mma_config(0, 0, 0)


@pytest.mark.parametrize("name,wt", FORMATS + [("iq4_xs", B.WTYPE_IQ4_XS)])
def test_formats_dequantize_bit_exact(name, wt):
    N, K = 70, 1536
    rng = np.random.default_rng([43, wt])
    w = synth.weights_for(wt, rng, N, K, 2e-3)
    f32, b16 = oracle.get().dequantize_wt(wt, w, N, K, bf16=True)
    out = torch.full((N, K), float("nan"), dtype=torch.float32, device="cuda")
    B.iq4xs_dequantize_wt(dev(w), wt, N, K, out)
    ob = torch.zeros((N, K), dtype=torch.bfloat16, device="cuda")
    B.iq4xs_dequantize_wt(dev(w), name, N, K, ob)
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().numpy().view(np.uint32), f32.view(np.uint32))
    assert np.array_equal(ob.view(torch.int16).cpu().numpy().view(np.uint16), b16)


def test_iq4nl_equals_iq4xs_with_uniform_scale_bitwise():
    """IQ4_XS blocks whose eight ls are all L equal IQ4_NL blocks with
    d' = d*(L-32) (exact in fp16): same weights, same integer dots and the
    same fp32 scales, so both kernels give the same bits on both paths."""
    N, K = 256, 1024
    rng = np.random.default_rng(44)
    d, L = np.float16(0.0078125), 45
    qs_bytes = rng.integers(0, 256, (N, K // 256, 128), dtype=np.uint8)
    xs = np.zeros((N, K // 256, 136), np.uint8)
    xs[:, :, 0:2] = np.frombuffer(d.tobytes(), np.uint8)
    ls = [L] * 8
    sh = sum(((v >> 4) & 3) << (2 * j) for j, v in enumerate(ls))
    xs[:, :, 2] = sh & 0xFF
    xs[:, :, 3] = sh >> 8
    for j, v in enumerate(ls):
        xs[:, :, 4 + j // 2] |= np.uint8((v & 0xF) << (4 * (j % 2)))
    xs[:, :, 8:] = qs_bytes
    nl = np.zeros((N, K // 32, 18), np.uint8)
    nl[:, :, 0:2] = np.frombuffer(np.float16(float(d) * (L - 32)).tobytes(), np.uint8)
    nl[:, :, 2:] = qs_bytes.reshape(N, K // 256, 8, 16).reshape(N, K // 32, 16)
    w_xs, w_nl = dev(xs.reshape(N, -1)), dev(nl.reshape(N, -1))
    x = synth.activations(rng, 40, K)
    for M in (1, 3, 40):
        qs, ds = quantize_gpu(x[:M])
        for path in (B.PATH_DP4A, B.PATH_TC, B.PATH_MMA):
            a = _matmul_wt(w_xs, B.WTYPE_IQ4_XS, N, K, qs, ds, M, path)
            b = _matmul_wt(w_nl, B.WTYPE_IQ4_NL, N, K, qs, ds, M, path)
            assert gate_written(a) is None
            assert np.array_equal(a, b), (M, path)
        op = prepare_gpu(x[:M])
        a = matmul_gpu(w_xs, N, K, None, None, M, "tcp", op=op, wtype=B.WTYPE_IQ4_XS)
        b = matmul_gpu(w_nl, N, K, None, None, M, "tcp", op=op, wtype=B.WTYPE_IQ4_NL)
        assert gate_written(a) is None
        assert np.array_equal(a, b), (M, "tcp")


@pytest.mark.parametrize("name,wt", FORMATS)
def test_formats_linear_one_call(name, wt):
    """iq4xs_linear for Q4_0 / IQ4_NL weights on the dispatcher's path per M
    (CUDA cores, warp MMA, tcgen05 with the prepared operand): against the
    oracle, and bitwise the separate quantize + matmul calls."""
    rng = np.random.default_rng([47, wt])
    N, K = 300, 2048
    w = synth.block32_weights(rng, N, K, 2e-3)
    wd = dev(w)
    names = {B.PATH_DP4A: "dp4a", B.PATH_MMA: "mma", B.PATH_TC: "tcp", B.PATH_BASELINE: "tcp"}
    for M in (1, 3, 8, 16, 40):
        x = synth.activations(rng, M, K, outlier_frac=0.01)
        xd = dev(x)
        ws = torch.full((B.iq4xs_linear_workspace_bytes(M, N, K),), 0xFF, dtype=torch.uint8, device="cuda")
        y = torch.full((M, N), float("nan"), device="cuda")
        B.iq4xs_linear(wd, N, K, xd, y, ws, wtype=wt)
        torch.cuda.synchronize()
        yl = y.cpu().numpy()
        assert gate_written(yl) is None
        qs_o, d_o, _ = oracle_q8(x)
        assert gate_parity(yl, _oracle_wt(wt, w, N, K, qs_o, d_o)) is None, (name, M)
        path = names[B.iq4xs_select_path(M, N, K)]
        qs, ds = quantize_gpu(x)
        if path == "tcp":
            y2 = matmul_gpu(wd, N, K, None, None, M, "tcp", op=prepare_gpu(x), wtype=wt)
        else:
            y2 = _matmul_wt(wd, wt, N, K, qs, ds, M, {"dp4a": B.PATH_DP4A, "mma": B.PATH_MMA}[path])
        assert np.array_equal(yl, y2), (name, M, path)
