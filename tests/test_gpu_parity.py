"""CUDA path vs the CPU oracle, through the C ABI (needs an sm_103 GPU).

Q8_1 codes and scales are compared bit for bit; the matmul per output row
within 1e-5 relative to the fp64 oracle; every output buffer is NaN-poisoned
before the call and must come back fully written; an independent fp32
dequantize + matmul must differ from the result by a nonzero amount within
2e-3.  Full-size shapes are checked on sampled weight rows in the launch
configuration the benchmark times.
"""
import numpy as np
import pytest
import torch

import oracle
from _gates import gate_independent, gate_parity, gate_written
from _gpu import (check_q8, dev, independent_fp32, matmul_gpu, oracle_matmul, oracle_q8, prepare_gpu,
                  quantize_gpu, run_and_gate, sample_rows)
from _pins import make_block, parse_q8_cases
from iq4_xs_quantized_gb300 import binding as B
from iq4_xs_quantized_gb300 import synth

pytestmark = pytest.mark.gpu

# dp4a; tcgen05 from the Q8_1 arrays; tcgen05 from the prepared operand;
# warp-level MMA
PATHS = ("dp4a", "tc", "tcp", "mma")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from iq4_xs_quantized_gb300 import build
    build.build()
    B.load()
    yield
    assert B.iq4xs_last_device_error() == 0


# --------------------------------------------------------------------------- Q8_1
@pytest.mark.parametrize("wl,M", [("tiny_256x1024", 8), ("square_4096x4096", 96),
                                  ("decoder27b_9proj", 64), ("prefill_sweep", 512)])
def test_quantize_bit_exact(wl, M):
    W = synth.WORKLOADS[wl]
    idx = 0 if wl != "prefill_sweep" else 1
    _, K = W.shapes[idx]
    x = synth.activations(W.rng(idx, 99), M, K, W.outlier_frac, bf16_round=W.bf16_round)
    qs, ds = quantize_gpu(x)
    check_q8(x, qs, ds)


def test_quantize_closed_forms():
    cases = parse_q8_cases()
    x = np.zeros((len(cases), 256), np.float32)
    for i, c in enumerate(cases):
        x[i, :32] = c["x"]
        x[i, 32:64] = -c["x"] * np.float32(0.125)
    qs, ds = quantize_gpu(x)
    check_q8(x, qs, ds)
    q = qs.cpu().numpy()
    for i, c in enumerate(cases):
        assert np.array_equal(q[i, :32], c["q"]), c["name"]


# ------------------------------------------------------------------ matmul, tiny
TINY_MS_TC = (1, 2, 3, 8, 16, 17, 31, 33, 48, 64, 80, 96, 112, 127, 128, 129, 200, 257)


@pytest.mark.parametrize("M", (1, 2, 3, 4, 5, 8, 9, 16))
def test_matmul_tiny_dp4a(M):
    w, x = synth.TINY.inputs(0, M=M)
    run_and_gate(w, 256, 1024, x, "dp4a")


@pytest.mark.parametrize("M", TINY_MS_TC)
@pytest.mark.parametrize("form", ("tc", "tcp"))
def test_matmul_tiny_tc(M, form):
    w, x = synth.TINY.inputs(0, M=M)
    run_and_gate(w, 256, 1024, x, form)


TINY_MS_MMA = (1, 2, 3, 4, 7, 8, 9, 15, 16, 17, 24, 25, 32, 33, 40, 64, 96)


@pytest.mark.parametrize("M", TINY_MS_MMA)
def test_matmul_tiny_mma(M):
    w, x = synth.TINY.inputs(0, M=M)
    run_and_gate(w, 256, 1024, x, "mma")


# Every tile height (32..256 weight rows per CTA: 1..8 fragments per warp,
# odd and even) and K split of the warp-MMA path, for every activation tile
# width (8, 16, 24, 32 rows), on a ragged N; K = 4608 is 9 super-block pairs,
# so the splits take unequal shares.
@pytest.mark.parametrize("rows", (32, 96, 128, 160, 224, 256))
@pytest.mark.parametrize("splits", (1, 3, 8))
def test_matmul_mma_configs(rows, splits):
    rng = np.random.default_rng([rows, splits])
    N, K = 300, 4608
    w = synth.iq4xs_weights(rng, N, K, 1e-3)
    B.iq4xs_test_mma_config(rows, splits, 1)
    try:
        for M in (5, 13, 21, 32):
            x = synth.activations(rng, M, K, outlier_frac=0.01)
            run_and_gate(w, N, K, x, "mma")
    finally:
        B.iq4xs_test_mma_config(0, 0, 0)


def test_mma_measured_launch_is_taken():
    """An installed launch-table entry decides the launch for its exact shape
    and tile height (and only there); the result still matches the oracle."""
    rng = np.random.default_rng(31)
    N, K = 600, 4608
    w = synth.iq4xs_weights(rng, N, K, 1e-3)
    try:
        B.iq4xs_set_mma_launch_table([(N, K, 16, 96, 3, 1), (N, K, 8, 64, 2, 2)])
        assert B.iq4xs_mma_launch_config(12, N, K) == (96, 3, 1)
        assert B.iq4xs_mma_launch_config(5, N, K) == (64, 2, 2)
        for M in (5, 12):
            run_and_gate(w, N, K, synth.activations(rng, M, K), "mma")
    finally:
        B.reset_dispatch()


def test_calibrated_launch_table_is_taken():
    """Every measured launch the calibration stored is one the kernel holds,
    and the call for that shape and tile height takes it."""
    from iq4_xs_quantized_gb300 import calibrate
    table = calibrate.load_table() or {}
    entries = table.get("mma_launch", [])
    B.reset_dispatch()
    for N, K, mt, R, S, occ in entries:
        assert B.iq4xs_mma_launch_config(mt, N, K) == (R, S, occ), (N, K, mt)


def test_mma_launch_config_reports_the_launch():
    """The reported launch is the forced one when forced, and the model's
    own choice covers N with at most 256 rows per CTA and at most 8 splits."""
    for c in ((96, 3, 1), (64, 2, 2), (256, 1, 1)):
        B.iq4xs_test_mma_config(*c)
        try:
            assert B.iq4xs_mma_launch_config(8, 4096, 4608) == c
        finally:
            B.iq4xs_test_mma_config(0, 0, 0)
    for M, N, K in ((1, 4096, 4096), (16, 34816, 5120), (32, 5120, 17408), (8, 300, 512)):
        r, sp, o = B.iq4xs_mma_launch_config(M, N, K)
        assert r % 32 == 0 and 32 <= r <= 256 and 1 <= sp <= min(8, K // 512) and o in (1, 2)


# The half-shared-memory tiles (two CTAs per SM): 32 and 64 rows at 8
# activation rows, 32 at 16 and 24 (M = 32 falls back to one CTA per SM).
@pytest.mark.parametrize("rows,splits", [(32, 1), (64, 2), (64, 5), (32, 8)])
def test_matmul_mma_two_ctas_per_sm(rows, splits):
    rng = np.random.default_rng([rows, splits, 2])
    N, K = 1000, 5120
    w = synth.iq4xs_weights(rng, N, K, 1e-3)
    B.iq4xs_test_mma_config(rows, splits, 2)
    try:
        for M in (1, 8, 9, 16, 24, 32):
            x = synth.activations(rng, M, K, outlier_frac=0.01)
            run_and_gate(w, N, K, x, "mma")
    finally:
        B.iq4xs_test_mma_config(0, 0, 0)


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("N", (1, 7, 130, 200, 383))
def test_matmul_ragged_n(path, N):
    rng = np.random.default_rng(N)
    w = synth.iq4xs_weights(rng, N, 1024, 2e-3)
    for M in (1, 5, 40):
        x = synth.activations(rng, M, 1024)
        run_and_gate(w, N, 1024, x, path)


# With 3 row tiles every split fits one wave, so the tcgen05 path takes the
# largest useful split: K = 512 / 1536 / 2560 / 3072 / 3584 / 4096 give
# clusters of 1 / 3 / 5 / 6 / 7 / 8 (uneven row shares of the split-K
# reduction at 3, 5, 6, 7), 5120 and 7168 clusters of 5 and 7.
@pytest.mark.parametrize("K", (512, 1536, 2560, 3072, 3584, 4096, 5120, 7168))
@pytest.mark.parametrize("path", PATHS)
def test_matmul_k_variants(K, path):
    rng = np.random.default_rng(K)
    w = synth.iq4xs_weights(rng, 384, K, 1e-3)
    for M in (3, 24):
        x = synth.activations(rng, M, K, outlier_frac=0.01)
        run_and_gate(w, 384, K, x, path)


def test_matmul_k256_dp4a_only():
    rng = np.random.default_rng(5)
    w = synth.iq4xs_weights(rng, 64, 256, 2e-3)
    x = synth.activations(rng, 4, 256)
    run_and_gate(w, 64, 256, x, "dp4a")
    for K in (768, 1280):  # an odd number of super-blocks: rows not 16-byte strided
        w2 = synth.iq4xs_weights(rng, 200, K, 2e-3)
        for M in (3, 20):
            run_and_gate(w2, 200, K, synth.activations(rng, M, K), "auto")
            assert B.iq4xs_select_path(M, 200, K) == B.PATH_DP4A
    qs, ds = quantize_gpu(x)
    y = torch.empty((4, 64), dtype=torch.float32, device="cuda")
    with pytest.raises(B.IQ4XSError) as e:
        B.iq4xs_matmul(dev(w), 64, 256, qs, ds, 4, y, "mma")
    assert e.value.status == B.ERR_SHAPE
    qs, ds = quantize_gpu(x)
    y = torch.empty((4, 64), dtype=torch.float32, device="cuda")
    with pytest.raises(B.IQ4XSError) as e:
        B.iq4xs_matmul(dev(w), 64, 256, qs, ds, 4, y, "tc")
    assert e.value.status == B.ERR_SHAPE
    with pytest.raises(B.IQ4XSError) as e:
        B.iq4xs_matmul_tc_operand(dev(w), 64, 256, prepare_gpu(x), 4, y)
    assert e.value.status == B.ERR_SHAPE


@pytest.mark.parametrize("path", PATHS)
def test_matmul_ldy_padding(path):
    w, x = synth.TINY.inputs(0, M=6)
    run_and_gate(w, 256, 1024, x, path, ldy=300)


# ---------------------------------------------------------- exactness, degenerate
@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("M", (1, 16, 96))
def test_matmul_integer_exact(path, M):
    """d = 1, ls = 33 and integer activations with a +-127 in every block make
    every scale 1: y is an integer below 2^24 and must match exactly."""
    rng = np.random.default_rng(M)
    N, K = 256, 1024
    w = np.stack([np.concatenate([make_block(1.0, [33] * 8, rng.integers(0, 256, 128))
                                  for _ in range(K // 256)]) for _ in range(N)])
    x = rng.integers(-126, 127, (M, K)).astype(np.float32)
    x[:, ::32] = 127 * rng.choice([-1, 1], (M, K // 32))
    y, yo = run_and_gate(w, N, K, x, path, independent=False)
    assert np.array_equal(y.astype(np.float64), yo)


@pytest.mark.parametrize("path", PATHS)
def test_matmul_zero_scales_and_zero_activations(path):
    rng = np.random.default_rng(3)
    N, K, M = 256, 1024, 20
    w = np.stack([np.concatenate([make_block(0.5, [32] * 8, rng.integers(0, 256, 128))
                                  for _ in range(K // 256)]) for _ in range(N)])
    x = rng.standard_normal((M, K)).astype(np.float32)
    y, _ = run_and_gate(w, N, K, x, path, independent=False)
    assert np.all(y == 0)
    w2, _ = synth.TINY.inputs(0, M=1)
    y2, _ = run_and_gate(w2, N, K, np.zeros((M, K), np.float32), path, independent=False)
    assert np.all(y2 == 0)


@pytest.mark.parametrize("path", PATHS)
def test_matmul_extreme_magnitudes(path):
    """Largest fp16 d with the largest |ls-32| and |kv|; activations near the
    top of the fp16 scale range and down in its subnormal range."""
    rng = np.random.default_rng(4)
    N, K, M = 128, 512, 4
    w = np.stack([np.concatenate([make_block(65504.0, rng.choice([0, 63], 8), rng.integers(0, 256, 128))
                                  for _ in range(K // 256)]) for _ in range(N)])
    x = (rng.standard_normal((M, K)) * 1e5).astype(np.float32)
    run_and_gate(w, N, K, x, path)
    # activation scales in the fp16 subnormal range
    run_and_gate(w, N, K, (x * np.float32(1e-10)).astype(np.float32), path)


# ------------------------------------------------ full-size shapes, sampled rows
def _full_case(wl, shape_index, M, path, nrows=48):
    W = synth.WORKLOADS[wl]
    N, K = W.shapes[shape_index]
    w, x = W.inputs(shape_index, M=M)
    run_and_gate(w, N, K, x, path, rows=sample_rows(N, nrows, seed=M))


@pytest.mark.parametrize("M", synth.SQUARE.ms)
def test_full_square(M):
    _full_case("square_4096x4096", 0, M, "auto")  # the dispatcher's choice, as the benchmark runs it
    _full_case("square_4096x4096", 0, M, "tcp")
    _full_case("square_4096x4096", 0, M, "mma")
    _full_case("square_4096x4096", 0, M, "tc")
    if M <= 16:
        _full_case("square_4096x4096", 0, M, "dp4a")


@pytest.mark.parametrize("shape_index", range(9))
def test_full_decoder_shapes(shape_index):
    # dp4a at M = 1 and 2 meets all three launch shapes across these grids
    # (1024 rows: 64 CTAs; 5120-6144: 320-384; 10240-34816: 640-2176)
    for M, path in ((1, "dp4a"), (2, "dp4a"), (16, "tc"), (64, "tc"), (16, "tcp"), (64, "tcp"),
                    (1, "mma"), (4, "mma"), (8, "mma"), (16, "mma"), (32, "mma")):
        _full_case("decoder27b_9proj", shape_index, M, path, nrows=24)


@pytest.mark.parametrize("M", (96, 256, 512))
@pytest.mark.parametrize("shape_index", (0, 1))
def test_full_prefill(shape_index, M):
    _full_case("prefill_sweep", shape_index, M, "tc", nrows=16)
    _full_case("prefill_sweep", shape_index, M, "tcp", nrows=16)


# ------------------------------------------------------------------- dequantize
def test_matmul_max_m_every_path():
    """The largest M the boundary takes (32768 rows: 1024 warp-MMA activation
    tiles, 256 tcgen05 tiles, 4096 dp4a passes) on a ragged N, every output
    against the oracle."""
    rng = np.random.default_rng(32768)
    M, N, K = 32768, 135, 512
    w = synth.iq4xs_weights(rng, N, K, 2e-3)
    x = synth.activations(rng, M, K)
    qs, ds = quantize_gpu(x)
    qs_o, d_o = check_q8(x, qs, ds)
    yo = oracle_matmul(w, N, K, qs_o, d_o)
    op = prepare_gpu(x, qs, ds)
    for path in PATHS:
        y = matmul_gpu(dev(w), N, K, qs, ds, M, path, op=op if path == "tcp" else None)
        assert gate_written(y) is None, path
        r = gate_parity(y, yo)
        assert r is None, (path, r)


def test_dequantize_bit_exact():
    rng = np.random.default_rng(21)
    N, K = 300, 2048
    w = synth.iq4xs_weights(rng, N, K, 2e-3)
    f32_o, b16_o = oracle.get().dequantize(w, N, K, bf16=True)
    wd = dev(w)
    out = torch.full((N, K), float("nan"), dtype=torch.float32, device="cuda")
    B.iq4xs_dequantize(wd, N, K, out)
    assert np.array_equal(out.cpu().numpy().view(np.uint32), f32_o.view(np.uint32))
    outb = torch.full((N, K), float("nan"), dtype=torch.bfloat16, device="cuda")
    B.iq4xs_dequantize(wd, N, K, outb)
    assert np.array_equal(outb.view(torch.int16).cpu().numpy().view(np.uint16), b16_o)


# --------------------------------------------------------------------- dispatch
def test_auto_matches_explicit_path():
    """AUTO runs exactly the kernel the installed crossovers name (outputs
    bit-identical to the explicit path's), classes overriding the defaults."""
    w, x = synth.TINY.inputs(0, M=8)
    qs, ds = quantize_gpu(x)
    wd = dev(w)
    try:
        B.iq4xs_set_crossover_classes([])
        B.iq4xs_set_mma_crossover_classes([])
        for cross, mma, expect in ((8, 8, "dp4a"), (2, 8, "mma"), (2, 4, "tc"), (9, 2, "dp4a")):
            B.iq4xs_set_crossover(cross)
            B.iq4xs_set_mma_crossover(mma)
            assert B.iq4xs_select_path(8, 256, 1024) == B.PATHS[expect]
            ya = matmul_gpu(wd, 256, 1024, qs, ds, 8, "auto")
            ye = matmul_gpu(wd, 256, 1024, qs, ds, 8, expect)
            assert np.array_equal(ya, ye), expect
        B.iq4xs_set_crossover(2)
        B.iq4xs_set_mma_crossover(4)
        B.iq4xs_set_mma_crossover_classes([(256 * 1024, 16)])  # this matrix's class: MMA to M = 16
        assert B.iq4xs_select_path(8, 256, 1024) == B.PATH_MMA
        assert B.iq4xs_select_path(8, 128, 1024) == B.PATH_TC  # below the class: the default
    finally:
        B.reset_dispatch()  # defaults, then the calibrated table


# ------------------------------------------------------------ negative controls
def test_gate_fires_when_no_kernel_runs():
    y = torch.full((4, 256), float("nan"), device="cuda").cpu().numpy()
    assert gate_written(y) is not None


@pytest.mark.parametrize("path", PATHS)
def test_gate_fires_on_one_corrupted_weight_byte(path):
    """Plant one flipped qs byte in the oracle's copy of W: the parity gate
    must fail for the row that holds it."""
    w, x = synth.TINY.inputs(0, M=4)
    qs, ds = quantize_gpu(x)
    qs_o, d_o, _ = oracle_q8(x)
    y = matmul_gpu(dev(w), 256, 1024, qs, ds, 4, path, op=prepare_gpu(x) if path == "tcp" else None)
    bad = w.copy()
    bad[17, 136 * 2 + 8 + 40] ^= 0x5A
    assert gate_parity(y, oracle_matmul(w, 256, 1024, qs_o, d_o)) is None
    assert gate_parity(y, oracle_matmul(bad, 256, 1024, qs_o, d_o)) is not None
