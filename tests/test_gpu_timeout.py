"""The tensor-core kernels' bounded waits, made to run out in the allowed
way: one W stage is left unissued (a barrier that nothing completes), so the
consumers' wait for it ends after its 2 s limit instead of hanging.  The call
returns, the device error word reports the stage timeout through
iq4xs_last_device_error (IQ4XS_ERR_TIMEOUT; code 0x101 on tcgen05, 0x10B on
the warp-MMA kernel, dense and persistent grouped), the CTAs drained their
copies (and freed their tensor memory), and the next ordinary call on the
same context is correct."""
import ctypes

import numpy as np
import pytest
import torch

from _gates import gate_parity, gate_written
from _gpu import dev, matmul_gpu, oracle_matmul, oracle_q8, quantize_gpu
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
    assert B.iq4xs_last_device_error() == 0
    yield
    B.iq4xs_test_skip_w_stage(-1)
    assert B.iq4xs_last_device_error() == 0


def test_unissued_w_stage_times_out_and_context_stays_usable():
    # K = 512: one W stage per CTA and no K split (one CTA per row tile);
    # 256 rows = two CTAs, both waiting on their unissued stage 0.
    rng = np.random.default_rng(9)
    N, K, M = 256, 512, 16
    w = synth.iq4xs_weights(rng, N, K, 2e-3)
    x = synth.activations(rng, M, K)
    wd = dev(w)
    qs, ds = quantize_gpu(x)
    y = torch.full((M, N), float("nan"), device="cuda")
    B.iq4xs_test_skip_w_stage(0)
    B.iq4xs_matmul(wd, N, K, qs, ds, M, y, "tc")
    torch.cuda.synchronize()  # returns: the wait was bounded
    code = ctypes.c_int(-1)
    assert B.load().iq4xs_last_device_error(ctypes.byref(code)) == B.ERR_TIMEOUT
    assert code.value == 0x101
    assert B.iq4xs_last_device_error() == 0  # read and cleared
    # the same context, the next ordinary calls: correct results
    qs_o, d_o, _ = oracle_q8(x)
    ref = oracle_matmul(w, N, K, qs_o, d_o)
    for path in ("tc", "dp4a", "tc"):
        y2 = matmul_gpu(wd, N, K, qs, ds, M, path)
        assert gate_written(y2) is None
        r = gate_parity(y2, ref)
        assert r is None, (path, r)
    assert B.iq4xs_last_device_error() == 0


def _expect_timeout(code_expected):
    code = ctypes.c_int(-1)
    assert B.load().iq4xs_last_device_error(ctypes.byref(code)) == B.ERR_TIMEOUT
    assert code.value == code_expected, hex(code.value)
    assert B.iq4xs_last_device_error() == 0  # read and cleared


def test_mma_unissued_stage_times_out_and_context_stays_usable():
    """The warp-MMA kernel (dense form, K = 512: one stage per CTA): its
    consumers' wait for the unissued stage runs out (code 0x10B), the CTAs
    drain and exit, and the next calls are correct."""
    rng = np.random.default_rng(10)
    N, K, M = 256, 512, 8
    w = synth.iq4xs_weights(rng, N, K, 2e-3)
    x = synth.activations(rng, M, K)
    wd = dev(w)
    qs, ds = quantize_gpu(x)
    y = torch.full((M, N), float("nan"), device="cuda")
    B.iq4xs_test_skip_w_stage(0)
    B.iq4xs_matmul(wd, N, K, qs, ds, M, y, "mma")
    torch.cuda.synchronize()  # returns: the wait was bounded
    _expect_timeout(0x10B)
    qs_o, d_o, _ = oracle_q8(x)
    ref = oracle_matmul(w, N, K, qs_o, d_o)
    for path in ("mma", "dp4a", "mma"):
        y2 = matmul_gpu(wd, N, K, qs, ds, M, path)
        assert gate_written(y2) is None
        r = gate_parity(y2, ref)
        assert r is None, (path, r)
    assert B.iq4xs_last_device_error() == 0


@pytest.mark.parametrize("stage", (2, 3))
def test_grouped_mma_unissued_stage_times_out_and_context_stays_usable(stage):
    """The persistent grouped warp-MMA form with more work items than CTAs
    (64 experts x 8 row tiles): each CTA's second item (stages 2 and 3 at
    K = 1024) loses its first stage -- the one that publishes the item's
    descriptor -- or its second.  Every consumer warp leaves the item loop
    together, the producer stops issuing and drains, the call returns with
    code 0x10B, and the next grouped call is correct."""
    W = synth.MoEWorkload("moe_timeout", seed=29, G=64, N=1024, K=1024, topk=4, tokens=(40,),
                          d_scale=2e-3)
    _, rows_x, offsets = W.inputs(40)
    w = W.weights()
    G, N, K = W.G, W.N, W.K
    stride = w.shape[1] * w.shape[2]
    wd = dev(w.reshape(G, -1))
    qs, ds = quantize_gpu(rows_x)
    off_d = dev(offsets.astype(np.int32))
    M = rows_x.shape[0]
    assert int((np.diff(offsets) > 0).sum()) * (N // 128) > 2 * 152  # several items per CTA
    y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    B.iq4xs_test_skip_w_stage(stage)
    B.iq4xs_matmul_grouped(wd, stride, G, N, K, qs, ds, off_d, y, path="mma")
    torch.cuda.synchronize()
    _expect_timeout(0x10B)
    y2 = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    B.iq4xs_matmul_grouped(wd, stride, G, N, K, qs, ds, off_d, y2, path="mma")
    torch.cuda.synchronize()
    yn = y2.cpu().numpy()
    assert gate_written(yn) is None
    qs_o, d_o, _ = oracle_q8(rows_x)
    for g in range(G):
        r0, r1 = int(offsets[g]), int(offsets[g + 1])
        if r1 > r0:
            r = gate_parity(yn[r0:r1], oracle_matmul(w[g], N, K, qs_o[r0:r1], d_o[r0:r1]))
            assert r is None, (g, r)
    assert B.iq4xs_last_device_error() == 0
