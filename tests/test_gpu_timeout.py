"""The tensor-core matmul's bounded waits, made to run out in the allowed way:
one W stage is left unissued (a barrier that nothing completes), so the
decoders' wait for it ends after its 2 s limit instead of hanging.  The call
returns, the device error word reports the W-stage timeout through
iq4xs_last_device_error (IQ4XS_ERR_TIMEOUT, code 0x101), the CTAs drained
their copies and freed their tensor memory, and the next ordinary call on
the same context is correct."""
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
