"""iq4xs_linear_static: the projection for callers that cannot allocate device
memory (a plugin whose host framework owns every allocation, or a serving
loop that must not allocate once running).  Its scratch is a fixed device
array inside the library; its output must match the workspace entry point,
iq4xs_linear, within the parity tolerance, over two calls in a row (the
second call finds the first call's contents in the shared scratch)."""
import numpy as np
import pytest
import torch

from _gates import gate_independent, gate_parity, gate_written
from _gpu import independent_fp32, oracle_matmul, oracle_q8, sample_rows
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


def _inputs(workload, M):
    w, x = workload.inputs(0, M=M)
    return torch.from_numpy(w).cuda(), torch.from_numpy(x).cuda()


def test_static_scratch_matches_workspace_entry_point_twice():
    # first call: tensor-core path on the square 4096 x 4096 projection;
    # second call: dp4a path on a small projection
    for workload, M in ((synth.SQUARE, 96), (synth.TINY, 3)):
        N, K = workload.shapes[0]
        assert B.iq4xs_linear_workspace_bytes(M, N, K) <= B.iq4xs_linear_static_max_bytes()  # prepared form
        wd, xd = _inputs(workload, M)
        y_static = torch.full((M, N), float("nan"), device="cuda")
        B.iq4xs_linear_static(wd, N, K, xd, y_static)
        ws = torch.empty((B.iq4xs_linear_workspace_bytes(M, N, K),), dtype=torch.uint8, device="cuda")
        y_ws = torch.full((M, N), float("nan"), device="cuda")
        B.iq4xs_linear(wd, N, K, xd, y_ws, ws)
        torch.cuda.synchronize()
        a, b = y_static.cpu().numpy(), y_ws.cpu().numpy()
        assert gate_written(a) is None, gate_written(a)
        r = gate_parity(a, b.astype(np.float64))
        assert r is None, r
        # and against the oracle and an independent fp32 dequantize + matmul
        w_np, x_np = workload.inputs(0, M=M)
        qs_o, d_o, _ = oracle_q8(x_np)
        rows = sample_rows(N, 32, seed=M) if N > 256 else None
        a_s = a if rows is None else a[:, rows]
        r = gate_parity(a_s, oracle_matmul(w_np, N, K, qs_o, d_o, rows))
        assert r is None, r
        r = gate_independent(a_s, independent_fp32(w_np, N, K, qs_o, d_o, rows))
        assert r is None, r


def _largest_m(N, K):
    cap = B.iq4xs_linear_static_max_bytes()
    m = 1
    while B.iq4xs_linear_workspace_min_bytes(m + 1, N, K) <= cap:
        m += 1
    return m


def test_static_scratch_size_limit_boundary():
    """At K = 17408 the 8 MiB scratch holds the Q8_1 codes and scales of 428
    rows: M = 428 runs (tensor-core path), M = 429 is refused before any
    launch and leaves y untouched."""
    N, K = 256, 17408
    assert _largest_m(N, K) == 428
    rng = np.random.default_rng(17)
    w_np = synth.iq4xs_weights(rng, N, K, 1e-3)
    wd = torch.from_numpy(w_np).cuda()
    x_np = synth.activations(rng, 429, K)
    xd = torch.from_numpy(x_np).cuda()
    y = torch.full((428, N), float("nan"), device="cuda")
    B.iq4xs_linear_static(wd, N, K, xd[:428], y)
    torch.cuda.synchronize()
    yn = y.cpu().numpy()
    assert gate_written(yn) is None
    qs_o, d_o, _ = oracle_q8(x_np[:428])
    r = gate_parity(yn, oracle_matmul(w_np, N, K, qs_o, d_o))
    assert r is None, r
    y2 = torch.full((429, N), float("nan"), device="cuda")
    with pytest.raises(B.IQ4XSError) as e:
        B.iq4xs_linear_static(wd, N, K, xd, y2)
    assert e.value.status == B.ERR_SHAPE
    torch.cuda.synchronize()
    assert torch.isnan(y2).all()  # nothing was launched


def test_static_scratch_rejects_requests_beyond_its_size():
    N, K, M = 17408, 5120, 2048
    assert B.iq4xs_linear_workspace_min_bytes(M, N, K) > B.iq4xs_linear_static_max_bytes()
    w = torch.zeros((N, K // 256 * 136), dtype=torch.uint8, device="cuda")
    x = torch.zeros((M, K), device="cuda")
    y = torch.full((M, N), float("nan"), device="cuda")
    with pytest.raises(B.IQ4XSError) as e:
        B.iq4xs_linear_static(w, N, K, x, y)
    assert e.value.status == B.ERR_SHAPE
    torch.cuda.synchronize()
    assert torch.isnan(y).all()  # nothing was launched
