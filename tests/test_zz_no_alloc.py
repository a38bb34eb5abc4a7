"""iq4xs_linear_static: the projection for callers that cannot allocate device
memory (a plugin whose host framework owns every allocation, or a serving
loop that must not allocate once running).  Its scratch is a fixed device
array inside the library; its output must match the workspace entry point,
iq4xs_linear, within the parity tolerance, over two calls in a row (the
second call finds the first call's contents in the shared scratch)."""
import numpy as np
import pytest
import torch

from _gates import gate_parity, gate_written
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
        assert B.iq4xs_linear_workspace_bytes(M, N, K) <= B.iq4xs_linear_static_max_bytes()
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


def test_static_scratch_rejects_requests_beyond_its_size():
    N, K, M = 17408, 5120, 512
    assert B.iq4xs_linear_workspace_bytes(M, N, K) > B.iq4xs_linear_static_max_bytes()
    w = torch.zeros((N, K // 256 * 136), dtype=torch.uint8, device="cuda")
    x = torch.zeros((M, K), device="cuda")
    y = torch.full((M, N), float("nan"), device="cuda")
    with pytest.raises(B.IQ4XSError) as e:
        B.iq4xs_linear_static(w, N, K, x, y)
    assert e.value.status == B.ERR_SHAPE
    torch.cuda.synchronize()
    assert torch.isnan(y).all()  # nothing was launched
