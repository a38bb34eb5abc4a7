"""Helpers for the GPU parity tests: move seeded inputs to the device, call the
C ABI through the binding with NaN-poisoned outputs, and get oracle results
(optionally on a sample of weight rows, for full-size shapes)."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from _gates import gate_independent, gate_parity, gate_written
from iq4_xs_quantized_gb300 import binding as B

BLOCK_BYTES = 136


def dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def quantize_gpu(x: np.ndarray):
    """Q8_1 on the GPU with every output poisoned first."""
    M, K = x.shape
    xd = dev(x)
    qs, ds = B.alloc_activations(M, K, "cuda")
    qs.fill_(0x55)
    ds.view(torch.int16).fill_(0x7E00)  # fp16 NaN
    B.iq4xs_quantize_q8_1(xd, qs, ds)
    return qs, ds


def prepare_gpu(x: np.ndarray, qs_ref=None, ds_ref=None):
    """The prepared tensor-core operand of x (poisoned first); the Q8_1
    arrays written beside it must equal iq4xs_quantize_q8_1's bit for bit."""
    M, K = x.shape
    qs, ds = B.alloc_activations(M, K, "cuda")
    op = B.alloc_tc_operand(M, K, "cuda")
    op.fill_(0xFF)  # fp16 NaN pattern / fp32 NaN in the scale part
    B.iq4xs_quantize_q8_1_tc(dev(x), qs, ds, op)
    if qs_ref is not None:
        assert torch.equal(qs, qs_ref) and torch.equal(ds.view(torch.int16), ds_ref.view(torch.int16))
    return op


def matmul_gpu(wd: torch.Tensor, N: int, K: int, qs, ds, M: int, path, ldy: int | None = None,
               op=None, wtype=0):
    """y [M, ldy] through the C ABI, NaN-poisoned first.  path "tcp": the
    tensor-core matmul from the prepared operand `op`."""
    ldy = N if ldy is None else ldy
    y = torch.full((M, ldy), float("nan"), dtype=torch.float32, device="cuda")
    if path == "tcp":
        B.iq4xs_matmul_tc_operand(wd, N, K, op, M, y, wtype)
    elif wtype:
        B.iq4xs_matmul_wt(wd, wtype, N, K, qs, ds, M, y, path)
    else:
        B.iq4xs_matmul(wd, N, K, qs, ds, M, y, path)
    torch.cuda.synchronize()
    return y.cpu().numpy()


def oracle_q8(x: np.ndarray):
    return oracle.get().quantize_q8_1(x)


def oracle_matmul(w: np.ndarray, N: int, K: int, qs: np.ndarray, d_h: np.ndarray, rows=None):
    """Oracle y [M, N] (fp64), or y[:, rows] computed on those rows only."""
    orc = oracle.get()
    nt = max(1, min(16, oracle.threads_available()))
    if rows is None:
        return orc.matmul(w, N, K, qs, d_h, nthreads=nt)
    wr = np.ascontiguousarray(w.reshape(N, -1)[rows])
    return orc.matmul(wr, len(rows), K, qs, d_h, nthreads=nt)


def sample_rows(N: int, count: int, seed: int = 0) -> np.ndarray:
    """Rows spanning the first and last 128-row tiles plus random ones."""
    rng = np.random.default_rng(seed)
    fixed = [0, 1, 127, 128, N // 2, N - 129, N - 2, N - 1]
    fixed = [r for r in fixed if 0 <= r < N]
    extra = rng.choice(N, size=min(N, max(0, count - len(fixed))), replace=False)
    return np.unique(np.concatenate([np.array(fixed, dtype=np.int64), extra.astype(np.int64)]))


def independent_fp32(w: np.ndarray, N: int, K: int, qs: np.ndarray, d_h: np.ndarray, rows=None):
    """Independent check path: the oracle's exact fp32 dequantization of W and
    the dequantized Q8_1 activations, multiplied by torch on the GPU in fp32
    with TF32 disabled (different code, different summation order)."""
    orc = oracle.get()
    wr = w.reshape(N, -1) if rows is None else np.ascontiguousarray(w.reshape(N, -1)[rows])
    n = wr.shape[0]
    W = orc.dequantize(wr, n, K)
    xhat = qs.astype(np.float32) * np.repeat(d_h.view(np.float16).astype(np.float32), 32, axis=1)
    prev = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = False
    try:
        y = (dev(xhat) @ dev(W).T).cpu().numpy()
    finally:
        torch.backends.cuda.matmul.allow_tf32 = prev
    return y


def check_q8(x, qs, ds):
    qs_o, d_o, s_o = oracle_q8(x)
    assert np.array_equal(qs.cpu().numpy(), qs_o)
    dsn = ds.cpu().numpy().view(np.uint16)
    assert np.array_equal(dsn[..., 0], d_o)
    assert np.array_equal(dsn[..., 1], s_o)
    return qs_o, d_o


def run_and_gate(w, N, K, x, path, rows=None, ldy=None, independent=True):
    qs, ds = quantize_gpu(x)
    qs_o, d_o = check_q8(x, qs, ds)
    M = x.shape[0]
    op = prepare_gpu(x, qs, ds) if path == "tcp" else None
    y = matmul_gpu(dev(w), N, K, qs, ds, M, path, ldy=ldy, op=op)
    assert gate_written(y[:, :N]) is None, gate_written(y[:, :N])
    if ldy is not None and ldy > N:
        assert np.all(np.isnan(y[:, N:])), "columns beyond N must not be written"
    y = y[:, :N]
    ys = y if rows is None else y[:, rows]
    yo = oracle_matmul(w, N, K, qs_o, d_o, rows)
    r = gate_parity(ys, yo)
    assert r is None, r
    if independent:
        yi = independent_fp32(w, N, K, qs_o, d_o, rows)
        # A handful of outputs can agree with the independent path exactly by
        # chance; the nonzero-error rule is applied to outputs of >= 256 values.
        r = gate_independent(ys, yi, require_nonzero=ys.size >= 256)
        assert r is None, r
    return y, yo
