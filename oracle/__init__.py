"""CPU oracle for the IQ4_XS x Q8_1 batched matmul -- TEST INFRASTRUCTURE.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline /
reference leg may import this package.  The product path (the CUDA library and
its Python binding) never imports, links or runs it, and this package imports
nothing from the product.

The arithmetic lives in ``iq4xs_oracle.c`` (plain C11, fp64 product, IEEE
half/bfloat16 conversions written from the definitions).  This module compiles
it with gcc on first use (``-ffp-contract=off``, no fast-math, no -march) and
wraps it with ctypes over numpy arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "iq4xs_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

QK = 256          # weights per IQ4_XS super-block
BLOCK_BYTES = 136  # bytes per super-block
SUB = 32          # weights per sub-block / per Q8_1 block
B18_BYTES = 18    # bytes per 32-weight Q4_0 / IQ4_NL block

# Weight formats: IQ4_XS (256-weight super-blocks), Q4_0 and IQ4_NL (32-weight
# blocks of 18 bytes).
WT_IQ4_XS, WT_Q4_0, WT_IQ4_NL = 0, 1, 2


def compile_oracle(src: str = _SRC, out: str = _LIB, extra_flags=()) -> str:
    """Compile the oracle C source to a shared library and return its path."""
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared",
           "-pthread", *extra_flags, src, "-o", out + ".tmp", "-lm"]
    subprocess.run(cmd, check=True, capture_output=True)
    os.replace(out + ".tmp", out)
    return out


def _needs_build() -> bool:
    return (not os.path.exists(_LIB)) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC)


def _bind(lib):
    c = ctypes
    p = c.c_void_p
    i64 = c.c_int64
    lib.oracle_kvalue.argtypes = [c.c_int]
    lib.oracle_kvalue.restype = c.c_int
    lib.oracle_f16_to_f32.argtypes = [c.c_uint16]
    lib.oracle_f16_to_f32.restype = c.c_float
    lib.oracle_f32_to_f16.argtypes = [c.c_float]
    lib.oracle_f32_to_f16.restype = c.c_uint16
    lib.oracle_bf16_to_f32.argtypes = [c.c_uint16]
    lib.oracle_bf16_to_f32.restype = c.c_float
    lib.oracle_f32_to_bf16.argtypes = [c.c_float]
    lib.oracle_f32_to_bf16.restype = c.c_uint16
    lib.oracle_iq4xs_ls.argtypes = [p, c.c_int]
    lib.oracle_iq4xs_ls.restype = c.c_int
    lib.oracle_iq4xs_subblock_scale.argtypes = [p, c.c_int]
    lib.oracle_iq4xs_subblock_scale.restype = c.c_float
    lib.oracle_iq4xs_code.argtypes = [p, c.c_int]
    lib.oracle_iq4xs_code.restype = c.c_int
    lib.oracle_iq4xs_decode.argtypes = [p, i64, i64, p]
    lib.oracle_iq4xs_decode.restype = c.c_int
    lib.oracle_iq4xs_dequantize.argtypes = [p, i64, i64, p, p]
    lib.oracle_iq4xs_dequantize.restype = c.c_int
    lib.oracle_quantize_q8_1.argtypes = [p, i64, i64, i64, p, p, p]
    lib.oracle_quantize_q8_1.restype = c.c_int
    lib.oracle_matmul.argtypes = [p, i64, i64, p, p, i64, p, c.c_int]
    lib.oracle_matmul.restype = c.c_int
    lib.oracle_subblock_dot.argtypes = [p, i64, p, i64, i64, i64, c.c_int]
    lib.oracle_subblock_dot.restype = c.c_int64
    lib.oracle_b18_code.argtypes = [c.c_int, p, c.c_int]
    lib.oracle_b18_code.restype = c.c_int
    lib.oracle_b18_scale.argtypes = [p]
    lib.oracle_b18_scale.restype = c.c_float
    lib.oracle_row_bytes.argtypes = [c.c_int, i64]
    lib.oracle_row_bytes.restype = c.c_int64
    lib.oracle_decode_wt.argtypes = [c.c_int, p, i64, i64, p]
    lib.oracle_decode_wt.restype = c.c_int
    lib.oracle_dequantize_wt.argtypes = [c.c_int, p, i64, i64, p, p]
    lib.oracle_dequantize_wt.restype = c.c_int
    lib.oracle_matmul_wt.argtypes = [c.c_int, p, i64, i64, p, p, i64, p, c.c_int]
    lib.oracle_matmul_wt.restype = c.c_int
    return lib


def load_library(path: str | None = None):
    """Load (building if needed) the oracle library.  ``path`` loads another
    build of it, e.g. a deliberately broken copy compiled by a test."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            if _needs_build():
                compile_oracle()
            _lib = _bind(ctypes.CDLL(_LIB))
    return _lib


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


class Oracle:
    """numpy-level wrapper over one oracle library build."""

    def __init__(self, lib=None):
        self.lib = lib if lib is not None else load_library()

    # -- conversions -------------------------------------------------------
    def f32_to_f16(self, x: np.ndarray) -> np.ndarray:
        x = np.asarray(x, dtype=np.float32).ravel()
        return np.array([self.lib.oracle_f32_to_f16(float(v)) for v in x], dtype=np.uint16)

    def f16_to_f32(self, h: np.ndarray) -> np.ndarray:
        h = np.asarray(h, dtype=np.uint16).ravel()
        return np.array([self.lib.oracle_f16_to_f32(int(v)) for v in h], dtype=np.float32)

    def f32_to_bf16(self, x: np.ndarray) -> np.ndarray:
        x = np.asarray(x, dtype=np.float32).ravel()
        return np.array([self.lib.oracle_f32_to_bf16(float(v)) for v in x], dtype=np.uint16)

    def kvalues(self) -> list[int]:
        return [self.lib.oracle_kvalue(i) for i in range(16)]

    # -- IQ4_XS ------------------------------------------------------------
    def decode(self, w: np.ndarray, N: int, K: int) -> np.ndarray:
        w = np.ascontiguousarray(w, dtype=np.uint8)
        assert w.size == N * (K // QK) * BLOCK_BYTES
        out = np.empty((N, K), dtype=np.float64)
        rc = self.lib.oracle_iq4xs_decode(_ptr(w), N, K, _ptr(out))
        if rc:
            raise ValueError(f"oracle decode failed: {rc}")
        return out

    def dequantize(self, w: np.ndarray, N: int, K: int, bf16: bool = False):
        w = np.ascontiguousarray(w, dtype=np.uint8)
        f32 = np.empty((N, K), dtype=np.float32)
        b16 = np.empty((N, K), dtype=np.uint16) if bf16 else None
        rc = self.lib.oracle_iq4xs_dequantize(_ptr(w), N, K, _ptr(f32),
                                              _ptr(b16) if bf16 else None)
        if rc:
            raise ValueError(f"oracle dequantize failed: {rc}")
        return (f32, b16) if bf16 else f32

    def ls(self, block: np.ndarray, j: int) -> int:
        block = np.ascontiguousarray(block, dtype=np.uint8)
        return self.lib.oracle_iq4xs_ls(_ptr(block), j)

    def subblock_scale(self, block: np.ndarray, j: int) -> float:
        block = np.ascontiguousarray(block, dtype=np.uint8)
        return self.lib.oracle_iq4xs_subblock_scale(_ptr(block), j)

    # -- Q8_1 ----------------------------------------------------------------
    def quantize_q8_1(self, x: np.ndarray):
        """x [M,K] fp32 -> (qs int8 [M,K], d_h uint16 [M,K/32], s_h uint16 [M,K/32])."""
        x = np.ascontiguousarray(x, dtype=np.float32)
        M, K = x.shape
        qs = np.empty((M, K), dtype=np.int8)
        d_h = np.empty((M, K // SUB), dtype=np.uint16)
        s_h = np.empty((M, K // SUB), dtype=np.uint16)
        rc = self.lib.oracle_quantize_q8_1(_ptr(x), M, K, K, _ptr(qs), _ptr(d_h), _ptr(s_h))
        if rc:
            raise ValueError(f"oracle quantize failed: {rc}")
        return qs, d_h, s_h

    # -- product -------------------------------------------------------------
    def matmul(self, w: np.ndarray, N: int, K: int, qs: np.ndarray, d_h: np.ndarray,
               nthreads: int = 1) -> np.ndarray:
        """y [M,N] fp64 = oracle product of IQ4_XS W and Q8_1 activations."""
        w = np.ascontiguousarray(w, dtype=np.uint8)
        qs = np.ascontiguousarray(qs, dtype=np.int8)
        d_h = np.ascontiguousarray(d_h, dtype=np.uint16)
        M = qs.shape[0]
        assert qs.shape == (M, K) and d_h.shape == (M, K // SUB)
        y = np.empty((M, N), dtype=np.float64)
        rc = self.lib.oracle_matmul(_ptr(w), N, K, _ptr(qs), _ptr(d_h), M, _ptr(y),
                                    int(nthreads))
        if rc:
            raise ValueError(f"oracle matmul failed: {rc}")
        return y

    # -- any weight format -------------------------------------------------
    def row_bytes(self, wtype: int, K: int) -> int:
        return self.lib.oracle_row_bytes(wtype, K)

    def b18_code(self, wtype: int, block: np.ndarray, i: int) -> int:
        block = np.ascontiguousarray(block, dtype=np.uint8)
        return self.lib.oracle_b18_code(wtype, _ptr(block), i)

    def b18_scale(self, block: np.ndarray) -> float:
        block = np.ascontiguousarray(block, dtype=np.uint8)
        return self.lib.oracle_b18_scale(_ptr(block))

    def decode_wt(self, wtype: int, w: np.ndarray, N: int, K: int) -> np.ndarray:
        w = np.ascontiguousarray(w, dtype=np.uint8)
        assert w.size == N * self.row_bytes(wtype, K)
        out = np.empty((N, K), dtype=np.float64)
        rc = self.lib.oracle_decode_wt(wtype, _ptr(w), N, K, _ptr(out))
        if rc:
            raise ValueError(f"oracle decode failed: {rc}")
        return out

    def dequantize_wt(self, wtype: int, w: np.ndarray, N: int, K: int, bf16: bool = False):
        w = np.ascontiguousarray(w, dtype=np.uint8)
        assert w.size == N * self.row_bytes(wtype, K)
        f32 = np.empty((N, K), dtype=np.float32)
        b16 = np.empty((N, K), dtype=np.uint16) if bf16 else None
        rc = self.lib.oracle_dequantize_wt(wtype, _ptr(w), N, K, _ptr(f32),
                                           _ptr(b16) if bf16 else None)
        if rc:
            raise ValueError(f"oracle dequantize failed: {rc}")
        return (f32, b16) if bf16 else f32

    def matmul_wt(self, wtype: int, w: np.ndarray, N: int, K: int, qs: np.ndarray,
                  d_h: np.ndarray, nthreads: int = 1) -> np.ndarray:
        """y [M,N] fp64 for weights in format ``wtype``."""
        w = np.ascontiguousarray(w, dtype=np.uint8)
        assert w.size == N * self.row_bytes(wtype, K)
        qs = np.ascontiguousarray(qs, dtype=np.int8)
        d_h = np.ascontiguousarray(d_h, dtype=np.uint16)
        M = qs.shape[0]
        assert qs.shape == (M, K) and d_h.shape == (M, K // SUB)
        y = np.empty((M, N), dtype=np.float64)
        rc = self.lib.oracle_matmul_wt(wtype, _ptr(w), N, K, _ptr(qs), _ptr(d_h), M, _ptr(y),
                                       int(nthreads))
        if rc:
            raise ValueError(f"oracle matmul failed: {rc}")
        return y

    def subblock_dot(self, w, K, qs, n, m, b, j) -> int:
        w = np.ascontiguousarray(w, dtype=np.uint8)
        qs = np.ascontiguousarray(qs, dtype=np.int8)
        return self.lib.oracle_subblock_dot(_ptr(w), K, _ptr(qs), n, m, b, j)


_default = None


def get() -> Oracle:
    """The shared oracle instance over the default build."""
    global _default
    if _default is None:
        _default = Oracle()
    return _default


def threads_available() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1
