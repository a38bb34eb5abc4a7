"""Correctness gates for the CUDA path, after the lessons the V100TPS engine
page draws from its broken batched route: the output buffer is poisoned
before every call and its error against an independent implementation must be
nonzero (an exact match means the same code or memory was compared with
itself), a call faster than its bytes allow did no work (the roofline gate),
and absolute thresholds give way to per-row relative ones on fixed seeds.

Each gate returns None when it passes and a short reason string when it fails,
so the negative-control tests can assert that a gate fires.
"""
from __future__ import annotations

import numpy as np

PARITY_RTOL = 1e-5       # per output row, against the fp64 oracle
INDEPENDENT_RTOL = 2e-3  # against an independent fp32 dequantize + matmul


def gate_written(y: np.ndarray):
    """The NaN poison must be fully overwritten."""
    bad = ~np.isfinite(y)
    if bad.any():
        return f"{int(bad.sum())} of {y.size} outputs not written (NaN/Inf left)"
    return None


def row_rel_errors(y: np.ndarray, ref: np.ndarray) -> np.ndarray:
    """Per row m: max_n |y - ref| / max_n |ref|  (inf if ref row is all zero
    but y is not; 0 if both are exactly zero)."""
    d = np.abs(y.astype(np.float64) - ref.astype(np.float64)).max(axis=1)
    s = np.abs(ref.astype(np.float64)).max(axis=1)
    out = np.zeros_like(d)
    nz = s > 0
    out[nz] = d[nz] / s[nz]
    out[~nz & (d > 0)] = np.inf
    return out


def gate_parity(y: np.ndarray, ref: np.ndarray, rtol: float = PARITY_RTOL):
    e = row_rel_errors(y, ref)
    if not np.all(e <= rtol):
        return f"per-row relative error {e.max():.3e} > {rtol:g} (row {int(e.argmax())})"
    return None


def gate_independent(y: np.ndarray, ref_ind: np.ndarray, rtol: float = INDEPENDENT_RTOL,
                     require_nonzero: bool = True):
    """Against an independent fp32 path: the error must be nonzero (zero means
    the two read the same memory or the same code ran) and within rtol."""
    d = np.abs(y.astype(np.float64) - ref_ind.astype(np.float64)).max()
    s = np.abs(ref_ind.astype(np.float64)).max()
    rel = d / s if s > 0 else (0.0 if d == 0 else np.inf)
    if require_nonzero and d == 0:
        return "error against the independent path is exactly zero"
    if rel > rtol:
        return f"relative error {rel:.3e} against the independent path > {rtol:g}"
    return None


def gate_roofline(bytes_moved: float, seconds: float, peak_bytes_per_s: float, slack: float = 1.10):
    """A call cannot move its algorithmic bytes faster than HBM allows."""
    if seconds <= 0:
        return "non-positive time"
    bw = bytes_moved / seconds
    if bw > slack * peak_bytes_per_s:
        return f"{bw / 1e9:.0f} GB/s exceeds {slack:g} x peak {peak_bytes_per_s / 1e9:.0f} GB/s"
    return None
