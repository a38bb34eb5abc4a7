"""Thin ctypes binding over libiq4xs.so (argument marshalling only).

The names match the C ABI in include/iq4xs.h.  Tensors are torch CUDA tensors
owned by the caller; streams default to torch's current stream.  Every step
of the computation runs in the library's CUDA kernels: there is no CPU or
PyTorch fallback, and a missing library raises immediately.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libiq4xs.so")
BOUNDS_LIB_PATH = os.path.join(_HERE, "libiq4xs_bounds.so")  # the bounds-checked debug build
HEADER = os.path.join(os.path.dirname(_HERE), "include", "iq4xs.h")

OK, ERR_ARG, ERR_ALIGN, ERR_SHAPE, ERR_DEVICE, ERR_CUDA, ERR_TIMEOUT, ERR_BOUNDS = range(8)
PATH_AUTO, PATH_DP4A, PATH_TC, PATH_BASELINE, PATH_MMA = 0, 1, 2, 3, 4
PATHS = {"auto": PATH_AUTO, "dp4a": PATH_DP4A, "tc": PATH_TC, "mma": PATH_MMA}
WTYPE_IQ4_XS, WTYPE_Q4_0, WTYPE_IQ4_NL = 0, 1, 2
WTYPES = {"iq4_xs": WTYPE_IQ4_XS, "q4_0": WTYPE_Q4_0, "iq4_nl": WTYPE_IQ4_NL}

_lock = threading.Lock()
_lib = None


class IQ4XSError(RuntimeError):
    def __init__(self, fn: str, status: int, msg: str):
        super().__init__(f"{fn} failed: status {status} ({msg})")
        self.status = status


def header_functions() -> list[str]:
    """Names of the functions declared in include/iq4xs.h."""
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.findall(r"^\s*(?:const\s+char\s*\*|int64_t|int)\s+(iq4xs_\w+)\s*\(", text, flags=re.M)


def load(path: str | None = None):
    """Load the CUDA library (built by ``iq4_xs_quantized_gb300.build``)."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(f"{p} is missing: build it with iq4_xs_quantized_gb300.build.build()")
        lib = ctypes.CDLL(p)
        i64, vp, ci = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
        lib.iq4xs_quantize_q8_1.argtypes = [vp, i64, i64, i64, vp, vp, i64]
        lib.iq4xs_quantize_q8_1_tc.argtypes = [vp, i64, i64, i64, vp, vp, vp, i64]
        lib.iq4xs_tc_operand_bytes.argtypes = [i64, i64]
        lib.iq4xs_tc_operand_bytes.restype = i64
        lib.iq4xs_matmul_tc_operand.argtypes = [vp, ci, i64, i64, vp, i64, vp, i64, i64]
        lib.iq4xs_linear_workspace_min_bytes.argtypes = [i64, i64, i64]
        lib.iq4xs_linear_workspace_min_bytes.restype = i64
        lib.iq4xs_matmul.argtypes = [vp, i64, i64, vp, vp, i64, vp, i64, ci, i64]
        lib.iq4xs_dequantize.argtypes = [vp, i64, i64, vp, ci, i64]
        lib.iq4xs_matmul_wt.argtypes = [vp, ci, i64, i64, vp, vp, i64, vp, i64, ci, i64]
        lib.iq4xs_dequantize_wt.argtypes = [vp, ci, i64, i64, vp, ci, i64]
        lib.iq4xs_weight_bytes.argtypes = [ci, i64, i64]
        lib.iq4xs_weight_bytes.restype = i64
        lib.iq4xs_matmul_grouped.argtypes = [vp, i64, i64, i64, i64, vp, vp, vp, i64, vp, i64, i64]
        lib.iq4xs_matmul_grouped_path.argtypes = [vp, i64, i64, i64, i64, vp, vp, vp, i64, vp, i64, ci, i64]
        lib.iq4xs_matmul_grouped_wt.argtypes = [vp, ci, i64, i64, i64, i64, vp, vp, vp, i64, vp, i64, ci, i64]
        lib.iq4xs_linear.argtypes = [vp, i64, i64, vp, i64, i64, vp, i64, vp, i64, i64]
        lib.iq4xs_linear_wt.argtypes = [vp, ci, i64, i64, vp, i64, i64, vp, i64, vp, i64, i64]
        lib.iq4xs_linear_workspace_bytes.argtypes = [i64, i64, i64]
        lib.iq4xs_linear_workspace_bytes.restype = i64
        lib.iq4xs_linear_static.argtypes = [vp, i64, i64, vp, i64, i64, vp, i64, i64]
        lib.iq4xs_linear_static.restype = ci
        lib.iq4xs_linear_static_max_bytes.argtypes = []
        lib.iq4xs_linear_static_max_bytes.restype = i64
        lib.iq4xs_select_path.argtypes = [i64, i64, i64, ctypes.POINTER(ci)]
        lib.iq4xs_select_grouped_path.argtypes = [i64, i64, i64, i64, ci, ctypes.POINTER(ci)]
        lib.iq4xs_set_crossover.argtypes = [i64]
        lib.iq4xs_set_baseline_threshold.argtypes = [i64]
        lib.iq4xs_set_crossover_classes.argtypes = [ctypes.POINTER(i64), ctypes.POINTER(i64), ci]
        lib.iq4xs_set_mma_crossover.argtypes = [i64]
        lib.iq4xs_test_mma_config.argtypes = [i64, i64, i64]
        lib.iq4xs_set_mma_crossover_classes.argtypes = [ctypes.POINTER(i64), ctypes.POINTER(i64), ci]
        lib.iq4xs_set_pdl.argtypes = [ci]
        lib.iq4xs_set_pdl.restype = ci
        lib.iq4xs_last_device_error.argtypes = [ctypes.POINTER(ci)]
        lib.iq4xs_test_skip_w_stage.argtypes = [i64]
        lib.iq4xs_bounds_checked.argtypes = [ctypes.POINTER(ci)]
        lib.iq4xs_mma_launch_config.argtypes = [i64, i64, i64, ctypes.POINTER(ci), ctypes.POINTER(ci),
                                                ctypes.POINTER(ci)]
        lib.iq4xs_set_mma_launch_table.argtypes = [ctypes.POINTER(i64), ci]
        lib.iq4xs_test_bounds_margin.argtypes = [i64]
        lib.iq4xs_status_string.argtypes = [ci]
        lib.iq4xs_status_string.restype = ctypes.c_char_p
        for name in ("iq4xs_quantize_q8_1", "iq4xs_matmul", "iq4xs_matmul_grouped", "iq4xs_matmul_grouped_path",
                     "iq4xs_matmul_grouped_wt", "iq4xs_linear_wt",
                     "iq4xs_dequantize", "iq4xs_linear", "iq4xs_matmul_wt", "iq4xs_dequantize_wt",
                     "iq4xs_select_path", "iq4xs_select_grouped_path", "iq4xs_set_crossover",
                     "iq4xs_set_baseline_threshold",
                     "iq4xs_set_crossover_classes", "iq4xs_test_skip_w_stage",
                     "iq4xs_set_mma_crossover", "iq4xs_set_mma_crossover_classes",
                     "iq4xs_test_mma_config",
                     "iq4xs_quantize_q8_1_tc", "iq4xs_matmul_tc_operand",
                     "iq4xs_last_device_error", "iq4xs_bounds_checked", "iq4xs_test_bounds_margin",
                     "iq4xs_mma_launch_config", "iq4xs_set_mma_launch_table"):
            getattr(lib, name).restype = ci
        if path is None:
            _lib = lib
            _install_calibration(lib)
        return lib


def use(path: str | None = None):
    """Route every call of this module through the library at ``path`` (None:
    the default build), e.g. the bounds-checked build; returns it."""
    global _lib
    lib = load(path or LIB_PATH)
    with _lock:
        _lib = lib
    _install_calibration(lib)
    return lib


def _install_calibration(lib):
    """Apply the measured crossovers (dp4a/tcgen05, and the M from which the
    dequantize + GEMM route is advised), if they have been calibrated."""
    from . import calibrate
    table = calibrate.load_table()
    if table and "crossover_m_max_dp4a" in table:
        lib.iq4xs_set_crossover(int(table["crossover_m_max_dp4a"]))
    if table and "crossover_classes" in table:
        _set_classes(lib, table["crossover_classes"])
    if table and "baseline_m_min" in table:
        lib.iq4xs_set_baseline_threshold(int(table["baseline_m_min"]))
    if table and "mma_m_max" in table:
        lib.iq4xs_set_mma_crossover(int(table["mma_m_max"]))
    if table and "mma_classes" in table:
        _set_classes(lib, table["mma_classes"], mma=True)
    if table and "mma_launch" in table:
        _set_launch_table(lib, table["mma_launch"])


def _set_launch_table(lib, entries):
    flat = [int(v) for e in entries for v in e]
    arr = (ctypes.c_int64 * max(1, len(flat)))(*flat)
    _check("iq4xs_set_mma_launch_table", lib.iq4xs_set_mma_launch_table(arr, len(entries)))


def iq4xs_set_mma_launch_table(entries) -> None:
    """Install measured warp-MMA launches: [(N, K, tile_rows, rows_per_cta, k_splits, ctas_per_sm), ...]."""
    _set_launch_table(load(), entries)


def reset_dispatch() -> None:
    """Dispatcher back to the library defaults (DP4A to M = 4, MMA to M = 8,
    no classes, no baseline advice, no measured launches), then the
    calibrated table if present."""
    lib = load()
    lib.iq4xs_set_crossover(4)
    lib.iq4xs_set_mma_crossover(8)
    _set_classes(lib, [])
    _set_classes(lib, [], mma=True)
    _set_launch_table(lib, [])
    lib.iq4xs_set_baseline_threshold(0)
    _install_calibration(lib)


def _set_classes(lib, classes, mma=False):
    n = len(classes)
    mins = (ctypes.c_int64 * max(n, 1))(*[int(c[0]) for c in classes])
    ms = (ctypes.c_int64 * max(n, 1))(*[int(c[1]) for c in classes])
    fn = lib.iq4xs_set_mma_crossover_classes if mma else lib.iq4xs_set_crossover_classes
    return fn(mins, ms, n)


def _check(fn: str, rc: int):
    if rc != OK:
        raise IQ4XSError(fn, rc, load().iq4xs_status_string(rc).decode())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


# --------------------------------------------------------------------------
# Entry points (same names as the C ABI).
# --------------------------------------------------------------------------
def iq4xs_quantize_q8_1(x, qs, ds, stream=None) -> None:
    """x fp32 [M, K] (row stride x.stride(0)) -> qs int8 [M, K], ds fp16 [M, K/32, 2]
    ({d, s})."""
    M, K = x.shape
    rc = load().iq4xs_quantize_q8_1(_ptr(x), M, K, x.stride(0), _ptr(qs), _ptr(ds), _stream(stream))
    _check("iq4xs_quantize_q8_1", rc)


def iq4xs_tc_operand_bytes(M: int, K: int) -> int:
    return int(load().iq4xs_tc_operand_bytes(M, K))


def iq4xs_quantize_q8_1_tc(x, qs, ds, tc_operand, stream=None) -> None:
    """iq4xs_quantize_q8_1 that also writes the prepared tensor-core operand
    (uint8 device tensor of iq4xs_tc_operand_bytes(M, K) bytes)."""
    M, K = x.shape
    rc = load().iq4xs_quantize_q8_1_tc(_ptr(x), M, K, x.stride(0), _ptr(qs), _ptr(ds),
                                       _ptr(tc_operand), _stream(stream))
    _check("iq4xs_quantize_q8_1_tc", rc)


def iq4xs_matmul_tc_operand(w, N: int, K: int, tc_operand, M: int, y, wtype=WTYPE_IQ4_XS,
                            stream=None) -> None:
    """The tensor-core matmul from the prepared operand."""
    rc = load().iq4xs_matmul_tc_operand(_ptr(w), _wtype(wtype), N, K, _ptr(tc_operand), M, _ptr(y),
                                        y.stride(0), _stream(stream))
    _check("iq4xs_matmul_tc_operand", rc)


def iq4xs_matmul(w, N: int, K: int, qs, ds, M: int, y, path=PATH_AUTO, stream=None) -> None:
    """y fp32 [M, ldy] = x . W^T from IQ4_XS bytes w and Q8_1 activations."""
    if isinstance(path, str):
        path = PATHS[path]
    ldy = y.stride(0)
    rc = load().iq4xs_matmul(_ptr(w), N, K, _ptr(qs), _ptr(ds), M, _ptr(y), ldy, int(path),
                             _stream(stream))
    _check("iq4xs_matmul", rc)


def _wtype(wtype) -> int:
    return WTYPES[wtype] if isinstance(wtype, str) else int(wtype)


def iq4xs_weight_bytes(wtype, N: int, K: int) -> int:
    return int(load().iq4xs_weight_bytes(_wtype(wtype), N, K))


def iq4xs_matmul_wt(w, wtype, N: int, K: int, qs, ds, M: int, y, path=PATH_AUTO,
                    stream=None) -> None:
    """iq4xs_matmul for weights in format ``wtype`` (WTYPE_* or its name)."""
    if isinstance(path, str):
        path = PATHS[path]
    rc = load().iq4xs_matmul_wt(_ptr(w), _wtype(wtype), N, K, _ptr(qs), _ptr(ds), M, _ptr(y),
                                y.stride(0), int(path), _stream(stream))
    _check("iq4xs_matmul_wt", rc)


def iq4xs_linear_workspace_bytes(M: int, N: int, K: int) -> int:
    return int(load().iq4xs_linear_workspace_bytes(M, N, K))


def iq4xs_linear_workspace_min_bytes(M: int, N: int, K: int) -> int:
    return int(load().iq4xs_linear_workspace_min_bytes(M, N, K))


def iq4xs_linear(w, N: int, K: int, x, y, workspace, stream=None, wtype=WTYPE_IQ4_XS) -> None:
    """y fp32 [M, ldy] = Q8_1(x) . W^T in one call (W in format ``wtype``);
    workspace: uint8 device tensor of at least
    iq4xs_linear_workspace_bytes(M, N, K) bytes."""
    M = x.shape[0]
    rc = load().iq4xs_linear_wt(_ptr(w), _wtype(wtype), N, K, _ptr(x), M, x.stride(0), _ptr(y), y.stride(0),
                                _ptr(workspace), workspace.numel() * workspace.element_size(),
                                _stream(stream))
    _check("iq4xs_linear_wt", rc)


def iq4xs_linear_static(w, N: int, K: int, x, y, stream=None) -> None:
    """iq4xs_linear with the library's fixed device scratch: nothing is
    allocated (for callers that cannot allocate device memory)."""
    M = x.shape[0]
    rc = load().iq4xs_linear_static(_ptr(w), N, K, _ptr(x), M, x.stride(0), _ptr(y), y.stride(0),
                                    _stream(stream))
    _check("iq4xs_linear_static", rc)


def iq4xs_linear_static_max_bytes() -> int:
    return int(load().iq4xs_linear_static_max_bytes())


def iq4xs_matmul_grouped(w, expert_stride: int, G: int, N: int, K: int, qs, ds, row_offsets, y,
                         stream=None, path=PATH_AUTO, wtype=WTYPE_IQ4_XS) -> None:
    """Mixture-of-experts matmul in one launch: expert g (W at byte
    g * expert_stride of w, format ``wtype``) over the Q8_1 rows
    [row_offsets[g], row_offsets[g+1]) (row_offsets: int32 device tensor
    [G+1]); y holds every row (its row count bounds the number of non-empty
    experts).  path: AUTO, DP4A, MMA or TC (iq4xs_matmul_grouped_wt)."""
    if row_offsets.dtype != torch.int32:
        raise TypeError("row_offsets must be int32")
    if isinstance(path, str):
        path = PATHS[path]
    rc = load().iq4xs_matmul_grouped_wt(_ptr(w), _wtype(wtype), int(expert_stride), G, N, K, _ptr(qs), _ptr(ds),
                                        _ptr(row_offsets), y.shape[0], _ptr(y), y.stride(0), int(path),
                                        _stream(stream))
    _check("iq4xs_matmul_grouped_wt", rc)


def iq4xs_dequantize(w, N: int, K: int, out, stream=None) -> None:
    """IQ4_XS -> dense [N, K]; out dtype float32 (exact) or bfloat16 (RNE)."""
    dt = {torch.float32: 0, torch.bfloat16: 1}[out.dtype]
    rc = load().iq4xs_dequantize(_ptr(w), N, K, _ptr(out), dt, _stream(stream))
    _check("iq4xs_dequantize", rc)


def iq4xs_dequantize_wt(w, wtype, N: int, K: int, out, stream=None) -> None:
    """Weights in format ``wtype`` -> dense [N, K] (float32 exact, or bfloat16 RNE)."""
    dt = {torch.float32: 0, torch.bfloat16: 1}[out.dtype]
    rc = load().iq4xs_dequantize_wt(_ptr(w), _wtype(wtype), N, K, _ptr(out), dt, _stream(stream))
    _check("iq4xs_dequantize_wt", rc)


def iq4xs_select_path(M: int, N: int, K: int) -> int:
    out = ctypes.c_int(-1)
    _check("iq4xs_select_path", load().iq4xs_select_path(M, N, K, ctypes.byref(out)))
    return out.value


def iq4xs_select_grouped_path(G: int, N: int, K: int, total_rows: int, wtype=WTYPE_IQ4_XS) -> int:
    """The form the grouped call takes with AUTO (PATH_DP4A, PATH_MMA or PATH_TC)."""
    out = ctypes.c_int(-1)
    _check("iq4xs_select_grouped_path",
           load().iq4xs_select_grouped_path(G, N, K, total_rows, _wtype(wtype), ctypes.byref(out)))
    return out.value


def iq4xs_set_crossover(m_max_dp4a: int) -> None:
    _check("iq4xs_set_crossover", load().iq4xs_set_crossover(int(m_max_dp4a)))


def iq4xs_set_crossover_classes(classes) -> None:
    """[(min_weights, m_max_dp4a), ...]: the crossover per weight-size class."""
    _check("iq4xs_set_crossover_classes", _set_classes(load(), list(classes)))


def iq4xs_set_mma_crossover(m_max_mma: int) -> None:
    _check("iq4xs_set_mma_crossover", load().iq4xs_set_mma_crossover(int(m_max_mma)))


def iq4xs_set_mma_crossover_classes(classes) -> None:
    """classes: [(min_weights, m_max_mma), ...]; [] clears them."""
    _check("iq4xs_set_mma_crossover_classes", _set_classes(load(), list(classes), mma=True))


def iq4xs_test_mma_config(rows_per_cta: int = 0, k_splits: int = 0, ctas_per_sm: int = 0) -> None:
    """Force the warp-MMA launch configuration (0 = the launch model's choice)."""
    _check("iq4xs_test_mma_config",
           load().iq4xs_test_mma_config(int(rows_per_cta), int(k_splits), int(ctas_per_sm)))


def iq4xs_mma_launch_config(M: int, N: int, K: int) -> tuple[int, int, int]:
    """(rows per CTA, K splits, CTAs per SM) of the warp-MMA launch for (M, N, K)."""
    r, s, o = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    _check("iq4xs_mma_launch_config",
           load().iq4xs_mma_launch_config(M, N, K, ctypes.byref(r), ctypes.byref(s), ctypes.byref(o)))
    return r.value, s.value, o.value


def iq4xs_set_baseline_threshold(m_min_baseline: int) -> None:
    _check("iq4xs_set_baseline_threshold", load().iq4xs_set_baseline_threshold(int(m_min_baseline)))


def iq4xs_set_pdl(enable: bool) -> None:
    _check("iq4xs_set_pdl", load().iq4xs_set_pdl(1 if enable else 0))


def iq4xs_last_device_error() -> int:
    """The device error word (0 = clean), read and cleared; a timeout or
    bounds code (status IQ4XS_ERR_TIMEOUT / IQ4XS_ERR_BOUNDS) is returned,
    not raised."""
    out = ctypes.c_int(-1)
    rc = load().iq4xs_last_device_error(ctypes.byref(out))
    if rc not in (ERR_TIMEOUT, ERR_BOUNDS):
        _check("iq4xs_last_device_error", rc)
    return out.value


def iq4xs_bounds_checked() -> bool:
    out = ctypes.c_int(-1)
    _check("iq4xs_bounds_checked", load().iq4xs_bounds_checked(ctypes.byref(out)))
    return out.value == 1


def iq4xs_test_bounds_margin(nbytes: int) -> None:
    _check("iq4xs_test_bounds_margin", load().iq4xs_test_bounds_margin(int(nbytes)))


def iq4xs_test_skip_w_stage(stage: int) -> None:
    _check("iq4xs_test_skip_w_stage", load().iq4xs_test_skip_w_stage(int(stage)))


def iq4xs_status_string(status: int) -> str:
    return load().iq4xs_status_string(status).decode()


# --------------------------------------------------------------------------
# Buffer helpers (allocation by torch; the library allocates nothing).
# --------------------------------------------------------------------------
def alloc_activations(M: int, K: int, device="cuda"):
    """Q8_1 buffers for M x K activations: (qs int8 [M, K], ds fp16 [M, K/32, 2])."""
    qs = torch.empty((M, K), dtype=torch.int8, device=device)
    ds = torch.empty((M, K // 32, 2), dtype=torch.float16, device=device)
    return qs, ds


def alloc_tc_operand(M: int, K: int, device="cuda"):
    """A uint8 device buffer for the prepared tensor-core operand."""
    return torch.empty(iq4xs_tc_operand_bytes(M, K), dtype=torch.uint8, device=device)


def linear(w, N: int, K: int, x, path=PATH_AUTO, stream=None, out=None, allow_baseline=False):
    """Convenience: quantize x [M, K] and return y [M, N] fp32 (two launches).

    With allow_baseline and the dispatcher advising BASELINE (M at or above
    the measured threshold), W is dequantized to bf16 by this library and the
    product is a dense bf16 GEMM (torch / cuBLAS): faster there, at bf16
    precision rather than the Q8_1 paths' exact sub-block dots."""
    M = x.shape[0]
    y = out if out is not None else torch.empty((M, N), dtype=torch.float32, device=x.device)
    if allow_baseline and path == PATH_AUTO and iq4xs_select_path(M, N, K) == PATH_BASELINE:
        wbf = torch.empty((N, K), dtype=torch.bfloat16, device=x.device)
        iq4xs_dequantize(w, N, K, wbf, stream)
        s = torch.cuda.current_stream() if stream is None else stream
        with torch.cuda.stream(s):
            y.copy_(torch.matmul(x.to(torch.bfloat16), wbf.t()).float())
        return y
    kpath = path
    if path == PATH_AUTO:
        sel = iq4xs_select_path(M, N, K)
        kpath = PATH_TC if sel == PATH_BASELINE else sel
    qs, ds = alloc_activations(M, K, x.device)
    iq4xs_quantize_q8_1(x, qs, ds, stream)
    iq4xs_matmul(w, N, K, qs, ds, M, y, kpath, stream)
    return y
