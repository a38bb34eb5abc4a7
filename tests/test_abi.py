"""The C ABI library on the host: it builds, loads, exports every function
include/iq4xs.h declares, and its host-only entry points (path selection,
argument validation) behave without touching a GPU."""
import ctypes
import os

import pytest

from iq4_xs_quantized_gb300 import binding as B
from iq4_xs_quantized_gb300 import build


@pytest.fixture(scope="module")
def lib():
    build.build()
    return B.load()


def test_header_declares_the_entry_points():
    names = set(B.header_functions())
    assert {"iq4xs_quantize_q8_1", "iq4xs_matmul", "iq4xs_dequantize", "iq4xs_select_path",
            "iq4xs_set_crossover", "iq4xs_set_baseline_threshold",
            "iq4xs_last_device_error",
            "iq4xs_status_string", "iq4xs_linear", "iq4xs_linear_workspace_bytes",
            "iq4xs_matmul_wt", "iq4xs_dequantize_wt", "iq4xs_weight_bytes"} <= names


def _prototype(name):
    """Parameter list of `name` in include/iq4xs.h, as (type, name) pairs."""
    import re
    text = re.sub(r"/\*.*?\*/", "", open(B.HEADER).read(), flags=re.S)
    m = re.search(r"\b" + name + r"\s*\(([^)]*)\)\s*;", text)
    assert m, name
    out = []
    for p in m.group(1).split(","):
        p = " ".join(p.replace("*", " * ").split())
        typ, _, pname = p.rpartition(" ")
        out.append((typ.replace(" *", "*"), pname))
    return out


def test_boundary_prototypes():
    """The four calls of the boundary, with exactly these parameters (plain
    pointers and sizes, stream as int64)."""
    assert _prototype("iq4xs_quantize_q8_1") == [
        ("const float*", "x"), ("int64_t", "M"), ("int64_t", "K"), ("int64_t", "ldx"),
        ("int8_t*", "qs"), ("void*", "ds"), ("int64_t", "stream")]
    assert _prototype("iq4xs_matmul") == [
        ("const void*", "w"), ("int64_t", "N"), ("int64_t", "K"), ("const int8_t*", "qs"),
        ("const void*", "ds"), ("int64_t", "M"), ("float*", "y"), ("int64_t", "ldy"),
        ("int", "path"), ("int64_t", "stream")]
    assert _prototype("iq4xs_dequantize") == [
        ("const void*", "w"), ("int64_t", "N"), ("int64_t", "K"), ("void*", "out"),
        ("int", "out_dtype"), ("int64_t", "stream")]
    assert _prototype("iq4xs_select_path") == [
        ("int64_t", "M"), ("int64_t", "N"), ("int64_t", "K"), ("int*", "path_out")]


def test_library_exports_every_declared_symbol(lib):
    for name in B.header_functions():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def _dispatch(dp4a, mma, baseline=0):
    B.iq4xs_set_crossover_classes([])
    B.iq4xs_set_mma_crossover_classes([])
    B.iq4xs_set_crossover(dp4a)
    B.iq4xs_set_mma_crossover(mma)
    B.iq4xs_set_baseline_threshold(baseline)


def test_select_path_and_crossover(lib):
    try:
        _dispatch(4, 8)  # DP4A to M = 4, MMA to M = 8, TC above
        sel = B.iq4xs_select_path
        assert [sel(m, 4096, 4096) for m in (1, 4, 5, 8, 9, 96)] == [
            B.PATH_DP4A, B.PATH_DP4A, B.PATH_MMA, B.PATH_MMA, B.PATH_TC, B.PATH_TC]
        # K % 512 != 0: neither tensor-core path (W rows not 16-byte strided)
        assert sel(2, 4096, 256 * 3) == B.PATH_DP4A
        assert sel(96, 4096, 256 * 3) == B.PATH_DP4A
        B.iq4xs_set_mma_crossover(0)  # no MMA range
        assert sel(5, 4096, 4096) == B.PATH_TC
        B.iq4xs_set_crossover(0)
        assert sel(1, 4096, 4096) == B.PATH_TC
        # per weight-size class: the largest class at or below N*K applies
        _dispatch(4, 8)
        B.iq4xs_set_mma_crossover_classes([(20_000_000, 16), (100_000_000, 4)])
        B.iq4xs_set_crossover_classes([(20_000_000, 2)])
        assert sel(12, 12288, 5120) == B.PATH_MMA   # 63M weights: MMA to 16
        assert sel(3, 12288, 5120) == B.PATH_MMA    # dp4a only to 2 there
        assert sel(12, 4096, 4096) == B.PATH_TC     # 16.8M: the defaults
        assert sel(3, 4096, 4096) == B.PATH_DP4A
        assert sel(8, 34816, 5120) == B.PATH_TC     # 178M: MMA only to 4
        out = ctypes.c_int()
        assert lib.iq4xs_select_path(0, 1, 256, ctypes.byref(out)) == B.ERR_SHAPE
        assert lib.iq4xs_select_path(1, 1, 100, ctypes.byref(out)) == B.ERR_SHAPE
        assert lib.iq4xs_select_path(1, 1, 256, None) == B.ERR_ARG
        assert lib.iq4xs_set_crossover(-1) == B.ERR_ARG
        assert lib.iq4xs_set_mma_crossover(-1) == B.ERR_ARG
        assert lib.iq4xs_set_mma_crossover(40000) == B.ERR_ARG
        bad = (ctypes.c_int64 * 1)(0)
        ok = (ctypes.c_int64 * 1)(4)
        assert lib.iq4xs_set_mma_crossover_classes(bad, ok, 1) == B.ERR_ARG
        assert lib.iq4xs_set_mma_crossover_classes(ok, ok, 17) == B.ERR_ARG
    finally:
        B.reset_dispatch()


def test_select_grouped_path_rule(lib):
    """The grouped AUTO rule (host only): the CUDA-core form below min(G, 24)
    rows unless the mean rows per expert leave the DP4A range, the warp-MMA
    form from there, tcgen05 from 32 mean rows per expert slot on (IQ4_XS
    only), and the CUDA-core form whenever K % 512 != 0."""
    try:
        _dispatch(1, 8)
        sel = B.iq4xs_select_grouped_path
        G, N, K = 128, 1536, 2048
        assert [sel(G, N, K, r) for r in (1, 16, 23, 24, 128, 3968, 3969, 32768)] == [
            B.PATH_DP4A, B.PATH_DP4A, B.PATH_DP4A, B.PATH_MMA, B.PATH_MMA, B.PATH_MMA, B.PATH_TC, B.PATH_TC]
        for wt in (B.WTYPE_Q4_0, B.WTYPE_IQ4_NL):
            assert sel(G, N, K, 4096, wt) == B.PATH_MMA  # no tcgen05 grouped form for these formats
            assert sel(G, N, K, 16, wt) == B.PATH_DP4A
        assert sel(8, N, K, 7) == B.PATH_DP4A      # fewer rows than the 8 experts: mean 1 row
        assert sel(8, N, K, 8) == B.PATH_MMA       # min(G, 24) = 8 rows
        assert sel(8, N, K, 248) == B.PATH_MMA     # mean 31 rows (rounded up)
        assert sel(8, N, K, 249) == B.PATH_TC      # mean 32 rows
        assert sel(G, N, 1280, 4096) == B.PATH_DP4A  # K % 512 != 0
        assert sel(32, N, K, 20) == B.PATH_DP4A    # 20 rows < min(32, 24)
        B.iq4xs_set_crossover(0)  # a matrix size without a DP4A range: one row already leaves it
        assert sel(G, N, K, 1) == B.PATH_MMA
        out = ctypes.c_int()
        assert lib.iq4xs_select_grouped_path(0, N, K, 8, 0, ctypes.byref(out)) == B.ERR_SHAPE
        assert lib.iq4xs_select_grouped_path(G, N, K, 0, 0, ctypes.byref(out)) == B.ERR_SHAPE
        assert lib.iq4xs_select_grouped_path(G, N, K, 32769, 0, ctypes.byref(out)) == B.ERR_SHAPE
        assert lib.iq4xs_select_grouped_path(G, N, K, 8, 3, ctypes.byref(out)) == B.ERR_ARG
        assert lib.iq4xs_select_grouped_path(G, N, K, 8, 0, None) == B.ERR_ARG
    finally:
        B.reset_dispatch()


def test_mma_config_hook_validation(lib):
    assert lib.iq4xs_test_mma_config(0, 0, 0) == B.OK
    for rows, splits, occ in ((16, 1, 0), (288, 1, 0), (-32, 1, 0), (64, 9, 0), (64, -1, 0), (64, 1, 3),
                              (64, 1, -1)):
        assert lib.iq4xs_test_mma_config(rows, splits, occ) == B.ERR_ARG
    assert lib.iq4xs_test_mma_config(256, 8, 2) == B.OK
    assert lib.iq4xs_test_mma_config(0, 0, 0) == B.OK


def test_baseline_threshold_is_advice_above_the_tc_range(lib):
    _dispatch(4, 0)  # no MMA range; baseline never
    assert B.iq4xs_select_path(512, 5120, 17408) == B.PATH_TC
    B.iq4xs_set_baseline_threshold(128)
    assert B.iq4xs_select_path(96, 5120, 17408) == B.PATH_TC
    assert B.iq4xs_select_path(128, 5120, 17408) == B.PATH_BASELINE
    assert B.iq4xs_select_path(512, 5120, 17408) == B.PATH_BASELINE
    # below the dp4a crossover the dp4a path stays
    B.iq4xs_set_baseline_threshold(1)
    assert B.iq4xs_select_path(2, 4096, 4096) == B.PATH_DP4A
    assert B.iq4xs_select_path(8, 4096, 4096) == B.PATH_BASELINE
    # shapes the tensor-core paths cannot take keep dp4a
    assert B.iq4xs_select_path(256, 4096, 256 * 3) == B.PATH_DP4A
    assert lib.iq4xs_set_baseline_threshold(-1) == B.ERR_ARG
    # the library's own calls never take the advice as an explicit path
    out = ctypes.c_int()
    rc = lib.iq4xs_matmul(ctypes.c_void_p(16), 256, 512, ctypes.c_void_p(16), ctypes.c_void_p(16),
                          8, ctypes.c_void_p(16), 256, B.PATH_BASELINE, 0)
    assert rc == B.ERR_ARG, rc
    B.reset_dispatch()


def test_tc_operand_bytes(lib):
    # M rounds up to a multiple of 16 (at most 128 per tile); q*d as an exact
    # fp16 pair (4 bytes) per padded activation, plus one fp32 power of two
    # per padded row and span of 1024 values
    assert B.iq4xs_tc_operand_bytes(1, 1024) == 16 * 1024 * 4 + 16 * 1 * 4
    assert B.iq4xs_tc_operand_bytes(96, 4096) == 96 * 4096 * 4 + 96 * 4 * 4
    assert B.iq4xs_tc_operand_bytes(129, 512) == 2 * 128 * 512 * 4 + 2 * 128 * 1 * 4
    assert B.iq4xs_tc_operand_bytes(0, 1024) == 0
    assert B.iq4xs_tc_operand_bytes(4, 1000) == 0


def test_prepared_form_argument_errors(lib):
    p = ctypes.c_void_p(0x10000)
    odd = ctypes.c_void_p(0x10008)
    assert lib.iq4xs_quantize_q8_1_tc(p, 1, 256, 256, p, p, None, 0) == B.ERR_ARG
    assert lib.iq4xs_quantize_q8_1_tc(p, 1, 256, 256, p, p, odd, 0) == B.ERR_ALIGN
    assert lib.iq4xs_quantize_q8_1_tc(p, 1, 300, 300, p, p, p, 0) == B.ERR_SHAPE
    assert lib.iq4xs_matmul_tc_operand(None, 0, 8, 512, p, 1, p, 8, 0) == B.ERR_ARG
    assert lib.iq4xs_matmul_tc_operand(p, 0, 8, 512, None, 1, p, 8, 0) == B.ERR_ARG
    assert lib.iq4xs_matmul_tc_operand(p, 3, 8, 512, p, 1, p, 8, 0) == B.ERR_ARG
    assert lib.iq4xs_matmul_tc_operand(p, 0, 8, 768, p, 1, p, 8, 0) == B.ERR_SHAPE
    assert lib.iq4xs_matmul_tc_operand(p, 0, 8, 512, p, 1, p, 4, 0) == B.ERR_ARG
    assert lib.iq4xs_matmul_tc_operand(p, 0, 8, 512, odd, 1, p, 8, 0) == B.ERR_ALIGN


def test_argument_errors_return_before_any_launch(lib):
    p = ctypes.c_void_p(0x10000)      # never dereferenced: validation fails first
    odd = ctypes.c_void_p(0x10008)
    vp = ctypes.c_void_p
    # null pointers
    assert lib.iq4xs_matmul(None, 8, 256, p, p, 1, p, 8, 0, 0) == B.ERR_ARG
    assert lib.iq4xs_matmul(p, 8, 256, None, p, 1, p, 8, 0, 0) == B.ERR_ARG
    assert lib.iq4xs_matmul(p, 8, 256, p, None, 1, p, 8, 0, 0) == B.ERR_ARG
    assert lib.iq4xs_matmul(p, 8, 256, p, p, 1, None, 8, 0, 0) == B.ERR_ARG
    assert lib.iq4xs_quantize_q8_1(None, 1, 256, 256, p, p, 0) == B.ERR_ARG
    assert lib.iq4xs_quantize_q8_1(p, 1, 256, 256, p, None, 0) == B.ERR_ARG
    assert lib.iq4xs_dequantize(p, 8, 256, None, 0, 0) == B.ERR_ARG
    # shapes
    assert lib.iq4xs_matmul(p, 8, 300, p, p, 1, p, 8, 0, 0) == B.ERR_SHAPE
    assert lib.iq4xs_matmul(p, 8, 256, p, p, 0, p, 8, 0, 0) == B.ERR_SHAPE
    assert lib.iq4xs_matmul(p, 0, 256, p, p, 1, p, 8, 0, 0) == B.ERR_SHAPE
    assert lib.iq4xs_quantize_q8_1(p, 1, 100, 100, p, p, 0) == B.ERR_SHAPE
    # bad ldy / ldx / path / dtype
    assert lib.iq4xs_matmul(p, 8, 256, p, p, 1, p, 4, 0, 0) == B.ERR_ARG
    assert lib.iq4xs_matmul(p, 8, 256, p, p, 1, p, 8, 7, 0) == B.ERR_ARG
    assert lib.iq4xs_quantize_q8_1(p, 1, 256, 255, p, p, 0) == B.ERR_ARG
    assert lib.iq4xs_dequantize(p, 8, 256, p, 5, 0) == B.ERR_ARG
    # alignment: W, qs (16 bytes), ds (4 bytes)
    assert lib.iq4xs_matmul(odd, 8, 256, p, p, 1, p, 8, 1, 0) == B.ERR_ALIGN
    assert lib.iq4xs_matmul(p, 8, 256, odd, p, 1, p, 8, 1, 0) == B.ERR_ALIGN
    assert lib.iq4xs_matmul(p, 8, 256, p, ctypes.c_void_p(0x10002), 1, p, 8, 1, 0) == B.ERR_ALIGN
    assert lib.iq4xs_quantize_q8_1(odd, 1, 256, 256, p, p, 0) == B.ERR_ALIGN
    # the tensor-core path needs K % 512 == 0
    assert lib.iq4xs_matmul(p, 8, 768, p, p, 1, p, 8, 2, 0) == B.ERR_SHAPE


def test_weight_formats_sizes_and_argument_errors(lib):
    # bytes per [N][K]: IQ4_XS 136 per 256 weights, Q4_0 / IQ4_NL 18 per 32
    assert B.iq4xs_weight_bytes("iq4_xs", 3, 512) == 3 * 2 * 136
    assert B.iq4xs_weight_bytes("q4_0", 3, 512) == 3 * 16 * 18
    assert B.iq4xs_weight_bytes("iq4_nl", 5, 4096) == 5 * 128 * 18
    assert B.iq4xs_weight_bytes(3, 3, 512) == 0 and B.iq4xs_weight_bytes(1, 3, 96) == 0
    p = ctypes.c_void_p(0x10000)
    for wt in (0, 1, 2):
        assert lib.iq4xs_matmul_wt(None, wt, 8, 256, p, p, 1, p, 8, 0, 0) == B.ERR_ARG
        assert lib.iq4xs_matmul_wt(p, wt, 8, 288, p, p, 1, p, 8, 0, 0) == B.ERR_SHAPE
        assert lib.iq4xs_matmul_wt(p, wt, 8, 768, p, p, 1, p, 8, 2, 0) == B.ERR_SHAPE
        assert lib.iq4xs_matmul_wt(ctypes.c_void_p(0x10004), wt, 8, 256, p, p, 1, p, 8, 1,
                                   0) == B.ERR_ALIGN
        assert lib.iq4xs_dequantize_wt(p, wt, 8, 256, p, 2, 0) == B.ERR_ARG
    for bad in (-1, 3, 99):
        assert lib.iq4xs_matmul_wt(p, bad, 8, 256, p, p, 1, p, 8, 0, 0) == B.ERR_ARG
        assert lib.iq4xs_dequantize_wt(p, bad, 8, 256, p, 0, 0) == B.ERR_ARG


@pytest.mark.skipif(os.path.exists("/dev/nvidia0"), reason="host without a GPU only")
def test_valid_call_without_gpu_reports_device_error(lib):
    p = ctypes.c_void_p(0x10000)
    assert lib.iq4xs_matmul(p, 8, 256, p, p, 1, p, 8, 1, 0) == B.ERR_DEVICE


def test_mma_launch_table_validation(lib):
    def put(entries):
        flat = [v for e in entries for v in e]
        arr = (ctypes.c_int64 * max(1, len(flat)))(*flat)
        return lib.iq4xs_set_mma_launch_table(arr, len(entries))
    good = (4096, 4096, 8, 128, 4, 1)
    assert put([good]) == B.OK
    for bad in ((0, 4096, 8, 128, 4, 1), (4096, 768, 8, 128, 4, 1), (4096, 4096, 12, 128, 4, 1),
                (4096, 4096, 8, 48, 4, 1), (4096, 4096, 8, 288, 4, 1), (4096, 4096, 8, 128, 9, 1),
                (4096, 4096, 8, 128, 0, 1), (4096, 4096, 8, 128, 4, 3)):
        assert put([good, bad]) == B.ERR_ARG, bad
    assert lib.iq4xs_set_mma_launch_table(None, 1) == B.ERR_ARG
    assert put([good] * 257) == B.ERR_ARG
    assert put([]) == B.OK
    B.reset_dispatch()


def test_mma_launch_config_validation(lib):
    r, sp, o = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    assert lib.iq4xs_mma_launch_config(8, 4096, 4096, None, ctypes.byref(sp), ctypes.byref(o)) == B.ERR_ARG
    for M, N, K in ((0, 4096, 4096), (8, 0, 4096), (8, 4096, 768), (8, 4096, 0), (40000, 4096, 4096)):
        assert lib.iq4xs_mma_launch_config(M, N, K, ctypes.byref(r), ctypes.byref(sp),
                                           ctypes.byref(o)) == B.ERR_SHAPE, (M, N, K)


def test_largest_m_is_32768(lib):
    p = ctypes.c_void_p(0x10000)
    out = ctypes.c_int(-1)
    assert lib.iq4xs_select_path(32769, 8, 256, ctypes.byref(out)) == B.ERR_SHAPE
    assert lib.iq4xs_matmul(p, 8, 256, p, p, 32769, p, 8, 0, 0) == B.ERR_SHAPE
    assert lib.iq4xs_quantize_q8_1(p, 32769, 256, 256, p, p, 0) == B.ERR_SHAPE
    assert lib.iq4xs_quantize_q8_1_tc(p, 32769, 256, 256, p, p, p, 0) == B.ERR_SHAPE
    assert lib.iq4xs_matmul_grouped(p, 16 * 136, 2, 8, 512, p, p, p, 32769, p, 8, 0) == B.ERR_SHAPE
    assert lib.iq4xs_select_path(32768, 8, 256, ctypes.byref(out)) == B.OK


def test_status_strings(lib):
    for s in range(8):
        assert B.iq4xs_status_string(s) != "unknown status"


def test_bounds_checked_build_exports_and_flags(lib):
    """The debug build with bounds checks builds from the same sources,
    exports every declared function and says which build it is; the margin
    hook is refused by the normal build."""
    blib = B.load(build.build(bounds_check=True))
    for name in B.header_functions():
        assert hasattr(blib, name), name
    out = ctypes.c_int(-1)
    assert blib.iq4xs_bounds_checked(ctypes.byref(out)) == B.OK and out.value == 1
    assert lib.iq4xs_bounds_checked(ctypes.byref(out)) == B.OK and out.value == 0
    assert lib.iq4xs_bounds_checked(None) == B.ERR_ARG
    assert lib.iq4xs_test_bounds_margin(16) == B.ERR_ARG
    assert blib.iq4xs_test_bounds_margin(-1) == B.ERR_ARG


def test_linear_workspace_and_validation(lib):
    _dispatch(4, 8)
    # the least: qs, then ds 16-byte aligned (1.125 bytes per activation);
    # the fastest form adds the prepared operand on the tensor-core path
    assert B.iq4xs_linear_workspace_bytes(2, 4096, 4096) == 2 * 4096 + 2 * 128 * 4
    assert B.iq4xs_linear_workspace_min_bytes(2, 4096, 4096) == 2 * 4096 + 2 * 128 * 4
    assert B.iq4xs_linear_workspace_min_bytes(96, 4096, 4096) == 96 * 4096 + 96 * 128 * 4
    assert (B.iq4xs_linear_workspace_bytes(96, 4096, 4096) ==
            96 * 4096 + 96 * 128 * 4 + B.iq4xs_tc_operand_bytes(96, 4096))
    assert B.iq4xs_linear_workspace_min_bytes(3, 8, 256) == 3 * 256 + 3 * 8 * 4
    assert B.iq4xs_linear_workspace_bytes(0, 8, 256) == 0
    p = ctypes.c_void_p(0x10000)
    need = B.iq4xs_linear_workspace_bytes(96, 4096, 4096)
    least = B.iq4xs_linear_workspace_min_bytes(96, 4096, 4096)
    assert lib.iq4xs_linear(p, 4096, 4096, p, 96, 4096, p, 4096, p, least - 1, 0) == B.ERR_ARG
    assert lib.iq4xs_linear(p, 4096, 4096, p, 96, 4096, p, 4096, None, need, 0) == B.ERR_ARG
    assert lib.iq4xs_linear(p, 4096, 300, p, 96, 4096, p, 4096, p, need, 0) == B.ERR_SHAPE
    B.reset_dispatch()


def test_grouped_argument_errors_return_before_any_launch(lib):
    p = ctypes.c_void_p(256)  # never dereferenced: validation fails first
    f = lib.iq4xs_matmul_grouped
    N, K, stride = 128, 512, 128 * 2 * 136
    assert f(None, stride, 2, N, K, p, p, p, 1, p, N, 0) == B.ERR_ARG
    assert f(p, stride, 2, N, K, p, p, None, 1, p, N, 0) == B.ERR_ARG
    assert f(p, stride, 0, N, K, p, p, p, 1, p, N, 0) == B.ERR_SHAPE
    assert f(p, stride, 70000, N, K, p, p, p, 1, p, N, 0) == B.ERR_SHAPE
    assert f(p, stride, 2, N, 500, p, p, p, 1, p, N, 0) == B.ERR_SHAPE
    assert f(p, stride - 16, 2, N, K, p, p, p, 1, p, N, 0) == B.ERR_ARG   # overlapping experts
    assert f(p, stride + 8, 2, N, K, p, p, p, 1, p, N, 0) == B.ERR_ARG    # stride not 16-byte
    assert f(p, stride, 2, N, K, p, p, p, 0, p, N, 0) == B.ERR_ARG        # no rows
    assert f(p, stride, 2, N, K, p, p, p, 1, p, N - 1, 0) == B.ERR_ARG    # ldy < N
    assert f(ctypes.c_void_p(264), stride, 2, N, K, p, p, p, 1, p, N, 0) == B.ERR_ALIGN


def test_crossover_classes(lib):
    _dispatch(4, 0)  # the DP4A / TC choice alone
    try:
        B.iq4xs_set_crossover_classes([(50_000_000, 2), (150_000_000, 6)])
        assert B.iq4xs_select_path(4, 4096, 4096) == B.PATH_DP4A      # below every class: 4
        assert B.iq4xs_select_path(5, 4096, 4096) == B.PATH_TC
        assert B.iq4xs_select_path(2, 12288, 5120) == B.PATH_DP4A     # 63M weights: 2
        assert B.iq4xs_select_path(3, 12288, 5120) == B.PATH_TC
        assert B.iq4xs_select_path(6, 34816, 5120) == B.PATH_DP4A     # 178M weights: 6
        assert B.iq4xs_select_path(7, 34816, 5120) == B.PATH_TC
        i64 = ctypes.c_int64
        assert lib.iq4xs_set_crossover_classes((i64 * 1)(0), (i64 * 1)(3), 1) == B.ERR_ARG
        assert lib.iq4xs_set_crossover_classes((i64 * 1)(5), (i64 * 1)(-1), 1) == B.ERR_ARG
        assert lib.iq4xs_set_crossover_classes(None, None, 17) == B.ERR_ARG
        assert B.iq4xs_select_path(2, 12288, 5120) == B.PATH_DP4A     # unchanged after errors
        B.iq4xs_set_crossover_classes([])
        assert B.iq4xs_select_path(4, 12288, 5120) == B.PATH_DP4A
    finally:
        B.reset_dispatch()
