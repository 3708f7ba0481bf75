"""The C-ABI library without a GPU: it loads, exports every function that
include/bfp8.h declares, and rejects bad arguments on the host before any CUDA
call (no launch happens for these cases, so they are safe anywhere)."""
import ctypes

import pytest

import blockwise_fp8_linear_weight_b300 as bfp8
from blockwise_fp8_linear_weight_b300 import build as bfp8_build

OK, EINVAL, EALIGN, ESHAPE = 0, -1, -2, -3
A = 0x10000  # a 16-byte-aligned fake device address; never dereferenced in these cases


@pytest.fixture(scope="module")
def lib():
    bfp8_build.build()
    return bfp8.load_library()


def test_exports_every_declared_function(lib):
    names = bfp8.header_functions()
    assert set(names) >= {"fp8_quantize_act", "fp8_quantize_weight", "fp8_quantize_transpose",
                          "fp8_quantize_act_transpose",
                          "fp8_block_gemm_fwd", "fp8_block_gemm_dgrad", "fp8_block_gemm_wgrad",
                          "fp8_block_gemm_wgrad_acc",
                          "bfp8_status_string", "bfp8_last_device_status", "bfp8_set_gemm_tile_n",
                          "bfp8_set_wait_limit_ns", "bfp8_test_stall_producers", "bfp8_kernel_launches",
                          "fp8_block_gemm_workspace_bytes",
                          "muonh_partials_len", "muonh_normalize", "muonh_apply", "muonh_apply_static",
                          "bf16_gemm_axpby", "muonh_newton_schulz_work_bytes", "muonh_newton_schulz"}
    cdll = ctypes.CDLL(bfp8.LIB_PATH)
    for n in names:
        assert hasattr(cdll, n), n


def test_status_strings(lib):
    for code, name in bfp8.STATUS.items():
        assert lib.bfp8_status_string(code).decode().startswith(name)
    assert lib.bfp8_status_string(12345) == b"unknown bfp8 status"


def test_tile_knob(lib):
    assert lib.bfp8_set_gemm_tile_n(64) == EINVAL
    prev = lib.bfp8_set_gemm_tile_n(256)
    assert lib.bfp8_set_gemm_tile_n(prev) == 256


def test_launch_counter(lib):
    n = ctypes.c_int64(-1)
    assert lib.bfp8_kernel_launches(None) == EINVAL
    assert lib.bfp8_kernel_launches(ctypes.byref(n)) == OK
    assert n.value >= 0
    # calls refused on the host launch nothing
    lib.fp8_block_gemm_fwd(A, 128, A, 4, A, 128, A, A, 128, 4, 130, 128, None, 0, None)
    m = ctypes.c_int64(-1)
    lib.bfp8_kernel_launches(ctypes.byref(m))
    assert m.value == n.value


def test_wait_limit_and_stall_switch_arguments(lib):
    assert lib.bfp8_set_wait_limit_ns(999) == EINVAL
    assert lib.bfp8_set_wait_limit_ns(-1) == EINVAL
    assert lib.bfp8_set_wait_limit_ns(60_000_000_001) == EINVAL
    assert lib.bfp8_set_wait_limit_ns(1000) == OK
    assert lib.bfp8_set_wait_limit_ns(0) == OK  # back to the default
    assert lib.bfp8_test_stall_producers(2) == EINVAL
    assert lib.bfp8_test_stall_producers(1) == 0
    assert lib.bfp8_test_stall_producers(0) == 1


def test_quantiser_argument_checks(lib):
    s = None
    # C not a multiple of 128
    assert lib.fp8_quantize_act(A, 4, 100, 128, A, 128, A, 4, s) == ESHAPE
    # empty input is a no-op
    assert lib.fp8_quantize_act(None, 0, 128, 128, None, 128, None, 0, s) == OK
    assert lib.fp8_quantize_act(A, -1, 128, 128, A, 128, A, 4, s) == EINVAL
    # null output, short leading dimension
    assert lib.fp8_quantize_act(A, 4, 128, 128, None, 128, A, 4, s) == EINVAL
    assert lib.fp8_quantize_act(A, 4, 256, 128, A, 256, A, 4, s) == EINVAL
    assert lib.fp8_quantize_act(A, 8, 128, 128, A, 128, A, 4, s) == EINVAL  # lds < R
    # misaligned input pointer / row stride
    assert lib.fp8_quantize_act(A + 2, 4, 128, 128, A, 128, A, 4, s) == EALIGN
    assert lib.fp8_quantize_act(A, 4, 128, 132, A, 128, A, 4, s) == EALIGN
    assert lib.fp8_quantize_weight(A, 100, 128, 128, A, 128, A, s) == ESHAPE
    assert lib.fp8_quantize_weight(A, 128, 128, 128, A + 4, 128, A, s) == EALIGN
    assert lib.fp8_quantize_transpose(A, 4, 120, 128, A, 128, A, 128, s) == ESHAPE
    assert lib.fp8_quantize_transpose(A, 200, 128, 128, A, 200, A, 128, s) == EINVAL  # ldqt < R128
    assert lib.fp8_quantize_transpose(A, 200, 128, 128, A, 264, A, 128, s) == EALIGN  # ldqt % 16
    assert lib.fp8_quantize_transpose(A, 200, 128, 128, A, 256, A + 4, 128, s) == EALIGN
    dual = lib.fp8_quantize_act_transpose
    assert dual(None, 0, 128, 128, None, 128, None, 0, None, 128, None, 128, s) == OK
    assert dual(A, 200, 100, 128, A, 128, A, 200, A, 256, A, 128, s) == ESHAPE
    assert dual(A, 200, 128, 128, A, 128, A, 200, A, 200, A, 128, s) == EINVAL   # ldqt < R128
    assert dual(A, 200, 128, 128, A, 128, A, 100, A, 256, A, 128, s) == EINVAL   # lds < R
    assert dual(A, 200, 128, 128, None, 128, A, 200, A, 256, A, 128, s) == EINVAL
    assert dual(A, 200, 128, 128, A, 128, A, 200, A + 8, 256, A, 128, s) == EALIGN
    assert dual(A + 2, 200, 128, 128, A, 128, A, 200, A, 256, A, 128, s) == EALIGN


def test_gemm_argument_checks(lib):
    s = None
    # fwd: N, K multiples of 128
    assert lib.fp8_block_gemm_fwd(A, 128, A, 4, A, 128, A, A, 128, 4, 130, 128, None, 0, s) == ESHAPE
    assert lib.fp8_block_gemm_fwd(A, 128, A, 4, A, 128, A, A, 128, 4, 128, 96, None, 0, s) == ESHAPE
    assert lib.fp8_block_gemm_fwd(A, 128, A, 4, A, 128, A, A, 128, 0, 128, 128, None, 0, s) == OK
    assert lib.fp8_block_gemm_fwd(None, 128, A, 4, A, 128, A, A, 128, 4, 128, 128, None, 0, s) == EINVAL
    assert lib.fp8_block_gemm_fwd(A, 128, A, 3, A, 128, A, A, 128, 4, 128, 128, None, 0, s) == EINVAL  # ldsx < M
    assert lib.fp8_block_gemm_fwd(A, 128, A, 6, A, 128, A, A, 128, 6, 128, 128, None, 0, s) == EALIGN  # ldsx % 4
    assert lib.fp8_block_gemm_fwd(A, 136, A, 4, A, 136, A, A, 128, 4, 128, 128, None, 0, s) == EALIGN  # ldq % 16
    assert lib.fp8_block_gemm_fwd(A, 128, A + 4, 4, A, 128, A, A, 128, 4, 128, 128, None, 0, s) == EALIGN
    assert lib.fp8_block_gemm_dgrad(A, 128, A, 4, A, 96, A, A, 96, 4, 128, 96, None, 0, s) == ESHAPE
    assert lib.fp8_block_gemm_dgrad(A, 128, A, 4, A, 128, A, A, 100, 4, 128, 128, None, 0, s) == EINVAL
    # wgrad: M >= 1, ld of transposed codes >= M128
    assert lib.fp8_block_gemm_wgrad(A, 128, A, 128, A, 128, A, 128, A, 128, 0, 128, 128, None, 0, s) == ESHAPE
    assert lib.fp8_block_gemm_wgrad(A, 128, A, 128, A, 128, A, 128, A, 128, 200, 128, 128, None, 0, s) == EINVAL
    assert lib.fp8_block_gemm_wgrad(A, 256, A, 126, A, 256, A, 128, A, 128, 200, 128, 128, None, 0, s) == EINVAL
    assert lib.fp8_block_gemm_wgrad(A, 256, A, 130, A, 256, A, 128, A, 128, 200, 128, 128, None, 0, s) == EALIGN
    # the optional workspace: a negative size or a misaligned pointer is refused
    assert lib.fp8_block_gemm_fwd(A, 128, A, 4, A, 128, A, A, 128, 4, 128, 128, A, -1, s) == EINVAL
    assert lib.fp8_block_gemm_fwd(A, 128, A, 4, A, 128, A, A, 128, 4, 128, 128, A + 8, 1 << 20, s) == EALIGN
    assert lib.fp8_block_gemm_dgrad(A, 128, A, 4, A, 128, A, A, 128, 4, 128, 128, A + 4, 1 << 20, s) == EALIGN
    assert lib.fp8_block_gemm_wgrad(A, 256, A, 128, A, 256, A, 128, A, 128, 200, 128, 128, A, -5, s) == EINVAL
    assert lib.fp8_block_gemm_workspace_bytes(None) == EINVAL
    # wgrad accumulating into FP32: same operand rules, FP32 main gradient with ldmg % 4 == 0
    acc = lib.fp8_block_gemm_wgrad_acc
    assert acc(A, 128, A, 128, A, 128, A, 128, A, 128, 0, 128, 128, s) == ESHAPE
    assert acc(A, 256, A, 128, A, 256, A, 128, A, 128, 200, 128, 96, s) == ESHAPE
    assert acc(A, 256, A, 128, A, 256, A, 128, None, 128, 200, 128, 128, s) == EINVAL
    assert acc(A, 256, A, 128, A, 256, A, 128, A, 100, 200, 128, 128, s) == EINVAL  # ldmg < K
    assert acc(A, 256, A, 128, A, 256, A, 128, A, 130, 200, 128, 128, s) == EALIGN  # ldmg % 4
    assert acc(A, 256, A, 128, A, 256, A, 128, A + 8, 128, 200, 128, 128, s) == EALIGN


def test_muonh_argument_checks(lib):
    s = None
    f = ctypes.c_float
    assert lib.muonh_partials_len(None) == EINVAL
    assert lib.muonh_normalize(A, 4, 6, 8, A, 8, A, 1 << 12, f(0.0), s) == ESHAPE       # cols % 4
    assert lib.muonh_normalize(None, 4, 8, 8, A, 8, A, 1 << 12, f(0.0), s) == EINVAL
    assert lib.muonh_normalize(A, 4, 8, 4, A, 8, A, 1 << 12, f(0.0), s) == EINVAL       # ldg < cols
    assert lib.muonh_normalize(A + 4, 4, 8, 8, A, 8, A, 1 << 12, f(0.0), s) == EALIGN
    assert lib.muonh_normalize(A, 4, 8, 8, A, 8, A, 1 << 12, f(-1.0), s) == EINVAL      # eps < 0
    assert lib.muonh_apply(A, 8, A, 8, 4, 8, A, 1 << 12, f(0.1), f(0.0), s) == EINVAL   # radius 0
    assert lib.muonh_apply(A, 8, A, 8, 4, 8, A, 1 << 12, f(-0.1), f(1.0), s) == EINVAL  # lr < 0
    assert lib.muonh_apply(A, 10, A, 8, 4, 8, A, 1 << 12, f(0.1), f(1.0), s) == EALIGN  # ldw % 4
    assert lib.muonh_apply(A, 8, A + 2, 8, 4, 8, A, 1 << 12, f(0.1), f(1.0), s) == EALIGN
    # a partials buffer shorter than muonh_partials_len() is refused (without a B300 the
    # device query refuses first)
    assert lib.muonh_normalize(A, 4, 8, 8, A, 8, A, 0, f(0.0), s) != OK
    assert lib.muonh_apply_static(A, 8, A, 8, 4, 8, f(0.1), f(0.0), s) == EINVAL   # radius 0
    assert lib.muonh_apply_static(A, 8, A, 8, 4, 6, f(0.1), f(1.0), s) == ESHAPE   # cols % 4


def test_bf16_gemm_and_newton_schulz_argument_checks(lib):
    import ctypes as ct
    g = lib.bf16_gemm_axpby
    f = ct.c_float
    assert g(A, 64, A, 64, 0, None, 0, A, 64, 0, 64, 64, f(1), f(0), None) == EINVAL       # M < 1
    assert g(A, 64, A, 64, 2, None, 0, A, 64, 64, 64, 64, f(1), f(0), None) == EINVAL      # bad layout flag
    assert g(A, 64, A, 64, 0, None, 0, A, 64, 64, 60, 64, f(1), f(0), None) == ESHAPE      # N % 8
    assert g(A, 64, A, 64, 0, None, 0, A, 64, 64, 64, 64, f(1), f(1), None) == EINVAL      # beta != 0, no C
    assert g(A, 32, A, 64, 0, None, 0, A, 64, 64, 64, 64, f(1), f(0), None) == EINVAL      # lda < K
    assert g(A + 8, 64, A, 64, 0, None, 0, A, 64, 64, 64, 64, f(1), f(0), None) == EALIGN  # misaligned a
    assert g(A, 68, A, 64, 0, None, 0, A, 64, 64, 64, 64, f(1), f(0), None) == EALIGN      # lda % 8
    n = ct.c_int64(0)
    assert lib.muonh_newton_schulz_work_bytes(64, 256, ct.byref(n)) == OK
    # A and B: 64 x 64, two Y buffers: 64 x 256, BF16
    assert n.value == 2 * (2 * 64 * 64 + 2 * 64 * 256)
    assert lib.muonh_newton_schulz_work_bytes(256, 64, ct.byref(n)) == OK and n.value == 2 * (2 * 64 * 64 + 2 * 64 * 256)
    assert lib.muonh_newton_schulz_work_bytes(0, 64, ct.byref(n)) == EINVAL
    ns = lib.muonh_newton_schulz
    need = 2 * (2 * 64 * 64 + 2 * 64 * 256)
    assert ns(A, 64, 256, 256, A, need - 1, 5, f(3.4445), f(-4.775), f(2.0315), None) == EINVAL  # short scratch
    assert ns(A, 60, 256, 256, A, need, 5, f(3.4445), f(-4.775), f(2.0315), None) == ESHAPE      # rows % 8
    assert ns(A, 64, 256, 200, A, need, 5, f(3.4445), f(-4.775), f(2.0315), None) == EINVAL      # ldx < cols
    assert ns(A, 64, 256, 260, A, need, 5, f(3.4445), f(-4.775), f(2.0315), None) == EALIGN      # ldx % 8
    assert ns(A, 64, 256, 256, A, need, -1, f(3.4445), f(-4.775), f(2.0315), None) == EINVAL     # steps < 0
