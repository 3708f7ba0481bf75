"""Pins for the oracle's three FP64 blockwise GEMMs (fwd, dgrad, wgrad).

Checked against facts fixed outside the oracle's own loops:
  * exact integer chunk sums (int64 on the integer reading of the codes) give
    bit-identical results, so the FP64 chunk sums are exact;
  * brute force: dequantise every operand with ml_dtypes' decoder, multiply
    with numpy in FP64 (a different summation order; agreement to ~1e-12);
  * closed forms: unit scales with small-integer codes give the exact integer
    GEMM; identity weight blocks return the dequantised activations;
  * dgrad is fwd with the weight codes and block scales transposed;
  * powers of two on the scales scale the result exactly;
  * end to end, quantise-then-GEMM approximates the BF16 product to within
    E4M3 precision (this catches a transposed operand or scale anywhere);
  * accumulating wgrad into an FP32 main gradient matches brute force plus the
    main gradient, and accumulating twice from zero doubles dW exactly.
"""
import ml_dtypes
import numpy as np
import pytest

import oracle
from workloads import bf16_bits, bits_to_f32, random_bits, random_codes, random_scales

TILE = 128


def deq(codes):
    return np.asarray(codes, dtype=np.uint8).view(ml_dtypes.float8_e4m3fn).astype(np.float64)


def brute_fwd(qx, sx, qw, sw):
    M, K = qx.shape
    N = qw.shape[0]
    X = deq(qx) * np.repeat(sx.astype(np.float64).T, TILE, axis=1)[:, :K]
    W = deq(qw) * np.kron(sw.astype(np.float64), np.ones((TILE, TILE)))
    return X @ W.T


def brute_dgrad(qdy, sdy, qw, sw):
    dY = deq(qdy) * np.repeat(sdy.astype(np.float64).T, TILE, axis=1)
    W = deq(qw) * np.kron(sw.astype(np.float64), np.ones((TILE, TILE)))
    return dY @ W


def brute_wgrad(qdyt, sdyt, qxt, sxt):
    dYt = deq(qdyt) * np.repeat(sdyt.astype(np.float64).T, TILE, axis=1)
    Xt = deq(qxt) * np.repeat(sxt.astype(np.float64).T, TILE, axis=1)
    return dYt @ Xt.T


def _operands(M, N, K, seed):
    qx = random_codes((M, K), seed)
    sx = random_scales((K // TILE, M), seed + 1)
    qw = random_codes((N, K), seed + 2)
    sw = random_scales((N // TILE, K // TILE), seed + 3)
    return qx, sx, qw, sw


def _close(a, b, rtol=1e-12):
    scale = np.abs(b).max() + 1e-300
    return np.abs(a - b).max() <= rtol * scale


@pytest.mark.parametrize("M,N,K", [(1, 128, 128), (37, 256, 384), (130, 128, 256)])
def test_fp64_chunk_sums_are_exact(oracle_lib, M, N, K):
    qx, sx, qw, sw = _operands(M, N, K, seed=M)
    a = oracle.gemm_fwd(qx, sx, qw, sw)
    b = oracle.gemm_fwd(qx, sx, qw, sw, exact_int=True)
    assert np.array_equal(a.view(np.uint64), b.view(np.uint64))


@pytest.mark.parametrize("M", [1, 5, 128, 200])
@pytest.mark.parametrize("nk", [(1, 1), (2, 3), (3, 2)])
def test_brute_force_all_passes(oracle_lib, M, nk):
    N, K = nk[0] * TILE, nk[1] * TILE
    qx, sx, qw, sw = _operands(M, N, K, seed=100 + M)
    assert _close(oracle.gemm_fwd(qx, sx, qw, sw), brute_fwd(qx, sx, qw, sw))
    qdy = random_codes((M, N), 7)
    sdy = random_scales((N // TILE, M), 8)
    assert _close(oracle.gemm_dgrad(qdy, sdy, qw, sw), brute_dgrad(qdy, sdy, qw, sw))
    M128 = (M + TILE - 1) // TILE * TILE
    qdyt = random_codes((N, M128), 9)
    qxt = random_codes((K, M128), 10)
    qdyt[:, M:] = 0
    qxt[:, M:] = 0
    sdyt = random_scales((M128 // TILE, N), 11)
    sxt = random_scales((M128 // TILE, K), 12)
    got = oracle.gemm_wgrad(qdyt, sdyt, qxt, sxt, M)
    assert _close(got, brute_wgrad(qdyt, sdyt, qxt, sxt))
    # the zero pad contributes nothing: brute force over the valid tokens only
    valid = brute_wgrad(qdyt[:, :M], sdyt, qxt[:, :M], sxt) if M % TILE == 0 else None
    if valid is not None:
        assert _close(got, valid)


def test_row_subset_matches_full(oracle_lib):
    qx, sx, qw, sw = _operands(64, 256, 256, seed=3)
    rows = np.array([0, 17, 63, 5])
    full = oracle.gemm_fwd(qx, sx, qw, sw)
    assert np.array_equal(oracle.gemm_fwd(qx, sx, qw, sw, rows=rows), full[rows])


def test_unit_scales_small_integers_is_integer_gemm(oracle_lib):
    rng = np.random.default_rng(4)
    ints = np.arange(-16, 17)
    code_of = {int(v): c for c in range(256) if (c & 0x7F) != 0x7F
               for v in [deq(np.array([c]))[0]] if float(v).is_integer() and abs(v) <= 16}
    code_of[0] = 0
    a = rng.choice(ints, size=(9, 256))
    b = rng.choice(ints, size=(128, 256))
    qa = np.vectorize(code_of.get)(a).astype(np.uint8)
    qb = np.vectorize(code_of.get)(b).astype(np.uint8)
    y = oracle.gemm_fwd(qa, np.ones((2, 9), np.float32), qb, np.ones((1, 2), np.float32))
    assert np.array_equal(y, (a.astype(np.int64) @ b.T.astype(np.int64)).astype(np.float64))


def test_identity_weight_returns_dequantised_input(oracle_lib):
    K = 256
    qx = random_codes((20, K), 5)
    sx = random_scales((K // TILE, 20), 6)
    qw = np.zeros((K, K), dtype=np.uint8)
    np.fill_diagonal(qw, 0x38)  # code 0x38 = 1.0
    y = oracle.gemm_fwd(qx, sx, qw, np.ones((2, 2), np.float32))
    expect = deq(qx) * np.repeat(sx.astype(np.float64).T, TILE, axis=1)
    assert np.array_equal(y, expect)


def test_dgrad_is_fwd_with_transposed_weight(oracle_lib):
    M, N, K = 33, 384, 256
    qdy = random_codes((M, N), 1)
    sdy = random_scales((N // TILE, M), 2)
    qw = random_codes((N, K), 3)
    sw = random_scales((N // TILE, K // TILE), 4)
    a = oracle.gemm_dgrad(qdy, sdy, qw, sw)
    b = oracle.gemm_fwd(qdy, sdy, np.ascontiguousarray(qw.T), np.ascontiguousarray(sw.T))
    assert np.array_equal(a, b)


def test_scales_times_powers_of_two(oracle_lib):
    qx, sx, qw, sw = _operands(17, 256, 384, seed=21)
    y = oracle.gemm_fwd(qx, sx, qw, sw)
    y2 = oracle.gemm_fwd(qx, sx * np.float32(2.0 ** 5), qw, sw * np.float32(2.0 ** -9))
    assert np.array_equal(y2, y * 2.0 ** -4)


def test_single_nonzero_chunk_is_one_dot_product(oracle_lib):
    qx, sx, qw, sw = _operands(3, 128, 384, seed=31)
    qx[:, :128] = 0
    qx[:, 256:] = 0
    y = oracle.gemm_fwd(qx, sx, qw, sw)
    dots = deq(qx[:, 128:256]) @ deq(qw[:, 128:256]).T
    expect = dots * sx[1].astype(np.float64)[:, None] * np.float64(sw[0, 1])
    assert _close(y, expect, 1e-15)


@pytest.mark.parametrize("M", [128, 200])
def test_quantise_then_gemm_approximates_bf16_product(oracle_lib, M):
    N, K = 256, 384
    x = random_bits((M, K), 41)
    w = random_bits((N, K), 42, std=0.02)
    dy = random_bits((M, N), 43)
    X, W, dY = (bits_to_f32(a).astype(np.float64) for a in (x, w, dy))

    def rel(a, b):
        return np.linalg.norm(a - b) / np.linalg.norm(b)

    qx, sx = oracle.quantize_act(x)
    qw, sw = oracle.quantize_weight(w)
    assert rel(oracle.gemm_fwd(qx, sx, qw, sw), X @ W.T) < 0.06
    qdy, sdy = oracle.quantize_act(dy)
    assert rel(oracle.gemm_dgrad(qdy, sdy, qw, sw), dY @ W) < 0.06
    qdyt, sdyt = oracle.quantize_transpose(dy)
    qxt, sxt = oracle.quantize_transpose(x)
    assert rel(oracle.gemm_wgrad(qdyt, sdyt, qxt, sxt, M), dY.T @ X) < 0.06


def _wgrad_operands(M, N, K, seed):
    M128 = (M + TILE - 1) // TILE * TILE
    qdyt = random_codes((N, M128), seed)
    qxt = random_codes((K, M128), seed + 1)
    qdyt[:, M:] = 0
    qxt[:, M:] = 0
    sdyt = random_scales((M128 // TILE, N), seed + 2)
    sxt = random_scales((M128 // TILE, K), seed + 3)
    return qdyt, sdyt, qxt, sxt


@pytest.mark.parametrize("M,N,K", [(1, 128, 128), (200, 256, 384)])
def test_wgrad_accumulate_is_main_plus_brute_force(oracle_lib, M, N, K):
    qdyt, sdyt, qxt, sxt = _wgrad_operands(M, N, K, seed=40 + M)
    main = np.random.default_rng(M).standard_normal((N, K)).astype(np.float32)
    got = oracle.gemm_wgrad_accumulate(main, qdyt, sdyt, qxt, sxt, M)
    want = main.astype(np.float64) + brute_wgrad(qdyt, sdyt, qxt, sxt)
    assert _close(got, want)
    rows = np.array([3, 0, N - 1])
    assert np.array_equal(oracle.gemm_wgrad_accumulate(main, qdyt, sdyt, qxt, sxt, M, rows=rows), got[rows])


def test_wgrad_accumulate_twice_from_zero_doubles(oracle_lib):
    qdyt, sdyt, qxt, sxt = _wgrad_operands(130, 128, 256, seed=77)
    zero = np.zeros((128, 256), dtype=np.float32)
    once = oracle.gemm_wgrad_accumulate(zero, qdyt, sdyt, qxt, sxt, 130)
    assert np.array_equal(once, oracle.gemm_wgrad(qdyt, sdyt, qxt, sxt, 130))
    # dW values are FP64 sums; adding a float32-rounded copy of dW back is what a
    # second call does to an FP32 main gradient, and doubling is exact in FP64
    assert np.array_equal(2.0 * once, once + once)
    twice = oracle.gemm_wgrad_accumulate(once.astype(np.float32), qdyt, sdyt, qxt, sxt, 130)
    assert _close(twice, 2.0 * once, rtol=1e-7)


@pytest.mark.parametrize("total", [1, 127, 128, 1000, 8192, 32768])
def test_tile_rows_cover_every_output_tile(total):
    """The parity tests' row sampler picks at least one row in every 128-row tile."""
    from helpers import tile_rows
    r = tile_rows(total, seed=total)
    assert r.min() == 0 and r.max() == total - 1 and np.all(np.diff(r) > 0)
    assert set(range((total + 127) // 128)) == set((r // 128).tolist())
