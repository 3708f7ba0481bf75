"""Pins for the oracle's three quantisers (1x128 activation tiles, 128x128 weight
blocks, transposed 1x128 tiles), checked against closed forms and invariants
that the definition fixes, not against a retyped copy of the formula:

  * block-max invariant: the largest magnitude of every non-zero tile encodes
    to +-448, because x/s = 448 (1 + e), |e| <= 2^-23, far from the 464 midpoint;
  * power-of-two round trip: a tile of +-2^e with maximum 2^E gets the exact
    codes 7 * 2^(6 - (E - e)) (for E - e <= 15) and dequantises back;
  * scale invariance: x * 2^k gives identical codes and scales * 2^k;
  * all-zero tiles: scale 0, signed-zero codes;
  * rounding bound: every code is within half an E4M3 step of x/s;
  * the three quantisers agree where their definitions coincide
    (transposed tiles are activation tiles of x^T; a weight block's scale is
    the largest of its rows' 1x128 scales; qt = q^T).
"""
import ml_dtypes
import numpy as np
import pytest

import oracle
from workloads import bf16_bits, bits_to_f32, random_bits

TILE = 128


def _tiles_act(x_bits):
    """Yield (values, codes, scale) per 1x128 activation tile from the oracle."""
    q, s = oracle.quantize_act(x_bits)
    xf = bits_to_f32(x_bits)
    R, C = x_bits.shape
    for r in range(R):
        for c in range((C + TILE - 1) // TILE):
            sl = slice(c * TILE, min((c + 1) * TILE, C))
            yield xf[r, sl], q[r, sl], s[c, r]


def _dist_inputs(seed):
    rng = np.random.default_rng(seed)
    return [
        bf16_bits(rng.standard_normal((24, 384)).astype(np.float32)),
        bf16_bits(rng.standard_t(3, size=(24, 384)).astype(np.float32)),
        bf16_bits((rng.standard_normal((24, 384)) * 1e-30).astype(np.float32)),  # tiny, s subnormal
        bf16_bits((rng.standard_normal((24, 384)) * 1e30).astype(np.float32)),   # huge
    ]


@pytest.mark.parametrize("seed", [0, 1])
def test_block_max_encodes_to_448(oracle_lib, seed):
    for x in _dist_inputs(seed):
        for vals, codes, s in _tiles_act(x):
            a = np.abs(vals).max()
            if a == 0:
                continue
            at_max = np.abs(vals) == a
            assert set(codes[at_max] & 0x7F) == {0x7E}
            assert s > 0


def test_block_max_weight_and_transpose(oracle_lib):
    w = random_bits((256, 384), seed=3, std=0.02)
    q, s = oracle.quantize_weight(w)
    wf = bits_to_f32(w)
    for bi in range(2):
        for bj in range(3):
            blk = wf[bi * 128:(bi + 1) * 128, bj * 128:(bj + 1) * 128]
            qb = q[bi * 128:(bi + 1) * 128, bj * 128:(bj + 1) * 128]
            a = np.abs(blk).max()
            assert set(qb[np.abs(blk) == a] & 0x7F) == {0x7E}
    x = random_bits((300, 256), seed=4)
    qt, st = oracle.quantize_transpose(x)
    xf = bits_to_f32(x)
    for c in range(256):
        for rb in range(3):
            col = xf[rb * 128:min((rb + 1) * 128, 300), c]
            a = np.abs(col).max()
            seg = qt[c, rb * 128: rb * 128 + col.size]
            assert set(seg[np.abs(col) == a] & 0x7F) == {0x7E}


@pytest.mark.parametrize("E", [-100, -20, 0, 5, 60])
def test_power_of_two_round_trip(oracle_lib, E):
    rng = np.random.default_rng(E & 0xFFFF)
    d = rng.integers(0, 16, size=128)
    d[rng.integers(0, 128)] = 0  # make sure the maximum 2^E is present
    sign = np.where(rng.random(128) < 0.5, -1.0, 1.0)
    x = (sign * np.ldexp(1.0, E - d)).astype(np.float32)
    q, s = oracle.quantize_act(bf16_bits(x[None, :]))
    vals = q[0].view(ml_dtypes.float8_e4m3fn).astype(np.float64)
    assert np.array_equal(vals, sign * 7.0 * np.ldexp(1.0, 6 - d))
    sd = float(s[0, 0])
    # FP64 dequantisation is x up to the scale's own rounding (2^-24 relative)
    assert np.all(np.abs(vals * sd - x) <= 2.0 ** -23 * np.abs(x))
    # the tile maximum comes back exactly through a binary32 product
    assert np.float32(np.float32(448.0) * np.float32(sd)) == np.float32(2.0 ** E)


def test_scale_invariance_under_powers_of_two(oracle_lib):
    x = random_bits((16, 512), seed=5)
    xf = bits_to_f32(x)
    q0, s0 = oracle.quantize_act(x)
    qt0, st0 = oracle.quantize_transpose(x)
    for k in (-7, 3, 20):
        xk = bf16_bits(xf * np.float32(2.0 ** k))  # exact: a power of two
        q1, s1 = oracle.quantize_act(xk)
        assert np.array_equal(q0, q1)
        assert np.array_equal(s1, (s0 * np.float32(2.0 ** k)).astype(np.float32))
        qt1, st1 = oracle.quantize_transpose(xk)
        assert np.array_equal(qt0, qt1)
        assert np.array_equal(st1, (st0 * np.float32(2.0 ** k)).astype(np.float32))
    w = random_bits((128, 256), seed=6, std=0.02)
    qw0, sw0 = oracle.quantize_weight(w)
    qw1, sw1 = oracle.quantize_weight(bf16_bits(bits_to_f32(w) * np.float32(2.0 ** -5)))
    assert np.array_equal(qw0, qw1) and np.array_equal(sw1, sw0 * np.float32(2.0 ** -5))


def test_all_zero_tiles(oracle_lib):
    x = np.zeros((4, 256), dtype=np.float32)
    x[1, :128] = -0.0
    x[2, 130] = 1.0  # second chunk of row 2 is non-zero
    xb = bf16_bits(x)
    q, s = oracle.quantize_act(xb)
    assert s[0, 0] == 0 and s[0, 1] == 0 and s[0, 2] == 0 and s[1, 2] == np.float32(1.0) / np.float32(448.0)
    assert (q[1, :128] == 0x80).all() and (q[0] == 0).all()
    assert q[2, 130] == 0x7E
    qt, st = oracle.quantize_transpose(xb)
    assert (st[0, :] == np.array([0] * 130 + [np.float32(1.0) / np.float32(448.0)] + [0] * 125,
                                 dtype=np.float32)).all()
    assert (qt[:128, 1] == 0x80).all()
    w = np.zeros((128, 128), dtype=np.float32)
    qw, sw = oracle.quantize_weight(bf16_bits(w))
    assert sw[0, 0] == 0 and (qw == 0).all()


def test_codes_within_half_a_step_of_the_quotient(oracle_lib):
    rng = np.random.default_rng(8)
    x = bf16_bits(rng.standard_t(2, size=(32, 640)).astype(np.float32))
    for vals, codes, s in _tiles_act(x):
        if s == 0:
            continue
        t = vals.astype(np.float64) / np.float64(s)
        v = codes.view(ml_dtypes.float8_e4m3fn).astype(np.float64)
        # E4M3 spacing at |t|: 2^(floor(log2|t|) - 3) for |t| >= 2^-6, else 2^-9
        at = np.maximum(np.abs(t), 2.0 ** -6)
        step = np.ldexp(1.0, np.floor(np.log2(at)).astype(int) - 3)
        # half a step, plus the binary32 rounding of the quotient (relative 2^-24)
        assert np.all(np.abs(v - t) <= step / 2 + np.abs(t) * 2.0 ** -23)


@pytest.mark.parametrize("R", [1, 127, 128, 300])
def test_transposed_tiles_are_activation_tiles_of_the_transpose(oracle_lib, R):
    x = random_bits((R, 256), seed=R)
    qt, st = oracle.quantize_transpose(x)
    R128 = (R + 127) // 128 * 128
    assert qt.shape == (256, R128) and st.shape == (R128 // 128, 256)
    qa, sa = oracle.quantize_act(np.ascontiguousarray(x.T))  # chunks along R, last may be partial
    assert np.array_equal(qt[:, :R], qa)
    assert (qt[:, R:] == 0).all()
    assert np.array_equal(st, sa)


def test_weight_block_scale_is_largest_row_scale(oracle_lib):
    w = random_bits((256, 384), seed=9, std=0.02)
    qw, sw, qt = oracle.quantize_weight(w, transposed=True)
    _, sa = oracle.quantize_act(w)  # [K/128][N]: one 1x128 scale per row and chunk
    for bi in range(2):
        for bj in range(3):
            assert sw[bi, bj] == sa[bj, bi * 128:(bi + 1) * 128].max()
    assert np.array_equal(qt, qw.T)


def test_ragged_last_chunk_uses_valid_elements_only(oracle_lib):
    x = random_bits((3, 200), seed=10)
    q, s = oracle.quantize_act(x)
    xf = bits_to_f32(x)
    for r in range(3):
        a = np.abs(xf[r, 128:200]).max()
        assert s[1, r] == np.float32(a) / np.float32(448.0)
