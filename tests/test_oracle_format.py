"""Pins for the oracle's number formats: bf16 widening and OCP E4M3FN encode/decode.

The oracle writes these from the format definitions; here they are checked
against facts fixed outside the oracle:
  * two independent library casts (ml_dtypes and torch, both OCP E4M3FN with
    round-to-nearest-even), exhaustively over every binary32 value in range;
  * a brute-force nearest-grid-point search over all 254 finite codes;
  * hand-derived landmark values (tests/golden/e4m3_landmarks.txt).
"""
import os

import ml_dtypes
import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_bf16_widening_every_pattern(oracle_lib):
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(ml_dtypes.bfloat16).astype(np.float32)
    got = np.array([oracle.bf16_to_f32(b) for b in bits], dtype=np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_e4m3_decode_every_code_matches_two_libraries(oracle_lib):
    codes = np.arange(256, dtype=np.uint8)
    mine = oracle.e4m3_values(codes)
    ml = codes.view(ml_dtypes.float8_e4m3fn).astype(np.float64)
    th = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for ref in (ml, th):
        nan = np.isnan(ref)
        assert nan.sum() == 2 and set(codes[nan]) == {0x7F, 0xFF}
        assert np.array_equal(np.isnan(mine), nan)
        assert np.array_equal(mine[~nan], ref[~nan])
    assert mine[0x7E] == 448.0 and mine[0xFE] == -448.0
    assert mine[0x01] == 2.0 ** -9 and mine[0x08] == 2.0 ** -6


def test_e4m3_integer_units_agree_with_values(oracle_lib):
    for c in range(256):
        if (c & 0x7F) == 0x7F:
            continue
        assert oracle.e4m3_units(c) * 2.0 ** -9 == oracle.e4m3_value(c)


def _exhaustive_range(sign_bit: int, chunk: int = 1 << 26):
    # every binary32 magnitude from +0 up to and including 464 (the last value
    # whose nearest-even rounding is still the finite 448)
    hi = int(np.array([464.0], dtype=np.float32).view(np.uint32)[0])
    for start in range(0, hi + 1, chunk):
        stop = min(start + chunk, hi + 1)
        u = np.arange(start, stop, dtype=np.uint32) | np.uint32(sign_bit)
        yield u.view(np.float32)


@pytest.mark.slow
@pytest.mark.parametrize("sign_bit", [0, 0x80000000])
def test_e4m3_encode_exhaustive_against_two_libraries(oracle_lib, sign_bit):
    n = 0
    for t in _exhaustive_range(sign_bit):
        mine = oracle.e4m3_encode_array(t)
        ml = t.astype(ml_dtypes.float8_e4m3fn).view(np.uint8)
        assert np.array_equal(mine, ml), "mismatch vs ml_dtypes"
        th = torch.from_numpy(t).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        assert np.array_equal(mine, th), "mismatch vs torch"
        n += t.size
    assert n == 0x43E80000 + 1


def test_e4m3_saturates_above_448(oracle_lib):
    rng = np.random.default_rng(7)
    big = np.concatenate([
        np.array([448.0001, 460.0, 464.0, 464.0001, 479.9, 480.0, 1e4, 3.0e38], dtype=np.float32),
        np.float32(2.0) ** rng.uniform(8.81, 127.9, 4096).astype(np.float32),
        np.array([np.inf], dtype=np.float32),
    ])
    assert (oracle.e4m3_encode_array(big) == 0x7E).all()
    assert (oracle.e4m3_encode_array(-big) == 0xFE).all()


def test_e4m3_signed_zero_kept(oracle_lib):
    t = np.array([0.0, -0.0, 2.0 ** -11, -(2.0 ** -11), 2.0 ** -10, -(2.0 ** -10), 1e-30, -1e-30],
                 dtype=np.float32)
    assert list(oracle.e4m3_encode_array(t)) == [0x00, 0x80, 0x00, 0x80, 0x00, 0x80, 0x00, 0x80]


def test_e4m3_encode_is_nearest_grid_point_ties_to_even(oracle_lib):
    """Brute force: among all finite codes pick the nearest value; on a tie the even mantissa."""
    finite = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    vals = finite.view(ml_dtypes.float8_e4m3fn).astype(np.float64)
    rng = np.random.default_rng(11)
    mags = np.concatenate([
        rng.uniform(0, 448, 3000),
        np.float64(2.0) ** rng.uniform(-14, 8.8, 3000),
        # exact midpoints between neighbouring grid values (tie cases)
        (np.unique(np.abs(vals))[1:] + np.unique(np.abs(vals))[:-1]) / 2,
    ])
    t = (mags * np.where(rng.random(mags.size) < 0.5, -1, 1)).astype(np.float32)
    got = oracle.e4m3_encode_array(t)
    for ti, gi in zip(t.astype(np.float64), got):
        d = np.abs(vals - ti)
        best = finite[d == d.min()]
        if best.size > 1:
            best = best[(best & 1) == 0]  # ties: even mantissa
            # two zeros (+0/-0) tie exactly; keep the one with t's sign
            if best.size > 1:
                best = best[(best & 0x80) == (0x80 if np.signbit(ti) else 0)]
        assert best.size == 1
        assert gi == best[0], (ti, hex(gi), hex(best[0]))


def test_e4m3_landmarks_from_the_format_definition(oracle_lib):
    """Hand-derived values, see tests/golden/e4m3_landmarks.txt for each derivation."""
    path = os.path.join(GOLDEN, "e4m3_landmarks.txt")
    n = 0
    with open(path) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            t_str, code_str = line.split()
            t = np.float32(float.fromhex(t_str) if "p" in t_str else float(t_str))
            assert oracle.e4m3_encode(t) == int(code_str, 16), line
            n += 1
    assert n >= 20
