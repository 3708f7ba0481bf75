"""Pins of the oracle's per-element quotient: code = e4m3(fl32(x / s)), s = fl32(amax / 448).

The blockwise FP8 of the Puro-2B recipe follows DeepSeek-V3's fine-grained block
quantisation (Puro-2B article on en.roboind.com, section on FP8 and the RTX
5090); the plain reading of "scale = amax / 448" is an IEEE binary32 division
for the scale and another for each element, then rounding to E4M3. Two
plausible slips give other codes on a small share of inputs: multiplying by a
rounded reciprocal, fl32(x * fl32(1/s)), and rounding the exact quotient only
once. tests/golden/quotient_cases.txt lists BF16 (amax, x) pairs on which each
slip changes the code; here every expected code is recomputed with exact
rational arithmetic (tests/golden/exact_e4m3.py, written from the formats'
definitions), and the oracle's three quantisers must reproduce it. Either slip
in the oracle fails these tests.
"""
import os
import sys

import numpy as np
import pytest

import oracle
import workloads as wl

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.join(HERE, "golden"))

import exact_e4m3 as ex  # noqa: E402

TILE = 128


def _cases():
    out = []
    with open(os.path.join(HERE, "golden", "quotient_cases.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            kind, a, x = line.split()
            out.append((kind, int(a, 16), int(x, 16)))
    return out


CASES = _cases()


def test_cases_discriminate_both_slips():
    kinds = {k for k, _, _ in CASES}
    assert kinds == {"reciprocal", "single"} and len(CASES) >= 40
    for kind, ab, xb in CASES:
        A, X = ex.bf16_value(ab), ex.bf16_value(xb)
        assert abs(X) <= A
        want = ex.code_by_definition(A, X)
        other = ex.code_by_reciprocal(A, X) if kind == "reciprocal" else ex.code_by_single_rounding(A, X)
        assert other != want, (kind, hex(ab), hex(xb))


def _expected(ab, xb):
    return ex.code_by_definition(ex.bf16_value(ab), ex.bf16_value(xb))


def test_activation_quantiser_on_golden_pairs():
    n = len(CASES)
    x = np.zeros((n, TILE), np.uint16)
    for i, (_, ab, xb) in enumerate(CASES):
        x[i, 0], x[i, 1] = ab, xb
    q, s = oracle.quantize_act(x)
    for i, (_, ab, xb) in enumerate(CASES):
        assert q[i, 1] == _expected(ab, xb), (hex(ab), hex(xb))
        assert q[i, 0] == 0x7E
        assert ex.Fraction(float(s[0, i])) == ex.tile_scale(ex.bf16_value(ab))


def test_transposed_quantiser_on_golden_pairs():
    n = len(CASES)
    x = np.zeros((TILE, n), np.uint16)  # tiles run down the columns
    for j, (_, ab, xb) in enumerate(CASES):
        x[0, j], x[1, j] = ab, xb
    qt, st = oracle.quantize_transpose(x)
    for j, (_, ab, xb) in enumerate(CASES):
        assert qt[j, 1] == _expected(ab, xb), (hex(ab), hex(xb))


def test_weight_quantiser_on_golden_pairs():
    for _, ab, xb in CASES[::4]:
        w = np.zeros((TILE, TILE), np.uint16)
        w[0, 0], w[5, 77] = ab, xb
        q, s = oracle.quantize_weight(w)
        assert q[5, 77] == _expected(ab, xb), (hex(ab), hex(xb))


@pytest.mark.parametrize("dist", ["student_t3", "normal"])
def test_random_tiles_match_exact_arithmetic_elementwise(dist):
    """Brute force: every code of 24 random 1x128 tiles equals the exact-arithmetic definition."""
    lin = wl.Linear("q", 24, TILE, TILE, dist, 5)
    x = wl.make_x(lin)
    q, s = oracle.quantize_act(x)
    for r in range(x.shape[0]):
        vals = [ex.bf16_value(int(b)) for b in x[r]]
        amax = max(abs(v) for v in vals)
        assert ex.Fraction(float(s[0, r])) == ex.tile_scale(amax)
        for j, v in enumerate(vals):
            neg0 = v == 0 and bool(x[r, j] & 0x8000)
            assert q[r, j] == ex.code_by_definition(amax, v, neg0), (r, j)
