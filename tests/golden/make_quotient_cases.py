"""Writes tests/golden/quotient_cases.txt: (amax, x) BF16 input pairs on which the
quantiser's reading of "scale = amax / 448" is decided.

The definition is code = e4m3(fl32(x / s)) with s = fl32(amax / 448): an IEEE
binary32 division, then a second rounding to E4M3 (the readings of the
DeepSeek-V3-style block quantisation that the Puro-2B recipe follows). Two
plausible mistakes give other codes on a small share of inputs:
  reciprocal  e4m3(fl32(x * fl32(1 / s)))  (a multiplication by a rounded reciprocal)
  single      e4m3(x / s)                  (the exact quotient rounded once)
This script searches seeded random BF16 pairs with numpy's binary32 arithmetic
for pairs on which a mistake changes the code, confirms each with exact
rational arithmetic (exact_e4m3.py), and writes the inputs only. The tests
recompute every expected code with exact arithmetic; no stored value is an
output of the code under test.

Usage: python tests/golden/make_quotient_cases.py
"""
from __future__ import annotations

import os
import sys

import ml_dtypes
import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, HERE)

import exact_e4m3 as ex  # noqa: E402

OUT = os.path.join(HERE, "quotient_cases.txt")
PER_KIND = 24


def bf16(a):
    return np.asarray(a, dtype=np.float32).astype(ml_dtypes.bfloat16)


def bits(a):
    return np.asarray(a).view(np.uint16)


def search(kind: str, rng, want: int):
    found = []
    seen = set()
    while len(found) < want:
        n = 1 << 20
        amax = bf16(np.abs(rng.standard_t(3, n)) * np.float32(2.0) ** rng.integers(-20, 20, n).astype(np.float32))
        amax = amax[amax.astype(np.float32) > 0]
        s = amax.astype(np.float32) / np.float32(448.0)
        if kind == "reciprocal":
            x = bf16(amax.astype(np.float32) * rng.uniform(-1, 1, amax.size).astype(np.float32))
            xf = x.astype(np.float32)
            keep = np.abs(xf) <= amax.astype(np.float32)
            t_div = xf / s
            t_rcp = xf * (np.float32(1.0) / s)
            c_div = t_div.astype(ml_dtypes.float8_e4m3fn).view(np.uint8)
            c_rcp = t_rcp.astype(ml_dtypes.float8_e4m3fn).view(np.uint8)
            cand = np.nonzero(keep & (c_div != c_rcp) & (np.abs(t_div) <= 448))[0]
        else:
            # aim x / s at a midpoint of the E4M3 grid, so that the binary32 quotient can land on it
            e = rng.integers(-6, 8, amax.size)
            mid = (np.float32(8.5) + rng.integers(0, 8, amax.size).astype(np.float32)) / np.float32(8.0) * \
                np.float32(2.0) ** e.astype(np.float32)
            x = bf16(mid * s * np.where(rng.random(amax.size) < 0.5, -1, 1).astype(np.float32))
            xf = x.astype(np.float32)
            keep = np.abs(xf) <= amax.astype(np.float32)
            t = xf / s
            scaled = np.abs(t.astype(np.float64)) * 16.0 / np.float64(2.0) ** np.floor(np.log2(np.abs(t) + 1e-30))
            on_mid = np.abs(scaled - np.round(scaled)) == 0
            cand = np.nonzero(keep & on_mid & (np.round(scaled) % 2 == 1) & (np.abs(t) < 448))[0]
        for i in cand:
            ab, xb = int(bits(amax[i])), int(bits(x[i]))
            if (ab, xb) in seen:
                continue
            A, X = ex.bf16_value(ab), ex.bf16_value(xb)
            want_code = ex.code_by_definition(A, X)
            other = ex.code_by_reciprocal(A, X) if kind == "reciprocal" else ex.code_by_single_rounding(A, X)
            if other != want_code:
                seen.add((ab, xb))
                found.append((ab, xb))
                if len(found) == want:
                    break
    return found


def main():
    rng = np.random.default_rng(20260101)
    rows = [("reciprocal", p) for p in search("reciprocal", rng, PER_KIND)]
    rows += [("single", p) for p in search("single", rng, PER_KIND)]
    with open(OUT, "w") as f:
        f.write("# (amax, x) BF16 bit patterns on which the quantiser's quotient reading is decided.\n")
        f.write("# Definition: code = e4m3_rn_satfinite(fl32(x / s)), s = fl32(amax / 448): the\n")
        f.write("# DeepSeek-V3-style fine-grained block quantisation that the Puro-2B recipe follows\n")
        f.write("# (Puro-2B article on en.roboind.com, section on FP8 and the RTX 5090), read plainly.\n")
        f.write("# kind 'reciprocal': e4m3(fl32(x * fl32(1/s))) gives another code; kind 'single':\n")
        f.write("# e4m3(x / s), one rounding, gives another code (fl32(x/s) is an E4M3 midpoint).\n")
        f.write("# Inputs only; written by tests/golden/make_quotient_cases.py; expected codes are\n")
        f.write("# recomputed by the tests with exact rational arithmetic (exact_e4m3.py).\n")
        f.write("# kind amax_bits x_bits\n")
        for kind, (ab, xb) in rows:
            f.write(f"{kind} 0x{ab:04x} 0x{xb:04x}\n")
    print(f"wrote {len(rows)} cases to {OUT}")


if __name__ == "__main__":
    main()
