"""Pins for the oracle's bf16 rounding (CPU only).

Three independent checks of ``oracle.round_bf16``:
  1. hand-derived cases (tests/golden/bf16_rounding_cases.json);
  2. brute force over the whole bf16 grid with exact rational arithmetic: the
     neighbours of x are found among all finite bf16 values and picked per mode;
  3. for binary32 inputs, the carry-based integer rule on the low 16 bits
     (written here, not taken from any other module), over every high half and a
     set of low halves that includes every tie and near-tie.
"""
import bisect
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

from oracle import round_bf16, ulp_distance

HERE = os.path.dirname(os.path.abspath(__file__))
MODES = ("rtne", "rtna", "rtz")


def _cases():
    with open(os.path.join(HERE, "golden", "bf16_rounding_cases.json")) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("case", _cases(), ids=lambda c: c["x"])
def test_hand_cases(case):
    x = eval(case["x"], {"float": float})  # fixture expressions are plain arithmetic
    for mode in MODES:
        got = int(round_bf16(np.array([x]), mode)[0])
        assert got == int(case[mode], 16), (case["x"], mode, hex(got), case["why"])


# --- 2. exact brute force over the bf16 grid ---------------------------------

def _bf16_value(bits):
    sign = -1 if bits & 0x8000 else 1
    e = (bits >> 7) & 0xFF
    f = bits & 0x7F
    if e == 0:
        return sign * Fraction(f, 2 ** 133)
    return sign * Fraction(128 + f, 128) * Fraction(2) ** (e - 127)


_POS = [(_bf16_value(b), b) for b in range(0x0000, 0x7F80)]  # 0 .. largest finite
_POS_VALS = [v for v, _ in _POS]
_TWO128 = Fraction(2) ** 128


def _exact_round(x: float, mode: str) -> int:
    if math.isnan(x):
        return 0x7FC0
    sign = 0x8000 if math.copysign(1.0, x) < 0 else 0
    if math.isinf(x):
        return sign | 0x7F80
    a = abs(Fraction(x))
    i = bisect.bisect_right(_POS_VALS, a) - 1  # largest grid value <= a
    lo_v, lo_b = _POS[i]
    if lo_v == a:
        return sign | lo_b
    if i + 1 < len(_POS):
        hi_v, hi_b = _POS[i + 1]
    else:  # above the largest finite: the next step is 2^128 (even significand)
        hi_v, hi_b = _TWO128, 0x7F80
    if mode == "rtz":
        return sign | lo_b
    dlo, dhi = a - lo_v, hi_v - a
    if dlo < dhi:
        pick = lo_b
    elif dhi < dlo:
        pick = hi_b
    elif mode == "rtna":
        pick = hi_b
    else:  # tie, to even significand
        pick = lo_b if (lo_b & 1) == 0 else hi_b
    if pick == 0x7F80 and mode == "rtz":
        pick = 0x7F7F
    return sign | pick


def _sample_doubles(n, seed=7):
    rng = np.random.default_rng(seed)
    e = rng.integers(-140, 130, n)
    m = rng.uniform(1.0, 2.0, n)
    x = np.ldexp(m, e) * np.where(rng.random(n) < 0.5, -1.0, 1.0)
    # exact ties and near-ties of the grid at random binades
    b = rng.integers(0, 0x7F7F, n // 4).astype(np.uint32)
    base = (b << 16).view(np.float32).astype(np.float64)
    step = np.ldexp(1.0, np.frexp(base)[1] - 9)
    ties = base + step
    near = ties + np.where(rng.random(n // 4) < 0.5, -1, 1) * step * 2.0 ** -20
    return np.concatenate([x, ties, near, [0.0, -0.0, 2.0 ** -1074, 3.4e38, 3.5e38]])


def test_exact_bruteforce_sample():
    xs = _sample_doubles(4000)
    for mode in MODES:
        got = round_bf16(xs, mode)
        want = np.array([_exact_round(float(x), mode) for x in xs], dtype=np.uint16)
        bad = np.nonzero(got != want)[0]
        assert bad.size == 0, [(float(xs[i]), mode, hex(got[i]), hex(want[i])) for i in bad[:5]]


# --- 3. binary32 inputs: carry rule on the low half ----------------------------

def _carry_rule(u32: np.ndarray, mode: str) -> np.ndarray:
    u = u32.astype(np.uint64)
    hi = u >> np.uint64(16)
    low = u & np.uint64(0xFFFF)
    if mode == "rtz":
        r = hi
    elif mode == "rtna":
        r = hi + (low >= 0x8000)
    else:
        r = hi + ((low > 0x8000) | ((low == 0x8000) & ((hi & np.uint64(1)) == 1)))
    exp_all = (u32 & np.uint32(0x7F800000)) == np.uint32(0x7F800000)
    nan = exp_all & ((u32 & np.uint32(0x007FFFFF)) != 0)
    r = r.astype(np.uint32)
    if mode == "rtz":
        pass  # truncation never carries into the Inf pattern
    r = np.where(nan, np.uint32(0x7FC0), r)
    return r.astype(np.uint16)


def test_binary32_carry_rule():
    hi = np.arange(0, 1 << 16, dtype=np.uint32) << np.uint32(16)
    lows = np.array([0x0000, 0x0001, 0x3FFF, 0x7FFF, 0x8000, 0x8001, 0xC000, 0xFFFF],
                    dtype=np.uint32)
    u = (hi[:, None] | lows[None, :]).reshape(-1)
    x = u.view(np.float32).astype(np.float64)
    for mode in MODES:
        got = round_bf16(x, mode)
        want = _carry_rule(u, mode)
        bad = np.nonzero(got != want)[0]
        assert bad.size == 0, [(hex(int(u[i])), mode, hex(int(got[i])), hex(int(want[i])))
                               for i in bad[:5]]


def test_ulp_distance():
    a = np.array([0x3F80, 0x3F80, 0x0000, 0x8000, 0x0001, 0x8001, 0x7F7F], dtype=np.uint16)
    b = np.array([0x3F81, 0x3F7F, 0x8000, 0x0001, 0x8001, 0x0001, 0x7F7E], dtype=np.uint16)
    assert ulp_distance(a, b).tolist() == [1, 1, 0, 1, 2, 2, 1]
