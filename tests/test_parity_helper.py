"""The comparison helper itself: correctly rounded values have zero excess error,
and an element two ULPs off is caught."""
import numpy as np

from oracle import round_bf16

from _parity import compare


def test_correct_rounding_has_no_excess_error():
    rng = np.random.default_rng(7)
    exact = rng.uniform(2.0, 4.0, 4096) * rng.choice([-1.0, 1.0], 4096)
    for mode in ("rtne", "rtna", "rtz"):
        st = compare(round_bf16(exact, mode), exact, mode)
        assert st["exact_match"] == 1.0
        assert st["max_excess_err"] <= 0.0
    # RTZ of values in [2, 4) misses by up to one ULP (2^-6), beyond 8e-3.
    assert compare(round_bf16(exact, "rtz"), exact, "rtz")["max_abs_err"] > 8e-3


def test_two_ulp_error_shows_as_excess():
    exact = np.full(16, 3.0 + 2.0 ** -9)
    bits = round_bf16(exact, "rtz")
    bits[3] += 2  # two ULPs (2^-5) too large in magnitude
    st = compare(bits, exact, "rtz")
    assert st["max_ulp"] == 2
    assert abs(st["max_excess_err"] - (2 * 2.0 ** -6 - 2.0 ** -9 - 2.0 ** -9)) < 1e-12


def test_one_ulp_rtz_miss_at_a_grid_point_is_not_excess():
    # Exact value just above 4.0; a kernel value just below 4.0 truncates one full
    # ULP (2^-6) lower. Within 1 ULP, so no excess error although |err| > 8e-3.
    exact = np.full(4, 4.0 + 2.0 ** -20)
    bits = round_bf16(exact, "rtz")
    bits[1] = round_bf16(np.array([4.0 - 2.0 ** -20]), "rtz")[0]
    st = compare(bits, exact, "rtz")
    assert st["max_ulp"] == 1 and st["max_abs_err"] > 8e-3
    assert st["max_excess_err"] == 0.0
