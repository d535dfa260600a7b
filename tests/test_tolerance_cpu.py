"""The bf16 output check of the GPU parity tests, checked on the CPU.

A stored bf16 value passes when some real within the tolerance of the fp64
oracle rounds (to nearest, ties to even) to it.  Here that rule is compared with
a brute-force scan of the bf16 numbers around random oracle values: the values
it accepts must be exactly those between round_bf16(oracle - tol) and
round_bf16(oracle + tol).
"""
import numpy as np

from gpu_common import OUT_TOL, _bf16_neighbours, bf16_store_excess, out_err_beyond_bf16_store
from oracle.moe import round_to_bf16


with np.errstate(invalid="ignore"):
    _ALL = (np.arange(0, 1 << 16, dtype=np.uint32) << 16).view(np.float32).astype(np.float64)
_ALL = np.unique(_ALL[np.isfinite(_ALL)])          # every finite bf16 value, sorted (-0 == +0)


def _bf16_grid(lo, hi):
    """Every bf16 value in [lo, hi] (float64)."""
    return _ALL[np.searchsorted(_ALL, lo, "left"):np.searchsorted(_ALL, hi, "right")]


def test_neighbours_are_adjacent_bf16_values():
    rng = np.random.default_rng(1)
    for x in np.concatenate([rng.standard_normal(200) * 4, [0.0, 1.0, 2.0, -2.0, 0.5, 1e-39]]):
        g = float(round_to_bf16(x))
        down, up = _bf16_neighbours(np.array([g]))
        grid = _bf16_grid(g - 1.0, g + 1.0) if g != 0 else _bf16_grid(-1e-30, 1e-30)
        i = int(np.searchsorted(grid, g))
        assert grid[i] == g
        assert down[0] == grid[i - 1] and up[0] == grid[i + 1], (x, g, down, up)


def test_interval_rule_equals_monotone_rounding_bounds():
    rng = np.random.default_rng(2)
    ys = np.concatenate([rng.standard_normal(300) * 3, rng.uniform(1.9, 8.5, 100),
                         rng.uniform(-0.05, 0.05, 50), [2.0, 4.0, -4.0, 0.0]])
    for tol in (OUT_TOL, 1e-3, 0.02):
        for y in ys:
            lo, hi = float(round_to_bf16(y - tol)), float(round_to_bf16(y + tol))
            cand = _bf16_grid(y - 4 * tol - 0.1, y + 4 * tol + 0.1)
            exc = bf16_store_excess(cand, np.full(cand.shape, y))
            ok = exc <= tol
            want = (cand >= lo) & (cand <= hi)
            # disagreement only where a candidate's rounding interval touches the
            # tolerance band in a single point (a tie that the rounding breaks to even)
            assert np.all(np.abs(exc[ok != want] - tol) < 1e-15), (y, tol, cand[ok != want])


def test_rule_rejects_what_arithmetic_cannot_explain():
    # 3.0 is a bf16 value (step 2^-6 in [2, 4)) whose rounding interval is [3 - 2^-7, 3 + 2^-7]
    assert out_err_beyond_bf16_store(np.array([3.0]), np.array([3.0 + 2 ** -7 + 0.0099])) <= OUT_TOL
    assert out_err_beyond_bf16_store(np.array([3.0]), np.array([3.0 + 2 ** -7 + 0.0101])) > OUT_TOL
    # a value stored one step away across a rounding midpoint is accepted when the
    # oracle is within the tolerance of that midpoint
    assert out_err_beyond_bf16_store(np.array([3.015625]), np.array([3.0077])) <= OUT_TOL
    # a non-finite stored value always fails
    assert np.isnan(out_err_beyond_bf16_store(np.array([np.nan]), np.array([0.0])))
