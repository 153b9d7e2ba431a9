"""Helpers shared by the tests: golden-file reader and tolerance checks."""

import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load_golden(name: str) -> dict:
    """Read ``key: numbers...`` lines of a golden fixture (``#`` starts a comment)."""
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, vals = line.split(":", 1)
            nums = [float(v) for v in vals.split()]
            out[key.strip()] = nums[0] if len(nums) == 1 else np.array(nums)
    return out


def assert_within_abs_sum(got, ref, abs_sum, rtol, what=""):
    """|got - ref| <= rtol * (sum of absolute summands) + 1e-30, elementwise.

    ``abs_sum`` is the sum of the absolute values of the terms that make up
    each reference element, so cancellation in a dot product or a sum does not
    turn rounding noise into a spurious failure.
    """
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    bound = rtol * np.asarray(abs_sum, dtype=np.float64) + 1e-30
    err = np.abs(got - ref)
    bad = err > bound
    if bad.any():
        i = np.flatnonzero(bad.ravel())[0]
        raise AssertionError(
            f"{what}: {bad.sum()} of {bad.size} elements outside tolerance; first at flat index "
            f"{i}: got {got.ravel()[i]!r}, ref {ref.ravel()[i]!r}, bound {bound.ravel()[i]!r}")
    return float((err / np.maximum(bound, 1e-300)).max()) if err.size else 0.0
