"""The seeded input generators: determinism and their published definitions."""

import math

import numpy as np
import pytest

from dlrm_embeddings_dot_gb300 import inputs

MASK = (1 << 64) - 1


def _splitmix64_int(seed: int, i: int) -> int:
    """splitmix64 with Python integers (Steele, Lea & Flood, OOPSLA 2014)."""
    z = (seed + (i + 1) * 0x9E3779B97F4A7C15) & MASK
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK
    return z ^ (z >> 31)


def test_splitmix64_matches_integer_definition():
    for seed in (0, 1, 1234567, 2**63 + 5):
        idx = np.array([0, 1, 2, 3, 1000, 2**40 + 7], dtype=np.uint64)
        got = inputs.splitmix64(seed, idx)
        for i, g in zip(idx.tolist(), got.tolist()):
            assert g == _splitmix64_int(seed, i)


def test_uniform_values_range_and_moments():
    v = inputs.uniform_values(3, np.arange(200000, dtype=np.uint64), 0.05)
    assert v.dtype == np.float32
    assert v.min() >= -0.05 and v.max() < 0.05
    assert abs(v.mean()) < 1e-3
    assert v.std() == pytest.approx(0.1 / math.sqrt(12), rel=1e-2)


def test_uniform_values_are_single_fp32_products():
    """x * c with x a 24-bit integer and c = fp32(a / 2^23): one rounding, so the
    exact product in float64 rounds to the same fp32 value."""
    e = np.arange(5000, dtype=np.uint64)
    z = inputs.splitmix64(11, e)
    x = (z >> np.uint64(40)).astype(np.int64) - (1 << 23)
    c = np.float32(0.05 / 8388608.0)
    exact = x.astype(np.float64) * np.float64(c)      # exact: 24-bit x 24-bit < 53 bits
    assert np.array_equal(inputs.uniform_values(11, e, 0.05), exact.astype(np.float32))


def test_table_rows_fp16_is_rounded_fp32():
    r32 = inputs.table_rows(9, np.array([0, 5, 77]), 16, inputs.F32)
    r16 = inputs.table_rows(9, np.array([0, 5, 77]), 16, inputs.F16)
    assert np.array_equal(r32.astype(np.float16), r16)


@pytest.mark.parametrize("alpha", [1.05, 1.2, 0.8])
@pytest.mark.parametrize("n", [1, 2, 20])
def test_bounded_zipf_pmf(alpha, n):
    rng = np.random.default_rng(0)
    k = inputs.BoundedZipf(n, alpha).sample(rng, 200000)
    assert k.min() >= 1 and k.max() <= n
    p = np.arange(1, n + 1, dtype=np.float64) ** -alpha
    p /= p.sum()
    freq = np.bincount(k, minlength=n + 1)[1:] / k.size
    # 200k draws: binomial standard error <= 0.0012
    assert np.abs(freq - p).max() < 0.006


def test_zipf_rows_is_a_permutation_of_ranks():
    rng = np.random.default_rng(1)
    rows = inputs.zipf_rows(rng, 97, 1.2, 50000)
    assert rows.min() >= 0 and rows.max() < 97
    # the most frequent row takes rank 1's share
    top = np.bincount(rows).max() / rows.size
    p1 = 1.0 / (np.arange(1, 98) ** -1.2).sum()
    assert top == pytest.approx(p1, abs=0.01)


def test_workloads_are_deterministic_and_well_formed():
    a = inputs.tiny_slice(seed=0)
    b = inputs.tiny_slice(seed=0)
    assert np.array_equal(a.indices, b.indices) and np.array_equal(a.dense, b.dense)
    assert a.B == 256 and a.F == 3 and a.D == 16 and a.out_cols == 22
    assert a.dense.shape == (256, 16) and (a.dense >= 0).all()
    assert np.array_equal(a.offsets, np.arange(3 * 256 + 1))
    w = inputs.dlrm_default(B=512, train=True)
    assert w.F == 26 and w.D == 128 and w.out_cols == 480
    assert (w.rows >= 10).all() and (w.rows <= 4_000_000).all()
    assert w.grad_out.shape == (512, 480)
    for t in range(w.F):
        seg = w.indices[w.offsets[t * w.B]:w.offsets[(t + 1) * w.B]]
        assert seg.min() >= 0 and seg.max() < w.rows[t]
    m = inputs.multi_hot(B=64, rows_per_table=1000)
    counts = np.diff(m.offsets)
    assert counts.min() >= 1 and counts.max() <= 100
    assert m.offsets[-1] == m.nnz


def test_fp16_dense_fits():
    w = inputs.dlrm_default(B=256, dtype=inputs.F16)
    assert np.array_equal(w.dense, w.dense.astype(np.float16).astype(np.float32))
