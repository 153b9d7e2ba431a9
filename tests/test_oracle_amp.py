"""Pins of the mixed-precision oracle helpers ("DLRM For PyTorch", §Mixed
precision training): one binary16 rounding of exact values."""

import numpy as np
import pytest

import oracle


@pytest.fixture(scope="module", autouse=True)
def _built():
    oracle.build()


def test_round_f16_matches_numpy_and_the_scalar_converter():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(20000) * 10.0 ** rng.integers(-9, 6, 20000),
                        [0.0, -0.0, 65504.0, 65520.0, -65520.0, 1e9, 2.0**-25, 2.0**-24, 3 * 2.0**-25]])
    # exact midpoints between neighbouring halves (ties go to even)
    h = rng.integers(0, 0x7BFF, 2000).astype(np.uint16).view(np.float16)
    lo, hi = h.astype(np.float64), np.nextafter(h, np.float16(np.inf)).astype(np.float64)
    x = np.concatenate([x, (lo + hi) / 2])
    got = oracle.round_f16(x)
    with np.errstate(over="ignore"):
        want = x.astype(np.float16)
    assert np.array_equal(got.view(np.uint16), want.view(np.uint16))
    for v in x[:200]:
        assert got[list(x).index(v)].view(np.uint16) == oracle.lib().oracle_f64_to_f16(float(v))


def test_pooling_to_fp16_rounds_once():
    # bag {r0, r1}: 1 + 2^-11 + 2^-12 is exact in fp32 but rounds to 1 + 2^-10 in fp16 only if
    # summed exactly (rounding 1 + 2^-11 first would give 1, a tie to even)
    tables = np.array([[1.0], [2.0**-11 + 2.0**-12]], np.float32)
    pooled, st = oracle.emb_fwd_f16out(tables, np.array([0, 2]), 1, 1, 1, np.array([0, 1], np.int32),
                                       np.array([0, 2], np.int32))
    assert st == 0 and pooled.dtype == np.float16 and float(pooled[0, 0, 0]) == 1 + 2.0**-10


def test_backward_f16_is_the_rounded_exact_backward():
    rng = np.random.default_rng(1)
    B, F, D, P = 3, 4, 8, 24
    dense = rng.standard_normal((B, D)).astype(np.float16)
    pooled = rng.standard_normal((B, F, D)).astype(np.float16)
    g = (rng.standard_normal((B, P)) * 1024).astype(np.float16)      # loss-scaled upstream gradient
    gd, gp = oracle.interact_bwd_f16(g, dense, pooled)
    # exact reference by brute force: M from the triangle, dZ = M Z
    W = D + F * (F + 1) // 2
    for b in range(B):
        Z = np.vstack([dense[b], pooled[b]]).astype(np.float64)
        M = np.zeros((F + 1, F + 1))
        k = D
        for i in range(1, F + 1):
            for j in range(i):
                M[i, j] = M[j, i] = float(g[b, k])
                k += 1
        assert k == W
        dZ = M @ Z
        assert np.array_equal(gd[b], (g[b, :D].astype(np.float64) + dZ[0]).astype(np.float16))
        assert np.array_equal(gp[b], dZ[1:].astype(np.float16))
