"""Pins for the CPU oracle: checks against facts fixed outside the oracle.

Each check is something the oracle's own code does not restate: hand-worked
examples (``tests/golden``), library routines that reach the same quantity by
another route (``np.add.at``, ``np.einsum``, ``np.tril_indices``, stable
``np.argsort``, numpy's binary16 conversion), closed forms and invariants
(symmetry of the Gram matrix, output width, exactness of central differences
on a quadratic), and special cases (one table, orthonormal vectors, lr = 0).
The model is the one of "DLRM For PyTorch", §Model architecture.
"""

import numpy as np
import pytest

import oracle
from helpers import load_golden

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


# --------------------------------------------------------------------------
# binary16 converter: exhaustive against numpy
# --------------------------------------------------------------------------
def test_f16_to_f64_exhaustive():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.f16_to_f64(b) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    # signed zeros keep their sign
    assert np.signbit(oracle.f16_to_f64(0x8000)) and not np.signbit(oracle.f16_to_f64(0))


def _f64_to_f16_many(xs):
    return np.array([oracle.f64_to_f16(x) for x in xs], dtype=np.uint16)


def test_f64_to_f16_exact_values_and_ties():
    finite = np.arange(0, 0x7C00, dtype=np.uint32).astype(np.uint16)
    vals = finite.view(np.float16).astype(np.float64)
    # exact values map back to themselves, both signs
    assert np.array_equal(_f64_to_f16_many(vals), finite)
    assert np.array_equal(_f64_to_f16_many(-vals), finite | np.uint16(0x8000))
    # midpoints between neighbours (ties -> even) and the doubles right beside them
    mids = (vals[:-1] + vals[1:]) / 2.0
    for xs in (mids, np.nextafter(mids, np.inf), np.nextafter(mids, -np.inf)):
        ref = xs.astype(np.float16).view(np.uint16)
        assert np.array_equal(_f64_to_f16_many(xs), ref)


def test_f64_to_f16_overflow_and_random():
    edge = np.array([65504.0, 65519.99, 65520.0, 1e6, np.inf, -np.inf, 2.0**-25, 2.0**-24 * 1.5,
                     2.0**-26, 5.96e-8, 6.1e-5, -0.0, 0.0])
    ref = edge.astype(np.float16).view(np.uint16)
    assert np.array_equal(_f64_to_f16_many(edge), ref)
    rng = np.random.default_rng(5)
    xs = rng.standard_normal(20000) * np.exp2(rng.integers(-30, 17, size=20000))
    ref = xs.astype(np.float16).view(np.uint16)
    assert np.array_equal(_f64_to_f16_many(xs), ref)
    assert oracle.f64_to_f16(float("nan")) & 0x7C00 == 0x7C00


# --------------------------------------------------------------------------
# embedding lookup with sum pooling
# --------------------------------------------------------------------------
def test_lookup_hand_example():
    g = load_golden("lookup_hand.txt")
    table = g["table"].astype(np.float32).reshape(int(g["rows"]), int(g["D"]))
    pooled, status = oracle.emb_fwd(table, [0, int(g["rows"])], 1, 2, 3,
                                    g["indices"], g["offsets"])
    assert status == 0
    assert np.array_equal(pooled.reshape(-1), g["pooled"].astype(np.float32))


def _random_bags(rng, F, B, rows, max_pool, allow_empty=True):
    counts = rng.integers(0 if allow_empty else 1, max_pool + 1, size=F * B)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    idx = np.empty(offsets[-1], dtype=np.int32)
    for t in range(F):
        lo, hi = offsets[t * B], offsets[(t + 1) * B]
        idx[lo:hi] = rng.integers(0, rows[t], size=hi - lo)
    return idx, offsets


def _brute_pool(table, row_base, F, B, D, idx, offsets):
    """np.add.at over (bag, row) pairs: a different route to the same sums."""
    out = np.zeros((B * F, D), dtype=np.float64)
    bag_of = np.repeat(np.arange(F * B), np.diff(offsets))
    t = bag_of // B
    b = bag_of % B
    rows = row_base[t] + idx.astype(np.int64)
    np.add.at(out, b * F + t, table[rows].astype(np.float64))
    return out.reshape(B, F, D)


@pytest.mark.parametrize("dtype", [np.float32, np.float16])
def test_lookup_matches_add_at(dtype):
    rng = np.random.default_rng(1)
    F, B, D = 4, 9, 8
    rows = np.array([5, 1, 17, 3])
    row_base = np.concatenate([[0], np.cumsum(rows)])
    table = rng.uniform(-1, 1, size=(row_base[-1], D)).astype(dtype)
    idx, off = _random_bags(rng, F, B, rows, 6)
    pooled, status = oracle.emb_fwd(table, row_base, F, D, B, idx, off)
    ref = _brute_pool(table, row_base, F, B, D, idx, off).astype(dtype)
    assert status == 0
    # few fp32/fp16 terms sum exactly in double, so one rounding on both sides
    assert np.array_equal(pooled, ref)


def test_lookup_single_hot_is_a_copy_and_empty_is_zero():
    rng = np.random.default_rng(2)
    F, B, D = 3, 5, 4
    rows = np.array([7, 7, 7])
    row_base = np.concatenate([[0], np.cumsum(rows)])
    table = rng.standard_normal((21, D)).astype(np.float32)
    idx = rng.integers(0, 7, size=F * B).astype(np.int32)
    off = np.arange(F * B + 1, dtype=np.int32)
    pooled, _ = oracle.emb_fwd(table, row_base, F, D, B, idx, off)
    for t in range(F):
        for b in range(B):
            assert np.array_equal(pooled[b, t], table[row_base[t] + idx[t * B + b]])
    pooled0, _ = oracle.emb_fwd(table, row_base, F, D, B, np.zeros(0, np.int32),
                                np.zeros(F * B + 1, np.int32))
    assert not pooled0.any()


def test_lookup_hashing_and_out_of_range():
    table = np.arange(10, dtype=np.float32).reshape(5, 2)
    row_base = [0, 5]
    idx = np.array([-1, 7, 12, -13], dtype=np.int32)
    off = np.array([0, 1, 2, 3, 4], dtype=np.int32)
    # hashing: non-negative remainder by the table size (np.mod has that sign rule)
    pooled, status = oracle.emb_fwd(table, row_base, 1, 2, 4, idx, off, flags=oracle.FLAG_HASH)
    assert status == 0
    assert np.array_equal(pooled[:, 0], table[np.mod(idx, 5)])
    # without hashing the out-of-range entries are skipped and flagged
    idx2 = np.array([4, 5, -1, 0], dtype=np.int32)
    pooled, status = oracle.emb_fwd(table, row_base, 1, 2, 4, idx2, off)
    assert status == oracle.STATUS_OOB
    assert np.array_equal(pooled[0, 0], table[4]) and np.array_equal(pooled[3, 0], table[0])
    assert not pooled[1].any() and not pooled[2].any()


def test_lookup_rejects_bad_offsets():
    t = np.zeros((2, 2), np.float32)
    with pytest.raises(ValueError):
        oracle.emb_fwd(t, [0, 2], 1, 2, 2, [0, 1], [0, 2, 1])
    with pytest.raises(ValueError):
        oracle.emb_fwd(t, [0, 2], 1, 2, 2, [0, 1], [0, 1, 3])


# --------------------------------------------------------------------------
# dot interaction
# --------------------------------------------------------------------------
def _golden_z(g, F):
    dense = g["dense"].reshape(1, -1)
    pooled = np.stack([g[f"emb{t}"] for t in range(F)])[None]
    return dense, pooled


@pytest.mark.parametrize("name", ["interact_f2_d2.txt", "interact_f3_d2.txt"])
@pytest.mark.parametrize("dtype", [np.float32, np.float16, np.float64])
def test_interaction_hand_examples(name, dtype):
    g = load_golden(name)
    F = int(g["F"])
    dense, pooled = _golden_z(g, F)
    out_cols = int(g.get("out_cols", g["out"].size))
    out = oracle.interact_fwd(dense.astype(dtype), pooled.astype(dtype), out_cols)
    assert np.array_equal(out[0].astype(np.float64), g["out"])


def _brute_interaction(dense, pooled):
    Z = np.concatenate([dense[:, None, :], pooled], axis=1).astype(np.float64)
    S = np.einsum("bik,bjk->bij", Z, Z)
    i, j = np.tril_indices(Z.shape[1], -1)
    return np.concatenate([Z[:, 0, :], S[:, i, j]], axis=1)


def test_interaction_matches_einsum_and_width():
    rng = np.random.default_rng(3)
    for F, D in [(1, 4), (3, 8), (5, 3), (26, 16)]:
        B = 3
        dense = rng.standard_normal((B, D))
        pooled = rng.standard_normal((B, F, D))
        W = D + F * (F + 1) // 2
        out = oracle.interact_fwd(dense, pooled, W + 3)
        ref = _brute_interaction(dense, pooled)
        assert ref.shape[1] == W
        np.testing.assert_allclose(out[:, :W], ref, rtol=1e-12, atol=1e-12)
        assert not out[:, W:].any()                         # padding is zero
        assert np.array_equal(out[:, :D], dense)           # dense copied first
        # fp32 inputs: one rounding of the double result
        o32 = oracle.interact_fwd(dense.astype(np.float32), pooled.astype(np.float32), W)
        r32 = _brute_interaction(dense.astype(np.float32), pooled.astype(np.float32))
        np.testing.assert_allclose(o32, r32.astype(np.float32), rtol=2**-23, atol=1e-30)


def test_interaction_single_table_is_a_dot():
    rng = np.random.default_rng(4)
    dense = rng.standard_normal((2, 5))
    pooled = rng.standard_normal((2, 1, 5))
    out = oracle.interact_fwd(dense, pooled, 6)
    for b in range(2):
        assert out[b, 5] == pytest.approx(np.dot(dense[b], pooled[b, 0]), rel=1e-14)


def test_interaction_orthonormal_rows_give_zero_triangle():
    q, _ = np.linalg.qr(np.random.default_rng(6).standard_normal((8, 8)))
    dense = q[0][None]
    pooled = q[1:6][None]
    out = oracle.interact_fwd(dense, pooled, 8 + 15)
    np.testing.assert_allclose(out[0, 8:], 0.0, atol=1e-14)


def test_gram_is_symmetric_and_holds_the_triangle():
    rng = np.random.default_rng(7)
    F, D, B = 6, 10, 2
    dense = rng.standard_normal((B, D))
    pooled = rng.standard_normal((B, F, D))
    out = oracle.interact_fwd(dense, pooled, D + F * (F + 1) // 2)
    for b in range(B):
        G = oracle.gram(dense, pooled, b)
        assert np.array_equal(G, G.T)
        i, j = np.tril_indices(F + 1, -1)
        assert np.array_equal(out[b, D:], G[i, j])
        assert np.all(np.diag(G) >= 0)


# --------------------------------------------------------------------------
# interaction backward
# --------------------------------------------------------------------------
def test_interaction_backward_hand_example():
    g = load_golden("interact_bwd_f1_d2.txt")
    dense, pooled = _golden_z(g, 1)
    gd, gp = oracle.interact_bwd(g["grad_out"][None], dense.astype(np.float32),
                                 pooled.astype(np.float32))
    assert np.array_equal(gd[0], g["grad_dense"].astype(np.float32))
    assert np.array_equal(gp[0, 0], g["grad_emb0"].astype(np.float32))


def test_interaction_backward_equals_central_differences():
    """The interaction is quadratic in Z, so a central difference is exact up
    to rounding: (f(Z + h e) - f(Z - h e)) / 2h = J e for any h."""
    rng = np.random.default_rng(8)
    F, D, B = 3, 4, 2
    W = D + F * (F + 1) // 2
    P = W + 2
    dense = rng.standard_normal((B, D))
    pooled = rng.standard_normal((B, F, D))
    G = rng.standard_normal((B, P))
    gd, gp = oracle.interact_bwd(G, dense, pooled)

    def loss(dn, pl):
        return float((oracle.interact_fwd(dn, pl, P) * G).sum())

    h = 0.25
    for b in range(B):
        for k in range(D):
            e = np.zeros_like(dense); e[b, k] = h
            fd = (loss(dense + e, pooled) - loss(dense - e, pooled)) / (2 * h)
            assert fd == pytest.approx(gd[b, k], rel=1e-12, abs=1e-12)
            for t in range(F):
                e = np.zeros_like(pooled); e[b, t, k] = h
                fd = (loss(dense, pooled + e) - loss(dense, pooled - e)) / (2 * h)
                assert fd == pytest.approx(gp[b, t, k], rel=1e-12, abs=1e-12)


def test_interaction_backward_ignores_padding():
    rng = np.random.default_rng(9)
    F, D, B = 4, 6, 3
    W = D + F * (F + 1) // 2
    dense = rng.standard_normal((B, D)).astype(np.float32)
    pooled = rng.standard_normal((B, F, D)).astype(np.float32)
    G = rng.standard_normal((B, W + 4)).astype(np.float32)
    a = oracle.interact_bwd(G, dense, pooled)
    G2 = G.copy(); G2[:, W:] = 1e6
    b = oracle.interact_bwd(G2, dense, pooled)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


# --------------------------------------------------------------------------
# sparse embedding gradient + SGD
# --------------------------------------------------------------------------
def test_sgd_hand_example():
    g = load_golden("sgd_hand.txt")
    rows, D, B = int(g["rows"]), int(g["D"]), int(g["B"])
    table = g["table"].astype(np.float32).reshape(rows, D)
    gp = g["grad_pooled"].astype(np.float32).reshape(B, 1, D)
    new, status, _, _ = oracle.emb_bwd_sgd(table, [0, rows], 1, D, B, g["indices"], g["offsets"],
                                           gp, g["lr"])
    assert status == 0
    assert np.array_equal(new.reshape(-1), g["table_after"].astype(np.float32))


def _keys_vals(row_base, F, B, idx, off):
    bag = np.repeat(np.arange(F * B), np.diff(off))
    t, b = bag // B, bag % B
    keys = (row_base[t] + idx.astype(np.int64)).astype(np.uint32)
    vals = (b * F + t).astype(np.uint32)
    return keys, vals


def test_sgd_matches_add_at_and_stable_sort():
    rng = np.random.default_rng(10)
    F, B, D = 3, 40, 4
    rows = np.array([6, 2, 9])
    row_base = np.concatenate([[0], np.cumsum(rows)])
    table = rng.uniform(-0.05, 0.05, size=(row_base[-1], D)).astype(np.float32)
    idx, off = _random_bags(rng, F, B, rows, 4)
    gp = rng.standard_normal((B, F, D)).astype(np.float32) * 1e-2
    lr = 0.1
    new, status, sk, sv = oracle.emb_bwd_sgd(table, row_base, F, D, B, idx, off, gp, lr)
    keys, vals = _keys_vals(row_base, F, B, idx, off)
    order = np.argsort(keys, kind="stable")
    assert np.array_equal(sk, keys[order]) and np.array_equal(sv, vals[order])
    # brute force: accumulate every occurrence's gradient row with np.add.at
    gsum = np.zeros((row_base[-1], D), dtype=np.float64)
    np.add.at(gsum, keys.astype(np.int64), gp.reshape(B * F, D)[vals].astype(np.float64))
    ref = (table.astype(np.float64) - np.float64(np.float32(lr)) * gsum).astype(np.float32)
    np.testing.assert_allclose(new, ref, rtol=2**-23, atol=1e-12)
    touched = np.zeros(row_base[-1], bool); touched[keys] = True
    assert np.array_equal(new[~touched], table[~touched])


def test_sgd_distinct_rows_lr_zero_and_skips():
    rng = np.random.default_rng(11)
    F, B, D = 1, 6, 3
    table = rng.standard_normal((10, D)).astype(np.float32)
    idx = np.array([9, 0, 4, 2, 7, 5], dtype=np.int32)
    off = np.arange(7, dtype=np.int32)
    gp = rng.standard_normal((B, 1, D)).astype(np.float32)
    new, _, _, _ = oracle.emb_bwd_sgd(table, [0, 10], F, D, B, idx, off, gp, 0.5)
    for b in range(B):
        want = (table[idx[b]].astype(np.float64) - 0.5 * gp[b, 0].astype(np.float64)).astype(np.float32)
        assert np.array_equal(new[idx[b]], want)
    same, _, _, _ = oracle.emb_bwd_sgd(table, [0, 10], F, D, B, idx, off, gp, 0.0)
    assert np.array_equal(same, table)
    bad = np.array([9, 10, -1, 2, 7, 5], dtype=np.int32)
    new, status, sk, sv = oracle.emb_bwd_sgd(table, [0, 10], F, D, B, bad, off, gp, 0.5)
    assert status == oracle.STATUS_OOB
    assert list(sk[-2:]) == [oracle.SKIP_KEY, oracle.SKIP_KEY] and list(sv[-2:]) == [1, 2]
    hashed, status, _, _ = oracle.emb_bwd_sgd(table, [0, 10], F, D, B, bad, off, gp, 0.5,
                                              flags=oracle.FLAG_HASH)
    assert status == 0
    ref = table.astype(np.float64).copy()
    gsum = np.zeros_like(ref)
    np.add.at(gsum, np.mod(bad, 10), gp[:, 0].astype(np.float64))
    touched = np.unique(np.mod(bad, 10))
    ref[touched] = ref[touched] - 0.5 * gsum[touched]
    assert np.array_equal(hashed, ref.astype(np.float32))
