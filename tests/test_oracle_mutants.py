"""The pins bite: plant one plausible mistake in a copy of the oracle, compile
it, and check that a pin from ``test_oracle_pins`` fails on it.

Mistakes are planted on the CPU only, in a temporary copy of ``oracle.c``;
each one keeps every memory access in bounds.
"""

import os
import subprocess

import pytest

import oracle
import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

MUTANTS = {
    # binary16 rounding truncates instead of rounding to nearest even
    "f16_truncates": ("double q = rint(ldexp(m, 11));", "double q = floor(ldexp(m, 11));",
                      [pins.test_f64_to_f16_exact_values_and_ties]),
    # pooling keeps the last row instead of summing
    "pool_overwrites": ("acc[k] += load_val(tables, dt, row * D + k);",
                        "acc[k] = load_val(tables, dt, row * D + k);",
                        [pins.test_lookup_hand_example]),
    # the pair loop reads the wrong second vector (transposed / shifted index)
    "pair_index_slip": ("s += z_at(dense, pooled, dt, F, D, b, i, k) * z_at(dense, pooled, dt, F, D, b, j, k);\n                store_val(out",
                        "s += z_at(dense, pooled, dt, F, D, b, i, k) * z_at(dense, pooled, dt, F, D, b, i - 1 - j, k);\n                store_val(out",
                        [lambda: pins.test_interaction_hand_examples("interact_f3_d2.txt", pins.np.float64)]),
    # the dense vector is not copied in front of the triangle
    "no_dense_copy": ("store_val(out, dt, o + k, z_at(dense, pooled, dt, F, D, b, 0, k));",
                      "store_val(out, dt, o + k, 0.0);",
                      [pins.test_interaction_matches_einsum_and_width]),
    # backward: wrong sign of the pair term
    "bwd_sign": ("s += g * z_at(", "s -= g * z_at(",
                 [pins.test_interaction_backward_equals_central_differences]),
    # backward: dense pass-through gradient dropped
    "bwd_no_passthrough": ("s += load_val(grad_out, gdt, o + k);", "s += 0.0;",
                           [pins.test_interaction_backward_hand_example]),
    # backward: triangle index transposed
    "bwd_transposed": ("o + D + hi * (hi - 1) / 2 + lo", "o + D + lo * (lo + 1) / 2 + hi - lo",
                       [pins.test_interaction_backward_equals_central_differences]),
    # sparse gradient: the bag id (t*B + b) used instead of the grad_pooled row (b*F + t)
    "sgd_bag_id": ("val[p] = (uint32_t)((int64_t)b * F + t);",
                   "val[p] = (uint32_t)((int64_t)t * B + b);",
                   [pins.test_sgd_matches_add_at_and_stable_sort]),
    # SGD ascends instead of descending
    "sgd_sign": ("(double)w[k] - (double)lr * g[k]", "(double)w[k] + (double)lr * g[k]",
                 [pins.test_sgd_hand_example]),
    # unstable merge (equal keys may swap)
    "sort_unstable": ("if (k[b] < k[a])", "if (k[b] <= k[a])",
                      [pins.test_sgd_matches_add_at_and_stable_sort]),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pin_catches_mutant(name, tmp_path):
    old, new, checks = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not unique"
    path = tmp_path / f"{name}.c"
    path.write_text(src.replace(old, new))
    so = tmp_path / f"lib{name}.so"
    subprocess.check_call(["gcc", "-O2", "-std=c99", "-ffp-contract=off", "-fPIC", "-shared",
                           "-o", str(so), str(path), "-lm"])
    oracle.use(oracle.load(str(so)))
    try:
        for check in checks:
            with pytest.raises(AssertionError):
                check()
    finally:
        oracle.use(None)
