"""Pins of the bottom-MLP oracle ("DLRM For PyTorch", §Model architecture;
--bottom_mlp_sizes; mixed precision keeps the tensors in fp16)."""

import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "mlp_hand.txt")


@pytest.fixture(scope="module", autouse=True)
def _built():
    oracle.build()


def _golden():
    g = {}
    for line in open(GOLDEN):
        if line.strip() and not line.startswith("#"):
            k, rest = line.split(None, 1)
            g[k] = np.array([[float(v) for v in r.split()] for r in rest.split(";")], dtype=np.float32)
    return g


def test_hand_worked_two_layers():
    g = _golden()
    W, b = [g["W1"], g["W2"]], [g["b1"][0], g["b2"][0]]
    assert np.array_equal(oracle.mlp_fwd(g["x"], W[:1], b[:1]), g["h1"].astype(np.float64))
    assert np.array_equal(oracle.mlp_fwd(g["x"], W, b), g["out"].astype(np.float64))
    assert np.array_equal(oracle.mlp_fwd(g["x"], W, b, half_io=True), g["out"].astype(np.float64))


def test_binary16_rounding_of_inputs_and_outputs():
    one = [np.ones((1, 1), np.float32)]
    zero = [np.zeros(1, np.float32)]
    # below half an ulp (2^-11 at 1.0): rounds down
    assert oracle.mlp_fwd(np.array([[1 + 2**-12]], np.float32), one, zero, half_io=True)[0, 0] == 1.0
    assert oracle.mlp_fwd(np.array([[1 + 2**-12]], np.float32), one, zero)[0, 0] == 1 + 2**-12
    # exact ties go to the even neighbour
    assert oracle.mlp_fwd(np.array([[1 + 2**-11]], np.float32), one, zero, half_io=True)[0, 0] == 1.0
    assert oracle.mlp_fwd(np.array([[1 + 3 * 2**-11]], np.float32), one, zero, half_io=True)[0, 0] == 1 + 2**-9
    # the output of a layer is rounded too: 1 * 1 + 2^-12 -> 1
    assert oracle.mlp_fwd(np.ones((1, 1), np.float32), one, [np.array([2**-12], np.float32)],
                          half_io=True)[0, 0] == 1.0


def test_identity_layers_are_relu():
    x = np.array([[1.5, -2.0, 0.0, 3.25]], np.float32)
    I = np.eye(4, dtype=np.float32)
    z = np.zeros(4, np.float32)
    assert np.array_equal(oracle.mlp_fwd(x, [I, I, I], [z, z, z]), np.maximum(x, 0).astype(np.float64))


def test_brute_force_small_random():
    rng = np.random.default_rng(0)
    dims = [5, 7, 4, 3]
    x = rng.standard_normal((6, dims[0])).astype(np.float32)
    W = [rng.standard_normal((dims[l + 1], dims[l])).astype(np.float32) for l in range(3)]
    b = [rng.standard_normal(dims[l + 1]).astype(np.float32) for l in range(3)]
    h = x.astype(np.float64)
    for l in range(3):
        h = np.maximum(h @ W[l].T.astype(np.float64) + b[l].astype(np.float64), 0.0)
    np.testing.assert_allclose(oracle.mlp_fwd(x, W, b), h, rtol=1e-13, atol=1e-13)
    assert (h == 0).any() and (h > 0).any()   # both sides of the ReLU occur


def test_default_widths():
    rng = np.random.default_rng(1)
    dims = [13, 512, 256, 128]
    W = [np.zeros((dims[l + 1], dims[l]), np.float32) for l in range(3)]
    b = [np.full(dims[l + 1], 0.5, np.float32) for l in range(3)]
    out = oracle.mlp_fwd(rng.standard_normal((3, 13)).astype(np.float32), W, b, half_io=True)
    assert out.shape == (3, 128) and np.all(out == 0.5)
