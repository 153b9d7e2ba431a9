"""The tensor-core bottom MLP (dlrm_bottom_mlp_fwd) against the oracle
("DLRM For PyTorch", §Model architecture; --bottom_mlp_sizes 512,256,128;
mixed precision: fp16 tensors, fp32 accumulation).

Layer by layer, each GPU layer is fed the GPU's own previous activation (read
from the documented workspace), so both sides start from the same fp16
numbers: they may differ by the fp32 accumulation (at most K 2^-23 of the sum
of absolute terms) and, where that moves a value across a rounding boundary,
by one binary16 ulp.  The whole chain is then compared with the oracle run
from x within 2^-8 of the absolute-value chain |W| ... |x| + |b| (errors
propagate through |W|; the ReLU is 1-Lipschitz)."""

import numpy as np
import pytest
import torch

import oracle
from dlrm_embeddings_dot_gb300 import inputs
from gpu_util import dev, to_dev

pytestmark = pytest.mark.gpu


def _ulp16(a):
    a = np.abs(np.asarray(a, np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0**-14)))
    return 2.0 ** (e - 10)


def _run(dl, x, dims, W, b):
    B = x.shape[0]
    wp, bp = inputs.mlp_pack(W, b)
    ws = torch.empty(dl.dlrm_bottom_mlp_workspace_size(B, dims), dtype=torch.uint8, device=dev())
    out = torch.empty(B, dims[-1], dtype=torch.float16, device=dev())
    status = torch.zeros(1, dtype=torch.int32, device=dev())
    dl.dlrm_bottom_mlp_fwd(to_dev(x), dims, to_dev(wp), to_dev(bp), out, ws, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    # workspace: x as fp16 [B][round_up(K0, 8)], then the hidden activations
    acts, off = [], 0
    widths = [(dims[0] + 7) // 8 * 8] + list(dims[1:-1])
    raw = ws.cpu().numpy()
    for wdt in widths:
        n = B * wdt * 2
        acts.append(raw[off:off + n].view(np.float16).reshape(B, wdt))
        off += (n + 255) // 256 * 256
    return acts, out.cpu().numpy()


def _check(x, dims, W, b, acts, out):
    K0 = dims[0]
    assert np.array_equal(acts[0][:, :K0], x.astype(np.float16)) and not acts[0][:, K0:].any()
    layers_out = acts[1:] + [out]
    h = acts[0][:, :K0]
    for l in range(len(W)):
        ref = oracle.mlp_fwd(h.astype(np.float32), [W[l].astype(np.float32)], [b[l]], half_io=True)
        got = layers_out[l].astype(np.float64)
        a = np.abs(h.astype(np.float64)) @ np.abs(W[l].astype(np.float64)).T + np.abs(b[l].astype(np.float64))
        tol = _ulp16(np.maximum(np.abs(ref), np.abs(got))) + W[l].shape[1] * 2.0**-23 * a
        bad = np.abs(got - ref) > tol
        assert not bad.any(), f"layer {l}: {bad.sum()} outputs off, worst {np.abs(got - ref).max()}"
        h = layers_out[l]
    # the chain, from x
    ref = oracle.mlp_fwd(x, [w.astype(np.float32) for w in W], b, half_io=True)
    chain = np.abs(x.astype(np.float16).astype(np.float64))
    for l in range(len(W)):
        chain = chain @ np.abs(W[l].astype(np.float64)).T + np.abs(b[l].astype(np.float64))
    assert np.all(np.abs(out.astype(np.float64) - ref) <= 2.0**-8 * chain)


def _run_layer_by_layer(dl, x, dims, W, b):
    """The same chain as one call per layer (the per-layer kernel, each layer's
    fp16 output passed on as fp32, which the next call rounds back exactly)."""
    h, acts = x, []
    for l in range(len(W)):
        a, o = _run(dl, h, [h.shape[1], dims[l + 1]], [W[l]], [b[l]])
        acts.append(a[0])
        h = o.astype(np.float32)
    return acts, o


@pytest.mark.parametrize("K0,B", [(13, 1), (13, 300), (13, 4096), (13, 4097), (16, 333), (9, 515)])
def test_default_bottom_mlp(cuda_lib, K0, B):
    """The pages' 13-512-256-128 shape (and any 9..16 inputs before the same
    layers) runs as one fused launch whose hidden activations stay on chip: its
    output equals the layer-by-layer chain bit for bit, and that chain is
    checked layer by layer against the oracle."""
    dims = [K0, 512, 256, 128]
    x = np.random.default_rng(B).lognormal(0.0, 1.0, size=(B, K0)).astype(np.float32)
    W, b = inputs.mlp_layers(dims, seed=0)
    _, out = _run(cuda_lib, x, dims, W, b)
    lacts, lout = _run_layer_by_layer(cuda_lib, x, dims, W, b)
    assert np.array_equal(out.view(np.uint16), lout.view(np.uint16)), "fused chain differs from the per-layer one"
    _check(x, dims, W, b, lacts, lout)
    assert (out > 0).any() and (out == 0).any()


@pytest.mark.parametrize("dims", [[16, 16], [5, 48], [70, 64, 32], [130, 1024, 16], [8, 272]])
def test_other_widths(cuda_lib, dims):
    """Padded first layer, K past one 64-wide block, every output tile width
    (N = 16, 48, 272 ... -> tiles of 16 up to 256)."""
    B = 257
    x = np.random.default_rng(len(dims)).standard_normal((B, dims[0])).astype(np.float32)
    W, b = inputs.mlp_layers(dims, seed=1)
    acts, out = _run(cuda_lib, x, dims, W, b)
    _check(x, dims, W, b, acts, out)


def test_full_batch_sampled_rows(cuda_lib):
    """64K rows in the launch shape the benchmark times; sampled rows checked."""
    dims = [13, 512, 256, 128]
    B = 65536
    x = np.random.default_rng(7).lognormal(0.0, 1.0, size=(B, 13)).astype(np.float32)
    W, b = inputs.mlp_layers(dims, seed=0)
    _, out = _run(cuda_lib, x, dims, W, b)
    _, lout = _run_layer_by_layer(cuda_lib, x, dims, W, b)
    assert np.array_equal(out.view(np.uint16), lout.view(np.uint16)), "fused chain differs from the per-layer one"
    rows = np.unique(np.concatenate([np.random.default_rng(8).choice(B, 64, replace=False), [0, B - 1]]))
    ref = oracle.mlp_fwd(x[rows], [w.astype(np.float32) for w in W], b, half_io=True)
    chain = np.abs(x[rows].astype(np.float16).astype(np.float64))
    for l in range(3):
        chain = chain @ np.abs(W[l].astype(np.float64)).T + np.abs(b[l].astype(np.float64))
    assert np.all(np.abs(out[rows].astype(np.float64) - ref) <= 2.0**-8 * chain)


def test_rejects_unsupported(cuda_lib):
    with pytest.raises(cuda_lib.DlrmError) as e:
        x = torch.zeros(4, 13, device=dev())
        cuda_lib.dlrm_bottom_mlp_fwd(x, [13, 40], torch.zeros(1024, dtype=torch.float16, device=dev()),
                                     torch.zeros(64, device=dev()), torch.empty(4, 40, dtype=torch.float16,
                                                                               device=dev()),
                                     torch.empty(4096, dtype=torch.uint8, device=dev()))
    assert e.value.code == cuda_lib.DLRM_ERR_UNSUPPORTED
