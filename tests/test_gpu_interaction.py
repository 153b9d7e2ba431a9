"""GPU parity of dlrm_interact_fwd / dlrm_interact_bwd against the oracle.

Bar: within rel 1e-5 (fp32) or 2e-2 (fp16 storage, fp32 accumulation) of the
sum of absolute products behind each output; the dense block and the zero
padding are bit-exact.  The fp16 tensor-core kernel is additionally held to
one fp16 rounding of the fp32-accurate result.
"""

import numpy as np
import pytest
import torch

import oracle
from dlrm_embeddings_dot_gb300 import inputs
from gpu_util import Compact, dev, device_tables, to_dev
from helpers import assert_within_abs_sum

pytestmark = pytest.mark.gpu


def abs_products(dense, pooled):
    """For every output column, the sum of |z_i[k] z_j[k]| over k."""
    Z = np.concatenate([dense[:, None, :], pooled], axis=1).astype(np.float64)
    A = np.einsum("bik,bjk->bij", np.abs(Z), np.abs(Z))
    i, j = np.tril_indices(Z.shape[1], -1)
    return np.concatenate([np.abs(Z[:, 0, :]), A[:, i, j]], axis=1)


def run_fwd(dl, dense, pooled, P, cuda_core=False):
    B, F, D = pooled.shape
    out = torch.full((B, P), float("nan"), dtype=dense.dtype, device=dev())
    status = torch.zeros(1, dtype=torch.int32, device=dev())
    if cuda_core:
        dl.dlrm_interact_fwd_cuda_core(dense, pooled, F, D, B, out, P)
    else:
        dl.dlrm_interact_fwd(dense, pooled, F, D, B, out, P, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return out.cpu().numpy()


def check_fwd(got, dense, pooled, P, rtol):
    B, F, D = pooled.shape
    W = D + F * (F + 1) // 2
    ref = oracle.interact_fwd(dense, pooled, P)
    assert np.array_equal(got[:, :D], dense)                  # dense block copied exactly
    assert not got[:, W:].any()                               # padding exactly zero
    assert_within_abs_sum(got[:, :W], ref[:, :W], abs_products(dense, pooled), rtol, "interaction")
    return ref


def test_tiny_slice_fp32(cuda_lib):
    w = inputs.tiny_slice(seed=0)
    pooled, _ = oracle.emb_fwd(w.full_tables(), w.row_base, w.F, w.D, w.B, w.indices, w.offsets)
    got = run_fwd(cuda_lib, to_dev(w.dense), to_dev(pooled), w.out_cols)
    check_fwd(got, w.dense, pooled, w.out_cols, 1e-5)


@pytest.mark.parametrize("B", [1, 3, 4, 5, 1021, 4096])
def test_tensor_core_default_shape(cuda_lib, B):
    """F = 26, D = 128, P = 480 fp16; B not a multiple of 4 exercises the
    partial last tile (its missing samples arrive as TMA zero fill)."""
    rng = np.random.default_rng(B)
    dense = np.abs(rng.standard_normal((B, 128))).astype(np.float16)
    pooled = rng.uniform(-0.05, 0.05, size=(B, 26, 128)).astype(np.float16)
    got = run_fwd(cuda_lib, to_dev(dense), to_dev(pooled), 480)
    ref = check_fwd(got, dense, pooled, 480, 2e-2)
    # tighter: at most one fp16 ulp from the oracle's correctly rounded value,
    # plus the fp32 accumulation error
    err = np.abs(got[:, 128:479].astype(np.float64) - ref[:, 128:479].astype(np.float64))
    scale = np.abs(ref[:, 128:479].astype(np.float64)) * 2.0**-10 + abs_products(dense, pooled)[:, 128:] * 1e-5
    assert (err <= scale + 2.0**-24).all()


@pytest.mark.parametrize("F,D", [(1, 64), (2, 64), (8, 128), (26, 64), (31, 192), (32, 256), (32, 128)])
def test_tensor_core_shapes(cuda_lib, F, D):
    rng = np.random.default_rng(F * 1000 + D)
    B = 37
    W = D + F * (F + 1) // 2
    P = (W + 7) // 8 * 8
    dense = rng.standard_normal((B, D)).astype(np.float16)
    pooled = rng.standard_normal((B, F, D)).astype(np.float16)
    got = run_fwd(cuda_lib, to_dev(dense), to_dev(pooled), P)
    check_fwd(got, dense, pooled, P, 2e-2)
    cc = run_fwd(cuda_lib, to_dev(dense), to_dev(pooled), P, cuda_core=True)
    check_fwd(cc, dense, pooled, P, 2e-2)


@pytest.mark.parametrize("B", [1, 5, 1021, 4099])
def test_register_kernel_default_shape_fp32(cuda_lib, B):
    """F = 26, D = 128, P = 480 fp32: the register-resident kernel (one warp
    per sample); B past 1216 makes warps take several samples, so the
    double-buffered staging of the next sample is exercised."""
    rng = np.random.default_rng(100 + B)
    dense = np.abs(rng.standard_normal((B, 128))).astype(np.float32)
    pooled = rng.standard_normal((B, 26, 128)).astype(np.float32)
    got = run_fwd(cuda_lib, to_dev(dense), to_dev(pooled), 480)
    check_fwd(got, dense, pooled, 480, 1e-5)


@pytest.mark.parametrize("F,D,P", [(3, 16, 22), (26, 128, 480), (5, 40, 60), (33, 64, 700), (26, 24, 400),
                                   (8, 128, 164), (8, 128, 192), (26, 128, 496), (26, 128, 484)])
@pytest.mark.parametrize("dt", [np.float32, np.float16])
def test_cuda_core_kernel(cuda_lib, F, D, P, dt):
    if dt == np.float16 and D % 8:
        pytest.skip("fp16 rows must be multiples of 16 bytes")
    rng = np.random.default_rng(F + D + P)
    B = 19
    dense = rng.standard_normal((B, D)).astype(dt)
    pooled = rng.standard_normal((B, F, D)).astype(dt)
    got = run_fwd(cuda_lib, to_dev(dense), to_dev(pooled), P)
    check_fwd(got, dense, pooled, P, 1e-5 if dt == np.float32 else 2e-2)


def test_default_workload_end_to_end_fp16(cuda_lib):
    """Real DLRM-default inputs (bottom-MLP dense, generated fp16 tables, Zipf
    indices): lookup then interaction on the device vs the oracle on a
    compacted copy of the same 512 samples."""
    w = inputs.dlrm_default(B=512, dtype=inputs.F16)
    tab = device_tables(cuda_lib, w)
    pooled = torch.empty(w.B, w.F, w.D, dtype=torch.float16, device=dev())
    cuda_lib.dlrm_emb_fwd(tab, to_dev(w.row_base), w.F, w.D, w.B, to_dev(w.indices), to_dev(w.offsets), pooled)
    dense = to_dev(w.dense.astype(np.float16))
    got = run_fwd(cuda_lib, dense, pooled, 480)
    c = Compact(w, np.arange(w.B))
    rp, _ = oracle.emb_fwd(c.tables, c.row_base, c.F, c.D, c.B, c.indices, c.offsets)
    check_fwd(got, c.dense, rp, 480, 2e-2)


# ---------------------------------------------------------------- backward
def abs_bwd(G, dense, pooled):
    """Sum of absolute terms behind each gradient element."""
    B, F, D = pooled.shape
    Z = np.concatenate([dense[:, None, :], pooled], axis=1).astype(np.float64)
    i, j = np.tril_indices(F + 1, -1)
    M = np.zeros((B, F + 1, F + 1))
    M[:, i, j] = np.abs(G[:, D:D + i.size])
    M = M + M.transpose(0, 2, 1)
    dz = np.einsum("bij,bjk->bik", M, np.abs(Z))
    return np.abs(G[:, :D]) + dz[:, 0], dz[:, 1:]


@pytest.mark.parametrize("F,D,P,B", [(3, 16, 22, 256), (26, 128, 480, 513), (1, 32, 40, 9),
                                     (15, 64, 200, 33), (31, 128, 640, 17),
                                     # fp32: the register kernel (F in {8, 26}, D = 128, P % 4 == 0), with
                                     # several samples per warp past 1824, and the staged kernel for P % 4 != 0
                                     (26, 128, 480, 4099), (26, 128, 1024, 37), (8, 128, 164, 2000),
                                     (26, 128, 481, 70)])
@pytest.mark.parametrize("dt", [np.float32, np.float16])
def test_backward(cuda_lib, F, D, P, B, dt):
    rng = np.random.default_rng(F * D + B)
    dense = rng.standard_normal((B, D)).astype(dt)
    pooled = rng.standard_normal((B, F, D)).astype(dt)
    G = (rng.standard_normal((B, P)) * 1e-2).astype(np.float32)
    gd = torch.full((B, D), float("nan"), device=dev())
    gp = torch.full((B, F, D), float("nan"), device=dev())
    cuda_lib.dlrm_interact_bwd(to_dev(G), to_dev(dense), to_dev(pooled), F, D, B, P, gd, gp)
    torch.cuda.synchronize()
    rd, rp = oracle.interact_bwd(G, dense, pooled)
    sd, sp = abs_bwd(G.astype(np.float64), dense, pooled)
    assert_within_abs_sum(gd.cpu().numpy(), rd, sd, 1e-5, "grad_dense")
    assert_within_abs_sum(gp.cpu().numpy(), rp, sp, 1e-5, "grad_pooled")


def test_backward_ignores_padding(cuda_lib):
    rng = np.random.default_rng(1)
    B, F, D, P = 8, 26, 128, 480
    dense = to_dev(rng.standard_normal((B, D)).astype(np.float32))
    pooled = to_dev(rng.standard_normal((B, F, D)).astype(np.float32))
    G = rng.standard_normal((B, P)).astype(np.float32)
    outs = []
    for pad in (0.0, 1e30):
        G[:, 479:] = pad
        gd = torch.empty(B, D, device=dev())
        gp = torch.empty(B, F, D, device=dev())
        cuda_lib.dlrm_interact_bwd(to_dev(G), dense, pooled, F, D, B, P, gd, gp)
        outs.append((gd.cpu().numpy(), gp.cpu().numpy()))
    assert np.array_equal(outs[0][0], outs[1][0]) and np.array_equal(outs[0][1], outs[1][1])
