"""The mixed-precision training pieces ("DLRM For PyTorch", §Mixed precision
training: fp16 interaction tensors, fp32 master tables, static loss scale,
--loss_scale 1024) against the oracle.

* fp16 pooling of fp32 rows (DLRM_FLAG_POOLED_F16): single-index bags are the
  correctly rounded row (bit-exact); larger bags within one binary16 ulp of
  the correctly rounded exact sum plus 1e-5 of the sum of absolute terms.
* dlrm_interact_bwd_f16 (tcgen05): the same one-ulp-plus-1e-5 bar against the
  oracle's exact gradient rounded once, and the 2e-2 fp16 bar of the sum of
  absolute terms; pad columns of the upstream gradient must not matter.
* fp16 gradients in the sparse SGD (DLRM_FLAG_GRAD_F16, lr / S): bit-identical
  to the fp32 path fed the same (exactly widened) gradients, and within rel
  1e-5 of the oracle.
"""

import numpy as np
import pytest
import torch

import oracle
from dlrm_embeddings_dot_gb300 import inputs
from gpu_util import dev, device_tables, to_dev
from helpers import assert_within_abs_sum
from test_gpu_interaction import abs_bwd
from test_gpu_sgd import abs_scale, run_sgd

pytestmark = pytest.mark.gpu

S = 1024.0   # static loss scale


def _ulp16(a):
    a = np.abs(np.asarray(a, np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0**-14)))
    return 2.0 ** (e - 10)


def _close16(got, ref, absum, what):
    got, ref = got.astype(np.float64), ref.astype(np.float64)
    tol = _ulp16(np.maximum(np.abs(got), np.abs(ref))) + 1e-5 * absum
    bad = np.abs(got - ref) > tol
    assert not bad.any(), f"{what}: {bad.sum()} elements beyond one fp16 ulp, worst {np.abs(got - ref).max()}"
    assert_within_abs_sum(got, ref, absum, 2e-2, what)


def _bwd16(dl, g, dense, pooled, P):
    B, F, D = pooled.shape
    gd = torch.full((B, D), float("nan"), dtype=torch.float16, device=dev())
    gp = torch.full((B, F, D), float("nan"), dtype=torch.float16, device=dev())
    status = torch.zeros(1, dtype=torch.int32, device=dev())
    dl.dlrm_interact_bwd_f16(to_dev(g), to_dev(dense), to_dev(pooled), F, D, B, P, gd, gp, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return gd.cpu().numpy(), gp.cpu().numpy()


def _case(B, F, D, P, seed):
    rng = np.random.default_rng(seed)
    dense = np.abs(rng.standard_normal((B, D))).astype(np.float16)
    pooled = rng.uniform(-0.05, 0.05, size=(B, F, D)).astype(np.float16)
    g = (rng.normal(0.0, 1e-2, size=(B, P)) * S).astype(np.float16)   # loss-scaled upstream gradient
    return dense, pooled, g


def _check_bwd(dl, B, F, D, P, seed):
    dense, pooled, g = _case(B, F, D, P, seed)
    gd, gp = _bwd16(dl, g, dense, pooled, P)
    rgd, rgp = oracle.interact_bwd_f16(g, dense, pooled)
    sd, sp = abs_bwd(g.astype(np.float64), dense, pooled)
    _close16(gd, rgd, sd, "grad_dense")
    _close16(gp, rgp, sp, "grad_pooled")
    # the pad columns of the upstream gradient are ignored
    W = D + F * (F + 1) // 2
    if P > W:
        g2 = g.copy()
        g2[:, W:] = np.float16(1000.0)
        gd2, gp2 = _bwd16(dl, g2, dense, pooled, P)
        assert np.array_equal(gd2, gd) and np.array_equal(gp2, gp)


@pytest.mark.parametrize("B", [1, 5, 1024, 4099])
def test_backward_default_shape(cuda_lib, B):
    _check_bwd(cuda_lib, B, 26, 128, 480, B)


@pytest.mark.parametrize("F,D", [(1, 64), (3, 128), (26, 64), (31, 192), (31, 256), (8, 128)])
def test_backward_shapes(cuda_lib, F, D):
    W = D + F * (F + 1) // 2
    _check_bwd(cuda_lib, 37, F, D, (W + 7) // 8 * 8 + 8, F * 100 + D)


def test_backward_rejects_unsupported(cuda_lib):
    z = torch.zeros(4096, dtype=torch.float16, device=dev())
    with pytest.raises(cuda_lib.DlrmError) as e:
        cuda_lib.dlrm_interact_bwd_f16(z, z, z, 32, 64, 1, 600, z, z)          # F = 32: no row left for dZ_0
    assert e.value.code == cuda_lib.DLRM_ERR_UNSUPPORTED
    with pytest.raises(cuda_lib.DlrmError) as e:
        cuda_lib.dlrm_interact_bwd_f16(z, z, z, 2, 64, 1, 67, z, z)            # out_cols not a multiple of 8
    assert e.value.code == cuda_lib.DLRM_ERR_UNSUPPORTED


def test_pooling_fp32_rows_to_fp16(cuda_lib):
    dl = cuda_lib
    rows = np.array([10, 1000, 70000, 5, 300])
    dense = np.zeros((777, 128), np.float32)
    w = inputs.make_workload("pool16", 777, 5, 128, inputs.F32, rows, alpha=1.05, dense=dense, out_cols=0,
                             seed=4, pool=(0, 4))
    tab = device_tables(dl, w)
    pooled = torch.empty(w.B, w.F, w.D, dtype=torch.float16, device=dev())
    status = torch.zeros(1, dtype=torch.int32, device=dev())
    dl.dlrm_emb_fwd(tab, to_dev(w.row_base), w.F, w.D, w.B, to_dev(w.indices), to_dev(w.offsets), pooled,
                    flags=dl.DLRM_FLAG_POOLED_F16, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    got = pooled.cpu().numpy()
    tables = inputs.table_rows(w.table_seed, np.arange(w.total_rows), w.D, inputs.F32)
    ref, _ = oracle.emb_fwd_f16out(tables, w.row_base, w.F, w.D, w.B, w.indices, w.offsets)
    counts = np.diff(w.offsets).reshape(w.F, w.B).T
    one = counts <= 1
    assert np.array_equal(got[one], ref[one]), "single-index and empty bags are the rounded row / zero"
    absum, _ = oracle.emb_fwd(np.abs(tables), w.row_base, w.F, w.D, w.B, w.indices, w.offsets)
    _close16(got[~one], ref[~one], absum[~one].astype(np.float64), "pooled")
    with pytest.raises(dl.DlrmError):   # the flag needs fp32 tables
        dl.dlrm_emb_fwd(tab.half(), to_dev(w.row_base), w.F, w.D, w.B, to_dev(w.indices), to_dev(w.offsets),
                        pooled, flags=dl.DLRM_FLAG_POOLED_F16)


def test_sgd_with_fp16_gradients(cuda_lib):
    dl = cuda_lib
    w = inputs.tiny_slice(seed=2, train=True)
    F, D, B = w.F, w.D, w.B
    tables = w.full_tables()
    rng = np.random.default_rng(9)
    g16 = (rng.normal(0.0, 1e-2, size=(B, F, D)) * S).astype(np.float16)
    lr = np.float32(w.lr / S)                        # exact: S is a power of two
    t16, st16, k16, v16 = run_sgd(dl, tables, w.row_base, F, D, B, w.indices, w.offsets, g16, lr,
                                  flags=dl.DLRM_FLAG_GRAD_F16)
    t32, st32, k32, v32 = run_sgd(dl, tables, w.row_base, F, D, B, w.indices, w.offsets, g16.astype(np.float32), lr)
    assert st16 == st32 == 0 and np.array_equal(k16, k32) and np.array_equal(v16, v32)
    assert np.array_equal(t16.cpu().numpy(), t32.cpu().numpy()), "fp16 gradients widen exactly"
    ref, _, _, _ = oracle.emb_bwd_sgd(tables, w.row_base, F, D, B, w.indices, w.offsets,
                                      g16.astype(np.float32), float(lr))
    assert_within_abs_sum(t16.cpu().numpy(), ref,
                          abs_scale(tables, w.row_base, F, B, D, w.indices, w.offsets, g16.astype(np.float32),
                                    float(lr)), 1e-5, "tables")


def test_amp_training_step_64k_sampled(cuda_lib):
    """The whole mixed-precision step at the 64K training shapes, in the launch
    shapes the benchmark times; sampled samples checked against the oracle."""
    dl = cuda_lib
    w = inputs.dlrm_default(B=65536, dtype=inputs.F32, alpha=1.2, train=True)
    F, D, B, P = w.F, w.D, w.B, w.out_cols
    tab = device_tables(dl, w)
    rb, idx, off = to_dev(w.row_base), to_dev(w.indices), to_dev(w.offsets)
    status = torch.zeros(1, dtype=torch.int32, device=dev())
    pooled = torch.empty(B, F, D, dtype=torch.float16, device=dev())
    dl.dlrm_emb_fwd(tab, rb, F, D, B, idx, off, pooled, flags=dl.DLRM_FLAG_POOLED_F16, status=status)
    dense16 = w.dense.astype(np.float16)
    g16 = (w.grad_out.astype(np.float64) * S).astype(np.float16)
    gd = torch.empty(B, D, dtype=torch.float16, device=dev())
    gp = torch.empty(B, F, D, dtype=torch.float16, device=dev())
    dl.dlrm_interact_bwd_f16(to_dev(g16), to_dev(dense16), pooled, F, D, B, P, gd, gp, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    rng = np.random.default_rng(11)
    samples = np.unique(np.concatenate([rng.choice(B, 48, replace=False), [0, B - 1]]))
    sel = torch.from_numpy(samples).to(dev())
    c = inputs.Compact(w, samples)
    rp, _ = oracle.emb_fwd_f16out(c.tables, c.row_base, c.F, c.D, c.B, c.indices, c.offsets)
    assert np.array_equal(pooled[sel].cpu().numpy(), rp), "single-hot fp16 pooling is the rounded row"
    rgd, rgp = oracle.interact_bwd_f16(g16[samples], dense16[samples], rp)
    sd, sp = abs_bwd(g16[samples].astype(np.float64), dense16[samples], rp)
    _close16(gd[sel].cpu().numpy(), rgd, sd, "grad_dense (sampled)")
    _close16(gp[sel].cpu().numpy(), rgp, sp, "grad_pooled (sampled)")


@pytest.mark.parametrize("B", [3000, 5000])   # 6,000 and 10,000 indices: both sort paths, D = 128
def test_sgd_with_fp16_gradients_both_sort_paths(cuda_lib, B):
    """fp16 gradients of 128-wide rows below and above the one-block sort's 8,192 indices:
    bit-identical to the same gradients widened to fp32, and within the oracle's bar."""
    dl = cuda_lib
    rng = np.random.default_rng(B)
    F, D = 2, 128
    rows = np.array([1500, 700])
    row_base = np.concatenate([[0], np.cumsum(rows)]).astype(np.int64)
    tables = rng.uniform(-0.05, 0.05, size=(row_base[-1], D)).astype(np.float32)
    idx = np.concatenate([np.where(rng.random(B) < 0.4, 3, rng.integers(0, n, size=B)) for n in rows]).astype(np.int32)
    off = np.arange(F * B + 1)
    g16 = (rng.normal(0.0, 1e-2, size=(B, F, D)) * S).astype(np.float16)
    lr = np.float32(0.1 / S)
    t16, st16, k16, v16 = run_sgd(dl, tables, row_base, F, D, B, idx, off, g16, lr, flags=dl.DLRM_FLAG_GRAD_F16)
    t32, st32, k32, v32 = run_sgd(dl, tables, row_base, F, D, B, idx, off, g16.astype(np.float32), lr)
    assert st16 == st32 == 0 and np.array_equal(k16, k32) and np.array_equal(v16, v32)
    assert np.array_equal(t16.cpu().numpy(), t32.cpu().numpy()), "fp16 gradients widen exactly"
    ref, _, rk, _ = oracle.emb_bwd_sgd(tables, row_base, F, D, B, idx, off, g16.astype(np.float32), float(lr))
    assert np.array_equal(k16, rk)
    assert_within_abs_sum(t16.cpu().numpy(), ref,
                          abs_scale(tables, row_base, F, B, D, idx, off, g16.astype(np.float32), float(lr)), 1e-5,
                          "tables")
