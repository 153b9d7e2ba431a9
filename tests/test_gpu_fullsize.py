"""Parity at the full workload sizes, in the launch configuration the benchmark
times, checked on sampled outputs the oracle computes one by one.

* DLRM-default forward: 65,536 samples, 26 fp16 tables (rows log-uniform in
  [10, 4e6]), Zipf 1.05, lookup + tensor-core interaction.
* The 64K training step: the same shapes with fp32 master tables, Zipf 1.2,
  upstream gradient N(0, 1e-2), SGD lr 0.1; the update of sampled rows
  (including the most frequent row) is recomputed from every occurrence of
  the row in the batch.
* Multi-hot: 16,384 samples, 26 fp32 tables of 1e6 rows, pooling U{1..100}.
* Large tables: 26 fp16 tables, three of 40M rows, at batch 1,048,576.

Sampled pooled rows are bit-exact for single-index bags; everything else
within the stated tolerances of the sum of absolute terms.
"""

import numpy as np
import pytest
import torch

import oracle
from dlrm_embeddings_dot_gb300 import inputs
from gpu_util import Compact, dev, device_tables, to_dev
from helpers import assert_within_abs_sum
from test_gpu_interaction import abs_bwd, abs_products

pytestmark = pytest.mark.gpu


def _samples(B, n, seed):
    rng = np.random.default_rng(seed)
    s = np.unique(np.concatenate([rng.choice(B, size=n, replace=False), [0, 1, B - 2, B - 1]]))
    return s


def _forward(dl, w, tab):
    F, D, B, P = w.F, w.D, w.B, w.out_cols
    tt = tab.dtype
    pooled = torch.empty(B, F, D, dtype=tt, device=dev())
    out = torch.empty(B, P, dtype=tt, device=dev())
    status = torch.zeros(1, dtype=torch.int32, device=dev())
    dense = to_dev(w.dense.astype(np.float16 if tt == torch.float16 else np.float32))
    dl.dlrm_emb_fwd(tab, to_dev(w.row_base), F, D, B, to_dev(w.indices), to_dev(w.offsets), pooled, status=status)
    dl.dlrm_interact_fwd(dense, pooled, F, D, B, out, P, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return dense, pooled, out


def _check_forward_samples(w, pooled, out, samples, tol):
    c = Compact(w, samples)
    rp, _ = oracle.emb_fwd(c.tables, c.row_base, c.F, c.D, c.B, c.indices, c.offsets)
    sel = torch.from_numpy(samples).to(dev())
    gp = pooled[sel].cpu().numpy()
    counts = np.diff(c.offsets).reshape(c.F, c.B).T          # [b][t] bag sizes
    single = counts == 1
    assert np.array_equal(gp[single], rp[single]), "single-index bags must be bit copies"
    if (~single).any():
        absum = np.zeros(rp.shape)
        for t in range(c.F):
            for k in range(c.B):
                g = t * c.B + k
                rows = c.row_base[t] + c.indices[c.offsets[g]:c.offsets[g + 1]].astype(np.int64)
                absum[k, t] = np.abs(c.tables[rows].astype(np.float64)).sum(axis=0)
        assert_within_abs_sum(gp, rp, absum, tol, "pooled (sampled)")
    if out is not None:
        ro = oracle.interact_fwd(c.dense, rp, w.out_cols)
        W = w.D + w.F * (w.F + 1) // 2
        go = out[sel].cpu().numpy()
        assert np.array_equal(go[:, :w.D], c.dense)
        assert not go[:, W:].any()
        assert_within_abs_sum(go[:, :W], ro[:, :W], abs_products(c.dense, rp), tol, "interaction (sampled)")
    return c, rp


def _occurrences(w, rows):
    """Positions (ascending) of every index that resolves to one of the global rows."""
    bag = np.repeat(np.arange(w.F * w.B), np.diff(w.offsets))
    t = bag // w.B
    keys = w.row_base[t] + w.indices.astype(np.int64)
    out = {}
    for r in rows:
        p = np.flatnonzero(keys == r)
        out[int(r)] = (p, bag[p] // w.B, bag[p] % w.B)         # positions, t, b
    return out


def _check_rows(dl, w, tab_after, table_seed_rows, occ, grad_of, lr):
    """Oracle update of each sampled row from all its occurrences, in position order."""
    for r, (p, t, b) in occ.items():
        g = grad_of(t, b)                                        # [n_occ][D] fp32
        w0 = inputs.table_rows(w.table_seed, np.array([r]), w.D, inputs.F32)
        n = p.size
        new, _, _, _ = oracle.emb_bwd_sgd(w0, np.array([0, 1]), 1, w.D, n, np.zeros(n, np.int32),
                                          np.arange(n + 1), g.reshape(n, 1, w.D), lr)
        got = tab_after[torch.tensor([r], device=dev())].cpu().numpy()
        scale = np.abs(w0.astype(np.float64)) + lr * np.abs(g.astype(np.float64)).sum(axis=0)
        assert_within_abs_sum(got, new, scale, 1e-5, f"row {r} ({n} occurrences)")


def test_default_forward_64k_fp16(cuda_lib):
    w = inputs.dlrm_default(B=65536, dtype=inputs.F16, alpha=1.05)
    tab = device_tables(cuda_lib, w)
    _, pooled, out = _forward(cuda_lib, w, tab)
    _check_forward_samples(w, pooled, out, _samples(w.B, 60, 1), 2e-2)
    del tab, pooled, out
    torch.cuda.empty_cache()


def test_training_step_64k_fp32(cuda_lib):
    dl = cuda_lib
    w = inputs.dlrm_default(B=65536, dtype=inputs.F32, alpha=1.2, train=True)
    F, D, B, P = w.F, w.D, w.B, w.out_cols
    tab = device_tables(dl, w)
    dense, pooled, out = _forward(dl, w, tab)
    gd = torch.empty(B, D, device=dev())
    gp = torch.empty(B, F, D, device=dev())
    go = to_dev(w.grad_out)
    dl.dlrm_interact_bwd(go, dense, pooled, F, D, B, P, gd, gp)
    ws = torch.empty(dl.dlrm_emb_bwd_sgd_workspace_size(w.nnz, D, w.total_rows), dtype=torch.uint8, device=dev())
    status = torch.zeros(1, dtype=torch.int32, device=dev())
    dl.dlrm_emb_bwd_sgd(tab, to_dev(w.row_base), w.total_rows, F, D, B, to_dev(w.indices), to_dev(w.offsets),
                        gp, w.lr, ws, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0

    # forward and interaction backward on sampled samples
    samples = _samples(B, 40, 2)
    c, rp = _check_forward_samples(w, pooled, out, samples, 1e-5)
    rgd, rgp = oracle.interact_bwd(c.grad_out, c.dense, rp)
    sel = torch.from_numpy(samples).to(dev())
    sd, sp = abs_bwd(c.grad_out.astype(np.float64), c.dense, rp)
    assert_within_abs_sum(gd[sel].cpu().numpy(), rgd, sd, 1e-5, "grad_dense (sampled)")
    assert_within_abs_sum(gp[sel].cpu().numpy(), rgp, sp, 1e-5, "grad_pooled (sampled)")

    # the sorted keys equal a stable sort (checked at full size: a property at any size)
    keys = ws[: 4 * w.nnz].view(torch.int32).cpu().numpy().view(np.uint32)
    off_v = dl.dlrm_ws_align(4 * w.nnz)
    vals = ws[off_v: off_v + 4 * w.nnz].view(torch.int32).cpu().numpy().view(np.uint32)
    bag = np.repeat(np.arange(F * B), np.diff(w.offsets))
    ref_keys = (w.row_base[bag // B] + w.indices.astype(np.int64)).astype(np.uint32)
    order = np.argsort(ref_keys, kind="stable")
    assert np.array_equal(keys, ref_keys[order])
    assert np.array_equal(vals, ((bag % B) * F + bag // B).astype(np.uint32)[order])

    # the SGD update of sampled rows, from every occurrence, with the oracle's own gradients
    uniq, cnt = np.unique(ref_keys, return_counts=True)
    rng = np.random.default_rng(3)
    rows = np.concatenate([[uniq[np.argmax(cnt)]], rng.choice(uniq, size=6, replace=False)])
    occ = _occurrences(w, rows)
    need = np.unique(np.concatenate([o[2] for o in occ.values()]))
    cn = Compact(w, need)
    pn, _ = oracle.emb_fwd(cn.tables, cn.row_base, cn.F, cn.D, cn.B, cn.indices, cn.offsets)
    _, gpn = oracle.interact_bwd(cn.grad_out, cn.dense, pn)
    pos_of = {int(s): k for k, s in enumerate(need)}

    def grad_of(t, b):
        return gpn[[pos_of[int(x)] for x in b], t]

    _check_rows(dl, w, tab, None, occ, grad_of, w.lr)
    # a sample of untouched rows is bit-identical to the generator
    untouched = np.setdiff1d(rng.integers(0, w.total_rows, size=2000), uniq)
    got = tab[torch.from_numpy(untouched).to(dev())].cpu().numpy()
    assert np.array_equal(got, inputs.table_rows(w.table_seed, untouched, D, inputs.F32))
    del tab, dense, pooled, out, gd, gp, go, ws
    torch.cuda.empty_cache()


def test_multi_hot_16k_fp32(cuda_lib):
    dl = cuda_lib
    w = inputs.multi_hot(B=16384)
    F, D, B = w.F, w.D, w.B
    tab = device_tables(dl, w)
    pooled = torch.empty(B, F, D, device=dev())
    status = torch.zeros(1, dtype=torch.int32, device=dev())
    dl.dlrm_emb_fwd(tab, to_dev(w.row_base), F, D, B, to_dev(w.indices), to_dev(w.offsets), pooled, status=status)
    torch.cuda.synchronize()
    _check_forward_samples(w, pooled, None, _samples(B, 12, 4), 1e-5)
    # backward + SGD with an upstream grad_pooled drawn N(0, 1e-2)
    grad = np.random.default_rng(5).normal(0, 1e-2, size=(B, F, D)).astype(np.float32)
    ws = torch.empty(dl.dlrm_emb_bwd_sgd_workspace_size(w.nnz, D, w.total_rows), dtype=torch.uint8, device=dev())
    dl.dlrm_emb_bwd_sgd(tab, to_dev(w.row_base), w.total_rows, F, D, B, to_dev(w.indices), to_dev(w.offsets),
                        to_dev(grad), w.lr, ws, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    bag = np.repeat(np.arange(F * B), np.diff(w.offsets))
    keys = (w.row_base[bag // B] + w.indices.astype(np.int64))
    uniq, cnt = np.unique(keys, return_counts=True)
    rng = np.random.default_rng(6)
    rows = np.concatenate([[uniq[np.argmax(cnt)]], rng.choice(uniq, size=6, replace=False)])
    occ = _occurrences(w, rows)
    _check_rows(dl, w, tab, None, occ, lambda t, b: grad[b, t], w.lr)
    del tab, pooled, ws
    torch.cuda.empty_cache()


def test_large_tables_1m_fp16(cuda_lib):
    B = 1 << 20
    w = inputs.dlrm_default(B=B, dtype=inputs.F16, alpha=1.05, rows=inputs.large_tables_rows())
    tab = device_tables(cuda_lib, w)
    _, pooled, out = _forward(cuda_lib, w, tab)
    _check_forward_samples(w, pooled, out, _samples(B, 40, 7), 2e-2)
    del tab, pooled, out
    torch.cuda.empty_cache()
