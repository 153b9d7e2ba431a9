"""GPU parity of dlrm_emb_bwd_sgd (sparse gradient + SGD) against the oracle.

Bar: the sorted (row, grad-row) pairs left in the workspace equal a stable
sort bit for bit; updated rows agree within rel 1e-5 of |w| + lr * sum|g|;
untouched rows are bit-identical; two runs give bit-identical tables.
"""

import numpy as np
import pytest
import torch

import oracle
from dlrm_embeddings_dot_gb300 import inputs
from gpu_util import Compact, dev, device_tables, to_dev
from helpers import assert_within_abs_sum

pytestmark = pytest.mark.gpu


def run_sgd(dl, tables_np_or_dev, row_base, F, D, B, indices, offsets, grad_pooled, lr, flags=0):
    tab = tables_np_or_dev if isinstance(tables_np_or_dev, torch.Tensor) else to_dev(tables_np_or_dev)
    nnz = indices.size
    # only well-formed CSR goes to the device
    assert offsets[0] == 0 and offsets[-1] == nnz and (np.diff(offsets) >= 0).all()
    total_rows = int(row_base[-1])
    wsb = dl.dlrm_emb_bwd_sgd_workspace_size(nnz, D, total_rows)
    ws = torch.empty(max(wsb, 256), dtype=torch.uint8, device=dev())
    status = torch.zeros(1, dtype=torch.int32, device=dev())
    dl.dlrm_emb_bwd_sgd(tab, to_dev(row_base), total_rows, F, D, B, to_dev(indices.astype(np.int32)),
                        to_dev(offsets.astype(np.int32)), to_dev(grad_pooled), lr, ws, flags=flags,
                        status=status)
    torch.cuda.synchronize()
    off_v = dl.dlrm_ws_align(4 * nnz)
    keys = ws[: 4 * nnz].view(torch.int32).cpu().numpy().view(np.uint32)
    vals = ws[off_v: off_v + 4 * nnz].view(torch.int32).cpu().numpy().view(np.uint32)
    return tab, int(status.item()), keys, vals


def abs_scale(tables, row_base, F, B, D, indices, offsets, grad_pooled, lr, flags=0):
    """|w| + lr * sum of |g| over the row's occurrences (tolerance scale)."""
    bag = np.repeat(np.arange(F * B), np.diff(offsets))
    t, b = bag // B, bag % B
    n = row_base[t + 1] - row_base[t]
    idx = indices.astype(np.int64)
    ok = (idx >= 0) & (idx < n) if not flags else np.ones_like(idx, bool)
    if flags:
        idx = np.mod(idx, n)
    s = np.zeros(tables.shape, dtype=np.float64)
    np.add.at(s, (row_base[t] + idx)[ok], np.abs(grad_pooled.reshape(B * F, D)[(b * F + t)[ok]]))
    return np.abs(tables.astype(np.float64)) + lr * s


def check(dl, tables, row_base, F, D, B, idx, off, gp, lr, flags=0):
    tab, status, keys, vals = run_sgd(dl, tables, row_base, F, D, B, idx, off, gp, lr, flags)
    ref, rstatus, rk, rv = oracle.emb_bwd_sgd(tables, row_base, F, D, B, idx, off, gp, lr, flags)
    assert status == rstatus
    assert np.array_equal(keys, rk), "sorted row keys differ from a stable sort"
    assert np.array_equal(vals, rv), "sorted grad rows differ from a stable sort"
    got = tab.cpu().numpy()
    assert_within_abs_sum(got, ref, abs_scale(tables, row_base, F, B, D, idx, off, gp, lr, flags), 1e-5, "tables")
    touched = np.zeros(tables.shape[0], bool)
    touched[rk[rk != oracle.SKIP_KEY]] = True
    assert np.array_equal(got[~touched], tables[~touched]), "untouched rows changed"
    return got


def test_tiny_training_slice(cuda_lib):
    w = inputs.tiny_slice(seed=0, train=True)
    tables = w.full_tables()
    pooled, _ = oracle.emb_fwd(tables, w.row_base, w.F, w.D, w.B, w.indices, w.offsets)
    _, gp = oracle.interact_bwd(w.grad_out, w.dense, pooled)
    check(cuda_lib, tables, w.row_base, w.F, w.D, w.B, w.indices, w.offsets, gp, w.lr)


@pytest.mark.parametrize("B", [50, 400])   # about 3K and 24K indices: the one-block sort and the multi-block one
@pytest.mark.parametrize("D", [4, 16, 128, 256, 512])
def test_multi_hot_random(cuda_lib, D, B):
    rng = np.random.default_rng(D + B)
    F = 4
    rows = np.array([3, 200, 40, 1])
    row_base = np.concatenate([[0], np.cumsum(rows)]).astype(np.int64)
    tables = rng.uniform(-0.05, 0.05, size=(row_base[-1], D)).astype(np.float32)
    counts = rng.integers(0, 30, size=F * B)
    off = np.concatenate([[0], np.cumsum(counts)])
    idx = np.concatenate([rng.integers(0, rows[g // B], size=c) for g, c in enumerate(counts)]).astype(np.int32)
    gp = (rng.standard_normal((B, F, D)) * 1e-2).astype(np.float32)
    check(cuda_lib, tables, row_base, F, D, B, idx, off, gp, 0.1)


@pytest.mark.parametrize("n", [31, 32, 33, 64, 65, 1000, 40000])
def test_one_hot_row_across_many_chunks(cuda_lib, n):
    """Every position hits the same row (and a few hit a second one), so runs
    cross 32-position chunk edges and go through the partial-sum fixup."""
    rng = np.random.default_rng(n)
    F, B, D = 1, n, 128
    tables = rng.uniform(-0.05, 0.05, size=(10, D)).astype(np.float32)
    idx = np.full(n, 7, dtype=np.int32)
    idx[rng.integers(0, n, size=max(1, n // 10))] = 3
    off = np.arange(n + 1)
    gp = (rng.standard_normal((B, F, D)) * 1e-2).astype(np.float32)
    check(cuda_lib, tables, np.array([0, 10]), F, D, B, idx, off, gp, 0.1)


def test_zipf_default_shapes_and_determinism(cuda_lib):
    """26 tables with log-uniform sizes, Zipf 1.2 (hot rows span many chunks),
    B = 3000; compared through a compacted table; run twice, bit-identical."""
    w = inputs.dlrm_default(B=3000, dtype=inputs.F32, alpha=1.2, train=True)
    c = Compact(w, np.arange(w.B))
    rng = np.random.default_rng(5)
    gp = (rng.standard_normal((w.B, w.F, w.D)) * 1e-2).astype(np.float32)
    got = check(cuda_lib, c.tables, c.row_base, c.F, c.D, c.B, c.indices, c.offsets, gp, 0.1)
    again, _, _, _ = run_sgd(cuda_lib, c.tables, c.row_base, c.F, c.D, c.B, c.indices, c.offsets, gp, 0.1)
    assert np.array_equal(again.cpu().numpy(), got)
    # full-size joint table on the device: untouched rows stay bit-identical
    tab = device_tables(cuda_lib, w)
    before = tab.clone()
    _, status, keys, _ = run_sgd(cuda_lib, tab, w.row_base, w.F, w.D, w.B, w.indices, w.offsets, gp, 0.1)
    assert status == 0
    touched = torch.zeros(w.total_rows, dtype=torch.bool, device=dev())
    touched[torch.from_numpy(keys.astype(np.int64)).to(dev())] = True
    assert torch.equal(tab[~touched], before[~touched])
    # the touched rows equal the compacted run's rows
    assert np.array_equal(tab[torch.from_numpy(c.global_rows).to(dev())].cpu().numpy(), got)


@pytest.mark.parametrize("B", [100, 5000])   # 200 and 10,000 indices: both sort paths
def test_hashing_out_of_range_and_lr_zero(cuda_lib, B):
    rng = np.random.default_rng(9)
    F, D = 2, 16
    row_base = np.array([0, 13, 20], dtype=np.int64)
    tables = rng.uniform(-0.05, 0.05, size=(20, D)).astype(np.float32)
    idx = rng.integers(-30, 30, size=F * B).astype(np.int32)
    off = np.arange(F * B + 1)
    gp = rng.standard_normal((B, F, D)).astype(np.float32)
    check(cuda_lib, tables, row_base, F, D, B, idx, off, gp, 0.1, flags=1)
    check(cuda_lib, tables, row_base, F, D, B, idx, off, gp, 0.1, flags=0)
    tab, _, _, _ = run_sgd(cuda_lib, tables, row_base, F, D, B, idx, off, gp, 0.0, flags=1)
    assert np.array_equal(tab.cpu().numpy(), tables)


@pytest.mark.parametrize("B", [3000, 9000])   # below and above the one-block sort's 8,192 keys
@pytest.mark.parametrize("total_rows", [1, 255, 256, 257, 70000, 20_000_000])
def test_key_width_edges(cuda_lib, total_rows, B):
    """The number of radix passes follows the key width; 1 row, byte edges."""
    rng = np.random.default_rng(total_rows + B)
    F, D = 1, 4
    idx = rng.integers(0, total_rows, size=B).astype(np.int32)
    idx[::5] = total_rows - 1
    uniq = np.unique(idx)
    tables_c = rng.uniform(-1, 1, size=(uniq.size, D)).astype(np.float32)
    off = np.arange(B + 1)
    gp = rng.standard_normal((B, F, D)).astype(np.float32)
    # full table on the device, only the used rows have known values
    tab = torch.zeros(total_rows, D, device=dev())
    tab[torch.from_numpy(uniq.astype(np.int64)).to(dev())] = to_dev(tables_c)
    tab, status, keys, vals = run_sgd(cuda_lib, tab, np.array([0, total_rows]), F, D, B, idx, off, gp, 0.5)
    order = np.argsort(idx, kind="stable")
    assert status == 0
    assert np.array_equal(keys, idx[order].astype(np.uint32)) and np.array_equal(vals, order.astype(np.uint32))
    ref, _, _, _ = oracle.emb_bwd_sgd(tables_c, np.array([0, uniq.size]), F, D, B,
                                      np.searchsorted(uniq, idx).astype(np.int32), off, gp, 0.5)
    got = tab[torch.from_numpy(uniq.astype(np.int64)).to(dev())].cpu().numpy()
    np.testing.assert_allclose(got, ref, rtol=1e-5, atol=1e-5)


def test_empty(cuda_lib):
    tab = torch.ones(4, 8, device=dev())
    _, status, _, _ = run_sgd(cuda_lib, tab, np.array([0, 4]), 1, 8, 5, np.zeros(0, np.int32),
                              np.zeros(6, np.int64), np.zeros((5, 1, 8), np.float32), 0.1)
    assert status == 0 and torch.equal(tab, torch.ones(4, 8, device=dev()))


@pytest.mark.parametrize("reps", [1, 1500])   # 6 and 9,000 indices: both sort paths
def test_malformed_offsets_are_clamped_and_flagged(cuda_lib, reps):
    """Malformed CSR reaches the sparse update: keys are clamped into [0, nnz],
    grad rows and table rows are range-checked, and the status bit is set."""
    F, B, D = 2, 4 * reps, 16
    tab = torch.zeros(5, D, device=dev())
    idx_np = np.tile(np.array([0, 1, 2, 0, 1, 1], dtype=np.int32), reps)
    bad_np = np.arange(F * B + 1, dtype=np.int64) * idx_np.size // (F * B)
    bad_np[:9] = [0, 2, 9, -3, 4, 3, 6, 100, 6]
    if reps > 1:
        bad_np[-1] = idx_np.size + 50
    idx, bad = to_dev(idx_np), to_dev(bad_np.astype(np.int32))
    ws = torch.zeros(cuda_lib.dlrm_emb_bwd_sgd_workspace_size(idx_np.size, D, 5), dtype=torch.uint8, device=dev())
    status = torch.zeros(1, dtype=torch.int32, device=dev())
    gp = torch.ones(B, F, D, device=dev())
    cuda_lib.dlrm_emb_bwd_sgd(tab, to_dev(np.array([0, 3, 5], dtype=np.int64)), 5, F, D, B, idx, bad, gp, 0.1,
                              ws, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & cuda_lib.DLRM_STATUS_BAD_OFFSETS
    assert torch.isfinite(tab).all()


@pytest.mark.parametrize("n,B", [(8192, 8192), (8193, 8193), (100, 40000)])
def test_one_block_sort_threshold(cuda_lib, n, B):
    """Batches of up to 8,192 indices over at most 32,768 bags are sorted by one
    block in shared memory, others by the multi-block passes: both sides of the
    edge give the stable sort and the oracle's rows (hot rows span many chunks)."""
    rng = np.random.default_rng(n + B)
    F, D = 1, 32
    rows = 70000   # three radix passes
    tables = rng.uniform(-0.05, 0.05, size=(rows, D)).astype(np.float32)
    counts = np.zeros(B, np.int64)
    counts[rng.choice(B, size=min(n, B), replace=False)] = 1
    np.add.at(counts, rng.integers(0, B, size=n - min(n, B)), 1)
    off = np.concatenate([[0], np.cumsum(counts)])
    idx = np.where(rng.random(n) < 0.3, 17, rng.integers(0, rows, size=n)).astype(np.int32)
    gp = (rng.standard_normal((B, F, D)) * 1e-2).astype(np.float32)
    check(cuda_lib, tables, np.array([0, rows]), F, D, B, idx, off, gp, 0.1)

