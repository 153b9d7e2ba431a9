"""GPU parity of dlrm_emb_fwd (embedding lookup with sum pooling) against the oracle.

Bar: single-index bags and all index handling are bit-exact; multi-index sums
agree within rel 1e-5 (fp32) or 2e-2 (fp16 storage, fp32 accumulation) of
the sum of absolute summands.
"""

import numpy as np
import pytest
import torch

import oracle
from dlrm_embeddings_dot_gb300 import inputs
from gpu_util import Compact, dev, device_tables, to_dev, torch_dtype
from helpers import assert_within_abs_sum

pytestmark = pytest.mark.gpu


def run_lookup(dl, tables, row_base, F, D, B, indices, offsets, flags=0):
    # only well-formed CSR goes to the device
    assert offsets[0] == 0 and offsets[-1] == indices.size and (np.diff(offsets) >= 0).all()
    pooled = torch.full((B, F, D), float("nan"), dtype=tables.dtype, device=dev())
    status = torch.zeros(1, dtype=torch.int32, device=dev())
    dl.dlrm_emb_fwd(tables, to_dev(row_base), F, D, B, to_dev(indices.astype(np.int32)),
                    to_dev(offsets.astype(np.int32)), pooled, flags=flags, status=status)
    torch.cuda.synchronize()
    return pooled.cpu().numpy(), int(status.item())


def abs_sum_pool(tables, row_base, F, B, D, indices, offsets):
    """Sum of |row| over each bag (the tolerance scale), by np.add.at."""
    out = np.zeros((B * F, D))
    bag = np.repeat(np.arange(F * B), np.diff(offsets))
    t, b = bag // B, bag % B
    np.add.at(out, b * F + t, np.abs(tables[row_base[t] + indices.astype(np.int64)].astype(np.float64)))
    return out.reshape(B, F, D)


def test_synth_tables_match_host_generator(cuda_lib):
    for dt in (inputs.F32, inputs.F16):
        t = torch.empty(3000, 16, dtype=torch_dtype(dt), device=dev())
        cuda_lib.dlrm_synth_fill_uniform(t, 12345, 0)
        ref = inputs.table_rows(12345, np.arange(3000), 16, dt)
        assert np.array_equal(t.cpu().numpy(), ref)
        # an offset start (first_elem) continues the same element numbering
        part = torch.empty(100, 16, dtype=torch_dtype(dt), device=dev())
        cuda_lib.dlrm_synth_fill_uniform(part, 12345, 16 * 2900)
        assert np.array_equal(part.cpu().numpy(), ref[2900:])


def test_tiny_slice_is_bit_exact(cuda_lib):
    w = inputs.tiny_slice(seed=0)
    tables = w.full_tables()
    got, status = run_lookup(cuda_lib, to_dev(tables), w.row_base, w.F, w.D, w.B, w.indices, w.offsets)
    ref, rstatus = oracle.emb_fwd(tables, w.row_base, w.F, w.D, w.B, w.indices, w.offsets)
    assert status == rstatus == 0
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("dt", [inputs.F32, inputs.F16])
def test_default_shapes_sampled_bit_exact(cuda_lib, dt):
    """26 single-hot tables, real log-uniform sizes; B = 1000 (ragged vs the
    4-bag groups); compared on every sample through compacted tables."""
    w = inputs.dlrm_default(B=1000, dtype=dt)
    tab = device_tables(cuda_lib, w)
    got, status = run_lookup(cuda_lib, tab, w.row_base, w.F, w.D, w.B, w.indices, w.offsets)
    c = Compact(w, np.arange(w.B))
    ref, _ = oracle.emb_fwd(c.tables, c.row_base, c.F, c.D, c.B, c.indices, c.offsets)
    assert status == 0
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("dt", [inputs.F32, inputs.F16])
@pytest.mark.parametrize("D", [16, 64, 128, 256])
def test_multi_hot_ragged_with_empty_bags(cuda_lib, dt, D):
    rng = np.random.default_rng(D)
    F, B = 5, 77
    rows = np.array([1, 50, 300, 7, 1000])
    row_base = np.concatenate([[0], np.cumsum(rows)]).astype(np.int64)
    tables = rng.uniform(-1, 1, size=(row_base[-1], D)).astype(np.float16 if dt else np.float32)
    counts = rng.integers(0, 40, size=F * B)
    counts[::7] = 0
    offsets = np.concatenate([[0], np.cumsum(counts)])
    idx = np.concatenate([rng.integers(0, rows[(g // B)], size=c) for g, c in enumerate(counts)]).astype(np.int32)
    got, status = run_lookup(cuda_lib, to_dev(tables), row_base, F, D, B, idx, offsets)
    ref, _ = oracle.emb_fwd(tables, row_base, F, D, B, idx, offsets)
    assert status == 0
    tol = 1e-5 if dt == inputs.F32 else 2e-2
    assert_within_abs_sum(got, ref, abs_sum_pool(tables, row_base, F, B, D, idx, offsets), tol, "pooled")
    # single-index bags are exact copies, empty bags exact zeros
    for g in np.flatnonzero(counts <= 1):
        t, b = g // B, g % B
        assert np.array_equal(got[b, t], ref[b, t])


def test_hashing_and_out_of_range(cuda_lib):
    rng = np.random.default_rng(3)
    F, B, D = 2, 64, 32
    rows = np.array([10, 3])
    row_base = np.array([0, 10, 13], dtype=np.int64)
    tables = rng.standard_normal((13, D)).astype(np.float32)
    idx = rng.integers(-40, 40, size=F * B).astype(np.int32)
    off = np.arange(F * B + 1)
    got, status = run_lookup(cuda_lib, to_dev(tables), row_base, F, D, B, idx, off, flags=1)
    ref, rs = oracle.emb_fwd(tables, row_base, F, D, B, idx, off, flags=oracle.FLAG_HASH)
    assert status == rs == 0 and np.array_equal(got, ref)
    got, status = run_lookup(cuda_lib, to_dev(tables), row_base, F, D, B, idx, off)
    ref, rs = oracle.emb_fwd(tables, row_base, F, D, B, idx, off)
    assert status == rs == oracle.STATUS_OOB and np.array_equal(got, ref)
    # multi-hot path with some bad entries
    off2 = np.concatenate([[0], np.cumsum(np.full(F * 8, 16))])
    idx2 = rng.integers(-40, 40, size=off2[-1]).astype(np.int32)
    got, status = run_lookup(cuda_lib, to_dev(tables), row_base, F, D, 8, idx2, off2)
    ref, rs = oracle.emb_fwd(tables, row_base, F, D, 8, idx2, off2)
    assert status == rs == oracle.STATUS_OOB
    np.testing.assert_allclose(got, ref, rtol=1e-5, atol=1e-5)


def test_empty_index_list(cuda_lib):
    F, B, D = 3, 10, 8
    tables = torch.ones(5, D, device=dev())
    got, status = run_lookup(cuda_lib, tables, np.array([0, 1, 3, 5]), F, D, B, np.zeros(0, np.int32),
                             np.zeros(F * B + 1, np.int64))
    assert status == 0 and not got.any()


def test_malformed_offsets_are_clamped_and_flagged(cuda_lib):
    """Offsets past nnz, negative or decreasing: the kernels clamp every bag
    into [0, nnz] (no access leaves the index list) and set the status bit."""
    F, B, D = 2, 4, 16
    tables = to_dev(np.arange(5 * D, dtype=np.float32).reshape(5, D))
    row_base = to_dev(np.array([0, 3, 5], dtype=np.int64))
    idx = to_dev(np.array([0, 1, 2, 0, 1, 1], dtype=np.int32))
    bad = to_dev(np.array([0, 2, 9, -3, 4, 3, 6, 100, 6], dtype=np.int32))
    pooled = torch.zeros(B, F, D, device=dev())
    status = torch.zeros(1, dtype=torch.int32, device=dev())
    cuda_lib.dlrm_emb_fwd(tables, row_base, F, D, B, idx, bad, pooled, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & cuda_lib.DLRM_STATUS_BAD_OFFSETS
    assert torch.isfinite(pooled).all()


# Rows one load instruction moves whole (32 lanes x 16 bytes): the single-hot
# kernel sums the bags of several indices of each 32-bag group as one list of
# positions, for every batch.
WHOLE_ROW = [(inputs.F32, 128), (inputs.F16, 256)]


@pytest.mark.parametrize("dt,D", WHOLE_ROW)
@pytest.mark.parametrize("flags", [0, 1])
def test_whole_row_mixed_bags_hashing_and_skips(cuda_lib, dt, D, flags):
    """Empty, single and several-index bags (up to 40: a bag's positions span
    several rounds of 32), indices outside the table skipped and flagged, or
    folded into it with DLRM_FLAG_HASH_INDICES; 633 bags, a ragged last group."""
    rng = np.random.default_rng(D + flags)
    F, B = 3, 211
    rows = np.array([10, 3, 50])
    row_base = np.concatenate([[0], np.cumsum(rows)]).astype(np.int64)
    tables = rng.uniform(-1, 1, size=(row_base[-1], D)).astype(np.float16 if dt == inputs.F16 else np.float32)
    counts = rng.choice([0, 1, 1, 2, 3, 7, 40], size=F * B)
    offsets = np.concatenate([[0], np.cumsum(counts)])
    idx = rng.integers(-60, 60, size=offsets[-1]).astype(np.int32)
    got, status = run_lookup(cuda_lib, to_dev(tables), row_base, F, D, B, idx, offsets, flags=flags)
    ref, rs = oracle.emb_fwd(tables, row_base, F, D, B, idx, offsets, flags=flags)
    absum, _ = oracle.emb_fwd(np.abs(tables).astype(np.float64), row_base, F, D, B, idx, offsets, flags=flags)
    assert status == rs == (0 if flags else oracle.STATUS_OOB)
    assert_within_abs_sum(got, ref, absum, 1e-5 if dt == inputs.F32 else 2e-2, "pooled")
    for g in np.flatnonzero(counts <= 1):   # copies of the row, or zeros
        t, b = g // B, g % B
        assert np.array_equal(got[b, t], ref[b, t])


@pytest.mark.parametrize("dt,D", WHOLE_ROW)
def test_whole_row_malformed_offsets(cuda_lib, dt, D):
    """Negative, decreasing and past-nnz offsets: each bag is clamped on its
    own (start into [0, nnz], end into [start, nnz]) and the status bit set;
    the result equals the oracle on the CSR rebuilt from the clamped bags."""
    rng = np.random.default_rng(11 + D)
    F, B = 2, 100
    rows = np.array([30, 20])
    row_base = np.concatenate([[0], np.cumsum(rows)]).astype(np.int64)
    tables = rng.uniform(-1, 1, size=(row_base[-1], D)).astype(np.float16 if dt == inputs.F16 else np.float32)
    counts = rng.choice([1, 2, 5], size=F * B)
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    nnz = int(off[-1])
    idx = rng.integers(0, 20, size=nnz).astype(np.int32)
    off[17] = 3            # bag 16 ends before it starts, bag 17 starts early
    off[40] = nnz + 50     # past the index list
    off[77] = -5           # negative
    pooled = torch.full((B, F, D), float("nan"), dtype=torch_dtype(dt), device=dev())
    status = torch.zeros(1, dtype=torch.int32, device=dev())
    cuda_lib.dlrm_emb_fwd(to_dev(tables), to_dev(row_base), F, D, B, to_dev(idx), to_dev(off.astype(np.int32)),
                          pooled, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & cuda_lib.DLRM_STATUS_BAD_OFFSETS
    s = np.clip(off[:-1], 0, nnz)
    e = np.minimum(np.maximum(off[1:], s), nnz)
    cidx = np.concatenate([idx[a:b] for a, b in zip(s, e)]).astype(np.int32)
    coff = np.concatenate([[0], np.cumsum(e - s)])
    ref, rs = oracle.emb_fwd(tables, row_base, F, D, B, cidx, coff)
    absum, _ = oracle.emb_fwd(np.abs(tables).astype(np.float64), row_base, F, D, B, cidx, coff)
    assert rs == 0
    got = pooled.cpu().numpy()
    assert_within_abs_sum(got, ref, absum, 1e-5 if dt == inputs.F32 else 2e-2, "pooled")
    for g in np.flatnonzero(e - s <= 1):
        t, b = g // B, g % B
        assert np.array_equal(got[b, t], ref[b, t])
