"""GPU parity of the fp32 lookup + interaction in one pass: the training
forward dlrm_emb_interact_fwd_train (pooled rows written for the backward)
and dlrm_emb_interact_fwd with fp32 tables (no pooled output); and of the
backward that gathers the pooled rows again, dlrm_emb_interact_bwd.

Both compute what dlrm_emb_fwd followed by dlrm_interact_fwd computes, with
the same arithmetic in the same order, so pooled rows, interaction output and
status bits are compared bit for bit with the two calls (whose oracle parity
test_gpu_lookup and test_gpu_interaction establish); one oracle comparison on
sampled rows is made here directly as well.
"""

import numpy as np
import pytest
import torch

import oracle
from dlrm_embeddings_dot_gb300 import inputs
from gpu_util import Compact, dev, device_tables, to_dev
from helpers import assert_within_abs_sum
from test_gpu_interaction import abs_products

pytestmark = pytest.mark.gpu


def two_calls(dl, tab, row_base, F, D, B, idx, off, dense, P, flags=0):
    pooled = torch.full((B, F, D), float("nan"), device=dev())
    out = torch.full((B, P), float("nan"), device=dev())
    st = torch.zeros(1, dtype=torch.int32, device=dev())
    dl.dlrm_emb_fwd(tab, row_base, F, D, B, idx, off, pooled, flags=flags, status=st)
    dl.dlrm_interact_fwd(dense, pooled, F, D, B, out, P, status=st)
    torch.cuda.synchronize()
    return pooled.cpu().numpy(), out.cpu().numpy(), int(st.item())


def fused_train(dl, tab, row_base, F, D, B, idx, off, dense, P, flags=0):
    pooled = torch.full((B, F, D), float("nan"), device=dev())
    out = torch.full((B, P), float("nan"), device=dev())
    st = torch.zeros(1, dtype=torch.int32, device=dev())
    dl.dlrm_emb_interact_fwd_train(tab, row_base, F, D, B, idx, off, dense, pooled, out, P, flags=flags, status=st)
    torch.cuda.synchronize()
    return pooled.cpu().numpy(), out.cpu().numpy(), int(st.item())


def fused_infer(dl, tab, row_base, F, D, B, idx, off, dense, P, flags=0):
    out = torch.full((B, P), float("nan"), device=dev())
    st = torch.zeros(1, dtype=torch.int32, device=dev())
    dl.dlrm_emb_interact_fwd(tab, row_base, F, D, B, idx, off, dense, out, P, flags=flags, status=st)
    torch.cuda.synchronize()
    return out.cpu().numpy(), int(st.item())


def _same(a, b):
    """Bit equality (NaN patterns included)."""
    return a.shape == b.shape and np.array_equal(a.view(np.uint32), b.view(np.uint32))


@pytest.mark.parametrize("B", [1, 5, 1021, 4099, 65536])
def test_default_shapes_match_two_calls_and_oracle(cuda_lib, B):
    """F = 26, D = 128, 480 columns, Zipf 1.2 single-hot fp32 (the training
    shapes); B past 1824 gives every warp several samples, so the staging of
    the next sample behind the current one is exercised."""
    w = inputs.dlrm_default(B=B, dtype=inputs.F32, alpha=1.2, train=True)
    tab = device_tables(cuda_lib, w)
    args = (tab, to_dev(w.row_base), w.F, w.D, w.B, to_dev(w.indices), to_dev(w.offsets), to_dev(w.dense),
            w.out_cols)
    p2, o2, s2 = two_calls(cuda_lib, *args)
    p1, o1, s1 = fused_train(cuda_lib, *args)
    oi, si = fused_infer(cuda_lib, *args)
    assert s1 == s2 == si == 0
    assert _same(p1, p2) and _same(o1, o2) and _same(oi, o2)
    samples = np.unique(np.concatenate([np.arange(min(B, 8)), [B // 2, B - 1]]))
    c = Compact(w, samples)
    rp, _ = oracle.emb_fwd(c.tables, c.row_base, c.F, c.D, c.B, c.indices, c.offsets)
    assert np.array_equal(p1[samples], rp), "single-hot fp32 pooling is a copy of the row"
    ro = oracle.interact_fwd(c.dense, rp, w.out_cols)
    W = w.D + w.F * (w.F + 1) // 2
    assert np.array_equal(o1[samples][:, :w.D], c.dense)
    assert not o1[samples][:, W:].any()
    assert_within_abs_sum(o1[samples][:, :W], ro[:, :W], abs_products(c.dense, rp), 1e-5, "fused vs oracle")


# bag sizes: "heavy" averages 4.2 indices per bag, so the training forward
# runs as two launches; "ragged" (1.67, with runs of several-index bags longer
# than one list chunk of 32 positions) and "mostly_single" (1.06) stay in one
# pass, whose several-index bags go through the staging ring
BAG_MIX = {"heavy": [0, 1, 2, 5, 9, 8], "ragged": [0, 1, 1, 1, 2, 5], "mostly_single": [1] * 13 + [0, 2, 3]}


@pytest.mark.parametrize("F,P", [(26, 480), (8, 164), (8, 192)])
@pytest.mark.parametrize("flags", [0, 1])
@pytest.mark.parametrize("mix", sorted(BAG_MIX))
def test_ragged_bags_hashing_and_skips(cuda_lib, F, P, flags, mix):
    """Empty bags, bags of several indices, indices outside the table (skipped
    with the status bit, or folded with DLRM_FLAG_HASH_INDICES)."""
    rng = np.random.default_rng(F * 11 + P + flags)
    B, D = 2111, 128
    rows = rng.integers(1, 50, size=F)
    row_base = np.concatenate([[0], np.cumsum(rows)]).astype(np.int64)
    tab = to_dev(rng.standard_normal((row_base[-1], D)).astype(np.float32))
    counts = rng.choice(BAG_MIX[mix], size=F * B)
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    idx = rng.integers(-60, 60, size=off[-1]).astype(np.int32)
    dense = to_dev(rng.standard_normal((B, D)).astype(np.float32))
    args = (tab, to_dev(row_base), F, D, B, to_dev(idx), to_dev(off), dense, P, flags)
    p2, o2, s2 = two_calls(cuda_lib, *args)
    p1, o1, s1 = fused_train(cuda_lib, *args)
    oi, si = fused_infer(cuda_lib, *args)
    assert s1 == s2 == si
    assert (s1 & cuda_lib.DLRM_STATUS_OOB_INDEX) == (0 if flags else cuda_lib.DLRM_STATUS_OOB_INDEX)
    assert _same(p1, p2) and _same(o1, o2) and _same(oi, o2)
    # and directly against the oracle on a few samples
    tables = tab.cpu().numpy()
    ref_p, ref_s = oracle.emb_fwd(tables, row_base, F, D, B, idx, off, flags=flags)
    absum, _ = oracle.emb_fwd(np.abs(tables), row_base, F, D, B, idx, off, flags=flags)
    assert ref_s == s1
    assert_within_abs_sum(p1, ref_p, absum.astype(np.float64), 1e-5, "pooled vs oracle")


def test_malformed_offsets_are_clamped_like_the_lookup(cuda_lib):
    rng = np.random.default_rng(5)
    F, D, B, P = 26, 128, 300, 480
    rows = np.full(F, 40)
    row_base = np.concatenate([[0], np.cumsum(rows)]).astype(np.int64)
    tab = to_dev(rng.standard_normal((row_base[-1], D)).astype(np.float32))
    off = np.arange(F * B + 1, dtype=np.int32)
    off[17] = 5                     # decreasing
    off[400] = 10**6                # past nnz
    idx = rng.integers(0, 40, size=F * B).astype(np.int32)
    dense = to_dev(rng.standard_normal((B, D)).astype(np.float32))
    args = (tab, to_dev(row_base), F, D, B, to_dev(idx), to_dev(off), dense, P)
    p2, o2, s2 = two_calls(cuda_lib, *args)
    p1, o1, s1 = fused_train(cuda_lib, *args)
    assert s1 == s2 and s1 & cuda_lib.DLRM_STATUS_BAD_OFFSETS
    assert _same(p1, p2) and _same(o1, o2)


def bwd_two_calls(dl, tab, row_base, F, D, B, idx, off, dense, go, P, flags=0):
    pooled = torch.empty(B, F, D, device=dev())
    gd = torch.full((B, D), float("nan"), device=dev())
    gp = torch.full((B, F, D), float("nan"), device=dev())
    st = torch.zeros(1, dtype=torch.int32, device=dev())
    dl.dlrm_emb_fwd(tab, row_base, F, D, B, idx, off, pooled, flags=flags, status=st)
    dl.dlrm_interact_bwd(go, dense, pooled, F, D, B, P, gd, gp)
    torch.cuda.synchronize()
    return gd.cpu().numpy(), gp.cpu().numpy(), int(st.item())


def bwd_gather(dl, tab, row_base, F, D, B, idx, off, dense, go, P, flags=0):
    gd = torch.full((B, D), float("nan"), device=dev())
    gp = torch.full((B, F, D), float("nan"), device=dev())
    st = torch.zeros(1, dtype=torch.int32, device=dev())
    dl.dlrm_emb_interact_bwd(tab, row_base, F, D, B, idx, off, go, dense, P, gd, gp, flags=flags, status=st)
    torch.cuda.synchronize()
    return gd.cpu().numpy(), gp.cpu().numpy(), int(st.item())


@pytest.mark.parametrize("B", [1, 5, 1021, 4099, 65536])
def test_gathering_backward_matches_two_calls(cuda_lib, B):
    """dlrm_emb_interact_bwd == dlrm_interact_bwd(dlrm_emb_fwd(...)) bit for bit at the training
    shapes; past 1824 samples every warp takes several, so the bag pipeline (bounds two samples
    ahead, index one ahead) is exercised; sampled rows against the oracle as well."""
    w = inputs.dlrm_default(B=B, dtype=inputs.F32, alpha=1.2, train=True)
    tab = device_tables(cuda_lib, w)
    args = (tab, to_dev(w.row_base), w.F, w.D, w.B, to_dev(w.indices), to_dev(w.offsets), to_dev(w.dense),
            to_dev(w.grad_out), w.out_cols)
    d2, p2, s2 = bwd_two_calls(cuda_lib, *args)
    d1, p1, s1 = bwd_gather(cuda_lib, *args)
    assert s1 == s2 == 0
    assert _same(d1, d2) and _same(p1, p2)
    samples = np.unique(np.concatenate([np.arange(min(B, 6)), [B - 1]]))
    c = Compact(w, samples)
    rp, _ = oracle.emb_fwd(c.tables, c.row_base, c.F, c.D, c.B, c.indices, c.offsets)
    rd, rg = oracle.interact_bwd(w.grad_out[samples], c.dense, rp)
    from test_gpu_interaction import abs_bwd
    sd, sp = abs_bwd(w.grad_out[samples].astype(np.float64), c.dense, rp)
    assert_within_abs_sum(d1[samples], rd, sd, 1e-5, "grad_dense vs oracle")
    assert_within_abs_sum(p1[samples], rg, sp, 1e-5, "grad_pooled vs oracle")


@pytest.mark.parametrize("F,P", [(26, 480), (8, 164), (26, 1024)])
@pytest.mark.parametrize("flags", [0, 1])
def test_gathering_backward_ragged_bags(cuda_lib, F, P, flags):
    rng = np.random.default_rng(F * 13 + P + flags)
    B, D = 2111, 128
    rows = rng.integers(1, 50, size=F)
    row_base = np.concatenate([[0], np.cumsum(rows)]).astype(np.int64)
    tab = to_dev(rng.standard_normal((row_base[-1], D)).astype(np.float32))
    counts = rng.choice([0, 1, 1, 1, 2, 5], size=F * B)
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    idx = rng.integers(-60, 60, size=off[-1]).astype(np.int32)
    dense = to_dev(rng.standard_normal((B, D)).astype(np.float32))
    go = to_dev((rng.standard_normal((B, P)) * 1e-2).astype(np.float32))
    args = (tab, to_dev(row_base), F, D, B, to_dev(idx), to_dev(off), dense, go, P, flags)
    d2, p2, s2 = bwd_two_calls(cuda_lib, *args)
    d1, p1, s1 = bwd_gather(cuda_lib, *args)
    assert s1 == s2
    assert _same(d1, d2) and _same(p1, p2)


def test_gathering_backward_malformed_offsets(cuda_lib):
    rng = np.random.default_rng(6)
    F, D, B, P = 26, 128, 300, 480
    row_base = np.concatenate([[0], np.cumsum(np.full(F, 40))]).astype(np.int64)
    tab = to_dev(rng.standard_normal((row_base[-1], D)).astype(np.float32))
    off = np.arange(F * B + 1, dtype=np.int32)
    off[17] = 5
    off[400] = 10**6
    idx = rng.integers(0, 40, size=F * B).astype(np.int32)
    dense = to_dev(rng.standard_normal((B, D)).astype(np.float32))
    go = to_dev((rng.standard_normal((B, P)) * 1e-2).astype(np.float32))
    args = (tab, to_dev(row_base), F, D, B, to_dev(idx), to_dev(off), dense, go, P)
    d2, p2, s2 = bwd_two_calls(cuda_lib, *args)
    d1, p1, s1 = bwd_gather(cuda_lib, *args)
    assert s1 == s2 and s1 & cuda_lib.DLRM_STATUS_BAD_OFFSETS
    assert _same(d1, d2) and _same(p1, p2)
