"""GPU parity of dlrm_emb_interact_fwd (lookup + interaction in one pass).

It computes the same thing as dlrm_emb_fwd followed by dlrm_interact_fwd, with
the same arithmetic, so the two are compared bit for bit; the oracle check of
the two-call path (test_gpu_lookup, test_gpu_interaction) carries over, and
one oracle comparison is made here directly.
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
    pooled = torch.empty(B, F, D, dtype=torch.float16, device=dev())
    out = torch.full((B, P), float("nan"), dtype=torch.float16, device=dev())
    st = torch.zeros(1, dtype=torch.int32, device=dev())
    dl.dlrm_emb_fwd(tab, row_base, F, D, B, idx, off, pooled, flags=flags, status=st)
    dl.dlrm_interact_fwd(dense, pooled, F, D, B, out, P, status=st)
    torch.cuda.synchronize()
    return out.cpu().numpy(), int(st.item())


def fused(dl, tab, row_base, F, D, B, idx, off, dense, P, flags=0):
    out = torch.full((B, P), float("nan"), dtype=torch.float16, device=dev())
    st = torch.zeros(1, dtype=torch.int32, device=dev())
    dl.dlrm_emb_interact_fwd(tab, row_base, F, D, B, idx, off, dense, out, P, flags=flags, status=st)
    torch.cuda.synchronize()
    return out.cpu().numpy(), int(st.item())


@pytest.mark.parametrize("B", [1, 5, 1000, 65536])
def test_default_shapes_match_two_calls_and_oracle(cuda_lib, B):
    w = inputs.dlrm_default(B=B, dtype=inputs.F16, alpha=1.05)
    tab = device_tables(cuda_lib, w)
    args = (tab, to_dev(w.row_base), w.F, w.D, w.B, to_dev(w.indices), to_dev(w.offsets),
            to_dev(w.dense.astype(np.float16)), w.out_cols)
    a, sa = two_calls(cuda_lib, *args)
    b, sb = fused(cuda_lib, *args)
    assert sa == sb == 0
    assert np.array_equal(a, b)
    samples = np.unique(np.concatenate([np.arange(min(B, 8)), [B - 1]]))
    c = Compact(w, samples)
    rp, _ = oracle.emb_fwd(c.tables, c.row_base, c.F, c.D, c.B, c.indices, c.offsets)
    ro = oracle.interact_fwd(c.dense, rp, w.out_cols)
    W = w.D + w.F * (w.F + 1) // 2
    assert_within_abs_sum(b[samples][:, :W], ro[:, :W], abs_products(c.dense, rp), 2e-2, "fused vs oracle")


# "heavy" (4.2 indices per bag) puts several chunks of 32 positions in a
# sample's list of several-index bags
BAG_MIX = {"ragged": [0, 1, 1, 1, 2, 5], "heavy": [0, 1, 2, 5, 9, 8]}


@pytest.mark.parametrize("mix", sorted(BAG_MIX))
@pytest.mark.parametrize("F,D", [(1, 64), (3, 128), (26, 64), (31, 192), (32, 256), (32, 128)])
def test_shapes_with_ragged_bags_hashing_and_skips(cuda_lib, F, D, mix):
    rng = np.random.default_rng(F * 7 + D)
    B = 37
    rows = rng.integers(1, 50, size=F)
    row_base = np.concatenate([[0], np.cumsum(rows)]).astype(np.int64)
    tab = to_dev(rng.standard_normal((row_base[-1], D)).astype(np.float16))
    counts = rng.choice(BAG_MIX[mix], size=F * B)
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    idx = rng.integers(-60, 60, size=off[-1]).astype(np.int32)
    dense = to_dev(rng.standard_normal((B, D)).astype(np.float16))
    W = D + F * (F + 1) // 2
    P = (W + 7) // 8 * 8
    for flags in (0, 1):
        args = (tab, to_dev(row_base), F, D, B, to_dev(idx), to_dev(off), dense, P, flags)
        a, sa = two_calls(cuda_lib, *args)
        b, sb = fused(cuda_lib, *args)
        assert sa == sb
        assert np.array_equal(a, b)


def test_rejects_unsupported_shapes(cuda_lib):
    t = torch.zeros(10, 16, dtype=torch.float32, device=dev())
    with pytest.raises(cuda_lib.DlrmError) as e:
        cuda_lib.dlrm_emb_interact_fwd(t, to_dev(np.array([0, 10])), 1, 16, 2, to_dev(np.zeros(2, np.int32)),
                                       to_dev(np.arange(3, dtype=np.int32)), torch.zeros(2, 16, device=dev()),
                                       torch.zeros(2, 24, device=dev()), 24)
    assert e.value.code == cuda_lib.DLRM_ERR_UNSUPPORTED
