"""dlrm_emb_bwd_sgd_noalloc: the sparse gradient + SGD entry point for callers
that cannot allocate device memory (for example a plugin run from a host
framework that owns all device memory and forbids allocation while it
executes).  Its scratch is an array built into the library instead of a
caller workspace.  This file is collected last on purpose, so that a run that
stops at the first failure has already run every other test.

Both entry points run the same kernels on the same inputs, so their tables
must agree bit for bit.
"""

import numpy as np
import pytest
import torch

from dlrm_embeddings_dot_gb300 import inputs

pytestmark = pytest.mark.gpu

S = 1024.0   # the static loss scale of the mixed-precision step


def _inputs(seed):
    w = inputs.dlrm_default(B=4096, dtype=inputs.F32, alpha=1.2, train=True, seed=seed,
                            rows=np.array([97, 5000, 1, 20000] + [300] * 22))
    rng = np.random.default_rng(seed)
    gp = (rng.standard_normal((w.B, w.F, w.D)) * 1e-2).astype(np.float32)
    return w, gp


def _same_bits(a, b):
    return np.array_equal(a.cpu().numpy().view(np.uint32), b.cpu().numpy().view(np.uint32))


@pytest.mark.parametrize("fp16_grad", [False, True])
def test_noalloc_matches_workspace_entry_point_on_two_calls(cuda_lib, fp16_grad):
    dl = cuda_lib
    dev = torch.device("cuda:0")
    w, _ = _inputs(0)
    tab_ws = torch.empty(w.total_rows, w.D, device=dev)
    dl.dlrm_synth_fill_uniform(tab_ws, w.table_seed, 0)
    tab_na = tab_ws.clone()
    ws = torch.empty(dl.dlrm_emb_bwd_sgd_workspace_size(w.nnz, w.D, w.total_rows), dtype=torch.uint8, device=dev)
    flags = dl.DLRM_FLAG_GRAD_F16 if fp16_grad else 0
    for call in range(2):          # two calls in a row: the shared scratch keeps the first call's contents
        wc, gp = _inputs(call)
        rb = torch.from_numpy(wc.row_base).to(dev)
        idx = torch.from_numpy(wc.indices).to(dev)
        off = torch.from_numpy(wc.offsets).to(dev)
        g = torch.from_numpy((gp * S).astype(np.float16) if fp16_grad else gp).to(dev)
        lr = np.float32(wc.lr / S) if fp16_grad else wc.lr
        st_ws = torch.zeros(1, dtype=torch.int32, device=dev)
        st_na = torch.zeros(1, dtype=torch.int32, device=dev)
        dl.dlrm_emb_bwd_sgd(tab_ws, rb, wc.total_rows, wc.F, wc.D, wc.B, idx, off, g, lr, ws, flags=flags,
                            status=st_ws)
        dl.dlrm_emb_bwd_sgd_noalloc(tab_na, rb, wc.total_rows, wc.F, wc.D, wc.B, idx, off, g, lr, flags=flags,
                                    status=st_na)
        torch.cuda.synchronize()
        assert int(st_ws.item()) == int(st_na.item()) == 0
        assert _same_bits(tab_na, tab_ws), f"call {call}: tables differ from dlrm_emb_bwd_sgd"


def test_noalloc_rejects_sizes_beyond_its_scratch(cuda_lib):
    dl = cuda_lib
    dev = torch.device("cuda:0")
    # the smallest index count whose workspace exceeds the built-in scratch at D = 128 over 10 rows
    lo, hi = 1, dl.DLRM_MAX_NNZ
    while lo < hi:
        mid = (lo + hi) // 2
        if dl.load().dlrm_emb_bwd_sgd_workspace_size(mid, 128, 10) > dl.DLRM_NOALLOC_SCRATCH_BYTES:
            hi = mid
        else:
            lo = mid + 1
    nnz = lo
    tab = torch.zeros(10, 128, device=dev)
    idx = torch.zeros(nnz, dtype=torch.int32, device=dev)
    off = torch.tensor([0, nnz], dtype=torch.int32, device=dev)
    gp = torch.zeros(1, 1, 128, device=dev)
    with pytest.raises(dl.DlrmError) as e:
        dl.dlrm_emb_bwd_sgd_noalloc(tab, torch.tensor([0, 10], device=dev), 10, 1, 128, 1, idx, off, gp, 0.1)
    assert e.value.code == dl.DLRM_ERR_UNSUPPORTED and "scratch" in str(e.value)
    assert torch.equal(tab, torch.zeros(10, 128, device=dev))
