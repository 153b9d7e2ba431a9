"""Failure detection on the GPU without a fault: the tensor-core kernels' bounded
waits are made to run out (a zero wait limit gives up at the first wait that is
not already complete), and each call must return with DLRM_STATUS_TIMEOUT set
after draining what it issued and freeing its tensor memory.  The next call with
the default limit, on the same stream, must then match the oracle: the context
is still usable and nothing of the aborted call is left behind."""

import numpy as np
import pytest
import torch

import oracle
from gpu_util import dev, to_dev
from helpers import assert_within_abs_sum

pytestmark = pytest.mark.gpu

S = 1024.0


def _inputs(B, F, D, seed):
    rng = np.random.default_rng(seed)
    dense = rng.uniform(-1, 1, size=(B, D)).astype(np.float16)
    pooled = rng.uniform(-1, 1, size=(B, F, D)).astype(np.float16)
    return dense, pooled


@pytest.fixture
def short_waits(cuda_lib):
    yield cuda_lib
    cuda_lib.dlrm_set_wait_limit(-1)


def test_wait_limit_setting_round_trips(cuda_lib):
    default = cuda_lib.dlrm_set_wait_limit(-1)
    assert default >= 10**9                       # about two seconds of SM clock
    assert cuda_lib.dlrm_set_wait_limit(500) == default
    assert cuda_lib.dlrm_set_wait_limit(-1) == 500
    assert cuda_lib.dlrm_set_wait_limit(-1) == default
    assert cuda_lib.dlrm_set_wait_limit(10**15) == default   # clamped to the default
    assert cuda_lib.dlrm_set_wait_limit(-1) == default


def test_interaction_forward_times_out_then_recovers(short_waits):
    dl = short_waits
    B, F, D, P = 2048, 26, 128, 480
    dense, pooled = _inputs(B, F, D, 1)
    d_dense, d_pooled = to_dev(dense), to_dev(pooled)
    out = torch.full((B, P), 7.0, dtype=torch.float16, device=dev())
    status = torch.zeros(1, dtype=torch.int32, device=dev())
    dl.dlrm_set_wait_limit(0)
    dl.dlrm_interact_fwd(d_dense, d_pooled, F, D, B, out, P, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & dl.DLRM_STATUS_TIMEOUT
    dl.dlrm_set_wait_limit(-1)
    status.zero_()
    dl.dlrm_interact_fwd(d_dense, d_pooled, F, D, B, out, P, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref = oracle.interact_fwd(dense.astype(np.float64), pooled.astype(np.float64), P)
    got = out.cpu().numpy().astype(np.float64)
    absum = oracle.interact_fwd(np.abs(dense.astype(np.float64)), np.abs(pooled.astype(np.float64)), P)
    # fp16 output of an fp32 sum: one fp16 rounding (2^-11 relative) plus the fp32 accumulation
    assert_within_abs_sum(got, ref, absum + np.abs(ref), 2.0**-10, "interaction after a timeout")


def test_interaction_backward_f16_times_out_then_recovers(short_waits):
    dl = short_waits
    B, F, D, P = 2048, 26, 128, 480
    dense, pooled = _inputs(B, F, D, 2)
    rng = np.random.default_rng(3)
    g = (rng.normal(0.0, 1e-2, size=(B, P)) * S).astype(np.float16)
    d_dense, d_pooled, d_g = to_dev(dense), to_dev(pooled), to_dev(g)
    gd = torch.zeros(B, D, dtype=torch.float16, device=dev())
    gp = torch.zeros(B, F, D, dtype=torch.float16, device=dev())
    status = torch.zeros(1, dtype=torch.int32, device=dev())
    dl.dlrm_set_wait_limit(0)
    dl.dlrm_interact_bwd_f16(d_g, d_dense, d_pooled, F, D, B, P, gd, gp, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & dl.DLRM_STATUS_TIMEOUT
    dl.dlrm_set_wait_limit(-1)
    status.zero_()
    dl.dlrm_interact_bwd_f16(d_g, d_dense, d_pooled, F, D, B, P, gd, gp, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    rgd, rgp = oracle.interact_bwd_f16(g, dense, pooled)
    # each result is the exact value rounded once to fp16, up to the fp32 accumulation
    for name, got, ref in (("grad_dense", gd, rgd), ("grad_pooled", gp, rgp)):
        a = got.cpu().numpy().astype(np.float64)
        r = ref.astype(np.float64)
        np.testing.assert_allclose(a, r, rtol=2.0**-9, atol=2.0**-14 * S, err_msg=name)
