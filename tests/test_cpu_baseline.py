"""The benchmark's all-cores CPU baseline computes exactly what one oracle call
computes: the oracle's functions run unchanged on disjoint parts of the step
(per table, per block of samples), so every output and every updated table row
is bit-identical to the single call's."""

import numpy as np

import bench
import oracle
from dlrm_embeddings_dot_gb300 import inputs
from dlrm_embeddings_dot_gb300.inputs import Compact


def test_threaded_oracle_step_equals_one_call():
    w = inputs.dlrm_default(B=700, dtype=inputs.F32, alpha=1.2, train=True,
                            rows=np.array([3, 50, 1, 2000] + [40] * 22))
    samples = np.arange(600)
    step = bench.ThreadedOracleStep(w, samples)
    step.run(4)
    got = step.outputs()
    c = Compact(w, samples)
    pooled, _ = oracle.emb_fwd(c.tables, c.row_base, c.F, c.D, c.B, c.indices, c.offsets)
    out = oracle.interact_fwd(c.dense, pooled, w.out_cols)
    gd, gp = oracle.interact_bwd(c.grad_out, c.dense, pooled)
    tables, _, _, _ = oracle.emb_bwd_sgd(c.tables, c.row_base, c.F, c.D, c.B, c.indices, c.offsets, gp, w.lr)
    for name, ref in (("pooled", pooled), ("out", out), ("gd", gd), ("gp", gp), ("tables", tables)):
        assert np.array_equal(got[name].view(np.uint32), np.asarray(ref, np.float32).view(np.uint32)), name
