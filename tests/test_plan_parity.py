"""The library's host-side planning calls (include/dlrm_plan.h) against the
placement oracle: identical placements, shards and exchange layouts, and
argument checks.  Host only: no GPU call."""

import math

import numpy as np
import pytest

import dlrm_embeddings_dot_gb300 as dl
from dlrm_embeddings_dot_gb300 import build as libbuild
from oracle import plan


@pytest.fixture(scope="module", autouse=True)
def _lib():
    libbuild.build()
    dl.load()


def _case(rng):
    n_gpus = int(rng.integers(1, 9))
    n_tables = int(rng.integers(0, 40))
    tables = [int(x) for x in rng.integers(0, 10**9, size=n_tables)]
    if rng.random() < 0.3 and n_tables:
        tables = [tables[0]] * n_tables                    # all equal: tie order matters
    scale = max(sum(tables), 1) // max(n_gpus - 1, 1)
    free = [int(x) for x in rng.integers(0, 2 * scale + 2, size=n_gpus)]
    if rng.random() < 0.3 and n_gpus > 2:
        free[1:] = [free[1]] * (n_gpus - 1)                # equal free memory
    return tables, free


def test_placement_matches_oracle_including_failures():
    rng = np.random.default_rng(11)
    fits = nofit = 0
    for _ in range(3000):
        tables, free = _case(rng)
        try:
            want, _ = plan.place_tables(tables, free)
        except plan.PlacementError:
            with pytest.raises(dl.DlrmError) as e:
                dl.dlrm_plan_tables(tables, free)
            assert e.value.code == dl.DLRM_ERR_NO_FIT
            nofit += 1
            continue
        assert dl.dlrm_plan_tables(tables, free) == want
        fits += 1
    assert fits > 500 and nofit > 500


def test_shards_and_layouts_match_oracle():
    rng = np.random.default_rng(12)
    for _ in range(300):
        N = int(rng.integers(1, 9))
        F = int(rng.integers(0, 30))
        dev = [int(x) for x in rng.integers(0, N, size=F)]
        B = int(rng.integers(0, 100))
        D = int(rng.integers(0, 200))
        for r in range(N):
            assert dl.dlrm_batch_shard(B, N, r) == plan.batch_shard(B, N, r)
            got = dl.dlrm_a2a_layout(dev, B, N, r, D)
            assert [list(x) for x in got] == [list(x) for x in plan.forward_layout(dev, B, N, r, D)]


def test_default_tables_on_eight_gpus():
    """The 26 DLRM-default fp32 tables (rows log-uniform in [10, 4e6]) over 8
    GPUs of 280 GB: GPUs 1..7 hold at most ceil(26/7) = 4 tables each."""
    from dlrm_embeddings_dot_gb300 import inputs
    w = inputs.dlrm_default(B=8, dtype=inputs.F32)
    tb = [int(r) * w.D * 4 for r in w.rows]
    dev = dl.dlrm_plan_tables(tb, [280 << 30] * 8)
    assert dev == plan.place_tables(tb, [280 << 30] * 8)[0]
    counts = np.bincount(dev, minlength=8)
    assert counts[0] == 0 and counts.max() <= math.ceil(26 / 7) and counts.sum() == 26


def test_argument_checks():
    with pytest.raises(dl.DlrmError) as e:
        dl.dlrm_plan_tables([1, -2], [10, 10])
    assert e.value.code == dl.DLRM_ERR_INVALID_ARG
    with pytest.raises(dl.DlrmError):
        dl.dlrm_plan_tables([1], [])
    with pytest.raises(dl.DlrmError):
        dl.dlrm_batch_shard(10, 2, 2)
    with pytest.raises(dl.DlrmError):
        dl.dlrm_a2a_layout([0, 3], 10, 2, 0, 4)           # table on a rank that does not exist
    assert dl.dlrm_plan_tables([], [5, 5]) == []
