"""Pins of the placement / all-to-all layout oracle ("DLRM For PyTorch",
§Embedding table placement and load balancing; §Hybrid-parallel multiGPU
with all-2-all communication): hand-worked cases and invariants."""

import math
import os

import numpy as np
import pytest

from oracle import plan

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "placement_hand.txt")


def _ints(s):
    s = s.strip()
    return [int(x) for x in s.split(",")] if s else []


def _golden(kind):
    out = []
    for line in open(GOLDEN):
        line = line.strip()
        if line.startswith(kind + " "):
            out.append([p.strip() for p in line[len(kind) + 1:].split("|")])
    return out


@pytest.mark.parametrize("case", _golden("place"))
def test_hand_worked_placements(case):
    tables, free, want = _ints(case[0]), _ints(case[1]), case[2]
    if want == "NOFIT":
        with pytest.raises(plan.PlacementError):
            plan.place_tables(tables, free)
    else:
        dev, mlp = plan.place_tables(tables, free)
        assert dev == _ints(want) and mlp == 0


@pytest.mark.parametrize("case", _golden("shard"))
def test_hand_worked_shards(case):
    B, N = _ints(case[0].replace(" ", ","))
    want = [tuple(int(x) for x in fc.split(":")) for fc in case[1].split()]
    assert [plan.batch_shard(B, N, r) for r in range(N)] == want


@pytest.mark.parametrize("case", _golden("layout"))
def test_hand_worked_layouts(case):
    head = case[0].split()
    dev, (B, N, D) = _ints(head[0]), [int(x) for x in head[1:]]
    rank = int(case[1])
    got = plan.forward_layout(dev, B, N, rank, D)
    assert list(got) == [_ints(c) for c in case[2:7]]


def _random_case(rng):
    n_gpus = int(rng.integers(1, 7))
    n_tables = int(rng.integers(1, 30))
    tables = [int(x) for x in rng.integers(1, 1000, size=n_tables)]
    if n_gpus == 1:
        free = [int(sum(tables) + rng.integers(0, 10))]
    else:
        cap = math.ceil(n_tables / (n_gpus - 1))
        roomy = int(sum(sorted(tables)[-cap:])) + 1   # any GPU can take its share of the largest tables
        free = [int(rng.integers(0, 100))] + [roomy + int(rng.integers(0, 1000)) for _ in range(n_gpus - 1)]
    return tables, free


def test_invariants_on_random_cases():
    rng = np.random.default_rng(0)
    for _ in range(500):
        tables, free = _random_case(rng)
        dev, _ = plan.place_tables(tables, free)
        n_gpus = len(free)
        assert len(dev) == len(tables)
        if n_gpus == 1:
            assert set(dev) == {0}
            continue
        cap = math.ceil(len(tables) / (n_gpus - 1))
        for g in range(n_gpus):
            mine = [t for t in range(len(tables)) if dev[t] == g]
            if g == 0:
                assert not mine, "GPU 0 holds the bottom MLP and no table"
            assert len(mine) <= cap
            assert sum(tables[t] for t in mine) <= free[g]


def test_layouts_are_consistent_between_ranks():
    """What rank r sends to d is exactly what d expects from r, and every rank
    ends with all F tables of its own samples."""
    rng = np.random.default_rng(1)
    for _ in range(100):
        tables, free = _random_case(rng)
        dev, _ = plan.place_tables(tables, free)
        N, F, D = len(free), len(tables), int(rng.integers(1, 5))
        B = int(rng.integers(0, 50))
        lay = [plan.forward_layout(dev, B, N, r, D) for r in range(N)]
        for r in range(N):
            sc, sd, rc, rd, slots = lay[r]
            assert sorted(slots) == list(range(F))
            assert sum(rc) == plan.batch_shard(B, N, r)[1] * F * D
            for d in range(N):
                assert sc[d] == lay[d][2][r]
            assert sd == list(np.cumsum([0] + sc[:-1])) and rd == list(np.cumsum([0] + rc[:-1]))
