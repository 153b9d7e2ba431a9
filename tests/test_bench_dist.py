"""bench.py's multi-rank helpers on world_size 2 gloo ranks (CPU): the max of
the per-rank step times over ranks, the barrier, the environment parsing, and
the reference arm that only rank 0 runs."""

import os
import socket
import traceback

import pytest


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, queue):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import torch.distributed as dist
    dist.init_process_group("gloo")
    try:
        import bench
        r, w, local = bench.dist_env()
        assert (r, w, local) == (rank, world, rank)
        got = bench.reduce_max(1.5 + 10.0 * rank, w)
        bench.barrier(w)
        queue.put((rank, "ok", got))
    except BaseException:
        queue.put((rank, traceback.format_exc(), None))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_barrier():
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = {}
    try:
        for _ in range(2):
            r, msg, v = q.get(timeout=180)
            out[r] = (msg, v)
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.kill()
    for r in range(2):
        assert out[r][0] == "ok", out[r][0]
        assert out[r][1] == 11.5          # every rank sees the slowest rank's time


def test_single_rank_helpers_are_identity(monkeypatch):
    import bench
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench.dist_env() == (0, 1, 0)
    assert bench.reduce_max(3.25, 1) == 3.25
    bench.barrier(1)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    bench.main(["--impl", "reference", "--steps", "1", "--warmup", "3"])
    assert capsys.readouterr().out == ""   # the other ranks exit without work


def test_packed_e2e_buffers_alias_their_parts():
    """The end-to-end loops copy one packed buffer per direction: every part sits at a 256-byte
    aligned offset, in order, and the views the calls take alias exactly its bytes."""
    import torch

    import bench

    offs, tot = bench._pack_layout([5, 256, 257, 0, 12])
    assert offs == [0, 256, 512, 1024, 1024] and tot == 1280
    parts = [("a", torch.arange(7, dtype=torch.int32)), ("b", torch.ones(3, 5, dtype=torch.float16)),
             ("c", torch.full((2, 2), 2.5, dtype=torch.float32))]
    buf, views = bench._packed_views(torch, torch.device("cpu"), parts)
    offs, tot = bench._pack_layout([t.numel() * t.element_size() for _, t in parts])
    assert buf.numel() == tot and buf.dtype == torch.uint8
    for (name, t), o in zip(parts, offs):
        v = views[name]
        assert v.shape == t.shape and v.dtype == t.dtype
        v.copy_(t)
        n = t.numel() * t.element_size()
        assert torch.equal(buf[o:o + n], t.contiguous().view(-1).view(torch.uint8))


def test_roofline_traffic_scales_a_smaller_capture_by_samples():
    """Each committed traffic capture names its batch; the bench scales a capture taken on a
    smaller batch to the launch it reports, by the samples processed."""
    import json
    import os

    import bench

    entries = json.load(open(os.path.join(bench.ROOT, "profiles", "traffic.json")))
    for name, e in entries.items():
        cb = e["captured_batch"]
        assert cb > 0
        got, note = bench.ncu_traffic(name, batch=4 * cb)
        if got is None:   # taken on an older source: the bench reports no traffic for it
            continue
        assert got == 4 * e["dram_bytes_per_launch"] and str(cb) in note
        assert bench.ncu_traffic(name, batch=cb)[0] == e["dram_bytes_per_launch"]
