"""CPU-rank simulation of the hybrid-parallel step ("DLRM For PyTorch",
§Hybrid-parallel multiGPU with all-2-all communication; §Embedding table
placement and load balancing) on world_size 2..4 gloo ranks.

Each rank owns the tables that dlrm_plan_tables puts on its GPU (the bottom
MLP, hence the dense rows, on rank 0).  The ranks' per-GPU work is done by
the CPU oracle; what is under test is the library's placement and exchange
layout (dlrm_batch_shard, dlrm_a2a_layout) driving real all_to_all_single
collectives:
  forward   table-sharded pooled [B][own tables][D] -> batch-sharded
            [B_r][F][D] in global table order; dense rows scattered from rank 0
  backward  batch-sharded grad_pooled -> each owner's [B][own tables][D],
            then the owner's sparse SGD on its own tables.
Every stage must equal the single-process oracle bit for bit: pooling,
interaction and the row updates are independent per table and per sample,
and each row's occurrences keep their order.
"""

import os
import socket
import traceback

import numpy as np
import pytest

B, F, D = 37, 7, 8
ROWS = [3, 50, 1000, 7, 200, 20, 5000]


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _workload():
    from dlrm_embeddings_dot_gb300 import inputs
    P = inputs.interaction_width(F, D)
    dense = np.random.default_rng(3).standard_normal((B, D)).astype(np.float32)
    return inputs.make_workload("a2a-sim", B, F, D, inputs.F32, np.array(ROWS), alpha=1.2, dense=dense,
                                out_cols=P, seed=5, pool=(1, 3), with_grad=True)


def _sub(w, tables, mine):
    """Tables, row_base and CSR of the bags of the tables in `mine` (ascending)."""
    rb = np.zeros(len(mine) + 1, dtype=np.int64)
    rb[1:] = np.cumsum(w.rows[mine]) if mine else []
    tabs = np.concatenate([tables[w.row_base[t]:w.row_base[t + 1]] for t in mine]) if mine else \
        np.zeros((0, D), np.float32)
    idx, counts = [], []
    for t in mine:
        lo, hi = int(w.offsets[t * B]), int(w.offsets[(t + 1) * B])
        idx.append(w.indices[lo:hi])
        counts.append(np.diff(w.offsets[t * B:(t + 1) * B + 1]))
    idx = np.concatenate(idx) if mine else np.zeros(0, np.int32)
    off = np.zeros(len(mine) * B + 1, dtype=np.int32)
    if mine:
        off[1:] = np.cumsum(np.concatenate(counts))
    return tabs, rb, idx.astype(np.int32), off


def _rank(rank, world, port, queue):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    import torch
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import dlrm_embeddings_dot_gb300 as dl
        import oracle
        from dlrm_embeddings_dot_gb300 import inputs
        w = _workload()
        P = w.out_cols
        tables = inputs.table_rows(w.table_seed, np.arange(int(w.row_base[-1])), D, inputs.F32)
        # the single-process step
        pooled_full, _ = oracle.emb_fwd(tables, w.row_base, F, D, B, w.indices, w.offsets)
        out_full = oracle.interact_fwd(w.dense, pooled_full, P)
        _, gp_full = oracle.interact_bwd(w.grad_out, w.dense, pooled_full)
        new_full = oracle.emb_bwd_sgd(tables, w.row_base, F, D, B, w.indices, w.offsets, gp_full, w.lr)[0]

        dev = dl.dlrm_plan_tables([r * D * 4 for r in ROWS], [1 << 40] * world)
        mine = [t for t in range(F) if dev[t] == rank]
        owned = [dev.count(s) for s in range(world)]
        first, cnt = dl.dlrm_batch_shard(B, world, rank)
        sc, sd, rc, rd, slots = dl.dlrm_a2a_layout(dev, B, world, rank, D)

        # ---- forward: this rank's tables for the whole batch, then the exchange
        stabs, srb, sidx, soff = _sub(w, tables, mine)
        if mine:
            pooled_mine, status = oracle.emb_fwd(stabs, srb, len(mine), D, B, sidx, soff)
            assert status == 0
        else:
            pooled_mine = np.zeros((B, 0, D), np.float32)
        send = torch.from_numpy(np.ascontiguousarray(pooled_mine).reshape(-1))
        recv = torch.empty(sum(rc))
        dist.all_to_all_single(recv, send, output_split_sizes=rc, input_split_sizes=sc)
        local = np.empty((cnt, F, D), np.float32)
        k = 0
        for s in range(world):
            block = recv[rd[s]:rd[s] + rc[s]].numpy().reshape(cnt, owned[s], D)
            local[:, slots[k:k + owned[s]], :] = block
            k += owned[s]
        assert np.array_equal(local, pooled_full[first:first + cnt]), "pooled shard"

        # ---- dense rows: the bottom MLP's output leaves rank 0 by shard
        if rank == 0:
            dsend = torch.from_numpy(np.ascontiguousarray(w.dense).reshape(-1))
            dsc = [dl.dlrm_batch_shard(B, world, d)[1] * D for d in range(world)]
        else:
            dsend, dsc = torch.empty(0), [0] * world
        drc = [cnt * D if s == 0 else 0 for s in range(world)]
        drecv = torch.empty(cnt * D)
        dist.all_to_all_single(drecv, dsend, output_split_sizes=drc, input_split_sizes=dsc)
        dense_local = drecv.numpy().reshape(cnt, D)
        assert np.array_equal(dense_local, w.dense[first:first + cnt])
        out_local = oracle.interact_fwd(dense_local, local, P)
        assert np.array_equal(out_local, out_full[first:first + cnt]), "interaction shard"

        # ---- backward: grad_pooled of this shard back to the tables' owners
        _, gp = oracle.interact_bwd(w.grad_out[first:first + cnt], dense_local, local)
        assert np.array_equal(gp, gp_full[first:first + cnt])
        parts, k = [], 0
        for s in range(world):
            parts.append(np.ascontiguousarray(gp[:, slots[k:k + owned[s]], :]).reshape(-1))
            k += owned[s]
        send2 = torch.from_numpy(np.concatenate(parts))
        recv2 = torch.empty(sum(sc))
        dist.all_to_all_single(recv2, send2, output_split_sizes=sc, input_split_sizes=rc)
        grad_mine = recv2.numpy().reshape(B, len(mine), D)
        assert np.array_equal(grad_mine, gp_full[:, mine, :]), "grad_pooled at the owner"
        if mine:
            new_mine = oracle.emb_bwd_sgd(stabs, srb, len(mine), D, B, sidx, soff, grad_mine, w.lr)[0]
            want = np.concatenate([new_full[w.row_base[t]:w.row_base[t + 1]] for t in mine])
            assert np.array_equal(new_mine, want), "updated rows"
        queue.put((rank, "ok", mine))
    except BaseException:
        queue.put((rank, traceback.format_exc(), None))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3, 4])
def test_hybrid_parallel_step_matches_single_process(world):
    import multiprocessing as mp
    from dlrm_embeddings_dot_gb300 import build as libbuild
    libbuild.build()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = {}
    try:
        for _ in range(world):
            rank, msg, mine = q.get(timeout=240)
            results[rank] = (msg, mine)
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.kill()
    for r in range(world):
        assert results[r][0] == "ok", f"rank {r}:\n{results[r][0]}"
    owned = sorted(t for r in range(world) for t in results[r][1])
    assert owned == list(range(F)) and results[0][1] == []   # every table once, none on rank 0
