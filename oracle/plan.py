"""Table placement and the all-to-all layout of the hybrid-parallel scheme,
restated plainly.

Test infrastructure, like the rest of ``oracle/``: only the test suite, the
package smoke check and the benchmark's CPU-baseline leg use it, and it
shares nothing with the library.

Source: "DLRM For PyTorch", §Hybrid-parallel multiGPU with all-2-all
communication and §Embedding table placement and load balancing.  The
embedding tables and the bottom MLP are model parallel; the interaction and
everything above it are data parallel, so one all-to-all turns the pooled
embeddings from table-sharded (each GPU holds its tables' bags for the whole
batch) into batch-sharded (each GPU holds every table's bags for its samples).

Readings where the pages leave a step open:
* With one GPU everything sits on GPU 0 (the heuristic describes the
  multi-GPU case; with one device there is nowhere else to put tables).
* With N > 1 GPUs the tables go to GPUs 1..N-1, so the per-GPU cap is
  ceil(tables / (N - 1)).
* Equal table sizes keep table-id order; equal free memory picks the lowest
  GPU id.
* The data-parallel batch shards are contiguous in sample order; the first
  B mod N ranks take one extra sample.
* Buffers are sample-major: a table-sharded block is [samples][own tables][D]
  with the rank's tables in ascending id; the receive side concatenates the
  sources' blocks in rank order.
"""

from __future__ import annotations

import math


class PlacementError(ValueError):
    """A table does not fit on the GPU the heuristic picked for it."""


def place_tables(table_bytes: list[int], gpu_free_bytes: list[int]) -> tuple[list[int], int]:
    """Device of every table, and the device of the bottom MLP (always 0)."""
    n_gpus = len(gpu_free_bytes)
    n_tables = len(table_bytes)
    if n_gpus < 1:
        raise ValueError("need at least one GPU")
    if n_gpus == 1:
        if sum(table_bytes) > gpu_free_bytes[0]:
            raise PlacementError("the tables do not fit on the only GPU")
        return [0] * n_tables, 0
    # the bottom MLP takes GPU 0, which receives no table
    available = list(range(1, n_gpus))
    max_tables_per_gpu = math.ceil(n_tables / len(available))
    # largest table first
    order = sorted(range(n_tables), key=lambda t: (-table_bytes[t], t))
    free = list(gpu_free_bytes)
    count = [0] * n_gpus
    device = [-1] * n_tables
    for t in order:
        # the available GPU with the most unallocated memory
        best = available[0]
        for g in available[1:]:
            if free[g] > free[best]:
                best = g
        if table_bytes[t] > free[best]:
            raise PlacementError(f"table {t} ({table_bytes[t]} bytes) does not fit on GPU {best} "
                                 f"({free[best]} bytes free)")
        device[t] = best
        free[best] -= table_bytes[t]
        count[best] += 1
        if count[best] == max_tables_per_gpu:
            available.remove(best)
    return device, 0


def batch_shard(B: int, n_ranks: int, rank: int) -> tuple[int, int]:
    """(first sample, sample count) of a rank's contiguous data-parallel shard."""
    base, extra = divmod(B, n_ranks)
    first = rank * base + min(rank, extra)
    return first, base + (1 if rank < extra else 0)


def tables_of(device: list[int], rank: int) -> list[int]:
    return [t for t, g in enumerate(device) if g == rank]


def forward_layout(device: list[int], B: int, n_ranks: int, rank: int, D: int):
    """Element counts and offsets of the forward all-to-all for one rank.

    Rank r sends destination d the rows of d's samples for r's own tables,
    [B_d][n_r][D]; it receives from every source s the rows of its own
    samples for s's tables, [B_r][n_s][D].  Also returns, for each receive
    slot (source-major, then the source's tables in ascending id), the global
    table it holds.
    """
    n_own = len(tables_of(device, rank))
    send_counts, recv_counts, slot_table = [], [], []
    _, my_count = batch_shard(B, n_ranks, rank)
    for other in range(n_ranks):
        _, other_count = batch_shard(B, n_ranks, other)
        send_counts.append(other_count * n_own * D)
        theirs = tables_of(device, other)
        recv_counts.append(my_count * len(theirs) * D)
        slot_table.extend(theirs)
    send_displs = [sum(send_counts[:i]) for i in range(n_ranks)]
    recv_displs = [sum(recv_counts[:i]) for i in range(n_ranks)]
    return send_counts, send_displs, recv_counts, recv_displs, slot_table
