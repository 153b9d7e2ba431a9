/*
 * dlrm_plan.h -- host-side planning of the hybrid-parallel layout.
 *
 * "DLRM For PyTorch", §Hybrid-parallel multiGPU with all-2-all communication:
 * the embedding tables and the bottom MLP are model parallel, the dot
 * interaction and the layers above it data parallel; one all-to-all turns the
 * pooled embeddings from table-sharded into batch-sharded (and the reverse one
 * brings grad_pooled back to the tables' owners before the sparse update).
 * §Embedding table placement and load balancing gives the placement heuristic.
 *
 * Everything here runs on the host, on host memory, and makes no CUDA call.
 * Readings of the pages fixed by these functions:
 *   - one GPU: every table (and the bottom MLP) on GPU 0;
 *   - N > 1 GPUs: the bottom MLP on GPU 0, the tables on GPUs 1..N-1, at most
 *     ceil(n_tables / (N - 1)) tables per GPU;
 *   - ties: equal table sizes keep table-id order, equal free memory takes
 *     the lower GPU id;
 *   - data-parallel shards are contiguous in sample order, the first
 *     batch mod N ranks taking one extra sample;
 *   - exchange buffers are sample-major: a rank's table-sharded block for
 *     destination d is [B_d][its tables, ascending id][row_elems]; a
 *     receive buffer is the sources' blocks in rank order.
 * Errors: DLRM_ERR_INVALID_ARG for a bad argument (message in
 * dlrm_last_error), DLRM_ERR_NO_FIT when the heuristic's GPU for a table
 * lacks the room (table_device is then undefined).
 */
#ifndef DLRM_GB300_PLAN_H
#define DLRM_GB300_PLAN_H

#include "dlrm.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Place n_tables tables of table_bytes[t] bytes on n_gpus GPUs with
 * gpu_free_bytes[g] free bytes each ("DLRM For PyTorch", §Embedding table
 * placement and load balancing): the largest unplaced table goes to the
 * available GPU with the most unallocated memory; a GPU stops taking tables
 * once it holds the per-GPU cap.  Writes table_device[t] (caller-owned host
 * array of n_tables ints).  The bottom MLP is on GPU 0. */
dlrm_status dlrm_plan_tables(int n_tables, const int64_t* table_bytes, int n_gpus, const int64_t* gpu_free_bytes,
                             int* table_device);

/* First sample and sample count of rank's contiguous data-parallel shard of
 * a batch of `batch` samples over n_ranks ranks (host out-pointers). */
dlrm_status dlrm_batch_shard(int64_t batch, int n_ranks, int rank, int64_t* first, int64_t* count);

/* Element counts and offsets of the forward all-to-all seen from `rank`
 * ("DLRM For PyTorch", §Hybrid-parallel multiGPU with all-2-all
 * communication), for tables placed by table_device[] and rows of row_elems
 * elements (D).  All outputs are caller-owned host arrays: send_counts,
 * send_displs, recv_counts, recv_displs of n_ranks entries each (elements,
 * displacements are exclusive prefix sums), and slot_table of n_tables
 * entries: the global table held by each receive slot (source rank by source
 * rank, ascending table id within a source).  The backward exchange of
 * grad_pooled is the same layout with send and receive swapped. */
dlrm_status dlrm_a2a_layout(int n_tables, const int* table_device, int64_t batch, int n_ranks, int rank,
                            int64_t row_elems, int64_t* send_counts, int64_t* send_displs, int64_t* recv_counts,
                            int64_t* recv_displs, int* slot_table);

#ifdef __cplusplus
}
#endif

#endif
