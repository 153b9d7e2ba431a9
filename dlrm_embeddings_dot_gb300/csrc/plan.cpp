// plan.cpp -- host-side placement of embedding tables and the all-to-all
// layout of the hybrid-parallel scheme ("DLRM For PyTorch", §Hybrid-parallel
// multiGPU with all-2-all communication; §Embedding table placement and load
// balancing).  No CUDA call; the readings of the pages are listed in
// include/dlrm_plan.h.
#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <vector>

#include "dlrm_plan.h"

namespace dlrm {
void set_error(const char* fmt, ...);
void clear_error();
}  // namespace dlrm

using namespace dlrm;

namespace {

dlrm_status plan_fail(dlrm_status code, const char* msg)
{
    set_error("%s", msg);
    return code;
}

void shard(int64_t batch, int n, int r, int64_t& first, int64_t& count)
{
    const int64_t base = batch / n, extra = batch % n;
    first = (int64_t)r * base + (r < extra ? r : extra);
    count = base + (r < extra ? 1 : 0);
}

}  // namespace

extern "C" dlrm_status dlrm_plan_tables(int n_tables, const int64_t* table_bytes, int n_gpus,
                                        const int64_t* gpu_free_bytes, int* table_device)
{
    clear_error();
    if (n_tables < 0 || n_gpus < 1) return plan_fail(DLRM_ERR_INVALID_ARG, "dlrm_plan_tables: need n_tables >= 0, n_gpus >= 1");
    if (!gpu_free_bytes || (n_tables > 0 && (!table_bytes || !table_device)))
        return plan_fail(DLRM_ERR_INVALID_ARG, "dlrm_plan_tables: null host pointer");
    for (int t = 0; t < n_tables; ++t)
        if (table_bytes[t] < 0) return plan_fail(DLRM_ERR_INVALID_ARG, "dlrm_plan_tables: negative table size");
    for (int g = 0; g < n_gpus; ++g)
        if (gpu_free_bytes[g] < 0) return plan_fail(DLRM_ERR_INVALID_ARG, "dlrm_plan_tables: negative free memory");
    if (n_gpus == 1) {   // one device holds everything
        int64_t total = 0;
        for (int t = 0; t < n_tables; ++t) {
            total += table_bytes[t];
            table_device[t] = 0;
        }
        if (total > gpu_free_bytes[0])
            return plan_fail(DLRM_ERR_NO_FIT, "dlrm_plan_tables: the tables do not fit on the only GPU");
        return DLRM_OK;
    }
    // GPU 0 runs the bottom MLP; GPUs 1..n-1 take the tables, at most `cap` each.
    const int table_gpus = n_gpus - 1;
    const int cap = (n_tables + table_gpus - 1) / table_gpus;
    std::vector<int> order(n_tables);
    for (int t = 0; t < n_tables; ++t) order[t] = t;
    std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return table_bytes[a] > table_bytes[b]; });
    std::vector<int64_t> free_bytes(gpu_free_bytes, gpu_free_bytes + n_gpus);
    std::vector<int> held(n_gpus, 0);
    std::vector<char> open(n_gpus, 1);
    open[0] = 0;
    for (int t : order) {
        int best = -1;
        for (int g = 1; g < n_gpus; ++g)
            if (open[g] && (best < 0 || free_bytes[g] > free_bytes[best])) best = g;
        if (best < 0) return plan_fail(DLRM_ERR_INVALID_ARG, "dlrm_plan_tables: no GPU left (internal)");
        if (table_bytes[t] > free_bytes[best]) {
            set_error("dlrm_plan_tables: table %d (%lld bytes) does not fit on GPU %d (%lld bytes free)", t,
                      (long long)table_bytes[t], best, (long long)free_bytes[best]);
            return DLRM_ERR_NO_FIT;
        }
        table_device[t] = best;
        free_bytes[best] -= table_bytes[t];
        if (++held[best] == cap) open[best] = 0;
    }
    return DLRM_OK;
}

extern "C" dlrm_status dlrm_batch_shard(int64_t batch, int n_ranks, int rank, int64_t* first, int64_t* count)
{
    clear_error();
    if (batch < 0 || n_ranks < 1 || rank < 0 || rank >= n_ranks || !first || !count)
        return plan_fail(DLRM_ERR_INVALID_ARG, "dlrm_batch_shard: need batch >= 0, 0 <= rank < n_ranks, outputs");
    shard(batch, n_ranks, rank, *first, *count);
    return DLRM_OK;
}

extern "C" dlrm_status dlrm_a2a_layout(int n_tables, const int* table_device, int64_t batch, int n_ranks, int rank,
                                       int64_t row_elems, int64_t* send_counts, int64_t* send_displs,
                                       int64_t* recv_counts, int64_t* recv_displs, int* slot_table)
{
    clear_error();
    if (n_tables < 0 || batch < 0 || n_ranks < 1 || rank < 0 || rank >= n_ranks || row_elems < 0)
        return plan_fail(DLRM_ERR_INVALID_ARG, "dlrm_a2a_layout: bad sizes or rank");
    if (!send_counts || !send_displs || !recv_counts || !recv_displs || (n_tables > 0 && (!table_device || !slot_table)))
        return plan_fail(DLRM_ERR_INVALID_ARG, "dlrm_a2a_layout: null host pointer");
    std::vector<int64_t> owned(n_ranks, 0);
    for (int t = 0; t < n_tables; ++t) {
        if (table_device[t] < 0 || table_device[t] >= n_ranks)
            return plan_fail(DLRM_ERR_INVALID_ARG, "dlrm_a2a_layout: table_device out of range");
        ++owned[table_device[t]];
    }
    int64_t my_first, my_count;
    shard(batch, n_ranks, rank, my_first, my_count);
    int64_t soff = 0, roff = 0;
    int slot = 0;
    for (int r = 0; r < n_ranks; ++r) {
        int64_t first, count;
        shard(batch, n_ranks, r, first, count);
        send_counts[r] = count * owned[rank] * row_elems;
        send_displs[r] = soff;
        soff += send_counts[r];
        recv_counts[r] = my_count * owned[r] * row_elems;
        recv_displs[r] = roff;
        roff += recv_counts[r];
        for (int t = 0; t < n_tables; ++t)
            if (table_device[t] == r) slot_table[slot++] = t;
    }
    return DLRM_OK;
}
