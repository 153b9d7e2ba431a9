// reg_gather.cuh -- a warp's view of one sample's bags for the one-warp-per-
// sample kernels that read table rows straight into shared memory (the
// one-pass forward and the backward that re-gathers the pooled rows).
//
// Lane t < F owns bag t of a sample: its CSR bounds (clamped into [0, nnz],
// malformed lists flagged DLRM_STATUS_BAD_OFFSETS, as in the lookup) and its
// source: a table row (32 bits: 2^32 rows of 512 bytes would not fit in
// memory), kRowZero (empty bag or rejected index) or kRowMulti (several
// indices).  gather() fills rows 1..F of a [R][32] float4 buffer: lane t
// copies its single-index bag's row with one 512-byte bulk copy counted on the
// warp's mbarrier; zero rows and bags of several indices (summed in fp32 in
// bag order, exactly as the lookup sums them) are stored by the lanes, each
// its own 16-byte column.  The caller adds its other copies, then
// __syncwarp() and one arrival.
#pragma once

#include "common.cuh"
#include "tcgen05.cuh"

namespace dlrm {

struct RegGather {
    const float* tables;
    const int64_t* row_base;
    const int32_t* indices;
    const int32_t* offsets;
    int64_t nnz;
    bool hash;
};

template <int F, int D>
struct BagLanes {
    static constexpr uint32_t kRowZero = 0xffffffffu, kRowMulti = 0xfffffffeu;
    RegGather ga;
    int B, lane;
    int64_t tbase, tn;   // lane t < F: table t's first row and row count
    uint32_t* status;

    __device__ __forceinline__ BagLanes(const RegGather& g, int B_, int lane_, uint32_t* st)
        : ga(g), B(B_), lane(lane_), tbase(0), tn(0), status(st)
    {
        if (lane < F) {
            tbase = ga.row_base[lane];
            tn = ga.row_base[lane + 1] - tbase;
        }
    }

    __device__ __forceinline__ void load_bounds(int64_t smp, int& a, int& e) const
    {
        a = e = 0;
        if (lane < F && smp < B) {
            a = ldg_early_s32(ga.offsets + (int64_t)lane * B + smp);
            e = ldg_early_s32(ga.offsets + (int64_t)lane * B + smp + 1);
        }
    }

    __device__ __forceinline__ void clamp(int& a, int& e) const
    {
        int64_t x = a, y = e;
        if (x < 0 || y < x || y > ga.nnz) {
            set_status(status, DLRM_STATUS_BAD_OFFSETS);
            x = x < 0 ? 0 : (x > ga.nnz ? ga.nnz : x);
            y = y < x ? x : (y > ga.nnz ? ga.nnz : y);
        }
        a = (int)x;
        e = (int)y;
    }

    // the index of a single-index bag, loaded where it is written (a sample ahead)
    __device__ __forceinline__ int early_index(int a, int e) const
    {
        return (lane < F && e - a == 1) ? ldg_early_s32(ga.indices + a) : 0;
    }

    __device__ __forceinline__ uint32_t resolve(int a, int e, int idx) const
    {
        if (lane >= F || e - a == 0) return kRowZero;
        if (e - a > 1) return kRowMulti;
        int64_t i = idx;
        if (ga.hash && tn > 0) {
            i %= tn;
            if (i < 0) i += tn;
        } else if (ga.hash || i < 0 || i >= tn || tbase + i >= (int64_t)kRowMulti) {
            set_status(status, DLRM_STATUS_OOB_INDEX);
            return kRowZero;
        }
        return (uint32_t)(tbase + i);
    }

    // kCopyAsync: every lane copies its 16-byte column of each single-index row
    // with cp.async (completion: cp.async.wait_group by the same lane, which
    // reads only the columns it copied) instead of lane t's bulk copy of row t.
    // kMultiU: positions of a several-index bag in flight (indices, then rows),
    // added in bag order; few enough that the caller's live registers are not
    // spilled
    template <bool kCopyAsync = false, int kMultiU = 4>
    __device__ __forceinline__ void gather(float4* buf, uint32_t src_row, int a, int e, uint64_t* bar) const
    {
        if constexpr (kCopyAsync) {
#pragma unroll
            for (int t = 0; t < F; ++t) {
                const uint32_t src = __shfl_sync(0xffffffffu, src_row, t);
                if (src < kRowMulti) {
                    const uint32_t d = (uint32_t)__cvta_generic_to_shared(buf + (t + 1) * kWarp + lane);
                    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d),
                                 "l"(ga.tables + (size_t)src * D + 4 * lane)
                                 : "memory");
                }
            }
            asm volatile("cp.async.commit_group;" ::: "memory");
        } else if (lane < F && src_row < kRowMulti) {
            tc::mbar_expect_tx_only(bar, D * 4);
            tc::bulk_g2s(buf + (lane + 1) * kWarp, ga.tables + (size_t)src_row * D, D * 4, bar);
        }
        for (uint32_t zero = __ballot_sync(0xffffffffu, lane < F && src_row == kRowZero); zero; zero &= zero - 1)
            buf[__ffs(zero) * kWarp + lane] = make_float4(0.f, 0.f, 0.f, 0.f);
        for (uint32_t multi = __ballot_sync(0xffffffffu, src_row == kRowMulti); multi; multi &= multi - 1) {
            const int t = __ffs(multi) - 1;
            const int s1 = __shfl_sync(0xffffffffu, a, t), e1 = __shfl_sync(0xffffffffu, e, t);
            const int64_t base = __shfl_sync(0xffffffffu, tbase, t), n = __shfl_sync(0xffffffffu, tn, t);
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int p0 = s1; p0 < e1; p0 += kMultiU) {
                int idx[kMultiU];
#pragma unroll
                for (int u = 0; u < kMultiU; ++u) idx[u] = p0 + u < e1 ? __ldg(ga.indices + p0 + u) : 0;
                uint32_t row[kMultiU];   // kRowZero: skipped or past the bag
                float4 r[kMultiU];
#pragma unroll
                for (int u = 0; u < kMultiU; ++u) {
                    int64_t i = idx[u];
                    row[u] = kRowZero;
                    if (p0 + u < e1) {
                        if (ga.hash && n > 0) {
                            i %= n;
                            if (i < 0) i += n;
                            row[u] = (uint32_t)(base + i);
                        } else if (ga.hash || i < 0 || i >= n) {
                            set_status(status, DLRM_STATUS_OOB_INDEX);
                        } else {
                            row[u] = (uint32_t)(base + i);
                        }
                    }
                    r[u] = row[u] != kRowZero ? u4_as_f4(ldg_nc_l1_v4(ga.tables + (size_t)row[u] * D + 4 * lane))
                                              : make_float4(0.f, 0.f, 0.f, 0.f);
                }
#pragma unroll
                for (int u = 0; u < kMultiU; ++u)
                    if (row[u] != kRowZero) {
                        acc.x += r[u].x;
                        acc.y += r[u].y;
                        acc.z += r[u].z;
                        acc.w += r[u].w;
                    }
            }
            buf[(t + 1) * kWarp + lane] = acc;
        }
    }
};

}  // namespace dlrm
