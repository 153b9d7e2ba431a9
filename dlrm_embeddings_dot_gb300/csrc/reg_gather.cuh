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
    // kMultiU: rows of the several-index bags in flight in registers, few
    // enough that the caller's live registers are not spilled; kRing > 0: in
    // flight through kRing rows of shared staging (ring: kRing x 32 float4,
    // free while gather runs) instead, which costs no registers.
    template <bool kCopyAsync = false, int kMultiU = 4, int kRing = 0>
    __device__ __forceinline__ void gather(float4* buf, uint32_t src_row, int a, int e, uint64_t* bar,
                                           float4* ring = nullptr) const
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
        // Bags of several indices: their positions form one list in bag order
        // (lane t < F holds bag t's count).  Each lane resolves one of 32
        // positions at a time (coalesced index loads), then the warp adds the
        // rows kMultiU at a time, each bag's in position order from zero in
        // fp32, and stores a bag's sum into its buffer row when the next bag
        // begins.  A row waits for one index load, not for the bags before it.
        const int cnt = (lane < F && src_row == kRowMulti) ? e - a : 0;
        if (!__any_sync(0xffffffffu, cnt > 0)) return;
        int incl = cnt;
#pragma unroll
        for (int o = 1; o < kWarp; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        const int excl = incl - cnt;
        const int total = __shfl_sync(0xffffffffu, incl, kWarp - 1);
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        int cur = -1;   // bag being summed (warp-uniform)
        // position q0 + lane: its bag (the last lane whose list offset is at
        // most the position) and its table row (kRowZero: skipped or past the list)
        auto locate = [&](int q0, int& k, uint32_t& row) {
            const int q = q0 + lane;
            k = 0;
#pragma unroll
            for (int step = kWarp / 2; step > 0; step >>= 1)
                if (__shfl_sync(0xffffffffu, excl, k + step) <= q) k += step;
            const int pos = __shfl_sync(0xffffffffu, a, k) + (q - __shfl_sync(0xffffffffu, excl, k));
            const int64_t base = __shfl_sync(0xffffffffu, tbase, k), n = __shfl_sync(0xffffffffu, tn, k);
            row = kRowZero;
            if (q < total) {
                int64_t i = __ldg(ga.indices + pos);
                if (ga.hash && n > 0) {
                    i %= n;
                    if (i < 0) i += n;
                    row = (uint32_t)(base + i);
                } else if (ga.hash || i < 0 || i >= n) {
                    set_status(status, DLRM_STATUS_OOB_INDEX);
                } else {
                    row = (uint32_t)(base + i);
                }
            }
        };
        auto add = [&](int kj, uint32_t rowj, const float4& v) {
            if (kj != cur) {
                if (cur >= 0) buf[(cur + 1) * kWarp + lane] = acc;
                acc = make_float4(0.f, 0.f, 0.f, 0.f);
                cur = kj;
            }
            if (rowj != kRowZero) {
                acc.x += v.x;
                acc.y += v.y;
                acc.z += v.z;
                acc.w += v.w;
            }
        };
        if constexpr (kRing > 0) {
            // Rows through a ring of kRing staging rows: lane l copies column l
            // of position j's row into slot j % kRing, one commit group per
            // position (empty past the list), so that waiting for all but the
            // kRing - 1 newest groups completes position j, and reads it back.
            // Every slot access is by the lane that owns the column, so no
            // other lane is involved; a slot is refilled only after the lane's
            // read of it was issued, and the copy writes it only once its
            // global load returns.  The positions stream across chunks of 32:
            // the next chunk's indices are resolved while this chunk's rows
            // are in flight.
            static_assert(kRing <= kWarp, "the ring reaches at most one chunk ahead");
            int kc, kn = 0;
            uint32_t rc, rn = kRowZero;
            locate(0, kc, rc);
            auto issue = [&](int j, int c0) {   // c0: first position of the current chunk
                const bool next = j >= c0 + kWarp;
                const uint32_t rowj = __shfl_sync(0xffffffffu, next ? rn : rc, j & (kWarp - 1));
                if (j < total && rowj != kRowZero) {
                    const uint32_t d = (uint32_t)__cvta_generic_to_shared(ring + (j % kRing) * kWarp + lane);
                    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d),
                                 "l"(ga.tables + (size_t)rowj * D + 4 * lane)
                                 : "memory");
                }
                asm volatile("cp.async.commit_group;" ::: "memory");
            };
#pragma unroll
            for (int j = 0; j < kRing; ++j) issue(j, 0);
            for (int c0 = 0; c0 < total; c0 += kWarp) {
                if (c0 + kWarp < total) locate(c0 + kWarp, kn, rn);
                const int m = total - c0 < kWarp ? total - c0 : kWarp;
                for (int jj = 0; jj < m; ++jj) {
                    asm volatile("cp.async.wait_group %0;" ::"n"(kRing - 1) : "memory");
                    const float4 v = ring[((c0 + jj) % kRing) * kWarp + lane];
                    add(__shfl_sync(0xffffffffu, kc, jj), __shfl_sync(0xffffffffu, rc, jj), v);
                    issue(c0 + jj + kRing, c0);
                }
                kc = kn;
                rc = rn;
            }
        } else {
            for (int q0 = 0; q0 < total; q0 += kWarp) {
                int k;
                uint32_t row;
                locate(q0, k, row);
                const int m = total - q0 < kWarp ? total - q0 : kWarp;
                for (int j0 = 0; j0 < m; j0 += kMultiU) {
                    uint32_t rj[kMultiU];
                    float4 r[kMultiU];
#pragma unroll
                    for (int u = 0; u < kMultiU; ++u) {
                        rj[u] = __shfl_sync(0xffffffffu, row, (j0 + u) & (kWarp - 1));
                        r[u] = (j0 + u < m && rj[u] != kRowZero)
                                   ? u4_as_f4(ldg_nc_l1_v4(ga.tables + (size_t)rj[u] * D + 4 * lane))
                                   : make_float4(0.f, 0.f, 0.f, 0.f);
                    }
#pragma unroll
                    for (int u = 0; u < kMultiU; ++u) {
                        const int kj = __shfl_sync(0xffffffffu, k, (j0 + u) & (kWarp - 1));
                        if (j0 + u >= m) break;
                        add(kj, rj[u], r[u]);
                    }
                }
            }
        }
        buf[(cur + 1) * kWarp + lane] = acc;
    }
};

}  // namespace dlrm
