// interact_tc.cu -- dot interaction on the 5th-generation tensor cores
// (tcgen05) for fp16 inputs with fp32 accumulation ("DLRM For PyTorch",
// §Model architecture; --interaction_op cuda_dot).
//
// Per sample, Z = [d; e_0 .. e_{F-1}] and the output needs z_i . z_j for
// i > j.  Four samples form one M = 128 tile: sample s's F embedding rows sit
// at rows 32s .. 32s+F-1, so the 128 x 128 product of the tile with itself
// holds each sample's E E^T in a 32 x 32 diagonal block.  Rows F..31 of a
// slot may hold anything: every product they enter is left unread.  The
// dense rows of the four samples are appended as B rows 128..131 (rows
// 132..143 zero), so one tcgen05.mma of M = 128, N = 144 per 16-wide K step
// also yields every e_r . d.  The 75 % of the product outside the diagonal
// blocks is wasted work the tensor pipe absorbs easily: this path is bound by
// HBM, not by tensor throughput.
//
// Data movement: TMA (cp.async.bulk.tensor) loads, per tile and per 64-wide K
// block, one 3-D box {64, 32, 4} of the pooled tensor viewed as [B][F][D]
// (rows F..31 of each sample fall outside the tensor and arrive as zeros) and
// one 2-D box {64, 4} of the dense tensor, both in the 128-byte swizzled
// K-major layout the MMA descriptors expect.  A persistent CTA per SM runs a
// warp-specialised pipeline:
//   warp 0      TMA producer over an NS-stage shared-memory ring
//   warp 1      TMEM allocation + single-thread MMA issue, commits to mbarriers
//   warps 2..5  epilogue: tcgen05.ld of the accumulator (TMEM lane quarter q
//               = warp % 4 holds sample q of the tile), triangle extraction
//               into a shared output row, coalesced 16-byte stores.
// Fused variant (dlrm_emb_interact_fwd, inference): each sample slot of a
// tile is filled by one gather warp straight from the table, so the pooled
// tensor never goes to HBM.  Twelve gather warps (warp 0 and warps 6..16, in
// teams of four) fill three tiles at once with 16-byte register loads, eight
// in flight per lane: a table row is only 256 bytes, and the TMA engine's
// rate for such small row gathers (tile::gather4) is several times below
// what the warps reach.  (At 64K: two teams with 13 loads in flight 0.1169
// ms, three with 8 0.1102, four with 8 0.1113; 10 or more with three teams
// spill.)
// Two TMEM accumulators (2 x 256 columns) let the MMA of tile i+1 overlap the
// epilogue of tile i.  Every mbarrier wait is bounded; on timeout the kernel
// sets DLRM_STATUS_TIMEOUT, drains what it issued, frees TMEM and returns.
#include <cuda.h>

#include "interact_tc.cuh"
#include "tcgen05.cuh"

namespace dlrm {
namespace {

using namespace tc;

constexpr int kGroup = 4;                         // samples per tile
constexpr int kSlot = 32;                         // rows per sample (F <= 32)
constexpr int kM = kGroup * kSlot;                // 128
constexpr int kDenseRows = 16;                    // B rows 128..143
constexpr int kN = kM + kDenseRows;               // 144
constexpr int kKB = 64;                           // fp16 elements per 128-byte row
constexpr int kEBytes = kM * 128;                 // 16 KB
constexpr int kDBytes = kDenseRows * 128;         // 2 KB
constexpr int kKBlockBytes = kEBytes + kDBytes;   // 18 KB (multiple of 1 KB)
constexpr int kTmemCols = 512;
constexpr int kAccStride = 256;
constexpr int kThreads = 192;
constexpr int kTeams = 3;                         // fused: tiles gathered at once, four warps each
constexpr int kThreadsFused = (5 + kGroup * kTeams) * 32;   // + gather warps 6.. (warp 0 gathers too)
constexpr int kGatherU = 8;                       // fused: 16-byte row loads in flight per lane
constexpr int kMaxStages = 8;
constexpr int kFusedStages = 4;
constexpr int kSqRow = 17;                        // words per row of the epilogue's product square
constexpr int kSmemLimit = 232448;                // 227 KB opt-in per block

// instruction descriptor, kind::f16: D = f32, A = B = f16, both K-major, N, M
constexpr uint32_t kIdesc = (1u << 4) | ((uint32_t)(kN >> 3) << 17) | ((uint32_t)(kM >> 4) << 24);

struct Layout {
    int stage_bytes, ns, sq_bytes, tri_bytes;
    size_t smem;
};

__host__ __device__ inline Layout make_layout(int KH, int P, int ns)
{
    Layout L;
    L.stage_bytes = KH * kKBlockBytes;
    L.ns = ns;
    L.sq_bytes = kGroup * kSlot * kSqRow * 4;
    L.tri_bytes = (kSlot * (kSlot + 1) / 2 + 7) / 8 * 16;
    L.smem = 1024 + (size_t)ns * L.stage_bytes + L.sq_bytes + L.tri_bytes + (2 * ns + 4) * 8 + 16;
    (void)P;
    return L;
}

// Operands of the fused lookup (kFused): the joint fp16 table and the CSR lists.
struct GatherArgs {
    const __half* tables;
    const int64_t* row_base;
    const int32_t* indices;
    const int32_t* offsets;
    int64_t nnz;
    bool hash;
};

// kCpr: 16-byte chunks per table row when fixed at compile time (fused
// gather, D = 64, 128, 256), else 0.
template <bool kFused, int kCpr>
__global__ void __launch_bounds__(kFused ? kThreadsFused : kThreads, 1)
interact_tc_kernel(const __grid_constant__ CUtensorMap map_pooled,
                   const __grid_constant__ CUtensorMap map_dense,
                   const __half* __restrict__ dense,
                   __half* __restrict__ out, int F, int D, int B, int P, int KH, int NS,
                   uint32_t* status, GatherArgs ga, long long wait_cycles)
{
    pdl_wait();
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    const Layout L = make_layout(KH, P, NS);
    uint8_t* stages = smem;
    // epilogue: per sample a 32 x kSqRow-word square of its products as
    // halves, and the triangle's offsets into it in output order
    uint32_t* square = reinterpret_cast<uint32_t*>(smem + (size_t)NS * L.stage_bytes);
    uint16_t* tri = reinterpret_cast<uint16_t*>(square + L.sq_bytes / 4);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)NS * L.stage_bytes + L.sq_bytes + L.tri_bytes);
    uint64_t* empty = full + NS;
    uint64_t* tfull = empty + NS;
    uint64_t* tempty = tfull + 2;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(tempty + 2);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
    const int nthreads = kFused ? kThreadsFused : kThreads;

    const int warp = threadIdx.x / kWarp;
    const int lane = threadIdx.x % kWarp;
    const int ntiles = (B + kGroup - 1) / kGroup;
    const int W = D + F * (F + 1) / 2;

    if (threadIdx.x == 0) {
        for (int i = 0; i < NS; ++i) {
            mbar_init(&full[i], kFused ? kGroup : 1);   // fused: one arrive per gather warp of the tile
            mbar_init(&empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&tfull[i], 1);
            mbar_init(&tempty[i], kGroup);
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    // B rows 132..143 (dense rows 4..15) are never written by TMA: zero them once.
    for (int s = 0; s < NS; ++s)
        for (int kb = 0; kb < KH; ++kb) {
            uint4* z = reinterpret_cast<uint4*>(stages + (size_t)s * L.stage_bytes + kb * kKBlockBytes +
                                                kEBytes + kGroup * 128);
            for (int x = threadIdx.x; x < (kDenseRows - kGroup) * 128 / 16; x += nthreads)
                z[x] = make_uint4(0, 0, 0, 0);
        }
    // Output pair k = i (i + 1) / 2 + j (0 <= j <= i < F) sits at halfword
    // i * 2 kSqRow + j of the square; tri[k] holds that offset, 0xffff (a
    // zero half) past the end, up to a multiple of 8 pairs.
    const int T = F * (F + 1) / 2;
    const int T8 = (T + 7) / 8 * 8;
    for (int k = threadIdx.x; k < T8; k += nthreads) {
        uint16_t off = 0xffffu;
        if (k < T) {
            int i = 0;
            while ((i + 1) * (i + 2) / 2 <= k) ++i;
            off = (uint16_t)(i * 2 * kSqRow + (k - i * (i + 1) / 2));
        }
        tri[k] = off;
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_holder)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;

    if (warp == 0 || warp >= 6) {
        if constexpr (!kFused) {
            if (lane == 0) {
                // ------------------------------------------------ TMA producer
                int it = 0;
                for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++it) {
                    const int stage = it % NS;
                    const uint32_t ph = (uint32_t)(it / NS) & 1u;
                    if (!mbar_wait(&empty[stage], ph ^ 1u, abort_flag, wait_cycles)) break;
                    uint8_t* sb = stages + (size_t)stage * L.stage_bytes;
                    mbar_expect_tx(&full[stage], (uint32_t)KH * (kEBytes + kGroup * 128));
                    for (int kb = 0; kb < KH; ++kb) {
                        tma_load_3d(sb + kb * kKBlockBytes, &map_pooled, kb * kKB, 0, tile * kGroup, &full[stage]);
                        tma_load_2d(sb + kb * kKBlockBytes + kEBytes, &map_dense, kb * kKB, tile * kGroup,
                                    &full[stage]);
                    }
                }
                if (*abort_flag) {   // let the copies already issued land before the CTA exits
                    for (int j = (it > NS ? it - NS : 0); j < it; ++j)
                        mbar_drain(&full[j % NS], (uint32_t)(j / NS) & 1u);
                }
            }
        } else {
            // ------------------------------------ gather warps
            // Warp gi (warp 0, then warps 6..) fills slot sm = gi % 4 of the
            // tiles of team gi / 4: tiles team, team + kTeams, ... of this CTA.
            // Lane t < F owns bag (t, b) of the slot's sample b.  Offsets are
            // read two tiles ahead and the index one tile ahead, so each tile
            // costs the warp one memory round trip: the table rows (16 lanes
            // per 256-byte row, 16-byte loads into registers) are in flight
            // before the warp waits for the stage, then stored swizzled.
            const int gi = warp == 0 ? 0 : warp - 5;
            const int team = gi / kGroup, sm = gi % kGroup;
            const int cpr = D / 8;                        // 16-byte chunks per row
            const int nchunks = F * cpr;
            int64_t tbase = 0, tn = 0;                    // lane t < F: table t's first row and row count
            if (lane < F) {
                tbase = ga.row_base[lane];
                tn = ga.row_base[lane + 1] - tbase;
            }
            const int64_t tstride = (int64_t)kTeams * gridDim.x;
            auto load_bounds = [&](int64_t tile, int& s0, int& e0) {
                s0 = e0 = 0;
                const int64_t b = tile * kGroup + sm;
                if (lane < F && tile < ntiles && b < B) {
                    s0 = ldg_early_s32(ga.offsets + (int64_t)lane * B + b);
                    e0 = ldg_early_s32(ga.offsets + (int64_t)lane * B + b + 1);
                }
            };
            auto clamp_bounds = [&](int& s0, int& e0) {   // into [0, nnz], flagging malformed lists
                int64_t a = s0, z = e0;
                if (a < 0 || z < a || z > ga.nnz) {
                    set_status(status, DLRM_STATUS_BAD_OFFSETS);
                    a = a < 0 ? 0 : (a > ga.nnz ? ga.nnz : a);
                    z = z < a ? a : (z > ga.nnz ? ga.nnz : z);
                }
                s0 = (int)a;
                e0 = (int)z;
            };
            // bag -> source: a table row (32 bits: a joint table of 2^32 rows of
            // at least 128 bytes would not fit in memory), kRowZero (empty bag,
            // rejected index) or kRowMulti (several indices)
            constexpr uint32_t kRowZero = 0xffffffffu, kRowMulti = 0xfffffffeu;
            auto resolve = [&](int a, int z, int idx) -> uint32_t {
                if (lane >= F || z - a == 0) return kRowZero;
                if (z - a > 1) return kRowMulti;
                int64_t i = idx;
                if (ga.hash && tn > 0) {
                    i %= tn;
                    if (i < 0) i += tn;
                } else if (ga.hash || i < 0 || i >= tn || tbase + i >= (int64_t)kRowMulti) {
                    set_status(status, DLRM_STATUS_OOB_INDEX);
                    return kRowZero;
                }
                return (uint32_t)(tbase + i);
            };
            // chunk k of this lane: row e of the slot, 16-byte column c.  With
            // 32 % cpr == 0 (D = 64, 128, 256) the column is fixed per lane.
            const int Dr = kCpr > 0 ? 8 * kCpr : D;
            auto chunk_of = [&](int k, int& e, int& c) {
                if constexpr (kCpr > 0 && kWarp % (kCpr > 0 ? kCpr : 1) == 0) {
                    e = lane / kCpr + k * (kWarp / kCpr);
                    c = lane % kCpr;
                } else {
                    const int x = lane + kWarp * k;
                    e = x / cpr;
                    c = x - e * cpr;
                }
            };
            const int nsteps = (nchunks + kWarp - 1) / kWarp;
            int64_t tile = blockIdx.x + (int64_t)team * gridDim.x;
            int it = team;
            int a0, z0, a1, z1, idx0 = 0;
            load_bounds(tile, a0, z0);
            load_bounds(tile + tstride, a1, z1);
            clamp_bounds(a0, z0);
            if (z0 - a0 == 1) idx0 = __ldg(ga.indices + a0);
            clamp_bounds(a1, z1);
            for (; tile < ntiles; tile += tstride, it += kTeams) {
                const int stage = it % NS;
                const uint32_t ph = (uint32_t)(it / NS) & 1u;
                const uint32_t row0 = resolve(a0, z0, idx0);
                // in flight together: next tile's index, the bounds two tiles on, this tile's rows
                int idx1 = 0, a2, z2;
                if (z1 - a1 == 1) idx1 = ldg_early_s32(ga.indices + a1);
                load_bounds(tile + 2 * tstride, a2, z2);
                const int64_t b = tile * kGroup + sm;
                uint8_t* sb = stages + (size_t)stage * L.stage_bytes;
                const uint32_t sbase = smem_u32(sb);
                uint4 dv = make_uint4(0, 0, 0, 0);
                if (lane < cpr && b < B) dv = ldg_nc_v4(dense + b * D + 8 * lane);
                bool ok = true;
                for (int k0 = 0; k0 < nsteps; k0 += kGatherU) {
                    uint4 v[kGatherU];
                    uint32_t store = 0;
#pragma unroll
                    for (int u = 0; u < kGatherU; ++u) {
                        int e, c;
                        chunk_of(k0 + u, e, c);          // e >= F past the last step
                        const uint32_t src = __shfl_sync(0xffffffffu, row0, e < F ? e : 0);
                        v[u] = make_uint4(0, 0, 0, 0);
                        if (e < F && src != kRowMulti) {
                            store |= 1u << u;
                            if (src != kRowZero) v[u] = ldg_nc_l1_v4(ga.tables + (size_t)src * Dr + 8 * c);
                        }
                    }
                    if (k0 == 0) {
                        int w = 1;
                        if (lane == 0) w = mbar_wait(&empty[stage], ph ^ 1u, abort_flag, wait_cycles);
                        ok = __shfl_sync(0xffffffffu, w, 0) != 0;
                        if (!ok) break;
                    }
#pragma unroll
                    for (int u = 0; u < kGatherU; ++u) {
                        if (!(store >> u & 1u)) continue;
                        int e, c;
                        chunk_of(k0 + u, e, c);
                        const int row = sm * kSlot + e;
                        const uint32_t dst = sbase + (c >> 3) * kKBlockBytes + row * 128 + (((c & 7) ^ (row & 7)) << 4);
                        asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(dst), "r"(v[u].x), "r"(v[u].y),
                                     "r"(v[u].z), "r"(v[u].w)
                                     : "memory");
                    }
                }
                if (!ok) break;
                if (lane < cpr) {   // dense row -> B row 128 + sm
                    const uint32_t dst = sbase + (lane >> 3) * kKBlockBytes + kEBytes + sm * 128 +
                                         (((lane & 7) ^ (sm & 7)) << 4);
                    asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(dst), "r"(dv.x), "r"(dv.y), "r"(dv.z),
                                 "r"(dv.w)
                                 : "memory");
                }
                // bags of several indices: fp32 sum in bag order, one rounding
                if constexpr (kCpr == 8 || kCpr == 16 || kCpr == 32) {
                    // Their positions form one list in bag order (lane t < F holds
                    // bag t's count); each lane resolves one of 32 positions at a
                    // time (coalesced index loads), then every lane adds its H
                    // halves of each row (all 32 lanes busy on one row), kMultiRows
                    // rows in flight, and a bag's sum is stored when the next begins.
                    constexpr int H = kCpr / 4;              // halves of a row per lane: 2, 4 or 8
                    constexpr int kMultiRows = 16;            // 8: 0.327 / 0.824 ms, 24: spills
                    const int cnt = (lane < F && row0 == kRowMulti) ? z0 - a0 : 0;
                    if (__any_sync(0xffffffffu, cnt > 0)) {
                        int incl = cnt;
#pragma unroll
                        for (int o = 1; o < kWarp; o <<= 1) {
                            const int y = __shfl_up_sync(0xffffffffu, incl, o);
                            if (lane >= o) incl += y;
                        }
                        const int excl = incl - cnt;
                        const int total = __shfl_sync(0xffffffffu, incl, kWarp - 1);
                        float acc[H];
#pragma unroll
                        for (int h = 0; h < H; ++h) acc[h] = 0.f;
                        int cur = -1;   // bag being summed (warp-uniform)
                        auto flush = [&](int t) {   // lane's H halves of bag t's row, rounded once
                            const int row = sm * kSlot + t;
                            const int c = lane * H / 8;
                            const uint32_t dst = sbase + (c >> 3) * kKBlockBytes + row * 128 +
                                                 (((c & 7) ^ (row & 7)) << 4) + (lane * H * 2) % 16;
                            uint32_t w[H / 2];
#pragma unroll
                            for (int h = 0; h < H / 2; ++h) {
                                const __half2 x = __floats2half2_rn(acc[2 * h], acc[2 * h + 1]);
                                w[h] = *reinterpret_cast<const uint32_t*>(&x);
                            }
                            if constexpr (H == 8)
                                asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(dst), "r"(w[0]), "r"(w[1]),
                                             "r"(w[2]), "r"(w[3])
                                             : "memory");
                            else if constexpr (H == 4)
                                asm volatile("st.shared.v2.u32 [%0], {%1,%2};" ::"r"(dst), "r"(w[0]), "r"(w[1])
                                             : "memory");
                            else
                                asm volatile("st.shared.u32 [%0], %1;" ::"r"(dst), "r"(w[0]) : "memory");
#pragma unroll
                            for (int h = 0; h < H; ++h) acc[h] = 0.f;
                        };
                        for (int q0 = 0; q0 < total; q0 += kWarp) {
                            const int q = q0 + lane;
                            int k = 0;   // the last lane whose list offset is at most q: its bag holds q
#pragma unroll
                            for (int step = kWarp / 2; step > 0; step >>= 1)
                                if (__shfl_sync(0xffffffffu, excl, k + step) <= q) k += step;
                            const int pos = __shfl_sync(0xffffffffu, a0, k) + (q - __shfl_sync(0xffffffffu, excl, k));
                            const int64_t base = __shfl_sync(0xffffffffu, tbase, k);
                            const int64_t n = __shfl_sync(0xffffffffu, tn, k);
                            uint32_t rowq = kRowZero;   // skipped, or past the list
                            if (q < total) {
                                int64_t i = __ldg(ga.indices + pos);
                                if (ga.hash && n > 0) {
                                    i %= n;
                                    if (i < 0) i += n;
                                    rowq = (uint32_t)(base + i);
                                } else if (ga.hash || i < 0 || i >= n) {
                                    set_status(status, DLRM_STATUS_OOB_INDEX);
                                } else {
                                    rowq = (uint32_t)(base + i);
                                }
                            }
                            const int m = total - q0 < kWarp ? total - q0 : kWarp;
                            for (int j0 = 0; j0 < m; j0 += kMultiRows) {
                                uint32_t rj[kMultiRows];
                                uint32_t v[kMultiRows][H / 2];
#pragma unroll
                                for (int u = 0; u < kMultiRows; ++u) {
                                    rj[u] = __shfl_sync(0xffffffffu, rowq, (j0 + u) & (kWarp - 1));
                                    const bool ld = j0 + u < m && rj[u] != kRowZero;
                                    const __half* src = ga.tables + (size_t)(ld ? rj[u] : 0) * D + lane * H;
                                    if constexpr (H == 8) {
                                        const uint4 x = ld ? ldg_nc_v4(src) : make_uint4(0, 0, 0, 0);
                                        v[u][0] = x.x;
                                        v[u][1] = x.y;
                                        v[u][2] = x.z;
                                        v[u][3] = x.w;
                                    } else if constexpr (H == 4) {
                                        const uint2 x = ld ? __ldg(reinterpret_cast<const uint2*>(src)) : make_uint2(0, 0);
                                        v[u][0] = x.x;
                                        v[u][1] = x.y;
                                    } else {
                                        v[u][0] = ld ? __ldg(reinterpret_cast<const uint32_t*>(src)) : 0u;
                                    }
                                }
#pragma unroll
                                for (int u = 0; u < kMultiRows; ++u) {
                                    const int kj = __shfl_sync(0xffffffffu, k, (j0 + u) & (kWarp - 1));
                                    if (j0 + u >= m) break;
                                    if (kj != cur) {
                                        if (cur >= 0) flush(cur);
                                        cur = kj;
                                    }
                                    if (rj[u] != kRowZero) {
#pragma unroll
                                        for (int h = 0; h < H / 2; ++h) {
                                            const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&v[u][h]));
                                            acc[2 * h] += f.x;
                                            acc[2 * h + 1] += f.y;
                                        }
                                    }
                                }
                            }
                        }
                        flush(cur);
                    }
                } else {
                    for (uint32_t multi = __ballot_sync(0xffffffffu, row0 == kRowMulti); multi; multi &= multi - 1) {
                        const int t = __ffs(multi) - 1;
                        const int s1 = __shfl_sync(0xffffffffu, a0, t), e1 = __shfl_sync(0xffffffffu, z0, t);
                        const int64_t base = __shfl_sync(0xffffffffu, tbase, t), n = __shfl_sync(0xffffffffu, tn, t);
                        const int row = sm * kSlot + t;
                        for (int c = lane; c < cpr; c += kWarp) {
                            float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
                            constexpr int kMultiU = 4;   // positions in flight, added in bag order
                            for (int p0 = s1; p0 < e1; p0 += kMultiU) {
                                int64_t row[kMultiU];
    #pragma unroll
                                for (int u = 0; u < kMultiU; ++u) row[u] = p0 + u < e1 ? __ldg(ga.indices + p0 + u) : -1;
                                uint4 r[kMultiU];
    #pragma unroll
                                for (int u = 0; u < kMultiU; ++u) {
                                    int64_t i = row[u];
                                    row[u] = -1;
                                    if (p0 + u < e1) {
                                        if (ga.hash && n > 0) {
                                            i %= n;
                                            if (i < 0) i += n;
                                            row[u] = base + i;
                                        } else if (ga.hash || i < 0 || i >= n) {
                                            set_status(status, DLRM_STATUS_OOB_INDEX);
                                        } else {
                                            row[u] = base + i;
                                        }
                                    }
                                    r[u] = row[u] >= 0 ? ldg_nc_v4(ga.tables + row[u] * D + 8 * c) : make_uint4(0, 0, 0, 0);
                                }
    #pragma unroll
                                for (int u = 0; u < kMultiU; ++u)
                                    if (row[u] >= 0) {
                                        float f[8];
                                        h8_to_f8(r[u], f);
    #pragma unroll
                                        for (int v = 0; v < 8; ++v) acc[v] += f[v];
                                    }
                            }
                            const uint4 w = f8_to_h8(acc);
                            const uint32_t dst = sbase + (c >> 3) * kKBlockBytes + row * 128 + (((c & 7) ^ (row & 7)) << 4);
                            asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(dst), "r"(w.x), "r"(w.y), "r"(w.z),
                                         "r"(w.w)
                                         : "memory");
                        }
                    }
                }
                // generic-proxy writes -> visible to the tensor core, then publish this slot
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (lane == 0) mbar_arrive(&full[stage]);
                a0 = a1;
                z0 = z1;
                idx0 = idx1;
                clamp_bounds(a2, z2);
                a1 = a2;
                z1 = z2;
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------------------------ MMA issuer
            int it = 0;
            for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++it) {
                const int stage = it % NS;
                const uint32_t ph = (uint32_t)(it / NS) & 1u;
                const int buf = it & 1;
                const uint32_t bph = (uint32_t)(it >> 1) & 1u;
                if (!mbar_wait(&tempty[buf], bph ^ 1u, abort_flag, wait_cycles)) break;
                tc_fence_after();
                if (!mbar_wait(&full[stage], ph, abort_flag, wait_cycles)) break;
                tc_fence_after();
                const uint32_t d = tmem_base + (uint32_t)(buf * kAccStride);
                const uint32_t sb = smem_u32(stages + (size_t)stage * L.stage_bytes);
                for (int kb = 0; kb < KH; ++kb)
#pragma unroll
                    for (int kk = 0; kk < kKB / 16; ++kk) {
                        const uint64_t desc = sw128_desc(sb + kb * kKBlockBytes + kk * 32);
                        tc_mma_f16(d, desc, desc, kIdesc, (kb | kk) != 0);
                    }
                tc_commit(&empty[stage]);
                tc_commit(&tfull[buf]);
            }
            if (*abort_flag && it > 0)   // MMAs already issued must finish before TMEM is freed
                mbar_drain(&tfull[(it - 1) & 1], (uint32_t)((it - 1) >> 1) & 1u);
        }
    } else if (warp < 6) {
        // ---------------------------------------------------- epilogue
        const int q = warp & 3;                     // TMEM lane quarter == sample in tile
        uint32_t* sq = square + q * kSlot * kSqRow;
        const __half* sqh = reinterpret_cast<const __half*>(sq);
        // The sample's dense row is copied to the output from registers, loaded
        // one tile ahead so its latency overlaps the wait for the accumulator.
        auto load_dense = [&](int tile) {
            const int64_t b = (int64_t)tile * kGroup + q;
            return (tile < ntiles && b < B && lane < D / 8) ? ldg_nc_v4(dense + b * D + 8 * lane)
                                                             : make_uint4(0u, 0u, 0u, 0u);
        };
        uint4 dnext = load_dense(blockIdx.x);
        int it = 0;
        for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++it) {
            const int buf = it & 1;
            const uint32_t bph = (uint32_t)(it >> 1) & 1u;
            const uint4 dcur = dnext;
            dnext = load_dense(tile + gridDim.x);
            if (!mbar_wait(&tfull[buf], bph, abort_flag, wait_cycles)) break;
            __syncwarp();
            tc_fence_after();
            const uint32_t taddr = tmem_base + ((uint32_t)(kSlot * q) << 16) + (uint32_t)(buf * kAccStride);
            uint32_t v[32];
            uint32_t dd;
            tmem_ld_x32(taddr + (uint32_t)(kSlot * q), v);
            tmem_ld_x1(taddr + (uint32_t)(kM + q), dd);
            tmem_wait_ld(v, dd);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[buf]);
            const int b = tile * kGroup + q;
            if (b < B) {
                // Lane i holds row i + 1 of Z against rows 0..31: h[0] = e_i . d,
                // h[j] = e_i . e_{j-1}.  It writes them as halves to row i of the
                // square (17-word rows: conflict-free), then the warp reads the
                // triangle back in output order and stores it coalesced.
                uint32_t* srow = sq + lane * kSqRow;
                srow[0] = h2_bits(__uint_as_float(dd), __uint_as_float(v[0]));
#pragma unroll
                for (int m = 1; m < 16; ++m)
                    srow[m] = h2_bits(__uint_as_float(v[2 * m - 1]), __uint_as_float(v[2 * m]));
                __syncwarp();
                __half* orow = out + (int64_t)b * P;
                if (lane < D / 8) stg_cs_v4(orow + 8 * lane, dcur);
                // lane: output pairs 8 (lane + 32 m) .. + 7, one 16-byte store each
                constexpr int kTriIters = (kSlot * (kSlot + 1) / 2 + 8 * kWarp - 1) / (8 * kWarp);
#pragma unroll
                for (int m = 0; m < kTriIters; ++m) {
                    const int k = 8 * (lane + kWarp * m);
                    if (k < T) {
                        const uint4 o = *reinterpret_cast<const uint4*>(tri + k);
                        const uint32_t ow[4] = {o.x, o.y, o.z, o.w};
                        uint32_t hw[4];
#pragma unroll
                        for (int h = 0; h < 4; ++h) {
                            const uint32_t o0 = ow[h] & 0xffffu, o1 = ow[h] >> 16;
                            const uint32_t lo = o0 == 0xffffu ? 0u : __half_as_ushort(sqh[o0]);
                            const uint32_t hi = o1 == 0xffffu ? 0u : __half_as_ushort(sqh[o1]);
                            hw[h] = lo | (hi << 16);
                        }
                        stg_cs_v4(orow + D + k, make_uint4(hw[0], hw[1], hw[2], hw[3]));
                    }
                }
                // zero padding past the triangle (rounded up to 8 pairs)
                for (int c = D + ((T + 7) & ~7) + 8 * lane; c < P; c += 8 * kWarp)
                    stg_cs_v4(orow + c, make_uint4(0u, 0u, 0u, 0u));
                __syncwarp();   // the square is rewritten for the next tile
            }
        }
        (void)W;
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(kTmemCols)
                     : "memory");
    }
    if (threadIdx.x == 0 && *abort_flag) set_status(status, DLRM_STATUS_TIMEOUT);
}

}  // namespace

bool tc_interact_supported(int F, int D, int out_cols, const void* dense, const void* pooled, const void* out)
{
    return F >= 1 && F <= kSlot && D % kKB == 0 && D >= kKB && D <= 4 * kKB && out_cols % 8 == 0 &&
           out_cols <= 2048 && aligned16(dense) && aligned16(pooled) && aligned16(out);
}

template <bool kFused, int kCpr>
dlrm_status launch_kernel(int grid, int threads, const Layout& L, const CUtensorMap& mp, const CUtensorMap& md,
                          const void* dense, void* out, int F, int D, int B, int P, int KH, int ns, uint32_t* status,
                          const GatherArgs& ga, cudaStream_t stream, const char* who)
{
    cudaError_t e = cudaFuncSetAttribute(interact_tc_kernel<kFused, kCpr>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)L.smem);
    if (e != cudaSuccess) return fail(DLRM_ERR_CUDA, "%s: %s", who, cudaGetErrorString(e));
    return check_launch_pdl(launch_pdl(interact_tc_kernel<kFused, kCpr>, grid, threads, L.smem, stream, mp, md,
                                       (const __half*)dense, (__half*)out, F, D, B, P, KH, ns, status, ga,
                                       wait_limit_cycles()),
                            "interact_tc_kernel");
}

// Tensor maps + launch of the tcgen05 kernel.  pooled == nullptr selects the
// fused lookup (rows gathered from ga.tables).
dlrm_status tc_launch(const void* dense, const void* pooled, const GatherArgs& ga, int F, int D, int B, void* out,
                      int out_cols, uint32_t* status, cudaStream_t stream, const char* who)
{
    EncodeTiledFn enc = encode_fn();
    if (!enc) return fail(DLRM_ERR_CUDA, "%s: cuTensorMapEncodeTiled unavailable", who);
    const int KH = D / kKB;
    // The fused kernel keeps to kFusedStages so that about 90 KB of the SM's
    // 256 KB stays L1: the Zipf-hot table rows then hit in L1.
    int ns = pooled ? kMaxStages : kFusedStages;
    while (ns > 1 && make_layout(KH, out_cols, ns).smem > (size_t)kSmemLimit) --ns;
    const Layout L = make_layout(KH, out_cols, ns);
    if (ns < 2 || L.smem > (size_t)kSmemLimit)
        return fail(DLRM_ERR_UNSUPPORTED, "%s: tensor-core tile does not fit shared memory", who);

    CUtensorMap mp, md;
    const cuuint32_t ones[3] = {1, 1, 1};
    const cuuint64_t ddims[2] = {(cuuint64_t)D, (cuuint64_t)B};
    const cuuint64_t dstr[1] = {(cuuint64_t)D * 2};
    const cuuint32_t dbox[2] = {(cuuint32_t)kKB, (cuuint32_t)kGroup};
    CUresult r = enc(&md, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(dense), ddims, dstr, dbox, ones,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(DLRM_ERR_CUDA, "%s: encoding the dense tensor map failed (%d)", who, (int)r);
    if (pooled) {
        const cuuint64_t pdims[3] = {(cuuint64_t)D, (cuuint64_t)F, (cuuint64_t)B};
        const cuuint64_t pstr[2] = {(cuuint64_t)D * 2, (cuuint64_t)F * D * 2};
        const cuuint32_t pbox[3] = {(cuuint32_t)kKB, (cuuint32_t)kSlot, (cuuint32_t)kGroup};
        r = enc(&mp, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void*>(pooled), pdims, pstr, pbox, ones,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS)
            return fail(DLRM_ERR_CUDA, "%s: encoding the pooled tensor map failed (%d)", who, (int)r);
    } else {
        mp = md;   // unused by the fused kernel
    }
    const int ntiles = (B + kGroup - 1) / kGroup;
    const int grid = ntiles < num_sms() ? ntiles : num_sms();
    if (pooled)
        return launch_kernel<false, 0>(grid, kThreads, L, mp, md, dense, out, F, D, B, out_cols, KH, ns, status, ga,
                                       stream, who);
    switch (D / 8) {
    case 8: return launch_kernel<true, 8>(grid, kThreadsFused, L, mp, md, dense, out, F, D, B, out_cols, KH, ns, status,
                                          ga, stream, who);
    case 16: return launch_kernel<true, 16>(grid, kThreadsFused, L, mp, md, dense, out, F, D, B, out_cols, KH, ns,
                                            status, ga, stream, who);
    case 32: return launch_kernel<true, 32>(grid, kThreadsFused, L, mp, md, dense, out, F, D, B, out_cols, KH, ns,
                                            status, ga, stream, who);
    default: return launch_kernel<true, 0>(grid, kThreadsFused, L, mp, md, dense, out, F, D, B, out_cols, KH, ns,
                                           status, ga, stream, who);
    }
}

dlrm_status tc_interact_fwd(const void* dense, const void* pooled, int F, int D, int B, void* out,
                            int out_cols, uint32_t* status, cudaStream_t stream)
{
    return tc_launch(dense, pooled, GatherArgs{}, F, D, B, out, out_cols, status, stream, "dlrm_interact_fwd");
}

}  // namespace dlrm

using namespace dlrm;

extern "C" dlrm_status dlrm_emb_interact_fwd(const void* d_tables, dlrm_dtype dtype, const int64_t* d_row_base,
                                             int F, int D, int B, const int32_t* d_indices,
                                             const int32_t* d_offsets, int64_t nnz, const void* d_dense,
                                             void* d_out, int out_cols, unsigned flags, uint32_t* d_status,
                                             void* stream)
{
    DLRM_API_RANGE("dlrm_emb_interact_fwd");
    clear_error();
    if (!dtype_ok(dtype)) return fail(DLRM_ERR_INVALID_ARG, "dlrm_emb_interact_fwd: bad dtype");
    if (F < 1 || D < 1 || B < 0)
        return fail(DLRM_ERR_INVALID_ARG, "dlrm_emb_interact_fwd: need F >= 1, D >= 1, B >= 0");
    if (nnz < 0 || nnz > DLRM_MAX_NNZ || (int64_t)F * B >= (int64_t)1 << 31)
        return fail(DLRM_ERR_INVALID_ARG, "dlrm_emb_interact_fwd: need nnz <= DLRM_MAX_NNZ and F*B < 2^31");
    const int64_t W = (int64_t)D + (int64_t)F * (F + 1) / 2;
    if (out_cols < W)
        return fail(DLRM_ERR_INVALID_ARG, "dlrm_emb_interact_fwd: out_cols %d < D + F(F+1)/2 = %lld", out_cols,
                    (long long)W);
    if (!d_tables || !d_row_base || !d_offsets || !d_dense || !d_out || (nnz > 0 && !d_indices))
        return fail(DLRM_ERR_INVALID_ARG, "dlrm_emb_interact_fwd: null device pointer");
    if (flags & ~DLRM_FLAG_HASH_INDICES)
        return fail(DLRM_ERR_INVALID_ARG, "dlrm_emb_interact_fwd: unknown flag bits 0x%x", flags);
    if (dtype == DLRM_F32) {
        if (!regs_emb_interact_supported(F, D, out_cols, d_tables, d_dense, nullptr, d_out))
            return fail(DLRM_ERR_UNSUPPORTED,
                        "dlrm_emb_interact_fwd: fp32 needs D = 128, F in {8, 26}, out_cols a multiple of 4 without "
                        "padding past the last group of 32 pairs, and 16-byte aligned pointers (use dlrm_emb_fwd + "
                        "dlrm_interact_fwd otherwise)");
        if (B == 0) return DLRM_OK;
        return regs_emb_interact_fwd((const float*)d_tables, d_row_base, F, D, B, d_indices, d_offsets, nnz,
                                     (const float*)d_dense, nullptr, (float*)d_out, out_cols,
                                     (flags & DLRM_FLAG_HASH_INDICES) != 0, d_status, as_stream(stream));
    }
    if (!tc_interact_supported(F, D, out_cols, d_dense, d_dense, d_out) || !aligned16(d_tables))
        return fail(DLRM_ERR_UNSUPPORTED,
                    "dlrm_emb_interact_fwd: fp16 needs F <= 32, D a multiple of 64 up to 256, out_cols a multiple "
                    "of 8 and 16-byte aligned pointers (use dlrm_emb_fwd + dlrm_interact_fwd otherwise)");
    if (B == 0) return DLRM_OK;
    GatherArgs ga;
    ga.tables = (const __half*)d_tables;
    ga.row_base = d_row_base;
    ga.indices = d_indices;
    ga.offsets = d_offsets;
    ga.nnz = nnz;
    ga.hash = (flags & DLRM_FLAG_HASH_INDICES) != 0;
    return tc_launch(d_dense, nullptr, ga, F, D, B, d_out, out_cols, d_status, as_stream(stream),
                     "dlrm_emb_interact_fwd");
}
