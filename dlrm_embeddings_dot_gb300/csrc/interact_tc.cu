// interact_tc.cu -- dot interaction on the 5th-generation tensor cores
// (tcgen05) for fp16 inputs with fp32 accumulation ("DLRM For PyTorch",
// §Model architecture; --interaction_op cuda_dot).
//
// Per sample, Z = [d; e_0 .. e_{F-1}] and the output needs z_i . z_j for
// i > j.  Four samples form one M = 128 tile: sample s's F embedding rows sit
// at rows 32s .. 32s+F-1 (rows F..31 zero), so the 128 x 128 product of the
// tile with itself holds each sample's E E^T in a 32 x 32 diagonal block.  The
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
// Fused variant (dlrm_emb_interact_fwd, inference): the producer warp gathers
// each bag's table row straight into the sample slots with cp.async, so the
// pooled tensor never goes to HBM.
// Two TMEM accumulators (2 x 256 columns) let the MMA of tile i+1 overlap the
// epilogue of tile i.  Every mbarrier wait is bounded; on timeout the kernel
// sets DLRM_STATUS_TIMEOUT, drains what it issued, frees TMEM and returns.
#include <cuda.h>

#include "interact_tc.cuh"

namespace dlrm {
namespace {

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
constexpr int kThreadsFused = 256;                // + two resolver warps
constexpr int kGatherDepth = 3;                   // tiles of cp.async gathers in flight
constexpr int kResolveBatch = 3;                  // tiles a resolver warp resolves at once
constexpr int kMetaSlots = 4 * kResolveBatch;     // rows-to-gather ring (two batches per resolver warp)
constexpr int kMaxStages = 8;
constexpr int kSmemLimit = 232448;                // 227 KB opt-in per block
constexpr long long kWaitCycles = 4000000000LL;   // about two seconds

// instruction descriptor, kind::f16: D = f32, A = B = f16, both K-major, N, M
constexpr uint32_t kIdesc = (1u << 4) | ((uint32_t)(kN >> 3) << 17) | ((uint32_t)(kM >> 4) << 24);

__device__ __forceinline__ uint32_t smem_u32(const void* p)
{
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

// Adds to the expected transaction bytes of the current phase without arriving.
__device__ __forceinline__ void mbar_add_tx(uint64_t* bar, uint32_t bytes)
{
    asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void cp_async16(uint32_t smem_dst, const void* gsrc)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_dst), "l"(gsrc) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait for the phase of `parity` to complete.  Returns false if the
// CTA is aborting or the bound is hit (which starts the abort).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag)
{
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    for (;;) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (clock64() - t0 > kWaitCycles) {
            *abort_flag = 1;
            return false;
        }
    }
}

// Bounded wait that ignores the abort flag (used to drain on the abort path).
__device__ __forceinline__ void mbar_drain(uint64_t* bar, uint32_t parity)
{
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity) && clock64() - t0 < kWaitCycles) {
    }
}

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int c0, int c1, int c2,
                                            uint64_t* bar)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
        "l"(map), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int c0, int c1, uint64_t* bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
        "l"(map), "r"(c0), "r"(c1), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tc_commit(uint64_t* bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void tc_mma_f16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                           uint32_t accumulate)
{
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups
// 1024 bytes apart (stride byte offset), descriptor version 1.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr)
{
    uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)1 << 16;                 // leading byte offset (unused for swizzled K-major)
    d |= (uint64_t)(1024 >> 4) << 32;       // stride byte offset
    d |= (uint64_t)1 << 46;                 // version
    d |= (uint64_t)2 << 61;                 // SWIZZLE_128B
    return d;
}

__device__ __forceinline__ void tmem_ld_x32(uint32_t taddr, uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld_x1(uint32_t taddr, uint32_t& r)
{
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];" : "=r"(r) : "r"(taddr));
}

// tcgen05.wait::ld, tied to the loaded registers so no use moves above it.
__device__ __forceinline__ void tmem_wait_ld(uint32_t (&r)[32], uint32_t& x)
{
    asm volatile(
        "tcgen05.wait::ld.sync.aligned;"
        : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
          "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]),
          "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]),
          "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]),
          "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31]), "+r"(x)
        :
        : "memory");
}

struct Layout {
    int stage_bytes, ns, out_bytes;
    size_t smem;
};

__host__ __device__ inline Layout make_layout(int KH, int P, int ns)
{
    Layout L;
    L.stage_bytes = KH * kKBlockBytes;
    L.ns = ns;
    L.out_bytes = (kGroup * P * 2 + 15) / 16 * 16;
    L.smem = 1024 + (size_t)ns * L.stage_bytes + L.out_bytes + (2 * ns + 4) * 8 + 16 +
             (size_t)kMetaSlots * (8 * kGroup * kSlot + 16);
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

template <bool kFused>
__global__ void __launch_bounds__(kFused ? kThreadsFused : kThreads, 1)
interact_tc_kernel(const __grid_constant__ CUtensorMap map_pooled,
                   const __grid_constant__ CUtensorMap map_dense, const __half* __restrict__ dense,
                   __half* __restrict__ out, int F, int D, int B, int P, int KH, int NS,
                   uint32_t* status, GatherArgs ga)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    const Layout L = make_layout(KH, P, NS);
    uint8_t* stages = smem;
    __half* ostage = reinterpret_cast<__half*>(smem + (size_t)NS * L.stage_bytes);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)NS * L.stage_bytes + L.out_bytes);
    uint64_t* empty = full + NS;
    uint64_t* tfull = empty + NS;
    uint64_t* tempty = tfull + 2;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(tempty + 2);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
    // fused mode: ring of kMetaSlots tiles' source rows per (sample, table)
    // (>= 0 row, -1 zero row, -2 several indices: summed by the producer),
    // filled by the resolver warps, and its full/empty barriers
    int64_t* ring = reinterpret_cast<int64_t*>(reinterpret_cast<uint8_t*>(tempty + 2) + 16);
    uint64_t* meta_full = reinterpret_cast<uint64_t*>(ring + kMetaSlots * kGroup * kSlot);
    uint64_t* meta_empty = meta_full + kMetaSlots;
    const int nthreads = kFused ? kThreadsFused : kThreads;

    const int warp = threadIdx.x / kWarp;
    const int lane = threadIdx.x % kWarp;
    const int ntiles = (B + kGroup - 1) / kGroup;
    const int W = D + F * (F + 1) / 2;

    if (threadIdx.x == 0) {
        for (int i = 0; i < NS; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&tfull[i], 1);
            mbar_init(&tempty[i], kGroup);
        }
        if (kFused)
            for (int i = 0; i < kMetaSlots; ++i) {
                mbar_init(&meta_full[i], 1);
                mbar_init(&meta_empty[i], 1);
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
    if (kFused) {   // rows F..31 of each sample slot are never written by the gather
        const int per_slot = (kSlot - F) * 8;   // 16-byte chunks of rows F..31 in one K block
        for (int s = 0; s < NS; ++s)
            for (int kb = 0; kb < KH; ++kb)
                for (int x = threadIdx.x; x < kGroup * per_slot; x += nthreads) {
                    const int slot = x / per_slot, r = F + (x % per_slot) / 8, c = x % 8;
                    *reinterpret_cast<uint4*>(stages + (size_t)s * L.stage_bytes + kb * kKBlockBytes +
                                              (slot * kSlot + r) * 128 + c * 16) = make_uint4(0, 0, 0, 0);
                }
    }
    for (int x = threadIdx.x; x < kGroup * P; x += nthreads) ostage[x] = __float2half_rn(0.f);
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

    if (warp == 0) {
        if constexpr (!kFused) {
            if (lane == 0) {
                // ------------------------------------------------ TMA producer
                int it = 0;
                for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++it) {
                    const int stage = it % NS;
                    const uint32_t ph = (uint32_t)(it / NS) & 1u;
                    if (!mbar_wait(&empty[stage], ph ^ 1u, abort_flag)) break;
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
            // ------------------------------------ gather producer (whole warp)
            // Table rows go straight from the table into the swizzled sample slots
            // with cp.async (16 lanes per 256-byte row, so every load is a full
            // sector); the dense rows come by TMA.  A tile's arrive on its full
            // barrier is posted kGatherDepth - 1 tiles later, after its copies
            // have landed and a proxy fence, so kGatherDepth tiles are in flight.
            const int cpr = D / 8;                       // 16-byte chunks per row
            int it = 0, published = 0;   // tiles [published, it) have copies in flight
            for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++it) {
                const int stage = it % NS;
                const uint32_t ph = (uint32_t)(it / NS) & 1u;
                int ok = 1;
                if (lane == 0) ok = mbar_wait(&empty[stage], ph ^ 1u, abort_flag);
                if (!__shfl_sync(0xffffffffu, ok, 0)) break;
                uint8_t* sb = stages + (size_t)stage * L.stage_bytes;
                if (lane == 0) {
                    mbar_add_tx(&full[stage], (uint32_t)KH * (kGroup * 128));
                    for (int kb = 0; kb < KH; ++kb)
                        tma_load_2d(sb + kb * kKBlockBytes + kEBytes, &map_dense, kb * kKB, tile * kGroup,
                                    &full[stage]);
                }
                // source rows of the tile's kGroup x F bags, from the resolver warps
                const int mslot = it % kMetaSlots;
                if (lane == 0) ok = mbar_wait(&meta_full[mslot], (uint32_t)(it / kMetaSlots) & 1u, abort_flag);
                if (!__shfl_sync(0xffffffffu, ok, 0)) break;
                const int64_t* rowsrc = ring + mslot * kGroup * kSlot;
                __syncwarp();
                const uint32_t sbase = smem_u32(sb);
                auto gather_chunk = [&](int sm, int t, int c) {
                    const int row = sm * kSlot + t;
                    const int64_t src = rowsrc[row];
                    const uint32_t dst = sbase + (c >> 3) * kKBlockBytes + row * 128 + (((c & 7) ^ (row & 7)) << 4);
                    if (src >= 0)
                        cp_async16(dst, ga.tables + src * D + 8 * c);
                    else if (src == -1)
                        asm volatile("st.shared.v4.u32 [%0], {%1,%1,%1,%1};" ::"r"(dst), "r"(0u) : "memory");
                };
                if (kWarp % cpr == 0) {
                    // each lane keeps one chunk column c; rows advance by 32 / cpr per step
                    const int step = kWarp / cpr, c = lane % cpr;
                    int sm = 0, t = lane / cpr;
                    for (int e = lane / cpr; e < kGroup * F; e += step) {
                        while (t >= F) {
                            t -= F;
                            ++sm;
                        }
                        gather_chunk(sm, t, c);
                        t += step;
                    }
                } else {
                    for (int x = lane; x < kGroup * F * cpr; x += kWarp) {
                        const int e = x / cpr, c = x - e * cpr;
                        const int sm = e / F;
                        gather_chunk(sm, e - sm * F, c);
                    }
                }
                // bags of several indices (rare): fp32 sum in bag order, one rounding
                bool any_multi = false;
                for (int e = lane; e < kGroup * F; e += kWarp) any_multi |= rowsrc[(e / F) * kSlot + e % F] == -2;
                for (int e = 0; __any_sync(0xffffffffu, any_multi) && e < kGroup * F; ++e) {
                    if (rowsrc[(e / F) * kSlot + e % F] != -2) continue;
                    const int sm = e / F, t = e - sm * F;
                    const int64_t bag = (int64_t)t * B + (int64_t)tile * kGroup + sm;
                    int64_t s0 = ga.offsets[bag], e0 = ga.offsets[bag + 1];
                    s0 = s0 < 0 ? 0 : (s0 > ga.nnz ? ga.nnz : s0);
                    e0 = e0 < s0 ? s0 : (e0 > ga.nnz ? ga.nnz : e0);
                    const int64_t base = ga.row_base[t], n = ga.row_base[t + 1] - base;
                    const int row = sm * kSlot + t;
                    for (int c = lane; c < cpr; c += kWarp) {
                        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
                        for (int64_t p = s0; p < e0; ++p) {
                            int64_t i = ga.indices[p];
                            if (ga.hash && n > 0) {
                                i %= n;
                                if (i < 0) i += n;
                            } else if (ga.hash || i < 0 || i >= n) {
                                set_status(status, DLRM_STATUS_OOB_INDEX);
                                continue;
                            }
                            float f[8];
                            h8_to_f8(ldg_nc_v4(ga.tables + (base + i) * D + 8 * c), f);
#pragma unroll
                            for (int u = 0; u < 8; ++u) acc[u] += f[u];
                        }
                        const uint4 v = f8_to_h8(acc);
                        const uint32_t dst = sbase + (c >> 3) * kKBlockBytes + row * 128 + (((c & 7) ^ (row & 7)) << 4);
                        asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(dst), "r"(v.x), "r"(v.y), "r"(v.z),
                                     "r"(v.w)
                                     : "memory");
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&meta_empty[mslot]);   // the ring slot has been read
                asm volatile("cp.async.commit_group;" ::: "memory");
                // (the stage ring must be deeper than the gathers in flight, or the
                // producer would wait on a stage whose tile it has not published yet)
                if (it + 1 - published >= (NS > kGatherDepth ? kGatherDepth : NS - 1)) {
                    // the oldest tile's rows have landed: publish it
                    if (NS > kGatherDepth)
                        asm volatile("cp.async.wait_group %0;" ::"n"(kGatherDepth - 1) : "memory");
                    else
                        asm volatile("cp.async.wait_group 0;" ::: "memory");
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&full[published % NS]);
                    ++published;
                }
            }
            asm volatile("cp.async.wait_all;" ::: "memory");
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            for (; published < it; ++published)
                if (lane == 0) mbar_arrive(&full[published % NS]);
            if (*abort_flag && lane == 0) {   // the dense copies already issued must land before exit
                for (int j = (it > NS ? it - NS : 0); j < it; ++j)
                    mbar_drain(&full[j % NS], (uint32_t)(j / NS) & 1u);
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
                if (!mbar_wait(&tempty[buf], bph ^ 1u, abort_flag)) break;
                tc_fence_after();
                if (!mbar_wait(&full[stage], ph, abort_flag)) break;
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
        __half* os = ostage + q * P;
        int it = 0;
        for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++it) {
            const int buf = it & 1;
            const uint32_t bph = (uint32_t)(it >> 1) & 1u;
            if (!mbar_wait(&tfull[buf], bph, abort_flag)) break;
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
                const __half* drow = dense + (int64_t)b * D;
                for (int c = lane; c < D / 8; c += kWarp)
                    *reinterpret_cast<uint4*>(os + 8 * c) = ldg_nc_v4(drow + 8 * c);
                if (lane < F) {
                    // row i = lane + 1 of Z: pairs (i, 0) .. (i, i-1)
                    const int base = D + (lane + 1) * lane / 2;
                    os[base] = __float2half_rn(__uint_as_float(dd));
#pragma unroll
                    for (int j = 1; j < 32; ++j)
                        if (j <= lane) os[base + j] = __float2half_rn(__uint_as_float(v[j - 1]));
                }
                __syncwarp();
                __half* orow = out + (int64_t)b * P;
                for (int c = lane; c < P / 8; c += kWarp)
                    stg_cs_v4(orow + 8 * c, *reinterpret_cast<const uint4*>(os + 8 * c));
                __syncwarp();
            }
        }
        (void)W;
    } else if constexpr (kFused) {
        // ---------------------------------------------------- resolvers
        // Warp 6 + r resolves batches of kResolveBatch consecutive tiles of this
        // CTA (batches r, r + 2, ...): offsets -> index -> hashed or checked
        // global row, with all offset loads and then all index loads of the
        // batch in flight together, into ring slots it % kMetaSlots.
        const int r = warp - 6;
        constexpr int kPer = (kGroup * kSlot + kWarp - 1) / kWarp;   // entries per lane per tile
        for (int g = r;; g += 2) {
            const int it0 = g * kResolveBatch;
            if (blockIdx.x + it0 * (int)gridDim.x >= ntiles) break;
            int ok = 1;
            if (lane == 0)
                for (int k = 0; k < kResolveBatch && ok; ++k) {
                    const int it = it0 + k;
                    if (blockIdx.x + it * (int)gridDim.x < ntiles)
                        ok = mbar_wait(&meta_empty[it % kMetaSlots], ((uint32_t)(it / kMetaSlots) & 1u) ^ 1u,
                                       abort_flag);
                }
            if (!__shfl_sync(0xffffffffu, ok, 0)) break;
            int64_t s0[kResolveBatch][kPer], e0[kResolveBatch][kPer];
#pragma unroll
            for (int k = 0; k < kResolveBatch; ++k)
#pragma unroll
                for (int u = 0; u < kPer; ++u) {
                    const int e = lane + u * kWarp;
                    const int64_t tile = (int64_t)blockIdx.x + (int64_t)(it0 + k) * gridDim.x;
                    s0[k][u] = e0[k][u] = 0;
                    if (e < kGroup * F && tile < ntiles) {
                        const int sm = e / F, t = e - sm * F;
                        const int64_t b = tile * kGroup + sm;
                        if (b < B) {
                            s0[k][u] = ga.offsets[(int64_t)t * B + b];
                            e0[k][u] = ga.offsets[(int64_t)t * B + b + 1];
                        }
                    }
                }
            int32_t idx[kResolveBatch][kPer];
#pragma unroll
            for (int k = 0; k < kResolveBatch; ++k)
#pragma unroll
                for (int u = 0; u < kPer; ++u) {
                    const int64_t a = s0[k][u];
                    idx[k][u] = (e0[k][u] - a == 1 && a >= 0 && a < ga.nnz) ? ga.indices[a] : 0;
                }
#pragma unroll
            for (int k = 0; k < kResolveBatch; ++k) {
                const int it = it0 + k;
                if (blockIdx.x + it * (int)gridDim.x >= ntiles) break;
                int64_t* rowsrc = ring + (it % kMetaSlots) * kGroup * kSlot;
#pragma unroll
                for (int u = 0; u < kPer; ++u) {
                    const int e = lane + u * kWarp;
                    if (e >= kGroup * F) continue;
                    const int sm = e / F, t = e - sm * F;
                    int64_t a = s0[k][u], z = e0[k][u];
                    if (a < 0 || z < a || z > ga.nnz) {
                        set_status(status, DLRM_STATUS_BAD_OFFSETS);
                        a = a < 0 ? 0 : (a > ga.nnz ? ga.nnz : a);
                        z = z < a ? a : (z > ga.nnz ? ga.nnz : z);
                    }
                    int64_t src = -1;
                    if (z - a == 1) {
                        if (e0[k][u] - s0[k][u] != 1) idx[k][u] = ga.indices[a];   // clamped bag
                        int64_t i = idx[k][u];
                        const int64_t base = ga.row_base[t], n = ga.row_base[t + 1] - base;
                        if (ga.hash && n > 0) {
                            i %= n;
                            if (i < 0) i += n;
                            src = base + i;
                        } else if (!ga.hash && i >= 0 && i < n) {
                            src = base + i;
                        } else {
                            set_status(status, DLRM_STATUS_OOB_INDEX);
                        }
                    } else if (z - a > 1) {
                        src = -2;
                    }
                    rowsrc[sm * kSlot + t] = src;
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&meta_full[it % kMetaSlots]);
            }
        }
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

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                                  CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                  CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

}  // namespace

bool tc_interact_supported(int F, int D, int out_cols, const void* dense, const void* pooled, const void* out)
{
    return F >= 1 && F <= kSlot && D % kKB == 0 && D >= kKB && D <= 4 * kKB && out_cols % 8 == 0 &&
           out_cols <= 2048 && aligned16(dense) && aligned16(pooled) && aligned16(out);
}

// Tensor maps + launch of the tcgen05 kernel.  pooled == nullptr selects the
// fused lookup (rows gathered from ga.tables).
dlrm_status tc_launch(const void* dense, const void* pooled, const GatherArgs& ga, int F, int D, int B, void* out,
                      int out_cols, uint32_t* status, cudaStream_t stream, const char* who)
{
    EncodeTiledFn enc = encode_fn();
    if (!enc) return fail(DLRM_ERR_CUDA, "%s: cuTensorMapEncodeTiled unavailable", who);
    const int KH = D / kKB;
    int ns = kMaxStages;
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
    if (pooled) {
        cudaError_t e = cudaFuncSetAttribute(interact_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)L.smem);
        if (e != cudaSuccess) return fail(DLRM_ERR_CUDA, "%s: %s", who, cudaGetErrorString(e));
        interact_tc_kernel<false><<<grid, kThreads, L.smem, stream>>>(mp, md, (const __half*)dense, (__half*)out, F,
                                                                      D, B, out_cols, KH, ns, status, ga);
    } else {
        cudaError_t e = cudaFuncSetAttribute(interact_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)L.smem);
        if (e != cudaSuccess) return fail(DLRM_ERR_CUDA, "%s: %s", who, cudaGetErrorString(e));
        interact_tc_kernel<true><<<grid, kThreadsFused, L.smem, stream>>>(mp, md, (const __half*)dense, (__half*)out, F,
                                                                     D, B, out_cols, KH, ns, status, ga);
    }
    return check_launch("interact_tc_kernel");
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
    clear_error();
    if (!dtype_ok(dtype)) return fail(DLRM_ERR_INVALID_ARG, "dlrm_emb_interact_fwd: bad dtype");
    if (F < 1 || D < 1 || B < 0)
        return fail(DLRM_ERR_INVALID_ARG, "dlrm_emb_interact_fwd: need F >= 1, D >= 1, B >= 0");
    if (nnz < 0 || nnz >= (int64_t)1 << 31 || (int64_t)F * B >= (int64_t)1 << 31)
        return fail(DLRM_ERR_INVALID_ARG, "dlrm_emb_interact_fwd: nnz and F*B must be below 2^31");
    const int64_t W = (int64_t)D + (int64_t)F * (F + 1) / 2;
    if (out_cols < W)
        return fail(DLRM_ERR_INVALID_ARG, "dlrm_emb_interact_fwd: out_cols %d < D + F(F+1)/2 = %lld", out_cols,
                    (long long)W);
    if (!d_tables || !d_row_base || !d_offsets || !d_dense || !d_out || (nnz > 0 && !d_indices))
        return fail(DLRM_ERR_INVALID_ARG, "dlrm_emb_interact_fwd: null device pointer");
    if (flags & ~DLRM_FLAG_HASH_INDICES)
        return fail(DLRM_ERR_INVALID_ARG, "dlrm_emb_interact_fwd: unknown flag bits 0x%x", flags);
    if (dtype != DLRM_F16 || !tc_interact_supported(F, D, out_cols, d_dense, d_dense, d_out) || !aligned16(d_tables))
        return fail(DLRM_ERR_UNSUPPORTED,
                    "dlrm_emb_interact_fwd: needs fp16, F <= 32, D a multiple of 64 up to 256, out_cols a multiple "
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
