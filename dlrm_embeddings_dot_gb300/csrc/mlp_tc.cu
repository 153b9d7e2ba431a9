// mlp_tc.cu -- the bottom MLP on the tcgen05 tensor cores ("DLRM For
// PyTorch", §Model architecture; --bottom_mlp_sizes 512,256,128; §Mixed
// precision training): each layer computes out = relu(in W^T + b) from fp16
// tensors with fp32 accumulation and an fp32 bias, and stores fp16.  The last
// layer's output is the `dense` operand of the dot interaction.
//
// One launch per layer: a persistent CTA per SM walks 128 x BN output tiles
// (BN = 256 for the 512- and 256-wide layers, 128 for the last one):
//   warp 0      TMA producer: per 64-wide K block, a {64, 128} box of the
//               input activations and a {64, BN} box of the weights (PyTorch's
//               [N][K] layout is exactly the K-major B operand), 128-byte
//               swizzle, into an NS-stage ring
//   warp 1      TMEM allocation and MMA issue: M = 128, N = BN, K = 16 steps
//   warps 2..9  epilogue: TMEM lane quarter q = warp % 4 holds rows
//               32q..32q+31, shared by two warps that take alternate 32-column
//               slices; each thread takes its row's slices, adds the bias and
//               applies the ReLU; the warp's 32 x 32 fp16 slice goes to a
//               swizzled shared-memory buffer (64-byte swizzle: conflict-free
//               16-byte stores) and leaves by a TMA tensor store, two buffers
//               per warp so the next slice is built while one is written
// Two TMEM accumulators let the MMAs of tile i+1 run under the epilogue of
// tile i.  K need not be a multiple of 64: TMA fills columns past the tensor
// with zeros, and the last block issues only the 16-wide steps it needs.  The
// first layer's fp32 input is converted and zero-padded to 8 columns by a
// small kernel.  Every mbarrier wait is bounded (DLRM_STATUS_TIMEOUT).
#include <type_traits>

#include "dlrm_mlp.h"
#include "tcgen05.cuh"

namespace dlrm {
namespace {

using namespace tc;

constexpr int kBM = 128;           // output rows per tile (the MMA's M)
constexpr int kKB = 64;            // fp16 K elements per 128-byte shared-memory row
constexpr int kEpiWarps = 8;       // two per TMEM lane quarter, alternate 32-column slices
constexpr int kThreads = (2 + kEpiWarps) * 32;
constexpr int kMaxStages = 8;
constexpr int kSmemLimit = 232448; // 227 KB opt-in per block

__host__ __device__ inline int round_up8(int x) { return (x + 7) / 8 * 8; }

constexpr int kStageOut = kEpiWarps * 2 * 32 * 64;   // epilogue: 2 buffers x 32 rows x 64 bytes per warp

__host__ __device__ inline size_t layer_smem(int BN, int ns)
{
    return 1024 + (size_t)ns * (kBM * 128 + BN * 128) + kStageOut + (size_t)(2 * ns + 4) * 8 + 16;
}

__global__ void __launch_bounds__(kThreads, 1)
mlp_layer_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_w,
                 const __grid_constant__ CUtensorMap map_out, const float* __restrict__ bias, int M, int N, int K,
                 int BN, int NS, uint32_t tmem_cols, uint32_t* status)
{
    pdl_wait();
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    const int a_bytes = kBM * 128, stage_bytes = a_bytes + BN * 128;
    uint8_t* stages = smem;
    uint8_t* stage_out = smem + (size_t)NS * stage_bytes;   // 1024-byte aligned
    uint64_t* full = reinterpret_cast<uint64_t*>(stage_out + kStageOut);
    uint64_t* empty = full + NS;
    uint64_t* tfull = empty + NS;
    uint64_t* tempty = tfull + 2;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(tempty + 2);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

    const int warp = threadIdx.x / kWarp, lane = threadIdx.x % kWarp;
    const int n_tiles = N / BN;
    const int tiles = (M + kBM - 1) / kBM * n_tiles;
    const int kblocks = (K + kKB - 1) / kKB;
    const int last_steps = (K - (kblocks - 1) * kKB + 15) / 16;   // 16-wide K steps in the last block
    const uint32_t idesc = idesc_f16(kBM, BN);

    if (threadIdx.x == 0) {
        for (int i = 0; i < NS; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&tfull[i], 1);
            mbar_init(&tempty[i], kEpiWarps);
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_holder)),
                     "r"(tmem_cols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------------------------------------------- TMA producer
            int q = 0;
            bool ok = true;
            for (int t = blockIdx.x; ok && t < tiles; t += gridDim.x) {
                const int m0 = t / n_tiles * kBM, n0 = t % n_tiles * BN;
                for (int kb = 0; kb < kblocks; ++kb, ++q) {
                    const int stage = q % NS;
                    const uint32_t ph = (uint32_t)(q / NS) & 1u;
                    if (!mbar_wait(&empty[stage], ph ^ 1u, abort_flag)) {
                        ok = false;
                        break;
                    }
                    uint8_t* sa = stages + (size_t)stage * stage_bytes;
                    mbar_expect_tx(&full[stage], (uint32_t)stage_bytes);
                    tma_load_2d(sa, &map_a, kb * kKB, m0, &full[stage]);
                    tma_load_2d(sa + a_bytes, &map_w, kb * kKB, n0, &full[stage]);
                }
            }
            if (*abort_flag)   // the copies already issued must land before the CTA exits
                for (int j = (q > NS ? q - NS : 0); j < q; ++j) mbar_drain(&full[j % NS], (uint32_t)(j / NS) & 1u);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------------------------------------------- MMA issuer
            int q = 0, it = 0;
            bool ok = true;
            for (int t = blockIdx.x; ok && t < tiles; t += gridDim.x, ++it) {
                const int buf = it & 1;
                if (!mbar_wait(&tempty[buf], ((uint32_t)(it >> 1) & 1u) ^ 1u, abort_flag)) break;
                tc_fence_after();
                const uint32_t d = tmem_base + (uint32_t)(buf * BN);
                for (int kb = 0; kb < kblocks; ++kb, ++q) {
                    const int stage = q % NS;
                    if (!mbar_wait(&full[stage], (uint32_t)(q / NS) & 1u, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = smem_u32(stages + (size_t)stage * stage_bytes);
                    const int steps = kb == kblocks - 1 ? last_steps : kKB / 16;
                    for (int kk = 0; kk < steps; ++kk)
                        tc_mma_f16(d, sw128_desc(sa + kk * 32), sw128_desc(sa + a_bytes + kk * 32), idesc,
                                   (kb | kk) != 0);
                    tc_commit(&empty[stage]);
                }
                if (ok) tc_commit(&tfull[buf]);
            }
            if (*abort_flag && it > 0)   // MMAs already issued must finish before TMEM is freed
                mbar_drain(&tfull[(it - 1) & 1], (uint32_t)((it - 1) >> 1) & 1u);
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int quarter = warp & 3;
        const int half = (warp - 2) / 4;                      // which of the quarter's two warps
        // slices of CW columns: 32 (64-byte rows, 64-byte swizzle) or, for a
        // 16-wide tile, 16 (32-byte rows, 32-byte swizzle); the swizzle XORs
        // the 16-byte chunk index with address bits 7.. (row >> 1 or row >> 2)
        const int CW = BN % 32 == 0 ? 32 : 16;
        const int xs = CW == 32 ? ((lane >> 1) & 3) : ((lane >> 2) & 1);
        uint8_t* myout = stage_out + (size_t)(warp - 2) * (2 * 32 * 64);
        int it = 0, k = 0;                                    // k counts this warp's slices (buffer k & 1)
        for (int t = blockIdx.x; t < tiles; t += gridDim.x, ++it) {
            const int buf = it & 1;
            if (!mbar_wait(&tfull[buf], (uint32_t)(it >> 1) & 1u, abort_flag)) break;
            __syncwarp();
            tc_fence_after();
            const int m0 = t / n_tiles * kBM, n0 = t % n_tiles * BN;
            const uint32_t taddr = tmem_base + ((uint32_t)(32 * quarter) << 16) + (uint32_t)(buf * BN);
            // NC-column slice of the row: load, + bias, ReLU, fp16 into the buffer, TMA store
            auto slice = [&](auto nc, int c0) {
                constexpr int NC = decltype(nc)::value;
                uint32_t v[NC];
                if constexpr (NC == 32)
                    tmem_ld_x32(taddr + (uint32_t)c0, v);
                else
                    tmem_ld_x16(taddr + (uint32_t)c0, v);
                tmem_wait_ld(v);
                const float4* bq = reinterpret_cast<const float4*>(bias + n0 + c0);
                uint32_t h[NC / 2];
#pragma unroll
                for (int j = 0; j < NC / 4; ++j) {
                    const float4 bb = __ldg(bq + j);
                    h[2 * j] = h2_relu_bits(__uint_as_float(v[4 * j]) + bb.x, __uint_as_float(v[4 * j + 1]) + bb.y);
                    h[2 * j + 1] =
                        h2_relu_bits(__uint_as_float(v[4 * j + 2]) + bb.z, __uint_as_float(v[4 * j + 3]) + bb.w);
                }
                uint8_t* sb = myout + (k & 1) * (32 * 64);
                if (lane == 0) bulk_wait_read<1>();           // the store that last used this buffer has read it
                __syncwarp();
#pragma unroll
                for (int j = 0; j < NC / 8; ++j) {
                    const uint32_t dst = smem_u32(sb + lane * (NC * 2) + ((j ^ xs) << 4));
                    asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(dst), "r"(h[4 * j]), "r"(h[4 * j + 1]),
                                 "r"(h[4 * j + 2]), "r"(h[4 * j + 3])
                                 : "memory");
                }
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (lane == 0) {   // rows past M are clipped by the tensor store
                    tma_store_2d(&map_out, n0 + c0, m0 + 32 * quarter, sb);
                    bulk_commit();
                }
                ++k;
            };
            if (CW == 32) {
                for (int c0 = 32 * half; c0 < BN; c0 += 64) slice(std::integral_constant<int, 32>{}, c0);
            } else if (half == 0) {
                slice(std::integral_constant<int, 16>{}, 0);   // BN == 16: one slice
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[buf]);
        }
        if (lane == 0) bulk_wait_all();   // this warp's stores are complete before the CTA exits
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(tmem_cols)
                     : "memory");
    }
    if (threadIdx.x == 0 && *abort_flag) set_status(status, DLRM_STATUS_TIMEOUT);
}

// ----------------------------------------------------------- fused 3 layers
// The pages' bottom MLP, 16 (9..16 padded) -> 512 -> 256 -> 128, in one
// persistent launch: a CTA per SM walks 128-row tiles, and each tile's
// activations live in tensor memory, where the next layer's MMA reads them as
// its A operand, so only x goes in and the 128-wide output comes out.
//   TMEM (512 columns): an fp32 accumulator in columns 0..255 and the fp16
//   activations packed two to a column in 256..511.  Layer 1 runs as two
//   N = 256 halves into 0..255, each converted (bias, ReLU, fp16) into A2 at
//   256..383 and 384..511; layer 2 (K = 512 from A2) accumulates into 0..255
//   and is converted into A3 at 256..383; layer 3 (K = 256 from A3) accumulates
//   into 384..511 and leaves through shared memory by TMA tensor stores.
//   Shared memory: the x tile and W1 (resident), both as 32-byte rows (one
//   16-wide K step, 32-byte swizzle); a 5-stage ring of 32 KB weight boxes fed
//   by TMA in the order the MMAs use them (W2's eight K blocks, W3's four);
//   the output staging; the biases.
//   warp 0      TMA producer of the weight ring (and W1 once)
//   warp 1      TMEM allocation and MMA issue
//   warps 2..17 conversion: four warps per TMEM lane quarter, each two of a
//               layer's eight 32-column slices (both loads in flight) into 16
//               packed columns each; for layer 3 one slice, out by TMA store
//   warp 18     builds each x tile from the fp32 input (coalesced 16-byte
//               loads of the tile's contiguous rows, rounded to fp16 at their
//               swizzled places) as soon as the previous tile's layer 1 has
//               read the buffer
// A column range is overwritten only after its last reader: layer 1's second
// half waits for every warp's conversion of the first (lread), layer 2 for
// the second (bread), the next tile's layer 1 for layer 2's conversion (a3);
// A3 replaces A2 once layer 2's MMAs are complete, and the next tile's A2
// replaces A3 and layer 3's accumulator only after the same warps have
// drained layer 3 (program order).  Bit-identical to the per-layer kernels.
constexpr int kF3K0 = 16, kF3N1 = 512, kF3N2 = 256, kF3N3 = 128;
constexpr int kF3Epi = 16;
constexpr int kF3Threads = (3 + kF3Epi) * 32;   // producer, MMA, conversion warps, x-tile warp
constexpr int kF3Stages = 5;
constexpr int kF3StageBytes = 256 * 128;
constexpr int kF3XOff = 0;
constexpr int kF3W1Off = kF3XOff + kBM * 32;
constexpr int kF3RingOff = kF3W1Off + kF3N1 * 32;
constexpr int kF3OutOff = kF3RingOff + kF3Stages * kF3StageBytes;
constexpr int kF3BiasOff = kF3OutOff + kF3Epi * 32 * 64;
constexpr int kF3BarOff = kF3BiasOff + (kF3N1 + kF3N2 + kF3N3) * 4;
// barriers: xfull, xempty, w1full, full[S], empty[S], l1a, l1b, l2, l3, lread, bread, a3, drain
constexpr int kF3Bars = 3 + 2 * kF3Stages + 8;
constexpr size_t kF3Smem = 1024 + kF3BarOff + kF3Bars * 8 + 16;

__global__ void __launch_bounds__(kF3Threads, 1)
mlp3_fused_kernel(const float* __restrict__ x, int K0, const __grid_constant__ CUtensorMap map_w1,
                  const __grid_constant__ CUtensorMap map_w2, const __grid_constant__ CUtensorMap map_w3,
                  const __grid_constant__ CUtensorMap map_out, const float* __restrict__ b1,
                  const float* __restrict__ b2, const float* __restrict__ b3, int M, uint32_t* status,
                  long long wait_cycles)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint8_t* xs = smem + kF3XOff;
    uint8_t* w1s = smem + kF3W1Off;
    uint8_t* ring = smem + kF3RingOff;
    uint8_t* stage_out = smem + kF3OutOff;
    float* bias_s = reinterpret_cast<float*>(smem + kF3BiasOff);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kF3BarOff);
    uint64_t* xfull = bars;
    uint64_t* xempty = bars + 1;
    uint64_t* w1full = bars + 2;
    uint64_t* full = bars + 3;
    uint64_t* empty = full + kF3Stages;
    uint64_t* l1a = empty + kF3Stages;
    uint64_t* l1b = l1a + 1;
    uint64_t* l2 = l1a + 2;
    uint64_t* l3 = l1a + 3;
    uint64_t* lread = l1a + 4;   // layer 1's first half drained into A2 columns 256..383
    uint64_t* bread = l1a + 5;   // layer 1's second half drained into A2 columns 384..511
    uint64_t* a3 = l1a + 6;      // layer 2 drained into A3 columns 256..383 (columns 0..255 free)
    uint64_t* drain = l1a + 7;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + kF3Bars);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

    const int warp = threadIdx.x / kWarp, lane = threadIdx.x % kWarp;
    const int tiles = (M + kBM - 1) / kBM;

    if (threadIdx.x == 0) {
        mbar_init(xfull, 1);
        mbar_init(xempty, 1);
        mbar_init(w1full, 1);
        for (int i = 0; i < kF3Stages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        for (int i = 0; i < 4; ++i) mbar_init(&l1a[i], 1);
        mbar_init(lread, kF3Epi);
        mbar_init(bread, kF3Epi);
        mbar_init(a3, kF3Epi);
        mbar_init(drain, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_holder)),
                     "r"(512)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    pdl_wait();
    for (int i = threadIdx.x; i < kBM * 8; i += blockDim.x) reinterpret_cast<uint32_t*>(xs)[i] = 0u;
    for (int i = threadIdx.x; i < kF3N1 + kF3N2 + kF3N3; i += blockDim.x)
        bias_s[i] = i < kF3N1 ? b1[i] : (i < kF3N1 + kF3N2 ? b2[i - kF3N1] : b3[i - kF3N1 - kF3N2]);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;

    if (warp == 0) {
        // ------------------------------------------------------- TMA producer
        int q = 0;   // ring loads issued
        bool ok = true;
        auto ring_load = [&](const CUtensorMap* map, int c0, int c1, uint32_t bytes) {
            const int st = q % kF3Stages;
            if (!mbar_wait(&empty[st], ((uint32_t)(q / kF3Stages) & 1u) ^ 1u, abort_flag, wait_cycles)) return false;
            mbar_expect_tx(&full[st], bytes);
            tma_load_2d(ring + (size_t)st * kF3StageBytes, map, c0, c1, &full[st]);
            ++q;
            return true;
        };
        if (lane == 0 && blockIdx.x < tiles) {
            mbar_expect_tx(w1full, kF3N1 * 32);
            tma_load_2d(w1s, &map_w1, 0, 0, w1full);
            tma_load_2d(w1s + 256 * 32, &map_w1, 0, 256, w1full);
        }
        if (lane == 0)
            for (int t = blockIdx.x; ok && t < tiles; t += gridDim.x) {
                for (int kb = 0; ok && kb < kF3N1 / kKB; ++kb) ok = ring_load(&map_w2, kb * kKB, 0, kF3StageBytes);
                for (int kb = 0; ok && kb < kF3N2 / kKB; ++kb) ok = ring_load(&map_w3, kb * kKB, 0, kF3N3 * 128);
            }
        if (lane == 0 && *abort_flag) {
            for (int j = (q > kF3Stages ? q - kF3Stages : 0); j < q; ++j)
                mbar_drain(&full[j % kF3Stages], (uint32_t)(j / kF3Stages) & 1u);
            if (blockIdx.x < tiles) mbar_drain(w1full, 0);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // --------------------------------------------------- MMA issuer
            int q = 0, it = 0;
            bool ok = true, issued = false;
            const uint32_t id256 = idesc_f16(kBM, 256), id128 = idesc_f16(kBM, 128);
            auto ring_wait = [&]() -> int {
                const int st = q % kF3Stages;
                if (!mbar_wait(&full[st], (uint32_t)(q / kF3Stages) & 1u, abort_flag, wait_cycles)) return -1;
                tc_fence_after();
                return st;
            };
            for (int t = blockIdx.x; ok && t < tiles; t += gridDim.x, ++it) {
                const uint32_t par = (uint32_t)it & 1u;
                // layer 1, first half -> columns 0..255 (free once the previous tile's layer 2 is drained)
                if ((it == 0 && !mbar_wait(w1full, 0, abort_flag, wait_cycles)) ||
                    !mbar_wait(xfull, par, abort_flag, wait_cycles) || !mbar_wait(a3, par ^ 1u, abort_flag, wait_cycles))
                    break;
                tc_fence_after();
                const uint64_t xd = sw32_desc(smem_u32(xs));
                tc_mma_f16(tmem_base, xd, sw32_desc(smem_u32(w1s)), id256, 0);
                issued = true;
                tc_commit(l1a);
                // second half -> columns 0..255 again, once the first is drained
                if (!mbar_wait(lread, par, abort_flag, wait_cycles)) break;
                tc_fence_after();
                tc_mma_f16(tmem_base, xd, sw32_desc(smem_u32(w1s + 256 * 32)), id256, 0);
                tc_commit(xempty);
                tc_commit(l1b);
                // layer 2: A = A2 in TMEM columns 256..511, accumulator columns 0..255
                if (!mbar_wait(bread, par, abort_flag, wait_cycles)) break;
                tc_fence_after();
                int st;
                for (int kb = 0; ok && kb < kF3N1 / kKB; ++kb) {
                    if ((st = ring_wait()) < 0) {
                        ok = false;
                        break;
                    }
                    const uint32_t wa = smem_u32(ring + (size_t)st * kF3StageBytes);
                    for (int kk = 0; kk < kKB / 16; ++kk)
                        tc_mma_f16_ts(tmem_base, tmem_base + 256 + (uint32_t)(32 * kb + 8 * kk), sw128_desc(wa + kk * 32),
                                      id256, (kb | kk) != 0);
                    tc_commit(&empty[st]);
                    ++q;
                }
                if (!ok) break;
                tc_commit(l2);
                // layer 3: A = A3 in TMEM columns 256..383, accumulator columns 384..511
                if (!mbar_wait(a3, par, abort_flag, wait_cycles)) break;
                tc_fence_after();
                for (int kb = 0; ok && kb < kF3N2 / kKB; ++kb) {
                    if ((st = ring_wait()) < 0) {
                        ok = false;
                        break;
                    }
                    const uint32_t wa = smem_u32(ring + (size_t)st * kF3StageBytes);
                    for (int kk = 0; kk < kKB / 16; ++kk)
                        tc_mma_f16_ts(tmem_base + 384, tmem_base + 256 + (uint32_t)(32 * kb + 8 * kk),
                                      sw128_desc(wa + kk * 32), id128, (kb | kk) != 0);
                    tc_commit(&empty[st]);
                    ++q;
                }
                if (!ok) break;
                tc_commit(l3);
            }
            if (*abort_flag && issued) {
                tc_commit(drain);
                mbar_drain(drain, 0);
            }
        }
    } else if (warp == 2 + kF3Epi) {
        // ----------------------------------------------------------- x tiles
        // each tile's x rows are one contiguous run of fp32: element i of it is
        // row i / K0, column i % K0, rounded to fp16 at its swizzled place
        const int64_t xn = (int64_t)M * K0;
        int it = 0;
        for (int t = blockIdx.x; t < tiles; t += gridDim.x, ++it) {
            int w = 1;
            if (lane == 0) w = mbar_wait(xempty, ((uint32_t)it & 1u) ^ 1u, abort_flag, wait_cycles);
            if (!__shfl_sync(0xffffffffu, w, 0)) break;
            const int64_t base = (int64_t)t * kBM * K0;
            const float4* x4 = reinterpret_cast<const float4*>(x + base);
            for (int u0 = 0; u0 < K0; u0 += 8) {
                float4 v[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int64_t i = base + 4 * (lane + kWarp * (u0 + u));
                    v[u] = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (u0 + u < K0) {
                        if (i + 4 <= xn) {
                            v[u] = __ldg(x4 + lane + kWarp * (u0 + u));
                        } else if (i < xn) {
                            v[u].x = x[i];
                            if (i + 1 < xn) v[u].y = x[i + 1];
                            if (i + 2 < xn) v[u].z = x[i + 2];
                        }
                    }
                }
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    if (u0 + u >= K0) break;
                    const float f[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int i = 4 * (lane + kWarp * (u0 + u)) + e;
                        const int r = i / K0, c = i - r * K0;
                        const uint32_t off = (uint32_t)r * 32 + ((uint32_t)((c >> 3) ^ ((r >> 2) & 1)) << 4) +
                                             (uint32_t)(c & 7) * 2;
                        *reinterpret_cast<__half*>(xs + off) = __float2half_rn(f[e]);
                    }
                }
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // generic writes -> the MMA
            __syncwarp();
            if (lane == 0) mbar_arrive(xfull);
        }
    } else {
        const int quarter = warp & 3;
        const int sub = (warp - 2) / 4;
        const uint32_t trow = tmem_base + ((uint32_t)(32 * quarter) << 16);
        const int xs64 = (lane >> 1) & 3;
        uint8_t* myout = stage_out + (size_t)(warp - 2) * (32 * 64);
        auto finish32 = [&](const uint32_t (&v)[32], const float* bias, uint32_t (&h)[16]) {
            const float4* bq = reinterpret_cast<const float4*>(bias);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float4 bb = bq[j];
                h[2 * j] = h2_relu_bits(__uint_as_float(v[4 * j]) + bb.x, __uint_as_float(v[4 * j + 1]) + bb.y);
                h[2 * j + 1] =
                    h2_relu_bits(__uint_as_float(v[4 * j + 2]) + bb.z, __uint_as_float(v[4 * j + 3]) + bb.w);
            }
        };
        // 256 accumulator columns (from 0) -> 128 packed columns from dst0: slices sub and sub + 4
        auto convert = [&](const float* bias, uint32_t dst0, uint64_t* done) {
            const int j0 = sub, j1 = sub + 4;
            uint32_t v0[32], v1[32], h[16];
            tmem_ld_x32(trow + (uint32_t)(32 * j0), v0);
            tmem_ld_x32(trow + (uint32_t)(32 * j1), v1);
            tmem_wait_ld2(v0, v1);
            finish32(v0, bias + 32 * j0, h);
            tmem_st_x16(trow + dst0 + (uint32_t)(16 * j0), h);
            finish32(v1, bias + 32 * j1, h);
            tmem_st_x16(trow + dst0 + (uint32_t)(16 * j1), h);
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(done);
        };
        int it = 0;
        for (int t = blockIdx.x; t < tiles; t += gridDim.x, ++it) {
            const uint32_t par = (uint32_t)it & 1u;
            const int m0 = t * kBM;
            if (!mbar_wait(l1a, par, abort_flag, wait_cycles)) break;
            __syncwarp();
            tc_fence_after();
            convert(bias_s, 256, lread);
            if (!mbar_wait(l1b, par, abort_flag, wait_cycles)) break;
            __syncwarp();
            tc_fence_after();
            convert(bias_s + 256, 384, bread);
            if (!mbar_wait(l2, par, abort_flag, wait_cycles)) break;
            __syncwarp();
            tc_fence_after();
            convert(bias_s + kF3N1, 256, a3);
            if (!mbar_wait(l3, par, abort_flag, wait_cycles)) break;
            __syncwarp();
            tc_fence_after();
            {
                const int c0 = 32 * sub;
                uint32_t v[32], h[16];
                tmem_ld_x32(trow + 384 + (uint32_t)c0, v);
                tmem_wait_ld(v);
                finish32(v, bias_s + kF3N1 + kF3N2 + c0, h);
                if (lane == 0) bulk_wait_read<0>();
                __syncwarp();
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint32_t dst = smem_u32(myout + lane * 64 + ((j ^ xs64) << 4));
                    asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(dst), "r"(h[4 * j]), "r"(h[4 * j + 1]),
                                 "r"(h[4 * j + 2]), "r"(h[4 * j + 3])
                                 : "memory");
                }
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (lane == 0) {
                    tma_store_2d(&map_out, c0, m0 + 32 * quarter, myout);
                    bulk_commit();
                }
            }
        }
        if (lane == 0) bulk_wait_all();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(512) : "memory");
    }
    if (threadIdx.x == 0 && *abort_flag) set_status(status, DLRM_STATUS_TIMEOUT);
}

// x (fp32 [M][K]) -> fp16 [M][Kp], pad columns zero.
__global__ void cast_pad_kernel(const float* __restrict__ x, int64_t M, int K, int Kp, __half* __restrict__ x16)
{
    pdl_wait();
    const int64_t n = M * Kp;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = i / Kp;
        const int c = (int)(i - r * Kp);
        x16[i] = c < K ? __float2half_rn(x[r * K + c]) : __float2half_rn(0.f);
    }
}

int tile_n(int N)
{
    for (int bn = 256; bn >= 16; bn /= 2)
        if (bn <= N && N % bn == 0) return bn;
    return 0;
}

dlrm_status launch_layer(const __half* a, int lda, const __half* w, const float* bias, __half* out, int M, int N,
                         uint32_t* status, cudaStream_t st)
{
    EncodeTiledFn enc = encode_fn();
    if (!enc) return fail(DLRM_ERR_CUDA, "dlrm_bottom_mlp_fwd: cuTensorMapEncodeTiled unavailable");
    const int BN = tile_n(N);
    int ns = kMaxStages;
    while (ns > 2 && layer_smem(BN, ns) > (size_t)kSmemLimit) --ns;
    const size_t smem = layer_smem(BN, ns);
    uint32_t tmem_cols = 32;
    while (tmem_cols < (uint32_t)(2 * BN)) tmem_cols *= 2;
    const cuuint32_t ones[2] = {1, 1};
    CUtensorMap ma, mw;
    const cuuint64_t adims[2] = {(cuuint64_t)lda, (cuuint64_t)M};
    const cuuint64_t astr[1] = {(cuuint64_t)lda * 2};
    const cuuint32_t abox[2] = {(cuuint32_t)kKB, (cuuint32_t)kBM};
    CUresult r = enc(&ma, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<__half*>(a), adims, astr, abox, ones,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(DLRM_ERR_CUDA, "dlrm_bottom_mlp_fwd: activation tensor map (%d)", (int)r);
    const cuuint64_t wdims[2] = {(cuuint64_t)lda, (cuuint64_t)N};
    const cuuint32_t wbox[2] = {(cuuint32_t)kKB, (cuuint32_t)BN};
    r = enc(&mw, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<__half*>(w), wdims, astr, wbox, ones,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(DLRM_ERR_CUDA, "dlrm_bottom_mlp_fwd: weight tensor map (%d)", (int)r);
    CUtensorMap mo;
    const int CW = BN % 32 == 0 ? 32 : 16;
    const cuuint64_t odims[2] = {(cuuint64_t)N, (cuuint64_t)M};
    const cuuint64_t ostr[1] = {(cuuint64_t)N * 2};
    const cuuint32_t obox[2] = {(cuuint32_t)CW, 32};
    r = enc(&mo, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, out, odims, ostr, obox, ones, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CW == 32 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(DLRM_ERR_CUDA, "dlrm_bottom_mlp_fwd: output tensor map (%d)", (int)r);
    const int tiles = (M + kBM - 1) / kBM * (N / BN);
    const int grid = tiles < num_sms() ? tiles : num_sms();
    cudaError_t e = cudaFuncSetAttribute(mlp_layer_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return fail(DLRM_ERR_CUDA, "dlrm_bottom_mlp_fwd: %s", cudaGetErrorString(e));
    return check_launch_pdl(launch_pdl(mlp_layer_kernel, grid, kThreads, smem, st, ma, mw, mo, bias, M, N, lda, BN, ns,
                                       tmem_cols, status),
                            "mlp_layer_kernel");
}

// The pages' 13 -> 512 -> 256 -> 128 shape (x padded to 16 columns) runs fused.
bool fused3_shape(int n_layers, const int* dims)
{
    return n_layers == 3 && round_up8(dims[0]) == kF3K0 && dims[1] == kF3N1 && dims[2] == kF3N2 && dims[3] == kF3N3;
}

dlrm_status launch_fused3(const float* x, int K0, const __half* w, const float* bias, __half* out, int M,
                          uint32_t* status, cudaStream_t st)
{
    EncodeTiledFn enc = encode_fn();
    if (!enc) return fail(DLRM_ERR_CUDA, "dlrm_bottom_mlp_fwd: cuTensorMapEncodeTiled unavailable");
    const cuuint32_t ones[2] = {1, 1};
    // K-major fp16 operand [rows][cols], {64, box_rows} boxes, 128-byte swizzle
    auto operand = [&](CUtensorMap* m, const __half* p, int cols, int rows, int box_rows) {
        const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
        const cuuint64_t str[1] = {(cuuint64_t)cols * 2};
        const cuuint32_t box[2] = {(cuuint32_t)kKB, (cuuint32_t)box_rows};
        return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<__half*>(p), dims, str, box, ones,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    };
    const __half* w1 = w;
    const __half* w2 = w1 + (size_t)kF3N1 * kF3K0;
    const __half* w3 = w2 + (size_t)kF3N2 * kF3N1;
    // 16-wide K operands: {16, box_rows} boxes of 32-byte rows, 32-byte swizzle
    auto narrow = [&](CUtensorMap* m, const __half* p, int rows, int box_rows) {
        const cuuint64_t dims[2] = {(cuuint64_t)kF3K0, (cuuint64_t)rows};
        const cuuint64_t str[1] = {(cuuint64_t)kF3K0 * 2};
        const cuuint32_t box[2] = {(cuuint32_t)kF3K0, (cuuint32_t)box_rows};
        return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<__half*>(p), dims, str, box, ones,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_32B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    };
    CUtensorMap m1, m2, m3, mo;
    CUresult r = narrow(&m1, w1, kF3N1, 256);
    if (r == CUDA_SUCCESS) r = operand(&m2, w2, kF3N1, kF3N2, 256);
    if (r == CUDA_SUCCESS) r = operand(&m3, w3, kF3N2, kF3N3, kF3N3);
    if (r != CUDA_SUCCESS) return fail(DLRM_ERR_CUDA, "dlrm_bottom_mlp_fwd: operand tensor map (%d)", (int)r);
    const cuuint64_t odims[2] = {(cuuint64_t)kF3N3, (cuuint64_t)M};
    const cuuint64_t ostr[1] = {(cuuint64_t)kF3N3 * 2};
    const cuuint32_t obox[2] = {32, 32};
    r = enc(&mo, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, out, odims, ostr, obox, ones, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(DLRM_ERR_CUDA, "dlrm_bottom_mlp_fwd: output tensor map (%d)", (int)r);
    const int tiles = (M + kBM - 1) / kBM;
    const int grid = tiles < num_sms() ? tiles : num_sms();
    cudaError_t e = cudaFuncSetAttribute(mlp3_fused_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kF3Smem);
    if (e != cudaSuccess) return fail(DLRM_ERR_CUDA, "dlrm_bottom_mlp_fwd: %s", cudaGetErrorString(e));
    return check_launch_pdl(launch_pdl(mlp3_fused_kernel, grid, kF3Threads, kF3Smem, st, x, K0, m1, m2, m3, mo, bias,
                                       bias + kF3N1, bias + kF3N1 + kF3N2, M, status, wait_limit_cycles()),
                            "mlp3_fused_kernel");
}

// Workspace: x as fp16 [B][round_up8(dims[0])], then each hidden layer's
// output [B][dims[l+1]], l = 0..n_layers-2, each piece 256-byte aligned.
bool mlp_dims_ok(int B, int n_layers, const int* dims)
{
    if (B < 0 || n_layers < 1 || n_layers > 64 || !dims) return false;
    for (int l = 0; l <= n_layers; ++l)
        if (dims[l] < 1 || dims[l] > 65536) return false;
    return true;
}

}  // namespace
}  // namespace dlrm

using namespace dlrm;

extern "C" size_t dlrm_bottom_mlp_workspace_size(int B, int n_layers, const int* dims)
{
    if (!mlp_dims_ok(B, n_layers, dims)) return 0;
    size_t bytes = dlrm_ws_align((size_t)B * round_up8(dims[0]) * 2);
    for (int l = 0; l + 1 < n_layers; ++l) bytes += dlrm_ws_align((size_t)B * dims[l + 1] * 2);
    return bytes;
}

extern "C" dlrm_status dlrm_bottom_mlp_fwd(const float* d_x, int B, int n_layers, const int* dims,
                                           const void* d_weights, const float* d_biases, void* d_out,
                                           void* d_workspace, size_t ws_bytes, uint32_t* d_status, void* stream)
{
    DLRM_API_RANGE("dlrm_bottom_mlp_fwd");
    clear_error();
    if (!mlp_dims_ok(B, n_layers, dims))
        return fail(DLRM_ERR_INVALID_ARG, "dlrm_bottom_mlp_fwd: need B >= 0, 1..64 layers, widths in [1, 65536]");
    for (int l = 1; l <= n_layers; ++l)
        if (dims[l] % 16 != 0)
            return fail(DLRM_ERR_UNSUPPORTED, "dlrm_bottom_mlp_fwd: layer widths must be multiples of 16 (dims[%d] = %d)",
                        l, dims[l]);
    if (B == 0) return DLRM_OK;
    if (!d_x || !d_weights || !d_biases || !d_out || !d_workspace)
        return fail(DLRM_ERR_INVALID_ARG, "dlrm_bottom_mlp_fwd: null device pointer");
    if (!aligned16(d_x) || !aligned16(d_weights) || !aligned16(d_biases) || !aligned16(d_out) ||
        ((uintptr_t)d_workspace & 255) != 0)
        return fail(DLRM_ERR_UNSUPPORTED, "dlrm_bottom_mlp_fwd: pointers must be 16-byte (workspace 256-byte) aligned");
    const size_t need = dlrm_bottom_mlp_workspace_size(B, n_layers, dims);
    if (ws_bytes < need)
        return fail(DLRM_ERR_WORKSPACE, "dlrm_bottom_mlp_fwd: workspace %zu bytes < %zu", ws_bytes, need);
    cudaStream_t st = as_stream(stream);
    if (fused3_shape(n_layers, dims))
        return launch_fused3(d_x, dims[0], static_cast<const __half*>(d_weights), d_biases,
                             static_cast<__half*>(d_out), B, d_status, st);
    uint8_t* ws = static_cast<uint8_t*>(d_workspace);
    const int Kp0 = round_up8(dims[0]);
    __half* x16 = reinterpret_cast<__half*>(ws);
    size_t off = dlrm_ws_align((size_t)B * Kp0 * 2);
    {
        const int64_t n = (int64_t)B * Kp0;
        int64_t blocks = (n + 255) / 256;
        if (blocks > (int64_t)num_sms() * 8) blocks = (int64_t)num_sms() * 8;
        const cudaError_t e = launch_pdl(cast_pad_kernel, (int)blocks, 256, 0, st, d_x, (int64_t)B, dims[0], Kp0, x16);
        if (e != cudaSuccess) return check_launch_pdl(e, "cast_pad_kernel");
        dlrm_status s = check_launch("cast_pad_kernel");
        if (s != DLRM_OK) return s;
    }
    const __half* in = x16;
    int lda = Kp0;
    const __half* w = static_cast<const __half*>(d_weights);
    const float* b = d_biases;
    for (int l = 0; l < n_layers; ++l) {
        const int N = dims[l + 1];
        __half* o = l + 1 == n_layers ? static_cast<__half*>(d_out) : reinterpret_cast<__half*>(ws + off);
        if (l + 1 < n_layers) off += dlrm_ws_align((size_t)B * N * 2);
        dlrm_status s = launch_layer(in, lda, w, b, o, B, N, d_status, st);
        if (s != DLRM_OK) return s;
        w += (size_t)N * lda;
        b += N;
        in = o;
        lda = N;
    }
    return DLRM_OK;
}
