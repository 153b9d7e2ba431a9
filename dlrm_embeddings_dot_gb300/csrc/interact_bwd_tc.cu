// interact_bwd_tc.cu -- gradient of the dot interaction on the tcgen05 tensor
// cores, fp16 tensors with fp32 accumulation ("DLRM For PyTorch", §Model
// architecture; §Mixed precision training: fp16 interaction, static loss
// scaling, so the gradients here carry the loss scale).
//
// Per sample, with G the upstream gradient row and M the symmetric
// (F+1)x(F+1) matrix M_pq = M_qp = G[D + p(p-1)/2 + q] (p > q), M_pp = 0:
//   dZ = M Z,  grad_dense = G[0..D) + dZ_0,  grad_pooled[t] = dZ_{t+1}.
//
// Four samples form one tile.  The B operand is exactly the forward's stage
// tile: per 64-feature block, rows 32s..32s+F-1 hold sample s's embedding
// rows (rows F..31 zero from TMA's fill) and rows 128..131 the dense rows
// (132..143 zero).  Read as an MN-major operand (features contiguous) it is
// Z^T with K = 144 rows: 128-byte swizzle, 8-row groups 1 KB apart (stride
// byte offset) and 64-feature blocks one stage block apart (leading byte
// offset).  The A operand (K-major, 128 x 144) holds, for sample s:
//   row 32s+i, i < F:   M_{i+1, j+1} at column 32s+j, M_{i+1, 0} at column 128+s
//   row 32s+31:         M_{0, j+1} at column 32s+j
// and zeros elsewhere, so one chain of 9 tcgen05.mma (M = 128, N = D, K = 16
// each) leaves dZ_{i+1} in TMEM lane 32s+i and dZ_0 in lane 32s+31.
//   warp 0      TMA producer of the Z tiles (as in the forward)
//   warp 1      TMEM allocation and MMA issue
//   warps 2..5  epilogue: lane quarter q = sample q; 64-feature blocks of the
//               32 rows staged swizzled, one TMA store each (rows F..31 fall
//               outside grad_pooled and are clipped); grad_dense by plain stores
//   warps 6..9  builders: sample s of the tile's G row (prefetched a tile
//               ahead) -> its rows of A
// Every mbarrier wait is bounded (DLRM_STATUS_TIMEOUT on expiry).
#include "interact_tc.cuh"
#include "tcgen05.cuh"

namespace dlrm {
namespace {

using namespace tc;

constexpr int kGroup = 4;                 // samples per tile
constexpr int kSlot = 32;                 // rows per sample slot (F <= 31: row 31 is dZ_0)
constexpr int kM = kGroup * kSlot;        // 128
constexpr int kDenseRows = 16;            // Z rows 128..143
constexpr int kK = kM + kDenseRows;       // 144
constexpr int kKB = 64;
constexpr int kZBlockBytes = (kM + kDenseRows) * 128;   // 18 KB per 64-feature block
constexpr int kABlockBytes = kM * 128;                  // 16 KB per 64-wide block of A's K
constexpr int kABytes = 3 * kABlockBytes;               // K = 144 in three 64-wide blocks
constexpr int kThreads = 320;
constexpr int kMaxStages = 4;
constexpr int kSmemLimit = 232448;

struct BwdLayout {
    int z_bytes, stage_bytes, ns;
    size_t smem;
};

constexpr int kOutStage = 4 * 2 * 32 * 128;   // epilogue: 4 warps x 2 buffers x 32 rows x 128 bytes
constexpr int kGdScratch = 4 * 512;           // epilogue: each warp's sample's G[0..D), D <= 256

__host__ __device__ inline size_t bwd_smem(int KH, int P, int ns)
{
    const size_t g_bytes = (size_t)kGroup * 2 * ((P * 2 + 15) / 16 * 16);   // two G rows per builder
    return 1024 + (size_t)ns * ((size_t)KH * kZBlockBytes + kABytes) + kOutStage + kGdScratch + g_bytes +
           (size_t)(3 * ns + 4) * 8 + 16;
}

__device__ __forceinline__ uint16_t ld_h(const uint16_t* g, int i) { return g[i]; }

__global__ void __launch_bounds__(kThreads, 1)
interact_bwd_tc_kernel(const __grid_constant__ CUtensorMap map_pooled, const __grid_constant__ CUtensorMap map_dense,
                       const __grid_constant__ CUtensorMap map_gpooled, const __half* __restrict__ grad_out,
                       __half* __restrict__ grad_dense, int F, int D, int B, int P, int KH, int NS,
                       uint32_t tmem_cols, uint32_t* status, long long wait_cycles)
{
    pdl_wait();
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    const int z_bytes = KH * kZBlockBytes;
    const int stage_bytes = z_bytes + kABytes;          // both multiples of 1 KB
    const int gpitch = (P * 2 + 15) / 16 * 16;          // bytes per staged G row
    uint8_t* stages = smem;
    uint8_t* ostage = smem + (size_t)NS * stage_bytes;      // 1 KB aligned
    uint8_t* gdscr = ostage + kOutStage;
    uint8_t* gstage = gdscr + kGdScratch;
    uint64_t* full = reinterpret_cast<uint64_t*>(gstage + kGroup * 2 * gpitch);   // Z copies landed
    uint64_t* built = full + NS;                                                    // A tile built
    uint64_t* empty = built + NS;
    uint64_t* tfull = empty + NS;
    uint64_t* tempty = tfull + 2;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(tempty + 2);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

    const int warp = threadIdx.x / kWarp, lane = threadIdx.x % kWarp;
    const int ntiles = (B + kGroup - 1) / kGroup;
    const uint32_t idesc = idesc_f16(kM, D) | (1u << 16);   // B operand MN-major

    if (threadIdx.x == 0) {
        for (int i = 0; i < NS; ++i) {
            mbar_init(&full[i], 1);        // the TMA producer's arrive.expect_tx
            mbar_init(&built[i], kGroup);  // the four builders (apart, so an abort can drain the copies alone)
            mbar_init(&empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&tfull[i], 1);
            mbar_init(&tempty[i], kGroup);
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    // Zero once: every A tile (only the diagonal blocks and dense columns are
    // rewritten per tile) and the Z rows 132..143 no copy writes.
    for (int s = 0; s < NS; ++s) {
        uint4* a = reinterpret_cast<uint4*>(stages + (size_t)s * stage_bytes + z_bytes);
        for (int x = threadIdx.x; x < kABytes / 16; x += kThreads) a[x] = make_uint4(0, 0, 0, 0);
        for (int kb = 0; kb < KH; ++kb) {
            uint4* z = reinterpret_cast<uint4*>(stages + (size_t)s * stage_bytes + kb * kZBlockBytes + kM * 128 +
                                                kGroup * 128);
            for (int x = threadIdx.x; x < (kDenseRows - kGroup) * 128 / 16; x += kThreads) z[x] = make_uint4(0, 0, 0, 0);
        }
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
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
            // ------------------------------------------------ TMA producer (Z)
            int it = 0;
            for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++it) {
                const int stage = it % NS;
                if (!mbar_wait(&empty[stage], ((uint32_t)(it / NS) & 1u) ^ 1u, abort_flag, wait_cycles)) break;
                uint8_t* sb = stages + (size_t)stage * stage_bytes;
                mbar_expect_tx(&full[stage], (uint32_t)KH * (kM * 128 + kGroup * 128));
                for (int kb = 0; kb < KH; ++kb) {
                    tma_load_3d(sb + kb * kZBlockBytes, &map_pooled, kb * kKB, 0, tile * kGroup, &full[stage]);
                    tma_load_2d(sb + kb * kZBlockBytes + kM * 128, &map_dense, kb * kKB, tile * kGroup, &full[stage]);
                }
            }
            if (*abort_flag)   // the copies already issued must land before the CTA exits
                for (int j = (it > NS ? it - NS : 0); j < it; ++j) mbar_drain(&full[j % NS], (uint32_t)(j / NS) & 1u);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------------------------ MMA issuer
            int it = 0;
            for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++it) {
                const int stage = it % NS, buf = it & 1;
                if (!mbar_wait(&tempty[buf], ((uint32_t)(it >> 1) & 1u) ^ 1u, abort_flag, wait_cycles)) break;
                tc_fence_after();
                if (!mbar_wait(&full[stage], (uint32_t)(it / NS) & 1u, abort_flag, wait_cycles)) break;
                if (!mbar_wait(&built[stage], (uint32_t)(it / NS) & 1u, abort_flag, wait_cycles)) break;
                tc_fence_after();
                const uint32_t zb = smem_u32(stages + (size_t)stage * stage_bytes);
                const uint32_t ab = zb + (uint32_t)z_bytes;
                const uint32_t d = tmem_base + (uint32_t)(buf * D);
#pragma unroll
                for (int kk = 0; kk < kK / 16; ++kk) {
                    const uint64_t adesc = sw128_desc(ab + (kk / 4) * kABlockBytes + (kk % 4) * 32);
                    const uint64_t bdesc = sw128_desc_mn(zb + kk * 2048, (uint32_t)kZBlockBytes, 1024);
                    tc_mma_f16(d, adesc, bdesc, idesc, kk != 0);
                }
                tc_commit(&empty[stage]);
                tc_commit(&tfull[buf]);
            }
            if (*abort_flag && it > 0) mbar_drain(&tfull[(it - 1) & 1], (uint32_t)((it - 1) >> 1) & 1u);
        }
    } else if (warp < 6) {
        // ---------------------------------------------------- epilogue
        // Lane i holds row i of the sample's 32-row slot.  Each 64-feature
        // block of rows 0..31 goes to a 128-byte-swizzled staging buffer and
        // leaves by one TMA store of the box {64, 32, 1} of grad_pooled viewed as
        // [B][F][D]: rows F..31 lie outside the tensor and are not written.
        // Row 31 (dZ_0) becomes grad_dense = G[0..D) + dZ_0 by plain stores.
        const int q = warp & 3;                     // TMEM lane quarter == sample in tile
        uint8_t* myout = ostage + (size_t)q * (2 * 32 * 128);
        uint4* gd_s = reinterpret_cast<uint4*>(gdscr + q * 512);
        // the sample's G[0..D) (the dense pass-through), loaded a tile ahead
        auto load_gd = [&](int tile) {
            const int64_t b = (int64_t)tile * kGroup + q;
            return (tile < ntiles && b < B && lane < D / 8) ? ldg_nc_v4(grad_out + b * P + 8 * lane)
                                                             : make_uint4(0, 0, 0, 0);
        };
        uint4 gnext = load_gd(blockIdx.x);
        int it = 0, k = 0;                          // k counts this warp's staged blocks (buffer k & 1)
        for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++it) {
            const int buf = it & 1;
            const uint4 gcur = gnext;
            gnext = load_gd(tile + gridDim.x);
            if (!mbar_wait(&tfull[buf], (uint32_t)(it >> 1) & 1u, abort_flag, wait_cycles)) break;
            if (lane < D / 8) gd_s[lane] = gcur;
            __syncwarp();
            tc_fence_after();
            const int64_t b = (int64_t)tile * kGroup + q;
            const bool live = b < B;
            const uint32_t taddr = tmem_base + ((uint32_t)(kSlot * q) << 16) + (uint32_t)(buf * D);
            for (int c0 = 0; c0 < D; c0 += kKB) {
                uint32_t h[32];
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    uint32_t v[32];
                    tmem_ld_x32(taddr + (uint32_t)(c0 + 32 * half), v);
                    tmem_wait_ld(v);
                    float add[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) add[j] = 0.f;
                    if (live && lane == kSlot - 1) {   // dense pass-through G[0..D)
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            float f[8];
                            h8_to_f8(gd_s[(c0 + 32 * half) / 8 + j], f);
#pragma unroll
                            for (int e = 0; e < 8; ++e) add[8 * j + e] = f[e];
                        }
                    }
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        h[16 * half + j] = h2_bits(__uint_as_float(v[2 * j]) + add[2 * j],
                                                   __uint_as_float(v[2 * j + 1]) + add[2 * j + 1]);
                }
                if (live && lane == kSlot - 1) {
                    uint4* o = reinterpret_cast<uint4*>(grad_dense + b * D + c0);
#pragma unroll
                    for (int j = 0; j < 8; ++j) stg_cs_v4(o + j, make_uint4(h[4 * j], h[4 * j + 1], h[4 * j + 2], h[4 * j + 3]));
                }
                uint8_t* sbuf = myout + (k & 1) * (32 * 128);
                if (lane == 0) bulk_wait_read<1>();   // the store that last used this buffer has read it
                __syncwarp();
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    *reinterpret_cast<uint4*>(sbuf + lane * 128 + ((j ^ (lane & 7)) << 4)) =
                        make_uint4(h[4 * j], h[4 * j + 1], h[4 * j + 2], h[4 * j + 3]);
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (lane == 0 && live) {
                    tma_store_3d(&map_gpooled, c0, 0, (int)b, sbuf);
                    bulk_commit();
                }
                ++k;
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[buf]);
        }
        if (lane == 0) bulk_wait_all();
    } else {
        // ---------------------------------------------------- builders of A
        const int s = warp - 6;                     // sample slot of the tile
        // The sample's G row is staged in shared memory, two buffers: the next
        // tile's row is loaded into registers while this tile's A is built.
        const int gchunks = gpitch / 16;            // <= 4 * kWarp (out_cols <= 1024)
        uint8_t* grows = gstage + s * 2 * gpitch;
        const int row = kSlot * s + lane;           // A row (TMEM lane) this lane builds
        auto load_g = [&](int64_t tile, uint4 (&r)[4]) {
            const int64_t b = tile * kGroup + s;
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int c = lane + kWarp * u;
                r[u] = (tile < ntiles && b < B && c < gchunks) ? ldg_nc_v4(grad_out + b * P + 8 * c)
                                                                : make_uint4(0, 0, 0, 0);
            }
        };
        auto put_g = [&](int bufi, const uint4 (&r)[4]) {
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int c = lane + kWarp * u;
                if (c < gchunks) *reinterpret_cast<uint4*>(grows + bufi * gpitch + 16 * c) = r[u];
            }
        };
        {
            uint4 r0[4];
            load_g(blockIdx.x, r0);
            put_g(0, r0);
        }
        int it = 0;
        for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++it) {
            const int stage = it % NS;
            uint4 rn[4];
            load_g((int64_t)tile + gridDim.x, rn);   // next tile's row, in flight during the build
            const uint16_t* gh = reinterpret_cast<const uint16_t*>(grows + (it & 1) * gpitch);
            __syncwarp();
            int ok = 1;
            if (lane == 0) ok = mbar_wait(&empty[stage], ((uint32_t)(it / NS) & 1u) ^ 1u, abort_flag, wait_cycles);
            if (!__shfl_sync(0xffffffffu, ok, 0)) break;
            __syncwarp();
            // Z index of this row: p = lane + 1 for embedding rows, 0 for row 31 (dZ_0)
            const bool live = lane < F || lane == kSlot - 1;
            const int p = lane == kSlot - 1 ? 0 : lane + 1;
            auto m_at = [&](int a, int c) -> uint16_t {   // M_ac, a != c
                const int hi = a > c ? a : c, lo = a > c ? c : a;
                return ld_h(gh, D + hi * (hi - 1) / 2 + lo);
            };
            uint8_t* ab = stages + (size_t)stage * stage_bytes + z_bytes;
            // own 32 columns: K = 32s..32s+31 -> block s/2, 16-byte chunks 4(s%2)..4(s%2)+3
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint16_t e[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const int j = 8 * c + k;       // column j of the slot: Z index j + 1
                    e[k] = (live && j < F && j + 1 != p) ? m_at(p, j + 1) : (uint16_t)0;
                }
                const int chunk = 4 * (s & 1) + c;
                *reinterpret_cast<uint4*>(ab + (s >> 1) * kABlockBytes + row * 128 + ((chunk ^ (row & 7)) << 4)) =
                    *reinterpret_cast<const uint4*>(e);
            }
            {   // dense column 128 + s: block 2, chunk 0, element s
                uint16_t e[8] = {0, 0, 0, 0, 0, 0, 0, 0};
                if (lane < F) e[s] = m_at(p, 0);
                *reinterpret_cast<uint4*>(ab + 2 * kABlockBytes + row * 128 + ((0 ^ (row & 7)) << 4)) =
                    *reinterpret_cast<const uint4*>(e);
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (lane == 0) mbar_arrive(&built[stage]);
            put_g((it + 1) & 1, rn);
        }
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

}  // namespace
}  // namespace dlrm

using namespace dlrm;

extern "C" dlrm_status dlrm_interact_bwd_f16(const void* d_grad_out, const void* d_dense, const void* d_pooled, int F,
                                             int D, int B, int out_cols, void* d_grad_dense, void* d_grad_pooled,
                                             uint32_t* d_status, void* stream)
{
    DLRM_API_RANGE("dlrm_interact_bwd_f16");
    clear_error();
    if (F < 1 || D < 1 || B < 0)
        return fail(DLRM_ERR_INVALID_ARG, "dlrm_interact_bwd_f16: need F >= 1, D >= 1, B >= 0");
    const int64_t W = (int64_t)D + (int64_t)F * (F + 1) / 2;
    if (out_cols < W)
        return fail(DLRM_ERR_INVALID_ARG, "dlrm_interact_bwd_f16: out_cols %d < D + F(F+1)/2 = %lld", out_cols,
                    (long long)W);
    if (F > kSlot - 1 || D % kKB != 0 || D > 4 * kKB || out_cols % 8 != 0 || out_cols > 1024)
        return fail(DLRM_ERR_UNSUPPORTED,
                    "dlrm_interact_bwd_f16: needs F <= 31, D a multiple of 64 up to 256, out_cols a multiple of 8 "
                    "up to 1024");
    if (B == 0) return DLRM_OK;
    if (!d_grad_out || !d_dense || !d_pooled || !d_grad_dense || !d_grad_pooled)
        return fail(DLRM_ERR_INVALID_ARG, "dlrm_interact_bwd_f16: null device pointer");
    if (!aligned16(d_grad_out) || !aligned16(d_dense) || !aligned16(d_pooled) || !aligned16(d_grad_dense) ||
        !aligned16(d_grad_pooled))
        return fail(DLRM_ERR_UNSUPPORTED, "dlrm_interact_bwd_f16: pointers must be 16-byte aligned");
    EncodeTiledFn enc = encode_fn();
    if (!enc) return fail(DLRM_ERR_CUDA, "dlrm_interact_bwd_f16: cuTensorMapEncodeTiled unavailable");
    const int KH = D / kKB;
    int ns = kMaxStages;
    while (ns > 1 && bwd_smem(KH, out_cols, ns) > (size_t)kSmemLimit) --ns;
    const size_t smem = bwd_smem(KH, out_cols, ns);
    if (smem > (size_t)kSmemLimit) return fail(DLRM_ERR_UNSUPPORTED, "dlrm_interact_bwd_f16: tile does not fit");
    uint32_t tmem_cols = 32;
    while (tmem_cols < (uint32_t)(2 * D)) tmem_cols *= 2;

    CUtensorMap mp, md;
    const cuuint32_t ones[3] = {1, 1, 1};
    const cuuint64_t ddims[2] = {(cuuint64_t)D, (cuuint64_t)B};
    const cuuint64_t dstr[1] = {(cuuint64_t)D * 2};
    const cuuint32_t dbox[2] = {(cuuint32_t)kKB, (cuuint32_t)kGroup};
    CUresult r = enc(&md, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(d_dense), ddims, dstr, dbox, ones,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(DLRM_ERR_CUDA, "dlrm_interact_bwd_f16: dense tensor map (%d)", (int)r);
    const cuuint64_t pdims[3] = {(cuuint64_t)D, (cuuint64_t)F, (cuuint64_t)B};
    const cuuint64_t pstr[2] = {(cuuint64_t)D * 2, (cuuint64_t)F * D * 2};
    const cuuint32_t pbox[3] = {(cuuint32_t)kKB, (cuuint32_t)kSlot, (cuuint32_t)kGroup};
    r = enc(&mp, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void*>(d_pooled), pdims, pstr, pbox, ones,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(DLRM_ERR_CUDA, "dlrm_interact_bwd_f16: pooled tensor map (%d)", (int)r);
    CUtensorMap mg;   // grad_pooled as [B][F][D]: boxes {64, 32, 1}, rows F..31 clipped
    const cuuint32_t gbox[3] = {(cuuint32_t)kKB, (cuuint32_t)kSlot, 1};
    r = enc(&mg, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, d_grad_pooled, pdims, pstr, gbox, ones,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(DLRM_ERR_CUDA, "dlrm_interact_bwd_f16: grad_pooled tensor map (%d)", (int)r);
    const int ntiles = (B + kGroup - 1) / kGroup;
    const int grid = ntiles < num_sms() ? ntiles : num_sms();
    cudaError_t e = cudaFuncSetAttribute(interact_bwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return fail(DLRM_ERR_CUDA, "dlrm_interact_bwd_f16: %s", cudaGetErrorString(e));
    return check_launch_pdl(launch_pdl(interact_bwd_tc_kernel, grid, kThreads, smem, as_stream(stream), mp, md, mg,
                                       (const __half*)d_grad_out, (__half*)d_grad_dense, F, D, B, out_cols, KH, ns,
                                       tmem_cols, d_status, wait_limit_cycles()),
                            "interact_bwd_tc_kernel");
}
