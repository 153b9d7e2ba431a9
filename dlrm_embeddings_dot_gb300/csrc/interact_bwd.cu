// interact_bwd.cu -- gradient of the dot interaction ("DLRM For PyTorch",
// §Model architecture: interaction output = dense vector followed by the
// pairwise dot products).  With G the upstream gradient row and M the
// symmetric (F+1)x(F+1) matrix holding G's triangle (zero diagonal),
//   dZ = M Z,  grad_dense = G[0..D) + dZ_0,  grad_pooled[t] = dZ_{t+1}.
//
// One warp per sample.  The sample's Z and upstream gradient row are staged
// in shared memory with cp.async, and the next sample's copy is issued as soon
// as the current one has been read into registers, so the loads run behind
// the arithmetic.  G's triangle is written into both halves of M (row stride
// padded to a multiple of 4 so a row is read with broadcast float4 loads);
// lane l owns columns 4l..4l+3 of a 128-column slab of Z, held in registers
// for all F+1 rows, so each output element is an in-register fp32 FMA chain
// over j (fixed order).  Outputs are 16-byte stores, 512 contiguous bytes per
// warp.
#include "common.cuh"
#include "interact_tc.cuh"
#include "reg_gather.cuh"
#include "tcgen05.cuh"

namespace dlrm {
namespace {

constexpr int kWarps = 4;

__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gsrc)
{
    const uint32_t d = (uint32_t)__cvta_generic_to_shared(smem_dst);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(gsrc) : "memory");
}

__device__ __forceinline__ void cp_async4(void* smem_dst, const void* gsrc)
{
    const uint32_t d = (uint32_t)__cvta_generic_to_shared(smem_dst);
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(d), "l"(gsrc) : "memory");
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Four consecutive elements of a staged row as fp32 (fp16 widened exactly).
template <typename T>
__device__ __forceinline__ float4 lds4(const T* p)
{
    if constexpr (sizeof(T) == 4) {
        return *reinterpret_cast<const float4*>(p);
    } else {
        const uint2 u = *reinterpret_cast<const uint2*>(p);
        const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&u.x));
        const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&u.y));
        return make_float4(a.x, a.y, b.x, b.y);
    }
}

__device__ __forceinline__ void fma4(float4& acc, float c, const float4& z)
{
    acc.x = fmaf(c, z.x, acc.x);
    acc.y = fmaf(c, z.y, acc.y);
    acc.z = fmaf(c, z.z, acc.z);
    acc.w = fmaf(c, z.w, acc.w);
}

struct BwdSmem {
    int z_bytes, g_floats, m_floats, warp_bytes;
};

template <int RMAX>
__host__ __device__ inline BwdSmem bwd_smem(int F, int D, int P, int es)
{
    BwdSmem m;
    m.z_bytes = ((F + 1) * D * es + 15) / 16 * 16;
    m.g_floats = (P + 3) / 4 * 4;
    m.m_floats = RMAX * ((RMAX + 3) / 4 * 4);
    m.warp_bytes = m.z_bytes + 4 * (m.g_floats + m.m_floats);
    return m;
}

// Copy sample b's Z (dense row, then the F pooled rows) and its upstream
// gradient row into this warp's staging area, all asynchronously.
template <typename T>
__device__ __forceinline__ void stage_bwd(unsigned char* zs, float* gs, const float* __restrict__ grad_out,
                                          const T* __restrict__ dense, const T* __restrict__ pooled, int64_t b,
                                          int F, int D, int P, int lane)
{
    const int dchunks = D * (int)sizeof(T) / 16;             // 16-byte chunks of one row
    const unsigned char* drow = reinterpret_cast<const unsigned char*>(dense + b * D);
    const unsigned char* prow = reinterpret_cast<const unsigned char*>(pooled + b * F * D);
    for (int x = lane; x < dchunks; x += kWarp) cp_async16(zs + 16 * x, drow + 16 * x);
    for (int x = lane; x < F * dchunks; x += kWarp) cp_async16(zs + 16 * (dchunks + x), prow + 16 * x);
    const float* G = grad_out + b * P;
    for (int x = lane; x < P; x += kWarp) cp_async4(gs + x, G + x);   // rows are only 4-byte aligned in general
}

template <typename T, int RMAX>
__global__ void __launch_bounds__(kWarps * kWarp)
interact_bwd_kernel(const float* __restrict__ grad_out, const T* __restrict__ dense,
                    const T* __restrict__ pooled, int F, int D, int B, int P,
                    float* __restrict__ grad_dense, float* __restrict__ grad_pooled)
{
    pdl_wait();
    constexpr int RS = (RMAX + 3) / 4 * 4;       // smem row stride of M (multiple of 4)
    extern __shared__ __align__(16) unsigned char bwd_smem_raw[];
    const int lane = threadIdx.x % kWarp;
    const int warp = threadIdx.x / kWarp;
    const int R = F + 1;
    const BwdSmem L = bwd_smem<RMAX>(F, D, P, (int)sizeof(T));
    unsigned char* zs = bwd_smem_raw + (size_t)warp * L.warp_bytes;
    float* gs = reinterpret_cast<float*>(zs + L.z_bytes);
    float* M = gs + L.g_floats;
    const int warps_total = gridDim.x * kWarps;

    // the diagonal and everything outside R x R stay zero for the whole kernel
    for (int x = lane; x < RMAX * RS; x += kWarp) M[x] = 0.f;

    int b = blockIdx.x * kWarps + warp;
    if (b < B) stage_bwd(zs, gs, grad_out, dense, pooled, (int64_t)b, F, D, P, lane);
    cp_async_commit();
    for (; b < B; b += warps_total) {
        cp_async_wait_all();
        __syncwarp();
        // row hi of the upstream triangle goes to M[hi][lo] and M[lo][hi]
#pragma unroll
        for (int hi = 1; hi < RMAX; ++hi) {
            if (hi < R && lane < hi) {
                const float v = gs[D + hi * (hi - 1) / 2 + lane];
                M[hi * RS + lane] = v;
                M[lane * RS + hi] = v;
            }
        }
        for (int c0 = 0; c0 < D; c0 += 4 * kWarp) {
            const int k = c0 + 4 * lane;              // this lane's 4 columns
            const bool on = k < D;
            float4 z[RMAX];
#pragma unroll
            for (int j = 0; j < RMAX; ++j) {
                z[j] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (j < R && on) z[j] = lds4(reinterpret_cast<const T*>(zs) + (int64_t)j * D + k);
            }
            float4 g0 = make_float4(0.f, 0.f, 0.f, 0.f);
            if (on) g0 = make_float4(gs[k], gs[k + 1], gs[k + 2], gs[k + 3]);
            __syncwarp();
            if (c0 + 4 * kWarp >= D) {
                // this sample's staging area has been read: fetch the next sample behind the arithmetic
                if (b + warps_total < B)
                    stage_bwd(zs, gs, grad_out, dense, pooled, (int64_t)(b + warps_total), F, D, P, lane);
                cp_async_commit();
            }
            for (int i = 0; i < R; ++i) {
                float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
                const float4* mrow = reinterpret_cast<const float4*>(M + i * RS);
#pragma unroll
                for (int j4 = 0; j4 < RS / 4; ++j4) {
                    const float4 c = mrow[j4];
                    if (4 * j4 + 0 < RMAX) fma4(acc, c.x, z[(4 * j4 + 0) % RMAX]);
                    if (4 * j4 + 1 < RMAX) fma4(acc, c.y, z[(4 * j4 + 1) % RMAX]);
                    if (4 * j4 + 2 < RMAX) fma4(acc, c.z, z[(4 * j4 + 2) % RMAX]);
                    if (4 * j4 + 3 < RMAX) fma4(acc, c.w, z[(4 * j4 + 3) % RMAX]);
                }
                if (on) {
                    if (i == 0) {
                        acc.x += g0.x;
                        acc.y += g0.y;
                        acc.z += g0.z;
                        acc.w += g0.w;
                        *reinterpret_cast<float4*>(grad_dense + (int64_t)b * D + k) = acc;
                    } else {
                        *reinterpret_cast<float4*>(grad_pooled + ((int64_t)b * F + (i - 1)) * D + k) = acc;
                    }
                }
            }
        }
        __syncwarp();   // M is rebuilt for the next sample
    }
}

// ------------------------------------------------------------ register kernel
// fp32, D = 128, R = F + 1 rows known at compile time.  One warp per sample;
// lane l holds features 4l..4l+3 of every row of Z in registers.  The sample
// arrives by three bulk copies on the warp's mbarrier (dense row, the F
// pooled rows, the upstream gradient row); the lanes expand G's triangle
// into M (one triangle element per lane per step, through a pair table
// built once per block), and output row i is an fp32 FMA chain over j in
// ascending order, with M's rows read by broadcast float4 loads.  The next
// sample's copies are issued as soon as this one's buffer has been read.
constexpr int kRegD = 128;

template <int R>
struct RegBwd {
    static constexpr int NP = R * (R - 1) / 2;             // triangle elements
    static constexpr int RS = (R + 3) / 4 * 4;             // M row stride
    static constexpr int z_bytes = R * kRegD * 4;
    static constexpr int m_bytes = R * RS * 4;
    // per-warp bytes for a gradient row of P floats
    __host__ __device__ static constexpr int warp_bytes(int P) { return z_bytes + (P * 4 + 15) / 16 * 16 + m_bytes; }
    // per-block bytes: warps, the pair table, the mbarriers
    __host__ __device__ static constexpr int block_bytes(int P)
    {
        return kWarps * warp_bytes(P) + (NP * 2 + 15) / 16 * 16 + kWarps * 8;
    }
};

// kGather: Z's pooled rows are gathered from the tables (ga) instead of read
// from a stored pooled tensor (pooled is then unused); the values are the
// same bits the lookup produced, so are the results.
// Gathered rows arrive by per-lane cp.async (the backward has room in the
// shared-memory pipe; 26 bulk copies per sample measured 3 % slower).
constexpr bool kRowsAsync = true;

template <int R, bool kGather>
__global__ void __launch_bounds__(kWarps * kWarp, 3)
interact_bwd_regs_kernel(const float* __restrict__ grad_out, const float* __restrict__ dense,
                         const float* __restrict__ pooled, RegGather ga, int B, int P, float* __restrict__ grad_dense,
                         float* __restrict__ grad_pooled, uint32_t* __restrict__ status)
{
    pdl_wait();
    using L = RegBwd<R>;
    constexpr int F = R - 1, D = kRegD, RS = L::RS, NP = L::NP;
    extern __shared__ __align__(16) unsigned char bwd_regs_raw[];
    const int lane = threadIdx.x % kWarp;
    const int warp = threadIdx.x / kWarp;
    const int wb = L::warp_bytes(P);
    unsigned char* base = bwd_regs_raw + (size_t)warp * wb;
    float4* zs = reinterpret_cast<float4*>(base);                       // [R][32] float4
    float* gs = reinterpret_cast<float*>(base + L::z_bytes);             // [P]
    float* M = reinterpret_cast<float*>(base + L::z_bytes + (P * 4 + 15) / 16 * 16);
    uint16_t* pair_ij = reinterpret_cast<uint16_t*>(bwd_regs_raw + (size_t)kWarps * wb);
    uint64_t* bar = reinterpret_cast<uint64_t*>(bwd_regs_raw + (size_t)kWarps * wb + (NP * 2 + 15) / 16 * 16) + warp;

    // pair table (i << 8 | j for triangle element p), M's diagonal stays zero
    for (int p = threadIdx.x; p < NP; p += blockDim.x) {
        int i = 1;
        while (i * (i + 1) / 2 <= p) ++i;
        pair_ij[p] = (uint16_t)(i << 8 | (p - i * (i - 1) / 2));
    }
    for (int x = lane; x < R * RS; x += kWarp) M[x] = 0.f;
    if (lane == 0) {
        tc::mbar_init(bar, 1);
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    __syncthreads();

    const int64_t stride = (int64_t)gridDim.x * kWarps;
    int64_t b = (int64_t)blockIdx.x * kWarps + warp;
    const BagLanes<F, D> bags(ga, B, lane, status);
    // sample smp's Z rows and gradient row, all counted on the warp's mbarrier
    auto stage = [&](int64_t smp, uint32_t src_row, int a, int e) {
        if constexpr (kGather) {
            bags.template gather<kRowsAsync, 2>(zs, src_row, a, e, bar);
            if (lane == F) {
                tc::mbar_expect_tx_only(bar, D * 4);
                tc::bulk_g2s(zs, dense + smp * D, D * 4, bar);
            } else if (lane == F + 1) {
                tc::mbar_expect_tx_only(bar, P * 4);
                tc::bulk_g2s(gs, grad_out + smp * P, P * 4, bar);
            }
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(bar);
        } else if (lane == 0) {
            tc::mbar_expect_tx(bar, R * D * 4 + P * 4);
            tc::bulk_g2s(zs, dense + smp * D, D * 4, bar);
            tc::bulk_g2s(zs + kWarp, pooled + smp * (int64_t)F * D, F * D * 4, bar);
            tc::bulk_g2s(gs, grad_out + smp * P, P * 4, bar);
        }
    };
    // bags: bounds two samples ahead, the index one sample ahead (used a
    // sample after it was requested)
    int a1 = 0, e1 = 0, a2 = 0, e2 = 0, idx1 = 0;
    if constexpr (kGather) {
        int a0, e0;
        bags.load_bounds(b, a0, e0);
        bags.load_bounds(b + stride, a1, e1);
        bags.load_bounds(b + 2 * stride, a2, e2);
        bags.clamp(a0, e0);
        if (b < B) stage(b, bags.resolve(a0, e0, bags.early_index(a0, e0)), a0, e0);
        bags.clamp(a1, e1);
        idx1 = bags.early_index(a1, e1);
    } else {
        if (b < B) stage(b, 0, 0, 0);
    }
    uint32_t phase = 0;
    for (; b < B; b += stride) {
        if constexpr (kGather && kRowsAsync) asm volatile("cp.async.wait_group 0;" ::: "memory");
        if (!tc::bounded_wait(bar, phase)) {
            if (lane == 0) set_status(status, DLRM_STATUS_TIMEOUT);
            return;
        }
        phase ^= 1u;
        // G's triangle into both halves of M
#pragma unroll
        for (int k = 0; k < (NP + kWarp - 1) / kWarp; ++k) {
            const int p = k * kWarp + lane;
            if (p < NP) {
                const float v = gs[D + p];
                const int ij = pair_ij[p];
                const int i = ij >> 8, j = ij & 0xff;
                M[i * RS + j] = v;
                M[j * RS + i] = v;
            }
        }
        float4 z[R];
#pragma unroll
        for (int r = 0; r < R; ++r) z[r] = zs[r * kWarp + lane];
        const float4 g0 = reinterpret_cast<const float4*>(gs)[lane];
        // M complete for every lane; the staging buffer has been read
        __syncwarp();
        if (b + stride < B) {
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            if constexpr (kGather)
                stage(b + stride, bags.resolve(a1, e1, idx1), a1, e1);
            else
                stage(b + stride, 0, 0, 0);
        }
        if constexpr (kGather) {   // advance the bag pipeline by one sample
            int a3, e3;
            bags.load_bounds(b + 3 * stride, a3, e3);
            bags.clamp(a2, e2);
            idx1 = bags.early_index(a2, e2);
            a1 = a2;
            e1 = e2;
            a2 = a3;
            e2 = e3;
        }
        // a rolled loop over the rows keeps the code small (the diagonal of M
        // is zero, so j = i adds an exact zero product)
#pragma unroll 1
        for (int i = 0; i < R; ++i) {
            const float4* mrow = reinterpret_cast<const float4*>(M + i * RS);
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            static_for<RS / 4>([&](auto J4) {
                constexpr int j0 = 4 * decltype(J4)::value;
                const float4 c = mrow[j0 / 4];
                if constexpr (j0 + 0 < R) fma4(acc, c.x, z[j0 + 0 < R ? j0 + 0 : 0]);
                if constexpr (j0 + 1 < R) fma4(acc, c.y, z[j0 + 1 < R ? j0 + 1 : 0]);
                if constexpr (j0 + 2 < R) fma4(acc, c.z, z[j0 + 2 < R ? j0 + 2 : 0]);
                if constexpr (j0 + 3 < R) fma4(acc, c.w, z[j0 + 3 < R ? j0 + 3 : 0]);
            });
            float* dst;
            if (i == 0) {
                acc.x += g0.x;
                acc.y += g0.y;
                acc.z += g0.z;
                acc.w += g0.w;
                dst = grad_dense + b * D;
            } else {
                dst = grad_pooled + (b * F + (i - 1)) * D;
            }
            reinterpret_cast<float4*>(dst)[lane] = acc;
        }
        __syncwarp();   // M is rebuilt for the next sample
    }
}

template <int R, bool kGather>
dlrm_status launch_regs(const float* grad_out, const float* dense, const float* pooled, const RegGather& ga, int B,
                        int P, float* gd, float* gp, uint32_t* status, cudaStream_t stream)
{
    const size_t smem = (size_t)RegBwd<R>::block_bytes(P);
    auto kern = interact_bwd_regs_kernel<R, kGather>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return fail(DLRM_ERR_CUDA, "dlrm_interact_bwd: %s", cudaGetErrorString(e));
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kWarps * kWarp, smem) != cudaSuccess ||
        per_sm < 1)
        per_sm = 1;
    int64_t blocks = ((int64_t)B + kWarps - 1) / kWarps;
    const int64_t cap = (int64_t)num_sms() * per_sm;
    if (blocks > cap) blocks = cap;
    return check_launch_pdl(launch_pdl(kern, (int)blocks, kWarps * kWarp, smem, stream, grad_out, dense, pooled, ga, B,
                                       P, gd, gp, status),
                            "interact_bwd_regs_kernel");
}

// Shapes the register kernel takes: fp32, D = 128, F in {8, 26}, gradient
// rows of a multiple of 4 floats, at most 1024 columns.
inline bool regs_bwd_supported(int F, int D, int P)
{
    return D == kRegD && (F == 8 || F == 26) && P % 4 == 0 && P <= 1024;
}

template <typename T, int RMAX>
dlrm_status launch(const float* grad_out, const void* dense, const void* pooled, int F, int D, int B, int P,
                   float* gd, float* gp, cudaStream_t stream)
{
    const BwdSmem L = bwd_smem<RMAX>(F, D, P, (int)sizeof(T));
    const size_t smem = (size_t)kWarps * L.warp_bytes;
    if (smem > 200 * 1024)
        return fail(DLRM_ERR_UNSUPPORTED, "dlrm_interact_bwd: (F+1) x D too large for the staged backward");
    auto kern = interact_bwd_kernel<T, RMAX>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return fail(DLRM_ERR_CUDA, "dlrm_interact_bwd: %s", cudaGetErrorString(e));
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kWarps * kWarp, smem) != cudaSuccess ||
        per_sm < 1)
        per_sm = 1;
    int64_t blocks = ((int64_t)B + kWarps - 1) / kWarps;
    const int64_t cap = (int64_t)num_sms() * per_sm;
    if (blocks > cap) blocks = cap;
    return check_launch_pdl(launch_pdl(kern, (int)blocks, kWarps * kWarp, smem, stream, grad_out, (const T*)dense,
                                       (const T*)pooled, F, D, B, P, gd, gp),
                            "interact_bwd_kernel");
}

template <typename T>
dlrm_status dispatch(const float* grad_out, const void* dense, const void* pooled, int F, int D, int B, int P,
                     float* gd, float* gp, cudaStream_t stream)
{
    const int R = F + 1;
    if (R <= 8) return launch<T, 8>(grad_out, dense, pooled, F, D, B, P, gd, gp, stream);
    if (R <= 16) return launch<T, 16>(grad_out, dense, pooled, F, D, B, P, gd, gp, stream);
    if (R <= 28) return launch<T, 28>(grad_out, dense, pooled, F, D, B, P, gd, gp, stream);
    if (R <= 32) return launch<T, 32>(grad_out, dense, pooled, F, D, B, P, gd, gp, stream);
    return fail(DLRM_ERR_UNSUPPORTED, "dlrm_interact_bwd: F > 31 is not implemented");
}

}  // namespace
}  // namespace dlrm

using namespace dlrm;

extern "C" dlrm_status dlrm_interact_bwd(const float* d_grad_out, const void* d_dense, const void* d_pooled,
                                         dlrm_dtype dtype, int F, int D, int B, int out_cols,
                                         float* d_grad_dense, float* d_grad_pooled, void* stream)
{
    DLRM_API_RANGE("dlrm_interact_bwd");
    clear_error();
    if (!dtype_ok(dtype)) return fail(DLRM_ERR_INVALID_ARG, "dlrm_interact_bwd: bad dtype");
    if (F < 1 || D < 1 || B < 0)
        return fail(DLRM_ERR_INVALID_ARG, "dlrm_interact_bwd: need F >= 1, D >= 1, B >= 0");
    const int64_t W = (int64_t)D + (int64_t)F * (F + 1) / 2;
    if (out_cols < W)
        return fail(DLRM_ERR_INVALID_ARG, "dlrm_interact_bwd: out_cols %d < D + F(F+1)/2 = %lld", out_cols,
                    (long long)W);
    if (!d_grad_out || !d_dense || !d_pooled || !d_grad_dense || !d_grad_pooled)
        return fail(DLRM_ERR_INVALID_ARG, "dlrm_interact_bwd: null device pointer");
    if (((int64_t)D * dtype_size(dtype)) % 16 != 0)
        return fail(DLRM_ERR_UNSUPPORTED, "dlrm_interact_bwd: D*%d bytes must be a multiple of 16",
                    dtype_size(dtype));
    if (!aligned16(d_grad_out) || !aligned16(d_dense) || !aligned16(d_pooled) || !aligned16(d_grad_dense) ||
        !aligned16(d_grad_pooled))
        return fail(DLRM_ERR_UNSUPPORTED, "dlrm_interact_bwd: pointers must be 16-byte aligned");
    if (B == 0) return DLRM_OK;
    cudaStream_t st = as_stream(stream);
    if (dtype == DLRM_F32 && regs_bwd_supported(F, D, out_cols)) {
        const float* d = static_cast<const float*>(d_dense);
        const float* p = static_cast<const float*>(d_pooled);
        const RegGather none{};
        return F == 26 ? launch_regs<27, false>(d_grad_out, d, p, none, B, out_cols, d_grad_dense, d_grad_pooled,
                                                nullptr, st)
                       : launch_regs<9, false>(d_grad_out, d, p, none, B, out_cols, d_grad_dense, d_grad_pooled,
                                               nullptr, st);
    }
    if (dtype == DLRM_F32)
        return dispatch<float>(d_grad_out, d_dense, d_pooled, F, D, B, out_cols, d_grad_dense, d_grad_pooled, st);
    return dispatch<__half>(d_grad_out, d_dense, d_pooled, F, D, B, out_cols, d_grad_dense, d_grad_pooled, st);
}

extern "C" dlrm_status dlrm_emb_interact_bwd(const void* d_tables, dlrm_dtype dtype, const int64_t* d_row_base,
                                            int F, int D, int B, const int32_t* d_indices, const int32_t* d_offsets,
                                            int64_t nnz, const float* d_grad_out, const void* d_dense, int out_cols,
                                            float* d_grad_dense, float* d_grad_pooled, unsigned flags,
                                            uint32_t* d_status, void* stream)
{
    DLRM_API_RANGE("dlrm_emb_interact_bwd");
    clear_error();
    if (!dtype_ok(dtype)) return fail(DLRM_ERR_INVALID_ARG, "dlrm_emb_interact_bwd: bad dtype");
    if (F < 1 || D < 1 || B < 0)
        return fail(DLRM_ERR_INVALID_ARG, "dlrm_emb_interact_bwd: need F >= 1, D >= 1, B >= 0");
    if (nnz < 0 || nnz > DLRM_MAX_NNZ || (int64_t)F * B >= (int64_t)1 << 31)
        return fail(DLRM_ERR_INVALID_ARG, "dlrm_emb_interact_bwd: need nnz <= DLRM_MAX_NNZ and F*B < 2^31");
    const int64_t W = (int64_t)D + (int64_t)F * (F + 1) / 2;
    if (out_cols < W)
        return fail(DLRM_ERR_INVALID_ARG, "dlrm_emb_interact_bwd: out_cols %d < D + F(F+1)/2 = %lld", out_cols,
                    (long long)W);
    if (!d_tables || !d_row_base || !d_offsets || !d_grad_out || !d_dense || !d_grad_dense || !d_grad_pooled ||
        (nnz > 0 && !d_indices))
        return fail(DLRM_ERR_INVALID_ARG, "dlrm_emb_interact_bwd: null device pointer");
    if (flags & ~DLRM_FLAG_HASH_INDICES)
        return fail(DLRM_ERR_INVALID_ARG, "dlrm_emb_interact_bwd: unknown flag bits 0x%x", flags);
    if (dtype != DLRM_F32 || !regs_bwd_supported(F, D, out_cols) || !aligned16(d_tables) || !aligned16(d_grad_out) ||
        !aligned16(d_dense) || !aligned16(d_grad_dense) || !aligned16(d_grad_pooled))
        return fail(DLRM_ERR_UNSUPPORTED,
                    "dlrm_emb_interact_bwd: needs fp32, D = 128, F in {8, 26}, out_cols a multiple of 4 up to 1024 "
                    "and 16-byte aligned pointers (use dlrm_emb_fwd + dlrm_interact_bwd otherwise)");
    if (B == 0) return DLRM_OK;
    const RegGather ga{(const float*)d_tables, d_row_base, d_indices, d_offsets, nnz,
                       (flags & DLRM_FLAG_HASH_INDICES) != 0};
    const float* d = static_cast<const float*>(d_dense);
    cudaStream_t st = as_stream(stream);
    return F == 26 ? launch_regs<27, true>(d_grad_out, d, nullptr, ga, B, out_cols, d_grad_dense, d_grad_pooled,
                                           d_status, st)
                   : launch_regs<9, true>(d_grad_out, d, nullptr, ga, B, out_cols, d_grad_dense, d_grad_pooled,
                                          d_status, st);
}
