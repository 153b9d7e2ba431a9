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
    kern<<<(int)blocks, kWarps * kWarp, smem, stream>>>(grad_out, (const T*)dense, (const T*)pooled, F, D, B, P,
                                                        gd, gp);
    return check_launch("interact_bwd_kernel");
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
    if (dtype == DLRM_F32)
        return dispatch<float>(d_grad_out, d_dense, d_pooled, F, D, B, out_cols, d_grad_dense, d_grad_pooled, st);
    return dispatch<__half>(d_grad_out, d_dense, d_pooled, F, D, B, out_cols, d_grad_dense, d_grad_pooled, st);
}
