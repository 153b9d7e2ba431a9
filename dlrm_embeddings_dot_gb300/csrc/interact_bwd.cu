// interact_bwd.cu -- gradient of the dot interaction ("DLRM For PyTorch",
// §Model architecture: interaction output = dense vector followed by the
// pairwise dot products).  With G the upstream gradient row and M the
// symmetric (F+1)x(F+1) matrix holding G's triangle (zero diagonal),
//   dZ = M Z,  grad_dense = G[0..D) + dZ_0,  grad_pooled[t] = dZ_{t+1}.
//
// One warp per sample.  G's triangle is fetched with all loads in flight and
// written straight into both halves of M in shared memory (row stride padded to a multiple
// of 4 so a row is read with broadcast float4 loads); lane l owns columns
// 4l..4l+3 of a 128-column slab of Z, held in registers for all F+1 rows, so
// each output element is an in-register fp32 FMA chain over j (fixed order).
// Every global access is a 16-byte vector, 512 contiguous bytes per warp.
#include "common.cuh"

namespace dlrm {
namespace {

constexpr int kWarps = 4;

// Four consecutive elements of a row as fp32 (fp16 widened exactly).
template <typename T>
__device__ __forceinline__ float4 ld4(const T* p)
{
    if constexpr (sizeof(T) == 4) {
        return __ldg(reinterpret_cast<const float4*>(p));
    } else {
        const uint2 u = __ldg(reinterpret_cast<const uint2*>(p));
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

template <typename T, int RMAX>
__global__ void __launch_bounds__(kWarps * kWarp)
interact_bwd_kernel(const float* __restrict__ grad_out, const T* __restrict__ dense,
                    const T* __restrict__ pooled, int F, int D, int B, int P,
                    float* __restrict__ grad_dense, float* __restrict__ grad_pooled)
{
    constexpr int RS = (RMAX + 3) / 4 * 4;       // smem row stride of M (multiple of 4)
    __shared__ __align__(16) float msh[kWarps][RMAX * RS];
    const int lane = threadIdx.x % kWarp;
    const int warp = threadIdx.x / kWarp;
    const int R = F + 1;
    float* M = msh[warp];
    const int warps_total = gridDim.x * kWarps;

    // the diagonal and everything outside R x R stay zero for the whole kernel
    for (int x = lane; x < RMAX * RS; x += kWarp) M[x] = 0.f;

    for (int b = blockIdx.x * kWarps + warp; b < B; b += warps_total) {
        const float* G = grad_out + (int64_t)b * P;
        __syncwarp();
        // row hi of the triangle goes to M[hi][lo] and M[lo][hi]; all loads in flight together
#pragma unroll
        for (int hi = 1; hi < RMAX; ++hi) {
            if (hi < R && lane < hi) {
                const float v = __ldg(G + D + hi * (hi - 1) / 2 + lane);
                M[hi * RS + lane] = v;
                M[lane * RS + hi] = v;
            }
        }
        __syncwarp();
        for (int c0 = 0; c0 < D; c0 += 4 * kWarp) {
            const int k = c0 + 4 * lane;              // this lane's 4 columns
            const bool on = k < D;
            float4 z[RMAX];
#pragma unroll
            for (int j = 0; j < RMAX; ++j) {
                z[j] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (j < R && on)
                    z[j] = ld4((j == 0) ? dense + (int64_t)b * D + k : pooled + ((int64_t)b * F + (j - 1)) * D + k);
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
                        // scalar loads: a grad_out row is only 4-byte aligned when out_cols % 4 != 0
                        acc.x += __ldg(G + k);
                        acc.y += __ldg(G + k + 1);
                        acc.z += __ldg(G + k + 2);
                        acc.w += __ldg(G + k + 3);
                        *reinterpret_cast<float4*>(grad_dense + (int64_t)b * D + k) = acc;
                    } else {
                        *reinterpret_cast<float4*>(grad_pooled + ((int64_t)b * F + (i - 1)) * D + k) = acc;
                    }
                }
            }
        }
    }
}

template <typename T, int RMAX>
dlrm_status launch(const float* grad_out, const void* dense, const void* pooled, int F, int D, int B, int P,
                   float* gd, float* gp, cudaStream_t stream)
{
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, interact_bwd_kernel<T, RMAX>, kWarps * kWarp, 0) !=
            cudaSuccess ||
        per_sm < 1)
        per_sm = 1;
    int64_t blocks = ((int64_t)B + kWarps - 1) / kWarps;
    const int64_t cap = (int64_t)num_sms() * per_sm;
    if (blocks > cap) blocks = cap;
    interact_bwd_kernel<T, RMAX><<<(int)blocks, kWarps * kWarp, 0, stream>>>(
        grad_out, (const T*)dense, (const T*)pooled, F, D, B, P, gd, gp);
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
