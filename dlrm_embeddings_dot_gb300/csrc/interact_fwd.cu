// interact_fwd.cu -- dot interaction ("DLRM For PyTorch", §Model
// architecture; --interaction_op cuda_dot): pairwise dot products among the
// bottom-MLP output and the F pooled embeddings, strict lower triangle in
// row-major order, concatenated after the dense vector, zero padded.
//
// This file holds the CUDA-core (FFMA) kernel, used for fp32 (tensor-core
// TF32 cannot meet fp32 accuracy) and for fp16 shapes the tensor-core kernel
// does not take, plus the entry point that picks between the two.
//
// FFMA kernel: one CTA of 4 warps per sample at a time.  Z = [dense; pooled
// rows] is staged in shared memory as fp32 (all 16-byte chunks of a sample in
// flight at once via cp.async), rows padded to a multiple of 4 and to
// 128-byte strides, with the 16-byte chunk index XOR-swizzled by (row / 4)
// so that the float4 reads of up to 8 row-blocks in one instruction hit
// distinct banks.  Lane l owns 4x4 blocks (I, J), J <= I, of the lower block
// triangle of Z Z^T; warp w covers the 16-byte chunks c = w, w+4, ... of K, so
// the four warps split K and their partial blocks are added in the fixed
// order w = 0..3 through shared memory.  A CTA holds one sample (about 23 KB
// for F = 26, D = 128), so ~9 CTAs (36 warps) share an SM and hide each
// other's staging latency.
#include "common.cuh"
#include "interact_tc.cuh"

namespace dlrm {
namespace {

constexpr int kSplit = 4;                     // warps per sample (K split)
constexpr int kFfmaThreads = kSplit * kWarp;

__host__ __device__ inline int round_up(int x, int m) { return (x + m - 1) / m * m; }

struct FfmaGeom {
    int R;        // F + 1 vectors
    int R4;       // rounded up to 4
    int ld;       // floats per smem row (multiple of 32)
    int nblocks;  // 4x4 blocks of the lower block triangle
    int z_floats; // R4 * ld
    int p_floats; // kSplit partial blocks: [kSplit][16][nblocks]
    int smem_floats;
};

__host__ __device__ inline FfmaGeom ffma_geom(int F, int D, int P)
{
    FfmaGeom g;
    g.R = F + 1;
    g.R4 = round_up(g.R, 4);
    g.ld = round_up(D, 32);
    const int nb = g.R4 / 4;
    g.nblocks = nb * (nb + 1) / 2;
    g.z_floats = g.R4 * g.ld;
    g.p_floats = kSplit * 16 * g.nblocks;
    g.smem_floats = g.z_floats + g.p_floats + round_up(P, 4);
    return g;
}

// float offset of 16-byte chunk c of row i (XOR swizzle within 128-byte segments)
__device__ __forceinline__ int zoff(int i, int c, int ld)
{
    return i * ld + (((c & ~7) | ((c ^ (i >> 2)) & 7)) << 2);
}

__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gsrc)
{
    const uint32_t d = (uint32_t)__cvta_generic_to_shared(smem_dst);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(gsrc) : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Stage Z of sample b (row 0 = dense[b], rows 1..F = pooled[b]) into zs with
// all threads of the CTA.  fp32: independent cp.async per 16-byte chunk;
// fp16: 16-byte loads widened to fp32 in registers.
template <typename T>
__device__ __forceinline__ void stage_sample(float* zs, int ld, const T* __restrict__ dense,
                                             const T* __restrict__ pooled, int64_t b, int F, int D, int tid)
{
    constexpr int V = 16 / sizeof(T);          // elements per 16-byte chunk
    const int cpr = D / V;                      // chunks per row
    const int total = (F + 1) * cpr;
    const T* prow = pooled + b * F * D;
    if constexpr (sizeof(T) == 4) {
        for (int x = tid; x < total; x += kFfmaThreads) {
            const int i = x / cpr, c = x - i * cpr;
            const float* src = i == 0 ? dense + b * D + 4 * c : prow + (int64_t)(i - 1) * D + 4 * c;
            cp_async16(zs + zoff(i, c, ld), src);
        }
        cp_async_wait_all();
    } else {
        for (int x0 = 0; x0 < total; x0 += 4 * kFfmaThreads) {
            uint4 v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int x = x0 + u * kFfmaThreads + tid;
                if (x < total) {
                    const int i = x / cpr, c = x - i * cpr;
                    const __half* src = i == 0 ? dense + b * D + 8 * c : prow + (int64_t)(i - 1) * D + 8 * c;
                    v[u] = ldg_nc_v4(src);
                }
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int x = x0 + u * kFfmaThreads + tid;
                if (x < total) {
                    const int i = x / cpr, c = x - i * cpr;
                    float f[8];
                    h8_to_f8(v[u], f);
                    *reinterpret_cast<float4*>(zs + zoff(i, 2 * c, ld)) = make_float4(f[0], f[1], f[2], f[3]);
                    *reinterpret_cast<float4*>(zs + zoff(i, 2 * c + 1, ld)) = make_float4(f[4], f[5], f[6], f[7]);
                }
            }
        }
    }
}

template <typename T>
__device__ __forceinline__ T to_out(float v)
{
    if constexpr (sizeof(T) == 4)
        return v;
    else
        return __float2half_rn(v);
}

template <typename T>
__global__ void __launch_bounds__(kFfmaThreads, 8)
interact_fwd_ffma_kernel(const T* __restrict__ dense, const T* __restrict__ pooled, int F, int D,
                         int B, T* __restrict__ out, int P)
{
    extern __shared__ __align__(16) float smem[];
    const FfmaGeom geo = ffma_geom(F, D, P);
    const int tid = threadIdx.x;
    const int lane = tid % kWarp;
    const int warp = tid / kWarp;
    float* zs = smem;
    float* part = smem + geo.z_floats;          // [kSplit][16][nblocks]
    float* os = part + geo.p_floats;
    const int W = D + F * (F + 1) / 2;
    const int C = D / 4;                        // 16-byte chunks of K

    // rows >= R and the output padding stay zero for the whole kernel
    for (int x = tid; x < (geo.R4 - geo.R) * geo.ld; x += kFfmaThreads) zs[geo.R * geo.ld + x] = 0.f;
    for (int x = W + tid; x < P; x += kFfmaThreads) os[x] = 0.f;

    for (int b = blockIdx.x; b < B; b += gridDim.x) {
        stage_sample(zs, geo.ld, dense, pooled, (int64_t)b, F, D, tid);
        __syncthreads();
        for (int k = tid; k < D; k += kFfmaThreads) os[k] = zs[zoff(0, k >> 2, geo.ld) + (k & 3)];
        for (int blk = lane; blk < geo.nblocks; blk += kWarp) {
            int I = 0;
            while ((I + 1) * (I + 2) / 2 <= blk) ++I;
            const int J = blk - I * (I + 1) / 2;
            float acc[4][4];
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int q = 0; q < 4; ++q) acc[r][q] = 0.f;
            const float* arow = zs + 4 * I * geo.ld;
            const float* brow = zs + 4 * J * geo.ld;
#pragma unroll 1
            for (int c = warp; c < C; c += kSplit) {
                const int ca = (((c & ~7) | ((c ^ I) & 7)) << 2);
                const int cb = (((c & ~7) | ((c ^ J) & 7)) << 2);
                float4 a[4], bq[4];
#pragma unroll
                for (int r = 0; r < 4; ++r) a[r] = *reinterpret_cast<const float4*>(arow + r * geo.ld + ca);
#pragma unroll
                for (int q = 0; q < 4; ++q) bq[q] = *reinterpret_cast<const float4*>(brow + q * geo.ld + cb);
#pragma unroll
                for (int r = 0; r < 4; ++r)
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        acc[r][q] = fmaf(a[r].x, bq[q].x, acc[r][q]);
                        acc[r][q] = fmaf(a[r].y, bq[q].y, acc[r][q]);
                        acc[r][q] = fmaf(a[r].z, bq[q].z, acc[r][q]);
                        acc[r][q] = fmaf(a[r].w, bq[q].w, acc[r][q]);
                    }
            }
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int q = 0; q < 4; ++q) part[(warp * 16 + r * 4 + q) * geo.nblocks + blk] = acc[r][q];
        }
        __syncthreads();
        // partial blocks of the four K quarters, added in a fixed order
        for (int x = tid; x < 16 * geo.nblocks; x += kFfmaThreads) {
            const int blk = x % geo.nblocks, rq = x / geo.nblocks;
            int I = 0;
            while ((I + 1) * (I + 2) / 2 <= blk) ++I;
            const int J = blk - I * (I + 1) / 2;
            const int i = 4 * I + (rq >> 2), j = 4 * J + (rq & 3);
            if (i < geo.R && j < i) {
                float v = part[rq * geo.nblocks + blk];
#pragma unroll
                for (int w = 1; w < kSplit; ++w) v += part[(w * 16 + rq) * geo.nblocks + blk];
                os[D + i * (i - 1) / 2 + j] = v;
            }
        }
        __syncthreads();
        T* orow = out + (int64_t)b * P;
        for (int x = tid; x < P; x += kFfmaThreads) orow[x] = to_out<T>(os[x]);
    }
}

template <typename T>
dlrm_status launch_ffma(const void* dense, const void* pooled, int F, int D, int B, void* out, int P,
                        cudaStream_t stream)
{
    const FfmaGeom g = ffma_geom(F, D, P);
    const size_t smem = (size_t)g.smem_floats * sizeof(float);
    if (smem > 200 * 1024)
        return fail(DLRM_ERR_UNSUPPORTED, "dlrm_interact_fwd: (F+1) x D too large for the CUDA-core kernel");
    cudaError_t e = cudaFuncSetAttribute(interact_fwd_ffma_kernel<T>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return fail(DLRM_ERR_CUDA, "dlrm_interact_fwd: %s", cudaGetErrorString(e));
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, interact_fwd_ffma_kernel<T>, kFfmaThreads, smem);
    if (e != cudaSuccess || per_sm < 1) per_sm = 1;
    int64_t blocks = B;
    const int64_t cap = (int64_t)num_sms() * per_sm;
    if (blocks > cap) blocks = cap;
    interact_fwd_ffma_kernel<T><<<(int)blocks, kFfmaThreads, smem, stream>>>(
        (const T*)dense, (const T*)pooled, F, D, B, (T*)out, P);
    return check_launch("interact_fwd_ffma_kernel");
}

}  // namespace
}  // namespace dlrm

using namespace dlrm;

extern "C" dlrm_status dlrm_interact_fwd(const void* d_dense, const void* d_pooled, dlrm_dtype dtype,
                                         int F, int D, int B, void* d_out, int out_cols,
                                         uint32_t* d_status, void* stream)
{
    clear_error();
    if (!dtype_ok(dtype)) return fail(DLRM_ERR_INVALID_ARG, "dlrm_interact_fwd: bad dtype");
    if (F < 1 || D < 1 || B < 0)
        return fail(DLRM_ERR_INVALID_ARG, "dlrm_interact_fwd: need F >= 1, D >= 1, B >= 0");
    const int64_t W = (int64_t)D + (int64_t)F * (F + 1) / 2;
    if (out_cols < W)
        return fail(DLRM_ERR_INVALID_ARG, "dlrm_interact_fwd: out_cols %d < D + F(F+1)/2 = %lld",
                    out_cols, (long long)W);
    if (!d_dense || !d_pooled || !d_out)
        return fail(DLRM_ERR_INVALID_ARG, "dlrm_interact_fwd: null device pointer");
    const int s = dtype_size(dtype);
    if (((int64_t)D * s) % 16 != 0)
        return fail(DLRM_ERR_UNSUPPORTED, "dlrm_interact_fwd: D*%d bytes must be a multiple of 16", s);
    if (!aligned16(d_dense) || !aligned16(d_pooled))
        return fail(DLRM_ERR_UNSUPPORTED, "dlrm_interact_fwd: dense and pooled must be 16-byte aligned");
    if (B == 0) return DLRM_OK;
    cudaStream_t st = as_stream(stream);
    if (dtype == DLRM_F16 && tc_interact_supported(F, D, out_cols, d_dense, d_pooled, d_out))
        return tc_interact_fwd(d_dense, d_pooled, F, D, B, d_out, out_cols, d_status, st);
    if (dtype == DLRM_F32) return launch_ffma<float>(d_dense, d_pooled, F, D, B, d_out, out_cols, st);
    return launch_ffma<__half>(d_dense, d_pooled, F, D, B, d_out, out_cols, st);
}

// CUDA-core path for any shape, exposed for tests of the tensor-core kernel.
extern "C" dlrm_status dlrm_interact_fwd_cuda_core(const void* d_dense, const void* d_pooled,
                                                   dlrm_dtype dtype, int F, int D, int B,
                                                   void* d_out, int out_cols, void* stream)
{
    clear_error();
    if (!dtype_ok(dtype) || F < 1 || D < 1 || B < 0 || !d_dense || !d_pooled || !d_out ||
        out_cols < (int64_t)D + (int64_t)F * (F + 1) / 2)
        return fail(DLRM_ERR_INVALID_ARG, "dlrm_interact_fwd_cuda_core: bad arguments");
    if (((int64_t)D * dtype_size(dtype)) % 16 != 0 || !aligned16(d_dense) || !aligned16(d_pooled))
        return fail(DLRM_ERR_UNSUPPORTED, "dlrm_interact_fwd_cuda_core: alignment");
    if (B == 0) return DLRM_OK;
    cudaStream_t st = as_stream(stream);
    if (dtype == DLRM_F32) return launch_ffma<float>(d_dense, d_pooled, F, D, B, d_out, out_cols, st);
    return launch_ffma<__half>(d_dense, d_pooled, F, D, B, d_out, out_cols, st);
}
