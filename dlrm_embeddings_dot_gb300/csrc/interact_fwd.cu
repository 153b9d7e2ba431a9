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
    int o_floats; // output row
    int smem_bytes;
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
    g.o_floats = round_up(P, 4);
    // + one int per partial-slot: the output column it lands in (or -1)
    g.smem_bytes = 4 * (g.z_floats + g.p_floats + g.o_floats + 16 * g.nblocks);
    return g;
}

// Float offset of 16-byte chunk c of row i: the low 3 bits of the chunk index
// are XOR-ed with (row / 4), a permutation within each 128-byte segment.
__device__ __forceinline__ int zoff(int i, int c, int ld)
{
    return i * ld + ((c ^ ((i >> 2) & 7)) << 2);
}

__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gsrc)
{
    const uint32_t d = (uint32_t)__cvta_generic_to_shared(smem_dst);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(gsrc) : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Lower-triangle 4x4 block number -> (I, J), J <= I.
__device__ __forceinline__ void block_ij(int blk, int& I, int& J)
{
    I = 0;
    while ((I + 1) * (I + 2) / 2 <= blk) ++I;
    J = blk - I * (I + 1) / 2;
}

template <typename T>
__device__ __forceinline__ T to_out(float v)
{
    if constexpr (sizeof(T) == 4)
        return v;
    else
        return __float2half_rn(v);
}

// One 4x4 block of Z Z^T over this warp's K chunks (c = warp, warp+4, ...).
template <int DT>
__device__ __forceinline__ void block_dot(const float* zs, int ld, int C, int warp, int I, int J, float (&acc)[4][4])
{
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[r][q] = 0.f;
    const float* arow = zs + 4 * I * ld;
    const float* brow = zs + 4 * J * ld;
    const int I7 = I & 7, J7 = J & 7;
    constexpr int CT = DT / 4;
#pragma unroll 1
    for (int c = warp; c < (DT ? CT : C); c += kSplit) {
        const float* pa = arow + ((c ^ I7) << 2);
        const float* pb = brow + ((c ^ J7) << 2);
        float4 a[4], bq[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) a[r] = *reinterpret_cast<const float4*>(pa + r * ld);
#pragma unroll
        for (int q = 0; q < 4; ++q) bq[q] = *reinterpret_cast<const float4*>(pb + q * ld);
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
}

// DT: D as a compile-time constant (0 = taken at run time).
template <typename T, int DT>
__global__ void __launch_bounds__(kFfmaThreads, 8)
interact_fwd_ffma_kernel(const T* __restrict__ dense, const T* __restrict__ pooled, int F, int D_rt,
                         int B, T* __restrict__ out, int P)
{
    extern __shared__ __align__(16) float smem[];
    const int D = DT ? DT : D_rt;
    const FfmaGeom geo = ffma_geom(F, D, P);
    const int ld = DT ? (DT + 31) / 32 * 32 : geo.ld;
    const int tid = threadIdx.x;
    const int lane = tid % kWarp;
    const int warp = tid / kWarp;
    float* zs = smem;
    float* part = smem + geo.z_floats;          // [kSplit][16][nblocks]
    float* os = part + geo.p_floats;
    int* slot_col = reinterpret_cast<int*>(os + geo.o_floats);
    const int W = D + F * (F + 1) / 2;
    const int C = D / 4;                        // 16-byte fp32 chunks of K
    constexpr int V = 16 / sizeof(T);           // elements per 16-byte global chunk
    const int cpr = D / V;                      // global chunks per row

    // ---- once per CTA: zero padding, partial-slot -> output column map
    for (int x = tid; x < (geo.R4 - geo.R) * ld; x += kFfmaThreads) zs[geo.R * ld + x] = 0.f;
    for (int x = W + tid; x < P; x += kFfmaThreads) os[x] = 0.f;
    for (int x = tid; x < 16 * geo.nblocks; x += kFfmaThreads) {
        int I, J;
        block_ij(x % geo.nblocks, I, J);
        const int rq = x / geo.nblocks;
        const int i = 4 * I + (rq >> 2), j = 4 * J + (rq & 3);
        slot_col[x] = (i < geo.R && j < i) ? D + i * (i - 1) / 2 + j : -1;
    }
    int myI = 0, myJ = 0;
    if (lane < geo.nblocks) block_ij(lane, myI, myJ);
    // staging: when 128 % cpr == 0 every thread owns one chunk column
    const bool fixed_col = (kFfmaThreads % cpr) == 0;
    const int c0 = tid % cpr, i0 = tid / cpr, istep = kFfmaThreads / cpr;
    __syncthreads();

    for (int b = blockIdx.x; b < B; b += gridDim.x) {
        const T* drow = dense + (int64_t)b * D;
        const T* prow = pooled + (int64_t)b * F * D - D;   // row i >= 1 of Z at prow + i*D
        // ---- stage Z (all chunks of the sample in flight)
        if constexpr (sizeof(T) == 4) {
            if (fixed_col) {
                for (int i = i0; i < geo.R; i += istep)
                    cp_async16(zs + zoff(i, c0, ld), (i == 0 ? drow : prow + (int64_t)i * D) + 4 * c0);
            } else {
                for (int x = tid; x < geo.R * cpr; x += kFfmaThreads) {
                    const int i = x / cpr, c = x - i * cpr;
                    cp_async16(zs + zoff(i, c, ld), (i == 0 ? drow : prow + (int64_t)i * D) + 4 * c);
                }
            }
            cp_async_wait_all();
        } else {
            for (int x = tid; x < geo.R * cpr; x += kFfmaThreads) {
                const int i = x / cpr, c = x - i * cpr;
                float f[8];
                h8_to_f8(ldg_nc_v4((i == 0 ? drow : prow + (int64_t)i * D) + 8 * c), f);
                *reinterpret_cast<float4*>(zs + zoff(i, 2 * c, ld)) = make_float4(f[0], f[1], f[2], f[3]);
                *reinterpret_cast<float4*>(zs + zoff(i, 2 * c + 1, ld)) = make_float4(f[4], f[5], f[6], f[7]);
            }
        }
        __syncthreads();
        for (int k = tid; k < D; k += kFfmaThreads) os[k] = zs[zoff(0, k >> 2, ld) + (k & 3)];
        // ---- this warp's quarter of K for every 4x4 block
        for (int blk = lane; blk < geo.nblocks; blk += kWarp) {
            int I = myI, J = myJ;
            if (blk != lane) block_ij(blk, I, J);
            float acc[4][4];
            block_dot<DT>(zs, ld, C, warp, I, J, acc);
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int q = 0; q < 4; ++q) part[(warp * 16 + r * 4 + q) * geo.nblocks + blk] = acc[r][q];
        }
        __syncthreads();
        // ---- the four K quarters, added in a fixed order
        const int nslot = 16 * geo.nblocks;
        for (int x = tid; x < nslot; x += kFfmaThreads) {
            const int col = slot_col[x];
            if (col >= 0) {
                float v = part[x];
#pragma unroll
                for (int w = 1; w < kSplit; ++w) v += part[w * nslot + x];
                os[col] = v;
            }
        }
        __syncthreads();
        T* orow = out + (int64_t)b * P;
        for (int x = tid; x < P; x += kFfmaThreads) orow[x] = to_out<T>(os[x]);
    }
}

template <typename T, int DT>
dlrm_status launch_ffma_t(const void* dense, const void* pooled, int F, int D, int B, void* out, int P,
                          cudaStream_t stream)
{
    const FfmaGeom g = ffma_geom(F, D, P);
    const size_t smem = (size_t)g.smem_bytes;
    if (smem > 200 * 1024)
        return fail(DLRM_ERR_UNSUPPORTED, "dlrm_interact_fwd: (F+1) x D too large for the CUDA-core kernel");
    auto kern = interact_fwd_ffma_kernel<T, DT>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return fail(DLRM_ERR_CUDA, "dlrm_interact_fwd: %s", cudaGetErrorString(e));
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kFfmaThreads, smem);
    if (e != cudaSuccess || per_sm < 1) per_sm = 1;
    int64_t blocks = B;
    const int64_t cap = (int64_t)num_sms() * per_sm;
    if (blocks > cap) blocks = cap;
    kern<<<(int)blocks, kFfmaThreads, smem, stream>>>((const T*)dense, (const T*)pooled, F, D, B, (T*)out, P);
    return check_launch("interact_fwd_ffma_kernel");
}

template <typename T>
dlrm_status launch_ffma(const void* dense, const void* pooled, int F, int D, int B, void* out, int P,
                        cudaStream_t stream)
{
    if (D == 128) return launch_ffma_t<T, 128>(dense, pooled, F, D, B, out, P, stream);
    return launch_ffma_t<T, 0>(dense, pooled, F, D, B, out, P, stream);
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
