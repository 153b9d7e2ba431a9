// interact_fwd.cu -- dot interaction ("DLRM For PyTorch", §Model
// architecture; --interaction_op cuda_dot): pairwise dot products among the
// bottom-MLP output and the F pooled embeddings, strict lower triangle in
// row-major order, concatenated after the dense vector, zero padded.
//
// This file holds the CUDA-core kernels, used for fp32 (a single TF32
// product cannot meet fp32 accuracy, and the three-product split measured
// slower than these kernels) and for fp16 shapes the tensor-core kernel does
// not take, plus the entry point that picks among them.
//
// Where every operand float must be read from shared memory, the shared-memory
// pipe bounds the arithmetic: a wavefront delivers 32 lane-words per clock
// while the FMA pipes consume 128 products, so a lane needs four products per
// float it loads (8x8 register tiles, which waste half their products on the
// triangle).  The kernel for the common fp32 shape therefore keeps the
// operands in registers and moves partial sums instead:
//
// Register kernel (fp32, D = 128, F + 1 rows of Z known at compile time): one
// warp per sample.  Lane l holds features 4l..4l+3 of every row of Z in
// registers and forms its four-feature partial dot products for all F(F+1)/2
// pairs (i, j), j < i, in output order, in groups of 32 -- no wasted product
// (two packed fp32x2 instructions and one add per pair).  Each group is
// finished by a transpose through a per-warp 32 x 36 shared scratch: lane l
// stores its 32 partials as row l (four 16-byte stores, no bank conflict with
// the 36-float pitch), and lane t adds column t (32 conflict-free 4-byte reads
// into 8 interleaved sums, then a 3-level tree: a dependent chain of 6 adds
// instead of 31), which leaves the dot product of the group's pair t in lane
// t: 32 consecutive output columns, one coalesced store.  The kernel is bound
// by each warp's own latency (its time scales with 1 / resident warps, which
// registers and shared memory cap at 12 per SM), so shorter chains and fewer
// instructions pay; moving part of the reduction to shuffles (fewer shared
// wavefronts, more instructions) measured slower.  A sample
// arrives in the warp's buffer by two bulk copies (the dense row, then the F
// pooled rows, contiguous in global memory) completing on the warp's
// mbarrier; the next sample's copy is issued after the first group, behind a
// warp barrier that orders the buffer's reads before the refill.
//
// Tile kernel (any shape): one CTA of 4 warps per sample at a time.  Z = [dense; pooled
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
#include <type_traits>
#include <utility>

#include "common.cuh"
#include "interact_tc.cuh"
#include "reg_gather.cuh"
#include "tcgen05.cuh"

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
    pdl_wait();
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

// ------------------------------------------------------------ register kernel
constexpr int kRegWarps = 4;     // warps per CTA, one sample each at a time
constexpr int kRegD = 128;       // 32 lanes x 4 features
constexpr int kPitch = 36;       // floats per row of the transpose scratch
constexpr int kGatherRing = 8;   // staging rows of the one-pass gather (8 x 512 bytes <= the scratch)
static_assert(kGatherRing * kRegD <= 32 * kPitch, "gather ring larger than the transpose scratch");

// Pair p of the strict lower triangle in row-major order: p = i(i-1)/2 + j.
constexpr int pair_row(int p)
{
    int i = 1;
    while (i * (i + 1) / 2 <= p) ++i;
    return i;
}

// Four-feature dot product with the packed two-lane fp32 instructions (each
// lane of mul/fma.rn.f32x2 rounds as the scalar instruction does): features
// (x, y) and (z, w) side by side, then the two halves added, in half the
// multiply-add instructions of four scalar ones.
__device__ __forceinline__ uint64_t pack2(float lo, float hi)
{
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}

__device__ __forceinline__ float dot4(const float4& a, const float4& b)
{
    uint64_t p;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(p) : "l"(pack2(a.x, a.y)), "l"(pack2(b.x, b.y)));
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(p) : "l"(pack2(a.z, a.w)), "l"(pack2(b.z, b.w)));
    float xz, yw;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(xz), "=f"(yw) : "l"(p));
    return xz + yw;
}

// Four-feature partial dot product of pair p (zero past the last pair).
template <int R, int p>
__device__ __forceinline__ float slot_dot(const float4 (&z)[R])
{
    if constexpr (p < R * (R - 1) / 2) {
        constexpr int i = pair_row(p);
        constexpr int j = p - i * (i - 1) / 2;
        return dot4(z[i], z[j]);
    } else {
        return 0.f;
    }
}

// Shared memory of one CTA: [kRegWarps][R rows][D floats] sample buffers,
// [kRegWarps][32][kPitch] transpose scratch, kRegWarps mbarriers.
template <int R>
constexpr size_t regs_smem_bytes()
{
    return (size_t)kRegWarps * R * kRegD * 4 + (size_t)kRegWarps * 32 * kPitch * 4 + kRegWarps * 8;
}

// The interaction of one sample whose Z rows (features 4l..4l+3 in lane l)
// are in z: the dense block and the F(F+1)/2 dot products of output row orow.
// after_first = work to start once the first group has passed its barrier
// (the sample buffer z came from may then be refilled).
template <int R, int kAfter = 0, typename Fn>
__device__ __forceinline__ void regs_sample(const float4 (&z)[R], float* orow, int P, int lane, float* scratch,
                                            Fn&& after_first)
{
    constexpr int NP = R * (R - 1) / 2;           // pairs
    constexpr int NG = (NP + 31) / 32;            // groups of 32 pairs
    constexpr int D = kRegD;
    *reinterpret_cast<float4*>(orow + 4 * lane) = z[0];
    static_for<NG>([&](auto G) {
        constexpr int g = decltype(G)::value;
        float v[32];
        static_for<32>([&](auto T) {
            constexpr int t = decltype(T)::value;
            v[t] = slot_dot<R, g * 32 + t>(z);
        });
        float* row = scratch + lane * kPitch;
#pragma unroll
        for (int q = 0; q < 8; ++q)
            *reinterpret_cast<float4*>(row + 4 * q) = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
        __syncwarp();
        float s8[8];
#pragma unroll
        for (int r = 0; r < 8; ++r) s8[r] = scratch[r * kPitch + lane];
#pragma unroll
        for (int r = 8; r < 32; ++r) s8[r & 7] += scratch[r * kPitch + lane];
        const float sum = ((s8[0] + s8[1]) + (s8[2] + s8[3])) + ((s8[4] + s8[5]) + (s8[6] + s8[7]));
        const int col = D + g * 32 + lane;
        if (col < P) orow[col] = sum;
        // orders this group's scratch reads before the next group's writes;
        // it also keeps the scheduler from hoisting later groups' products
        // into this group (which spills registers)
        __syncwarp();
        if constexpr (g == (kAfter < NG ? kAfter : NG - 1)) after_first();
    });
}

template <int R>
__global__ void __launch_bounds__(kRegWarps * kWarp, 3)
interact_fwd_regs_kernel(const float* __restrict__ dense, const float* __restrict__ pooled, int B,
                         float* __restrict__ out, int P, uint32_t* __restrict__ status)
{
    pdl_wait();
    constexpr int D = kRegD;
    extern __shared__ __align__(16) float4 zbuf[];
    const int lane = threadIdx.x % kWarp;
    const int warp = threadIdx.x / kWarp;
    float4* mine = zbuf + warp * R * kWarp;       // row r, features 4l..4l+3 at [r * 32 + l]
    float* const scratch_all = reinterpret_cast<float*>(zbuf + kRegWarps * R * kWarp);
    float* scratch = scratch_all + warp * 32 * kPitch;
    uint64_t* bar = reinterpret_cast<uint64_t*>(scratch_all + kRegWarps * 32 * kPitch) + warp;
    const int64_t stride = (int64_t)gridDim.x * kRegWarps;
    int64_t b = (int64_t)blockIdx.x * kRegWarps + warp;

    // row 0 of Z is the dense row, rows 1..F the sample's pooled rows
    auto stage = [&](int64_t s) {
        if (lane == 0) {
            tc::mbar_expect_tx(bar, R * D * 4);
            tc::bulk_g2s(mine, dense + s * D, D * 4, bar);
            tc::bulk_g2s(mine + kWarp, pooled + s * (int64_t)(R - 1) * D, (R - 1) * D * 4, bar);
        }
    };
    if (lane == 0) {
        tc::mbar_init(bar, 1);
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    __syncwarp();
    uint32_t phase = 0;
    if (b < B) stage(b);
    for (; b < B; b += stride) {
        if (!tc::bounded_wait(bar, phase)) {
            if (lane == 0) set_status(status, DLRM_STATUS_TIMEOUT);
            return;
        }
        phase ^= 1u;
        float4 z[R];
#pragma unroll
        for (int r = 0; r < R; ++r) z[r] = mine[r * kWarp + lane];
        const int64_t nb = b + stride;
        regs_sample<R>(z, out + b * P, P, lane, scratch, [&] {
            // the sample buffer was read before the group barrier
            if (nb < B) {
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                stage(nb);
            }
        });
    }
}

// ------------------------------------------- lookup + register kernel in one pass
// The same interaction, with the sample buffer filled straight from the
// tables: lane t < F resolves bag t of the warp's next sample (bounds two
// samples ahead, the index one sample ahead, as in the tensor-core fused
// kernel), then copies its single-index bag's row into the buffer with one
// bulk copy on the warp's mbarrier (the tensor-memory-access unit moves the
// rows, so the gather adds nothing to the shared-memory pipe that bounds the
// interaction); empty bags (and rejected indices) give zero rows, bags of
// several indices are summed in fp32 in bag order by the whole warp, their
// positions as one list streamed through the transpose scratch (free while
// the next sample is staged) eight rows at a time.
// The pooled rows (rows 1..F of the buffer) leave by one bulk store, so the
// lookup's output is written once and never read back.  Pooled rows and
// interaction are bit-identical to dlrm_emb_fwd + dlrm_interact_fwd.
// Shared memory: the same layout as the register kernel's.
template <int R>
constexpr size_t emb_regs_smem_bytes()
{
    return regs_smem_bytes<R>();
}

// kPooled: the pooled rows are stored (training).  The next sample is staged
// after group kAfter: right after the first group without the store, half way
// through with it, which leaves the bulk store time to read the buffer first
// (measured at 64K: 320 us staging after group 0, 282 us after group 5).
template <int R, bool kPooled>
__global__ void __launch_bounds__(kRegWarps * kWarp, 3)
emb_interact_regs_kernel(RegGather ga, const float* __restrict__ dense, int B, float* __restrict__ pooled,
                         float* __restrict__ out, int P, uint32_t* __restrict__ status)
{
    pdl_wait();
    constexpr int kAfter = kPooled ? (R * (R - 1) / 2 + 31) / 32 / 2 : 0;
    constexpr int F = R - 1;
    constexpr int D = kRegD;
    extern __shared__ __align__(16) float4 zbuf[];
    const int lane = threadIdx.x % kWarp;
    const int warp = threadIdx.x / kWarp;
    float4* mine = zbuf + warp * R * kWarp;
    float* const scratch_all = reinterpret_cast<float*>(zbuf + kRegWarps * R * kWarp);
    float* scratch = scratch_all + warp * 32 * kPitch;
    uint64_t* bar = reinterpret_cast<uint64_t*>(scratch_all + kRegWarps * 32 * kPitch) + warp;
    const int64_t stride = (int64_t)gridDim.x * kRegWarps;
    int64_t b = (int64_t)blockIdx.x * kRegWarps + warp;
    if (lane == 0) {
        tc::mbar_init(bar, 1);
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    __syncwarp();
    uint32_t phase = 0;
    const BagLanes<F, D> bags(ga, B, lane, status);
    // fill the buffer with sample smp: the bags' rows as rows 1..F, the dense
    // row (lane F's bulk copy) as row 0; lane 0 arrives once all are counted
    auto stage = [&](int64_t smp, uint32_t src_row, int a, int e) {
        // the transpose scratch is free while a sample is staged: it holds the
        // rows of several-index bags in flight
        bags.template gather<false, 4, kGatherRing>(mine, src_row, a, e, bar, reinterpret_cast<float4*>(scratch));
        if (lane == F) {
            tc::mbar_expect_tx_only(bar, D * 4);
            tc::bulk_g2s(mine, dense + smp * D, D * 4, bar);
        }
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(bar);
    };

    int a0, e0, a1, e1;
    bags.load_bounds(b, a0, e0);
    bags.load_bounds(b + stride, a1, e1);
    bags.clamp(a0, e0);
    if (b < B) stage(b, bags.resolve(a0, e0, bags.early_index(a0, e0)), a0, e0);
    bags.clamp(a1, e1);
    for (; b < B; b += stride) {
        const int64_t nb = b + stride;
        // in flight during this sample: the next sample's index, the bounds two samples on
        const int idx1 = bags.early_index(a1, e1);
        int a2, e2;
        bags.load_bounds(nb + stride, a2, e2);
        if (!tc::bounded_wait(bar, phase)) {
            if (lane == 0) {
                set_status(status, DLRM_STATUS_TIMEOUT);
                if (kPooled) tc::bulk_wait_all();
            }
            return;
        }
        phase ^= 1u;
        float4 z[R];
#pragma unroll
        for (int r = 0; r < R; ++r) z[r] = mine[r * kWarp + lane];
        if constexpr (kPooled) {
            // every lane's rows (cp.async and plain stores) -> visible to the bulk store
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (lane == 0) {
                tc::bulk_s2g(pooled + b * (int64_t)F * D, mine + kWarp, F * D * 4);
                tc::bulk_commit();
            }
        }
        regs_sample<R, kAfter>(z, out + b * P, P, lane, scratch, [&] {
            if constexpr (kPooled) {
                if (lane == 0) tc::bulk_wait_read<0>();   // the bulk store has read the buffer
                __syncwarp();
            }
            if (nb < B) {
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                stage(nb, bags.resolve(a1, e1, idx1), a1, e1);
            }
        });
        bags.clamp(a2, e2);
        a1 = a2;
        e1 = e2;
    }
    if (kPooled && lane == 0) tc::bulk_wait_all();
}

template <int R>
dlrm_status launch_regs(const float* dense, const float* pooled, int B, float* out, int P, uint32_t* status,
                        cudaStream_t stream)
{
    const size_t smem = regs_smem_bytes<R>();
    auto kern = interact_fwd_regs_kernel<R>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return fail(DLRM_ERR_CUDA, "dlrm_interact_fwd: %s", cudaGetErrorString(e));
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kRegWarps * kWarp, smem);
    if (e != cudaSuccess || per_sm < 1) per_sm = 1;
    const int64_t need = ((int64_t)B + kRegWarps - 1) / kRegWarps;
    const int64_t cap = (int64_t)num_sms() * per_sm;
    const int blocks = (int)(need < cap ? need : cap);
    return check_launch_pdl(launch_pdl(kern, blocks, kRegWarps * kWarp, smem, stream, dense, pooled, B, out, P, status),
                            "interact_fwd_regs_kernel");
}

template <int R, bool kPooled>
dlrm_status launch_emb_regs(const RegGather& ga, const float* dense, int B, float* pooled, float* out, int P,
                            uint32_t* status, cudaStream_t stream)
{
    const size_t smem = emb_regs_smem_bytes<R>();
    auto kern = emb_interact_regs_kernel<R, kPooled>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return fail(DLRM_ERR_CUDA, "dlrm_emb_interact_fwd: %s", cudaGetErrorString(e));
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kRegWarps * kWarp, smem);
    if (e != cudaSuccess || per_sm < 1) per_sm = 1;
    const int64_t need = ((int64_t)B + kRegWarps - 1) / kRegWarps;
    const int64_t cap = (int64_t)num_sms() * per_sm;
    const int blocks = (int)(need < cap ? need : cap);
    return check_launch_pdl(launch_pdl(kern, blocks, kRegWarps * kWarp, smem, stream, ga, dense, B, pooled, out, P,
                                       status),
                            "emb_interact_regs_kernel");
}

// Shapes the register kernel takes: fp32, D = 128, F in {8, 26}, rows of the
// output 16-byte aligned, and no padding column past the last group of 32
// pairs (the group's empty slots write the padding zeros).
inline bool regs_supported(int F, int D, int P, const void* out)
{
    const int groups = (F * (F + 1) / 2 + 31) / 32;
    return D == kRegD && (F == 8 || F == 26) && P % 4 == 0 && P <= kRegD + 32 * groups && aligned16(out);
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
    return check_launch_pdl(launch_pdl(kern, (int)blocks, kFfmaThreads, smem, stream, (const T*)dense, (const T*)pooled,
                                       F, D, B, (T*)out, P),
                            "interact_fwd_ffma_kernel");
}

template <typename T>
dlrm_status launch_ffma(const void* dense, const void* pooled, int F, int D, int B, void* out, int P,
                        uint32_t* status, cudaStream_t stream)
{
    if constexpr (sizeof(T) == 4) {
        if (regs_supported(F, D, P, out)) {
            const float* d = static_cast<const float*>(dense);
            const float* p = static_cast<const float*>(pooled);
            float* o = static_cast<float*>(out);
            return F == 26 ? launch_regs<27>(d, p, B, o, P, status, stream)
                           : launch_regs<9>(d, p, B, o, P, status, stream);
        }
    }
    if (D == 128) return launch_ffma_t<T, 128>(dense, pooled, F, D, B, out, P, stream);
    return launch_ffma_t<T, 0>(dense, pooled, F, D, B, out, P, stream);
}

}  // namespace

// fp32 lookup + interaction in one pass (pooled may be null); shapes as
// regs_supported, plus 16-byte-aligned tables and pooled.
bool regs_emb_interact_supported(int F, int D, int out_cols, const void* tables, const void* dense,
                                 const void* pooled, const void* out)
{
    return regs_supported(F, D, out_cols, out) && aligned16(tables) && aligned16(dense) &&
           (pooled == nullptr || aligned16(pooled));
}

dlrm_status regs_emb_interact_fwd(const float* tables, const int64_t* row_base, int F, int D, int B,
                                  const int32_t* indices, const int32_t* offsets, int64_t nnz, const float* dense,
                                  float* pooled, float* out, int out_cols, bool hash, uint32_t* status,
                                  cudaStream_t stream)
{
    (void)D;
    RegGather ga{tables, row_base, indices, offsets, nnz, hash};
    if (pooled)
        return F == 26 ? launch_emb_regs<27, true>(ga, dense, B, pooled, out, out_cols, status, stream)
                       : launch_emb_regs<9, true>(ga, dense, B, pooled, out, out_cols, status, stream);
    return F == 26 ? launch_emb_regs<27, false>(ga, dense, B, pooled, out, out_cols, status, stream)
                   : launch_emb_regs<9, false>(ga, dense, B, pooled, out, out_cols, status, stream);
}

}  // namespace dlrm

using namespace dlrm;

extern "C" dlrm_status dlrm_interact_fwd(const void* d_dense, const void* d_pooled, dlrm_dtype dtype,
                                         int F, int D, int B, void* d_out, int out_cols,
                                         uint32_t* d_status, void* stream)
{
    DLRM_API_RANGE("dlrm_interact_fwd");
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
    if (dtype == DLRM_F32) return launch_ffma<float>(d_dense, d_pooled, F, D, B, d_out, out_cols, d_status, st);
    return launch_ffma<__half>(d_dense, d_pooled, F, D, B, d_out, out_cols, d_status, st);
}

// CUDA-core path for any shape, exposed for tests of the tensor-core kernel.
extern "C" dlrm_status dlrm_interact_fwd_cuda_core(const void* d_dense, const void* d_pooled,
                                                   dlrm_dtype dtype, int F, int D, int B,
                                                   void* d_out, int out_cols, void* stream)
{
    DLRM_API_RANGE("dlrm_interact_fwd_cuda_core");
    clear_error();
    if (!dtype_ok(dtype) || F < 1 || D < 1 || B < 0 || !d_dense || !d_pooled || !d_out ||
        out_cols < (int64_t)D + (int64_t)F * (F + 1) / 2)
        return fail(DLRM_ERR_INVALID_ARG, "dlrm_interact_fwd_cuda_core: bad arguments");
    if (((int64_t)D * dtype_size(dtype)) % 16 != 0 || !aligned16(d_dense) || !aligned16(d_pooled))
        return fail(DLRM_ERR_UNSUPPORTED, "dlrm_interact_fwd_cuda_core: alignment");
    if (B == 0) return DLRM_OK;
    cudaStream_t st = as_stream(stream);
    if (dtype == DLRM_F32) return launch_ffma<float>(d_dense, d_pooled, F, D, B, d_out, out_cols, nullptr, st);
    return launch_ffma<__half>(d_dense, d_pooled, F, D, B, d_out, out_cols, nullptr, st);
}

extern "C" dlrm_status dlrm_emb_interact_fwd_train(const void* d_tables, dlrm_dtype dtype, const int64_t* d_row_base,
                                                   int F, int D, int B, const int32_t* d_indices,
                                                   const int32_t* d_offsets, int64_t nnz, const void* d_dense,
                                                   void* d_pooled, void* d_out, int out_cols, unsigned flags,
                                                   uint32_t* d_status, void* stream)
{
    DLRM_API_RANGE("dlrm_emb_interact_fwd_train");
    clear_error();
    if (!dtype_ok(dtype)) return fail(DLRM_ERR_INVALID_ARG, "dlrm_emb_interact_fwd_train: bad dtype");
    if (F < 1 || D < 1 || B < 0)
        return fail(DLRM_ERR_INVALID_ARG, "dlrm_emb_interact_fwd_train: need F >= 1, D >= 1, B >= 0");
    if (nnz < 0 || nnz > DLRM_MAX_NNZ || (int64_t)F * B >= (int64_t)1 << 31)
        return fail(DLRM_ERR_INVALID_ARG, "dlrm_emb_interact_fwd_train: need nnz <= DLRM_MAX_NNZ and F*B < 2^31");
    const int64_t W = (int64_t)D + (int64_t)F * (F + 1) / 2;
    if (out_cols < W)
        return fail(DLRM_ERR_INVALID_ARG, "dlrm_emb_interact_fwd_train: out_cols %d < D + F(F+1)/2 = %lld",
                    out_cols, (long long)W);
    if (!d_tables || !d_row_base || !d_offsets || !d_dense || !d_pooled || !d_out || (nnz > 0 && !d_indices))
        return fail(DLRM_ERR_INVALID_ARG, "dlrm_emb_interact_fwd_train: null device pointer");
    if (flags & ~DLRM_FLAG_HASH_INDICES)
        return fail(DLRM_ERR_INVALID_ARG, "dlrm_emb_interact_fwd_train: unknown flag bits 0x%x", flags);
    if (dtype != DLRM_F32 || !regs_emb_interact_supported(F, D, out_cols, d_tables, d_dense, d_pooled, d_out))
        return fail(DLRM_ERR_UNSUPPORTED,
                    "dlrm_emb_interact_fwd_train: needs fp32, D = 128, F in {8, 26}, out_cols a multiple of 4 "
                    "without padding past the last group of 32 pairs, and 16-byte aligned pointers (use "
                    "dlrm_emb_fwd + dlrm_interact_fwd otherwise)");
    if (B == 0) return DLRM_OK;
    const int64_t nbags = (int64_t)F * B;
    if (nnz > 3 * nbags) {
        // Many indices per bag: one warp per sample streams its sample's rows eight at a time, while
        // the lookup spreads the bags over all warps with more rows in flight (64K samples of 26 bags
        // over 1e6-row tables: one pass 0.427 against 0.465 ms as two launches at 1.5 indices per
        // bag, 0.730 against 0.700 at 4).  The two launches compute the same bits, so the choice is
        // by speed alone.
        dlrm_status s = dlrm_emb_fwd(d_tables, dtype, d_row_base, F, D, B, d_indices, d_offsets, nnz, d_pooled,
                                     flags, d_status, stream);
        if (s != DLRM_OK) return s;
        return dlrm_interact_fwd(d_dense, d_pooled, dtype, F, D, B, d_out, out_cols, d_status, stream);
    }
    return regs_emb_interact_fwd((const float*)d_tables, d_row_base, F, D, B, d_indices, d_offsets, nnz,
                                 (const float*)d_dense, (float*)d_pooled, (float*)d_out, out_cols,
                                 (flags & DLRM_FLAG_HASH_INDICES) != 0, d_status, as_stream(stream));
}
