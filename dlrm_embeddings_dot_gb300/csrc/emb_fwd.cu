// emb_fwd.cu -- embedding lookup with sum pooling ("DLRM For PyTorch",
// §Model architecture: one table per categorical feature; joint table layout
// of --embedding_type joint*; --hash_indices folds indices into the table).
//
// Design: a group of G lanes moves one row; each lane moves 16-byte chunks of
// it (D*s/16 chunks per row), so a row is read and written with fully
// coalesced 16-byte accesses.
//  * single-hot kernel (about one index per bag): a warp resolves 32 bags with
//    coalesced metadata loads, then keeps 8 row loads per lane in flight.  A
//    bag of one valid index is a bit copy of the row (the fp32 round trip of
//    one term is exact, so this equals the general sum).  Where one load
//    instruction moves a whole row (fp32 D of 68..128, fp16 D of 136..256),
//    the bags of several indices among the 32 are then summed as one list of
//    positions (pool_flat), and this kernel takes every batch: against one
//    bag per warp, at 64K samples of 26 bags over 1e6-row tables, 563 -> 247
//    us at 1.5 indices per bag, 694 -> 426 us at 4, bit-identical.
//  * multi-hot kernel (narrower rows): one bag per group, U = 4 positions in
//    flight, fp32 accumulation in bag order, one rounding to the table type.
// Bag bounds are clamped into [0, nnz]; malformed offsets set
// DLRM_STATUS_BAD_OFFSETS instead of reading outside the index list.
#include "common.cuh"

namespace dlrm {
namespace {

constexpr int kThreads = 256;

template <typename T> struct Vec;
template <> struct Vec<float> { static constexpr int n = 4; };
template <> struct Vec<__half> { static constexpr int n = 8; };

template <typename T>
__device__ __forceinline__ void acc_chunk(float* a, uint4 v)
{
    if constexpr (sizeof(T) == 4) {
        a[0] += __uint_as_float(v.x);
        a[1] += __uint_as_float(v.y);
        a[2] += __uint_as_float(v.z);
        a[3] += __uint_as_float(v.w);
    } else {
        float f[8];
        h8_to_f8(v, f);
#pragma unroll
        for (int i = 0; i < 8; ++i) a[i] += f[i];
    }
}

template <typename T>
__device__ __forceinline__ uint4 pack_chunk(const float* a)
{
    if constexpr (sizeof(T) == 4)
        return make_uint4(__float_as_uint(a[0]), __float_as_uint(a[1]), __float_as_uint(a[2]),
                          __float_as_uint(a[3]));
    else
        return f8_to_h8(a);
}

// Stores one chunk (Vec<T>::n elements) of a pooled row: as is, or fp32 -> fp16
// rounded to nearest (the fp16 pooled output of fp32 master rows).
template <typename T, typename TO>
__device__ __forceinline__ void store_chunk(TO* dst, uint4 v)
{
    if constexpr (sizeof(T) == sizeof(TO)) {
        *reinterpret_cast<uint4*>(dst) = v;
    } else {
        const __half2 lo = __floats2half2_rn(__uint_as_float(v.x), __uint_as_float(v.y));
        const __half2 hi = __floats2half2_rn(__uint_as_float(v.z), __uint_as_float(v.w));
        *reinterpret_cast<uint2*>(dst) =
            make_uint2(*reinterpret_cast<const uint32_t*>(&lo), *reinterpret_cast<const uint32_t*>(&hi));
    }
}

// Global row for index `i` of a table of n rows starting at `base`, or -1 if skipped.
__device__ __forceinline__ int64_t resolve_row(int64_t i, int64_t base, int64_t n, bool hash,
                                               uint32_t* status)
{
    if (hash) {
        if (n <= 0) {
            set_status(status, DLRM_STATUS_OOB_INDEX);
            return -1;
        }
        i %= n;
        if (i < 0) i += n;
    } else if (i < 0 || i >= n) {
        set_status(status, DLRM_STATUS_OOB_INDEX);
        return -1;
    }
    return base + i;
}

// Bag bounds [s, e) clamped into [0, nnz]; flags malformed offsets.
__device__ __forceinline__ void bag_bounds(const int32_t* __restrict__ offsets, int64_t bag, int64_t nnz,
                                           uint32_t* status, int64_t& s, int64_t& e)
{
    s = offsets[bag];
    e = offsets[bag + 1];
    if (s < 0 || e < s || e > nnz) {
        set_status(status, DLRM_STATUS_BAD_OFFSETS);
        s = s < 0 ? 0 : (s > nnz ? nnz : s);
        e = e < s ? s : (e > nnz ? nnz : e);
    }
}

// General sum over bag positions [s, e) for chunk `ch` of the row (U loads in flight).
template <typename T, int U>
__device__ __forceinline__ uint4 pool_bag(const T* __restrict__ tables, const int32_t* __restrict__ indices,
                                          int64_t s, int64_t e, int64_t base, int64_t n, int D, int ch,
                                          bool hash, uint32_t* status)
{
    constexpr int V = Vec<T>::n;
    float acc[V];
#pragma unroll
    for (int i = 0; i < V; ++i) acc[i] = 0.f;
    for (int64_t p = s; p < e; p += U) {
        const T* src[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            src[u] = nullptr;
            if (p + u < e) {
                int64_t r = resolve_row(indices[p + u], base, n, hash, status);
                if (r >= 0) src[u] = tables + r * D + (int64_t)ch * V;
            }
        }
        uint4 v[U];
#pragma unroll
        for (int u = 0; u < U; ++u) v[u] = src[u] ? ldg_nc_l1_v4(src[u]) : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (src[u]) acc_chunk<T>(acc, v[u]);
    }
    return pack_chunk<T>(acc);
}

template <typename T, typename TO, int G>
__global__ void __launch_bounds__(kThreads)
emb_fwd_multi_kernel(const T* __restrict__ tables, const int64_t* __restrict__ row_base, int F,
                     int D, int B, const int32_t* __restrict__ indices,
                     const int32_t* __restrict__ offsets, TO* __restrict__ pooled, bool hash,
                     uint32_t* status, int64_t nbags, int64_t nnz)
{
    pdl_wait();
    constexpr int V = Vec<T>::n;
    const int chunks = D / V;
    const int lane = threadIdx.x % G;
    const int64_t group = ((int64_t)blockIdx.x * kThreads + threadIdx.x) / G;
    const int64_t ngroups = (int64_t)gridDim.x * kThreads / G;
    for (int64_t g = group; g < nbags; g += ngroups) {
        const int b = (int)(g / F);
        const int t = (int)(g - (int64_t)b * F);
        const int64_t bag = (int64_t)t * B + b;
        int64_t s, e;
        bag_bounds(offsets, bag, nnz, status, s, e);
        const int64_t base = row_base[t], n = row_base[t + 1] - base;
        for (int ch = lane; ch < chunks; ch += G) {
            uint4 r = pool_bag<T, 4>(tables, indices, s, e, base, n, D, ch, hash, status);
            store_chunk<T, TO>(pooled + g * D + (int64_t)ch * V, r);
        }
    }
}

// The bags of several indices among the warp's 32 bags g0 + k (lane k holds
// bag k's length), one row per load instruction.  Their positions form one
// list in bag order: each lane takes one of 32 positions at a time, finds its
// bag (the last lane whose list offset is at most the position), loads and
// resolves its index; the warp then adds the rows kFlatU at a time, each bag's
// in position order from zero in fp32 exactly as pool_bag does, and stores a
// bag's sum when the next bag begins.  Index loads are coalesced and a row
// waits for one index load, not a bag's worth.
constexpr int kFlatU = 4;

template <typename T, typename TO>
__device__ __forceinline__ void pool_flat(const T* __restrict__ tables, const int64_t* __restrict__ row_base,
                                          const int32_t* __restrict__ indices, const int32_t* __restrict__ offsets,
                                          TO* __restrict__ pooled, int F, int D, int B, int64_t g0, int64_t nnz,
                                          int lane, int cl, bool active, int len, bool hash, uint32_t* status)
{
    constexpr int V = Vec<T>::n;
    const int cnt = len > 1 ? len : 0;
    // this lane's bag again (its bounds were loaded by the caller; fetched here, not kept live)
    int start = 0, tbl = 0;
    if (cnt > 0) {
        const int64_t g = g0 + lane;   // < nbags, as len > 1
        int64_t s, e;
        bag_bounds(offsets, g, nnz, status, s, e);
        start = (int)s;
        tbl = (int)(g / B);
    }
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < kWarp; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    const int excl = incl - cnt;
    const int total = __shfl_sync(0xffffffffu, incl, kWarp - 1);
    float acc[V];
#pragma unroll
    for (int i = 0; i < V; ++i) acc[i] = 0.f;
    int cur = -1;   // lane of the bag being summed (warp-uniform)
    auto flush = [&](int k) {   // bag g0 + k = t*B + b goes to pooled row b*F + t (F*B < 2^31)
        const int g = (int)(g0 + k), t = g / B;
        const int64_t o = (int64_t)(g - t * B) * F + t;
        if (active) store_chunk<T, TO>(pooled + o * D + (int64_t)cl * V, pack_chunk<T>(acc));
#pragma unroll
        for (int i = 0; i < V; ++i) acc[i] = 0.f;
    };
    for (int q0 = 0; q0 < total; q0 += kWarp) {
        const int q = q0 + lane;
        int k = 0;   // the last lane with excl <= q: its bag holds position q
#pragma unroll
        for (int step = kWarp / 2; step > 0; step >>= 1)
            if (__shfl_sync(0xffffffffu, excl, k + step) <= q) k += step;
        const int p = __shfl_sync(0xffffffffu, start, k) + (q - __shfl_sync(0xffffffffu, excl, k));
        const int t = __shfl_sync(0xffffffffu, tbl, k);
        int64_t r = -1;
        if (q < total) {
            const int64_t kb = row_base[t];
            r = resolve_row(indices[p], kb, row_base[t + 1] - kb, hash, status);
        }
        const int m = total - q0 < kWarp ? total - q0 : kWarp;
        for (int j0 = 0; j0 < m; j0 += kFlatU) {
            uint4 v[kFlatU];
            int64_t rj[kFlatU];
#pragma unroll
            for (int u = 0; u < kFlatU; ++u) {
                rj[u] = __shfl_sync(0xffffffffu, r, (j0 + u) & (kWarp - 1));
                v[u] = (j0 + u < m && rj[u] >= 0 && active) ? ldg_nc_l1_v4(tables + rj[u] * D + (int64_t)cl * V)
                                                            : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int u = 0; u < kFlatU; ++u) {
                const int kj = __shfl_sync(0xffffffffu, k, (j0 + u) & (kWarp - 1));
                if (j0 + u >= m) break;
                if (kj != cur) {
                    if (cur >= 0) flush(cur);
                    cur = kj;
                }
                if (rj[u] >= 0) acc_chunk<T>(acc, v[u]);
            }
        }
    }
    if (cur >= 0) flush(cur);
}

// Single-hot kernel.  A warp takes 32 consecutive bags in CSR order (bag
// g = t*B + b, so the offsets and indices of the 32 bags are read with one
// coalesced load each), resolves their rows, then moves the rows with
// RPI = 32/G rows per load instruction and U such instructions in flight per
// lane.  Writes go to pooled row b*F + t, a full row per group of lanes.
// Bags that do not hold exactly one index are summed afterwards by the
// whole warp (pool_flat where a load instruction moves a whole row).
template <typename T, typename TO, int G>
__device__ __forceinline__ void single_hot_body(const T* __restrict__ tables, const int64_t* __restrict__ row_base,
                                                int F, int D, int B, const int32_t* __restrict__ indices,
                                                const int32_t* __restrict__ offsets, TO* __restrict__ pooled,
                                                bool hash, uint32_t* status, int64_t nbags, int64_t nnz)
{
    pdl_wait();
    constexpr int V = Vec<T>::n;
    constexpr int RPI = kWarp / G;                // rows per load instruction
    constexpr int U = 8;                          // load instructions in flight per lane
    const int chunks = D / V;                     // <= G for this kernel
    const int lane = threadIdx.x % kWarp;
    const int sub = lane / G, cl = lane % G;
    const bool active = cl < chunks;
    const int64_t warp_id = ((int64_t)blockIdx.x * kThreads + threadIdx.x) / kWarp;
    const int64_t nwarps = (int64_t)gridDim.x * kThreads / kWarp;

    for (int64_t g0 = warp_id * kWarp; g0 < nbags; g0 += nwarps * kWarp) {
        // ---- metadata of bag g0 + lane
        const int64_t g = g0 + lane;
        int len = -1;                             // -1: no bag
        int64_t row = -1, orow = 0;
        if (g < nbags) {
            const int t = (int)(g / B);
            const int b = (int)(g - (int64_t)t * B);
            int64_t s, e;
            bag_bounds(offsets, g, nnz, status, s, e);
            len = (int)(e - s);
            orow = (int64_t)b * F + t;
            if (len == 1) {
                const int64_t base = row_base[t];
                row = resolve_row(indices[s], base, row_base[t + 1] - base, hash, status);
            }
        }
        // ---- rows of bags with at most one index (bit copies; zeros for empty or skipped)
#pragma unroll
        for (int k0 = 0; k0 < kWarp; k0 += RPI * U) {
            uint4 v[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int src_lane = k0 + u * RPI + sub;
                const int64_t r = __shfl_sync(0xffffffffu, row, src_lane);
                v[u] = (r >= 0 && active) ? ldg_nc_l1_v4(tables + r * D + (int64_t)cl * V) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int src_lane = k0 + u * RPI + sub;
                const int l = __shfl_sync(0xffffffffu, len, src_lane);
                const int64_t o = __shfl_sync(0xffffffffu, orow, src_lane);
                if (l >= 0 && l <= 1 && active) store_chunk<T, TO>(pooled + o * D + (int64_t)cl * V, v[u]);
            }
        }
        // ---- bags with several indices
        uint32_t multi = __ballot_sync(0xffffffffu, len > 1);
        if constexpr (RPI == 1) {
            if (multi)
                pool_flat<T, TO>(tables, row_base, indices, offsets, pooled, F, D, B, g0, nnz, lane, cl, active, len,
                                 hash, status);
        } else {
            // (several rows per load instruction) the whole warp, RPI bags at a time
            while (multi) {
                int pick[RPI];
#pragma unroll
                for (int q = 0; q < RPI; ++q) {
                    pick[q] = multi ? __ffs(multi) - 1 : -1;
                    if (multi) multi &= multi - 1;
                }
                const int mine = pick[sub];
                const int src = mine < 0 ? 0 : mine;
                const int64_t gg = g0 + src;
                const int64_t o = __shfl_sync(0xffffffffu, orow, src);
                if (mine >= 0 && active) {
                    const int t = (int)(gg / B);
                    int64_t s, e;
                    bag_bounds(offsets, gg, nnz, status, s, e);
                    const int64_t tb = row_base[t];
                    const uint4 r = pool_bag<T, 4>(tables, indices, s, e, tb, row_base[t + 1] - tb, D, cl, hash,
                                                   status);
                    store_chunk<T, TO>(pooled + o * D + (int64_t)cl * V, r);
                }
            }
        }
    }
}

template <typename T, typename TO, int G>
__global__ void __launch_bounds__(kThreads)
emb_fwd_single_kernel(const T* __restrict__ tables, const int64_t* __restrict__ row_base, int F, int D, int B,
                      const int32_t* __restrict__ indices, const int32_t* __restrict__ offsets,
                      TO* __restrict__ pooled, bool hash, uint32_t* status, int64_t nbags, int64_t nnz)
{
    single_hot_body<T, TO, G>(tables, row_base, F, D, B, indices, offsets, pooled, hash, status, nbags, nnz);
}

// Whole-row groups (the pool_flat path) without a type conversion: held to 64
// registers, 32 warps per SM (left to itself the compiler takes 73 and 24 warps,
// 2 % slower on single-hot batches).
template <typename T, typename TO>
__global__ void __launch_bounds__(kThreads, 4)
emb_fwd_single_row_kernel(const T* __restrict__ tables, const int64_t* __restrict__ row_base, int F, int D, int B,
                          const int32_t* __restrict__ indices, const int32_t* __restrict__ offsets,
                          TO* __restrict__ pooled, bool hash, uint32_t* status, int64_t nbags, int64_t nnz)
{
    single_hot_body<T, TO, kWarp>(tables, row_base, F, D, B, indices, offsets, pooled, hash, status, nbags, nnz);
}

int64_t grid_for(int64_t groups, int G)
{
    int64_t blocks = (groups * G + kThreads - 1) / kThreads;
    int64_t cap = (int64_t)num_sms() * (2048 / kThreads);
    if (blocks > cap) blocks = cap;
    return blocks < 1 ? 1 : blocks;
}

template <typename T, typename TO, int G>
void launch(const void* tables, const int64_t* row_base, int F, int D, int B,
            const int32_t* indices, const int32_t* offsets, void* pooled, bool hash,
            uint32_t* status, int64_t nbags, int64_t nnz, bool single_hot, cudaStream_t stream)
{
    const int blocks = (int)grid_for((nbags + kWarp - 1) / kWarp, kWarp);
    bool launched = false;
    if constexpr (G == kWarp && sizeof(T) == sizeof(TO)) {
        if (single_hot) {
            launch_pdl(emb_fwd_single_row_kernel<T, TO>, blocks, kThreads, 0, stream,
                (const T*)tables, row_base, F, D, B, indices, offsets, (TO*)pooled, hash, status, nbags, nnz);
            launched = true;
        }
    } else if (single_hot && D / Vec<T>::n <= G) {
        launch_pdl(emb_fwd_single_kernel<T, TO, G>, blocks, kThreads, 0, stream,
            (const T*)tables, row_base, F, D, B, indices, offsets, (TO*)pooled, hash, status, nbags, nnz);
        launched = true;
    }
    if (!launched)
        launch_pdl(emb_fwd_multi_kernel<T, TO, G>, (int)grid_for(nbags, G), kThreads, 0, stream,
            (const T*)tables, row_base, F, D, B, indices, offsets, (TO*)pooled, hash, status, nbags, nnz);
}

template <typename T, typename TO>
dlrm_status dispatch(const void* tables, const int64_t* row_base, int F, int D, int B,
                     const int32_t* indices, const int32_t* offsets, void* pooled, bool hash,
                     uint32_t* status, int64_t nbags, int64_t nnz, bool single_hot, cudaStream_t stream)
{
    const int chunks = D * (int)sizeof(T) / 16;
    if (chunks <= 4)
        launch<T, TO, 4>(tables, row_base, F, D, B, indices, offsets, pooled, hash, status, nbags, nnz, single_hot, stream);
    else if (chunks <= 8)
        launch<T, TO, 8>(tables, row_base, F, D, B, indices, offsets, pooled, hash, status, nbags, nnz, single_hot, stream);
    else if (chunks <= 16)
        launch<T, TO, 16>(tables, row_base, F, D, B, indices, offsets, pooled, hash, status, nbags, nnz, single_hot, stream);
    else
        launch<T, TO, 32>(tables, row_base, F, D, B, indices, offsets, pooled, hash, status, nbags, nnz, single_hot, stream);
    return check_launch("emb_fwd kernel");
}

}  // namespace
}  // namespace dlrm

using namespace dlrm;

extern "C" dlrm_status dlrm_emb_fwd(const void* d_tables, dlrm_dtype dtype,
                                    const int64_t* d_row_base, int F, int D, int B,
                                    const int32_t* d_indices, const int32_t* d_offsets,
                                    int64_t nnz, void* d_pooled, unsigned flags,
                                    uint32_t* d_status, void* stream)
{
    DLRM_API_RANGE("dlrm_emb_fwd");
    clear_error();
    if (!dtype_ok(dtype)) return fail(DLRM_ERR_INVALID_ARG, "dlrm_emb_fwd: bad dtype");
    if (F < 1 || D < 1 || B < 0)
        return fail(DLRM_ERR_INVALID_ARG, "dlrm_emb_fwd: need F >= 1, D >= 1, B >= 0 (got %d, %d, %d)",
                    F, D, B);
    if (nnz < 0 || nnz > DLRM_MAX_NNZ)
        return fail(DLRM_ERR_INVALID_ARG, "dlrm_emb_fwd: nnz must be in [0, DLRM_MAX_NNZ]");
    if ((int64_t)F * B >= (int64_t)1 << 31)
        return fail(DLRM_ERR_INVALID_ARG, "dlrm_emb_fwd: F*B must be below 2^31");
    if (!d_tables || !d_row_base || !d_offsets || !d_pooled || (nnz > 0 && !d_indices))
        return fail(DLRM_ERR_INVALID_ARG, "dlrm_emb_fwd: null device pointer");
    if (flags & ~(DLRM_FLAG_HASH_INDICES | DLRM_FLAG_POOLED_F16))
        return fail(DLRM_ERR_INVALID_ARG, "dlrm_emb_fwd: unknown flag bits 0x%x", flags);
    const bool out_f16 = (flags & DLRM_FLAG_POOLED_F16) != 0;
    if (out_f16 && dtype != DLRM_F32)
        return fail(DLRM_ERR_INVALID_ARG, "dlrm_emb_fwd: DLRM_FLAG_POOLED_F16 needs fp32 tables");
    const int s = dtype_size(dtype);
    if (((int64_t)D * s) % 16 != 0)
        return fail(DLRM_ERR_UNSUPPORTED, "dlrm_emb_fwd: D*%d bytes must be a multiple of 16", s);
    if (!aligned16(d_tables) || !aligned16(d_pooled))
        return fail(DLRM_ERR_UNSUPPORTED, "dlrm_emb_fwd: tables and pooled must be 16-byte aligned");
    const int64_t nbags = (int64_t)F * B;
    if (nbags == 0) return DLRM_OK;
    const bool hash = (flags & DLRM_FLAG_HASH_INDICES) != 0;
    // The single-hot kernel takes batches of about one index per bag and, where one load instruction
    // moves a whole row (its bags of several indices then go through pool_flat), every batch.
    const int chunks = D * dtype_size(dtype) / 16;
    const bool flat = chunks > 16 && chunks <= 32;
    const bool single_hot = flat || nnz <= nbags + nbags / 8;
    cudaStream_t st = as_stream(stream);
    if (dtype == DLRM_F32 && out_f16)
        return dispatch<float, __half>(d_tables, d_row_base, F, D, B, d_indices, d_offsets, d_pooled, hash,
                                       d_status, nbags, nnz, single_hot, st);
    if (dtype == DLRM_F32)
        return dispatch<float, float>(d_tables, d_row_base, F, D, B, d_indices, d_offsets, d_pooled, hash,
                                      d_status, nbags, nnz, single_hot, st);
    return dispatch<__half, __half>(d_tables, d_row_base, F, D, B, d_indices, d_offsets, d_pooled, hash,
                                    d_status, nbags, nnz, single_hot, st);
}
