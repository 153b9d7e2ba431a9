// emb_fwd.cu -- embedding lookup with sum pooling ("DLRM For PyTorch",
// §Model architecture: one table per categorical feature; joint table layout
// of --embedding_type joint*; --hash_indices folds indices into the table).
//
// Design: a group of G lanes owns one bag at a time; each lane moves 16-byte
// chunks of a row (D*s/16 chunks per row), so a row is read with fully
// coalesced 16-byte loads.  Bags are walked in [b][t] order so that
// consecutive groups write consecutive pooled rows.
//  * single-hot kernel (about one index per bag): a group keeps NB = 4 bags in
//    flight and is software pipelined: the offsets and indices of the next NB
//    bags are fetched while the current rows are in flight.  A bag of one
//    valid index is a bit copy of the row (the fp32 round trip of one term is
//    exact, so this equals the general sum); other bags take the general path.
//  * multi-hot kernel: one bag per group, U = 4 positions in flight, fp32
//    accumulation in bag order, one rounding to the table type.
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
        for (int u = 0; u < U; ++u) v[u] = src[u] ? ldg_nc_v4(src[u]) : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (src[u]) acc_chunk<T>(acc, v[u]);
    }
    return pack_chunk<T>(acc);
}

template <typename T, int G>
__global__ void __launch_bounds__(kThreads)
emb_fwd_multi_kernel(const T* __restrict__ tables, const int64_t* __restrict__ row_base, int F,
                     int D, int B, const int32_t* __restrict__ indices,
                     const int32_t* __restrict__ offsets, T* __restrict__ pooled, bool hash,
                     uint32_t* status, int64_t nbags, int64_t nnz)
{
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
            *reinterpret_cast<uint4*>(pooled + g * D + (int64_t)ch * V) = r;
        }
    }
}

// Metadata of one bag for the single-hot kernel: source row (or null) and its
// index count (-1 = no bag).
template <typename T>
__device__ __forceinline__ void single_meta(const T* __restrict__ tables, const int64_t* __restrict__ row_base,
                                            const int32_t* __restrict__ indices,
                                            const int32_t* __restrict__ offsets, int F, int D, int B,
                                            int64_t g, int64_t nbags, int64_t nnz, int lane, bool hash,
                                            uint32_t* status, const T*& src, int& len)
{
    constexpr int V = Vec<T>::n;
    src = nullptr;
    len = -1;
    if (g < nbags) {
        const int b = (int)(g / F);
        const int t = (int)(g - (int64_t)b * F);
        int64_t s, e;
        bag_bounds(offsets, (int64_t)t * B + b, nnz, status, s, e);
        len = (int)(e - s);
        if (len == 1) {
            const int64_t base = row_base[t];
            const int64_t r = resolve_row(indices[s], base, row_base[t + 1] - base, hash, status);
            if (r >= 0) src = tables + r * D + (int64_t)lane * V;
        }
    }
}

template <typename T, int G, int NB>
__global__ void __launch_bounds__(kThreads)
emb_fwd_single_kernel(const T* __restrict__ tables, const int64_t* __restrict__ row_base, int F,
                      int D, int B, const int32_t* __restrict__ indices,
                      const int32_t* __restrict__ offsets, T* __restrict__ pooled, bool hash,
                      uint32_t* status, int64_t nbags, int64_t nnz)
{
    constexpr int V = Vec<T>::n;
    const int chunks = D / V;       // <= G for this kernel
    const int lane = threadIdx.x % G;
    const bool active = lane < chunks;
    const int64_t group = ((int64_t)blockIdx.x * kThreads + threadIdx.x) / G;
    const int64_t ngroups = (int64_t)gridDim.x * kThreads / G;
    const int64_t stride = (int64_t)NB * ngroups;

    const T* src[NB];
    int len[NB];
#pragma unroll
    for (int k = 0; k < NB; ++k)
        single_meta(tables, row_base, indices, offsets, F, D, B, group + (int64_t)k * ngroups, nbags, nnz,
                    lane, hash, status, src[k], len[k]);
    for (int64_t g0 = group; g0 < nbags; g0 += stride) {
        uint4 v[NB];
#pragma unroll
        for (int k = 0; k < NB; ++k)
            v[k] = (src[k] && active) ? ldg_nc_v4(src[k]) : make_uint4(0, 0, 0, 0);
        // next bags' metadata while the rows are in flight
        const T* nsrc[NB];
        int nlen[NB];
#pragma unroll
        for (int k = 0; k < NB; ++k)
            single_meta(tables, row_base, indices, offsets, F, D, B, g0 + stride + (int64_t)k * ngroups, nbags,
                        nnz, lane, hash, status, nsrc[k], nlen[k]);
#pragma unroll
        for (int k = 0; k < NB; ++k) {
            const int64_t g = g0 + (int64_t)k * ngroups;
            if (len[k] >= 0 && active) {
                if (len[k] != 1) {                    // empty or multi-index bag: general sum
                    const int b = (int)(g / F);
                    const int t = (int)(g - (int64_t)b * F);
                    int64_t s, e;
                    bag_bounds(offsets, (int64_t)t * B + b, nnz, status, s, e);
                    const int64_t base = row_base[t];
                    v[k] = pool_bag<T, 4>(tables, indices, s, e, base, row_base[t + 1] - base, D, lane, hash,
                                          status);
                }
                *reinterpret_cast<uint4*>(pooled + g * D + (int64_t)lane * V) = v[k];
            }
            src[k] = nsrc[k];
            len[k] = nlen[k];
        }
    }
}

int64_t grid_for(int64_t groups, int G)
{
    int64_t blocks = (groups * G + kThreads - 1) / kThreads;
    int64_t cap = (int64_t)num_sms() * (2048 / kThreads);
    if (blocks > cap) blocks = cap;
    return blocks < 1 ? 1 : blocks;
}

template <typename T, int G>
void launch(const void* tables, const int64_t* row_base, int F, int D, int B,
            const int32_t* indices, const int32_t* offsets, void* pooled, bool hash,
            uint32_t* status, int64_t nbags, int64_t nnz, bool single_hot, cudaStream_t stream)
{
    constexpr int NB = 4;
    if (single_hot && D / Vec<T>::n <= G)
        emb_fwd_single_kernel<T, G, NB><<<(int)grid_for((nbags + NB - 1) / NB, G), kThreads, 0, stream>>>(
            (const T*)tables, row_base, F, D, B, indices, offsets, (T*)pooled, hash, status, nbags, nnz);
    else
        emb_fwd_multi_kernel<T, G><<<(int)grid_for(nbags, G), kThreads, 0, stream>>>(
            (const T*)tables, row_base, F, D, B, indices, offsets, (T*)pooled, hash, status, nbags, nnz);
}

template <typename T>
dlrm_status dispatch(const void* tables, const int64_t* row_base, int F, int D, int B,
                     const int32_t* indices, const int32_t* offsets, void* pooled, bool hash,
                     uint32_t* status, int64_t nbags, int64_t nnz, bool single_hot, cudaStream_t stream)
{
    const int chunks = D * (int)sizeof(T) / 16;
    if (chunks <= 4)
        launch<T, 4>(tables, row_base, F, D, B, indices, offsets, pooled, hash, status, nbags, nnz, single_hot, stream);
    else if (chunks <= 8)
        launch<T, 8>(tables, row_base, F, D, B, indices, offsets, pooled, hash, status, nbags, nnz, single_hot, stream);
    else if (chunks <= 16)
        launch<T, 16>(tables, row_base, F, D, B, indices, offsets, pooled, hash, status, nbags, nnz, single_hot, stream);
    else
        launch<T, 32>(tables, row_base, F, D, B, indices, offsets, pooled, hash, status, nbags, nnz, single_hot, stream);
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
    clear_error();
    if (!dtype_ok(dtype)) return fail(DLRM_ERR_INVALID_ARG, "dlrm_emb_fwd: bad dtype");
    if (F < 1 || D < 1 || B < 0)
        return fail(DLRM_ERR_INVALID_ARG, "dlrm_emb_fwd: need F >= 1, D >= 1, B >= 0 (got %d, %d, %d)",
                    F, D, B);
    if (nnz < 0 || nnz >= (int64_t)1 << 31)
        return fail(DLRM_ERR_INVALID_ARG, "dlrm_emb_fwd: nnz must be in [0, 2^31)");
    if ((int64_t)F * B >= (int64_t)1 << 31)
        return fail(DLRM_ERR_INVALID_ARG, "dlrm_emb_fwd: F*B must be below 2^31");
    if (!d_tables || !d_row_base || !d_offsets || !d_pooled || (nnz > 0 && !d_indices))
        return fail(DLRM_ERR_INVALID_ARG, "dlrm_emb_fwd: null device pointer");
    if (flags & ~DLRM_FLAG_HASH_INDICES)
        return fail(DLRM_ERR_INVALID_ARG, "dlrm_emb_fwd: unknown flag bits 0x%x", flags);
    const int s = dtype_size(dtype);
    if (((int64_t)D * s) % 16 != 0)
        return fail(DLRM_ERR_UNSUPPORTED, "dlrm_emb_fwd: D*%d bytes must be a multiple of 16", s);
    if (!aligned16(d_tables) || !aligned16(d_pooled))
        return fail(DLRM_ERR_UNSUPPORTED, "dlrm_emb_fwd: tables and pooled must be 16-byte aligned");
    const int64_t nbags = (int64_t)F * B;
    if (nbags == 0) return DLRM_OK;
    const bool hash = (flags & DLRM_FLAG_HASH_INDICES) != 0;
    const bool single_hot = nnz <= nbags + nbags / 8;   // about one index per bag
    cudaStream_t st = as_stream(stream);
    if (dtype == DLRM_F32)
        return dispatch<float>(d_tables, d_row_base, F, D, B, d_indices, d_offsets, d_pooled, hash,
                               d_status, nbags, nnz, single_hot, st);
    return dispatch<__half>(d_tables, d_row_base, F, D, B, d_indices, d_offsets, d_pooled, hash,
                            d_status, nbags, nnz, single_hot, st);
}
