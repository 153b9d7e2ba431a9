// emb_bwd_sgd.cu -- sparse embedding gradient fused with the SGD row update.
//
// The gradient of the sum pooling ("DLRM For PyTorch", §Model architecture)
// sends grad_pooled[b][t] to every row of bag (t, b); the tables are FP32
// (§Training process) and only touched rows change (--embedding_type
// joint_sparse).  No dense gradient table is formed:
//
//  1. keys: position p of bag (t, b) -> (key = global row, val = b*F + t);
//     skipped indices get key 0xFFFFFFFF.
//  2. stable LSD radix sort of (key, val) over the bits that can be set,
//     8 bits per pass, reduce-then-scan (no inter-block waiting):
//     per-tile digit histograms -> per-digit scan over tiles -> stable
//     scatter with warp-level ranking (match.any) in position order.
//  3. segments: the sorted array is cut into chunks of 32 positions; a warp
//     sums, in ascending position order, the grad rows of each run of equal
//     keys inside its chunk.  A run wholly inside the chunk updates its row
//     at once (w = fmaf(-lr, g, w)); a run crossing a chunk edge leaves one
//     partial sum per chunk it touches.
//     The chunk where such a run starts finds the run's last chunk (an
//     exponential probe of chunk heads, then 32-ary refinement) and files
//     the run with its number of pieces.
//  4. fixup (one kernel): runs of more than 64 pieces are summed by one block
//     each (16 warps add 16 contiguous slices of pieces, then the 16 sums in
//     slice order), the others by one warp each, pieces in chunk order; a
//     lane keeps up to 4 partial-sum loads in flight.
// Every order of summation is fixed by the data, so results are bitwise
// reproducible.  Workspace layout (256-byte aligned pieces):
//   keysA | valsA | keysB | valsB | hist[256][ntiles] | totals[256] |
//   partials[2 * nchunks][D] | split_list[nchunks] | long_list[nchunks] (64-bit) |
//   counters
// The sort ends in keysA/valsA, which the caller may read after the call.
#include <mutex>

#include "common.cuh"

namespace dlrm {
namespace {

constexpr uint32_t kSkipKey = 0xFFFFFFFFu;
constexpr int kSortThreads = 256;
constexpr int kItems = 4;                      // keys per thread (1,024-key tiles measured best: 2 to 16 tried)
constexpr int kTile = kSortThreads * kItems;   // 1024 keys per tile
constexpr int kChunk = 32;                     // positions per segment chunk
constexpr int kFixThreads = 512;

struct Ws {
    uint32_t *keys[2], *vals[2];
    uint32_t* hist;
    uint32_t* totals;
    float* partials;
    uint64_t* split_list;    // runs crossing a chunk edge: first chunk << 32 | pieces, up to kLongPieces pieces
    uint32_t* split_count;   // [0] entries of split_list, [1] entries of long_list
    uint64_t* long_list;     // the same for runs of more pieces
    size_t bytes;
};

Ws carve(void* base, int64_t nnz, int D)
{
    Ws w;
    const int64_t ntiles = (nnz + kTile - 1) / kTile;
    const int64_t nchunks = (nnz + kChunk - 1) / kChunk;
    uint8_t* p = static_cast<uint8_t*>(base);
    size_t off = 0;
    auto take = [&](size_t bytes) {
        uint8_t* q = p ? p + off : nullptr;
        off += dlrm_ws_align(bytes);
        return q;
    };
    w.keys[0] = (uint32_t*)take(4 * (size_t)nnz);
    w.vals[0] = (uint32_t*)take(4 * (size_t)nnz);
    w.keys[1] = (uint32_t*)take(4 * (size_t)nnz);
    w.vals[1] = (uint32_t*)take(4 * (size_t)nnz);
    w.hist = (uint32_t*)take(4 * 256 * (size_t)ntiles);
    w.totals = (uint32_t*)take(4 * 256);
    w.partials = (float*)take(4 * 2 * (size_t)nchunks * D);
    w.split_list = (uint64_t*)take(8 * (size_t)nchunks);
    w.long_list = (uint64_t*)take(8 * (size_t)nchunks);
    w.split_count = (uint32_t*)take(8);
    w.bytes = off;
    return w;
}

// ------------------------------------------------------------------ 1. keys
template <int G>
__global__ void __launch_bounds__(256)
keys_kernel(const int64_t* __restrict__ row_base, int F, int B, const int32_t* __restrict__ indices,
            const int32_t* __restrict__ offsets, bool hash, uint32_t* status, uint32_t* __restrict__ keys,
            uint32_t* __restrict__ vals, int64_t nbags, int64_t nnz, uint32_t* __restrict__ split_count)
{
    pdl_wait_and_release();
    if (blockIdx.x == 0 && threadIdx.x < 2) split_count[threadIdx.x] = 0;   // counters of the segment pass
    const int lane = threadIdx.x % G;
    const int64_t group = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) / G;
    const int64_t ngroups = (int64_t)gridDim.x * blockDim.x / G;
    for (int64_t g = group; g < nbags; g += ngroups) {   // g = t*B + b (feature-major, like offsets)
        const int t = (int)((uint32_t)g / (uint32_t)B);   // F * B < 2^31
        const int b = (int)g - t * B;
        const int64_t base = row_base[t], n = row_base[t + 1] - base;
        const uint32_t val = (uint32_t)((int64_t)b * F + t);
        int64_t s = offsets[g], e = offsets[g + 1];
        if (s < 0 || e < s || e > nnz) {   // malformed CSR: clamp, flag, stay in bounds
            set_status(status, DLRM_STATUS_BAD_OFFSETS);
            s = s < 0 ? 0 : (s > nnz ? nnz : s);
            e = e < s ? s : (e > nnz ? nnz : e);
        }
        for (int64_t p = s + lane; p < e; p += G) {
            int64_t i = indices[p];
            uint32_t key = kSkipKey;
            if (hash) {
                if (n > 0) {
                    i %= n;
                    if (i < 0) i += n;
                    key = (uint32_t)(base + i);
                } else {
                    set_status(status, DLRM_STATUS_OOB_INDEX);
                }
            } else if (i >= 0 && i < n) {
                key = (uint32_t)(base + i);
            } else {
                set_status(status, DLRM_STATUS_OOB_INDEX);
            }
            keys[p] = key;
            vals[p] = val;
        }
    }
}

// ------------------------------------------------------- block scan helper
// Exclusive scan of one value per thread over a block of kSortThreads threads.
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, uint32_t* warp_sums, uint32_t* total)
{
    const int lane = threadIdx.x % kWarp, warp = threadIdx.x / kWarp;
    uint32_t x = v;
#pragma unroll
    for (int o = 1; o < kWarp; o <<= 1) {
        uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == kWarp - 1) warp_sums[warp] = x;
    __syncthreads();
    if (warp == 0) {
        uint32_t w = lane < kSortThreads / kWarp ? warp_sums[lane] : 0;
#pragma unroll
        for (int o = 1; o < kWarp; o <<= 1) {
            uint32_t y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        if (lane < kSortThreads / kWarp) warp_sums[lane] = w;   // inclusive
    }
    __syncthreads();
    const uint32_t before = warp > 0 ? warp_sums[warp - 1] : 0;
    if (total) *total = warp_sums[kSortThreads / kWarp - 1];
    __syncthreads();
    return before + x - v;
}

// ------------------------------------------------------------ 2. radix sort
__global__ void __launch_bounds__(kSortThreads)
radix_upsweep(const uint32_t* __restrict__ keys, int64_t n, int shift, uint32_t mask, uint32_t* __restrict__ hist,
              int64_t ntiles)
{
    pdl_wait_and_release();
    __shared__ uint32_t h[256];
    h[threadIdx.x] = 0;
    __syncthreads();
    const int64_t base = (int64_t)blockIdx.x * kTile;
    const uint32_t lt = (1u << (threadIdx.x % kWarp)) - 1u;
    uint32_t d[kItems];
#pragma unroll
    for (int r = 0; r < kItems; ++r) {
        const int64_t p = base + r * kSortThreads + threadIdx.x;
        d[r] = p < n ? (keys[p] >> shift) & mask : 0x100u;
    }
    // Zipf-skewed keys repeat digits: one shared atomic per distinct digit per warp
#pragma unroll
    for (int r = 0; r < kItems; ++r) {
        const uint32_t peers = __match_any_sync(0xffffffffu, d[r]);
        if (d[r] < 0x100u && (peers & lt) == 0) atomicAdd(&h[d[r]], (uint32_t)__popc(peers));
    }
    __syncthreads();
    hist[(int64_t)threadIdx.x * ntiles + blockIdx.x] = h[threadIdx.x];
}

// One block per digit: exclusive scan of hist[d][0..ntiles) in place, total to totals[d].
__global__ void __launch_bounds__(kSortThreads)
radix_scan(uint32_t* __restrict__ hist, int64_t ntiles, uint32_t* __restrict__ totals)
{
    pdl_wait_and_release();
    __shared__ uint32_t warp_sums[kSortThreads / kWarp];
    __shared__ uint32_t chunk_total;
    uint32_t* row = hist + (int64_t)blockIdx.x * ntiles;
    uint32_t carry = 0;
    for (int64_t c0 = 0; c0 < ntiles; c0 += kTile) {
        uint32_t v[kItems];
        uint32_t s = 0;
#pragma unroll
        for (int r = 0; r < kItems; ++r) {
            const int64_t i = c0 + (int64_t)threadIdx.x * kItems + r;
            v[r] = i < ntiles ? row[i] : 0;
            s += v[r];
        }
        uint32_t ex = block_excl_scan(s, warp_sums, &chunk_total);
#pragma unroll
        for (int r = 0; r < kItems; ++r) {
            const int64_t i = c0 + (int64_t)threadIdx.x * kItems + r;
            if (i < ntiles) row[i] = carry + ex;
            ex += v[r];
        }
        carry += chunk_total;
    }
    if (threadIdx.x == 0) totals[blockIdx.x] = carry;
}

__global__ void __launch_bounds__(kSortThreads)
radix_downsweep(const uint32_t* __restrict__ keys_in, const uint32_t* __restrict__ vals_in,
                uint32_t* __restrict__ keys_out, uint32_t* __restrict__ vals_out, int64_t n, int shift,
                uint32_t mask, const uint32_t* __restrict__ hist, const uint32_t* __restrict__ totals,
                int64_t ntiles)
{
    pdl_wait_and_release();
    constexpr int kW = kSortThreads / kWarp;
    __shared__ uint32_t wcnt[kW][256];
    __shared__ uint32_t dbase[256];
    __shared__ uint32_t warp_sums[kW];
    const int lane = threadIdx.x % kWarp, warp = threadIdx.x / kWarp;
    const uint32_t lt = (1u << lane) - 1u;

    // global start of each digit in this tile
    const uint32_t ex = block_excl_scan(totals[threadIdx.x], warp_sums, nullptr);
    dbase[threadIdx.x] = ex + hist[(int64_t)threadIdx.x * ntiles + blockIdx.x];
#pragma unroll
    for (int w = 0; w < kW; ++w) wcnt[w][threadIdx.x] = 0;
    __syncthreads();

    uint32_t key[kItems], val[kItems], local[kItems];
    const int64_t wbase = (int64_t)blockIdx.x * kTile + (int64_t)warp * kWarp * kItems;
#pragma unroll
    for (int r = 0; r < kItems; ++r) {
        const int64_t p = wbase + r * kWarp + lane;
        const bool valid = p < n;
        key[r] = valid ? keys_in[p] : 0;
        val[r] = valid ? vals_in[p] : 0;
        const uint32_t d = (key[r] >> shift) & mask;
        const uint32_t peers = __match_any_sync(0xffffffffu, valid ? d : 0x100u);
        const uint32_t prior = valid ? wcnt[warp][d] : 0;
        __syncwarp();
        if (valid && (peers & lt) == 0) wcnt[warp][d] = prior + __popc(peers);
        __syncwarp();
        local[r] = prior + __popc(peers & lt);
    }
    __syncthreads();
    {   // exclusive scan over warps, per digit
        uint32_t s = 0;
#pragma unroll
        for (int w = 0; w < kW; ++w) {
            const uint32_t c = wcnt[w][threadIdx.x];
            wcnt[w][threadIdx.x] = s;
            s += c;
        }
    }
    __syncthreads();
#pragma unroll
    for (int r = 0; r < kItems; ++r) {
        const int64_t p = wbase + r * kWarp + lane;
        if (p < n) {
            const uint32_t d = (key[r] >> shift) & mask;
            const uint32_t pos = dbase[d] + wcnt[warp][d] + local[r];
            if (pos < n) {   // always true for consistent histograms; guards the write
                keys_out[pos] = key[r];
                vals_out[pos] = val[r];
            }
        }
    }
}

// ----------------------------------------------------------------- 4. fixup
constexpr int kLongPieces = 64;   // runs with more chunk pieces are summed by a whole block
constexpr int kFixRegs = 4;       // float4 partial-sum loads a lane has in flight

// Last chunk touched by the run of key K that starts in chunk c0 and continues
// past it.  Keys are sorted, so the run touches chunk c iff the first key of c
// is K, and the chunks it touches are c0..L.  Chunk c0 + 2 is probed first
// (one broadcast load); past it, one round probes c0 + 2^j for j = 0..31 (so
// 2^j <= L - c0 < 2^(j+1) for the last true j), then each round probes 32
// evenly spaced chunks of the remaining interval.
__device__ __forceinline__ int64_t run_last_chunk(const uint32_t* __restrict__ keys, int64_t n, int64_t nchunks,
                                                  int64_t c0, uint32_t K, int lane)
{
    auto touches = [&](int64_t c) { return c < nchunks && c * kChunk < n && keys[c * kChunk] == K; };
    if (!touches(c0 + 2)) return c0 + 1;      // most runs that cross an edge end in the next chunk
    const uint32_t m = __ballot_sync(0xffffffffu, touches(c0 + ((int64_t)1 << lane)));
    const int j = __popc(m) - 1;              // chunk c0 + 1 is touched, so j >= 0
    int64_t lo = c0 + ((int64_t)1 << j);      // touched
    int64_t hi = c0 + ((int64_t)2 << j);      // not touched (or past the end)
    while (hi - lo > 1) {
        const int64_t step = (hi - lo + kWarp - 1) / kWarp;
        const int64_t c = lo + step * (lane + 1);
        const uint32_t t = __ballot_sync(0xffffffffu, c < hi && touches(c));
        const int k = __popc(t);              // probes lo + step, ..., lo + k*step are touched
        const int64_t nlo = lo + step * k;
        hi = nlo + step < hi ? nlo + step : hi;
        lo = nlo;
    }
    return lo;
}

// --------------------------------------------------------- 3. segment sums
// A gradient chunk of four elements as loaded: fp32 as one float4, fp16 as
// the 8 loaded bytes (half the registers, so twice the loads fit in flight),
// widened exactly to fp32 where it is added.
template <typename GT>
struct GradRaw { using T = float4; };
template <>
struct GradRaw<__half> { using T = uint2; };

template <typename GT>
__device__ __forceinline__ typename GradRaw<GT>::T load_grad_raw(const GT* p)
{
    if constexpr (sizeof(GT) == 4) {
        return u4_as_f4(ldg_nc_v4(p));
    } else {
        uint2 r;
        asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(r.x), "=r"(r.y) : "l"(p));
        return r;
    }
}

__device__ __forceinline__ float4 widen(float4 v) { return v; }
__device__ __forceinline__ float4 widen(uint2 r)
{
    const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&r.x));
    const float2 c = __half22float2(*reinterpret_cast<const __half2*>(&r.y));
    return make_float4(a.x, a.y, c.x, c.y);
}

template <int MC, typename GT>
__global__ void __launch_bounds__(256, MC >= 8 ? 2 : 3)   // rows past 512 elements: registers for 8 float4 sums
segment_kernel(const uint32_t* __restrict__ keys, const uint32_t* __restrict__ vals, int64_t n,
               const GT* __restrict__ grad, int D, float* __restrict__ tables, int64_t total_rows, float lr,
               float* __restrict__ partials, uint64_t* __restrict__ split_list, uint32_t* split_count,
               uint64_t* __restrict__ long_list, int64_t nchunks, int64_t nbags)
{
    pdl_wait_and_release();
    // positions per batch: their gradient rows, and the table rows of the runs
    // that end (complete) among them, are all loaded before any is used (at
    // three blocks per SM and the 64K training shapes, 6 measured best for fp32
    // gradients; 8 for fp16, 243 against 281 us at 6)
    constexpr int U0 = sizeof(GT) == 2 && MC <= 2 ? 8 : 6;
    constexpr int U = MC >= 8 ? 1 : (U0 / MC > 0 ? U0 / MC : 1);
    const int lane = threadIdx.x % kWarp;
    const int64_t warp_id = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) / kWarp;
    const int64_t nwarps = (int64_t)gridDim.x * blockDim.x / kWarp;
    const int c4 = D / 4;   // float4 columns per row
    for (int64_t c = warp_id; c < nchunks; c += nwarps) {
        const int64_t p0 = c * kChunk;
        const int64_t p = p0 + lane;
        const uint32_t key = p < n ? keys[p] : kSkipKey;
        const uint32_t val = p < n ? vals[p] : 0;
        uint32_t prev = __shfl_up_sync(0xffffffffu, key, 1);
        if (lane == 0) prev = p0 > 0 ? keys[p0 - 1] : ~key;
        const uint32_t after = (p0 + kChunk < n) ? keys[p0 + kChunk] : kSkipKey;
        uint32_t next = __shfl_down_sync(0xffffffffu, key, 1);
        if (lane == kWarp - 1) next = after;
        const bool valid = key != kSkipKey;
        const uint32_t heads = __ballot_sync(0xffffffffu, valid && prev != key);
        const uint32_t vmask = __ballot_sync(0xffffffffu, valid);
        if (vmask == 0) continue;
        const int nvalid = 32 - __clz(vmask);             // valid lanes are a prefix
        const uint32_t starts = heads | 1u;               // lane 0 starts a run piece
        // pieces: a piece ends where the next position holds another key or
        // the chunk's valid prefix ends.  A piece that began with a head (its
        // run starts in this chunk) and whose run does not continue past the
        // chunk is a whole run: its row is updated here.
        const bool piece_end = valid && (next != key || lane == nvalid - 1);
        const int s_me = 31 - __clz(starts & (0xffffffffu >> (31 - lane)));
        const bool starts_here = (heads >> s_me) & 1u;
        const bool run_ends = lane < kWarp - 1 || after != key;
        const uint32_t ends = __ballot_sync(0xffffffffu, piece_end);
        const uint32_t whole = __ballot_sync(0xffffffffu, piece_end && starts_here && run_ends);
        const uint32_t complete = __ballot_sync(0xffffffffu, piece_end && starts_here && run_ends &&
                                                             (int64_t)key < total_rows);
        float4 acc[MC];
#pragma unroll
        for (int m = 0; m < MC; ++m) acc[m] = make_float4(0.f, 0.f, 0.f, 0.f);
        uint32_t file_key = kSkipKey;   // key of a run that starts here and crosses the chunk's end
        for (int q0 = 0; q0 < nvalid; q0 += U) {
            typename GradRaw<GT>::T v[U][MC];
            float4 w[U][MC];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int q = q0 + u;
                const uint32_t row = __shfl_sync(0xffffffffu, val, q & 31);
                const uint32_t qk = __shfl_sync(0xffffffffu, key, q & 31);
                const bool done = q < nvalid && ((complete >> (q & 31)) & 1u);
#pragma unroll
                for (int m = 0; m < MC; ++m) {
                    const int col = lane + m * kWarp;
                    v[u][m] = typename GradRaw<GT>::T{};
                    w[u][m] = make_float4(0.f, 0.f, 0.f, 0.f);
                    // row < nbags holds for pairs made from well-formed offsets
                    if (q < nvalid && col < c4 && (int64_t)row < nbags)
                        v[u][m] = load_grad_raw<GT>(grad + (int64_t)row * D + 4 * col);
                    if (done && col < c4) w[u][m] = *reinterpret_cast<const float4*>(tables + (int64_t)qk * D + 4 * col);
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int q = q0 + u;
                if (q >= nvalid) break;
#pragma unroll
                for (int m = 0; m < MC; ++m) {
                    const float4 g = widen(v[u][m]);
                    acc[m].x += g.x;
                    acc[m].y += g.y;
                    acc[m].z += g.z;
                    acc[m].w += g.w;
                }
                if (!((ends >> q) & 1u)) continue;
                const uint32_t qk = __shfl_sync(0xffffffffu, key, q);
                if ((complete >> q) & 1u) {
#pragma unroll
                    for (int m = 0; m < MC; ++m) {
                        const int col = lane + m * kWarp;
                        if (col < c4) {
                            float4 x = w[u][m];
                            x.x = fmaf(-lr, acc[m].x, x.x);
                            x.y = fmaf(-lr, acc[m].y, x.y);
                            x.z = fmaf(-lr, acc[m].z, x.z);
                            x.w = fmaf(-lr, acc[m].w, x.w);
                            *reinterpret_cast<float4*>(tables + (int64_t)qk * D + 4 * col) = x;
                        }
                    }
                } else if (!((whole >> q) & 1u)) {
                    // a piece of a run that crosses a chunk edge: its partial sum
                    // (a whole run whose key is out of range cannot be made above)
                    const bool piece_starts_here = __shfl_sync(0xffffffffu, starts_here, q);
                    const int64_t slot = 2 * c + (piece_starts_here ? 1 : 0);
#pragma unroll
                    for (int m = 0; m < MC; ++m) {
                        const int col = lane + m * kWarp;
                        if (col < c4) reinterpret_cast<float4*>(partials + slot * D)[col] = acc[m];
                    }
                    if (piece_starts_here) file_key = qk;   // filed after the chunk (at most one per chunk)
                }
#pragma unroll
                for (int m = 0; m < MC; ++m) acc[m] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
        if (file_key != kSkipKey) {   // this chunk files the run it starts, with its number of pieces
            const int64_t pieces = run_last_chunk(keys, n, nchunks, c, file_key, lane) - c + 1;
            if (lane == 0) {
                const uint64_t e = (uint64_t)c << 32 | (uint64_t)pieces;
                if (pieces > kLongPieces)
                    long_list[atomicAdd(split_count + 1, 1u)] = e;
                else
                    split_list[atomicAdd(split_count, 1u)] = e;
            }
        }
    }
}

template <int MC>
__device__ __forceinline__ void apply_sgd(float* __restrict__ tables, int64_t row, int D, float lr, int lane,
                                          const float4 (&g)[MC])
{
#pragma unroll
    for (int m = 0; m < MC; ++m) {
        const int col = lane + m * kWarp;
        if (col < D / 4) {
            float4* wp = reinterpret_cast<float4*>(tables + row * D + 4 * col);
            float4 x = *wp;
            x.x = fmaf(-lr, g[m].x, x.x);
            x.y = fmaf(-lr, g[m].y, x.y);
            x.z = fmaf(-lr, g[m].z, x.z);
            x.w = fmaf(-lr, g[m].w, x.w);
            *wp = x;
        }
    }
}

// Slot of piece j of the run that starts in chunk c0 (the first piece is the
// starting chunk's "continues" slot, the others are chunk-start slots).
__device__ __forceinline__ int64_t piece_slot(int64_t c0, int64_t j) { return j == 0 ? 2 * c0 + 1 : 2 * (c0 + j); }

// Pieces [j0, j1) of the run starting in chunk c0, added in order into acc.
template <int MC>
__device__ __forceinline__ void add_pieces(const float* __restrict__ partials, int64_t c0, int64_t j0, int64_t j1,
                                           int D, int lane, float4 (&acc)[MC])
{
    const int c4 = D / 4;
    constexpr int kFixBatch = kFixRegs / MC > 0 ? kFixRegs / MC : 1;   // pieces in flight
    for (int64_t j = j0; j < j1; j += kFixBatch) {
        float4 v[kFixBatch][MC];
#pragma unroll
        for (int u = 0; u < kFixBatch; ++u) {
            const int64_t slot = piece_slot(c0, j + u);
#pragma unroll
            for (int m = 0; m < MC; ++m) {
                const int col = lane + m * kWarp;
                v[u][m] = (j + u < j1 && col < c4) ? reinterpret_cast<const float4*>(partials + slot * D)[col]
                                                   : make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
#pragma unroll
        for (int u = 0; u < kFixBatch; ++u)
            if (j + u < j1)
#pragma unroll
                for (int m = 0; m < MC; ++m) {
                    acc[m].x += v[u][m].x;
                    acc[m].y += v[u][m].y;
                    acc[m].z += v[u][m].z;
                    acc[m].w += v[u][m].w;
                }
    }
}

// Runs that cross chunk edges.  Block i < (long runs) takes long run i: warp w
// adds the w-th of kW contiguous slices of its pieces, then warp 0 adds the
// kW slice sums in slice order and updates the row.  Then every warp takes
// short runs (pieces in order, one warp per run).
template <int MC>
__global__ void __launch_bounds__(kFixThreads)
fixup_kernel(const uint32_t* __restrict__ keys, const float* __restrict__ partials,
             const uint64_t* __restrict__ split_list, const uint64_t* __restrict__ long_list,
             const uint32_t* __restrict__ counts, int D, float* __restrict__ tables, int64_t total_rows, float lr)
{
    pdl_wait_and_release();
    constexpr int kW = kFixThreads / kWarp;
    extern __shared__ __align__(16) float red[];   // [kW][D]
    const int lane = threadIdx.x % kWarp, warp = threadIdx.x / kWarp;
    const int c4 = D / 4;
    const uint32_t nshort = counts[0], nlong = counts[1];
    for (uint32_t i = blockIdx.x; i < nlong; i += gridDim.x) {
        const uint64_t e = long_list[i];
        const int64_t c0 = (int64_t)(e >> 32), pieces = (int64_t)(e & 0xffffffffu);
        const uint32_t K = keys[c0 * kChunk + kChunk - 1];
        float4 acc[MC];
#pragma unroll
        for (int m = 0; m < MC; ++m) acc[m] = make_float4(0.f, 0.f, 0.f, 0.f);
        add_pieces<MC>(partials, c0, pieces * warp / kW, pieces * (warp + 1) / kW, D, lane, acc);
#pragma unroll
        for (int m = 0; m < MC; ++m) {
            const int col = lane + m * kWarp;
            if (col < c4) reinterpret_cast<float4*>(red + warp * D)[col] = acc[m];
        }
        __syncthreads();
        if (warp == 0) {
            float4 g[MC];
#pragma unroll
            for (int m = 0; m < MC; ++m) {
                const int col = lane + m * kWarp;
                g[m] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (col < c4) {
                    g[m] = reinterpret_cast<const float4*>(red)[col];
                    for (int w = 1; w < kW; ++w) {
                        const float4 v = reinterpret_cast<const float4*>(red + w * D)[col];
                        g[m].x += v.x;
                        g[m].y += v.y;
                        g[m].z += v.z;
                        g[m].w += v.w;
                    }
                }
            }
            if ((int64_t)K < total_rows) apply_sgd<MC>(tables, K, D, lr, lane, g);
        }
        __syncthreads();
    }
    const int64_t gw = (int64_t)blockIdx.x * kW + warp, nw = (int64_t)gridDim.x * kW;
    for (int64_t i = gw; i < nshort; i += nw) {
        const uint64_t e = split_list[i];
        const int64_t c0 = (int64_t)(e >> 32), pieces = (int64_t)(e & 0xffffffffu);
        const uint32_t K = keys[c0 * kChunk + kChunk - 1];
        float4 acc[MC];
#pragma unroll
        for (int m = 0; m < MC; ++m) acc[m] = make_float4(0.f, 0.f, 0.f, 0.f);
        add_pieces<MC>(partials, c0, 0, pieces, D, lane, acc);
        if ((int64_t)K < total_rows) apply_sgd<MC>(tables, K, D, lr, lane, acc);
    }
}

int key_bits(int64_t total_rows)
{
    int b = 0;
    while (b < 32 && ((uint64_t)1 << b) <= (uint64_t)total_rows) ++b;   // 2^b > total_rows
    return b;
}

template <int MC, typename GT>
dlrm_status launch_segments(const Ws& w, int64_t nnz, const GT* grad, int D, float* tables,
                            int64_t total_rows, float lr, int64_t nbags, cudaStream_t st)
{
    const int64_t nchunks = (nnz + kChunk - 1) / kChunk;
    int64_t blocks = (nchunks * kWarp + 255) / 256;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, segment_kernel<MC, GT>, 256, 0) != cudaSuccess ||
        per_sm < 1)
        per_sm = 1;
    const int64_t resident = (int64_t)num_sms() * per_sm;   // one wave of the grid-stride loop
    if (blocks > resident) blocks = resident;
    dlrm_status s = check_launch_pdl(launch_pdl(segment_kernel<MC, GT>, (int)blocks, 256, 0, st,
                                                (const uint32_t*)w.keys[0], (const uint32_t*)w.vals[0], nnz, grad, D,
                                                tables, total_rows, lr, w.partials, w.split_list, w.split_count,
                                                w.long_list, nchunks, nbags),
                                     "segment_kernel");
    if (s != DLRM_OK) return s;
    const size_t smem = (size_t)(kFixThreads / kWarp) * D * sizeof(float);
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(fixup_kernel<MC>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return fail(DLRM_ERR_CUDA, "dlrm_emb_bwd_sgd: %s", cudaGetErrorString(e));
    }
    int64_t fblocks = (int64_t)num_sms() * 4;
    const int64_t fneed = (nchunks * kWarp + kFixThreads - 1) / kFixThreads;   // one warp per chunk at most
    if (fblocks > fneed) fblocks = fneed;
    return check_launch_pdl(launch_pdl(fixup_kernel<MC>, (int)fblocks, kFixThreads, smem, st, (const uint32_t*)w.keys[0],
                                       (const float*)w.partials, (const uint64_t*)w.split_list,
                                       (const uint64_t*)w.long_list, (const uint32_t*)w.split_count, D, tables,
                                       total_rows, lr),
                            "fixup_kernel");
}

}  // namespace
}  // namespace dlrm

using namespace dlrm;

extern "C" size_t dlrm_emb_bwd_sgd_workspace_size(int64_t nnz, int D, int64_t total_rows)
{
    if (nnz < 0 || nnz > DLRM_MAX_NNZ || D < 1 || D % 4 != 0 || D > 1024 || total_rows < 1 ||
        total_rows >= 0xFFFFFFFFll)
        return 0;
    return carve(nullptr, nnz, D).bytes;
}

extern "C" dlrm_status dlrm_emb_bwd_sgd(float* d_tables, const int64_t* d_row_base, int64_t total_rows, int F,
                                        int D, int B, const int32_t* d_indices, const int32_t* d_offsets,
                                        int64_t nnz, const void* d_grad_pooled, float lr, void* d_workspace,
                                        size_t workspace_bytes, unsigned flags, uint32_t* d_status, void* stream)
{
    clear_error();
    if (F < 1 || D < 1 || B < 0)
        return fail(DLRM_ERR_INVALID_ARG, "dlrm_emb_bwd_sgd: need F >= 1, D >= 1, B >= 0");
    if (nnz < 0 || nnz > DLRM_MAX_NNZ)
        return fail(DLRM_ERR_INVALID_ARG, "dlrm_emb_bwd_sgd: nnz must be in [0, DLRM_MAX_NNZ]");
    if ((int64_t)F * B >= ((int64_t)1 << 31))
        return fail(DLRM_ERR_INVALID_ARG, "dlrm_emb_bwd_sgd: F*B must be below 2^31");
    if (total_rows < 1 || total_rows >= 0xFFFFFFFFll)
        return fail(DLRM_ERR_INVALID_ARG, "dlrm_emb_bwd_sgd: total_rows must be in [1, 2^32 - 1)");
    if (!d_tables || !d_row_base || !d_offsets || !d_grad_pooled || (nnz > 0 && (!d_indices || !d_workspace)))
        return fail(DLRM_ERR_INVALID_ARG, "dlrm_emb_bwd_sgd: null device pointer");
    if (flags & ~(DLRM_FLAG_HASH_INDICES | DLRM_FLAG_GRAD_F16))
        return fail(DLRM_ERR_INVALID_ARG, "dlrm_emb_bwd_sgd: unknown flag bits 0x%x", flags);
    if (D % 4 != 0 || D > 1024)
        return fail(DLRM_ERR_UNSUPPORTED, "dlrm_emb_bwd_sgd: D must be a multiple of 4, at most 1024");
    if (!aligned16(d_tables) || !aligned16(d_grad_pooled))
        return fail(DLRM_ERR_UNSUPPORTED, "dlrm_emb_bwd_sgd: tables and grad_pooled must be 16-byte aligned");
    if (nnz > 0 && (reinterpret_cast<uintptr_t>(d_workspace) & 255u))
        return fail(DLRM_ERR_UNSUPPORTED, "dlrm_emb_bwd_sgd: workspace must be 256-byte aligned");
    const size_t need = dlrm_emb_bwd_sgd_workspace_size(nnz, D, total_rows);
    if (nnz > 0 && workspace_bytes < need)
        return fail(DLRM_ERR_WORKSPACE, "dlrm_emb_bwd_sgd: workspace %zu bytes < %zu needed", workspace_bytes, need);
    if (nnz == 0 || B == 0) return DLRM_OK;

    cudaStream_t st = as_stream(stream);
    Ws w = carve(d_workspace, nnz, D);
    const int nbits = key_bits(total_rows);
    const int npasses = (nbits + 7) / 8;
    int cur = npasses & 1;   // the last pass lands in buffer 0

    const int64_t nbags = (int64_t)F * B;
    const bool multi = nnz > 2 * nbags;
    const bool hash = (flags & DLRM_FLAG_HASH_INDICES) != 0;
    {
        const int G = multi ? 32 : 1;
        int64_t blocks = (nbags * G + 255) / 256;
        const int64_t cap = (int64_t)num_sms() * 8;
        if (blocks > cap) blocks = cap;
        const cudaError_t e =
            multi ? launch_pdl(keys_kernel<32>, (int)blocks, 256, 0, st, d_row_base, F, B, d_indices, d_offsets, hash,
                               d_status, w.keys[cur], w.vals[cur], nbags, nnz, w.split_count)
                  : launch_pdl(keys_kernel<1>, (int)blocks, 256, 0, st, d_row_base, F, B, d_indices, d_offsets, hash,
                               d_status, w.keys[cur], w.vals[cur], nbags, nnz, w.split_count);
        dlrm_status s = check_launch_pdl(e, "keys_kernel");
        if (s != DLRM_OK) return s;
    }
    const int64_t ntiles = (nnz + kTile - 1) / kTile;
    for (int pass = 0; pass < npasses; ++pass) {
        const int shift = 8 * pass;
        const int bits = nbits - shift < 8 ? nbits - shift : 8;
        const uint32_t mask = (1u << bits) - 1u;
        cudaError_t e = launch_pdl(radix_upsweep, (int)ntiles, kSortThreads, 0, st, (const uint32_t*)w.keys[cur], nnz,
                                   shift, mask, w.hist, ntiles);
        if (e == cudaSuccess) e = launch_pdl(radix_scan, 256, kSortThreads, 0, st, w.hist, ntiles, w.totals);
        if (e == cudaSuccess)
            e = launch_pdl(radix_downsweep, (int)ntiles, kSortThreads, 0, st, (const uint32_t*)w.keys[cur],
                           (const uint32_t*)w.vals[cur], w.keys[cur ^ 1], w.vals[cur ^ 1], nnz, shift, mask,
                           (const uint32_t*)w.hist, (const uint32_t*)w.totals, ntiles);
        dlrm_status s = check_launch_pdl(e, "radix sort pass");
        if (s != DLRM_OK) return s;
        cur ^= 1;
    }
    if (flags & DLRM_FLAG_GRAD_F16) {
        const __half* grad = static_cast<const __half*>(d_grad_pooled);
        if (D <= 128) return launch_segments<1>(w, nnz, grad, D, d_tables, total_rows, lr, nbags, st);
        if (D <= 256) return launch_segments<2>(w, nnz, grad, D, d_tables, total_rows, lr, nbags, st);
        if (D <= 512) return launch_segments<4>(w, nnz, grad, D, d_tables, total_rows, lr, nbags, st);
        return launch_segments<8>(w, nnz, grad, D, d_tables, total_rows, lr, nbags, st);
    }
    const float* grad = static_cast<const float*>(d_grad_pooled);
    if (D <= 128) return launch_segments<1>(w, nnz, grad, D, d_tables, total_rows, lr, nbags, st);
    if (D <= 256) return launch_segments<2>(w, nnz, grad, D, d_tables, total_rows, lr, nbags, st);
    if (D <= 512) return launch_segments<4>(w, nnz, grad, D, d_tables, total_rows, lr, nbags, st);
    return launch_segments<8>(w, nnz, grad, D, d_tables, total_rows, lr, nbags, st);
}

// --------------------------------------------------------------------------
// Variant of dlrm_emb_bwd_sgd for callers that cannot allocate device memory
// (for example a plugin invoked from a host framework's execute callback,
// where the framework owns all device memory and forbids allocation while it
// runs).  The scratch lives in this file-scope device array instead of a
// caller-provided workspace.  Every GPU that loads the library holds it until
// the process exits.
// --------------------------------------------------------------------------
namespace dlrm {
namespace {

constexpr size_t kStaticScratchBytes = DLRM_NOALLOC_SCRATCH_BYTES;

static __device__ __align__(256) unsigned char g_sgd_scratch[kStaticScratchBytes];

// Device address of g_sgd_scratch for the current device.  In host code the
// array's name is only a host-side stand-in, so the address is queried once
// per device (with that device current) and cached.
dlrm_status static_scratch(void** out)
{
    static std::mutex mu;
    static void* cache[64] = {nullptr};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(DLRM_ERR_CUDA, "dlrm_emb_bwd_sgd_noalloc: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= 64) return fail(DLRM_ERR_UNSUPPORTED, "dlrm_emb_bwd_sgd_noalloc: device %d", dev);
    std::lock_guard<std::mutex> lock(mu);
    if (!cache[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_sgd_scratch);
        if (e != cudaSuccess || !p)
            return fail(DLRM_ERR_CUDA, "dlrm_emb_bwd_sgd_noalloc: cudaGetSymbolAddress: %s", cudaGetErrorString(e));
        cache[dev] = p;
    }
    *out = cache[dev];
    return DLRM_OK;
}

}  // namespace
}  // namespace dlrm

extern "C" dlrm_status dlrm_emb_bwd_sgd_noalloc(float* d_tables, const int64_t* d_row_base, int64_t total_rows,
                                                int F, int D, int B, const int32_t* d_indices,
                                                const int32_t* d_offsets, int64_t nnz,
                                                const float* d_grad_pooled, float lr, unsigned flags,
                                                uint32_t* d_status, void* stream)
{
    clear_error();
    const size_t need = dlrm_emb_bwd_sgd_workspace_size(nnz, D, total_rows);
    if (need == 0 && nnz != 0)
        return fail(DLRM_ERR_INVALID_ARG, "dlrm_emb_bwd_sgd_noalloc: invalid nnz, D or total_rows");
    if (need > dlrm::kStaticScratchBytes)
        return fail(DLRM_ERR_UNSUPPORTED,
                    "dlrm_emb_bwd_sgd_noalloc: needs %zu bytes of scratch, the built-in array holds %zu "
                    "(use dlrm_emb_bwd_sgd with a caller workspace)",
                    need, dlrm::kStaticScratchBytes);
    void* scratch = nullptr;
    dlrm_status s = dlrm::static_scratch(&scratch);
    if (s != DLRM_OK) return s;
    return dlrm_emb_bwd_sgd(d_tables, d_row_base, total_rows, F, D, B, d_indices, d_offsets, nnz, d_grad_pooled, lr,
                            scratch, dlrm::kStaticScratchBytes, flags, d_status, stream);
}
