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
//     Up to 8,192 keys one block forms the keys and sorts them in shared
//     memory instead (the same stable sort in one launch).
//  3. segments: the sorted array is cut into items of kSubs sub-chunks of 32
//     positions.  A warp takes items from a counter and walks their
//     sub-chunks (each position's key and gradient row number in one lane;
//     the next sub-chunk's loaded meanwhile); the gradient rows of a batch of
//     positions, and the table rows of the runs that complete among them, are
//     loaded before any is added.  Each run of equal keys is summed in
//     ascending position order; a run that starts and ends inside the item
//     updates its row (w = fmaf(-lr, g, w)); a run crossing an item edge
//     leaves one partial sum per item it touches, and the item where it
//     starts finds the run's last item and files the run with its number of
//     pieces.
//  4. fixup: each filed run's pieces are added in item order (a block of 16
//     warps over 16 contiguous slices for runs of many pieces, a warp for the
//     others) and the row is updated.
// Every order of summation is fixed by the data, so results are bitwise
// reproducible.  Workspace layout (256-byte aligned pieces):
//   keysA | valsA | keysB | valsB | hist[256][ntiles] | totals[256] | counters |
//   partials[2 * nitems][D] | split_list[nitems] | long_list[nitems]
// The sort ends in keysA/valsA, which the caller may read after the call.
#include <cuda.h>

#include <mutex>

#include "common.cuh"

namespace dlrm {
namespace {

constexpr uint32_t kSkipKey = 0xFFFFFFFFu;
constexpr int kSortThreads = 256;
constexpr int kItems = 6;                      // keys per thread (1,536-key tiles measured best: 2 to 16 tried)
constexpr int kTile = kSortThreads * kItems;   // 1,536 keys per tile

// segment pass
constexpr int kSubs = 8;                 // sub-chunks per item
constexpr int kSubsSmall = 1;            // ... for batches of the one-block sort (more items in flight)
constexpr int kFixThreads = 512;
constexpr int kLongPieces = 8;           // runs of more pieces are summed by a whole block

// counters
constexpr int kCtrSplit = 0;   // entries of split_list
constexpr int kCtrLong = 1;    // entries of long_list
constexpr int kCtrItem = 2;    // next segment item
constexpr int kNumCounters = 4;

int key_bits(int64_t total_rows)
{
    int b = 0;
    while (b < 32 && ((uint64_t)1 << b) <= (uint64_t)total_rows) ++b;   // 2^b > total_rows
    return b;
}

constexpr int kSmallMaxKeys = 8192;   // batches up to this many keys take the one-block sort

// Sub-chunks of 32 positions per segment item: a warp walks an item as a
// chain of dependent loads, so few keys are cut into short items.
inline int item_subs(int64_t nnz) { return nnz <= kSmallMaxKeys ? kSubsSmall : kSubs; }

struct Ws {
    uint32_t *keys[2], *vals[2];
    uint32_t* hist;
    uint32_t* totals;
    uint32_t* counters;
    float* partials;
    uint64_t* split_list;
    uint64_t* long_list;
    int64_t ntiles, nitems;
    size_t bytes;
};

Ws carve(void* base, int64_t nnz, int D)
{
    Ws w;
    w.ntiles = (nnz + kTile - 1) / kTile;
    const int64_t it = (int64_t)kWarp * item_subs(nnz);
    w.nitems = (nnz + it - 1) / it;
    // item buffers sized so that the workspace never shrinks as nnz grows:
    // short items stop at kSmallMaxKeys / 32 of them
    const int64_t it_big = (int64_t)kWarp * kSubs, short_max = kSmallMaxKeys / kWarp / kSubsSmall;
    const int64_t n_short = (nnz + kWarp * kSubsSmall - 1) / (kWarp * kSubsSmall);
    const int64_t n_big = (nnz + it_big - 1) / it_big;
    const int64_t nalloc = n_big > (n_short < short_max ? n_short : short_max) ? n_big
                                                                              : (n_short < short_max ? n_short : short_max);
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
    w.hist = (uint32_t*)take(4 * 256 * (size_t)w.ntiles);
    w.totals = (uint32_t*)take(4 * 256);
    w.counters = (uint32_t*)take(4 * kNumCounters);
    w.partials = (float*)take(4 * 2 * (size_t)nalloc * D);
    w.split_list = (uint64_t*)take(8 * (size_t)nalloc);
    w.long_list = (uint64_t*)take(8 * (size_t)nalloc);
    w.bytes = off;
    return w;
}

__device__ __forceinline__ uint32_t ldg_early_u32(const uint32_t* p)
{
    uint32_t r;
    asm volatile("ld.global.nc.u32 %0, [%1];" : "=r"(r) : "l"(p));
    return r;
}

// 16 bytes of a table row, loaded where written (the row is stored later by
// the same thread, so this is an ordinary coherent load, kept in order with
// the thread's other memory accesses).
__device__ __forceinline__ float4 ldg_row_early(const float* p)
{
    float4 r;
    asm volatile("ld.global.v4.f32 {%0,%1,%2,%3}, [%4];" : "=f"(r.x), "=f"(r.y), "=f"(r.z), "=f"(r.w) : "l"(p)
                 : "memory");
    return r;
}

// ------------------------------------------------------------------ 1. keys
// Block b owns bags [b * bpb, (b + 1) * bpb) (feature-major: bag g = t*B + b),
// writes the keys of their positions and counts the first radix digit
// (key & mask) of every key it writes: row b of the first pass's histogram.
// For well-formed offsets the block's positions are the contiguous range
// offsets[b * bpb] .. offsets[(b + 1) * bpb], the first pass's tile b.
// G = 1: a thread per bag, kKeyBags bags per thread in flight (bags of about
// one index); G = 32: a warp per bag.
constexpr int kKeyBags = 4;

template <int G>
__global__ void __launch_bounds__(kSortThreads)
keys_kernel(const int64_t* __restrict__ row_base, int F, int B, const int32_t* __restrict__ indices,
            const int32_t* __restrict__ offsets, bool hash, uint32_t* status, uint32_t* __restrict__ keys,
            uint32_t* __restrict__ vals, int64_t nbags, int64_t nnz, int64_t bpb, uint32_t mask,
            uint32_t* __restrict__ hist, int64_t ntiles, uint32_t* __restrict__ counters)
{
    __shared__ uint32_t h[256];
    h[threadIdx.x] = 0;
    pdl_wait();
    if (blockIdx.x == 0 && threadIdx.x < kNumCounters) counters[threadIdx.x] = 0;   // counters of the segment pass
    __syncthreads();
    const int lane = threadIdx.x % kWarp;
    const int64_t g0 = (int64_t)blockIdx.x * bpb;
    const int64_t g1 = g0 + bpb < nbags ? g0 + bpb : nbags;

    auto bounds = [&](int64_t& s, int64_t& e) {
        if (s < 0 || e < s || e > nnz) {   // malformed CSR: clamp, flag, stay in bounds
            set_status(status, DLRM_STATUS_BAD_OFFSETS);
            s = s < 0 ? 0 : (s > nnz ? nnz : s);
            e = e < s ? s : (e > nnz ? nnz : e);
        }
    };
    // one position of a bag of table (base, n): its key, stored with the bag's value and counted
    auto emit = [&](int64_t p, int32_t raw, int64_t base, int64_t n, uint32_t val) {
        int64_t i = raw;
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
        // Zipf-skewed keys repeat digits: one shared atomic per distinct digit per warp
        const uint32_t d = key & mask;
        const uint32_t peers = __match_any_sync(__activemask(), d);
        if ((peers & ((1u << lane) - 1u)) == 0) atomicAdd(&h[d], (uint32_t)__popc(peers));
    };

    if constexpr (G == 1) {
        for (int64_t gb = g0 + threadIdx.x; gb < g1; gb += (int64_t)kKeyBags * kSortThreads) {
            int64_t s[kKeyBags], e[kKeyBags];
            int32_t first[kKeyBags];
#pragma unroll
            for (int u = 0; u < kKeyBags; ++u) {
                const int64_t g = gb + (int64_t)u * kSortThreads;
                s[u] = e[u] = 0;
                if (g < g1) {
                    s[u] = ldg_early_s32(offsets + g);
                    e[u] = ldg_early_s32(offsets + g + 1);
                }
            }
#pragma unroll
            for (int u = 0; u < kKeyBags; ++u) {
                bounds(s[u], e[u]);
                first[u] = e[u] > s[u] ? ldg_early_s32(indices + s[u]) : 0;
            }
#pragma unroll
            for (int u = 0; u < kKeyBags; ++u) {
                const int64_t g = gb + (int64_t)u * kSortThreads;
                if (g < g1 && e[u] > s[u]) {
                    const int t = (int)((uint32_t)g / (uint32_t)B);   // F * B < 2^31
                    const int b = (int)g - t * B;
                    const int64_t base = row_base[t], n = row_base[t + 1] - base;
                    const uint32_t val = (uint32_t)((int64_t)b * F + t);
                    emit(s[u], first[u], base, n, val);
                    for (int64_t p = s[u] + 1; p < e[u]; ++p) emit(p, indices[p], base, n, val);
                }
            }
        }
    } else {
        for (int64_t g = g0 + threadIdx.x / kWarp; g < g1; g += kSortThreads / kWarp) {
            const int t = (int)((uint32_t)g / (uint32_t)B);
            const int b = (int)g - t * B;
            const int64_t base = row_base[t], n = row_base[t + 1] - base;
            const uint32_t val = (uint32_t)((int64_t)b * F + t);
            int64_t s = offsets[g], e = offsets[g + 1];
            bounds(s, e);
            for (int64_t p = s + lane; p < e; p += kWarp) emit(p, indices[p], base, n, val);
        }
    }
    __syncthreads();
    hist[(int64_t)threadIdx.x * ntiles + blockIdx.x] = h[threadIdx.x];
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
    pdl_wait();
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
    pdl_wait();
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

// One block per tile.  The first pass's tile b is the key kernel's block b:
// positions offsets[b * bpb] .. offsets[(b + 1) * bpb] (clamped), taken in
// sub-tiles of kTile keys, each digit's output offset advancing by the
// sub-tile's count; later passes' tiles are fixed ranges of kTile positions.
// kReorder (the first pass, whose input is in position order): each sub-tile
// is placed in shared memory by digit before it is written out, so that
// neighbouring threads write neighbouring places of a digit's output range
// (Zipf-hot keys spread over a warp otherwise make every write its own
// request); later passes read keys already grouped by their lower digits.
template <bool kReorder>
__global__ void __launch_bounds__(kSortThreads)
radix_downsweep(const uint32_t* __restrict__ keys_in, const uint32_t* __restrict__ vals_in,
                uint32_t* __restrict__ keys_out, uint32_t* __restrict__ vals_out, int64_t n, int shift,
                uint32_t mask, const uint32_t* __restrict__ hist, const uint32_t* __restrict__ totals,
                int64_t ntiles, const int32_t* __restrict__ offsets, int64_t bpb, int64_t nbags)
{
    pdl_wait();
    constexpr int kW = kSortThreads / kWarp;
    __shared__ uint32_t wcnt[kW][256];
    __shared__ uint32_t dbase[256];
    __shared__ uint32_t warp_sums[kW];
    __shared__ uint32_t tstart[kReorder ? 256 : 1];       // first place of each digit in the sub-tile
    __shared__ uint32_t skey[kReorder ? kTile : 1], sval[kReorder ? kTile : 1];
    const int lane = threadIdx.x % kWarp, warp = threadIdx.x / kWarp;
    const uint32_t lt = (1u << lane) - 1u;
    int64_t lo, hi;
    if (offsets) {
        const int64_t g0 = (int64_t)blockIdx.x * bpb;
        const int64_t g1 = g0 + bpb < nbags ? g0 + bpb : nbags;
        auto clampp = [&](int64_t x) { return x < 0 ? 0 : (x > n ? n : x); };
        lo = g0 < nbags ? clampp(offsets[g0]) : n;
        hi = g0 < nbags ? clampp(offsets[g1]) : n;
        if (hi < lo) hi = lo;
    } else {
        lo = (int64_t)blockIdx.x * kTile;
        hi = lo + kTile < n ? lo + kTile : n;
    }

    // global start of each digit in this tile
    const uint32_t ex = block_excl_scan(totals[threadIdx.x], warp_sums, nullptr);
    dbase[threadIdx.x] = ex + hist[(int64_t)threadIdx.x * ntiles + blockIdx.x];
    for (int64_t sub = lo; sub < hi; sub += kTile) {
#pragma unroll
        for (int w = 0; w < kW; ++w) wcnt[w][threadIdx.x] = 0;
        __syncthreads();

        uint32_t key[kItems], val[kItems], local[kItems];
        const int64_t wbase = sub + (int64_t)warp * kWarp * kItems;
#pragma unroll
        for (int r = 0; r < kItems; ++r) {
            const int64_t p = wbase + r * kWarp + lane;
            const bool valid = p < hi;
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
        uint32_t subtotal = 0;   // this sub-tile's count of digit threadIdx.x
#pragma unroll
        for (int w = 0; w < kW; ++w) {   // exclusive scan over warps, per digit
            const uint32_t c = wcnt[w][threadIdx.x];
            wcnt[w][threadIdx.x] = subtotal;
            subtotal += c;
        }
        if constexpr (kReorder) {
            // the sub-tile ordered by digit in shared memory first, then written out in that
            // order: consecutive threads write consecutive places of a digit's range
            tstart[threadIdx.x] = block_excl_scan(subtotal, warp_sums, nullptr);
            __syncthreads();
#pragma unroll
            for (int r = 0; r < kItems; ++r) {
                const int64_t p = wbase + r * kWarp + lane;
                if (p < hi) {
                    const uint32_t d = (key[r] >> shift) & mask;
                    const uint32_t lp = tstart[d] + wcnt[warp][d] + local[r];
                    if (lp < (uint32_t)kTile) {   // always true for consistent counts; guards the write
                        skey[lp] = key[r];
                        sval[lp] = val[r];
                    }
                }
            }
            __syncthreads();
            const int cnt = (int)(hi - sub < kTile ? hi - sub : kTile);
            for (int i = threadIdx.x; i < cnt; i += kSortThreads) {
                const uint32_t k2 = skey[i];
                const uint32_t d = (k2 >> shift) & mask;
                const uint32_t pos = dbase[d] + ((uint32_t)i - tstart[d]);
                if (pos < n) {
                    keys_out[pos] = k2;
                    vals_out[pos] = sval[i];
                }
            }
        } else {
            __syncthreads();
#pragma unroll
            for (int r = 0; r < kItems; ++r) {
                const int64_t p = wbase + r * kWarp + lane;
                if (p < hi) {
                    const uint32_t d = (key[r] >> shift) & mask;
                    const uint32_t pos = dbase[d] + wcnt[warp][d] + local[r];
                    if (pos < n) {   // always true for consistent histograms; guards the write
                        keys_out[pos] = key[r];
                        vals_out[pos] = val[r];
                    }
                }
            }
        }
        __syncthreads();
        dbase[threadIdx.x] += subtotal;
    }
}


// ------------------------------------------------ 2'. small batches: one block
// With few keys the chain of key, count, scan and scatter kernels is all
// launch and drain latency (about 50 us for a few hundred keys).  Up to
// kSmallMax keys one block of 32 warps does both steps in shared memory: the
// keys of every bag (as the key kernel forms them), then the same stable LSD
// passes -- warp w ranks positions [w * ni * 32, (w + 1) * ni * 32) in order
// by match.any, the per-digit counts are scanned over the warps and the
// digit totals over the digits, and each key goes to digit base + earlier
// warps' count + its rank in the warp -- and writes the sorted pairs where
// the multi-block sort leaves them.  The result is the same stable sort.
constexpr int kSmallThreads = 1024;
constexpr int kSmallWarps = kSmallThreads / kWarp;
constexpr int kSmallItems = 8;                             // keys per thread at most
constexpr int kSmallMax = kSmallThreads * kSmallItems;    // 8,192 keys
static_assert(kSmallMax == kSmallMaxKeys, "the one-block sort and the short segment items share the edge");
constexpr int64_t kSmallBags = 4 * (int64_t)kSmallMax;    // bags the block's key loop takes

// keys and values twice (cap each), per-warp digit counts, digit bases, scan carries
inline size_t small_sort_smem(int cap) { return 16 * (size_t)cap + 4 * (kSmallWarps * 256 + 256 + kSmallWarps); }

__global__ void __launch_bounds__(kSmallThreads, 1)
small_sort_kernel(const int64_t* __restrict__ row_base, int F, int B, const int32_t* __restrict__ indices,
                  const int32_t* __restrict__ offsets, bool hash, uint32_t* status, uint32_t* __restrict__ keys_out,
                  uint32_t* __restrict__ vals_out, int64_t nbags, int nnz, int ni, int nbits,
                  uint32_t* __restrict__ counters)
{
    extern __shared__ __align__(16) uint32_t ssm[];
    const int cap = ni * kSmallThreads;
    // buffer c (0 or 1): keys at ssm + 2 * c * cap, values cap further
    auto kbuf = [&](int c) { return ssm + 2 * c * cap; };
    auto vbuf = [&](int c) { return ssm + (2 * c + 1) * cap; };
    uint32_t* wcnt = ssm + 4 * cap;   // [kSmallWarps][256]
    uint32_t* dbase = wcnt + kSmallWarps * 256;
    uint32_t* wsum = dbase + 256;
    const int tid = threadIdx.x, lane = tid % kWarp, warp = tid / kWarp;
    const uint32_t lt = (1u << lane) - 1u;
    pdl_wait();
    if (tid < kNumCounters) counters[tid] = 0;   // counters of the segment pass
    // positions no bag covers (malformed offsets only) keep the skip key
    for (int p = tid; p < cap; p += kSmallThreads) {
        kbuf(0)[p] = kSkipKey;
        vbuf(0)[p] = 0;
    }
    __syncthreads();

    // ---- 1. keys, as the key kernel forms them
    auto emit = [&](int64_t p, int32_t raw, int64_t base, int64_t n, uint32_t val) {
        int64_t i = raw;
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
        kbuf(0)[p] = key;
        vbuf(0)[p] = val;
    };
    auto bag = [&](int64_t g, int64_t& s, int64_t& e, int64_t& base, int64_t& n, uint32_t& val) {
        const int t = (int)((uint32_t)g / (uint32_t)B);   // F * B < 2^31
        const int b = (int)g - t * B;
        base = row_base[t];
        n = row_base[t + 1] - base;
        val = (uint32_t)((int64_t)b * F + t);
        s = offsets[g];
        e = offsets[g + 1];
        if (s < 0 || e < s || e > nnz) {   // malformed CSR: clamp, flag, stay in bounds
            set_status(status, DLRM_STATUS_BAD_OFFSETS);
            s = s < 0 ? 0 : (s > nnz ? nnz : s);
            e = e < s ? s : (e > nnz ? nnz : e);
        }
    };
    if (nnz > 2 * nbags) {   // bags of several indices: a warp per bag
        for (int64_t g = warp; g < nbags; g += kSmallWarps) {
            int64_t s, e, base, n;
            uint32_t val;
            bag(g, s, e, base, n, val);
            for (int64_t p = s + lane; p < e; p += kWarp) emit(p, indices[p], base, n, val);
        }
    } else {
        for (int64_t g = tid; g < nbags; g += kSmallThreads) {
            int64_t s, e, base, n;
            uint32_t val;
            bag(g, s, e, base, n, val);
            for (int64_t p = s; p < e; ++p) emit(p, indices[p], base, n, val);
        }
    }
    __syncthreads();

    // ---- 2. stable LSD passes over the bits that can be set
    int cur = 0;
    for (int shift = 0; shift < nbits; shift += 8) {
        const uint32_t mask = (1u << (nbits - shift < 8 ? nbits - shift : 8)) - 1u;
        const uint32_t* kin = kbuf(cur);
        const uint32_t* vin = vbuf(cur);
        for (int x = tid; x < kSmallWarps * 256; x += kSmallThreads) wcnt[x] = 0;
        __syncthreads();
        uint32_t key[kSmallItems], val[kSmallItems], local[kSmallItems];
        const int wbase = warp * ni * kWarp;
#pragma unroll
        for (int r = 0; r < kSmallItems; ++r) {
            if (r < ni) {   // warp-uniform
                const int p = wbase + r * kWarp + lane;
                const bool valid = p < nnz;
                key[r] = valid ? kin[p] : 0;
                val[r] = valid ? vin[p] : 0;
                const uint32_t d = (key[r] >> shift) & mask;
                const uint32_t peers = __match_any_sync(0xffffffffu, valid ? d : 0x100u);
                const uint32_t prior = valid ? wcnt[warp * 256 + d] : 0;
                __syncwarp();
                if (valid && (peers & lt) == 0) wcnt[warp * 256 + d] = prior + __popc(peers);
                __syncwarp();
                local[r] = prior + __popc(peers & lt);
            }
        }
        __syncthreads();
        // per digit: exclusive scan over the warps, then over the digits
        uint32_t total = 0;
        if (tid < 256) {
            for (int w = 0; w < kSmallWarps; ++w) {
                const uint32_t c = wcnt[w * 256 + tid];
                wcnt[w * 256 + tid] = total;
                total += c;
            }
            uint32_t x = total;
#pragma unroll
            for (int o = 1; o < kWarp; o <<= 1) {
                const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
                if (lane >= o) x += y;
            }
            if (lane == kWarp - 1) wsum[warp] = x;
            dbase[tid] = x - total;   // exclusive within the warp's 32 digits
        }
        __syncthreads();
        if (tid < 256) {
            uint32_t before = 0;
            for (int w = 0; w < warp; ++w) before += wsum[w];
            dbase[tid] += before;
        }
        __syncthreads();
        uint32_t* kout = kbuf(cur ^ 1);
        uint32_t* vout = vbuf(cur ^ 1);
#pragma unroll
        for (int r = 0; r < kSmallItems; ++r) {
            if (r < ni) {
                const int p = wbase + r * kWarp + lane;
                if (p < nnz) {
                    const uint32_t d = (key[r] >> shift) & mask;
                    const uint32_t pos = dbase[d] + wcnt[warp * 256 + d] + local[r];
                    if (pos < (uint32_t)nnz) {   // always true for consistent counts; guards the write
                        kout[pos] = key[r];
                        vout[pos] = val[r];
                    }
                }
            }
        }
        __syncthreads();
        cur ^= 1;
    }
    for (int p = tid; p < nnz; p += kSmallThreads) {
        keys_out[p] = kbuf(cur)[p];
        vals_out[p] = vbuf(cur)[p];
    }
}

// ----------------------------------------------------------------- 4. fixup
constexpr int kFixRegs = 4;   // float4 partial-sum loads a lane keeps in flight

// Last item touched by the run of key K that starts in item c0 and continues
// past it.  Keys are sorted, so the run touches item c iff the first key of c
// is K, and the items it touches are c0..L.  Item c0 + 2 is probed first (one
// broadcast load); past it, one round probes c0 + 2^j for j = 0..31 (so
// 2^j <= L - c0 < 2^(j+1) for the last true j), then each round probes 32
// evenly spaced items of the remaining interval.
__device__ __forceinline__ int64_t run_last_item(const uint32_t* __restrict__ keys, int64_t n, int64_t nitems,
                                                 int64_t IT, int64_t c0, uint32_t K, int lane)
{
    auto touches = [&](int64_t c) { return c < nitems && c * IT < n && keys[c * IT] == K; };
    if (!touches(c0 + 2)) return c0 + 1;      // most runs that cross an edge end in the next item
    const uint32_t m = __ballot_sync(0xffffffffu, touches(c0 + ((int64_t)1 << lane)));
    const int j = __popc(m) - 1;              // item c0 + 1 is touched, so j >= 0
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

// Slot of piece j of the run that starts in item c0 (the first piece is the
// starting item's trailing slot, the others are the later items' leading slots).
__device__ __forceinline__ int64_t piece_slot(int64_t c0, int64_t j) { return j == 0 ? 2 * c0 + 1 : 2 * (c0 + j); }

// Pieces [j0, j1) of the run starting in item c0, added in order into acc.
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

// Runs that cross item edges.  Block i < (long runs) takes long run i: warp w
// adds the w-th of kW contiguous slices of its pieces, then warp 0 adds the
// kW slice sums in slice order and updates the row.  Then every warp takes
// short runs (pieces in order, one warp per run).
template <int MC>
__global__ void __launch_bounds__(kFixThreads)
fixup_kernel(const uint32_t* __restrict__ keys, const float* __restrict__ partials,
             const uint64_t* __restrict__ split_list, const uint64_t* __restrict__ long_list,
             const uint32_t* __restrict__ counters, int64_t IT, int D, float* __restrict__ tables,
             int64_t total_rows, float lr)
{
    pdl_wait();
    constexpr int kW = kFixThreads / kWarp;
    extern __shared__ __align__(16) float red[];   // [kW][D]
    const int lane = threadIdx.x % kWarp, warp = threadIdx.x / kWarp;
    const int c4 = D / 4;
    const uint32_t nshort = counters[kCtrSplit], nlong = counters[kCtrLong];
    for (uint32_t i = blockIdx.x; i < nlong; i += gridDim.x) {
        const uint64_t e = long_list[i];
        const int64_t c0 = (int64_t)(e >> 32), pieces = (int64_t)(e & 0xffffffffu);
        const uint32_t K = keys[c0 * IT + IT - 1];
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
        const uint32_t K = keys[c0 * IT + IT - 1];
        float4 acc[MC];
#pragma unroll
        for (int m = 0; m < MC; ++m) acc[m] = make_float4(0.f, 0.f, 0.f, 0.f);
        add_pieces<MC>(partials, c0, 0, pieces, D, lane, acc);
        if ((int64_t)K < total_rows) apply_sgd<MC>(tables, K, D, lr, lane, acc);
    }
}

// --------------------------------------------------------- 3. segment sums
__device__ __forceinline__ void add4(float4& a, const float4& b)
{
    a.x += b.x;
    a.y += b.y;
    a.z += b.z;
    a.w += b.w;
}

// A gradient chunk of four elements as loaded: fp32 as one float4, fp16 as
// the 8 loaded bytes (half the registers), widened exactly to fp32 where it
// is added.
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

// Positions per batch: their gradient rows, and the table rows of the runs
// that complete among them, are all loaded before any is added.
template <int MC, typename GT>
constexpr int seg_batch()
{
    return MC >= 8 ? 1 : (sizeof(GT) == 2 ? 8 : 6) / MC > 0 ? (sizeof(GT) == 2 ? 8 : 6) / MC : 1;
}

// Warps are independent: each takes items of IT = 32 * SUBS positions from a
// counter and walks their 32-position sub-chunks (lane q holds position q's
// key and gradient row number; the next sub-chunk's are loaded meanwhile).
// Rows are added column-wise: lane l holds four-element columns l, l + 32, ...
template <int MC, typename GT, int SUBS>
__global__ void __launch_bounds__(256, MC >= 2 ? 2 : 3)
segment_kernel(const uint32_t* __restrict__ keys, const uint32_t* __restrict__ vals, int64_t n,
               const GT* __restrict__ grad, int D, float* __restrict__ tables, int64_t total_rows, float lr,
               float* __restrict__ partials, uint64_t* __restrict__ split_list, uint64_t* __restrict__ long_list,
               uint32_t* __restrict__ counters, int64_t nitems, int64_t nbags)
{
    constexpr int U = seg_batch<MC, GT>();
    constexpr int64_t IT = (int64_t)kWarp * SUBS;
    const int lane = threadIdx.x % kWarp;
    const int c4 = D / 4;
    pdl_wait();

    auto fetch_item = [&]() -> int64_t {
        uint32_t v = 0;
        if (lane == 0) v = atomicAdd(&counters[kCtrItem], 1u);
        return (int64_t)__shfl_sync(0xffffffffu, v, 0);
    };
    auto load_sub = [&](int64_t item, int j, uint32_t& k, uint32_t& v) {
        const int64_t p = item * IT + (int64_t)j * kWarp + lane;
        k = kSkipKey;
        v = 0;
        if (item < nitems && p < n) {
            k = ldg_early_u32(keys + p);
            v = ldg_early_u32(vals + p);
        }
    };
    auto load_edges = [&](int64_t item, uint32_t& before, uint32_t& after) {
        before = after = kSkipKey;
        if (item < nitems) {
            if (item > 0) before = ldg_early_u32(keys + item * IT - 1);
            if ((item + 1) * IT < n) after = ldg_early_u32(keys + (item + 1) * IT);
        }
    };

    int64_t item = fetch_item();
    int64_t pending = item < nitems ? fetch_item() : nitems;
    uint32_t k_cur, v_cur, before, after;
    load_sub(item, 0, k_cur, v_cur);
    load_edges(item, before, after);
    while (item < nitems) {
        float4 acc[MC];
#pragma unroll
        for (int m = 0; m < MC; ++m) acc[m] = make_float4(0.f, 0.f, 0.f, 0.f);
        bool cs = false;            // the run continuing into this sub-chunk began inside the item
        uint32_t last_key = before;
        uint32_t k_nxt = kSkipKey, v_nxt = 0, before_nxt = kSkipKey, after_nxt = kSkipKey;
        for (int j = 0; j < SUBS; ++j) {
            // next sub-chunk (or the next item's first) in flight while this one is summed
            if (j + 1 < SUBS) {
                load_sub(item, j + 1, k_nxt, v_nxt);
            } else {
                load_sub(pending, 0, k_nxt, v_nxt);
                load_edges(pending, before_nxt, after_nxt);
            }
            const int64_t p = item * IT + (int64_t)j * kWarp + lane;
            const uint32_t k = k_cur;
            const bool valid = p < n && k != kSkipKey;
            const bool loaded = valid && (int64_t)v_cur < nbags;
            uint32_t prev = __shfl_up_sync(0xffffffffu, k, 1);
            if (lane == 0) prev = last_key;
            uint32_t next = __shfl_down_sync(0xffffffffu, k, 1);
            const uint32_t first_next = __shfl_sync(0xffffffffu, k_nxt, 0);
            if (lane == kWarp - 1) next = j + 1 < SUBS ? first_next : after;
            const bool head = valid && prev != k;
            const bool endq = valid && next != k;
            const uint32_t hm = __ballot_sync(0xffffffffu, head);
            const uint32_t em = __ballot_sync(0xffffffffu, endq);
            const uint32_t vm = __ballot_sync(0xffffffffu, valid);
            const uint32_t lm = __ballot_sync(0xffffffffu, loaded);
            const bool stq = (hm & ((2u << lane) - 1u)) != 0 || cs;   // the run through q began inside the item
            const uint32_t cm = __ballot_sync(0xffffffffu, endq && stq && (int64_t)k < total_rows);
            const uint32_t leadm = __ballot_sync(0xffffffffu, endq && !stq);
            const int qmax = vm ? 32 - __clz(vm) : 0;
            for (int q0 = 0; q0 < qmax; q0 += U) {
                typename GradRaw<GT>::T g[U][MC];
                float4 w[U][MC];
                const uint32_t bl = (lm >> q0) & ((1u << U) - 1u);
                const uint32_t bc = (cm >> q0) & ((1u << U) - 1u);
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const GT* src = grad + (int64_t)__shfl_sync(0xffffffffu, v_cur, (q0 + u) & 31) * D;
#pragma unroll
                    for (int m = 0; m < MC; ++m) {
                        const int col = lane + m * kWarp;
                        g[u][m] = typename GradRaw<GT>::T{};
                        if (((bl >> u) & 1u) && col < c4) g[u][m] = load_grad_raw<GT>(src + 4 * col);
                    }
                }
                if (bc) {
#pragma unroll
                    for (int u = 0; u < U; ++u) {
                        const float* trow = tables + (int64_t)__shfl_sync(0xffffffffu, k, (q0 + u) & 31) * D;
#pragma unroll
                        for (int m = 0; m < MC; ++m) {
                            const int col = lane + m * kWarp;
                            w[u][m] = make_float4(0.f, 0.f, 0.f, 0.f);
                            if (((bc >> u) & 1u) && col < c4) w[u][m] = ldg_row_early(trow + 4 * col);
                        }
                    }
                }
                const uint32_t be = (em >> q0) & ((1u << U) - 1u);
#pragma unroll
                for (int u = 0; u < U; ++u) {
#pragma unroll
                    for (int m = 0; m < MC; ++m) add4(acc[m], widen(g[u][m]));
                    if ((be >> u) & 1u) {   // a run piece ends at q0 + u
                        const int q = q0 + u;
                        if ((bc >> u) & 1u) {   // complete run: w = fmaf(-lr, g, w)
                            const uint32_t kk = __shfl_sync(0xffffffffu, k, q);
#pragma unroll
                            for (int m = 0; m < MC; ++m) {
                                const int col = lane + m * kWarp;
                                if (col < c4) {
                                    float4 x = w[u][m];
                                    x.x = fmaf(-lr, acc[m].x, x.x);
                                    x.y = fmaf(-lr, acc[m].y, x.y);
                                    x.z = fmaf(-lr, acc[m].z, x.z);
                                    x.w = fmaf(-lr, acc[m].w, x.w);
                                    *reinterpret_cast<float4*>(tables + (int64_t)kk * D + 4 * col) = x;
                                }
                            }
                        } else if ((leadm >> q) & 1u) {   // leading piece of a run that began in an earlier item
#pragma unroll
                            for (int m = 0; m < MC; ++m) {
                                const int col = lane + m * kWarp;
                                if (col < c4) reinterpret_cast<float4*>(partials + 2 * item * D)[col] = acc[m];
                            }
                        }
#pragma unroll
                        for (int m = 0; m < MC; ++m) acc[m] = make_float4(0.f, 0.f, 0.f, 0.f);
                    }
                }
            }
            // the run through the last valid position continues past this sub-chunk
            const int lastq = qmax - 1;
            const bool cont = vm != 0 && !((em >> lastq) & 1u);
            const bool st_last = __shfl_sync(0xffffffffu, stq, lastq < 0 ? 0 : lastq);
            if (cont) {
                cs = st_last;
                if (j == SUBS - 1) {   // it continues past the item: a trailing or middle piece
                    const int64_t slot = st_last ? 2 * item + 1 : 2 * item;
#pragma unroll
                    for (int m = 0; m < MC; ++m) {
                        const int col = lane + m * kWarp;
                        if (col < c4) reinterpret_cast<float4*>(partials + slot * D)[col] = acc[m];
                    }
                    if (st_last) {   // the run begins in this item: file it with its number of pieces
                        const uint32_t K = __shfl_sync(0xffffffffu, k, lastq);
                        const int64_t pieces = run_last_item(keys, n, nitems, IT, item, K, lane) - item + 1;
                        if (lane == 0) {
                            const uint64_t e = (uint64_t)item << 32 | (uint64_t)pieces;
                            if (pieces > kLongPieces)
                                long_list[atomicAdd(&counters[kCtrLong], 1u)] = e;
                            else
                                split_list[atomicAdd(&counters[kCtrSplit], 1u)] = e;
                        }
                    }
                }
            }
            last_key = __shfl_sync(0xffffffffu, k, kWarp - 1);
            k_cur = k_nxt;
            v_cur = v_nxt;
        }
        item = pending;
        pending = item < nitems ? fetch_item() : nitems;
        before = before_nxt;
        after = after_nxt;
    }
}

template <int MC, typename GT, int SUBS>
dlrm_status launch_segments_subs(const Ws& w, int64_t nnz, const GT* grad, int D, float* tables, int64_t total_rows,
                            float lr, int64_t nbags, cudaStream_t st)
{
    constexpr int64_t IT = (int64_t)kWarp * SUBS;
    const int64_t nitems = (nnz + IT - 1) / IT;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, segment_kernel<MC, GT, SUBS>, 256, 0) != cudaSuccess ||
        per_sm < 1)
        per_sm = 1;
    int64_t blocks = (int64_t)num_sms() * per_sm;   // one resident wave; warps take items from a counter
    const int64_t need = (nitems + 7) / 8;
    if (blocks > need) blocks = need;
    dlrm_status s = check_launch_pdl(launch_pdl(segment_kernel<MC, GT, SUBS>, (int)blocks, 256, 0, st,
                                                (const uint32_t*)w.keys[0], (const uint32_t*)w.vals[0], nnz, grad,
                                                D, tables, total_rows, lr, w.partials, w.split_list, w.long_list,
                                                w.counters, nitems, nbags),
                                     "segment_kernel");
    if (s != DLRM_OK) return s;
    cudaError_t e;
    const size_t fsmem = (size_t)(kFixThreads / kWarp) * D * sizeof(float);
    if (fsmem > 48 * 1024) {
        e = cudaFuncSetAttribute(fixup_kernel<MC>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)fsmem);
        if (e != cudaSuccess) return fail(DLRM_ERR_CUDA, "dlrm_emb_bwd_sgd: %s", cudaGetErrorString(e));
    }
    int64_t fblocks = (int64_t)num_sms() * 4;
    const int64_t fneed = (nitems * kWarp + kFixThreads - 1) / kFixThreads;   // one warp per item at most
    if (fblocks > fneed) fblocks = fneed;
    return check_launch_pdl(launch_pdl(fixup_kernel<MC>, (int)fblocks, kFixThreads, fsmem, st,
                                       (const uint32_t*)w.keys[0], (const float*)w.partials,
                                       (const uint64_t*)w.split_list, (const uint64_t*)w.long_list,
                                       (const uint32_t*)w.counters, IT, D, tables, total_rows, lr),
                            "fixup_kernel");
}

template <int MC, typename GT>
dlrm_status launch_segments(const Ws& w, int64_t nnz, const GT* grad, int D, float* tables, int64_t total_rows,
                            float lr, int64_t nbags, cudaStream_t st)
{
    if (item_subs(nnz) == kSubsSmall)
        return launch_segments_subs<MC, GT, kSubsSmall>(w, nnz, grad, D, tables, total_rows, lr, nbags, st);
    return launch_segments_subs<MC, GT, kSubs>(w, nnz, grad, D, tables, total_rows, lr, nbags, st);
}

// The segment pass and the fixup for the gradient type and width.
dlrm_status launch_all_segments(const Ws& w, int64_t nnz, const void* d_grad, unsigned flags, int D, float* tables,
                                int64_t total_rows, float lr, int64_t nbags, cudaStream_t st)
{
    if (flags & DLRM_FLAG_GRAD_F16) {
        const __half* grad = static_cast<const __half*>(d_grad);
        if (D <= 128) return launch_segments<1>(w, nnz, grad, D, tables, total_rows, lr, nbags, st);
        if (D <= 256) return launch_segments<2>(w, nnz, grad, D, tables, total_rows, lr, nbags, st);
        if (D <= 512) return launch_segments<4>(w, nnz, grad, D, tables, total_rows, lr, nbags, st);
        return launch_segments<8>(w, nnz, grad, D, tables, total_rows, lr, nbags, st);
    }
    const float* grad = static_cast<const float*>(d_grad);
    if (D <= 128) return launch_segments<1>(w, nnz, grad, D, tables, total_rows, lr, nbags, st);
    if (D <= 256) return launch_segments<2>(w, nnz, grad, D, tables, total_rows, lr, nbags, st);
    if (D <= 512) return launch_segments<4>(w, nnz, grad, D, tables, total_rows, lr, nbags, st);
    return launch_segments<8>(w, nnz, grad, D, tables, total_rows, lr, nbags, st);
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
    DLRM_API_RANGE("dlrm_emb_bwd_sgd");
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
    if ((flags & DLRM_FLAG_GRAD_F16) && D % 8 != 0)
        return fail(DLRM_ERR_UNSUPPORTED, "dlrm_emb_bwd_sgd: fp16 gradients need D a multiple of 8");
    if (!aligned16(d_tables) || !aligned16(d_grad_pooled))
        return fail(DLRM_ERR_UNSUPPORTED, "dlrm_emb_bwd_sgd: tables and grad_pooled must be 16-byte aligned");
    if (nnz > 0 && (reinterpret_cast<uintptr_t>(d_workspace) & 255u))
        return fail(DLRM_ERR_UNSUPPORTED, "dlrm_emb_bwd_sgd: workspace must be 256-byte aligned");
    const size_t need = dlrm_emb_bwd_sgd_workspace_size(nnz, D, total_rows);
    if (nnz > 0 && workspace_bytes < need)
        return fail(DLRM_ERR_WORKSPACE, "dlrm_emb_bwd_sgd: workspace %zu bytes < %zu needed", workspace_bytes, need);
    if (nnz == 0 || B == 0) return DLRM_OK;

    cudaStream_t st = as_stream(stream);
    const Ws w = carve(d_workspace, nnz, D);
    const int nbits = key_bits(total_rows);
    const int npasses = (nbits + 7) / 8;
    int cur = npasses & 1;   // the last pass lands in buffer 0

    const int64_t nbags = (int64_t)F * B;
    if (nnz <= kSmallMax && nbags <= kSmallBags) {   // one block sorts in shared memory
        const int ni = (int)((nnz + kSmallThreads - 1) / kSmallThreads);
        const size_t smem = small_sort_smem(ni * kSmallThreads);
        cudaError_t e = cudaFuncSetAttribute(small_sort_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)small_sort_smem(kSmallMax));
        if (e == cudaSuccess)
            e = launch_pdl(small_sort_kernel, 1, kSmallThreads, smem, st, d_row_base, F, B, d_indices, d_offsets,
                           (flags & DLRM_FLAG_HASH_INDICES) != 0, d_status, w.keys[0], w.vals[0], nbags, (int)nnz,
                           ni, nbits, w.counters);
        dlrm_status s = check_launch_pdl(e, "small_sort_kernel");
        if (s != DLRM_OK) return s;
        return launch_all_segments(w, nnz, d_grad_pooled, flags, D, d_tables, total_rows, lr, nbags, st);
    }
    const bool multi = nnz > 2 * nbags;
    const bool hash = (flags & DLRM_FLAG_HASH_INDICES) != 0;
    const int64_t ntiles = w.ntiles;
    const int64_t bpb = (nbags + ntiles - 1) / ntiles;   // bags per first-pass tile
    {
        const uint32_t mask0 = (1u << (nbits < 8 ? nbits : 8)) - 1u;
        const cudaError_t e =
            multi ? launch_pdl(keys_kernel<32>, (int)ntiles, kSortThreads, 0, st, d_row_base, F, B, d_indices,
                               d_offsets, hash, d_status, w.keys[cur], w.vals[cur], nbags, nnz, bpb, mask0, w.hist,
                               ntiles, w.counters)
                  : launch_pdl(keys_kernel<1>, (int)ntiles, kSortThreads, 0, st, d_row_base, F, B, d_indices,
                               d_offsets, hash, d_status, w.keys[cur], w.vals[cur], nbags, nnz, bpb, mask0, w.hist,
                               ntiles, w.counters);
        dlrm_status s = check_launch_pdl(e, "keys_kernel");
        if (s != DLRM_OK) return s;
    }
    for (int pass = 0; pass < npasses; ++pass) {
        const int shift = 8 * pass;
        const int bits = nbits - shift < 8 ? nbits - shift : 8;
        const uint32_t mask = (1u << bits) - 1u;
        cudaError_t e = cudaSuccess;
        if (pass > 0)   // the first pass's histogram comes from the key kernel
            e = launch_pdl(radix_upsweep, (int)ntiles, kSortThreads, 0, st, (const uint32_t*)w.keys[cur], nnz, shift,
                           mask, w.hist, ntiles);
        if (e == cudaSuccess) e = launch_pdl(radix_scan, 256, kSortThreads, 0, st, w.hist, ntiles, w.totals);
        if (e == cudaSuccess)
            e = launch_pdl(pass == 0 ? radix_downsweep<true> : radix_downsweep<false>, (int)ntiles, kSortThreads, 0,
                           st, (const uint32_t*)w.keys[cur],
                           (const uint32_t*)w.vals[cur], w.keys[cur ^ 1], w.vals[cur ^ 1], nnz, shift, mask,
                           (const uint32_t*)w.hist, (const uint32_t*)w.totals, ntiles,
                           pass == 0 ? d_offsets : (const int32_t*)nullptr, bpb, nbags);
        dlrm_status s = check_launch_pdl(e, "radix sort pass");
        if (s != DLRM_OK) return s;
        cur ^= 1;
    }
    return launch_all_segments(w, nnz, d_grad_pooled, flags, D, d_tables, total_rows, lr, nbags, st);
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

// Identity of the calling thread's current CUDA context (0 if there is none
// or the driver cannot say): cuCtxGetId numbers every context the process
// creates, so a context made after a device reset gets a new number.  The two
// driver calls are looked up through the runtime, so the library does not link
// the driver library directly.
unsigned long long current_context_id()
{
    using GetCurrentFn = CUresult (*)(CUcontext*);
    using GetIdFn = CUresult (*)(CUcontext, unsigned long long*);
    static GetCurrentFn get_current = nullptr;
    static GetIdFn get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        cudaDriverEntryPointQueryResult q;
        void* f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<GetCurrentFn>(f);
        f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<GetIdFn>(f);
    });
    if (!get_current || !get_id) return 0;
    CUcontext ctx = nullptr;
    if (get_current(&ctx) != CUDA_SUCCESS || !ctx) return 0;
    unsigned long long id = 0;
    return get_id(ctx, &id) == CUDA_SUCCESS ? id : 0;
}

// Device address of g_sgd_scratch for the current device.  In host code the
// array's name is only a host-side stand-in, so the address is queried with
// the device current (once per device and context) and cached.
dlrm_status static_scratch(void** out)
{
    struct Entry {
        unsigned long long ctx;
        void* ptr;
    };
    static std::mutex mu;
    static Entry cache[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(DLRM_ERR_CUDA, "dlrm_emb_bwd_sgd_noalloc: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= 64) return fail(DLRM_ERR_UNSUPPORTED, "dlrm_emb_bwd_sgd_noalloc: device %d", dev);
    std::lock_guard<std::mutex> lock(mu);
    const unsigned long long ctx = current_context_id();
    if (!cache[dev].ptr || ctx == 0 || cache[dev].ctx != ctx) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_sgd_scratch);
        if (e != cudaSuccess || !p)
            return fail(DLRM_ERR_CUDA, "dlrm_emb_bwd_sgd_noalloc: cudaGetSymbolAddress: %s", cudaGetErrorString(e));
        cache[dev].ptr = p;
        cache[dev].ctx = current_context_id();   // the lookup made the device's primary context current if needed
    }
    *out = cache[dev].ptr;
    return DLRM_OK;
}

}  // namespace
}  // namespace dlrm

extern "C" dlrm_status dlrm_emb_bwd_sgd_noalloc(float* d_tables, const int64_t* d_row_base, int64_t total_rows,
                                                int F, int D, int B, const int32_t* d_indices,
                                                const int32_t* d_offsets, int64_t nnz,
                                                const void* d_grad_pooled, float lr, unsigned flags,
                                                uint32_t* d_status, void* stream)
{
    DLRM_API_RANGE("dlrm_emb_bwd_sgd_noalloc");
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
