// common.cu -- error reporting, device queries and the seeded table synthesiser.
#include <cstring>
#include <atomic>
#include <mutex>

#include "common.cuh"
#include "dlrm_synth.h"

namespace dlrm {

static thread_local char g_last_error[512] = "";

void set_error(const char* fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
    va_end(ap);
}

void clear_error() { g_last_error[0] = '\0'; }

static std::atomic<long long> g_wait_limit{-1};   // negative: the default

long long wait_limit_cycles()
{
    const long long v = g_wait_limit.load(std::memory_order_relaxed);
    return v < 0 || v > kDefaultWaitCycles ? kDefaultWaitCycles : v;
}

long long set_wait_limit_cycles(long long cycles)
{
    const long long prev = wait_limit_cycles();
    g_wait_limit.store(cycles < 0 ? -1 : cycles, std::memory_order_relaxed);
    return prev;
}

int num_sms()
{
    static std::mutex mu;
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 152;
    std::lock_guard<std::mutex> lock(mu);
    if (cache[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            n = 152;
        cache[dev] = n;
    }
    return cache[dev];
}

// ------------------------------------------------------------------ synthesis
// splitmix64 (Steele, Lea & Flood, OOPSLA 2014): output e of the stream
// seeded with `seed` is mix(seed + (e + 1) * golden_gamma).
__device__ __forceinline__ uint64_t splitmix64_at(uint64_t seed, uint64_t e)
{
    uint64_t z = seed + (e + 1ull) * 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

template <typename T>
__global__ void synth_uniform_kernel(T* dst, uint64_t seed, int64_t first, int64_t count, float scale)
{
    int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < count; i += stride) {
        const uint64_t z = splitmix64_at(seed, (uint64_t)(first + i));
        const int x = (int)(z >> 40) - (1 << 23);               // exact in fp32
        const float f = __fmul_rn((float)x, scale);             // one rounding
        if constexpr (sizeof(T) == 2)
            dst[i] = __float2half_rn(f);
        else
            dst[i] = f;
    }
}

}  // namespace dlrm

using namespace dlrm;

extern "C" int64_t dlrm_set_wait_limit(int64_t cycles) { return set_wait_limit_cycles(cycles); }

extern "C" size_t dlrm_ws_align(size_t bytes) { return (bytes + 255) & ~(size_t)255; }

extern "C" const char* dlrm_last_error(void) { return g_last_error; }

extern "C" dlrm_status dlrm_synth_fill_uniform(void* d_dst, dlrm_dtype dtype, uint64_t seed,
                                               int64_t first_elem, int64_t count, double amplitude,
                                               void* stream)
{
    DLRM_API_RANGE("dlrm_synth_fill_uniform");
    clear_error();
    if (!d_dst) return fail(DLRM_ERR_INVALID_ARG, "dlrm_synth_fill_uniform: d_dst is NULL");
    if (count < 0 || first_elem < 0)
        return fail(DLRM_ERR_INVALID_ARG, "dlrm_synth_fill_uniform: negative count or first_elem");
    if (!dtype_ok(dtype)) return fail(DLRM_ERR_INVALID_ARG, "dlrm_synth_fill_uniform: bad dtype");
    if (count == 0) return DLRM_OK;
    const float scale = (float)(amplitude / 8388608.0);
    int threads = 256;
    int64_t want = (count + threads - 1) / threads;
    int blocks = (int)(want < (int64_t)num_sms() * 16 ? want : (int64_t)num_sms() * 16);
    if (dtype == DLRM_F16)
        synth_uniform_kernel<__half><<<blocks, threads, 0, as_stream(stream)>>>(
            (__half*)d_dst, seed, first_elem, count, scale);
    else
        synth_uniform_kernel<float><<<blocks, threads, 0, as_stream(stream)>>>(
            (float*)d_dst, seed, first_elem, count, scale);
    return check_launch("synth_uniform_kernel");
}
