// common.cuh -- shared host/device helpers of the CUDA library (not the oracle).
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <cstdarg>
#include <type_traits>
#include <utility>
#include <cstdio>

#include "dlrm.h"
#include <nvtx3/nvToolsExt.h>

namespace dlrm {

// ---------------------------------------------------------------- host side
void set_error(const char* fmt, ...);
void clear_error();

inline dlrm_status fail(dlrm_status code, const char* fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    set_error("%s", buf);
    return code;
}

inline dlrm_status check_launch(const char* what)
{
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(DLRM_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
    return DLRM_OK;
}

// Launch with programmatic stream serialization: the launch is processed
// while the previous kernel on the stream runs.  Every kernel launched this
// way calls pdl_wait() before touching global memory, so it still sees all of
// the previous kernel's writes and makes none the previous kernel could see.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

inline dlrm_status check_launch_pdl(cudaError_t e, const char* what)
{
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(DLRM_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
    }
    return check_launch(what);
}

// NVTX range around one C-ABI call (the host-side enqueue): profilers that
// record NVTX show each call by its name over the kernels it launched.
// Without a tool attached the push and pop cost a few nanoseconds.
struct ApiRange {
    explicit ApiRange(const char* name) { nvtxRangePushA(name); }
    ~ApiRange() { nvtxRangePop(); }
    ApiRange(const ApiRange&) = delete;
    ApiRange& operator=(const ApiRange&) = delete;
};
#define DLRM_API_RANGE(name) ::dlrm::ApiRange dlrm_api_range_(name)

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline int dtype_size(dlrm_dtype dt) { return dt == DLRM_F16 ? 2 : 4; }
inline bool dtype_ok(dlrm_dtype dt) { return dt == DLRM_F32 || dt == DLRM_F16; }
inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

int num_sms();   // SM count of the current device (cached per device)

// Cycles a bounded on-chip wait of the tensor-core kernels lasts before the
// kernel gives up (dlrm_set_wait_limit; about two seconds by default).
constexpr long long kDefaultWaitCycles = 4000000000LL;
long long wait_limit_cycles();
long long set_wait_limit_cycles(long long cycles);   // negative: the default; returns the previous limit

// -------------------------------------------------------------- device side
constexpr int kWarp = 32;

// Programmatic dependent launch: wait for the previous grid on the stream to
// complete (its writes visible).  A no-op for a grid launched without the
// attribute.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// No kernel triggers its dependents early (griddepcontrol.launch_dependents):
// the next grid is then scheduled only when this one completes, and the
// attribute still hides its launch processing.  With an early trigger the
// next grid's blocks took registers and shared memory on SMs as this grid's
// blocks left, and a one-wave persistent grid that followed (the one-pass
// forward after the sparse update, the backward after the forward) started
// with fewer blocks on those SMs: 0.851 ms per 64K fp32 training step with the
// trigger, 0.808 ms without, 0.839 ms with plain launches.

__device__ __forceinline__ void set_status(uint32_t* status, uint32_t bit)
{
    if (status) atomicOr(status, bit);
}

// 16-byte read-only load that does not allocate in L1 (rows are streamed).
__device__ __forceinline__ uint4 ldg_nc_v4(const void* p)
{
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// 4-byte read-only load issued where it is written: volatile, so the compiler
// neither sinks it to its first use nor reorders it with other volatile loads
// (used to start index reads a pipeline step ahead of their use).
__device__ __forceinline__ int ldg_early_s32(const int32_t* p)
{
    int r;
    asm volatile("ld.global.nc.s32 %0, [%1];" : "=r"(r) : "l"(p));
    return r;
}

// 16-byte read-only load that allocates in L1 (gathers of Zipf-hot rows).
__device__ __forceinline__ uint4 ldg_nc_l1_v4(const void* p)
{
    uint4 r;
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// 16-byte streaming store (evict-first: outputs are not re-read by this kernel).
__device__ __forceinline__ void stg_cs_v4(void* p, uint4 v)
{
    asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ float4 u4_as_f4(uint4 v)
{
    return make_float4(__uint_as_float(v.x), __uint_as_float(v.y), __uint_as_float(v.z),
                       __uint_as_float(v.w));
}

__device__ __forceinline__ uint4 f4_as_u4(float4 v)
{
    return make_uint4(__float_as_uint(v.x), __float_as_uint(v.y), __float_as_uint(v.z),
                      __float_as_uint(v.w));
}

// 8 halves packed in a uint4 -> 8 floats (exact widening).
__device__ __forceinline__ void h8_to_f8(uint4 v, float* f)
{
    const __half2* h = reinterpret_cast<const __half2*>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float2 t = __half22float2(h[i]);
        f[2 * i] = t.x;
        f[2 * i + 1] = t.y;
    }
}

// 8 floats -> 8 halves (round to nearest even) packed in a uint4.
__device__ __forceinline__ uint4 f8_to_h8(const float* f)
{
    uint4 v;
    __half2* h = reinterpret_cast<__half2*>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2half2_rn(f[2 * i], f[2 * i + 1]);
    return v;
}

template <typename Fn, int... Is>
__device__ __forceinline__ void static_for_impl(Fn& fn, std::integer_sequence<int, Is...>)
{
    (fn(std::integral_constant<int, Is>{}), ...);
}

// fn(std::integral_constant<int, 0>), ..., fn(std::integral_constant<int, N-1>):
// every index is a constant expression, so register arrays stay in registers.
template <int N, typename Fn>
__device__ __forceinline__ void static_for(Fn&& fn)
{
    static_for_impl(fn, std::make_integer_sequence<int, N>{});
}

}  // namespace dlrm
