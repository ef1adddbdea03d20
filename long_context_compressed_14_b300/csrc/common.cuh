// common.cuh -- device helpers shared by the library's kernels (not by the oracle).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/csa.h"

namespace csa {

constexpr int kD = 128;      // head dim
constexpr int kDI = 64;      // indexer dim
constexpr int kMaxTopk = 2048;

// Device status word (first error wins) and the abort flag raised with a timeout, which makes
// every other bounded wait give up at once. Both defined in api.cu, cleared by
// csa_device_status(reset).
extern __device__ int g_status;
extern __device__ int g_abort;

__device__ __forceinline__ void set_status(int code) { atomicCAS(&g_status, 0, code); }

// Programmatic dependent launch (the decode step's chain of kernels): a kernel launched with
// launch_pdl may be scheduled while the previous kernel of the stream is still running; it
// lets its own successor be scheduled at once (pdl_trigger) and waits for the previous kernel's
// completion and memory (pdl_wait) before it touches global memory. Both are no-ops in a kernel
// launched the ordinary way.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<Args &&>(args)...);
}
__device__ __forceinline__ void set_timeout() {
    atomicCAS(&g_status, 0, CSA_ERR_TIMEOUT);
    atomicExch(&g_abort, 1);
}

// ---- element loads / stores ------------------------------------------------------------
__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

// FP8 E4M3 ("fn") conversions through the hardware cvt instructions: round to nearest even,
// saturating finite values to +-448.
__device__ __forceinline__ uint8_t f32_to_e4m3(float x) {
    return (uint8_t)__nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3);
}
__device__ __forceinline__ float e4m3_to_f32(uint8_t c) {
    __half_raw h = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)c, __NV_E4M3);
    return __half2float(__half(h));
}

// Orderable key of a float score for a descending radix select: larger float -> larger key.
// -0 is folded onto +0 first; the invisible marker -inf maps below every finite score.
__device__ __forceinline__ uint32_t score_key(float s) {
    if (s == 0.0f) s = 0.0f;
    uint32_t u = __float_as_uint(s);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Two FP32 lanes in one 64-bit register pair (x in the low word) and the packed FMA on them:
// d.x = a.x * b.x + c.x, d.y = a.y * b.y + c.y, each rounded to nearest like fmaf.
__device__ __forceinline__ uint64_t f2_pack(float x, float y) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(x), "f"(y));
    return r;
}
__device__ __forceinline__ float2 f2_unpack(uint64_t r) {
    float2 v;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(v.x), "=f"(v.y) : "l"(r));
    return v;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__host__ __device__ __forceinline__ int64_t ceil_div64(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Number of entries visible to a query at position t (entry j visible iff (j+1)m-1 <= t).
__host__ __device__ __forceinline__ int visible_entries(int64_t t, int m, int ncap) {
    int64_t v = (t + 1) / m;
    return (int)(v < ncap ? v : ncap);
}

}  // namespace csa
