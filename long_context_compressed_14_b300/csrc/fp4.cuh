// fp4.cuh -- device helpers for FP4 (E2M1) rows: the hardware E2M1 conversions and the MXFP4
// quantisation of one 64-value row by a warp (used by the quantiser, the compression and the
// decode-state append). The format and its sources are described in fp4.cu.
#pragma once

#include <cuda_fp16.h>

#include "common.cuh"

namespace csa {

// two floats to one byte of E2M1 codes: lo in bits 0-3, hi in bits 4-7 (round to nearest even,
// saturated at +-6)
__device__ __forceinline__ uint8_t e2m1x2_from(float lo, float hi) {
    uint16_t d;
    asm("{.reg .b8 t; cvt.rn.satfinite.e2m1x2.f32 t, %1, %2; mov.b16 %0, {t, 0};}" : "=h"(d) : "f"(hi), "f"(lo));
    return (uint8_t)d;
}
// one byte of E2M1 codes to two floats (bits 0-3 -> .x, bits 4-7 -> .y)
__device__ __forceinline__ float2 e2m1x2_to(uint8_t v) {
    uint32_t r;
    asm("{.reg .b8 t; mov.b16 {t, _}, %1; cvt.rn.f16x2.e2m1x2 %0, t;}" : "=r"(r) : "h"((uint16_t)v));
    return __half22float2(*reinterpret_cast<__half2 *>(&r));
}

__device__ __forceinline__ int mx_block_exp(float amax) {
    if (!(amax > 0.0f)) return -127;
    const int e = ilogbf(amax) - 2;
    return e < -127 ? -127 : (e > 127 ? 127 : e);
}

// One warp quantises the 64 values of one row held as (x0, x1) = (element lane, element 32 +
// lane); lane 0 writes the two exponent bytes, even lanes the code bytes.
__device__ __forceinline__ void mxfp4_row_store(float x0, float x1, uint8_t *codes, uint8_t *e8) {
    const int lane = threadIdx.x & 31;
    const int e0 = mx_block_exp(warp_max(fabsf(x0))), e1 = mx_block_exp(warp_max(fabsf(x1)));
    const float v0 = ldexpf(x0, -e0), v1 = ldexpf(x1, -e1);
    const float n0 = __shfl_down_sync(0xffffffffu, v0, 1), n1 = __shfl_down_sync(0xffffffffu, v1, 1);
    if ((lane & 1) == 0) {
        codes[lane >> 1] = e2m1x2_from(v0, n0);
        codes[16 + (lane >> 1)] = e2m1x2_from(v1, n1);
    }
    if (lane == 0) {
        e8[0] = (uint8_t)(e0 + 127);
        e8[1] = (uint8_t)(e1 + 127);
    }
}

}  // namespace csa
