// fp4.cuh -- device helpers for the low-precision rows: the hardware E2M1 conversions, the MXFP4
// quantisation of one 64-value indexer row by a warp (format and sources in fp4.cu), the NVFP4
// entry row and the FP8 window row of the V4.1 cache variant (formats below), and their
// widening to BF16. Used by the quantisers, the compression, the decode-state append and the
// attention kernels.
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
// one byte of E2M1 codes to two halves (bits 0-3 -> .x, bits 4-7 -> .y), exact
__device__ __forceinline__ __half2 e2m1x2_to_h2(uint8_t v) {
    uint32_t r;
    asm("{.reg .b8 t; mov.b16 {t, _}, %1; cvt.rn.f16x2.e2m1x2 %0, t;}" : "=r"(r) : "h"((uint16_t)v));
    return *reinterpret_cast<__half2 *>(&r);
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

// ---- NVFP4 compressed entries (an 80-byte row per entry) --------------------------------
// Reading of the V4.1 cache format ([P3] "Технический отчёт DeepSeek-V4.1-Flash — часть 2/2":
// the KV cache is kept in NVFP4, quantised after RoPE): E2M1 elements in blocks of 16 with one
// E4M3 scale per block and one float scale per entry. Row layout: bytes [0, 64) the codes
// (dim 2i in the low nibble of byte i), [64, 72) the eight block scales, [72, 76) the row scale
// s = max|c| / (6 * 448) (so every block scale fits E4M3), [76, 80) zero. Block b: code
// E4M3(max_b / (6 s)), scale_b = E4M3 value * s; element = E2M1(c / scale_b) (0 when scale_b is
// 0). Value = E2M1 * scale_b.
constexpr int kNvfp4RowBytes = 80;

// A warp stores one 128-dim row held as c[e] = dim lane + 32 e (e < 4).
__device__ __forceinline__ void nvfp4_row_store(const float (&c)[4], uint8_t *row) {
    const int lane = threadIdx.x & 31;
    float am = fmaxf(fmaxf(fabsf(c[0]), fabsf(c[1])), fmaxf(fabsf(c[2]), fabsf(c[3])));
    am = warp_max(am);
    const float s = __fdiv_rn(am, 6.0f * 448.0f);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        float bm = fabsf(c[e]);  // max over the 16 lanes of this half-warp = block 2e + (lane >= 16)
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, o));
        const uint8_t sb = s > 0.0f ? f32_to_e4m3(__fdiv_rn(bm, 6.0f * s)) : (uint8_t)0;
        const float scale = e4m3_to_f32(sb) * s;
        const float q = scale > 0.0f ? __fdiv_rn(c[e], scale) : 0.0f;
        const float qn = __shfl_down_sync(0xffffffffu, q, 1);
        if ((lane & 1) == 0) row[(lane + 32 * e) >> 1] = e2m1x2_from(q, qn);
        if ((lane & 15) == 0) row[64 + 2 * e + (lane >> 4)] = sb;
    }
    if (lane == 0) {
        *reinterpret_cast<float *>(row + 72) = s;
        *reinterpret_cast<uint32_t *>(row + 76) = 0u;
    }
}

// ---- FP8 window rows (a 144-byte row per raw token) -------------------------------------
// Reading of the V4.1 window cache ([P3]: the SWA KV cache is kept in FP8): 128 E4M3 codes of
// the rotated raw row with one float scale s = max|x| / 448 at byte 128 (code = E4M3(x / s)),
// bytes [132, 144) zero. Value = code * s.
constexpr int kFp8WinRowBytes = 144;

// A warp stores one 128-dim window row held as c[e] = dim lane + 32 e (e < 4).
__device__ __forceinline__ void fp8win_row_store(const float (&c)[4], uint8_t *row) {
    const int lane = threadIdx.x & 31;
    const float am = warp_max(fmaxf(fmaxf(fabsf(c[0]), fabsf(c[1])), fmaxf(fabsf(c[2]), fabsf(c[3]))));
    const float s = __fdiv_rn(am, 448.0f);
#pragma unroll
    for (int e = 0; e < 4; ++e) row[lane + 32 * e] = s > 0.0f ? f32_to_e4m3(__fdiv_rn(c[e], s)) : (uint8_t)0;
    if (lane < 4) *reinterpret_cast<uint32_t *>(row + 128 + 4 * lane) = lane == 0 ? __float_as_uint(s) : 0u;
}

// ---- widening to BF16 (8 dims = one 16-byte chunk of a BF16 row) ------------------------
__device__ __forceinline__ uint32_t bf16x2_bits(float a, float b) {
    __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&v);
}

// eight E4M3 codes (byte i = dim i) times the row scale s, each product rounded to BF16
__device__ __forceinline__ uint4 fp8x8_to_bf16(uint32_t lo, uint32_t hi, float s) {
    const uint32_t w[2] = {lo, hi};
    uint32_t pk[4];
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const uint16_t two = (uint16_t)(w[h] >> (16 * e));
            __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)two, __NV_E4M3);
            const float2 f = __half22float2(__half2(hr));
            pk[2 * h + e] = bf16x2_bits(f.x * s, f.y * s);
        }
    return make_uint4(pk[0], pk[1], pk[2], pk[3]);
}

// eight E2M1 codes (dim 2i in the low nibble of byte i) of one NVFP4 block with block-scale code
// sb and entry scale s: value = E2M1 * (E4M3(sb) * s), rounded to BF16
__device__ __forceinline__ uint4 fp4x8_to_bf16(uint32_t codes, uint32_t sb, float s) {
    const float scale = e4m3_to_f32((uint8_t)sb) * s;
    uint32_t pk[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const float2 v = e2m1x2_to((uint8_t)(codes >> (8 * e)));
        pk[e] = bf16x2_bits(v.x * scale, v.y * scale);
    }
    return make_uint4(pk[0], pk[1], pk[2], pk[3]);
}

}  // namespace csa
