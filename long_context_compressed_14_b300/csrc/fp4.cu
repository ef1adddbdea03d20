// fp4.cu -- FP4 (E2M1) rows for the lightning indexer: MXFP4 quantisation and the lossless
// dequantisation to FP8 E4M3 rows that lets the FP8 tensor-core indexer consume them; and the
// quantisers of the low-precision caches: NVFP4 entry rows and FP8 window rows (formats in
// fp4.cuh).
//
// Sources: [P2] "DeepSeek-V4: Towards Highly Efficient Million-Token Context Intelligence"
// (wiki notes), 事後学習 §3 (the CSA indexer's QK path is quantised to FP4 (MXFP4); the FP4 to
// FP8 dequantisation is lossless, so the FP8 stack is reused) and 提案手法 §1 (the lightning
// indexer computes its scores in FP4); [P5] "deepseek V4 技术论文" 一.1 (低秩分解+FP4计算).
//
// MXFP4 rows of 64 values: two blocks of 32 E2M1 elements, each block with one E8M0 exponent
// byte e8 (scale 2^(e8 - 127)); e = floor(log2(block max)) - 2 (clamped to [-127, 127], 2 being
// the exponent of E2M1's largest value 6), elements = E2M1(v / 2^e), rounded to nearest even
// and saturated at 6 by the hardware conversion. Element 2i sits in the low nibble of byte i.
//
// FP8 form of an MXFP4 row (used by the FP8 indexer): with E = the row's larger block exponent,
// code_i = E4M3(v_i * 2^(e_blk - E + 6)) and the row scale 2^(E - 6). An E2M1 value times a power
// of two has at most two significant bits, and with e_blk - E >= -14 it stays inside E4M3's range
// (largest 6 * 2^6 = 384 <= 448, smallest 0.5 * 2^-8 = 2^-9, E4M3's least subnormal), so the
// conversion is exact for rows whose block exponents lie within 14 binades of each other.
#include "common.cuh"
#include "fp4.cuh"
#include "kernels.cuh"

namespace csa {

__global__ void quant_mxfp4_kernel(const float *__restrict__ x, int64_t rows, uint8_t *__restrict__ codes,
                                   uint8_t *__restrict__ e8) {
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t r = blockIdx.x * (int64_t)(blockDim.x >> 5) + (threadIdx.x >> 5); r < rows; r += warps) {
        const float *row = x + r * kDI;
        mxfp4_row_store(row[lane], row[32 + lane], codes + r * (kDI / 2), e8 + r * 2);
    }
}

// MXFP4 rows -> E4M3 rows with one float scale per row (lossless within 14 binades, above)
__global__ void mxfp4_to_fp8_kernel(const uint8_t *__restrict__ codes, const uint8_t *__restrict__ e8, int64_t rows,
                                    uint8_t *__restrict__ out, float *__restrict__ out_scale) {
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t r = blockIdx.x * (int64_t)(blockDim.x >> 5) + (threadIdx.x >> 5); r < rows; r += warps) {
        const int e0 = (int)e8[r * 2] - 127, e1 = (int)e8[r * 2 + 1] - 127;
        const int E = e0 > e1 ? e0 : e1;
        const uint8_t b0 = codes[r * (kDI / 2) + (lane >> 1)], b1 = codes[r * (kDI / 2) + 16 + (lane >> 1)];
        const float2 p0 = e2m1x2_to(b0), p1 = e2m1x2_to(b1);
        const float v0 = (lane & 1) ? p0.y : p0.x, v1 = (lane & 1) ? p1.y : p1.x;
        out[r * kDI + lane] = f32_to_e4m3(ldexpf(v0, e0 - E + 6));
        out[r * kDI + 32 + lane] = f32_to_e4m3(ldexpf(v1, e1 - E + 6));
        if (lane == 0) out_scale[r] = ldexpf(1.0f, E - 6);
    }
}

// NVFP4 entry rows and FP8 window rows of 128-dim float rows: one warp per row (fp4.cuh)
__global__ void quant_nvfp4_kernel(const float *__restrict__ x, int64_t rows, uint8_t *__restrict__ out) {
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t r = blockIdx.x * (int64_t)(blockDim.x >> 5) + (threadIdx.x >> 5); r < rows; r += warps) {
        const float c[4] = {x[r * kD + lane], x[r * kD + 32 + lane], x[r * kD + 64 + lane], x[r * kD + 96 + lane]};
        nvfp4_row_store(c, out + r * kNvfp4RowBytes);
    }
}

__global__ void quant_fp8win_kernel(const float *__restrict__ x, int64_t rows, uint8_t *__restrict__ out) {
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t r = blockIdx.x * (int64_t)(blockDim.x >> 5) + (threadIdx.x >> 5); r < rows; r += warps) {
        const float c[4] = {x[r * kD + lane], x[r * kD + 32 + lane], x[r * kD + 64 + lane], x[r * kD + 96 + lane]};
        fp8win_row_store(c, out + r * kFp8WinRowBytes);
    }
}

static int blocks_for(int64_t rows) {
    int64_t b = (rows + 7) / 8;
    if (b > 148 * 32) b = 148 * 32;
    return (int)(b < 1 ? 1 : b);
}

void launch_quant_mxfp4(const float *x, int64_t rows, uint8_t *codes, uint8_t *e8, cudaStream_t st) {
    if (rows <= 0) return;
    quant_mxfp4_kernel<<<blocks_for(rows), 256, 0, st>>>(x, rows, codes, e8);
    count_launches(1);
}

void launch_mxfp4_to_fp8(const uint8_t *codes, const uint8_t *e8, int64_t rows, uint8_t *out, float *out_scale,
                         cudaStream_t st) {
    if (rows <= 0) return;
    mxfp4_to_fp8_kernel<<<blocks_for(rows), 256, 0, st>>>(codes, e8, rows, out, out_scale);
    count_launches(1);
}

void launch_quant_nvfp4_entries(const float *x, int64_t rows, uint8_t *out, cudaStream_t st) {
    if (rows <= 0) return;
    quant_nvfp4_kernel<<<blocks_for(rows), 256, 0, st>>>(x, rows, out);
    count_launches(1);
}

void launch_quant_fp8_window(const float *x, int64_t rows, uint8_t *out, cudaStream_t st) {
    if (rows <= 0) return;
    quant_fp8win_kernel<<<blocks_for(rows), 256, 0, st>>>(x, rows, out);
    count_launches(1);
}

}  // namespace csa
