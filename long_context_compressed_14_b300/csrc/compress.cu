// compress.cu -- RoPE table, FP8 row quantisation and the fused overlapping compression.
//
// Sources: [P2] "DeepSeek-V4: Towards Highly Efficient Million-Token Context Intelligence"
// (wiki notes), 提案手法 §1 (CSA: weighted-average compression of every m = 4 tokens with
// overlap between adjacent blocks; HCA: m' = 128; partial RoPE on the last 64 dims) and
// 訓練インフラの革新 §5 (KV entries: RoPE dims BF16, other dims FP8); [P5] "deepseek V4
// 技术论文" 一.1 (C^b overlaps C^a); [P3] "Технический отчёт DeepSeek-V4.1-Flash — часть 2/2"
// (the V4.1 variant: entries in NVFP4, quantised after RoPE).
#include "common.cuh"
#include "fp4.cuh"
#include "kernels.cuh"

namespace csa {

// ---------------------------------------------------------------------------------------
// RoPE table: tab[pos][i] = (cos, sin)(pos * theta^(-i/half)), double math, float storage.
// ---------------------------------------------------------------------------------------
__global__ void rope_table_kernel(float2 *tab, int rope_len, int half, double theta) {
    const int64_t n = (int64_t)rope_len * half;
    for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < n;
         e += (int64_t)gridDim.x * blockDim.x) {
        const int64_t pos = e / half;
        const int i = (int)(e % half);
        const double freq = pow(theta, -(double)i / (double)half);
        double s, c;
        sincos((double)pos * freq, &s, &c);
        tab[e] = make_float2((float)c, (float)s);
    }
}

void launch_rope_table(float *tab, int rope_len, int d_rope, float theta, cudaStream_t st) {
    const int half = d_rope / 2;
    const int64_t n = (int64_t)rope_len * half;
    int blocks = (int)((n + 255) / 256);
    if (blocks > 148 * 16) blocks = 148 * 16;
    if (blocks < 1) blocks = 1;
    rope_table_kernel<<<blocks, 256, 0, st>>>(reinterpret_cast<float2 *>(tab), rope_len, half,
                                                (double)theta);
    count_launches(1);
}

// ---------------------------------------------------------------------------------------
// Per-row FP8 quantisation: one warp per row.
// ---------------------------------------------------------------------------------------
__global__ void quant_rows_kernel(const float *__restrict__ x, int64_t rows, int cols,
                                  uint8_t *__restrict__ codes, float *__restrict__ scales) {
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t r = blockIdx.x * (int64_t)(blockDim.x >> 5) + (threadIdx.x >> 5); r < rows; r += warps) {
        const float *row = x + r * cols;
        float amax = 0.0f;
        for (int c = lane; c < cols; c += 32) amax = fmaxf(amax, fabsf(row[c]));
        amax = warp_max(amax);
        const float scale = __fdiv_rn(amax, 448.0f);
        for (int c = lane; c < cols; c += 32)
            codes[r * cols + c] = scale > 0.0f ? f32_to_e4m3(__fdiv_rn(row[c], scale)) : (uint8_t)0;
        if (lane == 0) scales[r] = scale;
    }
}

void launch_quant_rows(const float *x, int64_t rows, int cols, uint8_t *codes, float *scales,
                       cudaStream_t st) {
    int64_t blocks = (rows + 7) / 8;
    if (blocks > 148 * 32) blocks = 148 * 32;
    if (blocks < 1) blocks = 1;
    quant_rows_kernel<<<(int)blocks, 256, 0, st>>>(x, rows, cols, codes, scales);
    count_launches(1);
}

// ---------------------------------------------------------------------------------------
// kv_compress: one CTA (4 warps) per entry j of sequence b.
//   window rows [(j-1)m, (j+1)m) ∩ [0, L); weight of row t = exp(z[t, set] - max) with set 0
//   for the own block (t >= jm) and set 1 for the previous block; normalised at the end.
//   Warp g accumulates the rows g, g+4, ...; lane l owns dims {l, l+32, l+64, l+96} of the
//   KV row (so that RoPE pairs (64+i, 96+i) sit in one lane) and dims {l, l+32} of the
//   indexer-key row.
// ---------------------------------------------------------------------------------------
constexpr int kMaxWindow = 2 * 1024;

template <typename ActT, int KV_T, int IDX_T, bool WITH_KI, bool WITH_KVROPE>
__global__ void __launch_bounds__(128)
kv_compress_kernel(const ActT *__restrict__ kv, const float *__restrict__ z,
                   const float *__restrict__ kI_raw, const float2 *__restrict__ rope,
                   void *__restrict__ c_data, __nv_bfloat16 *__restrict__ c_rope,
                   float *__restrict__ c_scale, void *__restrict__ ki_data,
                   float *__restrict__ ki_scale, uint8_t *__restrict__ ki_e8, ActT *__restrict__ kv_rope, int L,
                   int m, int N, int d_rope) {
    __shared__ float s_w[kMaxWindow];
    __shared__ float s_red[4][kD + kDI];
    __shared__ float s_scalar[8];

    const int j = blockIdx.x, b = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t lo = (int64_t)(j - 1) * m < 0 ? 0 : (int64_t)(j - 1) * m;
    const int64_t hi = (int64_t)(j + 1) * m > L ? (int64_t)L : (int64_t)(j + 1) * m;
    const int n = (int)(hi - lo);
    const int64_t own0 = (int64_t)j * m;
    const float *zb = z + (int64_t)b * L * 2;

    // softmax weights of the window
    float mx = -INFINITY;
    for (int i = threadIdx.x; i < n; i += 128) {
        const int64_t t = lo + i;
        const float l = zb[2 * t + (t >= own0 ? 0 : 1)];
        s_w[i] = l;
        mx = fmaxf(mx, l);
    }
    mx = warp_max(mx);
    if (lane == 0) s_scalar[warp] = mx;
    __syncthreads();
    mx = fmaxf(fmaxf(s_scalar[0], s_scalar[1]), fmaxf(s_scalar[2], s_scalar[3]));
    float den = 0.0f;
    for (int i = threadIdx.x; i < n; i += 128) {
        const float e = expf(s_w[i] - mx);
        s_w[i] = e;
        den += e;
    }
    den = warp_sum(den);
    __syncthreads();
    if (lane == 0) s_scalar[4 + warp] = den;
    __syncthreads();
    den = (s_scalar[4] + s_scalar[5]) + (s_scalar[6] + s_scalar[7]);

    const int half = d_rope / 2;  // 32 or 0
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    float acck[2] = {0.f, 0.f};
    const ActT *kvb = kv + (int64_t)b * L * kD;
    for (int i = warp; i < n; i += 4) {
        const int64_t t = lo + i;
        const float wt = s_w[i];
        float x[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) x[e] = to_f(kvb[t * kD + lane + 32 * e]);
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[e] = fmaf(wt, x[e], acc[e]);
        if (WITH_KI) {
            const float *kr = kI_raw + ((int64_t)b * L + t) * kDI;
            acck[0] = fmaf(wt, kr[lane], acck[0]);
            acck[1] = fmaf(wt, kr[lane + 32], acck[1]);
        }
        if (WITH_KVROPE && t >= own0) {
            // this raw row belongs to block j: write it rotated at its own position t
            float y[4] = {x[0], x[1], x[2], x[3]};
            if (half == 32) {
                const float2 cs = rope[t * half + lane];
                y[2] = x[2] * cs.x - x[3] * cs.y;
                y[3] = x[2] * cs.y + x[3] * cs.x;
            }
            ActT *dst = kv_rope + ((int64_t)b * L + t) * kD;
#pragma unroll
            for (int e = 0; e < 4; ++e) dst[lane + 32 * e] = from_f<ActT>(y[e]);
        }
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) s_red[warp][lane + 32 * e] = acc[e];
    if (WITH_KI) {
        s_red[warp][kD + lane] = acck[0];
        s_red[warp][kD + lane + 32] = acck[1];
    }
    __syncthreads();
    if (warp != 0) return;

    const float inv = 1.0f / den;
    float c[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const int dd = lane + 32 * e;
        c[e] = ((s_red[0][dd] + s_red[1][dd]) + (s_red[2][dd] + s_red[3][dd])) * inv;
    }
    if (half == 32) {
        const int64_t pos = (int64_t)(j + 1) * m - 1;
        const float2 cs = rope[pos * half + lane];
        const float a = c[2], bb = c[3];
        c[2] = a * cs.x - bb * cs.y;
        c[3] = a * cs.y + bb * cs.x;
    }
    const int64_t row = (int64_t)b * N + j;
    if (KV_T == CSA_F32) {
        float *dst = reinterpret_cast<float *>(c_data) + row * kD;
#pragma unroll
        for (int e = 0; e < 4; ++e) dst[lane + 32 * e] = c[e];
    } else if (KV_T == CSA_BF16) {
        __nv_bfloat16 *dst = reinterpret_cast<__nv_bfloat16 *>(c_data) + row * kD;
#pragma unroll
        for (int e = 0; e < 4; ++e) dst[lane + 32 * e] = __float2bfloat16_rn(c[e]);
    } else if (KV_T == CSA_NVFP4) {  // the whole rotated entry in NVFP4 (fp4.cuh)
        nvfp4_row_store(c, reinterpret_cast<uint8_t *>(c_data) + row * kNvfp4RowBytes);
    } else {  // MIXED: dims 0..63 FP8 + row scale, dims 64..127 BF16
        float amax = warp_max(fmaxf(fabsf(c[0]), fabsf(c[1])));
        const float scale = __fdiv_rn(amax, 448.0f);
        uint8_t *dst = reinterpret_cast<uint8_t *>(c_data) + row * 64;
        dst[lane] = scale > 0.0f ? f32_to_e4m3(__fdiv_rn(c[0], scale)) : (uint8_t)0;
        dst[lane + 32] = scale > 0.0f ? f32_to_e4m3(__fdiv_rn(c[1], scale)) : (uint8_t)0;
        if (lane == 0) c_scale[row] = scale;
        __nv_bfloat16 *rr = c_rope + row * 64;
        rr[lane] = __float2bfloat16_rn(c[2]);
        rr[lane + 32] = __float2bfloat16_rn(c[3]);
    }
    if (WITH_KI) {
        float k0 = ((s_red[0][kD + lane] + s_red[1][kD + lane]) + (s_red[2][kD + lane] + s_red[3][kD + lane])) * inv;
        float k1 = ((s_red[0][kD + lane + 32] + s_red[1][kD + lane + 32]) +
                    (s_red[2][kD + lane + 32] + s_red[3][kD + lane + 32])) * inv;
        if (IDX_T == CSA_F32) {
            float *dst = reinterpret_cast<float *>(ki_data) + row * kDI;
            dst[lane] = k0;
            dst[lane + 32] = k1;
        } else if (IDX_T == CSA_MXFP4) {
            mxfp4_row_store(k0, k1, reinterpret_cast<uint8_t *>(ki_data) + row * (kDI / 2), ki_e8 + row * 2);
        } else {
            const float amax = warp_max(fmaxf(fabsf(k0), fabsf(k1)));
            const float scale = __fdiv_rn(amax, 448.0f);
            uint8_t *dst = reinterpret_cast<uint8_t *>(ki_data) + row * kDI;
            dst[lane] = scale > 0.0f ? f32_to_e4m3(__fdiv_rn(k0, scale)) : (uint8_t)0;
            dst[lane + 32] = scale > 0.0f ? f32_to_e4m3(__fdiv_rn(k1, scale)) : (uint8_t)0;
            if (lane == 0) ki_scale[row] = scale;
        }
    }
}

template <typename ActT, int KV_T, int IDX_T>
static void launch_compress_t(const CompressArgs &a, cudaStream_t st) {
    dim3 grid(a.N, a.B);
    const ActT *kv = reinterpret_cast<const ActT *>(a.kv);
    ActT *kvr = reinterpret_cast<ActT *>(a.kv_rope);
    const float2 *rope = reinterpret_cast<const float2 *>(a.rope_tab);
    auto *cr = reinterpret_cast<__nv_bfloat16 *>(a.c_rope);
#define CSA_LAUNCH(KI, KVR)                                                                          \
    kv_compress_kernel<ActT, KV_T, IDX_T, KI, KVR><<<grid, 128, 0, st>>>(                            \
        kv, a.z, a.kI_raw, rope, a.c_data, cr, a.c_scale, a.ki_data, a.ki_scale, a.ki_e8, kvr, a.L, a.m, a.N, \
        a.d_rope)
    if (a.kI_raw && a.kv_rope) CSA_LAUNCH(true, true);
    else if (a.kI_raw) CSA_LAUNCH(true, false);
    else if (a.kv_rope) CSA_LAUNCH(false, true);
    else CSA_LAUNCH(false, false);
#undef CSA_LAUNCH
}

template <typename ActT, int KV_T>
static void launch_compress_k(const CompressArgs &a, cudaStream_t st) {
    if (a.idx_t == CSA_FP8E4M3) launch_compress_t<ActT, KV_T, CSA_FP8E4M3>(a, st);
    else if (a.idx_t == CSA_MXFP4) launch_compress_t<ActT, KV_T, CSA_MXFP4>(a, st);
    else launch_compress_t<ActT, KV_T, CSA_F32>(a, st);
}

template <typename ActT>
static void launch_compress_a(const CompressArgs &a, cudaStream_t st) {
    if (a.kv_t == CSA_F32) launch_compress_k<ActT, CSA_F32>(a, st);
    else if (a.kv_t == CSA_BF16) launch_compress_k<ActT, CSA_BF16>(a, st);
    else if (a.kv_t == CSA_NVFP4) launch_compress_k<ActT, CSA_NVFP4>(a, st);
    else launch_compress_k<ActT, CSA_MIXED>(a, st);
}

void launch_kv_compress(const CompressArgs &a, cudaStream_t st) {
    if (a.act_t == CSA_F32) launch_compress_a<float>(a, st);
    else launch_compress_a<__nv_bfloat16>(a, st);
    count_launches(1);
}

}  // namespace csa
