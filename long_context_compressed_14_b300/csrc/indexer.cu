// indexer.cu -- lightning-indexer scores on CUDA cores.
//
// Sources: [P2] "DeepSeek-V4: Towards Highly Efficient Million-Token Context Intelligence"
// (wiki notes), 提案手法 §1 CSA (a lightning indexer scores compressed entries for top-k);
// [P5] "deepseek V4 技术论文" 一.1 (low-rank, cheap); [P4] "EP 95 DeepSeek-V4論文を読む" 17:10
// (it looks at every entry, so it must be light).
//
// Score of query row t against entry j (visible iff (j+1)m-1 <= t):
//   s(t,j) = sum_h w[t,h] * ReLU(qI[t,h] . KI[j]).
// FP32 operands: the fixed order acc = fma(q_c, k_c, acc) (c ascending, from +0),
//   r = acc > 0 ? acc : 0, s = fma(w_h, r, s) (h ascending, from +0), -0 -> +0, so that a
//   top-k selection made from these scores is exactly reproducible.
// FP8 operands: s = sk_j * sum_h (w_h * sq_h) * ReLU(sum_c qcode_c * kcode_c) -- the row
//   scales factor out of the ReLU because they are positive.
// This file holds the CUDA-core kernels: the exact FP32 path and the decode scan (one query
// per sequence, HBM-bound). The FP8 prefill indexer, with the selection fused in, runs on the
// tensor cores (index_select.cu).
#include "common.cuh"
#include "kernels.cuh"

namespace csa {

constexpr int kIdxTQ = 32;   // query rows per CTA
constexpr int kIdxTJ = 64;   // entries per CTA

// Prefill: CTA = 32 query rows x 64 entries of sequence a.b; thread = 8 (row, entry) pairs.
template <int IDX_T>
__global__ void __launch_bounds__(256)
indexer_prefill_kernel(IndexArgs a) {
    extern __shared__ float smem[];
    const int H_I = a.H_I;
    float *q_s = smem;                                  // [32][H_I][64]
    float *w_s = q_s + kIdxTQ * H_I * kDI;              // [32][H_I]
    float *k_s = w_s + kIdxTQ * H_I;                    // [64][65]
    float *ks_s = k_s + kIdxTJ * (kDI + 1);             // [64]

    const int tq0 = a.t0 + blockIdx.y * kIdxTQ;
    const int nq = min(kIdxTQ, a.t0 + a.nrows - tq0);
    const int j0 = blockIdx.x * kIdxTJ;
    const int vis_max = visible_entries(tq0 + nq - 1, a.m, a.ncap);
    if (j0 >= vis_max) return;
    const int nj = min(kIdxTJ, vis_max - j0);
    const int64_t row0 = (int64_t)a.b * a.L + tq0;

    for (int e = threadIdx.x; e < kIdxTQ * H_I * kDI; e += 256) {
        const int r = e / (H_I * kDI);
        float v = 0.0f;
        if (r < nq) {
            if (IDX_T == CSA_F32) v = reinterpret_cast<const float *>(a.qI)[row0 * H_I * kDI + e];
            else v = e4m3_to_f32(reinterpret_cast<const uint8_t *>(a.qI)[row0 * H_I * kDI + e]);
        }
        q_s[e] = v;
    }
    for (int e = threadIdx.x; e < kIdxTQ * H_I; e += 256) {
        const int r = e / H_I;
        float v = 0.0f;
        if (r < nq) {
            v = a.w[row0 * H_I + e];
            if (IDX_T != CSA_F32) v = v * a.qI_scale[row0 * H_I + e];
        }
        w_s[e] = v;
    }
    const int64_t kbase = (int64_t)a.b * a.ncap + j0;
    for (int e = threadIdx.x; e < kIdxTJ * kDI; e += 256) {
        const int jj = e / kDI, c = e % kDI;
        float v = 0.0f;
        if (jj < nj) {
            if (IDX_T == CSA_F32) v = reinterpret_cast<const float *>(a.KI)[(kbase + jj) * kDI + c];
            else v = e4m3_to_f32(reinterpret_cast<const uint8_t *>(a.KI)[(kbase + jj) * kDI + c]);
        }
        k_s[jj * (kDI + 1) + c] = v;
    }
    if (IDX_T != CSA_F32)
        for (int e = threadIdx.x; e < kIdxTJ; e += 256) ks_s[e] = e < nj ? a.KI_scale[kbase + e] : 0.0f;
    __syncthreads();

    const int jj = threadIdx.x % kIdxTJ;
    const int j = j0 + jj;
    for (int r = threadIdx.x / kIdxTJ; r < nq; r += 256 / kIdxTJ) {
        const int t = tq0 + r;
        if (jj >= nj || j >= visible_entries(t, a.m, a.ncap)) continue;
        const float *q = q_s + r * H_I * kDI;
        const float *k = k_s + jj * (kDI + 1);
        float s = 0.0f;
        for (int h = 0; h < H_I; ++h) {
            float acc = 0.0f;
#pragma unroll 16
            for (int c = 0; c < kDI; ++c) acc = __fmaf_rn(q[h * kDI + c], k[c], acc);
            const float rl = acc > 0.0f ? acc : 0.0f;
            s = __fmaf_rn(w_s[r * H_I + h], rl, s);
        }
        if (IDX_T != CSA_F32) s = s * ks_s[jj];
        if (s == 0.0f) s = 0.0f;
        a.S[(int64_t)(t - a.t0) * a.ldS + j] = s;
    }
}

// Decode: one query per sequence; CTA = 256 entries of one sequence, thread = one entry.
template <int IDX_T>
__global__ void __launch_bounds__(256)
indexer_decode_kernel(IndexArgs a) {
    __shared__ float q_s[16 * kDI];
    __shared__ float w_s[16];
    const int b = blockIdx.y;
    const int H_I = a.H_I;
    const int64_t p = (int64_t)a.ctx[b] - 1;
    if (p < 0 || p >= a.L) return;  // reported by the attention kernel
    const int vis = visible_entries(p, a.m, a.ncap);
    const int j0 = blockIdx.x * 256;
    if (j0 >= vis) return;
    for (int e = threadIdx.x; e < H_I * kDI; e += 256) {
        if (IDX_T == CSA_F32) q_s[e] = reinterpret_cast<const float *>(a.qI)[(int64_t)b * H_I * kDI + e];
        else q_s[e] = e4m3_to_f32(reinterpret_cast<const uint8_t *>(a.qI)[(int64_t)b * H_I * kDI + e]);
    }
    if (threadIdx.x < H_I) {
        float v = a.w[b * H_I + threadIdx.x];
        if (IDX_T != CSA_F32) v = v * a.qI_scale[b * H_I + threadIdx.x];
        w_s[threadIdx.x] = v;
    }
    __syncthreads();
    const int j = j0 + threadIdx.x;
    if (j >= vis) return;
    const int64_t krow = (int64_t)b * a.ncap + j;
    float k[kDI];
    if (IDX_T == CSA_F32) {
        const float4 *src = reinterpret_cast<const float4 *>(reinterpret_cast<const float *>(a.KI) + krow * kDI);
#pragma unroll
        for (int v = 0; v < kDI / 4; ++v) {
            float4 x = src[v];
            k[4 * v] = x.x; k[4 * v + 1] = x.y; k[4 * v + 2] = x.z; k[4 * v + 3] = x.w;
        }
    } else {
        const uint4 *src = reinterpret_cast<const uint4 *>(reinterpret_cast<const uint8_t *>(a.KI) + krow * kDI);
#pragma unroll
        for (int v = 0; v < kDI / 16; ++v) {
            uint4 x = src[v];
            const uint32_t wd[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
            for (int q = 0; q < 4; ++q)
#pragma unroll
                for (int e = 0; e < 4; ++e) k[16 * v + 4 * q + e] = e4m3_to_f32((uint8_t)(wd[q] >> (8 * e)));
        }
    }
    float s = 0.0f;
    for (int h = 0; h < H_I; ++h) {
        float acc = 0.0f;
#pragma unroll
        for (int c = 0; c < kDI; ++c) acc = __fmaf_rn(q_s[h * kDI + c], k[c], acc);
        const float rl = acc > 0.0f ? acc : 0.0f;
        s = __fmaf_rn(w_s[h], rl, s);
    }
    if (IDX_T != CSA_F32) s = s * a.KI_scale[krow];
    if (s == 0.0f) s = 0.0f;
    a.S[(int64_t)b * a.ldS + j] = s;
}

void launch_indexer(const IndexArgs &a, cudaStream_t st) {
    if (a.decode) {
        dim3 grid((unsigned)ceil_div64(a.ncap, 256), a.B);
        if (a.idx_t == CSA_F32) indexer_decode_kernel<CSA_F32><<<grid, 256, 0, st>>>(a);
        else indexer_decode_kernel<CSA_FP8E4M3><<<grid, 256, 0, st>>>(a);
        count_launches(1);
        return;
    }
    const int last_vis = visible_entries((int64_t)a.t0 + a.nrows - 1, a.m, a.ncap);
    if (last_vis <= 0) return;
    dim3 grid((unsigned)ceil_div64(last_vis, kIdxTJ), (unsigned)ceil_div64(a.nrows, kIdxTQ));
    const size_t smem = sizeof(float) * ((size_t)kIdxTQ * a.H_I * kDI + kIdxTQ * a.H_I +
                                         kIdxTJ * (kDI + 1) + kIdxTJ);
    if (a.idx_t == CSA_F32) {
        cudaFuncSetAttribute(indexer_prefill_kernel<CSA_F32>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        indexer_prefill_kernel<CSA_F32><<<grid, 256, smem, st>>>(a);
    } else {
        cudaFuncSetAttribute(indexer_prefill_kernel<CSA_FP8E4M3>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        indexer_prefill_kernel<CSA_FP8E4M3><<<grid, 256, smem, st>>>(a);
    }
    count_launches(1);
}

}  // namespace csa
