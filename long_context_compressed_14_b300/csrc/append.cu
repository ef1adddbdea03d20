// append.cu -- incremental decode state: one new token per sequence appended to the sliding
// window, to the state cache of the incomplete block and, when the token completes a block, to
// the compressed caches.
//
// Sources: [P2] "DeepSeek-V4: Towards Highly Efficient Million-Token Context Intelligence"
// (wiki notes), 訓練インフラの革新 §5 (the inference KV cache is heterogeneous: a state cache of
// the recent raw tokens, whose incomplete block waits there, and the compressed KV cache) and
// 提案手法 §1 (overlapping compression: entry j averages the raw rows of blocks j-1 and j with
// softmax weights; sliding window of the last n_win raw tokens; partial RoPE); [P5] "deepseek V4
// 技术论文" 一.1 (C^b overlaps C^a); [P3] "Технический отчёт DeepSeek-V4.1-Flash — часть 2/2"
// (the V4.1 variant: entries in NVFP4 quantised after RoPE, the window cache in FP8).
//
// One CTA of 128 threads per sequence, thread = head dimension. For the new token at position u:
//   ring[u mod n_win]   = its raw row rotated at u (the window keys), in act_t or as an FP8 row;
//   state[u mod 2m]     = its raw row, its compression logits z and its raw indexer key (the last
//                         2m tokens: exactly the window rows [u - 2m + 1, u] an entry needs);
//   if u = (j+1)m - 1   entry j = sum_t alpha_t kv[t] over t in [(j-1)m, (j+1)m) ∩ [0, u], alpha =
//                       softmax of z[t, 0] (t in block j) or z[t, 1] (t in block j-1), rotated at
//                       (j+1)m - 1 and stored per kv_t; KI_j = sum_t alpha_t kI[t], stored per
//                       idx_t. The arithmetic follows kv_compress (float sums, row quantisation
//                       with scale = amax / 448).
// Entries of incomplete blocks are not written: no decode query can see them.
#include "common.cuh"
#include "fp4.cuh"
#include "kernels.cuh"

namespace csa {

template <typename ActT, int KV_T, int IDX_T>
__global__ void __launch_bounds__(128) kv_append_kernel(AppendArgs a) {
    __shared__ float s_x[kD];       // the new raw row / the entry before storage
    __shared__ float s_y[kD];       // a rotated row gathered for a warp's row quantiser
    __shared__ float s_w[2 * 1024]; // window weights
    __shared__ float s_red[8];
    const int b = blockIdx.x, d = threadIdx.x, lane = d & 31, warp = d >> 5;
    const int64_t u = (int64_t)a.ctx[b] - 1;
    if (u < 0 || u >= a.L) {
        if (d == 0) set_status(CSA_ERR_BOUNDS);
        return;
    }
    const int m = a.m, m2 = 2 * a.m;
    const int half = a.d_rope / 2;  // 32 or 0
    const float2 *rope = reinterpret_cast<const float2 *>(a.rope_tab);
    // 1. the new token into the state cache and (rotated) into the window ring
    const ActT *kvn = reinterpret_cast<const ActT *>(a.kv_new) + (int64_t)b * kD;
    const float x = to_f(kvn[d]);
    ActT *st_kv = reinterpret_cast<ActT *>(a.state_kv) + (int64_t)b * m2 * kD;
    st_kv[(u % m2) * kD + d] = kvn[d];
    if (d < 2) a.state_z[((int64_t)b * m2 + u % m2) * 2 + d] = a.z_new[(int64_t)b * 2 + d];
    if (a.kI_new && d < kDI) a.state_kI[((int64_t)b * m2 + u % m2) * kDI + d] = a.kI_new[(int64_t)b * kDI + d];
    s_x[d] = x;
    __syncthreads();
    float y = x;
    if (half == 32 && d >= kD - 64) {  // pairs (64 + i, 96 + i) rotated at u
        const int i = (d - 64) & 31;
        const float2 cs = rope[u * half + i];
        const float x0 = s_x[64 + i], x1 = s_x[96 + i];
        y = d < 96 ? x0 * cs.x - x1 * cs.y : x0 * cs.y + x1 * cs.x;
    }
    const int64_t slot = (int64_t)b * a.n_win + u % a.n_win;
    if (a.win_t == CSA_FP8E4M3) {  // an FP8 ring row (fp4.cuh): warp 0 quantises the whole row
        s_y[d] = y;
        __syncthreads();
        if (warp == 0) {
            const float r[4] = {s_y[lane], s_y[32 + lane], s_y[64 + lane], s_y[96 + lane]};
            fp8win_row_store(r, reinterpret_cast<uint8_t *>(a.ring) + slot * kFp8WinRowBytes);
        }
    } else {
        reinterpret_cast<ActT *>(a.ring)[slot * kD + d] = from_f<ActT>(y);
    }
    if ((u + 1) % m != 0) return;  // the token does not complete a block

    // 2. the token completes block j: entry j from the window rows held in the state cache
    __syncthreads();  // this CTA's state writes are visible to its threads
    const int64_t j = u / m;
    const int64_t lo = (j - 1) * m < 0 ? 0 : (j - 1) * m, own0 = j * m;
    const int n = (int)(u + 1 - lo);
    const float *sz = a.state_z + (int64_t)b * m2 * 2;
    float mx = -INFINITY;
    for (int i = d; i < n; i += 128) {
        const int64_t t = lo + i;
        const float l = sz[(t % m2) * 2 + (t >= own0 ? 0 : 1)];
        s_w[i] = l;
        mx = fmaxf(mx, l);
    }
    mx = warp_max(mx);
    if (lane == 0) s_red[warp] = mx;
    __syncthreads();
    mx = fmaxf(fmaxf(s_red[0], s_red[1]), fmaxf(s_red[2], s_red[3]));
    float den = 0.0f;
    for (int i = d; i < n; i += 128) {
        const float e = expf(s_w[i] - mx);
        s_w[i] = e;
        den += e;
    }
    den = warp_sum(den);
    __syncthreads();
    if (lane == 0) s_red[4 + warp] = den;
    __syncthreads();
    den = (s_red[4] + s_red[5]) + (s_red[6] + s_red[7]);
    const float inv = 1.0f / den;
    float c = 0.0f, ck = 0.0f;
    for (int i = 0; i < n; ++i) {
        const int64_t slot = (lo + i) % m2;
        const float wt = s_w[i];
        c = fmaf(wt, to_f(st_kv[slot * kD + d]), c);
        if (a.kI_new && d < kDI) ck = fmaf(wt, a.state_kI[((int64_t)b * m2 + slot) * kDI + d], ck);
    }
    c *= inv;
    ck *= inv;
    __syncthreads();
    s_x[d] = c;
    __syncthreads();
    if (half == 32 && d >= kD - 64) {  // the entry rotated at its position (j+1)m - 1 = u
        const int i = (d - 64) & 31;
        const float2 cs = rope[u * half + i];
        const float c0 = s_x[64 + i], c1 = s_x[96 + i];
        c = d < 96 ? c0 * cs.x - c1 * cs.y : c0 * cs.y + c1 * cs.x;
    }
    const int64_t row = (int64_t)b * a.ncap + j;
    if (KV_T == CSA_F32) {
        reinterpret_cast<float *>(a.c_data)[row * kD + d] = c;
    } else if (KV_T == CSA_BF16) {
        reinterpret_cast<__nv_bfloat16 *>(a.c_data)[row * kD + d] = __float2bfloat16_rn(c);
    } else if (KV_T == CSA_NVFP4) {  // the rotated entry in NVFP4 (fp4.cuh), stored by warp 0
        s_y[d] = c;
        __syncthreads();
        if (warp == 0) {
            const float r[4] = {s_y[lane], s_y[32 + lane], s_y[64 + lane], s_y[96 + lane]};
            nvfp4_row_store(r, reinterpret_cast<uint8_t *>(a.c_data) + row * kNvfp4RowBytes);
        }
    } else {  // MIXED: dims 0..63 FP8 with one scale, dims 64..127 BF16
        const float am = warp_max(d < 64 ? fabsf(c) : 0.0f);
        if (lane == 0) s_red[warp] = am;
        __syncthreads();
        const float scale = __fdiv_rn(fmaxf(s_red[0], s_red[1]), 448.0f);
        if (d < 64) {
            reinterpret_cast<uint8_t *>(a.c_data)[row * 64 + d] = scale > 0.0f ? f32_to_e4m3(__fdiv_rn(c, scale)) : (uint8_t)0;
            if (d == 0) a.c_scale[row] = scale;
        } else {
            a.c_rope[row * 64 + (d - 64)] = __float2bfloat16_rn(c);
        }
        __syncthreads();
    }
    if (a.kI_new) {
        if (IDX_T == CSA_F32) {
            if (d < kDI) reinterpret_cast<float *>(a.ki_data)[row * kDI + d] = ck;
        } else if (IDX_T == CSA_MXFP4) {
            // warp 0 holds dims 0..31, warp 1 dims 32..63: gather the row into warp 0
            __syncthreads();
            s_x[d] = ck;
            __syncthreads();
            if (warp == 0)
                mxfp4_row_store(s_x[lane], s_x[32 + lane], reinterpret_cast<uint8_t *>(a.ki_data) + row * (kDI / 2),
                                a.ki_e8 + row * 2);
        } else {
            const float am = warp_max(d < kDI ? fabsf(ck) : 0.0f);
            if (lane == 0) s_red[warp] = am;
            __syncthreads();
            const float scale = __fdiv_rn(fmaxf(s_red[0], s_red[1]), 448.0f);
            if (d < kDI) {
                reinterpret_cast<uint8_t *>(a.ki_data)[row * kDI + d] =
                    scale > 0.0f ? f32_to_e4m3(__fdiv_rn(ck, scale)) : (uint8_t)0;
                if (d == 0) a.ki_scale[row] = scale;
            }
        }
    }
}

template <typename ActT, int KV_T>
static void launch_append_k(const AppendArgs &a, cudaStream_t st) {
    if (a.idx_t == CSA_FP8E4M3) kv_append_kernel<ActT, KV_T, CSA_FP8E4M3><<<a.B, 128, 0, st>>>(a);
    else if (a.idx_t == CSA_MXFP4) kv_append_kernel<ActT, KV_T, CSA_MXFP4><<<a.B, 128, 0, st>>>(a);
    else kv_append_kernel<ActT, KV_T, CSA_F32><<<a.B, 128, 0, st>>>(a);
}

template <typename ActT>
static void launch_append_a(const AppendArgs &a, cudaStream_t st) {
    if (a.kv_t == CSA_F32) launch_append_k<ActT, CSA_F32>(a, st);
    else if (a.kv_t == CSA_BF16) launch_append_k<ActT, CSA_BF16>(a, st);
    else if (a.kv_t == CSA_NVFP4) launch_append_k<ActT, CSA_NVFP4>(a, st);
    else launch_append_k<ActT, CSA_MIXED>(a, st);
}

void launch_kv_append(const AppendArgs &a, cudaStream_t st) {
    if (a.act_t == CSA_F32) launch_append_a<float>(a, st);
    else launch_append_a<__nv_bfloat16>(a, st);
    count_launches(1);
}

}  // namespace csa
