// attn_simple.cu -- core attention on CUDA cores (FP32 math), any head count <= 64.
//
// Sources: [P2] "DeepSeek-V4: Towards Highly Efficient Million-Token Context Intelligence"
// (wiki notes), 提案手法 §1 (shared-KV multi-query attention; sliding-window branch with
// n_win = 128 for both CSA and HCA; an attention sink lets the total attention of a head be
// below 1; partial RoPE on the last 64 dims with inverse RoPE on the core output);
// [P5] "deepseek V4 技术论文" 一.1 (a compressed entry is both key and value).
//
// One CTA per query row (one token, all heads). The key list of the row is the compressed
// branch (CSA: its top-k entries; HCA: every visible entry) followed by the window rows
// [p - n_win + 1, p]. Keys stream through shared memory in tiles of 32; warp w owns heads
// w, w+8, ... with an online softmax per head; lane l owns output dims {l, l+32, l+64,
// l+96}, so each RoPE pair (64+i, 96+i) sits in one lane. The sink logit joins only the
// denominator. This kernel is the exact FP32 path and the reference-shaped path for any
// dtype; the tensor-core kernels take the BF16 workloads.
#include "common.cuh"
#include "kernels.cuh"

namespace csa {

constexpr int kTile = 32;
constexpr int kLd = kD + 1;

template <typename ActT, int KV_T>
__device__ __forceinline__ float load_entry(const AttnArgs &a, int64_t row, int c) {
    if (KV_T == CSA_F32) return reinterpret_cast<const float *>(a.c_data)[row * kD + c];
    if (KV_T == CSA_BF16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(a.c_data)[row * kD + c]);
    // MIXED
    if (c < kD / 2)
        return e4m3_to_f32(reinterpret_cast<const uint8_t *>(a.c_data)[row * (kD / 2) + c]) * a.c_scale[row];
    return __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(a.c_rope)[row * (kD / 2) + c - kD / 2]);
}

template <typename ActT, int KV_T>
__global__ void __launch_bounds__(256)
attn_simple_kernel(AttnArgs a) {
    extern __shared__ float sm[];
    float *qs = sm;                  // [H][128]
    float *ks = qs + a.H * kD;       // [32][129]
    __shared__ int s_nc;

    const int b = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int H = a.H;
    int64_t pos, row;
    if (a.decode) {
        pos = (int64_t)a.ctx[b] - 1;
        row = b;
    } else {
        pos = blockIdx.x;
        row = (int64_t)b * a.L + blockIdx.x;
    }
    if (pos < 0 || pos >= a.L) {  // decode ctx_len outside [1, capacity]: record and skip the row
        if (threadIdx.x == 0) set_status(CSA_ERR_BOUNDS);
        return;
    }
    const ActT *q = reinterpret_cast<const ActT *>(a.q) + row * H * kD;
    for (int e = threadIdx.x; e < H * kD; e += 256) qs[e] = to_f(q[e]);
    if (threadIdx.x == 0) {
        int nc;
        if (a.idx) {
            const int32_t *ir = a.idx + row * a.topk;
            nc = a.topk;
            while (nc > 0 && ir[nc - 1] < 0) --nc;  // the kept set is ascending, -1 padded
        } else {
            nc = visible_entries(pos, a.m, a.ncap);
        }
        s_nc = nc;
    }
    __syncthreads();
    const int half = a.d_rope / 2;
    const float2 *rope = reinterpret_cast<const float2 *>(a.rope_tab);
    if (half == 32) {
        for (int e = threadIdx.x; e < H * 32; e += 256) {
            const int h = e >> 5, i = e & 31;
            const float2 cs = rope[pos * 32 + i];
            const float x = qs[h * kD + 64 + i], y = qs[h * kD + 96 + i];
            qs[h * kD + 64 + i] = x * cs.x - y * cs.y;
            qs[h * kD + 96 + i] = x * cs.y + y * cs.x;
        }
    }
    const int nc = s_nc;
    const int ns = (int)min((int64_t)a.n_win, pos + 1);
    const int64_t u0 = pos - ns + 1;
    const int total = nc + ns;
    const int32_t *irow = a.idx ? a.idx + row * a.topk : nullptr;

    constexpr int HPW = 8;  // heads per warp (H <= 64)
    float mrun[HPW], lrun[HPW], o[HPW][4];
#pragma unroll
    for (int i = 0; i < HPW; ++i) {
        mrun[i] = -INFINITY;
        lrun[i] = 0.0f;
        o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.0f;
    }
    __syncthreads();

    for (int kt = 0; kt < total; kt += kTile) {
        for (int e = threadIdx.x; e < kTile * kD; e += 256) {
            const int kk = e / kD, c = e % kD;
            const int i = kt + kk;
            float v = 0.0f;
            if (i < nc) {
                const int j = irow ? irow[i] : i;
                if (j >= 0 && j < a.ncap) v = load_entry<ActT, KV_T>(a, (int64_t)b * a.ncap + j, c);
                else set_status(CSA_ERR_BOUNDS);
            } else if (i < total) {
                const int64_t u = u0 + (i - nc);
                const ActT *src = reinterpret_cast<const ActT *>(a.kv_rope);
                v = a.decode ? to_f(src[((int64_t)b * a.n_win + u % a.n_win) * kD + c])
                             : to_f(src[((int64_t)b * a.L + u) * kD + c]);
            }
            ks[kk * kLd + c] = v;
        }
        __syncthreads();
#pragma unroll
        for (int hi = 0; hi < HPW; ++hi) {
            const int h = warp + 8 * hi;
            if (h >= H) break;
            const float *qh = qs + h * kD;
            const float *kr = ks + lane * kLd;
            float dot = 0.0f;
#pragma unroll 16
            for (int c = 0; c < kD; ++c) dot = fmaf(qh[c], kr[c], dot);
            const float sc = (kt + lane < total) ? dot * a.scale : -INFINITY;
            const float mnew = fmaxf(mrun[hi], warp_max(sc));
            const float corr = expf(mrun[hi] - mnew);
            const float p = expf(sc - mnew);
            lrun[hi] = lrun[hi] * corr + warp_sum(p);
#pragma unroll
            for (int e = 0; e < 4; ++e) o[hi][e] *= corr;
            for (int kk = 0; kk < kTile; ++kk) {
                const float pk = __shfl_sync(0xffffffffu, p, kk);
#pragma unroll
                for (int e = 0; e < 4; ++e) o[hi][e] = fmaf(pk, ks[kk * kLd + lane + 32 * e], o[hi][e]);
            }
            mrun[hi] = mnew;
        }
        __syncthreads();
    }

    ActT *out = reinterpret_cast<ActT *>(a.out) + row * H * kD;
#pragma unroll
    for (int hi = 0; hi < HPW; ++hi) {
        const int h = warp + 8 * hi;
        if (h >= H) break;
        float f;
        if (a.sink) {
            const float s = a.sink[h];
            const float mf = fmaxf(mrun[hi], s);
            const float den = lrun[hi] * expf(mrun[hi] - mf) + expf(s - mf);
            f = expf(mrun[hi] - mf) / den;
        } else {
            f = 1.0f / lrun[hi];
        }
        float v[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) v[e] = o[hi][e] * f;
        if (half == 32) {
            const float2 cs = rope[pos * 32 + lane];
            const float x = v[2], y = v[3];
            v[2] = x * cs.x + y * cs.y;
            v[3] = -x * cs.y + y * cs.x;
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) out[h * kD + lane + 32 * e] = from_f<ActT>(v[e]);
        if (a.lse && lane == 0) a.lse[row * H + h] = mrun[hi] + logf(lrun[hi]);
    }
}

template <typename ActT>
static void launch_attn_a(const AttnArgs &a, cudaStream_t st) {
    dim3 grid(a.decode ? 1 : a.L, a.B);
    const size_t smem = sizeof(float) * ((size_t)a.H * kD + kTile * kLd);
    auto go = [&](auto kern) {
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        kern<<<grid, 256, smem, st>>>(a);
    };
    if (a.kv_t == CSA_F32) go(attn_simple_kernel<ActT, CSA_F32>);
    else if (a.kv_t == CSA_BF16) go(attn_simple_kernel<ActT, CSA_BF16>);
    else go(attn_simple_kernel<ActT, CSA_MIXED>);
}

void launch_attn_simple(const AttnArgs &a, cudaStream_t st) {
    if (a.act_t == CSA_F32) launch_attn_a<float>(a, st);
    else launch_attn_a<__nv_bfloat16>(a, st);
    count_launches(1);
}

}  // namespace csa
