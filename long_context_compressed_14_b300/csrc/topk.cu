// topk.cu -- per-query top-k selection by radix select in shared memory.
//
// Sources: [P5] "deepseek V4 技术论文" 一.1 CSA (each query attends only to its top-k
// compressed entries); [P4] "EP 95 DeepSeek-V4論文を読む" 17:10 (the indexer picks the top k).
//
// Result of a row with n visible scores: the k highest, ties broken towards the lower index;
// the kept set is written in ascending index order (which also gives the attention gather
// increasing addresses), padded with -1 when n < k. Deterministic: the selection is a
// function of the score bits only.
//
// One CTA per query row. Scores map to order-preserving 32-bit keys (score_key); four
// 8-bit radix passes find K*, the k-th largest key, and how many keys equal to K* are
// needed; a final ordered compaction (block-wide prefix sums) emits, in index order, every
// key > K* and the first `need` keys == K*. Rows that fit are staged in shared memory once.
#include "common.cuh"
#include "kernels.cuh"

namespace csa {

constexpr int kTopkThreads = 512;
constexpr int kTopkSmemRow = 12288;  // scores staged in shared memory when n <= this

// exclusive prefix sum of a 0/1 flag across the CTA; returns the prefix, *total = sum.
__device__ __forceinline__ int block_excl_scan(int flag, int *warp_tot, int *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const unsigned bal = __ballot_sync(0xffffffffu, flag);
    const int in_warp = __popc(bal & ((1u << lane) - 1u));
    if (lane == 0) warp_tot[warp] = __popc(bal);
    __syncthreads();
    int base = 0, tot = 0;
    for (int w = 0; w < kTopkThreads / 32; ++w) {
        const int v = warp_tot[w];
        base += (w < warp) ? v : 0;
        tot += v;
    }
    __syncthreads();
    *total = tot;
    return base + in_warp;
}

__global__ void __launch_bounds__(kTopkThreads)
topk_kernel(TopkArgs a) {
    extern __shared__ uint32_t s_keys[];
    __shared__ uint32_t hist[256];
    __shared__ int warp_tot[kTopkThreads / 32];
    __shared__ uint32_t s_sel[2];

    const int r = blockIdx.x;
    int64_t t;
    const float *S;
    int32_t *out;
    if (a.decode) {
        t = (int64_t)a.ctx[r] - 1;
        S = a.S + (int64_t)r * a.ldS;
        out = a.out + (int64_t)r * a.k;
    } else {
        t = (int64_t)a.t0 + r;
        S = a.S + (int64_t)r * a.ldS;
        out = a.out + ((int64_t)a.b * a.L + t) * a.k;
    }
    const int k = a.k;
    if (t < 0 || t >= a.L) {  // decode ctx_len outside [1, capacity]
        for (int i = threadIdx.x; i < k; i += kTopkThreads) out[i] = -1;
        return;
    }
    const int n = visible_entries(t, a.m, a.ncap);
    if (n <= k) {
        for (int i = threadIdx.x; i < k; i += kTopkThreads) out[i] = i < n ? i : -1;
        return;
    }
    const bool staged = n <= kTopkSmemRow;
    if (staged) {
        for (int i = threadIdx.x; i < n; i += kTopkThreads) s_keys[i] = score_key(S[i]);
        __syncthreads();
    }
    uint32_t prefix = 0, mask = 0;
    int remaining = k;
    for (int pass = 0; pass < 4; ++pass) {
        const int shift = 24 - 8 * pass;
        for (int i = threadIdx.x; i < 256; i += kTopkThreads) hist[i] = 0;
        __syncthreads();
        for (int i = threadIdx.x; i < n; i += kTopkThreads) {
            const uint32_t key = staged ? s_keys[i] : score_key(S[i]);
            if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1u);
        }
        __syncthreads();
        if (threadIdx.x < 32) {
            const int lane = threadIdx.x;
            // lane owns bins [8*lane, 8*lane+8); count of keys in bins above this lane's
            uint32_t mine = 0;
#pragma unroll
            for (int q = 0; q < 8; ++q) mine += hist[8 * lane + q];
            uint32_t suffix = 0;  // keys in the bins of lanes above this one
            for (int l2 = 31; l2 >= 0; --l2) {
                const uint32_t v = __shfl_sync(0xffffffffu, mine, l2);
                if (l2 > lane) suffix += v;
            }
            uint32_t run = suffix;
            for (int q = 7; q >= 0; --q) {
                const uint32_t h = hist[8 * lane + q];
                if (run < (uint32_t)remaining && run + h >= (uint32_t)remaining) {
                    s_sel[0] = (uint32_t)(8 * lane + q);
                    s_sel[1] = (uint32_t)remaining - run;
                }
                run += h;
            }
        }
        __syncthreads();
        prefix |= s_sel[0] << shift;
        mask |= 255u << shift;
        remaining = (int)s_sel[1];
        __syncthreads();
    }
    // prefix == K*; `remaining` keys equal to K* are taken, lowest indices first
    const uint32_t kstar = prefix;
    const int need_eq = remaining;
    int taken_eq = 0, written = 0;
    for (int i0 = 0; i0 < n; i0 += kTopkThreads) {
        const int i = i0 + threadIdx.x;
        uint32_t key = 0;
        if (i < n) key = staged ? s_keys[i] : score_key(S[i]);
        const int gt = (i < n) && key > kstar;
        const int eq = (i < n) && key == kstar;
        int tot_eq, tot_keep;
        const int eq_rank = block_excl_scan(eq, warp_tot, &tot_eq);
        const int keep = gt || (eq && taken_eq + eq_rank < need_eq);
        const int pos = block_excl_scan(keep, warp_tot, &tot_keep);
        if (keep) out[written + pos] = i;
        taken_eq += tot_eq;
        written += tot_keep;
        if (written >= k) break;
    }
    for (int i = written + threadIdx.x; i < k; i += kTopkThreads) out[i] = -1;
}

void launch_topk(const TopkArgs &a, cudaStream_t st) {
    const size_t smem = sizeof(uint32_t) * kTopkSmemRow;
    cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    topk_kernel<<<a.nrows, kTopkThreads, smem, st>>>(a);
    count_launches(1);
}

}  // namespace csa
