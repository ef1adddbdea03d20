// topk.cu -- per-query top-k selection of indexer scores.
//
// Sources: [P5] "deepseek V4 技术论文" 一.1 CSA (each query attends only to its top-k
// compressed entries); [P4] "EP 95 DeepSeek-V4論文を読む" 17:10 (the indexer picks the top k).
//
// Result of a row with n visible scores: the k highest, ties broken towards the lower index;
// the kept set is written in ascending index order (which also gives the attention gather
// increasing addresses), padded with -1 when n < k. Deterministic: the selection is a
// function of the score bits only.
//
// Scores map to order-preserving 32-bit keys (score_key). One CTA per query row:
//  1. histogram of the top 11 key bits (2048 bins) over the row, read once;
//  2. the bin holding the k-th largest key is found by a suffix scan; every key in a higher
//     bin is kept (a bit in a shared-memory bitmap), the keys of the threshold bin are
//     collected with their indices (second read of the row, normally served by L2);
//  3. an exact radix select over the low 21 bits of the collected keys gives K*, the k-th
//     largest key, and how many keys equal to K* are taken; they are marked in a second
//     bitmap (ties: lowest indices first, applied at emission);
//  4. emission in index order from the two bitmaps with block-wide prefix sums.
// A threshold bin too large for shared memory (heavy exact ties) is resolved by exact radix
// passes over the row in global memory instead. Rows of more than kMaxBitmapN entries use the
// plain four-pass radix select with an ordered compaction.
#include "common.cuh"
#include "kernels.cuh"

namespace csa {

namespace tk {
constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kBins = 2048;            // top 11 key bits
constexpr int kBinShift = 21;
constexpr int kCandCap = 4096;         // keys of the threshold bin kept in shared memory
constexpr int kMaxBitmapN = 1 << 18;   // rows up to this many entries use the bitmap kernel
}  // namespace tk

// ---------------------------------------------------------------------------------------
// block-wide scans (512 threads)
// ---------------------------------------------------------------------------------------

// Exclusive prefix sum of v across the CTA in thread order; *total = sum. Uses s_tmp[kWarps].
__device__ __forceinline__ int block_excl_sum(int v, int *s_tmp, int *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) s_tmp[warp] = x;
    __syncthreads();
    int base = 0, tot = 0;
#pragma unroll
    for (int w = 0; w < tk::kWarps; ++w) {
        const int t = s_tmp[w];
        base += w < warp ? t : 0;
        tot += t;
    }
    __syncthreads();
    *total = tot;
    return base + x - v;
}

// exclusive prefix sum of a 0/1 flag across the CTA (generic kernel)
__device__ __forceinline__ int block_excl_scan(int flag, int *warp_tot, int *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const unsigned bal = __ballot_sync(0xffffffffu, flag);
    const int in_warp = __popc(bal & ((1u << lane) - 1u));
    if (lane == 0) warp_tot[warp] = __popc(bal);
    __syncthreads();
    int base = 0, tot = 0;
    for (int w = 0; w < tk::kWarps; ++w) {
        const int v = warp_tot[w];
        base += (w < warp) ? v : 0;
        tot += v;
    }
    __syncthreads();
    *total = tot;
    return base + in_warp;
}

// Row location for a top-k launch; returns false (and fills the row with -1) for a decode
// position outside [0, L).
__device__ __forceinline__ bool topk_row(const TopkArgs &a, int r, int64_t *t, const float **S, int32_t **out) {
    if (a.decode) {
        *t = (int64_t)a.ctx[r] - 1;
        *S = a.S + (int64_t)r * a.ldS;
        *out = a.out + (int64_t)r * a.k;
    } else {
        *t = (int64_t)a.t0 + r;
        *S = a.S + (int64_t)r * a.ldS;
        *out = a.out + ((int64_t)a.b * a.L + *t) * a.k;
    }
    if (*t < 0 || *t >= a.L) {  // decode ctx_len outside [1, capacity]
        for (int i = threadIdx.x; i < a.k; i += tk::kThreads) (*out)[i] = -1;
        return false;
    }
    return true;
}

// Visits every score of the row once: fn(index, key). float4 loads (rows are 16-byte aligned).
template <typename F>
__device__ __forceinline__ void for_each_key(const float *S, int n, F &&fn) {
    const int n4 = n >> 2;
    const float4 *S4 = reinterpret_cast<const float4 *>(S);
    for (int i4 = threadIdx.x; i4 < n4; i4 += tk::kThreads) {
        const float4 v = __ldcg(S4 + i4);
        fn(4 * i4 + 0, score_key(v.x));
        fn(4 * i4 + 1, score_key(v.y));
        fn(4 * i4 + 2, score_key(v.z));
        fn(4 * i4 + 3, score_key(v.w));
    }
    for (int i = 4 * n4 + threadIdx.x; i < n; i += tk::kThreads) fn(i, score_key(__ldcg(S + i)));
}

// In a histogram of `nbins` bins (nbins / kThreads per thread), finds the bin b holding the
// `want`-th largest element (1-based, counted from the top bin down): *bin = b and
// *above = number of elements in bins above b. Block-wide; every thread gets the result.
__device__ __forceinline__ void find_threshold_bin(const uint32_t *hist, int nbins, int want, int *s_tmp,
                                                   int *s_res, int *bin, int *above) {
    const int per = nbins / tk::kThreads;  // 4 (2048 bins) or 1 (<= 512 bins, padded)
    // thread i owns bins [per*i, per*i + per); reverse order so that an exclusive prefix sum
    // in thread order counts the bins above
    const int owner = tk::kThreads - 1 - threadIdx.x;
    int mine = 0;
    for (int q = 0; q < per; ++q) mine += (int)hist[per * owner + q];
    int tot;
    const int before = block_excl_sum(mine, s_tmp, &tot);  // elements in bins above my range
    if (before < want && before + mine >= want) {
        int run = before;
        for (int q = per - 1; q >= 0; --q) {
            const int h = (int)hist[per * owner + q];
            if (run < want && run + h >= want) {
                s_res[0] = per * owner + q;
                s_res[1] = run;
            }
            run += h;
        }
    }
    __syncthreads();
    *bin = s_res[0];
    *above = s_res[1];
    __syncthreads();
}

// ---------------------------------------------------------------------------------------
// bitmap kernel
// ---------------------------------------------------------------------------------------

__global__ void __launch_bounds__(tk::kThreads) topk_bitmap_kernel(TopkArgs a) {
    using namespace tk;
    extern __shared__ uint32_t dyn[];
    uint32_t *hist = dyn;                              // [kBins]
    uint32_t *cand_key = hist + kBins;                 // [kCandCap]
    int32_t *cand_idx = reinterpret_cast<int32_t *>(cand_key + kCandCap);  // [kCandCap]
    uint32_t *bm_gt = reinterpret_cast<uint32_t *>(cand_idx + kCandCap);  // [nw]
    __shared__ int s_tmp[kWarps];
    __shared__ int s_res[2];
    __shared__ int s_ncand;

    int64_t t;
    const float *S;
    int32_t *out;
    if (!topk_row(a, blockIdx.x, &t, &S, &out)) return;
    const int k = a.k;
    const int n = visible_entries(t, a.m, a.ncap);
    if (n <= k) {
        for (int i = threadIdx.x; i < k; i += kThreads) out[i] = i < n ? i : -1;
        return;
    }
    const int nw = (n + 31) >> 5;
    uint32_t *bm_eq = bm_gt + nw;
    for (int i = threadIdx.x; i < kBins; i += kThreads) hist[i] = 0;
    for (int i = threadIdx.x; i < 2 * nw; i += kThreads) bm_gt[i] = 0;
    if (threadIdx.x == 0) s_ncand = 0;
    __syncthreads();

    // 1. histogram of the top 11 bits
    for_each_key(S, n, [&](int, uint32_t key) { atomicAdd(&hist[key >> kBinShift], 1u); });
    __syncthreads();
    int bstar, above;
    find_threshold_bin(hist, kBins, k, s_tmp, s_res, &bstar, &above);
    int need = k - above;  // keys still to take from bin bstar (>= 1)

    // 2. keys above the bin are kept; keys of the bin are collected
    for_each_key(S, n, [&](int i, uint32_t key) {
        const int bin = (int)(key >> kBinShift);
        if (bin > bstar) {
            atomicOr(&bm_gt[i >> 5], 1u << (i & 31));
        } else if (bin == bstar) {
            const int pos = atomicAdd(&s_ncand, 1);
            if (pos < kCandCap) {
                cand_key[pos] = key;
                cand_idx[pos] = i;
            }
        }
    });
    __syncthreads();
    const int nc = s_ncand;
    uint32_t kstar;
    if (nc <= kCandCap) {
        // 3. exact select inside the bin: low 21 bits in rounds of 7 bits (128 bins)
        uint32_t prefix = (uint32_t)bstar << kBinShift, mask = ~0u << kBinShift;
        for (int round = 0; round < 3; ++round) {
            const int shift = 14 - 7 * round;
            for (int i = threadIdx.x; i < kThreads; i += kThreads) hist[i] = 0;
            __syncthreads();
            for (int c = threadIdx.x; c < nc; c += kThreads) {
                const uint32_t key = cand_key[c];
                if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 127u], 1u);
            }
            __syncthreads();
            int b2, ab2;
            find_threshold_bin(hist, kThreads, need, s_tmp, s_res, &b2, &ab2);  // bins >= 128 are empty
            prefix |= (uint32_t)b2 << shift;
            mask |= 127u << shift;
            need -= ab2;
        }
        kstar = prefix;
        for (int c = threadIdx.x; c < nc; c += kThreads) {
            const uint32_t key = cand_key[c];
            const int i = cand_idx[c];
            if (key > kstar) atomicOr(&bm_gt[i >> 5], 1u << (i & 31));
            else if (key == kstar) atomicOr(&bm_eq[i >> 5], 1u << (i & 31));
        }
    } else {
        // heavy bin: exact radix rounds over the row in global memory (8 + 8 + 5 bits)
        uint32_t prefix = (uint32_t)bstar << kBinShift, mask = ~0u << kBinShift;
        const int shifts[3] = {13, 5, 0};
        const int widths[3] = {8, 8, 5};
        for (int round = 0; round < 3; ++round) {
            const int shift = shifts[round];
            const uint32_t wmask = (1u << widths[round]) - 1u;
            for (int i = threadIdx.x; i < kThreads; i += kThreads) hist[i] = 0;
            __syncthreads();
            for_each_key(S, n, [&](int, uint32_t key) {
                if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & wmask], 1u);
            });
            __syncthreads();
            int b2, ab2;
            find_threshold_bin(hist, kThreads, need, s_tmp, s_res, &b2, &ab2);
            prefix |= (uint32_t)b2 << shift;
            mask |= wmask << shift;
            need -= ab2;
        }
        kstar = prefix;
        for_each_key(S, n, [&](int i, uint32_t key) {
            if ((key >> kBinShift) != (uint32_t)bstar) return;
            if (key > kstar) atomicOr(&bm_gt[i >> 5], 1u << (i & 31));
            else if (key == kstar) atomicOr(&bm_eq[i >> 5], 1u << (i & 31));
        });
    }
    __syncthreads();

    // 4. emission in index order: every gt bit, and the first `need` eq bits
    const int per = (nw + kThreads - 1) / kThreads;
    const int w0 = threadIdx.x * per, w1 = min(nw, w0 + per);
    int my_eq = 0;
    for (int w = w0; w < w1; ++w) my_eq += __popc(bm_eq[w]);
    int tot_eq;
    int eq_before = block_excl_sum(my_eq, s_tmp, &tot_eq);
    int my_sel = 0;
    for (int w = w0; w < w1; ++w) {
        uint32_t e = bm_eq[w];
        const int take = max(0, min(__popc(e), need - eq_before));
        eq_before += __popc(e);
        // keep the lowest `take` set bits of e
        uint32_t kept = 0;
        for (int q = 0; q < take; ++q) {
            const uint32_t low = e & (~e + 1u);
            kept |= low;
            e ^= low;
        }
        bm_eq[w] = kept;
        my_sel += __popc(bm_gt[w] | kept);
    }
    int tot_sel;
    int pos = block_excl_sum(my_sel, s_tmp, &tot_sel);
    for (int w = w0; w < w1; ++w) {
        uint32_t s = bm_gt[w] | bm_eq[w];
        while (s) {
            const int bit = __ffs(s) - 1;
            s &= s - 1u;
            if (pos < k) out[pos] = 32 * w + bit;
            ++pos;
        }
    }
    if (tot_sel != k) set_status(CSA_ERR_BOUNDS);  // cannot happen: the select keeps exactly k
    for (int i = tot_sel + threadIdx.x; i < k; i += kThreads) out[i] = -1;
}

// ---------------------------------------------------------------------------------------
// generic kernel (rows longer than kMaxBitmapN): four 8-bit radix passes over the row and an
// ordered compaction
// ---------------------------------------------------------------------------------------

__global__ void __launch_bounds__(tk::kThreads) topk_radix_kernel(TopkArgs a) {
    using namespace tk;
    __shared__ uint32_t hist[256];
    __shared__ int warp_tot[kWarps];
    __shared__ uint32_t s_sel[2];

    int64_t t;
    const float *S;
    int32_t *out;
    if (!topk_row(a, blockIdx.x, &t, &S, &out)) return;
    const int k = a.k;
    const int n = visible_entries(t, a.m, a.ncap);
    if (n <= k) {
        for (int i = threadIdx.x; i < k; i += kThreads) out[i] = i < n ? i : -1;
        return;
    }
    uint32_t prefix = 0, mask = 0;
    int remaining = k;
    for (int pass = 0; pass < 4; ++pass) {
        const int shift = 24 - 8 * pass;
        for (int i = threadIdx.x; i < 256; i += kThreads) hist[i] = 0;
        __syncthreads();
        for (int i = threadIdx.x; i < n; i += kThreads) {
            const uint32_t key = score_key(S[i]);
            if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1u);
        }
        __syncthreads();
        if (threadIdx.x < 32) {
            const int lane = threadIdx.x;
            uint32_t mine = 0;
#pragma unroll
            for (int q = 0; q < 8; ++q) mine += hist[8 * lane + q];
            uint32_t suffix = 0;
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
    const uint32_t kstar = prefix;
    const int need_eq = remaining;
    int taken_eq = 0, written = 0;
    for (int i0 = 0; i0 < n; i0 += kThreads) {
        const int i = i0 + threadIdx.x;
        uint32_t key = 0;
        if (i < n) key = score_key(S[i]);
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
    for (int i = written + threadIdx.x; i < k; i += kThreads) out[i] = -1;
}

void launch_topk(const TopkArgs &a, cudaStream_t st) {
    using namespace tk;
    if (a.nrows <= 0) return;
    if (a.ncap <= kMaxBitmapN) {
        const int nw = (a.ncap + 31) / 32;
        const size_t smem = sizeof(uint32_t) * ((size_t)kBins + 2 * kCandCap + 2 * (size_t)nw);
        cudaFuncSetAttribute(topk_bitmap_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        topk_bitmap_kernel<<<a.nrows, kThreads, smem, st>>>(a);
    } else {
        topk_radix_kernel<<<a.nrows, kThreads, 0, st>>>(a);
    }
    count_launches(1);
}

}  // namespace csa
