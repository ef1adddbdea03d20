// topk_common.cuh -- block-wide pieces of the exact top-k selection shared by the top-k kernels
// (topk.cu) and the fused indexer selection (index_select.cu): block scans, histogram threshold
// search, the order-preserving key of a score, the exact full-row select and the emission of a
// selection in ascending index order from bitmaps. Every routine is block-wide over a CTA of NT
// threads (a template argument, tk::kThreads = 256 unless stated; NT a multiple of 256 up to
// 1024, so that a 2048-bin histogram splits evenly over the threads).
#pragma once

#include "common.cuh"

namespace csa {

namespace tk {
constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kBins = 2048;            // top 11 key bits
constexpr int kBinShift = 21;
constexpr int kCandCap = 3584;         // candidate keys kept in shared memory
constexpr int kMaxBitmapN = 1 << 18;   // rows up to this many entries use the bitmap kernel
}  // namespace tk

// ---------------------------------------------------------------------------------------
// block-wide scans
// ---------------------------------------------------------------------------------------

// Exclusive prefix sum of v across the CTA (NT threads) in thread order; *total = sum. Uses
// s_tmp[NT / 32].
template <int NT = tk::kThreads>
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
    for (int w = 0; w < NT / 32; ++w) {
        const int t = s_tmp[w];
        base += w < warp ? t : 0;
        tot += t;
    }
    __syncthreads();
    *total = tot;
    return base + x - v;
}

// exclusive prefix sum of a 0/1 flag across a CTA of tk::kThreads threads (generic kernel)
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

// Visits every score of the row once: fn(index, key). float4 loads (rows are 16-byte aligned).
template <int NT = tk::kThreads, typename F>
__device__ __forceinline__ void for_each_key(const float *S, int n, F &&fn) {
    const int n4 = n >> 2;
    const float4 *S4 = reinterpret_cast<const float4 *>(S);
    for (int i4 = threadIdx.x; i4 < n4; i4 += NT) {
        const float4 v = __ldcg(S4 + i4);
        fn(4 * i4 + 0, score_key(v.x));
        fn(4 * i4 + 1, score_key(v.y));
        fn(4 * i4 + 2, score_key(v.z));
        fn(4 * i4 + 3, score_key(v.w));
    }
    for (int i = 4 * n4 + threadIdx.x; i < n; i += NT) fn(i, score_key(__ldcg(S + i)));
}

// In a histogram of `nbins` bins (nbins / kThreads per thread), finds the bin b holding the
// `want`-th largest element (1-based, counted from the top bin down): *bin = b and
// *above = number of elements in bins above b; with `count`, also the elements in bin b (s_res
// then needs three ints). Block-wide; every thread gets the result.
template <int NT = tk::kThreads>
__device__ __forceinline__ void find_threshold_bin(const uint32_t *hist, int nbins, int want, int *s_tmp,
                                                   int *s_res, int *bin, int *above, int *count = nullptr) {
    const int per = nbins / NT;  // 4 (2048 bins) or 1 (<= 512 bins, padded)
    // thread i owns bins [per*i, per*i + per); reverse order so that an exclusive prefix sum
    // in thread order counts the bins above
    const int owner = NT - 1 - threadIdx.x;
    int mine = 0;
    for (int q = 0; q < per; ++q) mine += (int)hist[per * owner + q];
    int tot;
    const int before = block_excl_sum<NT>(mine, s_tmp, &tot);  // elements in bins above my range
    if (before < want && before + mine >= want) {
        int run = before;
        for (int q = per - 1; q >= 0; --q) {
            const int h = (int)hist[per * owner + q];
            if (run < want && run + h >= want) {
                s_res[0] = per * owner + q;
                s_res[1] = run;
                if (count) s_res[2] = h;
            }
            run += h;
        }
    }
    __syncthreads();
    *bin = s_res[0];
    *above = s_res[1];
    if (count) *count = s_res[2];
    __syncthreads();
}

// ---------------------------------------------------------------------------------------
// bitmap kernel
// ---------------------------------------------------------------------------------------

// Canonical order key of a score: -0 folded onto +0 by adding +0 (x + 0 = x otherwise), then
// the sign-magnitude bits mapped to an unsigned order (larger score -> larger key).
__device__ __forceinline__ uint32_t key_of(float s) {
    const uint32_t u = __float_as_uint(s + 0.0f);
    return u ^ ((uint32_t)((int32_t)u >> 31) | 0x80000000u);
}

// The smallest float whose key (key_of) is at least `key`: a float v (not NaN) has
// key_of(v) >= key exactly when v >= key_floor_value(key). Keys up to that of -inf give -inf.
__device__ __forceinline__ float key_floor_value(uint32_t key) {
    if (key <= 0x007FFFFFu) return -INFINITY;
    return __uint_as_float((key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key);
}

// Exact k-th largest key among the n scores of the row, by the full histogram path: keys in
// higher bins than the k-th are marked in bm_gt, the threshold bin's keys are collected and
// selected exactly (or, when that bin is too large for shared memory, by radix passes over the
// row). On return bm_gt holds every key > K*, bm_eq every key == K*; the result is the number
// of keys == K* to take (lowest indices first).
// The same when the histogram of the row's top 11 key bits is already known: hist (shared
// memory, kBins counters) holds it on entry and is reused as scratch.
template <int NT = tk::kThreads>
__device__ inline int select_from_hist(const float *S, int n, int k, uint32_t *hist, uint32_t *cand_key,
                                       int32_t *cand_idx, uint32_t *bm_gt, uint32_t *bm_eq, int *s_tmp, int *s_res,
                                       int *s_ncand);

template <int NT = tk::kThreads>
__device__ inline int select_full(const float *S, int n, int k, uint32_t *hist, uint32_t *cand_key, int32_t *cand_idx,
                           uint32_t *bm_gt, uint32_t *bm_eq, int *s_tmp, int *s_res, int *s_ncand) {
    using namespace tk;
    constexpr int kThreads = NT;
    for (int i = threadIdx.x; i < kBins; i += kThreads) hist[i] = 0;
    __syncthreads();
    for_each_key<NT>(S, n, [&](int, uint32_t key) { atomicAdd(&hist[key >> kBinShift], 1u); });
    __syncthreads();
    return select_from_hist<NT>(S, n, k, hist, cand_key, cand_idx, bm_gt, bm_eq, s_tmp, s_res, s_ncand);
}

template <int NT>
__device__ inline int select_from_hist(const float *S, int n, int k, uint32_t *hist, uint32_t *cand_key,
                                       int32_t *cand_idx, uint32_t *bm_gt, uint32_t *bm_eq, int *s_tmp, int *s_res,
                                       int *s_ncand) {
    using namespace tk;
    constexpr int kThreads = NT;
    if (threadIdx.x == 0) *s_ncand = 0;
    int bstar, above;
    find_threshold_bin<NT>(hist, kBins, k, s_tmp, s_res, &bstar, &above);
    int need = k - above;
    for_each_key<NT>(S, n, [&](int i, uint32_t key) {
        const int bin = (int)(key >> kBinShift);
        if (bin > bstar) {
            atomicOr(&bm_gt[i >> 5], 1u << (i & 31));
        } else if (bin == bstar) {
            const int pos = atomicAdd(s_ncand, 1);
            if (pos < kCandCap) {
                cand_key[pos] = key;
                cand_idx[pos] = i;
            }
        }
    });
    __syncthreads();
    const int nc = *s_ncand;
    uint32_t prefix = (uint32_t)bstar << kBinShift, mask = ~0u << kBinShift;
    if (nc <= kCandCap) {
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
            find_threshold_bin<NT>(hist, kThreads, need, s_tmp, s_res, &b2, &ab2);  // bins >= 128 are empty
            prefix |= (uint32_t)b2 << shift;
            mask |= 127u << shift;
            need -= ab2;
        }
        const uint32_t kstar = prefix;
        for (int c = threadIdx.x; c < nc; c += kThreads) {
            const uint32_t key = cand_key[c];
            const int i = cand_idx[c];
            if (key > kstar) atomicOr(&bm_gt[i >> 5], 1u << (i & 31));
            else if (key == kstar) atomicOr(&bm_eq[i >> 5], 1u << (i & 31));
        }
    } else {
        // heavy bin: exact radix rounds over the row in global memory (8 + 8 + 5 bits)
        const int shifts[3] = {13, 5, 0};
        const int widths[3] = {8, 8, 5};
        for (int round = 0; round < 3; ++round) {
            const int shift = shifts[round];
            const uint32_t wmask = (1u << widths[round]) - 1u;
            for (int i = threadIdx.x; i < kThreads; i += kThreads) hist[i] = 0;
            __syncthreads();
            for_each_key<NT>(S, n, [&](int, uint32_t key) {
                if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & wmask], 1u);
            });
            __syncthreads();
            int b2, ab2;
            find_threshold_bin<NT>(hist, kThreads, need, s_tmp, s_res, &b2, &ab2);
            prefix |= (uint32_t)b2 << shift;
            mask |= wmask << shift;
            need -= ab2;
        }
        const uint32_t kstar = prefix;
        for_each_key<NT>(S, n, [&](int i, uint32_t key) {
            if ((key >> kBinShift) != (uint32_t)bstar) return;
            if (key > kstar) atomicOr(&bm_gt[i >> 5], 1u << (i & 31));
            else if (key == kstar) atomicOr(&bm_eq[i >> 5], 1u << (i & 31));
        });
    }
    __syncthreads();
    return need;
}

// Emission in index order from the bitmaps: every gt bit and the first `need` eq bits.
template <int NT = tk::kThreads>
__device__ inline void emit_selection(uint32_t *bm_gt, uint32_t *bm_eq, int nw, int need, int k, int32_t *out, int *s_tmp) {
    using namespace tk;
    constexpr int kThreads = NT;
    const int per = (nw + kThreads - 1) / kThreads;
    const int w0 = threadIdx.x * per, w1 = min(nw, w0 + per);
    int my_eq = 0;
    for (int w = w0; w < w1; ++w) my_eq += __popc(bm_eq[w]);
    int tot_eq;
    int eq_before = block_excl_sum<NT>(my_eq, s_tmp, &tot_eq);
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
    int pos = block_excl_sum<NT>(my_sel, s_tmp, &tot_sel);
    for (int w = w0; w < w1; ++w) {
        uint32_t sl = bm_gt[w] | bm_eq[w];
        while (sl) {
            const int bit = __ffs(sl) - 1;
            sl &= sl - 1u;
            if (pos < k) out[pos] = 32 * w + bit;
            ++pos;
        }
    }
    if (tot_sel != k) set_status(CSA_ERR_BOUNDS);  // cannot happen: the select keeps exactly k
    for (int i = tot_sel + threadIdx.x; i < k; i += kThreads) out[i] = -1;
}

}  // namespace csa
