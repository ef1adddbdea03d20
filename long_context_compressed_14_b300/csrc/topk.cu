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
// Scores map to order-preserving 32-bit keys (-0 folded onto +0). One CTA of 256 threads per
// query row, four CTAs per SM:
//  1. a threshold from a sample of the row (the first 128-byte line of every eight): two
//     2048-bin histograms of the sampled keys (top 11 bits, then the next 11 inside the chosen
//     bin) give a 22-bit key that, with a 4-sigma margin on the sampled count, lies below the
//     k-th largest key;
//  2. one pass over the row, four float4 loads per thread in flight, compares every score with
//     the threshold and writes the indices of those at or above it (normally ~1.4 k) to shared
//     memory;
//  3. an exact radix select over the collected keys (gathered from the row, still in L2),
//     offset by the threshold, gives K*, the k-th largest key, and how many keys equal to K*
//     are taken; keys > K* and keys == K* are marked in two bitmaps;
//  4. emission in index order from the bitmaps with block-wide prefix sums (ties: lowest
//     indices first).
// When the sample misjudges (fewer than k or more than kCandCap keys collected) the exact full
// path runs instead: a histogram of the whole row, the threshold bin's keys collected (or, when
// that bin is too large for shared memory, radix passes over the row), then steps 3-4. Rows of
// more than kMaxBitmapN entries use the plain four-pass radix select with an ordered compaction.
#include "common.cuh"
#include "kernels.cuh"
#include "topk_common.cuh"

namespace csa {

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


// Visits the sampled float4s of a row: the first 128-byte line of every 8 (one eighth of the
// row, whole lines so that the sample costs one eighth of the row's DRAM sectors).
template <typename F>
__device__ __forceinline__ void for_each_sample(const float4 *S4, int n4, F &&fn) {
    for (int s = threadIdx.x;; s += tk::kThreads) {
        const int j = ((s >> 3) << 6) | (s & 7);
        if (j >= n4) break;
        fn(__ldcg(S4 + j));
    }
}
__device__ __forceinline__ int sample_count(int n4) {  // float4s visited by for_each_sample
    return 8 * (n4 >> 6) + min(8, n4 & 63);
}

// Main kernel, one CTA per row.
// A. (rows longer than kCandCap) threshold from the sample: histograms of the sampled keys'
//    top 11 bits and then of the next 11 bits inside the chosen bin give the 22-bit key prefix
//    where the sampled count from the top reaches the scaled k plus a 4-sigma margin.
// B. one pass over the row (four float4 per thread in flight) collects the indices of the
//    scores at or above the threshold into shared memory.
// C. when at least k and at most kCandCap keys were collected, the k-th largest key K* is among
//    them: radix rounds over d = key - threshold (the first round spans the collected range,
//    the next ones the remaining low bits, at most 11 per round) give K* and the number of keys
//    equal to it to take; keys above and equal to K* are marked in two bitmaps. Otherwise the
//    sample misjudged and the exact full path runs.
// D. emission in index order.
__global__ void __launch_bounds__(tk::kThreads, 4) topk_bitmap_kernel(TopkArgs a) {
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
    const int lane = threadIdx.x & 31;
    const int nw = (n + 31) >> 5;
    uint32_t *bm_eq = bm_gt + nw;
    for (int i = threadIdx.x; i < kBins; i += kThreads) hist[i] = 0;
    for (int i = threadIdx.x; i < 2 * nw; i += kThreads) bm_gt[i] = 0;
    if (threadIdx.x == 0) s_ncand = 0;
    __syncthreads();

    const int n4 = n >> 2;
    const float4 *S4 = reinterpret_cast<const float4 *>(S);
    // A. threshold
    uint32_t thr = 0;
    if (n > kCandCap) {
        for_each_sample(S4, n4, [&](float4 v) {
            atomicAdd(&hist[key_of(v.x) >> kBinShift], 1u);
            atomicAdd(&hist[key_of(v.y) >> kBinShift], 1u);
            atomicAdd(&hist[key_of(v.z) >> kBinShift], 1u);
            atomicAdd(&hist[key_of(v.w) >> kBinShift], 1u);
        });
        __syncthreads();
        const int ns = 4 * sample_count(n4);
        const float expect = (float)k * (float)ns / (float)n;
        const int ks = min(ns, (int)ceilf(expect + 4.0f * sqrtf(expect) + 4.0f));
        int bin, above;
        find_threshold_bin(hist, kBins, ks, s_tmp, s_res, &bin, &above);
        for (int i = threadIdx.x; i < kBins; i += kThreads) hist[i] = 0;
        __syncthreads();
        for_each_sample(S4, n4, [&](float4 v) {
            const uint32_t q[4] = {key_of(v.x), key_of(v.y), key_of(v.z), key_of(v.w)};
#pragma unroll
            for (int e = 0; e < 4; ++e)
                if ((int)(q[e] >> kBinShift) == bin) atomicAdd(&hist[(q[e] >> 10) & (kBins - 1)], 1u);
        });
        __syncthreads();
        int bin2, above2;
        find_threshold_bin(hist, kBins, ks - above, s_tmp, s_res, &bin2, &above2);
        thr = ((uint32_t)bin << kBinShift) | ((uint32_t)bin2 << 10);
    }
    // B. collection of the candidate indices. The threshold is compared as a float (the
    // smallest float whose key is thr); each lane covers four float4s per batch as a 16-bit
    // mask, one warp scan of the mask counts gives the positions and only the kept indices are
    // written. Keys are gathered for the candidates afterwards.
    const float thr_f = key_floor_value(thr);
    constexpr int kU = 4;
    for (int i0 = 0; i0 < n4; i0 += kU * kThreads) {
        float4 v[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int i4 = i0 + u * kThreads + threadIdx.x;
            v[u] = i4 < n4 ? __ldcs(S4 + i4) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        }
        uint32_t mask = 0;
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const uint32_t live = (i0 + u * kThreads + threadIdx.x < n4) ? 0xFu : 0u;
            const uint32_t m4 = (v[u].x >= thr_f ? 1u : 0u) | (v[u].y >= thr_f ? 2u : 0u) |
                                (v[u].z >= thr_f ? 4u : 0u) | (v[u].w >= thr_f ? 8u : 0u);
            mask |= (m4 & live) << (4 * u);
        }
        const int c = __popc(mask);
        if (__any_sync(0xffffffffu, c != 0)) {
            int x = c;  // inclusive warp scan of the counts
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, x, o);
                if (lane >= o) x += y;
            }
            int base = 0;
            if (lane == 31) base = atomicAdd(&s_ncand, x);
            int pos = __shfl_sync(0xffffffffu, base, 31) + x - c;
            const int ibase = 4 * (i0 + threadIdx.x);
            while (mask) {
                const int bit = __ffs(mask) - 1;
                mask &= mask - 1u;
                if (pos < kCandCap) cand_idx[pos] = ibase + (bit >> 2) * (4 * kThreads) + (bit & 3);
                ++pos;
            }
        }
    }
    if (threadIdx.x < 32) {  // the last n % 4 scores
        const int i = 4 * n4 + lane;
        const bool keep = i < n && __ldcg(S + i) >= thr_f;
        const unsigned m = __ballot_sync(0xffffffffu, keep);
        if (m != 0u) {
            int base = 0;
            if (lane == 0) base = atomicAdd(&s_ncand, __popc(m));
            const int pos = __shfl_sync(0xffffffffu, base, 0) + __popc(m & ((1u << lane) - 1u));
            if (keep && pos < kCandCap) cand_idx[pos] = i;
        }
    }
    __syncthreads();
    const int nc = s_ncand;
    __syncthreads();  // every thread has read the count before the full path may reset it
    int need;
    if (nc >= k && nc <= kCandCap) {
        // C. exact K* among the candidates, on d = key - thr (every candidate has key >= thr);
        // the candidates' keys are gathered from the row (still in L2)
        uint32_t dmax = 0;
        for (int c = threadIdx.x; c < nc; c += kThreads) {
            const uint32_t key = key_of(__ldcg(S + cand_idx[c]));
            cand_key[c] = key;
            dmax = max(dmax, key - thr);
        }
        dmax = __reduce_max_sync(0xffffffffu, dmax);
        if (lane == 0) s_tmp[threadIdx.x >> 5] = (int)dmax;
        __syncthreads();
        dmax = 0;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) dmax = max(dmax, (uint32_t)s_tmp[w]);
        __syncthreads();
        // round 1 bins d >> shift (< kBins); later rounds take the next <= 11 bits below
        int shift = dmax == 0u ? 0 : max(0, 32 - __clz(dmax) - 11);
        uint32_t prefix = 0, mask = 0, wmask = ~0u;
        need = k;
        while (true) {
            for (int i = threadIdx.x; i < kBins; i += kThreads) hist[i] = 0;
            __syncthreads();
            for (int c = threadIdx.x; c < nc; c += kThreads) {
                const uint32_t d = cand_key[c] - thr;
                if ((d & mask) == prefix) atomicAdd(&hist[(d >> shift) & wmask], 1u);
            }
            __syncthreads();
            int b2, ab2;
            find_threshold_bin(hist, kBins, need, s_tmp, s_res, &b2, &ab2);
            prefix |= (uint32_t)b2 << shift;
            mask |= wmask << shift;
            need -= ab2;
            if (shift == 0) break;
            const int next = max(0, shift - 11);
            wmask = (1u << (shift - next)) - 1u;
            shift = next;
        }
        const uint32_t dstar = prefix;
        for (int c = threadIdx.x; c < nc; c += kThreads) {
            const uint32_t d = cand_key[c] - thr;
            const int i = cand_idx[c];
            if (d > dstar) atomicOr(&bm_gt[i >> 5], 1u << (i & 31));
            else if (d == dstar) atomicOr(&bm_eq[i >> 5], 1u << (i & 31));
        }
        __syncthreads();
    } else {
        // the sample misjudged (too few or too many candidates): exact full path
        need = select_full(S, n, k, hist, cand_key, cand_idx, bm_gt, bm_eq, s_tmp, s_res, &s_ncand);
    }
    // D. emission in index order
    emit_selection(bm_gt, bm_eq, nw, need, k, out, s_tmp);
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

// Decode: one query row per sequence, so one CTA of 1024 threads per row (the rows are few and
// their latency is the step's): the exact full-row select (a histogram of the whole row, the
// threshold bin's keys collected and selected exactly) and emission in index order.
constexpr int kDecTopkThreads = 1024;

__global__ void __launch_bounds__(kDecTopkThreads) decode_topk_kernel(TopkArgs a) {
    using namespace tk;
    extern __shared__ uint32_t dyn[];
    uint32_t *hist = dyn;                                                   // [kBins]
    uint32_t *cand_key = hist + kBins;                                      // [kCandCap]
    int32_t *cand_idx = reinterpret_cast<int32_t *>(cand_key + kCandCap);  // [kCandCap]
    uint32_t *bm_gt = reinterpret_cast<uint32_t *>(cand_idx + kCandCap);   // [nw], bm_eq [nw]
    __shared__ int s_tmp[kDecTopkThreads / 32];
    __shared__ int s_res[2];
    __shared__ int s_ncand;
    const int r = blockIdx.x;
    const int64_t t = (int64_t)a.ctx[r] - 1;
    int32_t *out = a.out + (int64_t)r * a.k;
    const int k = a.k;
    if (t < 0 || t >= a.L) {  // decode ctx_len outside [1, capacity]: reported by the attention
        for (int i = threadIdx.x; i < k; i += kDecTopkThreads) out[i] = -1;
        return;
    }
    const int n = visible_entries(t, a.m, a.ncap);
    if (n <= k) {
        for (int i = threadIdx.x; i < k; i += kDecTopkThreads) out[i] = i < n ? i : -1;
        return;
    }
    const int nw = (n + 31) >> 5;
    uint32_t *bm_eq = bm_gt + nw;
    for (int i = threadIdx.x; i < 2 * nw; i += kDecTopkThreads) bm_gt[i] = 0;
    __syncthreads();
    const float *S = a.S + (int64_t)r * a.ldS;
    int need;
    if (a.hist) {  // the indexer scan already counted the row's keys
        for (int i = threadIdx.x; i < kBins; i += kDecTopkThreads) hist[i] = __ldcg(a.hist + (int64_t)r * kBins + i);
        __syncthreads();
        need = select_from_hist<kDecTopkThreads>(S, n, k, hist, cand_key, cand_idx, bm_gt, bm_eq, s_tmp, s_res,
                                                 &s_ncand);
    } else {
        need = select_full<kDecTopkThreads>(S, n, k, hist, cand_key, cand_idx, bm_gt, bm_eq, s_tmp, s_res, &s_ncand);
    }
    emit_selection<kDecTopkThreads>(bm_gt, bm_eq, nw, need, k, out, s_tmp);
}

// Decode top-k over a known key histogram (the tensor-core indexer scan counts each row's keys)
// in two launches, so that a row is not left to one SM:
//  collect (a number of CTAs per row, each over at most kDecMaxSlice scores): the threshold bin b* of the row's k-th largest key from the
//    histogram (the same in every CTA of the row); each CTA scans one slice of the row and
//    appends the indices of keys above bin b* to the row's `above` list and the (key, index)
//    pairs of keys in bin b* to the row's bin list (positions taken by warp-aggregated atomics;
//    the order does not matter, the selection is emitted in index order);
//  finish (one CTA per row): the exact k-th largest key among the bin's keys, then emission in
//    index order from bitmaps. A bin that overflows its list takes the exact full-row path.
constexpr int kDecBinCap = 4096;
constexpr int kDecMaxSlice = 4096;  // scores per collecting CTA at most (kept in registers)
constexpr int kDecFinishThreads = 512;

__global__ void __launch_bounds__(tk::kThreads) decode_collect_kernel(DecSelArgs a) {
    using namespace tk;
    __shared__ uint32_t hist[kBins];
    __shared__ int s_tmp[kWarps];
    __shared__ int s_res[2];
    pdl_trigger();
    pdl_wait();
    const int r = blockIdx.x / a.slices, g = blockIdx.x % a.slices;
    const int64_t t = (int64_t)a.ctx[r] - 1;
    int32_t *out = a.out + (int64_t)r * a.k;
    const int k = a.k;
    if (t < 0 || t >= a.L) {  // reported by the attention kernel
        if (g == 0)
            for (int i = threadIdx.x; i < k; i += kThreads) out[i] = -1;
        return;
    }
    const int n = visible_entries(t, a.m, a.ncap);
    if (n <= k) {
        if (g == 0)
            for (int i = threadIdx.x; i < k; i += kThreads) out[i] = i < n ? i : -1;
        return;
    }
    const int per = (n + a.slices - 1) / a.slices;
    const int i0 = g * per, i1 = min(n, i0 + per);
    const float *S = a.S + (int64_t)r * a.ldS;
    // the slice's keys stay in registers (loaded first, so that their reads overlap the
    // histogram's): one pass counts (per thread, then a block scan, then one atomic per list per
    // CTA), the second writes at the positions found
    constexpr int kPer = (kDecMaxSlice + kThreads - 1) / kThreads;
    uint32_t key[kPer];
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
        const int i = i0 + u * kThreads + (int)threadIdx.x;
        key[u] = i < i1 ? key_of(__ldcg(S + i)) : 0u;
    }
    for (int i = threadIdx.x; i < kBins; i += kThreads) hist[i] = __ldcg(a.hist + (int64_t)r * kBins + i);
    __syncthreads();
    int bstar, above;
    find_threshold_bin(hist, kBins, k, s_tmp, s_res, &bstar, &above);
    int ngt = 0, neq = 0;
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
        const int i = i0 + u * kThreads + (int)threadIdx.x;
        const int bin = i < i1 ? (int)(key[u] >> kBinShift) : -1;
        ngt += bin > bstar;
        neq += bin == bstar;
    }
    __shared__ int s_base[2];
    int tot_gt, tot_eq;
    int pg = block_excl_sum(ngt, s_tmp, &tot_gt);
    int pe = block_excl_sum(neq, s_tmp, &tot_eq);
    if (threadIdx.x == 0) {
        s_base[0] = tot_gt ? atomicAdd(a.cnt + 2 * r, tot_gt) : 0;
        s_base[1] = tot_eq ? atomicAdd(a.cnt + 2 * r + 1, tot_eq) : 0;
    }
    __syncthreads();
    pg += s_base[0];
    pe += s_base[1];
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
        const int i = i0 + u * kThreads + (int)threadIdx.x;
        if (i >= i1) continue;
        const int bin = (int)(key[u] >> kBinShift);
        if (bin > bstar) {
            if (pg < k) a.above[(int64_t)r * k + pg] = i;
            ++pg;
        } else if (bin == bstar) {
            if (pe < kDecBinCap) a.bin[(int64_t)r * kDecBinCap + pe] = make_uint2(key[u], (uint32_t)i);
            ++pe;
        }
    }
}

__global__ void __launch_bounds__(kDecFinishThreads) decode_finish_kernel(DecSelArgs a) {
    using namespace tk;
    constexpr int NT = kDecFinishThreads;
    pdl_trigger();
    pdl_wait();
    extern __shared__ uint32_t dyn[];
    uint32_t *hist = dyn;                                                    // [kBins]
    uint32_t *cand_key = hist + kBins;                                       // [kDecBinCap]
    int32_t *cand_idx = reinterpret_cast<int32_t *>(cand_key + kDecBinCap);  // [kDecBinCap]
    uint32_t *bm_gt = reinterpret_cast<uint32_t *>(cand_idx + kDecBinCap);   // [nw], bm_eq [nw]
    __shared__ int s_tmp[NT / 32];
    __shared__ int s_res[2];
    __shared__ int s_ncand;
    const int r = blockIdx.x;
    const int64_t t = (int64_t)a.ctx[r] - 1;
    if (t < 0 || t >= a.L) return;
    const int n = visible_entries(t, a.m, a.ncap);
    const int k = a.k;
    if (n <= k) return;  // written by the collect step
    int32_t *out = a.out + (int64_t)r * k;
    const int nw = (n + 31) >> 5;
    uint32_t *bm_eq = bm_gt + nw;
    for (int i = threadIdx.x; i < 2 * nw; i += NT) bm_gt[i] = 0;
    const int n_above = __ldcg(a.cnt + 2 * r), c = __ldcg(a.cnt + 2 * r + 1);
    int need;
    if (c > kDecBinCap || n_above >= k) {
        // the threshold bin holds more keys than the list (heavy ties): exact full-row path
        __syncthreads();
        need = select_full<NT>(a.S + (int64_t)r * a.ldS, n, k, hist, cand_key, cand_idx, bm_gt, bm_eq, s_tmp, s_res,
                               &s_ncand);
    } else {
        for (int i = threadIdx.x; i < c; i += NT) {
            const uint2 v = __ldcg(a.bin + (int64_t)r * kDecBinCap + i);
            cand_key[i] = v.x;
            cand_idx[i] = (int32_t)v.y;
        }
        __syncthreads();
        for (int i = threadIdx.x; i < n_above; i += NT) {
            const int j = __ldcg(a.above + (int64_t)r * k + i);
            atomicOr(&bm_gt[j >> 5], 1u << (j & 31));
        }
        // the bin's keys share their top 11 bits: radix rounds over the low 21 (7 bits each)
        need = k - n_above;
        uint32_t prefix = cand_key[0] & (~0u << kBinShift), mask = ~0u << kBinShift;
        for (int round = 0; round < 3; ++round) {
            const int shift = 14 - 7 * round;
            for (int i = threadIdx.x; i < NT; i += NT) hist[i] = 0;
            __syncthreads();
            for (int i = threadIdx.x; i < c; i += NT) {
                const uint32_t key = cand_key[i];
                if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 127u], 1u);
            }
            __syncthreads();
            int b2, ab2;
            find_threshold_bin<NT>(hist, NT, need, s_tmp, s_res, &b2, &ab2);  // bins >= 128 are empty
            prefix |= (uint32_t)b2 << shift;
            mask |= 127u << shift;
            need -= ab2;
        }
        for (int i = threadIdx.x; i < c; i += NT) {
            const uint32_t key = cand_key[i];
            const int j = cand_idx[i];
            if (key > prefix) atomicOr(&bm_gt[j >> 5], 1u << (j & 31));
            else if (key == prefix) atomicOr(&bm_eq[j >> 5], 1u << (j & 31));
        }
        __syncthreads();
    }
    emit_selection<NT>(bm_gt, bm_eq, nw, need, k, out, s_tmp);
}

// Layout of the selection lists after the two counters per row: the `above` list at
// decode_select_above_off, the bin list at decode_select_bin_off (both 256-byte aligned).
size_t decode_select_above_off(int B) { return ((size_t)B * 2 * sizeof(int) + 255) / 256 * 256; }
size_t decode_select_bin_off(int B, int k) {
    return (decode_select_above_off(B) + (size_t)B * k * sizeof(int32_t) + 255) / 256 * 256;
}
size_t decode_select_bytes(int B, int k) {
    return decode_select_bin_off(B, k) + (size_t)B * kDecBinCap * sizeof(uint2);
}

void launch_decode_select(const DecSelArgs &a, cudaStream_t st) {
    using namespace tk;
    DecSelArgs b = a;
    b.slices = (int)((a.ncap + kDecMaxSlice - 1) / kDecMaxSlice);  // each slice fits the registers
    if (b.slices < 16) b.slices = 16;
    launch_pdl(decode_collect_kernel, a.B * b.slices, kThreads, 0, st, b);
    const int nw = (a.ncap + 31) / 32;
    const size_t smem = sizeof(uint32_t) * ((size_t)kBins + 2 * (size_t)kDecBinCap + 2 * (size_t)nw);
    cudaFuncSetAttribute(decode_finish_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    launch_pdl(decode_finish_kernel, a.B, kDecFinishThreads, smem, st, b);
    count_launches(2);
}

void launch_topk(const TopkArgs &a, cudaStream_t st) {
    using namespace tk;
    if (a.nrows <= 0) return;
    if (a.decode && a.ncap <= kMaxBitmapN) {
        const int nw = (a.ncap + 31) / 32;
        const size_t smem = sizeof(uint32_t) * ((size_t)kBins + 2 * kCandCap + 2 * (size_t)nw);
        cudaFuncSetAttribute(decode_topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        decode_topk_kernel<<<a.nrows, kDecTopkThreads, smem, st>>>(a);
        count_launches(1);
        return;
    }
    if (a.ncap <= kMaxBitmapN) {
        const int nw = (a.ncap + 31) / 32;
        const size_t smem = sizeof(uint32_t) * ((size_t)kBins + 2 * kCandCap + 2 * (size_t)nw);
        cudaFuncSetAttribute(topk_bitmap_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        cudaFuncSetAttribute(topk_bitmap_kernel, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
        topk_bitmap_kernel<<<a.nrows, kThreads, smem, st>>>(a);
    } else {
        topk_radix_kernel<<<a.nrows, kThreads, 0, st>>>(a);
    }
    count_launches(1);
}

}  // namespace csa
