// index_select.cu -- FP8 lightning-indexer scores with the per-query top-k selection fused in:
// the full score matrix of a prefill (one float per visible (token, entry) pair) is never
// written out.
//
// Sources: [P2] "DeepSeek-V4: Towards Highly Efficient Million-Token Context Intelligence"
// (wiki notes), 提案手法 §1 CSA (a lightning indexer scores every compressed entry for the top-k
// selection, in low precision; it touches every entry, so it has to be light) and 事後学習 §3
// (the indexer's QK path in low precision); [P5] "deepseek V4 技术论文" 一.1 (each query attends
// only to its top-k entries; low-rank, cheap indexer); [P4] "EP 95 DeepSeek-V4論文を読む" 17:10.
//
// Score (FP8 form of sum_h w[t,h] ReLU(qI[t,h] . KI_j) with per-row scales, which are positive
// and leave the ReLU): s(t, j) = sk_j * sum_h (w[t,h] * sq[t,h]) * ReLU(qcode[t,h] . kcode_j).
// Selection: the k highest visible scores of the row, ties to the lower index, written in
// ascending index order and padded with -1.
//
// A chunk of query rows of one sequence takes five launches:
//  1. isel_tc_kernel<kSample>: the scores of every 16th entry tile (entries [16·128·s,
//     16·128·s + 128)), written densely to a sample buffer -- only for query tiles with rows that
//     see more than kCap entries;
//  2. sample_thr_kernel: per row with more than kCap visible entries, the threshold = the
//     ks-th largest sampled score (rounded down to a 22-bit key), ks = the sample's expected
//     share of the row's top k plus six standard deviations plus 4; rows with at most kCap
//     visible entries take all of them (threshold -inf);
//  3. isel_tc_kernel<kFilter>: every visible score on the tensor cores, compared with its row's
//     threshold in the epilogue; (entry, score) pairs at or above it are appended to the row's
//     candidates -- each epilogue warp to its own segment of the row (at most kSeg kept, all
//     counted), in entry order, with the counts in registers (lane q counts token q);
//  4. cand_select_kernel: exact top-k of each row's candidates (radix select on the order keys of
//     the scores, ties to the lower index, emission in index order from bitmaps). A row with
//     fewer than k candidates, or a segment that overflowed, is queued instead;
//  5. isel_fallback_kernel: each queued row's full score row on CUDA cores (float sums of the
//     exact FP8 products) and the exact full-row select.
// The result never depends on the sample being right: when a row holds at least k candidates and
// no segment overflowed, every score above the threshold is among them, so its top k are.
//
// Tensor-core kernel (persistent, one CTA per SM, 576 threads). One MMA tile: D[128 entries]
// [128 columns = TQ tokens x H_I heads] = KI_tile (128 x 64 E4M3) times qI_tile^T, K = 64 as
// two kind::f8f6f4 MMAs of K = 32, FP32 accumulation. Both operands are 64-byte rows with the
// 64-byte swizzle. D has four TMEM buffers of 128 columns; epilogue warpgroup g owns buffer g
// and takes the tiles n = g mod 4 of the CTA's tile sequence, one thread per entry (TMEM lane),
// so the four warpgroups never wait for each other inside a tile. Warp 16 loads query and
// entry tiles by TMA (query tiles double-buffered with their per-token data: w * q_scale,
// threshold, visible count, candidate counters), warp 17 lane 0 issues the MMAs. Query tiles
// are dealt to CTAs heaviest first (the last rows see the most entries); each walks only the
// entry tiles its last token can see. Every wait is bounded; a failure sets the device status,
// raises the abort flag and the CTA frees its TMEM and returns.
#include "common.cuh"
#include "kernels.cuh"
#include "tma_host.cuh"
#include "topk_common.cuh"
#include "umma.cuh"

namespace csa {
using namespace umma;

namespace isel {
constexpr int kWG = 4;                    // epilogue warpgroups = TMEM buffers
constexpr int kEpi = 128 * kWG;           // warps 0-15
constexpr int kEpiWarps = kEpi / 32;
constexpr int kProdWarp = kEpiWarps;      // warp 16: TMA + per-query-tile data
constexpr int kMmaWarp = kEpiWarps + 1;   // warp 17: MMA issue
constexpr int kThreads = kEpi + 64;       // 576
constexpr int kJ = 128;                   // entries per tile (M)
constexpr int kN = 128;                   // (token, head) columns per query tile (N)
constexpr int kNK = 6;                    // entry-tile ring
constexpr int kTileBytes = 128 * 64;      // one operand tile: 128 rows of 64 E4M3 codes
constexpr int kQOff = 0;                  // 2 query tiles
constexpr int kKOff = 2 * kTileBytes;     // kNK entry tiles
constexpr int kSmemBytes = kKOff + kNK * kTileBytes + 1024;
constexpr uint32_t kTmemCols = kWG * kN;  // 512
constexpr int kSample = 0, kFilter = 1;
constexpr int kFbCtas = 296;              // fallback CTAs (each owns one score-row slot)
constexpr size_t kBudget = (size_t)16 << 30;  // workspace bytes per chunk of rows (upper bound)
}  // namespace isel

struct IselTcParams {
    CUtensorMap mq;          // qI codes as [B*L*H_I][64] u8, box 64 x 128, 64-byte swizzle
    CUtensorMap mk;          // KI codes as [B*ncap][64] u8, box 64 x 128, 64-byte swizzle
    const float *q_scale;    // [B*L*H_I]
    const float *k_scale;    // [B*ncap]
    const float *w;          // [B*L*H_I]
    const float *thr;        // filter: [nrows] thresholds
    float *samp;             // sample: [nrows][ld_samp]
    int64_t ld_samp;
    uint2 *cand;             // filter: [nrows][16 warps][kIselSeg] (entry, score bits)
    int *cnt;                // filter: [nrows][16 warps] candidates found (may exceed kIselSeg)
    int L, m, ncap, b, t0, nrows, n_qt;
};

// Shared-memory matrix descriptor with the 64-byte swizzle (layout type 4): rows of 64 bytes,
// 8-row atoms of 512 bytes (stride-dimension offset 512).
__device__ __forceinline__ uint64_t isel_desc_sw64(uint32_t addr) {
    return (uint64_t)((addr >> 4) & 0x3FFFu) | (1ull << 16) | ((uint64_t)(512 >> 4) << 32) | (1ull << 46) |
           (4ull << 61);
}

// Sampled entries visible to a row that sees n entries: the entries of tiles 0, S, 2S, ... below n.
__host__ __device__ __forceinline__ int isel_sample_count(int n) {
    const int span = kIselSampleStride * 128;
    const int full = n / span;  // sample tiles wholly below n
    const int rest = n - full * span;
    return full * 128 + (rest < 128 ? rest : 128);
}

template <int HI, int MODE>
__global__ void __launch_bounds__(isel::kThreads, 1) isel_tc_kernel(const __grid_constant__ IselTcParams P) {
    using namespace isel;
    constexpr int TQ = kN / HI;  // tokens per query tile
    constexpr int CT = 16 / HI;  // tokens per 16-column TMEM chunk
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ __align__(8) uint64_t b_qfull[2], b_qempty[2], b_kfull[kNK], b_kempty[kNK], b_dfull[kWG],
        b_dempty[kWG];
    __shared__ uint32_t tmem_slot;
    __shared__ __align__(16) float s_wq[2][kN];  // w * q_scale / 2 per (token, head) of a query slot
    __shared__ __align__(16) float s_thr[2][TQ]; // per-token thresholds (filter)
    __shared__ __align__(16) int s_nvis[2][TQ];  // entries visible to each token (0 past the chunk)
    __shared__ int s_fin[2];                     // epilogue warps done with a query slot
    __shared__ int s_tq0[2];                     // first token of a query slot

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t s_base = smem_u32(sm);
    if (warp == 0) {
        tmem_alloc(smem_u32(&tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&b_qfull[i]), 1);
            mbar_init(smem_u32(&b_qempty[i]), 2);  // last MMA of the query tile + last epilogue warp
            s_fin[i] = 0;
        }
        for (int i = 0; i < kNK; ++i) {
            mbar_init(smem_u32(&b_kfull[i]), 1);
            mbar_init(smem_u32(&b_kempty[i]), 1);
        }
        for (int i = 0; i < kWG; ++i) {
            mbar_init(smem_u32(&b_dfull[i]), 1);
            mbar_init(smem_u32(&b_dempty[i]), 4);  // one arrival per warp of the owning warpgroup
        }
        mbar_fence_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    const int last_row = P.t0 + P.nrows - 1;
    // i-th query tile of this CTA (heaviest first; < 0 when done) and its number of tile items
    auto qt_of = [&](int i) { return P.n_qt - 1 - ((int)blockIdx.x + i * (int)gridDim.x); };
    auto items_of = [&](int qt) -> int {
        const int tq0 = P.t0 + qt * TQ;
        const int tql = min(tq0 + TQ - 1, last_row);
        const int nv = visible_entries(tql, P.m, P.ncap);
        const int net = (nv + kJ - 1) / kJ;
        if (MODE == kSample) return nv <= kIselCap ? 0 : (net + kIselSampleStride - 1) / kIselSampleStride;
        return net;
    };
    bool ok = true;

    if (warp == kProdWarp) {
        // ---- producer warp: per-query-tile data by all lanes, TMA copies by lane 0 ----
        auto pwait = [&](uint32_t bar, uint32_t par) -> bool {
            return __all_sync(0xffffffffu, mbar_wait(bar, par, kWaitNs, &g_abort));
        };
        int iq = 0, n = 0, q_issued = 0;
        for (int i = 0; ok; ++i) {
            const int qt = qt_of(i);
            if (qt < 0) break;
            const int net = items_of(qt);
            if (net == 0) continue;
            const int qs = iq & 1;
            if (iq >= 2 && !pwait(smem_u32(&b_qempty[qs]), ((iq >> 1) - 1) & 1)) { ok = false; break; }
            const int tq0 = P.t0 + qt * TQ;
            for (int rr = lane; rr < kN; rr += 32) {
                const int tok = tq0 + rr / HI;
                float v = 0.0f;
                if (tok <= last_row) {
                    const int64_t gr = ((int64_t)P.b * P.L + tok) * HI + rr % HI;
                    v = 0.5f * (P.w[gr] * P.q_scale[gr]);  // exact halving: pairs with x + |x| = 2 ReLU(x)
                }
                s_wq[qs][rr] = v;
            }
            if (lane < TQ) {
                const int tok = tq0 + lane;
                const bool in = tok <= last_row;
                s_nvis[qs][lane] = in ? visible_entries(tok, P.m, P.ncap) : 0;
                s_thr[qs][lane] = (MODE == kFilter && in) ? P.thr[tok - P.t0] : INFINITY;
            }
            if (lane == 0) s_tq0[qs] = tq0;
            __syncwarp();
            if (lane == 0) {
                mbar_expect_tx(smem_u32(&b_qfull[qs]), kTileBytes);
                tma_load_3d(s_base + kQOff + qs * kTileBytes, &P.mq, smem_u32(&b_qfull[qs]), 0,
                            (int)(((int64_t)P.b * P.L + tq0) * HI), 0);
            }
            ++q_issued;
            for (int e = 0; e < net; ++e, ++n) {
                const int kb = n % kNK;
                if (n >= kNK && !pwait(smem_u32(&b_kempty[kb]), ((n / kNK) - 1) & 1)) { ok = false; break; }
                const int et = MODE == kSample ? e * kIselSampleStride : e;
                if (lane == 0) {
                    mbar_expect_tx(smem_u32(&b_kfull[kb]), kTileBytes);
                    tma_load_3d(s_base + kKOff + kb * kTileBytes, &P.mk, smem_u32(&b_kfull[kb]), 0,
                                P.b * P.ncap + et * kJ, 0);
                }
            }
            ++iq;
        }
        if (!ok) {
            if (lane == 0) {
                set_timeout();
                // copies still in flight land before the CTA exits (bounded)
                for (int f = max(0, n - kNK); f < n; ++f)
                    mbar_wait(smem_u32(&b_kfull[f % kNK]), (f / kNK) & 1, kDrainNs);
                for (int f = max(0, q_issued - 2); f < q_issued; ++f)
                    mbar_wait(smem_u32(&b_qfull[f & 1]), (f >> 1) & 1, kDrainNs);
            }
            __syncwarp();
        }
    } else if (warp == kMmaWarp) {
        // ---- MMA issue (one thread) ----
        if (lane == 0) {
            const uint32_t idesc = idesc_e4m3(128, kN);
            int iq = 0, n = 0;
            for (int i = 0; ok; ++i) {
                const int qt = qt_of(i);
                if (qt < 0) break;
                const int net = items_of(qt);
                if (net == 0) continue;
                const int qs = iq & 1;
                if (!mbar_wait(smem_u32(&b_qfull[qs]), (iq >> 1) & 1, kWaitNs, &g_abort)) { ok = false; break; }
                for (int e = 0; e < net; ++e, ++n) {
                    const int kb = n % kNK, db = n & 3;
                    if (!mbar_wait(smem_u32(&b_kfull[kb]), (n / kNK) & 1, kWaitNs, &g_abort)) { ok = false; break; }
                    if (n >= kWG && !mbar_wait(smem_u32(&b_dempty[db]), ((n >> 2) - 1) & 1, kWaitNs, &g_abort)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < 2; ++kk)
                        mma_e4m3(tmem + db * kN, isel_desc_sw64(s_base + kKOff + kb * kTileBytes + kk * 32),
                                 isel_desc_sw64(s_base + kQOff + qs * kTileBytes + kk * 32), idesc, kk);
                    mma_commit(smem_u32(&b_dfull[db]));
                    mma_commit(smem_u32(&b_kempty[kb]));
                    if (e == net - 1) mma_commit(smem_u32(&b_qempty[qs]));
                }
                ++iq;
            }
            if (!ok) {
                set_timeout();
                // the MMAs already issued finish (in order) before TMEM is freed
                if (n > 0) mbar_wait(smem_u32(&b_dfull[(n - 1) & 3]), ((n - 1) >> 2) & 1, kDrainNs);
            }
        }
    } else {
        // ---- epilogue: warpgroup g owns TMEM buffer g; thread = entry jl of the tile ----
        const int g = warp >> 2, wl = warp & 3;
        const int jl = 32 * wl + lane;
        const uint32_t tb = tmem + ((uint32_t)(32 * wl) << 16) + g * kN;
        const float *kscale = P.k_scale + (int64_t)P.b * P.ncap;
        const unsigned lt_mask = (1u << lane) - 1u;
        auto wwait = [&](uint32_t bar, uint32_t par) -> bool {
            return __all_sync(0xffffffffu, mbar_wait(bar, par, kWaitNs, &g_abort));
        };
        int iq = 0, n = 0;
        for (int i = 0; ok; ++i) {
            const int qt = qt_of(i);
            if (qt < 0) break;
            const int net = items_of(qt);
            if (net == 0) continue;
            const int qs = iq & 1;
            if (!wwait(smem_u32(&b_qfull[qs]), (iq >> 1) & 1)) { ok = false; break; }
            const int tq0 = s_tq0[qs];
            // filter: this warp's candidates of token q go to its own segment of row q, in entry
            // order; lane q keeps the segment's count (no atomics, no shared state)
            int my_cnt = 0;
            const float4 *wq4 = reinterpret_cast<const float4 *>(s_wq[qs]);
            for (int nn = n + ((g - n) & 3); nn < n + net; nn += kWG) {
                const int e = nn - n;
                const int et = MODE == kSample ? e * kIselSampleStride : e;
                const int j = et * kJ + jl;
                const float sk = j < P.ncap ? __ldg(kscale + j) : 0.0f;
                if (!wwait(smem_u32(&b_dfull[g]), (nn >> 2) & 1)) { ok = false; break; }
                tc_fence_after();
                // scores of the CT tokens of one 16-column chunk from registers r. ReLU(x) * w is
                // formed as (x + |x|) * (w / 2) -- exact, and on the FMA pipe rather than the
                // half-rate ALU pipe that fmax would use. Tiles that every token of the query
                // tile sees in full skip the per-token visibility test.
                const bool full = (et + 1) * kJ * P.m - 1 <= tq0 && tq0 + TQ - 1 <= last_row;
                auto chunk = [&](const uint32_t (&r)[16], int c) {
                    float thr_c[CT];
                    int nv_c[CT];
#pragma unroll
                    for (int qq = 0; qq < CT; ++qq) {
                        thr_c[qq] = s_thr[qs][c * CT + qq];
                        nv_c[qq] = s_nvis[qs][c * CT + qq];
                    }
#pragma unroll
                    for (int qq = 0; qq < CT; ++qq) {
                        const int q = c * CT + qq;
                        uint64_t acc = 0;
#pragma unroll
                        for (int h4 = 0; h4 < HI / 4; ++h4) {
                            const float4 w4 = wq4[(q * HI) / 4 + h4];
                            const uint32_t *x = r + qq * HI + 4 * h4;
                            const float x0 = __uint_as_float(x[0]), x1 = __uint_as_float(x[1]);
                            const float x2 = __uint_as_float(x[2]), x3 = __uint_as_float(x[3]);
                            acc = f2_fma(f2_pack(w4.x, w4.y), f2_pack(x0 + fabsf(x0), x1 + fabsf(x1)), acc);
                            acc = f2_fma(f2_pack(w4.z, w4.w), f2_pack(x2 + fabsf(x2), x3 + fabsf(x3)), acc);
                        }
                        const float2 a2 = f2_unpack(acc);
                        const float s = fmaf(a2.x + a2.y, sk, 0.0f);  // + 0 turns -0 into +0
                        const bool vis = full || j < nv_c[qq];
                        const int64_t row = tq0 + q - P.t0;
                        if (MODE == kSample) {
                            if (vis) P.samp[row * P.ld_samp + e * kJ + jl] = s;
                        } else {
                            const bool hit = vis && s >= thr_c[qq];
                            const unsigned bal = __ballot_sync(0xffffffffu, hit);
                            if (bal != 0u) {
                                const int pos = __shfl_sync(0xffffffffu, my_cnt, q) + __popc(bal & lt_mask);
                                if (hit && pos < kIselSeg)
                                    P.cand[(row * kEpiWarps + warp) * kIselSeg + pos] =
                                        make_uint2((uint32_t)j, __float_as_uint(s));
                                if (lane == q) my_cnt += __popc(bal);
                            }
                        }
                    }
                };
                // eight 16-column chunks, the next one's TMEM load in flight while the current
                // one is computed; the buffer goes back to the MMA once the last is in registers
                uint32_t ra[16], rb[16];
                tmem_ld16_async(tb, ra);
#pragma unroll
                for (int c = 0; c < 8; c += 2) {
                    tmem_wait_hold16(ra);
                    tmem_ld16_async(tb + 16 * (c + 1), rb);
                    chunk(ra, c);
                    tmem_wait_hold16(rb);
                    if (c + 2 < 8) {
                        tmem_ld16_async(tb + 16 * (c + 2), ra);
                    } else {
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(smem_u32(&b_dempty[g]));
                    }
                    chunk(rb, c + 1);
                }
            }
            if (!ok) break;
            if (MODE == kFilter && lane < TQ && tq0 + lane <= last_row)
                P.cnt[(int64_t)(tq0 + lane - P.t0) * kEpiWarps + warp] = my_cnt;
            // this warp is done with the query slot; the last of the 16 warps frees it
            __syncwarp();
            int v = 0;
            if (lane == 0) {
                __threadfence_block();
                v = atomicAdd(&s_fin[qs], 1);
            }
            v = __shfl_sync(0xffffffffu, v, 0);
            if (v == kEpiWarps - 1) {
                if (lane == 0) {
                    s_fin[qs] = 0;
                    mbar_arrive(smem_u32(&b_qempty[qs]));
                }
            }
            n += net;
            ++iq;
        }
        if (!ok && lane == 0) set_timeout();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

// ---------------------------------------------------------------------------------------
// per-row threshold from the sample
// ---------------------------------------------------------------------------------------

struct IselRowArgs {
    const float *samp;
    int64_t ld_samp;
    float *thr;
    const uint2 *cand;
    const int *cnt;
    int *fb_rows;
    int *fb_count;
    int32_t *out;
    float *slots;       // fallback: [kFbCtas][ld_slot] score rows
    int64_t ld_slot;
    const void *qI;     // fallback scoring (codes, scales, weights, keys)
    const float *q_scale;
    const void *KI;
    const float *k_scale;
    const float *w;
    int L, m, ncap, k, b, t0, nrows, H_I;
};

__global__ void __launch_bounds__(tk::kThreads) sample_thr_kernel(IselRowArgs a) {
    using namespace tk;
    __shared__ uint32_t hist[kBins];
    __shared__ int s_tmp[kWarps];
    __shared__ int s_res[2];
    if (blockIdx.x == 0 && threadIdx.x == 0) *a.fb_count = 0;  // the queue of this chunk starts empty
    const int r = blockIdx.x;
    const int64_t t = (int64_t)a.t0 + r;
    const int n = visible_entries(t, a.m, a.ncap);
    if (n <= kIselCap) {
        if (threadIdx.x == 0) a.thr[r] = -INFINITY;
        return;
    }
    const int ns = isel_sample_count(n);
    const float expect = (float)a.k * (float)ns / (float)n;
    const int ks = min(ns, (int)ceilf(expect + 6.0f * sqrtf(expect) + 4.0f));
    const float *sr = a.samp + (int64_t)r * a.ld_samp;
    for (int i = threadIdx.x; i < kBins; i += kThreads) hist[i] = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < ns; i += kThreads) atomicAdd(&hist[key_of(__ldcs(sr + i)) >> kBinShift], 1u);
    __syncthreads();
    int bin, above;
    find_threshold_bin(hist, kBins, ks, s_tmp, s_res, &bin, &above);
    for (int i = threadIdx.x; i < kBins; i += kThreads) hist[i] = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < ns; i += kThreads) {
        const uint32_t key = key_of(__ldcs(sr + i));
        if ((int)(key >> kBinShift) == bin) atomicAdd(&hist[(key >> 10) & (kBins - 1)], 1u);
    }
    __syncthreads();
    int bin2, above2;
    find_threshold_bin(hist, kBins, ks - above, s_tmp, s_res, &bin2, &above2);
    if (threadIdx.x == 0) a.thr[r] = key_floor_value(((uint32_t)bin << kBinShift) | ((uint32_t)bin2 << 10));
}

// ---------------------------------------------------------------------------------------
// exact top-k among a row's candidates
// ---------------------------------------------------------------------------------------

constexpr int kSelPer = kIselCap / tk::kThreads;  // candidates per thread (registers): one per segment
static_assert(kSelPer == 16 && kIselSeg == tk::kThreads, "thread t holds slot t of every segment");

__global__ void __launch_bounds__(tk::kThreads, 5) cand_select_kernel(IselRowArgs a) {
    using namespace tk;
    extern __shared__ uint32_t dyn[];
    uint32_t *hist = dyn;                 // [kBins]
    uint32_t *bm_gt = hist + kBins;       // [nw], then bm_eq [nw]
    __shared__ int s_tmp[kWarps];
    __shared__ int s_res[3];
    const int r = blockIdx.x;
    const int64_t t = (int64_t)a.t0 + r;
    int32_t *out = a.out + ((int64_t)a.b * a.L + t) * a.k;
    const int k = a.k;
    const int n = visible_entries(t, a.m, a.ncap);
    if (n <= k) {
        for (int i = threadIdx.x; i < k; i += kThreads) out[i] = i < n ? i : -1;
        return;
    }
    // the row's candidates: 16 segments (one per filter warp) of up to kIselSeg entries
    const int *wc = a.cnt + (int64_t)r * 16;
    int c = 0;
    bool over = false;
#pragma unroll
    for (int u = 0; u < 16; ++u) {
        c += wc[u];
        over |= wc[u] > kIselSeg;
    }
    if (c < k || over) {  // the threshold misjudged the row: queue it for the exact path
        if (threadIdx.x == 0) a.fb_rows[atomicAdd(a.fb_count, 1)] = r;
        return;
    }
    const int nw = (n + 31) >> 5;
    uint32_t *bm_eq = bm_gt + nw;
    for (int i = threadIdx.x; i < 2 * nw; i += kThreads) bm_gt[i] = 0;
    uint32_t key[kSelPer];
    int32_t idx[kSelPer];
    const uint2 *cl = a.cand + (int64_t)r * kIselCap;
#pragma unroll
    for (int u = 0; u < kSelPer; ++u) {
        const bool live = (int)threadIdx.x < wc[u];
        const uint2 v = live ? __ldcs(cl + u * kIselSeg + threadIdx.x) : make_uint2(0u, 0u);
        key[u] = live ? key_of(__uint_as_float(v.y)) : 0u;
        idx[u] = live ? (int32_t)v.x : -1;
    }
    // radix rounds over the key bits 31..21, 20..10 and 9..0: the k-th largest key K* and how
    // many keys equal to it are taken. A round whose threshold bin is taken whole ends the
    // search: the key bits examined so far (under `mask`) already fix the selection.
    uint32_t prefix = 0, mask = 0;
    int need = k;
#pragma unroll 1
    for (int round = 0; round < 3; ++round) {
        const int shift = round == 0 ? 21 : (round == 1 ? 10 : 0);
        const uint32_t wm = round == 2 ? 1023u : 2047u;
        for (int i = threadIdx.x; i < kBins; i += kThreads) hist[i] = 0;
        __syncthreads();
#pragma unroll
        for (int u = 0; u < kSelPer; ++u)
            if (idx[u] >= 0 && (key[u] & mask) == prefix) atomicAdd(&hist[(key[u] >> shift) & wm], 1u);
        __syncthreads();
        int bb, above, cnt;
        find_threshold_bin(hist, kBins, need, s_tmp, s_res, &bb, &above, &cnt);
        prefix |= (uint32_t)bb << shift;
        mask |= wm << shift;
        need -= above;
        if (cnt == need) break;  // (the same in every thread)
    }
#pragma unroll
    for (int u = 0; u < kSelPer; ++u) {
        if (idx[u] < 0) continue;
        const int i = idx[u];
        const uint32_t km = key[u] & mask;
        if (km > prefix) atomicOr(&bm_gt[i >> 5], 1u << (i & 31));
        else if (km == prefix) atomicOr(&bm_eq[i >> 5], 1u << (i & 31));
    }
    __syncthreads();
    emit_selection(bm_gt, bm_eq, nw, need, k, out, s_tmp);
}

// ---------------------------------------------------------------------------------------
// exact path for the queued rows: full score row on CUDA cores, full-row select
// ---------------------------------------------------------------------------------------

__global__ void __launch_bounds__(tk::kThreads) isel_fallback_kernel(IselRowArgs a) {
    using namespace tk;
    extern __shared__ uint32_t dyn[];
    uint32_t *hist = dyn;                                                   // [kBins]
    uint32_t *cand_key = hist + kBins;                                      // [kCandCap]
    int32_t *cand_idx = reinterpret_cast<int32_t *>(cand_key + kCandCap);  // [kCandCap]
    uint32_t *bm_gt = reinterpret_cast<uint32_t *>(cand_idx + kCandCap);   // [nw], bm_eq [nw]
    __shared__ float q_s[16 * kDI];
    __shared__ float w_s[16];
    __shared__ int s_tmp[kWarps];
    __shared__ int s_res[2];
    __shared__ int s_ncand;
    const int nq = *a.fb_count;
    float *S = a.slots + (int64_t)blockIdx.x * a.ld_slot;
    const int HI = a.H_I;
    for (int qi = blockIdx.x; qi < nq; qi += gridDim.x) {
        const int r = a.fb_rows[qi];
        const int64_t t = (int64_t)a.t0 + r;
        const int n = visible_entries(t, a.m, a.ncap);
        const int64_t qrow = ((int64_t)a.b * a.L + t) * HI;
        __syncthreads();  // the previous row's shared data is no longer read
        for (int e = threadIdx.x; e < HI * kDI; e += kThreads)
            q_s[e] = e4m3_to_f32(reinterpret_cast<const uint8_t *>(a.qI)[qrow * kDI + e]);
        if (threadIdx.x < HI) w_s[threadIdx.x] = a.w[qrow + threadIdx.x] * a.q_scale[qrow + threadIdx.x];
        __syncthreads();
        for (int j = threadIdx.x; j < n; j += kThreads) {
            const int64_t er = (int64_t)a.b * a.ncap + j;
            const uint4 *src = reinterpret_cast<const uint4 *>(reinterpret_cast<const uint8_t *>(a.KI) + er * kDI);
            float kv[kDI];
#pragma unroll
            for (int v = 0; v < kDI / 16; ++v) {
                const uint4 x = src[v];
                const uint32_t wd[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                for (int q = 0; q < 4; ++q)
#pragma unroll
                    for (int e = 0; e < 4; ++e) kv[16 * v + 4 * q + e] = e4m3_to_f32((uint8_t)(wd[q] >> (8 * e)));
            }
            float s = 0.0f;
            for (int h = 0; h < HI; ++h) {
                float acc = 0.0f;
#pragma unroll
                for (int cc = 0; cc < kDI; ++cc) acc = fmaf(q_s[h * kDI + cc], kv[cc], acc);
                s = fmaf(w_s[h], fmaxf(acc, 0.0f), s);
            }
            S[j] = fmaf(s, a.k_scale[er], 0.0f);
        }
        __syncthreads();
        const int nw = (n + 31) >> 5;
        uint32_t *bm_eq = bm_gt + nw;
        for (int i = threadIdx.x; i < 2 * nw; i += kThreads) bm_gt[i] = 0;
        __syncthreads();
        const int need = select_full(S, n, a.k, hist, cand_key, cand_idx, bm_gt, bm_eq, s_tmp, s_res, &s_ncand);
        emit_selection(bm_gt, bm_eq, nw, need, a.k, a.out + ((int64_t)a.b * a.L + t) * a.k, s_tmp);
    }
}

// ---------------------------------------------------------------------------------------
// host
// ---------------------------------------------------------------------------------------

namespace {
inline size_t al256(size_t x) { return (x + 255) / 256 * 256; }
inline int64_t isel_ld_samp(int ncap) {
    const int64_t tiles = (ncap + 127) / 128;
    return (tiles + kIselSampleStride - 1) / kIselSampleStride * 128;
}
inline int64_t isel_ld_slot(int ncap) { return ((int64_t)ncap + 3) / 4 * 4; }
inline size_t isel_row_bytes(int ncap) {
    return sizeof(float) * (size_t)isel_ld_samp(ncap) + sizeof(uint2) * (size_t)kIselCap + 18 * sizeof(int);
}
}  // namespace

int64_t isel_chunk_rows(int L, int ncap) {
    int64_t rows = (int64_t)(isel::kBudget / isel_row_bytes(ncap));
    if (rows >= L) return L;
    rows = rows / 128 * 128;
    return rows < 128 ? 128 : rows;
}

size_t isel_workspace_bytes(int L, int ncap) {
    const size_t R = (size_t)isel_chunk_rows(L, ncap);
    return al256(sizeof(float) * R * (size_t)isel_ld_samp(ncap)) + al256(sizeof(float) * R) +
           al256(sizeof(uint2) * R * kIselCap) + al256(sizeof(int) * R * 16) + al256(sizeof(int) * R) + al256(16) +
           al256(sizeof(float) * (size_t)isel::kFbCtas * (size_t)isel_ld_slot(ncap));
}

bool isel_supported(const IselArgs &a) { return a.H_I == 4 || a.H_I == 8 || a.H_I == 16; }

int launch_index_select(const IselArgs &a, cudaStream_t st) {
    using namespace isel;
    if (!isel_supported(a)) return CSA_ERR_UNSUPPORTED;
    const int64_t R = isel_chunk_rows(a.L, a.ncap);
    char *p = reinterpret_cast<char *>(a.ws);
    auto take = [&](size_t bytes) {
        char *q = p;
        p += al256(bytes);
        return q;
    };
    float *samp = reinterpret_cast<float *>(take(sizeof(float) * R * isel_ld_samp(a.ncap)));
    float *thr = reinterpret_cast<float *>(take(sizeof(float) * R));
    uint2 *cand = reinterpret_cast<uint2 *>(take(sizeof(uint2) * R * kIselCap));
    int *cnt = reinterpret_cast<int *>(take(sizeof(int) * R * 16));
    int *fb_rows = reinterpret_cast<int *>(take(sizeof(int) * R));
    int *fb_count = reinterpret_cast<int *>(take(16));
    float *slots = reinterpret_cast<float *>(take(sizeof(float) * kFbCtas * isel_ld_slot(a.ncap)));

    IselTcParams P;
    memset(&P, 0, sizeof(P));
    const uint64_t qrows = (uint64_t)a.B * a.L * a.H_I;
    bool ok = make_map_3d(&P.mq, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, a.qI, 64, qrows, 1, 64, kN, CU_TENSOR_MAP_SWIZZLE_64B);
    ok = ok && make_map_3d(&P.mk, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, a.KI, 64, (uint64_t)a.B * a.ncap, 1, 64, kJ,
                           CU_TENSOR_MAP_SWIZZLE_64B);
    if (!ok) return CSA_ERR_UNSUPPORTED;
    P.q_scale = a.qI_scale;
    P.k_scale = a.KI_scale;
    P.w = a.w;
    P.thr = thr;
    P.samp = samp;
    P.ld_samp = isel_ld_samp(a.ncap);
    P.cand = cand;
    P.cnt = cnt;
    P.L = a.L; P.m = a.m; P.ncap = a.ncap;
    IselRowArgs ra{};
    ra.samp = samp; ra.ld_samp = P.ld_samp; ra.thr = thr; ra.cand = cand; ra.cnt = cnt;
    ra.fb_rows = fb_rows; ra.fb_count = fb_count; ra.out = a.out; ra.slots = slots;
    ra.ld_slot = isel_ld_slot(a.ncap);
    ra.qI = a.qI; ra.q_scale = a.qI_scale; ra.KI = a.KI; ra.k_scale = a.KI_scale; ra.w = a.w;
    ra.L = a.L; ra.m = a.m; ra.ncap = a.ncap; ra.k = a.k; ra.H_I = a.H_I;

    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int TQ = kN / a.H_I;
    const int nw_max = (a.ncap + 31) / 32;
    const size_t sel_smem = sizeof(uint32_t) * ((size_t)tk::kBins + 2 * (size_t)nw_max);
    const size_t fb_smem = sizeof(uint32_t) * ((size_t)tk::kBins + 2 * (size_t)tk::kCandCap + 2 * (size_t)nw_max);
    cudaFuncSetAttribute(cand_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sel_smem);
    cudaFuncSetAttribute(isel_fallback_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)fb_smem);
    auto tc = [&](auto kern, const IselTcParams &prm, int n_qt) {
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        kern<<<n_qt < sms ? n_qt : sms, kThreads, kSmemBytes, st>>>(prm);
    };
    int launches = 0;
    for (int b = 0; b < a.B; ++b) {
        for (int64_t t0 = 0; t0 < a.L; t0 += R) {
            const int nrows = (int)((a.L - t0) < R ? (a.L - t0) : R);
            const int last_vis = visible_entries(t0 + nrows - 1, a.m, a.ncap);
            ra.b = b; ra.t0 = (int)t0; ra.nrows = nrows;
            if (last_vis <= a.k) {
                // no row of the chunk sees more than k entries: the selection is every visible one
                cand_select_kernel<<<nrows, tk::kThreads, sel_smem, st>>>(ra);
                ++launches;
                continue;
            }
            P.b = b; P.t0 = (int)t0; P.nrows = nrows;
            P.n_qt = (nrows + TQ - 1) / TQ;
            if (last_vis > kIselCap) {
                if (a.H_I == 4) tc(isel_tc_kernel<4, kSample>, P, P.n_qt);
                else if (a.H_I == 8) tc(isel_tc_kernel<8, kSample>, P, P.n_qt);
                else tc(isel_tc_kernel<16, kSample>, P, P.n_qt);
                ++launches;
            }
            sample_thr_kernel<<<nrows, tk::kThreads, 0, st>>>(ra);
            if (a.H_I == 4) tc(isel_tc_kernel<4, kFilter>, P, P.n_qt);
            else if (a.H_I == 8) tc(isel_tc_kernel<8, kFilter>, P, P.n_qt);
            else tc(isel_tc_kernel<16, kFilter>, P, P.n_qt);
            cand_select_kernel<<<nrows, tk::kThreads, sel_smem, st>>>(ra);
            isel_fallback_kernel<<<kFbCtas, tk::kThreads, fb_smem, st>>>(ra);
            launches += 4;
        }
    }
    count_launches(launches);
    return CSA_OK;
}

}  // namespace csa
