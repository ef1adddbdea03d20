// indexer_tc.cu -- FP8 lightning-indexer scores on the tensor cores (tcgen05 kind::f8f6f4).
//
// Sources: [P2] "DeepSeek-V4: Towards Highly Efficient Million-Token Context Intelligence"
// (wiki notes), 提案手法 §1 CSA (a lightning indexer scores every compressed entry for the
// top-k selection, in low precision) and 事後学習 §3 (the indexer's QK path in low precision);
// [P5] "deepseek V4 技术论文" 一.1 (low-rank, cheap indexer).
//
// s(t, j) = sk_j * sum_h (w[t,h] * sq[t,h]) * ReLU(qcode[t,h] . kcode_j), the FP8 form of
// sum_h w[t,h] ReLU(qI[t,h] . KI_j) with per-row scales (positive, so they leave the ReLU).
//
// One MMA tile: D[128 entries][T_q tokens x H_I heads = 256] = KI_tile (128 x 64 E4M3) times
// qI_tile^T (256 x 64 E4M3), K = 64 as two MMAs of K = 32, FP32 accumulation in TMEM. Both
// operands are 64-byte rows, stored with the 64-byte swizzle (TMA SWIZZLE_64B, descriptor
// layout type 4). Entries sit on the MMA's M dimension so that one epilogue thread owns one
// entry: it reads its accumulators, applies ReLU and the per-head weight, sums the heads of
// each token and stores the token's score -- the 128 threads of a warpgroup write 128
// consecutive entries of one score row at a time.
//
// CTA (persistent, one per SM): warps 0-15 epilogue (four warpgroups, one per quarter of the
// tokens of a query tile), warp 16 lane 0 loads tiles by TMA and issues the MMAs. Query tiles
// are dealt round-robin; each walks only the entry tiles its last token can see (causal
// skipping). D is double-buffered in TMEM (2 x 256 columns), entry tiles flow through a 4-deep
// ring, query tiles through 2 buffers. The load cursor runs ahead of the MMA cursor and only
// blocks on a buffer when no MMA is pending; its other checks are non-blocking.
#include "common.cuh"
#include "kernels.cuh"
#include "tma_host.cuh"
#include "umma.cuh"

namespace csa {
using namespace umma;

namespace idx_tc {
constexpr int kEpiWG = 4;               // epilogue warpgroups
constexpr int kEpi = 128 * kEpiWG;      // epilogue threads (warps 0-15)
constexpr int kMmaWarp = kEpi / 32;     // warp 16: TMA loads + MMA issue
constexpr int kThreads = kEpi + 32;
constexpr int kJ = 128;                 // entries per tile (M)
constexpr int kN = 256;                 // (token, head) rows per query tile (N)
constexpr int kNK = 4;                  // entry-tile ring
constexpr int kKBytes = kJ * 64;        // 8 KB
constexpr int kQBytes = kN * 64;        // 16 KB
constexpr int kQOff = 0;                // 2 query tiles
constexpr int kKOff = 2 * kQBytes;      // kNK entry tiles
constexpr int kSmemBytes = kKOff + kNK * kKBytes + 1024;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kBarEpi = 1;
}  // namespace idx_tc

struct IndexTcParams {
    CUtensorMap mq;  // qI codes as [rows][64] u8, box 64 x 256, 64-byte swizzle
    CUtensorMap mk;  // KI codes as [B*ncap][64] u8, box 64 x 128, 64-byte swizzle
    const float *q_scale;  // [rows of (t, h)]
    const float *k_scale;  // [B*ncap]
    const float *w;        // [rows of (t, h)]
    float *S;
    int64_t ldS;
    int L, m, ncap, b, t0, nrows;
    int n_qt;  // query tiles in this launch
};

// Shared-memory matrix descriptor with the 64-byte swizzle (layout type 4): rows of 64 bytes,
// 8-row atoms of 512 bytes (stride-dimension offset 512).
__device__ __forceinline__ uint64_t sdesc_sw64(uint32_t addr) {
    return (uint64_t)((addr >> 4) & 0x3FFFu) | (1ull << 16) | ((uint64_t)(512 >> 4) << 32) | (1ull << 46) |
           (4ull << 61);
}

template <int HI>
__global__ void __launch_bounds__(idx_tc::kThreads, 1) indexer_tc_kernel(const __grid_constant__ IndexTcParams P) {
    using namespace idx_tc;
    constexpr int TQ = kN / HI;  // tokens per query tile
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ __align__(8) uint64_t b_qfull[2], b_qempty[2], b_kfull[kNK], b_kempty[kNK], b_dfull[2], b_dempty[2];
    __shared__ uint32_t tmem_slot;
    __shared__ __align__(16) float s_wq[kN];  // w * q_scale per (token, head) of the current query tile

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t s_base = smem_u32(sm);
    if (warp == 0) {
        tmem_alloc(smem_u32(&tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&b_qfull[i]), 1);
            mbar_init(smem_u32(&b_qempty[i]), 1);
            mbar_init(smem_u32(&b_dfull[i]), 1);
            mbar_init(smem_u32(&b_dempty[i]), kEpi / 32);  // one arrival per epilogue warp
        }
        for (int i = 0; i < kNK; ++i) {
            mbar_init(smem_u32(&b_kfull[i]), 1);
            mbar_init(smem_u32(&b_kempty[i]), 1);
        }
        mbar_fence_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    const int last_row = P.t0 + P.nrows - 1;
    auto n_et_of = [&](int qt) {
        const int tq0 = P.t0 + qt * TQ;
        const int tq_last = min(tq0 + TQ - 1, last_row);
        return (visible_entries(tq_last, P.m, P.ncap) + kJ - 1) / kJ;
    };
    bool ok = true;

    if (warp == kMmaWarp) {
        if (lane == 0) {
            // ---- producer + MMA issue (one thread) ----
            // Two cursors walk the same item sequence (query tiles of this CTA, each with its
            // visible entry tiles): the load cursor runs up to kNK items ahead of the MMA
            // cursor. It never blocks on a query buffer whose release needs an MMA that has not
            // been issued yet; it only blocks when nothing else can make progress.
            const uint32_t idesc = idesc_e4m3(128, kN);
            int lq = blockIdx.x, le = 0, lqn = 0, ln = 0;  // load cursor (qn counts non-empty tiles)
            int mq = blockIdx.x, me = 0, mqn = 0, mn = 0;  // MMA cursor
            while (lq < P.n_qt && n_et_of(lq) == 0) lq += gridDim.x;
            while (mq < P.n_qt && n_et_of(mq) == 0) mq += gridDim.x;
            while (mq < P.n_qt && ok) {
                while (lq < P.n_qt && ln - mn < kNK) {
                    const int net = n_et_of(lq);
                    const int kb = ln % kNK;
                    if (ln >= kNK) {
                        // the slot's last reader is MMA ln - kNK: block only when no MMA is
                        // pending, otherwise issue MMAs first and come back (checked before the
                        // query load so that nothing is issued twice)
                        const uint32_t par = ((ln / kNK) - 1) & 1;
                        if (ln == mn) {
                            if (!mbar_wait(smem_u32(&b_kempty[kb]), par, kWaitNs, &g_abort)) { ok = false; break; }
                        } else if (!mbar_test_wait(smem_u32(&b_kempty[kb]), par)) {
                            break;
                        }
                    }
                    if (le == 0) {
                        const int qb = lqn & 1;
                        if (lqn >= 2) {
                            const uint32_t par = ((lqn >> 1) - 1) & 1;
                            if (ln == mn) {
                                if (!mbar_wait(smem_u32(&b_qempty[qb]), par, kWaitNs, &g_abort)) { ok = false; break; }
                            } else if (!mbar_test_wait(smem_u32(&b_qempty[qb]), par)) {
                                break;  // do MMA work first
                            }
                        }
                        mbar_expect_tx(smem_u32(&b_qfull[qb]), kQBytes);
                        tma_load_3d(s_base + kQOff + qb * kQBytes, &P.mq, smem_u32(&b_qfull[qb]), 0,
                                    (int)(((int64_t)P.b * P.L + P.t0 + lq * TQ) * HI), 0);
                    }
                    mbar_expect_tx(smem_u32(&b_kfull[kb]), kKBytes);
                    tma_load_3d(s_base + kKOff + kb * kKBytes, &P.mk, smem_u32(&b_kfull[kb]), 0, P.b * P.ncap + le * kJ, 0);
                    ++ln;
                    if (++le == net) {
                        le = 0;
                        ++lqn;
                        do { lq += gridDim.x; } while (lq < P.n_qt && n_et_of(lq) == 0);
                    }
                }
                if (!ok) break;
                const int net = n_et_of(mq);
                const int qb = mqn & 1, kb = mn % kNK, db = mn & 1;
                if (me == 0 && !mbar_wait(smem_u32(&b_qfull[qb]), (mqn >> 1) & 1, kWaitNs, &g_abort)) { ok = false; break; }
                if (!mbar_wait(smem_u32(&b_kfull[kb]), (mn / kNK) & 1, kWaitNs, &g_abort)) { ok = false; break; }
                if (mn >= 2 && !mbar_wait(smem_u32(&b_dempty[db]), ((mn >> 1) - 1) & 1, kWaitNs, &g_abort)) { ok = false; break; }
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 2; ++kk)
                    mma_e4m3(tmem + db * kN, sdesc_sw64(s_base + kKOff + kb * kKBytes + kk * 32),
                             sdesc_sw64(s_base + kQOff + qb * kQBytes + kk * 32), idesc, kk);
                mma_commit(smem_u32(&b_dfull[db]));
                mma_commit(smem_u32(&b_kempty[kb]));
                if (me == net - 1) mma_commit(smem_u32(&b_qempty[qb]));
                ++mn;
                if (++me == net) {
                    me = 0;
                    ++mqn;
                    do { mq += gridDim.x; } while (mq < P.n_qt && n_et_of(mq) == 0);
                }
            }
            if (!ok) set_timeout();
        }
    } else {
        // ---- epilogue: warpgroup g = warp / 4 takes the columns [g*C, (g+1)*C) of D, i.e.
        // tokens [g*C/HI, (g+1)*C/HI) of the query tile; thread = one entry of the tile. The C
        // columns are read as two halves of 32: the second half's TMEM load and the next tile's
        // first half are in flight while the tokens of the half already in registers are
        // computed, and the entry scales are fetched one tile ahead. Warps only meet at the end
        // of a query tile; a failed wait is a warp-uniform decision ----
        constexpr int C = kN / kEpiWG;  // 64 columns
        constexpr int TW = C / HI;      // tokens per warpgroup
        constexpr int TH = TW / 2;      // tokens per 32-column half
        const int g = warp >> 2;
        const uint32_t tcol = tmem + ((uint32_t)(32 * (warp & 3)) << 16) + g * C;
        const float *kscale = P.k_scale + (int64_t)P.b * P.ncap;
        const int jl = 32 * (warp & 3) + lane;  // this thread's entry within a tile
        auto wwait = [&](uint32_t bar, uint32_t par) -> bool {
            return __all_sync(0xffffffffu, mbar_wait(bar, par, kWaitNs, &g_abort));
        };
        int n = 0;
        for (int qt = blockIdx.x; qt < P.n_qt && ok; qt += gridDim.x) {
            const int tq0 = P.t0 + qt * TQ;
            const int n_et = n_et_of(qt);
            if (n_et == 0) continue;
            // per (token, head) weights of this query tile (rows past the chunk weigh 0)
            for (int rr = tid; rr < kN; rr += kEpi) {  // rr = token * HI + head
                const int tok = tq0 + rr / HI;
                float v = 0.0f;
                if (tok <= last_row) {
                    const int64_t gr = ((int64_t)P.b * P.L + tok) * HI + rr % HI;
                    v = P.w[gr] * P.q_scale[gr];
                }
                s_wq[rr] = v;
            }
            named_sync(kBarEpi, kEpi);
            const int t_g = tq0 + g * TW;  // first token of this warpgroup
            float *srow0 = P.S + (int64_t)(t_g - P.t0) * P.ldS;
            const float4 *wq4 = reinterpret_cast<const float4 *>(s_wq + g * TW * HI);
            // scores of tokens [q0, q0 + TH) of entry j from one 32-column half; the heads are
            // summed as two interleaved partial sums (even and odd heads) in packed FP32 pairs.
            // `full`: every token of the warpgroup sees the whole tile and lies in the chunk
            auto tokens = [&](const uint32_t (&r)[32], int q0, int j, float sk, bool full) {
                const int t_first = (j + 1) * P.m - 1;  // first token that sees entry j
                float *dst = srow0 + (int64_t)q0 * P.ldS + j;
#pragma unroll
                for (int q = 0; q < TH; ++q) {
                    const int t = t_g + q0 + q;
                    uint64_t acc = 0;
#pragma unroll
                    for (int h4 = 0; h4 < HI / 4; ++h4) {
                        const float4 w4 = wq4[((q0 + q) * HI) / 4 + h4];
                        const uint32_t *x = r + q * HI + 4 * h4;
                        acc = f2_fma(f2_pack(w4.x, w4.y),
                                     f2_pack(fmaxf(__uint_as_float(x[0]), 0.0f), fmaxf(__uint_as_float(x[1]), 0.0f)), acc);
                        acc = f2_fma(f2_pack(w4.z, w4.w),
                                     f2_pack(fmaxf(__uint_as_float(x[2]), 0.0f), fmaxf(__uint_as_float(x[3]), 0.0f)), acc);
                    }
                    const float2 a2 = f2_unpack(acc);
                    const float s = fmaf(a2.x + a2.y, sk, 0.0f);  // + 0 turns -0 into +0
                    if (full || (t >= t_first && t <= last_row)) *dst = s;
                    dst += P.ldS;
                }
            };
            uint32_t ra[32], rb[32];
            float sk_next = jl < P.ncap ? kscale[jl] : 0.0f;
            if (wwait(smem_u32(&b_dfull[n & 1]), (n >> 1) & 1)) {
                tc_fence_after();
                tmem_ld32_async(tcol + (n & 1) * kN, ra);
            } else {
                ok = false;
                if (lane == 0) set_timeout();
            }
            for (int et = 0; et < n_et && ok; ++et, ++n) {
                const int db = n & 1;
                const int j = et * kJ + jl;
                const float sk = sk_next;
                // the last entry of the tile is visible to the warpgroup's first token
                const bool full = ((et + 1) * kJ) * P.m - 1 <= t_g && t_g + TW - 1 <= last_row;
                if (et + 1 < n_et) sk_next = j + kJ < P.ncap ? kscale[j + kJ] : 0.0f;
                tmem_wait_hold32(ra);
                tmem_ld32_async(tcol + db * kN + 32, rb);
                tokens(ra, 0, j, sk, full);
                tmem_wait_hold32(rb);
                // both halves are in registers: hand the TMEM buffer back to the MMA
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&b_dempty[db]));
                if (et + 1 < n_et) {
                    if (wwait(smem_u32(&b_dfull[db ^ 1]), ((n + 1) >> 1) & 1)) {
                        tc_fence_after();
                        tmem_ld32_async(tcol + (db ^ 1) * kN, ra);
                    } else {
                        ok = false;
                        if (lane == 0) set_timeout();
                    }
                }
                tokens(rb, TH, j, sk, full);
            }
            // s_wq is rewritten for the next query tile; a failure anywhere stops every warp
            ok = !named_sync_or(kBarEpi, kEpi, !ok);
        }
        if (!ok && tid == 0) set_timeout();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

bool launch_indexer_tc(const IndexArgs &a, cudaStream_t st) {
    using namespace idx_tc;
    if (a.decode || a.idx_t != CSA_FP8E4M3) return false;
    if (a.H_I != 4 && a.H_I != 8 && a.H_I != 16) return false;
    IndexTcParams P;
    memset(&P, 0, sizeof(P));
    const int TQ = kN / a.H_I;
    const uint64_t qrows = (uint64_t)a.B * a.L * a.H_I;
    bool ok = make_map_3d(&P.mq, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, a.qI, 64, qrows, 1, 64, kN,
                          CU_TENSOR_MAP_SWIZZLE_64B);
    ok = ok && make_map_3d(&P.mk, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, a.KI, 64, (uint64_t)a.B * a.ncap, 1, 64, kJ,
                           CU_TENSOR_MAP_SWIZZLE_64B);
    if (!ok) return false;
    P.q_scale = a.qI_scale;
    P.k_scale = a.KI_scale;
    P.w = a.w;
    P.S = a.S;
    P.ldS = a.ldS;
    P.L = a.L; P.m = a.m; P.ncap = a.ncap; P.b = a.b; P.t0 = a.t0; P.nrows = a.nrows;
    P.n_qt = (a.nrows + TQ - 1) / TQ;
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int grid = P.n_qt < sms ? P.n_qt : sms;
    auto go = [&](auto kern) {
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        kern<<<grid, kThreads, kSmemBytes, st>>>(P);
    };
    if (a.H_I == 4) go(indexer_tc_kernel<4>);
    else if (a.H_I == 8) go(indexer_tc_kernel<8>);
    else go(indexer_tc_kernel<16>);
    count_launches(1);
    return true;
}

}  // namespace csa
