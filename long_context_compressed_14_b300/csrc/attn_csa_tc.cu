// attn_csa_tc.cu -- CSA sparse attention on the 5th-generation tensor cores (tcgen05 + TMEM).
//
// Sources: [P2] "DeepSeek-V4: Towards Highly Efficient Million-Token Context Intelligence"
// (wiki notes), 提案手法 §1 (CSA: each query attends to its top-k compressed entries;
// shared-KV multi-query attention; sliding-window branch n_win = 128; attention sink;
// partial RoPE + inverse RoPE on the core output) and 訓練インフラの革新 §5 (mixed-precision
// entries); [P5] "deepseek V4 技术论文" 一.1 (an entry is both key and value).
//
// Every token has its own key list: its top-k entries (ascending, gathered by index) followed
// by the 128 raw rows of its window. All 64 heads of a token share that list, so the kernel
// puts the KEYS on the MMA's M dimension and the heads on N:
//   S^T[key, head] = K Q^T     (M = 128 keys, N = 64 heads, K = 128 dims)
//   O^T[dim, head] += V^T P^T  (M = 128 dims, N = 64 heads, K = 128 keys)
// which keeps both MMAs at M = 128 (full tensor-core rate). The key tile is one shared-memory
// buffer read as the K-major A operand of the first MMA and, through an MN-major descriptor,
// as V^T for the second; P^T is written by the softmax threads as 128-byte key rows and read as
// an MN-major B operand.
//
// One softmax thread owns one key (TMEM lane) and holds its 64 head logits; the per-head
// running max is shared across the 128 keys of a tile. It is kept lazily: a tile only triggers
// a CTA-wide max reduction when some logit exceeds the current max by more than 8 (log2
// units), which in practice happens on a token's first tile; O^T (in TMEM) and the partial
// sums are rescaled only then. Per-head sums are partial per thread and reduced once per
// token.
//
// Warp roles (256 threads, persistent over tokens):
//   warps 0-3  softmax and epilogue (they own TMEM lanes 0-127);
//   warp 4     MMA issue (one thread);
//   warps 5-7  producers: query rows by TMA + RoPE, top-k row, key tiles gathered with
//              cp.async (mixed entries: the FP8 half widened to BF16 by the threads), the
//              window tile by TMA (prefill) or gathered from the ring (decode).
// Pipelines: key tiles in a 3-buffer ring, S^T double-buffered in TMEM, P^T double-buffered in
// shared memory, query rows double-buffered; every wait is bounded.
#include "common.cuh"
#include "kernels.cuh"
#include "tma_host.cuh"
#include "umma.cuh"

namespace csa {
using namespace umma;

namespace csa_tc {
constexpr int kThreads = 256;
constexpr int kSoftmax = 128;                 // warps 0-3
constexpr int kMmaWarp = 4;
constexpr int kProd0 = 160;                   // first producer thread (warp 5)
constexpr int kProducers = 96;                // warps 5-7
constexpr int kH = 64;                        // heads (N of both MMAs)
constexpr int kTile = 128;                    // keys per tile
constexpr int kNB = 3;                        // key-tile buffers
constexpr int kQOff = 0;                      // Q: 2 buffers x 16 KB (two 64-dim halves of 8 KB)
constexpr int kKOff = 32768;                  // keys: kNB x 32 KB (two 64-dim halves of 16 KB)
constexpr int kPOff = kKOff + kNB * 32768;    // P^T: 2 x 16 KB
constexpr int kOsOff = kPOff + 2 * 16384;     // epilogue staging [64 heads][128 dims] float
constexpr int kIdxOff = kOsOff + 32768;       // top-k rows: 2 x kMaxTopk int32
constexpr int kSmemBytes = kIdxOff + 2 * kMaxTopk * 4 + 1024;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kOCol = 0;                 // O^T: columns [0, 64)
constexpr uint32_t kSCol = 64;                // S^T slots: [64, 128) and [128, 192)
constexpr float kRescaleThreshold = 8.0f;
// named barriers (0 is __syncthreads)
constexpr uint32_t kBarSoftmax = 1, kBarProd = 2;
}  // namespace csa_tc

struct CsaTcParams {
    CUtensorMap mq;    // q rows [rows*64][128] bf16, box 64 x 64
    CUtensorMap mkv;   // prefill: kv_rope [B][L][128] bf16, box 64 x 128
    const void *c_data;
    const __nv_bfloat16 *c_rope;
    const float *c_scale;
    const __nv_bfloat16 *win;   // decode: ring [B][n_win][128]
    const int32_t *idx;         // [rows][topk]
    const int32_t *ctx;         // decode: [B]
    const float *sink;
    const float2 *rope;
    __nv_bfloat16 *out;
    float *lse;
    int B, L, ncap, topk, n_win, d_rope, mixed, decode, rows;
    float scale_log2;
};

namespace {

struct TokenMeta {
    int n_sel;   // valid top-k entries
    int n_ct;    // compressed tiles
    int t;       // query position
    int b;       // sequence
    int n_win_t; // window rows that exist (<= n_win)
};

__device__ __forceinline__ uint32_t pack2(float a, float b) {
    __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&v);
}

}  // namespace

__global__ void __launch_bounds__(csa_tc::kThreads, 1) csa_tc_kernel(const __grid_constant__ CsaTcParams P) {
    using namespace csa_tc;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    // mbarriers
    __shared__ __align__(8) uint64_t b_qraw[2], b_qfull[2], b_qempty[2];
    __shared__ __align__(8) uint64_t b_kfull[kNB], b_kempty[kNB];
    __shared__ __align__(8) uint64_t b_sfull[2], b_sempty[2], b_pfull[2], b_pempty[2];
    __shared__ __align__(8) uint64_t b_ofull, b_oempty;
    __shared__ uint32_t tmem_slot;
    __shared__ TokenMeta meta[2];
    __shared__ float s_m[kH];          // running max per head (log2 units)
    __shared__ float s_f[kH];          // rescale factor per head of the current update
    __shared__ float s_red[4][kH];     // cross-warp reduction scratch
    __shared__ float s_fo[kH];         // final output factor per head
    __shared__ int s_cnt[3];           // producer warps' counts of valid top-k entries

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t s_base = smem_u32(sm);
    const int n_tok_cta = (P.rows - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x;

    if (warp == 0) {
        tmem_alloc(smem_u32(&tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&b_qraw[i]), 1);
            mbar_init(smem_u32(&b_qfull[i]), kProducers);
            // query slot free: the last S^T MMA of its token is done (commit) and the softmax
            // group has copied the token's metadata (128 arrivals)
            mbar_init(smem_u32(&b_qempty[i]), 1 + kSoftmax);
            mbar_init(smem_u32(&b_sfull[i]), 1);
            mbar_init(smem_u32(&b_sempty[i]), kSoftmax);
            mbar_init(smem_u32(&b_pfull[i]), kSoftmax);
            mbar_init(smem_u32(&b_pempty[i]), 1);
        }
        for (int i = 0; i < kNB; ++i) {
            mbar_init(smem_u32(&b_kfull[i]), kProducers);
            mbar_init(smem_u32(&b_kempty[i]), 1);
        }
        mbar_init(smem_u32(&b_ofull), 1);
        mbar_init(smem_u32(&b_oempty), kSoftmax);
        mbar_fence_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    bool ok = true;

    if (tid >= kProd0) {
        // =============================== producers ===============================
        const int ptid = tid - kProd0;
        // a wait whose outcome is the same for all producer threads (a timeout in one makes
        // them all leave together, so no named barrier is left short of threads)
        auto pwait = [&](uint32_t bar, uint32_t par) -> bool {
            const bool w = mbar_wait(bar, par, kMaxPolls, &g_abort);
            return !named_sync_or(kBarProd, kProducers, !w);
        };
        int n = 0;           // global tile item counter
        int pending = -1;    // item whose k_full arrival is outstanding
        // Fetch of a token's top-k row (bulk copy) and query rows (TMA) into slot it & 1, issued
        // by one thread as early as the slot is free, so it overlaps the previous token.
        auto fetch = [&](int it2) {
            const int row2 = (int)blockIdx.x + it2 * (int)gridDim.x;
            const int qs2 = it2 & 1;
            const uint32_t qb = smem_u32(&b_qraw[qs2]);
            mbar_expect_tx(qb, 2 * kH * 128 + P.topk * 4);
            bulk_load(s_base + kIdxOff + qs2 * kMaxTopk * 4, P.idx + (int64_t)row2 * P.topk, P.topk * 4, qb);
            tma_load_3d(s_base + kQOff + qs2 * 16384, &P.mq, qb, 0, row2 * kH, 0);
            tma_load_3d(s_base + kQOff + qs2 * 16384 + 8192, &P.mq, qb, 64, row2 * kH, 0);
        };
        int fetched = 0;  // tokens whose fetch has been issued
        if (ptid == 0 && n_tok_cta > 0) {
            fetch(0);
            fetched = 1;
        }
        for (int it = 0; it < n_tok_cta && ok; ++it) {
            const int row = (int)blockIdx.x + it * (int)gridDim.x;
            const int qs = it & 1;
            // flush the previous item before the per-token work
            if (pending >= 0) {
                cp_async_wait_all();
                fence_async_smem();
                mbar_arrive(smem_u32(&b_kfull[pending % kNB]));
                pending = -1;
            }
            if (ptid == 0 && fetched == it) {  // not prefetched: the slot must be free first
                if (it >= 2 && !mbar_wait(smem_u32(&b_qempty[qs]), ((it >> 1) - 1) & 1, kMaxPolls, &g_abort)) ok = false;
                if (ok) {
                    fetch(it);
                    fetched = it + 1;
                }
            }
            if (named_sync_or(kBarProd, kProducers, !ok)) { ok = false; break; }
            int b, t;
            if (P.decode) {
                b = row;
                t = P.ctx[b] - 1;
            } else {
                b = row / P.L;
                t = row % P.L;
            }
            const bool pos_ok = t >= 0 && t < P.L;
            if (!pwait(smem_u32(&b_qraw[qs]), (it >> 1) & 1)) { ok = false; break; }
            // count the valid prefix of the top-k row (ascending, -1 padded) in parallel
            int32_t *sidx = reinterpret_cast<int32_t *>(sm + kIdxOff) + qs * kMaxTopk;
            int cnt = 0;
            for (int i = ptid; i < P.topk; i += kProducers) cnt += (pos_ok && sidx[i] >= 0) ? 1 : 0;
            cnt = __reduce_add_sync(0xffffffffu, cnt);
            if ((ptid & 31) == 0) s_cnt[(tid - kProd0) >> 5] = cnt;
            named_sync(kBarProd, kProducers);
            TokenMeta mt;
            mt.n_sel = s_cnt[0] + s_cnt[1] + s_cnt[2];
            mt.n_ct = (mt.n_sel + kTile - 1) / kTile;
            mt.t = t;
            mt.b = b;
            mt.n_win_t = pos_ok ? min(P.n_win, t + 1) : 0;
            if (ptid == 0) meta[qs] = mt;
            // RoPE on dims 64..127 at position t: head h, chunk pair (c, c+4) of the second half
            if (P.d_rope == 64 && pos_ok) {
                uint8_t *q1 = sm + kQOff + qs * 16384 + 8192;
                for (int u = ptid; u < kH * 4; u += kProducers) {
                    const int h = u >> 2, c = u & 3;
                    uint4 *pa = reinterpret_cast<uint4 *>(q1 + sw128_off(h, c));
                    uint4 *pb = reinterpret_cast<uint4 *>(q1 + sw128_off(h, c + 4));
                    uint4 va = *pa, vb = *pb;
                    __nv_bfloat162 *a2 = reinterpret_cast<__nv_bfloat162 *>(&va);
                    __nv_bfloat162 *b2 = reinterpret_cast<__nv_bfloat162 *>(&vb);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 x = __bfloat1622float2(a2[e]);
                        const float2 y = __bfloat1622float2(b2[e]);
                        const float2 c0 = P.rope[(int64_t)t * 32 + 8 * c + 2 * e];
                        const float2 c1 = P.rope[(int64_t)t * 32 + 8 * c + 2 * e + 1];
                        a2[e] = __floats2bfloat162_rn(x.x * c0.x - y.x * c0.y, x.y * c1.x - y.y * c1.y);
                        b2[e] = __floats2bfloat162_rn(x.x * c0.y + y.x * c0.x, x.y * c1.y + y.y * c1.x);
                    }
                    *pa = va;
                    *pb = vb;
                }
            }
            fence_async_smem();
            mbar_arrive(smem_u32(&b_qfull[qs]));
            // key tiles: compressed tiles, then the window tile
            const int n_tiles = mt.n_ct + 1;
            for (int c = 0; c < n_tiles; ++c, ++n) {
                const int kb = n % kNB;
                if (n >= kNB && !pwait(smem_u32(&b_kempty[kb]), ((n / kNB) - 1) & 1)) {
                    ok = false;
                    break;
                }
                uint8_t *kbuf = sm + kKOff + kb * 32768;
                const uint32_t kbuf_s = s_base + kKOff + kb * 32768;
                if (c < mt.n_ct) {
                    for (int u = ptid; u < kTile * 16; u += kProducers) {
                        const int i = u >> 4, ch = u & 15;
                        const int pos = c * kTile + i;
                        const uint32_t off = (ch >> 3) * 16384 + sw128_off(i, ch & 7);
                        int j = pos < mt.n_sel ? sidx[pos] : -1;
                        if (j >= P.ncap) {
                            set_status(CSA_ERR_BOUNDS);
                            j = -1;
                        }
                        if (j < 0) {
                            *reinterpret_cast<uint4 *>(kbuf + off) = make_uint4(0, 0, 0, 0);
                            continue;
                        }
                        const int64_t er = (int64_t)mt.b * P.ncap + j;
                        if (!P.mixed) {
                            cp_async16(kbuf_s + off, reinterpret_cast<const __nv_bfloat16 *>(P.c_data) + er * 128 + ch * 8);
                        } else if (ch >= 8) {
                            cp_async16(kbuf_s + off, P.c_rope + er * 64 + (ch - 8) * 8);
                        } else {
                            const uint2 codes = *reinterpret_cast<const uint2 *>(
                                reinterpret_cast<const uint8_t *>(P.c_data) + er * 64 + ch * 8);
                            const float sc = P.c_scale[er];
                            const uint32_t cw[2] = {codes.x, codes.y};
                            uint32_t pk[4];
#pragma unroll
                            for (int q = 0; q < 2; ++q)
#pragma unroll
                                for (int e = 0; e < 2; ++e) {
                                    const uint16_t two = (uint16_t)(cw[q] >> (16 * e));
                                    __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)two, __NV_E4M3);
                                    const float2 f = __half22float2(__half2(hr));
                                    pk[2 * q + e] = pack2(f.x * sc, f.y * sc);
                                }
                            *reinterpret_cast<uint4 *>(kbuf + off) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                        }
                    }
                } else if (!P.decode) {
                    // window rows [t - 127, t] of sequence b by TMA (rows before 0 read as zeros)
                    if (ptid == 0) {
                        const uint32_t kf = smem_u32(&b_kfull[kb]);
                        mbar_expect_tx_only(kf, 2 * kTile * 128);
                        tma_load_3d(kbuf_s, &P.mkv, kf, 0, mt.t - kTile + 1, mt.b);
                        tma_load_3d(kbuf_s + 16384, &P.mkv, kf, 64, mt.t - kTile + 1, mt.b);
                    }
                } else {
                    // decode: window rows from the ring, row u at slot u mod n_win
                    for (int u = ptid; u < kTile * 16; u += kProducers) {
                        const int i = u >> 4, ch = u & 15;
                        const uint32_t off = (ch >> 3) * 16384 + sw128_off(i, ch & 7);
                        const int uu = mt.t - kTile + 1 + i;  // position of key row i
                        if (uu < 0 || uu <= mt.t - mt.n_win_t) {
                            *reinterpret_cast<uint4 *>(kbuf + off) = make_uint4(0, 0, 0, 0);
                            continue;
                        }
                        cp_async16(kbuf_s + off, P.win + ((int64_t)mt.b * P.n_win + (uu % P.n_win)) * 128 + ch * 8);
                    }
                }
                cp_async_commit();
                // fetch the next token's rows once its slot is free (never blocking here)
                if (ptid == 0 && fetched == it + 1 && it + 1 < n_tok_cta &&
                    (it + 1 < 2 || mbar_try_wait(smem_u32(&b_qempty[(it + 1) & 1]), (((it + 1) >> 1) - 1) & 1))) {
                    fetch(it + 1);
                    fetched = it + 2;
                }
                if (pending >= 0) {
                    cp_async_wait_1();
                    fence_async_smem();
                    mbar_arrive(smem_u32(&b_kfull[pending % kNB]));
                }
                pending = n;
            }
        }
        if (pending >= 0) {
            cp_async_wait_all();
            fence_async_smem();
            mbar_arrive(smem_u32(&b_kfull[pending % kNB]));
        }
    } else if (warp == kMmaWarp) {
        // =============================== MMA issue ===============================
        if (lane == 0) {
            const uint32_t idesc_s = idesc_bf16(128, kH, 0, 0);  // S^T = K Q^T
            const uint32_t idesc_o = idesc_bf16(128, kH, 1, 1);  // O^T = V^T P^T, both MN-major
            int n = 0;
            int prev_n = -1, prev_first = 0, prev_last = 0;  // the item whose P V is still to issue
            auto issue_pv = [&](int pn, bool first, bool last, int tok_it) -> bool {
                const int ps = pn & 1;
                if (!mbar_wait(smem_u32(&b_pfull[ps]), (pn >> 1) & 1, kMaxPolls, &g_abort)) return false;
                if (first && tok_it >= 1 &&
                    !mbar_wait(smem_u32(&b_oempty), (tok_it - 1) & 1, kMaxPolls, &g_abort))
                    return false;
                tc_fence_after();
                const uint32_t kb = s_base + kKOff + (pn % kNB) * 32768;
                const uint32_t pb = s_base + kPOff + ps * 16384;
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint64_t ad = sdesc_sw128(kb + kk * 2048, 16384, 1024);  // V^T, M = dims
                    const uint64_t bd = sdesc_sw128(pb + kk * 2048, 16384, 1024);  // P^T, N = heads
                    mma_bf16(tmem + kOCol, ad, bd, idesc_o, (!first || kk > 0) ? 1u : 0u);
                }
                mma_commit(smem_u32(&b_pempty[ps]));
                mma_commit(smem_u32(&b_kempty[pn % kNB]));
                if (last) mma_commit(smem_u32(&b_ofull));
                return true;
            };
            int prev_tok_it = 0;
            for (int it = 0; it < n_tok_cta && ok; ++it) {
                const int qs = it & 1;
                if (!mbar_wait(smem_u32(&b_qfull[qs]), (it >> 1) & 1, kMaxPolls, &g_abort)) { ok = false; break; }
                const int n_tiles = meta[qs].n_ct + 1;
                for (int c = 0; c < n_tiles; ++c, ++n) {
                    const int kb = n % kNB, ss = n & 1;
                    if (!mbar_wait(smem_u32(&b_kfull[kb]), (n / kNB) & 1, kMaxPolls, &g_abort)) { ok = false; break; }
                    if (n >= 2 && !mbar_wait(smem_u32(&b_sempty[ss]), ((n >> 1) - 1) & 1, kMaxPolls, &g_abort)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t kbuf = s_base + kKOff + kb * 32768;
                    const uint32_t qbuf = s_base + kQOff + qs * 16384;
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint64_t ad = sdesc_sw128(kbuf + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024);
                        const uint64_t bd = sdesc_sw128(qbuf + (kk >> 2) * 8192 + (kk & 3) * 32, 16, 1024);
                        mma_bf16(tmem + kSCol + ss * 64, ad, bd, idesc_s, kk > 0 ? 1u : 0u);
                    }
                    mma_commit(smem_u32(&b_sfull[ss]));
                    if (c == n_tiles - 1) mma_commit(smem_u32(&b_qempty[qs]));
                    if (prev_n >= 0 && !issue_pv(prev_n, prev_first, prev_last, prev_tok_it)) { ok = false; break; }
                    prev_n = n;
                    prev_first = c == 0;
                    prev_last = c == n_tiles - 1;
                    prev_tok_it = it;
                }
            }
            if (ok && prev_n >= 0) ok = issue_pv(prev_n, prev_first, prev_last, prev_tok_it);
            if (!ok) set_timeout();
        }
    } else if (warp < 4) {
        // ============================ softmax + epilogue ============================
        const uint32_t lane_base = (uint32_t)(32 * warp) << 16;
        // group-uniform wait (see the producers)
        auto swait = [&](uint32_t bar, uint32_t par) -> bool {
            const bool w = mbar_wait(bar, par, kMaxPolls, &g_abort);
            return !named_sync_or(kBarSoftmax, kSoftmax, !w);
        };
        float lpart[kH];
        int n = 0;
        for (int it = 0; it < n_tok_cta && ok; ++it) {
            const int qs = it & 1;
            if (!swait(smem_u32(&b_qfull[qs]), (it >> 1) & 1)) { ok = false; break; }
            const TokenMeta mt = meta[qs];
            mbar_arrive(smem_u32(&b_qempty[qs]));
            const int n_tiles = mt.n_ct + 1;
            for (int h = tid; h < kH; h += kSoftmax) s_m[h] = -INFINITY;
#pragma unroll
            for (int h = 0; h < kH; ++h) lpart[h] = 0.0f;
            named_sync(kBarSoftmax, kSoftmax);
            for (int c = 0; c < n_tiles; ++c, ++n) {
                const int ss = n & 1;
                if (!swait(smem_u32(&b_sfull[ss]), (n >> 1) & 1)) { ok = false; break; }
                tc_fence_after();
                // key validity of this thread's key (TMEM lane = key within the tile)
                bool valid;
                if (c < mt.n_ct) valid = c * kTile + tid < mt.n_sel;
                else valid = tid >= kTile - mt.n_win_t;  // key row tid is position t - 127 + tid
                float s[kH];
                {
                    float v[32];
                    tmem_ld32_sync(tmem + lane_base + kSCol + ss * 64, v);
#pragma unroll
                    for (int e = 0; e < 32; ++e) s[e] = valid ? v[e] * P.scale_log2 : -INFINITY;
                    tmem_ld32_sync(tmem + lane_base + kSCol + ss * 64 + 32, v);
#pragma unroll
                    for (int e = 0; e < 32; ++e) s[32 + e] = valid ? v[e] * P.scale_log2 : -INFINITY;
                }
                tc_fence_before();
                mbar_arrive(smem_u32(&b_sempty[ss]));
                // lazy max: reduce across the 128 keys only if some logit jumps the current max
                bool need = false;
#pragma unroll
                for (int h = 0; h < kH; ++h) need |= s[h] > s_m[h] + kRescaleThreshold;
                need = named_sync_or(kBarSoftmax, kSoftmax, need);
                if (need) {
                    // warp butterfly: after 5 steps lane holds the max of 2 heads over its warp
                    float v[kH];
#pragma unroll
                    for (int h = 0; h < kH; ++h) v[h] = s[h];
#pragma unroll
                    for (int step = 0; step < 5; ++step) {
                        const int o = 16 >> step;
                        const int w = kH >> (step + 1);  // values kept after this step
                        const bool upper = (lane & o) != 0;
#pragma unroll
                        for (int j = 0; j < w; ++j) {
                            const float keep = upper ? v[j + w] : v[j];
                            const float send = upper ? v[j] : v[j + w];
                            v[j] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, o));
                        }
                    }
                    // lane's heads: base = 32*b4 + 16*b3 + 8*b2 + 4*b1 + 2*b0
                    const int hb = ((lane >> 4) & 1) * 32 + ((lane >> 3) & 1) * 16 + ((lane >> 2) & 1) * 8 +
                                   ((lane >> 1) & 1) * 4 + (lane & 1) * 2;
                    s_red[warp][hb] = v[0];
                    s_red[warp][hb + 1] = v[1];
                    named_sync(kBarSoftmax, kSoftmax);
                    if (tid < kH) {
                        const float mnew = fmaxf(fmaxf(s_red[0][tid], s_red[1][tid]), fmaxf(s_red[2][tid], s_red[3][tid]));
                        const float mold = s_m[tid];
                        float f = 1.0f;
                        if (mnew > mold + kRescaleThreshold) {
                            f = exp2f(mold - mnew);  // 0 when mold is -inf
                            s_m[tid] = mnew;
                        }
                        s_f[tid] = f;
                    }
                    named_sync(kBarSoftmax, kSoftmax);
#pragma unroll
                    for (int h = 0; h < kH; ++h) lpart[h] *= s_f[h];
                    bool rescale_o = false;
                    if (c > 0) {
#pragma unroll
                        for (int h = 0; h < kH; ++h) rescale_o |= s_f[h] != 1.0f;
                    }
                    rescale_o = named_sync_or(kBarSoftmax, kSoftmax, rescale_o);
                    if (rescale_o) {
                        // O^T holds the P V of the previous tile of this token: wait for it
                        const int pn = n - 1;
                        if (!swait(smem_u32(&b_pempty[pn & 1]), (pn >> 1) & 1)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        for (int c0 = 0; c0 < kH; c0 += 32) {
                            float o[32];
                            tmem_ld32_sync(tmem + lane_base + kOCol + c0, o);
                            float o1[16], o2[16];
#pragma unroll
                            for (int e = 0; e < 16; ++e) {
                                o1[e] = o[e] * s_f[c0 + e];
                                o2[e] = o[16 + e] * s_f[c0 + 16 + e];
                            }
                            tmem_st16(tmem + lane_base + kOCol + c0, o1);
                            tmem_st16(tmem + lane_base + kOCol + c0 + 16, o2);
                        }
                        tmem_st_wait();
                    }
                }
                // P^T row of this key: exp2(s - m) for the 64 heads, BF16
                const int ps = n & 1;
                if (n >= 2 && !swait(smem_u32(&b_pempty[ps]), ((n >> 1) - 1) & 1)) {
                    ok = false;
                    break;
                }
                uint8_t *prow = sm + kPOff + ps * 16384;
#pragma unroll
                for (int ch = 0; ch < 8; ++ch) {
                    uint32_t pk[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int h = ch * 8 + 2 * e;
                        const float p0 = s[h] == -INFINITY ? 0.0f : fast_exp2(s[h] - s_m[h]);
                        const float p1 = s[h + 1] == -INFINITY ? 0.0f : fast_exp2(s[h + 1] - s_m[h + 1]);
                        lpart[h] += p0;
                        lpart[h + 1] += p1;
                        pk[e] = pack2(p0, p1);
                    }
                    *reinterpret_cast<uint4 *>(prow + sw128_off(tid, ch)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                }
                fence_async_smem();
                tc_fence_before();
                mbar_arrive(smem_u32(&b_pfull[ps]));
            }
            if (!ok) break;
            // ---- epilogue of the token: reduce the sums, normalise, inverse RoPE, store ----
            {
                float v[kH];
#pragma unroll
                for (int h = 0; h < kH; ++h) v[h] = lpart[h];
#pragma unroll
                for (int step = 0; step < 5; ++step) {
                    const int o = 16 >> step;
                    const int w = kH >> (step + 1);
                    const bool upper = (lane & o) != 0;
#pragma unroll
                    for (int j = 0; j < w; ++j) {
                        const float keep = upper ? v[j + w] : v[j];
                        const float send = upper ? v[j] : v[j + w];
                        v[j] = keep + __shfl_xor_sync(0xffffffffu, send, o);
                    }
                }
                const int hb = ((lane >> 4) & 1) * 32 + ((lane >> 3) & 1) * 16 + ((lane >> 2) & 1) * 8 +
                               ((lane >> 1) & 1) * 4 + (lane & 1) * 2;
                s_red[warp][hb] = v[0];
                s_red[warp][hb + 1] = v[1];
            }
            named_sync(kBarSoftmax, kSoftmax);
            if (tid < kH) {
                const float l = (s_red[0][tid] + s_red[1][tid]) + (s_red[2][tid] + s_red[3][tid]);
                const float m = s_m[tid];
                float f;
                if (P.sink) {
                    const float s2 = P.sink[tid] * 1.4426950408889634f;
                    const float mf = fmaxf(m, s2);
                    f = exp2f(m - mf) / (l * exp2f(m - mf) + exp2f(s2 - mf));
                } else {
                    f = 1.0f / l;
                }
                s_fo[tid] = f;
                if (P.lse && mt.t >= 0 && mt.t < P.L)
                    P.lse[(int64_t)((P.decode ? mt.b : mt.b * P.L + mt.t)) * kH + tid] = (m + log2f(l)) * 0.6931471805599453f;
            }
            if (!swait(smem_u32(&b_ofull), it & 1)) { ok = false; break; }
            tc_fence_after();
            named_sync(kBarSoftmax, kSoftmax);
            float *os = reinterpret_cast<float *>(sm + kOsOff);  // [h][d]
            {
                float o[32];
                tmem_ld32_sync(tmem + lane_base + kOCol, o);
#pragma unroll
                for (int e = 0; e < 32; ++e) os[e * 128 + tid] = o[e] * s_fo[e];
                tmem_ld32_sync(tmem + lane_base + kOCol + 32, o);
#pragma unroll
                for (int e = 0; e < 32; ++e) os[(32 + e) * 128 + tid] = o[e] * s_fo[32 + e];
            }
            tc_fence_before();
            mbar_arrive(smem_u32(&b_oempty));
            named_sync(kBarSoftmax, kSoftmax);
            if (mt.t >= 0 && mt.t < P.L) {
                const int64_t orow = P.decode ? (int64_t)mt.b : (int64_t)mt.b * P.L + mt.t;
                __nv_bfloat16 *out = P.out + orow * kH * 128;
                // thread tid always handles dims [8q, 8q+8), q = tid & 15, of heads (tid >> 4) + 8k,
                // so its RoPE factors are fetched once
                const int q = tid & 15;
                const bool rot = P.d_rope == 64 && q >= 8;
                const int i0 = 8 * ((q - 8) & 3);
                float2 cs[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) cs[e] = rot ? P.rope[(int64_t)mt.t * 32 + i0 + e] : make_float2(1.0f, 0.0f);
#pragma unroll
                for (int k = 0; k < kH / 8; ++k) {
                    const int h = (tid >> 4) + 8 * k;
                    const float *src = os + h * 128;
                    float y[8];
                    if (!rot) {
#pragma unroll
                        for (int e = 0; e < 8; ++e) y[e] = src[8 * q + e];
                    } else if (q < 12) {  // dims 64 + i, partner 96 + i
#pragma unroll
                        for (int e = 0; e < 8; ++e) y[e] = src[64 + i0 + e] * cs[e].x + src[96 + i0 + e] * cs[e].y;
                    } else {  // dims 96 + i
#pragma unroll
                        for (int e = 0; e < 8; ++e) y[e] = -src[64 + i0 + e] * cs[e].y + src[96 + i0 + e] * cs[e].x;
                    }
                    *reinterpret_cast<uint4 *>(out + h * 128 + 8 * q) =
                        make_uint4(pack2(y[0], y[1]), pack2(y[2], y[3]), pack2(y[4], y[5]), pack2(y[6], y[7]));
                }
            }
            named_sync(kBarSoftmax, kSoftmax);
        }
        if (!ok && tid == 0) set_timeout();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

bool csa_tc_supported(const AttnArgs &a) {
    if (a.act_t != CSA_BF16) return false;
    if (a.kv_t != CSA_BF16 && a.kv_t != CSA_MIXED) return false;
    if (a.H != csa_tc::kH || a.n_win != 128 || a.topk < 4 || a.topk > kMaxTopk || a.topk % 4 != 0) return false;
    if (a.d_rope != 0 && a.d_rope != 64) return false;
    // top-k rows are fetched with a bulk copy: 16-byte aligned rows
    return a.idx != nullptr && (reinterpret_cast<uintptr_t>(a.idx) & 15) == 0;
}

bool launch_csa_tc(const AttnArgs &a, cudaStream_t st) {
    using namespace csa_tc;
    if (!csa_tc_supported(a)) return false;
    CsaTcParams P;
    memset(&P, 0, sizeof(P));
    const int rows = a.decode ? a.B : a.B * a.L;
    bool ok = make_map_3d(&P.mq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.q, 128, (uint64_t)rows * kH, 1, 64, kH,
                          CU_TENSOR_MAP_SWIZZLE_128B);
    if (!a.decode)
        ok = ok && make_map_3d(&P.mkv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.kv_rope, 128, a.L, a.B, 64, kTile,
                               CU_TENSOR_MAP_SWIZZLE_128B);
    if (!ok) return false;
    P.c_data = a.c_data;
    P.c_rope = reinterpret_cast<const __nv_bfloat16 *>(a.c_rope);
    P.c_scale = a.c_scale;
    P.win = a.decode ? reinterpret_cast<const __nv_bfloat16 *>(a.kv_rope) : nullptr;
    P.idx = a.idx;
    P.ctx = a.ctx;
    P.sink = a.sink;
    P.rope = reinterpret_cast<const float2 *>(a.rope_tab);
    P.out = reinterpret_cast<__nv_bfloat16 *>(a.out);
    P.lse = a.lse;
    P.B = a.B; P.L = a.L; P.ncap = a.ncap; P.topk = a.topk; P.n_win = a.n_win; P.d_rope = a.d_rope;
    P.mixed = a.kv_t == CSA_MIXED; P.decode = a.decode; P.rows = rows;
    P.scale_log2 = a.scale * 1.4426950408889634f;
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaFuncSetAttribute(csa_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    const int grid = rows < sms ? rows : sms;
    csa_tc_kernel<<<grid, kThreads, kSmemBytes, st>>>(P);
    count_launches(1);
    return true;
}

}  // namespace csa
