// attn_hca_tc.cu -- HCA prefill attention on the 5th-generation tensor cores (tcgen05 + TMEM).
//
// Sources: [P2] "DeepSeek-V4: Towards Highly Efficient Million-Token Context Intelligence"
// (wiki notes), 提案手法 §1 (HCA: m' = 128 compression, no sparse selection, dense attention
// over the compressed entries; shared-KV MQA; sliding-window branch n_win = 128; attention
// sink; partial RoPE with inverse RoPE on the output) and 訓練インフラの革新 §5 (mixed-precision
// entries); [P5] "deepseek V4 技术论文" 一.1 (an entry is both key and value); [P3] "Технический
// отчёт DeepSeek-V4.1-Flash — часть 2/2" (NVFP4 entries).
//
// Every query head shares the one KV head, so a work item stacks T = 128 / H consecutive tokens
// x H heads into M = 128 query rows (row r = token t0 + r / H, head r % H) and walks one key
// list for all of them: compressed tiles of 128 entries [0, visible(last token)), then one
// window tile of the raw rows [t0 - 127, t0 + T - 1] (T + 127 <= 144 rows, padded to N = 144).
// Per key tile: S = Q K^T (M = 128, N = 128 or 144, K = 128) into TMEM; one thread per query row
// reads its S row, masks it (visibility / window), keeps a running row maximum in the log2
// domain (moved lazily, only when the tile maximum exceeds it by more than 8; O is then
// rescaled in TMEM), and writes P = exp2(s - max) as BF16 back into the first columns of the
// same TMEM slot (two values per 32-bit column); O += P V (M = 128, N = 128, K = keys)
// accumulates in TMEM with P read from TMEM as the A operand and V (the same key tile) from
// shared memory through an MN-major descriptor.
//
// Roles (192 threads, persistent over work items):
//   warps 0-3  softmax + epilogue (thread = query row = TMEM lane); the epilogue stages the
//              item's 128 output rows (BF16, 128-byte swizzle) in the item's query slot, whose
//              query rows are no longer needed, and writes them with two TMA tensor stores;
//   warp 4     MMA issue (one thread);
//   warp 5     producer: query rows by TMA (and RoPE on them, all 32 lanes), key tiles by TMA.
// S/P is double-buffered in TMEM, so the MMA computes the next tile's scores and the previous
// tile's P V while the softmax works on this one; a slot is rewritten by S(n + 2) only after
// P V(n) has read it, which the in-order tensor pipe guarantees (P V(n) is issued first). Key
// tiles flow through four buffers; query rows are double-buffered and fetched one item ahead.
// MIXED and NVFP4 entries are widened to BF16 once per call (caller workspace) before this
// kernel runs. Every wait is bounded, and every TMEM access and every wait whose result guards
// one sits in a warp-uniform branch (tcgen05.ld / st are .sync.aligned).
#include "common.cuh"
#include "kernels.cuh"
#include "tma_host.cuh"
#include "umma.cuh"

namespace csa {
using namespace umma;

namespace hca_tc {
constexpr int kRows = 128;                 // query rows per work item
constexpr int kMmaWarp = 4;
constexpr int kProdWarp = 5;
constexpr int kThreads = 192;
constexpr int kNB = 4;                     // key-tile buffers
constexpr int kMaxKeys = 144;              // rows of a key-tile buffer (the window tile needs <= 144)
constexpr int kSub = kMaxKeys * 128;       // bytes of one 64-dim half of a key-tile buffer (18 KB)
constexpr int kQOff = 0;                   // Q: 2 buffers of two 64-dim halves of 16 KB
constexpr int kKOff = 65536;               // key tiles: kNB buffers of 2 * kSub
constexpr int kSmemBytes = kKOff + kNB * 2 * kSub + 1024;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSStride = 160;         // S/P slots at columns [0, 144) and [160, 304)
constexpr uint32_t kOCol = 320;            // O: columns [320, 448)
constexpr float kOver = 8.0f;              // log2 of the largest unnormalised weight allowed
}  // namespace hca_tc

struct HcaTcParams {
    CUtensorMap mq;    // q viewed as [B][L*H][128] bf16, box 64 x 128
    CUtensorMap mo;    // out viewed as [B][L*H][128] bf16, box 64 x 128 (the epilogue's stores)
    CUtensorMap mc;    // BF16 entries [B][ncap][128], box 64 x 128
    CUtensorMap mkv;   // kv_rope [B][L][128] bf16, box 64 x 144
    const float *sink;
    const float2 *rope;
    __nv_bfloat16 *out;
    float *lse;
    int B, L, H, T, m, ncap, n_win, n_swa, d_rope, n_items, items_per_seq;
    float scale_log2;
};

namespace {

struct Item {
    int b, t0, n_ct, n_tiles;
};

__device__ __forceinline__ Item item_of(const HcaTcParams &P, int w) {
    Item it;
    it.b = w / P.items_per_seq;
    it.t0 = (w % P.items_per_seq) * P.T;
    const int t_last = min(it.t0 + P.T, P.L) - 1;
    it.n_ct = (visible_entries(t_last, P.m, P.ncap) + 127) / 128;
    it.n_tiles = it.n_ct + 1;
    return it;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
    __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&v);
}

}  // namespace

__global__ void __launch_bounds__(hca_tc::kThreads, 1) hca_tc_kernel(const __grid_constant__ HcaTcParams P) {
    using namespace hca_tc;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ __align__(8) uint64_t b_qraw[2], b_qfull[2], b_qempty[2];
    __shared__ __align__(8) uint64_t b_kfull[kNB], b_kempty[kNB];
    __shared__ __align__(8) uint64_t b_sfull[2], b_pfull[2], b_pvdone, b_ofull, b_oempty;
    __shared__ uint32_t tmem_slot;
    __shared__ float4 s_rope[16][16];  // RoPE (cos, sin) pairs of the item's tokens (T <= 16)

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t s_base = smem_u32(sm);
    const int n_it_cta = (P.n_items - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x;

    if (warp == 0) {
        tmem_alloc(smem_u32(&tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&b_qraw[i]), 1);
            mbar_init(smem_u32(&b_qfull[i]), 32);
            // query slot free: the item's last S MMA is done (commit) and the item's output,
            // staged in the slot by the epilogue, has been read by its bulk store
            mbar_init(smem_u32(&b_qempty[i]), 2);
        }
        for (int i = 0; i < kNB; ++i) {
            mbar_init(smem_u32(&b_kfull[i]), 1);
            mbar_init(smem_u32(&b_kempty[i]), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&b_sfull[i]), 1);
            mbar_init(smem_u32(&b_pfull[i]), kRows);
        }
        mbar_init(smem_u32(&b_pvdone), 1);
        mbar_init(smem_u32(&b_ofull), 1);
        mbar_init(smem_u32(&b_oempty), kRows);
        mbar_fence_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;

    if (warp == kProdWarp) {
        // =============================== producer ===============================
        bool ok = true;
        int n = 0;         // global key-tile counter
        int fetched = 0;   // items whose query rows have been requested
        int landed = 0;    // items whose query rows have been waited for
        auto fetch_q = [&](int it2) {  // lane 0
            const Item I2 = item_of(P, (int)blockIdx.x + it2 * (int)gridDim.x);
            const int qs2 = it2 & 1;
            const uint32_t qb = smem_u32(&b_qraw[qs2]);
            mbar_expect_tx(qb, 2 * kRows * 128);
            tma_load_3d(s_base + kQOff + qs2 * 32768, &P.mq, qb, 0, I2.t0 * P.H, I2.b);
            tma_load_3d(s_base + kQOff + qs2 * 32768 + 16384, &P.mq, qb, 64, I2.t0 * P.H, I2.b);
        };
        for (int it = 0; it < n_it_cta && ok; ++it) {
            const Item I = item_of(P, (int)blockIdx.x + it * (int)gridDim.x);
            const int qs = it & 1;
            if (lane == 0 && fetched == it) {  // not prefetched: the slot must be free first
                if (it >= 2 && !mbar_wait(smem_u32(&b_qempty[qs]), ((it >> 1) - 1) & 1, kWaitNs, &g_abort)) ok = false;
                if (ok) {
                    fetch_q(it);
                    fetched = it + 1;
                }
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            fetched = __shfl_sync(0xffffffffu, fetched, 0);
            if (!ok) break;
            if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&b_qraw[qs]), (it >> 1) & 1, kWaitNs, &g_abort))) {
                ok = false;
                break;
            }
            landed = it + 1;
            // RoPE on dims 64..127 of every query row at its token's position; the item's T rows of
            // the table are staged in shared memory first (one load per lane, no dependent chains)
            if (P.d_rope == 64) {
                for (int i = lane; i < P.T * 16; i += 32) {
                    const int t = I.t0 + (i >> 4);
                    s_rope[i >> 4][i & 15] =
                        t < P.L ? __ldg(reinterpret_cast<const float4 *>(P.rope + (int64_t)t * 32) + (i & 15))
                                : make_float4(1.0f, 0.0f, 1.0f, 0.0f);
                }
                __syncwarp();
                uint8_t *q1 = sm + kQOff + qs * 32768 + 16384;
                for (int u = lane; u < kRows * 4; u += 32) {
                    const int r = u >> 2, c = u & 3;
                    const int t = I.t0 + r / P.H;
                    if (t >= P.L) continue;
                    float4 rc[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) rc[e] = s_rope[r / P.H][4 * c + e];
                    uint4 *pa = reinterpret_cast<uint4 *>(q1 + sw128_off(r, c));
                    uint4 *pb = reinterpret_cast<uint4 *>(q1 + sw128_off(r, c + 4));
                    uint4 va = *pa, vb = *pb;
                    __nv_bfloat162 *a2 = reinterpret_cast<__nv_bfloat162 *>(&va);
                    __nv_bfloat162 *b2 = reinterpret_cast<__nv_bfloat162 *>(&vb);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 x = __bfloat1622float2(a2[e]);
                        const float2 y = __bfloat1622float2(b2[e]);
                        const float4 cs = rc[e];  // (cos, sin) of pairs 8c + 2e and 8c + 2e + 1
                        a2[e] = __floats2bfloat162_rn(x.x * cs.x - y.x * cs.y, x.y * cs.z - y.y * cs.w);
                        b2[e] = __floats2bfloat162_rn(x.x * cs.y + y.x * cs.x, x.y * cs.w + y.y * cs.z);
                    }
                    *pa = va;
                    *pb = vb;
                }
                __syncwarp();  // s_rope is rewritten for the next item
            }
            fence_async_smem();
            mbar_arrive(smem_u32(&b_qfull[qs]));
            __syncwarp();
            // key tiles (lane 0)
            if (lane == 0) {
                for (int c = 0; c < I.n_tiles; ++c, ++n) {
                    const int kb = n % kNB;
                    if (n >= kNB && !mbar_wait(smem_u32(&b_kempty[kb]), ((n / kNB) - 1) & 1, kWaitNs, &g_abort)) {
                        ok = false;
                        break;
                    }
                    const uint32_t kf = smem_u32(&b_kfull[kb]);
                    const uint32_t kdst = s_base + kKOff + kb * 2 * kSub;
                    if (c < I.n_ct) {
                        mbar_expect_tx(kf, 2 * 128 * 128);
                        tma_load_3d(kdst, &P.mc, kf, 0, c * 128, I.b);
                        tma_load_3d(kdst + kSub, &P.mc, kf, 64, c * 128, I.b);
                    } else {
                        // window rows [t0 - 127, t0 + 16] (rows before 0 read as zeros; the box
                        // always holds row t0, so it overlaps the tensor)
                        mbar_expect_tx(kf, 2 * kMaxKeys * 128);
                        tma_load_3d(kdst, &P.mkv, kf, 0, I.t0 - P.n_win + 1, I.b);
                        tma_load_3d(kdst + kSub, &P.mkv, kf, 64, I.t0 - P.n_win + 1, I.b);
                    }
                    // prefetch the next item's query rows once its slot is free (never blocking)
                    if (fetched == it + 1 && it + 1 < n_it_cta &&
                        (it + 1 < 2 || mbar_test_wait(smem_u32(&b_qempty[(it + 1) & 1]), (((it + 1) >> 1) - 1) & 1))) {
                        fetch_q(it + 1);
                        fetched = it + 2;
                    }
                }
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            n = __shfl_sync(0xffffffffu, n, 0);
            fetched = __shfl_sync(0xffffffffu, fetched, 0);
        }
        // after a failure: let query rows still in flight land (bounded) before the CTA exits
        if (!ok && lane == 0)
            for (int f = landed; f < fetched; ++f) mbar_wait(smem_u32(&b_qraw[f & 1]), (f >> 1) & 1, kDrainNs);
    } else if (warp == kMmaWarp) {
        // =============================== MMA issue ===============================
        if (lane == 0) {
            bool ok = true;
            int n = 0;
            int pv_n = -1, pv_kb = 0, pv_nkeys = 0;  // the tile whose P V is still to issue
            bool pv_first = false, pv_last = false;
            int pv_it = 0;
            const uint32_t idesc_pv = idesc_bf16(128, 128, 0, 1);  // A = P (TMEM), B = V MN-major
            auto issue_pv = [&]() -> bool {
                const int psb = pv_n & 1;
                if (!mbar_wait(smem_u32(&b_pfull[psb]), (pv_n >> 1) & 1, kWaitNs, &g_abort)) return false;
                if (pv_first && pv_it >= 1 && !mbar_wait(smem_u32(&b_oempty), (pv_it - 1) & 1, kWaitNs, &g_abort))
                    return false;
                tc_fence_after();
                const uint32_t kt = s_base + kKOff + pv_kb * 2 * kSub;
                for (int kk = 0; kk < pv_nkeys / 16; ++kk) {
                    const uint64_t bd = sdesc_sw128(kt + kk * 2048, kSub, 1024);
                    mma_bf16_ts(tmem + kOCol, tmem + psb * kSStride + kk * 8, bd, idesc_pv, (!pv_first || kk > 0) ? 1u : 0u);
                }
                mma_commit(smem_u32(&b_kempty[pv_kb]));
                mma_commit(smem_u32(&b_pvdone));
                if (pv_last) mma_commit(smem_u32(&b_ofull));
                return true;
            };
            for (int it = 0; it < n_it_cta && ok; ++it) {
                const Item I = item_of(P, (int)blockIdx.x + it * (int)gridDim.x);
                const int qs = it & 1;
                if (!mbar_wait(smem_u32(&b_qfull[qs]), (it >> 1) & 1, kWaitNs, &g_abort)) { ok = false; break; }
                const uint32_t qbuf = s_base + kQOff + qs * 32768;
                for (int c = 0; c < I.n_tiles; ++c, ++n) {
                    const int kb = n % kNB, sb = n & 1;
                    const int nkeys = c < I.n_ct ? 128 : P.n_swa;
                    if (!mbar_wait(smem_u32(&b_kfull[kb]), (n / kNB) & 1, kWaitNs, &g_abort)) { ok = false; break; }
                    // slot sb last held S(n - 2) / P(n - 2): the softmax had written P(n - 2) before
                    // P V(n - 2) was issued, and that P V was issued before this S on the same pipe
                    tc_fence_after();
                    const uint32_t kt = s_base + kKOff + kb * 2 * kSub;
                    const uint32_t idesc_s = idesc_bf16(128, nkeys, 0, 0);
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint64_t ad = sdesc_sw128(qbuf + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024);
                        const uint64_t bd = sdesc_sw128(kt + (kk >> 2) * kSub + (kk & 3) * 32, 16, 1024);
                        mma_bf16(tmem + sb * kSStride, ad, bd, idesc_s, kk > 0 ? 1u : 0u);
                    }
                    mma_commit(smem_u32(&b_sfull[sb]));
                    if (c == I.n_tiles - 1) mma_commit(smem_u32(&b_qempty[qs]));
                    if (pv_n >= 0 && !issue_pv()) { ok = false; break; }
                    pv_n = n;
                    pv_kb = kb;
                    pv_nkeys = nkeys;
                    pv_first = c == 0;
                    pv_last = c == I.n_tiles - 1;
                    pv_it = it;
                }
                // the item's last P V goes out now, not behind the next item's query rows, so
                // that the epilogue is not held up
                if (ok && pv_n >= 0) {
                    ok = issue_pv();
                    pv_n = -1;
                }
            }
            if (!ok) set_timeout();
        }
    } else {
        // ====================== softmax + epilogue (row per thread) ======================
        // Each thread runs its own row, but the TMEM loads and stores (tcgen05.ld/st .sync.aligned)
        // must be executed by all 32 threads of a warp together: every branch around them, and
        // every decision to leave after a failed wait, is therefore made per warp (__any_sync /
        // __all_sync). Warps are independent of each other (no named barrier).
        const int r = tid;
        const uint32_t lane_base = (uint32_t)(32 * warp) << 16;
        bool ok = true;
        int n = 0;
        int store_slot = -1;  // thread 0: query slot whose output stores are still to be confirmed
        for (int it = 0; it < n_it_cta && ok; ++it) {
            const Item I = item_of(P, (int)blockIdx.x + it * (int)gridDim.x);
            const int t = I.t0 + r / P.H, h = r % P.H;
            const bool row_ok = t < P.L;
            const int vis_t = row_ok ? visible_entries(t, P.m, P.ncap) : 0;
            float m_run = -INFINITY, l_run = 0.0f;
            for (int c = 0; c < I.n_tiles; ++c, ++n) {
                const int sb = n & 1;
                const bool ctile = c < I.n_ct;
                const int nk = ctile ? 128 : P.n_swa;
                // valid keys [lo, hi) of this row in the tile
                int lo, hi;
                if (ctile) {
                    lo = 0;
                    hi = min(128, vis_t - c * 128);
                } else {  // key k is raw row t0 - 127 + k
                    lo = max(t - I.t0, P.n_win - 1 - I.t0);
                    hi = min(nk, t - I.t0 + P.n_win);
                }
                if (!row_ok) hi = 0;
                if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&b_sfull[sb]), (n >> 1) & 1, kWaitNs, &g_abort))) {
                    ok = false;  // (the warps leave together at the item's epilogue barrier)
                    set_timeout();
                    break;
                }
                tc_fence_after();
                const uint32_t s_addr = tmem + lane_base + sb * kSStride;
                // the row's scores in registers: one TMEM load of 128 columns (+16 for the window)
                float sv[128], sx[16];
                tmem_ld128_sync(s_addr, sv);
                if (nk > 128) tmem_ld16_sync(s_addr + 128, sx);
                // masked keys become -inf; a warp whose rows all see the whole tile skips the masks
                const bool full = __all_sync(0xffffffffu, lo == 0 && hi >= 128 && nk == 128);
                if (!full) {
#pragma unroll
                    for (int e = 0; e < 128; ++e) sv[e] = (e >= lo && e < hi) ? sv[e] : -INFINITY;
#pragma unroll
                    for (int e = 0; e < 16; ++e) sx[e] = (nk > 128 && 128 + e >= lo && 128 + e < hi) ? sx[e] : -INFINITY;
                }
                // tile maximum with eight independent partial maxima (short dependency chains)
                float mx8[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) mx8[q] = full ? sv[q] : fmaxf(sv[q], sx[q]);
#pragma unroll
                for (int e = 8; e < 128; ++e) mx8[e & 7] = fmaxf(mx8[e & 7], sv[e]);
                if (!full) {
#pragma unroll
                    for (int e = 8; e < 16; ++e) mx8[e & 7] = fmaxf(mx8[e & 7], sx[e]);
                }
                float tmax = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                                   fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
                tmax *= P.scale_log2;  // the scale is positive: max(s) * scale = max(s * scale)
                const bool upd = tmax > m_run + kOver;
                if (__any_sync(0xffffffffu, upd)) {
                    // (warp-uniform branch) rows whose maximum moved rescale by f, the others by 1
                    const float f = upd ? exp2f(m_run - tmax) : 1.0f;  // 0 when m_run is -inf
                    l_run *= f;
                    if (c > 0) {
                        // O holds the P V of this item's earlier tiles: let the last one finish
                        if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&b_pvdone), (n - 1) & 1, kWaitNs, &g_abort))) {
                            ok = false;
                            set_timeout();
                            break;
                        }
                        tc_fence_after();
                        const uint32_t o_addr = tmem + lane_base + kOCol;
#pragma unroll 1
                        for (int c0 = 0; c0 < 128; c0 += 16) {
                            float o[16];
                            tmem_ld16_sync(o_addr + c0, o);
#pragma unroll
                            for (int e = 0; e < 16; ++e) o[e] *= f;
                            tmem_st16(o_addr + c0, o);
                        }
                        tmem_st_wait();
                    }
                    if (upd) m_run = tmax;
                }
                // P = exp2(scale * s - max) as BF16; masked keys are -inf and give exp2(-inf) = 0
                // (m_run is finite whenever the row has a valid key; a row with none in this
                // tile and m_run = -inf would give NaN, so such a row is zeroed explicitly)
                const float neg_m = -m_run;
                const bool row_live = m_run != -INFINITY;
                if (__all_sync(0xffffffffu, row_live)) {
                    // scale * s - max for two keys per packed FMA, then the hardware exp2
                    const uint64_t sc2 = f2_pack(P.scale_log2, P.scale_log2), nm2 = f2_pack(neg_m, neg_m);
#pragma unroll
                    for (int e = 0; e < 128; e += 2) {
                        const float2 x = f2_unpack(f2_fma(f2_pack(sv[e], sv[e + 1]), sc2, nm2));
                        sv[e] = fast_exp2(x.x);
                        sv[e + 1] = fast_exp2(x.y);
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < 128; ++e) sv[e] = row_live ? fast_exp2(fmaf(sv[e], P.scale_log2, neg_m)) : 0.0f;
                }
                if (nk > 128) {
#pragma unroll
                    for (int e = 0; e < 16; ++e) sx[e] = row_live ? fast_exp2(fmaf(sx[e], P.scale_log2, neg_m)) : 0.0f;
                }
                // P as BF16 pairs into the first columns of the slot (its scores are in registers);
                // the row sum in four packed pair accumulators
                uint64_t ls2[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
                for (int c0 = 0; c0 < 128; c0 += 32) {
                    float w[16];
#pragma unroll
                    for (int e = 0; e < 32; e += 2) {
                        ls2[(e >> 1) & 3] = f2_add(ls2[(e >> 1) & 3], f2_pack(sv[c0 + e], sv[c0 + e + 1]));
                        w[e >> 1] = __uint_as_float(pack_bf16x2(sv[c0 + e], sv[c0 + e + 1]));
                    }
                    tmem_st16(s_addr + (c0 >> 1), w);
                }
                if (nk > 128) {
                    float w[16];
#pragma unroll
                    for (int e = 0; e < 16; e += 2) {
                        ls2[(e >> 1) & 3] = f2_add(ls2[(e >> 1) & 3], f2_pack(sx[e], sx[e + 1]));
                        w[e >> 1] = __uint_as_float(pack_bf16x2(sx[e], sx[e + 1]));
                    }
#pragma unroll
                    for (int e = 8; e < 16; ++e) w[e] = 0.0f;  // columns 72..79: beyond the 144 keys' P
                    tmem_st16(s_addr + 64, w);
                }
                {
                    const float2 a = f2_unpack(f2_add(ls2[0], ls2[1])), b = f2_unpack(f2_add(ls2[2], ls2[3]));
                    l_run += (a.x + a.y) + (b.x + b.y);
                }
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(smem_u32(&b_pfull[sb]));
                if (store_slot >= 0) {
                    // the previous item's output stores have long read their staging by now: hand
                    // that query slot back to the producer
                    bulk_wait_read0();
                    mbar_arrive(smem_u32(&b_qempty[store_slot]));
                    store_slot = -1;
                }
            }
            // ---- epilogue of the item: O / (sum + exp(sink)), inverse RoPE, BF16 store ----
            // (the four warps meet here: a failure anywhere makes all of them leave)
            const bool got = ok && __all_sync(0xffffffffu, mbar_wait(smem_u32(&b_ofull), it & 1, kWaitNs, &g_abort));
            if (named_sync_or(1, kRows, !got)) {
                ok = false;
                break;
            }
            tc_fence_after();
            float f = 0.0f;
            if (row_ok) {
                if (P.sink) {
                    const float s2 = P.sink[h] * 1.4426950408889634f;
                    const float mf = fmaxf(m_run, s2);
                    f = exp2f(m_run - mf) / (l_run * exp2f(m_run - mf) + exp2f(s2 - mf));
                } else {
                    f = 1.0f / l_run;
                }
                if (P.lse) P.lse[((int64_t)I.b * P.L + t) * P.H + h] = (m_run + log2f(l_run)) * 0.6931471805599453f;
            }
            // staging: the item's query slot as two [128 rows][64 dims] BF16 halves in the 128-byte
            // swizzle of the output tensor map (row r, 16-byte chunk c at sw128_off(r, c))
            uint8_t *stage = sm + kQOff + (it & 1) * 32768;
            const uint32_t o_addr = tmem + lane_base + kOCol;
            {
                // dims 0..63: normalised, no rotation
                float o[64];
                tmem_ld64_sync(o_addr, o);
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    *reinterpret_cast<uint4 *>(stage + sw128_off(r, c)) =
                        make_uint4(pack_bf16x2(o[8 * c] * f, o[8 * c + 1] * f),
                                   pack_bf16x2(o[8 * c + 2] * f, o[8 * c + 3] * f),
                                   pack_bf16x2(o[8 * c + 4] * f, o[8 * c + 5] * f),
                                   pack_bf16x2(o[8 * c + 6] * f, o[8 * c + 7] * f));
            }
            {
                // dims 64..127: normalised, then rotated back at the row's position (pairs 64+i, 96+i)
                float o[64];
                tmem_ld64_sync(o_addr + 64, o);
                tc_fence_before();
                mbar_arrive(smem_u32(&b_oempty));
#pragma unroll
                for (int e = 0; e < 64; ++e) o[e] *= f;
                if (P.d_rope == 64 && row_ok) {
                    const float4 *rp = reinterpret_cast<const float4 *>(P.rope + (int64_t)t * 32);
#pragma unroll
                    for (int i2 = 0; i2 < 16; ++i2) {
                        const float4 cs = __ldg(rp + i2);  // (cos, sin) of pairs 2*i2 and 2*i2 + 1
                        const float x0 = o[2 * i2], y0 = o[32 + 2 * i2];
                        const float x1 = o[2 * i2 + 1], y1 = o[33 + 2 * i2];
                        o[2 * i2] = x0 * cs.x + y0 * cs.y;
                        o[32 + 2 * i2] = -x0 * cs.y + y0 * cs.x;
                        o[2 * i2 + 1] = x1 * cs.z + y1 * cs.w;
                        o[33 + 2 * i2] = -x1 * cs.w + y1 * cs.z;
                    }
                }
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    *reinterpret_cast<uint4 *>(stage + 16384 + sw128_off(r, c)) =
                        make_uint4(pack_bf16x2(o[8 * c], o[8 * c + 1]), pack_bf16x2(o[8 * c + 2], o[8 * c + 3]),
                                   pack_bf16x2(o[8 * c + 4], o[8 * c + 5]), pack_bf16x2(o[8 * c + 6], o[8 * c + 7]));
            }
            fence_async_smem();
            named_sync(1, kRows);
            if (tid == 0) {
                // rows past the sequence end (t >= L) lie outside the tensor map and are not written
                const uint32_t sb0 = s_base + kQOff + (it & 1) * 32768;
                tma_store_3d(&P.mo, sb0, 0, I.t0 * P.H, I.b);
                tma_store_3d(&P.mo, sb0 + 16384, 64, I.t0 * P.H, I.b);
                bulk_commit();
                store_slot = it & 1;  // released after the next item's first tile
            }
        }
        if (tid == 0) bulk_wait0();
        if (!ok) set_timeout();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

// Host: returns false when the configuration is outside what this kernel handles (the call is
// then refused as unsupported).
bool hca_tc_supported(const AttnArgs &a) {
    if (a.decode || a.act_t != CSA_BF16) return false;
    if (a.kv_t != CSA_BF16 && a.kv_t != CSA_MIXED && a.kv_t != CSA_NVFP4) return false;
    if (a.H != 16 && a.H != 32 && a.H != 64 && a.H != 128) return false;
    if (a.n_win != 128) return false;
    if (128 / a.H + a.n_win - 1 > hca_tc::kMaxKeys) return false;
    if (a.d_rope != 0 && a.d_rope != 64) return false;
    if ((reinterpret_cast<uintptr_t>(a.out) & 15) != 0) return false;
    if (csa_widen_bytes(a) > a.ws_bytes || (csa_widen_bytes(a) > 0 && !a.ws)) return false;
    return true;
}

bool launch_hca_tc(const AttnArgs &a, cudaStream_t st) {
    using namespace hca_tc;
    if (!hca_tc_supported(a)) return false;
    HcaTcParams P;
    memset(&P, 0, sizeof(P));
    const uint64_t L = a.L, H = a.H, B = a.B, ncap = a.ncap;
    const bool widen = a.kv_t == CSA_MIXED || a.kv_t == CSA_NVFP4;  // entries widened to BF16 into a.ws
    const void *entries = widen ? a.ws : a.c_data;
    bool ok = make_map_3d(&P.mq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.q, 128, L * H, B, 64, 128,
                          CU_TENSOR_MAP_SWIZZLE_128B);
    ok = ok && make_map_3d(&P.mo, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.out, 128, L * H, B, 64, 128,
                           CU_TENSOR_MAP_SWIZZLE_128B);
    ok = ok && make_map_3d(&P.mc, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, entries, 128, ncap, B, 64, 128,
                           CU_TENSOR_MAP_SWIZZLE_128B);
    ok = ok && make_map_3d(&P.mkv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.kv_rope, 128, L, B, 64, kMaxKeys,
                           CU_TENSOR_MAP_SWIZZLE_128B);
    if (!ok) return false;
    if (widen && a.ncap > 0) launch_widen_entries(a, st);
    P.sink = a.sink;
    P.rope = reinterpret_cast<const float2 *>(a.rope_tab);
    P.out = reinterpret_cast<__nv_bfloat16 *>(a.out);
    P.lse = a.lse;
    P.B = a.B; P.L = a.L; P.H = a.H; P.T = 128 / a.H; P.m = a.m; P.ncap = a.ncap; P.n_win = a.n_win;
    P.n_swa = ((P.T + a.n_win - 1) + 15) / 16 * 16;
    P.d_rope = a.d_rope;
    P.items_per_seq = (int)((L + P.T - 1) / P.T);
    P.n_items = P.items_per_seq * a.B;
    P.scale_log2 = a.scale * 1.4426950408889634f;
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaFuncSetAttribute(hca_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    const int grid = P.n_items < sms ? P.n_items : sms;
    hca_tc_kernel<<<grid, kThreads, kSmemBytes, st>>>(P);
    count_launches(1);
    return true;
}

}  // namespace csa
