// attn_csa_tc.cu -- CSA sparse attention on the 5th-generation tensor cores (tcgen05 + TMEM).
//
// Sources: [P2] "DeepSeek-V4: Towards Highly Efficient Million-Token Context Intelligence"
// (wiki notes), 提案手法 §1 (CSA: each query attends to its top-k compressed entries;
// shared-KV multi-query attention; sliding-window branch n_win = 128; attention sink;
// partial RoPE + inverse RoPE on the core output) and 訓練インフラの革新 §5 (mixed-precision
// entries); [P5] "deepseek V4 技术论文" 一.1 (an entry is both key and value); [P3] "Технический
// отчёт DeepSeek-V4.1-Flash — часть 2/2" (the V4.1 variant: NVFP4 entries, an FP8 window cache).
//
// Every token has its own key list: its top-k entries (ascending, gathered by index) followed
// by the 128 raw rows of its window. All 64 heads of a token share that list, so the kernel
// puts the KEYS on the MMA's M dimension and the heads on N:
//   S^T[key, head] = K Q^T     (M = 128 keys, N = 64 heads, K = 128 dims)
//   O^T[dim, head] += V^T P^T  (M = 128 dims, N = 64 heads, K = 128 keys)
// which keeps both MMAs at M = 128. The key tile is one shared-memory buffer read as the
// K-major A operand of the first MMA and, through an MN-major descriptor, as V^T for the
// second; P^T is written by the softmax threads as 128-byte key rows and read as an MN-major
// B operand.
//
// Softmax: two warpgroups, WG w owning heads [32w, 32w + 32); thread = one key (TMEM lane) x
// 32 heads. The per-head running maximum is shared by the 128 keys of a tile and kept lazily:
// P = exp2(s - m) is computed with the current maximum, and only when some value exceeds 2^8
// does the warpgroup reduce the tile's per-head maxima, move m, and rescale its partial sums
// and O^T (in TMEM). That happens on a token's first tile and rarely after. Per-head sums are
// partial per thread and reduced once per token.
//
// Warp roles (384 threads, persistent over tokens):
//   warps 0-7   softmax and epilogue (two warpgroups; TMEM lanes 0-127 each);
//   warp 8      MMA issue (one thread);
//   warps 9-11  producers: query rows by TMA + RoPE, top-k row by bulk copy, key tiles gathered
//               with cp.async, the window tile by TMA (prefill) or gathered from the ring
//               (decode). Decode tiles stored in a low-precision form (MIXED or NVFP4 entries,
//               an FP8 ring) are widened to BF16 by the producer threads: each thread loads a
//               group of its chunks, then converts and stores them.
// Pipelines: key tiles in a 3- or 4-buffer ring, four S^T slots and two O^T slots (by token) in
// TMEM, P^T double-buffered in shared memory, query rows double-buffered; every wait is bounded.
// The MMA warp issues the P V of tile n after the S^T of tile n + 2, so S^T work is queued on the
// tensor pipe while the softmax finishes a tile. The tensor pipe reads its operands from shared
// memory, whose bandwidth (with the gather's and the softmax's writes) bounds this kernel: an
// N = 64 MMA is operand-read bound, and the MMA issue loop builds each descriptor by adding a
// constant to a base descriptor.
// Epilogue: the per-head sums are reduced right after a token's last tile; the O part waits
// until the next token's first tile has been handed over (its P V has finished by then): O^T is
// normalised per head, the RoPE half is rotated back (the two dims of a pair live in different
// warps and meet in shared memory), staged as BF16 [head][dim] and written with one 16 KB bulk
// copy per token.
//
// Prefill with MIXED or NVFP4 entries first widens every entry to BF16 once (the dequantised
// value rounded to nearest even) into caller workspace; the gather then reads BF16 rows.
#include "common.cuh"
#include "fp4.cuh"
#include "kernels.cuh"
#include "tma_host.cuh"
#include "umma.cuh"

namespace csa {
using namespace umma;

namespace csa_tc {
constexpr int kSoftmax = 256;                 // warps 0-7
constexpr int kMmaWarp = 8;
constexpr int kProd0 = 288;                   // first producer thread (warp 9)
constexpr int kProducers = 96;                // warps 9-11
constexpr int kThreads = kProd0 + kProducers; // 384
constexpr int kH = 64;                        // heads (N of both MMAs)
constexpr int kTile = 128;                    // keys per tile
constexpr int kGatherPer = 22;                // 16-byte chunks of a key tile per producer thread
constexpr int kConvBatch = 8;                 // converted chunks whose loads are in flight together
// Shared memory (1024-aligned), for NB key-tile buffers:
//   Q       2 buffers x 16 KB (two 64-dim halves of 8 KB)
//   keys    NB x 32 KB (two 64-dim halves of 16 KB)
//   P^T     2 x 16 KB
//   output  staging [64 heads][128 dims] BF16, 16 KB; before that, in a token's epilogue, the
//           RoPE exchange [2 WG][2 halves][32 heads][32] float
//   top-k   2 rows of topk int32
constexpr int kQOff = 0;
constexpr int kKOff = 32768;
__host__ __device__ constexpr int p_off(int nb) { return kKOff + nb * 32768; }
__host__ __device__ constexpr int out_off(int nb) { return p_off(nb) + 2 * 16384; }
__host__ __device__ constexpr int idx_off(int nb) { return out_off(nb) + 16384; }
constexpr uint32_t kTmemCols = 512;
constexpr int kSSlots = 4;                    // S^T slots in TMEM
constexpr int kLag = 2;                       // the P V of tile n is issued after the S^T of tile n + kLag
constexpr uint32_t kSCol = 0;                 // S^T slots: [64 i, 64 i + 64), i < kSSlots
constexpr uint32_t kOCol = 256;               // O^T slots: [256, 320) and [320, 384)
constexpr float kOver = 8.0f;                 // log2 of the largest unnormalised weight allowed
// named barriers (0 is __syncthreads)
constexpr uint32_t kBarSoftmax = 1, kBarProd = 2, kBarWG0 = 3;  // kBarWG0 + w per warpgroup
}  // namespace csa_tc

struct CsaTcParams {
    CUtensorMap mq;    // q rows [rows*64][128] bf16, box 64 x 64
    CUtensorMap mkv;   // prefill: kv_rope [B][L][128] bf16, box 64 x 128
    const void *c_data;
    const __nv_bfloat16 *c_rope;
    const float *c_scale;
    const void *win;            // decode: ring [B][n_win][128] BF16, or [B][n_win] FP8 rows (win8)
    const int32_t *idx;         // [rows][topk]
    const int32_t *ctx;         // decode: [B]
    const float *sink;
    const float2 *rope;
    __nv_bfloat16 *out;
    float *lse;
    int B, L, ncap, topk, n_win, d_rope, decode, rows;
    int ent;        // entry storage read by the gather: 0 BF16, 1 MIXED, 2 NVFP4 (decode only)
    int win8;       // decode: the ring holds FP8 rows
    int dense, m;   // dense: keys are entries 0 .. visible(t) - 1 in order (no top-k row)
    float scale_log2;
    // split-KV decode: work item r = (sequence r / S, split r % S) takes the key tiles
    // [T * (r % S), T * (r % S) + T) of its sequence (compressed tiles, then the window tile) and
    // writes its unnormalised partial O and per-head (max, sum) instead of the output
    int split, S, T;
    float *part_o;     // [items][64 heads][128 dims] float
    float2 *part_ml;   // [items][64 heads] (running max in log2 units, sum of weights)
};

namespace {

struct TokenMeta {
    int n_sel;   // valid top-k entries
    int n_ct;    // compressed tiles
    int c0;      // first key tile of this work item (the window tile is tile n_ct)
    int n_tiles; // key tiles of this work item (>= 1)
    int t;       // query position
    int b;       // sequence
    int n_win_t; // window rows that exist (<= n_win)
    int pos_ok;  // 0: a decode position outside the cache (nothing is stored)
};

__device__ __forceinline__ uint32_t pack2(float a, float b) { return bf16x2_bits(a, b); }

// One 16-byte chunk (8 dims) of a key row as loaded from a low-precision store, widened to BF16
// when it is written to the key tile.
enum : int { kChZero = 0, kChBf16 = 1, kChFp8 = 2, kChFp4 = 3 };
struct RawChunk {
    uint4 v;   // BF16: the chunk; FP8: codes in v.x, v.y; FP4: codes in v.x, block-scale code in v.y
    float s;   // row scale (FP8, FP4)
    int kind;
};

__device__ __forceinline__ uint4 widen_chunk(const RawChunk &r) {
    if (r.kind == kChBf16) return r.v;
    if (r.kind == kChFp8) return fp8x8_to_bf16(r.v.x, r.v.y, r.s);
    if (r.kind == kChFp4) return fp4x8_to_bf16(r.v.x, r.v.y, r.s);
    return make_uint4(0, 0, 0, 0);
}

// chunk ch of entry row er: MIXED (ent 1) or NVFP4 (ent 2)
__device__ __forceinline__ void load_entry_chunk(const CsaTcParams &P, int64_t er, int ch, RawChunk &r) {
    if (P.ent == 2) {
        const uint8_t *row = reinterpret_cast<const uint8_t *>(P.c_data) + er * kNvfp4RowBytes;
        r.v.x = __ldg(reinterpret_cast<const uint32_t *>(row) + ch);
        r.v.y = __ldg(row + 64 + (ch >> 1));
        r.s = __ldg(reinterpret_cast<const float *>(row + 72));
        r.kind = kChFp4;
    } else if (ch >= 8) {
        r.v = __ldg(reinterpret_cast<const uint4 *>(P.c_rope + er * 64 + (ch - 8) * 8));
        r.kind = kChBf16;
    } else {
        const uint2 c = __ldg(reinterpret_cast<const uint2 *>(reinterpret_cast<const uint8_t *>(P.c_data) + er * 64) + ch);
        r.v.x = c.x;
        r.v.y = c.y;
        r.s = __ldg(P.c_scale + er);
        r.kind = kChFp8;
    }
}

// chunk ch of FP8 ring row `slot` (of all sequences' rows)
__device__ __forceinline__ void load_win8_chunk(const CsaTcParams &P, int64_t slot, int ch, RawChunk &r) {
    const uint8_t *row = reinterpret_cast<const uint8_t *>(P.win) + slot * kFp8WinRowBytes;
    const uint2 c = __ldg(reinterpret_cast<const uint2 *>(row) + ch);
    r.v.x = c.x;
    r.v.y = c.y;
    r.s = __ldg(reinterpret_cast<const float *>(row + 128));
    r.kind = kChFp8;
}

// bulk copy shared -> global (both 16-byte aligned, size a multiple of 16), bulk-group tracked
__device__ __forceinline__ void bulk_store(void *dst, uint32_t src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src), "r"(bytes)
                 : "memory");
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_read_all() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Transposed warp reduction of 32 values per lane: afterwards lane L holds the reduction of
// value L over the 32 lanes (the upper half of the lanes keeps the upper half of the values at
// every step, so the surviving index is the lane number). OP: 0 = max, 1 = sum.
template <int OP>
__device__ __forceinline__ float warp_transpose_reduce(float (&v)[32], int lane) {
#pragma unroll
    for (int step = 0; step < 5; ++step) {
        const int o = 16 >> step;
        const int w = 32 >> (step + 1);  // values kept after this step
        const bool upper = (lane & o) != 0;
#pragma unroll
        for (int j = 0; j < w; ++j) {
            const float keep = upper ? v[j + w] : v[j];
            const float send = upper ? v[j] : v[j + w];
            const float got = __shfl_xor_sync(0xffffffffu, send, o);
            v[j] = OP == 0 ? fmaxf(keep, got) : keep + got;
        }
    }
    return v[0];
}

// The same for 16 values: after four halving steps lanes 2i and 2i+1 hold value i over their
// half of the warp, and one more exchange combines the halves.
__device__ __forceinline__ float warp_transpose_max16(float (&v)[16], int lane) {
#pragma unroll
    for (int step = 0; step < 4; ++step) {
        const int o = 16 >> step;
        const int w = 16 >> (step + 1);
        const bool upper = (lane & o) != 0;
#pragma unroll
        for (int j = 0; j < w; ++j) {
            const float keep = upper ? v[j + w] : v[j];
            const float send = upper ? v[j] : v[j + w];
            v[j] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, o));
        }
    }
    return fmaxf(v[0], __shfl_xor_sync(0xffffffffu, v[0], 1));
}

}  // namespace

template <int kNB>
__global__ void __launch_bounds__(csa_tc::kThreads, 1) csa_tc_kernel(const __grid_constant__ CsaTcParams P) {
    using namespace csa_tc;
    constexpr int kPOff = p_off(kNB), kOutOff = out_off(kNB), kIdxOff = idx_off(kNB);
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    // mbarriers
    __shared__ __align__(8) uint64_t b_qraw[2], b_qfull[2], b_qempty[2];
    __shared__ __align__(8) uint64_t b_kfull[kNB], b_kempty[kNB];
    __shared__ __align__(8) uint64_t b_sfull[kSSlots], b_sempty[kSSlots], b_pfull[2], b_pempty[2];
    __shared__ __align__(8) uint64_t b_ofull[2], b_oempty[2];
    __shared__ uint32_t tmem_slot;
    __shared__ TokenMeta meta[2];
    __shared__ __align__(16) float s_m[kH];   // running max per head (log2 units)
    __shared__ __align__(16) float s_f[kH];   // rescale factor per head of the current update
    __shared__ float s_red[8][32];            // cross-warp reduction scratch
    __shared__ __align__(16) float s_fo[kH];  // final output factor per head
    __shared__ int s_cnt[3];                  // producer warps' counts of valid top-k entries
    __shared__ float4 s_rope[16];             // RoPE (cos, sin) pairs of the current token

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
            // threads have copied the token's metadata
            mbar_init(smem_u32(&b_qempty[i]), 1 + kSoftmax);
            mbar_init(smem_u32(&b_pfull[i]), kSoftmax);
            mbar_init(smem_u32(&b_pempty[i]), 1);
            mbar_init(smem_u32(&b_ofull[i]), 1);
            mbar_init(smem_u32(&b_oempty[i]), kSoftmax);
        }
        for (int i = 0; i < kNB; ++i) {
            mbar_init(smem_u32(&b_kfull[i]), kProducers);
            mbar_init(smem_u32(&b_kempty[i]), 1);
        }
        for (int i = 0; i < kSSlots; ++i) {
            mbar_init(smem_u32(&b_sfull[i]), 1);
            mbar_init(smem_u32(&b_sempty[i]), kSoftmax);
        }
        mbar_fence_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    pdl_trigger();
    pdl_wait();
    const uint32_t tmem = tmem_slot;
    bool ok = true;

    if (tid >= kProd0) {
        // =============================== producers ===============================
        const int ptid = tid - kProd0;
        // a wait whose outcome is the same for all producer threads (a timeout in one makes
        // them all leave together, so no named barrier is left short of threads)
        auto pwait = [&](uint32_t bar, uint32_t par) -> bool {
            const bool w = mbar_wait(bar, par, kWaitNs, &g_abort);
            return !named_sync_or(kBarProd, kProducers, !w);
        };
        int n = 0;           // global tile item counter
        // Fetch of a token's top-k row (bulk copy) and query rows (TMA) into slot it & 1, issued
        // by one thread as early as the slot is free, so it overlaps the previous token.
        auto fetch = [&](int it2) {
            const int item2 = (int)blockIdx.x + it2 * (int)gridDim.x;
            const int row2 = P.split ? item2 / P.S : item2;  // query row (token) of the item
            const int qs2 = it2 & 1;
            const uint32_t qb = smem_u32(&b_qraw[qs2]);
            mbar_expect_tx(qb, 2 * kH * 128 + (P.dense ? 0 : P.topk * 4));
            if (!P.dense)
                bulk_load(s_base + kIdxOff + qs2 * P.topk * 4, P.idx + (int64_t)row2 * P.topk, P.topk * 4, qb);
            tma_load_3d(s_base + kQOff + qs2 * 16384, &P.mq, qb, 0, row2 * kH, 0);
            tma_load_3d(s_base + kQOff + qs2 * 16384 + 8192, &P.mq, qb, 64, row2 * kH, 0);
        };
        int fetched = 0;  // tokens whose fetch has been issued
        int landed = 0;   // tokens whose fetch has been waited for
        if (ptid == 0 && n_tok_cta > 0) {
            fetch(0);
            fetched = 1;
        }
        for (int it = 0; it < n_tok_cta && ok; ++it) {
            const int row = (int)blockIdx.x + it * (int)gridDim.x;
            const int qs = it & 1;
            if (ptid == 0 && fetched == it) {  // not prefetched: the slot must be free first
                if (it >= 2 && !mbar_wait(smem_u32(&b_qempty[qs]), ((it >> 1) - 1) & 1, kWaitNs, &g_abort)) ok = false;
                if (ok) {
                    fetch(it);
                    fetched = it + 1;
                }
            }
            if (named_sync_or(kBarProd, kProducers, !ok)) { ok = false; break; }
            int b, t;
            if (P.decode) {
                b = P.split ? row / P.S : row;
                t = P.ctx[b] - 1;
            } else {
                b = row / P.L;
                t = row % P.L;
            }
            const bool pos_ok = t >= 0 && t < P.L;
            if (!pos_ok && ptid == 0) set_status(CSA_ERR_BOUNDS);
            if (!pwait(smem_u32(&b_qraw[qs]), (it >> 1) & 1)) { ok = false; break; }
            landed = it + 1;
            // count the valid prefix of the top-k row (ascending, -1 padded) in parallel
            const int32_t *sidx = reinterpret_cast<const int32_t *>(sm + kIdxOff) + qs * P.topk;
            if (ptid < 16)  // the token's row of the RoPE table, staged for the query rotation below
                s_rope[ptid] = pos_ok ? __ldg(reinterpret_cast<const float4 *>(P.rope + (int64_t)t * 32) + ptid)
                                      : make_float4(1.0f, 0.0f, 1.0f, 0.0f);
            int cnt = 0;
            if (!P.dense)
                for (int i = ptid; i < P.topk; i += kProducers) cnt += (pos_ok && sidx[i] >= 0) ? 1 : 0;
            cnt = __reduce_add_sync(0xffffffffu, cnt);
            if ((ptid & 31) == 0) s_cnt[ptid >> 5] = cnt;
            named_sync(kBarProd, kProducers);
            TokenMeta mt;
            mt.n_sel = P.dense ? (pos_ok ? visible_entries(t, P.m, P.ncap) : 0) : s_cnt[0] + s_cnt[1] + s_cnt[2];
            mt.n_ct = (mt.n_sel + kTile - 1) / kTile;
            mt.t = t;
            mt.b = b;
            mt.n_win_t = pos_ok ? min(P.n_win, t + 1) : 0;
            mt.pos_ok = pos_ok;
            mt.c0 = 0;
            mt.n_tiles = mt.n_ct + 1;
            if (P.split) {
                const int c0 = (row % P.S) * P.T;
                if (c0 < mt.n_ct + 1) {
                    mt.c0 = c0;
                    mt.n_tiles = min(P.T, mt.n_ct + 1 - c0);
                } else {  // nothing left for this split: one fully masked tile (no key is valid)
                    mt.c0 = mt.n_ct;
                    mt.n_tiles = 1;
                    mt.n_win_t = 0;
                }
            }
            if (ptid == 0) meta[qs] = mt;
            // RoPE on dims 64..127 at position t: head h, chunk pair (c, c+4) of the second half
            if (P.d_rope == 64 && pos_ok) {
                uint8_t *q1 = sm + kQOff + qs * 16384 + 8192;
                for (int u = ptid; u < kH * 4; u += kProducers) {
                    const int h = u >> 2, c = u & 3;
                    float4 rc[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) rc[e] = s_rope[4 * c + e];  // (cos, sin) of pairs 8c .. 8c+7
                    uint4 *pa = reinterpret_cast<uint4 *>(q1 + sw128_off(h, c));
                    uint4 *pb = reinterpret_cast<uint4 *>(q1 + sw128_off(h, c + 4));
                    uint4 va = *pa, vb = *pb;
                    __nv_bfloat162 *a2 = reinterpret_cast<__nv_bfloat162 *>(&va);
                    __nv_bfloat162 *b2 = reinterpret_cast<__nv_bfloat162 *>(&vb);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 x = __bfloat1622float2(a2[e]);
                        const float2 y = __bfloat1622float2(b2[e]);
                        const float4 cs = rc[e];  // (cos, sin) of pair 8c + 2e and 8c + 2e + 1
                        a2[e] = __floats2bfloat162_rn(x.x * cs.x - y.x * cs.y, x.y * cs.z - y.y * cs.w);
                        b2[e] = __floats2bfloat162_rn(x.x * cs.y + y.x * cs.x, x.y * cs.w + y.y * cs.z);
                    }
                    *pa = va;
                    *pb = vb;
                }
            }
            fence_async_smem();
            mbar_arrive(smem_u32(&b_qfull[qs]));
            // key tiles of this item: compressed tiles, then the window tile
            for (int cl = 0; cl < mt.n_tiles; ++cl, ++n) {
                const int c = mt.c0 + cl;
                const int kb = n % kNB;
                if (n >= kNB && !pwait(smem_u32(&b_kempty[kb]), ((n / kNB) - 1) & 1)) {
                    ok = false;
                    break;
                }
                uint8_t *kbuf = sm + kKOff + kb * 32768;
                const uint32_t kbuf_s = s_base + kKOff + kb * 32768;
                const uint32_t kf = smem_u32(&b_kfull[kb]);
                if (c < mt.n_ct && P.ent == 0) {
                    // gathered BF16 rows; an invalid slot reads nothing and is zero-filled (its
                    // weight is masked to 0 by the softmax). 96 threads: thread = chunk ch of keys
                    // i0 + 6q; all indices are read first so that the copies issue back to back.
                    static_assert(kProducers == 96 && kTile * 16 <= kProducers * kGatherPer, "gather split");
                    const int ch = ptid & 15, i0 = ptid >> 4;
                    int jj[kGatherPer];
                    bool bad = false;
#pragma unroll
                    for (int q = 0; q < kGatherPer; ++q) {
                        const int i = i0 + 6 * q;
                        const int pos = c * kTile + i;
                        const int j = (i < kTile && pos < mt.n_sel) ? (P.dense ? pos : sidx[pos]) : -1;
                        bad |= j >= P.ncap;
                        jj[q] = j >= P.ncap ? -1 : j;
                    }
                    if (bad) set_status(CSA_ERR_BOUNDS);
                    const __nv_bfloat16 *cbase =
                        reinterpret_cast<const __nv_bfloat16 *>(P.c_data) + (int64_t)mt.b * P.ncap * 128 + ch * 8;
                    const uint32_t dbase = kbuf_s + (ch >> 3) * 16384;
#pragma unroll
                    for (int q = 0; q < kGatherPer; ++q) {
                        const int i = i0 + 6 * q;
                        if (i < kTile) {
                            const int j = jj[q];
                            cp_async16_zfill(dbase + sw128_off(i, ch & 7), cbase + (int64_t)(j < 0 ? 0 : j) * 128,
                                             j < 0 ? 0u : 16u);
                        }
                    }
                    cp_async_mbar_arrive(kf);
                } else if (c < mt.n_ct || P.win8) {
                    // decode tiles in a low-precision store (MIXED / NVFP4 entries, an FP8 ring):
                    // widened by the threads; chunk u = ptid + 96 q (the BF16 gather's mapping),
                    // the loads of kConvBatch chunks issued before any is converted
                    const bool ents = c < mt.n_ct;
                    bool bad = false;
                    for (int q0 = 0; q0 < kGatherPer; q0 += kConvBatch) {
                        RawChunk r[kConvBatch];
#pragma unroll
                        for (int q = 0; q < kConvBatch; ++q) {
                            const int u = ptid + kProducers * (q0 + q);
                            r[q].kind = kChZero;
                            if (q0 + q >= kGatherPer || u >= kTile * 16) continue;
                            const int i = u >> 4, ch = u & 15;
                            if (ents) {
                                const int pos = c * kTile + i;
                                const int j = pos < mt.n_sel ? (P.dense ? pos : sidx[pos]) : -1;
                                bad |= j >= P.ncap;
                                if (j >= 0 && j < P.ncap) load_entry_chunk(P, (int64_t)mt.b * P.ncap + j, ch, r[q]);
                            } else {
                                const int uu = mt.t - kTile + 1 + i;  // position of window row i
                                if (!(uu < 0 || uu <= mt.t - mt.n_win_t))
                                    load_win8_chunk(P, (int64_t)mt.b * P.n_win + uu % P.n_win, ch, r[q]);
                            }
                        }
#pragma unroll
                        for (int q = 0; q < kConvBatch; ++q) {
                            const int u = ptid + kProducers * (q0 + q);
                            if (q0 + q >= kGatherPer || u >= kTile * 16) continue;
                            const int i = u >> 4, ch = u & 15;
                            *reinterpret_cast<uint4 *>(kbuf + (ch >> 3) * 16384 + sw128_off(i, ch & 7)) =
                                widen_chunk(r[q]);
                        }
                    }
                    if (bad) set_status(CSA_ERR_BOUNDS);
                    fence_async_smem();
                    mbar_arrive(kf);
                } else if (!P.decode) {
                    // window rows [t - 127, t] of sequence b by TMA (rows before 0 read as zeros)
                    if (ptid == 0) {
                        mbar_expect_tx_only(kf, 2 * kTile * 128);
                        tma_load_3d(kbuf_s, &P.mkv, kf, 0, mt.t - kTile + 1, mt.b);
                        tma_load_3d(kbuf_s + 16384, &P.mkv, kf, 64, mt.t - kTile + 1, mt.b);
                    }
                    mbar_arrive(kf);
                } else {
                    // decode: window rows from the ring, row u at slot u mod n_win
                    for (int u = ptid; u < kTile * 16; u += kProducers) {
                        const int i = u >> 4, ch = u & 15;
                        const int uu = mt.t - kTile + 1 + i;  // position of key row i
                        const bool have = !(uu < 0 || uu <= mt.t - mt.n_win_t);
                        const int64_t slot = have ? (uu % P.n_win) : 0;
                        cp_async16_zfill(kbuf_s + (ch >> 3) * 16384 + sw128_off(i, ch & 7),
                                         reinterpret_cast<const __nv_bfloat16 *>(P.win) +
                                             ((int64_t)mt.b * P.n_win + slot) * 128 + ch * 8,
                                         have ? 16u : 0u);
                    }
                    cp_async_mbar_arrive(kf);
                }
                // fetch the next token's rows once its slot is free (never blocking here)
                if (ptid == 0 && fetched == it + 1 && it + 1 < n_tok_cta &&
                    (it + 1 < 2 || mbar_test_wait(smem_u32(&b_qempty[(it + 1) & 1]), (((it + 1) >> 1) - 1) & 1))) {
                    fetch(it + 1);
                    fetched = it + 2;
                }
            }
        }
        // all copies of this thread have landed before the CTA may exit
        cp_async_wait_all();
        // after a failure: let copies still in flight into this CTA's shared memory land
        // (bounded) before the CTA exits
        if (!ok && ptid == 0)
            for (int f = landed; f < fetched; ++f) mbar_wait(smem_u32(&b_qraw[f & 1]), (f >> 1) & 1, kDrainNs);
    } else if (warp == kMmaWarp) {
        // =============================== MMA issue ===============================
        if (lane == 0) {
            const uint32_t idesc_s = idesc_bf16(128, kH, 0, 0);  // S^T = K Q^T
            const uint32_t idesc_o = idesc_bf16(128, kH, 1, 1);  // O^T = V^T P^T, both MN-major
            // descriptors of the buffers' first rows; within a buffer the start-address field
            // advances by (byte offset >> 4), which never carries out of the field (< 256 KB)
            const uint64_t dK0 = sdesc_sw128(s_base + kKOff, 16, 1024);     // key tile, K-major (S)
            const uint64_t dQ0 = sdesc_sw128(s_base + kQOff, 16, 1024);     // query rows, K-major
            const uint64_t dV0 = sdesc_sw128(s_base + kKOff, 16384, 1024);  // key tile, MN-major (P V)
            const uint64_t dP0 = sdesc_sw128(s_base + kPOff, 16384, 1024);  // P^T, MN-major
            // P V items waiting for their P^T, issued kLag = 2 tiles behind the S^T MMAs so that the
            // tensor pipe holds queued S^T work while the softmax finishes an earlier tile. Items
            // are consecutive tiles from pv_n on; pend0..2 hold (token << 2 | last << 1 | first).
            static_assert(kLag == 2, "three pending slots");
            int pv_n = 0, npend = 0, pend0 = 0, pend1 = 0, pend2 = 0;
            auto issue_pv = [&]() -> bool {
                const int pn = pv_n, fl = pend0, tok = pend0 >> 2;
                pend0 = pend1;
                pend1 = pend2;
                --npend;
                ++pv_n;
                const bool first = (fl & 1) != 0, last = (fl & 2) != 0;
                const int pb = pn & 1, ob = tok & 1;
                if (!mbar_wait(smem_u32(&b_pfull[pb]), (pn >> 1) & 1, kWaitNs, &g_abort)) return false;
                if (first && tok >= 2 && !mbar_wait(smem_u32(&b_oempty[ob]), ((tok >> 1) - 1) & 1, kWaitNs, &g_abort))
                    return false;
                tc_fence_after();
                const uint64_t ad = dV0 + (uint64_t)(((pn % kNB) * 32768) >> 4);
                const uint64_t bd = dP0 + (uint64_t)((pb * 16384) >> 4);
                const uint32_t d = tmem + kOCol + ob * kH;
                mma_bf16(d, ad, bd, idesc_o, first ? 0u : 1u);
#pragma unroll
                for (int kk = 1; kk < 8; ++kk) mma_bf16(d, ad + (kk * 2048 >> 4), bd + (kk * 2048 >> 4), idesc_o, 1u);
                mma_commit(smem_u32(&b_pempty[pb]));
                mma_commit(smem_u32(&b_kempty[pn % kNB]));
                if (last) mma_commit(smem_u32(&b_ofull[ob]));
                return true;
            };
            int n = 0;
            for (int it = 0; it < n_tok_cta && ok; ++it) {
                const int qs = it & 1;
                if (!mbar_wait(smem_u32(&b_qfull[qs]), (it >> 1) & 1, kWaitNs, &g_abort)) { ok = false; break; }
                const int n_tiles = meta[qs].n_tiles;
                const uint64_t bq = dQ0 + (uint64_t)((qs * 16384) >> 4);
                for (int c = 0; c < n_tiles; ++c, ++n) {
                    const int kb = n % kNB, sb = n % kSSlots;
                    if (!mbar_wait(smem_u32(&b_kfull[kb]), (n / kNB) & 1, kWaitNs, &g_abort)) { ok = false; break; }
                    if (n >= kSSlots &&
                        !mbar_wait(smem_u32(&b_sempty[sb]), ((n / kSSlots) - 1) & 1, kWaitNs, &g_abort)) {
                        ok = false;
                        break;
                    }
                    // the gathered rows were written by cp.async (generic proxy) and observed through
                    // the barrier; order them before the tensor core's reads (async proxy)
                    fence_async_smem();
                    tc_fence_after();
                    const uint64_t ak = dK0 + (uint64_t)((kb * 32768) >> 4);
                    const uint32_t d = tmem + kSCol + sb * kH;
                    mma_bf16(d, ak, bq, idesc_s, 0u);
#pragma unroll
                    for (int kk = 1; kk < 8; ++kk) {
                        const uint32_t off_k = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
                        const uint32_t off_q = ((kk >> 2) * 8192 + (kk & 3) * 32) >> 4;
                        mma_bf16(d, ak + off_k, bq + off_q, idesc_s, 1u);
                    }
                    mma_commit(smem_u32(&b_sfull[sb]));
                    if (c == n_tiles - 1) mma_commit(smem_u32(&b_qempty[qs]));
                    const int item = (it << 2) | (c == n_tiles - 1 ? 2 : 0) | (c == 0 ? 1 : 0);
                    if (npend == 0) pend0 = item;
                    else if (npend == 1) pend1 = item;
                    else pend2 = item;
                    ++npend;
                    if (npend > kLag && !issue_pv()) { ok = false; break; }
                }
            }
            while (ok && npend > 0) ok = issue_pv();
            if (!ok) set_timeout();
        }
    } else {
        // ============================ softmax + epilogue ============================
        const int wg = warp >> 2;                 // warpgroup: heads [32 wg, 32 wg + 32)
        const int kl = 32 * (warp & 3) + lane;    // this thread's key (TMEM lane) / output dim
        const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
        const uint32_t bar_wg = kBarWG0 + wg;
        const int h0 = 32 * wg;
        // Every wait result is kept in okl and acted upon only through an OR-reduction over all
        // softmax threads (once per token), so that all of them leave together and no named
        // barrier is ever left short of threads; a failed wait raises the abort flag at once, so
        // the remaining waits of the token return early.
        bool okl = true;
        auto note = [&](bool w) {
            if (!w && okl) set_timeout();
            okl = okl && w;
        };
        float lpart[32];
        int n = 0;
        // The O part of a token's epilogue (wait for its last P V, normalise, inverse RoPE,
        // store) is deferred until the next token's first tile has been handed to the MMA warp,
        // so the softmax threads do not idle while that P V runs. State of the deferred token:
        int pend_it = -1, pend_t = 0, pend_b = 0, pend_ok = 0;
        // returns false (in every softmax thread alike) after a failed wait
        auto o_epilogue = [&]() -> bool {
            const int ob = pend_it & 1;
            note(mbar_wait(smem_u32(&b_ofull[ob]), (pend_it >> 1) & 1, kWaitNs, &g_abort));
            if (named_sync_or(kBarSoftmax, kSoftmax, !okl)) return false;
            tc_fence_after();
            float o[32];
            tmem_ld32_sync(tmem + lane_base + kOCol + ob * kH + h0, o);  // lane kl = output dim
            tc_fence_before();
            mbar_arrive(smem_u32(&b_oempty[ob]));
            if (P.split) {
                // unnormalised partial O of this item: [head][dim], dims across the warp's lanes
                float *po = P.part_o + (((int64_t)blockIdx.x + (int64_t)pend_it * gridDim.x) * kH + h0) * 128 + kl;
#pragma unroll
                for (int e = 0; e < 32; ++e) __stcg(po + e * 128, o[e]);
                return true;
            }
            {
                const float4 *f4 = reinterpret_cast<const float4 *>(s_fo + h0);
#pragma unroll
                for (int e4 = 0; e4 < 8; ++e4) {
                    const float4 ff = f4[e4];
                    o[4 * e4] *= ff.x;
                    o[4 * e4 + 1] *= ff.y;
                    o[4 * e4 + 2] *= ff.z;
                    o[4 * e4 + 3] *= ff.w;
                }
            }
            // the staging buffer: the previous token's bulk store must have finished reading it
            if (tid == 0) bulk_wait_read_all();
            named_sync(kBarSoftmax, kSoftmax);
            if (P.d_rope == 64 && kl >= 64) {
                // dims 64 + i (warp 2) and 96 + i (warp 3) of a pair meet in the staging buffer
                const int half = (kl >> 5) & 1, i = kl & 31;
                float *x = reinterpret_cast<float *>(sm + kOutOff) + wg * 2048;
#pragma unroll
                for (int e = 0; e < 32; ++e) x[half * 1024 + e * 32 + i] = o[e];
                named_sync(kBarWG0 + 2 + wg, 64);  // warps 2 and 3 of this warpgroup
                const float2 cs = pend_ok ? P.rope[(int64_t)pend_t * 32 + i] : make_float2(1.0f, 0.0f);
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const float other = x[(half ^ 1) * 1024 + e * 32 + i];
                    o[e] = half == 0 ? o[e] * cs.x + other * cs.y : -other * cs.y + o[e] * cs.x;
                }
            }
            named_sync(kBarSoftmax, kSoftmax);  // the exchange is read before the staging writes
            {
                __nv_bfloat16 *os = reinterpret_cast<__nv_bfloat16 *>(sm + kOutOff);  // [h][d]
#pragma unroll
                for (int e = 0; e < 32; ++e) os[(h0 + e) * 128 + kl] = __float2bfloat16_rn(o[e]);
            }
            fence_async_smem();
            named_sync(kBarSoftmax, kSoftmax);
            if (tid == 0 && pend_ok) {
                const int64_t orow = P.decode ? (int64_t)pend_b : (int64_t)pend_b * P.L + pend_t;
                bulk_store(P.out + orow * kH * 128, s_base + kOutOff, kH * 128 * 2);
            }
            return true;
        };
        bool failed = false;
        for (int it = 0; it < n_tok_cta; ++it) {
            const int qs = it & 1;
            note(mbar_wait(smem_u32(&b_qfull[qs]), (it >> 1) & 1, kWaitNs, &g_abort));
            // each warpgroup's first warp resets its own heads' maxima: the same warp read them
            // last, in the previous token's reduction (the warpgroups are not in step there)
            if ((warp & 3) == 0) s_m[h0 + lane] = -INFINITY;
            if (named_sync_or(kBarSoftmax, kSoftmax, !okl)) break;
            const TokenMeta mt = meta[qs];
            mbar_arrive(smem_u32(&b_qempty[qs]));
            const int n_tiles = mt.n_tiles;
#pragma unroll
            for (int e = 0; e < 32; ++e) lpart[e] = 0.0f;
            for (int cl = 0; cl < n_tiles; ++cl, ++n) {
                const int c = mt.c0 + cl;
                const int sb = n % kSSlots, pb = n & 1;
                note(mbar_wait(smem_u32(&b_sfull[sb]), (n / kSSlots) & 1, kWaitNs, &g_abort));
                tc_fence_after();
                const uint32_t s_addr = tmem + lane_base + kSCol + sb * kH + h0;
                // key validity of this thread's key (TMEM lane = key within the tile)
                bool valid;
                if (c < mt.n_ct) valid = c * kTile + kl < mt.n_sel;
                else valid = kl >= kTile - mt.n_win_t;  // key row kl is position t - 127 + kl
                // p = exp2(scale * s - m) with the current maxima; the S^T slot stays held until
                // the P^T row is written, so the rare slow path can read the logits again. A
                // token's first tile always takes the slow path (no maximum yet): its speculative
                // pass is skipped.
                float p[32];
                bool over = cl == 0;
                if (cl > 0) {
                    tmem_ld32_sync(s_addr, p);
                    const float4 *m4 = reinterpret_cast<const float4 *>(s_m + h0);
                    if (__all_sync(0xffffffffu, valid)) {
                        // every key of the warp valid: two logits per packed FMA
                        const uint64_t sc2 = f2_pack(P.scale_log2, P.scale_log2);
#pragma unroll
                        for (int e4 = 0; e4 < 8; ++e4) {
                            const float4 mm = m4[e4];
                            const float2 x01 = f2_unpack(f2_fma(f2_pack(p[4 * e4], p[4 * e4 + 1]), sc2, f2_pack(-mm.x, -mm.y)));
                            const float2 x23 =
                                f2_unpack(f2_fma(f2_pack(p[4 * e4 + 2], p[4 * e4 + 3]), sc2, f2_pack(-mm.z, -mm.w)));
                            over |= x01.x > kOver;
                            over |= x01.y > kOver;
                            over |= x23.x > kOver;
                            over |= x23.y > kOver;
                            p[4 * e4] = fast_exp2(x01.x);
                            p[4 * e4 + 1] = fast_exp2(x01.y);
                            p[4 * e4 + 2] = fast_exp2(x23.x);
                            p[4 * e4 + 3] = fast_exp2(x23.y);
                        }
                    } else {
#pragma unroll
                        for (int e4 = 0; e4 < 8; ++e4) {
                            const float4 mm = m4[e4];
                            const float mv[4] = {mm.x, mm.y, mm.z, mm.w};
#pragma unroll
                            for (int q = 0; q < 4; ++q) {
                                const float x = valid ? fmaf(p[4 * e4 + q], P.scale_log2, -mv[q]) : -INFINITY;
                                over |= x > kOver;
                                p[4 * e4 + q] = fast_exp2(x);
                            }
                        }
                    }
                }
                if (n >= 2) note(mbar_wait(smem_u32(&b_pempty[pb]), ((n >> 1) - 1) & 1, kWaitNs, &g_abort));
                // the warpgroup owns its heads' maxima: the decision is the warpgroup's (rare: a
                // first tile or a jump of the maximum)
                over = named_sync_or(bar_wg, 128, over);
                if (over) {
                    // per-head maximum of this tile over the warpgroup's 128 keys, 16 heads at a time
#pragma unroll 1
                    for (int c0 = 0; c0 < 32; c0 += 16) {
                        float v[16];
                        tmem_ld16_sync(s_addr + c0, v);
#pragma unroll
                        for (int e = 0; e < 16; ++e) v[e] = valid ? v[e] * P.scale_log2 : -INFINITY;
                        const float wmax = warp_transpose_max16(v, lane);  // head c0 + lane / 2
                        if ((lane & 1) == 0) s_red[warp][c0 + (lane >> 1)] = wmax;
                    }
                    named_sync(bar_wg, 128);
                    if ((warp & 3) == 0) {
                        const int h = h0 + lane;
                        const float mnew = fmaxf(fmaxf(s_red[4 * wg][lane], s_red[4 * wg + 1][lane]),
                                                 fmaxf(s_red[4 * wg + 2][lane], s_red[4 * wg + 3][lane]));
                        const float mold = s_m[h];
                        float f = 1.0f;
                        if (mnew > mold + kOver) {
                            f = exp2f(mold - mnew);  // 0 when mold is -inf
                            s_m[h] = mnew;
                        }
                        s_f[h] = f;
                    }
                    named_sync(bar_wg, 128);
                    bool rescale_o = false;
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        const float f = s_f[h0 + e];
                        lpart[e] *= f;
                        rescale_o |= f != 1.0f;
                    }
                    rescale_o = cl > 0 && named_sync_or(bar_wg, 128, rescale_o);
                    if (rescale_o) {
                        // O^T holds the P V of the previous tiles of this token: wait for the last
                        note(mbar_wait(smem_u32(&b_pempty[(n - 1) & 1]), ((n - 1) >> 1) & 1, kWaitNs, &g_abort));
                        tc_fence_after();
#pragma unroll 1
                        for (int c0 = 0; c0 < 32; c0 += 16) {
                            float o[16];
                            tmem_ld16_sync(tmem + lane_base + kOCol + (it & 1) * kH + h0 + c0, o);
#pragma unroll
                            for (int e = 0; e < 16; ++e) o[e] *= s_f[h0 + c0 + e];
                            tmem_st16(tmem + lane_base + kOCol + (it & 1) * kH + h0 + c0, o);
                        }
                        tmem_st_wait();
                    }
                    tmem_ld32_sync(s_addr, p);
                    const float4 *m4 = reinterpret_cast<const float4 *>(s_m + h0);
#pragma unroll
                    for (int e4 = 0; e4 < 8; ++e4) {
                        const float4 mm = m4[e4];
                        const float mv[4] = {mm.x, mm.y, mm.z, mm.w};
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            p[4 * e4 + q] = fast_exp2(valid ? fmaf(p[4 * e4 + q], P.scale_log2, -mv[q]) : -INFINITY);
                    }
                }
                // the logits are no longer needed: release the S^T slot
                tc_fence_before();
                mbar_arrive(smem_u32(&b_sempty[sb]));
                // P^T row of this key: chunks 4 wg .. 4 wg + 3 (heads h0 .. h0 + 31), BF16
                uint8_t *prow = sm + kPOff + pb * 16384;
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4) {
                    uint32_t pk[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int h = 8 * c4 + 2 * e;
                        const float2 l2 = f2_unpack(f2_add(f2_pack(lpart[h], lpart[h + 1]), f2_pack(p[h], p[h + 1])));
                        lpart[h] = l2.x;
                        lpart[h + 1] = l2.y;
                        pk[e] = pack2(p[h], p[h + 1]);
                    }
                    *reinterpret_cast<uint4 *>(prow + sw128_off(kl, 4 * wg + c4)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                }
                fence_async_smem();
                tc_fence_before();
                mbar_arrive(smem_u32(&b_pfull[pb]));
                if (cl == 0 && pend_it >= 0) {
                    if (!o_epilogue()) {
                        failed = true;
                        break;
                    }
                    pend_it = -1;
                }
            }
            if (failed) break;
            // ---- epilogue of the token: reduce the sums into the per-head output factors; the
            // O part follows with the next token's first tile (or after the last token) ----
            {
                const float lsum = warp_transpose_reduce<1>(lpart, lane);
                s_red[warp][lane] = lsum;
            }
            named_sync(bar_wg, 128);
            if ((warp & 3) == 0) {
                const int h = h0 + lane;
                const float l = (s_red[4 * wg][lane] + s_red[4 * wg + 1][lane]) +
                                (s_red[4 * wg + 2][lane] + s_red[4 * wg + 3][lane]);
                const float m = s_m[h];
                float f = 1.0f;
                if (P.split) {
                    // the combine step merges the items of the sequence and applies the sink
                    P.part_ml[((int64_t)blockIdx.x + (int64_t)it * gridDim.x) * kH + h] = make_float2(m, l);
                } else if (P.sink) {
                    const float s2 = P.sink[h] * 1.4426950408889634f;
                    const float mf = fmaxf(m, s2);
                    f = exp2f(m - mf) / (l * exp2f(m - mf) + exp2f(s2 - mf));
                } else {
                    f = 1.0f / l;
                }
                s_fo[h] = f;
                if (P.lse && mt.pos_ok && !P.split)
                    P.lse[(int64_t)((P.decode ? mt.b : (int64_t)mt.b * P.L + mt.t)) * kH + h] =
                        (m + log2f(l)) * 0.6931471805599453f;
            }
            pend_it = it;
            pend_t = mt.t;
            pend_b = mt.b;
            pend_ok = mt.pos_ok;
        }
        if (!failed && pend_it >= 0) o_epilogue();
        if (tid == 0) bulk_wait_all();
        if (!okl) set_timeout();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

// MIXED or NVFP4 entries widened to BF16 rows (the dequantised value rounded to nearest even):
// MIXED dims [0, 64) = code * row scale, dims [64, 128) copied; NVFP4 every dim = E2M1 * block
// scale. Thread = one 16-byte output chunk.
__global__ void widen_entries_kernel(const uint8_t *__restrict__ codes, const __nv_bfloat16 *__restrict__ rope,
                                     const float *__restrict__ scale, int64_t rows, int nvfp4,
                                     __nv_bfloat16 *__restrict__ out) {
    const int64_t n = rows * 16;
    for (int64_t u = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; u < n; u += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = u >> 4;
        const int ch = (int)(u & 15);
        uint4 v;
        if (nvfp4) {
            const uint8_t *row = codes + r * kNvfp4RowBytes;
            v = fp4x8_to_bf16(reinterpret_cast<const uint32_t *>(row)[ch], row[64 + (ch >> 1)],
                              *reinterpret_cast<const float *>(row + 72));
        } else if (ch >= 8) {
            v = *reinterpret_cast<const uint4 *>(rope + r * 64 + (ch - 8) * 8);
        } else {
            const uint2 cw = *reinterpret_cast<const uint2 *>(codes + r * 64 + ch * 8);
            v = fp8x8_to_bf16(cw.x, cw.y, scale[r]);
        }
        *reinterpret_cast<uint4 *>(out + r * 128 + ch * 8) = v;
    }
}

size_t csa_widen_bytes(const AttnArgs &a) {
    return ((a.kv_t == CSA_MIXED || a.kv_t == CSA_NVFP4) && !a.decode) ? (size_t)a.B * (size_t)a.ncap * 128 * 2 : 0;
}

const void *launch_widen_entries(const AttnArgs &a, cudaStream_t st) {
    const int64_t erows = (int64_t)a.B * a.ncap;
    __nv_bfloat16 *wide = reinterpret_cast<__nv_bfloat16 *>(a.ws);
    int blocks = (int)ceil_div64(erows * 16, 256);
    if (blocks > 148 * 8) blocks = 148 * 8;
    if (blocks < 1) blocks = 1;
    widen_entries_kernel<<<blocks, 256, 0, st>>>(reinterpret_cast<const uint8_t *>(a.c_data),
                                                reinterpret_cast<const __nv_bfloat16 *>(a.c_rope), a.c_scale, erows,
                                                a.kv_t == CSA_NVFP4 ? 1 : 0, wide);
    count_launches(1);
    return wide;
}

bool csa_tc_supported(const AttnArgs &a) {
    if (a.act_t != CSA_BF16) return false;
    if (a.kv_t != CSA_BF16 && a.kv_t != CSA_MIXED && a.kv_t != CSA_NVFP4) return false;
    if (a.decode && a.win_t != CSA_BF16 && a.win_t != CSA_FP8E4M3) return false;
    if (a.H != csa_tc::kH || a.n_win != 128) return false;
    if (!a.dense && (a.topk < 4 || a.topk > kMaxTopk || a.topk % 4 != 0)) return false;
    if (a.dense && !a.decode && a.ncap != 0) return false;  // prefill: dense only as window-only (no entries)
    if (a.d_rope != 0 && a.d_rope != 64) return false;
    if (csa_widen_bytes(a) > a.ws_bytes || (csa_widen_bytes(a) > 0 && !a.ws)) return false;
    // outputs are stored with a bulk copy, top-k rows fetched with one: 16-byte aligned
    if ((reinterpret_cast<uintptr_t>(a.out) & 15) != 0) return false;
    return a.dense || (a.idx != nullptr && (reinterpret_cast<uintptr_t>(a.idx) & 15) == 0);
}

bool launch_csa_tc(const AttnArgs &a, cudaStream_t st) {
    using namespace csa_tc;
    if (!csa_tc_supported(a)) return false;
    CsaTcParams P;
    memset(&P, 0, sizeof(P));
    const int qrows = a.decode ? a.B : a.B * a.L;  // query rows (tokens)
    const bool split = a.decode && a.split_S > 0;
    const int rows = split ? a.B * a.split_S : qrows;  // work items
    bool ok = make_map_3d(&P.mq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.q, 128, (uint64_t)qrows * kH, 1, 64, kH,
                          CU_TENSOR_MAP_SWIZZLE_128B);
    if (!a.decode)
        ok = ok && make_map_3d(&P.mkv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.kv_rope, 128, a.L, a.B, 64, kTile,
                               CU_TENSOR_MAP_SWIZZLE_128B);
    if (!ok) return false;
    P.c_data = a.c_data;
    P.c_rope = reinterpret_cast<const __nv_bfloat16 *>(a.c_rope);
    P.c_scale = a.c_scale;
    P.ent = a.kv_t == CSA_MIXED ? 1 : (a.kv_t == CSA_NVFP4 ? 2 : 0);
    if (P.ent != 0 && !a.decode) {
        // prefill: widen every entry once; the attention then gathers BF16 rows
        if (a.ncap > 0) P.c_data = launch_widen_entries(a, st);
        P.c_rope = nullptr;
        P.c_scale = nullptr;
        P.ent = 0;
    }
    P.win = a.decode ? a.kv_rope : nullptr;
    P.win8 = a.decode && a.win_t == CSA_FP8E4M3 ? 1 : 0;
    P.idx = a.idx;
    P.ctx = a.ctx;
    P.sink = a.sink;
    P.rope = reinterpret_cast<const float2 *>(a.rope_tab);
    P.out = reinterpret_cast<__nv_bfloat16 *>(a.out);
    P.lse = a.lse;
    P.B = a.B; P.L = a.L; P.ncap = a.ncap; P.topk = a.topk; P.n_win = a.n_win; P.d_rope = a.d_rope;
    P.decode = a.decode; P.rows = rows;
    P.dense = a.dense; P.m = a.m;
    P.scale_log2 = a.scale * 1.4426950408889634f;
    P.split = split ? 1 : 0;
    P.S = split ? a.split_S : 1;
    P.T = split ? a.split_T : 1;
    P.part_o = a.part_o;
    P.part_ml = a.part_ml;
    int dev = 0, sms = 148, smem_max = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaDeviceGetAttribute(&smem_max, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    const int grid = rows < sms ? rows : sms;
    // four key-tile buffers when they fit next to the top-k rows, else three
    const int static_bytes = 4096;  // barriers, per-head vectors, reduction scratch (upper bound)
    const int idx_bytes = a.dense ? 0 : 2 * a.topk * 4;
    const int smem4 = 1024 + idx_off(4) + idx_bytes;
    const int smem3 = 1024 + idx_off(3) + idx_bytes;
    // decode: a programmatic dependent launch (it overlaps the previous kernel's tail)
    auto go = [&](auto kern, int smem) {
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (a.decode) launch_pdl(kern, grid, kThreads, smem, st, P);
        else kern<<<grid, kThreads, smem, st>>>(P);
    };
    if (smem4 + static_bytes <= smem_max) go(csa_tc_kernel<4>, smem4);
    else go(csa_tc_kernel<3>, smem3);
    count_launches(1);
    return true;
}


// ---------------------------------------------------------------------------------------
// split-KV decode: the plan and the combine step
// ---------------------------------------------------------------------------------------

// Key tiles of a decode token at most (compressed tiles, then the window tile), items per
// sequence S and tiles per item T, sized so that the B * S items fill about two waves of CTAs.
void decode_split_plan(int B, int topk, int ncap, int dense, int *S, int *T) {
    const int tiles = (dense ? (ncap + csa_tc::kTile - 1) / csa_tc::kTile
                             : (topk + csa_tc::kTile - 1) / csa_tc::kTile) + 1;
    int t = (int)ceil_div64((int64_t)tiles * B, 296);
    if (t < 1) t = 1;
    *T = t;
    *S = (tiles + t - 1) / t;
}

size_t decode_partial_bytes(int B, int S) {
    return (size_t)B * S * csa_tc::kH * (128 * sizeof(float) + sizeof(float2));
}

// One warp per (sequence, head): merges the S partial results of the sequence in a fixed order
// (max of the running maxima, rescaled sums and outputs), adds the sink to the denominator,
// normalises, rotates the RoPE half back by the query position and stores BF16. Lane i holds
// dims i, 32 + i, 64 + i and 96 + i, so a RoPE pair (64 + i, 96 + i) sits in one lane.
__global__ void __launch_bounds__(256) decode_combine_kernel(const float *__restrict__ part_o,
                                                             const float2 *__restrict__ part_ml,
                                                             const int32_t *__restrict__ ctx,
                                                             const float *__restrict__ sink,
                                                             const float2 *__restrict__ rope,
                                                             __nv_bfloat16 *__restrict__ out, float *__restrict__ lse,
                                                             int B, int S, int L, int d_rope) {
    pdl_trigger();
    pdl_wait();
    constexpr int kH = csa_tc::kH;
    const int lane = threadIdx.x & 31;
    const int gw = (int)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (gw >= B * kH) return;
    const int b = gw / kH, h = gw % kH;
    const int t = ctx[b] - 1;
    if (t < 0 || t >= L) return;  // reported by the attention kernel; nothing is stored
    const float2 *ml = part_ml + (int64_t)b * S * kH + h;
    float M = -INFINITY;
    for (int s = 0; s < S; ++s) M = fmaxf(M, ml[(int64_t)s * kH].x);
    const float s2 = sink ? sink[h] * 1.4426950408889634f : -INFINITY;
    const float Mf = fmaxf(M, s2);
    float l = 0.0f, o0 = 0.0f, o1 = 0.0f, o2 = 0.0f, o3 = 0.0f;
    for (int s = 0; s < S; ++s) {
        const float2 v = ml[(int64_t)s * kH];
        if (v.x == -INFINITY) continue;  // an item with no valid key
        const float wgt = exp2f(v.x - Mf);
        l = fmaf(v.y, wgt, l);
        const float *po = part_o + (((int64_t)b * S + s) * kH + h) * 128;
        o0 = fmaf(__ldcg(po + lane), wgt, o0);
        o1 = fmaf(__ldcg(po + 32 + lane), wgt, o1);
        o2 = fmaf(__ldcg(po + 64 + lane), wgt, o2);
        o3 = fmaf(__ldcg(po + 96 + lane), wgt, o3);
    }
    const float f = 1.0f / (l + (sink ? exp2f(s2 - Mf) : 0.0f));
    o0 *= f; o1 *= f; o2 *= f; o3 *= f;
    if (d_rope == 64) {  // inverse RoPE of the pair (64 + lane, 96 + lane) at position t
        const float2 cs = rope[(int64_t)t * 32 + lane];
        const float x = o2, y = o3;
        o2 = x * cs.x + y * cs.y;
        o3 = -x * cs.y + y * cs.x;
    }
    __nv_bfloat16 *orow = out + ((int64_t)b * kH + h) * 128;
    orow[lane] = __float2bfloat16_rn(o0);
    orow[32 + lane] = __float2bfloat16_rn(o1);
    orow[64 + lane] = __float2bfloat16_rn(o2);
    orow[96 + lane] = __float2bfloat16_rn(o3);
    if (lse && lane == 0) lse[(int64_t)b * kH + h] = (Mf + log2f(l)) * 0.6931471805599453f;
}

void launch_decode_combine(const AttnArgs &a, cudaStream_t st) {
    const int warps = a.B * csa_tc::kH;
    launch_pdl(decode_combine_kernel, (warps + 7) / 8, 256, 0, st, (const float *)a.part_o,
               (const float2 *)a.part_ml, a.ctx, a.sink, reinterpret_cast<const float2 *>(a.rope_tab),
               reinterpret_cast<__nv_bfloat16 *>(a.out), a.lse, a.B, a.split_S, a.L, a.d_rope);
    count_launches(1);
}

}  // namespace csa
