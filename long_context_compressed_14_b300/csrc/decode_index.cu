// decode_index.cu -- the decode indexer scan on the tensor cores: one new query per sequence
// scored against every visible entry of the sequence's FP8 indexer-key cache.
//
// Sources: [P2] "DeepSeek-V4: Towards Highly Efficient Million-Token Context Intelligence"
// (wiki notes), 提案手法 §1 CSA (the lightning indexer scores every compressed entry in low
// precision) and 訓練インフラの革新 §5 (decode against the compressed KV cache); [P5] "deepseek V4
// 技术论文" 一.1 (low-rank, cheap indexer).
//
// Score as in prefill: s(j) = sk_j * sum_h (w[h] * sq[h]) * ReLU(qcode[h] . kcode_j), for the
// entries j visible to the new token at p = ctx - 1 ((j+1)m - 1 <= p). The scan is bound by
// the bytes of the cache (64 code bytes + 4 scale bytes per entry), so the work is split into
// items of 128 entries of one sequence, dealt in contiguous blocks to three CTAs per SM:
//   MMA  D[128 entries][16] = KI_tile (128 x 64 E4M3) times qI^T (16 rows: the H_I heads of the
//        sequence's query, the rest of the 16 rows is ignored), K = 64 as two kind::f8f6f4 MMAs;
//   TMA  the entry tile and the query rows of the item into a ring of stages, with the entries'
//        scales copied by the producer lanes (cp.async) into the same stage;
//   epilogue (one warpgroup, thread = entry) the score, stored to the sequence's score row, and
//        the histogram of the scores' top 11 order-key bits per sequence, which the top-k kernel
//        then starts from. Each CTA takes a contiguous block of items (a stretch of one or two
//        sequences), counts in shared memory and adds its counts to the sequence's histogram in
//        global memory once per sequence, so the CTAs do not contend for the same counters.
// D has four 16-column TMEM buffers. Every wait is bounded; a failure sets the device status,
// raises the abort flag and the CTA frees its TMEM and returns.
#include <cuda_fp16.h>

#include "common.cuh"
#include "fp4.cuh"
#include "kernels.cuh"
#include "tma_host.cuh"
#include "topk_common.cuh"
#include "umma.cuh"

namespace csa {
using namespace umma;

namespace dix {
constexpr int kEpi = 128;                 // warps 0-3
constexpr int kProdWarp = 4;
constexpr int kMmaWarp = 5;
constexpr int kThreads = 192;
constexpr int kJ = 128;                   // entries per item (M)
constexpr int kN = 16;                    // query rows (N)
constexpr int kNS = 4;                    // ring stages (three CTAs fit one SM)
constexpr int kKBytes = kJ * 64;          // 8 KB
constexpr int kQBytes = kN * 64;          // 1 KB
constexpr int kSBytes = kJ * 4;           // the entries' FP8 scales
constexpr int kStage = kKBytes + kQBytes + kSBytes;
constexpr int kHistOff = kNS * kStage;   // per-warp key histograms [4][2048]
constexpr int kSmemBytes = kHistOff + 4 * 2048 * 4 + 1024;
constexpr int kNB = 4;                    // TMEM D buffers
constexpr uint32_t kTmemCols = 64;
}  // namespace dix

struct DixParams {
    CUtensorMap mk;          // KI codes [B*ncap][64] u8, box 64 x 128, 64-byte swizzle
    CUtensorMap mq;          // qI codes [B*H_I][64] u8, box 64 x 16, 64-byte swizzle
    const float *k_scale;    // [B*ncap]
    const float *q_scale;    // [B*H_I]
    const float *w;          // [B*H_I]
    const int32_t *ctx;      // [B]
    float *S;                // [B][ldS]
    int64_t ldS;
    uint32_t *hist;          // [B][2048] (zeroed by the caller's launch sequence)
    int B, L, m, ncap, HI, tiles;  // tiles = entry tiles per sequence (ceil(ncap / 128))
};

__device__ __forceinline__ uint64_t dix_desc_sw64(uint32_t addr) {
    return (uint64_t)((addr >> 4) & 0x3FFFu) | (1ull << 16) | ((uint64_t)(512 >> 4) << 32) | (1ull << 46) |
           (4ull << 61);
}

template <int HI>
__global__ void __launch_bounds__(dix::kThreads, 3) decode_index_tc_kernel(const __grid_constant__ DixParams P) {
    using namespace dix;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ __align__(8) uint64_t b_full[kNS], b_empty[kNS], b_dfull[kNB], b_dempty[kNB];
    __shared__ uint32_t tmem_slot;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t s_base = smem_u32(sm);
    if (warp == 0) {
        tmem_alloc(smem_u32(&tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int i = 0; i < kNS; ++i) {
            mbar_init(smem_u32(&b_full[i]), 1 + 32);  // TMA bytes + the producer lanes' scale copies
            mbar_init(smem_u32(&b_empty[i]), 1 + 4);  // the MMA commit + each epilogue warp
        }
        for (int i = 0; i < kNB; ++i) {
            mbar_init(smem_u32(&b_dfull[i]), 1);
            mbar_init(smem_u32(&b_dempty[i]), 4);
        }
        mbar_fence_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    pdl_trigger();
    pdl_wait();
    const uint32_t tmem = tmem_slot;
    const int n_items = P.B * P.tiles;
    const int per = (n_items + (int)gridDim.x - 1) / (int)gridDim.x;  // contiguous items per CTA
    const int it0 = (int)blockIdx.x * per, it1 = min(n_items, it0 + per);
    uint32_t *hist_all = reinterpret_cast<uint32_t *>(sm + kHistOff);
    // entries of item `it` visible to its sequence's new token (0: nothing to do)
    auto item_entries = [&](int it, int *b_out, int *et_out) -> int {
        const int b = it / P.tiles, et = it % P.tiles;
        *b_out = b;
        *et_out = et;
        const int64_t t = (int64_t)__ldg(P.ctx + b) - 1;
        if (t < 0 || t >= P.L) return 0;
        const int vis = visible_entries(t, P.m, P.ncap);
        return min(kJ, vis - et * kJ);
    };
    bool ok = true;

    if (warp == kProdWarp) {
        int n = 0;
        for (int it = it0; it < it1 && ok; ++it) {
            int b, et;
            const int ne = item_entries(it, &b, &et);
            if (ne <= 0) continue;
            const int s = n % kNS;
            if (n >= kNS && !__all_sync(0xffffffffu, mbar_wait(smem_u32(&b_empty[s]), ((n / kNS) - 1) & 1, kWaitNs,
                                                               &g_abort))) {
                ok = false;
                break;
            }
            const uint32_t st = s_base + s * kStage;
            if (lane == 0) {
                mbar_expect_tx(smem_u32(&b_full[s]), kKBytes + kQBytes);
                tma_load_3d(st, &P.mk, smem_u32(&b_full[s]), 0, b * P.ncap + et * kJ, 0);
                tma_load_3d(st + kKBytes, &P.mq, smem_u32(&b_full[s]), 0, b * HI, 0);
            }
            // the item's entry scales, 4 bytes per copy (rows of the cache need not be 16-byte
            // aligned), zero-filled past the visible entries; completion counted on the barrier
            const float *ks = P.k_scale + (int64_t)b * P.ncap + et * kJ;
#pragma unroll
            for (int q = 0; q < kJ / 32; ++q) {
                const int e = q * 32 + lane;
                asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(st + kKBytes + kQBytes + 4 * e),
                             "l"(ks + (e < ne ? e : 0)), "r"(e < ne ? 4u : 0u)
                             : "memory");
            }
            cp_async_mbar_arrive(smem_u32(&b_full[s]));
            ++n;
        }
        if (!ok) {
            if (lane == 0) {
                set_timeout();
                for (int f = max(0, n - kNS); f < n; ++f) mbar_wait(smem_u32(&b_full[f % kNS]), (f / kNS) & 1, kDrainNs);
            }
            cp_async_wait_all();
            __syncwarp();
        }
    } else if (warp == kMmaWarp) {
        if (lane == 0) {
            const uint32_t idesc = idesc_e4m3(128, kN);
            int n = 0;
            for (int it = it0; it < it1 && ok; ++it) {
                int b, et;
                if (item_entries(it, &b, &et) <= 0) continue;
                const int s = n % kNS, db = n % kNB;
                if (!mbar_wait(smem_u32(&b_full[s]), (n / kNS) & 1, kWaitNs, &g_abort)) { ok = false; break; }
                if (n >= kNB && !mbar_wait(smem_u32(&b_dempty[db]), ((n / kNB) - 1) & 1, kWaitNs, &g_abort)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t st = s_base + s * kStage;
#pragma unroll
                for (int kk = 0; kk < 2; ++kk)
                    mma_e4m3(tmem + db * kN, dix_desc_sw64(st + kk * 32), dix_desc_sw64(st + kKBytes + kk * 32), idesc,
                             kk);
                mma_commit(smem_u32(&b_dfull[db]));
                mma_commit(smem_u32(&b_empty[s]));
                ++n;
            }
            if (!ok) {
                set_timeout();
                if (n > 0) mbar_wait(smem_u32(&b_dfull[(n - 1) % kNB]), ((n - 1) / kNB) & 1, kDrainNs);
            }
        }
    } else {
        // epilogue: thread = entry jl of the item (TMEM lane)
        const int jl = tid;
        const uint32_t lane_base = (uint32_t)(32 * warp) << 16;
        int n = 0;
        // this warp's counts of the current sequence hb, added to the sequence's histogram in
        // global memory when the sequence changes (no barrier across warps: a warp that gives up
        // on a wait leaves without the others waiting for it)
        uint32_t *s_hist = hist_all + warp * tk::kBins;
        for (int i = lane; i < tk::kBins; i += 32) s_hist[i] = 0;
        __syncwarp();
        int hb = -1;
        float wq[HI];  // w * q_scale / 2 of sequence hb (kept in registers across its items)
        auto flush = [&]() {
            __syncwarp();
            for (int i = lane; i < tk::kBins; i += 32) {
                const uint32_t v = s_hist[i];
                if (v) {
                    atomicAdd(P.hist + (int64_t)hb * tk::kBins + i, v);
                    s_hist[i] = 0;
                }
            }
            __syncwarp();
        };
        for (int it = it0; it < it1 && ok; ++it) {
            int b, et;
            const int ne = item_entries(it, &b, &et);
            if (ne <= 0) continue;
            if (b != hb) {
                if (hb >= 0) flush();
                hb = b;
#pragma unroll
                for (int h = 0; h < HI; ++h) wq[h] = 0.5f * (__ldg(P.w + b * HI + h) * __ldg(P.q_scale + b * HI + h));
            }
            const int s = n % kNS, db = n % kNB;
            const int j = et * kJ + jl;
            // the stage's full barrier covers the scales the producer lanes copied (it has long
            // completed when the MMA result is there; its phase stays until this warp releases it)
            if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&b_full[s]), (n / kNS) & 1, kWaitNs, &g_abort) &&
                                             mbar_wait(smem_u32(&b_dfull[db]), (n / kNB) & 1, kWaitNs, &g_abort))) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t r[16];
            tmem_ld16_async(tmem + lane_base + db * kN, r);
            tmem_wait_hold16(r);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&b_dempty[db]));
            const float sk = reinterpret_cast<const float *>(sm + s * kStage + kKBytes + kQBytes)[jl];
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&b_empty[s]));  // this warp is done with the stage
            uint64_t acc = 0;
#pragma unroll
            for (int h2 = 0; h2 < HI / 2; ++h2) {
                const float x0 = __uint_as_float(r[2 * h2]), x1 = __uint_as_float(r[2 * h2 + 1]);
                acc = f2_fma(f2_pack(wq[2 * h2], wq[2 * h2 + 1]), f2_pack(x0 + fabsf(x0), x1 + fabsf(x1)), acc);
            }
            const float2 a2 = f2_unpack(acc);
            const float sc = fmaf(a2.x + a2.y, sk, 0.0f);
            const bool live = jl < ne;
            if (live) P.S[(int64_t)b * P.ldS + j] = sc;
            // histogram of the top 11 order-key bits, one atomic per distinct bin of the warp
            const uint32_t bin = key_of(sc) >> tk::kBinShift;
            const unsigned peers = __match_any_sync(0xffffffffu, live ? bin : 0xFFFFFFFFu);
            if (live && (__ffs(peers) - 1) == lane) atomicAdd(&s_hist[bin], (uint32_t)__popc(peers));
            ++n;
        }
        if (ok && hb >= 0) flush();
        if (!ok && lane == 0) set_timeout();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

bool decode_index_tc_supported(const IndexArgs &a) {
    return a.decode && a.idx_t == CSA_FP8E4M3 && (a.H_I == 4 || a.H_I == 8 || a.H_I == 16) &&
           (int64_t)a.B * a.H_I >= 16;
}

bool launch_decode_index_tc(const IndexArgs &a, uint32_t *hist, cudaStream_t st) {
    using namespace dix;
    if (!decode_index_tc_supported(a)) return false;
    DixParams P;
    memset(&P, 0, sizeof(P));
    bool ok = make_map_3d(&P.mk, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, a.KI, 64, (uint64_t)a.B * a.ncap, 1, 64, kJ,
                          CU_TENSOR_MAP_SWIZZLE_64B);
    ok = ok && make_map_3d(&P.mq, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, a.qI, 64, (uint64_t)a.B * a.H_I, 1, 64, kN,
                           CU_TENSOR_MAP_SWIZZLE_64B);
    if (!ok) return false;
    P.k_scale = a.KI_scale;
    P.q_scale = a.qI_scale;
    P.w = a.w;
    P.ctx = a.ctx;
    P.S = a.S;
    P.ldS = a.ldS;
    P.hist = hist;
    P.B = a.B; P.L = a.L; P.m = a.m; P.ncap = a.ncap; P.HI = a.H_I;
    P.tiles = (a.ncap + kJ - 1) / kJ;
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int items = a.B * P.tiles;
    const int grid = items < 3 * sms ? items : 3 * sms;  // three CTAs (pipelines) per SM
    auto go = [&](auto kern) {
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        launch_pdl(kern, grid, kThreads, kSmemBytes, st, P);
    };
    if (a.H_I == 4) go(decode_index_tc_kernel<4>);
    else if (a.H_I == 8) go(decode_index_tc_kernel<8>);
    else go(decode_index_tc_kernel<16>);
    count_launches(1);
    return true;
}

// ---------------------------------------------------------------------------------------
// MXFP4 decode scan: the packed FP4 cache read as stored (32 code bytes + 2 exponent bytes per
// entry, half the FP8 cache's bytes), on the CUDA cores. Thread = entry. Per head h and block
// b of 32 dims: the E2M1 products are summed in half precision in four partial sums of eight
// products each (an E2M1 product is a multiple of 1/4 of magnitude at most 36, so a sum of
// eight is at most 288 and exact in half precision), the partials are added in float and scaled
// by the two blocks' powers of two; s = sum_h w[h] ReLU(sum_b ...), stored to the sequence's score
// row and counted in the CTA's histogram of the top 11 order-key bits (added to the sequence's
// histogram in global memory when the CTA moves to the next sequence), as the tensor-core scan
// does for FP8 keys. Each CTA takes a contiguous block of 256-entry items.
// ---------------------------------------------------------------------------------------
namespace dix4 {
constexpr int kThreads = 256;
constexpr int kJ = 256;   // entries per item
}

template <int HI>
__global__ void __launch_bounds__(dix4::kThreads) decode_index_fp4_kernel(IndexArgs a, uint32_t *hist, int tiles) {
    using namespace dix4;
    __shared__ __align__(16) __half2 s_q[HI][32];  // the query's E2M1 values as half pairs
    __shared__ float s_qe[HI][2];                  // its block scales 2^(e8 - 127)
    __shared__ float s_w[HI];
    __shared__ uint32_t s_hist[tk::kBins];
    const int tid = threadIdx.x, lane = tid & 31;
    const int n_items = a.B * tiles;
    const int per = (n_items + (int)gridDim.x - 1) / (int)gridDim.x;
    const int it0 = (int)blockIdx.x * per, it1 = min(n_items, it0 + per);
    for (int i = tid; i < tk::kBins; i += kThreads) s_hist[i] = 0;
    pdl_trigger();
    pdl_wait();
    int hb = -1;
    auto flush = [&]() {
        __syncthreads();
        for (int i = tid; i < tk::kBins; i += kThreads) {
            const uint32_t v = s_hist[i];
            if (v) {
                atomicAdd(hist + (int64_t)hb * tk::kBins + i, v);
                s_hist[i] = 0;
            }
        }
    };
    const uint8_t *kc = reinterpret_cast<const uint8_t *>(a.KI);
    for (int it = it0; it < it1; ++it) {
        const int b = it / tiles, et = it % tiles;
        const int64_t t = (int64_t)__ldg(a.ctx + b) - 1;
        const int vis = (t < 0 || t >= a.L) ? 0 : visible_entries(t, a.m, a.ncap);
        if (et * kJ >= vis) continue;  // (uniform over the CTA)
        if (b != hb) {
            if (hb >= 0) flush();
            __syncthreads();  // the previous sequence's query is no longer read
            hb = b;
            const uint8_t *qc = reinterpret_cast<const uint8_t *>(a.qI) + (int64_t)b * HI * 32;
            for (int u = tid; u < HI * 32; u += kThreads) s_q[u / 32][u % 32] = e2m1x2_to_h2(qc[u]);  // dims 2i, 2i+1
            if (tid < HI * 2) s_qe[tid / 2][tid % 2] = ldexpf(1.0f, (int)a.qI_e8[(int64_t)b * HI * 2 + tid] - 127);
            if (tid < HI) s_w[tid] = __ldg(a.w + (int64_t)b * HI + tid);
            __syncthreads();
        }
        const int j = et * kJ + tid;
        const bool live = j < vis;
        float sc = 0.0f;
        if (live) {
            const int64_t row = (int64_t)b * a.ncap + j;
            const uint4 c0 = __ldg(reinterpret_cast<const uint4 *>(kc + row * 32));
            const uint4 c1 = __ldg(reinterpret_cast<const uint4 *>(kc + row * 32) + 1);
            const float ks[2] = {ldexpf(1.0f, (int)a.KI_e8[row * 2] - 127), ldexpf(1.0f, (int)a.KI_e8[row * 2 + 1] - 127)};
            const uint32_t cw[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
            __half2 kh[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) kh[i] = e2m1x2_to_h2((uint8_t)(cw[i >> 2] >> (8 * (i & 3))));
#pragma unroll
            for (int h = 0; h < HI; ++h) {
                float dot = 0.0f;
#pragma unroll
                for (int blk = 0; blk < 2; ++blk) {
                    __half2 p0 = __float2half2_rn(0.0f), p1 = p0;
#pragma unroll
                    for (int i = 0; i < 8; ++i) p0 = __hfma2(s_q[h][16 * blk + i], kh[16 * blk + i], p0);
#pragma unroll
                    for (int i = 8; i < 16; ++i) p1 = __hfma2(s_q[h][16 * blk + i], kh[16 * blk + i], p1);
                    const float2 f0 = __half22float2(p0), f1 = __half22float2(p1);
                    const float part = (f0.x + f0.y) + (f1.x + f1.y);
                    dot = fmaf(part, s_qe[h][blk] * ks[blk], dot);  // exact power-of-two scale
                }
                sc = fmaf(s_w[h], fmaxf(dot, 0.0f), sc);
            }
            sc += 0.0f;  // -0 -> +0
            a.S[(int64_t)b * a.ldS + j] = sc;
        }
        const uint32_t bin = key_of(sc) >> tk::kBinShift;
        const unsigned peers = __match_any_sync(0xffffffffu, live ? bin : 0xFFFFFFFFu);
        if (live && (__ffs(peers) - 1) == lane) atomicAdd(&s_hist[bin], (uint32_t)__popc(peers));
    }
    if (hb >= 0) flush();
}

bool decode_index_fp4_supported(const IndexArgs &a) {
    return a.decode && a.idx_t == CSA_MXFP4 && (a.H_I == 4 || a.H_I == 8 || a.H_I == 16) && a.qI_e8 && a.KI_e8;
}

bool launch_decode_index_fp4(const IndexArgs &a, uint32_t *hist, cudaStream_t st) {
    using namespace dix4;
    if (!decode_index_fp4_supported(a)) return false;
    const int tiles = (a.ncap + kJ - 1) / kJ;
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int items = a.B * tiles;
    const int grid = items < 4 * sms ? items : 4 * sms;
    if (a.H_I == 4) launch_pdl(decode_index_fp4_kernel<4>, grid, kThreads, 0, st, a, hist, tiles);
    else if (a.H_I == 8) launch_pdl(decode_index_fp4_kernel<8>, grid, kThreads, 0, st, a, hist, tiles);
    else launch_pdl(decode_index_fp4_kernel<16>, grid, kThreads, 0, st, a, hist, tiles);
    count_launches(1);
    return true;
}

}  // namespace csa
