// attn_hca_tc.cu -- HCA prefill attention on the 5th-generation tensor cores (tcgen05 + TMEM).
//
// Sources: [P2] "DeepSeek-V4: Towards Highly Efficient Million-Token Context Intelligence"
// (wiki notes), 提案手法 §1 (HCA: m' = 128 compression, no sparse selection, dense attention
// over the compressed entries; shared-KV MQA; sliding-window branch n_win = 128; attention
// sink; partial RoPE with inverse RoPE on the output) and 訓練インフラの革新 §5 (mixed-precision
// entries); [P5] "deepseek V4 技术论文" 一.1 (an entry is both key and value).
//
// Because every query head shares the one KV head, a CTA stacks T = 128 / H consecutive
// tokens x H heads into M = 128 query rows and walks one key list for all of them:
//   compressed tiles of 128 entries [0, visible(last token)), then one window tile of the raw
//   rows [t0 - n_win + 1, t0 + T - 1] (T + n_win - 1 <= 144 keys).
// Per key tile: S = Q K^T (M = 128, N = keys, K = 128) into TMEM; one thread per query row
// masks (visibility / window), keeps a running max in the log2 domain with lazy rescaling
// (the exponent base only moves when the max grows by more than 8, and then O is rescaled in
// TMEM), writes P = exp2(s - max) as BF16 into shared memory, and O += P V (M = 128, N = 128,
// K = keys) accumulates in TMEM, V being the same key tile read through an MN-major
// descriptor. Key tiles arrive by TMA (128-byte swizzle) into two buffers, the next tile
// loading while the current one is processed. Mixed-precision entries: the BF16 RoPE half
// arrives by TMA, the FP8 half is staged by TMA and widened to BF16 (code * row scale) by the
// threads. The epilogue divides by the softmax sum (plus exp(sink)), applies the inverse RoPE
// at each row's position and stores BF16.
#include "common.cuh"
#include "kernels.cuh"
#include "tma_host.cuh"
#include "umma.cuh"

namespace csa {
using namespace umma;

namespace hca_tc {
constexpr int kRows = 128;                 // query rows per CTA
constexpr int kCTile = 128;                // compressed entries per key tile
constexpr int kMaxKeys = 144;              // rows of a key-tile buffer (the window tile needs <= 144)
constexpr int kSub = kMaxKeys * 128;       // bytes of one 64-dim half of a key-tile buffer (18 KB)
constexpr int kQOff = 0;                   // Q: two 64-dim halves, 16 KB each
constexpr int kKOff = 32768;               // key tiles: two buffers of 2 * kSub
constexpr int kPOff = kKOff + 4 * kSub;    // P: three 64-key sub-tiles of 16 KB
constexpr int kStOff = kPOff + 3 * 16384;  // mixed: FP8 staging, two buffers of 8 KB
constexpr int kSmemBytes = kStOff + 2 * 8192 + 1024;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSCol = 0;              // S: columns [0, 144)
constexpr uint32_t kOCol = 256;            // O: columns [256, 384)
constexpr float kRescaleThreshold = 8.0f;  // log2 units
}  // namespace hca_tc

struct HcaTcParams {
    CUtensorMap mq;     // q viewed as [B][L*H][128] bf16, box 64 x 128
    CUtensorMap mc;     // BF16 entries [B][ncap][128] | MIXED RoPE half [B][ncap][64], box 64 x 128
    CUtensorMap mcode;  // MIXED FP8 half [B][ncap][64] u8, box 64 x 128, no swizzle
    CUtensorMap mkv;    // kv_rope [B][L][128] bf16, box 64 x 144
    const float *c_scale;
    const float *sink;
    const float2 *rope;
    __nv_bfloat16 *out;
    float *lse;
    int B, L, H, T, m, ncap, n_win, n_swa, d_rope, mixed;
    float scale_log2;
};

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
    __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&v);
}

__global__ void __launch_bounds__(128, 1) hca_tc_kernel(const __grid_constant__ HcaTcParams P) {
    using namespace hca_tc;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ __align__(8) uint64_t bars[4];  // 0: Q, 1-2: key-tile buffers, 3: MMA completion
    __shared__ uint32_t tmem_slot;

    const int tid = threadIdx.x, warp = tid >> 5;
    const int b = blockIdx.y;
    const int H = P.H, T = P.T;
    const int t0 = blockIdx.x * T;
    const int t_last = min(t0 + T, P.L) - 1;
    const int vis_hi = visible_entries(t_last, P.m, P.ncap);
    const int n_ct = (vis_hi + kCTile - 1) / kCTile;
    const int n_tiles = n_ct + 1;
    const int u_lo = t0 - P.n_win + 1;
    const uint32_t s_base = smem_u32(sm);
    const uint32_t bar_q = smem_u32(&bars[0]), bar_mma = smem_u32(&bars[3]);

    if (warp == 0) {
        tmem_alloc(smem_u32(&tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int i = 0; i < 4; ++i) mbar_init(smem_u32(&bars[i]), 1);
        mbar_fence_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;

    auto issue_tile = [&](int i) {  // one thread
        const int buf = i & 1;
        const uint32_t bar = smem_u32(&bars[1 + buf]);
        const uint32_t kdst = s_base + kKOff + buf * 2 * kSub;
        if (i < n_ct) {
            const int j0 = i * kCTile;
            if (!P.mixed) {
                mbar_expect_tx(bar, 2 * kCTile * 128);
                tma_load_3d(kdst, &P.mc, bar, 0, j0, b);
                tma_load_3d(kdst + kSub, &P.mc, bar, 64, j0, b);
            } else {
                mbar_expect_tx(bar, kCTile * 64 + kCTile * 128);
                tma_load_3d(s_base + kStOff + buf * 8192, &P.mcode, bar, 0, j0, b);
                tma_load_3d(kdst + kSub, &P.mc, bar, 0, j0, b);
            }
        } else {
            mbar_expect_tx(bar, 2 * kMaxKeys * 128);
            tma_load_3d(kdst, &P.mkv, bar, 0, u_lo, b);
            tma_load_3d(kdst + kSub, &P.mkv, bar, 64, u_lo, b);
        }
    };

    if (tid == 0) {
        mbar_expect_tx(bar_q, 2 * kRows * 128);
        tma_load_3d(s_base + kQOff, &P.mq, bar_q, 0, t0 * H, b);
        tma_load_3d(s_base + kQOff + 16384, &P.mq, bar_q, 64, t0 * H, b);
        issue_tile(0);
        if (n_tiles > 1) issue_tile(1);
    }

    // this thread's query row
    const int r = tid;
    const int t = t0 + r / H;
    const int h = r % H;
    const bool row_ok = t < P.L;
    const int vis_t = row_ok ? visible_entries(t, P.m, P.ncap) : 0;
    const uint32_t lane_base = (uint32_t)(32 * warp) << 16;
    bool ok = true;

    // Q: wait, then rotate dims 64..127 at position t (pairs (64+i, 96+i)) in shared memory
    ok = __syncthreads_and(mbar_wait(bar_q, 0, kWaitNs, &g_abort));
    if (ok && P.d_rope == 64 && row_ok) {
        uint8_t *q1 = sm + kQOff + 16384;  // dims 64..127
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            uint4 *pa = reinterpret_cast<uint4 *>(q1 + sw128_off(r, c));
            uint4 *pb = reinterpret_cast<uint4 *>(q1 + sw128_off(r, c + 4));
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
    __syncthreads();

    float m_run = -INFINITY, l_run = 0.0f;
    uint32_t ph_mma = 0;
    const uint32_t idesc_pv = idesc_bf16(128, 128, 0, 1);
    for (int i = 0; i < n_tiles && ok; ++i) {
        const int buf = i & 1;
        const bool ctile = i < n_ct;
        const int n_i = ctile ? kCTile : P.n_swa;
        const uint32_t kbuf = s_base + kKOff + buf * 2 * kSub;
        // a timed-out wait is made block-uniform so every thread leaves the loop together
        if (!__syncthreads_and(mbar_wait(smem_u32(&bars[1 + buf]), (i >> 1) & 1, kWaitNs, &g_abort))) { ok = false; break; }
        if (ctile && P.mixed) {
            // widen the FP8 half: row r of the tile = entry j0 + r
            const int j = i * kCTile + r;
            const float sc = j < P.ncap ? P.c_scale[(int64_t)b * P.ncap + j] : 0.0f;
            const uint8_t *src = sm + kStOff + buf * 8192 + r * 64;
            uint8_t *dst = sm + kKOff + buf * 2 * kSub;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const uint2 codes = *reinterpret_cast<const uint2 *>(src + 8 * c);
                const uint32_t cw[2] = {codes.x, codes.y};
                uint32_t packed[4];
#pragma unroll
                for (int q = 0; q < 2; ++q) {
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const uint16_t two = (uint16_t)(cw[q] >> (16 * e));
                        __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)two, __NV_E4M3);
                        const float2 f = __half22float2(__half2(hr));
                        packed[2 * q + e] = pack_bf16x2(f.x * sc, f.y * sc);
                    }
                }
                *reinterpret_cast<uint4 *>(dst + sw128_off(r, c)) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
            }
            fence_async_smem();
            __syncthreads();
        }
        // S = Q K^T
        if (tid == 0) {
            tc_fence_after();
            const uint32_t idesc = idesc_bf16(128, n_i, 0, 0);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint64_t ad = sdesc_sw128(s_base + kQOff + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024);
                const uint64_t bd = sdesc_sw128(kbuf + (kk >> 2) * kSub + (kk & 3) * 32, 16, 1024);
                mma_bf16(tmem + kSCol, ad, bd, idesc, kk > 0);
            }
            mma_commit(bar_mma);
        }
        if (!__syncthreads_and(mbar_wait(bar_mma, ph_mma, kWaitNs, &g_abort))) { ok = false; break; }
        ph_mma ^= 1;
        tc_fence_after();
        // the previous P V is complete: its key buffer takes tile i + 1
        if (tid == 0 && i >= 1 && i + 1 < n_tiles) issue_tile(i + 1);

        // ---- softmax of row r over keys [0, n_i) ----
        int lo, hi;  // valid key range [lo, hi) of this row in the tile
        if (ctile) {
            lo = 0;
            hi = row_ok ? max(0, min(kCTile, vis_t - i * kCTile)) : 0;
        } else {
            lo = max(t - t0, -u_lo);  // u >= t - n_win + 1 and u >= 0
            hi = row_ok ? (t - t0 + P.n_win) : 0;
            hi = min(hi, n_i);
        }
        float tmax = -INFINITY;
        for (int c0 = 0; c0 < n_i; c0 += 16) {
            float v[16];
            tmem_ld16_sync(tmem + lane_base + kSCol + c0, v);
#pragma unroll
            for (int e = 0; e < 16; ++e)
                if (c0 + e >= lo && c0 + e < hi) tmax = fmaxf(tmax, v[e] * P.scale_log2);
        }
        float factor = 1.0f;
        bool rescale_o = false;
        if (tmax > m_run + kRescaleThreshold) {
            factor = exp2f(m_run - tmax);  // 0 when m_run is -inf
            rescale_o = (i > 0) && (m_run != -INFINITY);
            l_run *= factor;
            m_run = tmax;
        }
        if (__any_sync(0xffffffffu, rescale_o)) {
            const float f = rescale_o ? factor : 1.0f;
            for (int c0 = 0; c0 < 128; c0 += 16) {
                float v[16];
                tmem_ld16_sync(tmem + lane_base + kOCol + c0, v);
#pragma unroll
                for (int e = 0; e < 16; ++e) v[e] *= f;
                tmem_st16(tmem + lane_base + kOCol + c0, v);
            }
            tmem_st_wait();
        }
        uint8_t *sp = sm + kPOff;
        for (int c0 = 0; c0 < n_i; c0 += 16) {
            float v[16];
            tmem_ld16_sync(tmem + lane_base + kSCol + c0, v);
            uint32_t pk[8];
#pragma unroll
            for (int e = 0; e < 16; e += 2) {
                const float p0 = (c0 + e >= lo && c0 + e < hi) ? fast_exp2(v[e] * P.scale_log2 - m_run) : 0.0f;
                const float p1 = (c0 + e + 1 >= lo && c0 + e + 1 < hi) ? fast_exp2(v[e + 1] * P.scale_log2 - m_run) : 0.0f;
                l_run += p0 + p1;
                pk[e >> 1] = pack_bf16x2(p0, p1);
            }
            const int sub = c0 >> 6, ch = (c0 & 63) >> 3;
            uint8_t *base = sp + sub * 16384;
            *reinterpret_cast<uint4 *>(base + sw128_off(r, ch)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            *reinterpret_cast<uint4 *>(base + sw128_off(r, ch + 1)) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        // O += P V
        if (tid == 0) {
            for (int kk = 0; kk < n_i / 16; ++kk) {
                const uint64_t ad = sdesc_sw128(s_base + kPOff + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024);
                const uint64_t bd = sdesc_sw128(kbuf + kk * 2048, kSub, 1024);
                mma_bf16(tmem + kOCol, ad, bd, idesc_pv, (i > 0 || kk > 0) ? 1u : 0u);
            }
        }
    }
    if (ok) {
        if (tid == 0) mma_commit(bar_mma);
        ok = __syncthreads_and(mbar_wait(bar_mma, ph_mma, kWaitNs, &g_abort));
        tc_fence_after();
    }
    if (!ok) {
        if (tid == 0) set_timeout();
        // let in-flight copies land before the shared memory is released (bounded)
        for (int q = 0; q < 3; ++q) mbar_wait(smem_u32(&bars[q]), 0, kDrainNs);
    } else {
        // ---- epilogue of row r. The TMEM loads are warp-collective (.sync.aligned), so every
        // thread executes them; only rows inside the sequence store. ----
        float f = 0.0f;
        if (row_ok) {
            if (P.sink) {
                const float s2 = P.sink[h] * 1.4426950408889634f;
                const float mf = fmaxf(m_run, s2);
                const float den = l_run * exp2f(m_run - mf) + exp2f(s2 - mf);
                f = exp2f(m_run - mf) / den;
            } else {
                f = 1.0f / l_run;
            }
        }
        __nv_bfloat16 *orow = P.out + (((int64_t)b * P.L + (row_ok ? t : 0)) * H + h) * 128;
        float lo_[32], hi_[32];
        // dims 0..63: no rotation
        for (int c0 = 0; c0 < 64; c0 += 32) {
            float v[32];
            tmem_ld32_sync(tmem + lane_base + kOCol + c0, v);
            uint32_t pk[16];
#pragma unroll
            for (int e = 0; e < 32; e += 2) pk[e >> 1] = pack_bf16x2(v[e] * f, v[e + 1] * f);
            if (row_ok) {
                uint4 *dst = reinterpret_cast<uint4 *>(orow + c0);
#pragma unroll
                for (int q = 0; q < 4; ++q) dst[q] = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
            }
        }
        tmem_ld32_sync(tmem + lane_base + kOCol + 64, lo_);
        tmem_ld32_sync(tmem + lane_base + kOCol + 96, hi_);
        if (row_ok) {
#pragma unroll
            for (int e = 0; e < 32; ++e) {
                const float x = lo_[e] * f, y = hi_[e] * f;
                if (P.d_rope == 64) {
                    const float2 cs = P.rope[(int64_t)t * 32 + e];
                    lo_[e] = x * cs.x + y * cs.y;
                    hi_[e] = -x * cs.y + y * cs.x;
                } else {
                    lo_[e] = x;
                    hi_[e] = y;
                }
            }
            uint32_t pk[16];
#pragma unroll
            for (int e = 0; e < 32; e += 2) pk[e >> 1] = pack_bf16x2(lo_[e], lo_[e + 1]);
            uint4 *dst = reinterpret_cast<uint4 *>(orow + 64);
#pragma unroll
            for (int q = 0; q < 4; ++q) dst[q] = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
#pragma unroll
            for (int e = 0; e < 32; e += 2) pk[e >> 1] = pack_bf16x2(hi_[e], hi_[e + 1]);
            dst = reinterpret_cast<uint4 *>(orow + 96);
#pragma unroll
            for (int q = 0; q < 4; ++q) dst[q] = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
            if (P.lse) P.lse[((int64_t)b * P.L + t) * H + h] = (m_run + log2f(l_run)) * 0.6931471805599453f;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

// Host: returns false when the configuration is outside what this kernel handles (the caller
// then uses the CUDA-core kernel).
bool hca_tc_supported(const AttnArgs &a) {
    if (a.decode || a.act_t != CSA_BF16) return false;
    if (a.kv_t != CSA_BF16 && a.kv_t != CSA_MIXED) return false;
    if (a.H != 16 && a.H != 32 && a.H != 64 && a.H != 128) return false;
    const int T = 128 / a.H;
    if (T + a.n_win - 1 > hca_tc::kMaxKeys) return false;
    if (a.d_rope != 0 && a.d_rope != 64) return false;
    return true;
}

bool launch_hca_tc(const AttnArgs &a, cudaStream_t st) {
    using namespace hca_tc;
    if (!hca_tc_supported(a)) return false;
    HcaTcParams P;
    memset(&P, 0, sizeof(P));
    const uint64_t L = a.L, H = a.H, B = a.B, ncap = a.ncap;
    bool ok = make_map_3d(&P.mq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.q, 128, L * H, B, 64, 128,
                          CU_TENSOR_MAP_SWIZZLE_128B);
    ok = ok && make_map_3d(&P.mkv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.kv_rope, 128, L, B, 64, kMaxKeys,
                           CU_TENSOR_MAP_SWIZZLE_128B);
    if (a.kv_t == CSA_BF16) {
        ok = ok && make_map_3d(&P.mc, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.c_data, 128, ncap, B, 64, kCTile,
                               CU_TENSOR_MAP_SWIZZLE_128B);
    } else {
        ok = ok && make_map_3d(&P.mc, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.c_rope, 64, ncap, B, 64, kCTile,
                               CU_TENSOR_MAP_SWIZZLE_128B);
        ok = ok && make_map_3d(&P.mcode, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, a.c_data, 64, ncap, B, 64, kCTile,
                               CU_TENSOR_MAP_SWIZZLE_NONE);
    }
    if (!ok) return false;
    P.c_scale = a.c_scale;
    P.sink = a.sink;
    P.rope = reinterpret_cast<const float2 *>(a.rope_tab);
    P.out = reinterpret_cast<__nv_bfloat16 *>(a.out);
    P.lse = a.lse;
    P.B = a.B; P.L = a.L; P.H = a.H; P.T = 128 / a.H; P.m = a.m; P.ncap = a.ncap; P.n_win = a.n_win;
    P.n_swa = ((P.T + a.n_win - 1) + 15) / 16 * 16;
    P.d_rope = a.d_rope; P.mixed = a.kv_t == CSA_MIXED;
    P.scale_log2 = a.scale * 1.4426950408889634f;
    cudaFuncSetAttribute(hca_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    dim3 grid((unsigned)((a.L + P.T - 1) / P.T), (unsigned)a.B);
    hca_tc_kernel<<<grid, 128, kSmemBytes, st>>>(P);
    count_launches(1);
    return true;
}

}  // namespace csa
