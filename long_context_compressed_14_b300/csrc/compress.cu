// compress.cu -- RoPE table, FP8 row quantisation and the fused overlapping compression.
//
// Sources: [P2] "DeepSeek-V4: Towards Highly Efficient Million-Token Context Intelligence"
// (wiki notes), 提案手法 §1 (CSA: weighted-average compression of every m = 4 tokens with
// overlap between adjacent blocks; HCA: m' = 128; partial RoPE on the last 64 dims) and
// 訓練インフラの革新 §5 (KV entries: RoPE dims BF16, other dims FP8); [P5] "deepseek V4
// 技术论文" 一.1 (C^b overlaps C^a); [P3] "Технический отчёт DeepSeek-V4.1-Flash — часть 2/2"
// (the V4.1 variant: entries in NVFP4, quantised after RoPE).
#include "common.cuh"
#include "fp4.cuh"
#include "kernels.cuh"
#include "umma.cuh"

namespace csa {

// ---------------------------------------------------------------------------------------
// RoPE table: tab[pos][i] = (cos, sin)(pos * theta^(-i/half)), double math, float storage.
// ---------------------------------------------------------------------------------------
__global__ void rope_table_kernel(float2 *tab, int rope_len, int half, double theta) {
    const int64_t n = (int64_t)rope_len * half;
    for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < n;
         e += (int64_t)gridDim.x * blockDim.x) {
        const int64_t pos = e / half;
        const int i = (int)(e % half);
        const double freq = pow(theta, -(double)i / (double)half);
        double s, c;
        sincos((double)pos * freq, &s, &c);
        tab[e] = make_float2((float)c, (float)s);
    }
}

void launch_rope_table(float *tab, int rope_len, int d_rope, float theta, cudaStream_t st) {
    const int half = d_rope / 2;
    const int64_t n = (int64_t)rope_len * half;
    int blocks = (int)((n + 255) / 256);
    if (blocks > 148 * 16) blocks = 148 * 16;
    if (blocks < 1) blocks = 1;
    rope_table_kernel<<<blocks, 256, 0, st>>>(reinterpret_cast<float2 *>(tab), rope_len, half,
                                                (double)theta);
    count_launches(1);
}

// ---------------------------------------------------------------------------------------
// Per-row FP8 quantisation: one warp per row.
// ---------------------------------------------------------------------------------------
__global__ void quant_rows_kernel(const float *__restrict__ x, int64_t rows, int cols,
                                  uint8_t *__restrict__ codes, float *__restrict__ scales) {
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t r = blockIdx.x * (int64_t)(blockDim.x >> 5) + (threadIdx.x >> 5); r < rows; r += warps) {
        const float *row = x + r * cols;
        float amax = 0.0f;
        for (int c = lane; c < cols; c += 32) amax = fmaxf(amax, fabsf(row[c]));
        amax = warp_max(amax);
        const float scale = __fdiv_rn(amax, 448.0f);
        for (int c = lane; c < cols; c += 32)
            codes[r * cols + c] = scale > 0.0f ? f32_to_e4m3(__fdiv_rn(row[c], scale)) : (uint8_t)0;
        if (lane == 0) scales[r] = scale;
    }
}

// Rows of 64 (the indexer's query rows): a half-warp per row, each lane one 16-byte chunk of four
// values, two rows per warp instruction and kQ64Unroll row pairs per warp in flight; the same
// arithmetic as quant_rows_kernel (float scale amax / 448, float division per element).
constexpr int kQ64Unroll = 4;
__global__ void __launch_bounds__(256) quant_rows64_kernel(const float4 *__restrict__ x, int64_t rows,
                                                           uint32_t *__restrict__ codes, float *__restrict__ scales) {
    const int lane = threadIdx.x & 31, c = lane & 15, h = lane >> 4;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    const int64_t gw = blockIdx.x * (int64_t)(blockDim.x >> 5) + (threadIdx.x >> 5);
    for (int64_t r0 = gw * 2 * kQ64Unroll; r0 < rows; r0 += warps * 2 * kQ64Unroll) {
        float4 v[kQ64Unroll];
#pragma unroll
        for (int u = 0; u < kQ64Unroll; ++u) {
            const int64_t r = r0 + 2 * u + h;
            v[u] = r < rows ? __ldcs(x + r * 16 + c) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        }
#pragma unroll
        for (int u = 0; u < kQ64Unroll; ++u) {
            const int64_t r = r0 + 2 * u + h;
            float amax = fmaxf(fmaxf(fabsf(v[u].x), fabsf(v[u].y)), fmaxf(fabsf(v[u].z), fabsf(v[u].w)));
#pragma unroll
            for (int o = 8; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
            const float scale = __fdiv_rn(amax, 448.0f);
            uint32_t w = 0;
            if (scale > 0.0f)
                w = (uint32_t)f32_to_e4m3(__fdiv_rn(v[u].x, scale)) | ((uint32_t)f32_to_e4m3(__fdiv_rn(v[u].y, scale)) << 8) |
                    ((uint32_t)f32_to_e4m3(__fdiv_rn(v[u].z, scale)) << 16) |
                    ((uint32_t)f32_to_e4m3(__fdiv_rn(v[u].w, scale)) << 24);
            if (r < rows) {
                codes[r * 16 + c] = w;
                if (c == 0) scales[r] = scale;
            }
        }
    }
}

void launch_quant_rows(const float *x, int64_t rows, int cols, uint8_t *codes, float *scales,
                       cudaStream_t st) {
    if (cols == 64 && reinterpret_cast<uintptr_t>(x) % 16 == 0 && reinterpret_cast<uintptr_t>(codes) % 4 == 0) {
        int64_t blocks = (rows + 8 * 2 * kQ64Unroll - 1) / (8 * 2 * kQ64Unroll);
        if (blocks > 148 * 8) blocks = 148 * 8;
        quant_rows64_kernel<<<(int)blocks, 256, 0, st>>>(reinterpret_cast<const float4 *>(x), rows,
                                                         reinterpret_cast<uint32_t *>(codes), scales);
        count_launches(1);
        return;
    }
    int64_t blocks = (rows + 7) / 8;
    if (blocks > 148 * 32) blocks = 148 * 32;
    if (blocks < 1) blocks = 1;
    quant_rows_kernel<<<(int)blocks, 256, 0, st>>>(x, rows, cols, codes, scales);
    count_launches(1);
}

// ---------------------------------------------------------------------------------------
// kv_compress: entry j of sequence b is the softmax-weighted sum of the window rows
//   [(j-1)m, (j+1)m) ∩ [0, L), weight of row t = exp(z[t, set] - max) with set 0 for the own
//   block (t >= jm) and set 1 for the previous block, normalised at the end; then RoPE at the
//   entry position (j+1)m - 1 and the storage format. Rows of the own block are also written
//   back rotated at their own position (kv_rope; the two dims of a RoPE pair sit in 16-byte
//   chunks 32 / V apart and meet by a shuffle). Consecutive entries share a block, so both
//   kernels below walk runs of consecutive entries block by block and read each raw row once.
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ void store16(float *p, const float (&y)[4]) {
    *reinterpret_cast<float4 *>(p) = make_float4(y[0], y[1], y[2], y[3]);
}
__device__ __forceinline__ void store16(__nv_bfloat16 *p, const float (&y)[8]) {
    uint32_t w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        __nv_bfloat162 b2 = __floats2bfloat162_rn(y[2 * k], y[2 * k + 1]);
        w[k] = *reinterpret_cast<uint32_t *>(&b2);
    }
    *reinterpret_cast<uint4 *>(p) = make_uint4(w[0], w[1], w[2], w[3]);
}

// The end of an entry, by one warp holding c[e] = dim lane + 32 e of the weighted sum (before
// RoPE) and (k0, k1) = indexer dims (lane, lane + 32): RoPE at the entry position (j+1)m - 1
// (rope_pos: that position's row of the table, in global or shared memory; null without RoPE)
// and storage per KV_T and IDX_T.
template <int KV_T, int IDX_T, bool WITH_KI>
__device__ __forceinline__ void finish_entry(float (&c)[4], float k0, float k1, int j, int b, int N,
                                             const float2 *rope_pos, void *__restrict__ c_data,
                                             __nv_bfloat16 *__restrict__ c_rope, float *__restrict__ c_scale,
                                             void *__restrict__ ki_data, float *__restrict__ ki_scale,
                                             uint8_t *__restrict__ ki_e8) {
    const int lane = threadIdx.x & 31;
    if (rope_pos) {
        const float2 cs = rope_pos[lane];
        const float a = c[2], bb = c[3];
        c[2] = a * cs.x - bb * cs.y;
        c[3] = a * cs.y + bb * cs.x;
    }
    const int64_t row = (int64_t)b * N + j;
    if (KV_T == CSA_F32) {
        float *dst = reinterpret_cast<float *>(c_data) + row * kD;
#pragma unroll
        for (int e = 0; e < 4; ++e) dst[lane + 32 * e] = c[e];
    } else if (KV_T == CSA_BF16) {
        __nv_bfloat16 *dst = reinterpret_cast<__nv_bfloat16 *>(c_data) + row * kD;
#pragma unroll
        for (int e = 0; e < 4; ++e) dst[lane + 32 * e] = __float2bfloat16_rn(c[e]);
    } else if (KV_T == CSA_NVFP4) {  // the whole rotated entry in NVFP4 (fp4.cuh)
        nvfp4_row_store(c, reinterpret_cast<uint8_t *>(c_data) + row * kNvfp4RowBytes);
    } else {  // MIXED: dims 0..63 FP8 + row scale, dims 64..127 BF16
        float amax = warp_max(fmaxf(fabsf(c[0]), fabsf(c[1])));
        const float scale = __fdiv_rn(amax, 448.0f);
        uint8_t *dst = reinterpret_cast<uint8_t *>(c_data) + row * 64;
        dst[lane] = scale > 0.0f ? f32_to_e4m3(__fdiv_rn(c[0], scale)) : (uint8_t)0;
        dst[lane + 32] = scale > 0.0f ? f32_to_e4m3(__fdiv_rn(c[1], scale)) : (uint8_t)0;
        if (lane == 0) c_scale[row] = scale;
        __nv_bfloat16 *rr = c_rope + row * 64;
        rr[lane] = __float2bfloat16_rn(c[2]);
        rr[lane + 32] = __float2bfloat16_rn(c[3]);
    }
    if (WITH_KI) {
        if (IDX_T == CSA_F32) {
            float *dst = reinterpret_cast<float *>(ki_data) + row * kDI;
            dst[lane] = k0;
            dst[lane + 32] = k1;
        } else if (IDX_T == CSA_MXFP4) {
            mxfp4_row_store(k0, k1, reinterpret_cast<uint8_t *>(ki_data) + row * (kDI / 2), ki_e8 + row * 2);
        } else {
            const float amax = warp_max(fmaxf(fabsf(k0), fabsf(k1)));
            const float scale = __fdiv_rn(amax, 448.0f);
            uint8_t *dst = reinterpret_cast<uint8_t *>(ki_data) + row * kDI;
            dst[lane] = scale > 0.0f ? f32_to_e4m3(__fdiv_rn(k0, scale)) : (uint8_t)0;
            dst[lane + 32] = scale > 0.0f ? f32_to_e4m3(__fdiv_rn(k1, scale)) : (uint8_t)0;
            if (lane == 0) ki_scale[row] = scale;
        }
    }
}

// kv_compress for m <= 8, streamed. One warp walks a run of up to kStreamE consecutive entries
// j0 .. j0 + E - 1 block by block (block beta = rows [beta m, (beta + 1) m)), from block j0 - 1
// (the run's halo: it only feeds entry j0) to block j0 + E - 1. Each block's KV rows,
// indexer-key rows and RoPE-table rows (contiguous in memory) are copied into the warp's ring of
// shared-memory slots kStreamD - 1 blocks ahead of their use by three bulk copies that complete
// on the slot's mbarrier, so every raw row is read from HBM once (plus one halo block per run)
// with several blocks in flight per warp. A block feeds two entries: entry beta (its own block,
// logits of set 0) and entry beta + 1 (its previous block, set 1). The warp keeps the two
// running sums; after block beta, entry beta is complete and is stored by finish_entry. The
// window weights of the run's entries are computed first, lane i for entry j0 + i.
constexpr int kStreamE = 16;     // entries per warp at most (ew: the launch's run length)
constexpr int kStreamWarps = 4;  // warps per CTA
constexpr int kStreamD = 3;      // ring slots per warp (blocks in flight: kStreamD - 1)
constexpr int kStreamMaxM = 8;

__device__ __forceinline__ void lds16(const float *p, float (&x)[4]) {
    const float4 v = *reinterpret_cast<const float4 *>(p);
    x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
}
__device__ __forceinline__ void lds16(const __nv_bfloat16 *p, float (&x)[8]) {
    const uint4 v = *reinterpret_cast<const uint4 *>(p);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w[k]));
        x[2 * k] = f.x;
        x[2 * k + 1] = f.y;
    }
}

// bytes of one ring slot (one block of m rows)
__host__ __device__ __forceinline__ int stream_slot_bytes(int m, int act_bytes, bool with_ki, bool rot) {
    return m * (kD * act_bytes + (with_ki ? kDI * 4 : 0) + (rot ? 32 * 8 : 0));
}

template <typename ActT, int KV_T, int IDX_T, bool WITH_KI, bool WITH_KVROPE>
__global__ void __launch_bounds__(kStreamWarps * 32, 5)
kv_compress_stream_kernel(const ActT *__restrict__ kv, const float *__restrict__ z,
                          const float *__restrict__ kI_raw, const float2 *__restrict__ rope,
                          void *__restrict__ c_data, __nv_bfloat16 *__restrict__ c_rope,
                          float *__restrict__ c_scale, void *__restrict__ ki_data,
                          float *__restrict__ ki_scale, uint8_t *__restrict__ ki_e8, ActT *__restrict__ kv_rope,
                          int L, int m, int N, int d_rope, int ew) {
    using namespace umma;
    constexpr int V = 16 / (int)sizeof(ActT);    // dims per 16-byte chunk
    constexpr int CPR = kD / V;                  // chunks per KV row
    constexpr int RPW = 32 / CPR;                // KV rows per warp instruction
    constexpr int KVB = kD * (int)sizeof(ActT);  // bytes per KV row
    constexpr int KIB = kDI * 4;                 // bytes per indexer-key row
    extern __shared__ __align__(16) uint8_t s_ring[];
    __shared__ float s_e[kStreamWarps][kStreamE][2 * kStreamMaxM];
    __shared__ float s_inv[kStreamWarps][kStreamE];
    __shared__ __align__(16) float s_c[kStreamWarps][kD + kDI];
    __shared__ __align__(8) uint64_t s_bar[kStreamWarps][kStreamD];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = blockIdx.y;
    const int j0 = (blockIdx.x * kStreamWarps + warp) * ew;
    if (j0 >= N) return;  // (the warp leaves as a whole; nothing below is CTA-wide)
    const int jn = min(N, j0 + ew);
    const bool rot = d_rope == 64;
    // slot: KV rows [m][KVB], indexer-key rows [m][KIB], RoPE rows [m][32 float2]
    const int kv_bytes = m * KVB, ki_bytes = WITH_KI ? m * KIB : 0;
    const int slot_bytes = stream_slot_bytes(m, (int)sizeof(ActT), WITH_KI, rot);
    uint8_t *ring = s_ring + (size_t)warp * kStreamD * slot_bytes;
    const uint32_t ring_u32 = smem_u32(ring);
    const ActT *kvb = kv + (int64_t)b * L * kD;
    const float *kib = WITH_KI ? kI_raw + (int64_t)b * L * kDI : nullptr;
    ActT *kvrb = WITH_KVROPE ? kv_rope + (int64_t)b * L * kD : nullptr;
    if (lane == 0) {
        for (int s = 0; s < kStreamD; ++s) mbar_init(smem_u32(&s_bar[warp][s]), 1);
        mbar_fence_init();
    }
    __syncwarp();

    // blocks of the run: beta = jb0 .. jn - 1, block i into slot i % kStreamD by three bulk copies
    // (lane 0) completing on the slot's barrier; rows past L are not copied and never read
    const int jb0 = j0 > 0 ? j0 - 1 : 0;
    const int nblk = jn - jb0;
    auto issue = [&](int i) {
        if (lane == 0 && i < nblk) {
            const int64_t t0 = (int64_t)(jb0 + i) * m;
            const int rows = (int)min((int64_t)m, (int64_t)L - t0);  // >= 1
            const uint32_t dst = ring_u32 + (uint32_t)((i % kStreamD) * slot_bytes);
            const uint32_t bar = smem_u32(&s_bar[warp][i % kStreamD]);
            mbar_expect_tx(bar, (uint32_t)(rows * KVB + (WITH_KI ? rows * KIB : 0) + (rot ? m * 256 : 0)));
            bulk_load(dst, kvb + t0 * kD, (uint32_t)(rows * KVB), bar);
            if (WITH_KI) bulk_load(dst + kv_bytes, kib + t0 * kDI, (uint32_t)(rows * KIB), bar);
            // the table holds every position below ceil(L / m) m
            if (rot) bulk_load(dst + kv_bytes + ki_bytes, rope + t0 * 32, (uint32_t)(m * 256), bar);
        }
    };
#pragma unroll
    for (int i = 0; i < kStreamD - 1; ++i) issue(i);

    // window weights of entry j0 + lane: s_e[.][r] = exp(logit - max) for window row r (r < m:
    // the previous block, set 1; r >= m: the own block, set 0); rows outside [0, L) weigh 0
    if (lane < ew) {
        const int j = j0 + lane;
        float lg[2 * kStreamMaxM];
        float mx = -INFINITY;
#pragma unroll
        for (int r = 0; r < 2 * kStreamMaxM; ++r) {
            const int64_t t = (int64_t)(j - 1) * m + r;
            const bool in = j < N && r < 2 * m && t >= 0 && t < L;
            lg[r] = in ? z[((int64_t)b * L + t) * 2 + (r < m ? 1 : 0)] : -INFINITY;
            mx = fmaxf(mx, lg[r]);
        }
        float den = 0.0f;
#pragma unroll
        for (int r = 0; r < 2 * kStreamMaxM; ++r) {
            const int64_t t = (int64_t)(j - 1) * m + r;
            const bool in = j < N && r < 2 * m && t >= 0 && t < L;
            const float e = in ? expf(lg[r] - mx) : 0.0f;
            den += e;
            s_e[warp][lane][r] = e;
        }
        s_inv[warp][lane] = 1.0f / den;
    }

    const int cl = lane % CPR, rl = lane / CPR, d0 = cl * V;
    const int kc = lane & 15, kr = lane >> 4;
    // running sums as float pairs (packed FMA): acc for entry beta, nxt for entry beta + 1
    uint64_t acc[V / 2], nxt[V / 2], ak[2], nk[2];
#pragma unroll
    for (int k = 0; k < V / 2; ++k) acc[k] = nxt[k] = 0ull;
    ak[0] = ak[1] = nk[0] = nk[1] = 0ull;
    // an indexer-key row chunk of window row r into the two sums
    auto ki_row = [&](const uint8_t *slot, int64_t t0, int r, float wo, float wn) {
        if (r < m && t0 + r < L) {
            const float4 x = *reinterpret_cast<const float4 *>(slot + kv_bytes + r * KIB + kc * 16);
            const uint64_t wo2 = f2_pack(wo, wo), wn2 = f2_pack(wn, wn);
            const uint64_t x01 = f2_pack(x.x, x.y), x23 = f2_pack(x.z, x.w);
            ak[0] = f2_fma(wo2, x01, ak[0]);
            ak[1] = f2_fma(wo2, x23, ak[1]);
            nk[0] = f2_fma(wn2, x01, nk[0]);
            nk[1] = f2_fma(wn2, x23, nk[1]);
        }
    };

    bool ok = true;
    int i = 0;
    for (; i < nblk; ++i) {
        issue(i + kStreamD - 1);
        if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&s_bar[warp][i % kStreamD]), (i / kStreamD) & 1, kWaitNs,
                                               &g_abort))) {
            ok = false;
            break;
        }
        const int beta = jb0 + i;
        const uint8_t *slot = ring + (size_t)(i % kStreamD) * slot_bytes;
        const float2 *slot_rope = reinterpret_cast<const float2 *>(slot + kv_bytes + ki_bytes);
        const bool own = beta >= j0;          // entry beta is in the run (else: the halo block)
        const bool has_next = beta + 1 < jn;  // entry beta + 1 is in the run
        const float *e_own = s_e[warp][own ? beta - j0 : 0] + m;
        const float *e_nxt = s_e[warp][has_next ? beta + 1 - j0 : 0];
        const int64_t t0 = (int64_t)beta * m;
        for (int r0 = 0; r0 < m; r0 += RPW) {
            const int r = r0 + rl;
            const bool have = r < m && t0 + r < L;
            float x[V];
            if (have) {
                lds16(reinterpret_cast<const ActT *>(slot + r * KVB) + d0, x);
            } else {
#pragma unroll
                for (int k = 0; k < V; ++k) x[k] = 0.0f;
            }
            const float wo = own && have ? e_own[r] : 0.0f;
            const float wn = has_next && have ? e_nxt[r] : 0.0f;
            const uint64_t wo2 = f2_pack(wo, wo), wn2 = f2_pack(wn, wn);
#pragma unroll
            for (int k = 0; k < V / 2; ++k) {
                const uint64_t x2 = f2_pack(x[2 * k], x[2 * k + 1]);
                acc[k] = f2_fma(wo2, x2, acc[k]);
                nxt[k] = f2_fma(wn2, x2, nxt[k]);
            }
            // BF16 rows: the indexer-key row of the same window row sits in the same lanes' half
            if (WITH_KI && RPW == 2) ki_row(slot, t0, r, wo, wn);
            if (WITH_KVROPE && own) {  // the row back, rotated at its own position t0 + r
                float y[V];
#pragma unroll
                for (int k = 0; k < V; ++k) y[k] = x[k];
                if (rot) {
                    float other[V];
#pragma unroll
                    for (int k = 0; k < V; ++k) other[k] = __shfl_xor_sync(0xffffffffu, x[k], 32 / V);
                    if (have && d0 >= 64) {
                        // dims 64 + i (first of the pair): x cos - x' sin; 96 + i: x cos + x' sin
                        const float sg = d0 < 96 ? -1.0f : 1.0f;
                        const int ip = (d0 - 64) & 31;  // pair index of the chunk's first dim
                        const float4 *r4 = reinterpret_cast<const float4 *>(slot_rope + r * 32 + ip);
#pragma unroll
                        for (int k2 = 0; k2 < V / 2; ++k2) {
                            const float4 cs = r4[k2];  // (cos, sin) of pairs ip + 2 k2 and ip + 2 k2 + 1
                            y[2 * k2] = fmaf(sg * other[2 * k2], cs.y, x[2 * k2] * cs.x);
                            y[2 * k2 + 1] = fmaf(sg * other[2 * k2 + 1], cs.w, x[2 * k2 + 1] * cs.z);
                        }
                    }
                }
                if (have) store16(kvrb + (t0 + r) * kD + d0, y);
            }
        }
        if (WITH_KI && RPW == 1) {
            for (int r0 = 0; r0 < m; r0 += 2) {
                const int r = r0 + kr;
                const bool have = r < m && t0 + r < L;
                ki_row(slot, t0, r, own && have ? e_own[r] : 0.0f, has_next && have ? e_nxt[r] : 0.0f);
            }
        }
        if (own) {  // entry beta is complete
            float a[V];
#pragma unroll
            for (int k = 0; k < V / 2; ++k) {
                const float2 f = f2_unpack(acc[k]);
                a[2 * k] = f.x;
                a[2 * k + 1] = f.y;
            }
            if (RPW == 2) {
#pragma unroll
                for (int k = 0; k < V; ++k) a[k] += __shfl_xor_sync(0xffffffffu, a[k], 16);
            }
            if (rl == 0) {
#pragma unroll
                for (int k = 0; k < V; ++k) s_c[warp][d0 + k] = a[k];
            }
            if (WITH_KI) {
                float q[4];
                const float2 f0 = f2_unpack(ak[0]), f1 = f2_unpack(ak[1]);
                q[0] = f0.x; q[1] = f0.y; q[2] = f1.x; q[3] = f1.y;
#pragma unroll
                for (int k = 0; k < 4; ++k) q[k] += __shfl_xor_sync(0xffffffffu, q[k], 16);
                if (kr == 0) {
#pragma unroll
                    for (int k = 0; k < 4; ++k) s_c[warp][kD + kc * 4 + k] = q[k];
                }
            }
            __syncwarp();
            const float inv = s_inv[warp][beta - j0];
            float c[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) c[q] = s_c[warp][lane + 32 * q] * inv;
            const float k0 = WITH_KI ? s_c[warp][kD + lane] * inv : 0.0f;
            const float k1 = WITH_KI ? s_c[warp][kD + lane + 32] * inv : 0.0f;
            // the entry position (beta + 1) m - 1 is the block's last row: its RoPE row is in the slot
            finish_entry<KV_T, IDX_T, WITH_KI>(c, k0, k1, beta, b, N, rot ? slot_rope + (m - 1) * 32 : nullptr,
                                               c_data, c_rope, c_scale, ki_data, ki_scale, ki_e8);
        }
#pragma unroll
        for (int k = 0; k < V / 2; ++k) {
            acc[k] = nxt[k];
            nxt[k] = 0ull;
        }
        ak[0] = nk[0]; ak[1] = nk[1];
        nk[0] = nk[1] = 0ull;
        __syncwarp();  // slot i and s_c are free for reuse
    }
    if (!ok) {
        set_timeout();
        // copies still in flight land before the warp leaves (bounded)
        if (lane == 0)
            for (int f = i; f < min(nblk, i + kStreamD); ++f)
                mbar_wait(smem_u32(&s_bar[warp][f % kStreamD]), (f / kStreamD) & 1, kDrainNs);
        __syncwarp();
    }
}

// kv_compress for m > 8, streamed by CTAs. A CTA of kRunThreads walks a run of up to kRunE
// consecutive entries j0 .. j0 + E - 1 over blocks j0 - 1 .. j0 + E - 1 (block beta = rows
// [beta m, (beta + 1) m); block j0 - 1 is the run's halo and only feeds entry j0), in stages of
// kRunG rows: thread 0 bulk-copies a stage's KV rows, indexer-key rows and (outside the halo)
// RoPE-table rows into a ring of kRunS shared-memory slots kRunS - 1 stages ahead, completing on
// the slot's mbarrier. Every thread adds its 16-byte chunks of the stage's rows into two running
// sums (entry beta with the set-0 weights of its own block, entry beta + 1 with the set-1 weights
// of its previous block) and writes its rows of the own blocks back rotated (kv_rope). After a
// block's last stage the partial sums meet in shared memory and warp 0 stores entry beta. The
// window weights of the run's entries are computed first, one warp per entry.
constexpr int kRunThreads = 256;
constexpr int kRunWarps = kRunThreads / 32;
constexpr int kRunE = 4;   // entries per CTA at most (ec: the launch's run length)
constexpr int kRunG = 64;  // rows per stage
constexpr int kRunS = 3;   // ring slots (stages in flight: kRunS - 1)

__host__ __device__ __forceinline__ int run_stage_bytes(int act_bytes, bool with_ki, bool rot) {
    return kRunG * (kD * act_bytes + (with_ki ? kDI * 4 : 0) + (rot ? 32 * 8 : 0));
}
__host__ __device__ __forceinline__ int run_smem_bytes(int m, int act_bytes, bool with_ki, bool rot) {
    return kRunS * run_stage_bytes(act_bytes, with_ki, rot) + kRunE * 2 * m * 4 + kRunE * 4 +
           kRunWarps * (kD + kDI) * 4;
}

template <typename ActT, int KV_T, int IDX_T, bool WITH_KI, bool WITH_KVROPE>
__global__ void __launch_bounds__(kRunThreads)
kv_compress_run_kernel(const ActT *__restrict__ kv, const float *__restrict__ z,
                       const float *__restrict__ kI_raw, const float2 *__restrict__ rope,
                       void *__restrict__ c_data, __nv_bfloat16 *__restrict__ c_rope,
                       float *__restrict__ c_scale, void *__restrict__ ki_data,
                       float *__restrict__ ki_scale, uint8_t *__restrict__ ki_e8, ActT *__restrict__ kv_rope,
                       int L, int m, int N, int d_rope, int ec) {
    using namespace umma;
    constexpr int V = 16 / (int)sizeof(ActT);    // dims per 16-byte chunk
    constexpr int CPR = kD / V;                  // chunks per KV row
    constexpr int RPW = 32 / CPR;                // KV rows per warp instruction
    constexpr int KVB = kD * (int)sizeof(ActT);  // bytes per KV row
    constexpr int KIB = kDI * 4;                 // bytes per indexer-key row
    constexpr int RG = kRunWarps * RPW;          // KV rows per CTA pass (row groups)
    extern __shared__ __align__(16) uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t s_bar[kRunS];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int b = blockIdx.y;
    const int j0 = blockIdx.x * ec;
    const int jn = min(N, j0 + ec);
    const bool rot = d_rope == 64;
    const int kv_bytes = kRunG * KVB, ki_bytes = WITH_KI ? kRunG * KIB : 0;
    const int stage_bytes = run_stage_bytes((int)sizeof(ActT), WITH_KI, rot);
    uint8_t *ring = smem_raw;
    float *s_e = reinterpret_cast<float *>(smem_raw + kRunS * stage_bytes);  // [kRunE][2m]
    float *s_inv = s_e + kRunE * 2 * m;                                       // [kRunE]
    float *s_red = s_inv + kRunE;  // [kRunWarps][kD]: KV partial sums, then [kRunWarps][kDI] keys
    float *s_redk = s_red + kRunWarps * kD;
    const ActT *kvb = kv + (int64_t)b * L * kD;
    const float *kib = WITH_KI ? kI_raw + (int64_t)b * L * kDI : nullptr;
    ActT *kvrb = WITH_KVROPE ? kv_rope + (int64_t)b * L * kD : nullptr;
    if (tid == 0) {
        for (int q = 0; q < kRunS; ++q) mbar_init(smem_u32(&s_bar[q]), 1);
        mbar_fence_init();
    }
    __syncthreads();

    // stages: block jb0 + q / ns, rows [(q % ns) G, min((q % ns + 1) G, m)) of it
    const int jb0 = j0 > 0 ? j0 - 1 : 0;
    const int ns = (m + kRunG - 1) / kRunG;
    const int nq = (jn - jb0) * ns;
    auto issue = [&](int q) {  // by thread 0
        if (q < nq) {
            const int beta = jb0 + q / ns, s0 = (q % ns) * kRunG;
            const int64_t t0 = (int64_t)beta * m + s0;
            // rows of the stage below L (a stage of the last block may have none: its barrier
            // phase then completes by a plain arrival)
            const int rows = (int)min((int64_t)min(kRunG, m - s0), (int64_t)L - t0);
            const uint32_t bar = smem_u32(&s_bar[q % kRunS]);
            if (rows <= 0) {
                mbar_arrive(bar);
                return;
            }
            const bool rr = rot && beta >= j0;  // RoPE rows: own blocks only
            const uint32_t dst = smem_u32(ring + (q % kRunS) * stage_bytes);
            mbar_expect_tx(bar, (uint32_t)(rows * KVB + (WITH_KI ? rows * KIB : 0) + (rr ? rows * 256 : 0)));
            bulk_load(dst, kvb + t0 * kD, (uint32_t)(rows * KVB), bar);
            if (WITH_KI) bulk_load(dst + kv_bytes, kib + t0 * kDI, (uint32_t)(rows * KIB), bar);
            if (rr) bulk_load(dst + kv_bytes + ki_bytes, rope + t0 * 32, (uint32_t)(rows * 256), bar);
        }
    };
    if (tid == 0)
        for (int q = 0; q < kRunS - 1; ++q) issue(q);

    // window weights: s_e[e][r] = exp(logit - max) of window row r of entry j0 + e (r < m: the
    // previous block, set 1; r >= m: the own block, set 0); rows outside [0, L) weigh 0. Logits
    // of the rows [(j0 - 1) m, jn m) first, by every thread: row i of that range (block
    // j0 - 1 + i / m) is an own row of entry j0 + i / m - 1 and a previous row of the next one.
    const int ne = jn - j0;
    const int nrow = (ne + 1) * m;
#pragma unroll 4
    for (int i = tid; i < nrow; i += kRunThreads) {
        const int64_t t = (int64_t)(j0 - 1) * m + i;
        const bool in = t >= 0 && t < L;
        const float z0 = in ? z[((int64_t)b * L + t) * 2] : -INFINITY;
        const float z1 = in ? z[((int64_t)b * L + t) * 2 + 1] : -INFINITY;
        const int e = i / m - 1, rb = i - (i / m) * m;  // e = -1: the halo block
        if (e >= 0) s_e[e * 2 * m + m + rb] = z0;
        if (e + 1 < ne) s_e[(e + 1) * 2 * m + rb] = z1;
    }
    __syncthreads();
    for (int e = warp; e < ne; e += kRunWarps) {
        float *we = s_e + e * 2 * m;
        float mx = -INFINITY;
        for (int r = lane; r < 2 * m; r += 32) mx = fmaxf(mx, we[r]);
        mx = warp_max(mx);
        float den = 0.0f;
        for (int r = lane; r < 2 * m; r += 32) {
            const float w = we[r] == -INFINITY ? 0.0f : expf(we[r] - mx);
            we[r] = w;
            den += w;
        }
        den = warp_sum(den);
        if (lane == 0) s_inv[e] = 1.0f / den;
    }
    __syncthreads();

    const int cl = lane % CPR, rl = lane / CPR, d0 = cl * V;
    const int kc = lane & 15, kr = lane >> 4;
    uint64_t acc[V / 2], nxt[V / 2], ak[2], nk[2];
#pragma unroll
    for (int k = 0; k < V / 2; ++k) acc[k] = nxt[k] = 0ull;
    ak[0] = ak[1] = nk[0] = nk[1] = 0ull;
    bool ok = true;
    int q = 0;
    for (; q < nq; ++q) {
        if (tid == 0) issue(q + kRunS - 1);
        const bool got = mbar_wait(smem_u32(&s_bar[q % kRunS]), (q / kRunS) & 1, kWaitNs, &g_abort);
        if (!__syncthreads_and(got)) {
            ok = false;
            break;
        }
        const int beta = jb0 + q / ns, s0 = (q % ns) * kRunG;
        const int64_t t0 = (int64_t)beta * m + s0;
        const int rows = (int)min((int64_t)min(kRunG, m - s0), (int64_t)L - t0);
        const uint8_t *slot = ring + (q % kRunS) * stage_bytes;
        const float2 *slot_rope = reinterpret_cast<const float2 *>(slot + kv_bytes + ki_bytes);
        const bool own = beta >= j0, has_next = beta + 1 < jn;
        const float *e_own = s_e + (own ? beta - j0 : 0) * 2 * m + m + s0;
        const float *e_nxt = s_e + (has_next ? beta + 1 - j0 : 0) * 2 * m + s0;
        for (int r0 = warp * RPW; r0 < rows; r0 += RG) {  // (uniform over the warp)
            const int r = r0 + rl;
            const bool have = r < rows;
            float x[V];
            if (have) {
                lds16(reinterpret_cast<const ActT *>(slot + r * KVB) + d0, x);
            } else {
#pragma unroll
                for (int k = 0; k < V; ++k) x[k] = 0.0f;
            }
            const float wo = own && have ? e_own[r] : 0.0f, wn = has_next && have ? e_nxt[r] : 0.0f;
            const uint64_t wo2 = f2_pack(wo, wo), wn2 = f2_pack(wn, wn);
#pragma unroll
            for (int k = 0; k < V / 2; ++k) {
                const uint64_t x2 = f2_pack(x[2 * k], x[2 * k + 1]);
                acc[k] = f2_fma(wo2, x2, acc[k]);
                nxt[k] = f2_fma(wn2, x2, nxt[k]);
            }
            if (WITH_KVROPE && own) {  // the row back, rotated at its own position t0 + r
                float y[V];
#pragma unroll
                for (int k = 0; k < V; ++k) y[k] = x[k];
                if (rot) {
                    float other[V];  // the partner chunk (dims 32 apart): lane ^ (32 / V)
#pragma unroll
                    for (int k = 0; k < V; ++k) other[k] = __shfl_xor_sync(0xffffffffu, x[k], 32 / V);
                    if (have && d0 >= 64) {
                        const float sg = d0 < 96 ? -1.0f : 1.0f;
                        const int ip = (d0 - 64) & 31;
                        const float4 *r4 = reinterpret_cast<const float4 *>(slot_rope + r * 32 + ip);
#pragma unroll
                        for (int k2 = 0; k2 < V / 2; ++k2) {
                            const float4 cs = r4[k2];
                            y[2 * k2] = fmaf(sg * other[2 * k2], cs.y, x[2 * k2] * cs.x);
                            y[2 * k2 + 1] = fmaf(sg * other[2 * k2 + 1], cs.w, x[2 * k2 + 1] * cs.z);
                        }
                    }
                }
                if (have) store16(kvrb + (t0 + r) * kD + d0, y);
            }
        }
        if (WITH_KI) {
            for (int r = warp * 2 + kr; r < rows; r += kRunWarps * 2) {
                const float4 x = *reinterpret_cast<const float4 *>(slot + kv_bytes + r * KIB + kc * 16);
                const float wo = own ? e_own[r] : 0.0f, wn = has_next ? e_nxt[r] : 0.0f;
                const uint64_t wo2 = f2_pack(wo, wo), wn2 = f2_pack(wn, wn);
                const uint64_t x01 = f2_pack(x.x, x.y), x23 = f2_pack(x.z, x.w);
                ak[0] = f2_fma(wo2, x01, ak[0]);
                ak[1] = f2_fma(wo2, x23, ak[1]);
                nk[0] = f2_fma(wn2, x01, nk[0]);
                nk[1] = f2_fma(wn2, x23, nk[1]);
            }
        }
        if (own && q % ns == ns - 1) {  // entry beta is complete: partial sums meet, warp 0 stores it
            float a[V];
#pragma unroll
            for (int k = 0; k < V / 2; ++k) {
                const float2 f = f2_unpack(acc[k]);
                a[2 * k] = f.x;
                a[2 * k + 1] = f.y;
            }
            if (RPW == 2) {
#pragma unroll
                for (int k = 0; k < V; ++k) a[k] += __shfl_xor_sync(0xffffffffu, a[k], 16);
            }
            if (rl == 0) {
#pragma unroll
                for (int k = 0; k < V; ++k) s_red[warp * kD + d0 + k] = a[k];
            }
            if (WITH_KI) {
                const float2 f0 = f2_unpack(ak[0]), f1 = f2_unpack(ak[1]);
                float qk[4] = {f0.x, f0.y, f1.x, f1.y};
#pragma unroll
                for (int k = 0; k < 4; ++k) qk[k] += __shfl_xor_sync(0xffffffffu, qk[k], 16);
                if (kr == 0) {
#pragma unroll
                    for (int k = 0; k < 4; ++k) s_redk[warp * kDI + kc * 4 + k] = qk[k];
                }
            }
            __syncthreads();
            if (warp == 0) {
                const float inv = s_inv[beta - j0];
                float c[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                float k0 = 0.0f, k1 = 0.0f;
                for (int w = 0; w < kRunWarps; ++w) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) c[e] += s_red[w * kD + lane + 32 * e];
                    if (WITH_KI) {
                        k0 += s_redk[w * kDI + lane];
                        k1 += s_redk[w * kDI + lane + 32];
                    }
                }
#pragma unroll
                for (int e = 0; e < 4; ++e) c[e] *= inv;
                k0 *= inv;
                k1 *= inv;
                // the entry position (beta + 1) m - 1: the last row of the block
                finish_entry<KV_T, IDX_T, WITH_KI>(c, k0, k1, beta, b, N,
                                                   rot ? rope + ((int64_t)(beta + 1) * m - 1) * 32 : nullptr, c_data,
                                                   c_rope, c_scale, ki_data, ki_scale, ki_e8);
            }
        }
        if (q % ns == ns - 1) {  // the next block: entry beta + 1's sum so far, a new one after it
#pragma unroll
            for (int k = 0; k < V / 2; ++k) {
                acc[k] = nxt[k];
                nxt[k] = 0ull;
            }
            ak[0] = nk[0]; ak[1] = nk[1];
            nk[0] = nk[1] = 0ull;
        }
        __syncthreads();  // slot q and the partial sums are free for reuse
    }
    if (!ok) {
        if (tid == 0) {
            set_timeout();
            // copies still in flight land before the CTA leaves (bounded)
            for (int f = q; f < min(nq, q + kRunS); ++f) mbar_wait(smem_u32(&s_bar[f % kRunS]), (f / kRunS) & 1, kDrainNs);
        }
        __syncthreads();
    }
}

template <typename ActT, int KV_T, int IDX_T>
static void launch_compress_t(const CompressArgs &a, cudaStream_t st) {
    const ActT *kv = reinterpret_cast<const ActT *>(a.kv);
    ActT *kvr = reinterpret_cast<ActT *>(a.kv_rope);
    const float2 *rope = reinterpret_cast<const float2 *>(a.rope_tab);
    auto *cr = reinterpret_cast<__nv_bfloat16 *>(a.c_rope);
    // m <= 8: runs of entries per warp; larger m: runs of entries per CTA
    const bool rot = a.d_rope == 64, with_ki = a.kI_raw != nullptr;
    const int wsmem = kStreamWarps * kStreamD * stream_slot_bytes(a.m, (int)sizeof(ActT), with_ki, rot);
    // run lengths: the longest (fewest halo blocks) that still gives every SM a few CTAs
    const int64_t units = (int64_t)a.N * a.B;
    const int ew = (int)std::max<int64_t>(1, std::min<int64_t>(kStreamE, units / (4 * kStreamWarps * 148)));
    const int ec = (int)std::max<int64_t>(1, std::min<int64_t>(kRunE, units / (2 * 148)));
    const dim3 wgrid((a.N + ew * kStreamWarps - 1) / (ew * kStreamWarps), a.B);
    const int csmem = run_smem_bytes(a.m, (int)sizeof(ActT), with_ki, rot);
    const dim3 cgrid((a.N + ec - 1) / ec, a.B);
#define CSA_LAUNCH(KI, KVR)                                                                                   \
    do {                                                                                                      \
    if (a.m <= kStreamMaxM) {                                                                                 \
        auto kern = kv_compress_stream_kernel<ActT, KV_T, IDX_T, KI, KVR>;                                    \
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, wsmem);                       \
        kern<<<wgrid, kStreamWarps * 32, wsmem, st>>>(kv, a.z, a.kI_raw, rope, a.c_data, cr, a.c_scale, a.ki_data, \
                                                       a.ki_scale, a.ki_e8, kvr, a.L, a.m, a.N, a.d_rope, ew);  \
    } else {                                                                                                  \
        auto kern = kv_compress_run_kernel<ActT, KV_T, IDX_T, KI, KVR>;                                       \
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, csmem);                       \
        kern<<<cgrid, kRunThreads, csmem, st>>>(kv, a.z, a.kI_raw, rope, a.c_data, cr, a.c_scale, a.ki_data,   \
                                                a.ki_scale, a.ki_e8, kvr, a.L, a.m, a.N, a.d_rope, ec);         \
    }                                                                                                         \
    } while (0)
    if (a.kI_raw && a.kv_rope) CSA_LAUNCH(true, true);
    else if (a.kI_raw) CSA_LAUNCH(true, false);
    else if (a.kv_rope) CSA_LAUNCH(false, true);
    else CSA_LAUNCH(false, false);
#undef CSA_LAUNCH
}

template <typename ActT, int KV_T>
static void launch_compress_k(const CompressArgs &a, cudaStream_t st) {
    if (a.idx_t == CSA_FP8E4M3) launch_compress_t<ActT, KV_T, CSA_FP8E4M3>(a, st);
    else if (a.idx_t == CSA_MXFP4) launch_compress_t<ActT, KV_T, CSA_MXFP4>(a, st);
    else launch_compress_t<ActT, KV_T, CSA_F32>(a, st);
}

template <typename ActT>
static void launch_compress_a(const CompressArgs &a, cudaStream_t st) {
    if (a.kv_t == CSA_F32) launch_compress_k<ActT, CSA_F32>(a, st);
    else if (a.kv_t == CSA_BF16) launch_compress_k<ActT, CSA_BF16>(a, st);
    else if (a.kv_t == CSA_NVFP4) launch_compress_k<ActT, CSA_NVFP4>(a, st);
    else launch_compress_k<ActT, CSA_MIXED>(a, st);
}

void launch_kv_compress(const CompressArgs &a, cudaStream_t st) {
    if (a.act_t == CSA_F32) launch_compress_a<float>(a, st);
    else launch_compress_a<__nv_bfloat16>(a, st);
    count_launches(1);
}

}  // namespace csa
