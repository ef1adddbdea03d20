// gemm.cu -- BF16 GEMM on the tensor cores for the projections on either side of the attention
// core: the hidden-state projections to the layer's inputs and the grouped output projection.
//
// Sources: [P2] "DeepSeek-V4: Towards Highly Efficient Million-Token Context Intelligence"
// (wiki notes), 概要 (V4-Flash hidden size 4096) and 提案手法 §1 CSA (shared-KV multi-query
// attention with a grouped output projection); [P5] "deepseek V4 技术论文" 一.1 (共享KV MQA与分组
// 输出投影: the grouped projection further cuts the compute).
//
// C[M, N] = A[M, K] B[N, K]^T, BF16 operands (both K-major, rows of A and B with their own
// strides), FP32 accumulation in TMEM. With groups > 1 the product is block-diagonal: output
// columns [g N/groups, (g+1) N/groups) read A's columns [g K, (g+1) K) (A has groups*K columns),
// i.e. each group of heads is projected by its own matrix, stacked in B. The output columns are
// written to up to four segments, each a row-major BF16 or FP32 tensor of its own (so that one
// product can produce q, kv and the indexer inputs as separate contiguous tensors).
//
// Persistent kernel, one CTA per SM, 192 threads: warps 0-3 epilogue (TMEM lanes = tile rows),
// warp 4 TMA producer, warp 5 lane 0 MMA issue. Tiles of 128 x 256 (MMA M = 128, N = 256), K in
// steps of 64 (128-byte rows, 128-byte swizzle), four A/B stages in shared memory, the
// accumulator double-buffered in TMEM (2 x 256 columns) so that a tile's epilogue overlaps the
// next tile's MMAs. Every wait is bounded.
#include "common.cuh"
#include "kernels.cuh"
#include "tma_host.cuh"
#include "umma.cuh"

namespace csa {
using namespace umma;

namespace gm {
constexpr int kBM = 128, kBN = 256, kBK = 64;
constexpr int kStages = 4;
constexpr int kABytes = kBM * kBK * 2;   // 16 KB
constexpr int kBBytes = kBN * kBK * 2;   // 32 KB
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kSmemBytes = kStages * kStageBytes + 1024;
constexpr int kThreads = 192;
constexpr int kProdWarp = 4, kMmaWarp = 5;
constexpr uint32_t kTmemCols = 512;
}  // namespace gm

struct GemmParams {
    CUtensorMap ma;   // A [M][groups*K] bf16, box 64 x 128, 128-byte swizzle
    CUtensorMap mb;   // B [N][K] bf16, box 64 x 256, 128-byte swizzle
    GemmOut out[4];
    int n_out;
    int M, N, K, groups, n_per_group;
    int tiles_m, tiles_n;
};

template <typename F>
__device__ __forceinline__ void gemm_tile_of(const GemmParams &P, int tile, F &&fn) {
    const int tn = tile % P.tiles_n, tm = tile / P.tiles_n;  // consecutive tiles share A rows
    fn(tm * gm::kBM, tn * gm::kBN);
}

__global__ void __launch_bounds__(gm::kThreads, 1) gemm_bf16_kernel(const __grid_constant__ GemmParams P) {
    using namespace gm;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ __align__(8) uint64_t b_full[kStages], b_empty[kStages], b_afull[2], b_aempty[2];
    __shared__ uint32_t tmem_slot;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t s_base = smem_u32(sm);
    if (warp == 0) {
        tmem_alloc(smem_u32(&tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(smem_u32(&b_full[i]), 1);
            mbar_init(smem_u32(&b_empty[i]), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&b_afull[i]), 1);
            mbar_init(smem_u32(&b_aempty[i]), 4);
        }
        mbar_fence_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    const int n_tiles = P.tiles_m * P.tiles_n;
    const int ksteps = P.K / kBK;
    bool ok = true;

    if (warp == kProdWarp) {
        if (lane == 0) {
            int s = 0;
            for (int tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x) {
                int m0 = 0, n0 = 0;
                gemm_tile_of(P, tile, [&](int a, int b) { m0 = a; n0 = b; });
                const int akoff = P.groups > 1 ? (n0 / P.n_per_group) * P.K : 0;
                for (int kk = 0; kk < ksteps; ++kk, ++s) {
                    const int st = s % kStages;
                    if (s >= kStages && !mbar_wait(smem_u32(&b_empty[st]), ((s / kStages) - 1) & 1, kWaitNs, &g_abort)) {
                        ok = false;
                        break;
                    }
                    const uint32_t dst = s_base + st * kStageBytes;
                    mbar_expect_tx(smem_u32(&b_full[st]), kStageBytes);
                    tma_load_3d(dst, &P.ma, smem_u32(&b_full[st]), akoff + kk * kBK, m0, 0);
                    tma_load_3d(dst + kABytes, &P.mb, smem_u32(&b_full[st]), kk * kBK, n0, 0);
                }
            }
            if (!ok) {
                set_timeout();
                for (int f = max(0, s - kStages); f < s; ++f)
                    mbar_wait(smem_u32(&b_full[f % kStages]), (f / kStages) & 1, kDrainNs);
            }
        }
    } else if (warp == kMmaWarp) {
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16(kBM, kBN, 0, 0);
            int s = 0, t = 0;
            for (int tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x, ++t) {
                const int ab = t & 1;
                if (t >= 2 && !mbar_wait(smem_u32(&b_aempty[ab]), ((t >> 1) - 1) & 1, kWaitNs, &g_abort)) {
                    ok = false;
                    break;
                }
                for (int kk = 0; kk < ksteps; ++kk, ++s) {
                    const int st = s % kStages;
                    if (!mbar_wait(smem_u32(&b_full[st]), (s / kStages) & 1, kWaitNs, &g_abort)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t a = s_base + st * kStageBytes, b = a + kABytes;
#pragma unroll
                    for (int k4 = 0; k4 < kBK / 16; ++k4)
                        mma_bf16(tmem + ab * kBN, sdesc_sw128(a + k4 * 32, 16, 1024), sdesc_sw128(b + k4 * 32, 16, 1024),
                                 idesc, (kk > 0 || k4 > 0) ? 1u : 0u);
                    mma_commit(smem_u32(&b_empty[st]));
                }
                if (!ok) break;
                mma_commit(smem_u32(&b_afull[ab]));
            }
            if (!ok) {
                set_timeout();
                if (s > 0) mbar_wait(smem_u32(&b_empty[(s - 1) % kStages]), ((s - 1) / kStages) & 1, kDrainNs);
            }
        }
    } else {
        // epilogue: thread = one row of the tile (TMEM lane), 32 columns at a time
        const uint32_t lane_base = (uint32_t)(32 * warp) << 16;
        int t = 0;
        for (int tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x, ++t) {
            int m0 = 0, n0 = 0;
            gemm_tile_of(P, tile, [&](int a, int b) { m0 = a; n0 = b; });
            const int ab = t & 1;
            if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&b_afull[ab]), (t >> 1) & 1, kWaitNs, &g_abort))) {
                ok = false;
                break;
            }
            tc_fence_after();
            const int row = m0 + tid;
#pragma unroll 1
            for (int c0 = 0; c0 < kBN; c0 += 32) {
                float v[32];
                tmem_ld32_sync(tmem + lane_base + ab * kBN + c0, v);
                if (c0 + 32 == kBN) {  // the accumulator is in registers: release it
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(&b_aempty[ab]));
                }
                if (row >= P.M) continue;
                // columns n0 + c0 .. n0 + c0 + 31 into their segments: 16-byte stores when the
                // chunk lies in one segment at an aligned address, else element by element
                const int cb = n0 + c0;
#pragma unroll 1
                for (int o = 0; o < P.n_out; ++o) {
                    const GemmOut &g = P.out[o];
                    const int lo = max(g.col0, cb), hi = min(g.col1, min(cb + 32, P.N));
                    if (lo >= hi) continue;
                    if (g.dtype == CSA_F32) {
                        float *dst = reinterpret_cast<float *>(g.ptr) + (int64_t)row * g.ld - g.col0;
                        if (lo == cb && hi == cb + 32 && ((reinterpret_cast<uintptr_t>(dst + cb)) & 15) == 0) {
#pragma unroll
                            for (int c = 0; c < 32; c += 4)
                                *reinterpret_cast<float4 *>(dst + cb + c) = make_float4(v[c], v[c + 1], v[c + 2], v[c + 3]);
                        } else {
#pragma unroll
                            for (int c = 0; c < 32; ++c)
                                if (cb + c >= lo && cb + c < hi) dst[cb + c] = v[c];
                        }
                    } else {
                        __nv_bfloat16 *dst = reinterpret_cast<__nv_bfloat16 *>(g.ptr) + (int64_t)row * g.ld - g.col0;
                        if (lo == cb && hi == cb + 32 && ((reinterpret_cast<uintptr_t>(dst + cb)) & 15) == 0) {
#pragma unroll
                            for (int c = 0; c < 32; c += 8) {
                                uint4 w;
                                __nv_bfloat162 *w2 = reinterpret_cast<__nv_bfloat162 *>(&w);
#pragma unroll
                                for (int e = 0; e < 4; ++e) w2[e] = __floats2bfloat162_rn(v[c + 2 * e], v[c + 2 * e + 1]);
                                *reinterpret_cast<uint4 *>(dst + cb + c) = w;
                            }
                        } else {
#pragma unroll
                            for (int c = 0; c < 32; ++c)
                                if (cb + c >= lo && cb + c < hi) dst[cb + c] = __float2bfloat16_rn(v[c]);
                        }
                    }
                }
            }
        }
        if (!ok && lane == 0) set_timeout();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

int launch_gemm_bf16(const GemmArgs &a, cudaStream_t st) {
    using namespace gm;
    if (a.M < 1 || a.N < 1 || a.K < kBK || a.K % kBK != 0 || a.groups < 1 || a.N % a.groups != 0) return CSA_ERR_INVALID;
    if (a.groups > 1 && (a.N / a.groups) % kBN != 0) return CSA_ERR_UNSUPPORTED;  // a tile stays in one group
    if (a.n_out < 1 || a.n_out > 4) return CSA_ERR_INVALID;
    GemmParams P;
    memset(&P, 0, sizeof(P));
    // row strides in bytes must be multiples of 16 for the tensor maps
    if ((a.lda * 2) % 16 != 0 || (a.ldb * 2) % 16 != 0) return CSA_ERR_INVALID;
    const uint64_t acols = (uint64_t)a.K * a.groups;
    EncodeTiledFn fn = encode_fn();
    if (!fn) return CSA_ERR_UNSUPPORTED;
    auto map2d = [&](CUtensorMap *m, const void *base, uint64_t cols, uint64_t rows, uint64_t ld, uint32_t box_rows) {
        cuuint64_t dims[3] = {cols, rows, 1};
        cuuint64_t strides[2] = {ld * 2, ld * 2 * rows};
        cuuint32_t box[3] = {(cuuint32_t)kBK, box_rows, 1};
        cuuint32_t es[3] = {1, 1, 1};
        return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    };
    if (!map2d(&P.ma, a.A, acols, (uint64_t)a.M, (uint64_t)a.lda, kBM)) return CSA_ERR_UNSUPPORTED;
    if (!map2d(&P.mb, a.B, (uint64_t)a.K, (uint64_t)a.N, (uint64_t)a.ldb, kBN)) return CSA_ERR_UNSUPPORTED;
    for (int i = 0; i < a.n_out; ++i) P.out[i] = a.out[i];
    P.n_out = a.n_out;
    P.M = a.M; P.N = a.N; P.K = a.K; P.groups = a.groups; P.n_per_group = a.N / a.groups;
    P.tiles_m = (a.M + kBM - 1) / kBM;
    P.tiles_n = (a.N + kBN - 1) / kBN;
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int n_tiles = P.tiles_m * P.tiles_n;
    cudaFuncSetAttribute(gemm_bf16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    gemm_bf16_kernel<<<n_tiles < sms ? n_tiles : sms, kThreads, kSmemBytes, st>>>(P);
    count_launches(1);
    return CSA_OK;
}

}  // namespace csa
