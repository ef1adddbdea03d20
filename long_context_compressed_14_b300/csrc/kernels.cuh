// kernels.cuh -- launch interfaces between the C-ABI layer (api.cu) and the kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/csa.h"

namespace csa {

struct CompressArgs {
    const void *kv;
    const float *z;
    const float *kI_raw;
    const float *rope_tab;
    void *c_data;
    void *c_rope;
    float *c_scale;
    void *ki_data;
    float *ki_scale;
    uint8_t *ki_e8;        // MXFP4 keys: E8M0 exponents [B, N, 2]
    void *kv_rope;
    int B, L, m, N, d_rope, act_t, kv_t, idx_t;
};

// Indexer scores of a block of query rows of ONE sequence (prefill) or of one query per
// sequence (decode) into S[r][j], r = local row, j < visible(row).
struct IndexArgs {
    const void *qI;        // rows [.., H_I, d_I] (F32 float, FP8 codes or MXFP4 codes)
    const float *qI_scale; // FP8: [.., H_I]
    const uint8_t *qI_e8;  // MXFP4: [.., H_I, d_I / 32] E8M0 block exponents
    const void *KI;        // [B, ncap, d_I]
    const float *KI_scale; // FP8: [B, ncap]
    const uint8_t *KI_e8;  // MXFP4: [B, ncap, d_I / 32]
    const float *w;        // [.., H_I]
    const int32_t *ctx;    // decode: [B]
    float *S;              // [rows, ldS]
    int64_t ldS;
    int B, L, H_I, m, ncap, idx_t;
    int b, t0, nrows;      // prefill: sequence and row range of this launch
    int decode;
};

struct TopkArgs {
    const float *S;
    const uint32_t *hist;  // decode: [rows][2048] histogram of the rows' top 11 key bits, or NULL
    int64_t ldS;
    const int32_t *ctx;    // decode positions (ctx-1) or NULL for prefill
    int32_t *out;          // prefill: out + ((b*L)+t)*k; decode: out + b*k
    int L, m, ncap, k;
    int b, t0, nrows;
    int decode;
};

struct AttnArgs {
    const void *q;         // prefill [B, L, H, d]; decode [B, H, d]
    const void *kv_rope;   // prefill [B, L, d]; decode ring [B, n_win, d]
    const void *c_data;    // entries
    const void *c_rope;
    const float *c_scale;
    const int32_t *idx;    // CSA: [B, L, k] / [B, k]; HCA: NULL
    const int32_t *ctx;    // decode: [B]
    const float *sink;     // [H] or NULL
    const float *rope_tab; // [rope_len, half, 2]
    void *out;
    float *lse;
    void *ws;              // prefill with MIXED / NVFP4 entries: room for the entries widened to BF16
    size_t ws_bytes;
    int B, L, H, m, topk, n_win, d_rope, ncap;
    float scale;
    int decode, act_t, kv_t;
    int win_t;             // decode ring: act_t rows, or FP8 rows of 144 bytes (CSA_FP8E4M3)
    int dense;             // 1: the key list is every visible entry in order (HCA decode), no idx
    // split-KV decode (0 = off): S work items per sequence, T key tiles per item; partial results
    // in part_o [B*S, H, 128] float and part_ml [B*S, H] (max, sum), merged by the combine step
    int split_S, split_T;
    float *part_o;
    float2 *part_ml;
};

// FP8 prefill indexer with the top-k selection fused in (index_select.cu).
constexpr int kIselSeg = 256;          // candidates kept per query row and filter warp
constexpr int kIselCap = 16 * kIselSeg; // candidates kept per query row (16 filter warps)
constexpr int kIselSampleStride = 16;  // the threshold sample holds every 16th entry tile
struct IselArgs {
    const void *qI;        // FP8 codes [B, L, H_I, d_I]
    const float *qI_scale; // [B, L, H_I]
    const void *KI;        // FP8 codes [B, ncap, d_I]
    const float *KI_scale; // [B, ncap]
    const float *w;        // [B, L, H_I]
    int32_t *out;          // [B, L, k]
    void *ws;              // isel_workspace_bytes(L, ncap) bytes, 256-byte aligned
    int B, L, H_I, m, ncap, k;
};
size_t isel_workspace_bytes(int L, int ncap);
int64_t isel_chunk_rows(int L, int ncap);
bool isel_supported(const IselArgs &a);
int launch_index_select(const IselArgs &a, cudaStream_t st);  // returns a csa_status

// Incremental decode state (append.cu): one new token per sequence into the window ring, the
// state cache of the last 2m raw tokens and, when it completes a block, the compressed caches.
struct AppendArgs {
    const void *kv_new;    // [B, d] act_t, before RoPE
    const float *z_new;    // [B, 2]
    const float *kI_new;   // [B, d_I] or NULL
    const int32_t *ctx;    // [B]: tokens including the new one
    const float *rope_tab;
    void *ring;            // [B, n_win, d] act_t, or [B, n_win, 144] bytes of FP8 rows (win_t)
    void *state_kv;        // [B, 2m, d] act_t
    float *state_z;        // [B, 2m, 2]
    float *state_kI;       // [B, 2m, d_I]
    void *c_data;
    __nv_bfloat16 *c_rope;
    float *c_scale;
    void *ki_data;
    float *ki_scale;
    uint8_t *ki_e8;
    int B, L, m, ncap, n_win, d_rope, act_t, kv_t, idx_t, win_t;
};
void launch_kv_append(const AppendArgs &a, cudaStream_t st);

// BF16 GEMM for the projections around the core (gemm.cu): C = A B^T, output columns split into
// up to four segments (csa_gemm_out), optionally block-diagonal over `groups`.
using GemmOut = csa_gemm_out;
struct GemmArgs {
    const void *A;
    int64_t lda;
    const void *B;
    int64_t ldb;
    int M, N, K, groups;
    GemmOut out[4];
    int n_out;
};
int launch_gemm_bf16(const GemmArgs &a, cudaStream_t st);  // returns a csa_status

// host-side count of kernel launches (every launch_* adds the kernels it launched)
void count_launches(int n);
uint64_t launch_counter();

void launch_status_reset(cudaStream_t st);
void launch_probe_ffma(int blocks, int iters, float *out, cudaStream_t st);
void launch_probe_read(const void *buf, int64_t bytes, int reps, int blocks, float *out, cudaStream_t st);
void launch_wait_selftest(uint64_t limit_ns, cudaStream_t st);
void launch_rope_table(float *tab, int rope_len, int d_rope, float theta, cudaStream_t st);
void launch_quant_rows(const float *x, int64_t rows, int cols, uint8_t *codes, float *scales,
                       cudaStream_t st);
// MXFP4 rows of 64 values (fp4.cu): quantisation, and the exact FP8 form (codes + row scale)
void launch_quant_mxfp4(const float *x, int64_t rows, uint8_t *codes, uint8_t *e8, cudaStream_t st);
void launch_mxfp4_to_fp8(const uint8_t *codes, const uint8_t *e8, int64_t rows, uint8_t *out, float *out_scale,
                         cudaStream_t st);
// NVFP4 entry rows (80 bytes) and FP8 window rows (144 bytes) of 128-dim float rows (fp4.cu)
void launch_quant_nvfp4_entries(const float *x, int64_t rows, uint8_t *out, cudaStream_t st);
void launch_quant_fp8_window(const float *x, int64_t rows, uint8_t *out, cudaStream_t st);
void launch_kv_compress(const CompressArgs &a, cudaStream_t st);
void launch_indexer(const IndexArgs &a, cudaStream_t st);
void launch_topk(const TopkArgs &a, cudaStream_t st);
// decode top-k from the scan's key histogram: a collect launch over slices of every row and a
// finishing launch per row (topk.cu). cnt [B][2] must be zero before the launch.
struct DecSelArgs {
    const float *S;
    int64_t ldS;
    const uint32_t *hist;  // [B][2048]
    const int32_t *ctx;
    int32_t *out;          // [B][k]
    int *cnt;              // [B][2]: keys above the threshold bin, keys in it
    int32_t *above;        // [B][k]
    uint2 *bin;            // [B][4096] (key, index)
    int L, m, ncap, k, B;
    int slices;            // collecting CTAs per row (set by the launcher)
};
size_t decode_select_bytes(int B, int k);
size_t decode_select_above_off(int B);
size_t decode_select_bin_off(int B, int k);
void launch_decode_select(const DecSelArgs &a, cudaStream_t st);
// decode indexer scan on the tensor cores (FP8, H_I in {4, 8, 16}, B * H_I >= 16): scores into
// a.S and the per-row key histogram into hist [B][2048] (zeroed before the launch); false when
// the layer is outside what it handles (launching nothing)
bool decode_index_tc_supported(const IndexArgs &a);
bool launch_decode_index_tc(const IndexArgs &a, uint32_t *hist, cudaStream_t st);
// the same scan for MXFP4 operands read as stored (packed E2M1 + E8M0), on the CUDA cores
bool decode_index_fp4_supported(const IndexArgs &a);
bool launch_decode_index_fp4(const IndexArgs &a, uint32_t *hist, cudaStream_t st);
void launch_attn_simple(const AttnArgs &a, cudaStream_t st);
// tensor-core kernels: return false (launching nothing) when the configuration is outside
// what they handle
bool launch_hca_tc(const AttnArgs &a, cudaStream_t st);
bool launch_csa_tc(const AttnArgs &a, cudaStream_t st);
// MIXED or NVFP4 entries (prefill) widened to BF16 rows [B, ncap, 128] in a.ws (csa_widen_bytes
// bytes); returns the widened array.
size_t csa_widen_bytes(const AttnArgs &a);
// split-KV decode plan (items per sequence S, tiles per item T), partial-result bytes, combine
void decode_split_plan(int B, int topk, int ncap, int dense, int *S, int *T);
size_t decode_partial_bytes(int B, int S);
void launch_decode_combine(const AttnArgs &a, cudaStream_t st);
const void *launch_widen_entries(const AttnArgs &a, cudaStream_t st);

}  // namespace csa
