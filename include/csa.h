/*
 * csa.h -- C ABI of the hybrid compressed attention library (libcsa.so, CUDA sm_103a).
 *
 * The library computes the attention layer of DeepSeek-V4's hybrid compressed attention:
 * Compressed Sparse Attention (CSA) and Heavily Compressed Attention (HCA).
 *
 * Sources (prose only; the pages print no formula):
 *  [P2] "DeepSeek-V4: Towards Highly Efficient Million-Token Context Intelligence"
 *       (wiki notes): 提案手法 §1 "ハイブリッドアテンション (CSA + HCA)";
 *       訓練インフラの革新 §5 "推論フレームワーク" (state cache + compressed KV cache,
 *       KV entries with BF16 RoPE dims and FP8 other dims).
 *  [P4] "EP 95 DeepSeek-V4論文を読む" (podcast), segment 17:10 (indexer and top-k).
 *  [P5] "deepseek V4 技术论文", 一.1 "混合注意力机制：CSA + HCA".
 *
 * Conventions for every call
 *  - All tensor pointers are DEVICE pointers owned by the caller, row-major and
 *    contiguous, 16-byte aligned. The library allocates nothing: scratch memory comes from
 *    the caller's workspace, sized by csa_workspace_bytes().
 *  - Every call is asynchronous on `stream` and returns a csa_status. Shapes, dtypes, null
 *    pointers, alignment and the workspace size are checked on the host before anything is
 *    launched; a failed check returns CSA_ERR_INVALID / CSA_ERR_WORKSPACE / CSA_ERR_UNSUPPORTED
 *    and launches nothing. No C++ exception crosses the ABI.
 *  - Device-side conditions (an index out of range that was skipped, a bounded wait that gave
 *    up) are recorded in a device status word, read with csa_device_status().
 *  - Fixed sizes: head dim d = 128, indexer dim d_I = 64, d_rope in {0, 64}.
 *  - Positions: in prefill, the query of row t of a sequence has position t. In decode, the
 *    caller has already appended the new token: ctx_len[b] counts it and its position is
 *    p = ctx_len[b] - 1.
 */
#ifndef CSA_H
#define CSA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *csa_stream_t; /* a cudaStream_t; NULL = the legacy default stream */

/* Element types. */
typedef enum {
    CSA_F32 = 0,     /* float32 */
    CSA_BF16 = 1,    /* bfloat16 */
    CSA_FP8E4M3 = 2, /* FP8 E4M3 ("fn": no infinities, max 448), with a float scale per row */
    CSA_MIXED = 3,   /* compressed entry: dims [0, d-d_rope) FP8 E4M3 + row scale, RoPE dims BF16 */
    CSA_MXFP4 = 4,   /* indexer operand rows in MXFP4: E2M1 elements, one E8M0 exponent per 32 */
    CSA_NVFP4 = 5    /* compressed entry in NVFP4: E2M1 elements, one E4M3 scale per 16, a float
                        scale per entry (an 80-byte row, layout at csa_entries) */
} csa_dtype;

typedef enum {
    CSA_OK = 0,
    CSA_ERR_INVALID = 1,     /* bad shape, dtype, null pointer or misaligned pointer */
    CSA_ERR_WORKSPACE = 2,   /* workspace smaller than csa_workspace_bytes() */
    CSA_ERR_UNSUPPORTED = 3, /* well-formed but not provided (e.g. d != 128) */
    CSA_ERR_LAUNCH = 4,      /* a kernel launch failed */
    CSA_ERR_TIMEOUT = 5,     /* device: a bounded wait gave up (kernel returned early) */
    CSA_ERR_BOUNDS = 6,      /* device: an out-of-range index was skipped */
    CSA_ERR_CUDA = 7         /* another CUDA runtime error */
} csa_status;

/* Layer description shared by all calls. */
typedef struct {
    int B;          /* sequences */
    int L;          /* prefill: tokens per sequence; decode: cache capacity in raw tokens */
    int H;          /* query heads (all share one KV head) */
    int d;          /* head dim; must be 128 */
    int d_rope;     /* RoPE dims, the last d_rope of d: 64, or 0 for no RoPE */
    int m;          /* compression ratio of this layer: m = 4 (CSA) or m' = 128 (HCA) */
    int topk;       /* CSA: entries selected per query (0 disables the compressed branch) */
    int n_win;      /* sliding-window length (128) */
    int H_I;        /* CSA indexer heads */
    int d_I;        /* CSA indexer dim; must be 64 */
    float scale;    /* softmax scale of the logits (1/sqrt(d)) */
    int act_t;      /* csa_dtype of q, raw kv, kv_rope and the output: F32 | BF16 */
    int kv_t;       /* csa_dtype of compressed entries: F32 | BF16 | MIXED | NVFP4 (BF16 act_t) */
    int idx_t;      /* csa_dtype of the indexer operands: F32 | FP8E4M3 | MXFP4 */
    int rope_len;   /* rows of the RoPE table (positions 0 .. rope_len-1) */
    int win_t;      /* csa_dtype of the decode SWA ring: act_t, or FP8E4M3 with BF16 act_t (the
                       ring's rows then are 144-byte FP8 rows, layout at csa_decode) */
} csa_params;

/* Compressed entries of B sequences, N_cap = ceil(L / m) rows per sequence.
 *  F32 / BF16: data = [B, N_cap, d];  rope = scale = NULL.
 *  MIXED     : data = [B, N_cap, d - d_rope] FP8 E4M3 codes, rope = [B, N_cap, d_rope] BF16,
 *              scale = [B, N_cap] float; value = decode(code) * scale on the first dims.
 *  NVFP4     : data = [B, N_cap, 80] bytes, one row per entry; rope = scale = NULL. Row: bytes
 *              [0, 64) E2M1 codes (dim 2i in the low nibble of byte i), [64, 72) one E4M3 scale
 *              code per block of 16 dims, [72, 76) the float entry scale s = max|c| / (6 * 448),
 *              [76, 80) zero. Block b: scale_b = E4M3(code_b) * s (float product); dim value =
 *              E2M1 * scale_b. Quantised after RoPE. ([P3] "Технический отчёт DeepSeek-V4.1-Flash
 *              — часть 2/2": the V4.1 KV cache in NVFP4, quantised after RoPE; the block of 16
 *              with an E4M3 scale is the NVFP4 format, the float scale per entry is this
 *              library's reading of its second-level scale.)
 * Entries hold RoPE already applied at the entry position (j+1)m - 1. */
typedef struct {
    void *data;
    void *rope;
    float *scale;
} csa_entries;

/* Rows of indexer operands (queries [.., H_I, d_I] or keys [.., d_I]).
 *  F32     : data = float rows, scale = NULL.
 *  FP8E4M3 : data = uint8 E4M3 codes, scale = one float per row of d_I values.
 *  MXFP4   : data = uint8 [.., d_I / 2] E2M1 codes (element 2i in the low nibble of byte i),
 *            mx_scale = uint8 [.., d_I / 32] E8M0 exponents (one per block of 32 elements:
 *            value = E2M1 * 2^(e8 - 127)); scale = NULL. ([P2] 事後学習 §3: the indexer's QK
 *            path in FP4 (MXFP4); FP4 -> FP8 dequantisation is lossless, so the library runs
 *            the FP8 indexer on the exact FP8 form of these rows.) */
typedef struct {
    void *data;
    float *scale;
    uint8_t *mx_scale;
} csa_index_rows;

/* Operation selector for csa_workspace_bytes. */
typedef enum {
    CSA_OP_INDEX_TOPK = 0,
    CSA_OP_CSA_PREFILL = 1,
    CSA_OP_HCA_PREFILL = 2,
    CSA_OP_CSA_DECODE = 3,
    CSA_OP_HCA_DECODE = 4,
    CSA_OP_SPARSE_ATTENTION = 5
} csa_op;

/* Human-readable text of a status code (static storage). */
const char *csa_strerror(int status);

/* Library ABI version (major * 100 + minor). */
int csa_version(void);

/* Bytes of caller workspace the operation needs for this layer; 0 if none. (size_t)-1 when
 * the parameters are invalid. Pure host function. */
size_t csa_workspace_bytes(const csa_params *p, int op);

/* Host-only validation of a layer description; returns CSA_OK or CSA_ERR_INVALID /
 * CSA_ERR_UNSUPPORTED without touching the GPU. `op` as in csa_workspace_bytes. */
int csa_check_params(const csa_params *p, int op);

/* RoPE table for partial RoPE ([P2] 提案手法 §1, last bullet: RoPE on the last 64 dims).
 * tab [rope_len, d_rope/2, 2] float receives (cos, sin) of pos * theta^(-i/(d_rope/2)),
 * evaluated in double precision on the device and rounded to float. */
int csa_rope_table(float *tab, int rope_len, int d_rope, float theta, csa_stream_t stream);

/* Per-row FP8 E4M3 quantisation of x [rows, cols] float (the indexer's low-precision
 * operands, [P2] 提案手法 §1 CSA): scale[r] = max|x[r,:]| / 448 (float), codes[r,c] =
 * E4M3(x[r,c] / scale[r]) rounded to nearest even with saturation to +-448; a zero row gets
 * scale 0 and zero codes. codes [rows, cols] uint8; scales [rows] float. */
int csa_quant_fp8_rows(const float *x, int64_t rows, int cols, uint8_t *codes, float *scales,
                       csa_stream_t stream);

/* NVFP4 entry rows (layout at csa_entries) of x [rows, 128] float: s = max|x[r,:]| / (6 * 448)
 * (float division), block code_b = E4M3(max_b / (6 s)) (E4M3 rounded to nearest even,
 * saturated), scale_b = E4M3(code_b) * s, element = E2M1(x / scale_b) rounded to nearest even
 * and saturated at 6 (0 when scale_b is 0). out [rows, 80] bytes, 16-byte aligned. Used to
 * build an entry cache from rows that already hold RoPE (the library's own compression writes
 * NVFP4 entries itself). */
int csa_quant_nvfp4_entries(const float *x, int64_t rows, uint8_t *out, csa_stream_t stream);

/* FP8 SWA-ring rows of x [rows, 128] float (RoPE already applied): bytes [0, 128) E4M3 codes
 * E4M3(x / s) with s = max|x[r,:]| / 448, bytes [128, 132) the float s, [132, 144) zero; a zero
 * row gets s = 0 and zero codes. out [rows, 144] bytes, 16-byte aligned. ([P3]: the V4.1
 * sliding-window KV cache in FP8.) Used for the prefill -> decode hand-over of the ring;
 * kv_append writes ring rows in this form itself when win_t = FP8E4M3. */
int csa_quant_fp8_window_rows(const float *x, int64_t rows, uint8_t *out, csa_stream_t stream);

/* Per-row MXFP4 quantisation of x [rows, 64] float (the indexer's FP4 operands, [P2] 事後学習
 * §3): per block of 32 values, e = floor(log2(max |x|)) - 2 clamped to [-127, 127] (a block of
 * zeros: e = -127), E8M0 byte e + 127, codes = E2M1(x / 2^e) rounded to nearest even and
 * saturated at 6. codes [rows, 32] uint8 (two elements per byte, the even one in the low
 * nibble); e8 [rows, 2] uint8. cols must be 64. */
int csa_quant_mxfp4_rows(const float *x, int64_t rows, int cols, uint8_t *codes, uint8_t *e8,
                         csa_stream_t stream);

/* Overlapping compression, one layer ([P2] 提案手法 §1 CSA/HCA: one entry per m tokens by a
 * weighted average with overlap between adjacent blocks; [P5] 一.1: C^b overlaps C^a).
 * Entry j of a sequence = sum over t in [(j-1)m, (j+1)m) ∩ [0, L) of alpha_t * kv[t], with
 * alpha = softmax over those tokens of z[t,0] (t in block j) or z[t,1] (t in block j-1).
 * Then RoPE at position (j+1)m - 1, then storage per p->kv_t. The same weights compress the
 * raw indexer keys (if kI_raw is given) into KI, stored per p->idx_t (FP8: one scale per
 * entry). Optionally writes kv_rope: the raw rows with RoPE at their own positions (the
 * sliding-window keys), in p->act_t.
 *   kv [B, L, d] act_t;  z [B, L, 2] float;  kI_raw [B, L, d_I] float or NULL;
 *   rope_tab: csa_rope_table with rope_len >= ceil(L/m) * m;
 *   C: entries [B, ceil(L/m), ...];  KI: [B, ceil(L/m), d_I] (ignored if kI_raw is NULL);
 *   kv_rope [B, L, d] act_t or NULL. kv, kI_raw, kv_rope and rope_tab must be 16-byte aligned
 *   (they are read and written in 16-byte chunks); otherwise CSA_ERR_INVALID. */
int kv_compress(const csa_params *p, const void *kv, const float *z, const float *kI_raw,
                const float *rope_tab, const csa_entries *C, const csa_index_rows *KI,
                void *kv_rope, csa_stream_t stream);

/* Incremental decode state ([P2] 訓練インフラの革新 §5: a heterogeneous inference cache -- a
 * state cache of the recent raw tokens, where the incomplete block waits, and the compressed
 * KV cache; 提案手法 §1: overlapping compression, sliding window, partial RoPE). Appends the
 * new token of each sequence, at position u = ctx_len[b] - 1:
 *  - ring[b][u mod n_win] = its raw row rotated by RoPE at u (the sliding-window keys that
 *    csa_decode / hca_decode read);
 *  - state_kv[b][u mod 2m] = its raw row, state_z[b][u mod 2m] = z, state_kI[b][u mod 2m] = its
 *    raw indexer key (when kI_new is given): the last 2m raw tokens, the window of the next entry;
 *  - when u completes block j = u / m (that is, (u + 1) % m == 0): entry j, computed from the
 *    state as kv_compress computes it (softmax weights over rows [(j-1)m, (j+1)m) with z[.,0]
 *    in block j and z[.,1] in block j-1, RoPE at (j+1)m - 1), is written to C per kv_t, and KI_j
 *    (the same weights over the indexer keys) to KI per idx_t. Entries of incomplete blocks are
 *    not written (no decode query sees them).
 * A prefill of L0 tokens hands over to decode with: C and KI from kv_compress, ring slots filled
 * from kv_rope (the last n_win rows; through csa_quant_fp8_window_rows for an FP8 ring), and the
 * state from the last 2m raw rows of kv, z and kI.
 *   kv_new [B, d] act_t (before RoPE); z_new [B, 2] float; kI_new [B, d_I] float or NULL;
 *   ctx_len [B] int32 (device; counts the new token; 1 <= ctx_len <= L, the cache capacity);
 *   ring [B, n_win, d] act_t, or FP8 rows [B, n_win, 144] bytes when win_t = FP8E4M3 (the row
 *   quantised as csa_quant_fp8_window_rows does); state_kv [B, 2m, d] act_t; state_z [B, 2m, 2] float;
 *   state_kI [B, 2m, d_I] float (NULL when kI_new is NULL); C, KI: caches [B, ceil(L/m), ...].
 * A position outside [0, L) is skipped and recorded as CSA_ERR_BOUNDS. */
int kv_append(const csa_params *p, const void *kv_new, const float *z_new, const float *kI_new,
              const int32_t *ctx_len, const float *rope_tab, void *ring, void *state_kv, float *state_z,
              float *state_kI, const csa_entries *C, const csa_index_rows *KI, csa_stream_t stream);

/* Lightning-indexer score and top-k selection for prefill rows ([P2] 提案手法 §1 CSA;
 * [P5] 一.1: each query attends only to its top-k compressed entries; [P4] 17:10).
 * s(t, j) = sum_h w[t,h] * ReLU(qI[t,h] . KI[j]) over the entries visible to t
 * ((j+1)m - 1 <= t). F32: fixed order -- acc = fma(q_c, k_c, acc) over c from +0,
 * r = acc > 0 ? acc : 0, s = fma(w_h, r, s) over h from +0 -- so the selection is exactly
 * reproducible. FP8: E4M3 operands with row scales, products accumulated in float.
 * Selection: the k highest scores, ties to the lower index; written in ascending index
 * order, padded with -1 when fewer than k entries are visible.
 *   qI rows [B, L, H_I, d_I] (FP8 scale [B, L, H_I]); KI rows [B, N, d_I] (scale [B, N]);
 *   w [B, L, H_I] float; topk_out [B, L, topk] int32. */
int csa_index_topk(const csa_params *p, const csa_index_rows *qI, const csa_index_rows *KI,
                   const float *w, int32_t *topk_out, void *ws, size_t ws_bytes,
                   csa_stream_t stream);

/* CSA prefill ([P2] 提案手法 §1 CSA + sliding window + sink + partial RoPE; [P5] 一.1).
 * Per query row t and head h: one softmax over (a) the top-k entries of t (indexer as in
 * csa_index_topk), (b) the raw rows u in [max(0, t - n_win + 1), t] (kv_rope), and (c) the
 * sink logit sink[h] (denominator only). Logits = scale * RoPE(q[t,h], t) . key; a key is
 * also its value. The output is the weighted sum with dims [d-d_rope, d) rotated back by
 * the inverse RoPE at t.
 *   q [B, L, H, d] act_t (before RoPE); kv_rope [B, L, d] act_t; C entries [B, N, ...];
 *   qI, KI, w as in csa_index_topk; sink [H] float or NULL (no sink);
 *   topk_out [B, L, topk] int32 or NULL; out [B, L, H, d] act_t;
 *   lse_out [B, L, H] float or NULL: natural log of the sum of exp(logit) over keys
 *   (sink excluded), so the weights of a head sum to exp(lse) / (exp(lse) + exp(sink)). */
int csa_prefill(const csa_params *p, const void *q, const void *kv_rope, const csa_entries *C,
                const csa_index_rows *qI, const csa_index_rows *KI, const float *w,
                const float *sink, const float *rope_tab, int32_t *topk_out, void *out,
                float *lse_out, void *ws, size_t ws_bytes, csa_stream_t stream);

/* The attention stage of csa_prefill with the selection given by the caller: topk_idx
 * [B, L, topk] int32 as written by csa_index_topk (ascending, -1 padded). Everything else as
 * in csa_prefill. Workspace: csa_workspace_bytes(p, CSA_OP_SPARSE_ATTENTION) bytes (non-zero
 * only for mixed-precision entries, which are widened to BF16 once per call); ws may be NULL
 * when that is 0. */
int csa_sparse_attention(const csa_params *p, const void *q, const void *kv_rope,
                         const csa_entries *C, const int32_t *topk_idx, const float *sink,
                         const float *rope_tab, void *out, float *lse_out, void *ws,
                         size_t ws_bytes, csa_stream_t stream);

/* HCA prefill ([P2] 提案手法 §1 HCA: m' = 128, no sparse selection, dense attention over the
 * compressed entries; plus sliding window and sink as for CSA). Key set of row t: every
 * entry visible to t, then the raw rows of the window. Arguments as in csa_prefill. */
int hca_prefill(const csa_params *p, const void *q, const void *kv_rope, const csa_entries *C,
                const float *sink, const float *rope_tab, void *out, float *lse_out, void *ws,
                size_t ws_bytes, csa_stream_t stream);

/* CSA decode step, one new query per sequence against the caches ([P2] 訓練インフラの革新
 * §5: state cache of recent raw tokens + compressed KV cache).
 *   q [B, H, d] act_t (before RoPE); ctx_len [B] int32 (device), 1 <= ctx_len[b] <= L;
 *   C: entry cache [B, ceil(L/m), ...] (entries j < ctx_len/m are read);
 *   qI rows [B, H_I, d_I] (+scale [B, H_I]); KI cache rows [B, ceil(L/m), d_I] (+scale);
 *   w [B, H_I]; swa_ring [B, n_win, d] act_t (win_t = act_t) or [B, n_win, 144] bytes of FP8
 *   rows (win_t = FP8E4M3; row layout at csa_quant_fp8_window_rows): the raw row of position
 *   u, after RoPE at u, at slot u mod n_win, for u in [max(0, p - n_win + 1), p];
 *   topk_out [B, topk] or NULL; out [B, H, d]; lse_out [B, H] or NULL. */
int csa_decode(const csa_params *p, const void *q, const int32_t *ctx_len, const csa_entries *C,
               const csa_index_rows *qI, const csa_index_rows *KI, const float *w,
               const void *swa_ring, const float *sink, const float *rope_tab,
               int32_t *topk_out, void *out, float *lse_out, void *ws, size_t ws_bytes,
               csa_stream_t stream);

/* csa_decode for callers that cannot allocate device memory. Examples: a host application
 * whose device memory is owned by another framework's allocator, which hands out no scratch
 * buffers; a real-time serving loop that must not call cudaMalloc, because it can synchronise
 * the device and take unbounded time; a caller held to a fixed device-memory budget. This
 * entry point has no counterpart in the paper; it exists only for such callers.
 * It computes exactly what csa_decode computes, with the same arguments minus the workspace:
 * the scratch it needs (indexer scores, selected indices and the split-KV partial results)
 * comes from one fixed array of
 * CSA_STATIC_SCRATCH_BYTES inside the library, which every GPU that loads the library holds
 * until the process exits. It allocates nothing.
 *  - A layer whose scratch (csa_workspace_bytes(p, CSA_OP_CSA_DECODE)) exceeds the array is
 *    refused with CSA_ERR_WORKSPACE before anything is launched; use csa_decode for it.
 *  - The first call made on a device looks up the array's device address for that device
 *    (cudaGetSymbolAddress, with the device current); make that first call before any stream
 *    capture begins.
 *  - All calls on a device share the array: calls that overlap on the GPU (unordered streams)
 *    race on it. Nothing in it needs to start at zero: each call writes the scores and indices
 *    before it reads them. */
#define CSA_STATIC_SCRATCH_BYTES (8u << 20)
int csa_decode_static_scratch(const csa_params *p, const void *q, const int32_t *ctx_len,
                              const csa_entries *C, const csa_index_rows *qI,
                              const csa_index_rows *KI, const float *w, const void *swa_ring,
                              const float *sink, const float *rope_tab, int32_t *topk_out,
                              void *out, float *lse_out, csa_stream_t stream);

/* HCA decode step ([P2] 提案手法 §1 HCA: m' = 128, dense attention over every compressed entry,
 * plus the sliding window and sink; 訓練インフラの革新 §5: state cache of recent raw tokens +
 * compressed KV cache). Key set of the new token at p = ctx_len[b] - 1: every cached entry j with
 * (j+1)m - 1 <= p, in order, then the window rows of the ring. Arguments as csa_decode (no
 * indexer operands, no workspace: ws may be NULL). */
int hca_decode(const csa_params *p, const void *q, const int32_t *ctx_len, const csa_entries *C,
               const void *swa_ring, const float *sink, const float *rope_tab, void *out,
               float *lse_out, void *ws, size_t ws_bytes, csa_stream_t stream);

/* The projections on either side of the attention core ([P2] 概要: V4-Flash hidden size 4096;
 * 提案手法 §1 CSA: shared-KV multi-query attention with a grouped output projection; [P5] 一.1
 * 共享KV MQA与分组输出投影), as one BF16 GEMM on the tensor cores with FP32 accumulation:
 *   C[M, N] = A[M, K] B[N, K]^T, A and B row-major BF16 with row strides lda, ldb (elements,
 *   multiples of 8), K a multiple of 64.
 *   groups > 1: the block-diagonal (grouped) product -- output columns [g N/groups, (g+1)
 *   N/groups) read A's columns [g K, (g+1) K), so A has groups * K columns and B stacks the
 *   groups' [N/groups, K] matrices; N/groups must be a multiple of 256.
 * The output columns go to up to four segments: segment s receives columns [col0, col1) into a
 * row-major tensor `ptr` (row stride ld elements, dtype CSA_BF16 or CSA_F32, column col0 at
 * offset 0), so that one product can write several separate tensors (q, kv, the indexer
 * inputs). Device pointers; asynchronous on stream. */
typedef struct {
    void *ptr;
    int64_t ld;
    int col0, col1;
    int dtype;
} csa_gemm_out;
int csa_gemm_bf16(const void *A, int64_t lda, const void *B, int64_t ldb, int M, int N, int K, int groups,
                  const csa_gemm_out *outs, int n_outs, csa_stream_t stream);

/* Number of kernels this library has launched in the process so far (host counter). */
uint64_t csa_launch_count(void);

/* Waits for the work queued on `stream`, then returns the device status word in *status:
 * CSA_OK or the first device-side code recorded since the last reset (CSA_ERR_TIMEOUT: a bounded
 * wait gave up and the kernel returned early, so its outputs are incomplete; CSA_ERR_BOUNDS: an
 * out-of-range index or decode position was skipped). The word is shared by every stream of the
 * device; it is cleared, together with the abort flag that makes every later bounded wait give
 * up at once, when reset != 0 (a stream-ordered reset on `stream`). A timeout therefore stays
 * visible, and keeps later kernels from waiting, until the caller resets it. */
int csa_device_status(int *status, int reset, csa_stream_t stream);

/* Diagnostic, no counterpart on the pages: launches one CTA that waits on an mbarrier that
 * never receives its arrival, through the same bounded wait the library's kernels use, with a
 * limit of limit_ns nanoseconds (1 .. 1e9). The wait gives up, records CSA_ERR_TIMEOUT in the
 * device status word and raises the abort flag, which csa_device_status(reset = 1) clears.
 * It exists so that the error path of a stalled pipeline can be exercised without a fault. */
int csa_selftest_wait_timeout(uint64_t limit_ns, csa_stream_t stream);

/* Measurement kernels, no counterpart on the pages: roofline denominators for the library's
 * kernels, timed by the caller with CUDA events on `stream`.
 * csa_probe_ffma: `blocks` CTAs of 256 threads, each thread 16 independent FP32 FMA chains of
 *   `iters` steps (32 * iters FLOP per thread); out [blocks * 256] float receives the results.
 * csa_probe_read: `blocks` CTAs of 512 threads read the device buffer buf (`bytes`, a multiple
 *   of 16, 16-byte aligned) `reps` times with 16-byte loads that may hit L2 (smaller than L2:
 *   the L2 read bandwidth; larger: HBM); out [blocks] float (zeroed by the caller) receives one
 *   sum per CTA. */
int csa_probe_ffma(int blocks, int iters, float *out, csa_stream_t stream);
int csa_probe_read(const void *buf, int64_t bytes, int reps, int blocks, float *out, csa_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* CSA_H */
