// api.cu -- the C ABI of libcsa.so: host-side validation, workspace carving and launches.
// Declarations and argument contracts are in include/csa.h.
#include <math.h>
#include <string.h>

#include <atomic>

#include "common.cuh"
#include "kernels.cuh"

namespace csa {
__device__ int g_status = 0;
__device__ int g_abort = 0;
static std::atomic<uint64_t> g_launches{0};
void count_launches(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }
uint64_t launch_counter() { return g_launches.load(std::memory_order_relaxed); }
}

using namespace csa;

namespace {

constexpr size_t kScoreBudget = (size_t)1 << 31;  // bytes of indexer scores per chunk
constexpr size_t kAlign = 256;

inline size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

inline bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

inline int64_t ncap_of(const csa_params *p) { return ceil_div64(p->L, p->m); }

// Stride of a score row in floats (kept a multiple of 4 so rows stay 16-byte aligned).
inline int64_t score_ld(const csa_params *p) { return (ncap_of(p) + 3) / 4 * 4; }

// Prefill rows whose scores share one workspace chunk.
inline int64_t score_chunk_rows(const csa_params *p) {
    int64_t rows = (int64_t)(kScoreBudget / (sizeof(float) * (size_t)score_ld(p)));
    if (rows >= p->L) return p->L;
    rows = rows / 32 * 32;
    return rows < 32 ? 32 : rows;
}

bool is_csa(int op) {
    return op == CSA_OP_INDEX_TOPK || op == CSA_OP_CSA_PREFILL || op == CSA_OP_CSA_DECODE ||
           op == CSA_OP_SPARSE_ATTENTION;
}
bool is_decode(int op) { return op == CSA_OP_CSA_DECODE || op == CSA_OP_HCA_DECODE; }

int check(const csa_params *p, int op) {
    if (!p) return CSA_ERR_INVALID;
    if (op < CSA_OP_INDEX_TOPK || op > CSA_OP_SPARSE_ATTENTION) return CSA_ERR_INVALID;
    if (p->B < 1 || p->L < 1 || p->H < 1 || p->m < 1 || p->n_win < 1) return CSA_ERR_INVALID;
    if (!(p->scale > 0.0f) || !isfinite(p->scale)) return CSA_ERR_INVALID;
    if (p->d != kD) return CSA_ERR_UNSUPPORTED;
    if (p->d_rope != 0 && p->d_rope != 64) return CSA_ERR_UNSUPPORTED;
    if (p->H > 64) return CSA_ERR_UNSUPPORTED;
    if (p->m > 1024) return CSA_ERR_UNSUPPORTED;
    if (p->act_t != CSA_F32 && p->act_t != CSA_BF16) return CSA_ERR_INVALID;
    if (p->kv_t != CSA_F32 && p->kv_t != CSA_BF16 && p->kv_t != CSA_MIXED && p->kv_t != CSA_NVFP4)
        return CSA_ERR_INVALID;
    if (p->kv_t == CSA_MIXED && p->d_rope != 64) return CSA_ERR_INVALID;
    if (p->win_t != p->act_t && p->win_t != CSA_FP8E4M3) return CSA_ERR_INVALID;
    // the NVFP4 entries and the FP8 ring are read by the tensor-core (BF16) kernels only
    if ((p->kv_t == CSA_NVFP4 || p->win_t == CSA_FP8E4M3) && p->act_t != CSA_BF16) return CSA_ERR_UNSUPPORTED;
    if ((int64_t)p->B * p->L > ((int64_t)1 << 40)) return CSA_ERR_UNSUPPORTED;
    if (p->d_rope > 0) {
        // positions used: raw rows < L, entries at (j+1)m-1 < ceil(L/m)*m
        const int64_t need = ncap_of(p) * p->m;
        if (p->rope_len < need || p->rope_len < p->L) return CSA_ERR_INVALID;
    }
    if (is_csa(op)) {
        if (p->topk < 0 || p->topk > kMaxTopk) return CSA_ERR_UNSUPPORTED;
        if (op == CSA_OP_INDEX_TOPK && p->topk < 1) return CSA_ERR_INVALID;
        if (p->topk > 0) {
            if (p->d_I != kDI) return CSA_ERR_UNSUPPORTED;
            if (p->H_I < 1 || p->H_I > 16) return CSA_ERR_UNSUPPORTED;
            if (p->idx_t != CSA_F32 && p->idx_t != CSA_FP8E4M3 && p->idx_t != CSA_MXFP4) return CSA_ERR_INVALID;
        }
    }
    return CSA_OK;
}

// Bytes of the entries widened to BF16 (prefill with MIXED or NVFP4 entries).
size_t widen_bytes(const csa_params *p) {
    return (p->kv_t == CSA_MIXED || p->kv_t == CSA_NVFP4) ? align_up((size_t)p->B * (size_t)ncap_of(p) * kD * 2) : 0;
}

// Bytes of the exact FP8 form of `rows` MXFP4 indexer rows (codes + one float scale per row).
size_t fp8_rows_bytes(int64_t rows) {
    return align_up((size_t)rows * kDI) + align_up((size_t)rows * sizeof(float));
}

// Workspace of the prefill indexer + top-k: the FP8 path keeps per-row candidate lists (the
// fused selection), the exact FP32 path a chunk of full score rows.
size_t index_ws_bytes(const csa_params *p) {
    if (p->idx_t == CSA_MXFP4)  // the FP8 form of the query and key rows, then the FP8 path's
        return fp8_rows_bytes((int64_t)p->B * p->L * p->H_I) + fp8_rows_bytes((int64_t)p->B * ncap_of(p)) +
               align_up(isel_workspace_bytes(p->L, (int)ncap_of(p)));
    if (p->idx_t == CSA_FP8E4M3) return align_up(isel_workspace_bytes(p->L, (int)ncap_of(p)));
    return align_up(sizeof(float) * (size_t)score_chunk_rows(p) * (size_t)score_ld(p));
}

// Partial results of the split-KV decode attention (BF16 activations, the tensor-core path).
size_t decode_split_bytes(const csa_params *p, int dense) {
    if (p->act_t != CSA_BF16) return 0;
    int S = 1, T = 1;
    decode_split_plan(p->B, p->topk, (int)ncap_of(p), dense, &S, &T);
    return align_up(decode_partial_bytes(p->B, S));
}

size_t ws_bytes(const csa_params *p, int op) {
    switch (op) {
    case CSA_OP_INDEX_TOPK:
        return index_ws_bytes(p);
    case CSA_OP_CSA_PREFILL:
        if (p->topk == 0) return 0;
        return index_ws_bytes(p) + align_up(sizeof(int32_t) * (size_t)p->B * p->L * p->topk) + widen_bytes(p);
    case CSA_OP_SPARSE_ATTENTION:
        return p->topk > 0 ? widen_bytes(p) : 0;
    case CSA_OP_HCA_PREFILL:
        return widen_bytes(p);
    case CSA_OP_CSA_DECODE:
        return (p->topk > 0 && p->idx_t == CSA_MXFP4
                    ? fp8_rows_bytes((int64_t)p->B * p->H_I) + fp8_rows_bytes((int64_t)p->B * ncap_of(p))
                    : 0) +
               (p->topk == 0 ? 0
                             : align_up(sizeof(float) * (size_t)p->B * (size_t)score_ld(p)) +
                                   align_up(sizeof(int32_t) * (size_t)p->B * p->topk) +
                                   align_up(sizeof(uint32_t) * (size_t)p->B * 2048) +
                                   align_up(decode_select_bytes(p->B, p->topk))) +
               decode_split_bytes(p, 0);
    case CSA_OP_HCA_DECODE:
        return decode_split_bytes(p, 1);
    default:
        return 0;
    }
}

int launch_status() {
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? CSA_OK : CSA_ERR_LAUNCH;
}

inline cudaStream_t cs(csa_stream_t s) { return reinterpret_cast<cudaStream_t>(s); }

bool entries_ok(const csa_params *p, const csa_entries *C) {
    if (!C || !C->data || !aligned16(C->data)) return false;
    if (p->kv_t == CSA_MIXED) return C->rope && C->scale && aligned16(C->rope) && aligned16(C->scale);
    return true;
}

bool index_rows_ok(const csa_params *p, const csa_index_rows *r) {
    if (!r || !r->data || !aligned16(r->data)) return false;
    if (p->idx_t == CSA_FP8E4M3) return r->scale && aligned16(r->scale);
    if (p->idx_t == CSA_MXFP4) return r->mx_scale != nullptr;
    return true;
}

// MXFP4 rows converted to their exact FP8 form in workspace at `ws`; the FP8 rows are returned
// in `out` (data = codes, scale = row scales).
void mxfp4_rows_to_fp8(const csa_index_rows *in, int64_t rows, void *ws, csa_index_rows *out, cudaStream_t st) {
    uint8_t *codes = reinterpret_cast<uint8_t *>(ws);
    float *scales = reinterpret_cast<float *>(reinterpret_cast<char *>(ws) + align_up((size_t)rows * kDI));
    launch_mxfp4_to_fp8(reinterpret_cast<const uint8_t *>(in->data), in->mx_scale, rows, codes, scales, st);
    out->data = codes;
    out->scale = scales;
    out->mx_scale = nullptr;
}

// indexer + top-k over all prefill rows: FP8 through the fused selection, FP32 (exact, the
// bit-exact workload) chunked through a workspace of full score rows
int run_index_topk(const csa_params *p, const csa_index_rows *qI, const csa_index_rows *KI,
                   const float *w, int32_t *idx_out, float *S, cudaStream_t st) {
    const int ncap = (int)ncap_of(p);
    if (p->idx_t == CSA_MXFP4) {
        // the exact FP8 form of the FP4 rows, then the FP8 path
        const int64_t qrows = (int64_t)p->B * p->L * p->H_I, krows = (int64_t)p->B * ncap;
        char *w8 = reinterpret_cast<char *>(S);
        csa_index_rows q8{}, k8{};
        mxfp4_rows_to_fp8(qI, qrows, w8, &q8, st);
        mxfp4_rows_to_fp8(KI, krows, w8 + fp8_rows_bytes(qrows), &k8, st);
        csa_params p8 = *p;
        p8.idx_t = CSA_FP8E4M3;
        return run_index_topk(&p8, &q8, &k8, w, idx_out,
                              reinterpret_cast<float *>(w8 + fp8_rows_bytes(qrows) + fp8_rows_bytes(krows)), st);
    }
    if (p->idx_t == CSA_FP8E4M3) {
        IselArgs ia{};
        ia.qI = qI->data; ia.qI_scale = qI->scale; ia.KI = KI->data; ia.KI_scale = KI->scale; ia.w = w;
        ia.out = idx_out; ia.ws = S;
        ia.B = p->B; ia.L = p->L; ia.H_I = p->H_I; ia.m = p->m; ia.ncap = ncap; ia.k = p->topk;
        const int s = launch_index_select(ia, st);
        return s ? s : launch_status();
    }
    const int64_t chunk = score_chunk_rows(p);
    for (int b = 0; b < p->B; ++b) {
        for (int64_t t0 = 0; t0 < p->L; t0 += chunk) {
            const int nrows = (int)((p->L - t0) < chunk ? (p->L - t0) : chunk);
            IndexArgs ia{};
            ia.qI = qI->data;
            ia.qI_scale = qI->scale;
            ia.KI = KI->data;
            ia.KI_scale = KI->scale;
            ia.w = w;
            ia.S = S;
            ia.ldS = score_ld(p);
            ia.B = p->B; ia.L = p->L; ia.H_I = p->H_I; ia.m = p->m; ia.ncap = ncap;
            ia.idx_t = p->idx_t;
            ia.b = b; ia.t0 = (int)t0; ia.nrows = nrows;
            launch_indexer(ia, st);
            TopkArgs ta{};
            ta.S = S;
            ta.ldS = score_ld(p);
            ta.out = idx_out;
            ta.L = p->L; ta.m = p->m; ta.ncap = ncap; ta.k = p->topk;
            ta.b = b; ta.t0 = (int)t0; ta.nrows = nrows;
            launch_topk(ta, st);
        }
    }
    return launch_status();
}

AttnArgs attn_args(const csa_params *p, const void *q, const void *kvr, const csa_entries *C,
                   const int32_t *idx, const int32_t *ctx, const float *sink, const float *rope,
                   void *out, float *lse, int decode, int topk, void *ws = nullptr, size_t wsb = 0) {
    AttnArgs a{};
    a.ws = ws;
    a.ws_bytes = wsb;
    a.q = q;
    a.kv_rope = kvr;
    a.c_data = C ? C->data : nullptr;
    a.c_rope = C ? C->rope : nullptr;
    a.c_scale = C ? C->scale : nullptr;
    a.idx = idx;
    a.ctx = ctx;
    a.sink = sink;
    a.rope_tab = rope;
    a.out = out;
    a.lse = lse;
    a.B = p->B; a.L = p->L; a.H = p->H; a.m = p->m; a.topk = topk; a.n_win = p->n_win;
    a.d_rope = p->d_rope; a.ncap = (int)ncap_of(p); a.scale = p->scale;
    a.decode = decode; a.act_t = p->act_t; a.kv_t = p->kv_t; a.win_t = p->win_t;
    return a;
}

// Attention kernel choice (no silent second backend): FP32 activations run the CUDA-core
// kernel (the exact FP32 workload); BF16 activations run the tensor-core kernels, and a BF16
// layer those do not take is refused with CSA_ERR_UNSUPPORTED before anything is launched.
int run_csa_attention(const AttnArgs &a, cudaStream_t st) {
    if (a.act_t == CSA_F32) {
        launch_attn_simple(a, st);
        return launch_status();
    }
    if (!launch_csa_tc(a, st)) return CSA_ERR_UNSUPPORTED;
    return launch_status();
}

// Decode: BF16 runs split-KV on the tensor cores (work items over the key tiles, partial results
// in the workspace at `part`) followed by the combine step; FP32 the CUDA-core kernel.
int run_decode_attention(AttnArgs a, void *part, cudaStream_t st) {
    if (a.act_t == CSA_F32) {
        launch_attn_simple(a, st);
        return launch_status();
    }
    decode_split_plan(a.B, a.topk, a.ncap, a.dense, &a.split_S, &a.split_T);
    a.part_o = reinterpret_cast<float *>(part);
    a.part_ml = reinterpret_cast<float2 *>(reinterpret_cast<char *>(part) +
                                           (size_t)a.B * a.split_S * 64 * 128 * sizeof(float));
    if (!launch_csa_tc(a, st)) return CSA_ERR_UNSUPPORTED;
    launch_decode_combine(a, st);
    return launch_status();
}

int run_hca_attention(const AttnArgs &a, cudaStream_t st) {
    if (a.act_t == CSA_F32) {
        launch_attn_simple(a, st);
        return launch_status();
    }
    if (!launch_hca_tc(a, st)) return CSA_ERR_UNSUPPORTED;
    return launch_status();
}

}  // namespace

extern "C" {

const char *csa_strerror(int s) {
    switch (s) {
    case CSA_OK: return "ok";
    case CSA_ERR_INVALID: return "invalid argument (shape, dtype, null or misaligned pointer)";
    case CSA_ERR_WORKSPACE: return "workspace too small";
    case CSA_ERR_UNSUPPORTED: return "unsupported configuration";
    case CSA_ERR_LAUNCH: return "kernel launch failed";
    case CSA_ERR_TIMEOUT: return "device wait timed out";
    case CSA_ERR_BOUNDS: return "device index out of range (skipped)";
    case CSA_ERR_CUDA: return "CUDA runtime error";
    default: return "unknown status";
    }
}

int csa_version(void) { return 110; }

int csa_check_params(const csa_params *p, int op) { return check(p, op); }

size_t csa_workspace_bytes(const csa_params *p, int op) {
    if (check(p, op) != CSA_OK) return (size_t)-1;
    return ws_bytes(p, op);
}

int csa_rope_table(float *tab, int rope_len, int d_rope, float theta, csa_stream_t stream) {
    if (!tab || !aligned16(tab) || rope_len < 1 || (d_rope != 64 && d_rope != 0) || !(theta > 1.0f))
        return CSA_ERR_INVALID;
    if (d_rope == 0) return CSA_OK;
    launch_rope_table(tab, rope_len, d_rope, theta, cs(stream));
    return launch_status();
}

int csa_quant_mxfp4_rows(const float *x, int64_t rows, int cols, uint8_t *codes, uint8_t *e8,
                         csa_stream_t stream) {
    if (!x || !codes || !e8 || rows < 0 || cols != kDI) return CSA_ERR_INVALID;
    launch_quant_mxfp4(x, rows, codes, e8, cs(stream));
    return launch_status();
}

int csa_quant_nvfp4_entries(const float *x, int64_t rows, uint8_t *out, csa_stream_t stream) {
    if (!x || !out || rows < 0 || !aligned16(out)) return CSA_ERR_INVALID;
    launch_quant_nvfp4_entries(x, rows, out, cs(stream));
    return launch_status();
}

int csa_quant_fp8_window_rows(const float *x, int64_t rows, uint8_t *out, csa_stream_t stream) {
    if (!x || !out || rows < 0 || !aligned16(out)) return CSA_ERR_INVALID;
    launch_quant_fp8_window(x, rows, out, cs(stream));
    return launch_status();
}

int csa_quant_fp8_rows(const float *x, int64_t rows, int cols, uint8_t *codes, float *scales,
                       csa_stream_t stream) {
    if (!x || !codes || !scales || rows < 0 || cols < 1) return CSA_ERR_INVALID;
    if (rows == 0) return CSA_OK;
    launch_quant_rows(x, rows, cols, codes, scales, cs(stream));
    return launch_status();
}

int kv_compress(const csa_params *p, const void *kv, const float *z, const float *kI_raw,
                const float *rope_tab, const csa_entries *C, const csa_index_rows *KI,
                void *kv_rope, csa_stream_t stream) {
    int s = check(p, CSA_OP_HCA_PREFILL);
    if (s) return s;
    if (!kv || !z || !aligned16(kv) || !entries_ok(p, C)) return CSA_ERR_INVALID;
    if (p->d_rope > 0 && (!rope_tab || !aligned16(rope_tab))) return CSA_ERR_INVALID;
    if (kI_raw) {
        if (p->idx_t != CSA_F32 && p->idx_t != CSA_FP8E4M3 && p->idx_t != CSA_MXFP4) return CSA_ERR_INVALID;
        if (!index_rows_ok(p, KI) || p->d_I != kDI || !aligned16(kI_raw)) return CSA_ERR_INVALID;
    }
    if (kv_rope && !aligned16(kv_rope)) return CSA_ERR_INVALID;
    CompressArgs a{};
    a.kv = kv; a.z = z; a.kI_raw = kI_raw; a.rope_tab = rope_tab;
    a.c_data = C->data; a.c_rope = C->rope; a.c_scale = C->scale;
    a.ki_data = kI_raw ? KI->data : nullptr;
    a.ki_scale = kI_raw ? KI->scale : nullptr;
    a.ki_e8 = kI_raw ? KI->mx_scale : nullptr;
    a.kv_rope = kv_rope;
    a.B = p->B; a.L = p->L; a.m = p->m; a.N = (int)ncap_of(p); a.d_rope = p->d_rope;
    a.act_t = p->act_t; a.kv_t = p->kv_t; a.idx_t = p->idx_t;
    launch_kv_compress(a, cs(stream));
    return launch_status();
}

int kv_append(const csa_params *p, const void *kv_new, const float *z_new, const float *kI_new,
              const int32_t *ctx_len, const float *rope_tab, void *ring, void *state_kv, float *state_z,
              float *state_kI, const csa_entries *C, const csa_index_rows *KI, csa_stream_t stream) {
    int s = check(p, CSA_OP_HCA_DECODE);
    if (s) return s;
    if (!kv_new || !z_new || !ctx_len || !ring || !state_kv || !state_z || !entries_ok(p, C)) return CSA_ERR_INVALID;
    if (!aligned16(kv_new) || !aligned16(ring) || !aligned16(state_kv)) return CSA_ERR_INVALID;
    if (p->d_rope > 0 && !rope_tab) return CSA_ERR_INVALID;
    if (kI_new) {
        if (!state_kI || p->d_I != kDI || !index_rows_ok(p, KI)) return CSA_ERR_INVALID;
        if (p->idx_t != CSA_F32 && p->idx_t != CSA_FP8E4M3 && p->idx_t != CSA_MXFP4) return CSA_ERR_INVALID;
    }
    AppendArgs a{};
    a.kv_new = kv_new; a.z_new = z_new; a.kI_new = kI_new; a.ctx = ctx_len; a.rope_tab = rope_tab;
    a.ring = ring; a.state_kv = state_kv; a.state_z = state_z; a.state_kI = state_kI;
    a.c_data = C->data; a.c_rope = reinterpret_cast<__nv_bfloat16 *>(C->rope); a.c_scale = C->scale;
    a.ki_data = kI_new ? KI->data : nullptr; a.ki_scale = kI_new ? KI->scale : nullptr;
    a.ki_e8 = kI_new ? KI->mx_scale : nullptr;
    a.B = p->B; a.L = p->L; a.m = p->m; a.ncap = (int)ncap_of(p); a.n_win = p->n_win; a.d_rope = p->d_rope;
    a.act_t = p->act_t; a.kv_t = p->kv_t; a.idx_t = p->idx_t; a.win_t = p->win_t;
    launch_kv_append(a, cs(stream));
    return launch_status();
}

int csa_index_topk(const csa_params *p, const csa_index_rows *qI, const csa_index_rows *KI,
                   const float *w, int32_t *topk_out, void *ws, size_t wsb, csa_stream_t stream) {
    int s = check(p, CSA_OP_INDEX_TOPK);
    if (s) return s;
    if (!index_rows_ok(p, qI) || !index_rows_ok(p, KI) || !w || !topk_out) return CSA_ERR_INVALID;
    if (wsb < ws_bytes(p, CSA_OP_INDEX_TOPK) || !ws || !aligned16(ws)) return CSA_ERR_WORKSPACE;
    return run_index_topk(p, qI, KI, w, topk_out, reinterpret_cast<float *>(ws), cs(stream));
}

int csa_prefill(const csa_params *p, const void *q, const void *kv_rope, const csa_entries *C,
                const csa_index_rows *qI, const csa_index_rows *KI, const float *w,
                const float *sink, const float *rope_tab, int32_t *topk_out, void *out,
                float *lse_out, void *ws, size_t wsb, csa_stream_t stream) {
    int s = check(p, CSA_OP_CSA_PREFILL);
    if (s) return s;
    if (!q || !kv_rope || !out || !aligned16(q) || !aligned16(kv_rope) || !aligned16(out))
        return CSA_ERR_INVALID;
    if (p->d_rope > 0 && !rope_tab) return CSA_ERR_INVALID;
    if (p->topk > 0) {
        if (!entries_ok(p, C) || !index_rows_ok(p, qI) || !index_rows_ok(p, KI) || !w) return CSA_ERR_INVALID;
        if (wsb < ws_bytes(p, CSA_OP_CSA_PREFILL) || !ws || !aligned16(ws)) return CSA_ERR_WORKSPACE;
    }
    cudaStream_t st = cs(stream);
    int32_t *idx = nullptr;
    void *wide = nullptr;
    if (p->topk > 0) {
        float *S = reinterpret_cast<float *>(ws);
        const size_t sbytes = index_ws_bytes(p);
        const size_t ibytes = align_up(sizeof(int32_t) * (size_t)p->B * p->L * p->topk);
        idx = topk_out ? topk_out : reinterpret_cast<int32_t *>(reinterpret_cast<char *>(ws) + sbytes);
        wide = reinterpret_cast<char *>(ws) + sbytes + ibytes;
        s = run_index_topk(p, qI, KI, w, idx, S, st);
        if (s) return s;
    }
    AttnArgs a = attn_args(p, q, kv_rope, p->topk > 0 ? C : nullptr, idx, nullptr, sink, rope_tab, out,
                           lse_out, 0, p->topk, wide, widen_bytes(p));
    if (p->topk == 0) {
        a.ncap = 0;
        a.dense = 1;  // no compressed branch: the key list is the window alone
    }
    return run_csa_attention(a, st);
}

int csa_sparse_attention(const csa_params *p, const void *q, const void *kv_rope,
                         const csa_entries *C, const int32_t *topk_idx, const float *sink,
                         const float *rope_tab, void *out, float *lse_out, void *ws, size_t wsb,
                         csa_stream_t stream) {
    int s = check(p, CSA_OP_SPARSE_ATTENTION);
    if (s) return s;
    if (!q || !kv_rope || !out || !aligned16(q) || !aligned16(kv_rope) || !aligned16(out)) return CSA_ERR_INVALID;
    if (p->d_rope > 0 && !rope_tab) return CSA_ERR_INVALID;
    if (p->topk > 0 && (!entries_ok(p, C) || !topk_idx)) return CSA_ERR_INVALID;
    const size_t need = ws_bytes(p, CSA_OP_SPARSE_ATTENTION);
    if (need > 0 && (wsb < need || !ws || !aligned16(ws))) return CSA_ERR_WORKSPACE;
    AttnArgs a = attn_args(p, q, kv_rope, p->topk > 0 ? C : nullptr, p->topk > 0 ? topk_idx : nullptr, nullptr, sink,
                           rope_tab, out, lse_out, 0, p->topk, ws, wsb);
    if (p->topk == 0) {
        a.ncap = 0;
        a.dense = 1;
    }
    return run_csa_attention(a, cs(stream));
}

int hca_prefill(const csa_params *p, const void *q, const void *kv_rope, const csa_entries *C,
                const float *sink, const float *rope_tab, void *out, float *lse_out, void *ws,
                size_t wsb, csa_stream_t stream) {
    int s = check(p, CSA_OP_HCA_PREFILL);
    if (s) return s;
    if (!q || !kv_rope || !out || !aligned16(q) || !aligned16(kv_rope) || !aligned16(out) ||
        !entries_ok(p, C))
        return CSA_ERR_INVALID;
    if (p->d_rope > 0 && !rope_tab) return CSA_ERR_INVALID;
    const size_t need = ws_bytes(p, CSA_OP_HCA_PREFILL);
    if (need > 0 && (wsb < need || !ws || !aligned16(ws))) return CSA_ERR_WORKSPACE;
    AttnArgs a = attn_args(p, q, kv_rope, C, nullptr, nullptr, sink, rope_tab, out, lse_out, 0, 0, ws, wsb);
    return run_hca_attention(a, cs(stream));
}

int csa_decode(const csa_params *p, const void *q, const int32_t *ctx_len, const csa_entries *C,
               const csa_index_rows *qI, const csa_index_rows *KI, const float *w,
               const void *swa_ring, const float *sink, const float *rope_tab, int32_t *topk_out,
               void *out, float *lse_out, void *ws, size_t wsb, csa_stream_t stream) {
    int s = check(p, CSA_OP_CSA_DECODE);
    if (s) return s;
    if (!q || !ctx_len || !swa_ring || !out || !aligned16(q) || !aligned16(swa_ring) || !aligned16(out))
        return CSA_ERR_INVALID;
    if (p->d_rope > 0 && !rope_tab) return CSA_ERR_INVALID;
    if (p->topk > 0 && (!entries_ok(p, C) || !index_rows_ok(p, qI) || !index_rows_ok(p, KI) || !w))
        return CSA_ERR_INVALID;
    const size_t need = ws_bytes(p, CSA_OP_CSA_DECODE);
    if (need > 0 && (wsb < need || !ws || !aligned16(ws))) return CSA_ERR_WORKSPACE;
    cudaStream_t st = cs(stream);
    int32_t *idx = nullptr;
    const int ncap = (int)ncap_of(p);
    const size_t sbytes = p->topk > 0 ? align_up(sizeof(float) * (size_t)p->B * (size_t)score_ld(p)) : 0;
    const size_t ibytes = p->topk > 0 ? align_up(sizeof(int32_t) * (size_t)p->B * p->topk) : 0;
    const size_t hbytes = p->topk > 0 ? align_up(sizeof(uint32_t) * (size_t)p->B * 2048) : 0;
    const size_t dbytes = p->topk > 0 ? align_up(decode_select_bytes(p->B, p->topk)) : 0;
    char *wsc = reinterpret_cast<char *>(ws);
    uint32_t *hist = p->topk > 0 ? reinterpret_cast<uint32_t *>(wsc + sbytes + ibytes) : nullptr;
    // selection lists: the two counters per row right after the histogram (one memset clears both)
    int *sel_cnt = p->topk > 0 ? reinterpret_cast<int *>(wsc + sbytes + ibytes + hbytes) : nullptr;
    void *part = need > 0 ? wsc + sbytes + ibytes + hbytes + dbytes : nullptr;
    // MXFP4 indexer operands: read as stored by the FP4 scan; otherwise (head counts it does
    // not take) their exact FP8 form, after the split-KV partials, for the FP8 scan
    IndexArgs ia{};
    ia.qI = qI ? qI->data : nullptr; ia.qI_scale = qI ? qI->scale : nullptr; ia.qI_e8 = qI ? qI->mx_scale : nullptr;
    ia.KI = KI ? KI->data : nullptr; ia.KI_scale = KI ? KI->scale : nullptr; ia.KI_e8 = KI ? KI->mx_scale : nullptr;
    ia.w = w; ia.ctx = ctx_len; ia.ldS = score_ld(p);
    ia.B = p->B; ia.L = p->L; ia.H_I = p->H_I; ia.m = p->m; ia.ncap = ncap; ia.idx_t = p->idx_t;
    ia.decode = 1;
    const bool fp4_scan = p->topk > 0 && decode_index_fp4_supported(ia);
    csa_index_rows q8{}, k8{};
    if (p->topk > 0 && p->idx_t == CSA_MXFP4 && !fp4_scan) {
        char *w8 = wsc + sbytes + ibytes + hbytes + dbytes + decode_split_bytes(p, 0);
        mxfp4_rows_to_fp8(qI, (int64_t)p->B * p->H_I, w8, &q8, st);
        mxfp4_rows_to_fp8(KI, (int64_t)p->B * ncap, w8 + fp8_rows_bytes((int64_t)p->B * p->H_I), &k8, st);
        ia.qI = q8.data; ia.qI_scale = q8.scale; ia.KI = k8.data; ia.KI_scale = k8.scale;
        ia.idx_t = CSA_FP8E4M3;
    }
    if (p->topk > 0) {
        float *S = reinterpret_cast<float *>(ws);
        idx = topk_out ? topk_out : reinterpret_cast<int32_t *>(reinterpret_cast<char *>(ws) + sbytes);
        ia.S = S;
        // FP8 keys: the tensor-core scan and MXFP4 keys the FP4 scan, which also count each
        // row's keys for the top-k; the exact FP32 scan (and FP8 batches of fewer than 16 query
        // rows) on CUDA cores
        bool counted = false;
        if (fp4_scan) {
            if (cudaMemsetAsync(hist, 0, hbytes + 2 * sizeof(int) * (size_t)p->B, st) != cudaSuccess)
                return CSA_ERR_CUDA;
            counted = launch_decode_index_fp4(ia, hist, st);
            if (!counted) return CSA_ERR_UNSUPPORTED;
        } else if (decode_index_tc_supported(ia)) {
            if (cudaMemsetAsync(hist, 0, hbytes + 2 * sizeof(int) * (size_t)p->B, st) != cudaSuccess)
                return CSA_ERR_CUDA;
            counted = launch_decode_index_tc(ia, hist, st);
            if (!counted) return CSA_ERR_UNSUPPORTED;
        } else {
            launch_indexer(ia, st);
        }
        if (counted) {
            DecSelArgs da{};
            da.S = S; da.ldS = score_ld(p); da.hist = hist; da.ctx = ctx_len; da.out = idx;
            da.cnt = sel_cnt;
            da.above = reinterpret_cast<int32_t *>(reinterpret_cast<char *>(sel_cnt) + decode_select_above_off(p->B));
            da.bin = reinterpret_cast<uint2 *>(reinterpret_cast<char *>(sel_cnt) + decode_select_bin_off(p->B, p->topk));
            da.L = p->L; da.m = p->m; da.ncap = ncap; da.k = p->topk; da.B = p->B;
            launch_decode_select(da, st);
        } else {
            TopkArgs ta{};
            ta.S = S; ta.ldS = score_ld(p); ta.ctx = ctx_len; ta.out = idx;
            ta.L = p->L; ta.m = p->m; ta.ncap = ncap; ta.k = p->topk; ta.nrows = p->B; ta.decode = 1;
            launch_topk(ta, st);
        }
    }
    AttnArgs a = attn_args(p, q, swa_ring, p->topk > 0 ? C : nullptr, idx, ctx_len, sink, rope_tab, out,
                           lse_out, 1, p->topk);
    if (p->topk == 0) {
        a.ncap = 0;
        a.dense = 1;
    }
    return run_decode_attention(a, part, st);
}

int hca_decode(const csa_params *p, const void *q, const int32_t *ctx_len, const csa_entries *C,
               const void *swa_ring, const float *sink, const float *rope_tab, void *out,
               float *lse_out, void *ws, size_t wsb, csa_stream_t stream) {
    int s = check(p, CSA_OP_HCA_DECODE);
    if (s) return s;
    if (!q || !ctx_len || !swa_ring || !out || !aligned16(q) || !aligned16(swa_ring) || !aligned16(out) ||
        !entries_ok(p, C))
        return CSA_ERR_INVALID;
    if (p->d_rope > 0 && !rope_tab) return CSA_ERR_INVALID;
    const size_t need = ws_bytes(p, CSA_OP_HCA_DECODE);
    if (need > 0 && (wsb < need || !ws || !aligned16(ws))) return CSA_ERR_WORKSPACE;
    AttnArgs a = attn_args(p, q, swa_ring, C, nullptr, ctx_len, sink, rope_tab, out, lse_out, 1, 0);
    a.dense = 1;  // every visible entry, in order
    return run_decode_attention(a, ws, cs(stream));
}

int csa_gemm_bf16(const void *A, int64_t lda, const void *B, int64_t ldb, int M, int N, int K, int groups,
                  const csa_gemm_out *outs, int n_outs, csa_stream_t stream) {
    if (!A || !B || !outs || n_outs < 1 || n_outs > 4 || !aligned16(A) || !aligned16(B)) return CSA_ERR_INVALID;
    GemmArgs g{};
    g.A = A; g.lda = lda; g.B = B; g.ldb = ldb; g.M = M; g.N = N; g.K = K; g.groups = groups; g.n_out = n_outs;
    for (int i = 0; i < n_outs; ++i) {
        const csa_gemm_out &o = outs[i];
        if (!o.ptr || o.col0 < 0 || o.col1 <= o.col0 || o.col1 > N || o.ld < o.col1 - o.col0) return CSA_ERR_INVALID;
        if (o.dtype != CSA_F32 && o.dtype != CSA_BF16) return CSA_ERR_INVALID;
        g.out[i] = o;
    }
    const int s = launch_gemm_bf16(g, cs(stream));
    return s ? s : launch_status();
}

uint64_t csa_launch_count(void) { return launch_counter(); }

int csa_device_status(int *status, int reset, csa_stream_t stream) {
    if (!status) return CSA_ERR_INVALID;
    cudaStream_t st = cs(stream);
    if (cudaStreamSynchronize(st) != cudaSuccess) return CSA_ERR_CUDA;
    int v = 0;
    if (cudaMemcpyFromSymbolAsync(&v, g_status, sizeof(int), 0, cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return CSA_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return CSA_ERR_CUDA;
    *status = v;
    if (reset) {
        launch_status_reset(st);
        if (cudaStreamSynchronize(st) != cudaSuccess) return CSA_ERR_CUDA;
    }
    return CSA_OK;
}

int csa_probe_ffma(int blocks, int iters, float *out, csa_stream_t stream) {
    if (blocks < 1 || iters < 1 || !out) return CSA_ERR_INVALID;
    launch_probe_ffma(blocks, iters, out, cs(stream));
    return launch_status();
}

int csa_probe_read(const void *buf, int64_t bytes, int reps, int blocks, float *out, csa_stream_t stream) {
    if (!buf || !aligned16(buf) || bytes < 16 || bytes % 16 != 0 || reps < 1 || blocks < 1 || !out)
        return CSA_ERR_INVALID;
    launch_probe_read(buf, bytes, reps, blocks, out, cs(stream));
    return launch_status();
}

int csa_selftest_wait_timeout(uint64_t limit_ns, csa_stream_t stream) {
    if (limit_ns == 0 || limit_ns > 1000000000ull) return CSA_ERR_INVALID;
    launch_wait_selftest(limit_ns, cs(stream));
    return launch_status();
}

}  // extern "C"
