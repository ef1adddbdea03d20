/*
 * csa_oracle.c -- plain, slow CPU reference of hybrid compressed attention (CSA / HCA).
 *
 * TEST INFRASTRUCTURE. This file is the oracle that the CUDA library is checked against.
 * Only the test-suite, the smoke check and the benchmark's CPU-baseline leg load it; the
 * library's own code path never does, and the two share no code, headers or tables.
 *
 * Sources (the method is described in prose only; no page prints a formula):
 *  [P2] "DeepSeek-V4: Towards Highly Efficient Million-Token Context Intelligence"
 *       (wiki notes), section 提案手法, item 1 "ハイブリッドアテンション (CSA + HCA)", and
 *       section 訓練インフラの革新, item 5 "推論フレームワーク" (mixed-precision KV entries).
 *  [P4] "EP 95 DeepSeek-V4論文を読む" (podcast transcript), segments
 *       "Sparse Attentionを構成する3つの中核コンポーネント 12:10" and
 *       "KV cacheを扱うLightning Indexerとtop-k選択 17:10".
 *  [P5] "deepseek V4 技术论文", section 一.1 "混合注意力机制：CSA + HCA".
 *
 * Where the pages leave a step open, the reading taken is stated beside the function.
 *
 * Arithmetic is double precision, except
 *   - orc_index_scores_f32: the FP32 lightning-indexer score in a fixed single-precision
 *     fma order, so a top-k decision can be compared bit for bit with the GPU;
 *   - the FP8 E4M3 codec and the per-row scale, which are defined on float values;
 *   - the FP4 (E2M1 / MXFP4) codec, whose encoder takes its input in double;
 *   - orc_round_bf16, the storage rounding of a float to bfloat16.
 * Build with -ffp-contract=off so that the compiler adds no fused operations of its own.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------------------ */
/* Partial RoPE.                                                                         */
/* [P2] 提案手法 §1, last bullet: RoPE acts on the last 64 dimensions only, and the core  */
/* attention output is rotated back (inverse RoPE) so that it carries relative position. */
/* Reading: half-split pairs (base+i, base+half+i), i < half, base = d - d_rope,         */
/* frequency theta^(-i/half); angle = pos * frequency in double.                          */
/* sign = +1 rotates forward, -1 applies the inverse rotation.                           */
/* ------------------------------------------------------------------------------------ */
void orc_rope(double *x, int64_t rows, int d, int d_rope, const int64_t *pos,
              double theta, int sign)
{
    if (d_rope <= 0) return;
    const int half = d_rope / 2, base = d - d_rope;
    for (int64_t r = 0; r < rows; ++r) {
        double *row = x + r * d;
        for (int i = 0; i < half; ++i) {
            double freq = pow(theta, -(double)i / (double)half);
            double ang = (double)sign * (double)pos[r] * freq;
            double c = cos(ang), s = sin(ang);
            double a = row[base + i], b = row[base + half + i];
            row[base + i] = a * c - b * s;
            row[base + half + i] = a * s + b * c;
        }
    }
}

/* ------------------------------------------------------------------------------------ */
/* Overlapping weighted-average compression.                                             */
/* [P2] 提案手法 §1 CSA: one entry per m tokens by a weighted average, with overlapping  */
/* compression between adjacent blocks; HCA: the same with m' = 128. [P5] 一.1: the      */
/* second set C^b overlaps C^a. [P4] 17:10: two sets are built and then combined.        */
/* Reading: entry j draws on the window [(j-1)m, (j+1)m) clipped to [0, L). A token of   */
/* block j (set a) contributes logit z[t,0]; a token of block j-1 (set b) contributes    */
/* z[t,1]. The weights are one softmax over the tokens present, so entry j is a convex   */
/* combination of at most 2m raw rows. There are ceil(L/m) entries.                      */
/* ------------------------------------------------------------------------------------ */
int64_t orc_num_entries(int64_t L, int m) { return (L + m - 1) / m; }

void orc_compress(const double *x, int64_t L, int dx, const double *z, int m, double *out)
{
    const int64_t N = orc_num_entries(L, m);
    for (int64_t j = 0; j < N; ++j) {
        int64_t lo = (j - 1) * m, hi = (j + 1) * m;
        if (lo < 0) lo = 0;
        if (hi > L) hi = L;
        double mx = -INFINITY;
        for (int64_t t = lo; t < hi; ++t) {
            double l = (t >= j * m) ? z[2 * t + 0] : z[2 * t + 1];
            if (l > mx) mx = l;
        }
        double den = 0.0;
        for (int64_t t = lo; t < hi; ++t) {
            double l = (t >= j * m) ? z[2 * t + 0] : z[2 * t + 1];
            den += exp(l - mx);
        }
        double *o = out + j * dx;
        for (int c = 0; c < dx; ++c) o[c] = 0.0;
        for (int64_t t = lo; t < hi; ++t) {
            double l = (t >= j * m) ? z[2 * t + 0] : z[2 * t + 1];
            double a = exp(l - mx) / den;
            for (int c = 0; c < dx; ++c) o[c] += a * x[t * dx + c];
        }
    }
}

/* Position given to compressed entry j: the last token it covers, (j+1)m - 1, which is  */
/* also the first query position allowed to see it (reading; the pages are silent).     */
int64_t orc_entry_pos(int64_t j, int m) { return (j + 1) * (int64_t)m - 1; }

/* Number of entries a query at position t may see: entry j is visible iff             */
/* (j+1)m - 1 <= t, i.e. every token it covers is at or before t.                      */
int64_t orc_visible(int64_t t, int m, int64_t N)
{
    int64_t v = (t + 1) / m;
    return v < N ? v : N;
}

/* ------------------------------------------------------------------------------------ */
/* Storage roundings.                                                                    */
/* ------------------------------------------------------------------------------------ */

/* Round a float to the nearest bfloat16 (ties to even), returned as a float.            */
/* bfloat16 keeps the sign, the 8 exponent bits and the top 7 mantissa bits of binary32. */
float orc_round_bf16(float x)
{
    if (isnan(x)) return x;
    uint32_t u;
    memcpy(&u, &x, 4);
    uint32_t lower = u & 0xFFFFu;
    uint32_t upper = u & 0xFFFF0000u;
    uint32_t lsb = (u >> 16) & 1u;
    if (lower > 0x8000u || (lower == 0x8000u && lsb)) upper += 0x10000u;
    float r;
    memcpy(&r, &upper, 4);
    return r;
}

/* FP8 E4M3 ("fn" variant of the OCP 8-bit floating-point specification): 1 sign bit,   */
/* 4 exponent bits with bias 7, 3 mantissa bits; exponent field 0 holds subnormals       */
/* (mantissa/8 * 2^-6); no infinities; S.1111.111 is NaN; the largest finite is 448.     */
float orc_fp8_decode(uint8_t code)
{
    int sgn = code >> 7, e = (code >> 3) & 0xF, mt = code & 7;
    double v;
    if (e == 0xF && mt == 7) return NAN;
    if (e == 0) v = ldexp((double)mt / 8.0, -6);
    else v = ldexp(1.0 + (double)mt / 8.0, e - 7);
    return (float)(sgn ? -v : v);
}

/* Encode by direct search: the nearest of the 127 finite non-negative codes, ties to   */
/* the code with an even mantissa, magnitudes above 448 saturate to 448.                 */
uint8_t orc_fp8_encode(float x)
{
    if (isnan(x)) return 0x7F;
    uint8_t sgn = signbit(x) ? 0x80 : 0x00;
    double a = fabs((double)x);
    if (a >= 448.0) return sgn | 0x7E;
    int best = 0;
    double best_err = INFINITY;
    for (int c = 0; c <= 0x7E; ++c) {
        double v = (double)orc_fp8_decode((uint8_t)c);
        double err = fabs(v - a);
        if (err < best_err || (err == best_err && (c & 1) == 0 && (best & 1) == 1)) {
            best = c;
            best_err = err;
        }
    }
    return sgn | (uint8_t)best;
}

/* Per-row FP8 quantisation (reading: one float scale per row, scale = amax / 448 in     */
/* float; code = E4M3(x / scale) with the division in float; a row of zeros gets scale 0 */
/* and all-zero codes). Dequantised value = decode(code) * scale.                        */
void orc_quant_rows_fp8(const float *x, int64_t rows, int cols, uint8_t *codes, float *scales)
{
    for (int64_t r = 0; r < rows; ++r) {
        const float *row = x + r * cols;
        float amax = 0.0f;
        for (int c = 0; c < cols; ++c) {
            float a = fabsf(row[c]);
            if (a > amax) amax = a;
        }
        float scale = amax / 448.0f;
        scales[r] = scale;
        for (int c = 0; c < cols; ++c) {
            codes[r * cols + c] = (scale > 0.0f) ? orc_fp8_encode(row[c] / scale) : 0;
        }
    }
}

/* ------------------------------------------------------------------------------------ */
/* FP4: E2M1 elements and the MXFP4 block format.                                        */
/* [P2] 事後学習 §3: the CSA indexer's QK path is quantised to FP4 (MXFP4); dequantising  */
/* FP4 to FP8 is lossless, so the FP8 stack is reused. [P3] (V4.1): the KV cache is       */
/* stored in NVFP4, quantised after RoPE.                                                 */
/* E2M1 (OCP microscaling formats): 1 sign bit, 2 exponent bits with bias 1, 1 mantissa  */
/* bit, no infinities or NaN. Codes 0..7 are the magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6;  */
/* bit 3 is the sign. Encoding rounds to nearest, ties to the even code, and saturates   */
/* at 6. MXFP4: blocks of 32 elements share a power-of-two scale X = 2^e stored as an    */
/* E8M0 byte (e + 127); e = floor(log2(max |v|)) - 2 (2 = the exponent of E2M1's largest */
/* value), elements = E2M1(v / X). Reading: a block of zeros gets the byte 0 (X = 2^-127) */
/* and zero codes.                                                                        */
/* ------------------------------------------------------------------------------------ */

double orc_e2m1_decode(uint8_t code)
{
    static const double mag[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};
    const double v = mag[code & 7];
    return (code & 8) ? -v : v;
}

uint8_t orc_e2m1_encode(double x)
{
    const uint8_t sgn = signbit(x) ? 8 : 0;
    const double a = fabs(x);
    if (a >= 6.0) return sgn | 7;
    int best = 0;
    double best_err = INFINITY;
    for (int c = 0; c < 8; ++c) {
        const double err = fabs(orc_e2m1_decode((uint8_t)c) - a);
        if (err < best_err || (err == best_err && (c & 1) == 0 && (best & 1) == 1)) {
            best = c;
            best_err = err;
        }
    }
    return sgn | (uint8_t)best;
}

/* Per-row MXFP4 quantisation of x [rows, cols] (cols a multiple of 32): codes [rows,     */
/* cols/2] with element 2i in the low nibble of byte i and element 2i+1 in the high one, */
/* and one E8M0 byte per block [rows, cols/32]. Dequantised value = E2M1 * 2^(byte-127). */
void orc_quant_rows_mxfp4(const float *x, int64_t rows, int cols, uint8_t *codes, uint8_t *e8)
{
    for (int64_t r = 0; r < rows; ++r) {
        for (int blk = 0; blk < cols / 32; ++blk) {
            const float *v = x + r * cols + blk * 32;
            double amax = 0.0;
            for (int i = 0; i < 32; ++i) amax = fmax(amax, fabs((double)v[i]));
            int e = -127;
            if (amax > 0.0) {
                int ex;
                frexp(amax, &ex);  /* amax = f * 2^ex, f in [0.5, 1): floor(log2 amax) = ex - 1 */
                e = ex - 1 - 2;
                if (e < -127) e = -127;
                if (e > 127) e = 127;
            }
            e8[r * (cols / 32) + blk] = (uint8_t)(e + 127);
            for (int i = 0; i < 32; ++i) {
                const uint8_t q = amax > 0.0 ? orc_e2m1_encode(ldexp((double)v[i], -e)) : 0;
                uint8_t *byte = codes + r * (cols / 2) + blk * 16 + i / 2;
                if (i % 2 == 0) *byte = q; else *byte |= (uint8_t)(q << 4);
            }
        }
    }
}

/* NVFP4 rows (reading of [P3] "Технический отчёт DeepSeek-V4.1-Flash — часть 2/2": the   */
/* V4.1 KV cache is stored in NVFP4, quantised after RoPE). NVFP4: blocks of 16 E2M1      */
/* elements, each with an E4M3 scale. Reading of its second-level scale: one float per    */
/* row, s = amax / (6 * 448) in float, so that every block scale fits E4M3 (6 = E2M1's    */
/* largest value, 448 = E4M3's). Block b with max |x| = bmax: code_b = E4M3(bmax / (6 s)) */
/* (the product 6 s and the division in float); scale_b = decode(code_b) * s in float;    */
/* element = E2M1(x / scale_b), the division in float, 0 when scale_b is 0 (also when the */
/* block scale underflows E4M3). Dequantised value = E2M1 * scale_b.                     */
/* x [rows, cols] (cols a multiple of 16) -> codes [rows, cols/2] (element 2i in the low   */
/* nibble of byte i), block codes [rows, cols/16], row scales [rows].                     */
void orc_quant_rows_nvfp4(const float *x, int64_t rows, int cols, uint8_t *codes, uint8_t *bcode, float *rs)
{
    for (int64_t r = 0; r < rows; ++r) {
        const float *row = x + r * cols;
        float amax = 0.0f;
        for (int c = 0; c < cols; ++c) amax = fmaxf(amax, fabsf(row[c]));
        const float s = amax / 2688.0f;
        rs[r] = s;
        for (int blk = 0; blk < cols / 16; ++blk) {
            const float *v = row + blk * 16;
            float bmax = 0.0f;
            for (int i = 0; i < 16; ++i) bmax = fmaxf(bmax, fabsf(v[i]));
            const float six_s = 6.0f * s;
            const uint8_t bc = s > 0.0f ? orc_fp8_encode(bmax / six_s) : 0;
            bcode[r * (cols / 16) + blk] = bc;
            const float scale = orc_fp8_decode(bc) * s;
            for (int i = 0; i < 16; ++i) {
                const uint8_t q = scale > 0.0f ? orc_e2m1_encode((double)(v[i] / scale)) : 0;
                uint8_t *byte = codes + r * (cols / 2) + blk * 8 + i / 2;
                if (i % 2 == 0) *byte = q; else *byte |= (uint8_t)(q << 4);
            }
        }
    }
}

/* ------------------------------------------------------------------------------------ */
/* Lightning indexer score.                                                              */
/* [P2] 提案手法 §1 CSA: a lightning indexer scores the compressed entries so that top-k */
/* can be chosen; [P5] 一.1: low-rank, cheap; [P4] 17:10 and 21:36: it must look at all  */
/* entries, so it has to be light, and it is nearly the indexer of DeepSeek Sparse       */
/* Attention.                                                                            */
/* Reading: s(t,j) = sum_h w[t,h] * ReLU(qI[t,h] . KI[j]) over H_I indexer heads with   */
/* one indexer key per entry; entries not visible to t score -inf.                      */
/* ------------------------------------------------------------------------------------ */

/* FP32 form in a fixed order: acc = fma(q_c, k_c, acc) over c = 0..dI-1 from +0;      */
/* r = acc > 0 ? acc : 0; s = fma(w_h, r, s) over h = 0..HI-1 from +0; -0 becomes +0.   */
/* qI [nrows, HI, dI] and w [nrows, HI] hold the query rows; pos[r] is the position of   */
/* row r (visibility); KI [N, dI]; s [nrows, N].                                         */
void orc_index_scores_f32(const float *qI, const float *KI, const float *w, int64_t N,
                          int HI, int dI, int m, const int64_t *pos, int64_t nrows,
                          float *s)
{
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t r = 0; r < nrows; ++r) {
        const int64_t t = pos[r];
        const int64_t vis = orc_visible(t, m, N);
        for (int64_t j = 0; j < N; ++j) {
            if (j >= vis) { s[r * N + j] = -INFINITY; continue; }
            float acc_s = 0.0f;
            for (int h = 0; h < HI; ++h) {
                const float *q = qI + (r * HI + h) * dI;
                const float *k = KI + j * dI;
                float acc = 0.0f;
                for (int c = 0; c < dI; ++c) acc = fmaf(q[c], k[c], acc);
                float rl = acc > 0.0f ? acc : 0.0f;
                acc_s = fmaf(w[r * HI + h], rl, acc_s);
            }
            if (acc_s == 0.0f) acc_s = 0.0f;
            s[r * N + j] = acc_s;
        }
    }
}

/* Double form, used with dequantised FP8 operands. */
void orc_index_scores_f64(const double *qI, const double *KI, const double *w, int64_t N,
                          int HI, int dI, int m, const int64_t *pos, int64_t nrows,
                          double *s)
{
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t r = 0; r < nrows; ++r) {
        const int64_t t = pos[r];
        const int64_t vis = orc_visible(t, m, N);
        for (int64_t j = 0; j < N; ++j) {
            if (j >= vis) { s[r * N + j] = -INFINITY; continue; }
            double acc_s = 0.0;
            for (int h = 0; h < HI; ++h) {
                const double *q = qI + (r * HI + h) * dI;
                const double *k = KI + j * dI;
                double acc = 0.0;
                for (int c = 0; c < dI; ++c) acc += q[c] * k[c];
                acc_s += w[r * HI + h] * (acc > 0.0 ? acc : 0.0);
            }
            s[r * N + j] = acc_s;
        }
    }
}

/* ------------------------------------------------------------------------------------ */
/* Top-k selection.                                                                      */
/* [P5] 一.1 CSA: every query token attends only to its top-k compressed entries;        */
/* [P4] 17:10: the indexer picks the top k and attention runs on those k only.           */
/* Reading: among the n visible entries, order by (score descending, index ascending)    */
/* and keep the first min(k, n); the kept set is returned in ascending index order and   */
/* padded with -1.                                                                       */
/* ------------------------------------------------------------------------------------ */
typedef struct { double s; int64_t j; } orc_cand;

static int orc_cand_cmp(const void *a, const void *b)
{
    const orc_cand *x = (const orc_cand *)a, *y = (const orc_cand *)b;
    if (x->s > y->s) return -1;
    if (x->s < y->s) return 1;
    return (x->j < y->j) ? -1 : (x->j > y->j);
}

static int orc_i32_cmp(const void *a, const void *b)
{
    int32_t x = *(const int32_t *)a, y = *(const int32_t *)b;
    return (x > y) - (x < y);
}

void orc_topk(const double *s, int64_t N, int m, const int64_t *pos, int64_t nrows, int k,
              int32_t *idx)
{
#pragma omp parallel
    {
        orc_cand *c = (orc_cand *)malloc(sizeof(orc_cand) * (size_t)(N > 0 ? N : 1));
#pragma omp for schedule(dynamic, 4)
        for (int64_t r = 0; r < nrows; ++r) {
            const int64_t vis = orc_visible(pos[r], m, N);
            for (int64_t j = 0; j < vis; ++j) { c[j].s = s[r * N + j]; c[j].j = j; }
            qsort(c, (size_t)vis, sizeof(orc_cand), orc_cand_cmp);
            const int64_t keep = vis < k ? vis : k;
            int32_t *o = idx + r * k;
            for (int64_t i = 0; i < keep; ++i) o[i] = (int32_t)c[i].j;
            qsort(o, (size_t)keep, sizeof(int32_t), orc_i32_cmp);
            for (int64_t i = keep; i < k; ++i) o[i] = -1;
        }
        free(c);
    }
}

/* ------------------------------------------------------------------------------------ */
/* Core attention of one query token over an explicit key set.                           */
/* [P2] 提案手法 §1: shared-KV multi-query attention (one KV head for all query heads);  */
/* [P5] 一.1: a compressed entry serves as both key and value; an attention sink lets a  */
/* head release part of its attention, so the weights of one head may sum to less than  */
/* 1 ([P2] §1: the total attention score of each query head can be made < 1).            */
/* Reading: logits = scale * q_h . key_i; the per-head sink logit enters the softmax     */
/* denominator only (as exp(sink_h)), with no value; value_i = key_i. sink == NULL means */
/* no sink (weights sum to exactly 1). psum_h receives the sum of the weights.           */
/* ------------------------------------------------------------------------------------ */
void orc_attend_one(const double *q, int H, int d, const double *keys, int64_t nk,
                    const double *sink, double scale, double *o, double *psum, double *lg)
{
    for (int h = 0; h < H; ++h) {
        const double *qh = q + (int64_t)h * d;
        double mx = -INFINITY;
        for (int64_t i = 0; i < nk; ++i) {
            double acc = 0.0;
            for (int c = 0; c < d; ++c) acc += qh[c] * keys[i * d + c];
            lg[i] = scale * acc;
            if (lg[i] > mx) mx = lg[i];
        }
        if (sink && sink[h] > mx) mx = sink[h];
        double den = sink ? exp(sink[h] - mx) : 0.0;
        for (int64_t i = 0; i < nk; ++i) den += exp(lg[i] - mx);
        double *oh = o + (int64_t)h * d;
        for (int c = 0; c < d; ++c) oh[c] = 0.0;
        double ps = 0.0;
        for (int64_t i = 0; i < nk; ++i) {
            double p = exp(lg[i] - mx) / den;
            ps += p;
            for (int c = 0; c < d; ++c) oh[c] += p * keys[i * d + c];
        }
        if (psum) psum[h] = ps;
    }
}

/* ------------------------------------------------------------------------------------ */
/* One attention layer for selected query rows (prefill).                                */
/* Key set of query t: the compressed branch (CSA: its top-k entries, skipping -1; HCA:  */
/* every visible entry), followed by the sliding-window branch, the raw rows u with      */
/* max(0, t - n_win + 1) <= u <= t. [P2] §1: both CSA and HCA get an auxiliary sliding-  */
/* window branch with n_win = 128; [P5] 一.1: an independent branch over recent tokens.  */
/* Reading: the branches share one softmax; no de-duplication between them.              */
/*                                                                                       */
/* q   [nrows, H, d] query rows before RoPE; pos[r] is the position t of row r           */
/* kvr [L, d]  raw rows after RoPE at their positions; C [N, d] entries after RoPE      */
/* idx [nrows, k] top-k (NULL = dense, HCA)                                             */
/* o   [nrows, H, d] output after inverse RoPE at t; psum [nrows, H] (nullable).        */
/* ------------------------------------------------------------------------------------ */
void orc_attention_rows(const double *q, const double *kvr, const double *C, int64_t N,
                        const int32_t *idx, int k, int m, int H, int d, int d_rope,
                        double theta, int n_win, const double *sink, double scale,
                        const int64_t *pos_rows, int64_t nrows, double *o, double *psum)
{
#pragma omp parallel
    {
        int64_t cap = (idx ? (int64_t)k : N) + n_win + 1;
        double *keys = (double *)malloc(sizeof(double) * (size_t)(cap * d));
        double *lg = (double *)malloc(sizeof(double) * (size_t)cap);
        double *qt = (double *)malloc(sizeof(double) * (size_t)H * d);
        int64_t *pos = (int64_t *)malloc(sizeof(int64_t) * (size_t)H);
#pragma omp for schedule(dynamic, 2)
        for (int64_t r = 0; r < nrows; ++r) {
            const int64_t t = pos_rows[r];
            int64_t nk = 0;
            if (idx) {
                for (int i = 0; i < k; ++i) {
                    int32_t j = idx[r * k + i];
                    if (j < 0) continue;
                    memcpy(keys + nk * d, C + (int64_t)j * d, sizeof(double) * d);
                    ++nk;
                }
            } else {
                const int64_t vis = orc_visible(t, m, N);
                for (int64_t j = 0; j < vis; ++j) {
                    memcpy(keys + nk * d, C + j * d, sizeof(double) * d);
                    ++nk;
                }
            }
            int64_t u0 = t - n_win + 1;
            if (u0 < 0) u0 = 0;
            for (int64_t u = u0; u <= t; ++u) {
                memcpy(keys + nk * d, kvr + u * d, sizeof(double) * d);
                ++nk;
            }
            memcpy(qt, q + r * (int64_t)H * d, sizeof(double) * (size_t)H * d);
            for (int h = 0; h < H; ++h) pos[h] = t;
            orc_rope(qt, H, d, d_rope, pos, theta, +1);
            double *orow = o + r * (int64_t)H * d;
            orc_attend_one(qt, H, d, keys, nk, sink, scale, orow, psum ? psum + r * H : NULL, lg);
            orc_rope(orow, H, d, d_rope, pos, theta, -1);
        }
        free(keys);
        free(lg);
        free(qt);
        free(pos);
    }
}

/* ------------------------------------------------------------------------------------ */
/* One decode step: one new query per sequence against caches.                          */
/* [P2] 訓練インフラの革新 §5: the inference KV cache is split into a state cache (recent */
/* uncompressed tokens) and a compressed KV cache.                                       */
/* Reading: ctx already counts the new token, whose position is p = ctx - 1; entries    */
/* j < floor(ctx / m) are visible; the sliding window holds raw rows after RoPE, the row */
/* of position u at ring slot u mod n_win, for u in [max(0, p - n_win + 1), p].          */
/* q [H, d] before RoPE; C [Ncap, d] after RoPE; ring [n_win, d]; idx [k] (NULL = HCA). */
/* ------------------------------------------------------------------------------------ */
void orc_decode_one(const double *q, int64_t ctx, const double *C, int64_t Ncap,
                    const int32_t *idx, int k, int m, const double *ring, int H, int d,
                    int d_rope, double theta, int n_win, const double *sink, double scale,
                    double *o, double *psum)
{
    const int64_t p = ctx - 1;
    int64_t vis = ctx / m;
    if (vis > Ncap) vis = Ncap;
    int64_t cap = (idx ? (int64_t)k : vis) + n_win + 1;
    double *keys = (double *)malloc(sizeof(double) * (size_t)(cap * d));
    double *lg = (double *)malloc(sizeof(double) * (size_t)cap);
    double *qt = (double *)malloc(sizeof(double) * (size_t)H * d);
    int64_t *pos = (int64_t *)malloc(sizeof(int64_t) * (size_t)H);
    int64_t nk = 0;
    if (idx) {
        for (int i = 0; i < k; ++i) {
            if (idx[i] < 0) continue;
            memcpy(keys + nk * d, C + (int64_t)idx[i] * d, sizeof(double) * d);
            ++nk;
        }
    } else {
        for (int64_t j = 0; j < vis; ++j) {
            memcpy(keys + nk * d, C + j * d, sizeof(double) * d);
            ++nk;
        }
    }
    int64_t u0 = p - n_win + 1;
    if (u0 < 0) u0 = 0;
    for (int64_t u = u0; u <= p; ++u) {
        memcpy(keys + nk * d, ring + (u % n_win) * d, sizeof(double) * d);
        ++nk;
    }
    memcpy(qt, q, sizeof(double) * (size_t)H * d);
    for (int h = 0; h < H; ++h) pos[h] = p;
    orc_rope(qt, H, d, d_rope, pos, theta, +1);
    orc_attend_one(qt, H, d, keys, nk, sink, scale, o, psum, lg);
    orc_rope(o, H, d, d_rope, pos, theta, -1);
    free(keys);
    free(lg);
    free(qt);
    free(pos);
}

int orc_num_threads(void)
{
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}
