"""The method's steps strung together, per sequence -- TEST INFRASTRUCTURE (oracle).

Sources: [P2] "DeepSeek-V4: Towards Highly Efficient Million-Token Context Intelligence"
(wiki notes), 提案手法 §1 and 訓練インフラの革新 §5; [P5] "deepseek V4 技术论文" 一.1.

Storage formats that the configurations fix are applied exactly where the data would be
stored, because they are approximations the result depends on:
  * compressed entries ("c_store"): 'f32', 'bf16', 'mixed' -- [P2] 訓練インフラの革新 §5:
    a KV entry keeps its RoPE dimensions in BF16 and its other dimensions in FP8 (reading:
    E4M3 with one float scale per entry row, amax/448) -- or 'nvfp4' -- [P3] "Технический
    отчёт DeepSeek-V4.1-Flash — часть 2/2": the V4.1 KV cache in NVFP4, quantised after RoPE
    (blocks of 16 E2M1 values with an E4M3 scale; reading: one float scale per entry row);
  * window rows: as the activations ('f32', 'bf16') or, for the V4.1 decode ring ([P3]: the
    SWA cache in FP8), 'fp8' rows with one scale each;
  * indexer operands ("idx_store"): 'f32', 'fp8' (E4M3, one scale per row of d_I values) or
    'mxfp4' (E2M1 elements, one power-of-two scale per 32 -- the pages' own indexer precision,
    [P2] 事後学習 §3; the configurations ask for FP32 and FP8);
  * raw rows after RoPE ("q_store"): 'f32' or 'bf16', the activation dtype.
Everything else is double precision.
"""
from __future__ import annotations

import numpy as np

from . import (attention_rows, compress, decode_one, dequant_fp8, dequant_mxfp4, dequant_nvfp4, entry_pos,
               index_scores_f32, index_scores_f64, num_entries, quant_rows_fp8, quant_rows_mxfp4, quant_rows_nvfp4,
               rope, round_bf16_fast, topk)

__all__ = ["store_rows", "kv_compress", "indexer_topk", "csa_rows", "hca_rows", "csa_decode",
           "hca_decode", "project", "grouped_output_projection"]


def store_rows(x: np.ndarray, store: str, d_rope: int = 0):
    """Apply a storage format to rows x [..., d] (double in, double out).

    Returns (values, extra) where values are the dequantised doubles and extra holds the
    stored representation for the formats that have one (codes and scales)."""
    x = np.asarray(x, np.float64)
    if store == "f64":
        return x, None
    if store == "f32":
        return x.astype(np.float32).astype(np.float64), None
    if store == "bf16":
        return round_bf16_fast(x.astype(np.float32)).astype(np.float64), None
    if store == "fp8":
        codes, scales = quant_rows_fp8(x.astype(np.float32))
        return dequant_fp8(codes, scales), (codes, scales)
    if store == "mxfp4":
        codes, e8 = quant_rows_mxfp4(x.astype(np.float32))
        return dequant_mxfp4(codes, e8), (codes, e8)
    if store == "nvfp4":
        codes, bcode, rs = quant_rows_nvfp4(x.astype(np.float32))
        return dequant_nvfp4(codes, bcode, rs), (codes, bcode, rs)
    if store == "mixed":
        d = x.shape[-1]
        nope = x[..., : d - d_rope]
        codes, scales = quant_rows_fp8(nope.astype(np.float32))
        out = np.empty_like(x)
        out[..., : d - d_rope] = dequant_fp8(codes, scales)
        out[..., d - d_rope:] = round_bf16_fast(x[..., d - d_rope:].astype(np.float32))
        return out, (codes, scales)
    raise ValueError(store)


def kv_compress(kv, z, kI_raw, m, d_rope, theta, c_store="f64", idx_store="f64", q_store="f64"):
    """Compression of one sequence.

    kv [L, d] raw shared-KV rows (before RoPE); z [L, 2] compression logits (set a, set b);
    kI_raw [L, dI] raw indexer-key rows or None.
    Returns dict with
      C      [N, d]  entries after RoPE at (j+1)m-1, in c_store (as doubles),
      C_raw  stored representation for 'mixed' (codes, scales) and 'nvfp4' (codes, block
             codes, row scales), else None,
      KI     [N, dI] compressed indexer keys in idx_store (as doubles) or None,
      KI_raw stored representation for 'fp8', else None,
      kv_rope [L, d] raw rows after RoPE at their own positions, in q_store (the window
             keys; q_store 'fp8' gives the rows of an FP8 decode ring).
    """
    kv = np.asarray(kv, np.float64)
    L, d = kv.shape
    N = num_entries(L, m)
    C = compress(kv, z, m)
    C = rope(C, entry_pos(N, m), d_rope, theta, +1)
    C, C_raw = store_rows(C, c_store, d_rope)
    KI = KI_raw = None
    if kI_raw is not None:
        KI, KI_raw = store_rows(compress(kI_raw, z, m), idx_store)
    kvr, _ = store_rows(rope(kv, np.arange(L), d_rope, theta, +1), q_store)
    return dict(C=C, C_raw=C_raw, KI=KI, KI_raw=KI_raw, kv_rope=kvr, N=N)


def indexer_topk(qI_rows, KI, w_rows, m, k, pos, idx_store):
    """Indexer scores and top-k for query rows at positions pos.

    idx_store 'f32': qI_rows, KI float32 values, fixed-order FP32 score.
    idx_store 'fp8': qI_rows are quantised here per (row, head) and the score is taken in
    double on the dequantised values; KI must already be the dequantised FP8 keys.
    Returns (scores [nrows, N], idx [nrows, k])."""
    if idx_store == "f32":
        s = index_scores_f32(np.asarray(qI_rows, np.float32), np.asarray(KI, np.float32),
                             np.asarray(w_rows, np.float32), m, pos)
    elif idx_store in ("fp8", "mxfp4", "f64"):
        q = np.asarray(qI_rows, np.float64)
        if idx_store != "f64":
            q, _ = store_rows(q, idx_store)
        s = index_scores_f64(q, np.asarray(KI, np.float64), np.asarray(w_rows, np.float64), m, pos)
    else:
        raise ValueError(idx_store)
    return s, topk(s, m, pos, k)


def csa_rows(q_rows, kv_rope, C, qI_rows, KI, w_rows, sink, pos, *, m, k, d_rope, theta, n_win,
             scale, idx_store):
    """CSA attention for query rows (at positions pos) of one sequence.

    Returns dict(scores, idx, o, psum)."""
    if k > 0:
        s, idx = indexer_topk(qI_rows, KI, w_rows, m, k, pos, idx_store)
    else:
        s, idx = None, np.zeros((len(pos), 0), np.int32)
    o, ps = attention_rows(q_rows, kv_rope, C, idx, k, m, d_rope, theta, n_win, sink, scale, pos)
    return dict(scores=s, idx=idx, o=o, psum=ps)


def hca_rows(q_rows, kv_rope, C, sink, pos, *, m, d_rope, theta, n_win, scale):
    """HCA attention (dense over every visible entry) for query rows of one sequence."""
    o, ps = attention_rows(q_rows, kv_rope, C, None, 0, m, d_rope, theta, n_win, sink, scale, pos)
    return dict(o=o, psum=ps)


def csa_decode(q, ctx, C, qI, KI, w, ring, sink, *, m, k, d_rope, theta, n_win, scale, idx_store):
    """One CSA decode step of one sequence: q [H, d], qI [HI, dI], w [HI]; ctx counts the
    new token (position ctx - 1). C [Ncap, d] and KI [Ncap, dI] are the caches (values)."""
    p = ctx - 1
    s, idx = indexer_topk(np.asarray(qI)[None], KI, np.asarray(w)[None], m, k, np.array([p]), idx_store)
    o, ps = decode_one(q, ctx, C, idx[0], k, m, ring, d_rope, theta, n_win, sink, scale)
    return dict(scores=s[0], idx=idx[0], o=o, psum=ps)


def hca_decode(q, ctx, C, ring, sink, *, m, d_rope, theta, n_win, scale):
    o, ps = decode_one(q, ctx, C, None, 0, m, ring, d_rope, theta, n_win, sink, scale)
    return dict(o=o, psum=ps)


def project(x, W):
    """A projection of rows: x [rows, K] times W [N, K] transposed -> [rows, N], in double
    (the hidden-state projections to the layer's inputs; [P2] 概要: hidden size 4096)."""
    return np.asarray(x, np.float64) @ np.asarray(W, np.float64).T


def grouped_output_projection(o, Wg, Wo, groups):
    """The grouped output projection ([P2] 提案手法 §1 CSA; [P5] 一.1 分组输出投影). o [rows, H, d]:
    the heads are split into `groups` consecutive groups; group g's heads, concatenated
    ([rows, H/groups * d]), are projected by its own matrix Wg[g] ([d_g, H/groups * d]); the
    group outputs, concatenated in group order ([rows, groups * d_g]), are projected by Wo
    ([hidden, groups * d_g]). Wg is given stacked: [groups * d_g, H/groups * d]."""
    o = np.asarray(o, np.float64)
    rows, H, d = o.shape
    hg = H // groups
    dg = Wg.shape[0] // groups
    y = np.empty((rows, groups * dg), np.float64)
    for g in range(groups):
        og = o[:, g * hg:(g + 1) * hg, :].reshape(rows, hg * d)
        y[:, g * dg:(g + 1) * dg] = project(og, Wg[g * dg:(g + 1) * dg])
    return y, project(y, Wo)
