"""Seeded synthetic inputs for hybrid compressed attention (a module of its own).

This module only draws random numbers and names shapes; it holds none of the method's
arithmetic. Both the CUDA library's tests/benchmark and the CPU oracle take their inputs
from here, so the two sides always see the same values.

Recipe: every tensor is N(0, 1) float32 drawn with ``torch.Generator('cpu')`` and then cast
(round-to-nearest-even, by torch) to the workload's dtype. A tensor is drawn in chunks of
``CHUNK_ROWS`` leading rows (its dims before the last one or two flattened), chunk c of
tensor number n seeded with ``seed * 1_000_003 + n * 7_919 + c``; any chunk can therefore be
redrawn alone, which lets the oracle rebuild sampled query rows of a workload without
drawing the whole tensor. Tensor numbers follow the fixed order
q, kv, z, qI, kI_raw, w, sink (then the decode caches), per attention layer.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import torch

CHUNK_ROWS = 4096

DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16}


@dataclasses.dataclass(frozen=True)
class Workload:
    """One attention workload (shapes, dtypes, seed)."""
    name: str
    kind: str            # 'csa' | 'hca' | 'pair' (CSA layer + HCA layer) | 'decode'
    B: int
    L: int               # prefill length, or cached context for decode
    H: int
    seed: int
    d: int = 128
    d_rope: int = 64
    m: int = 4           # CSA compression ratio
    m_hca: int = 128     # HCA compression ratio
    H_I: int = 8
    d_I: int = 64
    topk: int = 512
    n_win: int = 128
    theta: float = 1.0e4
    hidden: int = 4096   # hidden size the layer's inputs are projected from (V4-Flash width)
    groups: int = 8      # output-projection head groups
    d_g: int = 512       # output-projection width per group
    q_t: str = "bf16"    # activations: q, raw kv, outputs
    c_t: str = "bf16"    # compressed entries: 'f32' | 'bf16' | 'mixed' | 'nvfp4'
    idx_t: str = "fp8"   # indexer operands: 'f32' | 'fp8' | 'mxfp4'
    w_t: str = ""        # decode window ring: '' (as the activations) | 'fp8'

    @property
    def scale(self) -> float:
        return self.d ** -0.5

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five workloads of the method's benchmark set, plus a profiler-sized copy of the pair.
WORKLOADS = {
    # CSA prefill, one sequence, fp32 end to end (bit-exact top-k workload).
    "csa_f32_L2048": Workload("csa_f32_L2048", "csa", B=1, L=2048, H=8, seed=0, H_I=4, topk=32,
                              q_t="f32", c_t="f32", idx_t="f32"),
    # HCA prefill, one sequence, bf16, 16 heads.
    "hca_bf16_L16384": Workload("hca_bf16_L16384", "hca", B=1, L=16384, H=16, seed=1, m=128),
    # CSA prefill, 4 x 32768, bf16, FP8 indexer, top-512.
    "csa_bf16_4x32768": Workload("csa_bf16_4x32768", "csa", B=4, L=32768, H=64, seed=2),
    # CSA + HCA decode, 16 sequences with 131072 cached tokens each.
    "decode_b16_ctx131072": Workload("decode_b16_ctx131072", "decode", B=16, L=131072, H=64, seed=3),
    # The same decode step on the V4.1 cache: NVFP4 entries, an FP8 window ring.
    "decode_v41_b16_ctx131072": Workload("decode_v41_b16_ctx131072", "decode", B=16, L=131072, H=64, seed=3,
                                         c_t="nvfp4", w_t="fp8"),
    # ... and with the indexer in FP4 as well (MXFP4 keys and queries): the pages' low-precision formats.
    "decode_fp4_b16_ctx131072": Workload("decode_fp4_b16_ctx131072", "decode", B=16, L=131072, H=64, seed=3,
                                         c_t="nvfp4", w_t="fp8", idx_t="mxfp4"),
    # Interleaved CSA + HCA layer pair, L = 262144, mixed-precision KV entries, top-1024.
    "pair_mixed_L262144": Workload("pair_mixed_L262144", "pair", B=1, L=262144, H=64, seed=4,
                                   topk=1024, c_t="mixed"),
    # The same layer pair at one eighth of the length: a profiler-sized case of the same kernels
    # (identical per-token configuration; the compressed caches fit L2 at both lengths).
    "pair_mixed_L32768": Workload("pair_mixed_L32768", "pair", B=1, L=32768, H=64, seed=4,
                                  topk=1024, c_t="mixed"),
}


def _chunk_seed(seed: int, tensor_no: int, chunk: int) -> int:
    return (seed * 1_000_003 + tensor_no * 7_919 + chunk) % (2**63 - 1)


def randn_rows(seed: int, tensor_no: int, shape, dtype: str = "f32",
               rows: Optional[torch.Tensor] = None, pin: bool = False) -> torch.Tensor:
    """Draw tensor `tensor_no` of shape `shape`; leading dims = shape[:-1] flattened into
    rows of shape[-1] values. With `rows` (1-D int64 of flat row ids), only those rows are
    returned, as [len(rows), shape[-1]]."""
    shape = tuple(int(s) for s in shape)
    row_len = shape[-1]
    n_rows = 1
    for s in shape[:-1]:
        n_rows *= s
    out_dtype = DTYPES[dtype]
    if rows is None:
        out = torch.empty((n_rows, row_len), dtype=out_dtype, pin_memory=pin)
        for c0 in range(0, n_rows, CHUNK_ROWS):
            c1 = min(n_rows, c0 + CHUNK_ROWS)
            g = torch.Generator("cpu").manual_seed(_chunk_seed(seed, tensor_no, c0 // CHUNK_ROWS))
            out[c0:c1] = torch.randn((c1 - c0, row_len), generator=g, dtype=torch.float32).to(out_dtype)
        return out.view(shape)
    rows = torch.as_tensor(rows, dtype=torch.int64)
    out = torch.empty((rows.numel(), row_len), dtype=out_dtype)
    chunks = torch.unique(rows // CHUNK_ROWS)
    for c in chunks.tolist():
        c0 = c * CHUNK_ROWS
        c1 = min(n_rows, c0 + CHUNK_ROWS)
        g = torch.Generator("cpu").manual_seed(_chunk_seed(seed, tensor_no, c))
        block = torch.randn((c1 - c0, row_len), generator=g, dtype=torch.float32).to(out_dtype)
        sel = (rows // CHUNK_ROWS) == c
        out[sel] = block[rows[sel] - c0]
    return out


# Tensor numbers (fixed order per layer; a layer pair offsets the HCA layer by 16).
T_Q, T_KV, T_Z, T_QI, T_KIRAW, T_W, T_SINK = range(7)
T_CACHE_C, T_CACHE_KI, T_RING, T_CTX = 7, 8, 9, 10
LAYER_STRIDE = 16


def prefill_layer(wl: Workload, layer: int = 0, csa: bool = True, pin: bool = False) -> dict:
    """Inputs of one prefill attention layer, as CPU tensors:
    q [B,L,H,d] (q_t), kv [B,L,d] (q_t), z [B,L,2] f32, sink [H] f32 and, for CSA,
    qI [B,L,H_I,d_I] f32, kI_raw [B,L,d_I] f32, w [B,L,H_I] f32."""
    base = layer * LAYER_STRIDE
    B, L = wl.B, wl.L
    out = {
        "q": randn_rows(wl.seed, base + T_Q, (B, L, wl.H, wl.d), wl.q_t, pin=pin),
        "kv": randn_rows(wl.seed, base + T_KV, (B, L, wl.d), wl.q_t, pin=pin),
        "z": randn_rows(wl.seed, base + T_Z, (B, L, 2), "f32", pin=pin),
    }
    if csa:
        out["qI"] = randn_rows(wl.seed, base + T_QI, (B, L, wl.H_I, wl.d_I), "f32", pin=pin)
        out["kI_raw"] = randn_rows(wl.seed, base + T_KIRAW, (B, L, wl.d_I), "f32", pin=pin)
        out["w"] = randn_rows(wl.seed, base + T_W, (B, L, wl.H_I), "f32", pin=pin)
    out["sink"] = randn_rows(wl.seed, base + T_SINK, (wl.H,), "f32", pin=pin)
    return out


def prefill_query_rows(wl: Workload, b: int, ts, layer: int = 0, csa: bool = True) -> dict:
    """The per-query inputs of rows ts of sequence b (same values as prefill_layer)."""
    base = layer * LAYER_STRIDE
    ts = torch.as_tensor(ts, dtype=torch.int64)
    L = wl.L
    flat_t = b * L + ts
    out = {"q": randn_rows(wl.seed, base + T_Q, (wl.B, L, wl.H, wl.d), wl.q_t,
                           rows=(flat_t[:, None] * wl.H + torch.arange(wl.H)[None]).reshape(-1)
                           ).view(len(ts), wl.H, wl.d)}
    if csa:
        out["qI"] = randn_rows(wl.seed, base + T_QI, (wl.B, L, wl.H_I, wl.d_I), "f32",
                               rows=(flat_t[:, None] * wl.H_I + torch.arange(wl.H_I)[None]).reshape(-1)
                               ).view(len(ts), wl.H_I, wl.d_I)
        out["w"] = randn_rows(wl.seed, base + T_W, (wl.B, L, wl.H_I), "f32", rows=flat_t)
    return out


def decode_layer(wl: Workload, layer: int = 0, csa: bool = True, pin: bool = False) -> dict:
    """Inputs of one decode step of one layer, as CPU tensors. Cache contents are synthetic
    N(0,1) rows standing for entries/raw rows already rotated by RoPE.
      q [B,H,d] (q_t); ctx [B] int32 (= L for every sequence); ring [B,n_win,d] (q_t);
      C [B,Ncap,d] (q_t) with Ncap = L / m (CSA) or L / m_hca (HCA); sink [H] f32;
      CSA only: KI [B,Ncap,d_I] f32 (quantised by each side), qI [B,H_I,d_I] f32, w [B,H_I] f32."""
    base = layer * LAYER_STRIDE
    B = wl.B
    m = wl.m if csa else wl.m_hca
    ncap = -(-wl.L // m)
    out = {
        "q": randn_rows(wl.seed, base + T_Q, (B, wl.H, wl.d), wl.q_t, pin=pin),
        "ctx": torch.full((B,), wl.L, dtype=torch.int32),
        "C": randn_rows(wl.seed, base + T_CACHE_C, (B, ncap, wl.d), wl.q_t, pin=pin),
        "ring": randn_rows(wl.seed, base + T_RING, (B, wl.n_win, wl.d), wl.q_t, pin=pin),
        "sink": randn_rows(wl.seed, base + T_SINK, (wl.H,), "f32", pin=pin),
    }
    if csa:
        out["KI"] = randn_rows(wl.seed, base + T_CACHE_KI, (B, ncap, wl.d_I), "f32", pin=pin)
        out["qI"] = randn_rows(wl.seed, base + T_QI, (B, wl.H_I, wl.d_I), "f32", pin=pin)
        out["w"] = randn_rows(wl.seed, base + T_W, (B, wl.H_I), "f32", pin=pin)
    return out


def sample_rows(L: int, n: int, seed: int, first: int = 256, last: int = 128) -> torch.Tensor:
    """Stratified query-row sample of a length-L sequence: the first `first` rows, the last
    `last` rows and the rest uniformly at random without replacement (seeded), sorted."""
    if n >= L:
        return torch.arange(L, dtype=torch.int64)
    head = torch.arange(min(first, L))
    tail = torch.arange(max(0, L - last), L)
    mid_lo, mid_hi = int(head.numel()), L - int(tail.numel())
    k = max(0, n - head.numel() - tail.numel())
    g = torch.Generator("cpu").manual_seed(seed * 31 + 17)
    mid = torch.randperm(max(0, mid_hi - mid_lo), generator=g)[:k] + mid_lo
    return torch.unique(torch.cat([head, tail, mid])).to(torch.int64)


T_X, T_WQ, T_WKV, T_WIDX, T_WG, T_WO = 11, 12, 13, 14, 15, 16  # projections (per layer, + LAYER_STRIDE)


def projection_inputs(wl: Workload, layer: int = 0, csa: bool = True, rows: Optional[int] = None) -> dict:
    """Hidden states and projection weights of one layer, BF16 (CPU tensors): x [rows, hidden];
    Wq [H*d, hidden]; Wkv [d, hidden]; Widx [n_idx, hidden] with n_idx = H_I*d_I + d_I + H_I + 2
    (CSA: the indexer queries, indexer key, weights and compression logits) or 2 (HCA: the
    compression logits); Wg [groups*d_g, (H/groups)*d] (the groups' output matrices, stacked);
    Wo [hidden, groups*d_g]. Weights are N(0, 1) / sqrt(fan_in), so every projection has unit
    scale like the layer inputs drawn directly."""
    base = layer * LAYER_STRIDE
    rows = wl.B * wl.L if rows is None else rows
    hd = wl.hidden
    n_idx = (wl.H_I * wl.d_I + wl.d_I + wl.H_I + 2) if csa else 2
    hg = wl.H // wl.groups

    def w(no, shape, fan_in):
        return (randn_rows(wl.seed, base + no, shape, "f32") * fan_in ** -0.5).to(torch.bfloat16)
    return {
        "x": randn_rows(wl.seed, base + T_X, (rows, hd), "bf16"),
        "Wq": w(T_WQ, (wl.H * wl.d, hd), hd),
        "Wkv": w(T_WKV, (wl.d, hd), hd),
        "Widx": w(T_WIDX, (n_idx, hd), hd),
        "Wg": w(T_WG, (wl.groups * wl.d_g, hg * wl.d), hg * wl.d),
        "Wo": w(T_WO, (hd, wl.groups * wl.d_g), wl.groups * wl.d_g),
    }
