"""One attention layer end to end through the C ABI: buffer allocation (torch) and the
sequence of library calls. No arithmetic happens here.

Prefill layer (CSA):  csa_quant_fp8_rows(qI)  [FP8 indexer only]
                      kv_compress(kv, z, kI_raw) -> entries C, indexer keys KI, kv_rope
                      csa_prefill(q, kv_rope, C, qI, KI, w, sink) -> out
Prefill layer (HCA):  kv_compress(kv, z) -> C, kv_rope;  hca_prefill(q, kv_rope, C, sink) -> out
Decode layer:         csa_quant_fp8_rows(qI);  csa_decode(...) / hca_decode(...)
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional

import torch

from . import (FP8E4M3, MIXED, MXFP4, NVFP4, OP_CSA_DECODE, OP_CSA_PREFILL, OP_HCA_DECODE, OP_HCA_PREFILL, Params,
               alloc_entries, alloc_index_rows, alloc_ring, alloc_workspace, csa_decode, csa_prefill,
               csa_quant_fp8_rows, csa_quant_fp8_window_rows, csa_quant_mxfp4_rows, csa_quant_nvfp4_entries,
               hca_decode, hca_prefill, kv_compress, make_params, rope_table, torch_dtype)


def quantise_index_rows(p: Params, x: torch.Tensor, buf, stream=None):
    """Indexer operand rows in the layer's format: FP8 or MXFP4 codes written into buf by the
    library's quantisers, float rows as they are."""
    if p.idx_t == FP8E4M3:
        csa_quant_fp8_rows(x, buf[0], buf[1], stream)
        return buf
    if p.idx_t == MXFP4:
        csa_quant_mxfp4_rows(x, buf[0], buf[2], stream)
        return buf
    return (x, None)


def layer_params(wl, csa: bool) -> Params:
    """csa_params of one layer of a workload (see synth.Workload)."""
    m = wl.m if csa else wl.m_hca
    return make_params(B=wl.B, L=wl.L, H=wl.H, m=m, topk=wl.topk if csa else 0, n_win=wl.n_win,
                       H_I=wl.H_I, d_I=wl.d_I, d=wl.d, d_rope=wl.d_rope, act=wl.q_t, kv=wl.c_t,
                       idx=wl.idx_t if csa else "f32", win=getattr(wl, "w_t", "") or None)


@dataclass
class PrefillLayer:
    p: Params
    csa: bool
    theta: float
    device: str = "cuda"

    @classmethod
    def create(cls, wl, csa: bool, device="cuda") -> "PrefillLayer":
        self = cls(layer_params(wl, csa), csa, wl.theta, device)
        p = self.p
        self.rope = rope_table(p, wl.theta, device)
        self.C = alloc_entries(p, device)
        adt = torch_dtype(wl.q_t)
        self.kv_rope = torch.empty((p.B, p.L, p.d), dtype=adt, device=device)
        self.out = torch.empty((p.B, p.L, p.H, p.d), dtype=adt, device=device)
        self.lse = torch.empty((p.B, p.L, p.H), dtype=torch.float32, device=device)
        ncap = -(-p.L // p.m)
        if csa and p.topk > 0:
            self.KI = alloc_index_rows(p, (p.B, ncap), device)
            self.qI = alloc_index_rows(p, (p.B, p.L, p.H_I), device)
            self.topk = torch.empty((p.B, p.L, p.topk), dtype=torch.int32, device=device)
            self.ws = alloc_workspace(p, OP_CSA_PREFILL, device)
        else:
            self.KI = self.qI = self.topk = None
            self.ws = alloc_workspace(p, OP_HCA_PREFILL, device)
        return self

    def run(self, inp: dict, stream=None, want_lse: bool = False, want_topk: bool = True) -> torch.Tensor:
        """inp: device tensors q, kv, z, sink and (CSA) qI, kI_raw, w."""
        p = self.p
        lse = self.lse if want_lse else None
        if self.csa and p.topk > 0:
            qI = quantise_index_rows(p, inp["qI"], self.qI, stream)
            kv_compress(p, inp["kv"], inp["z"], inp["kI_raw"], self.rope, self.C, self.KI, self.kv_rope, stream)
            csa_prefill(p, inp["q"], self.kv_rope, self.C, qI, self.KI, inp["w"], inp.get("sink"), self.rope,
                        self.topk if want_topk else None, self.out, lse, self.ws, stream)
        else:
            kv_compress(p, inp["kv"], inp["z"], None, self.rope, self.C, None, self.kv_rope, stream)
            if self.csa:
                csa_prefill(p, inp["q"], self.kv_rope, None, None, None, None, inp.get("sink"), self.rope, None,
                            self.out, lse, self.ws, stream)
            else:
                hca_prefill(p, inp["q"], self.kv_rope, self.C, inp.get("sink"), self.rope, self.out, lse, self.ws,
                            stream)
        return self.out


@dataclass
class DecodeLayer:
    p: Params
    csa: bool
    theta: float
    device: str = "cuda"

    @classmethod
    def create(cls, wl, csa: bool, device="cuda") -> "DecodeLayer":
        self = cls(layer_params(wl, csa), csa, wl.theta, device)
        p = self.p
        self.rope = rope_table(p, wl.theta, device)
        adt = torch_dtype(wl.q_t)
        self.out = torch.empty((p.B, p.H, p.d), dtype=adt, device=device)
        self.lse = torch.empty((p.B, p.H), dtype=torch.float32, device=device)
        ncap = -(-p.L // p.m)
        if csa:
            self.KI = alloc_index_rows(p, (p.B, ncap), device)
            self.qI = alloc_index_rows(p, (p.B, p.H_I), device)
            self.topk = torch.empty((p.B, p.topk), dtype=torch.int32, device=device)
            self.ws = alloc_workspace(p, OP_CSA_DECODE, device)
        else:
            self.ws = alloc_workspace(p, OP_HCA_DECODE, device)
        return self

    def load_caches(self, inp: dict, stream=None):
        """Cache set-up (not part of a decode step): the FP8 indexer-key cache is quantised
        from the float keys; a mixed-precision entry cache is stored from the given rows (the
        first d - d_rope dims as FP8 codes with one scale per entry, the RoPE dims as they are),
        an NVFP4 entry cache and an FP8 ring by the library's quantisers; other entry caches and
        the ring are used as given."""
        self.C = None
        self.ring = None
        if self.p.win_t == FP8E4M3:
            self.ring = alloc_ring(self.p, inp["ring"].device)
            csa_quant_fp8_window_rows(inp["ring"].float().contiguous(), self.ring, stream)
        if self.p.kv_t == NVFP4:
            C = inp["C"]
            codes = torch.empty(C.shape[:-1] + (80,), dtype=torch.uint8, device=C.device)
            csa_quant_nvfp4_entries(C.float().contiguous(), codes, stream)
            self.C = (codes, None, None)
        if self.p.kv_t == MIXED:
            C = inp["C"]
            nope = self.p.d - self.p.d_rope
            codes = torch.empty(C.shape[:-1] + (nope,), dtype=torch.uint8, device=C.device)
            scales = torch.empty(C.shape[:-1], dtype=torch.float32, device=C.device)
            csa_quant_fp8_rows(C[..., :nope].float().contiguous(), codes, scales, stream)
            self.C = (codes, C[..., nope:].to(torch.bfloat16).contiguous(), scales)
        if self.csa:
            self.KI = quantise_index_rows(self.p, inp["KI"], self.KI, stream)

    def run(self, inp: dict, stream=None, want_lse: bool = False, want_topk: bool = True) -> torch.Tensor:
        p = self.p
        lse = self.lse if want_lse else None
        if getattr(self, "C", None) is not None:
            C = self.C
        else:
            C = inp["C"] if isinstance(inp["C"], (tuple, list)) else (inp["C"], None, None)
        ring = self.ring if getattr(self, "ring", None) is not None else inp["ring"]
        if self.csa:
            qI = quantise_index_rows(p, inp["qI"], self.qI, stream)
            csa_decode(p, inp["q"], inp["ctx"], C, qI, self.KI, inp["w"], ring, inp.get("sink"), self.rope,
                       self.topk if want_topk else None, self.out, lse, self.ws, stream)
        else:
            hca_decode(p, inp["q"], inp["ctx"], C, ring, inp.get("sink"), self.rope, self.out, lse, self.ws,
                       stream)
        return self.out


def to_device(inp: dict, device="cuda", non_blocking=False) -> dict:
    return {k: (v.to(device, non_blocking=non_blocking) if isinstance(v, torch.Tensor) else v)
            for k, v in inp.items()}


class Projections:
    """The projections on either side of one attention layer, as library GEMM calls (plumbing:
    buffers and the call sequence). inputs(): hidden states -> q, kv (BF16) and, for CSA, the
    indexer queries, indexer key, weights and compression logits (FP32; HCA: the logits only),
    each its own contiguous tensor. output(): the attention output -> the grouped output
    projection -> the hidden size."""

    def __init__(self, wl, csa: bool, weights: dict, device="cuda"):
        self.wl, self.csa = wl, csa
        self.W = {k: v.to(device) for k, v in weights.items() if k.startswith("W")}
        # one stacked weight per product: q | kv (BF16 outputs), the indexer inputs (FP32)
        self.W_bf16 = torch.cat([self.W["Wq"], self.W["Wkv"]]).contiguous()
        self.device = device

    def inputs(self, x: torch.Tensor, stream=None) -> dict:
        from . import csa_gemm_bf16
        wl, rows = self.wl, x.shape[0]
        dev = self.device
        q = torch.empty((rows, wl.H, wl.d), dtype=torch.bfloat16, device=dev)
        kv = torch.empty((rows, wl.d), dtype=torch.bfloat16, device=dev)
        nq = wl.H * wl.d
        csa_gemm_bf16(x, self.W_bf16, [(q.view(rows, nq), 0, nq), (kv, nq, nq + wl.d)], stream=stream)
        out = {"q": q, "kv": kv}
        z = torch.empty((rows, 2), dtype=torch.float32, device=dev)
        if self.csa:
            ni = wl.H_I * wl.d_I
            qI = torch.empty((rows, wl.H_I, wl.d_I), dtype=torch.float32, device=dev)
            kI = torch.empty((rows, wl.d_I), dtype=torch.float32, device=dev)
            w = torch.empty((rows, wl.H_I), dtype=torch.float32, device=dev)
            segs = [(qI.view(rows, ni), 0, ni), (kI, ni, ni + wl.d_I), (w, ni + wl.d_I, ni + wl.d_I + wl.H_I),
                    (z, ni + wl.d_I + wl.H_I, ni + wl.d_I + wl.H_I + 2)]
            csa_gemm_bf16(x, self.W["Widx"], segs, stream=stream)
            out.update(qI=qI, kI_raw=kI, w=w)
        else:
            csa_gemm_bf16(x, self.W["Widx"], [(z, 0, 2)], stream=stream)
        out["z"] = z
        return out

    def output(self, o: torch.Tensor, stream=None) -> torch.Tensor:
        """o [rows, H, d] BF16 -> [rows, hidden] BF16 through the grouped projection."""
        from . import csa_gemm_bf16
        wl, rows = self.wl, o.shape[0]
        y = torch.empty((rows, wl.groups * wl.d_g), dtype=torch.bfloat16, device=self.device)
        csa_gemm_bf16(o.view(rows, wl.H * wl.d), self.W["Wg"], [(y, 0, y.shape[1])], groups=wl.groups, stream=stream)
        h = torch.empty((rows, wl.hidden), dtype=torch.bfloat16, device=self.device)
        csa_gemm_bf16(y, self.W["Wo"], [(h, 0, wl.hidden)], stream=stream)
        return h
