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

from . import (FP8E4M3, MIXED, OP_CSA_DECODE, OP_CSA_PREFILL, OP_HCA_DECODE, OP_HCA_PREFILL, Params,
               alloc_entries, alloc_index_rows, alloc_workspace, csa_decode, csa_prefill,
               csa_quant_fp8_rows, hca_decode, hca_prefill, kv_compress, make_params, rope_table,
               torch_dtype)


def layer_params(wl, csa: bool) -> Params:
    """csa_params of one layer of a workload (see synth.Workload)."""
    m = wl.m if csa else wl.m_hca
    return make_params(B=wl.B, L=wl.L, H=wl.H, m=m, topk=wl.topk if csa else 0, n_win=wl.n_win,
                       H_I=wl.H_I, d_I=wl.d_I, d=wl.d, d_rope=wl.d_rope, act=wl.q_t, kv=wl.c_t,
                       idx=wl.idx_t if csa else "f32")


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
            if p.idx_t == FP8E4M3:
                csa_quant_fp8_rows(inp["qI"], self.qI[0], self.qI[1], stream)
                qI = self.qI
            else:
                qI = (inp["qI"], None)
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
        first d - d_rope dims as FP8 codes with one scale per entry, the RoPE dims as they are);
        other entry caches and the ring are used as given."""
        self.C = None
        if self.p.kv_t == MIXED:
            C = inp["C"]
            nope = self.p.d - self.p.d_rope
            codes = torch.empty(C.shape[:-1] + (nope,), dtype=torch.uint8, device=C.device)
            scales = torch.empty(C.shape[:-1], dtype=torch.float32, device=C.device)
            csa_quant_fp8_rows(C[..., :nope].float().contiguous(), codes, scales, stream)
            self.C = (codes, C[..., nope:].to(torch.bfloat16).contiguous(), scales)
        if self.csa:
            if self.p.idx_t == FP8E4M3:
                csa_quant_fp8_rows(inp["KI"], self.KI[0], self.KI[1], stream)
            else:
                self.KI = (inp["KI"], None)

    def run(self, inp: dict, stream=None, want_lse: bool = False, want_topk: bool = True) -> torch.Tensor:
        p = self.p
        lse = self.lse if want_lse else None
        if getattr(self, "C", None) is not None:
            C = self.C
        else:
            C = inp["C"] if isinstance(inp["C"], (tuple, list)) else (inp["C"], None, None)
        if self.csa:
            if p.idx_t == FP8E4M3:
                csa_quant_fp8_rows(inp["qI"], self.qI[0], self.qI[1], stream)
                qI = self.qI
            else:
                qI = (inp["qI"], None)
            csa_decode(p, inp["q"], inp["ctx"], C, qI, self.KI, inp["w"], inp["ring"], inp.get("sink"), self.rope,
                       self.topk if want_topk else None, self.out, lse, self.ws, stream)
        else:
            hca_decode(p, inp["q"], inp["ctx"], C, inp["ring"], inp.get("sink"), self.rope, self.out, lse, self.ws,
                       stream)
        return self.out


def to_device(inp: dict, device="cuda", non_blocking=False) -> dict:
    return {k: (v.to(device, non_blocking=non_blocking) if isinstance(v, torch.Tensor) else v)
            for k, v in inp.items()}
