"""Hybrid compressed attention (CSA / HCA) on B300: Python binding of libcsa.so.

Every call forwards to the C ABI declared in include/csa.h under the same name; this module
only marshals torch tensors to pointers and raises on a non-zero status. All compute runs in
the CUDA kernels of libcsa.so -- there is no Python or CPU fallback: the first call without
the built library raises ImportError, and calls need CUDA tensors. (The library is loaded on
first use so that `python -m long_context_compressed_14_b300.build` can (re)build it.)

Sources of the method: "DeepSeek-V4: Towards Highly Efficient Million-Token Context
Intelligence" (wiki notes), 提案手法 §1 and 訓練インフラの革新 §5; "deepseek V4 技术论文" 一.1.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libcsa.so")

# csa_dtype
F32, BF16, FP8E4M3, MIXED, MXFP4, NVFP4 = 0, 1, 2, 3, 4, 5
NVFP4_ROW_BYTES = 80      # an NVFP4 entry row (layout in include/csa.h, csa_entries)
FP8_WIN_ROW_BYTES = 144   # an FP8 window-ring row (layout in include/csa.h)
# csa_op
OP_INDEX_TOPK, OP_CSA_PREFILL, OP_HCA_PREFILL, OP_CSA_DECODE, OP_HCA_DECODE, OP_SPARSE_ATTENTION = range(6)
# csa_status
OK, ERR_INVALID, ERR_WORKSPACE, ERR_UNSUPPORTED, ERR_LAUNCH, ERR_TIMEOUT, ERR_BOUNDS, ERR_CUDA = range(8)

_DT = {"f32": F32, "bf16": BF16, "fp8": FP8E4M3, "mixed": MIXED, "mxfp4": MXFP4, "nvfp4": NVFP4}


class CsaError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {csa_strerror(status)} (status {status})")


class Params(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in ("B", "L", "H", "d", "d_rope", "m", "topk", "n_win", "H_I", "d_I")] + \
               [("scale", ctypes.c_float)] + \
               [(n, ctypes.c_int) for n in ("act_t", "kv_t", "idx_t", "rope_len", "win_t")]


class Entries(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("rope", ctypes.c_void_p), ("scale", ctypes.c_void_p)]


class GemmOut(ctypes.Structure):
    _fields_ = [("ptr", ctypes.c_void_p), ("ld", ctypes.c_int64), ("col0", ctypes.c_int), ("col1", ctypes.c_int),
                ("dtype", ctypes.c_int)]


class IndexRows(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("scale", ctypes.c_void_p), ("mx_scale", ctypes.c_void_p)]


_lib = None


def _load():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"libcsa.so is not built ({LIB_PATH}); run "
                              "`python -m long_context_compressed_14_b300.build`")
        lib = ctypes.CDLL(LIB_PATH)
        P, I, I64, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
        PP = ctypes.POINTER(Params)
        PE = ctypes.POINTER(Entries)
        PI = ctypes.POINTER(IndexRows)
        sig = {
            "csa_strerror": (ctypes.c_char_p, [I]),
            "csa_version": (I, []),
            "csa_workspace_bytes": (Z, [PP, I]),
            "csa_check_params": (I, [PP, I]),
            "csa_rope_table": (I, [P, I, I, ctypes.c_float, P]),
            "csa_quant_fp8_rows": (I, [P, I64, I, P, P, P]),
            "csa_quant_mxfp4_rows": (I, [P, I64, I, P, P, P]),
            "csa_quant_nvfp4_entries": (I, [P, I64, P, P]),
            "csa_quant_fp8_window_rows": (I, [P, I64, P, P]),
            "kv_compress": (I, [PP, P, P, P, P, PE, PI, P, P]),
            "kv_append": (I, [PP, P, P, P, P, P, P, P, P, P, PE, PI, P]),
            "csa_index_topk": (I, [PP, PI, PI, P, P, P, Z, P]),
            "csa_prefill": (I, [PP, P, P, PE, PI, PI, P, P, P, P, P, P, P, Z, P]),
            "hca_prefill": (I, [PP, P, P, PE, P, P, P, P, P, Z, P]),
            "csa_decode": (I, [PP, P, P, PE, PI, PI, P, P, P, P, P, P, P, P, Z, P]),
            "hca_decode": (I, [PP, P, P, PE, P, P, P, P, P, P, Z, P]),
            "csa_sparse_attention": (I, [PP, P, P, PE, P, P, P, P, P, P, ctypes.c_size_t, P]),
            "csa_decode_static_scratch": (I, [PP, P, P, PE, PI, PI, P, P, P, P, P, P, P, P]),
            "csa_launch_count": (ctypes.c_uint64, []),
            "csa_gemm_bf16": (I, [P, I64, P, I64, I, I, I, I, ctypes.POINTER(GemmOut), I, P]),
            "csa_device_status": (I, [ctypes.POINTER(ctypes.c_int), I, P]),
            "csa_selftest_wait_timeout": (I, [ctypes.c_uint64, P]),
            "csa_probe_ffma": (I, [I, I, P, P]),
            "csa_probe_read": (I, [P, I64, I, I, P, P]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib




def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError("expected a torch.Tensor")
    if not t.is_contiguous():
        raise ValueError("tensors passed to libcsa must be contiguous")
    return t.data_ptr()


def _nbytes(t: Optional[torch.Tensor]) -> int:
    return 0 if t is None else t.numel() * t.element_size()


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream if torch.cuda.is_available() else None
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else stream


def _ok(status: int, what: str):
    if status != OK:
        raise CsaError(status, what)


def _entries(C: Optional[Sequence]) -> Optional[Entries]:
    if C is None:
        return None
    data, rope, scale = (list(C) + [None, None, None])[:3]
    return Entries(_ptr(data), _ptr(rope), _ptr(scale))


def _rows(R: Optional[Sequence]) -> Optional[IndexRows]:
    if R is None:
        return None
    data, scale, mx = (list(R) + [None, None, None])[:3]
    return IndexRows(_ptr(data), _ptr(scale), _ptr(mx))


def _byref(x):
    return None if x is None else ctypes.byref(x)


# ---------------------------------------------------------------------------------------
# The C ABI, same names
# ---------------------------------------------------------------------------------------

def csa_strerror(status: int) -> str:
    return _load().csa_strerror(status).decode()


def csa_version() -> int:
    return _load().csa_version()


def csa_workspace_bytes(p: Params, op: int) -> int:
    n = _load().csa_workspace_bytes(ctypes.byref(p), op)
    if n == ctypes.c_size_t(-1).value:
        raise CsaError(ERR_INVALID, "csa_workspace_bytes")
    return n


def csa_check_params(p: Params, op: int) -> int:
    return _load().csa_check_params(ctypes.byref(p), op)


def csa_rope_table(tab: torch.Tensor, rope_len: int, d_rope: int, theta: float, stream=None):
    _ok(_load().csa_rope_table(_ptr(tab), rope_len, d_rope, theta, _stream(stream)), "csa_rope_table")


def csa_quant_fp8_rows(x: torch.Tensor, codes: torch.Tensor, scales: torch.Tensor, stream=None):
    rows = x.numel() // x.shape[-1]
    _ok(_load().csa_quant_fp8_rows(_ptr(x), rows, x.shape[-1], _ptr(codes), _ptr(scales), _stream(stream)),
        "csa_quant_fp8_rows")


def csa_quant_mxfp4_rows(x: torch.Tensor, codes: torch.Tensor, e8: torch.Tensor, stream=None):
    rows = x.numel() // x.shape[-1]
    _ok(_load().csa_quant_mxfp4_rows(_ptr(x), rows, x.shape[-1], _ptr(codes), _ptr(e8), _stream(stream)),
        "csa_quant_mxfp4_rows")


def csa_quant_nvfp4_entries(x: torch.Tensor, out: torch.Tensor, stream=None):
    """x [.., 128] float -> NVFP4 entry rows out [.., 80] uint8."""
    rows = x.numel() // x.shape[-1]
    if x.shape[-1] != 128 or out.numel() != rows * NVFP4_ROW_BYTES:
        raise ValueError("csa_quant_nvfp4_entries: x [.., 128] float, out [.., 80] uint8")
    _ok(_load().csa_quant_nvfp4_entries(_ptr(x), rows, _ptr(out), _stream(stream)), "csa_quant_nvfp4_entries")


def csa_quant_fp8_window_rows(x: torch.Tensor, out: torch.Tensor, stream=None):
    """x [.., 128] float -> FP8 window rows out [.., 144] uint8."""
    rows = x.numel() // x.shape[-1]
    if x.shape[-1] != 128 or out.numel() != rows * FP8_WIN_ROW_BYTES:
        raise ValueError("csa_quant_fp8_window_rows: x [.., 128] float, out [.., 144] uint8")
    _ok(_load().csa_quant_fp8_window_rows(_ptr(x), rows, _ptr(out), _stream(stream)), "csa_quant_fp8_window_rows")


def kv_compress(p: Params, kv, z, kI_raw, rope_tab, C, KI, kv_rope, stream=None):
    _ok(_load().kv_compress(ctypes.byref(p), _ptr(kv), _ptr(z), _ptr(kI_raw), _ptr(rope_tab),
                            _byref(_entries(C)), _byref(_rows(KI)), _ptr(kv_rope), _stream(stream)),
        "kv_compress")


def kv_append(p: Params, kv_new, z_new, kI_new, ctx_len, rope_tab, ring, state_kv, state_z, state_kI, C, KI,
              stream=None):
    _ok(_load().kv_append(ctypes.byref(p), _ptr(kv_new), _ptr(z_new), _ptr(kI_new), _ptr(ctx_len), _ptr(rope_tab),
                          _ptr(ring), _ptr(state_kv), _ptr(state_z), _ptr(state_kI), _byref(_entries(C)),
                          _byref(_rows(KI)), _stream(stream)),
        "kv_append")


def csa_index_topk(p: Params, qI, KI, w, topk_out, ws, stream=None):
    _ok(_load().csa_index_topk(ctypes.byref(p), _byref(_rows(qI)), _byref(_rows(KI)), _ptr(w), _ptr(topk_out),
                               _ptr(ws), 0 if ws is None else ws.numel() * ws.element_size(), _stream(stream)),
        "csa_index_topk")


def csa_prefill(p: Params, q, kv_rope, C, qI, KI, w, sink, rope_tab, topk_out, out, lse_out, ws, stream=None):
    _ok(_load().csa_prefill(ctypes.byref(p), _ptr(q), _ptr(kv_rope), _byref(_entries(C)), _byref(_rows(qI)),
                            _byref(_rows(KI)), _ptr(w), _ptr(sink), _ptr(rope_tab), _ptr(topk_out), _ptr(out),
                            _ptr(lse_out), _ptr(ws), 0 if ws is None else ws.numel() * ws.element_size(),
                            _stream(stream)),
        "csa_prefill")


def csa_sparse_attention(p: Params, q, kv_rope, C, topk_idx, sink, rope_tab, out, lse_out, ws=None, stream=None):
    _ok(_load().csa_sparse_attention(ctypes.byref(p), _ptr(q), _ptr(kv_rope), _byref(_entries(C)), _ptr(topk_idx),
                                     _ptr(sink), _ptr(rope_tab), _ptr(out), _ptr(lse_out), _ptr(ws), _nbytes(ws),
                                     _stream(stream)),
        "csa_sparse_attention")


def csa_gemm_bf16(A: torch.Tensor, B: torch.Tensor, outs, groups: int = 1, stream=None):
    """C = A B^T on the tensor cores (BF16 in, FP32 accumulate). A [M, groups*K], B [N, K] BF16;
    outs: list of (tensor, col0, col1): columns [col0, col1) of C into that row-major tensor
    (BF16 or FP32, rows of col1 - col0 values)."""
    M, N, K = A.shape[0], B.shape[0], B.shape[1]
    arr = (GemmOut * len(outs))()
    for i, (t, c0, c1) in enumerate(outs):
        arr[i] = GemmOut(_ptr(t), t.shape[-1], c0, c1, _DT["f32" if t.dtype == torch.float32 else "bf16"])
    _ok(_load().csa_gemm_bf16(_ptr(A), A.stride(0), _ptr(B), B.stride(0), M, N, K, groups, arr, len(outs),
                              _stream(stream)), "csa_gemm_bf16")


def csa_launch_count() -> int:
    return int(_load().csa_launch_count())


def hca_prefill(p: Params, q, kv_rope, C, sink, rope_tab, out, lse_out, ws, stream=None):
    _ok(_load().hca_prefill(ctypes.byref(p), _ptr(q), _ptr(kv_rope), _byref(_entries(C)), _ptr(sink),
                            _ptr(rope_tab), _ptr(out), _ptr(lse_out), _ptr(ws),
                            0 if ws is None else ws.numel() * ws.element_size(), _stream(stream)),
        "hca_prefill")


def csa_decode(p: Params, q, ctx_len, C, qI, KI, w, swa_ring, sink, rope_tab, topk_out, out, lse_out, ws,
               stream=None):
    _ok(_load().csa_decode(ctypes.byref(p), _ptr(q), _ptr(ctx_len), _byref(_entries(C)), _byref(_rows(qI)),
                           _byref(_rows(KI)), _ptr(w), _ptr(swa_ring), _ptr(sink), _ptr(rope_tab),
                           _ptr(topk_out), _ptr(out), _ptr(lse_out), _ptr(ws),
                           0 if ws is None else ws.numel() * ws.element_size(), _stream(stream)),
        "csa_decode")


STATIC_SCRATCH_BYTES = 8 << 20  # CSA_STATIC_SCRATCH_BYTES in include/csa.h


def csa_decode_static_scratch(p: Params, q, ctx_len, C, qI, KI, w, swa_ring, sink, rope_tab, topk_out, out, lse_out,
                              stream=None):
    """csa_decode without a workspace argument, for callers that cannot allocate device
    memory: the scratch lives in a fixed array inside the library (see include/csa.h)."""
    _ok(_load().csa_decode_static_scratch(ctypes.byref(p), _ptr(q), _ptr(ctx_len), _byref(_entries(C)),
                                          _byref(_rows(qI)), _byref(_rows(KI)), _ptr(w), _ptr(swa_ring), _ptr(sink),
                                          _ptr(rope_tab), _ptr(topk_out), _ptr(out), _ptr(lse_out), _stream(stream)),
        "csa_decode_static_scratch")


def hca_decode(p: Params, q, ctx_len, C, swa_ring, sink, rope_tab, out, lse_out, ws, stream=None):
    _ok(_load().hca_decode(ctypes.byref(p), _ptr(q), _ptr(ctx_len), _byref(_entries(C)), _ptr(swa_ring),
                           _ptr(sink), _ptr(rope_tab), _ptr(out), _ptr(lse_out), _ptr(ws),
                           0 if ws is None else ws.numel() * ws.element_size(), _stream(stream)),
        "hca_decode")


def csa_device_status(reset: bool = True, stream=None) -> int:
    """Device status word after the work queued on `stream` (0 = ok); cleared when reset."""
    v = ctypes.c_int(0)
    _ok(_load().csa_device_status(ctypes.byref(v), int(reset), _stream(stream)), "csa_device_status")
    return v.value


def csa_probe_ffma(blocks: int, iters: int, out: torch.Tensor, stream=None):
    _ok(_load().csa_probe_ffma(blocks, iters, _ptr(out), _stream(stream)), "csa_probe_ffma")


def csa_probe_read(buf: torch.Tensor, reps: int, blocks: int, out: torch.Tensor, stream=None):
    _ok(_load().csa_probe_read(_ptr(buf), _nbytes(buf), reps, blocks, _ptr(out), _stream(stream)), "csa_probe_read")


def csa_selftest_wait_timeout(limit_ns: int, stream=None):
    _ok(_load().csa_selftest_wait_timeout(int(limit_ns), _stream(stream)), "csa_selftest_wait_timeout")


# ---------------------------------------------------------------------------------------
# Small conveniences (plumbing only: parameter structs and torch allocations)
# ---------------------------------------------------------------------------------------

def make_params(*, B, L, H, m, topk=0, n_win=128, H_I=8, d_I=64, d=128, d_rope=64, scale=None,
                act="bf16", kv="bf16", idx="fp8", rope_len=None, win=None) -> Params:
    """win: the decode ring's dtype, the activation dtype (default) or "fp8"."""
    ncap = -(-L // m)
    if rope_len is None:
        rope_len = max(L, ncap * m)
    return Params(B, L, H, d, d_rope, m, topk, n_win, H_I, d_I, float(d ** -0.5 if scale is None else scale),
                  _DT[act], _DT[kv], _DT[idx], rope_len, _DT[act if win is None else win])


def torch_dtype(name: str):
    return {"f32": torch.float32, "bf16": torch.bfloat16}[name]


def alloc_entries(p: Params, device="cuda"):
    """Entry buffers for a layer: (data, rope, scale) per p.kv_t."""
    ncap = -(-p.L // p.m)
    if p.kv_t == MIXED:
        return (torch.empty((p.B, ncap, p.d - p.d_rope), dtype=torch.uint8, device=device),
                torch.empty((p.B, ncap, p.d_rope), dtype=torch.bfloat16, device=device),
                torch.empty((p.B, ncap), dtype=torch.float32, device=device))
    if p.kv_t == NVFP4:
        return (torch.empty((p.B, ncap, NVFP4_ROW_BYTES), dtype=torch.uint8, device=device), None, None)
    dt = torch.float32 if p.kv_t == F32 else torch.bfloat16
    return (torch.empty((p.B, ncap, p.d), dtype=dt, device=device), None, None)


def alloc_ring(p: Params, device="cuda") -> torch.Tensor:
    """The decode SWA ring per p.win_t: [B, n_win, d] in the activation dtype, or FP8 rows
    [B, n_win, 144] uint8."""
    if p.win_t == FP8E4M3:
        return torch.zeros((p.B, p.n_win, FP8_WIN_ROW_BYTES), dtype=torch.uint8, device=device)
    dt = torch.float32 if p.act_t == F32 else torch.bfloat16
    return torch.zeros((p.B, p.n_win, p.d), dtype=dt, device=device)


def alloc_index_rows(p: Params, rows_shape, device="cuda"):
    """Indexer operand buffers of shape rows_shape + [d_I] per p.idx_t: (data, scale) for F32 /
    FP8, (codes [.., d_I/2], None, E8M0 exponents [.., d_I/32]) for MXFP4."""
    if p.idx_t == MXFP4:
        return (torch.empty(tuple(rows_shape) + (p.d_I // 2,), dtype=torch.uint8, device=device), None,
                torch.empty(tuple(rows_shape) + (p.d_I // 32,), dtype=torch.uint8, device=device))
    if p.idx_t == FP8E4M3:
        return (torch.empty(tuple(rows_shape) + (p.d_I,), dtype=torch.uint8, device=device),
                torch.empty(tuple(rows_shape), dtype=torch.float32, device=device))
    return (torch.empty(tuple(rows_shape) + (p.d_I,), dtype=torch.float32, device=device), None)


def alloc_workspace(p: Params, op: int, device="cuda") -> Optional[torch.Tensor]:
    n = csa_workspace_bytes(p, op)
    return torch.empty(max(n, 16), dtype=torch.uint8, device=device)


def rope_table(p: Params, theta: float = 1.0e4, device="cuda", stream=None) -> torch.Tensor:
    half = max(p.d_rope // 2, 1)
    tab = torch.empty((p.rope_len, half, 2), dtype=torch.float32, device=device)
    if p.d_rope > 0:
        csa_rope_table(tab, p.rope_len, p.d_rope, theta, stream)
    return tab
