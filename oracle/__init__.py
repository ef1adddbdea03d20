"""CPU oracle for hybrid compressed attention (CSA / HCA) -- TEST INFRASTRUCTURE.

This package is the plain, slow reference the CUDA library is checked against. Only the
test-suite, the smoke check and the benchmark's CPU-baseline leg may import it; the
library never does, and the two share no code. The arithmetic lives in ``csa_oracle.c``
(double precision, see that file for the sources and the readings of each step); this
module marshals numpy arrays to it and strings the steps together in the order the method
describes them:

  compression -> (indexer score -> top-k) -> attention with sliding window and sink,
  with partial RoPE on keys/queries and inverse RoPE on the output.

Parity pins for every function are in ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "csa_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")

CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off", "-fno-fast-math"]


def build(force: bool = False) -> str:
    """Compile csa_oracle.c into oracle/_build/liboracle.so (gcc, OpenMP)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", *CFLAGS, _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


_lib = None

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_INT = ctypes.c_int
_DBL = ctypes.c_double


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        sig = {
            "orc_rope": (None, [_P, _I64, _INT, _INT, _P, _DBL, _INT]),
            "orc_num_entries": (_I64, [_I64, _INT]),
            "orc_compress": (None, [_P, _I64, _INT, _P, _INT, _P]),
            "orc_entry_pos": (_I64, [_I64, _INT]),
            "orc_visible": (_I64, [_I64, _INT, _I64]),
            "orc_round_bf16": (ctypes.c_float, [ctypes.c_float]),
            "orc_fp8_decode": (ctypes.c_float, [ctypes.c_uint8]),
            "orc_fp8_encode": (ctypes.c_uint8, [ctypes.c_float]),
            "orc_quant_rows_fp8": (None, [_P, _I64, _INT, _P, _P]),
            "orc_e2m1_decode": (_DBL, [ctypes.c_uint8]),
            "orc_e2m1_encode": (ctypes.c_uint8, [_DBL]),
            "orc_quant_rows_mxfp4": (None, [_P, _I64, _INT, _P, _P]),
            "orc_quant_rows_nvfp4": (None, [_P, _I64, _INT, _P, _P, _P]),
            "orc_index_scores_f32": (None, [_P, _P, _P, _I64, _INT, _INT, _INT, _P, _I64, _P]),
            "orc_index_scores_f64": (None, [_P, _P, _P, _I64, _INT, _INT, _INT, _P, _I64, _P]),
            "orc_topk": (None, [_P, _I64, _INT, _P, _I64, _INT, _P]),
            "orc_attend_one": (None, [_P, _INT, _INT, _P, _I64, _P, _DBL, _P, _P, _P]),
            "orc_attention_rows": (None, [_P, _P, _P, _I64, _P, _INT, _INT, _INT, _INT, _INT,
                                          _DBL, _INT, _P, _DBL, _P, _I64, _P, _P]),
            "orc_decode_one": (None, [_P, _I64, _P, _I64, _P, _INT, _INT, _P, _INT, _INT,
                                      _INT, _DBL, _INT, _P, _DBL, _P, _P]),
            "orc_num_threads": (_INT, []),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def _c(a: np.ndarray, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


def _ptr(a):
    return None if a is None else a.ctypes.data


def num_threads() -> int:
    return int(_load().orc_num_threads())


# ----------------------------------------------------------------------------------------
# Elementary steps
# ----------------------------------------------------------------------------------------

def num_entries(L: int, m: int) -> int:
    return int(_load().orc_num_entries(L, m))


def visible(t: int, m: int, N: int) -> int:
    return int(_load().orc_visible(t, m, N))


def entry_pos(N: int, m: int) -> np.ndarray:
    lib = _load()
    return np.array([lib.orc_entry_pos(j, m) for j in range(N)], dtype=np.int64)


def rope(x: np.ndarray, pos: np.ndarray, d_rope: int, theta: float, sign: int = +1) -> np.ndarray:
    """Rotate the last d_rope dims of each row of x [rows, d] by its position (copy)."""
    x = _c(x, np.float64).copy()
    rows, d = x.shape
    pos = _c(np.broadcast_to(pos, (rows,)), np.int64)
    _load().orc_rope(_ptr(x), rows, d, d_rope, _ptr(pos), float(theta), int(sign))
    return x


def compress(x: np.ndarray, z: np.ndarray, m: int) -> np.ndarray:
    """Overlapping softmax-weighted compression of x [L, dx] with logits z [L, 2]."""
    x = _c(x, np.float64)
    z = _c(z, np.float64)
    L, dx = x.shape
    N = num_entries(L, m)
    out = np.zeros((N, dx), dtype=np.float64)
    _load().orc_compress(_ptr(x), L, dx, _ptr(z), m, _ptr(out))
    return out


def round_bf16(x: np.ndarray) -> np.ndarray:
    lib = _load()
    x = _c(x, np.float32)
    flat = x.reshape(-1)
    out = np.empty_like(flat)
    for i in range(flat.size):
        out[i] = lib.orc_round_bf16(float(flat[i]))
    return out.reshape(x.shape)


def round_bf16_fast(x: np.ndarray) -> np.ndarray:
    """Vectorised twin of round_bf16 (same bit rule: RNE on the top 16 bits of binary32);
    pinned against the scalar C routine in the tests."""
    x = _c(x, np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    lower = u & 0xFFFF
    lsb = (u >> 16) & 1
    up = u & 0xFFFF0000
    bump = (lower > 0x8000) | ((lower == 0x8000) & (lsb == 1))
    up = np.where(bump, up + 0x10000, up).astype(np.uint32)
    out = up.view(np.float32)
    return np.where(np.isnan(x), x, out).astype(np.float32)


def fp8_decode(codes: np.ndarray) -> np.ndarray:
    lib = _load()
    table = np.array([lib.orc_fp8_decode(c) for c in range(256)], dtype=np.float32)
    return table[_c(codes, np.uint8)]


def fp8_encode(x: np.ndarray) -> np.ndarray:
    lib = _load()
    flat = _c(x, np.float32).reshape(-1)
    return np.array([lib.orc_fp8_encode(float(v)) for v in flat], dtype=np.uint8).reshape(np.shape(x))


def quant_rows_fp8(x: np.ndarray):
    """Per-row FP8 E4M3 quantisation -> (codes uint8 [rows, cols], scales float32 [rows])."""
    x = _c(x, np.float32)
    shp = x.shape
    x2 = x.reshape(-1, shp[-1])
    codes = np.zeros(x2.shape, dtype=np.uint8)
    scales = np.zeros(x2.shape[0], dtype=np.float32)
    _load().orc_quant_rows_fp8(_ptr(x2), x2.shape[0], x2.shape[1], _ptr(codes), _ptr(scales))
    return codes.reshape(shp), scales.reshape(shp[:-1])


def e2m1_decode(codes: np.ndarray) -> np.ndarray:
    lib = _load()
    table = np.array([lib.orc_e2m1_decode(c) for c in range(16)], dtype=np.float64)
    return table[_c(codes, np.uint8) & 15]


def e2m1_encode(x: np.ndarray) -> np.ndarray:
    lib = _load()
    flat = _c(x, np.float64).reshape(-1)
    return np.array([lib.orc_e2m1_encode(float(v)) for v in flat], dtype=np.uint8).reshape(np.shape(x))


def quant_rows_mxfp4(x: np.ndarray):
    """Per-row MXFP4 quantisation -> (codes uint8 [rows, cols/2] (element 2i in the low nibble),
    block exponents uint8 [rows, cols/32] (E8M0))."""
    x = _c(x, np.float32)
    shp = x.shape
    x2 = x.reshape(-1, shp[-1])
    codes = np.zeros((x2.shape[0], shp[-1] // 2), dtype=np.uint8)
    e8 = np.zeros((x2.shape[0], shp[-1] // 32), dtype=np.uint8)
    _load().orc_quant_rows_mxfp4(_ptr(x2), x2.shape[0], x2.shape[1], _ptr(codes), _ptr(e8))
    return codes.reshape(shp[:-1] + (shp[-1] // 2,)), e8.reshape(shp[:-1] + (shp[-1] // 32,))


def dequant_mxfp4(codes: np.ndarray, e8: np.ndarray) -> np.ndarray:
    """Values of MXFP4 rows: E2M1 element times 2^(e8 - 127) of its 32-element block."""
    codes = np.asarray(codes, np.uint8)
    elems = np.empty(codes.shape[:-1] + (codes.shape[-1] * 2,), dtype=np.uint8)
    elems[..., 0::2] = codes & 15
    elems[..., 1::2] = codes >> 4
    scale = np.exp2(np.asarray(e8, np.float64) - 127.0)
    return e2m1_decode(elems) * np.repeat(scale, 32, axis=-1)


def quant_rows_nvfp4(x: np.ndarray):
    """Per-row NVFP4 quantisation -> (codes uint8 [rows, cols/2] (element 2i in the low nibble),
    block-scale codes uint8 [rows, cols/16] (E4M3), row scales float32 [rows])."""
    x = _c(x, np.float32)
    shp = x.shape
    x2 = x.reshape(-1, shp[-1])
    codes = np.zeros((x2.shape[0], shp[-1] // 2), dtype=np.uint8)
    bcode = np.zeros((x2.shape[0], shp[-1] // 16), dtype=np.uint8)
    rs = np.zeros(x2.shape[0], dtype=np.float32)
    _load().orc_quant_rows_nvfp4(_ptr(x2), x2.shape[0], x2.shape[1], _ptr(codes), _ptr(bcode), _ptr(rs))
    return (codes.reshape(shp[:-1] + (shp[-1] // 2,)), bcode.reshape(shp[:-1] + (shp[-1] // 16,)),
            rs.reshape(shp[:-1]))


def dequant_nvfp4(codes: np.ndarray, bcode: np.ndarray, rs: np.ndarray) -> np.ndarray:
    """Values of NVFP4 rows: E2M1 element times its block's scale, the float product
    E4M3(block code) * row scale."""
    codes = np.asarray(codes, np.uint8)
    elems = np.empty(codes.shape[:-1] + (codes.shape[-1] * 2,), dtype=np.uint8)
    elems[..., 0::2] = codes & 15
    elems[..., 1::2] = codes >> 4
    scale = (fp8_decode(bcode).astype(np.float32) * np.asarray(rs, np.float32)[..., None]).astype(np.float64)
    return e2m1_decode(elems) * np.repeat(scale, 16, axis=-1)


def dequant_fp8(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    return fp8_decode(codes).astype(np.float64) * np.asarray(scales, np.float64)[..., None]


def index_scores_f32(qI_rows, KI, w_rows, m: int, pos) -> np.ndarray:
    """FP32 indexer scores in the fixed fma order.

    qI_rows [nrows,HI,dI] and w_rows [nrows,HI] are the query rows at positions pos [nrows];
    KI [N,dI]. Returns [nrows, N] float32 (-inf where not visible)."""
    qI = _c(qI_rows, np.float32)
    KI = _c(KI, np.float32)
    w = _c(w_rows, np.float32)
    pos = _c(pos, np.int64)
    nr, HI, dI = qI.shape
    N = KI.shape[0]
    s = np.zeros((nr, N), dtype=np.float32)
    _load().orc_index_scores_f32(_ptr(qI), _ptr(KI), _ptr(w), N, HI, dI, m, _ptr(pos), nr, _ptr(s))
    return s


def index_scores_f64(qI_rows, KI, w_rows, m: int, pos) -> np.ndarray:
    """Double-precision indexer scores (used with dequantised FP8 operands)."""
    qI = _c(qI_rows, np.float64)
    KI = _c(KI, np.float64)
    w = _c(w_rows, np.float64)
    pos = _c(pos, np.int64)
    nr, HI, dI = qI.shape
    N = KI.shape[0]
    s = np.zeros((nr, N), dtype=np.float64)
    _load().orc_index_scores_f64(_ptr(qI), _ptr(KI), _ptr(w), N, HI, dI, m, _ptr(pos), nr, _ptr(s))
    return s


def topk(s: np.ndarray, m: int, pos, k: int) -> np.ndarray:
    """Top-k per row of s [nrows, N] among the entries visible at pos[r]; the kept set in
    ascending index order, padded with -1."""
    s = _c(s, np.float64)
    pos = _c(pos, np.int64)
    N = s.shape[1]
    idx = np.zeros((pos.size, k), dtype=np.int32)
    if k > 0:
        _load().orc_topk(_ptr(s), N, m, _ptr(pos), pos.size, k, _ptr(idx))
    return idx


def attend_one(q, keys, sink, scale):
    """One query [H, d] (post-RoPE) over keys [nk, d]; returns (o [H, d], psum [H])."""
    q = _c(q, np.float64)
    keys = _c(keys, np.float64)
    H, d = q.shape
    nk = keys.shape[0]
    sink_a = None if sink is None else _c(sink, np.float64)
    o = np.zeros((H, d), dtype=np.float64)
    ps = np.zeros(H, dtype=np.float64)
    lg = np.zeros(max(nk, 1), dtype=np.float64)
    _load().orc_attend_one(_ptr(q), H, d, _ptr(keys), nk, _ptr(sink_a), float(scale), _ptr(o), _ptr(ps), _ptr(lg))
    return o, ps


def attention_rows(q_rows, kvr, C, idx, k, m, d_rope, theta, n_win, sink, scale, pos):
    """Attention for query rows of one sequence.

    q_rows [nrows,H,d] pre-RoPE at positions pos [nrows]; kvr [L,d] post-RoPE raw rows;
    C [N,d] post-RoPE entries; idx [nrows,k] (CSA) or None (HCA: all visible entries).
    Returns (o [nrows,H,d] after inverse RoPE, psum [nrows,H] = sum of the weights)."""
    q = _c(q_rows, np.float64)
    kvr = _c(kvr, np.float64)
    C = _c(C, np.float64) if C is not None and C.size else np.zeros((0, q.shape[2]), np.float64)
    rows = _c(pos, np.int64)
    nr, H, d = q.shape
    N = C.shape[0]
    idx_a = None if idx is None else _c(idx, np.int32)
    sink_a = None if sink is None else _c(sink, np.float64)
    o = np.zeros((rows.size, H, d), dtype=np.float64)
    ps = np.zeros((rows.size, H), dtype=np.float64)
    _load().orc_attention_rows(_ptr(q), _ptr(kvr), _ptr(C), N, _ptr(idx_a), int(k), int(m), H, d,
                               int(d_rope), float(theta), int(n_win), _ptr(sink_a), float(scale),
                               _ptr(rows), rows.size, _ptr(o), _ptr(ps))
    return o, ps


def decode_one(q, ctx, C, idx, k, m, ring, d_rope, theta, n_win, sink, scale):
    """Decode of one sequence: q [H,d] pre-RoPE, ctx = tokens incl. the new one."""
    q = _c(q, np.float64)
    C = _c(C, np.float64)
    ring = _c(ring, np.float64)
    H, d = q.shape
    idx_a = None if idx is None else _c(idx, np.int32)
    sink_a = None if sink is None else _c(sink, np.float64)
    o = np.zeros((H, d), dtype=np.float64)
    ps = np.zeros(H, dtype=np.float64)
    _load().orc_decode_one(_ptr(q), int(ctx), _ptr(C), C.shape[0], _ptr(idx_a), int(k), int(m), _ptr(ring),
                           H, d, int(d_rope), float(theta), int(n_win), _ptr(sink_a), float(scale),
                           _ptr(o), _ptr(ps))
    return o, ps


from .method import *  # noqa: E402,F401,F403  (the step-by-step pipelines)
