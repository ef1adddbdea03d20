"""The C ABI on the host (CPU only): the library loads, exports every function that
include/csa.h declares, and rejects bad arguments before launching anything."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _header_functions():
    text = open(os.path.join(ROOT, "include", "csa.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", text, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "return")))


@pytest.fixture(scope="module")
def csa():
    from long_context_compressed_14_b300 import build
    build.build()
    import long_context_compressed_14_b300 as m
    return m


def test_header_declares_the_boundary():
    fns = _header_functions()
    for name in ["kv_compress", "csa_prefill", "csa_decode", "hca_prefill", "hca_decode", "csa_index_topk",
                 "csa_quant_fp8_rows", "csa_rope_table", "csa_workspace_bytes", "csa_device_status"]:
        assert name in fns


def test_library_exports_every_declared_symbol(csa):
    lib = ctypes.CDLL(csa.LIB_PATH)
    missing = [f for f in _header_functions() if not hasattr(lib, f)]
    assert not missing, missing


def _p(csa, **kw):
    base = dict(B=1, L=2048, H=8, m=4, topk=32, H_I=4, act="f32", kv="f32", idx="f32")
    base.update(kw)
    return csa.make_params(**base)


def test_valid_params_pass(csa):
    for op in range(5):
        assert csa.csa_check_params(_p(csa), op) == csa.OK


@pytest.mark.parametrize("field,value,code", [
    ("d", 64, 3), ("d_rope", 32, 3), ("H", 65, 3), ("m", 0, 1), ("m", 2048, 3), ("B", 0, 1), ("L", 0, 1),
    ("n_win", 0, 1), ("act_t", 2, 1), ("kv_t", 2, 1), ("scale", 0.0, 1), ("rope_len", 100, 1),
])
def test_bad_params_rejected(csa, field, value, code):
    p = _p(csa)
    setattr(p, field, value)
    assert csa.csa_check_params(p, csa.OP_CSA_PREFILL) == code


def test_csa_only_fields(csa):
    p = _p(csa, topk=4096)
    assert csa.csa_check_params(p, csa.OP_CSA_PREFILL) == csa.ERR_UNSUPPORTED
    assert csa.csa_check_params(p, csa.OP_HCA_PREFILL) == csa.OK  # HCA ignores topk
    p = _p(csa, H_I=17)
    assert csa.csa_check_params(p, csa.OP_CSA_PREFILL) == csa.ERR_UNSUPPORTED
    p = _p(csa, kv="mixed", d_rope=0)
    assert csa.csa_check_params(p, csa.OP_HCA_PREFILL) == csa.ERR_INVALID


def test_workspace_sizes(csa):
    p = _p(csa)
    n = csa.csa_workspace_bytes(p, csa.OP_CSA_PREFILL)
    # scores of the whole sequence (2048 x 512 floats) plus the top-k indices
    assert n >= 2048 * 512 * 4 + 2048 * 32 * 4
    assert csa.csa_workspace_bytes(p, csa.OP_HCA_PREFILL) == 0
    big = csa.make_params(B=1, L=262144, H=64, m=4, topk=1024)
    nb = csa.csa_workspace_bytes(big, csa.OP_CSA_PREFILL)
    # the FP8 indexer keeps per-row candidate lists (48 KB per row at this length; rows are
    # chunked past 16 GiB): never the 34 GB score matrix (the top-k indices themselves are 1 GiB)
    assert nb < 18 * 2 ** 30
    with pytest.raises(csa.CsaError):
        csa.csa_workspace_bytes(_p(csa, d=96), csa.OP_CSA_PREFILL)


def test_null_pointers_rejected_before_launch(csa):
    # No CUDA call happens on these paths, so they run without a GPU.
    lib = csa._load()
    p = _p(csa)
    assert lib.csa_prefill(ctypes.byref(p), None, None, None, None, None, None, None, None, None, None, None,
                           None, 0, None) == csa.ERR_INVALID
    assert lib.hca_prefill(ctypes.byref(p), None, None, None, None, None, None, None, None, 0, None) == csa.ERR_INVALID
    assert lib.kv_compress(ctypes.byref(p), None, None, None, None, None, None, None, None) == csa.ERR_INVALID
    assert lib.csa_decode(ctypes.byref(p), None, None, None, None, None, None, None, None, None, None, None, None,
                          None, 0, None) == csa.ERR_INVALID
    assert lib.csa_quant_fp8_rows(None, 4, 64, None, None, None) == csa.ERR_INVALID
    assert lib.csa_rope_table(None, 16, 64, 1e4, None) == csa.ERR_INVALID
    assert lib.csa_prefill(None, None, None, None, None, None, None, None, None, None, None, None, None, 0,
                           None) == csa.ERR_INVALID
    # misaligned pointers are rejected too
    fake = ctypes.c_void_p(0x1000 + 8)
    ok = ctypes.c_void_p(0x1000)
    assert lib.hca_prefill(ctypes.byref(p), fake, ok, None, None, None, ok, None, None, 0, None) == csa.ERR_INVALID


def test_workspace_too_small_rejected(csa):
    lib = csa._load()
    p = _p(csa)
    fake = ctypes.c_void_p(0x10000)
    E = csa.Entries(0x10000, None, None)
    R = csa.IndexRows(0x10000, None)
    s = lib.csa_prefill(ctypes.byref(p), fake, fake, ctypes.byref(E), ctypes.byref(R), ctypes.byref(R), fake, None,
                        fake, None, fake, None, fake, 16, None)
    assert s == csa.ERR_WORKSPACE


def test_strerror(csa):
    assert csa.csa_strerror(0) == "ok"
    assert "workspace" in csa.csa_strerror(csa.ERR_WORKSPACE)
