"""Incremental decode state on the GPU (kv_append, through the C ABI): a prefill of L0 tokens
hands over to decode, then every further token is appended and decoded one at a time. Each
decoded row must equal the oracle's prefill row of the whole sequence at that position (the
cache conventions and the append path pinned together), and the compressed caches built by the
appends must equal the oracle's compression of the whole sequence."""
import math

import numpy as np
import pytest
import torch

import oracle
import synth
from _helpers import attention_on_gpu_selection, check_topk_by_score, np64, oracle_prefill, rel_l2, unpack_nvfp4

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("csa,c_t,w_t,L0,L1", [
    (True, "bf16", "", 301, 363),    # CSA m = 4: a block completes every 4 appends
    (True, "mixed", "", 255, 300),
    (False, "bf16", "", 200, 400),   # HCA m' = 128: blocks complete at 255 and 383
    (True, "nvfp4", "fp8", 301, 350),  # the V4.1 cache: NVFP4 entries, FP8 window ring
    (False, "nvfp4", "fp8", 200, 300),
])
def test_prefill_then_append_decode_continuity(lib, csa, c_t, w_t, L0, L1):
    from long_context_compressed_14_b300.pipeline import layer_params
    if csa:
        wl = synth.WORKLOADS["csa_bf16_4x32768"].replace(B=1, L=L1, topk=64, c_t=c_t, w_t=w_t)
    else:
        wl = synth.WORKLOADS["hca_bf16_L16384"].replace(B=1, L=L1, H=64, c_t=c_t, w_t=w_t)
    m = wl.m if csa else wl.m_hca
    inp = synth.prefill_layer(wl, csa=csa)
    d = {k: v.cuda() for k, v in inp.items()}
    p = layer_params(wl, csa)                      # capacity L1
    p0 = layer_params(wl.replace(L=L0), csa)       # the prefill part
    rope = lib.rope_table(p)
    C = lib.alloc_entries(p)
    ncap = math.ceil(L1 / m)
    KI = lib.alloc_index_rows(p, (1, ncap)) if csa else None
    kv_rope = torch.empty((1, L0, 128), dtype=torch.bfloat16, device="cuda")
    # prefill: entries of the first L0 tokens (B = 1, so they are a prefix of the capacity cache)
    lib.kv_compress(p0, d["kv"][:, :L0].contiguous(), d["z"][:, :L0].contiguous(),
                    d["kI_raw"][:, :L0].contiguous() if csa else None, rope, C, KI, kv_rope)
    # hand-over: the window ring from kv_rope (an FP8 ring through the library's quantiser), the
    # state cache from the last 2m raw tokens
    ring = torch.zeros((1, wl.n_win, 128), dtype=torch.bfloat16, device="cuda")
    for u in range(max(0, L0 - wl.n_win), L0):
        ring[0, u % wl.n_win] = kv_rope[0, u]
    if w_t == "fp8":
        ring8 = lib.alloc_ring(p)
        lib.csa_quant_fp8_window_rows(ring.float().contiguous(), ring8)
        ring = ring8
    st_kv = torch.zeros((1, 2 * m, 128), dtype=torch.bfloat16, device="cuda")
    st_z = torch.zeros((1, 2 * m, 2), dtype=torch.float32, device="cuda")
    st_kI = torch.zeros((1, 2 * m, 64), dtype=torch.float32, device="cuda") if csa else None
    for u in range(max(0, L0 - 2 * m), L0):
        st_kv[0, u % (2 * m)] = d["kv"][0, u]
        st_z[0, u % (2 * m)] = d["z"][0, u]
        if csa:
            st_kI[0, u % (2 * m)] = d["kI_raw"][0, u]
    ws = lib.alloc_workspace(p, lib.OP_CSA_DECODE if csa else lib.OP_HCA_DECODE)
    n = L1 - L0
    out = torch.empty((n, 64, 128), dtype=torch.bfloat16, device="cuda")
    idx = torch.empty((n, wl.topk), dtype=torch.int32, device="cuda") if csa else None
    qI = lib.alloc_index_rows(p, (1, wl.H_I)) if csa else None
    for i, u in enumerate(range(L0, L1)):
        ctx = torch.tensor([u + 1], dtype=torch.int32, device="cuda")
        lib.kv_append(p, d["kv"][:, u].contiguous(), d["z"][:, u].contiguous(),
                      d["kI_raw"][:, u].contiguous() if csa else None, ctx, rope, ring, st_kv, st_z, st_kI, C, KI)
        q = d["q"][:, u].contiguous()
        if csa:
            lib.csa_quant_fp8_rows(d["qI"][:, u].contiguous(), qI[0], qI[1])
            lib.csa_decode(p, q, ctx, C, qI, KI, d["w"][:, u].contiguous(), ring, d["sink"], rope, idx[i:i + 1],
                           out[i:i + 1], None, ws)
        else:
            lib.hca_decode(p, q, ctx, C, ring, d["sink"], rope, out[i:i + 1], None, ws)
    torch.cuda.synchronize()
    assert lib.csa_device_status() == 0

    rows = np.arange(L0, L1)
    # the oracle's window rows stored as the ring stores them
    res = oracle_prefill(wl, inp, 0, rows, csa=csa, w_store="fp8" if w_t == "fp8" else None)
    got = np64(out)
    if csa:
        gidx = idx.cpu().numpy()
        frac = check_topk_by_score(gidx, res["scores"], rows, m, wl.topk)
        assert frac >= 0.95, frac
        o_own = attention_on_gpu_selection(wl, res, np64(inp["q"][0][rows]), gidx, rows, np64(inp["sink"]))
        assert rel_l2(got, o_own) <= 2e-2
    assert rel_l2(got, res["o"]) <= 2e-2

    # the caches the appends completed equal the oracle's compression of the whole sequence
    full = L1 // m
    comp = res["comp"]
    if c_t == "mixed":
        # (entries past the appended ones were never written: only the first `full` are read)
        gc = np.concatenate([oracle.dequant_fp8(C[0][0][:full].cpu().numpy(), C[2][0][:full].cpu().numpy()),
                             np64(C[1][0][:full])], axis=1)
        assert rel_l2(gc, comp["C"][:full]) < 1e-2
    elif c_t == "nvfp4":
        gc, gb, gs, _ = unpack_nvfp4(C[0][0][:full])
        oc, ob, os_ = comp["C_raw"]
        assert np.mean(gc == oc[:full]) >= 0.99 and np.mean(gb == ob[:full]) >= 0.99
        np.testing.assert_allclose(gs, os_[:full], rtol=1e-6)
        assert rel_l2(oracle.dequant_nvfp4(gc, gb, gs), comp["C"][:full]) < 2e-2
    else:
        np.testing.assert_allclose(np64(C[0][0][:full]), comp["C"][:full], rtol=2 ** -7, atol=4e-6)
    if csa:
        gk = oracle.dequant_fp8(KI[0][0][:full].cpu().numpy(), KI[1][0][:full].cpu().numpy())
        assert rel_l2(gk, comp["KI"][:full]) < 1e-2
