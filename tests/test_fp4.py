"""The FP4 (MXFP4) indexer on the GPU through the C ABI: the quantiser bit for bit against the
oracle's codec, the indexer + top-k by score against the oracle's double-precision scores of the
dequantised rows, a CSA prefill layer and compressed indexer keys in MXFP4.

Tolerances as in test_gpu_parity: the MXFP4 codes from identical float inputs are bit-exact
(one codec definition, the same float inputs); the selection is judged by score; outputs
relative-L2 <= 2e-2."""
import math

import numpy as np
import pytest
import torch

import oracle
import synth
from _helpers import check_csa_rows, check_topk_by_score, np64, oracle_prefill, rel_l2

pytestmark = pytest.mark.gpu


def test_quant_mxfp4_rows_bit_exact(lib):
    g = torch.Generator().manual_seed(8)
    x = torch.randn((3000, 64), generator=g) * torch.exp(torch.randn((3000, 1), generator=g) * 4)
    x[:, 32:] *= torch.exp2(torch.randint(-12, 12, (3000, 1), generator=g).float())
    x[7] = 0.0                  # a zero row
    x[8, :32] = 0.0             # one zero block
    x[9, 3] = 1e30              # a huge element
    x[10, 40] = -5.0 * 2 ** -3  # an exact midpoint of the E2M1 grid after scaling
    codes = torch.empty((3000, 32), dtype=torch.uint8, device="cuda")
    e8 = torch.empty((3000, 2), dtype=torch.uint8, device="cuda")
    lib.csa_quant_mxfp4_rows(x.cuda(), codes, e8)
    oc, oe = oracle.quant_rows_mxfp4(x.numpy())
    np.testing.assert_array_equal(e8.cpu().numpy(), oe)
    np.testing.assert_array_equal(codes.cpu().numpy(), oc)


def test_index_topk_mxfp4(lib):
    L, m, H_I, k = 20000, 4, 8, 512  # rows past 16384 take the sampled threshold
    g = torch.Generator().manual_seed(12)
    N = L // m
    qI = torch.randn((1, L, H_I, 64), generator=g)
    KI = torch.randn((1, N, 64), generator=g)
    w = torch.randn((1, L, H_I), generator=g)
    p = lib.make_params(B=1, L=L, H=64, m=m, topk=k, H_I=H_I, act="bf16", kv="bf16", idx="mxfp4")
    qd = lib.alloc_index_rows(p, (1, L, H_I))
    kd = lib.alloc_index_rows(p, (1, N))
    lib.csa_quant_mxfp4_rows(qI.cuda(), qd[0], qd[2])
    lib.csa_quant_mxfp4_rows(KI.cuda(), kd[0], kd[2])
    out = torch.empty((1, L, k), dtype=torch.int32, device="cuda")
    lib.csa_index_topk(p, qd, kd, w.cuda(), out, lib.alloc_workspace(p, lib.OP_INDEX_TOPK))
    torch.cuda.synchronize()
    assert lib.csa_device_status() == 0
    kc, ke = oracle.quant_rows_mxfp4(KI[0].numpy())
    rows = np.unique(np.concatenate([np.arange(0, 60), np.arange(16370, 16400), np.arange(L - 30, L),
                                     np.random.default_rng(1).integers(0, L, 40)]))
    s, _ = oracle.indexer_topk(qI[0].numpy()[rows], oracle.dequant_mxfp4(kc, ke), w[0].numpy()[rows], m, k, rows,
                               "mxfp4")
    frac = check_topk_by_score(out.cpu().numpy()[0][rows], s, rows, m, k)
    assert frac >= 0.95, frac


@pytest.mark.parametrize("L", [3001, 1030])
def test_csa_prefill_mxfp4_indexer(lib, L):
    # the whole CSA layer with the indexer in MXFP4: compression writes the FP4 keys, the queries
    # are quantised by the library, attention checked twice on every sampled row
    wl = synth.WORKLOADS["csa_bf16_4x32768"].replace(B=1, L=L, topk=64, idx_t="mxfp4")
    from long_context_compressed_14_b300.pipeline import PrefillLayer
    inp = synth.prefill_layer(wl, csa=True)
    layer = PrefillLayer.create(wl, csa=True)
    out = layer.run({k: v.cuda() for k, v in inp.items()})
    torch.cuda.synchronize()
    assert lib.csa_device_status() == 0
    rows = synth.sample_rows(L, 256, seed=3).numpy()
    res = oracle_prefill(wl, inp, 0, rows, csa=True)
    gidx = layer.topk.cpu().numpy()[0][rows]
    frac = check_topk_by_score(gidx, res["scores"], rows, wl.m, wl.topk)
    assert frac >= 0.95, frac
    check_csa_rows(wl, inp, 0, rows, np64(out[0][rows]), gidx, res)
    # compressed indexer keys: FP4 codes of the float keys (the float sums of the GPU and the
    # double sums of the oracle may sit on either side of a rounding boundary now and then)
    N = math.ceil(L / wl.m)
    gk = oracle.dequant_mxfp4(layer.KI[0][0].cpu().numpy(), layer.KI[2][0].cpu().numpy())
    assert gk.shape == (N, 64)
    same = np.mean(gk == res["comp"]["KI"])
    assert same >= 0.99, same
    assert rel_l2(gk, res["comp"]["KI"]) < 2e-2
