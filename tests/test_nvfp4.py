"""The V4.1 cache variant on the GPU through the C ABI: NVFP4 compressed entries (quantised after
RoPE) and an FP8 sliding-window ring. The quantisers bit for bit against the oracle's codecs
(one definition each, the same float inputs), and CSA / HCA prefill layers whose compression
writes NVFP4 entries, checked against the oracle with the same storage formats. Decode on these
caches is covered by test_gpu_parity.test_decode, the prefill -> append -> decode hand-over by
test_append.

Tolerances as in test_gpu_parity: codes and scales bit-exact from identical float inputs;
outputs relative-L2 <= 2e-2, checked twice on every sampled CSA row."""
import numpy as np
import pytest
import torch

import oracle
import synth
from _helpers import (check_csa_rows, check_topk_by_score, np64, oracle_prefill, rel_l2, unpack_fp8_window,
                      unpack_nvfp4)

pytestmark = pytest.mark.gpu


def _rows(n, seed):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn((n, 128), generator=g) * torch.exp(torch.randn((n, 1), generator=g) * 4)
    # blocks of very different size within a row: small blocks get subnormal or zero E4M3 scales
    x *= torch.exp2(torch.randint(-14, 4, (n, 8), generator=g).float()).repeat_interleave(16, dim=1)
    x[7] = 0.0                  # a zero row
    x[8, 16:32] = 0.0           # a zero block
    x[9, 3] = 1e30              # a huge element: every other block underflows
    x[10, :16] = torch.tensor([2688.0, 1000.0, -700.0, 224.0] + [0.0] * 12)  # the hand-worked block
    x[11, 20] = 5.0 * 2 ** -3   # an exact E2M1 midpoint of its block
    return x


def test_quant_nvfp4_entries_bit_exact(lib):
    x = _rows(3000, 21)
    out = torch.empty((3000, 80), dtype=torch.uint8, device="cuda")
    lib.csa_quant_nvfp4_entries(x.cuda(), out)
    torch.cuda.synchronize()
    gc, gb, gs, pad = unpack_nvfp4(out)
    oc, ob, os_ = oracle.quant_rows_nvfp4(x.numpy())
    np.testing.assert_array_equal(gs, os_)
    np.testing.assert_array_equal(gb, ob)
    np.testing.assert_array_equal(gc, oc)
    assert np.all(pad == 0)


def test_quant_fp8_window_rows_bit_exact(lib):
    x = _rows(2000, 22)
    out = torch.empty((2000, 144), dtype=torch.uint8, device="cuda")
    lib.csa_quant_fp8_window_rows(x.cuda(), out)
    torch.cuda.synchronize()
    gc, gs, pad = unpack_fp8_window(out)
    oc, os_ = oracle.quant_rows_fp8(x.numpy())
    np.testing.assert_array_equal(gs, os_)
    np.testing.assert_array_equal(gc, oc)
    assert np.all(pad == 0)


@pytest.mark.parametrize("csa,L", [(True, 3001), (True, 1030), (False, 2000)])
def test_prefill_nvfp4_entries(lib, csa, L):
    # the whole layer: the compression writes NVFP4 entries, the attention widens them to BF16;
    # the oracle stores its entries in NVFP4 too
    from long_context_compressed_14_b300.pipeline import PrefillLayer
    if csa:
        wl = synth.WORKLOADS["csa_bf16_4x32768"].replace(B=1, L=L, topk=64, c_t="nvfp4")
    else:
        wl = synth.WORKLOADS["hca_bf16_L16384"].replace(B=1, L=L, c_t="nvfp4")
    inp = synth.prefill_layer(wl, csa=csa)
    layer = PrefillLayer.create(wl, csa=csa)
    out = layer.run({k: v.cuda() for k, v in inp.items()})
    torch.cuda.synchronize()
    assert lib.csa_device_status() == 0
    rows = synth.sample_rows(L, 256, seed=4).numpy()
    res = oracle_prefill(wl, inp, 0, rows, csa=csa)
    if csa:
        gidx = layer.topk.cpu().numpy()[0][rows]
        frac = check_topk_by_score(gidx, res["scores"], rows, wl.m, wl.topk)
        assert frac >= 0.95, frac
        check_csa_rows(wl, inp, 0, rows, np64(out[0][rows]), gidx, res)
    else:
        assert rel_l2(np64(out[0][rows]), res["o"]) <= 2e-2
    # the entries' codes (an element or block code moves by one step where the float and double
    # sums fall on either side of a rounding boundary; the row scale by the last bits of the sum)
    gc, gb, gs, _ = unpack_nvfp4(layer.C[0][0])
    oc, ob, os_ = res["comp"]["C_raw"]
    assert np.mean(gc == oc) >= 0.99 and np.mean(gb == ob) >= 0.99
    np.testing.assert_allclose(gs, os_, rtol=1e-6)
    assert rel_l2(oracle.dequant_nvfp4(gc, gb, gs), res["comp"]["C"]) < 2e-2
