"""The allocation-free decode entry point (csa_decode_static_scratch), on the GPU.

Some callers cannot allocate device memory (their device memory belongs to another
framework's allocator, or a real-time loop must not call cudaMalloc because it can synchronise
the device), so the library offers csa_decode with its scratch in a fixed array inside the
library. These tests call it through the C ABI twice in a row and compare it with
csa_decode given a caller workspace; they also check that a layer too large for the array is
refused. This file is collected last so that a failure here comes after every other test.
"""
import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu


def _decode_setup(lib, B=4, L=8192, topk=256, c_t="bf16"):
    from long_context_compressed_14_b300.pipeline import DecodeLayer
    wl = synth.WORKLOADS["decode_b16_ctx131072"].replace(B=B, L=L, topk=topk, c_t=c_t)
    inp = synth.decode_layer(wl, csa=True)
    inp["ctx"] = torch.tensor([L, 1, 77, L - 3191][:B], dtype=torch.int32)
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    layer = DecodeLayer.create(wl, csa=True)
    layer.load_caches(d)
    lib.csa_quant_fp8_rows(d["qI"], layer.qI[0], layer.qI[1])
    return wl, d, layer


@pytest.mark.parametrize("c_t", ["bf16", "mixed"])
def test_static_scratch_decode_matches_workspace_decode(lib, c_t):
    wl, d, layer = _decode_setup(lib, c_t=c_t)
    p = layer.p
    assert lib.csa_workspace_bytes(p, lib.OP_CSA_DECODE) <= lib.STATIC_SCRATCH_BYTES
    C = layer.C if layer.C is not None else (d["C"], None, None)
    ref = torch.empty_like(layer.out)
    ref_idx = torch.empty_like(layer.topk)
    lib.csa_decode(p, d["q"], d["ctx"], C, layer.qI, layer.KI, d["w"], d["ring"], d["sink"], layer.rope, ref_idx, ref,
                   None, layer.ws)
    for _ in range(2):  # two calls in a row share the fixed array
        out = torch.full_like(layer.out, float("nan"))
        idx = torch.full_like(layer.topk, -7)
        lib.csa_decode_static_scratch(p, d["q"], d["ctx"], C, layer.qI, layer.KI, d["w"], d["ring"], d["sink"],
                                      layer.rope, idx, out, None)
        torch.cuda.synchronize()
        assert torch.equal(idx, ref_idx)
        a = out.float().cpu().numpy().astype(np.float64)
        b = ref.float().cpu().numpy().astype(np.float64)
        assert np.linalg.norm(a - b) / np.linalg.norm(b) <= 2e-2
    assert lib.csa_device_status() == 0


def test_static_scratch_refuses_a_layer_larger_than_the_array(lib):
    # 16 sequences x 131072 cached tokens at m = 4 fit (2 MiB of scores, 2.7 MB of split-KV
    # partial results); a 1M-token cache (16 x 262144 float scores = 16 MiB) does not and is
    # refused before any launch.
    fits = lib.make_params(B=16, L=131072, H=64, m=4, topk=512)
    assert lib.csa_workspace_bytes(fits, lib.OP_CSA_DECODE) <= lib.STATIC_SCRATCH_BYTES
    big = lib.make_params(B=16, L=1 << 20, H=64, m=4, topk=512)
    assert lib.csa_workspace_bytes(big, lib.OP_CSA_DECODE) > lib.STATIC_SCRATCH_BYTES
    with pytest.raises(lib.CsaError) as e:
        lib.csa_decode_static_scratch(big, torch.empty(1, device="cuda"), None, None, None, None, None, None, None,
                                      None, None, None, None)
    assert e.value.status == lib.ERR_WORKSPACE
