"""The projections on either side of the attention core on the GPU (csa_gemm_bf16 through the C
ABI) against the oracle's double-precision products of the same BF16 values.

Tolerances: FP32 outputs relative-L2 <= 2e-5 (the products of BF16 values are exact in FP32 and
a K-term FP32 sum errs by ~sqrt(K) * 2^-24 relative: 4e-6 at K = 4096); BF16 outputs <= 5e-3
(one BF16 rounding, at most 2^-9 relative per element); a product of a BF16-rounded product
(the grouped projection's final stage) <= 1e-2."""
import numpy as np
import pytest
import torch

import oracle
import synth
from _helpers import np64, rel_l2

pytestmark = pytest.mark.gpu


def test_gemm_ragged_shapes_and_output_segments(lib):
    g = torch.Generator().manual_seed(1)
    M, N, K = 300, 384, 256  # neither M nor N a multiple of the tile
    A = torch.randn((M, K), generator=g).to(torch.bfloat16)
    B = torch.randn((N, K), generator=g).to(torch.bfloat16)
    o1 = torch.full((M, 200), float("nan"), dtype=torch.bfloat16, device="cuda")
    o2 = torch.full((M, 184), float("nan"), dtype=torch.float32, device="cuda")
    lib.csa_gemm_bf16(A.cuda(), B.cuda(), [(o1, 0, 200), (o2, 200, 384)])
    torch.cuda.synchronize()
    want = oracle.project(np64(A), np64(B))
    assert rel_l2(np64(o1), want[:, :200]) <= 5e-3
    assert rel_l2(np64(o2), want[:, 200:]) <= 2e-5


def test_grouped_output_projection(lib):
    g = torch.Generator().manual_seed(2)
    M, H, d, groups, dg, hidden = 256, 64, 128, 8, 256, 512
    o = torch.randn((M, H, d), generator=g).to(torch.bfloat16)
    Wg = (torch.randn((groups * dg, (H // groups) * d), generator=g) * 0.03).to(torch.bfloat16)
    Wo = (torch.randn((hidden, groups * dg), generator=g) * 0.03).to(torch.bfloat16)
    od = o.cuda()
    y = torch.empty((M, groups * dg), dtype=torch.bfloat16, device="cuda")
    h = torch.empty((M, hidden), dtype=torch.bfloat16, device="cuda")
    lib.csa_gemm_bf16(od.view(M, H * d), Wg.cuda(), [(y, 0, groups * dg)], groups=groups)
    lib.csa_gemm_bf16(y, Wo.cuda(), [(h, 0, hidden)])
    torch.cuda.synchronize()
    wy, wh = oracle.grouped_output_projection(np64(o), np64(Wg), np64(Wo), groups)
    assert rel_l2(np64(y), wy) <= 5e-3
    assert rel_l2(np64(h), wh) <= 1e-2


@pytest.mark.parametrize("csa", [True, False])
def test_layer_projections_at_the_pair_workload_widths(lib, csa):
    # hidden 4096 -> q (64 x 128), kv (128) and the indexer inputs / logits, and the grouped
    # output projection back to 4096, on 640 rows of the layer-pair workload's shapes
    from long_context_compressed_14_b300.pipeline import Projections
    wl = synth.WORKLOADS["pair_mixed_L262144"]
    rows = 640
    P = synth.projection_inputs(wl, 0 if csa else 1, csa=csa, rows=rows)
    proj = Projections(wl, csa, P)
    got = proj.inputs(P["x"].cuda())
    torch.cuda.synchronize()
    x = np64(P["x"])
    assert rel_l2(np64(got["q"]).reshape(rows, -1), oracle.project(x, np64(P["Wq"]))) <= 5e-3
    assert rel_l2(np64(got["kv"]), oracle.project(x, np64(P["Wkv"]))) <= 5e-3
    idx = oracle.project(x, np64(P["Widx"]))
    if csa:
        ni = wl.H_I * wl.d_I
        assert rel_l2(np64(got["qI"]).reshape(rows, -1), idx[:, :ni]) <= 2e-5
        assert rel_l2(np64(got["kI_raw"]), idx[:, ni:ni + wl.d_I]) <= 2e-5
        assert rel_l2(np64(got["w"]), idx[:, ni + wl.d_I:ni + wl.d_I + wl.H_I]) <= 2e-5
        assert rel_l2(np64(got["z"]), idx[:, ni + wl.d_I + wl.H_I:]) <= 2e-5
    else:
        assert rel_l2(np64(got["z"]), idx) <= 2e-5
    h = proj.output(got["q"])
    torch.cuda.synchronize()
    _, wh = oracle.grouped_output_projection(np64(got["q"]), np64(P["Wg"]), np64(P["Wo"]), wl.groups)
    assert rel_l2(np64(h), wh) <= 1e-2
    assert lib.csa_device_status() == 0
