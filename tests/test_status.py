"""The device status word on the GPU: a bounded wait that runs out, a skipped out-of-range
index, and the reset that clears both (through the C ABI).

No GPU is faulted or hung here: the wait that runs out is the library's own bounded wait on an
mbarrier that never receives its arrival (1 ms limit), and the out-of-range index is skipped by
the attention kernel's own bounds check."""
import math

import numpy as np
import pytest
import torch

import synth
from _helpers import np64, oracle_prefill, rel_l2

pytestmark = pytest.mark.gpu


def _hca_parity(lib):
    from long_context_compressed_14_b300.pipeline import PrefillLayer
    wl = synth.WORKLOADS["hca_bf16_L16384"].replace(L=400)
    inp = synth.prefill_layer(wl, csa=False)
    out = PrefillLayer.create(wl, csa=False).run({k: v.cuda() for k, v in inp.items()})
    res = oracle_prefill(wl, inp, 0, np.arange(wl.L), csa=False)
    return rel_l2(np64(out[0]), res["o"])


def test_bounded_wait_times_out_then_reset_restores(lib):
    torch.cuda.synchronize()
    assert lib.csa_device_status() == 0
    lib.csa_selftest_wait_timeout(1_000_000)  # 1 ms
    assert lib.csa_device_status(reset=False) == lib.ERR_TIMEOUT
    assert lib.csa_device_status(reset=False) == lib.ERR_TIMEOUT  # sticky until reset
    assert lib.csa_device_status(reset=True) == lib.ERR_TIMEOUT
    assert lib.csa_device_status() == 0  # status word and abort flag cleared
    # the context is usable: a normal call afterwards runs to completion and matches the oracle
    assert _hca_parity(lib) <= 2e-2
    assert lib.csa_device_status() == 0


def test_out_of_range_index_is_skipped_and_reported(lib):
    wl = synth.WORKLOADS["csa_bf16_4x32768"].replace(B=1, L=300, topk=64)
    N = math.ceil(wl.L / wl.m)
    p = lib.make_params(B=1, L=wl.L, H=64, m=wl.m, topk=wl.topk)
    rope = lib.rope_table(p)
    g = torch.Generator().manual_seed(3)
    q = torch.randn((1, wl.L, 64, 128), generator=g).to(torch.bfloat16).cuda()
    kvr = torch.randn((1, wl.L, 128), generator=g).to(torch.bfloat16).cuda()
    C = torch.randn((1, N, 128), generator=g).to(torch.bfloat16).cuda()
    idx = torch.full((1, wl.L, wl.topk), -1, dtype=torch.int32)
    for t in range(wl.L):
        v = min((t + 1) // wl.m, wl.topk)
        idx[0, t, :v] = torch.arange(v)
    idx[0, wl.L - 1, wl.topk - 1] = N + 1000  # out of range: skipped, reported
    out = torch.empty((1, wl.L, 64, 128), dtype=torch.bfloat16, device="cuda")
    torch.cuda.synchronize()
    assert lib.csa_device_status() == 0
    lib.csa_sparse_attention(p, q, kvr, (C,), idx.cuda(), None, rope, out, None)
    assert lib.csa_device_status(reset=True) == lib.ERR_BOUNDS
    assert lib.csa_device_status() == 0
    assert torch.isfinite(out.float()).all()
