"""Pins of the CPU oracle to things other than itself (CPU only).

Each test checks one oracle step against a closed form, an invariant, a special case that
reduces to a library routine (torch SDPA, torch dtype casts), brute force on tiny inputs,
or a hand-worked fixture in tests/golden/. They are chosen so that a plausible slip in the
oracle -- a dropped term, a wrong sign or index, a transposed operand -- fails one of them.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
RNG = np.random.default_rng(1234)


# ---------------------------------------------------------------------------------------
# Compression
# ---------------------------------------------------------------------------------------

@pytest.mark.parametrize("L,m", [(1, 4), (3, 4), (4, 4), (5, 4), (2048, 4), (16384, 128),
                                 (127, 128), (129, 128), (7, 1)])
def test_compressed_length_is_ceil(L, m):
    x = RNG.standard_normal((L, 3))
    z = RNG.standard_normal((L, 2))
    assert oracle.compress(x, z, m).shape == (math.ceil(L / m), 3)


def test_compress_constant_rows_give_the_constant():
    # The weights of an entry sum to 1: constant raw rows compress to that constant.
    for L, m in [(37, 4), (300, 128), (5, 2)]:
        x = np.tile(RNG.standard_normal(8), (L, 1))
        z = RNG.standard_normal((L, 2)) * 3
        C = oracle.compress(x, z, m)
        np.testing.assert_allclose(C, np.tile(x[0], (C.shape[0], 1)), rtol=0, atol=1e-13)


@pytest.mark.parametrize("L,m", [(22, 4), (21, 4), (300, 128), (9, 2)])
def test_compress_one_hot_logit_selects_window_and_set(L, m):
    # A logit of +60 on one token and set dominates every entry whose window uses that
    # token with that set: own block (set a) -> entry t // m, previous block (set b) ->
    # entry t // m + 1. This fixes the window bounds and which set each half uses.
    x = RNG.standard_normal((L, 5))
    N = math.ceil(L / m)
    for t0 in [0, m - 1, m, L // 2, L - 1]:
        for s in (0, 1):
            z = np.zeros((L, 2))
            z[t0, s] = 60.0
            C = oracle.compress(x, z, m)
            j = t0 // m + s
            if j < N:
                np.testing.assert_allclose(C[j], x[t0], rtol=0, atol=1e-12)
            # an entry whose window does not contain t0 is not dominated by it
            other = t0 // m + (1 - s)
            if other < N:
                assert not np.allclose(C[other], x[t0], atol=1e-6)


def test_compress_m1_without_previous_block_is_identity():
    L = 17
    x = RNG.standard_normal((L, 4))
    z = np.stack([RNG.standard_normal(L), np.full(L, -400.0)], axis=1)
    np.testing.assert_allclose(oracle.compress(x, z, 1), x, rtol=0, atol=1e-150)


def test_compress_hand_worked_fixture():
    with open(os.path.join(GOLDEN, "compress_hand_m2.txt")) as f:
        lines = [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]
    for parts in lines:
        L, m = int(parts[0]), int(parts[1])
        expect = [float(Fraction(p)) for p in parts[2:]]
        x = (np.arange(L, dtype=np.float64) + 1.0)[:, None]
        z = np.stack([np.zeros(L), np.full(L, math.log(2.0))], axis=1)
        C = oracle.compress(x, z, m)[:, 0]
        np.testing.assert_allclose(C, expect, rtol=1e-14)


def test_visibility_rule():
    # entry j covers tokens up to (j+1)m-1; visible iff that is <= t
    m, N = 4, 10
    for t in range(45):
        v = oracle.visible(t, m, N)
        for j in range(N):
            assert (j < v) == ((j + 1) * m - 1 <= t)
    assert list(oracle.entry_pos(3, 4)) == [3, 7, 11]


@pytest.mark.parametrize("m", [4, 128])
def test_entry_rotation_position_is_its_last_raw_row(m):
    # An entry whose weights all sit on the last raw row u = (j+1)m-1 of its block (a +60
    # set-a logit there, every other logit 0) is that raw row; rotated at the entry position it
    # must equal the sliding-window copy of row u, which is rotated at u itself. So its logit
    # against any query equals row u's window logit. Rotating entries at jm (the block start)
    # or at (j+1)m (one past it) breaks this.
    L, d, d_rope, theta = 5 * m + 3, 128, 64, 1.0e4
    rng = np.random.default_rng(m)
    kv = rng.standard_normal((L, d))
    N = oracle.num_entries(L, m)
    for j in range(N - 1):  # complete blocks
        u = (j + 1) * m - 1
        z = np.zeros((L, 2))
        z[u, 0] = 60.0
        comp = oracle.kv_compress(kv, z, None, m, d_rope, theta)
        np.testing.assert_allclose(comp["C"][j], comp["kv_rope"][u], rtol=0, atol=1e-12)
        q = rng.standard_normal((3, d))
        np.testing.assert_allclose(q @ comp["C"][j], q @ comp["kv_rope"][u], rtol=0, atol=1e-10)
        # a rotation at the block start would not agree (the RoPE half moves)
        wrong = oracle.rope(kv[u:u + 1], np.array([j * m]), d_rope, theta)[0]
        assert np.abs(wrong[d - d_rope:] - comp["C"][j][d - d_rope:]).max() > 1e-3


# ---------------------------------------------------------------------------------------
# RoPE
# ---------------------------------------------------------------------------------------

def test_rope_unit_vectors_and_pairing():
    d, d_rope, theta = 128, 64, 1.0e4
    half = d_rope // 2
    base = d - d_rope
    for i in [0, 1, 7, half - 1]:
        for p in [0, 1, 5, 1000, 262143]:
            e = np.zeros((1, d))
            e[0, base + i] = 1.0
            r = oracle.rope(e, np.array([p]), d_rope, theta)
            ang = p * theta ** (-i / half)
            assert abs(r[0, base + i] - math.cos(ang)) < 1e-12
            assert abs(r[0, base + half + i] - math.sin(ang)) < 1e-12
            mask = np.ones(d, bool)
            mask[[base + i, base + half + i]] = False
            assert np.all(r[0, mask] == 0.0)
    # the lowest frequency pair turns by exactly one radian per position
    e = np.zeros((1, d))
    e[0, base] = 1.0
    r = oracle.rope(e, np.array([3]), d_rope, theta)
    assert abs(math.atan2(r[0, base + half], r[0, base]) - 3.0) < 1e-12


def test_rope_is_a_rotation_on_the_last_dims_only():
    x = RNG.standard_normal((50, 128))
    pos = RNG.integers(0, 300000, 50)
    r = oracle.rope(x, pos, 64, 1e4)
    np.testing.assert_array_equal(r[:, :64], x[:, :64])
    np.testing.assert_allclose(np.linalg.norm(r[:, 64:], axis=1), np.linalg.norm(x[:, 64:], axis=1), rtol=1e-13)
    back = oracle.rope(r, pos, 64, 1e4, sign=-1)
    np.testing.assert_allclose(back, x, atol=1e-12)
    np.testing.assert_array_equal(oracle.rope(x, np.zeros(50, np.int64), 64, 1e4), x)


def test_rope_dot_depends_on_relative_position_only():
    a = RNG.standard_normal((1, 128))
    b = RNG.standard_normal((1, 128))
    for p1, p2, delta in [(10, 3, 1000), (500, 500, 77), (0, 9, 123456)]:
        d0 = float((oracle.rope(a, np.array([p1]), 64, 1e4) @ oracle.rope(b, np.array([p2]), 64, 1e4).T)[0, 0])
        d1 = float((oracle.rope(a, np.array([p1 + delta]), 64, 1e4) @ oracle.rope(b, np.array([p2 + delta]), 64, 1e4).T)[0, 0])
        assert abs(d0 - d1) < 1e-9


# ---------------------------------------------------------------------------------------
# Storage roundings
# ---------------------------------------------------------------------------------------

def test_bf16_rounding_matches_torch_cast():
    x = np.concatenate([RNG.standard_normal(20000).astype(np.float32) * 10.0 ** RNG.integers(-30, 30, 20000),
                        np.array([0.0, -0.0, 1.0, 65504.0, 3.0e38, 1e-40], np.float32)]).astype(np.float32)
    want = torch.from_numpy(x).to(torch.bfloat16).float().numpy()
    np.testing.assert_array_equal(oracle.round_bf16_fast(x), want)
    np.testing.assert_array_equal(oracle.round_bf16(x[:2000]), want[:2000])
    # halfway cases: 1 + 2^-8 lies halfway between 1 and 1 + 2^-7 -> even (1.0)
    assert oracle.round_bf16(np.array([1.0 + 2.0 ** -8], np.float32))[0] == 1.0
    assert oracle.round_bf16(np.array([1.0 + 3 * 2.0 ** -8], np.float32))[0] == 1.0 + 2.0 ** -6


def test_fp8_spec_points_and_rne():
    with open(os.path.join(GOLDEN, "fp8_e4m3_spec_points.txt")) as f:
        lines = [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]
    for parts in lines:
        if parts[0] == "rne":
            assert int(oracle.fp8_encode(np.array([float(parts[1])], np.float32))[0]) == int(parts[2], 16), parts
        else:
            code, val = int(parts[0], 16), float(parts[1])
            got = float(oracle.fp8_decode(np.array([code], np.uint8))[0])
            assert got == val and math.copysign(1, got) == math.copysign(1, val), parts
    assert np.isnan(oracle.fp8_decode(np.array([0x7F, 0xFF], np.uint8))).all()


def test_fp8_exhaustive_roundtrip_and_torch():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    vals = oracle.fp8_decode(codes)
    np.testing.assert_array_equal(oracle.fp8_encode(vals), codes)
    # decode agrees with torch's float8_e4m3fn for every code
    tv = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).float().numpy()
    np.testing.assert_array_equal(vals, tv)
    # encode agrees with torch's round-to-nearest-even cast inside the finite range
    x = (RNG.standard_normal(30000) * 10.0 ** RNG.uniform(-3.5, 2.6, 30000)).astype(np.float32)
    x = x[np.abs(x) < 448.0]
    want = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(oracle.fp8_encode(x), want)


def test_quant_rows_scale_and_error_bound():
    x = RNG.standard_normal((300, 64)).astype(np.float32)
    x[5] = 0.0
    codes, scales = oracle.quant_rows_fp8(x)
    amax = np.abs(x).max(axis=1)
    np.testing.assert_array_equal(scales, (amax / np.float32(448.0)).astype(np.float32))
    assert scales[5] == 0 and np.all(codes[5] == 0)
    deq = oracle.dequant_fp8(codes, scales)
    # the largest element of each nonzero row lands on +-448 exactly
    r = np.arange(300) != 5
    am = np.abs(x).argmax(axis=1)
    np.testing.assert_array_equal(np.abs(oracle.fp8_decode(codes[np.arange(300), am]))[r], 448.0)
    # relative error of E4M3 round-to-nearest: at most 2^-4 of the value for normals,
    # at most half a subnormal step (2^-10 * scale) below 2^-6 * scale
    err = np.abs(deq - x)
    bound = np.maximum(np.abs(x) * 2.0 ** -4, 2.0 ** -10 * scales[:, None]) * (1 + 1e-6)
    assert np.all(err <= bound)


# ---------------------------------------------------------------------------------------
# Indexer score and top-k
# ---------------------------------------------------------------------------------------

def test_index_scores_exact_on_small_integers():
    # With small-integer operands every product and sum is exact in float32, so the fixed-
    # order FP32 score must equal exact integer arithmetic: sum_h w * max(0, q . k).
    L, N, HI, dI, m = 13, 4, 3, 8, 3
    qI = RNG.integers(-3, 4, (L, HI, dI)).astype(np.float32)
    KI = RNG.integers(-3, 4, (N, dI)).astype(np.float32)
    w = RNG.integers(-2, 3, (L, HI)).astype(np.float32)
    pos = np.arange(L)
    s = oracle.index_scores_f32(qI, KI, w, m, pos)
    for t in range(L):
        for j in range(N):
            if (j + 1) * m - 1 > t:
                assert s[t, j] == -np.inf
                continue
            want = sum(int(w[t, h]) * max(0, int(qI[t, h].astype(np.int64) @ KI[j].astype(np.int64)))
                       for h in range(HI))
            assert s[t, j] == want
    s64 = oracle.index_scores_f64(qI, KI, w, m, pos)
    np.testing.assert_array_equal(s64, s.astype(np.float64))


def test_index_scores_f32_close_to_double():
    L, N, HI, dI, m = 40, 10, 4, 64, 4
    qI = RNG.standard_normal((L, HI, dI)).astype(np.float32)
    KI = RNG.standard_normal((N, dI)).astype(np.float32)
    w = RNG.standard_normal((L, HI)).astype(np.float32)
    pos = np.arange(L)
    s32 = oracle.index_scores_f32(qI, KI, w, m, pos)
    s64 = oracle.index_scores_f64(qI, KI, w, m, pos)
    fin = np.isfinite(s64)
    assert np.array_equal(fin, np.isfinite(s32))
    assert np.max(np.abs(s32[fin] - s64[fin])) < 1e-4


def test_topk_hand_fixture():
    with open(os.path.join(GOLDEN, "topk_hand.txt")) as f:
        lines = [ln for ln in f if ln.strip() and not ln.startswith("#")]
    for ln in lines:
        head, sc, ex = ln.split("|")
        m, t, k = (int(v) for v in head.split())
        s = np.array([[float(v) for v in sc.split()]])
        want = [int(v) for v in ex.split()]
        assert list(oracle.topk(s, m, [t], k)[0]) == want, ln


def test_topk_brute_force_tiny():
    # Against an exhaustive ranking: j is kept iff fewer than k visible entries beat it
    # under (score desc, index asc).
    for trial in range(200):
        N = int(RNG.integers(1, 12))
        m = int(RNG.integers(1, 4))
        k = int(RNG.integers(1, 8))
        t = int(RNG.integers(0, N * m + 2))
        s = RNG.integers(-3, 4, (1, N)).astype(np.float64)  # many ties
        got = oracle.topk(s, m, [t], k)[0]
        vis = min((t + 1) // m, N)
        keep = []
        for j in range(vis):
            beats = sum(1 for i in range(vis) if s[0, i] > s[0, j] or (s[0, i] == s[0, j] and i < j))
            if beats < k:
                keep.append(j)
        want = keep + [-1] * (k - len(keep))
        assert list(got) == want


# ---------------------------------------------------------------------------------------
# Attention
# ---------------------------------------------------------------------------------------

def _sdpa(q, k, v, mask):
    """torch SDPA in float64 with a boolean (True = attend) or additive float mask."""
    return torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q), torch.from_numpy(k), torch.from_numpy(v),
        attn_mask=torch.from_numpy(mask), scale=1.0 / math.sqrt(q.shape[-1])).numpy()


@pytest.mark.parametrize("d_rope", [0, 64])
@pytest.mark.parametrize("L", [1, 9, 128])
def test_swa_only_equals_causal_attention(L, d_rope):
    # With no compressed branch (CSA, top-k = 0), no sink and L <= n_win, the layer is
    # exact causal attention with one shared K = V head (library routine: torch SDPA).
    H, d, theta, n_win = 4, 128, 1e4, 128
    q = RNG.standard_normal((L, H, d))
    kv = RNG.standard_normal((L, d))
    kvr = oracle.rope(kv, np.arange(L), d_rope, theta)
    o, ps = oracle.attention_rows(q, kvr, None, np.zeros((L, 0), np.int32), 0, 4, d_rope, theta, n_win,
                                  None, d ** -0.5, np.arange(L))
    qr = np.stack([oracle.rope(q[:, h], np.arange(L), d_rope, theta) for h in range(H)])  # [H, L, d]
    ref = _sdpa(qr, np.broadcast_to(kvr, (H, L, d)).copy(), np.broadcast_to(kvr, (H, L, d)).copy(),
                np.tril(np.ones((L, L), bool)))
    ref = np.stack([oracle.rope(ref[h], np.arange(L), d_rope, theta, sign=-1) for h in range(H)], axis=1)
    np.testing.assert_allclose(o, ref, atol=1e-12)
    np.testing.assert_allclose(ps, 1.0, atol=1e-13)


def _dense_reference(q, kvr, C, m, n_win, sink, d_rope, theta):
    """HCA layer via torch SDPA: keys = [entries; raw rows; one zero 'sink' key], boolean
    visibility and window turned into an additive mask, the sink logit as the additive mask
    of the zero key (its logit is 0 before the mask and its value is 0)."""
    L, H, d = q.shape
    N = C.shape[0]
    keys = np.concatenate([C, kvr, np.zeros((1, d))])
    t = np.arange(L)[:, None]
    vis = ((np.arange(N)[None] + 1) * m - 1) <= t
    u = np.arange(L)[None]
    win = (u <= t) & (u > t - n_win)
    allowed = np.concatenate([vis, win, np.ones((L, 1), bool)], axis=1)
    add = np.where(allowed, 0.0, -np.inf)
    masks = np.repeat(add[None], H, axis=0)
    masks[:, :, -1] = -np.inf if sink is None else np.asarray(sink)[:, None]
    qr = np.stack([oracle.rope(q[:, h], np.arange(L), d_rope, theta) for h in range(H)])
    K = np.broadcast_to(keys, (H,) + keys.shape).copy()
    out = _sdpa(qr, K, K, masks)
    return np.stack([oracle.rope(out[h], np.arange(L), d_rope, theta, sign=-1) for h in range(H)], axis=1)


@pytest.mark.parametrize("with_sink", [False, True])
def test_hca_equals_masked_dense_attention(with_sink):
    L, H, d, m, n_win, theta = 300, 3, 128, 8, 16, 1e4
    q = RNG.standard_normal((L, H, d))
    kvr = oracle.rope(RNG.standard_normal((L, d)), np.arange(L), 64, theta)
    C = RNG.standard_normal((math.ceil(L / m), d))
    sink = RNG.standard_normal(H) if with_sink else None
    o, _ = oracle.attention_rows(q, kvr, C, None, 0, m, 64, theta, n_win, sink, d ** -0.5, np.arange(L))
    ref = _dense_reference(q, kvr, C, m, n_win, sink, 64, theta)
    np.testing.assert_allclose(o, ref, atol=1e-11)


def test_csa_with_k_at_least_visible_equals_dense():
    L, H, d, m, n_win, theta = 200, 2, 128, 4, 32, 1e4
    q = RNG.standard_normal((L, H, d))
    kvr = RNG.standard_normal((L, d))
    C = RNG.standard_normal((L // m, d))
    sink = RNG.standard_normal(H)
    HI, dI = 3, 64
    qI = RNG.standard_normal((L, HI, dI)).astype(np.float32)
    KI = RNG.standard_normal((L // m, dI)).astype(np.float32)
    w = RNG.standard_normal((L, HI)).astype(np.float32)
    k = L // m
    res = oracle.csa_rows(q, kvr, C, qI, KI, w, sink, np.arange(L), m=m, k=k, d_rope=64, theta=theta,
                          n_win=n_win, scale=d ** -0.5, idx_store="f32")
    ref = _dense_reference(q, kvr, C, m, n_win, sink, 64, theta)
    np.testing.assert_allclose(res["o"], ref, atol=1e-11)
    # and with a smaller k the selected set is exactly the top-k of the scores
    res2 = oracle.csa_rows(q, kvr, C, qI, KI, w, sink, np.arange(L), m=m, k=5, d_rope=64, theta=theta,
                           n_win=n_win, scale=d ** -0.5, idx_store="f32")
    for t in [4, 50, 199]:
        vis = (t + 1) // m
        order = sorted(range(vis), key=lambda j: (-res2["scores"][t, j], j))[:5]
        assert sorted(order) == [j for j in res2["idx"][t] if j >= 0]


def test_sink_weights_sum():
    H, d = 3, 16
    q = RNG.standard_normal((H, d))
    keys = RNG.standard_normal((7, d))
    _, ps = oracle.attend_one(q, keys, None, 0.25)
    np.testing.assert_allclose(ps, 1.0, atol=1e-15)
    sink = np.array([-1.0, 0.5, 3.0])
    _, ps2 = oracle.attend_one(q, keys, sink, 0.25)
    assert np.all(ps2 < 1.0)
    z = np.exp(0.25 * q @ keys.T).sum(axis=1)
    np.testing.assert_allclose(ps2, z / (z + np.exp(sink)), rtol=1e-13)
    _, ps3 = oracle.attend_one(q, keys, np.full(H, -1e4), 0.25)
    np.testing.assert_allclose(ps3, 1.0, atol=1e-15)
    # a lone key with a sink: weight = e^l / (e^l + e^s)
    o, ps4 = oracle.attend_one(q, keys[:1], sink, 0.25)
    lg = 0.25 * q @ keys[0]
    np.testing.assert_allclose(ps4, np.exp(lg) / (np.exp(lg) + np.exp(sink)), rtol=1e-13)
    np.testing.assert_allclose(o, ps4[:, None] * keys[:1], rtol=1e-13)


def test_attention_is_invariant_to_a_common_position_shift():
    # RoPE on queries and keys plus inverse RoPE on the output: shifting every position by
    # delta leaves the output unchanged (decode form: raw rows rotated at their positions).
    H, d, n_win, theta = 4, 128, 16, 1e4
    raw = RNG.standard_normal((n_win, d))
    q = RNG.standard_normal((H, d))
    outs = []
    for ctx in [40, 40 + 1000, 40 + 98765]:
        p = ctx - 1
        us = np.arange(p - n_win + 1, p + 1)
        ring = np.zeros((n_win, d))
        ring[us % n_win] = oracle.rope(raw, us, 64, theta)
        o, _ = oracle.decode_one(q, ctx, np.zeros((0, d)), None, 0, 1 << 30, ring, 64, theta, n_win,
                                 None, d ** -0.5)
        outs.append(o)
    np.testing.assert_allclose(outs[1], outs[0], atol=1e-9)
    np.testing.assert_allclose(outs[2], outs[0], atol=1e-9)
    # while a RoPE that forgot the inverse on the output would not be shift-invariant
    assert not np.allclose(oracle.rope(outs[0], np.array([39]), 64, theta),
                           oracle.rope(outs[1], np.array([1039]), 64, theta), atol=1e-3)


@pytest.mark.parametrize("idx_store,c_store", [("f32", "f32"), ("fp8", "mixed"), ("mxfp4", "nvfp4")])
def test_decode_equals_last_prefill_row(idx_store, c_store):
    # Decode at ctx = L against caches built from the same raw rows equals row L-1 of a
    # prefill of length L (CSA and HCA).
    L, H, d, m, mh, n_win, k, theta = 203, 4, 128, 4, 16, 32, 6, 1e4
    HI, dI = 3, 64
    kv = RNG.standard_normal((L, d))
    z = RNG.standard_normal((L, 2))
    kI = RNG.standard_normal((L, dI))
    q = RNG.standard_normal((L, H, d))
    qI = RNG.standard_normal((L, HI, dI))
    w = RNG.standard_normal((L, HI))
    sink = RNG.standard_normal(H)
    kw = dict(d_rope=64, theta=theta, n_win=n_win, scale=d ** -0.5)
    comp = oracle.kv_compress(kv, z, kI, m, 64, theta, c_store=c_store, idx_store=idx_store)
    pre = oracle.csa_rows(q[L - 1:], comp["kv_rope"], comp["C"], qI[L - 1:], comp["KI"], w[L - 1:], sink,
                          np.array([L - 1]), m=m, k=k, idx_store=idx_store, **kw)
    ring = np.zeros((n_win, d))
    us = np.arange(L - n_win, L)
    ring[us % n_win] = comp["kv_rope"][us]
    dec = oracle.csa_decode(q[L - 1], L, comp["C"], qI[L - 1], comp["KI"], w[L - 1], ring, sink, m=m, k=k,
                            idx_store=idx_store, **kw)
    np.testing.assert_array_equal(dec["idx"], pre["idx"][0])
    np.testing.assert_allclose(dec["o"], pre["o"][0], atol=1e-12)
    comph = oracle.kv_compress(kv, z, None, mh, 64, theta, c_store=c_store)
    preh = oracle.hca_rows(q[L - 1:], comph["kv_rope"], comph["C"], sink, np.array([L - 1]), m=mh, **kw)
    dech = oracle.hca_decode(q[L - 1], L, comph["C"], ring, sink, m=mh, **kw)
    np.testing.assert_allclose(dech["o"], preh["o"][0], atol=1e-12)


def test_mixed_storage_rows():
    x = RNG.standard_normal((50, 128)) * 3
    vals, (codes, scales) = oracle.store_rows(x, "mixed", d_rope=64)
    np.testing.assert_array_equal(vals[:, 64:], oracle.round_bf16_fast(x[:, 64:].astype(np.float32)))
    np.testing.assert_array_equal(vals[:, :64], oracle.dequant_fp8(codes, scales))
    assert codes.shape == (50, 64) and scales.shape == (50,)


# ---------------------------------------------------------------------------------------
# Projections around the core
# ---------------------------------------------------------------------------------------

def test_projection_identity_and_block_diagonal_grouping():
    # identity weights give the rows back; the grouped output projection equals one dense
    # projection with the groups' matrices on the block diagonal (a group-to-columns slip, e.g.
    # group g reading the heads of another group, breaks it)
    rng = np.random.default_rng(7)
    x = rng.standard_normal((5, 16))
    np.testing.assert_allclose(oracle.project(x, np.eye(16)), x, rtol=0, atol=0)
    rows, H, d, groups, dg, hidden = 6, 8, 4, 4, 3, 5
    o = rng.standard_normal((rows, H, d))
    Wg = rng.standard_normal((groups * dg, (H // groups) * d))
    Wo = rng.standard_normal((hidden, groups * dg))
    y, h = oracle.grouped_output_projection(o, Wg, Wo, groups)
    dense = np.zeros((groups * dg, H * d))
    hw = (H // groups) * d
    for g in range(groups):
        dense[g * dg:(g + 1) * dg, g * hw:(g + 1) * hw] = Wg[g * dg:(g + 1) * dg]
    np.testing.assert_allclose(y, o.reshape(rows, H * d) @ dense.T, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(h, y @ Wo.T, rtol=1e-13, atol=1e-13)
    # one head group alone: the other groups' columns of y are untouched by it
    o2 = o.copy()
    o2[:, : H // groups] += 1.0
    y2, _ = oracle.grouped_output_projection(o2, Wg, Wo, groups)
    np.testing.assert_allclose(y2[:, dg:], y[:, dg:], rtol=0, atol=0)
    assert np.abs(y2[:, :dg] - y[:, :dg]).max() > 1e-3


# ---------------------------------------------------------------------------------------
# FP4 (E2M1, MXFP4) codec
# ---------------------------------------------------------------------------------------

def test_e2m1_values_and_round_trip():
    vals = oracle.e2m1_decode(np.arange(16))
    np.testing.assert_array_equal(vals[:8], [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    np.testing.assert_array_equal(vals[8:], -vals[:8])
    assert np.all(oracle.e2m1_encode(vals[1:8]) == np.arange(1, 8))
    assert np.all(oracle.e2m1_encode(vals[9:]) == np.arange(9, 16))


def test_e2m1_rounding_fixture():
    rows = [l.split() for l in open(os.path.join(GOLDEN, "e2m1_rounding.txt")) if l.strip() and not l.startswith("#")]
    x = np.array([float(r[0]) for r in rows])
    want = np.array([float(r[1]) for r in rows])
    np.testing.assert_array_equal(oracle.e2m1_decode(oracle.e2m1_encode(x)), want)


def test_mxfp4_block_exponent_rule_and_error_bound():
    # the block exponent is floor(log2(block max)) - 2, so the block max lands in [4, 8) and a
    # max of 6 * 2^e is exact; a zero block gets exponent byte 0 and zero codes
    x = np.zeros((3, 64), np.float32)
    x[0, 0], x[0, 32:35] = 12.0, [1.0, 2.0, 3.0]
    x[1, 5] = 6.0
    codes, e8 = oracle.quant_rows_mxfp4(x)
    np.testing.assert_array_equal(e8, [[128, 126], [127, 0], [0, 0]])
    deq = oracle.dequant_mxfp4(codes, e8)
    np.testing.assert_array_equal(deq[0, [0, 32, 33, 34]], [12.0, 1.0, 2.0, 3.0])
    assert deq[1, 5] == 6.0 and np.all(deq[2] == 0.0)
    # random rows: below 6 * 2^e an element errs by at most half a gap (at most 1 * 2^e,
    # between 4 and 6); above it -- the block max lies in [4, 8) * 2^e -- it saturates at 6 * 2^e,
    # an error below 2 * 2^e; the block max is never exceeded
    rng = np.random.default_rng(3)
    r = (rng.standard_normal((200, 64)) * np.exp(rng.standard_normal((200, 1)) * 4)).astype(np.float32)
    c, e = oracle.quant_rows_mxfp4(r)
    d = oracle.dequant_mxfp4(c, e)
    scale = np.repeat(np.exp2(e.astype(np.float64) - 127), 32, axis=1)
    inside = np.abs(r) <= 6 * scale
    assert np.all(np.abs(d - r)[inside] <= 1.0 * scale[inside])
    assert np.all(np.abs(d - r)[~inside] < 2.0 * scale[~inside])
    assert np.all(np.abs(d[~inside]) == 6 * scale[~inside])
    blkmax = np.repeat(np.abs(r.reshape(200, 2, 32)).max(axis=2), 32, axis=1)
    assert np.all(np.abs(d) <= np.maximum(blkmax, 6 * scale) + 1e-300)


def test_mxfp4_to_fp8_is_exact():
    # [P2] 事後学習 §3: FP4 -> FP8 dequantisation is lossless. With E the row's larger block
    # exponent, every element times 2^(e_blk - E + 6) is an E4M3 value (checked with the
    # oracle's E4M3 codec, pinned against torch), so codes * 2^(E - 6) reproduce the row exactly
    rng = np.random.default_rng(4)
    r = (rng.standard_normal((300, 64)) * np.exp(rng.standard_normal((300, 1)) * 3)).astype(np.float32)
    r[:, 32:] *= np.exp2(rng.integers(-10, 10, (300, 1))).astype(np.float32)
    c, e = oracle.quant_rows_mxfp4(r)
    v = oracle.dequant_mxfp4(c, e)
    E = e.astype(np.int64).max(axis=1, keepdims=True) - 127
    scaled = v * np.exp2(6.0 - E)
    codes8 = oracle.fp8_encode(scaled.astype(np.float32))
    back = oracle.fp8_decode(codes8).astype(np.float64) * np.exp2(E - 6.0)
    np.testing.assert_array_equal(back, v)


# ---------------------------------------------------------------------------------------
# NVFP4 entries and FP8 window rows (the V4.1 cache variant)
# ---------------------------------------------------------------------------------------

def _nvfp4_fixture():
    x = np.zeros(128, np.float32)
    want = np.zeros(128)
    scale, blocks = None, None
    for line in open(os.path.join(GOLDEN, "nvfp4_row_hand.txt")):
        f = line.split()
        if not f or f[0].startswith("#"):
            continue
        if f[0] == "scale":
            scale = float(f[1])
        elif f[0] == "blocks":
            blocks = [int(v, 16) for v in f[1:]]
        else:
            x[int(f[0])], want[int(f[0])] = float(f[1]), float(f[2])
    return x, want, scale, blocks


def test_nvfp4_hand_worked_row():
    x, want, scale, blocks = _nvfp4_fixture()
    codes, bcode, rs = oracle.quant_rows_nvfp4(x[None])
    assert rs[0] == scale
    np.testing.assert_array_equal(bcode[0], blocks)
    np.testing.assert_array_equal(oracle.dequant_nvfp4(codes, bcode, rs)[0], want)


def test_nvfp4_exact_on_representable_rows():
    # rows built from the format itself -- s a power of two, block scale c_b an E4M3 value, the
    # block's elements E2M1 values (one of them +-6) times c_b s, one block with c_b = 448 -- come
    # back exactly, with block codes E4M3(c_b) and row scale s (a wrong 6 or 448, a block of
    # 32 instead of 16, or a misplaced scale breaks it)
    rng = np.random.default_rng(11)
    grid = oracle.e2m1_decode(np.arange(16))
    e4m3 = oracle.fp8_decode(np.arange(0x08, 0x7F)).astype(np.float64)  # normal E4M3 values
    rows = np.zeros((64, 128))
    cb = np.zeros((64, 8))
    s = np.exp2(rng.integers(-20, 10, 64)).astype(np.float64)
    for r in range(64):
        cb[r] = rng.choice(e4m3, 8)
        cb[r, rng.integers(0, 8)] = 448.0
        for b in range(8):
            el = rng.choice(grid, 16)
            el[rng.integers(0, 16)] = rng.choice([-6.0, 6.0])
            rows[r, 16 * b:16 * b + 16] = el * cb[r, b] * s[r]
    x = rows.astype(np.float32)
    assert np.array_equal(x.astype(np.float64), rows)
    codes, bcode, rs = oracle.quant_rows_nvfp4(x)
    np.testing.assert_array_equal(rs, s.astype(np.float32))
    np.testing.assert_array_equal(oracle.fp8_decode(bcode), cb)
    np.testing.assert_array_equal(oracle.dequant_nvfp4(codes, bcode, rs), rows)


def test_nvfp4_error_bound_on_random_rows():
    # each element errs by at most half a gap of the E2M1 grid (at most 1 x the block scale,
    # between 4 and 6) when inside 6 x scale, and saturates to +-6 x scale outside it, which the
    # block-scale rounding (relative 2^-4 for a normal E4M3 code) keeps below 6.4 x scale
    rng = np.random.default_rng(12)
    x = (rng.standard_normal((300, 128)) * np.exp(rng.standard_normal((300, 1)) * 3)).astype(np.float32)
    codes, bcode, rs = oracle.quant_rows_nvfp4(x)
    d = oracle.dequant_nvfp4(codes, bcode, rs)
    scale = np.repeat((oracle.fp8_decode(bcode).astype(np.float32) * rs[:, None]).astype(np.float64), 16, axis=1)
    normal = np.repeat(bcode >= 0x08, 16, axis=1)
    xs = x.astype(np.float64)
    inside = normal & (np.abs(xs) <= 6 * scale)
    assert np.all(np.abs(d - xs)[inside] <= 1.0 * scale[inside])
    out = normal & ~inside
    assert np.all(np.abs(d[out]) == 6 * scale[out]) and np.all(np.abs(xs[out]) <= 6.4 * scale[out])
    # the whole row: relative L2 error of a 4-bit format, well below 0.2
    rel = np.linalg.norm(d - xs, axis=1) / np.linalg.norm(xs, axis=1)
    assert rel.max() < 0.2


def test_nvfp4_and_fp8_window_storage_rows():
    # store_rows applies the formats: 'nvfp4' is the quantiser's dequantised row, 'fp8' the
    # per-row FP8 of the window ring
    x = RNG.standard_normal((20, 128)) * 3
    vals, (codes, bcode, rs) = oracle.store_rows(x, "nvfp4")
    np.testing.assert_array_equal(vals, oracle.dequant_nvfp4(codes, bcode, rs))
    assert codes.shape == (20, 64) and bcode.shape == (20, 8) and rs.shape == (20,)
    v8, (c8, s8) = oracle.store_rows(x, "fp8")
    np.testing.assert_array_equal(s8, (np.abs(x.astype(np.float32)).max(axis=1) / np.float32(448)).astype(np.float32))
    np.testing.assert_array_equal(v8, oracle.dequant_fp8(c8, s8))
