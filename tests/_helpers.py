"""Shared helpers of the parity tests: run the oracle on synth inputs, compare results."""
from __future__ import annotations

import numpy as np
import torch

import oracle


def np64(t: torch.Tensor) -> np.ndarray:
    """Exact float64 copy of a float32/bfloat16 tensor."""
    return t.detach().float().cpu().numpy().astype(np.float64)


def np32(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy()


def rel_l2(a, b) -> float:
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def oracle_prefill(wl, inp: dict, b: int, rows, csa: bool, q_rows=None, w_store=None):
    """Oracle result of one prefill layer for rows of sequence b (CPU torch inputs). w_store:
    the storage of the window rows (default: the activation dtype; 'fp8' for rows read from an
    FP8 decode ring)."""
    m = wl.m if csa else wl.m_hca
    rows = np.asarray(rows, np.int64)
    comp = oracle.kv_compress(np64(inp["kv"][b]), np64(inp["z"][b]),
                              np64(inp["kI_raw"][b]) if csa and wl.topk > 0 else None, m, wl.d_rope, wl.theta,
                              c_store=wl.c_t, idx_store=wl.idx_t if csa else "f64", q_store=w_store or wl.q_t)
    qr = np64(inp["q"][b][rows]) if q_rows is None else q_rows
    kw = dict(d_rope=wl.d_rope, theta=wl.theta, n_win=wl.n_win, scale=wl.scale)
    sink = np64(inp["sink"]) if inp.get("sink") is not None else None
    if csa:
        if wl.topk > 0:
            res = oracle.csa_rows(qr, comp["kv_rope"], comp["C"], np32(inp["qI"][b][rows]), comp["KI"],
                                  np32(inp["w"][b][rows]), sink, rows, m=m, k=wl.topk, idx_store=wl.idx_t, **kw)
        else:
            res = oracle.csa_rows(qr, comp["kv_rope"], comp["C"], None, None, None, sink, rows, m=m, k=0,
                                  idx_store=wl.idx_t, **kw)
    else:
        res = oracle.hca_rows(qr, comp["kv_rope"], comp["C"], sink, rows, m=m, **kw)
    res["comp"] = comp
    return res


def check_topk_by_score(gpu_idx, scores, pos, m, k, rel_eps=1e-3, min_overlap=0.99):
    """Selections that differ only by near-ties are both correct. Checks that every
    GPU-selected index is visible and has an oracle score >= (oracle k-th score - eps), with
    eps = rel_eps * max |score| of the row, that the GPU set has the right size and is
    ascending, and that the mean set overlap with the oracle's selection is >= min_overlap.
    Returns the fraction of rows whose sets agree exactly."""
    gpu_idx = np.asarray(gpu_idx)
    same = 0
    overlap = []
    for r in range(gpu_idx.shape[0]):
        t = int(pos[r])
        vis = min((t + 1) // m, scores.shape[1])
        g = gpu_idx[r]
        kept = g[g >= 0]
        assert len(kept) == min(k, vis), (r, len(kept), min(k, vis))
        assert np.all(np.diff(kept) > 0), "kept set must be ascending"
        assert np.all(g[len(kept):] == -1)
        if len(kept) == 0:
            same += 1
            overlap.append(1.0)
            continue
        assert kept.max() < vis
        s = scores[r, :vis]
        kth = np.sort(s)[::-1][min(k, vis) - 1]
        eps = rel_eps * max(np.abs(s).max(), 1e-30)
        assert np.all(s[kept] >= kth - eps), (r, s[kept].min(), kth)
        order = np.sort(np.lexsort((np.arange(vis), -s))[:k])
        same += int(np.array_equal(order, kept))
        overlap.append(len(np.intersect1d(order, kept)) / len(kept))
    ov = float(np.mean(overlap)) if overlap else 1.0
    assert ov >= min_overlap, ("mean set overlap", ov)
    return same / max(gpu_idx.shape[0], 1)


def attention_on_gpu_selection(wl, res, q_rows, gpu_idx, rows, sink, csa=True):
    """The oracle's attention for query rows, run on the GPU's own top-k selection (the
    'checked twice' step: isolates the attention kernel from near-tie selection differences)."""
    m = wl.m if csa else wl.m_hca
    o, _ = oracle.attention_rows(q_rows, res["comp"]["kv_rope"], res["comp"]["C"], np.asarray(gpu_idx, np.int32),
                                 wl.topk, m, wl.d_rope, wl.theta, wl.n_win, sink, wl.scale, rows)
    return o


def check_csa_rows(wl, inp, b, rows, gpu_out_rows, gpu_idx_rows, res, tol=2e-2):
    """CSA output checked twice: (1) against the oracle's attention on the GPU's own selection,
    every row; (2) end to end against the oracle's own selection, every row."""
    q_rows = np64(inp["q"][b][rows])
    sink = np64(inp["sink"]) if inp.get("sink") is not None else None
    o_own = attention_on_gpu_selection(wl, res, q_rows, gpu_idx_rows, rows, sink)
    e1 = rel_l2(gpu_out_rows, o_own)
    e2 = rel_l2(gpu_out_rows, res["o"])
    assert e1 <= tol, ("attention on the GPU selection", e1)
    assert e2 <= tol, ("end to end", e2)
    return e1, e2


def unpack_nvfp4(rows: torch.Tensor):
    """NVFP4 entry rows [.., 80] uint8 (layout in include/csa.h) -> (codes [.., 64], block codes
    [.., 8], row scales [..] float32, pad bytes [.., 4])."""
    r = rows.cpu().numpy()
    return r[..., :64], r[..., 64:72], np.ascontiguousarray(r[..., 72:76]).view(np.float32)[..., 0], r[..., 76:80]


def unpack_fp8_window(rows: torch.Tensor):
    """FP8 window rows [.., 144] uint8 -> (codes [.., 128], scales [..] float32, pad [.., 12])."""
    r = rows.cpu().numpy()
    return r[..., :128], np.ascontiguousarray(r[..., 128:132]).view(np.float32)[..., 0], r[..., 132:144]
