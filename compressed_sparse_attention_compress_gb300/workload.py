"""Algorithmic work accounting for the benchmark (counts only; no method arithmetic).

Per-unit figures ("DeepSeek-V4 Attention Training Systems", §2 phase table
cost model, §5.5 replicated-state size):
  attention  4*H*d FLOPs per (query, candidate key)   QK^T + PV
  attn bwd   10*H*d FLOPs per (query, candidate key)  S recompute, dP, dQ, dK, dV
  index bwd  2*H*d + 6*H_I*d_I FLOPs per (query, C_t entry)  teacher recompute (once), dw, dqI, dkI
  indexer    2*H_I*d_I FLOPs per (query, visible entry)
  teacher    2*H*d FLOPs per (query, C_t entry), counted once
  compress   read x and z (2 B each per channel) + write one row per r tokens;
             the "v4" compressor also reads the previous-half x and z
"""
from __future__ import annotations

import numpy as np


def compressed_state_bytes(tokens: int, ratio: int, dims: int, bytes_per_elem: int = 2) -> int:
    """Bytes of compressed state for ``tokens`` raw tokens at ``ratio`` (complete groups only)."""
    return (tokens // ratio) * dims * bytes_per_elem


def _per_query(lengths, ratio, window, topk):
    vis, win = [], []
    for L in lengths:
        t = np.arange(L, dtype=np.int64)
        v = (t + 1) // ratio if ratio > 0 else np.zeros(L, np.int64)
        vis.append(v)
        win.append(np.minimum(t + 1, window))
    return np.concatenate(vis), np.concatenate(win)


def counts(wl) -> dict:
    """Exact pair counts and algorithmic FLOPs / bytes of one forward of ``wl``."""
    vis, win = _per_query(wl.lengths, wl.ratio, wl.window, wl.topk)
    H, d = wl.H, wl.d
    if wl.H_I > 0:
        sel = np.minimum(vis, wl.topk)
        cmp_keys = sel
    elif wl.ratio > 0:
        sel = vis
        cmp_keys = vis
    else:
        sel = np.zeros_like(vis)
        cmp_keys = sel
    attn_pairs = int((cmp_keys + win).sum())
    out = {
        "queries": int(wl.T),
        "visible_pairs": int(vis.sum()),
        "attn_pairs": attn_pairs,
        "attn_flops": 4 * H * d * attn_pairs,
        "attn_bwd_flops": 10 * H * d * attn_pairs,
    }
    if wl.H_I > 0:
        out["indexer_flops"] = 2 * wl.H_I * wl.d_I * int(vis.sum())
        out["topk_bytes"] = int(wl.T) * (2 * wl.H_I * wl.d_I + 2 * wl.H_I) + int(wl.T) * 4 * wl.k_pad
    else:
        out["indexer_flops"] = 0
        out["topk_bytes"] = 0
    if wl.kl_mode == "dense":
        out["teacher_pairs"] = int(vis.sum())
    elif wl.kl_mode == "sparse":
        out["teacher_pairs"] = int(sel.sum())
    else:
        out["teacher_pairs"] = 0
    out["teacher_flops"] = 2 * H * d * out["teacher_pairs"]
    out["indexer_bwd_flops"] = (2 * H * d + 6 * wl.H_I * wl.d_I) * out["teacher_pairs"]
    comp = 0
    if wl.ratio > 0:
        comp += wl.T * 4 * d + wl.n_cmp * 2 * d + wl.span * d * 4
        if wl.H_I > 0:
            comp += wl.T * 4 * wl.d_I + wl.n_cmp * 2 * wl.d_I + wl.span * wl.d_I * 4
        if wl.compressor == "v4" and wl.overlap:   # previous-half x and z streams
            comp += wl.T * 4 * (wl.d + (wl.d_I if wl.H_I > 0 else 0))
    out["compress_bytes"] = int(comp)
    out["gather_bytes"] = attn_pairs * d * 2
    out["total_flops"] = out["attn_flops"] + out["indexer_flops"] + out["teacher_flops"]
    return out
