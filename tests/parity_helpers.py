"""Helpers for the GPU parity tests: run the C-ABI path, feed the same values to
the oracle stage by stage, compare within the tolerances the method fixes.

Tolerances (bf16 inputs, fp32 accumulation):
  compress / attention outputs / lse : max-abs 1e-2 against the fp64 oracle, on
                                       the stored values (a bf16 output's own
                                       rounding counts against the bound)
  top-k index sets                   : bit-exact, except entries whose oracle
                                       score lies within 1e-4 relative of the
                                       oracle's k-th score (near-ties)
  KL sum                             : 1e-3 relative
"""
from __future__ import annotations

import os

import numpy as np
import torch

import oracle
from compressed_sparse_attention_compress_gb300.inputs import bf16_round

ATOL = 1e-2
TIE_RTOL = 1e-4
KL_RTOL = 1e-3


# raw max-abs errors observed by the checks: (test id, quantity, error)
ERRORS: list = []


def record(what: str, err: float) -> float:
    """Keep an observed error for the session summary (written by conftest)."""
    test = os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0]
    ERRORS.append((test, what, float(err)))
    return err


def np32(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy()


def operand(t: torch.Tensor) -> np.ndarray:
    """A GPU intermediate as the next kernel consumes it: rounded to bf16 on load
    (a no-op for bf16 tensors; float32 I/O rounds its compressed rows)."""
    return bf16_round(np32(t))


def bf16_half_ulp(x: np.ndarray) -> np.ndarray:
    """Half the spacing of bf16 values at |x| (the largest round-to-nearest error)."""
    ax = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(ax, 2.0 ** -126)))
    return np.ldexp(1.0, (e - 8).astype(np.int64))


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    """The spacing of bf16 values in the binade of |x|."""
    ax = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(ax, 2.0 ** -126)))
    return np.ldexp(1.0, (e - 7).astype(np.int64))


def check_stored_bf16(got: np.ndarray, ref: np.ndarray, what: str) -> float:
    """A bf16 output against the exact value.  Where |x| < 4 a bf16 value lies
    within 1e-2 of any x (spacing <= 1/64), and the plain max-abs 1e-2 applies.
    Where |x| >= 4 the spacing is 1/32 or more, so no stored value can be within
    1e-2 of every x: there the value must be one of the two bf16 values that
    bracket x (within one spacing); the float32-output path of the same kernel
    is held to the plain bound separately."""
    d = np.abs(got - ref)
    err = record(what, d.max() if d.size else 0.0)
    small = np.abs(ref) < 4.0
    e_small = record(what + "[|x|<4]", d[small].max() if small.any() else 0.0)
    assert e_small <= ATOL, f"{what} max-abs {e_small} where |x| < 4"
    if (~small).any():
        over = d[~small] - bf16_ulp(ref[~small])
        record(what + "[|x|>=4] - spacing", over.max())
        assert np.all(over < 0), f"{what}: a stored value at |x| >= 4 is not a bracketing bf16"
    return err


def check_compress(gpu_out: torch.Tensor, x, z, P, cu, ratio, overlap, n_c):
    ref = oracle.compress(x, z, P, cu, ratio, overlap)
    got = np32(gpu_out[:n_c]).astype(np.float64)
    if gpu_out.dtype == torch.bfloat16 and ref.size:
        return check_stored_bf16(got, ref, "compress")
    err = record("compress_fp32" if gpu_out.dtype == torch.float32 else "compress",
                 np.abs(got - ref).max() if ref.size else 0.0)
    assert err <= ATOL, f"compress max-abs {err}"
    return err


def check_compress_ex(gpu_out: torch.Tensor, x, z, P, cu, ratio, overlap, n_c, **extras):
    """The compressor variant (previous-half stream, RMSNorm, RoPE) against the oracle."""
    ref = oracle.compress_ex(x, z, P, cu, ratio, overlap, **extras)
    got = np32(gpu_out[:n_c]).astype(np.float64)
    if gpu_out.dtype == torch.bfloat16:
        return check_stored_bf16(got, ref, "compress_ex")
    err = record("compress_ex_fp32", np.abs(got - ref).max() if ref.size else 0.0)
    assert err <= ATOL, f"compress_ex max-abs {err}"
    return err


def check_topk(idx_gpu: np.ndarray, qI, w, kI, cu, ratio, topk, rows):
    """Compare GPU index rows (global compressed rows) with the oracle's on ``rows``."""
    idx_ref = oracle.indexer_topk(qI, w, kI, cu, ratio, topk, idx_gpu.shape[1], rows)
    bad = []
    mismatched_rows = 0
    for qi, row in enumerate(rows):
        g, o = idx_gpu[row], idx_ref[qi]
        if np.array_equal(g, o):
            continue
        mismatched_rows += 1
        # same count, same padding layout required; differing members must be near-ties
        ng, no = (g >= 0).sum(), (o >= 0).sum()
        assert ng == no, f"row {row}: {ng} selected vs oracle {no}"
        assert np.all(np.diff(g[:ng]) > 0), f"row {row}: not ascending"
        b = int(np.searchsorted(cu, row, side="right") - 1)
        cmp0 = int(oracle.compressed_offsets(cu, ratio)[b])
        nvis = (row - int(cu[b]) + 1) // ratio
        logits, _ = oracle.indexer_logits(qI, w, kI, cu, ratio, [row], max(nvis, 1))
        s = logits[0, :nvis]
        kth = np.sort(s)[::-1][min(topk, nvis) - 1]
        tol = TIE_RTOL * max(abs(kth), 1e-30)
        diff = np.setxor1d(g[:ng], o[:no]) - cmp0
        for j in diff:
            if abs(s[j] - kth) > tol:
                bad.append((row, int(j), float(s[j]), float(kth)))
    assert not bad, f"top-k mismatches beyond near-ties: {bad[:5]}"
    record("topk_rows_differing_by_near_ties", mismatched_rows)
    return mismatched_rows


def check_attention(kind, out, lse, lse_cmp, q, k_cmp, v_cmp, k_raw, v_raw, cu, ratio, window, scale, idx,
                    rows, sink=None):
    o_ref, lse_ref, lsec_ref, err = oracle.attention(kind, q, k_cmp, v_cmp, k_raw, v_raw, cu, ratio, window,
                                                     scale, idx=idx, sink=sink, rows=rows)
    assert not err.any(), "oracle saw out-of-range indices"
    o = np32(out[rows]).astype(np.float64)
    e_o = record("attention_out", np.abs(o - o_ref).max())
    l = np32(lse[rows]).astype(np.float64)
    fin = np.isfinite(lse_ref)
    assert np.array_equal(np.isfinite(l), fin), "lse finiteness differs"
    e_l = record("attention_lse", np.abs(l[fin] - lse_ref[fin]).max() if fin.any() else 0.0)
    e_c = 0.0
    if lse_cmp is not None:
        lc = np32(lse_cmp[rows]).astype(np.float64)
        finc = np.isfinite(lsec_ref)
        assert np.array_equal(np.isfinite(lc), finc), "lse_cmp finiteness differs"
        e_c = record("attention_lse_cmp", np.abs(lc[finc] - lsec_ref[finc]).max() if finc.any() else 0.0)
    assert e_o <= ATOL and e_l <= ATOL and e_c <= ATOL, f"attention errs o={e_o} lse={e_l} lse_cmp={e_c}"
    return e_o, e_l, e_c


def check_kl(kl_sum_gpu: float, kl_rows_gpu: np.ndarray, q, k_cmp, qI, w, kI, cu, ratio, scale, idx, rows,
             full: bool):
    kl_ref, csize, err = oracle.indexer_kl(q, k_cmp, qI, w, kI, cu, ratio, scale, idx=idx, rows=rows)
    assert not err.any()
    per = kl_rows_gpu[rows].astype(np.float64)
    e_rows = record("kl_rows", np.abs(per - kl_ref).max() if len(rows) else 0.0)
    # per-query values: absolute 1e-3 on O(1) quantities, sum: 1e-3 relative
    assert e_rows <= 1e-3 + KL_RTOL * np.abs(kl_ref).max(), f"per-query KL err {e_rows}"
    if full:
        ref_sum = kl_ref.sum()
        rel = record("kl_sum_rel", abs(kl_sum_gpu - ref_sum) / max(abs(ref_sum), 1e-30))
        assert rel <= KL_RTOL, f"KL sum rel err {rel} ({kl_sum_gpu} vs {ref_sum})"
        return rel
    return e_rows
