"""ctypes wrapper around the C oracle (``csa_oracle.c``).

Test infrastructure only (see the package docstring).  Every function takes
numpy arrays holding the exact values the GPU receives (bf16 values widened to
float32, float32 parameters) and returns float64 results.  Query-level
functions take an explicit list of packed query rows so that large workloads
can be checked on a sample of queries.

Definitions and citations are in ``csa_oracle.c``; the page is
"DeepSeek-V4 Attention Training Systems" (Megatron V4 notes).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "csa_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "libcsa_oracle.so")

KIND_CSA, KIND_HCA, KIND_WINDOW = 0, 1, 2

_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP when available).  Returns the .so path."""
    os.makedirs(_BUILD, exist_ok=True)
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= os.path.getmtime(_SRC):
        return _SO
    tmp = _SO + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math", "-ffp-contract=off"]
    try:
        subprocess.run(base + ["-fopenmp", _SRC, "-o", tmp, "-lm"], check=True,
                       capture_output=True, text=True)
    except subprocess.CalledProcessError:
        subprocess.run(base + [_SRC, "-o", tmp, "-lm"], check=True, capture_output=True, text=True)
    os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i32, i64, f64 = ctypes.c_int, ctypes.c_int64, ctypes.c_double
        lib.oracle_num_threads.restype = i32
        lib.oracle_set_num_threads.argtypes = [i32]
        lib.oracle_compressed_offsets.argtypes = [P, i32, i32, P]
        lib.oracle_compressed_offsets.restype = i64
        lib.oracle_compress.argtypes = [P, P, P, P, P, i32, i32, i32, i32, P]
        lib.oracle_compress_ex.argtypes = [P, P, P, P, P, P, ctypes.c_float, i32, f64, i64, i64, P, P,
                                           i32, i32, i32, i32, P]
        lib.oracle_indexer_logits.argtypes = [P, P, P, P, P, i32, i32, i32, i32, P, i32, i64, P, P]
        lib.oracle_indexer_topk.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i32, i32, P, i32, P]
        lib.oracle_attention.argtypes = [i32, P, P, P, P, P, P, i32, P, P, P, i32, i32, i32, i32,
                                         i32, f64, P, i32, P, P, P, P]
        lib.oracle_attention_bwd.argtypes = [i32, P, P, P, P, P, P, i32, P, P, P, i32, i32, i32, i32, i32,
                                             f64, P, P, i32, P, P, P, P, P, P, P]
        lib.oracle_indexer_kl.argtypes = [P, P, P, P, P, P, i32, P, P, i32, i32, i32, i32, i32,
                                          i32, f64, P, i32, P, P, P]
        lib.oracle_indexer_kl_bwd.argtypes = [P, P, P, P, P, P, i32, P, P, i32, i32, i32, i32, i32, i32,
                                              f64, f64, P, i32, P, P, P, P]
        lib.oracle_quantize_fp8.argtypes = [P, i64, i32, P, P]
        lib.oracle_e4m3_value.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_value.restype = f64
        _lib = lib
        return lib


def _f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


def _i32(a):
    return np.ascontiguousarray(a, dtype=np.int32)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def set_num_threads(n: int) -> None:
    _load().oracle_set_num_threads(int(n))


def _rows(rows, T):
    if rows is None:
        rows = np.arange(T, dtype=np.int64)
    return np.ascontiguousarray(rows, dtype=np.int64)


def compressed_offsets(cu_seqlens, ratio: int) -> np.ndarray:
    """cu_cmp[b] = sum over earlier sequences of floor(L_b / ratio)."""
    cu = _i32(cu_seqlens)
    B = cu.shape[0] - 1
    out = np.zeros(B + 1, dtype=np.int32)
    _load().oracle_compressed_offsets(_ptr(cu), B, int(ratio), _ptr(out))
    return out


def compress(x, z, P, cu_seqlens, ratio: int, overlap: bool) -> np.ndarray:
    """Softmax-gated block compression; returns float64 [N_c, D]."""
    x, z, P, cu = _f32(x), _f32(z), _f32(P), _i32(cu_seqlens)
    D = x.shape[1]
    S = 2 * ratio if overlap else ratio
    assert z.shape == x.shape and P.shape == (S, D)
    cu_cmp = compressed_offsets(cu, ratio)
    out = np.zeros((int(cu_cmp[-1]), D), dtype=np.float64)
    _load().oracle_compress(_ptr(x), _ptr(z), _ptr(P), _ptr(cu), _ptr(cu_cmp), cu.shape[0] - 1,
                            D, int(ratio), int(bool(overlap)), _ptr(out))
    return out


def compress_ex(x, z, P, cu_seqlens, ratio: int, overlap: bool, x_prev=None, z_prev=None,
                gamma=None, eps: float = 1e-6, rope_dim: int = 0, theta: float = 10000.0,
                pos_stride: int = 1, pos_offset: int = 0) -> np.ndarray:
    """Compressor variant: optional separate (x_prev, z_prev) stream for the
    previous-block half of an overlapping span, then RMSNorm (gamma), then RoPE
    on the trailing rope_dim channels; returns float64 [N_c, D]."""
    x, z, P, cu = _f32(x), _f32(z), _f32(P), _i32(cu_seqlens)
    D = x.shape[1]
    S = 2 * ratio if overlap else ratio
    assert z.shape == x.shape and P.shape == (S, D)
    x_prev = None if x_prev is None else _f32(x_prev)
    z_prev = None if z_prev is None else _f32(z_prev)
    assert (x_prev is None) == (z_prev is None)
    if x_prev is not None:
        assert x_prev.shape == x.shape and z_prev.shape == x.shape
    gamma = None if gamma is None else _f32(gamma)
    assert gamma is None or gamma.shape == (D,)
    assert 0 <= rope_dim <= D and rope_dim % 2 == 0
    cu_cmp = compressed_offsets(cu, ratio)
    out = np.zeros((int(cu_cmp[-1]), D), dtype=np.float64)
    _load().oracle_compress_ex(_ptr(x), _ptr(z), _ptr(x_prev), _ptr(z_prev), _ptr(P), _ptr(gamma),
                               float(eps), int(rope_dim), float(theta), int(pos_stride), int(pos_offset),
                               _ptr(cu), _ptr(cu_cmp), cu.shape[0] - 1, D, int(ratio),
                               int(bool(overlap)), _ptr(out))
    return out


def indexer_logits(qI, w, kI, cu_seqlens, ratio: int, rows, max_vis: int):
    """Indexer logits of the given query rows; returns (logits[nq, max_vis], nvis[nq])."""
    qI, w, kI, cu = _f32(qI), _f32(w), _f32(kI), _i32(cu_seqlens)
    T, H_I, dI = qI.shape
    rows = _rows(rows, T)
    cu_cmp = compressed_offsets(cu, ratio)
    logits = np.full((rows.shape[0], max_vis), np.nan, dtype=np.float64)
    nvis = np.zeros(rows.shape[0], dtype=np.int32)
    _load().oracle_indexer_logits(_ptr(qI), _ptr(w), _ptr(kI), _ptr(cu), _ptr(cu_cmp),
                                  cu.shape[0] - 1, H_I, dI, int(ratio), _ptr(rows),
                                  rows.shape[0], int(max_vis), _ptr(logits), _ptr(nvis))
    return logits, nvis


def indexer_topk(qI, w, kI, cu_seqlens, ratio: int, topk: int, k_pad: int, rows=None):
    """Top-k global compressed rows per query row (ascending, -1 padded): int32 [nq, k_pad]."""
    qI, w, kI, cu = _f32(qI), _f32(w), _f32(kI), _i32(cu_seqlens)
    T, H_I, dI = qI.shape
    rows = _rows(rows, T)
    cu_cmp = compressed_offsets(cu, ratio)
    idx = np.full((rows.shape[0], k_pad), -1, dtype=np.int32)
    _load().oracle_indexer_topk(_ptr(qI), _ptr(w), _ptr(kI), _ptr(cu), _ptr(cu_cmp),
                                cu.shape[0] - 1, H_I, dI, int(ratio), int(topk), int(k_pad),
                                _ptr(rows), rows.shape[0], _ptr(idx))
    return idx


def attention(kind: int, q, k_cmp, v_cmp, k_raw, v_raw, cu_seqlens, ratio: int, window: int,
              scale: float, idx=None, sink=None, rows=None):
    """Selected / HCA / window attention; returns (o[nq,H,d], lse[nq,H], lse_cmp[nq,H], err[nq]).

    ``idx`` is the full [T, k_pad] index array (indexed by packed row);
    ``k_cmp``/``v_cmp`` may be None for window-only attention.
    """
    q, k_raw, cu = _f32(q), _f32(k_raw), _i32(cu_seqlens)
    v_raw = k_raw if v_raw is None else _f32(v_raw)
    T, H, d = q.shape
    if k_cmp is None:
        k_cmp = np.zeros((1, d), np.float32)
    k_cmp = _f32(k_cmp)
    v_cmp = k_cmp if v_cmp is None else _f32(v_cmp)
    rows = _rows(rows, T)
    cu_cmp = compressed_offsets(cu, ratio if kind != KIND_WINDOW else 0)
    if kind == KIND_CSA:
        idx = _i32(idx)
        k_pad = idx.shape[1]
    else:
        idx, k_pad = None, 0
    sink = None if sink is None else _f32(sink)
    nq = rows.shape[0]
    o = np.zeros((nq, H, d), np.float64)
    lse = np.zeros((nq, H), np.float64)
    lse_cmp = np.zeros((nq, H), np.float64)
    err = np.zeros(nq, np.int32)
    _load().oracle_attention(int(kind), _ptr(q), _ptr(k_cmp), _ptr(v_cmp), _ptr(k_raw),
                             _ptr(v_raw), _ptr(idx), int(k_pad), _ptr(sink), _ptr(cu),
                             _ptr(cu_cmp), cu.shape[0] - 1, H, d, int(ratio), int(window),
                             float(scale), _ptr(rows), nq, _ptr(o), _ptr(lse), _ptr(lse_cmp),
                             _ptr(err))
    return o, lse, lse_cmp, err


def attention_bwd(kind: int, q, k_cmp, v_cmp, k_raw, v_raw, cu_seqlens, ratio: int, window: int,
                  scale: float, dout, idx=None, sink=None, rows=None, want_kv: bool = True):
    """Gradients of the attention forward for upstream ``dout`` [T, H, d].

    Returns a dict: ``dq`` [nq, H, d] for the given rows, and (``want_kv``) the
    key / value gradients accumulated over those rows -- ``dk_cmp``, ``dv_cmp``
    [rows of k_cmp, d], ``dk_raw``, ``dv_raw`` [T, d] -- and ``dsink`` [H]
    (None without a sink), plus ``err`` [nq].  With K = V (v_cmp / v_raw None)
    the gradient of the shared array is dk + dv.
    """
    q, k_raw, cu, dout = _f32(q), _f32(k_raw), _i32(cu_seqlens), _f32(dout)
    v_raw = k_raw if v_raw is None else _f32(v_raw)
    T, H, d = q.shape
    if k_cmp is None:
        k_cmp = np.zeros((1, d), np.float32)
    k_cmp = _f32(k_cmp)
    v_cmp = k_cmp if v_cmp is None else _f32(v_cmp)
    rows = _rows(rows, T)
    cu_cmp = compressed_offsets(cu, ratio if kind != KIND_WINDOW else 0)
    if kind == KIND_CSA:
        idx = _i32(idx)
        k_pad = idx.shape[1]
    else:
        idx, k_pad = None, 0
    sink = None if sink is None else _f32(sink)
    nq = rows.shape[0]
    dq = np.zeros((nq, H, d), np.float64)
    out = {"dq": dq}
    if want_kv:
        out["dk_cmp"] = np.zeros(k_cmp.shape, np.float64)
        out["dv_cmp"] = np.zeros(v_cmp.shape, np.float64)
        out["dk_raw"] = np.zeros(k_raw.shape, np.float64)
        out["dv_raw"] = np.zeros(v_raw.shape, np.float64)
        out["dsink"] = np.zeros(H, np.float64) if sink is not None else None
    err = np.zeros(nq, np.int32)
    g = out.get
    _load().oracle_attention_bwd(int(kind), _ptr(q), _ptr(k_cmp), _ptr(v_cmp), _ptr(k_raw), _ptr(v_raw),
                                 _ptr(idx), int(k_pad), _ptr(sink), _ptr(cu), _ptr(cu_cmp), cu.shape[0] - 1, H, d,
                                 int(ratio), int(window), float(scale), _ptr(dout), _ptr(rows), nq, _ptr(dq),
                                 _ptr(g("dk_cmp")), _ptr(g("dv_cmp")), _ptr(g("dk_raw")), _ptr(g("dv_raw")),
                                 _ptr(g("dsink")), _ptr(err))
    out["err"] = err
    return out


def indexer_kl(q, k_cmp, qI, w, kI, cu_seqlens, ratio: int, scale: float, idx=None, rows=None):
    """Indexer KL per query row; returns (kl[nq], csize[nq], err[nq]).  idx None = dense teacher."""
    q, k_cmp, qI, w, kI, cu = _f32(q), _f32(k_cmp), _f32(qI), _f32(w), _f32(kI), _i32(cu_seqlens)
    T, H, d = q.shape
    _, H_I, dI = qI.shape
    rows = _rows(rows, T)
    cu_cmp = compressed_offsets(cu, ratio)
    if idx is not None:
        idx = _i32(idx)
        k_pad = idx.shape[1]
    else:
        k_pad = 0
    nq = rows.shape[0]
    kl = np.zeros(nq, np.float64)
    csize = np.zeros(nq, np.int32)
    err = np.zeros(nq, np.int32)
    _load().oracle_indexer_kl(_ptr(q), _ptr(k_cmp), _ptr(qI), _ptr(w), _ptr(kI), _ptr(idx),
                              int(k_pad), _ptr(cu), _ptr(cu_cmp), cu.shape[0] - 1, H, d, H_I, dI,
                              int(ratio), float(scale), _ptr(rows), nq, _ptr(kl), _ptr(csize),
                              _ptr(err))
    return kl, csize, err


def indexer_kl_bwd(q, k_cmp, qI, w, kI, cu_seqlens, ratio: int, scale: float, idx=None, rows=None,
                   grad_scale: float = 1.0, want_kI: bool = True):
    """Gradients of the indexer KL loss (teacher detached) for upstream
    ``grad_scale``: dict with ``dqI`` [nq, H_I, dI], ``dw`` [nq, H_I], ``dkI``
    [rows of kI, dI] (accumulated over the given rows; None unless want_kI)
    and ``err`` [nq].  idx None = dense teacher over every visible entry."""
    q, k_cmp, qI, w, kI, cu = _f32(q), _f32(k_cmp), _f32(qI), _f32(w), _f32(kI), _i32(cu_seqlens)
    T, H, d = q.shape
    _, H_I, dI = qI.shape
    rows = _rows(rows, T)
    cu_cmp = compressed_offsets(cu, ratio)
    if idx is not None:
        idx = _i32(idx)
        k_pad = idx.shape[1]
    else:
        k_pad = 0
    nq = rows.shape[0]
    dqI = np.zeros((nq, H_I, dI), np.float64)
    dw = np.zeros((nq, H_I), np.float64)
    dkI = np.zeros(kI.shape, np.float64) if want_kI else None
    err = np.zeros(nq, np.int32)
    _load().oracle_indexer_kl_bwd(_ptr(q), _ptr(k_cmp), _ptr(qI), _ptr(w), _ptr(kI), _ptr(idx), int(k_pad),
                                  _ptr(cu), _ptr(cu_cmp), cu.shape[0] - 1, H, d, H_I, dI, int(ratio), float(scale),
                                  float(grad_scale), _ptr(rows), nq, _ptr(dqI), _ptr(dw), _ptr(dkI), _ptr(err))
    return {"dqI": dqI, "dw": dw, "dkI": dkI, "err": err}


def quantize_fp8(x):
    """Per-row E4M3 codes (uint8 [rows, cols]) and power-of-two scales (float32 [rows])
    of a float32 array viewed as [rows, cols] (cols = its last dimension)."""
    x = _f32(x)
    cols = x.shape[-1]
    flat = x.reshape(-1, cols)
    codes = np.zeros(flat.shape, np.uint8)
    scales = np.zeros(flat.shape[0], np.float32)
    _load().oracle_quantize_fp8(_ptr(flat), flat.shape[0], cols, _ptr(codes), _ptr(scales))
    return codes.reshape(x.shape), scales.reshape(x.shape[:-1])


def e4m3_value(code: int) -> float:
    return float(_load().oracle_e4m3_value(int(code)))


def dequantize_fp8(codes, scales) -> np.ndarray:
    """codes * scale as float32 (exact: the scale is a power of two)."""
    table = np.array([e4m3_value(c) for c in range(256)], np.float64)
    return (table[np.asarray(codes)] * np.asarray(scales, np.float64)[..., None]).astype(np.float32)
