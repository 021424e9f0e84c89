"""Thin ctypes binding over libcsa.so.

Argument marshalling only: every step of the forward runs in the library's
CUDA kernels.  torch supplies device memory and the current stream.  The
functions carry the C names of include/csa.h and return the status code after
raising ``CSAError`` on a failure; outputs are written into the caller's
tensors.  Importing this module loads the library and fails loudly if it has
not been built (``compressed_sparse_attention_compress_gb300.build``).
"""
from __future__ import annotations

import ctypes
import os
import re

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libcsa.so")
HEADER = os.path.join(os.path.dirname(_HERE), "include", "csa.h")

CSA_BF16, CSA_FP32 = 0, 1
STATUS = {0: "CSA_OK", -1: "CSA_ERR_INVALID_ARG", -2: "CSA_ERR_UNSUPPORTED", -3: "CSA_ERR_WORKSPACE",
          -4: "CSA_ERR_CUDA", -5: "CSA_ERR_DEVICE_TIMEOUT", -6: "CSA_ERR_DEVICE_BOUNDS"}


class CSAError(RuntimeError):
    def __init__(self, name, code):
        super().__init__(f"{name} failed: {STATUS.get(code, code)}")
        self.code = code


def declared_symbols(header: str = HEADER) -> list:
    """Names of the functions include/csa.h declares."""
    text = open(header).read()
    return re.findall(r"^(?:csa_status_t|size_t|const char\*)\s+(\w+)\s*\(", text, flags=re.M)


def _load():
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                           "`python -m compressed_sparse_attention_compress_gb300.build`")
    lib = ctypes.CDLL(LIB_PATH)
    P, I, F, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    sig = {
        "csa_create": [I, P],
        "csa_destroy": [P],
        "csa_get_device_status": [P, P, P],
        "csa_set_position_offsets": [P, P, I],
        "csa_compressed_offsets": [P, P, I, I, P, P],
        "csa_compress": [P, P, P, P, P, P, I, I, I, I, I, I, I, P, P],
        "csa_compress_pair": [P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, I, P, P, P, P],
        "csa_compress_ex": [P, P, P, P, P, P, P, F, I, F, I, I, P, P, I, I, I, I, I, I, I, P, P],
        "csa_indexer_topk": [P, P, P, P, P, P, I, I, I, I, I, I, I, I, I, P, P],
        "csa_sparse_attn_fwd": [P, P, P, P, P, P, P, I, P, P, P, I, I, I, I, I, I, I, F, I, P, P, P, P],
        "hca_attn_fwd": [P, P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, F, I, P, P, P, P],
        "window_attn_fwd": [P, P, P, P, P, P, I, I, I, I, I, I, F, I, P, P, P],
        "csa_sparse_attn_bwd": [P, P, P, P, P, P, P, I, P, P, P, I, I, I, I, I, I, I, F, I, P, P, P, P, P, P, P, P,
                                P, P, P],
        "hca_attn_bwd": [P, P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, F, I, P, P, P, P, P, P, P, P, P, P, P],
        "window_attn_bwd": [P, P, P, P, P, P, I, I, I, I, I, I, F, I, P, P, P, P, P, P, P, P, P],
        "csa_indexer_kl_bwd": [P, P, P, P, P, P, P, I, P, P, P, P, I, I, I, I, I, I, I, I, F, F, I, P, P, P, P],
        "csa_indexer_kl_ex": [P, P, P, P, P, P, P, I, P, P, P, I, I, I, I, I, I, I, I, F, I, P, P, P, P, Z, P, P, P],
        "csa_quantize_fp8": [P, P, ctypes.c_int64, I, I, P, P, P],
        "csa_indexer_topk_fp8": [P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, I, I, P, P],
        "csa_indexer_kl": [P, P, P, P, P, P, P, I, P, P, P, I, I, I, I, I, I, I, I, F, I, P, P, P, P, Z, P],
        "csa_indexer_kl_static_scratch": [P, P, P, P, P, P, P, I, P, P, P, I, I, I, I, I, I, I, I, F, I, P, P, P, P],
    }
    for name, args in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = I
    lib.csa_status_string.argtypes = [I]
    lib.csa_status_string.restype = ctypes.c_char_p
    lib.csa_indexer_kl_workspace.argtypes = [I]
    lib.csa_indexer_kl_workspace.restype = Z
    return lib


LIB = _load()


def _p(t):
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors passed to libcsa must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _dtype(t) -> int:
    if t.dtype == torch.bfloat16:
        return CSA_BF16
    if t.dtype == torch.float32:
        return CSA_FP32
    raise TypeError(f"unsupported activation dtype {t.dtype}")


def _check(name, code):
    if code != 0:
        raise CSAError(name, code)
    return code


class Handle:
    """Owns a csa_handle_t (device properties + device status word)."""

    def __init__(self, device: int = 0):
        h = ctypes.c_void_p()
        _check("csa_create", LIB.csa_create(int(device), ctypes.byref(h)))
        self._h = h
        self.device = device

    @property
    def ptr(self):
        return self._h

    def device_status(self, stream=None) -> int:
        v = ctypes.c_int(0)
        _check("csa_get_device_status", LIB.csa_get_device_status(self._h, _stream(stream), ctypes.byref(v)))
        return v.value

    def set_position_offsets(self, pos0=None, cmp_rows: int = 0):
        """Per-sequence position of the first packed row (device int32 [B]) for the
        query calls made with this handle from now on; None restores 0."""
        _check("csa_set_position_offsets", LIB.csa_set_position_offsets(self._h, _p(pos0), int(cmp_rows)))

    def close(self):
        if self._h:
            LIB.csa_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def csa_compressed_offsets(h: Handle, cu_seqlens, ratio: int, cu_cmp, stream=None):
    B = cu_seqlens.numel() - 1
    return _check("csa_compressed_offsets",
                  LIB.csa_compressed_offsets(h.ptr, _p(cu_seqlens), B, int(ratio), _p(cu_cmp), _stream(stream)))


def csa_compress(h: Handle, x, z, pos_bias, cu_seqlens, cu_cmp, max_seqlen: int, ratio: int, overlap: bool,
                 out, stream=None):
    T_cap, D = x.shape
    return _check("csa_compress", LIB.csa_compress(
        h.ptr, _p(x), _p(z), _p(pos_bias), _p(cu_seqlens), _p(cu_cmp), cu_seqlens.numel() - 1, T_cap,
        int(max_seqlen), D, int(ratio), int(bool(overlap)), _dtype(x), _p(out), _stream(stream)))


def csa_compress_pair(h: Handle, x_kv, z_kv, pos_bias_kv, x_I, z_I, pos_bias_I, cu_seqlens, max_seqlen: int,
                      ratio: int, overlap: bool, cu_cmp, kv_cmp, kI_cmp, stream=None):
    """Both compressors of a layer and the compressed offsets in one launch."""
    T_cap, D = x_kv.shape
    d_I = x_I.shape[1]
    return _check("csa_compress_pair", LIB.csa_compress_pair(
        h.ptr, _p(x_kv), _p(z_kv), _p(pos_bias_kv), _p(x_I), _p(z_I), _p(pos_bias_I), _p(cu_seqlens),
        cu_seqlens.numel() - 1, T_cap, int(max_seqlen), D, d_I, int(ratio), int(bool(overlap)), _dtype(x_kv),
        _p(cu_cmp), _p(kv_cmp), _p(kI_cmp), _stream(stream)))


def csa_compress_ex(h: Handle, x, z, pos_bias, cu_seqlens, cu_cmp, max_seqlen: int, ratio: int, overlap: bool,
                    out, x_prev=None, z_prev=None, norm_weight=None, norm_eps: float = 1e-6, rope_dim: int = 0,
                    rope_theta: float = 10000.0, rope_pos_stride: int = 1, rope_pos_offset: int = 0, stream=None):
    T_cap, D = x.shape
    return _check("csa_compress_ex", LIB.csa_compress_ex(
        h.ptr, _p(x), _p(z), _p(x_prev), _p(z_prev), _p(pos_bias), _p(norm_weight), float(norm_eps),
        int(rope_dim), float(rope_theta), int(rope_pos_stride), int(rope_pos_offset), _p(cu_seqlens),
        _p(cu_cmp), cu_seqlens.numel() - 1, T_cap, int(max_seqlen), D, int(ratio), int(bool(overlap)),
        _dtype(x), _p(out), _stream(stream)))


def csa_indexer_topk(h: Handle, qI, w, kI, cu_seqlens, cu_cmp, max_seqlen: int, ratio: int, topk: int, idx,
                     stream=None):
    T_cap, H_I, d_I = qI.shape
    k_pad = idx.shape[1]
    return _check("csa_indexer_topk", LIB.csa_indexer_topk(
        h.ptr, _p(qI), _p(w), _p(kI), _p(cu_seqlens), _p(cu_cmp), cu_seqlens.numel() - 1, T_cap,
        int(max_seqlen), H_I, d_I, int(ratio), int(topk), k_pad, _dtype(qI), _p(idx), _stream(stream)))


def csa_sparse_attn_fwd(h: Handle, q, kv_cmp, kv_raw, idx, cu_seqlens, cu_cmp, max_seqlen: int, ratio: int,
                        window: int, softmax_scale: float, out, lse, lse_cmp=None, v_cmp=None, v_raw=None,
                        sink=None, stream=None):
    T_cap, H, d = q.shape
    return _check("csa_sparse_attn_fwd", LIB.csa_sparse_attn_fwd(
        h.ptr, _p(q), _p(kv_cmp), _p(v_cmp), _p(kv_raw), _p(v_raw), _p(idx), idx.shape[1], _p(sink),
        _p(cu_seqlens), _p(cu_cmp), cu_seqlens.numel() - 1, T_cap, int(max_seqlen), H, d, int(ratio),
        int(window), float(softmax_scale), _dtype(q), _p(out), _p(lse), _p(lse_cmp), _stream(stream)))


def hca_attn_fwd(h: Handle, q, kv_cmp, kv_raw, cu_seqlens, cu_cmp, max_seqlen: int, ratio: int, window: int,
                 softmax_scale: float, out, lse, lse_cmp=None, v_cmp=None, v_raw=None, sink=None, stream=None):
    T_cap, H, d = q.shape
    return _check("hca_attn_fwd", LIB.hca_attn_fwd(
        h.ptr, _p(q), _p(kv_cmp), _p(v_cmp), _p(kv_raw), _p(v_raw), _p(sink), _p(cu_seqlens), _p(cu_cmp),
        cu_seqlens.numel() - 1, T_cap, int(max_seqlen), H, d, int(ratio), int(window), float(softmax_scale),
        _dtype(q), _p(out), _p(lse), _p(lse_cmp), _stream(stream)))


def window_attn_fwd(h: Handle, q, kv_raw, cu_seqlens, max_seqlen: int, window: int, softmax_scale: float, out,
                    lse, v_raw=None, sink=None, stream=None):
    T_cap, H, d = q.shape
    return _check("window_attn_fwd", LIB.window_attn_fwd(
        h.ptr, _p(q), _p(kv_raw), _p(v_raw), _p(sink), _p(cu_seqlens), cu_seqlens.numel() - 1, T_cap,
        int(max_seqlen), H, d, int(window), float(softmax_scale), _dtype(q), _p(out), _p(lse), _stream(stream)))


def csa_sparse_attn_bwd(h: Handle, q, kv_cmp, kv_raw, idx, cu_seqlens, cu_cmp, max_seqlen: int, ratio: int,
                        window: int, softmax_scale: float, out, lse, dout, dq, dkv_cmp, dkv_raw, delta,
                        v_cmp=None, v_raw=None, dv_cmp=None, dv_raw=None, sink=None, dsink=None, stream=None):
    T_cap, H, d = q.shape
    return _check("csa_sparse_attn_bwd", LIB.csa_sparse_attn_bwd(
        h.ptr, _p(q), _p(kv_cmp), _p(v_cmp), _p(kv_raw), _p(v_raw), _p(idx), idx.shape[1], _p(sink),
        _p(cu_seqlens), _p(cu_cmp), cu_seqlens.numel() - 1, T_cap, int(max_seqlen), H, d, int(ratio),
        int(window), float(softmax_scale), _dtype(q), _p(out), _p(lse), _p(dout), _p(dq), _p(dkv_cmp),
        _p(dv_cmp), _p(dkv_raw), _p(dv_raw), _p(dsink), _p(delta), _stream(stream)))


def hca_attn_bwd(h: Handle, q, kv_cmp, kv_raw, cu_seqlens, cu_cmp, max_seqlen: int, ratio: int, window: int,
                 softmax_scale: float, out, lse, dout, dq, dkv_cmp, dkv_raw, delta, v_cmp=None, v_raw=None,
                 dv_cmp=None, dv_raw=None, sink=None, dsink=None, stream=None):
    T_cap, H, d = q.shape
    return _check("hca_attn_bwd", LIB.hca_attn_bwd(
        h.ptr, _p(q), _p(kv_cmp), _p(v_cmp), _p(kv_raw), _p(v_raw), _p(sink), _p(cu_seqlens), _p(cu_cmp),
        cu_seqlens.numel() - 1, T_cap, int(max_seqlen), H, d, int(ratio), int(window), float(softmax_scale),
        _dtype(q), _p(out), _p(lse), _p(dout), _p(dq), _p(dkv_cmp), _p(dv_cmp), _p(dkv_raw), _p(dv_raw),
        _p(dsink), _p(delta), _stream(stream)))


def window_attn_bwd(h: Handle, q, kv_raw, cu_seqlens, max_seqlen: int, window: int, softmax_scale: float, out,
                    lse, dout, dq, dkv_raw, delta, v_raw=None, dv_raw=None, sink=None, dsink=None, stream=None):
    T_cap, H, d = q.shape
    return _check("window_attn_bwd", LIB.window_attn_bwd(
        h.ptr, _p(q), _p(kv_raw), _p(v_raw), _p(sink), _p(cu_seqlens), cu_seqlens.numel() - 1, T_cap,
        int(max_seqlen), H, d, int(window), float(softmax_scale), _dtype(q), _p(out), _p(lse), _p(dout), _p(dq),
        _p(dkv_raw), _p(dv_raw), _p(dsink), _p(delta), _stream(stream)))


def csa_indexer_kl_workspace(T_cap: int) -> int:
    return int(LIB.csa_indexer_kl_workspace(int(T_cap)))


def csa_indexer_kl(h: Handle, q, kv_cmp, qI, w, kI, cu_seqlens, cu_cmp, max_seqlen: int, ratio: int,
                   softmax_scale: float, kl_sum, ws, idx=None, lse_cmp=None, kl_per_query=None, n_valid=None,
                   stream=None):
    T_cap, H, d = q.shape
    _, H_I, d_I = qI.shape
    k_pad = idx.shape[1] if idx is not None else 0
    return _check("csa_indexer_kl", LIB.csa_indexer_kl(
        h.ptr, _p(q), _p(kv_cmp), _p(qI), _p(w), _p(kI), _p(idx), k_pad, _p(lse_cmp), _p(cu_seqlens),
        _p(cu_cmp), cu_seqlens.numel() - 1, T_cap, int(max_seqlen), H, d, H_I, d_I, int(ratio),
        float(softmax_scale), _dtype(q), _p(kl_sum), _p(kl_per_query), _p(n_valid), _p(ws),
        ws.numel() * ws.element_size(), _stream(stream)))


def csa_indexer_kl_ex(h: Handle, q, kv_cmp, qI, w, kI, cu_seqlens, cu_cmp, max_seqlen: int, ratio: int,
                      softmax_scale: float, kl_sum, ws, teacher_lse=None, student_lse=None, idx=None, lse_cmp=None,
                      kl_per_query=None, n_valid=None, stream=None):
    T_cap, H, d = q.shape
    _, H_I, d_I = qI.shape
    k_pad = idx.shape[1] if idx is not None else 0
    return _check("csa_indexer_kl_ex", LIB.csa_indexer_kl_ex(
        h.ptr, _p(q), _p(kv_cmp), _p(qI), _p(w), _p(kI), _p(idx), k_pad, _p(lse_cmp), _p(cu_seqlens),
        _p(cu_cmp), cu_seqlens.numel() - 1, T_cap, int(max_seqlen), H, d, H_I, d_I, int(ratio),
        float(softmax_scale), _dtype(q), _p(kl_sum), _p(kl_per_query), _p(n_valid), _p(ws),
        ws.numel() * ws.element_size(), _p(teacher_lse), _p(student_lse), _stream(stream)))


def csa_indexer_kl_static_scratch(h: Handle, q, kv_cmp, qI, w, kI, cu_seqlens, cu_cmp, max_seqlen: int, ratio: int,
                                  softmax_scale: float, kl_sum, idx=None, lse_cmp=None, kl_per_query=None,
                                  n_valid=None, stream=None):
    """csa_indexer_kl without a workspace argument: the library's own static
    device scratch is used (for callers that cannot allocate device memory)."""
    T_cap, H, d = q.shape
    _, H_I, d_I = qI.shape
    k_pad = idx.shape[1] if idx is not None else 0
    return _check("csa_indexer_kl_static_scratch", LIB.csa_indexer_kl_static_scratch(
        h.ptr, _p(q), _p(kv_cmp), _p(qI), _p(w), _p(kI), _p(idx), k_pad, _p(lse_cmp), _p(cu_seqlens),
        _p(cu_cmp), cu_seqlens.numel() - 1, T_cap, int(max_seqlen), H, d, H_I, d_I, int(ratio),
        float(softmax_scale), _dtype(q), _p(kl_sum), _p(kl_per_query), _p(n_valid), _stream(stream)))


def csa_indexer_kl_bwd(h: Handle, q, kv_cmp, qI, w, kI, cu_seqlens, cu_cmp, max_seqlen: int, ratio: int,
                       softmax_scale: float, dqI, dw, dkI, idx=None, lse_cmp=None, grad_scale: float = 1.0,
                       student_lse=None, stream=None):
    T_cap, H, d = q.shape
    _, H_I, d_I = qI.shape
    k_pad = idx.shape[1] if idx is not None else 0
    return _check("csa_indexer_kl_bwd", LIB.csa_indexer_kl_bwd(
        h.ptr, _p(q), _p(kv_cmp), _p(qI), _p(w), _p(kI), _p(idx), k_pad, _p(lse_cmp), _p(student_lse),
        _p(cu_seqlens), _p(cu_cmp), cu_seqlens.numel() - 1, T_cap, int(max_seqlen), H, d, H_I, d_I, int(ratio),
        float(softmax_scale), float(grad_scale), _dtype(q), _p(dqI), _p(dw), _p(dkI), _stream(stream)))


def csa_quantize_fp8(h: Handle, x, codes, scales, stream=None):
    """E4M3 codes (uint8, x's shape) and per-row scales (float32, x.shape[:-1]) of x."""
    cols = x.shape[-1]
    return _check("csa_quantize_fp8", LIB.csa_quantize_fp8(
        h.ptr, _p(x), x.numel() // cols, cols, _dtype(x), _p(codes), _p(scales), _stream(stream)))


def csa_indexer_topk_fp8(h: Handle, qI, qI_scale, w, kI, kI_scale, cu_seqlens, cu_cmp, max_seqlen: int, ratio: int,
                         topk: int, idx, stream=None):
    T_cap, H_I, d_I = qI.shape
    return _check("csa_indexer_topk_fp8", LIB.csa_indexer_topk_fp8(
        h.ptr, _p(qI), _p(qI_scale), _p(w), _p(kI), _p(kI_scale), _p(cu_seqlens), _p(cu_cmp),
        cu_seqlens.numel() - 1, T_cap, int(max_seqlen), H_I, d_I, int(ratio), int(topk), idx.shape[1],
        _dtype(w), _p(idx), _stream(stream)))
