"""Seeded synthetic inputs shared by the CUDA path's tests/benchmark and the oracle tests.

This module draws random numbers and rounds them to bf16; it holds none of the
method's arithmetic.  Every tensor comes from its own ``numpy`` generator
stream, spawned in a fixed order from ``SeedSequence(seed)``:

    x_kv, z_kv, P_kv, x_I, z_I, P_I, q, qI, w, v,
    x_kv_prev, z_kv_prev, x_I_prev, z_I_prev, g_kv, g_I

Each bf16 tensor is ``standard_normal`` float32 rounded to bf16
(round-to-nearest-even); the rounded values are what both the GPU and the
oracle consume.  The compressor positional biases ``P_kv``/``P_I`` are float32
parameters and are not rounded.  Workloads with the DeepSeek-V4 style
compressor (``compressor="v4"``) also draw the previous-half projections
``*_prev`` (overlapping spans) and the float32 RMSNorm gains ``g_kv``/``g_I``
as 1 + 0.1 N(0, 1).

Workloads follow the shapes of the DeepSeek-V4 CSA/HCA layers described in
"DeepSeek-V4 Attention Training Systems" (§2 phase table, §4 THD packing,
§5.1 spans and window): ratio 4 with an overlapping span of 8 tokens for CSA,
ratio 128 with a span of 128 for HCA, a local window of 128 raw tokens.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

STREAMS = ("x_kv", "z_kv", "P_kv", "x_I", "z_I", "P_I", "q", "qI", "w", "v",
           "x_kv_prev", "z_kv_prev", "x_I_prev", "z_I_prev", "g_kv", "g_I")


def bf16_bits(a: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns (uint16), round-to-nearest-even; NaN kept quiet."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32)
    rounded = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    nan = np.isnan(a)
    if nan.any():
        rounded = np.where(nan, (u >> np.uint32(16)) | np.uint32(0x40), rounded)
    return rounded.astype(np.uint16)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float32 (exact)."""
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def bf16_round(a: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bf16 value, returned as float32."""
    return bf16_to_f32(bf16_bits(a))


@dataclass
class Workload:
    """Shape description of one synthetic workload."""
    name: str
    lengths: list            # per-sequence token counts
    ratio: int               # compression ratio r (0 = window-only layer)
    overlap: bool            # overlapping span (2r) or not (r)
    H: int                   # query heads (one shared KV head)
    d: int                   # head dim
    window: int              # local window W
    H_I: int = 0             # indexer heads (0 = no indexer)
    d_I: int = 0             # indexer head dim
    topk: int = 0
    k_pad: int = 0
    separate_v: bool = False # separate value stream (else K = V)
    io_fp32: bool = False    # float32 I/O arrays holding bf16 values
    kl_mode: str = "none"    # "sparse" (selected set), "dense" (all visible) or "none"
    cap_align: int = 1       # T_cap = total rounded up to this
    compressor: str = "plain"  # "plain" gate only; "v4": previous-half stream + RMSNorm + RoPE
    indexer: str = "bf16"      # "bf16" or "fp8" (E4M3 operands with per-row scales) for scoring + top-k
    notes: str = ""
    extra: dict = field(default_factory=dict)

    @property
    def B(self) -> int:
        return len(self.lengths)

    @property
    def T(self) -> int:
        return int(sum(self.lengths))

    @property
    def T_cap(self) -> int:
        a = self.cap_align
        return ((self.T + a - 1) // a) * a

    @property
    def cu_seqlens(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.lengths)]).astype(np.int32)

    @property
    def span(self) -> int:
        return (2 * self.ratio if self.overlap else self.ratio) if self.ratio > 0 else 0

    @property
    def scale(self) -> float:
        return 1.0 / float(np.sqrt(self.d))

    # compressor extras of the "v4" compressor: RMSNorm eps, RoPE band and base
    norm_eps = 1e-6
    rope_theta = 10000.0

    @property
    def rope_kv(self) -> int:
        return min(64, self.d // 2)

    @property
    def rope_I(self) -> int:
        return min(64, self.d_I // 2)

    @property
    def n_cmp(self) -> int:
        return int(sum(L // self.ratio for L in self.lengths)) if self.ratio > 0 else 0


def _thd_lengths(seed: int = 0, n: int = 16, lo: int = 1024, hi: int = 16384) -> list:
    return [int(v) for v in np.random.default_rng(seed).integers(lo, hi + 1, n)]


WORKLOADS = {
    # one sequence L=512, r=4, 4 heads x 64, indexer 2 x 32, top-k 16, W=64, fp32 I/O
    "tiny": Workload("tiny", [512], 4, True, 4, 64, 64, H_I=2, d_I=32, topk=16, k_pad=16,
                     separate_v=True, io_fp32=True, kl_mode="sparse"),
    # CSA sparse mode: L=8192, r=4, 64 x 128, indexer 8 x 64, top-k 512, W=128
    "csa8k": Workload("csa8k", [8192], 4, True, 64, 128, 128, H_I=8, d_I=64, topk=512,
                      k_pad=512, kl_mode="sparse"),
    # HCA: L=65536, r=128 (no overlap), 64 x 128, W=128, no indexer
    "hca64k": Workload("hca64k", [65536], 128, False, 64, 128, 128),
    # packed THD varlen CSA: 16 sequences, lengths uniform in [1024, 16384] from seed 0
    "thd128k": Workload("thd128k", _thd_lengths(), 4, True, 64, 128, 128, H_I=8, d_I=64,
                        topk=1024, k_pad=1024, kl_mode="none", cap_align=128),
    # the sparse warm-up layer at L=8192 with k=512 (a small case of the headline
    # layer for profiling and parity: every query past 2048 tokens runs the selection)
    "warmup8k": Workload("warmup8k", [8192], 4, True, 64, 128, 128, H_I=8, d_I=64,
                         topk=512, k_pad=512, kl_mode="dense"),
    # sparse warm-up: L=32768, r=4, 64 x 128, indexer 8 x 64, top-k 2048, W=128,
    # sparse main output + dense teacher over all visible entries
    "warmup32k": Workload("warmup32k", [32768], 4, True, 64, 128, 128, H_I=8, d_I=64,
                          topk=2048, k_pad=2048, kl_mode="dense"),
}


def custom(name="custom", **kw) -> Workload:
    """A workload with explicit fields (tests use small ragged shapes)."""
    return Workload(name=name, **kw)


def generate(wl: Workload, seed: int = 0) -> dict:
    """Draw every input stream of ``wl`` (float32 arrays holding bf16 values).

    Returns a dict with the arrays and ``cu_seqlens``.  Streams the workload
    does not use are not drawn (their generator is still spawned so that the
    other streams do not move).
    """
    ss = np.random.SeedSequence(seed).spawn(len(STREAMS))
    gens = {name: np.random.default_rng(s) for name, s in zip(STREAMS, ss)}
    T = wl.T_cap
    out = {"cu_seqlens": wl.cu_seqlens}

    def normal(name, shape, round_bf16=True):
        a = gens[name].standard_normal(shape, dtype=np.float32)
        return bf16_round(a) if round_bf16 else a

    out["x_kv"] = normal("x_kv", (T, wl.d))
    if wl.ratio > 0:
        out["z_kv"] = normal("z_kv", (T, wl.d))
        out["P_kv"] = normal("P_kv", (wl.span, wl.d), round_bf16=False)
    if wl.H_I > 0:
        out["x_I"] = normal("x_I", (T, wl.d_I))
        out["z_I"] = normal("z_I", (T, wl.d_I))
        out["P_I"] = normal("P_I", (wl.span, wl.d_I), round_bf16=False)
    out["q"] = normal("q", (T, wl.H, wl.d))
    if wl.H_I > 0:
        out["qI"] = normal("qI", (T, wl.H_I, wl.d_I))
        out["w"] = normal("w", (T, wl.H_I))
    if wl.separate_v:
        out["v"] = normal("v", (T, wl.d))
    if wl.compressor == "v4" and wl.ratio > 0:
        if wl.overlap:
            out["x_kv_prev"] = normal("x_kv_prev", (T, wl.d))
            out["z_kv_prev"] = normal("z_kv_prev", (T, wl.d))
        out["g_kv"] = 1.0 + 0.1 * normal("g_kv", (wl.d,), round_bf16=False)
        if wl.H_I > 0:
            if wl.overlap:
                out["x_I_prev"] = normal("x_I_prev", (T, wl.d_I))
                out["z_I_prev"] = normal("z_I_prev", (T, wl.d_I))
            out["g_I"] = 1.0 + 0.1 * normal("g_I", (wl.d_I,), round_bf16=False)
    return out


COMPRESS_EX_STREAMS = ("x", "z", "x_prev", "z_prev", "P", "gamma")


def generate_compress_ex(lengths, D: int, ratio: int, overlap: bool, two: bool, seed: int = 0,
                         cap_align: int = 1) -> dict:
    """Inputs of the compressor variant: bf16-valued x, z (and x_prev, z_prev
    when ``two``) [T_cap, D] standard normal, a float32 positional bias [S, D]
    standard normal and a float32 RMSNorm gain [D] drawn as 1 + 0.1 N(0, 1).
    Each stream has its own generator spawned from ``SeedSequence(seed)``."""
    ss = np.random.SeedSequence(seed).spawn(len(COMPRESS_EX_STREAMS))
    gens = {name: np.random.default_rng(s) for name, s in zip(COMPRESS_EX_STREAMS, ss)}
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    T = int(cu[-1])
    T_cap = ((T + cap_align - 1) // cap_align) * cap_align
    S = 2 * ratio if overlap else ratio
    out = {"cu_seqlens": cu}
    for name in ("x", "z") + (("x_prev", "z_prev") if two else ()):
        out[name] = bf16_round(gens[name].standard_normal((T_cap, D), dtype=np.float32))
    out["P"] = gens["P"].standard_normal((S, D), dtype=np.float32)
    out["gamma"] = (1.0 + 0.1 * gens["gamma"].standard_normal(D)).astype(np.float32)
    return out


ATTN_BWD_STREAMS = ("q", "k_cmp", "k_raw", "v_cmp", "v_raw", "sel", "sink", "dout")


def random_index_sets(lengths, ratio: int, topk: int, k_pad: int, rng, T_cap: int | None = None) -> np.ndarray:
    """[T_cap, k_pad] int32: for every query a uniformly random set of
    min(topk, |V_t|) of its visible compressed entries (global rows, ascending,
    -1 padded); capacity rows are all -1.  Drawn as the smallest of per-entry
    uniform keys, a block of queries at a time."""
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    cu_cmp = np.concatenate([[0], np.cumsum([L // ratio for L in lengths])]).astype(np.int64)
    T = int(cu[-1])
    idx = np.full((T if T_cap is None else T_cap, k_pad), -1, np.int32)
    for b, L in enumerate(lengths):
        n_b = L // ratio
        if n_b == 0:
            continue
        for t0 in range(0, L, 256):
            t = np.arange(t0, min(L, t0 + 256))
            nvis = (t + 1) // ratio
            keys = rng.random((t.size, n_b))
            keys[np.arange(n_b)[None, :] >= nvis[:, None]] = 2.0   # not visible
            m = min(topk, n_b)
            part = np.argpartition(keys, m - 1, axis=1)[:, :m] if m < n_b else np.tile(np.arange(n_b), (t.size, 1))
            for i, tt in enumerate(t):
                c = part[i][keys[i, part[i]] < 2.0]
                c.sort()
                idx[cu[b] + tt, :c.size] = cu_cmp[b] + c
    return idx


def generate_attention_bwd(lengths, H: int, d: int, ratio: int, topk: int = 0, k_pad: int = 0,
                           separate_v: bool = False, sink: bool = False, seed: int = 0, cap_align: int = 1) -> dict:
    """Inputs of an attention backward test: bf16-valued q, dout [T_cap, H, d],
    compressed and raw key (and value) rows, a random valid index set per
    query (``topk`` > 0) and a float32 sink [H].  One generator per stream
    spawned from ``SeedSequence(seed)``."""
    ss = np.random.SeedSequence(seed).spawn(len(ATTN_BWD_STREAMS))
    gens = {name: np.random.default_rng(s) for name, s in zip(ATTN_BWD_STREAMS, ss)}
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    T = int(cu[-1])
    T_cap = ((T + cap_align - 1) // cap_align) * cap_align
    n_cap = max(1, T_cap // ratio) if ratio > 0 else 1
    out = {"cu_seqlens": cu}

    def normal(name, shape):
        return bf16_round(gens[name].standard_normal(shape, dtype=np.float32))

    out["q"] = normal("q", (T_cap, H, d))
    out["dout"] = normal("dout", (T_cap, H, d))
    out["k_raw"] = normal("k_raw", (T_cap, d))
    out["k_cmp"] = normal("k_cmp", (n_cap, d))
    if separate_v:
        out["v_raw"] = normal("v_raw", (T_cap, d))
        out["v_cmp"] = normal("v_cmp", (n_cap, d))
    if sink:
        out["sink"] = gens["sink"].standard_normal(H, dtype=np.float32)
    if topk > 0:
        out["idx"] = random_index_sets(lengths, ratio, topk, k_pad, gens["sel"], T_cap)
    return out


INDEXER_BWD_STREAMS = ("q", "k_cmp", "qI", "w", "k_I", "sel", "k_raw")


def generate_indexer_bwd(lengths, H: int, d: int, H_I: int, d_I: int, ratio: int, topk: int = 0, k_pad: int = 0,
                         seed: int = 0, cap_align: int = 1) -> dict:
    """Inputs of an indexer backward test: bf16-valued q [T_cap, H, d], compressed
    main KV [n_cap, d], qI [T_cap, H_I, d_I], w [T_cap, H_I], indexer keys
    [n_cap, d_I], raw KV rows [T_cap, d] (for the forward that gives lse_cmp)
    and, with ``topk`` > 0, a random valid index set per query."""
    ss = np.random.SeedSequence(seed).spawn(len(INDEXER_BWD_STREAMS))
    gens = {name: np.random.default_rng(s) for name, s in zip(INDEXER_BWD_STREAMS, ss)}
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    T = int(cu[-1])
    T_cap = ((T + cap_align - 1) // cap_align) * cap_align
    n_cap = max(1, T_cap // ratio)

    def normal(name, shape):
        return bf16_round(gens[name].standard_normal(shape, dtype=np.float32))

    out = {"cu_seqlens": cu, "q": normal("q", (T_cap, H, d)), "k_cmp": normal("k_cmp", (n_cap, d)),
           "qI": normal("qI", (T_cap, H_I, d_I)), "w": normal("w", (T_cap, H_I)),
           "k_I": normal("k_I", (n_cap, d_I)), "k_raw": normal("k_raw", (T_cap, d))}
    if topk > 0:
        out["idx"] = random_index_sets(lengths, ratio, topk, k_pad, gens["sel"], T_cap)
    return out
