"""One full CSA / HCA / window-only forward through the C ABI.

``Forward`` holds the device buffers of one workload (capacity-sized, as the
static-capacity contract of "DeepSeek-V4 Attention Training Systems" §4.1
asks) and enqueues the calls in the order of the page's fused training
forward (§8.2): compress main KV and indexer K, indexer score + top-k,
selected attention (O, LSE), indexer KL.  HCA layers skip the indexer; window
layers skip the compressor too.  Every step is a libcsa.so kernel; this class
only allocates buffers and passes pointers.
"""
from __future__ import annotations

import math

import torch

from . import api


class Forward:
    def __init__(self, wl, inputs: dict, device: int = 0, handle: api.Handle | None = None):
        """``inputs``: torch tensors on the device (bf16, or float32 when wl.io_fp32)."""
        self.wl = wl
        self.dev = torch.device("cuda", device)
        self.h = handle or api.Handle(device)
        self.x = inputs
        if wl.compressor == "v4" and wl.separate_v:
            raise ValueError("the v4 compressor takes K = V (one compressed KV stream)")
        dt = torch.float32 if wl.io_fp32 else torch.bfloat16
        T, H, d = wl.T_cap, wl.H, wl.d
        self.cu = inputs["cu_seqlens"]
        self.max_seqlen = max(wl.lengths) if wl.lengths else 0
        self.scale = 1.0 / math.sqrt(d)
        B = wl.B
        if wl.ratio > 0:
            n_cap = max(1, T // wl.ratio)
            self.cu_cmp = torch.zeros(B + 1, dtype=torch.int32, device=self.dev)
            self.kv_cmp = torch.zeros(n_cap, d, dtype=dt, device=self.dev)
            self.v_cmp = torch.zeros(n_cap, d, dtype=dt, device=self.dev) if wl.separate_v else None
            if wl.H_I > 0:
                self.kI = torch.zeros(n_cap, wl.d_I, dtype=dt, device=self.dev)
                self.idx = torch.empty(T, wl.k_pad, dtype=torch.int32, device=self.dev)
        self.out = torch.empty(T, H, d, dtype=dt, device=self.dev)
        self.lse = torch.empty(T, H, dtype=torch.float32, device=self.dev)
        self.lse_cmp = torch.empty(T, H, dtype=torch.float32, device=self.dev) if wl.ratio > 0 else None
        if wl.kl_mode != "none":
            self.kl_sum = torch.zeros(1, dtype=torch.float32, device=self.dev)
            self.kl_rows = torch.zeros(T, dtype=torch.float32, device=self.dev)
            self.n_valid = torch.zeros(1, dtype=torch.int32, device=self.dev)
            self.ws = torch.empty(api.csa_indexer_kl_workspace(T), dtype=torch.uint8, device=self.dev)

    # individual stages -----------------------------------------------------
    def compress(self, stream=None):
        wl, x = self.wl, self.x
        if (wl.compressor != "v4" and self.v_cmp is None and wl.H_I > 0
                and (wl.d, wl.d_I) in ((128, 64), (64, 32))):
            # both compressors and the compressed offsets in one launch
            api.csa_compress_pair(self.h, x["x_kv"], x["z_kv"], x["P_kv"], x["x_I"], x["z_I"], x["P_I"], self.cu,
                                  self.max_seqlen, wl.ratio, wl.overlap, self.cu_cmp, self.kv_cmp, self.kI, stream)
            return
        api.csa_compressed_offsets(self.h, self.cu, wl.ratio, self.cu_cmp, stream)
        if wl.compressor == "v4":
            # previous-half stream (overlapping spans), RMSNorm and RoPE fused in
            api.csa_compress_ex(self.h, x["x_kv"], x["z_kv"], x["P_kv"], self.cu, self.cu_cmp, self.max_seqlen,
                                wl.ratio, wl.overlap, self.kv_cmp, x_prev=x.get("x_kv_prev"),
                                z_prev=x.get("z_kv_prev"), norm_weight=x["g_kv"], norm_eps=wl.norm_eps,
                                rope_dim=wl.rope_kv, rope_theta=wl.rope_theta, stream=stream)
            if wl.H_I > 0:
                api.csa_compress_ex(self.h, x["x_I"], x["z_I"], x["P_I"], self.cu, self.cu_cmp, self.max_seqlen,
                                    wl.ratio, wl.overlap, self.kI, x_prev=x.get("x_I_prev"),
                                    z_prev=x.get("z_I_prev"), norm_weight=x["g_I"], norm_eps=wl.norm_eps,
                                    rope_dim=wl.rope_I, rope_theta=wl.rope_theta, stream=stream)
            return
        api.csa_compress(self.h, x["x_kv"], x["z_kv"], x["P_kv"], self.cu, self.cu_cmp, self.max_seqlen,
                         wl.ratio, wl.overlap, self.kv_cmp, stream)
        if self.v_cmp is not None:
            api.csa_compress(self.h, x["v"], x["z_kv"], x["P_kv"], self.cu, self.cu_cmp, self.max_seqlen,
                             wl.ratio, wl.overlap, self.v_cmp, stream)
        if wl.H_I > 0:
            api.csa_compress(self.h, x["x_I"], x["z_I"], x["P_I"], self.cu, self.cu_cmp, self.max_seqlen,
                             wl.ratio, wl.overlap, self.kI, stream)

    def topk(self, stream=None):
        wl, x = self.wl, self.x
        if wl.indexer == "fp8":
            if getattr(self, "qI8", None) is None:
                self.qI8 = torch.empty(x["qI"].shape, dtype=torch.uint8, device=self.dev)
                self.qIs = torch.empty(x["qI"].shape[:-1], dtype=torch.float32, device=self.dev)
                self.kI8 = torch.empty(self.kI.shape, dtype=torch.uint8, device=self.dev)
                self.kIs = torch.empty(self.kI.shape[:-1], dtype=torch.float32, device=self.dev)
            api.csa_quantize_fp8(self.h, x["qI"], self.qI8, self.qIs, stream)
            api.csa_quantize_fp8(self.h, self.kI, self.kI8, self.kIs, stream)
            api.csa_indexer_topk_fp8(self.h, self.qI8, self.qIs, x["w"], self.kI8, self.kIs, self.cu, self.cu_cmp,
                                     self.max_seqlen, wl.ratio, wl.topk, self.idx, stream)
            return
        api.csa_indexer_topk(self.h, x["qI"], x["w"], self.kI, self.cu, self.cu_cmp, self.max_seqlen, wl.ratio,
                             wl.topk, self.idx, stream)

    def attend(self, stream=None, sink=None):
        wl, x = self.wl, self.x
        v_raw = x.get("v") if wl.separate_v else None
        if wl.ratio == 0:
            api.window_attn_fwd(self.h, x["q"], x["x_kv"], self.cu, self.max_seqlen, wl.window, self.scale,
                                self.out, self.lse, v_raw=v_raw, sink=sink, stream=stream)
        elif wl.H_I > 0:
            api.csa_sparse_attn_fwd(self.h, x["q"], self.kv_cmp, x["x_kv"], self.idx, self.cu, self.cu_cmp,
                                    self.max_seqlen, wl.ratio, wl.window, self.scale, self.out, self.lse,
                                    self.lse_cmp, v_cmp=self.v_cmp, v_raw=v_raw, sink=sink, stream=stream)
        else:
            api.hca_attn_fwd(self.h, x["q"], self.kv_cmp, x["x_kv"], self.cu, self.cu_cmp, self.max_seqlen,
                             wl.ratio, wl.window, self.scale, self.out, self.lse, self.lse_cmp,
                             v_cmp=self.v_cmp, v_raw=v_raw, sink=sink, stream=stream)

    keep_stats = False   # kl() keeps the normalisers for indexer_backward by default

    def kl(self, stream=None, save_stats: bool | None = None):
        """The indexer KL loss; with ``save_stats`` (default ``keep_stats``) it also
        keeps the teacher's and the student's log normalisers for
        ``indexer_backward``, which then takes one pass instead of two."""
        wl, x = self.wl, self.x
        save_stats = self.keep_stats if save_stats is None else save_stats
        sparse = wl.kl_mode == "sparse"
        # the teacher computes its own exact normaliser; the attention's lse_cmp (that of
        # its bf16-rounded weights) serves as the reference of that computation
        kw = dict(idx=self.idx if sparse else None, lse_cmp=self.lse_cmp if sparse else None,
                  kl_per_query=self.kl_rows, n_valid=self.n_valid, stream=stream)
        if not save_stats:
            api.csa_indexer_kl(self.h, x["q"], self.kv_cmp, x["qI"], x["w"], self.kI, self.cu, self.cu_cmp,
                               self.max_seqlen, wl.ratio, self.scale, self.kl_sum, self.ws, **kw)
            return
        if getattr(self, "teacher_lse", None) is None:
            self.teacher_lse = torch.empty(wl.T_cap, wl.H, dtype=torch.float32, device=self.dev)
            self.student_lse = torch.empty(wl.T_cap, dtype=torch.float32, device=self.dev)
        api.csa_indexer_kl_ex(self.h, x["q"], self.kv_cmp, x["qI"], x["w"], self.kI, self.cu, self.cu_cmp,
                              self.max_seqlen, wl.ratio, self.scale, self.kl_sum, self.ws,
                              teacher_lse=self.teacher_lse, student_lse=self.student_lse, **kw)

    def backward(self, dout, stream=None, sink=None, dsink=None):
        """Gradients of the attention stage for upstream ``dout`` [T_cap, H, d],
        from the saved output and LSE of the last forward: ``dq`` (I/O dtype),
        float32 ``dkv_cmp`` / ``dkv_raw`` (dK + dV of the shared KV rows, or dK
        with ``dv_cmp`` / ``dv_raw`` for a separate V) and ``dsink`` when given."""
        wl, x = self.wl, self.x
        if getattr(self, "dq", None) is None:
            T, d = wl.T_cap, wl.d
            self.dq = torch.empty_like(self.out)
            self.dkv_raw = torch.empty(T, d, dtype=torch.float32, device=self.dev)
            self.dv_raw = torch.empty(T, d, dtype=torch.float32, device=self.dev) if wl.separate_v else None
            if wl.ratio > 0:
                n_cap = max(1, T // wl.ratio)
                self.dkv_cmp = torch.empty(n_cap, d, dtype=torch.float32, device=self.dev)
                self.dv_cmp = torch.empty(n_cap, d, dtype=torch.float32, device=self.dev) if wl.separate_v else None
            self.delta = torch.empty(T, wl.H, dtype=torch.float32, device=self.dev)
        v_raw = x.get("v") if wl.separate_v else None
        common = dict(v_raw=v_raw, dv_raw=self.dv_raw, sink=sink, dsink=dsink, stream=stream)
        if wl.ratio == 0:
            api.window_attn_bwd(self.h, x["q"], x["x_kv"], self.cu, self.max_seqlen, wl.window, self.scale,
                                self.out, self.lse, dout, self.dq, self.dkv_raw, self.delta, **common)
        elif wl.H_I > 0:
            api.csa_sparse_attn_bwd(self.h, x["q"], self.kv_cmp, x["x_kv"], self.idx, self.cu, self.cu_cmp,
                                    self.max_seqlen, wl.ratio, wl.window, self.scale, self.out, self.lse, dout,
                                    self.dq, self.dkv_cmp, self.dkv_raw, self.delta, v_cmp=self.v_cmp,
                                    dv_cmp=self.dv_cmp, **common)
        else:
            api.hca_attn_bwd(self.h, x["q"], self.kv_cmp, x["x_kv"], self.cu, self.cu_cmp, self.max_seqlen,
                             wl.ratio, wl.window, self.scale, self.out, self.lse, dout, self.dq, self.dkv_cmp,
                             self.dkv_raw, self.delta, v_cmp=self.v_cmp, dv_cmp=self.dv_cmp, **common)

    def indexer_backward(self, grad_scale: float = 1.0, stream=None):
        """Gradients of the indexer KL loss (teacher detached) with respect to
        qI, w (I/O dtype) and the compressed indexer keys (float32), for the
        upstream gradient ``grad_scale``: the step the page runs eagerly inside
        the forward (§8.2)."""
        wl, x = self.wl, self.x
        if getattr(self, "dqI", None) is None:
            self.dqI = torch.empty_like(x["qI"])
            self.dw = torch.empty_like(x["w"])
            self.dkI = torch.empty(max(1, wl.T_cap // wl.ratio), wl.d_I, dtype=torch.float32, device=self.dev)
        sparse = wl.kl_mode == "sparse"
        stats = getattr(self, "teacher_lse", None) is not None   # normalisers kept by kl(save_stats=True)
        api.csa_indexer_kl_bwd(self.h, x["q"], self.kv_cmp, x["qI"], x["w"], self.kI, self.cu, self.cu_cmp,
                               self.max_seqlen, wl.ratio, self.scale, self.dqI, self.dw, self.dkI,
                               idx=self.idx if sparse else None,
                               lse_cmp=self.teacher_lse if stats else None,
                               student_lse=self.student_lse if stats else None,
                               grad_scale=grad_scale, stream=stream)

    def run(self, stream=None, sink=None):
        """The whole hot path of one forward, enqueued on ``stream``."""
        if self.wl.ratio > 0:
            self.compress(stream)
            if self.wl.H_I > 0:
                self.topk(stream)
        self.attend(stream, sink=sink)
        if self.wl.kl_mode != "none":
            self.kl(stream)


    # inputs each stage needs first, in the order the stages run
    _STAGE_INPUTS = (("cu_seqlens", "x_kv", "z_kv", "P_kv", "x_I", "z_I", "P_I", "v", "x_kv_prev", "z_kv_prev",
                      "x_I_prev", "z_I_prev", "g_kv", "g_I"), ("qI", "w"), ("q",))

    attend_chunks = 4   # run_from_host: selected attention in up to this many row chunks

    def run_from_host(self, host: dict, stream=None, copy_stream=None):
        """The forward with its inputs still in (pinned) host memory.

        The inputs are copied into this object's device buffers on
        ``copy_stream`` in the order the stages need them, and each stage
        waits only for its own inputs: the compressor's and the indexer's
        inputs first, then the queries (537 MB at the 32K layer) in row
        chunks, last rows first.  The selected attention runs chunk by chunk
        as the queries arrive (``_attention_chunks``); the KL loss, which
        needs all of them, follows.  The previous forward on ``stream`` must
        be done with the buffers before they are overwritten: the copy stream
        waits for it first.  ``host`` holds this workload's inputs (the same
        packing as ``wl``; the chunks are planned from it).
        """
        main = stream if stream is not None else torch.cuda.current_stream()
        cs = copy_stream if copy_stream is not None else self._copy_stream()
        cs.wait_stream(main)
        chunks = self._attention_chunks()
        ready = []
        with torch.cuda.stream(cs):
            for si, names in enumerate(self._STAGE_INPUTS):
                if si == 2 and chunks:   # the queries, chunk by chunk (each row once)
                    for c in chunks:
                        self.x["q"][c["copy"][0]:c["copy"][1]].copy_(host["q"][c["copy"][0]:c["copy"][1]],
                                                                    non_blocking=True)
                        c["ready"].record(cs)
                for k in names:
                    if k in host and k in self.x and not (si == 2 and chunks):
                        self.x[k].copy_(host[k], non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(cs)
                ready.append(ev)
        with torch.cuda.stream(main):
            main.wait_event(ready[0])
            if self.wl.ratio > 0:
                self.compress(main)
                if self.wl.H_I > 0:
                    main.wait_event(ready[1])
                    self.topk(main)
            main.wait_event(ready[1])
            if chunks:
                for c in chunks:
                    main.wait_event(c["ready"])
                    self._attend_rows(c, main)
            else:
                main.wait_event(ready[2])
                self.attend(main)
            main.wait_event(ready[2])
            if self.wl.kl_mode != "none":
                self.kl(main)

    def _attention_chunks(self):
        """Row chunks of the selected attention for ``run_from_host``, last first.

        Chunk k owns the packed rows [a_k, a_{k+1}) (the last one up to T_cap,
        so it also writes the capacity rows).  Its call sees the rows
        [lo_k, a_{k+1}) with lo_k up to W rows earlier inside a_k's sequence:
        the raw rows of its first queries' windows.  That view is a packing of
        its own -- one segment per sequence, each with the position of its
        first row (csa_set_position_offsets), the global compressed offsets and
        the global top-k rows -- so its queries see exactly what they see in
        the whole call ("DeepSeek-V4 Attention Training Systems" §5: the
        contiguous context-parallel layout with a boundary of W raw rows).  The
        rows [lo_k, a_k) are computed again with a truncated window; the chunks
        run last to first, so their owner (the next chunk run) writes them
        after.  Queries are copied as [lo_k, lo_{k+1}): each row once, before
        the first chunk that reads it.  Empty when chunking does not apply."""
        wl = self.wl
        if getattr(self, "_chunks", None) is not None:
            return self._chunks
        self._chunks = []
        if wl.ratio <= 0 or wl.H_I <= 0 or wl.separate_v or wl.k_pad % 4 != 0:
            return self._chunks
        cu = [int(v) for v in wl.cu_seqlens]   # the workload's packing: no device read
        for c in attention_chunk_plan(cu, wl.T_cap, wl.window, int(self.attend_chunks)):
            self._chunks.append(dict(
                lo=c["lo"], hi=c["hi"], copy=c["copy"], max_len=c["max_len"],
                cu=torch.tensor(c["cu"], dtype=torch.int32, device=self.dev),
                pos0=torch.tensor(c["pos0"], dtype=torch.int32, device=self.dev),
                ready=torch.cuda.Event()))
        return self._chunks

    def _attend_rows(self, c, stream):
        """The selected attention of one chunk of ``_attention_chunks``."""
        wl, x = self.wl, self.x
        lo, hi = c["lo"], c["hi"]
        self.h.set_position_offsets(c["pos0"], self.kv_cmp.shape[0])
        try:
            api.csa_sparse_attn_fwd(self.h, x["q"][lo:hi], self.kv_cmp, x["x_kv"][lo:hi], self.idx[lo:hi], c["cu"],
                                    self.cu_cmp, c["max_len"], wl.ratio, wl.window, self.scale, self.out[lo:hi],
                                    self.lse[lo:hi], self.lse_cmp[lo:hi], stream=stream)
        finally:
            self.h.set_position_offsets(None)

    def copy_from_host(self, dst, src):
        """Queue a host-to-device copy on the copy stream, behind the inputs
        ``run_from_host`` queued there (so it overlaps the forward's compute),
        and return the event a consumer waits for.  An upstream gradient for
        ``backward`` is the use: the next ``run_from_host`` waits for the
        stream it was given before the copy stream rewrites anything."""
        cs = self._copy_stream()
        with torch.cuda.stream(cs):
            dst.copy_(src, non_blocking=True)
            ev = torch.cuda.Event()
            ev.record(cs)
        return ev

    def _copy_stream(self):
        if getattr(self, "_cs", None) is None:
            self._cs = torch.cuda.Stream(device=self.dev)
        return self._cs


def attention_chunk_plan(cu: list, T_cap: int, W: int, n: int) -> list:
    """Host plan of ``Forward._attention_chunks``, in the order the chunks run
    (last rows first).  ``cu``: the packing's offsets [B + 1].  Each chunk:
    ``lo``, ``hi`` (the rows its call sees), ``own`` (the rows whose outputs it
    leaves in place), ``copy`` (the query rows copied for
    it), ``cu`` (its own packing, one segment per sequence), ``pos0`` (each
    segment's first position in its sequence) and ``max_len`` (a bound on the
    positions in the view, the calls' max_seqlen).  Chunk starts
    are multiples of 16 rows; fewer than 8 W rows per chunk: no chunks."""
    T = cu[-1]
    B = len(cu) - 1
    if n < 2 or T < n * 8 * max(W, 16):
        return []
    a = [((T * k) // n) // 16 * 16 for k in range(n)] + [T_cap]
    los = [0]
    for k in range(1, n):
        b0 = max(b for b in range(B) if cu[b] <= a[k])   # the sequence holding row a_k
        los.append(max(cu[b0], a[k] - W))
    plan = []
    for k in reversed(range(n)):
        lo, hi = los[k], a[k + 1]
        seg = [max(0, min(hi, cu[b + 1]) - max(lo, cu[b])) for b in range(B)]
        cu_l = [0]
        for L in seg:
            cu_l.append(cu_l[-1] + L)
        pos0 = [max(lo, cu[b]) - cu[b] if seg[b] > 0 else 0 for b in range(B)]
        plan.append(dict(lo=lo, hi=hi, own=(a[k], hi), copy=(los[k], los[k + 1] if k + 1 < n else T_cap), cu=cu_l,
                         pos0=pos0, max_len=max([p + L for p, L in zip(pos0, seg)] + [1])))
    return plan


def to_device(arrs: dict, io_fp32: bool, device: int = 0) -> dict:
    """numpy float32 (bf16-valued) inputs -> device tensors in the I/O dtype."""
    dev = torch.device("cuda", device)
    out = {}
    for k, v in arrs.items():
        t = torch.from_numpy(v)
        if k == "cu_seqlens":
            out[k] = t.to(dev, torch.int32)
        elif k.startswith(("P_", "g_")):
            out[k] = t.to(dev, torch.float32)
        else:
            out[k] = t.to(dev, torch.float32 if io_fp32 else torch.bfloat16)
    return out
