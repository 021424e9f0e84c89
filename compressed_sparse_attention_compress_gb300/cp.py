"""Contiguous context parallelism for the CSA forward, and its single-process emulation.

"DeepSeek-V4 Attention Training Systems" §5 (contiguous CP: each rank holds a
contiguous range of every sequence's queries; it receives max(W, S) raw rows
from its left neighbour -- the boundary -- compresses the complete blocks that
end in its own range, and the compressed main KV and indexer K are
all-gathered), §5.1 (S = 8 for the overlapping ratio-4 span, W = 128), §12
invariant 4 (selected ids must map to the right physical rows).

The host logic here is independent of where the ranks run:
``partition`` cuts every sequence into rank ranges (multiples of ``align``),
``rank_layout`` builds a rank's local packing (boundary + own rows, with the
position of each segment's first row), ``owned_entries`` picks the compressed
rows a rank owns, and ``gather_compressed`` puts every rank's owned rows back
into the global packed order -- by local copies in one process, or by an
all-gather on a process group.  With the gathered rows in global order a
selected id is the physical row itself (the lowering is the identity).
``emulate`` runs the ranks one after another on one GPU through the C ABI:
the compressor on each rank's local rows, then top-k, attention and the KL
loss with the handle's position offsets (csa_set_position_offsets), and
returns each rank's own rows.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

from . import api


@dataclass
class RankLayout:
    """One rank's local packing: per sequence the rows [lo, end) of the sequence."""
    lo: list            # first local row of each sequence segment (its position in the sequence)
    start: list         # first owned query position
    end: list           # one past the last owned position
    cu_local: np.ndarray  # int32 [B + 1] offsets of the segments in the local buffer

    def own_local_rows(self) -> np.ndarray:
        """Local row numbers of the owned queries, in sequence order."""
        rows = [np.arange(self.cu_local[b] + (s - lo), self.cu_local[b] + (e - lo))
                for b, (lo, s, e) in enumerate(zip(self.lo, self.start, self.end))]
        return np.concatenate(rows) if rows else np.zeros(0, np.int64)


def partition(lengths, P: int, align: int):
    """[(start, end)] per rank per sequence: contiguous ranges whose cut points
    are multiples of ``align`` (so every compressed block has one owner)."""
    out = []
    for L in lengths:
        chunk = -(-L // (P * align)) * align if L > 0 else align
        out.append([(min(p * chunk, L), min((p + 1) * chunk, L)) for p in range(P)])
    return out


def rank_layout(lengths, parts, p: int, boundary: int) -> RankLayout:
    lo, st, en, segs = [], [], [], []
    for b, L in enumerate(lengths):
        s, e = parts[b][p]
        low = max(0, s - boundary) if e > s else s
        lo.append(low)
        st.append(s)
        en.append(e)
        segs.append(e - low)
    cu = np.concatenate([[0], np.cumsum(segs)]).astype(np.int32)
    return RankLayout(lo, st, en, cu)


def owned_entries(lay: RankLayout, ratio: int):
    """Per sequence: (local first entry, count) of the compressed rows this rank
    owns -- the complete blocks ending in its range [start, end)."""
    out = []
    for lo, s, e in zip(lay.lo, lay.start, lay.end):
        g0, g1 = -(-s // ratio), e // ratio   # blocks whose last token lies in [s, e)
        g0 = s // ratio if s % ratio == 0 else g0
        out.append((g0 - lo // ratio, max(0, g1 - g0)))
    return out


def gather_compressed(owned_rows, n_seq: int, group=None):
    """Global packed order from each rank's owned rows.

    ``owned_rows``: in one process, the list over ranks of lists over sequences
    of [n, D] tensors; with a process group, this rank's list over sequences
    (the other ranks' are all-gathered)."""
    if group is not None:
        import torch.distributed as dist
        world = dist.get_world_size(group)
        mine = owned_rows
        counts = torch.tensor([t.shape[0] for t in mine], dtype=torch.int64)
        all_counts = [torch.zeros_like(counts) for _ in range(world)]
        dist.all_gather(all_counts, counts, group=group)
        D = mine[0].shape[1] if mine else 0
        flat = torch.cat(mine) if mine else torch.zeros(0, D)
        width = int(max(int(c.sum()) for c in all_counts))
        pad = torch.zeros(width, D, dtype=flat.dtype)
        pad[:flat.shape[0]] = flat
        bufs = [torch.zeros_like(pad) for _ in range(world)]
        dist.all_gather(bufs, pad, group=group)
        owned_rows = []
        for r in range(world):
            offs = np.concatenate([[0], np.cumsum(all_counts[r].numpy())])
            owned_rows.append([bufs[r][offs[b]:offs[b + 1]] for b in range(n_seq)])
    return torch.cat([owned_rows[r][b] for b in range(n_seq) for r in range(len(owned_rows))])


def emulate(wl, dev: dict, P: int, boundary: int | None = None):
    """Run the CSA forward of ``wl`` as P contiguous-CP ranks on one GPU.

    ``dev``: the workload's inputs on the device (as for Forward).  Returns a dict
    with, per output, the rank-local values of the owned queries concatenated in
    global row order: ``idx``, ``out``, ``lse``, ``lse_cmp`` and (with a KL mode)
    ``kl_rows``; plus the gathered ``kv_cmp`` and ``kI``."""
    assert wl.ratio > 0 and wl.H_I > 0 and not wl.separate_v
    r, S, W = wl.ratio, wl.span, wl.window
    boundary = boundary if boundary is not None else max(W, S)
    align = int(np.lcm(r, 4))
    assert boundary % r == 0
    lengths = list(wl.lengths)
    parts = partition(lengths, P, align)
    cu_g = wl.cu_seqlens
    dvc = dev["x_kv"].device
    h = api.Handle(dvc.index or 0)
    ranks = [rank_layout(lengths, parts, p, boundary) for p in range(P)]

    def local(name, lay, width):
        rows = [dev[name][cu_g[b] + lo:cu_g[b] + e] for b, (lo, e) in enumerate(zip(lay.lo, lay.end))]
        t = torch.cat(rows) if rows else dev[name][:0]
        return t.reshape(-1, *width).contiguous() if width else t.contiguous()

    # ---- each rank compresses its local rows (boundary included) and keeps what it owns ----
    owned_kv, owned_I = [], []
    for lay in ranks:
        T_l = int(lay.cu_local[-1])
        cu_l = torch.from_numpy(lay.cu_local).to(dvc)
        cmp_l = torch.zeros(len(lengths) + 1, dtype=torch.int32, device=dvc)
        api.csa_compressed_offsets(h, cu_l, r, cmp_l)
        kv_l = torch.zeros(max(1, T_l // r), wl.d, dtype=dev["x_kv"].dtype, device=dvc)
        kI_l = torch.zeros(max(1, T_l // r), wl.d_I, dtype=dev["x_I"].dtype, device=dvc)
        ms = max([e - lo for lo, e in zip(lay.lo, lay.end)] + [1])
        api.csa_compress(h, local("x_kv", lay, None), local("z_kv", lay, None), dev["P_kv"], cu_l, cmp_l, ms, r,
                         wl.overlap, kv_l)
        api.csa_compress(h, local("x_I", lay, None), local("z_I", lay, None), dev["P_I"], cu_l, cmp_l, ms, r,
                         wl.overlap, kI_l)
        cmp_np = cmp_l.cpu().numpy()
        own = owned_entries(lay, r)
        owned_kv.append([kv_l[cmp_np[b] + j0:cmp_np[b] + j0 + n] for b, (j0, n) in enumerate(own)])
        owned_I.append([kI_l[cmp_np[b] + j0:cmp_np[b] + j0 + n] for b, (j0, n) in enumerate(own)])
    # ---- all-gather (local copies): the compressed rows in global packed order ----
    kv_g = gather_compressed(owned_kv, len(lengths))
    kI_g = gather_compressed(owned_I, len(lengths))
    n_c = kv_g.shape[0]
    # capacity buffers: the tensor-core kernels read whole tiles of up to
    # max(n_c, T_local / r) rows, so the gathered rows sit in zero-padded buffers
    cap = max(1, n_c, max(int(lay.cu_local[-1]) // r for lay in ranks))
    kv_cmp = torch.zeros(cap, wl.d, dtype=kv_g.dtype, device=dvc)
    kI = torch.zeros(cap, wl.d_I, dtype=kI_g.dtype, device=dvc)
    kv_cmp[:n_c] = kv_g
    kI[:n_c] = kI_g
    cu_cmp = torch.from_numpy(np.concatenate([[0], np.cumsum([L // r for L in lengths])]).astype(np.int32)).to(dvc)
    # ---- each rank's queries at their true positions ----
    res = {k: [] for k in ("rows", "idx", "out", "lse", "lse_cmp", "kl_rows")}
    max_pos = max(lengths + [1])
    for lay in ranks:
        T_l = int(lay.cu_local[-1])
        if T_l == 0:
            continue
        cu_l = torch.from_numpy(lay.cu_local).to(dvc)
        pos0 = torch.tensor(lay.lo, dtype=torch.int32, device=dvc)
        h.set_position_offsets(pos0, cap)
        q = local("q", lay, (wl.H, wl.d))
        qI = local("qI", lay, (wl.H_I, wl.d_I))
        w = local("w", lay, (wl.H_I,))
        kv_raw = local("x_kv", lay, None)
        idx = torch.empty(T_l, wl.k_pad, dtype=torch.int32, device=dvc)
        api.csa_indexer_topk(h, qI, w, kI, cu_l, cu_cmp, max_pos, r, wl.topk, idx)
        out = torch.empty_like(q)
        lse = torch.empty(T_l, wl.H, dtype=torch.float32, device=dvc)
        lse_c = torch.empty_like(lse)
        scale = 1.0 / float(np.sqrt(wl.d))
        api.csa_sparse_attn_fwd(h, q, kv_cmp, kv_raw, idx, cu_l, cu_cmp, max_pos, r, W, scale, out, lse, lse_c)
        if wl.kl_mode != "none":
            sparse = wl.kl_mode == "sparse"
            kl_sum = torch.zeros(1, device=dvc)
            kl_rows = torch.zeros(T_l, device=dvc)
            ws = torch.empty(api.csa_indexer_kl_workspace(T_l), dtype=torch.uint8, device=dvc)
            api.csa_indexer_kl(h, q, kv_cmp, qI, w, kI, cu_l, cu_cmp, max_pos, r, scale, kl_sum, ws,
                               idx=idx if sparse else None, lse_cmp=lse_c if sparse else None, kl_per_query=kl_rows)
            res["kl_rows"].append(kl_rows)
        own = torch.from_numpy(lay.own_local_rows()).to(dvc)
        grow = np.concatenate([np.arange(cu_g[b] + s, cu_g[b] + e) for b, (s, e) in enumerate(zip(lay.start, lay.end))])
        res["rows"].append(grow)
        res["idx"].append(idx[own])
        res["out"].append(out[own])
        res["lse"].append(lse[own])
        res["lse_cmp"].append(lse_c[own])
        if res["kl_rows"]:
            res["kl_rows"][-1] = res["kl_rows"][-1][own]
        h.set_position_offsets(None)
    torch.cuda.synchronize()
    status = h.device_status()
    rows = np.concatenate(res.pop("rows"))
    order = torch.from_numpy(np.argsort(rows, kind="stable")).to(dvc)
    merged = {k: torch.cat(v)[order] for k, v in res.items() if v}
    merged.update(rows=np.sort(rows), kv_cmp=kv_cmp[:n_c], kI=kI[:n_c], status=status)
    return merged
