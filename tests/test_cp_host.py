"""Host logic of contiguous context parallelism on CPU (no GPU).

"DeepSeek-V4 Attention Training Systems" §5: a rank holds a contiguous query
range of every sequence, receives max(W, S) boundary rows from its left
neighbour, compresses the complete blocks ending in its range, and the
compressed rows are all-gathered.  Here the partition, the local layouts, the
ownership and the all-gather (two gloo ranks on 127.0.0.1) run with the CPU
oracle as the compressor; the gathered rows must equal the oracle's
compression of the whole packed batch, and every entry must have exactly one
owner.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
from compressed_sparse_attention_compress_gb300 import cp
from compressed_sparse_attention_compress_gb300.inputs import bf16_round

LENGTHS = [1000, 0, 37, 2050, 300]
R, W = 4, 128
S = 2 * R


def _data(seed=0):
    rng = np.random.default_rng(seed)
    T = sum(LENGTHS)
    x = bf16_round(rng.standard_normal((T, 16)).astype(np.float32))
    z = bf16_round(rng.standard_normal((T, 16)).astype(np.float32))
    P = rng.standard_normal((S, 16)).astype(np.float32)
    return x, z, P


def _local_compress(lay, x, z, P, cu):
    rows = np.concatenate([np.arange(cu[b] + lo, cu[b] + e) for b, (lo, e) in enumerate(zip(lay.lo, lay.end))])
    out = oracle.compress(x[rows], z[rows], P, lay.cu_local, R, True)
    cmp = oracle.compressed_offsets(lay.cu_local, R)
    own = cp.owned_entries(lay, R)
    return [torch.from_numpy(out[cmp[b] + j0:cmp[b] + j0 + n]) for b, (j0, n) in enumerate(own)]


@pytest.mark.parametrize("P", [1, 2, 3, 5])
def test_every_entry_has_one_owner_and_local_copies_reassemble(P):
    x, z, Pb = _data()
    cu = np.concatenate([[0], np.cumsum(LENGTHS)]).astype(np.int32)
    parts = cp.partition(LENGTHS, P, R)
    for b, L in enumerate(LENGTHS):       # ranges tile [0, L), cut points on block boundaries
        ends = [e for _, e in parts[b]]
        assert parts[b][0][0] == 0 and ends[-1] == L
        assert all(parts[b][p][1] == parts[b][p + 1][0] for p in range(P - 1))
        assert all(s % R == 0 for s, _ in parts[b])
    lays = [cp.rank_layout(LENGTHS, parts, p, max(W, S)) for p in range(P)]
    counts = np.zeros(len(LENGTHS), np.int64)
    for lay in lays:
        for b, (_, n) in enumerate(cp.owned_entries(lay, R)):
            counts[b] += n
    assert list(counts) == [L // R for L in LENGTHS]
    got = cp.gather_compressed([_local_compress(lay, x, z, Pb, cu) for lay in lays], len(LENGTHS))
    np.testing.assert_array_equal(got.numpy(), oracle.compress(x, z, Pb, cu, R, True))


def _worker(rank, world, port, result_path):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        x, z, Pb = _data()
        cu = np.concatenate([[0], np.cumsum(LENGTHS)]).astype(np.int32)
        parts = cp.partition(LENGTHS, world, R)
        lay = cp.rank_layout(LENGTHS, parts, rank, max(W, S))
        mine = _local_compress(lay, x, z, Pb, cu)
        got = cp.gather_compressed(mine, len(LENGTHS), group=dist.group.WORLD)
        if rank == 0:
            np.save(result_path, got.numpy())
    finally:
        dist.destroy_process_group()


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_all_gather_on_two_gloo_ranks(tmp_path):
    path = str(tmp_path / "gathered.npy")
    mp.spawn(_worker, args=(2, _free_port(), path), nprocs=2, join=True)
    x, z, Pb = _data()
    cu = np.concatenate([[0], np.cumsum(LENGTHS)]).astype(np.int32)
    np.testing.assert_array_equal(np.load(path), oracle.compress(x, z, Pb, cu, R, True))
