"""Host logic of the chunked host-input forward (no GPU).

``attention_chunk_plan`` cuts the packed queries into row chunks for the
selected attention that runs while the queries are still being copied
("DeepSeek-V4 Attention Training Systems" §5: a contiguous range of each
sequence plus a boundary of W raw rows, with each segment's position).  The
checks: the owned ranges partition the rows, every owned query sees its whole
window inside its chunk's view, boundary rows are owned by a chunk that runs
later, every query row is copied once and before the first chunk that reads
it, and each chunk's packing and positions describe exactly its view.
"""
import numpy as np
import pytest

from compressed_sparse_attention_compress_gb300.forward import attention_chunk_plan


def _packings():
    rng = np.random.default_rng(17)
    out = [([8192], 8192), ([32768], 32768), ([3000, 1, 2500, 700, 1900], 8192), ([0, 5000, 0, 3100], 8200)]
    for _ in range(40):
        lengths = [int(v) for v in rng.integers(0, 3000, rng.integers(1, 9))]
        lengths[int(rng.integers(len(lengths)))] = int(rng.integers(0, 2))   # an empty or one-token sequence
        T = sum(lengths)
        out.append((lengths, T + int(rng.integers(0, 300))))
    return out


@pytest.mark.parametrize("n", [2, 3, 4, 6])
@pytest.mark.parametrize("W", [64, 128])
def test_plan_invariants(n, W):
    for lengths, T_cap in _packings():
        cu = [0] + list(np.cumsum(lengths).astype(int))
        T = cu[-1]
        plan = attention_chunk_plan(cu, T_cap, W, n)
        if T < n * 8 * W:
            assert plan == []
            continue
        assert len(plan) == n
        seq_of = np.searchsorted(np.asarray(cu), np.arange(T_cap), side="right") - 1
        owner = np.full(T_cap, -1)
        copied = np.zeros(T_cap, np.int64)
        for order, c in enumerate(plan):
            lo, hi, (a, b) = c["lo"], c["hi"], c["own"]
            assert lo <= a < b == hi and a % 16 == 0
            assert (owner[a:b] == -1).all()
            owner[a:b] = order
            copied[c["copy"][0]:c["copy"][1]] += 1
            assert copied[lo:hi].all()                      # copied by now
            # its packing: one segment per sequence, the intersection with [lo, min(hi, T))
            B = len(cu) - 1
            assert len(c["cu"]) == B + 1 and len(c["pos0"]) == B
            for s in range(B):
                s0, s1 = max(lo, cu[s]), min(hi, cu[s + 1])
                L = max(0, s1 - s0)
                assert c["cu"][s + 1] - c["cu"][s] == L
                if L:
                    assert c["cu"][s] == s0 - lo and c["pos0"][s] == s0 - cu[s]
            assert c["cu"][-1] == min(hi, T) - lo
            # max_seqlen bounds every position the view holds, and no more than the longest sequence
            assert all(p + (c["cu"][s + 1] - c["cu"][s]) <= c["max_len"] for s, p in enumerate(c["pos0"]))
            assert c["max_len"] <= max(lengths + [1])
            # owned queries see their whole window inside the view
            for t in range(a, min(b, T)):
                s = seq_of[t]
                assert max(cu[s], t - W + 1) >= lo
        assert (owner >= 0).all() and (copied == 1).all()
        # rows a chunk computes but does not own are owned by a chunk that runs after it
        for order, c in enumerate(plan):
            assert (owner[c["lo"]:c["own"][0]] > order).all()
