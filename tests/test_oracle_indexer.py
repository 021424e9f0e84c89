"""Pins for the oracle's lightning-indexer logits and per-query top-k (CPU only).

Logit form sum_h w[t,h] * ReLU(qI[t,h,:] . kI[j,:]) over the causally visible
compressed entries; top-k with ties to the smaller index, emitted ascending as
global compressed rows and padded with -1 ("DeepSeek-V4 Attention Training
Systems", §3, §4, §8.1, §8.2).  Pins: numpy matmul special cases, linearity in
w, ReLU behaviour, a numpy lexsort brute force, and visibility invariants.
"""
import numpy as np
import pytest

import oracle
from compressed_sparse_attention_compress_gb300.inputs import bf16_round

rng = np.random.default_rng(99)


def _rand(*shape, positive=False):
    a = rng.standard_normal(shape).astype(np.float32)
    return bf16_round(np.abs(a) if positive else a)


def _setup(lengths, r, H_I, dI):
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    T = int(cu[-1])
    n_c = int(oracle.compressed_offsets(cu, r)[-1])
    return cu, T, _rand(T, H_I, dI), _rand(T, H_I), _rand(max(n_c, 1), dI)


def test_single_head_nonnegative_is_matmul():
    # H_I = 1, w = 1, nonnegative operands: ReLU is the identity and the
    # logits are the plain product qI kI^T restricted to visible entries.
    L, r, dI = 64, 4, 16
    qI = _rand(L, 1, dI, positive=True)
    kI = _rand(L // r, dI, positive=True)
    w = np.ones((L, 1), np.float32)
    logits, nvis = oracle.indexer_logits(qI, w, kI, [0, L], r, None, L // r)
    ref = qI[:, 0, :].astype(np.float64) @ kI.astype(np.float64).T
    for t in range(L):
        assert nvis[t] == (t + 1) // r
        np.testing.assert_allclose(logits[t, :nvis[t]], ref[t, :nvis[t]], rtol=1e-13)


def test_head_weight_linearity_and_relu():
    # One-hot w picks one head: logits = ReLU(qI_h kI^T) (numpy matmul +
    # maximum); logits are linear in w.
    L, r, H_I, dI = 48, 4, 3, 8
    cu, T, qI, w, kI = _setup([L], r, H_I, dI)
    rows = np.arange(L)
    per_head = []
    for h in range(H_I):
        wh = np.zeros((L, H_I), np.float32)
        wh[:, h] = 1.0
        lg, nvis = oracle.indexer_logits(qI, wh, kI, cu, r, rows, L // r)
        ref = np.maximum(qI[:, h, :].astype(np.float64) @ kI.astype(np.float64).T, 0.0)
        for t in range(L):
            np.testing.assert_allclose(lg[t, :nvis[t]], ref[t, :nvis[t]], rtol=1e-13, atol=1e-14)
        per_head.append(np.nan_to_num(lg))
    full, nvis = oracle.indexer_logits(qI, w, kI, cu, r, rows, L // r)
    combo = sum(w[:, h:h + 1].astype(np.float64) * per_head[h] for h in range(H_I))
    for t in range(L):
        np.testing.assert_allclose(full[t, :nvis[t]], combo[t, :nvis[t]], rtol=1e-12, atol=1e-13)


def test_negative_head_contributes_nothing():
    L, r, H_I, dI = 40, 4, 2, 8
    cu, T, qI, w, kI = _setup([L], r, H_I, dI)
    kI = np.abs(kI)
    qI[:, 1, :] = -np.abs(qI[:, 1, :])        # head 1: every dot product <= 0
    w2 = w.copy()
    w2[:, 1] = 0.0
    a, _ = oracle.indexer_logits(qI, w, kI, cu, r, None, L // r)
    b, _ = oracle.indexer_logits(qI, w2, kI, cu, r, None, L // r)
    np.testing.assert_array_equal(np.nan_to_num(a), np.nan_to_num(b))


@pytest.mark.parametrize("lengths,r,topk,k_pad", [([70], 4, 5, 8), ([33, 0, 51, 9], 4, 3, 4),
                                                  ([300], 128, 1, 2), ([90], 2, 64, 64)])
def test_topk_matches_lexsort_brute_force(lengths, r, topk, k_pad):
    H_I, dI = 2, 8
    cu, T, qI, w, kI = _setup(lengths, r, H_I, dI)
    cu_cmp = oracle.compressed_offsets(cu, r)
    idx = oracle.indexer_topk(qI, w, kI, cu, r, topk, k_pad)
    maxvis = max(1, max(L // r for L in lengths))
    logits, nvis = oracle.indexer_logits(qI, w, kI, cu, r, None, maxvis)
    for t in range(T):
        b = int(np.searchsorted(cu, t, side="right") - 1)
        n = int(nvis[t])
        m = min(topk, n)
        s = logits[t, :n]
        order = np.lexsort((np.arange(n), -s))            # score desc, index asc
        want = np.sort(order[:m]) + cu_cmp[b]
        got = idx[t]
        np.testing.assert_array_equal(got[:m], want)
        assert np.all(got[m:] == -1)
        # characterisation: every chosen score >= every unchosen score
        if 0 < m < n:
            chosen = np.zeros(n, bool)
            chosen[got[:m] - cu_cmp[b]] = True
            assert s[chosen].min() >= s[~chosen].max()


def test_ties_go_to_smaller_index_and_k_covers_visible():
    L, r, dI = 64, 4, 8
    qI = _rand(L, 1, dI)
    w = np.ones((L, 1), np.float32)
    kI = np.repeat(_rand(1, dI), L // r, axis=0)        # every entry ties
    idx = oracle.indexer_topk(qI, w, kI, [0, L], r, 3, 4)
    for t in range(L):
        n = (t + 1) // r
        m = min(3, n)
        assert list(idx[t, :m]) == list(range(m))
        assert np.all(idx[t, m:] == -1)
    # k >= |V_t| returns exactly the visible set (dense mode)
    cu, T, qI, w, kI = _setup([L], r, 2, dI)
    idx = oracle.indexer_topk(qI, w, kI, cu, r, L, L)
    for t in range(L):
        n = (t + 1) // r
        assert list(idx[t, :n]) == list(range(n)) and np.all(idx[t, n:] == -1)


def test_no_entry_visible_before_its_block_completes_and_capacity_rows():
    lengths, r = [37, 50], 4
    cu, T, qI, w, kI = _setup(lengths, r, 2, 8)
    cu_cmp = oracle.compressed_offsets(cu, r)
    rows = np.arange(T + 5)          # 5 capacity rows past the last sequence
    qI = np.concatenate([qI, _rand(5, 2, 8)])
    w = np.concatenate([w, _rand(5, 2)])
    idx = oracle.indexer_topk(qI, w, kI, cu, r, 6, 8, rows)
    for row in range(T):
        b = int(np.searchsorted(cu, row, side="right") - 1)
        t = row - cu[b]
        valid = idx[row][idx[row] >= 0]
        assert np.all(valid >= cu_cmp[b]) and np.all(valid < cu_cmp[b] + (t + 1) // r)
        assert np.all(np.diff(valid) > 0)
    assert np.all(idx[T:] == -1)


def test_packed_equals_separate():
    lengths, r = [29, 44, 16], 4
    cu, T, qI, w, kI = _setup(lengths, r, 2, 8)
    cu_cmp = oracle.compressed_offsets(cu, r)
    packed = oracle.indexer_topk(qI, w, kI, cu, r, 4, 4)
    for b, L in enumerate(lengths):
        s = slice(cu[b], cu[b + 1])
        alone = oracle.indexer_topk(qI[s], w[s], kI[cu_cmp[b]:cu_cmp[b + 1]], [0, L], r, 4, 4)
        alone = np.where(alone >= 0, alone + cu_cmp[b], -1)
        np.testing.assert_array_equal(packed[s], alone)
