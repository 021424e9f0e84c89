"""Pins for the oracle's indexer KL loss (CPU only).

L_I = sum_t KL(Softmax(a_{t,C_t}) || Softmax(i_{t,C_t})) with C_t the selected
set (sparse mode) or every visible entry (dense-loss warm-up)
("DeepSeek-V4 Attention Training Systems", §2 phase table, §3 equation, §9).
Teacher reading: a_{t,j} = log of the head average of per-head softmaxes over
C_t.  Pins: scipy softmax + rel_entr brute force, the two-entry closed form,
KL >= 0, KL = 0 when the indexer reproduces the teacher, dense == sparse when
k covers the visible set.
"""
import numpy as np
import pytest
from scipy.special import rel_entr, softmax

import oracle
from compressed_sparse_attention_compress_gb300.inputs import bf16_round

rng = np.random.default_rng(2024)


def _rand(*shape, positive=False):
    a = rng.standard_normal(shape).astype(np.float32)
    return bf16_round(np.abs(a) if positive else a)


def _case(L=48, r=4, H=3, d=16, H_I=2, dI=8):
    n_c = L // r
    return _rand(L, H, d), _rand(n_c, d), _rand(L, H_I, dI), _rand(L, H_I), _rand(n_c, dI)


def _random_idx(L, r, k, k_pad):
    idx = np.full((L, k_pad), -1, np.int32)
    for t in range(L):
        n = (t + 1) // r
        m = min(k, n)
        if m:
            idx[t, :m] = np.sort(rng.choice(n, m, replace=False))
    return idx


@pytest.mark.parametrize("dense", [False, True])
def test_matches_scipy_brute_force(dense):
    L, r, H = 48, 4, 3
    q, kc, qI, w, kI = _case(L, r, H)
    scale = 0.25
    idx = None if dense else _random_idx(L, r, 4, 6)
    kl, csize, err = oracle.indexer_kl(q, kc, qI, w, kI, [0, L], r, scale, idx=idx)
    logits, nvis = oracle.indexer_logits(qI, w, kI, [0, L], r, None, L // r)
    assert not err.any()
    for t in range(L):
        C = np.arange(nvis[t]) if dense else idx[t][idx[t] >= 0]
        assert csize[t] == len(C)
        if len(C) == 0:
            assert kl[t] == 0
            continue
        s = scale * (q[t].astype(np.float64) @ kc[C].astype(np.float64).T)     # [H, |C|]
        p = softmax(s, axis=1).mean(0)
        qq = softmax(logits[t, C])
        np.testing.assert_allclose(kl[t], rel_entr(p, qq).sum(), rtol=1e-11, atol=1e-14)
        assert kl[t] >= -1e-15


def test_two_entry_closed_form():
    # |C_t| = 2, one head: teacher and student are Bernoulli distributions.
    L, r = 12, 4
    q, kc, qI, w, kI = _case(L, r, H=1)
    idx = np.full((L, 2), -1, np.int32)
    idx[11] = [0, 2]
    kl, _, _ = oracle.indexer_kl(q, kc, qI, w, kI, [0, L], r, 0.5, idx=idx, rows=[11])
    logits, _ = oracle.indexer_logits(qI, w, kI, [0, L], r, [11], 3)
    s = 0.5 * (q[11, 0].astype(np.float64) @ kc[[0, 2]].astype(np.float64).T)
    p = 1 / (1 + np.exp(s[1] - s[0]))
    qq = 1 / (1 + np.exp(logits[0, 2] - logits[0, 0]))
    want = p * np.log(p / qq) + (1 - p) * np.log((1 - p) / (1 - qq))
    np.testing.assert_allclose(kl[0], want, rtol=1e-12)


@pytest.mark.parametrize("H", [1, 4])
def test_zero_when_indexer_reproduces_teacher(H):
    # H_I = 1, w = 1, qI = scale * q, kI = K with nonnegative operands (ReLU is
    # the identity) and identical heads: i_{t,j} = a_{t,j} up to a constant.
    L, r, d = 40, 4, 64
    scale = 1 / 8                              # exact in bf16
    q1 = _rand(L, 1, d, positive=True)
    q = np.repeat(q1, H, axis=1)
    kc = _rand(L // r, d, positive=True)
    qI = q1 * np.float32(scale)
    w = np.ones((L, 1), np.float32)
    for dense in (True, False):
        idx = None if dense else _random_idx(L, r, 3, 3)
        kl, csize, _ = oracle.indexer_kl(q, kc, qI, w, kc, [0, L], r, scale, idx=idx)
        assert np.all(np.abs(kl) < 1e-12)
        assert csize.sum() > 0


def test_dense_equals_sparse_when_k_covers_visible():
    L, r = 44, 4
    q, kc, qI, w, kI = _case(L, r)
    full = _random_idx(L, r, L, L // r)
    a, ca, _ = oracle.indexer_kl(q, kc, qI, w, kI, [0, L], r, 0.3, idx=full)
    b, cb, _ = oracle.indexer_kl(q, kc, qI, w, kI, [0, L], r, 0.3, idx=None)
    np.testing.assert_allclose(a, b, rtol=1e-13, atol=1e-15)
    np.testing.assert_array_equal(ca, cb)


def test_nonnegative_and_capacity_rows():
    lengths, r = [30, 19], 4
    cu = np.array([0, 30, 49], np.int32)
    T = 52
    q, qI, w = _rand(T, 2, 8), _rand(T, 2, 8), _rand(T, 2)
    n_c = int(oracle.compressed_offsets(cu, r)[-1])
    kc, kI = _rand(n_c, 8), _rand(n_c, 8)
    kl, csize, err = oracle.indexer_kl(q, kc, qI, w, kI, cu, r, 0.3)
    assert np.all(kl >= -1e-15) and np.all(kl[49:] == 0) and np.all(csize[49:] == 0)
    assert csize[0] == 0 and csize[3] == 1          # query t=3 sees entry 0 only
    assert abs(kl[3]) < 1e-15                        # one entry: both distributions are 1
