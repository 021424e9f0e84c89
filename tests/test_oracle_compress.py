"""Pins for the oracle's block compressor (CPU only).

The compressor is a softmax-gated weighted sum over a span of tokens
("DeepSeek-V4 Attention Training Systems", §4, §5.1, §8.2).  These tests pin
the oracle to closed forms, to the span widths the page states, and to the
packing/causality invariants -- never to a retyped copy of its own formula.
"""
import json
import os

import numpy as np
import pytest
from scipy.special import softmax

import oracle
from compressed_sparse_attention_compress_gb300.inputs import bf16_round

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "paper_facts.json")))
rng = np.random.default_rng(1234)


def _rand(*shape):
    return bf16_round(rng.standard_normal(shape).astype(np.float32))


def _span_rows(j, r, overlap, L):
    S = 2 * r if overlap else r
    first = r * j + r - S
    return [t for t in range(first, first + S) if 0 <= t < L]


@pytest.mark.parametrize("lengths,r", [([0, 1, 3, 4, 5, 8, 127, 128, 129, 257], 4),
                                       ([0, 127, 128, 129, 300, 1000], 128),
                                       ([7, 9], 1)])
def test_complete_groups_only(lengths, r):
    # §4: n_b = floor(L_b / r); the tail creates no entry.
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    cu_cmp = oracle.compressed_offsets(cu, r)
    assert cu_cmp[0] == 0
    assert list(np.diff(cu_cmp)) == [L // r for L in lengths]


@pytest.mark.parametrize("r,overlap", [(4, True), (4, False), (128, False), (2, True)])
def test_constant_gate_is_mean_of_available_rows(r, overlap):
    L, D = 9 * r + 3, 16
    x = _rand(L, D)
    z = np.full((L, D), 0.375, np.float32)
    S = 2 * r if overlap else r
    P = np.zeros((S, D), np.float32)
    out = oracle.compress(x, z, P, [0, L], r, overlap)
    assert out.shape == (L // r, D)
    for j in range(L // r):
        rows = _span_rows(j, r, overlap, L)
        np.testing.assert_allclose(out[j], x[rows].astype(np.float64).mean(0), rtol=0, atol=1e-12)


@pytest.mark.parametrize("via", ["z", "P"])
@pytest.mark.parametrize("r,overlap", [(4, True), (128, False)])
def test_one_hot_logit_copies_that_row(via, r, overlap):
    # A logit 80 above the others makes the gate one-hot (e^-80 ~ 1e-35):
    # the entry equals that token's row.  Via P this pins the position index u.
    L, D = 6 * r, 8
    S = 2 * r if overlap else r
    x = _rand(L, D)
    z = np.zeros((L, D), np.float32)
    P = np.zeros((S, D), np.float32)
    u_star = S - 3
    if via == "P":
        P[u_star] = 80.0
    out = oracle.compress(x, z if via == "P" else z, P, [0, L], r, overlap)
    for j in range(L // r):
        first = r * j + r - S
        t_star = first + u_star
        if via == "z":
            zz = np.zeros((L, D), np.float32)
            zz[t_star] = 80.0
            out_j = oracle.compress(x, zz, P, [0, L], r, overlap)[j]
        else:
            out_j = out[j]
        if t_star < 0:
            continue
        np.testing.assert_allclose(out_j, x[t_star], rtol=0, atol=1e-20)


def test_per_token_gate_matches_library_softmax():
    # A gate that is the same for every channel gives one weight per token:
    # out[j] = softmax(g over the span) @ x[span] (scipy softmax, numpy matmul).
    r, L, D = 4, 41, 12
    x = _rand(L, D)
    g = _rand(L)
    z = np.repeat(g[:, None], D, axis=1)
    P = np.zeros((2 * r, D), np.float32)
    out = oracle.compress(x, z, P, [0, L], r, True)
    for j in range(L // r):
        rows = _span_rows(j, r, True, L)
        wts = softmax(g[rows].astype(np.float64))
        np.testing.assert_allclose(out[j], wts @ x[rows].astype(np.float64), rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("key", ["D_compress_overlapping_ratio4", "D_compress_hca_ratio128"])
def test_span_width_matches_page(key):
    # Perturb one token at a time and record which entries move: every entry
    # away from the sequence start depends on exactly D_compress tokens, the
    # last of which is its own final token r(j+1)-1 (no future token).
    fact = GOLD[key]
    r, overlap, Dc = fact["ratio"], fact["overlap"], fact["value"]
    L, D = 5 * r + 2, 4
    x, z = _rand(L, D), _rand(L, D)
    P = _rand(2 * r if overlap else r, D)
    base = oracle.compress(x, z, P, [0, L], r, overlap)
    deps = [set() for _ in range(L // r)]
    for t in range(L):
        x2 = x.copy()
        x2[t] += 1.0
        moved = np.abs(oracle.compress(x2, z, P, [0, L], r, overlap) - base).max(1) > 0
        for j in np.nonzero(moved)[0]:
            deps[j].add(t)
    for j, dset in enumerate(deps):
        assert max(dset) == r * (j + 1) - 1
        if r * (j + 1) - Dc >= 0:
            assert len(dset) == Dc, (j, sorted(dset))
            assert min(dset) == r * (j + 1) - Dc
        else:
            assert min(dset) == 0 and len(dset) == r * (j + 1)


def test_first_overlapping_entry_drops_missing_left_half():
    # Entry 0 of an overlapping span has no previous block; it must equal the
    # non-overlapping entry 0 computed with the current-block half of P.
    r, L, D = 4, 23, 10
    x, z = _rand(L, D), _rand(L, D)
    P = _rand(2 * r, D)
    a = oracle.compress(x, z, P, [0, L], r, True)[0]
    b = oracle.compress(x, z, np.ascontiguousarray(P[r:]), [0, L], r, False)[0]
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-14)


def test_tail_tokens_never_contribute_and_packing_resets():
    # §4: compression resets at packed-sample boundaries; the L mod r tail is
    # reachable only through the window.
    r, D = 4, 8
    lengths = [13, 4, 22, 3]
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    T = int(cu[-1])
    x, z = _rand(T, D), _rand(T, D)
    P = _rand(2 * r, D)
    packed = oracle.compress(x, z, P, cu, r, True)
    cu_cmp = oracle.compressed_offsets(cu, r)
    for b, L in enumerate(lengths):
        s = slice(cu[b], cu[b + 1])
        alone = oracle.compress(x[s], z[s], P, [0, L], r, True)
        np.testing.assert_array_equal(packed[cu_cmp[b]:cu_cmp[b + 1]], alone)
        # tail perturbation leaves everything unchanged
        if L % r:
            x2 = x.copy()
            x2[cu[b + 1] - 1] += 3.0
            np.testing.assert_array_equal(oracle.compress(x2, z, P, cu, r, True), packed)
