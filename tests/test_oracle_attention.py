"""Pins for the oracle's selected / HCA / window attention (CPU only).

Per (query, head): softmax over the compressed candidates (top-k rows, or all
visible entries for HCA, none for window-only) together with the local window,
optional FP32 sink in the denominator, output and LSE ("DeepSeek-V4 Attention
Training Systems", §2 phase table, §5.3, §8.2, §9).  The oracle is pinned to
torch's scaled_dot_product_attention (float64, CPU) with an explicit boolean
mask built from the candidate sets, to torch.logsumexp, to closed forms for
the sink, and to the dense-mode / window-only reductions.
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from compressed_sparse_attention_compress_gb300.inputs import bf16_round

rng = np.random.default_rng(7)


def _rand(*shape):
    return bf16_round(rng.standard_normal(shape).astype(np.float32))


def _mask_reference(q, keys, vals, mask, scale, sink=None):
    """SDPA over an explicit [T, n_keys] boolean mask; lse via torch.logsumexp."""
    qt = torch.from_numpy(q.astype(np.float64)).permute(1, 0, 2)           # [H, T, d]
    kt = torch.from_numpy(keys.astype(np.float64))[None].expand(q.shape[1], -1, -1)
    vt = torch.from_numpy(vals.astype(np.float64))[None].expand(q.shape[1], -1, -1)
    mt = torch.from_numpy(mask)[None]
    o = F.scaled_dot_product_attention(qt, kt, vt, attn_mask=mt, scale=scale)
    s = torch.einsum("htd,kd->htk", qt, kt[0]) * scale
    lse = torch.logsumexp(s.masked_fill(~mt, float("-inf")), dim=-1)      # [H, T]
    o, lse = o.permute(1, 0, 2).numpy(), lse.T.numpy()
    if sink is not None:   # closed form: the sink only adds exp(sink) to the denominator
        lse_s = np.logaddexp(lse, sink[None, :].astype(np.float64))
        o = o * np.exp(lse - lse_s)[:, :, None]
        lse = lse_s
    return o, lse, s


def _window_mask(T, W):
    t = np.arange(T)
    return (t[None, :] <= t[:, None]) & (t[None, :] > t[:, None] - W)


@pytest.mark.parametrize("W", [1000, 17])
def test_window_only_is_banded_causal_sdpa(W):
    L, H, d = 60, 3, 16
    q, kv, v = _rand(L, H, d), _rand(L, d), _rand(L, d)
    scale = 0.25
    o, lse, lse_c, err = oracle.attention(oracle.KIND_WINDOW, q, None, None, kv, v, [0, L], 0, W, scale)
    ref_o, ref_lse, _ = _mask_reference(q, kv, v, _window_mask(L, W), scale)
    np.testing.assert_allclose(o, ref_o, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse, ref_lse, rtol=1e-12, atol=1e-12)
    assert np.all(np.isneginf(lse_c)) and not err.any()
    if W >= L:   # textbook causal attention
        qt = torch.from_numpy(q.astype(np.float64)).permute(1, 0, 2)
        kt = torch.from_numpy(kv.astype(np.float64))[None].expand(H, -1, -1)
        vt = torch.from_numpy(v.astype(np.float64))[None].expand(H, -1, -1)
        causal = F.scaled_dot_product_attention(qt, kt, vt, is_causal=True, scale=scale)
        np.testing.assert_allclose(o, causal.permute(1, 0, 2).numpy(), rtol=1e-12, atol=1e-13)


def _csa_case(L=80, r=4, H=4, d=16, W=9, k=5, k_pad=8, seed_rows=None):
    n_c = L // r
    q = _rand(L, H, d)
    kc, vc = _rand(n_c, d), _rand(n_c, d)
    kr, vr = _rand(L, d), _rand(L, d)
    idx = np.full((L, k_pad), -1, np.int32)
    for t in range(L):
        n = (t + 1) // r
        m = min(k, n)
        idx[t, :m] = np.sort(rng.choice(n, m, replace=False)) if m else []
    return q, kc, vc, kr, vr, idx


def test_selected_attention_matches_masked_sdpa():
    L, r, W = 80, 4, 9
    q, kc, vc, kr, vr, idx = _csa_case(L, r, W=W)
    scale = 1 / 4
    o, lse, lse_c, err = oracle.attention(oracle.KIND_CSA, q, kc, vc, kr, vr, [0, L], r, W, scale, idx=idx)
    n_c = kc.shape[0]
    mask = np.zeros((L, n_c + L), bool)
    for t in range(L):
        sel = idx[t][idx[t] >= 0]
        mask[t, sel] = True
    mask[:, n_c:] = _window_mask(L, W)
    keys, vals = np.concatenate([kc, kr]), np.concatenate([vc, vr])
    ref_o, ref_lse, s = _mask_reference(q, keys, vals, mask, scale)
    np.testing.assert_allclose(o, ref_o, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse, ref_lse, rtol=1e-12, atol=1e-12)
    # lse_cmp: logsumexp over the selected compressed keys only
    cm = torch.from_numpy(mask[:, :n_c])[None]
    ref_c = torch.logsumexp(s[:, :, :n_c].masked_fill(~cm, float("-inf")), -1).T.numpy()
    np.testing.assert_allclose(lse_c, ref_c, rtol=1e-12, atol=1e-12)
    assert not err.any()


def test_hca_equals_selected_with_every_visible_entry():
    # §2: dense mode / HCA send every completed entry into the candidate list.
    L, r, W = 70, 4, 6
    q, kc, vc, kr, vr, _ = _csa_case(L, r, W=W)
    full = np.full((L, L // r), -1, np.int32)
    for t in range(L):
        n = (t + 1) // r
        full[t, :n] = np.arange(n)
    a = oracle.attention(oracle.KIND_CSA, q, kc, vc, kr, vr, [0, L], r, W, 0.3, idx=full)
    b = oracle.attention(oracle.KIND_HCA, q, kc, vc, kr, vr, [0, L], r, W, 0.3)
    for x, y in zip(a[:3], b[:3]):
        np.testing.assert_allclose(x, y, rtol=1e-14, atol=1e-15)


def test_sink_closed_forms():
    L, r, W, H = 40, 4, 8, 3
    q, kc, vc, kr, vr, idx = _csa_case(L, r, H=H, W=W)
    base = oracle.attention(oracle.KIND_CSA, q, kc, vc, kr, vr, [0, L], r, W, 0.25, idx=idx)
    far = oracle.attention(oracle.KIND_CSA, q, kc, vc, kr, vr, [0, L], r, W, 0.25, idx=idx,
                           sink=np.full(H, -1e30, np.float32))
    for x, y in zip(base[:3], far[:3]):
        np.testing.assert_array_equal(x, y)
    sink = np.array([0.5, -2.0, 3.0], np.float32)
    s_o, s_lse, s_c, _ = oracle.attention(oracle.KIND_CSA, q, kc, vc, kr, vr, [0, L], r, W, 0.25,
                                          idx=idx, sink=sink)
    want_lse = np.logaddexp(base[1], sink[None, :].astype(np.float64))
    np.testing.assert_allclose(s_lse, want_lse, rtol=1e-13)
    np.testing.assert_allclose(s_o, base[0] * np.exp(base[1] - want_lse)[:, :, None], rtol=1e-12, atol=1e-14)
    np.testing.assert_array_equal(s_c, base[2])      # lse_cmp ignores the sink


def test_single_key_output_is_that_value():
    # query 0 of a sequence sees only itself (window, no completed group)
    L, H, d = 5, 2, 8
    q, kv, v = _rand(L, H, d), _rand(L, d), _rand(L, d)
    o, lse, _, _ = oracle.attention(oracle.KIND_WINDOW, q, None, None, kv, v, [0, L], 0, 4, 0.5)
    np.testing.assert_allclose(o[0], np.repeat(v[0:1].astype(np.float64), H, 0), rtol=1e-15)
    np.testing.assert_allclose(lse[0], 0.5 * (q[0].astype(np.float64) @ kv[0].astype(np.float64)), rtol=1e-14)


def test_packing_capacity_rows_and_bad_indices():
    lengths, r, W, H, d = [21, 34], 4, 5, 2, 8
    cu = np.array([0, 21, 55], np.int32)
    T = 55 + 3
    q = _rand(T, H, d)
    kr = _rand(T, d)
    cu_cmp = oracle.compressed_offsets(cu, r)
    kc = _rand(int(cu_cmp[-1]), d)
    idx = np.full((T, 4), -1, np.int32)
    for row in range(55):
        b = int(row >= 21)
        t = row - cu[b]
        n = (t + 1) // r
        m = min(3, n)
        idx[row, :m] = np.sort(rng.choice(n, m, replace=False)) + cu_cmp[b] if m else []
    o, lse, lse_c, err = oracle.attention(oracle.KIND_CSA, q, kc, None, kr, None, cu, r, W, 0.3, idx=idx)
    assert np.all(o[55:] == 0) and np.all(np.isneginf(lse[55:])) and not err.any()
    for b, L in enumerate(lengths):
        s = slice(cu[b], cu[b + 1])
        loc = np.where(idx[s] >= 0, idx[s] - cu_cmp[b], -1)
        a = oracle.attention(oracle.KIND_CSA, q[s], kc[cu_cmp[b]:cu_cmp[b + 1]], None, kr[s], None,
                             [0, L], r, W, 0.3, idx=loc)
        np.testing.assert_array_equal(a[0], o[s])
        np.testing.assert_array_equal(a[1], lse[s])
    bad = idx.copy()
    bad[30, 0] = cu_cmp[-1] - 1        # an entry the query cannot see yet
    *_, err = oracle.attention(oracle.KIND_CSA, q, kc, None, kr, None, cu, r, W, 0.3, idx=bad)
    assert err[30] == 1 and err.sum() == 1
