"""Pins for the oracle's attention backward (CPU only).

The backward of the selected / HCA / window attention ("DeepSeek-V4 Attention
Training Systems", §8.2 main attention backward: Q, KV and attention-sink
gradients from saved output and LSE) is pinned to torch autograd (float64)
through a dense masked formulation of the forward -- torch's
scaled_dot_product_attention without a sink, torch.softmax over the scores
and the sink logit with one -- to central finite differences of the forward
oracle, and to two identities of the chain rule that hold at any size.
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from compressed_sparse_attention_compress_gb300.inputs import bf16_round

rng = np.random.default_rng(11)


def _rand(*shape):
    return bf16_round(rng.standard_normal(shape).astype(np.float32))


def _case(kind, lengths, r=4, W=8, H=4, d=16, k=5, k_pad=8, separate_v=False, sink=False):
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    T = int(cu[-1])
    cu_cmp = oracle.compressed_offsets(cu, r if kind != oracle.KIND_WINDOW else 0)
    n_c = max(1, int(cu_cmp[-1]))
    c = dict(kind=kind, cu=cu, cu_cmp=cu_cmp, r=r, W=W, q=_rand(T, H, d), kc=_rand(n_c, d), kr=_rand(T, d),
             vc=_rand(n_c, d) if separate_v else None, vr=_rand(T, d) if separate_v else None,
             dout=_rand(T, H, d), scale=1.0 / np.sqrt(d), idx=None,
             sink=rng.standard_normal(H).astype(np.float32) if sink else None)
    if kind == oracle.KIND_CSA:
        idx = np.full((T, k_pad), -1, np.int32)
        for b in range(len(lengths)):
            for t in range(lengths[b]):
                nvis = (t + 1) // r
                pick = rng.choice(nvis, min(k, nvis), replace=False) if nvis else []
                idx[cu[b] + t, :len(pick)] = np.sort(cu_cmp[b] + np.asarray(pick, np.int64))
        c["idx"] = idx
    return c


def _mask(c):
    """[T, n_c + T] candidate mask: compressed rows first, then raw rows."""
    cu, cu_cmp, r, W = c["cu"], c["cu_cmp"], c["r"], c["W"]
    T, n_c = c["q"].shape[0], c["kc"].shape[0]
    m = np.zeros((T, n_c + T), bool)
    for b in range(len(cu) - 1):
        for t in range(cu[b + 1] - cu[b]):
            row = cu[b] + t
            nvis = (t + 1) // r if c["kind"] != oracle.KIND_WINDOW else 0
            if c["kind"] == oracle.KIND_CSA:
                for g in c["idx"][row]:
                    if g >= 0:
                        m[row, g] = True
            elif c["kind"] == oracle.KIND_HCA:
                m[row, cu_cmp[b]:cu_cmp[b] + nvis] = True
            w0 = max(0, t - W + 1)
            m[row, n_c + cu[b] + w0:n_c + cu[b] + t + 1] = True
    return m


def _torch_grads(c):
    f64 = lambda a: torch.tensor(a, dtype=torch.float64, requires_grad=True)  # noqa: E731
    q, kc, kr = f64(c["q"]), f64(c["kc"]), f64(c["kr"])
    vc = f64(c["vc"]) if c["vc"] is not None else kc
    vr = f64(c["vr"]) if c["vr"] is not None else kr
    sink = f64(c["sink"]) if c["sink"] is not None else None
    keys, vals = torch.cat([kc, kr]), torch.cat([vc, vr])
    mask = torch.from_numpy(_mask(c))
    H = q.shape[1]
    qh = q.permute(1, 0, 2)                                            # [H, T, d]
    if sink is None:
        o = F.scaled_dot_product_attention(qh, keys[None].expand(H, -1, -1), vals[None].expand(H, -1, -1),
                                           attn_mask=mask[None], scale=c["scale"])
    else:
        s = torch.einsum("htd,kd->htk", qh, keys) * c["scale"]
        s = s.masked_fill(~mask[None], float("-inf"))
        s = torch.cat([s, sink[:, None, None].expand(-1, s.shape[1], 1)], dim=-1)
        p = torch.softmax(s, dim=-1)[..., :-1]
        o = torch.einsum("htk,kd->htd", p, vals)
    loss = (o.permute(1, 0, 2) * torch.from_numpy(c["dout"].astype(np.float64))).sum()
    loss.backward()
    g = {"dq": q.grad.numpy(), "dk_cmp": kc.grad.numpy(), "dk_raw": kr.grad.numpy()}
    if c["vc"] is not None:
        g["dv_cmp"], g["dv_raw"] = vc.grad.numpy(), vr.grad.numpy()
    if sink is not None:
        g["dsink"] = sink.grad.numpy()
    return g


def _oracle_grads(c, rows=None):
    return oracle.attention_bwd(c["kind"], c["q"], c["kc"], c["vc"], c["kr"], c["vr"], c["cu"], c["r"], c["W"],
                                c["scale"], c["dout"], idx=c["idx"], sink=c["sink"], rows=rows)


KINDS = [oracle.KIND_CSA, oracle.KIND_HCA, oracle.KIND_WINDOW]


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("separate_v", [False, True])
@pytest.mark.parametrize("sink", [False, True])
def test_matches_torch_autograd(kind, separate_v, sink):
    c = _case(kind, [37, 0, 50, 3], separate_v=separate_v, sink=sink)
    got, ref = _oracle_grads(c), _torch_grads(c)
    assert not got["err"].any()
    np.testing.assert_allclose(got["dq"], ref["dq"], rtol=1e-10, atol=1e-12)
    if separate_v:
        pairs = [("dk_cmp", "dk_cmp"), ("dk_raw", "dk_raw"), ("dv_cmp", "dv_cmp"), ("dv_raw", "dv_raw")]
        for a, b in pairs:
            np.testing.assert_allclose(got[a], ref[b], rtol=1e-10, atol=1e-12, err_msg=a)
    else:  # K = V: the shared array's gradient is dk + dv
        np.testing.assert_allclose(got["dk_cmp"] + got["dv_cmp"], ref["dk_cmp"], rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(got["dk_raw"] + got["dv_raw"], ref["dk_raw"], rtol=1e-10, atol=1e-12)
    if sink:
        np.testing.assert_allclose(got["dsink"], ref["dsink"], rtol=1e-10, atol=1e-12)


def _loss(c, **over):
    cc = dict(c, **over)
    o, _, _, _ = oracle.attention(cc["kind"], cc["q"], cc["kc"], cc["vc"], cc["kr"], cc["vr"], cc["cu"], cc["r"],
                                  cc["W"], cc["scale"], idx=cc["idx"], sink=cc["sink"])
    return float((o * cc["dout"].astype(np.float64)).sum())


@pytest.mark.parametrize("kind", KINDS)
def test_central_differences_of_the_forward_oracle(kind):
    # the forward oracle takes float32 inputs, so perturb by a step that float32
    # represents exactly around values of order 1 and compare to 1e-4
    c = _case(kind, [21, 14], separate_v=True, sink=True, d=8, H=2)
    g = _oracle_grads(c)
    h = 2.0 ** -10
    picks = [("q", "dq", (5, 1, 3)), ("q", "dq", (30, 0, 7)), ("kr", "dk_raw", (12, 2)),
             ("vr", "dv_raw", (19, 5)), ("sink", "dsink", (1,))]
    if kind != oracle.KIND_WINDOW:
        picks += [("kc", "dk_cmp", (1, 4)), ("vc", "dv_cmp", (2, 0))]
    for name, gname, at in picks:
        a = c[name]
        ap, am = a.copy(), a.copy()
        ap[at] += h
        am[at] -= h
        fd = (_loss(c, **{name: ap}) - _loss(c, **{name: am})) / (2 * h)
        assert abs(fd - g[gname][at]) <= 1e-4 * max(1.0, abs(fd)), (name, at, fd, g[gname][at])


@pytest.mark.parametrize("kind", KINDS)
def test_chain_rule_identities(kind):
    # sum_j dK_j . K_j = sum_{t,h} dq_{t,h} . q_{t,h}   (both are scale * sum ds * s / scale)
    # sum_j dV_j . V_j = sum_{t,h} dout_{t,h} . o_{t,h}
    c = _case(kind, [40, 25], separate_v=True, sink=True)
    g = _oracle_grads(c)
    o, _, _, _ = oracle.attention(c["kind"], c["q"], c["kc"], c["vc"], c["kr"], c["vr"], c["cu"], c["r"], c["W"],
                                  c["scale"], idx=c["idx"], sink=c["sink"])
    lhs_k = (g["dk_cmp"] * c["kc"]).sum() + (g["dk_raw"] * c["kr"]).sum()
    rhs_k = (g["dq"] * c["q"]).sum()
    lhs_v = (g["dv_cmp"] * c["vc"]).sum() + (g["dv_raw"] * c["vr"]).sum()
    rhs_v = (o * c["dout"]).sum()
    np.testing.assert_allclose(lhs_k, rhs_k, rtol=1e-10)
    np.testing.assert_allclose(lhs_v, rhs_v, rtol=1e-10)


def test_row_subsets_add_up_and_capacity_rows_are_inert():
    c = _case(oracle.KIND_CSA, [30, 22])
    T = c["q"].shape[0]
    full = _oracle_grads(c)
    a = _oracle_grads(c, rows=np.arange(0, T, 2))
    b = _oracle_grads(c, rows=np.arange(1, T, 2))
    for k in ("dk_cmp", "dv_cmp", "dk_raw", "dv_raw"):
        np.testing.assert_allclose(a[k] + b[k], full[k], rtol=1e-12, atol=1e-13)
    np.testing.assert_array_equal(a["dq"], full["dq"][0::2])
    # a capacity row (past cu[B]) has no candidates: zero dq, no contribution
    c2 = dict(c, q=np.concatenate([c["q"], _rand(2, *c["q"].shape[1:])]),
              dout=np.concatenate([c["dout"], _rand(2, *c["q"].shape[1:])]),
              kr=np.concatenate([c["kr"], _rand(2, c["kr"].shape[1])]),
              idx=np.concatenate([c["idx"], np.full((2, c["idx"].shape[1]), -1, np.int32)]))
    cap = _oracle_grads(c2, rows=np.array([T, T + 1]))
    assert not cap["dq"].any() and not cap["dk_cmp"].any() and not cap["dk_raw"].any()
