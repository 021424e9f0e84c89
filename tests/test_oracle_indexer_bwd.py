"""Pins for the oracle's indexer backward (CPU only).

The indexer is trained only through the KL auxiliary loss ("DeepSeek-V4
Attention Training Systems" §3 equation, §8.2 "indexer backward ... a separate
auxiliary-gradient path"; the teacher operands are detached).  The oracle's
gradients with respect to qI, w and kI are pinned to torch autograd (float64)
of the loss written with torch.log_softmax and torch.relu, to central
differences of the forward KL oracle, and to the identities that positive
homogeneity of ReLU gives at any size.
"""
import numpy as np
import pytest
import torch

import oracle
from compressed_sparse_attention_compress_gb300.inputs import bf16_round

rng = np.random.default_rng(21)


def _rand(*shape):
    return bf16_round(rng.standard_normal(shape).astype(np.float32))


def _case(lengths, r=4, H=4, d=16, H_I=2, dI=8, sparse=True, k=6, k_pad=8):
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    T = int(cu[-1])
    cu_cmp = oracle.compressed_offsets(cu, r)
    n_c = max(1, int(cu_cmp[-1]))
    c = dict(cu=cu, cu_cmp=cu_cmp, r=r, q=_rand(T, H, d), kc=_rand(n_c, d), qI=_rand(T, H_I, dI),
             w=_rand(T, H_I), kI=_rand(n_c, dI), scale=1.0 / np.sqrt(d), idx=None)
    if sparse:
        idx = np.full((T, k_pad), -1, np.int32)
        for b in range(len(lengths)):
            for t in range(lengths[b]):
                nvis = (t + 1) // r
                pick = rng.choice(nvis, min(k, nvis), replace=False) if nvis else []
                idx[cu[b] + t, :len(pick)] = np.sort(cu_cmp[b] + np.asarray(pick, np.int64))
        c["idx"] = idx
    return c


def _sets(c):
    T = c["q"].shape[0]
    out = []
    for row in range(T):
        b = int(np.searchsorted(c["cu"], row, side="right") - 1)
        t = row - c["cu"][b]
        nvis = (t + 1) // c["r"]
        if c["idx"] is not None:
            js = [g for g in c["idx"][row] if g >= 0]
        else:
            js = list(range(c["cu_cmp"][b], c["cu_cmp"][b] + nvis))
        out.append(np.asarray(js, np.int64))
    return out


def _torch_grads(c, grad_scale=1.0):
    f64 = lambda a, g=False: torch.tensor(a, dtype=torch.float64, requires_grad=g)  # noqa: E731
    q, kc = f64(c["q"]), f64(c["kc"])
    qI, w, kI = f64(c["qI"], True), f64(c["w"], True), f64(c["kI"], True)
    loss = torch.zeros((), dtype=torch.float64)
    for row, js in enumerate(_sets(c)):
        if js.size == 0:
            continue
        jt = torch.from_numpy(js)
        with torch.no_grad():   # the teacher is detached
            p = torch.softmax(c["scale"] * q[row] @ kc[jt].T, dim=-1).mean(0)
        i = (w[row][:, None] * torch.relu(qI[row] @ kI[jt].T)).sum(0)
        loss = loss + (p * (torch.log(p) - torch.log_softmax(i, dim=-1))).sum()
    (grad_scale * loss).backward()
    return {"dqI": qI.grad.numpy(), "dw": w.grad.numpy(), "dkI": kI.grad.numpy()}


def _oracle(c, **kw):
    return oracle.indexer_kl_bwd(c["q"], c["kc"], c["qI"], c["w"], c["kI"], c["cu"], c["r"], c["scale"],
                                 idx=c["idx"], **kw)


@pytest.mark.parametrize("sparse", [True, False])
def test_matches_torch_autograd(sparse):
    c = _case([37, 0, 50, 3], sparse=sparse)
    got, ref = _oracle(c, grad_scale=0.75), _torch_grads(c, grad_scale=0.75)
    assert not got["err"].any()
    for k in ("dqI", "dw", "dkI"):
        np.testing.assert_allclose(got[k], ref[k], rtol=1e-10, atol=1e-12, err_msg=k)


def _kl_sum(c, **over):
    cc = dict(c, **over)
    kl, _, _ = oracle.indexer_kl(cc["q"], cc["kc"], cc["qI"], cc["w"], cc["kI"], cc["cu"], cc["r"], cc["scale"],
                                 idx=cc["idx"])
    return float(kl.sum())


def test_central_differences_of_the_forward_kl():
    c = _case([26, 19], sparse=True)
    g = _oracle(c)
    h = 2.0 ** -10
    for name, gname, at in [("qI", "dqI", (9, 1, 3)), ("qI", "dqI", (30, 0, 0)), ("w", "dw", (17, 1)),
                            ("w", "dw", (40, 0)), ("kI", "dkI", (2, 5)), ("kI", "dkI", (6, 1))]:
        a = c[name]
        ap, am = a.copy(), a.copy()
        ap[at] += h
        am[at] -= h
        fd = (_kl_sum(c, **{name: ap}) - _kl_sum(c, **{name: am})) / (2 * h)
        assert abs(fd - g[gname][at]) <= 1e-5 * max(1.0, abs(fd)), (name, at, fd, g[gname][at])


@pytest.mark.parametrize("sparse", [True, False])
def test_homogeneity_identities(sparse):
    # ReLU is positively homogeneous, so scaling w, qI or kI by a scales every
    # indexer logit by a: each of sum w.dw, sum qI.dqI and sum kI.dkI equals
    # sum_t sum_{j in C_t} g_tj i_tj
    c = _case([44, 31], sparse=sparse)
    g = _oracle(c)
    logits = []
    for row, js in enumerate(_sets(c)):
        if js.size:
            i = (c["w"][row].astype(np.float64)[:, None] *
                 np.maximum(c["qI"][row].astype(np.float64) @ c["kI"][js].astype(np.float64).T, 0)).sum(0)
            logits.append((row, js, i))
    # g_tj from the definition q - p, with the teacher from the attention oracle's per-head softmax
    total = 0.0
    for row, js, i in logits:
        s = c["scale"] * c["q"][row].astype(np.float64) @ c["kc"][js].astype(np.float64).T
        p = np.exp(s - s.max(1, keepdims=True))
        p = (p / p.sum(1, keepdims=True)).mean(0)
        qd = np.exp(i - i.max())
        qd /= qd.sum()
        total += ((qd - p) * i).sum()
    np.testing.assert_allclose((g["dw"] * c["w"]).sum(), total, rtol=1e-10)
    np.testing.assert_allclose((g["dqI"] * c["qI"]).sum(), total, rtol=1e-10)
    np.testing.assert_allclose((g["dkI"] * c["kI"]).sum(), total, rtol=1e-10)


def test_rows_without_entries_and_linearity_in_the_upstream_gradient():
    c = _case([3, 30])
    a = _oracle(c, grad_scale=1.0)
    b = _oracle(c, grad_scale=-2.5)
    for k in ("dqI", "dw", "dkI"):
        np.testing.assert_allclose(b[k], -2.5 * a[k], rtol=1e-12, atol=1e-15)
    assert not a["dqI"][:3].any() and not a["dw"][:3].any()   # t < r - 1: no visible entry
