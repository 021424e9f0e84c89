"""GPU parity of the indexer backward (csa_indexer_kl_bwd) against the fp64 oracle.

"DeepSeek-V4 Attention Training Systems" §8.2: the indexer is trained through
its KL auxiliary loss only, with the teacher detached.  Inputs are synthetic
(random rows and random valid index sets); in sparse mode the per-head
normaliser lse_cmp comes from the GPU attention forward on the same inputs,
as the product path passes it.

Tolerance.  The teacher scores run on bf16 tensor-core operands and the
exponentials in float32, so g = q - p carries absolute errors of about 1e-3 of
the largest probability; each gradient tensor is compared elementwise as
|gpu - ref| <= 1e-2 max|ref| + 2e-2 |ref| (+ the half-ulp of bf16 outputs).
"""
import numpy as np
import pytest
import torch

import oracle
from compressed_sparse_attention_compress_gb300 import inputs as I
from tests import parity_helpers as ph

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # the CPU suite never collects GPU work
    pytest.skip("no CUDA device", allow_module_level=True)

from compressed_sparse_attention_compress_gb300 import api  # noqa: E402


def _close(name, got, ref, quant=0.0):
    got, ref = np.asarray(got, np.float64), np.asarray(ref, np.float64)
    if ref.size == 0:
        return
    bound = 1e-2 * np.abs(ref).max() + 2e-2 * np.abs(ref) + quant
    bad = np.abs(got - ref) > bound
    assert not bad.any(), f"{name}: {bad.sum()} of {ref.size} outside, worst {np.abs(got - ref).max()}"


def _run(lengths, mode, H=64, d=128, H_I=8, d_I=64, ratio=4, topk=96, k_pad=128, fp32=False, seed=0,
         grad_scale=1.0, cap_align=64, rows=None, check_kI=True, stats=False, check_stats=True):
    sparse = mode != "dense"
    a = I.generate_indexer_bwd(lengths, H, d, H_I, d_I, ratio, topk if sparse else 0, k_pad, seed, cap_align)
    cu_np = a["cu_seqlens"]
    T_cap = a["q"].shape[0]
    dev = lambda k: (torch.from_numpy(a[k]).cuda() if fp32 else torch.from_numpy(a[k]).cuda().to(torch.bfloat16))  # noqa: E731
    h = api.Handle(0)
    cu = torch.from_numpy(cu_np).cuda()
    cmp_np = oracle.compressed_offsets(cu_np, ratio)
    cu_cmp = torch.from_numpy(cmp_np).cuda()
    q, kc, qI, w, kI = dev("q"), dev("k_cmp"), dev("qI"), dev("w"), dev("k_I")
    idx = torch.from_numpy(a["idx"]).cuda() if sparse else None
    scale = 1.0 / np.sqrt(d)
    ms = max(lengths + [1])
    lse_cmp = None
    if mode == "sparse_lse":   # the per-head normaliser over C_t from the attention forward
        kr = dev("k_raw")
        out = torch.empty_like(q)
        lse = torch.empty(T_cap, H, dtype=torch.float32, device="cuda")
        lse_cmp = torch.empty_like(lse)
        api.csa_sparse_attn_fwd(h, q, kc, kr, idx, cu, cu_cmp, ms, ratio, 128, scale, out, lse, lse_cmp)
    student_lse = None
    if stats:   # the KL forward keeps both normalisers; the backward then takes one pass
        teacher_lse = torch.full((T_cap, H), 7.0, dtype=torch.float32, device="cuda")
        student_lse = torch.full((T_cap,), 7.0, dtype=torch.float32, device="cuda")
        kl_sum = torch.zeros(1, device="cuda")
        ws = torch.empty(api.csa_indexer_kl_workspace(T_cap), dtype=torch.uint8, device="cuda")
        api.csa_indexer_kl_ex(h, q, kc, qI, w, kI, cu, cu_cmp, ms, ratio, scale, kl_sum, ws, teacher_lse=teacher_lse,
                              student_lse=student_lse, idx=idx, lse_cmp=lse_cmp)
        torch.cuda.synchronize()
        if check_stats:
            _check_stats(a, cu_np, ratio, scale, idx, teacher_lse, student_lse)
        lse_cmp = teacher_lse
    dqI = torch.full_like(qI, 5.0)
    dw = torch.full_like(w, 5.0)
    dkI = torch.full((max(1, T_cap // ratio), d_I), 3.0, dtype=torch.float32, device="cuda")
    api.csa_indexer_kl_bwd(h, q, kc, qI, w, kI, cu, cu_cmp, ms, ratio, scale, dqI, dw, dkI, idx=idx,
                           lse_cmp=lse_cmp, student_lse=student_lse, grad_scale=grad_scale)
    torch.cuda.synchronize()
    assert h.device_status() == 0
    T = int(cu_np[-1])
    rows = np.arange(T_cap) if rows is None else np.asarray(rows)
    ref = oracle.indexer_kl_bwd(a["q"], a["k_cmp"], a["qI"], a["w"], a["k_I"], cu_np, ratio, scale,
                                idx=a.get("idx"), rows=rows, grad_scale=grad_scale, want_kI=check_kI)
    bf = not fp32
    _close("dqI", ph.np32(dqI)[rows], ref["dqI"], ph.bf16_half_ulp(ref["dqI"]) if bf else 0.0)
    _close("dw", ph.np32(dw)[rows], ref["dw"], ph.bf16_half_ulp(ref["dw"]) if bf else 0.0)
    assert not ph.np32(dqI)[rows][rows >= T].any()
    if check_kI:
        n_c = int(cmp_np[-1])
        _close("dkI", ph.np32(dkI)[:n_c], ref["dkI"][:n_c])
        assert not ph.np32(dkI)[n_c:].any()
    return dict(dqI=dqI, dw=dw, dkI=dkI, qI=qI, w=w, kI=kI, n_c=int(cmp_np[-1]))


def _check_stats(a, cu_np, ratio, scale, idx, teacher_lse, student_lse):
    """teacher_lse against the attention oracle's compressed-only normaliser (the
    same logsumexp over C_t), student_lse against logsumexp of the oracle's
    indexer logits over C_t."""
    T_cap = a["q"].shape[0]
    T = int(cu_np[-1])
    idx_np = idx.cpu().numpy() if idx is not None else None
    kind = oracle.KIND_CSA if idx_np is not None else oracle.KIND_HCA
    _, _, ref_t, _ = oracle.attention(kind, a["q"], a["k_cmp"], None, a["k_raw"], None, cu_np, ratio, 1, scale,
                                      idx=idx_np)
    got_t = ph.np32(teacher_lse)
    fin = np.isfinite(ref_t)
    assert np.array_equal(fin, np.isfinite(got_t))
    np.testing.assert_allclose(got_t[fin], ref_t[fin], rtol=0, atol=1e-2)
    max_vis = max(1, int(np.diff(cu_np).max()) // ratio)
    logits, nvis = oracle.indexer_logits(a["qI"], a["w"], a["k_I"], cu_np, ratio, None, max_vis)
    cmp_np = oracle.compressed_offsets(cu_np, ratio)
    got_s = ph.np32(student_lse)
    for row in range(T_cap):
        if row >= T:
            assert got_s[row] == -np.inf
            continue
        b = int(np.searchsorted(cu_np, row, side="right") - 1)
        js = (np.arange(nvis[row]) if idx_np is None else idx_np[row][idx_np[row] >= 0] - cmp_np[b])
        if js.size == 0:
            assert got_s[row] == -np.inf
            continue
        ref = np.logaddexp.reduce(logits[row, js])
        assert abs(got_s[row] - ref) <= 1e-3 * max(1.0, abs(ref)), (row, got_s[row], ref)


RAGGED = [700, 0, 301, 1029, 5]


@pytest.mark.parametrize("mode", ["sparse", "sparse_lse", "dense"])
def test_64_heads_bf16_ragged(mode):
    _run(RAGGED, mode)


@pytest.mark.parametrize("mode", ["sparse", "dense"])
def test_one_pass_with_the_forward_normalisers(mode):
    _run(RAGGED, mode, stats=True, seed=4)


@pytest.mark.parametrize("mode", ["sparse", "dense"])
def test_small_shapes_fp32(mode):
    _run([389, 120, 3], mode, H=16, d=64, H_I=4, d_I=32, topk=40, k_pad=64, fp32=True, seed=3)


@pytest.mark.parametrize("H,H_I", [(4, 1), (128, 8)])
def test_head_counts(H, H_I):
    _run([517, 64], "sparse", H=H, H_I=H_I, topk=50, k_pad=64, seed=5, grad_scale=-3.0)


@pytest.mark.parametrize("grad_scale", [1.0, -3.0])
def test_one_pass_dense_tensor_core_path_ragged(grad_scale):
    # the dense teacher with both forward normalisers at 64 x 128 heads and an
    # 8 x 64 indexer runs the tcgen05 kernel: blocks of 4 queries, ragged ends,
    # an empty sequence, prefixes of 1 to 9 tiles
    _run([1029, 3, 0, 517, 130, 4600], "dense", stats=True, seed=6, grad_scale=grad_scale)


@pytest.mark.parametrize("grad_scale", [1.0, -3.0])
def test_one_pass_sparse_tensor_core_path_several_tiles(grad_scale):
    # the selected teacher with both forward normalisers at 64 x 128 heads and an
    # 8 x 64 indexer runs the tcgen05 kernel: gathered 128-entry tiles, one to
    # three per query (holes where a slot is -1), an empty sequence and
    # sequences shorter than one compressed block; every row against the oracle
    _run([900, 3, 0, 517, 1300], "sparse", topk=300, k_pad=384, stats=True, seed=7, grad_scale=grad_scale)


def test_full_size_sparse_layer_sampled():
    # the selected teacher at L = 8192, k = 512 (the CSA sparse-mode layer, one
    # pass on the tensor cores): dqI and dw on sampled rows against the oracle;
    # dkI through the homogeneity identity sum kI.dkI = sum w.dw
    L = 8192
    rng = np.random.default_rng(2)
    rows = np.sort(np.concatenate([rng.choice(L, 24, replace=False), [3, 4, 2047, L - 1]]))
    res = _run([L], "sparse", topk=512, k_pad=512, rows=rows, check_kI=False, cap_align=128, stats=True,
               check_stats=False, seed=8)
    f64 = lambda t: t.double()  # noqa: E731
    lhs = (f64(res["dkI"][:res["n_c"]]) * f64(res["kI"][:res["n_c"]])).sum()
    rhs = (f64(res["dw"]) * f64(res["w"])).sum()
    assert abs(float(lhs - rhs)) <= 2e-2 * max(1e-3, float((f64(res["dw"]).abs() * f64(res["w"]).abs()).sum()))


@pytest.mark.parametrize("stats", [False, True])
def test_full_size_dense_warmup_layer_sampled(stats):
    # the dense teacher at L = 32768 (with the forward's normalisers: the
    # one-pass tensor-core kernel): dqI and dw on sampled rows against the
    # oracle; dkI through the homogeneity identity sum kI.dkI = sum w.dw, which
    # holds for the whole tensors at any size
    L = 32768
    rng = np.random.default_rng(1)
    rows = np.sort(np.concatenate([rng.choice(L, 24, replace=False), [3, 4, 8191, L - 1]]))
    res = _run([L], "dense", rows=rows, check_kI=False, cap_align=128, stats=stats, check_stats=False)
    f64 = lambda t: t.double()  # noqa: E731
    lhs = (f64(res["dkI"][:res["n_c"]]) * f64(res["kI"][:res["n_c"]])).sum()
    rhs = (f64(res["dw"]) * f64(res["w"])).sum()
    assert abs(float(lhs - rhs)) <= 2e-2 * max(1e-3, float((f64(res["dw"]).abs() * f64(res["w"]).abs()).sum()))


def test_one_pass_dense_tensor_core_path_tiny_sequences():
    # many sequences of 0-9 tokens (blocks of 1-4 queries, prefixes of 0-2
    # entries: empty blocks, partial tiles) around one of three tiles
    _run([1, 2, 3, 4, 5, 0, 6, 7, 8, 9, 1500, 3, 4, 2], "dense", stats=True, seed=8)


def test_one_pass_dense_tensor_core_path_zero_upstream_gradient():
    res = _run([900, 77], "dense", stats=True, seed=2, grad_scale=0.0)
    for k in ("dqI", "dw", "dkI"):
        assert not bool(res[k].float().abs().sum()), k
