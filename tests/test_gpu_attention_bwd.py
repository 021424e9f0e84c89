"""GPU parity of the attention backward (csa_sparse_attn_bwd, hca_attn_bwd,
window_attn_bwd) against the fp64 oracle.

"DeepSeek-V4 Attention Training Systems" §8.2: the main attention backward
consumes the saved output and LSE and produces Q, KV and attention-sink
gradients.  The GPU forward produces out and LSE, the GPU backward consumes
them; the oracle recomputes everything from the same synthetic inputs (random
rows and random valid index sets, never a GPU result).

Tolerance.  The kernels round P and scale*dS to bf16 for the tensor-core
products (relative error 2^-9 per term) and sum in float32; with n terms of
mixed sign the error of a gradient entry is about 2^-9 sqrt(n) times a typical
term, far below the largest entry of the tensor.  Each gradient tensor G is
compared elementwise as |gpu - ref| <= 1e-2 max|ref| + 2e-2 |ref|; bf16 dq
also gets the half-ulp of its own storage rounding.
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

ATOL_FRAC, RTOL = 1e-2, 2e-2


def _close(name, got, ref, quant=0.0):
    got, ref = np.asarray(got, np.float64), np.asarray(ref, np.float64)
    if ref.size == 0:
        return
    bound = ATOL_FRAC * np.abs(ref).max() + RTOL * np.abs(ref) + quant
    bad = np.abs(got - ref) > bound
    assert not bad.any(), f"{name}: {bad.sum()} of {ref.size} outside, worst {np.abs(got - ref).max()}"


def _dev(a, fp32):
    t = torch.from_numpy(np.ascontiguousarray(a)).cuda()
    return t if fp32 else t.to(torch.bfloat16)


def _run(kind, lengths, H=64, d=128, ratio=4, window=128, topk=96, k_pad=128, separate_v=False, sink=False,
         fp32=False, seed=0, cap_align=64, rows=None, check_kv=True):
    K = oracle.KIND_CSA if kind == "csa" else oracle.KIND_HCA if kind == "hca" else oracle.KIND_WINDOW
    r = ratio if K != oracle.KIND_WINDOW else 0
    a = I.generate_attention_bwd(lengths, H, d, ratio if r else 1, topk if K == oracle.KIND_CSA else 0, k_pad,
                                 separate_v, sink, seed, cap_align)
    cu_np = a["cu_seqlens"]
    T_cap = a["q"].shape[0]
    h = api.Handle(0)
    cu = torch.from_numpy(cu_np).cuda()
    cmp_np = oracle.compressed_offsets(cu_np, r) if r else np.zeros(len(lengths) + 1, np.int32)
    cu_cmp = torch.from_numpy(cmp_np).cuda()
    q, g = _dev(a["q"], fp32), _dev(a["dout"], fp32)
    kr, kc = _dev(a["k_raw"], fp32), _dev(a["k_cmp"], fp32)
    vr = _dev(a["v_raw"], fp32) if separate_v else None
    vc = _dev(a["v_cmp"], fp32) if separate_v else None
    sk = torch.from_numpy(a["sink"]).cuda() if sink else None
    idx = torch.from_numpy(a["idx"]).cuda() if K == oracle.KIND_CSA else None
    scale = 1.0 / np.sqrt(d)
    ms = max(lengths + [1])
    out = torch.empty_like(q)
    lse = torch.empty(T_cap, H, dtype=torch.float32, device="cuda")
    lse_c = torch.empty_like(lse)
    dq = torch.full_like(q, 5.0)
    n_cap = max(1, T_cap // ratio)
    dkc = torch.full((n_cap, d), 3.0, dtype=torch.float32, device="cuda")     # the call zeroes them
    dkr = torch.full((T_cap, d), 3.0, dtype=torch.float32, device="cuda")
    dvc = torch.full_like(dkc, 3.0) if separate_v else None
    dvr = torch.full_like(dkr, 3.0) if separate_v else None
    dsink = torch.full((H,), 9.0, dtype=torch.float32, device="cuda") if sink else None
    delta = torch.empty(T_cap, H, dtype=torch.float32, device="cuda")
    if K == oracle.KIND_CSA:
        api.csa_sparse_attn_fwd(h, q, kc, kr, idx, cu, cu_cmp, ms, ratio, window, scale, out, lse, lse_c,
                                v_cmp=vc, v_raw=vr, sink=sk)
        api.csa_sparse_attn_bwd(h, q, kc, kr, idx, cu, cu_cmp, ms, ratio, window, scale, out, lse, g, dq, dkc, dkr,
                                delta, v_cmp=vc, v_raw=vr, dv_cmp=dvc, dv_raw=dvr, sink=sk, dsink=dsink)
    elif K == oracle.KIND_HCA:
        api.hca_attn_fwd(h, q, kc, kr, cu, cu_cmp, ms, ratio, window, scale, out, lse, lse_c, v_cmp=vc, v_raw=vr,
                         sink=sk)
        api.hca_attn_bwd(h, q, kc, kr, cu, cu_cmp, ms, ratio, window, scale, out, lse, g, dq, dkc, dkr, delta,
                         v_cmp=vc, v_raw=vr, dv_cmp=dvc, dv_raw=dvr, sink=sk, dsink=dsink)
    else:
        api.window_attn_fwd(h, q, kr, cu, ms, window, scale, out, lse, v_raw=vr, sink=sk)
        api.window_attn_bwd(h, q, kr, cu, ms, window, scale, out, lse, g, dq, dkr, delta, v_raw=vr, dv_raw=dvr,
                            sink=sk, dsink=dsink)
    torch.cuda.synchronize()
    assert h.device_status() == 0
    T = int(cu_np[-1])
    rows = np.arange(T_cap) if rows is None else np.asarray(rows)
    ref = oracle.attention_bwd(K, a["q"], a["k_cmp"] if r else None, a.get("v_cmp") if r else None, a["k_raw"],
                               a.get("v_raw"), cu_np, r, window, scale, a["dout"], idx=a.get("idx"),
                               sink=a.get("sink"), rows=rows, want_kv=check_kv)
    dq_np = ph.np32(dq)[rows]
    _close("dq", dq_np, ref["dq"], ph.bf16_half_ulp(ref["dq"]) if not fp32 else 0.0)
    assert not np.any(dq_np[rows >= T])     # capacity rows
    if check_kv:
        n_c = int(cmp_np[-1])
        if separate_v:
            if r:
                _close("dk_cmp", ph.np32(dkc)[:n_c], ref["dk_cmp"][:n_c])
                _close("dv_cmp", ph.np32(dvc)[:n_c], ref["dv_cmp"][:n_c])
            _close("dk_raw", ph.np32(dkr)[:T], ref["dk_raw"][:T])
            _close("dv_raw", ph.np32(dvr)[:T], ref["dv_raw"][:T])
        else:
            if r:
                _close("dkv_cmp", ph.np32(dkc)[:n_c], ref["dk_cmp"][:n_c] + ref["dv_cmp"][:n_c])
            _close("dkv_raw", ph.np32(dkr)[:T], ref["dk_raw"][:T] + ref["dv_raw"][:T])
        assert not ph.np32(dkr)[T:].any()
        if r:
            assert not ph.np32(dkc)[n_c:].any()
        if sink:
            _close("dsink", ph.np32(dsink), ref["dsink"])
    return dict(q=q, out=out, dout=g, dq=dq, dkc=dkc, dkr=dkr, kc=kc, kr=kr, T=T, n_c=int(cmp_np[-1]))


RAGGED = [700, 0, 301, 1029, 5]


@pytest.mark.parametrize("kind", ["csa", "hca", "window"])
@pytest.mark.parametrize("sink", [False, True])
def test_64_heads_bf16_ragged(kind, sink):
    _run(kind, RAGGED, sink=sink, ratio=4 if kind != "hca" else 128, window=128 if kind != "window" else 100)


@pytest.mark.parametrize("kind", ["csa", "hca", "window"])
def test_separate_v_fp32_small_heads(kind):
    _run(kind, [389, 120, 3], H=4, d=64, ratio=4, window=37, topk=40, k_pad=64, separate_v=True, sink=True,
         fp32=True, seed=3)


@pytest.mark.parametrize("H,d", [(16, 64), (32, 128), (128, 128)])
def test_head_shapes(H, d):
    _run("csa", [517, 64], H=H, d=d, topk=50, k_pad=64, seed=5)


def test_k_covers_every_visible_entry():
    _run("csa", [600], topk=150, k_pad=152, seed=8)


def test_full_size_warmup_layer_sampled_rows_and_identity():
    # the sparse warm-up layer at L = 32768 (k = 2048): dq on sampled rows
    # against the oracle; the key gradients through the chain-rule identity
    # sum_j dKV_j . KV_j = sum_{t,h} (dq . q + dout . out), which holds for the
    # whole tensors at any size
    L = 32768
    rng = np.random.default_rng(0)
    rows = np.sort(np.concatenate([rng.choice(L, 48, replace=False), [0, 3, 4, 8191, L - 1]]))
    res = _run("csa", [L], topk=2048, k_pad=2048, rows=rows, check_kv=False, cap_align=128)
    f64 = lambda t: t.double()  # noqa: E731
    lhs = (f64(res["dkc"][:res["n_c"]]) * f64(res["kc"][:res["n_c"]])).sum() + \
        (f64(res["dkr"][:res["T"]]) * f64(res["kr"][:res["T"]])).sum()
    rhs = (f64(res["dq"]) * f64(res["q"])).sum() + (f64(res["dout"]) * f64(res["out"])).sum()
    assert abs(float(lhs - rhs)) <= 1e-2 * max(1.0, abs(float(rhs))), (float(lhs), float(rhs))


def test_argument_errors():
    h = api.Handle(0)
    T, H, d = 64, 64, 128
    cu = torch.tensor([0, T], dtype=torch.int32, device="cuda")
    cu_cmp = torch.tensor([0, T // 4], dtype=torch.int32, device="cuda")
    q = torch.zeros(T, H, d, dtype=torch.bfloat16, device="cuda")
    kv = torch.zeros(T, d, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(T, H, device="cuda")
    f = torch.zeros(T, d, device="cuda")
    idx = torch.zeros(T, 4, dtype=torch.int32, device="cuda")
    with pytest.raises(api.CSAError) as e:   # separate V without its gradient buffer
        api.csa_sparse_attn_bwd(h, q, kv, kv, idx, cu, cu_cmp, T, 4, 16, 0.1, q, lse, q, q, f, f, lse,
                                v_cmp=kv, v_raw=kv)
    assert e.value.code == -1
    q96 = torch.zeros(T, H, 96, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(api.CSAError) as e:   # head dim 96 has no kernel
        api.window_attn_bwd(h, q96, kv, cu, T, 16, 0.1, q96, lse, q96, q96, f, lse)
    assert e.value.code == -2
    assert h.device_status() == 0
