"""GPU parity: the C-ABI path against the oracle, stage by stage (needs a GPU).

Each stage is fed the values the previous GPU stage produced (its bf16
compressed rows, its index lists), so bf16 rounding in one stage cannot flip a
top-k decision in the next one.  Small cases are checked on every query and
span several tiles with ragged tails; the full-size workloads are checked on a
sample of queries (all, for the KL sum where the oracle is cheap enough).
"""
import dataclasses

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
from compressed_sparse_attention_compress_gb300.forward import Forward, to_device  # noqa: E402


def _run(wl, seed=0, sink=None):
    arrs = I.generate(wl, seed)
    dev = to_device(arrs, wl.io_fp32)
    f = Forward(wl, dev)
    s = None if sink is None else torch.from_numpy(sink).cuda()
    f.run(sink=s)
    torch.cuda.synchronize()
    assert f.h.device_status() == 0
    return f, arrs


def _check_all(f, arrs, wl, rows=None, sink=None, kl_full=True):
    cu = arrs["cu_seqlens"]
    T = wl.T_cap
    rows = np.arange(T) if rows is None else np.asarray(rows)
    if wl.ratio > 0:
        cu_cmp = ph.np32(f.cu_cmp).astype(np.int64)
        assert np.array_equal(cu_cmp, oracle.compressed_offsets(cu, wl.ratio))
        n_c = int(cu_cmp[-1])
        if wl.compressor == "v4":
            ph.check_compress_ex(f.kv_cmp, arrs["x_kv"], arrs["z_kv"], arrs["P_kv"], cu, wl.ratio, wl.overlap, n_c,
                                 x_prev=arrs.get("x_kv_prev"), z_prev=arrs.get("z_kv_prev"), gamma=arrs["g_kv"],
                                 eps=wl.norm_eps, rope_dim=wl.rope_kv, theta=wl.rope_theta)
        else:
            ph.check_compress(f.kv_cmp, arrs["x_kv"], arrs["z_kv"], arrs["P_kv"], cu, wl.ratio, wl.overlap, n_c)
        kv_cmp = ph.operand(f.kv_cmp[:n_c])
        v_cmp = None
        if wl.separate_v:
            ph.check_compress(f.v_cmp, arrs["v"], arrs["z_kv"], arrs["P_kv"], cu, wl.ratio, wl.overlap, n_c)
            v_cmp = ph.operand(f.v_cmp[:n_c])
    v_raw = arrs.get("v") if wl.separate_v else None
    if wl.ratio == 0:
        ph.check_attention(oracle.KIND_WINDOW, f.out, f.lse, None, arrs["q"], None, None, arrs["x_kv"], v_raw,
                           cu, 0, wl.window, f.scale, None, rows, sink=sink)
        return
    if wl.H_I > 0:
        if wl.compressor == "v4":
            ph.check_compress_ex(f.kI, arrs["x_I"], arrs["z_I"], arrs["P_I"], cu, wl.ratio, wl.overlap, n_c,
                                 x_prev=arrs.get("x_I_prev"), z_prev=arrs.get("z_I_prev"), gamma=arrs["g_I"],
                                 eps=wl.norm_eps, rope_dim=wl.rope_I, theta=wl.rope_theta)
        else:
            ph.check_compress(f.kI, arrs["x_I"], arrs["z_I"], arrs["P_I"], cu, wl.ratio, wl.overlap, n_c)
        kI = ph.operand(f.kI[:n_c])
        idx = f.idx.cpu().numpy()
        ph.check_topk(idx, arrs["qI"], arrs["w"], kI, cu, wl.ratio, wl.topk, rows)
        ph.check_attention(oracle.KIND_CSA, f.out, f.lse, f.lse_cmp, arrs["q"], kv_cmp, v_cmp, arrs["x_kv"],
                           v_raw, cu, wl.ratio, wl.window, f.scale, idx, rows, sink=sink)
        if wl.kl_mode != "none":
            kl_idx = idx if wl.kl_mode == "sparse" else None
            ph.check_kl(float(f.kl_sum.item()), ph.np32(f.kl_rows), arrs["q"], kv_cmp, arrs["qI"], arrs["w"], kI,
                        cu, wl.ratio, f.scale, kl_idx, rows, full=kl_full)
            if kl_full:
                starts = cu[np.searchsorted(cu, np.arange(wl.T), side="right") - 1]
                want = int((((np.arange(wl.T) - starts) + 1) // wl.ratio > 0).sum())
                assert int(f.n_valid.item()) == want
    else:
        ph.check_attention(oracle.KIND_HCA, f.out, f.lse, f.lse_cmp, arrs["q"], kv_cmp, v_cmp, arrs["x_kv"],
                           v_raw, cu, wl.ratio, wl.window, f.scale, None, rows, sink=sink)


def test_tiny_fp32_workload():
    """The tiny CSA workload: L=512, r=4, 4 heads x 64, indexer 2 x 32, k=16, W=64, fp32 I/O."""
    wl = I.WORKLOADS["tiny"]
    f, arrs = _run(wl)
    _check_all(f, arrs, wl)


RAGGED = [
    # several tiles + ragged tails, packed THD with an empty sequence and capacity rows
    I.custom("ragged_csa", lengths=[700, 0, 301, 1029, 5], ratio=4, overlap=True, H=64, d=128, window=128,
             H_I=8, d_I=64, topk=96, k_pad=128, kl_mode="sparse", cap_align=64),
    I.custom("ragged_dense_kl", lengths=[389, 1200], ratio=4, overlap=True, H=16, d=64, window=37, H_I=4,
             d_I=32, topk=40, k_pad=64, kl_mode="dense", cap_align=128),
    I.custom("hca_small", lengths=[2000, 700], ratio=128, overlap=False, H=64, d=128, window=128, cap_align=32),
    I.custom("window_small", lengths=[333, 129, 64], ratio=0, overlap=False, H=32, d=128, window=100),
    I.custom("csa_sepv_h8", lengths=[517], ratio=4, overlap=True, H=8, d=128, window=64, H_I=1, d_I=64,
             topk=200, k_pad=256, separate_v=True, kl_mode="sparse"),
    # a separate value stream at 64 heads x 128 (the tcgen05 kernel that stages K and V)
    I.custom("csa_sepv_h64", lengths=[517, 0, 130], ratio=4, overlap=True, H=64, d=128, window=128, H_I=8,
             d_I=64, topk=96, k_pad=128, separate_v=True, kl_mode="sparse", cap_align=64),
]


@pytest.mark.parametrize("wl", RAGGED, ids=[w.name for w in RAGGED])
def test_ragged_workloads(wl):
    f, arrs = _run(wl, seed=3)
    _check_all(f, arrs, wl)


def test_sink():
    wl = RAGGED[0]
    sink = np.random.default_rng(5).standard_normal(wl.H).astype(np.float32)
    f, arrs = _run(wl, seed=4, sink=sink)
    _check_all(f, arrs, wl, sink=sink)


def test_topk_covers_visible_is_dense_mode():
    # k >= |V_t|: every visible entry is selected (the dense-mode candidate list)
    wl = I.custom("dense_mode", lengths=[600], ratio=4, overlap=True, H=16, d=128, window=64, H_I=2, d_I=64,
                  topk=150, k_pad=152, kl_mode="sparse")
    f, arrs = _run(wl, seed=8)
    idx = f.idx.cpu().numpy()
    for t in range(600):
        n = (t + 1) // 4
        assert np.array_equal(idx[t, :n], np.arange(n)) and np.all(idx[t, n:] == -1)
    _check_all(f, arrs, wl)


def _sample_rows(wl, n=96, seed=0):
    rng = np.random.default_rng(seed)
    cu = wl.cu_seqlens
    rows = set(rng.choice(wl.T, n, replace=False).tolist())
    for b in range(wl.B):  # first/last queries of each sequence, and a capacity row
        rows.update([int(cu[b]), int(cu[b + 1]) - 1])
    if wl.T_cap > wl.T:
        rows.add(wl.T_cap - 1)
    return np.array(sorted(r for r in rows if 0 <= r < wl.T_cap))


@pytest.mark.parametrize("name", ["csa8k", "hca64k", "thd128k", "warmup32k"])
def test_full_size_workloads_sampled(name):
    wl = I.WORKLOADS[name]
    f, arrs = _run(wl, seed=0)
    rows = _sample_rows(wl)
    _check_all(f, arrs, wl, rows=rows, kl_full=False)


def test_csa8k_kl_sum_over_every_query_against_the_oracle():
    """Sparse mode at full size: the KL sum of all 8192 queries (the selected-set
    teacher over the GPU's own index lists) within 1e-3 relative of the oracle's,
    and every per-query value."""
    wl = I.WORKLOADS["csa8k"]
    f, arrs = _run(wl, seed=0)
    cu = arrs["cu_seqlens"]
    n_c = int(f.cu_cmp[-1].item())
    kv_cmp, kI = ph.operand(f.kv_cmp[:n_c]), ph.operand(f.kI[:n_c])
    idx = f.idx.cpu().numpy()
    ph.check_kl(float(f.kl_sum.item()), ph.np32(f.kl_rows), arrs["q"], kv_cmp, arrs["qI"], arrs["w"], kI, cu,
                wl.ratio, f.scale, idx, np.arange(wl.T_cap), full=True)
    assert int(f.n_valid.item()) == wl.T - (wl.ratio - 1)   # queries t >= r - 1 see an entry


def test_warmup32k_kl_sum_is_the_fixed_order_sum_of_its_rows():
    """The dense-teacher step at full size: the loss the finalising reduction
    returns equals the float64 sum of the per-query values it was given."""
    wl = I.WORKLOADS["warmup32k"]
    f, _ = _run(wl, seed=0)
    rows = ph.np32(f.kl_rows).astype(np.float64)
    want = rows.sum()
    rel = ph.record("kl_sum_vs_rows_rel", abs(float(f.kl_sum.item()) - want) / abs(want))
    assert rel <= 1e-6, (float(f.kl_sum.item()), want)


V4 = [
    # the DeepSeek-V4 style compressor (previous-half stream, RMSNorm, RoPE) feeding the whole step
    I.custom("v4_ragged_csa", lengths=[700, 0, 301, 1029, 5], ratio=4, overlap=True, H=64, d=128, window=128,
             H_I=8, d_I=64, topk=96, k_pad=128, kl_mode="sparse", cap_align=64, compressor="v4"),
    I.custom("v4_hca", lengths=[2000, 700], ratio=128, overlap=False, H=64, d=128, window=128, cap_align=32,
             compressor="v4"),
]


@pytest.mark.parametrize("wl", V4, ids=[w.name for w in V4])
def test_v4_compressor_workloads(wl):
    f, arrs = _run(wl, seed=6)
    _check_all(f, arrs, wl)


def test_v4_compressor_full_size_packed_sampled():
    wl = dataclasses.replace(I.WORKLOADS["thd128k"], compressor="v4")
    f, arrs = _run(wl, seed=0)
    _check_all(f, arrs, wl, rows=_sample_rows(wl), kl_full=False)


def test_host_side_argument_errors():
    h = api.Handle(0)
    cu = torch.tensor([0, 64], dtype=torch.int32, device="cuda")
    cu_cmp = torch.zeros(2, dtype=torch.int32, device="cuda")
    x = torch.zeros(64, 96, dtype=torch.bfloat16, device="cuda")
    P = torch.zeros(8, 96, dtype=torch.float32, device="cuda")
    out = torch.zeros(16, 96, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(api.CSAError) as e:   # D = 96 has no kernel
        api.csa_compress(h, x, x, P, cu, cu_cmp, 64, 4, True, out)
    assert e.value.code == -2
    q = torch.zeros(64, 64, 96, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(api.CSAError) as e:   # head dim 96 unsupported
        api.window_attn_fwd(h, q, x, cu, 64, 16, 0.1, torch.empty_like(q), torch.empty(64, 64, device="cuda"))
    assert e.value.code == -2
    q = torch.zeros(64, 64, 128, dtype=torch.bfloat16, device="cuda")
    kv = torch.zeros(64 * 128 + 1, dtype=torch.bfloat16, device="cuda")[1:].view(64, 128)  # 2-byte offset
    with pytest.raises(api.CSAError) as e:
        api.window_attn_fwd(h, q, kv, cu, 64, 16, 0.1, torch.empty_like(q), torch.empty(64, 64, device="cuda"))
    assert e.value.code == -1
    idx = torch.zeros(64, 4, dtype=torch.int32, device="cuda")
    qI = torch.zeros(64, 8, 64, dtype=torch.bfloat16, device="cuda")
    w = torch.zeros(64, 8, dtype=torch.bfloat16, device="cuda")
    kI = torch.zeros(16, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(api.CSAError) as e:   # k_pad < topk
        api.csa_indexer_topk(h, qI, w, kI, cu, cu_cmp, 64, 4, 8, idx)
    assert e.value.code == -1
    kl = torch.zeros(1, device="cuda")
    with pytest.raises(api.CSAError) as e:   # workspace too small
        kv_c = torch.zeros(16, 128, dtype=torch.bfloat16, device="cuda")
        api.csa_indexer_kl(h, q, kv_c, qI, w, kI, cu, cu_cmp, 64, 4, 0.1, kl,
                           torch.empty(16, dtype=torch.uint8, device="cuda"))
    assert e.value.code == -3
    assert h.device_status() == 0


def test_device_bounds_error_is_reported_not_faulted():
    # an index the query cannot see yet: the kernel skips it and raises the status word
    wl = I.custom("bounds", lengths=[256], ratio=4, overlap=True, H=16, d=128, window=32, H_I=2, d_I=64,
                  topk=8, k_pad=8)
    f, arrs = _run(wl, seed=1)
    bad = f.idx.clone()
    bad[10, 0] = 60                          # query t=10 sees entries 0..1 only
    api.csa_sparse_attn_fwd(f.h, f.x["q"], f.kv_cmp, f.x["x_kv"], bad, f.cu, f.cu_cmp, 256, 4, 32, f.scale,
                            f.out, f.lse, f.lse_cmp)
    assert f.h.device_status() == -6
    assert f.h.device_status() == 0          # reading resets the word
    assert torch.isfinite(f.lse[10]).all()


def test_packed_equals_separate_sequences():
    wl = I.custom("pack", lengths=[300, 517], ratio=4, overlap=True, H=16, d=128, window=64, H_I=4, d_I=64,
                  topk=32, k_pad=32, kl_mode="sparse")
    f, arrs = _run(wl, seed=11)
    for b, L in enumerate(wl.lengths):
        s = slice(int(wl.cu_seqlens[b]), int(wl.cu_seqlens[b + 1]))
        one = I.custom("one", lengths=[L], ratio=4, overlap=True, H=16, d=128, window=64, H_I=4, d_I=64, topk=32,
                       k_pad=32, kl_mode="sparse")
        sub = {k: (v[s] if k not in ("cu_seqlens", "P_kv", "P_I") else v) for k, v in arrs.items()}
        sub["cu_seqlens"] = one.cu_seqlens
        g = Forward(one, to_device(sub, False))
        g.run()
        torch.cuda.synchronize()
        assert torch.equal(g.out, f.out[s])
        assert torch.equal(g.lse, f.lse[s])
        cmp0 = int(f.cu_cmp[b].item())
        gi = g.idx.clone()
        gi[gi >= 0] += cmp0
        assert torch.equal(gi, f.idx[s])


def test_run_from_host_matches_device_run():
    """Inputs copied from pinned host memory stage by stage give the same outputs
    as a forward on inputs already on the device; a second call reuses the buffers."""
    wl = I.custom("host", lengths=[700, 1300], ratio=4, overlap=True, H=64, d=128, window=128, H_I=8, d_I=64,
                  topk=64, k_pad=64, kl_mode="dense")
    arrs = I.generate(wl, 5)
    ref = Forward(wl, to_device(arrs, False))
    ref.run()
    zeros = {k: torch.zeros_like(v) for k, v in to_device(arrs, False).items()}
    g = Forward(wl, zeros)
    host = {k: v.cpu().pin_memory() for k, v in to_device(arrs, False).items()}
    for _ in range(2):
        g.run_from_host(host)
        torch.cuda.synchronize()
        assert g.h.device_status() == 0
        assert torch.equal(g.out, ref.out)
        assert torch.equal(g.lse, ref.lse)
        assert torch.equal(g.idx, ref.idx)
        assert torch.equal(g.kl_sum, ref.kl_sum)
