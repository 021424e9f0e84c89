"""Both backward calls on row ranges with per-sequence position offsets.

"DeepSeek-V4 Attention Training Systems" §5 (contiguous context parallelism:
each rank holds a contiguous range of every sequence's queries, W raw rows of
boundary from its left neighbour, the compressed rows all-gathered) and §8.2
(the attention and indexer backward).  The queries of one sequence are cut at
row a; the range [a, T) runs as its own packing whose first row sits at
position a - W (attention: the boundary rows with a zero upstream gradient,
so they add nothing) or a (indexer: no raw rows needed), set with
csa_set_position_offsets.  Per-query gradients (dq, dqI, dw) must be bit for
bit those of the whole call; the key-side gradients (float32 sums over
queries, added in a different order) must sum to the whole call's within a
rounding bound.
"""
import numpy as np
import pytest
import torch

from compressed_sparse_attention_compress_gb300 import inputs as I

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # the CPU suite never collects GPU work
    pytest.skip("no CUDA device", allow_module_level=True)

from compressed_sparse_attention_compress_gb300 import api  # noqa: E402
from compressed_sparse_attention_compress_gb300.forward import Forward, to_device  # noqa: E402


def _sums_close(name, got, ref):
    got, ref = got.double(), ref.double()
    bound = 2e-5 * ref.abs().max() + 1e-4 * ref.abs()
    bad = (got - ref).abs() > bound
    assert not bool(bad.any()), f"{name}: {int(bad.sum())} of {ref.numel()} outside, worst {(got - ref).abs().max()}"


@pytest.mark.parametrize("L,a", [(4096, 1536), (6000, 4000)])
def test_backward_on_offset_ranges(L, a):
    wl = I.custom("bwd_offsets", lengths=[L], ratio=4, overlap=True, H=64, d=128, window=128, H_I=8, d_I=64,
                  topk=256, k_pad=256, kl_mode="dense")
    W, r, T = wl.window, wl.ratio, wl.T
    dev = to_device(I.generate(wl, 9), wl.io_fp32)
    f = Forward(wl, dev)
    f.keep_stats = True
    f.run()
    g = torch.Generator(device="cpu").manual_seed(4)
    dout = (torch.randn(f.out.shape, generator=g) * 0.5).to(f.out.dtype).cuda()
    f.backward(dout)
    f.indexer_backward(grad_scale=1.0)
    torch.cuda.synchronize()
    assert f.h.device_status() == 0
    h = f.h
    n_cap = f.kv_cmp.shape[0]
    x = f.x

    # ---- attention backward: [0, a) plain, [a - W, T) at position a - W ----
    dq = torch.empty_like(f.out)
    dkv_cmp = torch.zeros(n_cap, wl.d, dtype=torch.float32, device="cuda")
    dkv_raw = torch.zeros(T, wl.d, dtype=torch.float32, device="cuda")
    for lo, own, hi in ((0, 0, a), (a - W, a, T)):
        n = hi - lo
        cu_l = torch.tensor([0, n], dtype=torch.int32, device="cuda")
        d_l = dout[lo:hi].clone()
        d_l[:own - lo] = 0            # boundary queries: no upstream gradient
        dq_l = torch.empty(n, wl.H, wl.d, dtype=f.out.dtype, device="cuda")
        dc_l = torch.empty(n_cap, wl.d, dtype=torch.float32, device="cuda")
        dr_l = torch.empty(n, wl.d, dtype=torch.float32, device="cuda")
        delta = torch.empty(n, wl.H, dtype=torch.float32, device="cuda")
        h.set_position_offsets(torch.tensor([lo], dtype=torch.int32, device="cuda"), n_cap)
        try:
            api.csa_sparse_attn_bwd(h, x["q"][lo:hi], f.kv_cmp, x["x_kv"][lo:hi], f.idx[lo:hi], cu_l, f.cu_cmp, L,
                                    r, W, f.scale, f.out[lo:hi], f.lse[lo:hi], d_l, dq_l, dc_l, dr_l, delta)
        finally:
            h.set_position_offsets(None)
        torch.cuda.synchronize()
        assert h.device_status() == 0
        dq[own:hi] = dq_l[own - lo:]
        dkv_cmp += dc_l
        dkv_raw[lo:hi] += dr_l
    assert torch.equal(dq[:T].view(torch.int16), f.dq[:T].view(torch.int16))
    _sums_close("dkv_cmp", dkv_cmp, f.dkv_cmp)
    _sums_close("dkv_raw", dkv_raw, f.dkv_raw[:T])

    # ---- indexer backward (one pass with the forward's normalisers): [0, a), [a, T) at position a ----
    dqI = torch.empty_like(x["qI"])
    dw = torch.empty_like(x["w"])
    dkI = torch.zeros(n_cap, wl.d_I, dtype=torch.float32, device="cuda")
    for lo, hi in ((0, a), (a, T)):
        n = hi - lo
        cu_l = torch.tensor([0, n], dtype=torch.int32, device="cuda")
        dqI_l = torch.empty(n, wl.H_I, wl.d_I, dtype=x["qI"].dtype, device="cuda")
        dw_l = torch.empty(n, wl.H_I, dtype=x["w"].dtype, device="cuda")
        dkI_l = torch.empty(n_cap, wl.d_I, dtype=torch.float32, device="cuda")
        h.set_position_offsets(torch.tensor([lo], dtype=torch.int32, device="cuda"), n_cap)
        try:
            api.csa_indexer_kl_bwd(h, x["q"][lo:hi], f.kv_cmp, x["qI"][lo:hi], x["w"][lo:hi], f.kI, cu_l, f.cu_cmp,
                                   L, r, f.scale, dqI_l, dw_l, dkI_l, lse_cmp=f.teacher_lse[lo:hi],
                                   student_lse=f.student_lse[lo:hi], grad_scale=1.0)
        finally:
            h.set_position_offsets(None)
        torch.cuda.synchronize()
        assert h.device_status() == 0
        dqI[lo:hi] = dqI_l
        dw[lo:hi] = dw_l
        dkI += dkI_l
    assert torch.equal(dqI[:T].view(torch.int16), f.dqI[:T].view(torch.int16))
    assert torch.equal(dw[:T].view(torch.int16), f.dw[:T].view(torch.int16))
    _sums_close("dkI", dkI, f.dkI)
    assert np.isfinite(dkI.cpu().numpy()).all()
