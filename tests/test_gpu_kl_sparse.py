"""The selected-set (sparse-mode) indexer KL on the tensor cores, against the oracle.

"DeepSeek-V4 Attention Training Systems" §3 (KL of the indexer against the
head-averaged teacher over C_t), §2 phase table (sparse mode: C_t is the
selected set).  At 64 heads x 128 with an 8 x 64 indexer in bf16 and a
reference normaliser (the attention's lse_cmp), csa_indexer_kl runs the
tcgen05 two-pass kernel.  These cases give it index rows with holes (-1 in
the middle), rows whose selected set is empty, sequences shorter than one
block and several tiles per query, and compare every row with the oracle; the
same call without the reference (the warp-level kernel) must agree with it,
and a reference far below the true normaliser must raise the bounds status.
A selected set of up to four tiles keeps its scores in tensor memory between
the passes; a longer one is gathered and multiplied again: both are covered.
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
from compressed_sparse_attention_compress_gb300.forward import Forward, to_device  # noqa: E402

WL = I.custom("kl_sparse", lengths=[1500, 3, 0, 777], ratio=4, overlap=True, H=64, d=128, window=128, H_I=8,
              d_I=64, topk=300, k_pad=384, kl_mode="sparse", cap_align=64)
# more than four tiles per query: the scores are gathered and multiplied again in pass 2
WL_LONG = I.custom("kl_sparse_long", lengths=[3100, 3, 0, 777], ratio=4, overlap=True, H=64, d=128, window=128,
                   H_I=8, d_I=64, topk=600, k_pad=640, kl_mode="sparse", cap_align=64)


def _setup(seed=2, wl=WL):
    arrs = I.generate(wl, seed)
    f = Forward(wl, to_device(arrs, False))
    f.run()
    torch.cuda.synchronize()
    assert f.h.device_status() == 0
    return f, arrs


def _holes(f):
    """The index rows with every third selected entry dropped (holes inside the
    rows), and the rows of a few queries emptied."""
    idx = f.idx.clone()
    idx[:, 1::3] = -1
    idx[[5, 600, 1501], :] = -1
    return idx


def _kl(f, idx, lse_cmp, T_cap):
    kl_sum = torch.zeros(1, device="cuda")
    rows = torch.full((T_cap,), 7.0, device="cuda")
    n_valid = torch.zeros(1, dtype=torch.int32, device="cuda")
    tl = torch.full((T_cap, f.wl.H), 7.0, device="cuda")
    sl = torch.full((T_cap,), 7.0, device="cuda")
    api.csa_indexer_kl_ex(f.h, f.x["q"], f.kv_cmp, f.x["qI"], f.x["w"], f.kI, f.cu, f.cu_cmp, f.max_seqlen,
                          f.wl.ratio, f.scale, kl_sum, f.ws, teacher_lse=tl, student_lse=sl, idx=idx,
                          lse_cmp=lse_cmp, kl_per_query=rows, n_valid=n_valid)
    torch.cuda.synchronize()
    return kl_sum, rows, n_valid, tl, sl


@pytest.mark.parametrize("wl", [WL, WL_LONG], ids=["keep", "long"])
@pytest.mark.parametrize("with_reference", [True, False])
def test_selected_set_kl_with_holes_and_empty_rows(with_reference, wl):
    f, arrs = _setup(wl=wl)
    idx = _holes(f)
    kl_sum, rows, n_valid, tl, sl = _kl(f, idx, f.lse_cmp if with_reference else None, wl.T_cap)
    assert f.h.device_status() == 0
    cu = arrs["cu_seqlens"]
    n_c = int(f.cu_cmp[-1].item())
    kv_cmp, kI = ph.operand(f.kv_cmp[:n_c]), ph.operand(f.kI[:n_c])
    idx_np = idx.cpu().numpy()
    every = np.arange(wl.T_cap)
    ph.check_kl(float(kl_sum.item()), ph.np32(rows), arrs["q"], kv_cmp, arrs["qI"], arrs["w"], kI, cu, wl.ratio,
                f.scale, idx_np, every, full=True)
    sizes = (idx_np >= 0).sum(1)
    assert int(n_valid.item()) == int((sizes > 0).sum())
    # the exact per-head teacher normaliser and the student's, against float64 sums
    q = arrs["q"].astype(np.float64)
    qI, w = arrs["qI"].astype(np.float64), arrs["w"].astype(np.float64)
    tl_np, sl_np = ph.np32(tl), ph.np32(sl)
    for row in [0, 4, 5, 700, 1499, 1500, 1502, 2000, wl.T - 1, wl.T_cap - 1]:
        sel = idx_np[row][idx_np[row] >= 0]
        if sel.size == 0:
            assert np.all(np.isneginf(tl_np[row])) and np.isneginf(sl_np[row]) and ph.np32(rows)[row] == 0
            continue
        K = kv_cmp[sel].astype(np.float64)
        s = f.scale * q[row] @ K.T
        ref_t = np.log(np.exp(s - s.max(1, keepdims=True)).sum(1)) + s.max(1)
        assert np.abs(tl_np[row] - ref_t).max() < 1e-3
        logit = (w[row][:, None] * np.maximum(qI[row] @ kI[sel].astype(np.float64).T, 0)).sum(0)
        ref_s = np.log(np.exp(logit - logit.max()).sum()) + logit.max()
        assert abs(sl_np[row] - ref_s) < 1e-3


def test_tensor_core_and_warp_level_kernels_agree():
    f, _ = _setup(seed=4)
    a_sum, a_rows, _, a_tl, _ = _kl(f, f.idx, f.lse_cmp, WL.T_cap)
    b_sum, b_rows, _, b_tl, _ = _kl(f, f.idx, None, WL.T_cap)
    assert f.h.device_status() == 0
    assert abs(a_sum.item() - b_sum.item()) <= 1e-4 * abs(b_sum.item())
    assert torch.allclose(a_rows, b_rows, atol=1e-4, rtol=1e-4)
    fin = torch.isfinite(b_tl)
    assert torch.equal(fin, torch.isfinite(a_tl))
    assert torch.allclose(a_tl[fin], b_tl[fin], atol=1e-4)


def test_reference_far_below_the_normaliser_is_reported():
    f, _ = _setup(seed=5)
    _kl(f, f.idx, f.lse_cmp - 100.0, WL.T_cap)
    assert f.h.device_status() == -6
    assert f.h.device_status() == 0
