"""Single-process emulation of contiguous context parallelism on the GPU.

"DeepSeek-V4 Attention Training Systems" §5 (contiguous CP: boundary rows from
the left neighbour, compressed rows all-gathered), §12 invariant 4 (selected
ids must map to the right physical rows).  P virtual ranks run one after
another through the C ABI: each compresses its own rows plus the boundary and
keeps the entries it owns, the owned entries are gathered by local copies, and
each rank's top-k, attention and KL run on its local rows with the handle's
position offsets.  Every owned query must reproduce the one-GPU forward bit
for bit: the per-query arithmetic is the same, only the rows around it moved.
The emulated ranks' results are also compared with the oracle on every row
(gathered compressed rows, index sets, outputs and LSEs, per-query KL and its
sum), within the same tolerances as the one-GPU parity tests.
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

from compressed_sparse_attention_compress_gb300 import cp  # noqa: E402
from compressed_sparse_attention_compress_gb300.forward import Forward, to_device  # noqa: E402

CASES = [
    (I.custom("cp_dense", lengths=[3000, 0, 1500, 37], ratio=4, overlap=True, H=64, d=128, window=128, H_I=8, d_I=64,
              topk=256, k_pad=256, kl_mode="dense"), 3),
    (I.custom("cp_sparse", lengths=[4096], ratio=4, overlap=True, H=64, d=128, window=128, H_I=8, d_I=64,
              topk=128, k_pad=128, kl_mode="sparse"), 4),
    (I.custom("cp_small_heads", lengths=[700, 901], ratio=4, overlap=True, H=16, d=64, window=64, H_I=4, d_I=32,
              topk=40, k_pad=64, kl_mode="sparse"), 2),
]


@pytest.mark.parametrize("wl,P", CASES, ids=[c[0].name for c in CASES])
def test_cp_ranks_reproduce_the_single_gpu_forward(wl, P):
    arrs = I.generate(wl, 11)
    dev = to_device(arrs, wl.io_fp32)
    f = Forward(wl, dev)
    f.run()
    torch.cuda.synchronize()
    assert f.h.device_status() == 0
    res = cp.emulate(wl, dev, P)
    assert res["status"] == 0
    T = wl.T
    assert np.array_equal(res["rows"], np.arange(T))
    n_c = wl.n_cmp
    assert torch.equal(res["kv_cmp"], f.kv_cmp[:n_c])
    assert torch.equal(res["kI"], f.kI[:n_c])
    assert torch.equal(res["idx"], f.idx[:T])
    assert torch.equal(res["out"], f.out[:T])
    assert torch.equal(res["lse"], f.lse[:T])
    assert torch.equal(res["lse_cmp"], f.lse_cmp[:T])
    if wl.kl_mode != "none":
        assert torch.equal(res["kl_rows"], f.kl_rows[:T])


@pytest.mark.parametrize("wl,P", CASES, ids=[c[0].name for c in CASES])
def test_cp_ranks_match_the_oracle(wl, P):
    arrs = I.generate(wl, 11)
    dev = to_device(arrs, wl.io_fp32)
    res = cp.emulate(wl, dev, P)
    assert res["status"] == 0
    cu = arrs["cu_seqlens"]
    T, n_c = wl.T, wl.n_cmp
    rows = np.arange(T)
    # gathered compressed rows (each rank compressed its own rows plus the boundary)
    ph.check_compress(res["kv_cmp"], arrs["x_kv"], arrs["z_kv"], arrs["P_kv"], cu, wl.ratio, wl.overlap, n_c)
    ph.check_compress(res["kI"], arrs["x_I"], arrs["z_I"], arrs["P_I"], cu, wl.ratio, wl.overlap, n_c)
    kv_cmp, kI = ph.operand(res["kv_cmp"]), ph.operand(res["kI"])
    idx = res["idx"].cpu().numpy()
    ph.check_topk(idx, arrs["qI"], arrs["w"], kI, cu, wl.ratio, wl.topk, rows)
    scale = 1.0 / float(np.sqrt(wl.d))
    ph.check_attention(oracle.KIND_CSA, res["out"], res["lse"], res["lse_cmp"], arrs["q"], kv_cmp, None,
                       arrs["x_kv"], None, cu, wl.ratio, wl.window, scale, idx, rows)
    kl_rows = ph.np32(res["kl_rows"])
    kl_idx = idx if wl.kl_mode == "sparse" else None
    ph.check_kl(float(kl_rows.astype(np.float64).sum()), kl_rows, arrs["q"], kv_cmp, arrs["qI"], arrs["w"], kI,
                cu, wl.ratio, scale, kl_idx, rows, full=True)
