"""The dense-teacher indexer KL on the tensor cores when a row's scores climb far
above those of its first key tile, against the oracle.

"DeepSeek-V4 Attention Training Systems": §3 (L_I = sum_t KL(Softmax(a_{t,C_t})
|| Softmax(i_{t,C_t})), C_t every visible compressed entry in the dense phase),
§9 (FP32 loss math).  The kernel's first pass keeps each (query, head) row's
normaliser against a reference that it fixes on the row's first tile and moves
only for a tile whose terms reach 2^64 against it; the planted keys below make
many rows do that on a later tile.
"""
import numpy as np
import pytest
import torch

from compressed_sparse_attention_compress_gb300 import inputs as I
from tests import parity_helpers as ph

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # the CPU suite never collects GPU work
    pytest.skip("no CUDA device", allow_module_level=True)

from compressed_sparse_attention_compress_gb300 import api  # noqa: E402
from compressed_sparse_attention_compress_gb300.forward import Forward, to_device  # noqa: E402

WL = I.custom("kl_dense_climb", lengths=[1500, 3, 0, 777], ratio=4, overlap=True, H=64, d=128, window=128,
              H_I=8, d_I=64, topk=64, k_pad=64, kl_mode="dense", cap_align=64)
# compressed entries of sequence 0 past its first 128-entry tile (it has 375), scaled by 256
# (exact in bf16): their scores reach about a hundred natural units, far above the first tile's
PLANTED = (131, 200, 290, 374)


def test_dense_kl_with_scores_far_above_the_first_tile():
    arrs = I.generate(WL, 4)
    f = Forward(WL, to_device(arrs, False))
    f.run()
    torch.cuda.synchronize()
    assert f.h.device_status() == 0
    for e in PLANTED:
        f.kv_cmp[e] *= 256
    T_cap = WL.T_cap
    kl_sum = torch.zeros(1, device="cuda")
    rows = torch.full((T_cap,), 7.0, device="cuda")
    n_valid = torch.zeros(1, dtype=torch.int32, device="cuda")
    tl = torch.full((T_cap, WL.H), 7.0, device="cuda")
    sl = torch.full((T_cap,), 7.0, device="cuda")
    api.csa_indexer_kl_ex(f.h, f.x["q"], f.kv_cmp, f.x["qI"], f.x["w"], f.kI, f.cu, f.cu_cmp, f.max_seqlen,
                          WL.ratio, f.scale, kl_sum, f.ws, teacher_lse=tl, student_lse=sl, kl_per_query=rows,
                          n_valid=n_valid)
    torch.cuda.synchronize()
    assert f.h.device_status() == 0
    cu = arrs["cu_seqlens"]
    n_c = int(f.cu_cmp[-1].item())
    kv_cmp, kI = ph.operand(f.kv_cmp[:n_c]), ph.operand(f.kI[:n_c])
    ph.check_kl(float(kl_sum.item()), ph.np32(rows), arrs["q"], kv_cmp, arrs["qI"], arrs["w"], kI, cu, WL.ratio,
                f.scale, None, np.arange(T_cap), full=True)
    # every head's normaliser against a float64 sum over the visible prefix; the rows checked
    # see the planted entries, and the test asserts that some (row, head) pairs gain more than
    # 64 in log2 units over the first tile there
    q = arrs["q"].astype(np.float64)
    tl_np = ph.np32(tl)
    climbs = 0
    for row in (527, 800, 1163, 1499):
        n = (row + 1) // WL.ratio
        s = f.scale * q[row] @ kv_cmp[:n].astype(np.float64).T
        ref = np.log(np.exp(s - s.max(1, keepdims=True)).sum(1)) + s.max(1)
        assert np.abs(tl_np[row] - ref).max() < 1e-3
        climbs += int(((s.max(1) - s[:, :128].max(1)) * np.log2(np.e) > 64).sum())
    assert climbs >= 16
