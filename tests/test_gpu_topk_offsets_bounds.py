"""Top-k with position offsets and a max_seqlen that does not bound the positions.

With csa_set_position_offsets, query t of a sequence sees (t + p0 + 1) / r
entries ("DeepSeek-V4 Attention Training Systems" §4 visibility, §5 contiguous
CP offsets), and max_seqlen must bound t + p0 (it sizes the on-chip score
rows).  A call that breaks this contract must raise CSA_ERR_DEVICE_BOUNDS on
the handle's status word and keep every access inside the score rows, on both
the warp-level kernel (other indexer shapes) and the tcgen05 kernel
(indexer 8 x 64, bf16).
"""
import pytest
import torch

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # the CPU suite never collects GPU work
    pytest.skip("no CUDA device", allow_module_level=True)

from compressed_sparse_attention_compress_gb300 import api  # noqa: E402


@pytest.mark.parametrize("H_I,d_I", [(4, 32), (2, 64), (8, 64)])
def test_offsets_beyond_max_seqlen_raise_bounds(H_I, d_I):
    h = api.Handle(0)
    L, p0, r, k = 300, 200, 4, 16
    g = torch.Generator().manual_seed(3)
    n_cmp = (L + p0) // r
    cu = torch.tensor([0, L], dtype=torch.int32, device="cuda")
    cu_cmp = torch.zeros(2, dtype=torch.int32, device="cuda")
    qI = torch.randn(L, H_I, d_I, generator=g).to("cuda", torch.bfloat16)
    w = torch.randn(L, H_I, generator=g).to("cuda", torch.bfloat16)
    kI = torch.randn(n_cmp, d_I, generator=g).to("cuda", torch.bfloat16)
    idx = torch.empty(L, k, dtype=torch.int32, device="cuda")
    pos = torch.tensor([p0], dtype=torch.int32, device="cuda")
    h.set_position_offsets(pos, n_cmp)
    try:
        # max_seqlen = L bounds t but not t + p0: the last queries see 125 > 75 entries
        api.csa_indexer_topk(h, qI, w, kI, cu, cu_cmp, L, r, k, idx)
        assert h.device_status() == -6
        # a bound on the positions: the same call is clean, and every row holds k ascending visible entries
        api.csa_indexer_topk(h, qI, w, kI, cu, cu_cmp, L + p0, r, k, idx)
        assert h.device_status() == 0
    finally:
        h.set_position_offsets(None)
    rows = idx.cpu()
    for t in range(L):
        n = (t + p0 + 1) // r
        sel = rows[t][rows[t] >= 0]
        assert sel.numel() == min(k, n)
        assert torch.all(sel < n) and torch.all(sel[1:] > sel[:-1])
