"""Top-k with exact ties in the indexer scores (needs a GPU).

"DeepSeek-V4 Attention Training Systems" §8 / §8.2 (radix top-k with a fixed
capacity).  The selection takes the min(k, |V_t|) largest logits with ties
going to the smaller entry index, in ascending order.  Random operands almost
never tie, so these cases build them: all-zero query operands (every logit
0: the first k entries), and compressed keys drawn from a handful of distinct
rows (many equal logits around the threshold).  Both are compared with the
oracle's (-logit, index) order bit for bit, on every query, over several tiles.
"""
import numpy as np
import pytest
import torch

import oracle
from compressed_sparse_attention_compress_gb300 import inputs as I

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # the CPU suite never collects GPU work
    pytest.skip("no CUDA device", allow_module_level=True)

from compressed_sparse_attention_compress_gb300 import api  # noqa: E402


def _run(qI, w, kI, lengths, ratio, topk, k_pad):
    cu_np = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    h = api.Handle(0)
    cu = torch.from_numpy(cu_np).cuda()
    cu_cmp = torch.from_numpy(oracle.compressed_offsets(cu_np, ratio).astype(np.int32)).cuda()
    T = int(cu_np[-1])
    idx = torch.full((T, k_pad), 7, dtype=torch.int32, device="cuda")
    api.csa_indexer_topk(h, torch.from_numpy(qI).cuda().bfloat16(), torch.from_numpy(w).cuda().bfloat16(),
                         torch.from_numpy(kI).cuda().bfloat16(), cu, cu_cmp, max(lengths), ratio, topk, idx)
    torch.cuda.synchronize()
    assert h.device_status() == 0
    ref = oracle.indexer_topk(qI, w, kI, cu_np, ratio, topk, k_pad, np.arange(T))
    return idx.cpu().numpy(), ref


@pytest.mark.parametrize("H_I,d_I", [(8, 64), (4, 32)])
def test_all_logits_equal_take_the_first_entries(H_I, d_I):
    lengths, r, k = [3000, 517], 4, 200
    rng = np.random.default_rng(1)
    T = sum(lengths)
    qI = np.zeros((T, H_I, d_I), np.float32)
    w = I.bf16_round(rng.standard_normal((T, H_I)).astype(np.float32))
    kI = I.bf16_round(rng.standard_normal((T // r, d_I)).astype(np.float32))
    got, ref = _run(qI, w, kI, lengths, r, k, 256)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("distinct", [2, 5])
def test_keys_from_a_few_distinct_rows(distinct):
    lengths, r, k = [6000, 1100], 4, 300
    rng = np.random.default_rng(2)
    T = sum(lengths)
    qI = I.bf16_round(rng.standard_normal((T, 8, 64)).astype(np.float32))
    w = I.bf16_round(rng.standard_normal((T, 8)).astype(np.float32))
    rows = I.bf16_round(rng.standard_normal((distinct, 64)).astype(np.float32))
    kI = rows[rng.integers(0, distinct, T // r)]
    got, ref = _run(qI, w, kI, lengths, r, k, 320)
    assert np.array_equal(got, ref)
