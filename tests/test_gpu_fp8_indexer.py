"""GPU parity of the FP8 indexer: E4M3 quantisation (csa_quantize_fp8) and the
tensor-core scoring + top-k on codes (csa_indexer_topk_fp8).

"DeepSeek-V4 Attention Training Systems" §1 and §9 name an FP8 indexer for the
index-search term.  The codes and scales are compared bit for bit with the
oracle's quantisation of the same synthetic inputs; the selected index sets
with the oracle's top-k over the oracle's dequantised operands (exact in
float32 since the scales are powers of two), bit-exact except entries within
1e-4 relative of the k-th score (near-ties), as for the bf16 indexer.
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


def _quant_gpu(h, x):
    codes = torch.empty(x.shape, dtype=torch.uint8, device="cuda")
    scales = torch.empty(x.shape[:-1], dtype=torch.float32, device="cuda")
    api.csa_quantize_fp8(h, x, codes, scales)
    return codes, scales


@pytest.mark.parametrize("fp32", [False, True])
def test_quantisation_is_bit_exact(fp32):
    h = api.Handle(0)
    rng = np.random.default_rng(2)
    x = (rng.standard_normal((3000, 64)) * np.exp(2 * rng.standard_normal((3000, 1)))).astype(np.float32)
    x[7] = 0.0
    x[9, :] = 1e-30
    x = I.bf16_round(x) if not fp32 else x
    t = torch.from_numpy(x).cuda()
    t = t if fp32 else t.to(torch.bfloat16)
    codes, scales = _quant_gpu(h, t)
    torch.cuda.synchronize()
    ref_c, ref_s = oracle.quantize_fp8(x)
    np.testing.assert_array_equal(codes.cpu().numpy(), ref_c)
    np.testing.assert_array_equal(scales.cpu().numpy(), ref_s)


def _run(wl, seed=0, rows=None):
    arrs = I.generate(wl, seed)
    h = api.Handle(0)
    cu_np = wl.cu_seqlens
    cu = torch.from_numpy(cu_np).cuda()
    cmp_np = oracle.compressed_offsets(cu_np, wl.ratio)
    cu_cmp = torch.from_numpy(cmp_np).cuda()
    n_cap = max(1, wl.T_cap // wl.ratio)
    # compressed indexer keys: synthetic bf16 rows (the compressor is tested elsewhere)
    kI_np = I.bf16_round(np.random.default_rng(seed + 100).standard_normal((n_cap, wl.d_I)).astype(np.float32))
    qI = torch.from_numpy(arrs["qI"]).cuda().to(torch.bfloat16)
    w = torch.from_numpy(arrs["w"]).cuda().to(torch.bfloat16)
    kI = torch.from_numpy(kI_np).cuda().to(torch.bfloat16)
    qc, qs = _quant_gpu(h, qI)
    kc, ks = _quant_gpu(h, kI)
    idx = torch.full((wl.T_cap, wl.k_pad), 7, dtype=torch.int32, device="cuda")
    api.csa_indexer_topk_fp8(h, qc, qs, w, kc, ks, cu, cu_cmp, max(wl.lengths), wl.ratio, wl.topk, idx)
    torch.cuda.synchronize()
    assert h.device_status() == 0
    # the oracle quantises the same inputs itself and scores the dequantised values
    rq_c, rq_s = oracle.quantize_fp8(arrs["qI"])
    rk_c, rk_s = oracle.quantize_fp8(kI_np)
    np.testing.assert_array_equal(qc.cpu().numpy(), rq_c)
    np.testing.assert_array_equal(kc.cpu().numpy(), rk_c)
    qI_deq = oracle.dequantize_fp8(rq_c, rq_s)
    kI_deq = oracle.dequantize_fp8(rk_c, rk_s)
    rows = np.arange(wl.T_cap) if rows is None else rows
    ph.check_topk(idx.cpu().numpy(), qI_deq, arrs["w"], kI_deq, cu_np, wl.ratio, wl.topk, rows)
    return idx


RAGGED = [
    I.custom("fp8_ragged", lengths=[700, 0, 301, 1029, 5], ratio=4, overlap=True, H=64, d=128, window=128,
             H_I=8, d_I=64, topk=96, k_pad=128, kl_mode="none", cap_align=64),
    I.custom("fp8_dense_mode", lengths=[600], ratio=4, overlap=True, H=16, d=128, window=64, H_I=8, d_I=64,
             topk=150, k_pad=152, kl_mode="none"),
]


@pytest.mark.parametrize("wl", RAGGED, ids=[w.name for w in RAGGED])
def test_fp8_topk_matches_oracle_every_query(wl):
    _run(wl, seed=3)


def test_fp8_topk_warmup_layer_sampled():
    wl = I.WORKLOADS["warmup32k"]
    rng = np.random.default_rng(0)
    rows = np.sort(np.concatenate([rng.choice(wl.T, 64, replace=False), [0, 8190, 8191, wl.T - 1]]))
    _run(wl, seed=0, rows=rows)


def test_argument_errors():
    h = api.Handle(0)
    T = 64
    cu = torch.tensor([0, T], dtype=torch.int32, device="cuda")
    cu_cmp = torch.tensor([0, T // 4], dtype=torch.int32, device="cuda")
    qc = torch.zeros(T, 4, 64, dtype=torch.uint8, device="cuda")       # H_I = 4: no FP8 kernel
    qs = torch.ones(T, 4, device="cuda")
    w = torch.zeros(T, 4, dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros(16, 64, dtype=torch.uint8, device="cuda")
    ks = torch.ones(16, device="cuda")
    idx = torch.zeros(T, 8, dtype=torch.int32, device="cuda")
    with pytest.raises(api.CSAError) as e:
        api.csa_indexer_topk_fp8(h, qc, qs, w, kc, ks, cu, cu_cmp, T, 4, 8, idx)
    assert e.value.code == -2
    x = torch.zeros(4, 300, dtype=torch.bfloat16, device="cuda")          # rows longer than 256
    with pytest.raises(api.CSAError) as e:
        _quant_gpu(h, x)
    assert e.value.code == -2
    assert h.device_status() == 0
