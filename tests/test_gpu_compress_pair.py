"""Both compressors of a layer in one launch (csa_compress_pair), on the GPU.

"DeepSeek-V4 Attention Training Systems" §3 (the indexer keys have their own
compressor), §4 (complete groups only, reset at packed-sample boundaries),
§5.1 (spans D_compress = 8 / 128).  The fused call must give the compressed
offsets and both streams' rows exactly as csa_compressed_offsets and one
csa_compress per stream do (bit for bit: the same arithmetic), and both
within the tolerance of the oracle; ragged lengths cover empty sequences,
sequences shorter than one block, tails of L mod r tokens and runs that end
mid-CTA.
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

LENGTHS = [0, 1, 3, 4, 5, 8, 127, 128, 129, 257, 1000, 4099, 20000]


@pytest.mark.parametrize("fp32", [False, True])
@pytest.mark.parametrize("D,d_I", [(128, 64), (64, 32)])
@pytest.mark.parametrize("ratio,overlap", [(4, True), (128, False), (4, False)])
def test_pair_equals_separate_calls_and_the_oracle(D, d_I, ratio, overlap, fp32):
    rng = np.random.default_rng(D + ratio)
    cu_np = np.concatenate([[0], np.cumsum(LENGTHS)]).astype(np.int32)
    T = int(cu_np[-1])
    S = 2 * ratio if overlap else ratio
    dt = torch.float32 if fp32 else torch.bfloat16

    def draw(shape):
        return I.bf16_round(rng.standard_normal(shape).astype(np.float32))

    x, z, xi, zi = draw((T, D)), draw((T, D)), draw((T, d_I)), draw((T, d_I))
    P = rng.standard_normal((S, D)).astype(np.float32)
    Pi = rng.standard_normal((S, d_I)).astype(np.float32)
    dev = lambda a, t=dt: torch.from_numpy(np.ascontiguousarray(a)).cuda().to(t)
    h = api.Handle(0)
    cu = dev(cu_np, torch.int32)
    n_cap = T // ratio + 2
    ref_cmp = oracle.compressed_offsets(cu_np, ratio)
    n_c = int(ref_cmp[-1])
    # fused
    cu_cmp = torch.full((len(LENGTHS) + 1,), -5, dtype=torch.int32, device="cuda")
    kv = torch.full((n_cap, D), 7.0, dtype=dt, device="cuda")
    ki = torch.full((n_cap, d_I), 7.0, dtype=dt, device="cuda")
    api.csa_compress_pair(h, dev(x), dev(z), dev(P, torch.float32), dev(xi), dev(zi), dev(Pi, torch.float32), cu,
                          max(LENGTHS), ratio, overlap, cu_cmp, kv, ki)
    # separate calls
    cu_cmp2 = torch.zeros_like(cu_cmp)
    kv2 = torch.full_like(kv, 7.0)
    ki2 = torch.full_like(ki, 7.0)
    api.csa_compressed_offsets(h, cu, ratio, cu_cmp2)
    api.csa_compress(h, dev(x), dev(z), dev(P, torch.float32), cu, cu_cmp2, max(LENGTHS), ratio, overlap, kv2)
    api.csa_compress(h, dev(xi), dev(zi), dev(Pi, torch.float32), cu, cu_cmp2, max(LENGTHS), ratio, overlap, ki2)
    torch.cuda.synchronize()
    assert h.device_status() == 0
    assert np.array_equal(cu_cmp.cpu().numpy(), ref_cmp)
    assert torch.equal(cu_cmp, cu_cmp2)
    assert torch.equal(kv, kv2) and torch.equal(ki, ki2)
    assert torch.all(kv[n_c:] == 7.0) and torch.all(ki[n_c:] == 7.0)
    ph.check_compress(kv, x, z, P, cu_np, ratio, overlap, n_c)
    ph.check_compress(ki, xi, zi, Pi, cu_np, ratio, overlap, n_c)


def test_pair_rejects_other_widths():
    h = api.Handle(0)
    cu = torch.tensor([0, 64], dtype=torch.int32, device="cuda")
    x = torch.zeros(64, 256, dtype=torch.bfloat16, device="cuda")
    xi = torch.zeros(64, 64, dtype=torch.bfloat16, device="cuda")
    P = torch.zeros(8, 256, device="cuda")
    Pi = torch.zeros(8, 64, device="cuda")
    with pytest.raises(api.CSAError) as e:
        api.csa_compress_pair(h, x, x, P, xi, xi, Pi, cu, 64, 4, True, torch.zeros(2, dtype=torch.int32,
                                                                                  device="cuda"),
                              torch.zeros(16, 256, dtype=torch.bfloat16, device="cuda"),
                              torch.zeros(16, 64, dtype=torch.bfloat16, device="cuda"))
    assert e.value.code == -2
