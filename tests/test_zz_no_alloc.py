"""The no-allocation KL entry point (needs a GPU).

csa_indexer_kl_static_scratch serves callers that cannot allocate device
memory (their allocations are owned by a host framework or frozen after
start-up): it uses a scratch array inside the library instead of a caller
workspace.  It must give the same result as csa_indexer_kl with a workspace,
on consecutive calls that leave different contents in the shared scratch.
This file is collected last so that a failure here cannot hide the others.
"""
import numpy as np
import pytest
import torch

from compressed_sparse_attention_compress_gb300 import inputs as I

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

from compressed_sparse_attention_compress_gb300 import api  # noqa: E402
from compressed_sparse_attention_compress_gb300.forward import Forward, to_device  # noqa: E402

KL_RTOL = 1e-3


def _forward(kl_mode, seed):
    wl = I.custom("noalloc", lengths=[700, 333, 1030], ratio=4, overlap=True, H=64, d=128, window=128, H_I=8,
                  d_I=64, topk=64, k_pad=64, kl_mode=kl_mode, cap_align=64)
    f = Forward(wl, to_device(I.generate(wl, seed), False))
    f.run()
    return f


def _both(f, sparse):
    wl = f.wl
    args = (f.h, f.x["q"], f.kv_cmp, f.x["qI"], f.x["w"], f.kI, f.cu, f.cu_cmp, f.max_seqlen, wl.ratio, f.scale)
    extra = dict(idx=f.idx if sparse else None, lse_cmp=f.lse_cmp if sparse else None)
    ref_sum = torch.zeros(1, device="cuda")
    ref_rows = torch.zeros(wl.T_cap, device="cuda")
    ref_n = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.empty(api.csa_indexer_kl_workspace(wl.T_cap), dtype=torch.uint8, device="cuda")
    api.csa_indexer_kl(*args, ref_sum, ws, kl_per_query=ref_rows, n_valid=ref_n, **extra)
    got_sum = torch.full((1,), float("nan"), device="cuda")
    got_n = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    api.csa_indexer_kl_static_scratch(*args, got_sum, n_valid=got_n, **extra)   # per-query rows in scratch
    torch.cuda.synchronize()
    assert f.h.device_status() == 0
    r, g = float(ref_sum.item()), float(got_sum.item())
    assert np.isfinite(g) and abs(g - r) <= KL_RTOL * abs(r), (g, r)
    assert int(got_n.item()) == int(ref_n.item())
    return g


def test_static_scratch_matches_workspace_on_consecutive_calls():
    dense = _forward("dense", seed=21)
    sparse = _forward("sparse", seed=22)
    a = _both(dense, sparse=False)     # first call on this device: scratch lookup
    b = _both(sparse, sparse=True)     # second call: different contents in the shared scratch
    assert a != b


def test_static_scratch_rejects_oversized_capacity():
    h = api.Handle(0)
    T = 262144 + 64
    q = torch.zeros(T, 4, 64, dtype=torch.bfloat16, device="cuda")
    qI = torch.zeros(T, 1, 32, dtype=torch.bfloat16, device="cuda")
    w = torch.zeros(T, 1, dtype=torch.bfloat16, device="cuda")
    kv = torch.zeros(16, 64, dtype=torch.bfloat16, device="cuda")
    kI = torch.zeros(16, 32, dtype=torch.bfloat16, device="cuda")
    cu = torch.tensor([0, 64], dtype=torch.int32, device="cuda")
    cu_cmp = torch.tensor([0, 16], dtype=torch.int32, device="cuda")
    with pytest.raises(api.CSAError) as e:
        api.csa_indexer_kl_static_scratch(h, q, kv, qI, w, kI, cu, cu_cmp, 64, 4, 0.125,
                                          torch.zeros(1, device="cuda"))
    assert e.value.code == -3
