"""The host-input forward (``Forward.run_from_host``) against the resident one.

``run_from_host`` copies the queries in row chunks and runs the selected
attention chunk by chunk as they arrive, each chunk a packing of its own with
per-segment position offsets and a boundary of W raw rows ("DeepSeek-V4
Attention Training Systems" §5, the contiguous context-parallel layout; §4.1,
static capacity).  Every output must be bit for bit the one of ``Forward.run``
on device-resident inputs: the per-query arithmetic is the same, only the rows
around it moved.  Cases: one long sequence, and a ragged packing with a
one-token sequence, chunk starts inside sequences and capacity rows.
"""
import numpy as np
import pytest
import torch

from compressed_sparse_attention_compress_gb300 import inputs as I

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # the CPU suite never collects GPU work
    pytest.skip("no CUDA device", allow_module_level=True)

from compressed_sparse_attention_compress_gb300.forward import Forward, to_device  # noqa: E402

CASES = [
    I.WORKLOADS["warmup8k"],
    I.custom("ragged_dense", lengths=[3000, 1, 2500, 700, 1900], ratio=4, overlap=True, H=64, d=128, window=128,
             H_I=8, d_I=64, topk=256, k_pad=256, kl_mode="dense", cap_align=128),
    I.custom("ragged_sparse", lengths=[1200, 4100, 20, 2999], ratio=4, overlap=True, H=64, d=128, window=128,
             H_I=8, d_I=64, topk=512, k_pad=512, kl_mode="sparse", cap_align=64),
]


@pytest.mark.parametrize("wl", CASES, ids=[c.name for c in CASES])
def test_chunked_host_forward_is_bitwise_the_resident_forward(wl):
    arrs = I.generate(wl, 5)
    dev = to_device(arrs, wl.io_fp32)
    f = Forward(wl, dev)
    f.run()
    torch.cuda.synchronize()
    assert f.h.device_status() == 0
    names = ["out", "lse", "lse_cmp", "idx", "kl_sum", "kl_rows"]
    ref = {k: getattr(f, k).clone() for k in names}
    host = {k: v.cpu().pin_memory() for k, v in dev.items()}
    chunks = f._attention_chunks()
    assert len(chunks) == f.attend_chunks   # the chunked path is the one under test
    # every query row is copied exactly once, and before the first chunk that reads it
    copied = np.zeros(wl.T_cap, np.int32)
    for c in chunks:
        copied[c["copy"][0]:c["copy"][1]] += 1
        assert copied[c["lo"]:c["hi"]].all()
    assert (copied == 1).all()
    # stale device state: queries and outputs overwritten before the host run
    dev["q"].fill_(3.0)
    for k in names:
        getattr(f, k).fill_(-7)
    f.run_from_host(host)
    torch.cuda.synchronize()
    assert f.h.device_status() == 0
    for k in names:
        got, exp = getattr(f, k), ref[k]
        if got.dtype.is_floating_point:
            assert torch.equal(got.view(torch.int16 if got.element_size() == 2 else torch.int32),
                               exp.view(torch.int16 if exp.element_size() == 2 else torch.int32)), k
        else:
            assert torch.equal(got, exp), k
