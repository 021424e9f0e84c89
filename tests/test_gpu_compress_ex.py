"""GPU parity of the compressor variant (csa_compress_ex) against the oracle.

The variant adds a separate previous-half stream, a post-compression RMSNorm
and a rotary embedding on compressed coordinates to the softmax-gated
compressor ("DeepSeek-V4 Attention Training Systems", §10, §12 invariants 2
and 3).  Every case compares all entries with the fp64 oracle: float32
outputs within max-abs 1e-2; bf16 outputs within max-abs 1e-2 where |x| < 4,
and at |x| >= 4 (bf16 spacing 1/32, after the RMSNorm) one of the two bf16
values bracketing the exact one; ragged lengths
cover empty sequences, sequences shorter than one block, a tail of L mod r
tokens and runs that end mid-CTA.
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

RAGGED = [0, 1, 3, 4, 5, 8, 127, 128, 129, 257, 1000, 4099]


def _dev(a, fp32):
    t = torch.from_numpy(np.ascontiguousarray(a)).cuda()
    return t if fp32 else t.to(torch.bfloat16)


def _run(lengths, D, ratio, overlap, two, norm, rope_dim, fp32=False, stride=1, offset=0, theta=10000.0,
         seed=0, eps=1e-6):
    arrs = I.generate_compress_ex(lengths, D, ratio, overlap, two, seed=seed)
    cu_np = arrs["cu_seqlens"]
    cu_cmp_np = oracle.compressed_offsets(cu_np, ratio)
    n_c = int(cu_cmp_np[-1])
    h = api.Handle(0)
    cu = torch.from_numpy(cu_np).cuda()
    cu_cmp = torch.from_numpy(cu_cmp_np).cuda()
    x, z = _dev(arrs["x"], fp32), _dev(arrs["z"], fp32)
    xp = _dev(arrs["x_prev"], fp32) if two else None
    zp = _dev(arrs["z_prev"], fp32) if two else None
    P = torch.from_numpy(arrs["P"]).cuda()
    g = torch.from_numpy(arrs["gamma"]).cuda() if norm else None
    out = torch.full((max(n_c, 1) + 3, D), 7.0, dtype=x.dtype, device="cuda")  # rows past n_c stay 7
    api.csa_compress_ex(h, x, z, P, cu, cu_cmp, max(lengths + [1]), ratio, overlap, out, x_prev=xp, z_prev=zp,
                        norm_weight=g, norm_eps=eps, rope_dim=rope_dim, rope_theta=theta,
                        rope_pos_stride=stride, rope_pos_offset=offset)
    torch.cuda.synchronize()
    assert h.device_status() == 0
    assert torch.all(out[n_c:] == 7.0)
    ref = oracle.compress_ex(arrs["x"], arrs["z"], arrs["P"], cu_np, ratio, overlap,
                             x_prev=arrs.get("x_prev"), z_prev=arrs.get("z_prev"),
                             gamma=arrs["gamma"] if norm else None, eps=eps, rope_dim=rope_dim, theta=theta,
                             pos_stride=stride, pos_offset=offset)
    got = ph.np32(out[:n_c]).astype(np.float64)
    if fp32:
        err = ph.record("compress_ex_fp32", np.abs(got - ref).max() if ref.size else 0.0)
        assert err <= ph.ATOL, f"compress_ex max-abs {err}"
    elif ref.size:
        ph.check_stored_bf16(got, ref, "compress_ex")
    return out[:n_c], (h, x, z, P, cu, cu_cmp)


@pytest.mark.parametrize("D", [32, 64, 128, 256, 512])
@pytest.mark.parametrize("two", [True, False])
def test_csa_overlap_norm_rope(D, two):
    _run(RAGGED, D, 4, True, two, norm=True, rope_dim=min(64, D // 2))


@pytest.mark.parametrize("D", [256, 512])
def test_fp32_output_of_the_widest_norm_rope_cases(D):
    """The unrounded (float32-output) values of the cases whose RMSNorm outputs
    reach |x| >= 4: the arithmetic itself within the plain max-abs 1e-2."""
    _run(RAGGED, D, 4, True, True, norm=True, rope_dim=64, fp32=True)


@pytest.mark.parametrize("fp32", [False, True])
@pytest.mark.parametrize("norm,rope_dim", [(True, 0), (False, 64), (False, 0), (True, 128)])
def test_each_step_alone(fp32, norm, rope_dim):
    _run(RAGGED, 128, 4, True, True, norm=norm, rope_dim=rope_dim, fp32=fp32)


@pytest.mark.parametrize("D", [64, 128, 256])
def test_hca_ratio128_norm_rope(D):
    _run([127, 128, 129, 1000, 5000, 0, 300], D, 128, False, False, norm=True, rope_dim=64, stride=128)


def test_long_positions_keep_the_angle_exact():
    # positions up to ~4e6 (offset + stride * j): the rotation is reduced in
    # turns, so the angle of the fastest pair stays accurate
    _run([65536, 9000], 128, 4, True, True, norm=True, rope_dim=64, stride=4, offset=3_900_000, theta=160000.0)


def test_packed_128k_tokens_full_compare():
    # 16 packed sequences, 1K..16K tokens each (the packed THD workload's mix)
    _run(I.WORKLOADS["thd128k"].lengths, 128, 4, True, True, norm=True, rope_dim=64)


def test_without_extras_matches_csa_compress_bit_for_bit():
    lengths = [5, 1000, 4099, 0, 77]
    out_ex, (h, x, z, P, cu, cu_cmp) = _run(lengths, 128, 4, True, False, norm=False, rope_dim=0)
    out = torch.empty_like(out_ex)
    api.csa_compress(h, x, z, P, cu, cu_cmp, max(lengths), 4, True, out)
    torch.cuda.synchronize()
    assert torch.equal(out, out_ex)


def test_argument_errors():
    h = api.Handle(0)
    T, D = 64, 128
    cu = torch.tensor([0, T], dtype=torch.int32, device="cuda")
    cu_cmp = torch.zeros(2, dtype=torch.int32, device="cuda")
    x = torch.zeros(T, D, dtype=torch.bfloat16, device="cuda")
    P = torch.zeros(8, D, dtype=torch.float32, device="cuda")
    P4 = torch.zeros(4, D, dtype=torch.float32, device="cuda")
    out = torch.zeros(16, D, dtype=torch.bfloat16, device="cuda")

    def code(**kw):
        args = dict(ratio=4, overlap=True, pos=P)
        args.update(kw)
        try:
            api.csa_compress_ex(h, args.pop("x", x), x, args.pop("pos"), cu, cu_cmp, T, args.pop("ratio"),
                                args.pop("overlap"), out, **args)
        except api.CSAError as e:
            return e.code
        return 0

    assert code(x_prev=x) == -1                                  # z_prev missing
    assert code(x_prev=x, z_prev=x, overlap=False, pos=P4) == -1  # previous half without overlap
    assert code(rope_dim=63) == -1                               # odd band
    assert code(rope_dim=256) == -1                              # band wider than D
    assert code(rope_dim=64, rope_theta=1.0) == -1
    assert code(norm_eps=-1.0) == -1
    x96 = torch.zeros(T, 96, dtype=torch.bfloat16, device="cuda")
    assert code(x=x96, pos=torch.zeros(8, 96, device="cuda")) == -2  # D = 96 has no kernel
    x512 = torch.zeros(256, 512, dtype=torch.bfloat16, device="cuda")
    hca = torch.zeros(128, 512, dtype=torch.float32, device="cuda")
    assert code(x=x512, pos=hca, ratio=128, overlap=False) == -2  # ratio-128 span at D = 512
    assert h.device_status() == 0
