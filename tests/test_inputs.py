"""The seeded input generator shared by the GPU tests, the bench and the oracle tests (no GPU).

Both sides consume the generator's bf16-rounded values, so its rounding is
pinned to a library routine (torch's float32 -> bfloat16 conversion, round to
nearest even) on random values, exact ties, subnormals, infinities and NaN.
Its streams are independent: one generator per tensor, spawned in a fixed
order, so a workload that draws more tensors (the v4 compressor's extra
streams) leaves the shared ones unchanged, and a seed fixes every value.
"""
import dataclasses

import numpy as np
import torch

from compressed_sparse_attention_compress_gb300 import inputs as I


def _torch_bits(a):
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(torch.bfloat16).view(torch.int16).numpy() \
        .view(np.uint16)


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(7)
    a = (rng.standard_normal(200_000) * np.exp(rng.uniform(-40, 40, 200_000))).astype(np.float32)
    np.testing.assert_array_equal(I.bf16_bits(a), _torch_bits(a))
    # exact ties between neighbouring bf16 values go to the even mantissa
    base = rng.standard_normal(5000).astype(np.float32)
    hi = base.view(np.uint32) & np.uint32(0xFFFF0000)
    ties = (hi | np.uint32(0x8000)).view(np.float32)
    np.testing.assert_array_equal(I.bf16_bits(ties), _torch_bits(ties))
    assert np.all(I.bf16_bits(ties) & 1 == 0)
    # subnormals, signed zeros, infinities, the largest finite values
    special = np.array([1e-40, -1e-40, 0.0, -0.0, np.inf, -np.inf, 3.3895e38, -3.3895e38], np.float32)
    np.testing.assert_array_equal(I.bf16_bits(special), _torch_bits(special))
    # NaN stays NaN
    assert np.isnan(I.bf16_round(np.array([np.nan], np.float32)))[0]


def test_rounded_values_are_bf16_values():
    a = np.random.default_rng(3).standard_normal(10_000).astype(np.float32)
    r = I.bf16_round(a)
    assert np.all(r.view(np.uint32) & np.uint32(0xFFFF) == 0)
    assert np.all(np.abs(r - a) <= np.abs(a) * 2.0 ** -8)


def test_streams_are_independent_and_seeded():
    wl = I.custom("gen", lengths=[300, 5, 0, 77], ratio=4, overlap=True, H=4, d=64, window=64, H_I=2, d_I=32,
                  topk=16, k_pad=16, kl_mode="dense")
    plain = I.generate(wl, 11)
    again = I.generate(wl, 11)
    v4 = I.generate(dataclasses.replace(wl, compressor="v4"), 11)
    other = I.generate(wl, 12)
    for k in ("x_kv", "z_kv", "P_kv", "x_I", "z_I", "P_I", "q", "qI", "w"):
        np.testing.assert_array_equal(plain[k], again[k])      # a seed fixes every value
        np.testing.assert_array_equal(plain[k], v4[k])         # extra streams leave these unchanged
        assert not np.array_equal(plain[k], other[k])
    for k in ("x_kv_prev", "z_kv_prev", "x_I_prev", "z_I_prev", "g_kv", "g_I"):
        assert k in v4 and k not in plain
    np.testing.assert_array_equal(plain["cu_seqlens"], [0, 300, 305, 305, 382])
    assert plain["q"].shape == (wl.T_cap, 4, 64) and plain["P_kv"].shape == (8, 64)
