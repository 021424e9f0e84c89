"""Pins for the oracle's FP8 (E4M3) quantisation of the indexer operands (CPU only).

"DeepSeek-V4 Attention Training Systems" §1 and §9 name an FP8 indexer for the
index-search term and fix nothing else; the reading taken is E4M3 codes with
one power-of-two scale per row (the smallest 2^e with max|x| / 2^e <= 448),
round to nearest even.  The codes are pinned to torch's float8_e4m3fn
conversion (a library routine) on random rows, on exact ties, on subnormals
and at the top of the range; the scale to its defining inequalities.
"""
import numpy as np
import pytest
import torch

import oracle

rng = np.random.default_rng(31)


def _torch_codes(x, scales):
    y = torch.from_numpy((x.astype(np.float64) / scales.astype(np.float64)[..., None]).astype(np.float32))
    return y.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


@pytest.mark.parametrize("spread", [1.0, 1e-3, 1e3, 1e-30])
def test_codes_match_torch_float8_e4m3fn(spread):
    x = (rng.standard_normal((257, 64)) * spread * np.exp(rng.standard_normal((257, 1)))).astype(np.float32)
    x[3] = 0.0                                   # an all-zero row
    codes, scales = oracle.quantize_fp8(x)
    np.testing.assert_array_equal(codes, _torch_codes(x, scales))


def test_ties_round_to_even_and_subnormals():
    # values exactly halfway between neighbouring E4M3 values, in the normal and
    # the subnormal range, with a fixed scale of 1 (the row maximum is 448)
    table = np.array([oracle.e4m3_value(c) for c in range(0x7f)])      # positive finite codes
    mids = (table[:-1] + table[1:]) / 2
    x = np.concatenate([[448.0], mids[:63]]).astype(np.float32)[None, :]
    codes, scales = oracle.quantize_fp8(x)
    assert scales[0] == 1.0
    np.testing.assert_array_equal(codes, _torch_codes(x, scales))
    # each tie went to the code with an even mantissa
    assert np.all(codes[0, 1:] % 2 == 0)


def test_signed_zeros_keep_their_sign():
    x = np.array([[-0.0, 0.0, -1e-30, 1e-30, 1.0]], np.float32)
    codes, scales = oracle.quantize_fp8(x)
    np.testing.assert_array_equal(codes, _torch_codes(x, scales))
    assert codes[0, 0] == 0x80 and codes[0, 1] == 0x00


def test_scale_is_the_smallest_power_of_two_that_fits():
    x = (rng.standard_normal((500, 32)) * np.exp(3 * rng.standard_normal((500, 1)))).astype(np.float32)
    _, scales = oracle.quantize_fp8(x)
    amax = np.abs(x).max(1).astype(np.float64)
    m, e = np.frexp(scales)
    assert np.all(m == 0.5)                                   # powers of two
    assert np.all(amax / scales <= 448.0)
    assert np.all(amax / (scales / 2) > 448.0)                # half the scale would not fit


def test_dequantised_values_are_exact_and_within_half_a_step():
    x = rng.standard_normal((64, 64)).astype(np.float32)
    codes, scales = oracle.quantize_fp8(x)
    deq = oracle.dequantize_fp8(codes, scales)
    table = np.array([oracle.e4m3_value(c) for c in range(256)])
    exact = table[codes] * scales[:, None].astype(np.float64)
    np.testing.assert_array_equal(deq.astype(np.float64), exact)          # no rounding in float32
    # the error is at most half the spacing of E4M3 values at that magnitude
    y = np.abs(x.astype(np.float64)) / scales[:, None]
    step = np.where(y < 2.0 ** -6, 2.0 ** -9, 2.0 ** (np.floor(np.log2(np.maximum(y, 2.0 ** -6))) - 3))
    assert np.all(np.abs(deq - x) / scales[:, None] <= step / 2 + 1e-12)
