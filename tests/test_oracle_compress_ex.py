"""Pins for the oracle's compressor variant (CPU only).

The variant adds three things around the softmax-gated compressor
("DeepSeek-V4 Attention Training Systems", §9 FP32 positional parameter, §10
"compressor softmax and normalization intermediates", §12 invariant 2 "RoPE
mode is per layer and per compressed coordinate system"): a separate (x, z)
projection for the previous-block half of an overlapping span, a
post-compression RMSNorm and a rotary embedding on compressed coordinates.
Each step is pinned to something other than the oracle's own formula: the
single-stream oracle, brute-force dependency sets, torch's RMSNorm, the
complex-number form of the rotary embedding (Su et al., "RoFormer", 2021) and
its relative-position property.
"""
import numpy as np
import pytest
import torch

import oracle
from compressed_sparse_attention_compress_gb300.inputs import bf16_round

rng = np.random.default_rng(4321)


def _rand(*shape):
    return bf16_round(rng.standard_normal(shape).astype(np.float32))


def _case(r, overlap, L, D):
    S = 2 * r if overlap else r
    return _rand(L, D), _rand(L, D), _rand(L, D), _rand(L, D), _rand(S, D)


@pytest.mark.parametrize("r,overlap", [(4, True), (4, False), (128, False), (2, True)])
def test_same_stream_twice_is_the_single_stream_compressor(r, overlap):
    L, D = 7 * r + 3, 12
    x, z, _, _, P = _case(r, overlap, L, D)
    base = oracle.compress(x, z, P, [0, L], r, overlap)
    np.testing.assert_array_equal(oracle.compress_ex(x, z, P, [0, L], r, overlap), base)
    np.testing.assert_array_equal(oracle.compress_ex(x, z, P, [0, L], r, overlap, x_prev=x, z_prev=z), base)


@pytest.mark.parametrize("which", ["x", "z"])
def test_previous_half_reads_the_previous_stream(which):
    # Brute force: perturb one token of one stream and record which entries
    # move.  Token t of the previous-half stream feeds only entry t//r + 1 (it
    # sits in block j-1 of that entry); token t of the current stream feeds only
    # entry t//r.
    r, L, D = 4, 6 * 4 + 3, 6
    x, z, xp, zp, P = _case(r, True, L, D)
    n = L // r
    base = oracle.compress_ex(x, z, P, [0, L], r, True, x_prev=xp, z_prev=zp)
    for t in range(L):
        for stream in ("prev", "cur"):
            args = dict(x=x, z=z, x_prev=xp, z_prev=zp)
            key = (which + "_prev") if stream == "prev" else which
            a = args[key].copy()
            a[t] += 1.0
            args[key] = a
            out = oracle.compress_ex(args["x"], args["z"], P, [0, L], r, True,
                                     x_prev=args["x_prev"], z_prev=args["z_prev"])
            moved = set(np.nonzero(np.abs(out - base).max(1) > 0)[0].tolist())
            j = t // r + (1 if stream == "prev" else 0)
            assert moved == ({j} if j < n else set()), (stream, t, moved)


@pytest.mark.parametrize("u_star", [0, 3, 4, 7])
def test_one_hot_position_copies_the_row_of_its_half(u_star):
    r, L, D = 4, 9 * 4, 8
    x, _, xp, _, _ = _case(r, True, L, D)
    z = np.zeros((L, D), np.float32)
    P = np.zeros((2 * r, D), np.float32)
    P[u_star] = 80.0
    out = oracle.compress_ex(x, z, P, [0, L], r, True, x_prev=xp, z_prev=z)
    for j in range(L // r):
        t = r * j - r + u_star
        if t < 0:
            continue
        want = xp[t] if u_star < r else x[t]
        np.testing.assert_allclose(out[j], want, rtol=0, atol=1e-20)


@pytest.mark.parametrize("eps", [0.0, 1e-6, 0.25])
def test_rmsnorm_matches_torch_rms_norm(eps):
    r, L, D = 4, 61, 32
    x, z, xp, zp, P = _case(r, True, L, D)
    gamma = (1.0 + 0.1 * rng.standard_normal(D)).astype(np.float32)
    base = oracle.compress_ex(x, z, P, [0, L], r, True, x_prev=xp, z_prev=zp)
    got = oracle.compress_ex(x, z, P, [0, L], r, True, x_prev=xp, z_prev=zp, gamma=gamma, eps=eps)
    want = torch.nn.functional.rms_norm(torch.from_numpy(base), (D,),
                                        weight=torch.from_numpy(gamma.astype(np.float64)),
                                        eps=float(np.float32(eps))).numpy()
    np.testing.assert_allclose(got, want, rtol=1e-13, atol=1e-14)


def test_rmsnorm_with_unit_gain_and_no_eps_gives_unit_rms():
    r, L, D = 128, 3 * 128 + 5, 16
    x, z, _, _, P = _case(r, False, L, D)
    got = oracle.compress_ex(x, z, P, [0, L], r, False, gamma=np.ones(D, np.float32), eps=0.0)
    np.testing.assert_allclose(np.mean(got * got, axis=1), 1.0, rtol=1e-13)


@pytest.mark.parametrize("rope_dim,theta,stride,offset", [(8, 10000.0, 1, 0), (16, 10000.0, 4, 3),
                                                          (4, 160000.0, 1, 1000), (16, 10000.0, 128, 0)])
def test_rope_matches_complex_rotation(rope_dim, theta, stride, offset):
    # RoFormer's complex form: the pair (y_{2i}, y_{2i+1}) of the rotated band is
    # the complex number y_{2i} + i y_{2i+1} multiplied by exp(i p theta^(-2i/d)).
    r, L, D = 4, 83, 16
    x, z, xp, zp, P = _case(r, True, L, D)
    gamma = (1.0 + 0.1 * rng.standard_normal(D)).astype(np.float32)
    kw = dict(x_prev=xp, z_prev=zp, gamma=gamma, eps=1e-6)
    base = oracle.compress_ex(x, z, P, [0, L], r, True, **kw)
    got = oracle.compress_ex(x, z, P, [0, L], r, True, rope_dim=rope_dim, theta=theta,
                             pos_stride=stride, pos_offset=offset, **kw)
    lo = D - rope_dim
    np.testing.assert_array_equal(got[:, :lo], base[:, :lo])   # channels outside the band untouched
    zc = base[:, lo::2] + 1j * base[:, lo + 1::2]
    pos = np.arange(base.shape[0], dtype=np.float64) * stride + offset
    freqs = theta ** (-np.arange(0, rope_dim, 2, dtype=np.float64) / rope_dim)
    rot = zc * np.exp(1j * pos[:, None] * freqs[None, :])
    np.testing.assert_allclose(got[:, lo::2], rot.real, rtol=0, atol=1e-12)
    np.testing.assert_allclose(got[:, lo + 1::2], rot.imag, rtol=0, atol=1e-12)


def test_rope_is_a_relative_position_encoding():
    # Shifting every position by the same amount leaves the band's pairwise
    # dot products unchanged and keeps each pair's norm; position 0 is the
    # identity.
    r, L, D, rope = 4, 64, 16, 8
    x, z, _, _, P = _case(r, True, L, D)
    plain = oracle.compress_ex(x, z, P, [0, L], r, True)
    a = oracle.compress_ex(x, z, P, [0, L], r, True, rope_dim=rope, pos_offset=0)
    b = oracle.compress_ex(x, z, P, [0, L], r, True, rope_dim=rope, pos_offset=777)
    band = slice(D - rope, D)
    np.testing.assert_allclose(a[:, band] @ a[:, band].T, b[:, band] @ b[:, band].T, rtol=0, atol=1e-11)
    pn = lambda y: y[:, D - rope::2] ** 2 + y[:, D - rope + 1::2] ** 2  # noqa: E731
    np.testing.assert_allclose(pn(a), pn(plain), rtol=1e-12)
    np.testing.assert_array_equal(a[0], plain[0])


def test_packed_sequences_restart_streams_and_positions():
    # §4 / §12: packed sample boundaries reset the compressor, and the
    # compressed coordinate of each sequence starts again at 0.
    r, D = 4, 8
    lengths = [13, 4, 0, 22, 3, 9]
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    T = int(cu[-1])
    x, z, xp, zp, P = _case(r, True, T, D)
    gamma = (1.0 + 0.1 * rng.standard_normal(D)).astype(np.float32)
    kw = dict(gamma=gamma, eps=1e-6, rope_dim=4, pos_stride=1, pos_offset=5)
    packed = oracle.compress_ex(x, z, P, cu, r, True, x_prev=xp, z_prev=zp, **kw)
    cu_cmp = oracle.compressed_offsets(cu, r)
    for b, L in enumerate(lengths):
        s = slice(cu[b], cu[b + 1])
        alone = oracle.compress_ex(x[s], z[s], P, [0, L], r, True, x_prev=xp[s], z_prev=zp[s], **kw)
        np.testing.assert_array_equal(packed[cu_cmp[b]:cu_cmp[b + 1]], alone)


def test_previous_stream_is_ignored_without_overlap():
    r, L, D = 4, 30, 8
    x, z, xp, zp, P = _case(r, False, L, D)
    np.testing.assert_array_equal(oracle.compress_ex(x, z, P, [0, L], r, False, x_prev=xp, z_prev=zp),
                                  oracle.compress(x, z, P, [0, L], r, False))
