"""Pins for the oracle's FP8 (e4m3) KV quantisation (CPU only).

The codec is pinned to the e4m3 format's definition (closed-form values of
named codes, the count of finite values, a round trip over every code) and
to an independent library routine (torch's float8_e4m3fn cast, which rounds
to nearest even); the per-token quantiser to the error bound the format
fixes; the fp8 decode to the float64 decode of the dequantised pool.
"""

import numpy as np
import pytest
import torch

import oracle
from oracle import quant as Q


def test_named_codes_have_their_closed_form_values():
    v = Q.e4m3_decode(np.array([0x00, 0x80, 0x01, 0x07, 0x08, 0x38, 0x39, 0x7E, 0xFE, 0x7F, 0xFF], np.uint8))
    assert v[0] == 0 and v[1] == 0 and np.signbit(v[1])
    assert v[2] == 2.0 ** -9                       # smallest subnormal
    assert v[3] == 7 * 2.0 ** -9                   # largest subnormal
    assert v[4] == 2.0 ** -6                       # smallest normal
    assert v[5] == 1.0 and v[6] == 1.125           # bias 7, 3 mantissa bits
    assert v[7] == 448.0 and v[8] == -448.0        # largest finite
    assert np.isnan(v[9]) and np.isnan(v[10])      # the only NaN patterns


def test_code_space_counts_and_ordering():
    vals = Q.e4m3_decode(np.arange(256, dtype=np.uint8))
    finite = vals[~np.isnan(vals)]
    assert len(finite) == 254
    assert len(np.unique(finite)) == 253            # +0 and -0 compare equal
    pos = vals[:0x7F]
    assert np.all(np.diff(pos) > 0)                 # codes 0..0x7E increase
    # spacing: 2**-9 through the subnormals and the first normal binade, then doubling
    assert np.allclose(np.diff(pos)[:15], 2.0 ** -9)


def test_round_trip_of_every_finite_code():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    assert np.array_equal(Q.e4m3_encode(Q.e4m3_decode(codes)), codes)


def test_encoder_matches_torch_float8_cast():
    rng = np.random.default_rng(0)
    mags = np.exp2(rng.uniform(-12, np.log2(460), size=200_000))
    x = (mags * rng.choice([-1.0, 1.0], size=mags.size)).astype(np.float32)
    # every exact tie between neighbouring finite values, and the subnormal ties
    pos = Q.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    ties = ((pos[:-1] + pos[1:]) / 2).astype(np.float32)
    x = np.concatenate([x, ties, -ties, np.float32([448.0, 463.9, 0.0])])
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = Q.e4m3_encode(x)
    assert np.array_equal(got, ref)


def test_encoder_saturates_instead_of_nan():
    assert Q.e4m3_encode(np.float32([500.0, -1e6]).astype(np.float64)).tolist() == [0x7E, 0xFE]


@pytest.mark.parametrize("seed", range(4))
def test_per_token_quantisation_error_bound(seed):
    rng = np.random.default_rng(seed)
    x = (rng.standard_normal((8, 128)) * rng.uniform(0.01, 100)).astype(np.float32)
    codes, s = Q.quantize_token(x)
    assert codes.shape == x.shape and codes.dtype == np.uint8 and s.dtype == np.float32
    xh = Q.e4m3_decode(codes) * np.float64(s)
    # the largest magnitude lands on +-448 exactly
    i = np.unravel_index(np.argmax(np.abs(x)), x.shape)
    assert codes[i] & 0x7F == 0x7E
    # normals: half an ulp (2**-4 relative); subnormals: half of 2**-9 times the scale;
    # plus the float32 rounding of x * (448/amax) and of the scale
    bound = np.maximum(2.0 ** -4 * np.abs(x), 2.0 ** -10 * float(s)) * (1 + 1e-6) + 4 * 2.0 ** -24 * np.abs(x)
    assert np.all(np.abs(xh - x) <= bound)


def test_zero_vector_gives_zero_scale_and_codes():
    codes, s = Q.quantize_token(np.zeros((2, 4), np.float32))
    assert s == 0 and not codes.any()


def test_append_fp8_writes_only_addressed_slots():
    rng = np.random.default_rng(3)
    NB, bs, H, D = 5, 4, 2, 8
    kc = rng.integers(0, 256, size=(NB, bs, H, D), dtype=np.uint8)
    vc = rng.integers(0, 256, size=(NB, bs, H, D), dtype=np.uint8)
    ks, vs = rng.random((NB, bs)).astype(np.float32), rng.random((NB, bs)).astype(np.float32)
    key = rng.standard_normal((3, H, D)).astype(np.float32)
    val = rng.standard_normal((3, H, D)).astype(np.float32)
    slots = np.array([6, -1, 17])
    kc2, vc2, ks2, vs2 = Q.reshape_and_cache_fp8(key, val, slots, kc, vc, ks, vs)
    c, s = Q.quantize_token(key[0])
    assert np.array_equal(kc2[1, 2], c) and ks2[1, 2] == s
    c, s = Q.quantize_token(val[2])
    assert np.array_equal(vc2[4, 1], c) and vs2[4, 1] == s
    mask = np.ones((NB, bs), bool)
    mask[1, 2] = mask[4, 1] = False
    assert np.array_equal(kc2[mask], kc[mask]) and np.array_equal(ks2[mask], ks[mask])
    assert np.array_equal(vc2[mask], vc[mask]) and np.array_equal(vs2[mask], vs[mask])


def test_fp8_decode_is_decode_of_the_dequantised_pool_and_close_to_full_precision():
    rng = np.random.default_rng(5)
    NB, bs, H, D, B = 12, 4, 2, 16, 2
    k = rng.standard_normal((NB, bs, H, D)).astype(np.float32)
    v = rng.standard_normal((NB, bs, H, D)).astype(np.float32)
    kc = np.zeros(k.shape, np.uint8)
    vc = np.zeros(v.shape, np.uint8)
    ks = np.zeros((NB, bs), np.float32)
    vs = np.zeros((NB, bs), np.float32)
    for b in range(NB):
        for o in range(bs):
            kc[b, o], ks[b, o] = Q.quantize_token(k[b, o])
            vc[b, o], vs[b, o] = Q.quantize_token(v[b, o])
    tables = np.array([[3, 7, 1, 0], [10, 2, 5, 0]])
    lens = np.array([11, 9])
    q = rng.standard_normal((B, 2 * H, D))
    sc = 1 / np.sqrt(D)
    got = Q.paged_decode_fp8(q, kc, vc, ks, vs, tables, lens, sc)
    # the same thing by the walk over an explicitly dequantised pool
    kd = Q.e4m3_decode(kc) * ks[:, :, None, None].astype(np.float64)
    vd = Q.e4m3_decode(vc) * vs[:, :, None, None].astype(np.float64)
    walk = oracle.paged_decode(q, kd, vd, tables, lens, sc, method="walk")
    assert np.abs(got - walk).max() <= 1e-12
    # quantisation keeps the result near the full-precision one (3 mantissa bits)
    full = oracle.paged_decode(q, k.astype(np.float64), v.astype(np.float64), tables, lens, sc)
    assert np.abs(got - full).max() < 0.1
    assert np.abs(got - full).mean() < 0.02


def test_planted_codec_mistakes_are_caught():
    rng = np.random.default_rng(9)
    x = np.exp2(rng.uniform(-11, 8.7, size=20000)).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()

    def trunc(v):                                  # rounding toward zero
        a = np.abs(v.astype(np.float64))
        _, ex = np.frexp(np.where(a > 0, a, 1.0))
        qn = np.exp2(np.maximum(ex - 1, -6) - 3.0)
        return Q.e4m3_encode(np.floor(a / qn) * qn)

    def half_away(v):                              # ties away from zero
        a = np.abs(v.astype(np.float64))
        _, ex = np.frexp(np.where(a > 0, a, 1.0))
        qn = np.exp2(np.maximum(ex - 1, -6) - 3.0)
        return Q.e4m3_encode(np.floor(a / qn + 0.5) * qn)

    pos = Q.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    ties = ((pos[:-1] + pos[1:]) / 2).astype(np.float32)
    ref_t = torch.from_numpy(ties).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert not np.array_equal(trunc(x), ref)
    assert not np.array_equal(half_away(ties), ref_t)
    # a decoder with bias 8 instead of 7 halves every normal value: the
    # named-code pin (0x38 -> 1.0, 0x7E -> 448) rejects it
    def bias8(c):
        return (8 + (c & 7)) * 2.0 ** (((c >> 3) & 15) - 11)
    assert bias8(0x38) != 1.0 and bias8(0x7E) != 448.0
