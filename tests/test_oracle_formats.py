"""Pins for the oracle's element codecs (E2M1, E4M3FN, bf16).

Each codec is checked against something other than itself: exhaustive
enumeration of every code, a brute-force nearest-value search written
independently of the oracle's binade arithmetic, the tie cases the OCP
definitions fix, and (for bf16) the library's own float32 -> bfloat16 cast.
"""
import numpy as np
import pytest
import torch

from oracle import formats as F


# Magnitudes written out from the OCP definitions (not from the oracle code).
E2M1_MAGS = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def _e4m3_mags():
    out = []
    for e in range(16):
        for m in range(8):
            if e == 15 and m == 7:
                continue                      # S.1111.111 is NaN
            out.append(m * 2.0 ** -9 if e == 0 else 2.0 ** (e - 7) * (1 + m / 8))
    return out


E4M3_MAGS = _e4m3_mags()


def _brute_round(x, mags):
    """Nearest magnitude index by exhaustive search; ties go to the even code
    (even mantissa bit, which is the even index in an ordered code list);
    beyond the largest magnitude, saturate."""
    a = abs(x)
    if a >= mags[-1]:
        return len(mags) - 1
    best, bestd = None, None
    for i, m in enumerate(mags):
        d = abs(a - m)
        if bestd is None or d < bestd or (d == bestd and i % 2 == 0):
            best, bestd = i, d
    return best


def test_e2m1_decode_exhaustive():
    vals = F.e2m1_decode(np.arange(16))
    assert list(vals[:8]) == E2M1_MAGS
    assert list(vals[8:]) == [-m for m in E2M1_MAGS]


def test_e4m3_decode_exhaustive():
    vals = F.e4m3_decode(np.arange(256))
    pos = vals[:127]
    assert list(pos) == E4M3_MAGS
    assert np.isnan(vals[127]) and np.isnan(vals[255])
    assert list(vals[128:255]) == [-m for m in E4M3_MAGS]
    assert pos.max() == 448.0 and pos[1] == 2.0 ** -9


def test_e2m1_encode_roundtrips_every_code():
    codes = np.arange(16)
    back = F.e2m1_encode(F.e2m1_decode(codes))
    assert np.array_equal(back, codes)


def test_e4m3_encode_roundtrips_every_finite_code():
    codes = np.array([c for c in range(256) if c not in (127, 255)])
    back = F.e4m3_encode(F.e4m3_decode(codes))
    assert np.array_equal(back, codes)


@pytest.mark.parametrize("x,code", [(0.25, 0), (0.75, 2), (1.25, 2), (1.75, 4), (2.5, 4),
                                    (3.5, 6), (5.0, 6), (6.5, 7), (1e9, 7), (0.2499, 0),
                                    (0.2501, 1), (-0.75, 10), (-5.0, 14)])
def test_e2m1_ties_to_even_and_saturates(x, code):
    assert int(F.e2m1_encode(np.array([x]))[0]) == code


def test_e2m1_matches_brute_force_on_dense_sweep():
    rng = np.random.default_rng(7)
    xs = np.concatenate([np.linspace(-7, 7, 4001), rng.uniform(-8, 8, 2000),
                         np.array(E2M1_MAGS) + 0.0, (np.array(E2M1_MAGS[1:]) + np.array(E2M1_MAGS[:-1])) / 2])
    xs = F.f32(xs)
    got = F.e2m1_encode(xs)
    for x, c in zip(xs, got):
        want = _brute_round(x, E2M1_MAGS) | (8 if np.signbit(x) else 0)
        assert int(c) == want, (x, c, want)


def test_e4m3_matches_brute_force_on_dense_sweep():
    rng = np.random.default_rng(8)
    mags = np.array(E4M3_MAGS)
    mids = (mags[1:] + mags[:-1]) / 2
    xs = np.concatenate([mags, mids, mids * (1 + 1e-7), mids * (1 - 1e-7),
                         np.exp(rng.uniform(np.log(1e-4), np.log(600), 3000)), [460.0, 464.0, 1e6]])
    xs = F.f32(xs)
    got = F.e4m3_encode(xs)
    for x, c in zip(xs, got):
        assert int(c) == _brute_round(x, E4M3_MAGS), (x, c)


def test_negative_zero_keeps_sign():
    assert int(F.e2m1_encode(np.array([-0.1]))[0]) == 0x8
    assert int(F.e2m1_encode(np.array([0.1]))[0]) == 0x0
    assert int(F.e4m3_encode(np.array([-1e-6]))[0]) == 0x80


def test_bf16_round_matches_torch_cast():
    rng = np.random.default_rng(9)
    x = np.concatenate([rng.standard_normal(20000) * np.exp(rng.uniform(-20, 20, 20000)),
                        [0.0, -0.0, 1.0, 1.00390625, 1.001953125, 3.0e38, 1e-40]]).astype(np.float32)
    want = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    got = F.bf16_round(x)
    assert np.array_equal(got, want)


def test_bf16_bits_roundtrip():
    x = F.bf16_round(np.random.default_rng(1).standard_normal(1000))
    assert np.array_equal(F.bf16_from_bits(F.bf16_bits(x)), x)


def test_f32_is_ieee_binary32():
    x = np.random.default_rng(2).standard_normal(1000) * 1e3
    assert np.array_equal(F.f32(x), x.astype(np.float32).astype(np.float64))
