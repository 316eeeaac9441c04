"""Pins of the per-tensor FP8 (E4M3) KV encoder and its page layout.

The encoder (oracle/fp8.py) multiplies by the correctly rounded reciprocal of
the per-tensor scale and rounds to E4M3 with ties to even and saturation.
These tests check it against things fixed independently of that code: every
finite code round-trips, an exhaustive nearest-value search on the code grid,
the half-spacing error bound, saturation, the sign of zero, and byte offsets
worked out by hand.
"""
import numpy as np
import pytest

from oracle import fp8 as F
from oracle import paged as PG
from oracle.formats import e4m3_decode

D = 256
FINITE = np.array([c for c in range(256) if (c & 0x7F) != 0x7F])  # all codes but the two NaNs


@pytest.mark.parametrize("g", [1.0, 0.25, 0.01, 3.7e-3])
def test_every_finite_code_round_trips(g):
    g32 = float(np.float32(g))
    x = e4m3_decode(FINITE) * g32
    got = F.quantize(x, g)
    # +0 and -0 both decode to 0; the sign bit of zero follows the input's sign
    assert np.array_equal(got, FINITE.astype(np.uint8))
    assert np.array_equal(F.dequantize(got, g), x)


def test_nearest_code_by_exhaustive_search():
    rng = np.random.default_rng(5)
    g = 0.0123
    r = float(np.float32(1.0 / np.float64(np.float32(g))))
    x = rng.standard_normal(20000) * rng.choice([1e-3, 0.05, 1.0, 5.0], 20000)
    xs = (x * r).astype(np.float32).astype(np.float64)      # the fp32 product
    grid = e4m3_decode(np.arange(127))                       # non-negative finite values
    for xi, si, c in zip(x[:4000], xs[:4000], F.quantize(x[:4000], g)):
        a = min(abs(si), 448.0)
        dist = np.abs(grid - a)
        best = np.flatnonzero(dist == dist.min())
        want = best[0] if len(best) == 1 else best[np.argmin(best % 2 == 1)]  # ties: even mantissa
        assert (c & 0x7F) == want
        assert (c >> 7) == (1 if np.signbit(si) else 0)


def test_error_bound_and_saturation():
    rng = np.random.default_rng(6)
    g = 0.02
    x = rng.uniform(-448 * g, 448 * g, 50000)
    xh = F.dequantize(F.quantize(x, g), g)
    # half the E4M3 spacing at |x| (3 fraction bits; subnormal spacing 2^-9), times g,
    # plus the fp32 product's own rounding
    e = np.maximum(np.floor(np.log2(np.maximum(np.abs(x) / g, 2.0 ** -6))), -6)
    half = 0.5 * 2.0 ** (e - 3) * g
    assert np.all(np.abs(xh - x) <= half * (1 + 1e-6) + 1e-12)
    big = np.array([500 * g, -1e6 * g])
    g32 = float(np.float32(g))
    assert np.array_equal(F.dequantize(F.quantize(big, g), g), np.array([448 * g32, -448 * g32]))


def test_sign_of_zero():
    assert F.quantize(np.array([-1e-30, 1e-30, -0.0, 0.0]), 1.0).tolist() == [0x80, 0x00, 0x80, 0x00]


def test_fp8_page_layout_offsets_by_hand():
    """Token 37 of a sequence whose page table is [5, 2, 9] lives in page 9,
    slot 5 (an odd slot of pair 2).  For KV head 1 of an FP8 page (8,192
    bytes per head record): K codes at 8192 + 5*256; V codes at 8192 + 4096 +
    2*512 + 2d + 1 (the odd slot's bytes of pair 2)."""
    pool = PG.new_pool(12, PG.FP8, 4, D)
    assert pool.shape == (12, 32768)
    k = np.zeros((1, 4, D))
    v = np.zeros((1, 4, D))
    k[0, 1, :] = 1.0                      # 1.0 / g with g = 0.5 -> 2.0 = E4M3 0x40
    v[0, 1, :] = -0.75                    # -0.75 / 0.25 = -3.0 -> 0xC4
    PG.scatter_tokens(pool, PG.FP8, 4, D, np.array([[5, 2, 9]]), [0], [37], k, v, 0.5, 0.25)
    nz = np.flatnonzero(pool.reshape(-1))
    assert set(nz // 32768) == {9}
    off = nz % 32768
    kc = set(range(8192 + 1280, 8192 + 1536))
    vc = set(8192 + 4096 + 1024 + 2 * d + 1 for d in range(D))
    assert set(off) == kc | vc
    assert np.all(pool[9, 8192 + 1280: 8192 + 1536] == 0x40)
    assert np.all(pool[9, 8192 + 4096 + 1024 + 1: 8192 + 4096 + 1536: 2] == 0xC4)
    # the even slot of the same pair fills the other byte of each 2-byte pair
    v[0, 1, :] = 0.5                      # 0.5 / 0.25 = 2.0 -> 0x40
    PG.scatter_tokens(pool, PG.FP8, 4, D, np.array([[5, 2, 9]]), [0], [36], k, v, 0.5, 0.25)
    assert np.all(pool[9, 8192 + 4096 + 1024: 8192 + 4096 + 1536: 2] == 0x40)
    assert np.all(pool[9, 8192 + 4096 + 1024 + 1: 8192 + 4096 + 1536: 2] == 0xC4)
