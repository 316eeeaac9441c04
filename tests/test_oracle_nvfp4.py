"""Pins for the oracle's two-level NVFP4 block quantiser.

Pinned against: exact round trips of blocks built from representable values,
the zero block, a brute-force choice of every element code and block scale
(nearest representable value, searched exhaustively), the per-element error
bound the rounding implies, and the nibble packing order.
"""
import numpy as np
import pytest

from oracle import nvfp4 as N
from oracle.formats import bf16_round, e2m1_decode, e4m3_decode, f32

E2M1_MAGS = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def _nearest_code(y):
    """Exhaustive nearest E2M1 code of a binary32 value (ties: even code)."""
    best, bestd = None, None
    for c in range(8):
        d = abs(abs(y) - E2M1_MAGS[c])
        if bestd is None or d < bestd or (d == bestd and c % 2 == 0):
            best, bestd = c, d
    if abs(y) > 6.0:
        best = 7
    return best | (8 if np.signbit(y) else 0)


def test_representable_blocks_roundtrip_exactly():
    rng = np.random.default_rng(11)
    for trial in range(300):
        g = 2.0 ** int(rng.integers(-12, 2))              # power-of-two tensor scale
        s_code = int(rng.integers(8, 120))                # a normal E4M3 scale
        s = float(e4m3_decode(s_code))
        codes = rng.integers(0, 16, 16)
        codes[int(rng.integers(0, 16))] = 7 | (8 * int(rng.integers(0, 2)))   # one |value| = 6
        x = e2m1_decode(codes) * s * g
        assert np.array_equal(bf16_round(x), x)            # the block is bf16-representable
        q, sc = N.quantize(x[None, :], g)
        assert int(sc[0, 0]) == s_code
        # values equal to +-0 may come back as either zero code; compare values
        xh = N.dequantize(q, sc, g)[0]
        assert np.array_equal(xh, x), trial


def test_zero_block():
    q, s = N.quantize(np.zeros((3, 32)), 0.01)
    assert not q.any() and not s.any()
    assert not N.dequantize(q, s, 0.01).any()


def test_block_too_small_for_scale_is_zero():
    g = 1.0
    x = np.full((1, 16), 2.0 ** -20)                      # a * e far below 2**-10
    q, s = N.quantize(x, g)
    assert not q.any() and not s.any()


def test_codes_and_scales_match_brute_force():
    rng = np.random.default_rng(12)
    g = float(np.float32(0.0031))
    x = bf16_round(rng.standard_normal((40, 64)) * np.exp(rng.uniform(-3, 3, (40, 1))))
    q, s = N.quantize(x, g)
    e = float(f32(1.0 / (6.0 * g)))
    for r in range(40):
        for b in range(4):
            blk = x[r, 16 * b:16 * b + 16]
            a = np.max(np.abs(blk))
            target = float(f32(a * e))
            # exhaustive nearest E4M3 (ties to even code, saturating at 448)
            vals = e4m3_decode(np.arange(127))
            d = np.abs(vals - target)
            cands = np.flatnonzero(d == d.min())
            want_s = int(cands[0] if len(cands) == 1 else cands[cands % 2 == 0][0])
            if target >= 448.0:
                want_s = 126
            assert int(s[r, b]) == want_s
            dec = float(f32(vals[want_s] * g))
            rcp = float(f32(1.0 / dec))
            for i in range(16):
                y = float(f32(blk[i] * rcp))
                assert int(q[r, 16 * b + i]) == _nearest_code(y), (r, b, i)


def test_error_bound():
    """|x - x_hat| <= d * half the E2M1 step at |x|/d, plus the saturation
    overshoot when the block scale rounded down (bounded by the E4M3 relative
    rounding, 1/16 of 6 d)."""
    rng = np.random.default_rng(13)
    g = float(np.float32(0.01))                        # keeps every block scale normal
    x = bf16_round(rng.standard_normal((200, 256)) * 3.0)
    q, s = N.quantize(x, g)
    xh = N.dequantize(q, s, g)
    d = np.repeat(e4m3_decode(s) * g, 16, axis=-1)
    y = np.abs(x) / d
    half_step = np.where(y < 2, 0.25, np.where(y < 4, 0.5, 1.0))
    over = np.maximum(y - 6.0, 0.0)
    assert np.all(np.abs(x - xh) <= d * (half_step + over) * (1 + 1e-6))
    assert np.all(over <= 6.0 / 16 + 1e-6)


def test_nibble_packing_order():
    codes = np.array([[1, 2, 3, 4, 15, 0, 8, 7]])
    packed = N.pack_nibbles(codes)
    assert list(packed[0]) == [0x21, 0x43, 0x0F, 0x78]
    assert np.array_equal(N.unpack_nibbles(packed), codes)


def test_encode_scale_is_one_rounding():
    for g in (1.0, 0.1, 3.7e-4, 1.2345e-3):
        g32 = float(np.float32(g))
        e = N.encode_scale(g)
        assert e == float(np.float32(1.0 / (6.0 * g32)))
