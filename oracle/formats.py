"""Element codecs: E2M1 (FP4), E4M3FN (FP8) and bf16, written from the format
definitions.  Test infrastructure only (see ``oracle/__init__.py``).

NVFP4 stores each KV element as an E2M1 code with one E4M3 scale per 16
elements ("262,144 Tokens on One RTX 5090 ...", section "Why NVFP4 KV changes
the math"; the block size and scale type are the ones of the NVFP4 format the
page names).  The codecs below follow the OCP definitions:

E2M1: 1 sign bit (bit 3), 2 exponent bits (bits 2..1), 1 mantissa bit (bit 0),
      exponent bias 1, no infinities or NaN.  Exponent field 0 is subnormal:
      value = m * 2**-1.  Otherwise value = 2**(e-1) * (1 + m/2).
      Magnitudes: 0, 0.5, 1, 1.5, 2, 3, 4, 6.
E4M3FN: 1 sign bit (bit 7), 4 exponent bits, 3 mantissa bits, bias 7.
      Exponent field 0 is subnormal: value = m * 2**-9.  Otherwise
      value = 2**(e-7) * (1 + m/8).  S.1111.111 is NaN; there are no
      infinities; the largest finite magnitude is 448.

Rounding to either format is round-to-nearest, ties to an even mantissa bit,
with saturation to the largest finite magnitude ("satfinite").  The sign of a
value that rounds to zero is kept (a negative input gives the negative-zero
code), as IEEE-style conversions do.
"""
import numpy as np

E2M1_MAX = 6.0
E4M3_MAX = 448.0


def e2m1_decode(codes):
    """E2M1 code (0..15, any integer array) -> float64 value."""
    c = np.asarray(codes).astype(np.int64) & 0xF
    sign = np.where(c & 0x8, -1.0, 1.0)
    e = (c >> 1) & 0x3
    m = c & 0x1
    mag = np.where(e == 0, 0.5 * m, np.ldexp(1.0 + 0.5 * m, (e - 1).astype(np.int32)))
    return sign * mag


def e4m3_decode(codes):
    """E4M3FN byte (0..255) -> float64 value; NaN codes decode to NaN."""
    c = np.asarray(codes).astype(np.int64) & 0xFF
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    mag = np.where(e == 0, m * 2.0 ** -9,
                   np.ldexp(1.0 + m / 8.0, (e - 7).astype(np.int32)))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return sign * mag


def _round_to_format(x, mant_bits, emin, maxval):
    """Round |x| (float64 array, values exactly representable in float64) to the
    nearest value with ``mant_bits`` fraction bits whose binade exponent is at
    least ``emin`` (subnormals below 2**emin), ties to even, saturating to
    ``maxval``.  Returns the rounded magnitude as float64 (exact)."""
    a = np.abs(np.asarray(x, dtype=np.float64))
    # exponent of the binade containing a (a = f * 2**k, 0.5 <= f < 1)
    _, k = np.frexp(a)
    e = np.maximum(k - 1, emin)
    quantum = np.ldexp(1.0, (e - mant_bits).astype(np.int32))
    # a / quantum is exact (power-of-two division); rint is round-half-even
    q = np.rint(a / quantum) * quantum
    q = np.where(a == 0.0, 0.0, q)
    return np.minimum(q, maxval)


def e2m1_encode(x):
    """float values -> E2M1 codes, RNE with satfinite; sign of zero kept."""
    x = np.asarray(x, dtype=np.float64)
    mag = _round_to_format(x, mant_bits=1, emin=0, maxval=E2M1_MAX)
    # magnitude -> code via the format definition's value list
    table = e2m1_decode(np.arange(8))
    idx = np.searchsorted(table, mag)
    assert np.all(table[np.minimum(idx, 7)] == mag), "e2m1 rounding off-grid"
    sign = np.signbit(x).astype(np.int64) << 3
    return (idx.astype(np.int64) | sign).astype(np.uint8)


def e4m3_encode(x):
    """float values -> E4M3FN bytes, RNE with satfinite; sign of zero kept."""
    x = np.asarray(x, dtype=np.float64)
    mag = _round_to_format(x, mant_bits=3, emin=-6, maxval=E4M3_MAX)
    table = e4m3_decode(np.arange(127))          # all finite non-negative codes
    idx = np.searchsorted(table, mag)
    assert np.all(table[np.minimum(idx, 126)] == mag), "e4m3 rounding off-grid"
    sign = np.signbit(x).astype(np.int64) << 7
    return (idx.astype(np.int64) | sign).astype(np.uint8)


def f32(x):
    """Round float64 values to IEEE binary32 (round to nearest even)."""
    return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)


def bf16_round(x):
    """Round binary32-representable values to bfloat16 (RNE), returned as
    float64.  bf16 keeps the top 16 bits of the binary32 encoding; the
    discarded low half rounds to nearest, ties to an even kept half."""
    u = np.asarray(x, dtype=np.float64).astype(np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) & 0xFFFF0000).astype(np.uint32)
    return r.view(np.float32).astype(np.float64)


def bf16_bits(x):
    """bf16-representable float values -> their 16-bit encodings (uint16)."""
    u = np.asarray(x, dtype=np.float64).astype(np.float32).view(np.uint32)
    assert np.all((u & 0xFFFF) == 0), "value is not bf16-representable"
    return (u >> 16).astype(np.uint16)


def bf16_from_bits(b):
    """16-bit bf16 encodings -> float64 values."""
    u = np.asarray(b).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)
