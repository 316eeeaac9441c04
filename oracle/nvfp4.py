"""Two-level NVFP4 block quantisation of KV rows.  Test infrastructure only
(see ``oracle/__init__.py``).

The page "262,144 Tokens on One RTX 5090 ...", sections "Why NVFP4 KV
changes the math" and "The stack, for the impatient", quantises the KV cache
itself to NVFP4: E2M1 element codes with an FP8 E4M3 scale per 16 contiguous
elements, and one binary32 scale per tensor.  The page is silent on the
encoder arithmetic; the reading used here (the standard two-level NVFP4
recipe) fixes every rounding point so that a GPU encoder can match it bit for
bit:

  g    caller-given per-tensor *decode* scale (binary32, > 0)
  e    = fp32(1 / (6 * g))                  (one rounding, computed in float64)
  a    = max |x_i| over the 16-element block (exact)
  S    = E4M3_RNE_satfinite( fp32(a * e) )
  if decode(S) == 0: all 16 codes are +0 and the scale byte is 0
  d    = fp32(decode(S) * g)
  r    = fp32(1 / d)
  q_i  = E2M1_RNE_satfinite( fp32(x_i * r) )

and dequantisation is x_hat_i = E2M1(q_i) * decode(S) * g, exact in float64.
Element 2k of a block is stored in the low nibble of byte k, element 2k+1 in
the high nibble.

Every binary32 rounding is emulated by a float64 operation on
binary32-representable operands followed by one rounding to binary32; for
+, -, *, / this equals the correctly rounded binary32 result because float64
carries more than 2*24 + 2 significand bits (double rounding is innocuous).
"""
import numpy as np

from .formats import e2m1_decode, e2m1_encode, e4m3_decode, e4m3_encode, f32

BLOCK = 16


def encode_scale(g):
    """e = fp32(1 / (6 g)) for a binary32 per-tensor decode scale g."""
    g = float(np.float32(g))
    return float(f32(1.0 / (6.0 * g)))


def quantize(x, g):
    """Quantise rows of bf16-valued ``x`` [..., D] (D a multiple of 16).

    Returns (codes uint8 [..., D] with values 0..15, scales uint8 [..., D/16])."""
    x = np.asarray(x, dtype=np.float64)
    g = float(np.float32(g))
    e = encode_scale(g)
    shp = x.shape
    blocks = x.reshape(*shp[:-1], shp[-1] // BLOCK, BLOCK)
    a = np.max(np.abs(blocks), axis=-1)
    s_byte = e4m3_encode(f32(a * e))
    s_val = e4m3_decode(s_byte)
    zero = s_val == 0.0
    d = f32(s_val * g)
    d_safe = np.where(zero, 1.0, d)
    r = f32(1.0 / d_safe)
    q = e2m1_encode(f32(blocks * r[..., None]))
    q = np.where(zero[..., None], 0, q).astype(np.uint8)
    s_byte = np.where(zero, 0, s_byte).astype(np.uint8)
    return q.reshape(shp), s_byte


def dequantize(codes, scales, g):
    """x_hat = E2M1(code) * E4M3(scale) * g, float64, shape of ``codes``."""
    codes = np.asarray(codes)
    shp = codes.shape
    vals = e2m1_decode(codes).reshape(*shp[:-1], shp[-1] // BLOCK, BLOCK)
    s = e4m3_decode(scales)[..., None]
    return (vals * s * float(np.float32(g))).reshape(shp)


def pack_nibbles(codes):
    """codes [..., D] (0..15) -> bytes [..., D/2]; element 2k low nibble."""
    c = np.asarray(codes).astype(np.uint8)
    return (c[..., 0::2] | (c[..., 1::2] << 4)).astype(np.uint8)


def unpack_nibbles(packed):
    """bytes [..., D/2] -> codes [..., D]."""
    p = np.asarray(packed).astype(np.uint8)
    out = np.empty(p.shape[:-1] + (p.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = p & 0xF
    out[..., 1::2] = p >> 4
    return out
