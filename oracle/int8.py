"""INT8 group-64 KV: symmetric 8-bit codes with one fp16 scale per 64
contiguous elements.  Test infrastructure only (see ``oracle/__init__.py``).

"NInfer -- Windows 11 TP2 fork" README, sections "Dual-GPU (TP2) and YaRN
1M context" and "Memory, per GPU": the 1M-token configuration stores the KV
cache as INT8 group-64 and the pool is 16.5 KiB per token per device,
quantisation-scale planes included.  With 16 full-attention layers, 2 KV
heads per device, K and V, and a 256-dim head that is 16 KiB of codes plus
512 B of scales, i.e. one 2-byte scale per 64-element group: fp16 here.
The page gives no encoder arithmetic; the reading used here is symmetric
absmax scaling, every rounding point fixed:

  a    = max |x_i| over the 64-element group (exact)
  s    = fp16_RNE_satfinite( fp32(a / 127) )
  if s == 0: all 64 codes are 0 and the scale is +0
  d    = fp32(s)                            (exact)
  r    = fp32(1 / d)
  q_i  = clamp( RNE( fp32(x_i * r) ), -127, 127 )

and dequantisation is x_hat_i = q_i * d, exact in float64.
"""
import numpy as np

from .formats import f32

GROUP = 64
QMAX = 127
F16_MAX = 65504.0


def f16_round(x):
    """Round binary32-representable float64 values to binary16 (RNE),
    saturating to +-65504; returned as float64."""
    x = np.asarray(x, dtype=np.float64)
    h = np.clip(x, -F16_MAX, F16_MAX).astype(np.float16)
    # numpy's float64 -> float16 cast rounds to nearest even; values
    # between 65504 and 65520 would round to inf without the clip
    return h.astype(np.float64)


def quantize(x, group=GROUP):
    """bf16-valued ``x`` [..., D] (D a multiple of 64) -> (codes int8 [..., D],
    scales as float16 bit patterns uint16 [..., D/64])."""
    x = np.asarray(x, dtype=np.float64)
    shp = x.shape
    g = x.reshape(*shp[:-1], shp[-1] // group, group)
    a = np.max(np.abs(g), axis=-1)
    s = f16_round(f32(a / QMAX))
    zero = s == 0.0
    d = np.where(zero, 1.0, s)             # fp16 values are exact in binary32
    r = f32(1.0 / d)
    q = np.rint(f32(g * r[..., None]))     # rint rounds half to even
    q = np.clip(q, -QMAX, QMAX)
    q = np.where(zero[..., None], 0, q).astype(np.int8)
    s = np.where(zero, 0.0, s)
    return q.reshape(shp), s.astype(np.float16).view(np.uint16)


def dequantize(codes, scale_bits, group=GROUP):
    """x_hat = q * d (float64), shape of ``codes``."""
    codes = np.asarray(codes).astype(np.int8).astype(np.float64)
    shp = codes.shape
    d = np.asarray(scale_bits, dtype=np.uint16).view(np.float16).astype(np.float64)
    return (codes.reshape(*shp[:-1], shp[-1] // group, group) * d[..., None]).reshape(shp)
