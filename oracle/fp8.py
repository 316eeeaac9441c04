"""FP8 (E4M3) KV with one binary32 scale per tensor.  Test infrastructure only
(see ``oracle/__init__.py``).

The page "A 1,048,576-token context on two RTX 5090s", section "Against vLLM:
prefill loses, decode wins, and one surprise", runs the comparison engine
with an fp8 KV cache: every K and V element is one E4M3 byte, with one scale
per tensor.  The page is silent on the encoder arithmetic; the reading used
here takes the same steps as this library's NVFP4 encoder (a caller-given
binary32 *decode* scale g, multiplication by its correctly rounded
reciprocal, E4M3 round-to-nearest-even with saturation):

  g    caller-given per-tensor decode scale (binary32, > 0)
  r    = fp32(1 / g)                        (one rounding, computed in float64)
  q_i  = E4M3_RNE_satfinite( fp32(x_i * r) )

and dequantisation is x_hat_i = E4M3(q_i) * g, exact in float64.  A negative
value that rounds to zero keeps its sign (code 0x80).
"""
import numpy as np

from .formats import e4m3_decode, e4m3_encode, f32


def reciprocal(g):
    """r = fp32(1 / g) for a binary32 per-tensor decode scale g."""
    g = float(np.float32(g))
    return float(f32(1.0 / g))


def quantize(x, g):
    """bf16-valued ``x`` [...] -> E4M3 codes (uint8, same shape)."""
    x = np.asarray(x, dtype=np.float64)
    return e4m3_encode(f32(x * reciprocal(g)))


def dequantize(codes, g):
    """x_hat = E4M3(code) * g (float64)."""
    return e4m3_decode(codes) * float(np.float32(g))
