"""YaRN rotary scaling: inverse frequencies, attention temperature, cos/sin
tables and rope.  Test infrastructure only (see ``oracle/__init__.py``).

What the pages fix:
* "A 1,048,576-token context on two RTX 5090s ...", section "YaRN, and
  matching what vLLM actually does": the deployed stack multiplies the
  original context length by the scaling factor before it computes the
  correction range, which gives the range (16, 24) instead of the (14, 22)
  the published formula gives for the same parameters; mscale is applied
  inside the rope on the rotary dimensions and there is no other
  attention-level scale.
* "ninfer-windows-tp2" README, section "YaRN reference and drift guard":
  range (16, 24), mscale 1.13863 applied to cos/sin over the 64 rotary
  dimensions of each 256-dimension head.
* The published YaRN method (Peng et al., 2023), NTK-by-parts section: the
  correction dimension of a wavelength ratio, the floor/ceil range, the linear
  ramp over pair indices, the blend of interpolated and original frequencies,
  and the temperature 0.1*ln(s) + 1.

Readings where the pages are silent: rotate-half pairing (j, j + R/2) within
the first R dims; the angle p*inv_freq is formed in float64 and cos/sin are
evaluated in float64, times mscale, rounded once to binary32; rope arithmetic
is binary32 with one rounding per product and per sum, then the result is
rounded to bf16.
"""
import math

import numpy as np

from .formats import bf16_round, f32


def correction_dim(n_rot, rotary_dim, theta, context_len):
    """Pair-index position at which a rotation count ``n_rot`` over
    ``context_len`` positions is reached (YaRN, NTK-by-parts):
    R * ln(L / (2*pi*n)) / (2 * ln(theta))."""
    return rotary_dim * math.log(context_len / (n_rot * 2.0 * math.pi)) / (2.0 * math.log(theta))


def correction_range(theta, factor, original_max, beta_fast, beta_slow, rotary_dim,
                     deployed=True):
    """(low, high) pair indices of the ramp.  ``deployed=True`` uses
    original_max * factor as the context length (the range the serving stack
    actually used); ``deployed=False`` uses original_max (the paper's)."""
    ctx = original_max * factor if deployed else original_max
    low = math.floor(correction_dim(beta_fast, rotary_dim, theta, ctx))
    high = math.ceil(correction_dim(beta_slow, rotary_dim, theta, ctx))
    return max(low, 0), min(high, rotary_dim - 1)


def mscale(factor):
    """YaRN attention temperature: 0.1 * ln(s) + 1 for s > 1, else 1."""
    return 1.0 if factor <= 1.0 else 0.1 * math.log(factor) + 1.0


def inv_freq(theta, factor, original_max, beta_fast, beta_slow, rotary_dim, deployed=True):
    """float64 inverse frequency of each rotary pair i = 0 .. R/2 - 1."""
    half = rotary_dim // 2
    i = np.arange(half, dtype=np.float64)
    # original ("extrapolation") frequency theta**(-2i/R), one libm pow each
    f_orig = np.array([math.pow(theta, -2.0 * k / rotary_dim) for k in range(half)])
    f_interp = f_orig / factor
    low, high = correction_range(theta, factor, original_max, beta_fast, beta_slow,
                                 rotary_dim, deployed)
    if low == high:
        high = high + 0.001
    ramp = np.clip((i - low) / (high - low), 0.0, 1.0)
    keep_orig = 1.0 - ramp            # 1 below the range, 0 above it
    return f_interp * (1.0 - keep_orig) + f_orig * keep_orig


def rope_tables(params, max_pos):
    """cos/sin tables, binary32 values in float64 arrays of shape
    [max_pos, R/2]: table[p, i] = fp32(mscale * cos(p * inv_freq_i))."""
    f = inv_freq(params["theta"], params["factor"], params["original_max"],
                 params["beta_fast"], params["beta_slow"], params["rotary_dim"],
                 params.get("deployed", True))
    m = mscale(params["factor"])
    p = np.arange(max_pos, dtype=np.float64)[:, None]
    ang = p * f[None, :]
    return f32(m * np.cos(ang)), f32(m * np.sin(ang))


def rope_rows(x, pos, cos_t, sin_t, rotary_dim):
    """Apply rope to bf16-valued ``x`` of shape [n, ..., D] (first axis:
    tokens) at positions ``pos`` [n] with binary32 tables; returns
    bf16-rounded float64 values of the same shape.

    For pair j < R/2 (partner j + R/2), at table row p:
      x'_j       = fp32( fp32(x_j * c) - fp32(x_{j+R/2} * s) )
      x'_{j+R/2} = fp32( fp32(x_{j+R/2} * c) + fp32(x_j * s) )
    then every element is rounded to bf16; dims >= R pass through."""
    x = np.asarray(x, dtype=np.float64)
    pos = np.asarray(pos, dtype=np.int64)
    half = rotary_dim // 2
    shape = [len(pos)] + [1] * (x.ndim - 2) + [half]
    c = cos_t[pos].reshape(shape)
    s = sin_t[pos].reshape(shape)
    lo = x[..., :half]
    hi = x[..., half:rotary_dim]
    out = x.copy()
    out[..., :half] = f32(f32(lo * c) - f32(hi * s))
    out[..., half:rotary_dim] = f32(f32(hi * c) + f32(lo * s))
    return bf16_round(out)
