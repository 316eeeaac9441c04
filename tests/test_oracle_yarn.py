"""Pins for the oracle's YaRN frequencies, tables and rope.

Pinned against: the values the pages print (tests/golden/yarn_pins.json), the
closed form s = 1 (plain RoPE), the defining property of the correction
dimension (a pair at that index turns exactly beta times over the window),
unit-vector rotations compared with libm cos/sin, the rotation's norm
(times mscale), and the relative-position property of rotary logits.
"""
import json
import math
import os

import numpy as np
import pytest

from oracle import yarn as Y
from oracle.formats import bf16_round, f32

HERE = os.path.dirname(os.path.abspath(__file__))
P = dict(theta=1.0e7, factor=4.0, original_max=262144, beta_fast=32.0, beta_slow=1.0,
         rotary_dim=64, deployed=True)


def _pins():
    with open(os.path.join(HERE, "golden", "yarn_pins.json")) as f:
        return {p["name"]: p for p in json.load(f)["pins"]}


def test_correction_ranges_match_pages():
    pins = _pins()
    dep = Y.correction_range(1e7, 4.0, 262144, 32.0, 1.0, 64, deployed=True)
    txt = Y.correction_range(1e7, 4.0, 262144, 32.0, 1.0, 64, deployed=False)
    assert list(dep) == pins["correction_range_deployed"]["value"]
    assert list(txt) == pins["correction_range_textbook"]["value"]


def test_mscale_matches_page_and_closed_form():
    pin = _pins()["mscale_x4"]
    m = Y.mscale(4.0)
    assert round(m, pin["decimals"]) == pin["value"]
    assert m == 0.1 * math.log(4.0) + 1.0
    assert Y.mscale(1.0) == 1.0


def test_correction_dim_turns_beta_times():
    # A pair i rotates by theta**(-2i/R) rad per position; over L positions
    # it turns L * theta**(-2i/R) / (2 pi) times.  At the correction dimension
    # for beta that count is beta (the definition the formula inverts).
    for beta in (32.0, 1.0, 7.5):
        for L in (262144, 4 * 262144):
            d = Y.correction_dim(beta, 64, 1e7, L)
            turns = L * 1e7 ** (-2.0 * d / 64) / (2 * math.pi)
            assert abs(turns - beta) < 1e-9 * beta


def test_factor_one_is_plain_rope():
    q = dict(P, factor=1.0)
    f = Y.inv_freq(q["theta"], 1.0, q["original_max"], q["beta_fast"], q["beta_slow"], 64)
    plain = np.array([1e7 ** (-2.0 * i / 64) for i in range(32)])
    assert np.allclose(f, plain, rtol=1e-15, atol=0)
    cos_t, sin_t = Y.rope_tables(q, 300)
    p = np.arange(300)[:, None]
    assert np.max(np.abs(cos_t - np.cos(p * plain))) <= 2 ** -24
    assert np.max(np.abs(sin_t - np.sin(p * plain))) <= 2 ** -24


def test_inv_freq_regions():
    f = Y.inv_freq(**{k: P[k] for k in ("theta", "factor", "original_max", "beta_fast",
                                        "beta_slow", "rotary_dim")})
    orig = np.array([1e7 ** (-2.0 * i / 64) for i in range(32)])
    # below the range: original frequency; above it: divided by the factor
    assert np.array_equal(f[:17], orig[:17])
    assert np.allclose(f[24:], orig[24:] / 4.0, rtol=1e-15, atol=0)
    # middle of the range (16, 24): pair 20 sits halfway on the ramp,
    # 0.5 * f/4 + 0.5 * f = 0.625 f
    assert abs(f[20] / orig[20] - 0.625) < 1e-15
    # pair 18 is a quarter up the ramp: 0.25 * f/4 + 0.75 * f = 0.8125 f
    assert abs(f[18] / orig[18] - 0.8125) < 1e-15
    assert np.all(np.diff(f) < 0)


def test_textbook_range_shifts_the_ramp():
    f = Y.inv_freq(1e7, 4.0, 262144, 32.0, 1.0, 64, deployed=False)
    orig = np.array([1e7 ** (-2.0 * i / 64) for i in range(32)])
    assert np.array_equal(f[:15], orig[:15])
    assert np.allclose(f[22:], orig[22:] / 4.0, rtol=1e-15, atol=0)
    assert abs(f[18] / orig[18] - 0.625) < 1e-15


def test_table_values_pair0_is_libm():
    cos_t, sin_t = Y.rope_tables(P, 5000)
    m = Y.mscale(4.0)
    for p in (0, 1, 17, 4095, 4999):
        assert cos_t[p, 0] == float(np.float32(m * math.cos(p)))
        assert sin_t[p, 0] == float(np.float32(m * math.sin(p)))
    # cos^2 + sin^2 = m^2 up to binary32 rounding
    r = cos_t ** 2 + sin_t ** 2
    assert np.max(np.abs(r - m * m)) < 4 * 2 ** -23 * m * m


def test_rope_unit_vectors():
    """e_j at position p rotates in the (j, j+32) plane: out[j] = c, out[j+32] = s
    (rotate-half convention), everything else untouched, rounded to bf16."""
    cos_t, sin_t = Y.rope_tables(P, 1000)
    for j in (0, 5, 31):
        x = np.zeros((1, 1, 256))
        x[0, 0, j] = 1.0
        out = Y.rope_rows(x, np.array([777]), cos_t, sin_t, 64)[0, 0]
        assert out[j] == bf16_round(cos_t[777, j])
        assert out[j + 32] == bf16_round(sin_t[777, j])
        assert np.count_nonzero(out) == 2
        y = np.zeros((1, 1, 256))
        y[0, 0, j + 32] = 1.0
        out = Y.rope_rows(y, np.array([777]), cos_t, sin_t, 64)[0, 0]
        assert out[j] == bf16_round(-sin_t[777, j])
        assert out[j + 32] == bf16_round(cos_t[777, j])
    # dims 64..255 pass through
    z = bf16_round(np.random.default_rng(3).standard_normal((4, 2, 256)))
    out = Y.rope_rows(z, np.array([1, 2, 3, 999]), cos_t, sin_t, 64)
    assert np.array_equal(out[..., 64:], z[..., 64:])


def test_rope_norm_scaled_by_mscale():
    rng = np.random.default_rng(4)
    cos_t, sin_t = Y.rope_tables(P, 70000)
    x = bf16_round(rng.standard_normal((50, 3, 256)))
    pos = rng.integers(0, 70000, 50)
    out = Y.rope_rows(x, pos, cos_t, sin_t, 64)
    n0 = np.linalg.norm(x[..., :64], axis=-1)
    n1 = np.linalg.norm(out[..., :64], axis=-1)
    assert np.max(np.abs(n1 / n0 - Y.mscale(4.0))) < 3e-3    # bf16 output rounding


def test_rope_logits_depend_on_relative_position():
    rng = np.random.default_rng(5)
    cos_t, sin_t = Y.rope_tables(P, 1 << 20)
    q = bf16_round(rng.standard_normal((1, 1, 256)))
    k = bf16_round(rng.standard_normal((1, 1, 256)))
    ref = None
    for shift in (0, 1000, 500000, 1048000):
        qa = Y.rope_rows(q, np.array([100 + shift]), cos_t, sin_t, 64)[0, 0, :64]
        ka = Y.rope_rows(k, np.array([40 + shift]), cos_t, sin_t, 64)[0, 0, :64]
        z = float(qa @ ka)
        if ref is None:
            ref = z
        assert abs(z - ref) < 0.05 * (1 + abs(ref))   # bf16 rounding of both vectors
    # and a different relative offset gives a clearly different logit
    qa = Y.rope_rows(q, np.array([100]), cos_t, sin_t, 64)[0, 0, :64]
    kb = Y.rope_rows(k, np.array([90]), cos_t, sin_t, 64)[0, 0, :64]
    assert abs(float(qa @ kb) - ref) > 0.1
