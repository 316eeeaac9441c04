"""Pins for the NVFP4-query prefill reading (oracle/fp4_prefill.py).

Pinned against: the plain dot product of the dequantised operands (the
blockwise block-scaled form must equal it), exactness of the block sums and
of their scaling in binary32 (exhaustive over the E4M3 scale pairs), queries
that are exactly NVFP4-representable (the reading then reduces to the plain
attention), and a brute-force softmax built on the blockwise logits.
"""
import math

import numpy as np

from oracle import fp4_prefill as F
from oracle import nvfp4 as N
from oracle.attention import attention_dense
from oracle.formats import bf16_round, e2m1_decode, e4m3_decode, f32

D = 256


def _finite_scale_bytes(rng, shape):
    b = rng.integers(0, 127, shape)            # 0x00 .. 0x7E: finite, non-negative
    return b.astype(np.uint8)


def test_block_scaled_dot_equals_plain_dot():
    rng = np.random.default_rng(41)
    for trial in range(20):
        R, L = 5, 7
        qc = rng.integers(0, 16, (R, D)).astype(np.uint8)
        kc = rng.integers(0, 16, (L, D)).astype(np.uint8)
        qs = _finite_scale_bytes(rng, (R, D // 16))
        ks = _finite_scale_bytes(rng, (L, D // 16))
        g_q = float(np.float32(rng.uniform(1e-4, 1e-1)))
        g_k = float(np.float32(rng.uniform(1e-4, 1e-1)))
        got = F.block_scaled_dot(qc, qs, g_q, kc, ks, g_k)
        want = N.dequantize(qc, qs, g_q) @ N.dequantize(kc, ks, g_k).T
        assert np.allclose(got, want, rtol=1e-12, atol=1e-300)
        # a scale taken from the wrong block changes the result
        ks_shift = np.roll(ks, 1, axis=1)
        if not np.array_equal(ks_shift, ks):
            assert not np.allclose(F.block_scaled_dot(qc, qs, g_q, kc, ks_shift, g_k), want)


def test_block_sums_and_scaling_exact_in_binary32():
    rng = np.random.default_rng(42)
    blocks = [np.full(16, 7), np.full(16, 15), rng.integers(0, 16, 16), rng.integers(0, 16, 16)]
    other = [np.full(16, 7), np.full(16, 7), rng.integers(0, 16, 16), rng.integers(0, 16, 16)]
    sums = [float(np.sum(e2m1_decode(a) * e2m1_decode(b))) for a, b in zip(blocks, other)]
    assert sums[0] == 576.0 and sums[1] == -576.0
    s = e4m3_decode(np.arange(127))                       # every finite non-negative scale
    pair = (s[:, None] * s[None, :]).reshape(-1)
    for b in sums:
        assert f32(b) == b and (4 * b) == int(4 * b)
        prod = b * pair
        assert np.array_equal(f32(prod), prod)


def test_representable_queries_reduce_to_plain_attention():
    rng = np.random.default_rng(43)
    g_q = 2.0 ** -7
    R, L = 6, 40
    codes = rng.integers(0, 16, (R, D))
    sc = rng.integers(40, 110, (R, D // 16))
    codes[:, ::16] = 7                                     # one |value| = 6 per block
    q = (e2m1_decode(codes).reshape(R, D // 16, 16) * e4m3_decode(sc)[..., None]).reshape(R, D) * g_q
    assert np.array_equal(bf16_round(q), q)
    assert np.array_equal(F.dequantized_queries(q, g_q), q)
    k = bf16_round(rng.standard_normal((L, D)))
    v = bf16_round(rng.standard_normal((L, D)))
    vis = np.array([40, 33, 1, 17, 40, 2])
    o1, l1 = F.prefill_attention_fp4q(q, g_q, k, v, 1 / 16, vis)
    o2, l2 = attention_dense(q, k, v, 1 / 16, vis)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_softmax_over_blockwise_logits_brute_force():
    """Tiny case: quantise q and K, take the logits from the blockwise form,
    do the softmax and P.V with explicit loops; the oracle must agree."""
    rng = np.random.default_rng(44)
    R, L = 3, 9
    q = bf16_round(rng.standard_normal((R, D)) * 2.0)
    k = bf16_round(rng.standard_normal((L, D)))
    v = bf16_round(rng.standard_normal((L, D)))
    g_q = float(np.float32(np.max(np.abs(q)) / (6 * 448)))
    g_k = float(np.float32(np.max(np.abs(k)) / (6 * 448)))
    qc, qs = F.quantize_queries(q, g_q)
    kc, ks = N.quantize(k, g_k)
    k_hat = N.dequantize(kc, ks, g_k)
    z = F.block_scaled_dot(qc, qs, g_q, kc, ks, g_k) / 16.0
    vis = [9, 4, 1]
    o_bf = np.zeros((R, D))
    lse_bf = np.zeros(R)
    for r in range(R):
        m = max(z[r, t] for t in range(vis[r]))
        w = [math.exp(z[r, t] - m) for t in range(vis[r])]
        ssum = sum(w)
        for t in range(vis[r]):
            o_bf[r] += (w[t] / ssum) * v[t]
        lse_bf[r] = m + math.log(ssum)
    o, lse = F.prefill_attention_fp4q(q, g_q, k_hat, v, 1 / 16, np.array(vis))
    assert np.max(np.abs(o - o_bf)) < 1e-12 and np.max(np.abs(lse - lse_bf)) < 1e-12
    # and the query quantisation is really applied: the plain attention differs
    o_plain, _ = attention_dense(q, k_hat, v, 1 / 16, np.array(vis))
    assert np.max(np.abs(o_plain - o)) > 1e-6
