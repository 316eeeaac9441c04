"""Pins for the oracle's attention, split-KV combine and paged gather.

Pinned against: a pure-Python triple loop on tiny inputs, closed forms (all
logits equal -> mean of V and LSE = ln n; V = 1 -> O = 1; one-hot V columns
-> the softmax weights, which sum to 1), split + combine == one pass,
causal row j == decode over its prefix, multi-chunk == single-chunk
evaluation, hand-computed byte offsets of the page layout, and invariance of
the paged result under a permutation of the pool's pages (bitwise).
"""
import math

import numpy as np
import pytest

from oracle import attention as A
from oracle import paged as PG
from oracle.formats import bf16_round

D = 256


def _rand(rng, *shape, scale=1.0):
    return bf16_round(rng.standard_normal(shape) * scale)


def test_dense_matches_brute_force():
    rng = np.random.default_rng(21)
    q, k, v = _rand(rng, 3, D), _rand(rng, 40, D), _rand(rng, 40, D)
    vis = [40, 17, 1]
    o1, l1 = A.attention_dense(q, k, v, 1 / 16, vis)
    o2, l2 = A.attention_brute_force(q.tolist(), k.tolist(), v.tolist(), 1 / 16, vis)
    assert np.max(np.abs(o1 - o2)) < 1e-12
    assert np.max(np.abs(l1 - l2)) < 1e-12


def test_closed_forms():
    rng = np.random.default_rng(22)
    n = 37
    k, v = _rand(rng, n, D), _rand(rng, n, D)
    o, lse = A.attention_dense(np.zeros((1, D)), k, v, 1 / 16)
    assert np.allclose(o[0], v.mean(axis=0), atol=1e-12)
    assert abs(lse[0] - math.log(n)) < 1e-12
    q = _rand(rng, 4, D)
    o, _ = A.attention_dense(q, k, np.ones((n, D)), 1 / 16)
    assert np.allclose(o, 1.0, atol=1e-12)
    # one-hot V columns recover the softmax weights; they sum to 1
    o, lse = A.attention_dense(q, k, np.eye(n, D), 1 / 16)
    w = o[:, :n]
    assert np.allclose(w.sum(axis=1), 1.0, atol=1e-12)
    z = (q @ k.T) / 16
    assert np.allclose(w, np.exp(z - lse[:, None]), atol=1e-12)


def test_no_visible_keys():
    o, lse = A.attention_dense(np.ones((1, D)), np.ones((3, D)), np.ones((3, D)), 1.0, [0])
    assert not o.any() and lse[0] == -math.inf


def test_split_then_combine_equals_one_pass():
    rng = np.random.default_rng(23)
    q, k, v = _rand(rng, 5, D), _rand(rng, 100, D, scale=2), _rand(rng, 100, D)
    vis = [100, 96, 97, 98, 99]
    o_ref, l_ref = A.attention_dense(q, k, v, 1 / 16, vis)
    for bounds in ([0, 100], [0, 16, 32, 48, 64, 80, 96, 100], [0, 97, 98, 100], [0, 50, 99, 100]):
        op, lp = A.split_attention(q, k, v, 1 / 16, vis, bounds)
        o, l = A.combine(op, lp)
        assert np.max(np.abs(o - o_ref)) < 1e-12
        assert np.max(np.abs(l - l_ref)) < 1e-12


def test_combine_ignores_empty_splits():
    rng = np.random.default_rng(24)
    op = rng.standard_normal((3, 2, D))
    lp = np.array([[0.5, -np.inf], [-np.inf, -np.inf], [1.5, 2.0]])
    o, l = A.combine(op, lp)
    w = np.exp(np.array([0.5, 1.5]) - 1.5)
    assert np.allclose(o[0], (w[0] * op[0, 0] + w[1] * op[2, 0]) / w.sum(), atol=1e-14)
    assert np.allclose(o[1], op[2, 1], atol=1e-14) and l[1] == 2.0
    o, l = A.combine(op[:2, :1], np.array([[-np.inf], [-np.inf]]))
    assert not o.any() and l[0] == -np.inf


def test_causal_rows_equal_prefix_decode():
    rng = np.random.default_rng(25)
    n, nq = 50, 5
    q, k, v = _rand(rng, nq, D), _rand(rng, n, D), _rand(rng, n, D)
    vis = [n - nq + j + 1 for j in range(nq)]
    o, l = A.attention_dense(q, k, v, 1 / 16, vis)
    for j in range(nq):
        oj, lj = A.attention_dense(q[j:j + 1], k[:vis[j]], v[:vis[j]], 1 / 16)
        assert np.max(np.abs(o[j] - oj[0])) < 1e-12 and abs(l[j] - lj[0]) < 1e-12


def test_chunked_equals_dense(monkeypatch):
    monkeypatch.setattr(A, "CHUNK", 7)
    rng = np.random.default_rng(26)
    q, k, v = _rand(rng, 4, D), _rand(rng, 45, D), _rand(rng, 45, D)
    vis = np.array([45, 44, 30, 1])
    o1, l1 = A.attention_dense(q, k, v, 1 / 16, vis)
    o2, l2 = A.attention_chunked(q, lambda s, e: (k[s:e], v[s:e]), 1 / 16, vis)
    assert np.max(np.abs(o1 - o2)) < 1e-12 and np.max(np.abs(l1 - l2)) < 1e-12


def test_page_layout_offsets_by_hand():
    """Token 37 of a sequence whose page table is [5, 2, 9] lives in page 9,
    slot 5.  For KV head 1 of an NVFP4 page (4,608 bytes per head record):
    K codes at 4608 + 5*128, K scales at 4608 + 2048 + 5*16, V codes in the
    high nibbles (odd slot) of slot pair 2 at 4608 + 2304 + 2*256, V scales at
    4608 + 4352 + 5*16."""
    pool = PG.new_pool(12, PG.NVFP4, 4, D)
    assert pool.shape == (12, 18432)
    k = np.zeros((1, 4, D))
    v = np.zeros((1, 4, D))
    k[0, 1, :] = 1.0
    v[0, 1, :] = -1.0
    PG.scatter_tokens(pool, PG.NVFP4, 4, D, np.array([[5, 2, 9]]), [0], [37], k, v, 1.0, 1.0)
    nz = np.flatnonzero(pool.reshape(-1))
    pages = set(nz // 18432)
    assert pages == {9}
    off = nz % 18432
    kc = range(4608 + 640, 4608 + 768)
    ks = range(4608 + 2048 + 80, 4608 + 2048 + 96)
    vc = range(4608 + 2304 + 512, 4608 + 2304 + 768)
    vs = range(4608 + 4352 + 80, 4608 + 4352 + 96)
    assert set(off) == set(kc) | set(ks) | set(vc) | set(vs)
    # 1.0 with g = 1: scale = e4m3(1/6) (code 0x23 = 2**-3 * 1.375 = 0.171875),
    # element 1/0.171875 = 5.82 -> code 7 (6.0); both nibbles -> 0x77; V -1.0
    # -> code 15 in the high nibble of every byte of the pair row -> 0xF0
    assert pool[9, 4608 + 640] == 0x77
    assert np.all(pool[9, 4608 + 2304 + 512: 4608 + 2304 + 768] == 0xF0)
    assert pool[9, 4608 + 2048 + 80] == 0x23 and pool[9, 4608 + 4352 + 80] == 0x23
    # the even slot of the same pair fills the low nibbles without touching
    # the odd slot's
    v[0, 1, :] = 1.0
    PG.scatter_tokens(pool, PG.NVFP4, 4, D, np.array([[5, 2, 9]]), [0], [36], k, v, 1.0, 1.0)
    assert np.all(pool[9, 4608 + 2304 + 512: 4608 + 2304 + 768] == 0xF7)


def test_bf16_page_layout_offsets_by_hand():
    pool = PG.new_pool(4, PG.BF16, 4, D)
    assert pool.shape == (4, 65536)
    k = np.zeros((1, 4, D))
    v = np.zeros((1, 4, D))
    k[0, 3, 0] = 1.0                      # bf16 0x3F80, little-endian: 80 3F
    v[0, 3, 255] = -2.0                   # bf16 0xC000
    PG.scatter_tokens(pool, PG.BF16, 4, D, np.array([[2, 0]]), [0], [17], k, v)
    base = 3 * 16384
    assert pool[0, base + 1 * 512] == 0x80 and pool[0, base + 1 * 512 + 1] == 0x3F
    assert pool[0, base + 8192 + 1 * 512 + 510] == 0x00 and pool[0, base + 8192 + 512 + 511] == 0xC0
    assert np.count_nonzero(pool) == 3


@pytest.mark.parametrize("dtype", [PG.NVFP4, PG.FP8, PG.INT8, PG.BF16])
def test_scatter_gather_roundtrip_and_fast_path(dtype):
    rng = np.random.default_rng(27)
    L, H = 70, 4
    k, v = _rand(rng, L, H, D, scale=2), _rand(rng, L, H, D)
    table = rng.permutation(8).astype(np.int32)[None, :5]
    p1 = PG.new_pool(8, dtype, H, D)
    p2 = PG.new_pool(8, dtype, H, D)
    # per-tensor scales that put the data's range at the top of the codes
    gk, gv = (0.004, 0.003) if dtype != PG.FP8 else (0.024, 0.018)
    PG.scatter_tokens(p1, dtype, H, D, table, np.zeros(L, int), np.arange(L), k, v, gk, gv)
    PG.scatter_sequence_fast(p2, dtype, H, D, table[0], 0, k, v, gk, gv)
    assert np.array_equal(p1, p2)
    for h in range(H):
        kk, vv = PG.gather_sequence(p1, dtype, H, D, table[0], L, h, gk, gv)
        if dtype == PG.BF16:
            assert np.array_equal(kk, k[:, h]) and np.array_equal(vv, v[:, h])
        else:
            assert np.max(np.abs(kk - k[:, h])) < 0.5 * np.abs(k).max()
            assert np.corrcoef(kk.ravel(), k[:, h].ravel())[0, 1] > 0.98


@pytest.mark.parametrize("dtype", [PG.NVFP4, PG.FP8, PG.INT8, PG.BF16])
def test_paged_decode_matches_dense_and_is_permutation_invariant(dtype):
    rng = np.random.default_rng(28)
    H, G, lens, qlen = 2, 3, [40, 23], [1, 5]
    Hq = H * G
    g_k, g_v = (0.003, 0.002) if dtype != PG.FP8 else (0.018, 0.012)
    tot = sum(lens)
    npg = [(n + 15) // 16 for n in lens]
    perm = rng.permutation(sum(npg)).astype(np.int32)
    table = np.full((2, max(npg)), -1, np.int32)
    table[0, :npg[0]] = perm[:npg[0]]
    table[1, :npg[1]] = perm[npg[0]:]
    pool = PG.new_pool(sum(npg), dtype, H, D)
    ks = [_rand(rng, n, H, D, scale=2) for n in lens]
    vs = [_rand(rng, n, H, D) for n in lens]
    for b in range(2):
        PG.scatter_sequence_fast(pool, dtype, H, D, table[b], 0, ks[b], vs[b], g_k, g_v)
    q = _rand(rng, sum(qlen), Hq, D)
    indptr = np.array([0, 1, 6])
    res = A.paged_decode(pool, dtype, H, D, q, indptr, table, np.array(lens), Hq, True, g_k, g_v)
    # dense reference from the gathered (dequantised) K/V
    for b in range(2):
        for hk in range(H):
            kk, vv = PG.gather_sequence(pool, dtype, H, D, table[b], lens[b], hk, g_k, g_v)
            for t in range(indptr[b], indptr[b + 1]):
                j = t - indptr[b]
                vis = lens[b] - qlen[b] + j + 1
                for h in range(hk * G, hk * G + G):
                    o, l = A.attention_dense(q[t, h][None], kk, vv, 1 / 16, [vis])
                    assert np.max(np.abs(res[(t, h)][0] - o[0])) < 1e-12
                    assert abs(res[(t, h)][1] - l[0]) < 1e-12
    # permute the pool's pages and the table with them: identical bits
    sigma = rng.permutation(pool.shape[0])
    pool2 = np.empty_like(pool)
    pool2[sigma] = pool
    table2 = np.where(table >= 0, sigma[np.maximum(table, 0)], -1).astype(np.int32)
    res2 = A.paged_decode(pool2, dtype, H, D, q, indptr, table2, np.array(lens), Hq, True, g_k, g_v)
    for key in res:
        assert np.array_equal(res[key][0], res2[key][0]) and res[key][1] == res2[key][1]
