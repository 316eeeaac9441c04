"""Pins of the INT8 group-64 KV encoder and its page layout.

The encoder (oracle/int8.py): per 64-element group a = max|x|, scale
s = fp16_rn_satfinite(fp32(a / 127)), codes RNE(fp32(x * fp32(1/s))) clamped
to +-127.  Checked here against things fixed independently of that code:
exact round trips of representable groups, a neighbour search on the fp16
grid for the scale, a brute-force nearest integer for every code, the
half-step error bound, zero and saturated groups, and byte offsets worked out
by hand.
"""
import numpy as np

from oracle import int8 as I
from oracle import paged as PG
from oracle.formats import f32

D = 256


def test_representable_groups_round_trip():
    rng = np.random.default_rng(11)
    for _ in range(50):
        d = float(np.float16(rng.uniform(1e-3, 50.0)))          # an fp16 scale
        q = rng.integers(-127, 128, (3, 64))
        q[:, 0] = rng.choice([-127, 127], 3)                     # the group's max is 127 * d
        x = q * d
        got, s = I.quantize(x.reshape(1, 192))
        assert np.array_equal(got.reshape(3, 64), q)
        assert np.all(s.view(np.float16).astype(np.float64) == d)
        assert np.array_equal(I.dequantize(got, s).reshape(3, 64), x)


def test_scale_is_the_nearest_fp16_of_a_over_127():
    rng = np.random.default_rng(12)
    a = rng.uniform(0, 1, 3000) * 10.0 ** rng.integers(-6, 6, 3000)
    x = np.zeros((3000, 64))
    x[:, 5] = a
    _, s = I.quantize(x)
    s = s.view(np.float16).astype(np.float64)[:, 0]
    t = f32(a / 127.0)
    for si, ti in zip(s, t):
        h = np.float16(si)
        lo = float(np.nextafter(h, np.float16(-np.inf)))
        hi = float(np.nextafter(h, np.float16(np.inf)))
        # no fp16 neighbour is closer to t; on a tie the even significand wins
        assert abs(si - ti) <= abs(lo - ti) and abs(si - ti) <= abs(hi - ti)
        if abs(si - ti) == abs(hi - ti) or abs(si - ti) == abs(lo - ti):
            assert np.float16(si).view(np.uint16) % 2 == 0


def test_codes_are_nearest_integers_and_error_is_half_a_step():
    rng = np.random.default_rng(13)
    x = rng.standard_normal((200, D)) * rng.uniform(0.01, 30, (200, 1))
    q, s = I.quantize(x)
    d = s.view(np.float16).astype(np.float64)
    r = f32(1.0 / d)
    y = f32(x.reshape(200, 4, 64) * r[..., None])
    for qi, yi in zip(q.reshape(-1)[:20000], y.reshape(-1)[:20000]):
        cand = np.arange(-127, 128)
        dist = np.abs(cand - yi)
        best = cand[dist == dist.min()]
        want = best[0] if len(best) == 1 else best[best % 2 == 0][0]
        assert qi == want
    err = np.abs(I.dequantize(q, s) - x).reshape(200, 4, 64)
    assert np.all(err <= 0.5 * d[..., None] * (1 + 1e-6))


def test_zero_tiny_and_saturated_groups():
    x = np.zeros((1, D))
    x[0, 64:128] = 1e-40                       # a / 127 rounds to fp16 zero
    x[0, 128] = 1e9                            # scale saturates at 65504
    x[0, 129] = -5e6
    q, s = I.quantize(x)
    assert np.all(q[0, :128] == 0) and np.all(s[0, :2] == 0)
    assert s[0, 2].view(np.float16) == np.float16(65504.0)
    assert q[0, 128] == 127 and q[0, 129] == -76    # -5e6 / 65504 = -76.3


def test_int8_positions_by_hand():
    # K: dim d of a slot row at 64*((d%16)//4) + 4*(d//16) + d%4
    assert [int(PG.int8_k_position(d)) for d in (0, 1, 3, 4, 15, 16, 63, 255)] == \
        [0, 1, 3, 64, 195, 4, 207, 255]
    # V: dim d at pair position 32*(d%8) + d//8
    assert [int(PG.int8_v_position(d)) for d in (0, 1, 7, 8, 9, 255)] == [0, 32, 224, 1, 33, 255]
    # both are permutations
    assert sorted(PG.int8_k_position(np.arange(D))) == list(range(D))
    assert sorted(PG.int8_v_position(np.arange(D))) == list(range(D))


def test_int8_page_layout_offsets_by_hand():
    """Token 37 (page table [5, 2, 9]) lives in page 9, slot 5.  KV head 1 of
    an INT8 page (8,448 bytes per head record): K codes at 8448 + 5*256, K
    scales at 8448 + 4096 + 5*8, V codes at 8448 + 4224 + 2*512 + 2p + 1,
    V scales at 8448 + 8320 + 5*8."""
    pool = PG.new_pool(12, PG.INT8, 4, D)
    assert pool.shape == (12, 33792)
    k = np.zeros((1, 4, D))
    v = np.zeros((1, 4, D))
    k[0, 1, 16] = 2.0                         # group 0: a = 2, s = fp16(2/127), code 127
    v[0, 1, 9] = -1.0                         # group 0: code -127 at V position 33
    PG.scatter_tokens(pool, PG.INT8, 4, D, np.array([[5, 2, 9]]), [0], [37], k, v)
    base = 8448
    s2 = np.float16(np.float32(2.0) / np.float32(127.0)).view(np.uint16)
    s1 = np.float16(np.float32(1.0) / np.float32(127.0)).view(np.uint16)
    nz = {int(o): int(pool[9, o]) for o in np.flatnonzero(pool[9])}
    want = {base + 5 * 256 + 4: 127,                              # dim 16 -> byte 4
            base + 4096 + 40: int(s2 & 0xFF), base + 4096 + 41: int(s2 >> 8),
            base + 4224 + 1024 + 2 * 33 + 1: 0x81,                 # -127, odd slot
            base + 8320 + 40: int(s1 & 0xFF), base + 8320 + 41: int(s1 >> 8)}
    assert nz == {o: b for o, b in want.items() if b != 0}
    assert np.count_nonzero(pool) == len(nz)
