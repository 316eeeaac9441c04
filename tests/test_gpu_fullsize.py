"""Parity at the five workloads' full sizes, on sampled outputs the oracle can
compute one by one.

For each workload the whole step runs on the GPU exactly as bench.py runs it
(cache fill, append of the new tokens, decode or prefill tile, combine).
Checked against the oracle:
  - roped queries of every new token: bit-exact (given the GPU rope table);
  - pool bytes of sampled pages (the new tokens' pages, the first and last
    pages, seeded random pages): bit-exact;
  - attention of sampled (token, head) rows over their full key range,
    recomputed by the oracle from the GPU's pool: fp32 output within 1e-2
    max-abs and 5e-3 mean-abs, bf16 output = RNE of the fp32 output;
  - the device error word stays 0.
These runs hold up to ~2.5 GB on the device and take minutes of oracle time
on the host cores.
"""
import numpy as np
import pytest
import torch

import oracle_path

pytestmark = pytest.mark.gpu

MAX_ABS, MEAN_ABS = 1e-2, 5e-3


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _run(w):
    from paged_nvfp4_kv_gb300.engine import DecodeSession
    s = DecodeSession(w)
    s.fill()
    s.append()
    out32 = s.attend(out_fp32=True).clone()
    out16 = s.attend(out_fp32=False).clone()
    torch.cuda.synchronize()
    return s, out32, out16


def _check(w, s, out32, out16, rows, sample_pages):
    assert s.error_word() == 0
    cos_t, sin_t = s.cos.double().cpu().numpy(), s.sin.double().cpu().numpy()
    q = s.q_roped.float().cpu().numpy().astype(np.float64)
    assert np.array_equal(q, oracle_path.roped_new_q(w, cos_t, sin_t))
    pool = s.cache.pool.cpu().numpy().reshape(w.num_pages, -1)
    for b, positions in sample_pages.items():
        for page, (want, used) in oracle_path.pool_pages(w, cos_t, sin_t, b, positions).items():
            # every byte of the page, zeros included: a partly filled last page's
            # unwritten slots stay as the zero-filled pool left them
            assert np.array_equal(pool[page], want), (b, page, used)
    ref = oracle_path.attention(w, pool, q, rows=set(rows))
    o = out32.cpu().numpy()
    errs = np.concatenate([np.abs(o[t, h] - ref[(t, h)][0]) for (t, h) in rows])
    assert errs.max() <= MAX_ABS, errs.max()
    assert errs.mean() <= MEAN_ABS, errs.mean()
    want16 = torch.from_numpy(o).to(torch.bfloat16)
    assert torch.equal(out16.cpu().view(torch.int16), want16.view(torch.int16))


def _pages_of(w, b, rng, extra=8):
    n = int(w.seq_lens[b])
    pos = [0, n - 1] + list(range(int(w.cached[b]), n)) + list(rng.integers(0, n, extra))
    return pos


def test_tiny_decode_full():
    from paged_nvfp4_kv_gb300 import workloads as W
    w = W.tiny_decode()
    s, o32, o16 = _run(w)
    rows = [(0, h) for h in range(24)]
    _check(w, s, o32, o16, rows, {0: list(range(0, 4096, 16))})


def test_native_window_decode_full():
    from paged_nvfp4_kv_gb300 import workloads as W
    w = W.native_window_decode()
    s, o32, o16 = _run(w)
    rows = [(0, h) for h in (0, 5, 13)]  # three KV heads' worth of rows
    _check(w, s, o32, o16, rows, {0: _pages_of(w, 0, np.random.default_rng(2))})


def test_million_token_decode_full():
    from paged_nvfp4_kv_gb300 import workloads as W
    w = W.million_token_decode()
    s, o32, o16 = _run(w)
    rows = [(0, h) for h in (2, 7, 23)]
    _check(w, s, o32, o16, rows, {0: _pages_of(w, 0, np.random.default_rng(3))})


def test_million_token_decode_fp8_full():
    """The million-token decode with an FP8 (E4M3, per-tensor scale) pool."""
    from paged_nvfp4_kv_gb300 import workloads as W
    w = W.million_token_decode_fp8()
    s, o32, o16 = _run(w)
    rows = [(0, h) for h in (4, 11, 19)]
    _check(w, s, o32, o16, rows, {0: _pages_of(w, 0, np.random.default_rng(7))})


def test_million_token_decode_int8_full():
    """The million-token decode with an INT8 group-64 pool."""
    from paged_nvfp4_kv_gb300 import workloads as W
    w = W.million_token_decode_int8()
    s, o32, o16 = _run(w)
    rows = [(0, h) for h in (1, 12, 22)]
    _check(w, s, o32, o16, rows, {0: _pages_of(w, 0, np.random.default_rng(8))})


def test_multi_session_verify_full():
    from paged_nvfp4_kv_gb300 import workloads as W
    w = W.multi_session_verify()
    s, o32, o16 = _run(w)
    order = np.argsort(w.seq_lens)
    picks = [int(order[0]), int(order[-1])]  # shortest and longest session
    rows = []
    for b in picks:
        t0 = int(w.qo_indptr[b])
        rows += [(t0 + j, h) for j in range(5) for h in (1, 17)]
    rng = np.random.default_rng(4)
    _check(w, s, o32, o16, rows, {b: _pages_of(w, b, rng, extra=4) for b in picks})


def test_chunked_prefill_full():
    """The tensor-core tile path: 256 seeded (query token, head) rows of the
    8,192-token chunk over up to 1,048,576 keys."""
    from paged_nvfp4_kv_gb300 import workloads as W
    w = W.chunked_prefill()
    s, o32, o16 = _run(w)
    rng = np.random.default_rng(1005)
    toks = rng.integers(0, 8192, 256)
    heads = rng.integers(0, 24, 256)
    rows = sorted(set(zip(toks.tolist(), heads.tolist())))
    _check(w, s, o32, o16, rows, {0: [0, 1040383, 1040384, 1044000, 1048575]
                                       + list(rng.integers(0, 1048576, 8))})


def test_chunked_prefill_fp4q_full():
    """The FP4-query tile (block-scaled FP4 QK^T): 256 seeded rows of the
    8,192-token chunk over up to 1,048,576 keys against the oracle's
    attention with the queries' NVFP4 round trip."""
    from oracle import fp4_prefill as FP
    from paged_nvfp4_kv_gb300 import workloads as W
    from paged_nvfp4_kv_gb300.engine import DecodeSession
    w = W.chunked_prefill()
    s = DecodeSession(w)
    s.fill()
    s.append()
    out32 = s.attend(out_fp32=True, q_scale=w.g_q).clone()
    out16 = s.attend(out_fp32=False, q_scale=w.g_q).clone()
    torch.cuda.synchronize()
    assert s.error_word() == 0
    rng = np.random.default_rng(1005)
    toks = rng.integers(0, 8192, 256)
    heads = rng.integers(0, 24, 256)
    rows = sorted(set(zip(toks.tolist(), heads.tolist())))
    q = s.q_roped.float().cpu().numpy().astype(np.float64)
    q_hat = FP.dequantized_queries(q, w.g_q)
    pool = s.cache.pool.cpu().numpy().reshape(w.num_pages, -1)
    ref = oracle_path.attention(w, pool, q_hat, rows=set(rows))
    o = out32.cpu().numpy()
    errs = np.concatenate([np.abs(o[t, h] - ref[(t, h)][0]) for (t, h) in rows])
    assert errs.max() <= MAX_ABS, errs.max()
    assert errs.mean() <= MEAN_ABS, errs.mean()
    want16 = torch.from_numpy(o).to(torch.bfloat16)
    assert torch.equal(out16.cpu().view(torch.int16), want16.view(torch.int16))
