"""The roofline accounting in bench.py against the oracle's page layout and a
brute-force count: algorithmic bytes per token are one record's bytes per
token over the KV heads, and the tensor-path FLOP count is the causal-exact
number of (query row, visible key) pairs x head dim x 4."""
from types import SimpleNamespace

import numpy as np

import bench
from oracle import paged as PG


def test_algorithmic_bytes_per_token_match_the_page_layout():
    for dtype in (PG.NVFP4, PG.FP8, PG.INT8, PG.BF16):
        assert bench.ALGO_BYTES_PER_TOKEN[dtype] == PG.page_head_bytes(dtype, 256) // PG.PAGE * 4


def _brute_pairs(seq_lens, qlen, causal):
    pairs = 0
    for n, nq in zip(seq_lens, qlen):
        for j in range(nq):
            pairs += (n - nq + j + 1) if causal else n
    return pairs


def test_attention_flops_brute_force():
    for causal in (0, 1):
        w = SimpleNamespace(batch=3, seq_lens=np.array([40, 7, 1000]), qlen=np.array([5, 7, 1]),
                            causal=causal, num_q_heads=24, head_dim=256)
        want = _brute_pairs(w.seq_lens, w.qlen, causal) * 24 * 256 * 4
        assert bench.attention_flops(w) == want


def test_chunked_prefill_flops():
    # 8,192 causal query tokens after 1,040,384 cached keys: 2.10e14 FLOP
    w = SimpleNamespace(batch=1, seq_lens=np.array([1040384 + 8192]), qlen=np.array([8192]),
                        causal=1, num_q_heads=24, head_dim=256)
    f = bench.attention_flops(w)
    assert f == (1040384 * 8192 + 8192 * 8193 // 2) * 24 * 256 * 4
    assert round(f / 1e14, 2) == 2.10


def test_fp4q_tile_peak_is_the_harmonic_mix():
    """With NVFP4 queries the FLOPs split evenly between a block-scaled FP4
    QK^T and an fp16 P V: the peak is the rate at which that mix runs, i.e.
    the harmonic combination of the two rates (FP4 = bf16 x 13.5 / 2.25)."""
    w = SimpleNamespace(batch=1, seq_lens=np.array([1040384 + 8192]), qlen=np.array([8192]),
                        causal=1, num_q_heads=24, num_kv_heads=4, head_dim=256, kv_dtype="nvfp4")
    f16 = bench.roofline_of(w, 100.0)
    fp4 = bench.roofline_of(w, 100.0, fp4q=True)
    p = f16["peak"]
    assert abs(fp4["peak"] - 2.0 / (1.0 / (6.0 * p) + 1.0 / p)) < 1e-9 * p
    # half of the work at the f16 rate alone takes half the f16 time, the
    # other half a sixth of that: the mix runs at 12/7 of the f16 rate
    assert abs(fp4["peak"] / p - 12.0 / 7.0) < 1e-12
    assert fp4["achieved"] == f16["achieved"]
