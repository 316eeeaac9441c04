"""The CPU oracle run over a seeded workload: rope tables, roped queries and
keys, the encoded pool and the attention outputs, stage by stage.

Test infrastructure: it imports only the oracle and the seeded input
generator, never the CUDA binding, so its results can stand against the GPU
path's.  Each stage can also be fed the GPU's previous-stage output (the
rope table, the pool) so that a stage is compared on identical inputs.
"""
import numpy as np

from oracle import attention as OA
from oracle import paged as OP
from oracle import yarn as OY


def tables(w, max_pos=None):
    return OY.rope_tables(w.yarn, int(max_pos or w.max_pos))


def roped_new_q(w, cos_t, sin_t):
    """Roped bf16 queries of the step's new tokens [total_q, Hq, D] (float64)."""
    seq, pos = w.new_tokens()
    q = np.concatenate([w.q_rows(b) for b in range(w.batch)]).astype(np.float64)
    return OY.rope_rows(q, pos, cos_t, sin_t, w.yarn["rotary_dim"])


def pool(w, cos_t, sin_t, sequences=None, chunk=65536):
    """The pool after the cache fill and the step's append, built by the
    oracle: K roped with the given tables, then encoded into its pages."""
    dtype = {"nvfp4": OP.NVFP4, "fp8": OP.FP8, "int8": OP.INT8, "bf16": OP.BF16}[w.kv_dtype]
    P = OP.new_pool(w.num_pages, dtype, w.num_kv_heads, w.head_dim)
    R = w.yarn["rotary_dim"]
    for b in (range(w.batch) if sequences is None else sequences):
        n = int(w.seq_lens[b])
        for s in range(0, n, chunk):
            e = min(n, s + chunk)
            k = w.k_rows(b, s, e).astype(np.float64)
            v = w.v_rows(b, s, e).astype(np.float64)
            kr = OY.rope_rows(k, np.arange(s, e), cos_t, sin_t, R)
            OP.scatter_sequence_fast(P, dtype, w.num_kv_heads, w.head_dim, w.page_table[b], s, kr,
                                     v, w.g_k, w.g_v)
    return P


def pool_pages(w, cos_t, sin_t, b, positions):
    """Oracle bytes of the pages holding ``positions`` of sequence b (used for
    sampled checks at full size).  Returns {page id: bytes}."""
    dtype = {"nvfp4": OP.NVFP4, "fp8": OP.FP8, "int8": OP.INT8, "bf16": OP.BF16}[w.kv_dtype]
    R = w.yarn["rotary_dim"]
    pages = sorted(set(int(p) // 16 for p in positions))
    out = {}
    for pi in pages:
        s, e = pi * 16, min(pi * 16 + 16, int(w.seq_lens[b]))
        P = OP.new_pool(1, dtype, w.num_kv_heads, w.head_dim)
        k = w.k_rows(b, s, e).astype(np.float64)
        v = w.v_rows(b, s, e).astype(np.float64)
        kr = OY.rope_rows(k, np.arange(s, e), cos_t, sin_t, R)
        table = np.zeros(pi + 1, dtype=np.int32)
        OP.scatter_sequence_fast(P, dtype, w.num_kv_heads, w.head_dim, table, s, kr, v, w.g_k,
                                 w.g_v)
        out[int(w.page_table[b][pi])] = (P[0], e - s)
    return out


def attention(w, pool_bytes, q_roped, rows=None):
    """{(token, head): (o [D], lse)} over the given pool bytes."""
    dtype = {"nvfp4": OP.NVFP4, "fp8": OP.FP8, "int8": OP.INT8, "bf16": OP.BF16}[w.kv_dtype]
    return OA.paged_decode(pool_bytes, dtype, w.num_kv_heads, w.head_dim, q_roped, w.qo_indptr,
                           w.page_table, w.seq_lens, w.num_q_heads, w.causal, w.g_k, w.g_v,
                           rows=rows)
