"""Decode attention over a paged KV cache, its split-KV partials and their
log-sum-exp combine.  Test infrastructure only (see ``oracle/__init__.py``).

The plain definition (float64): for query row q (the bf16 roped query) and
the visible keys t of its sequence,
    z_t = (q . k_t) * sm_scale,        sm_scale = 1 / sqrt(D)
    w_t = exp(z_t - max z) / sum_t' exp(z_t' - max z)
    O   = sum_t w_t v_t,               LSE = ln sum_t exp(z_t)
with k_t, v_t dequantised from the cached codes (bf16 cache: the stored
values).  GQA: query head h reads KV head h // (Hq / Hkv).  A causal query
chunk of n_q rows at the end of a sequence of n keys lets row j see keys
0 .. n - n_q + j.  The first page ("A 1,048,576-token context on two RTX
5090s ...", section "YaRN, and matching what vLLM actually does") states
there is no attention-level scale besides the rope's mscale, so sm_scale is
the plain 1/sqrt(D).

Split-KV ("ninfer-windows-tp2" README, section "Limitations": the decode key
range is split; the split policy is the engine's): each split s over a key
subset produces a normalised partial O_s and LSE_s; the combine is
    M = max_s LSE_s,  O = sum_s e^(LSE_s - M) O_s / sum_s e^(LSE_s - M),
    LSE = M + ln sum_s e^(LSE_s - M),
with an empty split carrying LSE = -inf and weight 0.

Long sequences are evaluated in two passes over 65,536-key chunks (first the
maximum logit, then the sums) so that a million keys fit in host memory; this
changes no arithmetic of the definition beyond float64 summation order.
"""
import math

import numpy as np

from .paged import gather_sequence

CHUNK = 65536


def attention_dense(q, k, v, sm_scale, visible=None):
    """q [R, D], k/v [L, D] (float64); ``visible[r]`` = number of leading keys
    row r sees (default all).  Returns O [R, D], LSE [R] (natural log);
    rows that see no key get O = 0, LSE = -inf."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    R, L = q.shape[0], k.shape[0]
    vis = np.full(R, L) if visible is None else np.asarray(visible)
    z = (q @ k.T) * sm_scale
    mask = np.arange(L)[None, :] < vis[:, None]
    z = np.where(mask, z, -np.inf)
    o = np.zeros((R, q.shape[1]))
    lse = np.full(R, -np.inf)
    for r in range(R):
        if vis[r] <= 0:
            continue
        m = np.max(z[r])
        w = np.exp(z[r] - m)
        s = np.sum(w)
        o[r] = (w @ v) / s
        lse[r] = m + math.log(s)
    return o, lse


def attention_chunked(q, kv_chunks, sm_scale, visible):
    """Same result as ``attention_dense`` for keys supplied by the callable
    ``kv_chunks(start, stop) -> (k, v)``; two passes over CHUNK-key chunks."""
    q = np.asarray(q, dtype=np.float64)
    R, D = q.shape
    vis = np.asarray(visible)
    L = int(vis.max()) if R else 0
    m = np.full(R, -np.inf)
    for s in range(0, L, CHUNK):
        k, _ = kv_chunks(s, min(s + CHUNK, L))
        z = (q @ k.T) * sm_scale
        z = np.where(np.arange(s, s + k.shape[0])[None, :] < vis[:, None], z, -np.inf)
        m = np.maximum(m, z.max(axis=1))
    acc = np.zeros((R, D))
    ssum = np.zeros(R)
    for s in range(0, L, CHUNK):
        k, v = kv_chunks(s, min(s + CHUNK, L))
        z = (q @ k.T) * sm_scale
        z = np.where(np.arange(s, s + k.shape[0])[None, :] < vis[:, None], z, -np.inf)
        w = np.exp(z - np.where(np.isfinite(m), m, 0.0)[:, None])
        ssum += w.sum(axis=1)
        acc += w @ v
    o = np.zeros((R, D))
    lse = np.full(R, -np.inf)
    ok = vis > 0
    o[ok] = acc[ok] / ssum[ok, None]
    lse[ok] = m[ok] + np.log(ssum[ok])
    return o, lse


def attention_brute_force(q, k, v, sm_scale, visible=None):
    """Triple loop in pure Python for tiny inputs (test pin for the above)."""
    R, D = len(q), len(q[0])
    L = len(k)
    vis = [L] * R if visible is None else list(visible)
    o = [[0.0] * D for _ in range(R)]
    lse = [-math.inf] * R
    for r in range(R):
        n = vis[r]
        if n <= 0:
            continue
        z = []
        for t in range(n):
            acc = 0.0
            for d in range(D):
                acc += q[r][d] * k[t][d]
            z.append(acc * sm_scale)
        m = max(z)
        e = [math.exp(x - m) for x in z]
        s = sum(e)
        for d in range(D):
            o[r][d] = sum(e[t] * v[t][d] for t in range(n)) / s
        lse[r] = m + math.log(s)
    return np.array(o), np.array(lse)


def combine(o_parts, lse_parts):
    """Log-sum-exp merge of split partials: o_parts [S, R, D], lse_parts [S, R]."""
    o_parts = np.asarray(o_parts, dtype=np.float64)
    lse_parts = np.asarray(lse_parts, dtype=np.float64)
    M = lse_parts.max(axis=0)
    finite = np.isfinite(M)
    Ms = np.where(finite, M, 0.0)
    w = np.where(np.isfinite(lse_parts), np.exp(lse_parts - Ms[None, :]), 0.0)
    ssum = w.sum(axis=0)
    o = np.zeros(o_parts.shape[1:])
    o[finite] = (w[:, finite, None] * o_parts[:, finite, :]).sum(axis=0) / ssum[finite, None]
    lse = np.where(finite, Ms + np.log(np.where(finite, ssum, 1.0)), -np.inf)
    return o, lse


def split_attention(q, k, v, sm_scale, visible, bounds):
    """Partials over key ranges [bounds[i], bounds[i+1]) (split-KV), each a
    normalised (O_s, LSE_s); combine them with ``combine``."""
    R = q.shape[0]
    o_parts, l_parts = [], []
    for a, b in zip(bounds[:-1], bounds[1:]):
        vis = np.clip(np.asarray(visible) - a, 0, b - a)
        o, l = attention_dense(q, k[a:b], v[a:b], sm_scale, vis)
        o_parts.append(o)
        l_parts.append(l)
    return np.array(o_parts).reshape(len(o_parts), R, -1), np.array(l_parts)


def paged_decode(pool, dtype, num_kv_heads, head_dim, q_roped, qo_indptr, page_table, seq_lens,
                 num_q_heads, causal=True, g_k=None, g_v=None, rows=None):
    """Attention of every query row of a batch over its paged sequence.

    q_roped [T_total, Hq, D] (bf16 values); qo_indptr [B+1]; page_table rows
    per sequence; seq_lens [B] keys per sequence (new tokens included).
    ``rows`` optionally restricts the evaluation to a list of
    (token_index, q_head) pairs (sampled check at full size); otherwise every
    (token, head).  Returns dict {(t, h): (o [D], lse)}."""
    G = num_q_heads // num_kv_heads
    sm_scale = 1.0 / math.sqrt(head_dim)
    want = {}
    B = len(seq_lens)
    for b in range(B):
        for t in range(int(qo_indptr[b]), int(qo_indptr[b + 1])):
            for h in range(num_q_heads):
                if rows is None or (t, h) in rows:
                    want.setdefault((b, h // G), []).append((t, h))
    out = {}
    for (b, hk), items in want.items():
        n = int(seq_lens[b])
        nq = int(qo_indptr[b + 1] - qo_indptr[b])
        qs = np.stack([q_roped[t, h] for t, h in items]).astype(np.float64)
        vis = np.array([(n - nq + (t - int(qo_indptr[b])) + 1) if causal else n
                        for t, h in items])
        vis = np.clip(vis, 0, n)

        def chunks(s, e, b=b, hk=hk):
            return gather_sequence(pool, dtype, num_kv_heads, head_dim, page_table[b], e, hk,
                                   g_k, g_v, start=s)
        o, lse = attention_chunked(qs, chunks, sm_scale, vis)
        for i, key in enumerate(items):
            out[key] = (o[i], lse[i])
    return out
