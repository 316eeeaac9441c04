"""Seeded synthetic workloads for the paged NVFP4 KV decode path.

This module only draws inputs: shapes, positions, page tables, per-channel
scales and bf16-rounded Gaussian values.  It holds none of the path's
arithmetic (no rope, no quantisation, no attention) and imports neither the
CUDA binding nor the CPU oracle, so both sides can be fed the same inputs.

Geometry and YaRN parameters are the ones of the 27B-class attention layer
the pages run: 24 query heads, 4 KV heads of dimension 256, rotary on the
first 64 dims, theta = 1e7, YaRN factor 4 over an original 262,144-token
window, beta_fast = 32, beta_slow = 1 ("ninfer-windows-tp2" README, sections
"YaRN reference and drift guard" and "Running"; "262,144 Tokens on One RTX
5090 ...", section "Why NVFP4 KV changes the math").

Value recipe (identical for every workload): Q, K, V ~ N(0, 1) * c[head, dim]
with ln c ~ U(ln 0.5, ln 4) drawn once per tensor, rounded to bf16.  Values
are drawn in chunks of 65,536 positions from generators keyed by
(seed, tensor, sequence, chunk), so any token range can be re-drawn on its own.
"""
import math
from dataclasses import dataclass, field

import numpy as np

PAGE = 16
CHUNK = 65536
HQ, HKV, HEAD_DIM, ROTARY_DIM = 24, 4, 256, 64
YARN = dict(theta=1.0e7, factor=4.0, original_max=262144, beta_fast=32.0, beta_slow=1.0,
            rotary_dim=ROTARY_DIM, deployed=True)
E4M3_TOP, E2M1_TOP = 448.0, 6.0

_TENSOR_ID = {"q": 1, "k": 2, "v": 3, "scale": 4, "pages": 5, "lens": 6}


def bf16_values(x):
    """Round binary32 values to the nearest bf16 (ties to even), as float32."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = ((u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000).astype(np.uint32)
    return u.view(np.float32)


def bf16_to_u16(x):
    """bf16-valued float32 array -> uint16 bit patterns."""
    return (np.ascontiguousarray(x, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)


@dataclass
class Workload:
    """A batch of sequences: ``cached[b]`` tokens already in the pool at
    positions 0..cached[b]-1, plus ``qlen[b]`` new tokens at the following
    positions that the step appends and attends with."""
    name: str
    seed: int
    kv_dtype: str                     # "nvfp4", "fp8", "int8" or "bf16"
    cached: np.ndarray                # [B] int64
    qlen: np.ndarray                  # [B] int64
    num_q_heads: int = HQ
    num_kv_heads: int = HKV
    head_dim: int = HEAD_DIM
    causal: bool = True
    yarn: dict = field(default_factory=lambda: dict(YARN))
    page_table: np.ndarray = None     # [B, max_pages] int32 (-1 = unused)
    num_pages: int = 0
    c_q: np.ndarray = None
    c_k: np.ndarray = None
    c_v: np.ndarray = None

    # ---- derived sizes -------------------------------------------------
    @property
    def batch(self):
        return len(self.cached)

    @property
    def seq_lens(self):
        """Keys each sequence attends over (cached + new)."""
        return (self.cached + self.qlen).astype(np.int64)

    @property
    def qo_indptr(self):
        return np.concatenate([[0], np.cumsum(self.qlen)]).astype(np.int64)

    @property
    def total_q(self):
        return int(self.qlen.sum())

    @property
    def max_pos(self):
        return int(self.seq_lens.max())

    @property
    def _code_top(self):
        """Largest encodable magnitude per unit of g: E2M1 x E4M3 for NVFP4,
        E4M3 for FP8."""
        return E2M1_TOP * E4M3_TOP if self.kv_dtype == "nvfp4" else E4M3_TOP

    @property
    def g_k(self):
        """Per-tensor K decode scale: a 6-sigma value of the widest channel,
        after the rope's mscale and the sqrt(2) a rotation can add, maps to
        the top of the code range."""
        m = 0.1 * math.log(self.yarn["factor"]) + 1.0 if self.yarn["factor"] > 1 else 1.0
        return float(np.float32(6.0 * float(self.c_k.max()) * m * math.sqrt(2.0) / self._code_top))

    @property
    def g_q(self):
        """Per-tensor decode scale for NVFP4-encoded queries (the FP4-query
        prefill): as g_k, from the widest query channel (E2M1 x E4M3 range)."""
        m = 0.1 * math.log(self.yarn["factor"]) + 1.0 if self.yarn["factor"] > 1 else 1.0
        return float(np.float32(6.0 * float(self.c_q.max()) * m * math.sqrt(2.0) / (E2M1_TOP * E4M3_TOP)))

    @property
    def g_v(self):
        return float(np.float32(6.0 * float(self.c_v.max()) / self._code_top))

    # ---- values ----------------------------------------------------------
    def _rng(self, tensor, b, chunk):
        return np.random.default_rng([self.seed, _TENSOR_ID[tensor], b, chunk])

    def _draw(self, tensor, b, start, stop, heads, scale, base=0):
        """bf16 values of ``tensor`` for positions start..stop-1 of seq b;
        chunk c covers positions base + c*CHUNK .. base + (c+1)*CHUNK - 1 and
        only the prefix of a chunk that is needed is drawn."""
        out = np.empty((stop - start, heads, self.head_dim), dtype=np.float32)
        if stop <= start:
            return out
        c0, c1 = (start - base) // CHUNK, (stop - 1 - base) // CHUNK
        for c in range(c0, c1 + 1):
            lo = base + c * CHUNK
            a, z = max(start, lo), min(stop, lo + CHUNK)
            x = self._rng(tensor, b, c).standard_normal(
                (z - lo, heads, self.head_dim), dtype=np.float32)
            out[a - start:z - start] = x[a - lo:]
        return bf16_values(out * scale[None])

    def k_rows(self, b, start, stop):
        """Un-roped K, [n, Hkv, D] bf16 values (float32)."""
        return self._draw("k", b, start, stop, self.num_kv_heads, self.c_k)

    def v_rows(self, b, start, stop):
        return self._draw("v", b, start, stop, self.num_kv_heads, self.c_v)

    def q_rows(self, b):
        """Un-roped Q of the new tokens of sequence b, [qlen, Hq, D]."""
        s = int(self.cached[b])
        return self._draw("q", b, s, s + int(self.qlen[b]), self.num_q_heads, self.c_q, base=s)

    def new_tokens(self):
        """(seq index, position) of every new token, in qo order."""
        seq = np.repeat(np.arange(self.batch), self.qlen)
        pos = np.concatenate([np.arange(int(c), int(c) + int(n))
                              for c, n in zip(self.cached, self.qlen)]) if self.total_q else \
            np.zeros(0, dtype=np.int64)
        return seq.astype(np.int32), pos.astype(np.int32)


def _log_uniform(rng, lo, hi, size):
    return np.exp(rng.uniform(math.log(lo), math.log(hi), size=size))


def build(name, seed, kv_dtype, cached, qlen, num_q_heads=HQ, num_kv_heads=HKV,
          head_dim=HEAD_DIM, interleave=True, extra_pages=0, causal=True, yarn=None):
    """Assemble a Workload: channel scales and a page table that deals a
    seeded random permutation of the pool's pages to the sequences,
    round-robin over page index (sequences' pages interleave in the pool)."""
    cached = np.asarray(cached, dtype=np.int64)
    qlen = np.asarray(qlen, dtype=np.int64)
    w = Workload(name=name, seed=seed, kv_dtype=kv_dtype, cached=cached, qlen=qlen,
                 num_q_heads=num_q_heads, num_kv_heads=num_kv_heads, head_dim=head_dim,
                 causal=causal, yarn=dict(yarn or YARN))
    srng = np.random.default_rng([seed, _TENSOR_ID["scale"]])
    w.c_q = _log_uniform(srng, 0.5, 4.0, (num_q_heads, head_dim)).astype(np.float32)
    w.c_k = _log_uniform(srng, 0.5, 4.0, (num_kv_heads, head_dim)).astype(np.float32)
    w.c_v = _log_uniform(srng, 0.5, 4.0, (num_kv_heads, head_dim)).astype(np.float32)
    npages = (w.seq_lens + PAGE - 1) // PAGE
    w.num_pages = int(npages.sum()) + extra_pages
    prng = np.random.default_rng([seed, _TENSOR_ID["pages"]])
    perm = prng.permutation(w.num_pages).astype(np.int32)
    maxp = int(npages.max()) if len(npages) else 0
    table = np.full((w.batch, max(maxp, 1)), -1, dtype=np.int32)
    k = 0
    if interleave:
        for p in range(maxp):
            for b in range(w.batch):
                if p < npages[b]:
                    table[b, p] = perm[k]
                    k += 1
    else:
        for b in range(w.batch):
            table[b, :npages[b]] = perm[k:k + npages[b]]
            k += int(npages[b])
    w.page_table = table
    return w


# ---- the five workloads the method is measured on ------------------------------

def tiny_decode(seed=1001):
    """1 sequence, 4,096 keys (4,095 cached + 1 new), bf16 KV."""
    return build("tiny decode (4,096 bf16 keys)", seed, "bf16", [4095], [1])


def native_window_decode(seed=1002):
    """1 sequence, 262,144 keys, bf16 KV."""
    return build("native-window decode (262,144 bf16 keys)", seed, "bf16", [262143], [1])


def million_token_decode(seed=1003):
    """1 sequence, 1,048,576 keys (1,048,575 cached + 1 appended), NVFP4 KV."""
    return build("million-token decode (1,048,576 NVFP4 keys)", seed, "nvfp4", [1048575], [1])


def multi_session_verify(seed=1004, sessions=16):
    """16 sequences, cached lengths log-uniform in [8,192, 524,288], 5 new
    tokens each (1 + 4 draft tokens, causal within the 5), NVFP4 KV."""
    rng = np.random.default_rng([seed, _TENSOR_ID["lens"]])
    lens = np.floor(_log_uniform(rng, 8192, 524288, sessions)).astype(np.int64)
    return build("multi-session verify (16 x qlen 5, NVFP4)", seed, "nvfp4", lens,
                 [5] * sessions)


def multi_session_verify_reduced(seed=1004, sessions=16):
    """The multi-session verify shape at a quarter of its lengths (log-uniform
    in [2,048, 131,072], about 0.5M keys, pool larger than L2), for kernel
    profiles that must stay small (profiling only)."""
    rng = np.random.default_rng([seed, _TENSOR_ID["lens"]])
    lens = np.floor(_log_uniform(rng, 2048, 131072, sessions)).astype(np.int64)
    return build("multi-session verify, reduced (16 x qlen 5, NVFP4)", seed, "nvfp4", lens,
                 [5] * sessions)


def chunked_prefill(seed=1005):
    """1 sequence with 1,040,384 cached NVFP4 tokens plus an 8,192-token chunk."""
    return build("chunked prefill (8,192 queries over 1,048,576 NVFP4 keys)", seed, "nvfp4",
                 [1040384], [8192])


def chunked_prefill_reduced(seed=1005):
    """The chunked-prefill shape at a size an ncu capture finishes in seconds:
    200,000 cached NVFP4 tokens plus a 1,024-token chunk (profiling only)."""
    return build("chunked prefill, reduced (1,024 queries over 201,024 NVFP4 keys)", seed, "nvfp4",
                 [200000], [1024])


def million_token_decode_fp8(seed=1003):
    """The million-token decode with an FP8 (E4M3, per-tensor scale) cache."""
    return build("million-token decode (1,048,576 FP8 keys)", seed, "fp8", [1048575], [1])


def million_token_decode_int8(seed=1003):
    """The million-token decode with an INT8 group-64 cache."""
    return build("million-token decode (1,048,576 INT8 group-64 keys)", seed, "int8", [1048575], [1])


WORKLOADS = {1: tiny_decode, 2: native_window_decode, 3: million_token_decode,
           4: multi_session_verify, 5: chunked_prefill, 6: chunked_prefill_reduced,
           7: million_token_decode_fp8, 8: million_token_decode_int8,
           9: multi_session_verify_reduced}
