"""A decode step over one attention layer, built from the four library calls.

``DecodeSession`` owns the device buffers of one workload (pool, page table,
rope tables, partial buffers, the step's new tokens) and issues, on one
stream:

    kv_append_nvfp4 -> paged_decode_attention -> split_kv_combine

``fill()`` writes a workload's cached tokens into the pool with the same
append kernel (positions 0 .. cached-1 of every sequence, no queries).
"""
import math

import numpy as np
import torch

from . import (Cache, decode_slots, kv_append_nvfp4, paged_decode_attention,
               paged_prefill_attention_fp4q, split_kv_combine, work_meta_ints, yarn_params,
               yarn_rope_tables)


def to_bf16(x, device):
    """bf16-valued float32 numpy array -> bf16 device tensor (exact)."""
    return torch.from_numpy(np.ascontiguousarray(x)).to(device=device, dtype=torch.bfloat16)


class DecodeSession:
    def __init__(self, w, device="cuda", max_pos=None, stream=None, tables=None, inputs=None):
        """``tables``: (cos, sin) of another session to share; ``inputs``: a
        session whose new-token tensors (q, k, v) and index tensors to share."""
        self.w = w
        self.device = device
        self.stream = stream
        self.cache = Cache(w.num_pages, w.kv_dtype, w.num_kv_heads, w.head_dim, w.g_k, w.g_v,
                           device=device)
        self.page_table = torch.from_numpy(w.page_table).to(device)
        y = w.yarn
        self.rotary_dim = y["rotary_dim"]
        self.yarn = yarn_params(y["theta"], y["factor"], y["original_max"], y["beta_fast"],
                                y["beta_slow"], y["rotary_dim"], y.get("deployed", True))
        self.max_pos = int(max_pos or w.max_pos)
        half = self.rotary_dim // 2
        if tables is not None:
            self.cos, self.sin = tables
        else:
            self.cos = torch.empty(self.max_pos, half, dtype=torch.float32, device=device)
            self.sin = torch.empty(self.max_pos, half, dtype=torch.float32, device=device)
            yarn_rope_tables(self.yarn, self.max_pos, self.cos, self.sin, stream)
        self.dev_err = torch.zeros(1, dtype=torch.int32, device=device)
        self.max_qlen = int(w.qlen.max())
        self.group = w.num_q_heads // w.num_kv_heads
        slots = decode_slots(self.cache, w.batch, w.num_q_heads, self.max_qlen)
        rows = self.group * self.max_qlen
        self.o_part = torch.empty(slots, rows, w.head_dim, dtype=torch.float32, device=device)
        self.lse_part = torch.empty(slots, rows, dtype=torch.float32, device=device)
        self.work_meta = torch.zeros(work_meta_ints(w.batch, w.num_kv_heads), dtype=torch.int32,
                                     device=device)
        self.qo_indptr = torch.from_numpy(w.qo_indptr.astype(np.int32)).to(device)
        self.seq_lens = torch.from_numpy(w.seq_lens.astype(np.int32)).to(device)
        seq, pos = w.new_tokens()
        self.tok_seq = torch.from_numpy(seq).to(device)
        self.tok_pos = torch.from_numpy(pos).to(device)
        self.total_q = w.total_q
        # the step's new tokens (un-roped Q, K, V)
        if inputs is not None:
            self.q, self.k, self.v = inputs.q, inputs.k, inputs.v
        elif self.total_q:
            self.q = to_bf16(np.concatenate([w.q_rows(b) for b in range(w.batch)]), device)
            self.k = to_bf16(np.concatenate([w.k_rows(b, int(w.cached[b]), int(w.seq_lens[b]))
                                             for b in range(w.batch)]), device)
            self.v = to_bf16(np.concatenate([w.v_rows(b, int(w.cached[b]), int(w.seq_lens[b]))
                                             for b in range(w.batch)]), device)
        self.q_roped = torch.empty_like(self.q)
        self.out = torch.empty(self.total_q, w.num_q_heads, w.head_dim, dtype=torch.bfloat16,
                               device=device)
        self.out32 = torch.empty(self.total_q, w.num_q_heads, w.head_dim, dtype=torch.float32,
                                 device=device)
        self.lse = torch.empty(self.total_q, w.num_q_heads, dtype=torch.float32, device=device)
        self.sm_scale = 1.0 / math.sqrt(w.head_dim)

    # -- cache fill -------------------------------------------------------------
    def fill(self, chunk=65536):
        """Append every cached token of every sequence (K roped, K/V encoded)."""
        w = self.w
        for b in range(w.batch):
            n = int(w.cached[b])
            for s in range(0, n, chunk):
                e = min(n, s + chunk)
                k = to_bf16(w.k_rows(b, s, e), self.device)
                v = to_bf16(w.v_rows(b, s, e), self.device)
                seq = torch.full((e - s,), b, dtype=torch.int32, device=self.device)
                pos = torch.arange(s, e, dtype=torch.int32, device=self.device)
                kv_append_nvfp4(self.cache, self.page_table, w.batch, seq, pos, None, None, k, v,
                                self.cos, self.sin, self.rotary_dim, self.dev_err, self.stream)

    # -- one step ---------------------------------------------------------------
    def append(self):
        kv_append_nvfp4(self.cache, self.page_table, self.w.batch, self.tok_seq, self.tok_pos,
                        self.q, self.q_roped, self.k, self.v, self.cos, self.sin, self.rotary_dim,
                        self.dev_err, self.stream)

    def attend(self, out_fp32=False, q_scale=None):
        """Attention of the step's roped queries -> combined output.  With
        ``q_scale`` (a prefill chunk on an NVFP4 pool) the queries are NVFP4-
        encoded with that decode scale and QK^T runs block-scaled in FP4."""
        self.partials(q_scale)
        return self.combine(out_fp32)

    def partials(self, q_scale=None):
        """The attention call alone: per-split partials into o_part/lse_part."""
        w = self.w
        if q_scale is None:
            paged_decode_attention(self.cache, self.q_roped, self.qo_indptr, self.page_table,
                                   self.seq_lens, w.num_q_heads, self.max_qlen, self.sm_scale,
                                   w.causal, self.o_part, self.lse_part, self.work_meta,
                                   self.dev_err, self.stream)
        else:
            paged_prefill_attention_fp4q(self.cache, self.q_roped, self.qo_indptr, self.page_table,
                                         self.seq_lens, w.num_q_heads, self.max_qlen, self.sm_scale,
                                         w.causal, q_scale, self.o_part, self.lse_part,
                                         self.work_meta, self.dev_err, self.stream)

    def combine(self, out_fp32=False):
        """The log-sum-exp merge of the partials -> out (bf16) or out32."""
        w = self.w
        out = self.out32 if out_fp32 else self.out
        split_kv_combine(self.o_part, self.lse_part, self.work_meta, self.qo_indptr, self.total_q,
                         w.num_q_heads, w.num_kv_heads, self.max_qlen, out, self.lse, self.stream)
        return out

    def step(self, out_fp32=False, q_scale=None):
        self.append()
        return self.attend(out_fp32, q_scale)

    def error_word(self):
        return int(self.dev_err.item())


class DecodeStack:
    """Attention layers of one geometry, each with its own pool, stepped
    together; the step can be captured in a CUDA graph and replayed (the
    library allocates nothing and every call is stream-ordered, so a captured
    step is the same launches with the same arguments).

    ``workloads`` holds one workload per layer: each layer has its own seeded
    K/V, new tokens, page table and per-tensor scales, and is filled from its
    own workload.  ``replicated(w, layers)`` builds a stack whose layers
    start as byte copies of layer 0's pool and append layer 0's new tokens
    (distinct memory, identical contents): the same work per layer, for timing
    deep stacks without drawing every layer's cache on the host."""

    def __init__(self, workloads, device="cuda", _replicas=0):
        first = DecodeSession(workloads[0], device=device,
                              max_pos=max(w.max_pos for w in workloads))
        self.sessions = [first]
        self.replicated_from_first = _replicas > 0
        for _ in range(_replicas):
            self.sessions.append(DecodeSession(workloads[0], device=device, max_pos=first.max_pos,
                                               tables=(first.cos, first.sin), inputs=first))
        for w in workloads[1:]:
            if w.yarn != workloads[0].yarn:
                raise ValueError("the layers of a stack share one rope table: YaRN parameters differ")
            self.sessions.append(DecodeSession(w, device=device, max_pos=first.max_pos,
                                               tables=(first.cos, first.sin)))
        self.graph = None

    @classmethod
    def replicated(cls, w, layers=16, device="cuda"):
        return cls([w], device=device, _replicas=layers - 1)

    def fill(self):
        first = self.sessions[0]
        first.fill()
        for s in self.sessions[1:]:
            if self.replicated_from_first:
                s.cache.pool.copy_(first.cache.pool)
            else:
                s.fill()

    def step(self, out_fp32=False):
        return [s.step(out_fp32) for s in self.sessions]

    def capture(self, out_fp32=False):
        """Capture one step of every layer in a CUDA graph (after one eager
        step on the capture stream, which sets kernel attributes)."""
        stream = torch.cuda.Stream()
        stream.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(stream):
            self.step(out_fp32)
        stream.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph, stream=stream):
            self.step(out_fp32)
        torch.cuda.current_stream().wait_stream(stream)
        return self.graph

    def replay(self):
        self.graph.replay()

    def outputs(self, out_fp32=False):
        return [s.out32 if out_fp32 else s.out for s in self.sessions]

    def error_word(self):
        e = 0
        for s in self.sessions:
            e |= s.error_word()
        return e
