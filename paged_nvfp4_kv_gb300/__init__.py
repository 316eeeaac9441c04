"""GB300-native paged NVFP4 KV decode attention with YaRN rotary scaling.

Thin Python binding over libpnkv (include/pnkv.h): the functions below carry
the C entry points' names and only marshal torch tensors into pointers and
sizes; every step of the path runs in the library's CUDA kernels.  torch is
used for device memory and streams.
"""
import ctypes

import torch

from . import _lib
from ._lib import PNKV_KV_BF16, PNKV_KV_FP8, PNKV_KV_INT8, PNKV_KV_NVFP4, CacheDesc, YarnParams

__all__ = ["Cache", "YarnParams", "yarn_params", "yarn_rope_tables", "kv_append_nvfp4",
           "paged_decode_attention", "paged_prefill_attention_fp4q", "split_kv_combine", "decode_slots", "work_meta_ints",
           "page_bytes", "set_wait_limit_ns", "PNKV_KV_BF16", "PNKV_KV_NVFP4", "PNKV_KV_FP8", "PNKV_KV_INT8", "decode_dev_err"]

_DTYPES = {"bf16": PNKV_KV_BF16, "nvfp4": PNKV_KV_NVFP4, "fp8": PNKV_KV_FP8, "int8": PNKV_KV_INT8}


def _ptr(t):
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def yarn_params(theta=1.0e7, factor=4.0, original_max=262144, beta_fast=32.0, beta_slow=1.0,
                rotary_dim=64, deployed=True):
    return YarnParams(theta, factor, original_max, beta_fast, beta_slow, rotary_dim,
                      1 if deployed else 0)


class Cache:
    """A paged KV pool (one layer) and its C descriptor.

    ``pool`` is a caller-owned uint8 device tensor of num_pages * page bytes;
    ``k_scale``/``v_scale`` are the NVFP4 or FP8 per-tensor decode scales
    (INT8 pools carry their scales per 64-element group and ignore them)."""

    def __init__(self, num_pages, dtype="nvfp4", num_kv_heads=4, head_dim=256, k_scale=1.0,
                 v_scale=1.0, pool=None, device="cuda"):
        self.dtype = dtype
        self.num_kv_heads = num_kv_heads
        self.head_dim = head_dim
        self.num_pages = num_pages
        desc = CacheDesc(None, num_pages, 16, num_kv_heads, head_dim, _DTYPES[dtype],
                         float(k_scale), float(v_scale))
        self.page_bytes = page_bytes(desc)
        if pool is None:
            pool = torch.zeros(num_pages * self.page_bytes, dtype=torch.uint8, device=device)
        self.pool = pool
        desc.pool = pool.data_ptr()
        self.desc = desc

    @property
    def k_scale(self):
        return self.desc.k_scale

    @property
    def v_scale(self):
        return self.desc.v_scale


def page_bytes(desc):
    out = ctypes.c_int64(0)
    d = CacheDesc(desc.pool or 128, desc.num_pages, desc.page_size, desc.num_kv_heads,
                  desc.head_dim, desc.dtype, desc.k_scale, desc.v_scale)
    _lib.check(_lib.load().pnkv_page_bytes(ctypes.byref(d), ctypes.byref(out)), "pnkv_page_bytes")
    return out.value


def yarn_rope_tables(params, max_pos, cos_out, sin_out, stream=None):
    """fp32 cos/sin tables [max_pos, R/2] (mscale folded in)."""
    st = _lib.load().yarn_rope_tables(ctypes.byref(params), int(max_pos), _ptr(cos_out),
                                      _ptr(sin_out), _stream(stream))
    _lib.check(st, "yarn_rope_tables")


def kv_append_nvfp4(cache, page_table, batch, tok_seq, tok_pos, q, q_out, k, v, cos_t, sin_t,
                    rotary_dim, dev_err, stream=None):
    """Rope q (-> q_out) and k, quantise k/v into their pages."""
    n = tok_seq.numel()
    hq = q.shape[1] if q is not None else 0
    st = _lib.load().kv_append_nvfp4(
        ctypes.byref(cache.desc), _ptr(page_table), page_table.shape[1], int(batch), _ptr(tok_seq),
        _ptr(tok_pos), n, _ptr(q), _ptr(q_out), hq, _ptr(k), _ptr(v), _ptr(cos_t), _ptr(sin_t),
        cos_t.shape[0], int(rotary_dim), _ptr(dev_err), _stream(stream))
    _lib.check(st, "kv_append_nvfp4")


def decode_slots(cache, batch, num_q_heads, max_qlen):
    v = _lib.load().pnkv_decode_slots(ctypes.byref(cache.desc), int(batch), int(num_q_heads),
                                      int(max_qlen))
    if v < 0:
        _lib.check(int(v), "pnkv_decode_slots")
    return int(v)


def work_meta_ints(batch, num_kv_heads):
    v = _lib.load().pnkv_work_meta_ints(int(batch), int(num_kv_heads))
    if v < 0:
        _lib.check(int(v), "pnkv_work_meta_ints")
    return int(v)


def paged_decode_attention(cache, q_roped, qo_indptr, page_table, seq_lens, num_q_heads, max_qlen,
                           sm_scale, causal, o_part, lse_part, work_meta, dev_err, stream=None):
    batch = seq_lens.numel()
    slots = lse_part.shape[0]
    st = _lib.load().paged_decode_attention(
        ctypes.byref(cache.desc), _ptr(q_roped), _ptr(qo_indptr), _ptr(page_table),
        page_table.shape[1], _ptr(seq_lens), batch, q_roped.shape[0], int(num_q_heads), int(max_qlen),
        float(sm_scale), 1 if causal else 0, _ptr(o_part), _ptr(lse_part), slots, _ptr(work_meta),
        _ptr(dev_err), _stream(stream))
    _lib.check(st, "paged_decode_attention")


def paged_prefill_attention_fp4q(cache, q_roped, qo_indptr, page_table, seq_lens, num_q_heads,
                                 max_qlen, sm_scale, causal, q_scale, o_part, lse_part, work_meta,
                                 dev_err, stream=None):
    """Prefill chunk with NVFP4-encoded queries (decode scale ``q_scale``):
    block-scaled FP4 QK^T on the tensor cores; partials as for
    paged_decode_attention."""
    batch = seq_lens.numel()
    slots = lse_part.shape[0]
    st = _lib.load().paged_prefill_attention_fp4q(
        ctypes.byref(cache.desc), _ptr(q_roped), _ptr(qo_indptr), _ptr(page_table),
        page_table.shape[1], _ptr(seq_lens), batch, q_roped.shape[0], int(num_q_heads),
        int(max_qlen), float(sm_scale), 1 if causal else 0, float(q_scale), _ptr(o_part),
        _ptr(lse_part), slots, _ptr(work_meta), _ptr(dev_err), _stream(stream))
    _lib.check(st, "paged_prefill_attention_fp4q")


def split_kv_combine(o_part, lse_part, work_meta, qo_indptr, total_q, num_q_heads, num_kv_heads,
                     max_qlen, out, lse_out=None, stream=None):
    batch = qo_indptr.numel() - 1
    st = _lib.load().split_kv_combine(
        _ptr(o_part), _ptr(lse_part), _ptr(work_meta), _ptr(qo_indptr), batch, int(total_q),
        int(num_q_heads), int(num_kv_heads), 256, int(max_qlen), _ptr(out),
        1 if out.dtype == torch.float32 else 0, _ptr(lse_out), _stream(stream))
    _lib.check(st, "split_kv_combine")


def set_wait_limit_ns(ns):
    """Bound of every pipeline wait in kernels launched from now on (a
    diagnostic and test knob; default 2 s).  Returns the previous bound."""
    v = _lib.load().pnkv_set_wait_limit_ns(int(ns))
    if v < 0:
        _lib.check(int(v), "pnkv_set_wait_limit_ns")
    return int(v)


def decode_dev_err(word):
    """Names of the bits set in a device error word."""
    return [name for bit, name in _lib.DEV_ERR_BITS.items() if word & bit]
