"""Paged KV pool: byte layout, scatter of new tokens, gather of a sequence.
Test infrastructure only (see ``oracle/__init__.py``).

The pages describe the pool only as fixed-size blocks in one shared pool
sized at start-up and not divided among request lanes ("NInfer -- Windows 11 TP2
fork" README, section "Limitations"), with a head-major ("HND") layout inside a
block ("262,144 Tokens on One RTX 5090 ...", section "The stack, for the
impatient").  The byte layout below is this library's own choice; it is the
definition the GPU encoder is checked against, byte for byte.

A page holds PAGE = 16 consecutive token positions of one sequence.  Token t
of sequence b lives in page ``page_table[b][t // 16]``, slot ``t % 16``.
Inside a page the record of each KV head h is contiguous, heads in order:

  NVFP4 (4,608 bytes per page-head, D = 256):
    K codes   [16 slots][D/2 bytes]   element 2k in the low nibble of byte k
    K scales  [16 slots][D/16 bytes]  E4M3, one per 16 contiguous elements
    V codes   [8 slot pairs][D bytes] byte d of pair i: element d of slot
                                      2i in the low nibble, of slot 2i+1 in
                                      the high nibble
    V scales  [16 slots][D/16 bytes]
  (V pairs slots rather than elements because the P.V product reduces over
  tokens: one byte then widens to the two consecutive-token values a
  tensor-core operand register holds.)
  FP8 (8,192 bytes per page-head; E4M3 codes, one scale per tensor):
    K codes   [16 slots][D bytes]     element d of slot s at byte d
    V codes   [8 slot pairs][D][2]    bytes 2d, 2d+1 of pair i: element d
                                      of slots 2i, 2i+1 (the same pairing as
                                      NVFP4, one byte per element)
  INT8 group-64 (8,448 bytes per page-head; int8 codes, fp16 scale per 64
  contiguous elements of a slot):
    K codes   [16 slots][D bytes]     dim d at byte 64*((d%16)//4) + 4*(d//16)
                                      + d%4 of the slot's row (the 64 bytes a
                                      tensor-core lane quarter reads for its
                                      16 k-steps are contiguous)
    K scales  [16 slots][D/64] fp16
    V codes   [8 slot pairs][D][2]    position p = 32*(d%8) + d//8 holds dim d;
                                      bytes 2p, 2p+1 of pair i: element d of
                                      slots 2i, 2i+1
    V scales  [16 slots][D/64] fp16
  bf16 (16,384 bytes per page-head):
    K [16 slots][D] bf16 (little-endian), then V [16 slots][D] bf16
"""
import numpy as np

from . import fp8, int8
from .formats import bf16_bits, bf16_from_bits
from .nvfp4 import dequantize, pack_nibbles, quantize, unpack_nibbles

PAGE = 16
NVFP4 = "nvfp4"
FP8 = "fp8"
INT8 = "int8"
BF16 = "bf16"


def int8_k_position(d):
    """Byte of a slot's K row holding dim d (INT8 pages)."""
    d = np.asarray(d)
    return 64 * ((d % 16) // 4) + 4 * (d // 16) + d % 4


def int8_v_position(d):
    """Position (2-byte pair) of a pair row holding dim d (INT8 pages)."""
    d = np.asarray(d)
    return 32 * (d % 8) + d // 8


def page_head_bytes(dtype, head_dim):
    if dtype == NVFP4:
        return 2 * PAGE * (head_dim // 2 + head_dim // 16)
    if dtype == FP8:
        return 2 * PAGE * head_dim
    if dtype == INT8:
        return 2 * PAGE * (head_dim + 2 * (head_dim // int8.GROUP))
    return 2 * PAGE * head_dim * 2


def page_bytes(dtype, num_kv_heads, head_dim):
    return num_kv_heads * page_head_bytes(dtype, head_dim)


def _sections(dtype, head_dim):
    """(offset, row_bytes) of K-data, K-scale, V-data, V-scale sections.
    For NVFP4 the V-data "row" is a slot pair (head_dim bytes)."""
    if dtype == NVFP4:
        cb, sb = head_dim // 2, head_dim // 16
        k0 = 0
        ks = k0 + PAGE * cb
        v0 = ks + PAGE * sb
        vs = v0 + PAGE * cb
        return (k0, cb), (ks, sb), (v0, head_dim), (vs, sb)
    if dtype == FP8:
        return (0, head_dim), None, (PAGE * head_dim, 2 * head_dim), None
    if dtype == INT8:
        sb = 2 * (head_dim // int8.GROUP)
        k0 = 0
        ks = PAGE * head_dim
        v0 = ks + PAGE * sb
        vs = v0 + PAGE * head_dim
        return (k0, head_dim), (ks, sb), (v0, 2 * head_dim), (vs, sb)
    rb = head_dim * 2
    return (0, rb), None, (PAGE * rb, rb), None


def new_pool(num_pages, dtype, num_kv_heads, head_dim):
    return np.zeros((num_pages, page_bytes(dtype, num_kv_heads, head_dim)), dtype=np.uint8)


def scatter_tokens(pool, dtype, num_kv_heads, head_dim, page_table, seq_of_tok, pos_of_tok,
                   k, v, g_k=None, g_v=None):
    """Write new tokens into the pool.

    ``k``, ``v``: bf16-valued float arrays [T, Hkv, D] (K already roped).
    For NVFP4 they are quantised with per-tensor decode scales g_k, g_v.
    Returns the pool (modified in place)."""
    phb = page_head_bytes(dtype, head_dim)
    (k0, kb), ks, (v0, vb), vs = _sections(dtype, head_dim)
    if dtype == NVFP4:
        kq, kscale = quantize(k, g_k)
        vq, vscale = quantize(v, g_v)
        krow = pack_nibbles(kq)
    elif dtype == FP8:
        krow = fp8.quantize(k, g_k)
        vq = fp8.quantize(v, g_v)
    elif dtype == INT8:
        kq, kscale = int8.quantize(k)
        vq, vscale = int8.quantize(v)
        krow = np.zeros(kq.shape, np.uint8)
        krow[..., int8_k_position(np.arange(head_dim))] = kq.view(np.uint8)
        kscale, vscale = kscale.view(np.uint8), vscale.view(np.uint8)   # little-endian fp16
        vpos = int8_v_position(np.arange(head_dim))
    else:
        krow = bf16_bits(k).view(np.uint8).reshape(k.shape[0], num_kv_heads, -1)
        vrow = bf16_bits(v).view(np.uint8).reshape(v.shape[0], num_kv_heads, -1)
    for t in range(len(seq_of_tok)):
        b, p = int(seq_of_tok[t]), int(pos_of_tok[t])
        page = int(page_table[b][p // PAGE])
        slot = p % PAGE
        for h in range(num_kv_heads):
            base = h * phb
            pool[page, base + k0 + slot * kb: base + k0 + (slot + 1) * kb] = krow[t, h]
            if dtype == NVFP4:
                # this slot's nibble of every byte of its pair's row
                row = pool[page, base + v0 + (slot // 2) * vb: base + v0 + (slot // 2 + 1) * vb]
                if slot % 2 == 0:
                    row[:] = (row & 0xF0) | vq[t, h]
                else:
                    row[:] = (row & 0x0F) | (vq[t, h] << 4)
                (ko, ksb), (vo, vsb) = ks, vs
                pool[page, base + ko + slot * ksb: base + ko + (slot + 1) * ksb] = kscale[t, h]
                pool[page, base + vo + slot * vsb: base + vo + (slot + 1) * vsb] = vscale[t, h]
            elif dtype == FP8:
                # byte 2d + (slot odd) of the pair's row
                row0 = base + v0 + (slot // 2) * vb + (slot % 2)
                pool[page, row0: row0 + vb: 2] = vq[t, h]
            elif dtype == INT8:
                # byte 2 p(d) + (slot odd) of the pair's row
                pool[page, base + v0 + (slot // 2) * vb + 2 * vpos + (slot % 2)] = vq[t, h].view(np.uint8)
                (ko, ksb), (vo, vsb) = ks, vs
                pool[page, base + ko + slot * ksb: base + ko + (slot + 1) * ksb] = kscale[t, h].reshape(-1)
                pool[page, base + vo + slot * vsb: base + vo + (slot + 1) * vsb] = vscale[t, h].reshape(-1)
            else:
                pool[page, base + v0 + slot * vb: base + v0 + (slot + 1) * vb] = vrow[t, h]
    return pool


def scatter_sequence_fast(pool, dtype, num_kv_heads, head_dim, pages_of_seq, start_pos, k, v,
                          g_k=None, g_v=None):
    """Write tokens start_pos .. start_pos+T-1 of one sequence (vectorised
    form of ``scatter_tokens`` for long fills; same bytes)."""
    T = k.shape[0]
    phb = page_head_bytes(dtype, head_dim)
    (k0, kb), ks, (v0, vb), vs = _sections(dtype, head_dim)
    pos = start_pos + np.arange(T)
    pages = np.asarray(pages_of_seq)[pos // PAGE]
    slots = pos % PAGE
    if dtype == NVFP4:
        kq, kscale = quantize(k, g_k)
        vq, vscale = quantize(v, g_v)
        krow = pack_nibbles(kq)
    elif dtype == FP8:
        krow = fp8.quantize(k, g_k)
        vq = fp8.quantize(v, g_v)
    elif dtype == INT8:
        kq, kscale = int8.quantize(k)
        vq, vscale = int8.quantize(v)
        krow = np.zeros(kq.shape, np.uint8)
        krow[..., int8_k_position(np.arange(head_dim))] = kq.view(np.uint8)
        kscale = kscale.view(np.uint8).reshape(T, num_kv_heads, -1)
        vscale = vscale.view(np.uint8).reshape(T, num_kv_heads, -1)
        vq = vq.view(np.uint8)
        vpos = int8_v_position(np.arange(head_dim))
    else:
        krow = bf16_bits(k).view(np.uint8).reshape(T, num_kv_heads, -1)
        vrow = bf16_bits(v).view(np.uint8).reshape(T, num_kv_heads, -1)
    for h in range(num_kv_heads):
        base = h * phb
        for j in range(kb):
            pool[pages, base + k0 + slots * kb + j] = krow[:, h, j]
        if dtype == NVFP4:
            # even slots, then odd slots (the two halves of a pair share bytes)
            for parity in (0, 1):
                sel = (slots % 2) == parity
                pg, sl = pages[sel], slots[sel]
                for j in range(vb):
                    col = base + v0 + (sl // 2) * vb + j
                    old = pool[pg, col]
                    if parity == 0:
                        pool[pg, col] = (old & 0xF0) | vq[sel, h, j]
                    else:
                        pool[pg, col] = (old & 0x0F) | (vq[sel, h, j] << 4)
            (ko, ksb), (vo, vsb) = ks, vs
            for j in range(ksb):
                pool[pages, base + ko + slots * ksb + j] = kscale[:, h, j]
                pool[pages, base + vo + slots * vsb + j] = vscale[:, h, j]
        elif dtype == FP8:
            for d in range(head_dim):
                pool[pages, base + v0 + (slots // 2) * vb + 2 * d + (slots % 2)] = vq[:, h, d]
        elif dtype == INT8:
            for d in range(head_dim):
                pool[pages, base + v0 + (slots // 2) * vb + 2 * vpos[d] + (slots % 2)] = vq[:, h, d]
            (ko, ksb), (vo, vsb) = ks, vs
            for j in range(ksb):
                pool[pages, base + ko + slots * ksb + j] = kscale[:, h, j]
                pool[pages, base + vo + slots * vsb + j] = vscale[:, h, j]
        else:
            for j in range(vb):
                pool[pages, base + v0 + slots * vb + j] = vrow[:, h, j]
    return pool


def gather_sequence(pool, dtype, num_kv_heads, head_dim, pages_of_seq, seq_len, head,
                    g_k=None, g_v=None, start=0):
    """Dequantised K, V of one sequence and KV head, tokens start..seq_len-1,
    as float64 [L, D] each.  Token t is read from page pages_of_seq[t // 16],
    slot t % 16."""
    phb = page_head_bytes(dtype, head_dim)
    (k0, kb), ks, (v0, vb), vs = _sections(dtype, head_dim)
    t = np.arange(start, seq_len)
    pages = np.asarray(pages_of_seq)[t // PAGE]
    slots = t % PAGE
    base = head * phb
    kcols = base + k0 + slots[:, None] * kb + np.arange(kb)[None, :]
    krow = pool[pages[:, None], kcols]
    if dtype == NVFP4:
        (ko, ksb), (vo, vsb) = ks, vs
        kscol = base + ko + slots[:, None] * ksb + np.arange(ksb)[None, :]
        vscol = base + vo + slots[:, None] * vsb + np.arange(vsb)[None, :]
        vcols = base + v0 + (slots[:, None] // 2) * vb + np.arange(vb)[None, :]
        vbytes = pool[pages[:, None], vcols]
        vcodes = np.where((slots % 2 == 0)[:, None], vbytes & 0xF, vbytes >> 4)
        kk = dequantize(unpack_nibbles(krow), pool[pages[:, None], kscol], g_k)
        vv = dequantize(vcodes, pool[pages[:, None], vscol], g_v)
        return kk, vv
    if dtype == FP8:
        vcols = (base + v0 + (slots[:, None] // 2) * vb + 2 * np.arange(head_dim)[None, :]
                 + (slots % 2)[:, None])
        return fp8.dequantize(krow, g_k), fp8.dequantize(pool[pages[:, None], vcols], g_v)
    if dtype == INT8:
        (ko, ksb), (vo, vsb) = ks, vs
        dims = np.arange(head_dim)
        kq = krow[:, int8_k_position(dims)].view(np.int8)
        vcols = (base + v0 + (slots[:, None] // 2) * vb + 2 * int8_v_position(dims)[None, :]
                 + (slots % 2)[:, None])
        vq = pool[pages[:, None], vcols].view(np.int8)
        kscol = base + ko + slots[:, None] * ksb + np.arange(ksb)[None, :]
        vscol = base + vo + slots[:, None] * vsb + np.arange(vsb)[None, :]
        ksc = np.ascontiguousarray(pool[pages[:, None], kscol]).view(np.uint16)
        vsc = np.ascontiguousarray(pool[pages[:, None], vscol]).view(np.uint16)
        return int8.dequantize(kq, ksc), int8.dequantize(vq, vsc)
    vcols = base + v0 + slots[:, None] * vb + np.arange(vb)[None, :]
    vrow = pool[pages[:, None], vcols]
    kk = bf16_from_bits(krow.view(np.uint16))
    vv = bf16_from_bits(vrow.view(np.uint16))
    return kk, vv
