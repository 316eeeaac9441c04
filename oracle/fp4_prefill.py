"""Prefill attention with NVFP4 queries: QK^T as a block-scaled FP4 x FP4
contraction.  Test infrastructure only (see ``oracle/__init__.py``).

"262,144 Tokens on One RTX 5090 ...", sections "Why NVFP4 KV changes the
math" and "The stack, for the impatient", keeps K and V as NVFP4 (E2M1 codes,
one E4M3 scale per 16 contiguous elements, one binary32 scale per tensor).  A
tensor-core product that reads those codes directly, with the block scales
applied inside the contraction, needs the other operand in the same format,
so the queries are quantised too.  The pages print no such prefill; the
reading used here is the plainest one that the rest supports:

  (qc, qs) = NVFP4 encoding of the roped bf16 query row with a caller-given
             per-tensor decode scale g_Q -- the same encoder as the cache
             (``nvfp4.quantize``: e = fp32(1/(6 g_Q)), S = E4M3(fp32(a e)),
             d = fp32(E4M3(S) g_Q), r = fp32(1/d), codes E2M1(fp32(x r)))
  q_hat    = E2M1(qc) * E4M3(qs) * g_Q, exact in float64
  z_t      = (q_hat . k_hat_t) * sm_scale
  softmax, P.V, LSE and the causal rule as in ``attention.py`` (V dequantised)

A block-scaled contraction computes, for each 16-element block b,
    B_b = sum_{i in b} E2M1(qc_i) * E2M1(kc_i)
and then sum_b B_b * E4M3(qs_b) * E4M3(ks_b), times g_Q * g_K.  Each product
of two E2M1 values is a multiple of 1/4 of magnitude at most 36, so |B_b| <=
576 is a multiple of 1/4 (at most 12 significant bits) and exact in binary32;
B_b times the two scales has at most 12 + 4 + 4 significant bits and no
exponent below 2^-20, so it is exact too.  The blockwise sum is
therefore q_hat . k_hat up to the rounding of the accumulation over blocks:
the reading is the plain definition with q_hat in place of q, and
``block_scaled_dot`` writes the blockwise form out so that the identity can
be checked.
"""
import numpy as np

from .attention import attention_dense
from .formats import e2m1_decode, e4m3_decode
from .nvfp4 import BLOCK, dequantize, quantize


def quantize_queries(q, g_q):
    """NVFP4 codes (uint8 [..., D], values 0..15) and scale bytes (uint8
    [..., D/16]) of bf16-valued roped queries ``q`` [..., D]."""
    return quantize(q, g_q)


def dequantized_queries(q, g_q):
    """q_hat = the NVFP4 round trip of ``q`` (float64, shape of ``q``)."""
    codes, scales = quantize_queries(q, g_q)
    return dequantize(codes, scales, g_q)


def block_scaled_dot(q_codes, q_scales, g_q, k_codes, k_scales, g_k):
    """The blockwise form: for each query row r and key t,
    g_Q g_K sum_b E4M3(qs[r,b]) E4M3(ks[t,b]) sum_{i in b} E2M1(qc[r,i]) E2M1(kc[t,i]).
    q_codes [R, D], q_scales [R, D/16], k_codes [L, D], k_scales [L, D/16];
    returns [R, L] (float64)."""
    qe = e2m1_decode(np.asarray(q_codes))
    ke = e2m1_decode(np.asarray(k_codes))
    R, D = qe.shape
    L = ke.shape[0]
    nb = D // BLOCK
    qb = qe.reshape(R, nb, BLOCK)
    kb = ke.reshape(L, nb, BLOCK)
    block_sums = np.einsum("rbi,tbi->rtb", qb, kb)          # B_b per (r, t)
    sq = e4m3_decode(np.asarray(q_scales))                    # [R, nb]
    sk = e4m3_decode(np.asarray(k_scales))                    # [L, nb]
    scaled = block_sums * sq[:, None, :] * sk[None, :, :]
    return scaled.sum(axis=-1) * float(np.float32(g_q)) * float(np.float32(g_k))


def prefill_attention_fp4q(q, g_q, k_hat, v_hat, sm_scale, visible=None):
    """Attention of bf16-valued queries ``q`` [R, D] over dequantised keys and
    values [L, D] with the queries replaced by their NVFP4 round trip;
    ``visible[r]`` = number of leading keys row r sees.  Returns O [R, D] and
    the natural-log LSE [R]."""
    return attention_dense(dequantized_queries(q, g_q), k_hat, v_hat, sm_scale, visible)
