/*
 * pnkv.h -- C ABI of libpnkv: long-context decode attention over a paged
 * NVFP4 (or bf16) KV cache with YaRN rotary scaling, for one sm_103a GPU.
 *
 * The four calls of the decode path, in the order a step issues them:
 *
 *   yarn_rope_tables        once per (YaRN parameters, maximum position)
 *   kv_append_nvfp4         rope the step's new queries and keys, quantise
 *                           K and V, write them into their pages
 *   paged_decode_attention  split-KV GQA attention of every new query row
 *                           over its sequence's pages -> per-split partials
 *   split_kv_combine        log-sum-exp merge of the partials -> output
 *
 * Conventions shared by every call:
 *   - Every pointer argument named as device memory must be device memory of
 *     the current CUDA device, allocated and owned by the caller; the library
 *     never allocates, frees or retains memory and keeps no state between
 *     calls except a per-device cache of the device's SM count, the pipeline
 *     wait bound (pnkv_set_wait_limit_ns) and the fixed scratch of
 *     paged_decode_attention_noalloc.
 *   - Every call is asynchronous and stream-ordered on `stream` (a
 *     cudaStream_t; NULL is the legacy default stream).  A call returns once
 *     its kernels are enqueued.
 *   - Kernel attributes (the shared-memory limit of the large kernels) are
 *     set on the current device at its first call there, so one process may
 *     drive several devices.
 *   - Return value: PNKV_OK, or a negative pnkv status.  Argument errors that
 *     the host can see return PNKV_ERR_INVALID_ARG before anything is
 *     launched; a failed launch returns PNKV_ERR_CUDA.
 *   - Errors only the device can see (a page id outside the pool, a position
 *     past the page table or the rope table, a sequence longer than its page
 *     table row, an inconsistent qo_indptr, a pipeline wait that timed out)
 *     are OR-ed into the caller's device word `dev_err` (PNKV_DEV_ERR_* bits);
 *     the offending page, token or sequence is skipped and the kernel
 *     completes.  Read `dev_err` after synchronising the stream.  The outputs
 *     of a flagged sequence are unspecified (a skipped sequence reads as no
 *     visible key: zeros and LSE -inf); after a timeout all outputs of that
 *     call are unspecified.  Other sequences' outputs are unaffected, and the
 *     context stays usable.
 *   - bf16 tensors are passed as uint16_t bit patterns.
 *
 * Sources (pages on the method; the library restates them, it copies none):
 *   [YaRN-page]  "A 1,048,576-token context on two RTX 5090s: forking a C++
 *                inference engine for tensor-parallel and YaRN", section
 *                "YaRN, and matching what vLLM actually does".
 *   [TP2-README] "NInfer -- Windows 11 TP2 fork" README, sections "YaRN
 *                reference and drift guard", "Usage" and "Limitations".
 *   [NVFP4-page] "262,144 Tokens on One RTX 5090: Qwen3.8-27B with an NVFP4
 *                KV Cache That Actually Works", sections "Why NVFP4 KV changes
 *                the math" and "The stack, for the impatient".
 *   [YaRN-paper] Peng et al., 2023, "YaRN: Efficient Context Window Extension
 *                of Large Language Models" (cited by [YaRN-page]).
 */
#ifndef PNKV_H
#define PNKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------ */
enum {
  PNKV_OK = 0,
  PNKV_ERR_INVALID_ARG = -1, /* a host-visible argument is out of contract  */
  PNKV_ERR_UNSUPPORTED = -2, /* valid request this build does not implement  */
  PNKV_ERR_CUDA = -3         /* a CUDA runtime/driver call or launch failed  */
};

/* ---- device error word bits (OR-ed into *dev_err) ----------------------- */
enum {
  PNKV_DEV_ERR_PAGE_ID = 1,    /* page table entry outside [0, num_pages)    */
  PNKV_DEV_ERR_POSITION = 2,   /* token position >= rope table rows, or < 0  */
  PNKV_DEV_ERR_SEQ_LEN = 4,    /* position or seq_len beyond pt_stride * 16  */
  PNKV_DEV_ERR_QO_INDPTR = 8,  /* qlen < 0, > max_qlen or > seq_len, or the
                                  sequence's rows end past total_q          */
  PNKV_DEV_ERR_TIMEOUT = 16,   /* a bounded pipeline wait gave up            */
  PNKV_DEV_ERR_SEQ_INDEX = 32  /* tok_seq outside [0, batch)                 */
};

/* ---- KV cache element formats ------------------------------------------- */
enum {
  PNKV_KV_BF16 = 0,  /* K, V stored as bf16                                  */
  PNKV_KV_NVFP4 = 1, /* E2M1 codes + E4M3 scale per 16 elements + fp32
                        per-tensor scale ([NVFP4-page])                      */
  PNKV_KV_FP8 = 2,   /* E4M3 codes + fp32 per-tensor scale (the comparison
                        engine's fp8 cache, [YaRN-page] section "Against
                        vLLM: prefill loses, decode wins, and one surprise") */
  PNKV_KV_INT8 = 3   /* int8 codes + fp16 scale per 64 elements ([TP2-README]
                        "Dual-GPU (TP2) and YaRN 1M context", "Memory, per
                        GPU": the million-token cache)                      */
};

/* YaRN parameters ([YaRN-paper], NTK-by-parts; [YaRN-page]; [TP2-README]).
 * Validation follows the [TP2-README] "Usage" rules: factor finite in
 * [1, 64]; original_max * factor a whole number <= 1,048,576.  Also theta >
 * 1, beta_fast > beta_slow > 0, rotary_dim in {16, 32, 64, 128, 256}.
 * deployed_range = 1 computes the correction range over original_max *
 * factor positions (the range the deployed serving stack uses, (16, 24) for
 * theta 1e7, R 64, s 4, original 262,144 -- [YaRN-page]); 0 uses
 * original_max (the paper's formula, (14, 22) for the same parameters). */
typedef struct {
  double theta;          /* rope base, e.g. 1e7                              */
  double factor;         /* YaRN scale s, e.g. 4                             */
  int64_t original_max;  /* native window, e.g. 262,144                      */
  double beta_fast;      /* e.g. 32                                          */
  double beta_slow;      /* e.g. 1                                           */
  int32_t rotary_dim;    /* R: dims 0..R-1 of a head are rotated, e.g. 64    */
  int32_t deployed_range;
} pnkv_yarn_params;

/* The paged KV pool: one layer's K and V in fixed 16-token pages.
 *
 * Byte layout (this library's own; the pages fix only "fixed-size blocks
 * in one shared pool" [TP2-README "Limitations"] and a head-major layout
 * [NVFP4-page "The stack, for the impatient"]).  A page holds 16 consecutive
 * positions of one sequence; token t of sequence b lives in page
 * page_table[b * pt_stride + t / 16], slot t % 16.  Inside a page the records
 * of the KV heads follow each other in head order.  One head's record:
 *   NVFP4, head_dim 256 (4,608 bytes):
 *     K codes  [16 slots][128 B]  element 2k in the low nibble of byte k
 *     K scales [16 slots][16 B]   E4M3, one per 16 contiguous elements
 *     V codes  [8 slot pairs][256 B]  byte d of pair i: element d of slot 2i
 *                                  in the low nibble, of slot 2i+1 in the high
 *     V scales [16 slots][16 B]
 *   FP8, head_dim 256 (8,192 bytes):
 *     K codes  [16 slots][256 B]  E4M3, element d of a slot at byte d
 *     V codes  [8 slot pairs][256][2 B]  bytes 2d, 2d+1 of pair i: element
 *                                  d of slots 2i and 2i+1
 *   INT8 group-64, head_dim 256 (8,448 bytes):
 *     K codes  [16 slots][256 B]  int8; dim d at byte 64*((d%16)/4) +
 *                                  4*(d/16) + d%4 of the slot's row
 *     K scales [16 slots][4] fp16 (one per 64 contiguous dims)
 *     V codes  [8 slot pairs][256][2 B]  position p = 32*(d%8) + d/8 holds
 *                                  dim d; bytes 2p, 2p+1 of pair i: element
 *                                  d of slots 2i and 2i+1
 *     V scales [16 slots][4] fp16
 *   bf16, head_dim 256 (16,384 bytes):
 *     K [16 slots][256] bf16, then V [16 slots][256] bf16
 * A page is num_kv_heads * record bytes (18,432 B NVFP4, 32,768 B FP8,
 * 33,792 B INT8 or 65,536 B bf16 for 4 KV heads).  `pool` must be 128-byte
 * aligned.
 *
 * NVFP4 decode of element i of a block with scale byte S: E2M1(code_i) *
 * E4M3(S) * k_scale (K) or * v_scale (V); k_scale and v_scale are the
 * per-tensor fp32 decode scales, calibrated by the caller.  FP8 decode:
 * E4M3(code) * k_scale (or v_scale); the encoder writes E4M3_rn_satfinite(x *
 * fp32(1/scale)).  FP8 precondition: bytes of slots not written yet hold no
 * E4M3 NaN code (0x7F, 0xFF); a zero-filled pool satisfies it.  INT8 decode:
 * code * fp16 group scale (k_scale and v_scale are not used). */
typedef struct {
  void* pool;            /* device, num_pages * page bytes                   */
  int64_t num_pages;
  int32_t page_size;     /* must be 16                                       */
  int32_t num_kv_heads;  /* 1..16                                            */
  int32_t head_dim;      /* must be 256                                      */
  int32_t dtype;         /* PNKV_KV_BF16, _NVFP4, _FP8 or _INT8              */
  float k_scale;         /* NVFP4/FP8: per-tensor K decode scale (> 0)       */
  float v_scale;         /* NVFP4/FP8: per-tensor V decode scale (> 0)       */
                         /* (INT8 and bf16 pools ignore both)                */
} pnkv_cache;

/* Bytes of one page of `cache` (written to *out).  Host only. */
int pnkv_page_bytes(const pnkv_cache* cache, int64_t* out);

/* YaRN cos/sin tables ([YaRN-paper]; [YaRN-page]; [TP2-README] "YaRN
 * reference and drift guard").  For pair i = 0 .. R/2-1 the inverse
 * frequency blends theta^(-2i/R) and theta^(-2i/R)/s along the linear ramp
 * over the correction range; mscale = 0.1 ln s + 1 (1 for s = 1) multiplies
 * cos and sin, so no other attention-level scale is applied:
 *   cos_out[p * R/2 + i] = fp32(mscale * cos(p * inv_freq_i))
 *   sin_out[p * R/2 + i] = fp32(mscale * sin(p * inv_freq_i))
 * for p = 0 .. max_pos-1, with the angle and cos/sin in double precision and
 * one rounding to fp32.
 *   params   host pointer, validated as described at pnkv_yarn_params
 *   max_pos  rows, 1 .. 2^31-1
 *   cos_out, sin_out  device, fp32 [max_pos, R/2] each, 4-byte aligned */
int yarn_rope_tables(const pnkv_yarn_params* params, int64_t max_pos,
                     float* cos_out, float* sin_out, void* stream);

/* Rope the step's new tokens and write their K/V into the pool.
 * ([YaRN-page]: mscale applied inside the rope on the rotary dims;
 * [NVFP4-page]: NVFP4 cache writer.)
 *
 * For new token n (0 .. num_tokens-1) of sequence b = tok_seq[n] at position
 * p = tok_pos[n], with c = cos_t[p * R/2 + i], s = sin_t[p * R/2 + i]:
 *   x'_i      = fp32(fp32(x_i * c) - fp32(x_{i+R/2} * s))     i < R/2
 *   x'_{i+R/2} = fp32(fp32(x_{i+R/2} * c) + fp32(x_i * s))
 * (rotate-half pairing within the first R dims; dims >= R unchanged), then
 * rounded to bf16.  Roped queries go to q_out; roped K and raw V go to page
 * page_table[b * pt_stride + p / 16], slot p % 16, as bf16 or NVFP4:
 *   e = fp32(1 / (6 g)); a = max |x| over the 16-element block;
 *   S = E4M3_rn_satfinite(fp32(a * e)); if E4M3(S) == 0 the block is all
 *   zero codes with scale byte 0; else d = fp32(E4M3(S) * g),
 *   r = fp32(1 / d), code_i = E2M1_rn_satfinite(fp32(x_i * r)), the sign of
 *   a value that rounds to zero kept (g = k_scale for K, v_scale for V);
 * or FP8: code_i = E4M3_rn_satfinite(fp32(x_i * fp32(1 / g))), the sign of a
 * value that rounds to zero kept; or INT8: per 64-element group a = max |x|,
 * s = fp16_rn_satfinite(fp32(a / 127)), zero group if s == 0, else code_i =
 * clamp(RNE(fp32(x_i * fp32(1 / s))), -127, 127).  (The name keeps the NVFP4 path's; the
 * pool's dtype selects the encoder.)  NVFP4 and FP8 scales must lie in
 * [2^-100, 2^100].
 *
 *   cache        host pointer to the pool descriptor
 *   page_table   device int32 [batch, pt_stride]
 *   tok_seq, tok_pos  device int32 [num_tokens]
 *   q            device bf16 [num_tokens, num_q_heads, 256], or NULL
 *   q_out        device bf16, same shape (NULL iff q is NULL); may equal q
 *   k, v         device bf16 [num_tokens, num_kv_heads, 256]
 *   cos_t, sin_t device fp32 [table_rows, rotary_dim/2]
 *   dev_err      device int32 word (see PNKV_DEV_ERR_*)
 * All tensors contiguous and 16-byte aligned.  Tokens whose page, position
 * or sequence index is out of range are skipped and flagged. */
int kv_append_nvfp4(const pnkv_cache* cache, const int32_t* page_table,
                    int64_t pt_stride, int32_t batch, const int32_t* tok_seq,
                    const int32_t* tok_pos, int64_t num_tokens,
                    const uint16_t* q, uint16_t* q_out, int32_t num_q_heads,
                    const uint16_t* k, const uint16_t* v, const float* cos_t,
                    const float* sin_t, int64_t table_rows, int32_t rotary_dim,
                    int32_t* dev_err, void* stream);

/* Number of partial slots paged_decode_attention writes at most, for this
 * device and geometry (host only; queries the current device).  The caller
 * sizes o_part as slots * num_q_heads/num_kv_heads * max_qlen * head_dim
 * floats and lse_part as slots * num_q_heads/num_kv_heads * max_qlen floats.
 * Returns a negative status on bad arguments. */
int64_t pnkv_decode_slots(const pnkv_cache* cache, int32_t batch,
                          int32_t num_q_heads, int32_t max_qlen);

/* int32 entries paged_decode_attention writes into work_meta. */
int64_t pnkv_work_meta_ints(int32_t batch, int32_t num_kv_heads);

/* Split-KV GQA attention of the new query rows over their paged sequences
 * ([TP2-README] "Limitations": split-KV decode; the split here is
 * stream-K over all (sequence, KV head, page) units, balanced across the
 * GPU's SMs).
 *
 * Sequence b has seq_lens[b] keys (the new tokens already appended) and
 * qlen_b = qo_indptr[b+1] - qo_indptr[b] query tokens, the last qlen_b
 * positions.  Query head h reads KV head h / (num_q_heads / num_kv_heads).
 * With causal != 0, query row j of sequence b sees keys 0 .. seq_lens[b] -
 * qlen_b + j; otherwise all seq_lens[b] keys.  Logits are
 * z = (q . k) * sm_scale with q the roped bf16 query and k, v the cache
 * values (NVFP4, FP8, INT8: dequantised), softmax in fp32 with fp16 probabilities in
 * the P.V product.  Each split writes its normalised partial output and
 * natural-log LSE; empty splits write LSE = -inf.
 * Query precision: on NVFP4, FP8 and INT8 pools the tensor-core products take
 * the roped query in fp16 (the cache values are exact in fp16), so the
 * query's bf16 elements must lie within the fp16 range (|q| <= 65,504); a
 * larger element becomes infinite.  Elements below 2^-14 in magnitude keep
 * fewer mantissa bits (fp16 subnormals; an error of at most 2^-25 per element),
 * which the logit tolerance absorbs.  bf16 pools take the query unchanged.
 *
 *   q_roped     device bf16 [total_q, num_q_heads, 256]
 *   qo_indptr   device int32 [batch + 1], non-decreasing, qo_indptr[0] = 0,
 *               qo_indptr[batch] <= total_q (a sequence whose rows end past
 *               total_q is skipped and flagged PNKV_DEV_ERR_QO_INDPTR)
 *   total_q     rows of q_roped (host copy of qo_indptr[batch])
 *   page_table  device int32 [batch, pt_stride]
 *   seq_lens    device int32 [batch]
 *   max_qlen    host bound on every qlen_b (1 .. 8192); num_q_heads /
 *               num_kv_heads * max_qlen rows per slot
 *   o_part      device fp32 [slots, rows_per_slot, 256]  (pnkv_decode_slots)
 *   lse_part    device fp32 [slots, rows_per_slot]
 *   part_slots  capacity of o_part/lse_part in slots
 *   work_meta   device int32 [pnkv_work_meta_ints(batch, num_kv_heads)]:
 *               where each (sequence, KV head)'s partials are; read by
 *               split_kv_combine
 *   dev_err     device int32 word
 * The pool must hold NVFP4, FP8, INT8 or bf16 pages with head_dim 256 and
 * 16-token pages; num_q_heads / num_kv_heads in 1..8 rows per query token.
 * More than 64 rows per KV head (a prefill chunk) run the tensor-core tile,
 * built for NVFP4 pools; other pools return PNKV_ERR_UNSUPPORTED there.
 * The pool is read through a TMA map of 128-byte rows with 32-bit signed row
 * coordinates: num_pages * num_kv_heads * rows per record (NVFP4 36, FP8 64,
 * INT8 66, bf16 128) must stay below 2^31 (about 14.9M NVFP4 pages of 4 KV
 * heads, 275 GB), else PNKV_ERR_INVALID_ARG. */
int paged_decode_attention(const pnkv_cache* cache, const uint16_t* q_roped,
                           const int32_t* qo_indptr, const int32_t* page_table,
                           int64_t pt_stride, const int32_t* seq_lens,
                           int32_t batch, int64_t total_q, int32_t num_q_heads, int32_t max_qlen,
                           float sm_scale, int32_t causal, float* o_part,
                           float* lse_part, int64_t part_slots,
                           int32_t* work_meta, int32_t* dev_err, void* stream);

/* Chunked prefill with NVFP4-encoded queries: the chunk's QK^T as a
 * block-scaled FP4 x FP4 tensor-core product on the cache's own codes.
 * ([NVFP4-page] "Why NVFP4 KV changes the math": K is E2M1 codes with an E4M3
 * scale per 16 elements and an fp32 per-tensor scale -- the operand format of
 * the block-scaled FP4 product; [YaRN-page] "Against vLLM: prefill loses,
 * decode wins, and one surprise": the long-context engines prefill in
 * chunks.  The pages print no such kernel; the query encoding below is this
 * library's reading.)
 *
 * Same arguments, layouts and results as paged_decode_attention (partials,
 * work_meta, dev_err, combine with split_kv_combine), except the logits:
 * each roped bf16 query row is first encoded with the cache's NVFP4 encoder
 * under the per-tensor decode scale q_scale (e = fp32(1 / (6 q_scale)); per
 * 16-element block S = E4M3_rn_satfinite(fp32(amax * e)), zero block if
 * E4M3(S) = 0, else codes E2M1_rn_satfinite(fp32(x * fp32(1 / fp32(E4M3(S) *
 * q_scale))))), and z = (q_hat . k) * sm_scale with q_hat = E2M1(code) *
 * E4M3(S) * q_scale, the query's round trip.  The block sums and their scaling
 * are exact in binary32, so z equals the plain dot product of q_hat and the
 * dequantised k up to the accumulation's rounding.  Softmax, P.V (fp16 P,
 * dequantised V), LSE and the causal rule are paged_decode_attention's.
 *   q_scale   per-tensor decode scale g_Q of the queries, in [2^-100, 2^100];
 *             the caller calibrates it (e.g. amax(q) / (6 * 448))
 * Only NVFP4 pools, and only requests with more than 64 query rows per KV
 * head (num_q_heads / num_kv_heads * max_qlen > 64: a prefill chunk, the
 * tensor-core tile path); anything else returns PNKV_ERR_UNSUPPORTED. */
int paged_prefill_attention_fp4q(const pnkv_cache* cache, const uint16_t* q_roped,
                                 const int32_t* qo_indptr, const int32_t* page_table,
                                 int64_t pt_stride, const int32_t* seq_lens, int32_t batch,
                                 int64_t total_q, int32_t num_q_heads, int32_t max_qlen,
                                 float sm_scale, int32_t causal, float q_scale, float* o_part,
                                 float* lse_part, int64_t part_slots, int32_t* work_meta,
                                 int32_t* dev_err, void* stream);

/* Log-sum-exp merge of the split partials ([TP2-README] "Limitations",
 * split-KV decode; the merge is the standard one):
 *   M = max_s lse_s,  out = sum_s e^(lse_s - M) o_s / sum_s e^(lse_s - M),
 *   lse = M + ln sum_s e^(lse_s - M),
 * splits with lse_s = -inf weigh 0; a row with no visible key gets out = 0,
 * lse = -inf.
 *   o_part, lse_part, work_meta  as written by paged_decode_attention
 *   qo_indptr   device int32 [batch + 1] (the same as for the decode call)
 *   total_q     qo_indptr[batch] (host copy)
 *   out         device [total_q, num_q_heads, head_dim], bf16 (RNE of the
 *               fp32 result) or fp32 when out_is_fp32
 *   lse_out     device fp32 [total_q, num_q_heads], natural log, or NULL */
int split_kv_combine(const float* o_part, const float* lse_part,
                     const int32_t* work_meta, const int32_t* qo_indptr,
                     int32_t batch, int64_t total_q, int32_t num_q_heads,
                     int32_t num_kv_heads, int32_t head_dim, int32_t max_qlen,
                     void* out, int32_t out_is_fp32, float* lse_out,
                     void* stream);

/* Bytes of the fixed device scratch behind paged_decode_attention_noalloc. */
#define PNKV_NOALLOC_SCRATCH_BYTES (8u << 20)

/* paged_decode_attention followed by split_kv_combine, allocating nothing.
 * (No counterpart in the pages: this is a convenience of this library.)
 *
 * For callers that cannot allocate device memory for the split-KV partials:
 * an engine whose device memory is all reserved up front by its own
 * allocator and that does not let libraries call cudaMalloc, a
 * latency-critical loop in which cudaMalloc could synchronise the device,
 * or C code with no tensor library at hand.  The partials live instead in a
 * fixed scratch array of PNKV_NOALLOC_SCRATCH_BYTES (8 MiB) inside the
 * library's own device memory; every GPU that loads the library holds it
 * until the process exits.  The caller passes only inputs and outputs.
 *   - Arguments and results are those of paged_decode_attention and
 *     split_kv_combine (total_q = qo_indptr[batch], host copy; out bf16, or
 *     fp32 when out_is_fp32; lse_out may be NULL).
 *   - Requests whose partials do not fit the scratch -- pnkv_decode_slots(...)
 *     slots of num_q_heads / num_kv_heads * max_qlen rows of 257 floats, plus
 *     the work metadata -- return PNKV_ERR_INVALID_ARG before anything is
 *     launched.  On the split-KV path (at most 64 rows per KV head) the slot
 *     count is batch * num_kv_heads + SM count; on the tensor-core tile path
 *     (more rows) it is batch * num_kv_heads * key splits, which for a
 *     prefill chunk of thousands of tokens normally exceeds the scratch.
 *   - The first call on a device looks up the scratch's device address with
 *     that device current; make that first call before any stream capture.
 *   - No scratch content needs to start at zero: each call writes every
 *     metadata entry and partial that its own combine reads.
 *   - All calls share the one scratch: calls that overlap on the GPU (on
 *     different streams, or from several threads) race and corrupt each
 *     other's results; serialise them.
 *   - Calls no cudaMalloc, cudaFree or allocating library routine. */
int paged_decode_attention_noalloc(const pnkv_cache* cache, const uint16_t* q_roped,
                                   const int32_t* qo_indptr, const int32_t* page_table,
                                   int64_t pt_stride, const int32_t* seq_lens, int32_t batch,
                                   int32_t num_q_heads, int32_t max_qlen, float sm_scale,
                                   int32_t causal, int64_t total_q, void* out,
                                   int32_t out_is_fp32, float* lse_out, int32_t* dev_err,
                                   void* stream);

/* Bound, in nanoseconds, of every pipeline wait (an mbarrier wait between
 * the roles of a CTA) in kernels launched after this call; returns the
 * previous bound, or PNKV_ERR_INVALID_ARG for ns outside [1,000, 6e10].
 * Default 2e9 (2 s): generous, because a shared GPU may be time-sliced.
 * When a wait runs out the kernel sets PNKV_DEV_ERR_TIMEOUT in dev_err, its
 * other warps stop at their next wait, and it returns; waits for bulk copies
 * or MMAs already issued keep the 2 s bound, so no CTA exits with work in
 * flight.  Process-wide, for every device; a diagnostic and test knob (a
 * short bound makes ordinary waits run out). */
int64_t pnkv_set_wait_limit_ns(int64_t ns);

/* Static text for a status code. */
const char* pnkv_status_string(int status);

/* ABI version of this library (major * 100 + minor). */
int pnkv_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PNKV_H */
