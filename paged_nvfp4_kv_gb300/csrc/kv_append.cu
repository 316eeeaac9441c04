// kv_append_nvfp4: fused rope + quantise + page scatter for the step's new
// tokens (NVFP4, FP8, INT8 group-64 or bf16 pools).
//
// Rope with the YaRN table, mscale already inside cos/sin ("A 1,048,576-token
// context on two RTX 5090s", section "YaRN, and matching what vLLM actually
// does": the scale is applied in the rope kernel on the rotary dims), then the
// two-level NVFP4 encoding of the cache ("262,144 Tokens on One RTX 5090",
// section "Why NVFP4 KV changes the math": E2M1 codes with an FP8 E4M3 scale
// per 16 elements and one fp32 scale per tensor).  Every fp32 step is one
// IEEE operation with round-to-nearest (no contraction into FMAs), so the
// bytes written are a pure function of the inputs.  An FP8 pool (the fp8 KV
// cache of the comparison engine in "A 1,048,576-token context on two RTX
// 5090s", section "Against vLLM: prefill loses, decode wins, and one
// surprise") stores E4M3(x * fp32(1/g)) per element with one scale g per
// tensor.  An INT8 pool (the TP2 README's million-token cache, sections
// "Dual-GPU (TP2) and YaRN 1M context" and "Memory, per GPU": INT8 with one
// scale per 64 elements) stores s = fp16_rn_satfinite(fp32(a / 127)) per
// 64-element group and codes RNE(fp32(x * fp32(1/s))) clamped to +-127.
//
// One warp per (token, head) row of 256 elements: lane l owns elements
// 8l .. 8l+7 (one 16-byte load).  Rope partners (j, j + R/2) sit R/16 lanes
// apart; an NVFP4 block of 16 elements is the lane pair (2m, 2m+1).
#include "device_common.cuh"
#include "host_common.h"

namespace pnkv {

int check_yarn(const pnkv_yarn_params* p);

namespace {

struct AppendArgs {
  uint8_t* pool;
  int64_t num_pages;
  int64_t page_bytes;
  int64_t rec_bytes;
  int32_t num_kv_heads;
  int32_t dtype;
  float k_scale, v_scale;
  const int32_t* page_table;
  int64_t pt_stride;
  int32_t batch;
  const int32_t* tok_seq;
  const int32_t* tok_pos;
  int64_t num_tokens;
  const uint16_t* q;
  uint16_t* q_out;
  int32_t num_q_heads;
  const uint16_t* k;
  const uint16_t* v;
  const float* cos_t;
  const float* sin_t;
  int64_t table_rows;
  int32_t rotary_dim;
  int32_t* dev_err;
};

// E4M3 code of a binary32 value: round to nearest even, saturate at 448; the
// sign bit is the value's (tiny negatives give code 0x80 whatever the
// conversion does with the sign of a zero result).
__device__ __forceinline__ uint32_t e4m3_code(float y) {
  return (f32_to_e4m3_satfinite(y) & 0xFFu) | ((__float_as_uint(y) >> 31) << 7);
}

// INT8 group-64: this lane's 8 elements are part of the group of lanes
// 8m .. 8m+7.  Returns the 8 codes (two words, element i in byte i % 4 of
// word i / 4); *scale gets the group's fp16 scale bits.
__device__ __forceinline__ uint2 quantize8_int8(const float (&x)[8], uint32_t* scale) {
  float a = 0.f;
#pragma unroll
  for (int e = 0; e < 8; ++e) a = fmaxf(a, fabsf(x[e]));
  a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
  a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
  a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 4));
  // satfinite: values past the largest fp16 clamp to it before the rounding
  const __half s16 = __float2half_rn(fminf(__fdiv_rn(a, 127.0f), 65504.0f));
  const float d = __half2float(s16);
  uint2 out = make_uint2(0, 0);
  if (d != 0.f) {
    const float r = __frcp_rn(d);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int q = max(-127, min(127, __float2int_rn(__fmul_rn(x[e], r))));
      const uint32_t b = static_cast<uint32_t>(q) & 0xFFu;
      if (e < 4) out.x |= b << (8 * e);
      else out.y |= b << (8 * (e - 4));
    }
    *scale = __half_as_ushort(s16);
  } else {
    *scale = 0;
  }
  return out;
}

// Quantise this lane's 8 elements (part of the 16-element block shared with
// lane ^ 1).  Returns 8 packed nibbles; *scale_byte gets the block's E4M3
// scale byte.
__device__ __forceinline__ uint32_t quantize8(const float (&x)[8], float g, uint32_t* scale_byte) {
  float a = 0.f;
#pragma unroll
  for (int e = 0; e < 8; ++e) a = fmaxf(a, fabsf(x[e]));
  a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
  const float enc = __double2float_rn(1.0 / (6.0 * static_cast<double>(g)));
  float r;
  *scale_byte = nvfp4_block_scale(a, g, enc, &r);
  uint32_t codes = 0;
  if (*scale_byte != 0) {
#pragma unroll
    for (int e = 0; e < 8; ++e) codes |= e2m1_code(__fmul_rn(x[e], r)) << (4 * e);
  }
  return codes;
}

__device__ __forceinline__ void unpack_bf16x8(const uint4& w, float (&x)[8]) {
  const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    x[2 * i] = __uint_as_float(ws[i] << 16);
    x[2 * i + 1] = __uint_as_float(ws[i] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ uint4 pack_bf16x8(const float (&x)[8]) {
  uint32_t ws[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) ws[i] = f32_to_bf16_bits(x[2 * i]) | (f32_to_bf16_bits(x[2 * i + 1]) << 16);
  return make_uint4(ws[0], ws[1], ws[2], ws[3]);
}

// Rope this lane's 8 elements in place (x holds the bf16 values as fp32).
__device__ __forceinline__ void rope8(float (&x)[8], const uint4& raw, int lane, int64_t pos,
                                      const AppendArgs& a) {
  const int R = a.rotary_dim;
  const int half = R >> 1;
  const int partner = R >> 4;  // lanes between j and j + R/2
  // every lane takes part in the shuffles; only lanes below R/8 use them
  uint4 other;
  other.x = __shfl_xor_sync(0xffffffffu, raw.x, partner);
  other.y = __shfl_xor_sync(0xffffffffu, raw.y, partner);
  other.z = __shfl_xor_sync(0xffffffffu, raw.z, partner);
  other.w = __shfl_xor_sync(0xffffffffu, raw.w, partner);
  if (8 * lane >= R) return;
  float y[8];
  unpack_bf16x8(other, y);
  const bool first = 8 * lane < half;
  const int i0 = first ? 8 * lane : 8 * lane - half;
  const float4* cp = reinterpret_cast<const float4*>(a.cos_t + pos * half + i0);
  const float4* sp = reinterpret_cast<const float4*>(a.sin_t + pos * half + i0);
  const float4 c0 = __ldg(cp), c1 = __ldg(cp + 1), s0 = __ldg(sp), s1 = __ldg(sp + 1);
  const float c[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
  const float s[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    // first half:  x_j c - x_{j+R/2} s ; second half: x_j c + x_{j-R/2} s
    const float xc = __fmul_rn(x[e], c[e]);
    const float ys = __fmul_rn(y[e], s[e]);
    x[e] = first ? __fsub_rn(xc, ys) : __fadd_rn(xc, ys);
  }
#pragma unroll
  for (int e = 0; e < 8; ++e) x[e] = __uint_as_float(f32_to_bf16_bits(x[e]) << 16);
}

__global__ void __launch_bounds__(256) kv_append_kernel(AppendArgs a) {
  griddep_wait();
  griddep_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int warps_per_block = blockDim.x >> 5;
  const int hq = a.q ? a.num_q_heads : 0;
  const int rows_per_tok = hq + a.num_kv_heads;
  const int64_t rows = a.num_tokens * rows_per_tok;
  for (int64_t row = static_cast<int64_t>(blockIdx.x) * warps_per_block + (threadIdx.x >> 5); row < rows;
       row += static_cast<int64_t>(gridDim.x) * warps_per_block) {
    const int64_t n = row / rows_per_tok;
    const int h = static_cast<int>(row - n * rows_per_tok);
    const int32_t b = __ldg(a.tok_seq + n);
    const int32_t pos = __ldg(a.tok_pos + n);
    if (pos < 0 || pos >= a.table_rows) {
      if (lane == 0) flag_error(a.dev_err, PNKV_DEV_ERR_POSITION);
      continue;
    }
    if (h < hq) {  // ---- query row: rope only
      const uint4 raw = __ldg(reinterpret_cast<const uint4*>(a.q + (n * hq + h) * 256) + lane);
      float x[8];
      unpack_bf16x8(raw, x);
      rope8(x, raw, lane, pos, a);
      reinterpret_cast<uint4*>(a.q_out + (n * hq + h) * 256)[lane] = pack_bf16x8(x);
      continue;
    }
    // ---- KV row
    const int kh = h - hq;
    if (b < 0 || b >= a.batch) {
      if (lane == 0) flag_error(a.dev_err, PNKV_DEV_ERR_SEQ_INDEX);
      continue;
    }
    if ((pos >> 4) >= a.pt_stride) {
      if (lane == 0) flag_error(a.dev_err, PNKV_DEV_ERR_SEQ_LEN);
      continue;
    }
    const int32_t page = __ldg(a.page_table + b * a.pt_stride + (pos >> 4));
    if (page < 0 || page >= a.num_pages) {
      if (lane == 0) flag_error(a.dev_err, PNKV_DEV_ERR_PAGE_ID);
      continue;
    }
    const int slot = pos & 15;
    const int64_t kv_off = (n * a.num_kv_heads + kh) * 256;
    const uint4 kraw = __ldg(reinterpret_cast<const uint4*>(a.k + kv_off) + lane);
    const uint4 vraw = __ldg(reinterpret_cast<const uint4*>(a.v + kv_off) + lane);
    float kx[8], vx[8];
    unpack_bf16x8(kraw, kx);
    unpack_bf16x8(vraw, vx);
    rope8(kx, kraw, lane, pos, a);
    uint8_t* rec = a.pool + page * a.page_bytes + static_cast<int64_t>(kh) * a.rec_bytes;
    if (a.dtype == PNKV_KV_BF16) {
      reinterpret_cast<uint4*>(rec + slot * 512)[lane] = pack_bf16x8(kx);
      reinterpret_cast<uint4*>(rec + 8192 + slot * 512)[lane] = vraw;
    } else if (a.dtype == PNKV_KV_INT8) {
      // K codes [16][256]: dim 8*lane + i at 64*(2*(lane & 1) + i/4) +
      // 4*(lane/2) + i%4 of the slot's row (two 4-byte runs); V codes
      // [8 pairs][256 positions][2]: dim 8*lane + i at position 32*i + lane;
      // scales [16][4] fp16 after each
      uint32_t ks, vs;
      const uint2 kc = quantize8_int8(kx, &ks);
      const uint2 vc = quantize8_int8(vx, &vs);
      const int p0 = 128 * (lane & 1) + 4 * (lane >> 1);
      *reinterpret_cast<uint32_t*>(rec + slot * 256 + p0) = kc.x;
      *reinterpret_cast<uint32_t*>(rec + slot * 256 + p0 + 64) = kc.y;
      uint8_t* vrow = rec + 4224 + (slot >> 1) * 512 + 2 * lane + (slot & 1);
#pragma unroll
      for (int i = 0; i < 8; ++i) vrow[64 * i] = static_cast<uint8_t>(((i < 4 ? vc.x : vc.y) >> (8 * (i & 3))) & 0xFFu);
      if ((lane & 7) == 0) {
        reinterpret_cast<uint16_t*>(rec + 4096 + slot * 8)[lane >> 3] = static_cast<uint16_t>(ks);
        reinterpret_cast<uint16_t*>(rec + 8320 + slot * 8)[lane >> 3] = static_cast<uint16_t>(vs);
      }
    } else if (a.dtype == PNKV_KV_FP8) {
      // K codes [16][256]: bytes 8*lane .. +7 of the slot's row; V codes
      // [8 pairs][256][2]: byte 2d + (slot odd) of the pair's row
      const float rk = __frcp_rn(a.k_scale), rv = __frcp_rn(a.v_scale);
      uint32_t lo = 0, hi = 0;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        lo |= e4m3_code(__fmul_rn(kx[e], rk)) << (8 * e);
        hi |= e4m3_code(__fmul_rn(kx[e + 4], rk)) << (8 * e);
      }
      reinterpret_cast<uint2*>(rec + slot * 256)[lane] = make_uint2(lo, hi);
      uint8_t* vrow = rec + 4096 + (slot >> 1) * 512 + (slot & 1);
#pragma unroll
      for (int e = 0; e < 8; ++e) vrow[2 * (8 * lane + e)] = static_cast<uint8_t>(e4m3_code(__fmul_rn(vx[e], rv)));
    } else {
      uint32_t ks, vs;
      const uint32_t kc = quantize8(kx, a.k_scale, &ks);
      const uint32_t vc = quantize8(vx, a.v_scale, &vs);
      reinterpret_cast<uint32_t*>(rec + slot * 128)[lane] = kc;
      // V codes: this slot's nibble of bytes 8*lane .. 8*lane+7 of its pair
      // row; the pair's other slot may be written concurrently, so the two
      // nibble sets are replaced with atomics that leave the other untouched
      uint64_t bits = 0;
#pragma unroll
      for (int e = 0; e < 8; ++e) bits |= static_cast<uint64_t>((vc >> (4 * e)) & 0xFu) << (8 * e);
      const int sh = 4 * (slot & 1);
      unsigned long long* vw = reinterpret_cast<unsigned long long*>(rec + 2304 + (slot >> 1) * 256) + lane;
      atomicAnd(vw, ~(0x0F0F0F0F0F0F0F0Full << sh));
      atomicOr(vw, static_cast<unsigned long long>(bits << sh));
      if ((lane & 1) == 0) {
        rec[2048 + slot * 16 + (lane >> 1)] = static_cast<uint8_t>(ks);
        rec[4352 + slot * 16 + (lane >> 1)] = static_cast<uint8_t>(vs);
      }
    }
  }
}

}  // namespace
}  // namespace pnkv

extern "C" int kv_append_nvfp4(const pnkv_cache* cache, const int32_t* page_table, int64_t pt_stride,
                               int32_t batch, const int32_t* tok_seq, const int32_t* tok_pos,
                               int64_t num_tokens, const uint16_t* q, uint16_t* q_out,
                               int32_t num_q_heads, const uint16_t* k, const uint16_t* v,
                               const float* cos_t, const float* sin_t, int64_t table_rows,
                               int32_t rotary_dim, int32_t* dev_err, void* stream) {
  using namespace pnkv;
  int st = check_cache(cache);
  if (st != PNKV_OK) return st;
  if (cache->dtype == PNKV_KV_NVFP4 || cache->dtype == PNKV_KV_FP8) {
    // keep d = E4M3(S) * g (NVFP4), 1/g (FP8) and 1/d normal binary32 numbers
    const float lo = 7.8886091e-31f, hi = 1.2676506e30f;  // 2^-100, 2^100
    if (cache->k_scale < lo || cache->k_scale > hi || cache->v_scale < lo || cache->v_scale > hi)
      return PNKV_ERR_INVALID_ARG;
  }
  if (num_tokens < 0 || pt_stride < 1 || batch < 1 || table_rows < 1) return PNKV_ERR_INVALID_ARG;
  if (!(rotary_dim == 16 || rotary_dim == 32 || rotary_dim == 64 || rotary_dim == 128 ||
        rotary_dim == 256))
    return PNKV_ERR_INVALID_ARG;
  if ((q == nullptr) != (q_out == nullptr)) return PNKV_ERR_INVALID_ARG;
  if (q && (num_q_heads < 1 || num_q_heads > 256)) return PNKV_ERR_INVALID_ARG;
  if (num_tokens == 0) return PNKV_OK;
  if (!page_table || !tok_seq || !tok_pos || !k || !v || !cos_t || !sin_t || !dev_err)
    return PNKV_ERR_INVALID_ARG;
  if (!aligned(k, 16) || !aligned(v, 16) || !aligned(cos_t, 16) || !aligned(sin_t, 16) ||
      (q && (!aligned(q, 16) || !aligned(q_out, 16))))
    return PNKV_ERR_INVALID_ARG;
  AppendArgs a;
  a.pool = static_cast<uint8_t*>(cache->pool);
  a.num_pages = cache->num_pages;
  a.rec_bytes = head_record_bytes(cache->dtype);
  a.page_bytes = a.rec_bytes * cache->num_kv_heads;
  a.num_kv_heads = cache->num_kv_heads;
  a.dtype = cache->dtype;
  a.k_scale = cache->k_scale;
  a.v_scale = cache->v_scale;
  a.page_table = page_table;
  a.pt_stride = pt_stride;
  a.batch = batch;
  a.tok_seq = tok_seq;
  a.tok_pos = tok_pos;
  a.num_tokens = num_tokens;
  a.q = q;
  a.q_out = q_out;
  a.num_q_heads = q ? num_q_heads : 0;
  a.k = k;
  a.v = v;
  a.cos_t = cos_t;
  a.sin_t = sin_t;
  a.table_rows = table_rows;
  a.rotary_dim = rotary_dim;
  a.dev_err = dev_err;
  int sms = 0;
  if ((st = device_sm_count(&sms)) != PNKV_OK) return st;
  const int64_t rows = num_tokens * (a.num_q_heads + a.num_kv_heads);
  int64_t blocks = (rows + 7) / 8;
  const int64_t cap = static_cast<int64_t>(sms) * 16;
  if (blocks > cap) blocks = cap;
  return launch_pdl(kv_append_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0,
                    as_stream(stream), a);
}
