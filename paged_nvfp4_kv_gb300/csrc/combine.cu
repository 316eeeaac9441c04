// split_kv_combine: log-sum-exp merge of the split-KV partials.
//
// For an output row with split partials (o_s, lse_s), s = 1..n ("NInfer --
// Windows 11 TP2 fork" README, section "Limitations": split-KV decode; the
// merge is the standard identity for a softmax split over disjoint key sets):
//   M = max_s lse_s,  w_s = e^(lse_s - M),  out = sum_s w_s o_s / sum_s w_s,
//   lse = M + ln sum_s w_s.
// A split with lse_s = -inf (no visible key) weighs 0; a row with no visible
// key at all gets out = 0 and lse = -inf.
//
// The partials are read once, coalesced (1 KiB per split per row).
#include <cmath>

#include "device_common.cuh"
#include "host_common.h"

namespace pnkv {
namespace {

struct CombineArgs {
  const float* o_part;
  const float* lse_part;
  const int32_t* meta;
  const int32_t* qo_indptr;
  int32_t batch;
  int64_t total_q;
  int32_t hq, hkv, group, rows_per_slot;
  void* out;
  int32_t out_fp32;
  float* lse_out;
};

// One 256-thread block per output row.  The row's split LSEs are read once
// into shared memory (max, then weights); then four groups of 64 threads each
// stream every fourth split (thread j of a group owns dims 4j .. 4j+3), so
// four times as many loads are in flight, and the groups' sums are added in a
// fixed order.
constexpr int kThreads = 256;
constexpr int kGroups = kThreads / 64;
constexpr int kMaxCached = 1024;  // splits whose LSE and weight fit in shared memory

__device__ __forceinline__ float block_reduce(float v, bool is_max, float* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float x = __shfl_xor_sync(0xffffffffu, v, o);
    v = is_max ? fmaxf(v, x) : v + x;
  }
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float r = red[0];
#pragma unroll
  for (int i = 1; i < kThreads / 32; ++i) r = is_max ? fmaxf(r, red[i]) : r + red[i];
  __syncthreads();
  return r;
}

__global__ void __launch_bounds__(kThreads) combine_kernel(const CombineArgs a) {
  __shared__ float w_s[kMaxCached];
  __shared__ float red[kThreads / 32];
  __shared__ float4 part[kGroups - 1][64];
  griddep_wait();
  griddep_launch_dependents();
  const int tid = threadIdx.x;
  const int64_t row = blockIdx.x;
  const int64_t t = row / a.hq;
  const int h = static_cast<int>(row - t * a.hq);
  // sequence of token t: last b with qo_indptr[b] <= t
  int lo = 0, hi = a.batch - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(a.qo_indptr + mid) <= t) lo = mid;
    else hi = mid - 1;
  }
  const int b = lo;
  const int64_t seg = static_cast<int64_t>(b) * a.hkv + h / a.group;
  const int32_t first = __ldg(a.meta + 4 + 2 * seg);
  int32_t cnt = __ldg(a.meta + 4 + 2 * seg + 1);
  const int r = static_cast<int>((t - __ldg(a.qo_indptr + b)) * a.group + h % a.group);
  if (!(cnt > 0 && first >= 0 && r < a.rows_per_slot)) cnt = 0;
  const float* lse = a.lse_part + static_cast<int64_t>(first) * a.rows_per_slot + r;
  auto lse_at = [&](int s) -> float {
    return s < kMaxCached ? w_s[s] : __ldg(lse + static_cast<int64_t>(s) * a.rows_per_slot);
  };

  // M = max_s lse_s (the LSEs are kept in w_s)
  float M = -INFINITY;
  for (int s = tid; s < cnt; s += kThreads) {
    const float l = __ldg(lse + static_cast<int64_t>(s) * a.rows_per_slot);
    if (s < kMaxCached) w_s[s] = l;
    M = fmaxf(M, l);
  }
  M = block_reduce(M, true, red);
  // weights e^(lse_s - M) in place, and their sum
  float wsum = 0.f;
  if (M != -INFINITY) {
    for (int s = tid; s < cnt; s += kThreads) {
      const float l = lse_at(s);
      const float w = (l == -INFINITY) ? 0.f : expf(l - M);
      if (s < kMaxCached) w_s[s] = w;
      wsum += w;
    }
  }
  wsum = block_reduce(wsum, false, red);  // (its barrier also publishes w_s)

  const int g = tid >> 6, j = tid & 63;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (wsum > 0.f) {
    const float4* src = reinterpret_cast<const float4*>(
        a.o_part + (static_cast<int64_t>(first) * a.rows_per_slot + r) * 256) + j;
    const int64_t step = static_cast<int64_t>(a.rows_per_slot) * 64;  // float4s per slot
#pragma unroll 4
    for (int s = g; s < cnt; s += kGroups) {
      float w;
      if (s < kMaxCached) {
        w = w_s[s];
      } else {
        const float l = __ldg(lse + static_cast<int64_t>(s) * a.rows_per_slot);
        w = (l == -INFINITY) ? 0.f : expf(l - M);
      }
      const float4 x = __ldg(src + s * step);
      acc.x += w * x.x;
      acc.y += w * x.y;
      acc.z += w * x.z;
      acc.w += w * x.w;
    }
  }
  if (g > 0) part[g - 1][j] = acc;
  __syncthreads();
  if (g == 0) {
#pragma unroll
    for (int k = 0; k < kGroups - 1; ++k) {
      const float4 x = part[k][j];
      acc.x += x.x;
      acc.y += x.y;
      acc.z += x.z;
      acc.w += x.w;
    }
    if (wsum > 0.f) {
      const float inv = 1.f / wsum;
      acc.x *= inv;
      acc.y *= inv;
      acc.z *= inv;
      acc.w *= inv;
    }
    const int64_t base = row * 256 + 4 * j;
    if (a.out_fp32) {
      *reinterpret_cast<float4*>(static_cast<float*>(a.out) + base) = acc;
    } else {
      const uint32_t w0 = f32_to_bf16_bits(acc.x) | (f32_to_bf16_bits(acc.y) << 16);
      const uint32_t w1 = f32_to_bf16_bits(acc.z) | (f32_to_bf16_bits(acc.w) << 16);
      *reinterpret_cast<uint2*>(static_cast<uint16_t*>(a.out) + base) = make_uint2(w0, w1);
    }
    if (a.lse_out && j == 0) a.lse_out[row] = wsum > 0.f ? M + logf(wsum) : -INFINITY;
  }
}

}  // namespace
}  // namespace pnkv

extern "C" int split_kv_combine(const float* o_part, const float* lse_part, const int32_t* work_meta,
                                const int32_t* qo_indptr, int32_t batch, int64_t total_q,
                                int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                int32_t max_qlen, void* out, int32_t out_is_fp32, float* lse_out,
                                void* stream) {
  using namespace pnkv;
  if (!o_part || !lse_part || !work_meta || !qo_indptr || !out) return PNKV_ERR_INVALID_ARG;
  if (batch < 1 || total_q < 0 || num_kv_heads < 1 || num_q_heads < 1 ||
      num_q_heads % num_kv_heads != 0 || head_dim != 256 || max_qlen < 1 || max_qlen > 8192)
    return PNKV_ERR_INVALID_ARG;
  if (!aligned(o_part, 16) || !aligned(out, 16)) return PNKV_ERR_INVALID_ARG;
  if (total_q == 0) return PNKV_OK;
  CombineArgs a;
  a.o_part = o_part;
  a.lse_part = lse_part;
  a.meta = work_meta;
  a.qo_indptr = qo_indptr;
  a.batch = batch;
  a.total_q = total_q;
  a.hq = num_q_heads;
  a.hkv = num_kv_heads;
  a.group = num_q_heads / num_kv_heads;
  a.rows_per_slot = a.group * max_qlen;
  a.out = out;
  a.out_fp32 = out_is_fp32 ? 1 : 0;
  a.lse_out = lse_out;
  const int64_t rows = total_q * num_q_heads;
  if (rows > 2147483647LL) return PNKV_ERR_INVALID_ARG;
  return launch_pdl(combine_kernel, dim3(static_cast<unsigned>(rows)), dim3(kThreads), 0,
                    as_stream(stream), a);
}
