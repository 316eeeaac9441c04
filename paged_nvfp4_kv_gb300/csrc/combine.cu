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
// One warp per (query token, query head) row; lane l owns dims 8l .. 8l+7.
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

__global__ void __launch_bounds__(256) combine_kernel(const CombineArgs a) {
  const int lane = threadIdx.x & 31;
  const int64_t rows = a.total_q * a.hq;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  if (row >= rows) return;
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
  const int32_t cnt = __ldg(a.meta + 4 + 2 * seg + 1);
  const int r = static_cast<int>((t - __ldg(a.qo_indptr + b)) * a.group + h % a.group);
  const bool ok = cnt > 0 && first >= 0 && r < a.rows_per_slot;

  float M = -INFINITY;
  if (ok)
    for (int s = lane; s < cnt; s += 32) M = fmaxf(M, __ldg(a.lse_part + static_cast<int64_t>(first + s) * a.rows_per_slot + r));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));

  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  float wsum = 0.f;
  if (ok && M != -INFINITY) {
    for (int s = 0; s < cnt; ++s) {
      const int64_t pr = static_cast<int64_t>(first + s) * a.rows_per_slot + r;
      const float l = __ldg(a.lse_part + pr);
      if (l == -INFINITY) continue;
      const float w = expf(l - M);
      wsum += w;
      const float4* src = reinterpret_cast<const float4*>(a.o_part + pr * 256) + 2 * lane;
      const float4 x = __ldg(src), y = __ldg(src + 1);
      acc[0] += w * x.x; acc[1] += w * x.y; acc[2] += w * x.z; acc[3] += w * x.w;
      acc[4] += w * y.x; acc[5] += w * y.y; acc[6] += w * y.z; acc[7] += w * y.w;
    }
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
#pragma unroll
  for (int e = 0; e < 8; ++e) acc[e] *= inv;
  const int64_t base = row * 256 + 8 * lane;
  if (a.out_fp32) {
    float4* dst = reinterpret_cast<float4*>(static_cast<float*>(a.out) + base);
    dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
  } else {
    uint32_t w[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) w[e] = f32_to_bf16_bits(acc[2 * e]) | (f32_to_bf16_bits(acc[2 * e + 1]) << 16);
    *reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.out) + base) = make_uint4(w[0], w[1], w[2], w[3]);
  }
  if (a.lse_out && lane == 0) a.lse_out[row] = wsum > 0.f ? M + logf(wsum) : -INFINITY;
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
  const int64_t blocks = (rows + 7) / 8;
  if (blocks > 2147483647LL) return PNKV_ERR_INVALID_ARG;
  combine_kernel<<<static_cast<unsigned>(blocks), 256, 0, as_stream(stream)>>>(a);
  return launch_status();
}
