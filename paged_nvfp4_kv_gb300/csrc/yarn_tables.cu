// yarn_rope_tables: YaRN cos/sin tables on the device.
//
// The method (YaRN, Peng et al. 2023, "NTK-by-parts" interpolation and the
// attention temperature; "A 1,048,576-token context on two RTX 5090s",
// section "YaRN, and matching what vLLM actually does"; "NInfer -- Windows 11
// TP2 fork" README, section "YaRN reference and drift guard"):
//   f_i       = theta^(-2i/R)                      original frequency of pair i
//   corr(n)   = R ln(L / (2 pi n)) / (2 ln theta)  pair index that turns n
//                                                  times over L positions
//   L         = original_max * s (deployed range) or original_max (paper)
//   low, high = max(floor(corr(beta_fast)), 0), min(ceil(corr(beta_slow)), R-1)
//   ramp_i    = clamp((i - low) / (high - low), 0, 1)   (high += 0.001 if equal)
//   inv_i     = (f_i / s) * ramp_i + f_i * (1 - ramp_i)
//   mscale    = 0.1 ln s + 1  (1 when s <= 1), folded into cos and sin
//   table     = fp32(mscale * cos(p * inv_i)), fp32(mscale * sin(p * inv_i))
// Everything before the final rounding is double precision.
#include <cmath>

#include "device_common.cuh"
#include "host_common.h"

namespace pnkv {
namespace {

struct YarnArgs {
  double theta, factor, ctx_len, beta_fast, beta_slow;
  int rotary_dim;
};

__device__ double correction_dim(double n_rot, const YarnArgs& a) {
  return a.rotary_dim * log(a.ctx_len / (n_rot * 2.0 * 3.14159265358979323846)) /
         (2.0 * log(a.theta));
}

__global__ void __launch_bounds__(256) yarn_tables_kernel(YarnArgs a, int64_t max_pos,
                                                          float* __restrict__ cos_out,
                                                          float* __restrict__ sin_out) {
  __shared__ double inv_freq[128];
  __shared__ double msc;
  const int half = a.rotary_dim / 2;
  if (threadIdx.x == 0) msc = a.factor <= 1.0 ? 1.0 : __dadd_rn(__dmul_rn(0.1, log(a.factor)), 1.0);
  if (threadIdx.x < half) {
    const int i = threadIdx.x;
    double low = floor(correction_dim(a.beta_fast, a));
    double high = ceil(correction_dim(a.beta_slow, a));
    low = fmax(low, 0.0);
    high = fmin(high, static_cast<double>(a.rotary_dim - 1));
    if (low == high) high += 0.001;
    double ramp = (static_cast<double>(i) - low) / (high - low);
    ramp = fmin(fmax(ramp, 0.0), 1.0);
    const double f = pow(a.theta, -2.0 * i / a.rotary_dim);
    const double keep = 1.0 - ramp;
    // separate roundings (no fused multiply-add), as the definition reads
    inv_freq[i] = __dadd_rn(__dmul_rn(f / a.factor, 1.0 - keep), __dmul_rn(f, keep));
  }
  __syncthreads();
  const int shift = __ffs(half) - 1;  // half is a power of two
  const int64_t total = max_pos * half;
  const double m = msc;
  for (int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; idx < total;
       idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t pos = idx >> shift;
    const int i = static_cast<int>(idx & (half - 1));
    const double ang = static_cast<double>(pos) * inv_freq[i];
    double s, c;
    sincos(ang, &s, &c);
    cos_out[idx] = __double2float_rn(m * c);
    sin_out[idx] = __double2float_rn(m * s);
  }
}

bool valid_rotary_dim(int r) { return r == 16 || r == 32 || r == 64 || r == 128 || r == 256; }

}  // namespace

// Validation shared with the append call ("NInfer -- Windows 11 TP2 fork"
// README, section "Usage": factor finite in [1, 64], original window times
// factor a whole token count no larger than 1,048,576).
int check_yarn(const pnkv_yarn_params* p) {
  if (!p) return PNKV_ERR_INVALID_ARG;
  if (!std::isfinite(p->factor) || p->factor < 1.0 || p->factor > 64.0) return PNKV_ERR_INVALID_ARG;
  if (p->original_max <= 0) return PNKV_ERR_INVALID_ARG;
  const double window = static_cast<double>(p->original_max) * p->factor;
  if (window != std::floor(window) || window > 1048576.0) return PNKV_ERR_INVALID_ARG;
  if (!std::isfinite(p->theta) || !(p->theta > 1.0)) return PNKV_ERR_INVALID_ARG;
  if (!std::isfinite(p->beta_fast) || !std::isfinite(p->beta_slow) || !(p->beta_slow > 0.0) ||
      !(p->beta_fast > p->beta_slow))
    return PNKV_ERR_INVALID_ARG;
  if (!valid_rotary_dim(p->rotary_dim)) return PNKV_ERR_INVALID_ARG;
  if (p->deployed_range != 0 && p->deployed_range != 1) return PNKV_ERR_INVALID_ARG;
  return PNKV_OK;
}

}  // namespace pnkv

extern "C" int yarn_rope_tables(const pnkv_yarn_params* params, int64_t max_pos, float* cos_out,
                                float* sin_out, void* stream) {
  using namespace pnkv;
  int st = check_yarn(params);
  if (st != PNKV_OK) return st;
  if (max_pos < 1 || max_pos > 2147483647LL || !cos_out || !sin_out || !aligned(cos_out, 4) ||
      !aligned(sin_out, 4))
    return PNKV_ERR_INVALID_ARG;
  YarnArgs a;
  a.theta = params->theta;
  a.factor = params->factor;
  a.ctx_len = params->deployed_range ? static_cast<double>(params->original_max) * params->factor
                                     : static_cast<double>(params->original_max);
  a.beta_fast = params->beta_fast;
  a.beta_slow = params->beta_slow;
  a.rotary_dim = params->rotary_dim;
  int sms = 0;
  if ((st = device_sm_count(&sms)) != PNKV_OK) return st;
  const int64_t total = max_pos * (params->rotary_dim / 2);
  int64_t blocks = (total + 255) / 256;
  const int64_t cap = static_cast<int64_t>(sms) * 8;
  if (blocks > cap) blocks = cap;
  yarn_tables_kernel<<<static_cast<unsigned>(blocks), 256, 0, as_stream(stream)>>>(a, max_pos, cos_out,
                                                                                 sin_out);
  return launch_status();
}
