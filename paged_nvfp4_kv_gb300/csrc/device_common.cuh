// Device-side building blocks shared by the libpnkv kernels (sm_103a):
// bounded mbarrier waits, 2-D TMA tensor loads, fp8/fp4 conversions and the
// m16n8k16 tensor-core MMA, all as inline PTX.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda.h>

#include "pnkv.h"

namespace pnkv {

// ---------------------------------------------------------------- errors --
__device__ __forceinline__ void flag_error(int32_t* dev_err, int bits) {
  if (dev_err) atomicOr(dev_err, bits);
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// Default bound of a pipeline wait (the GPU is shared and may be
// time-sliced, so the bound is generous); on expiry the kernel flags
// PNKV_DEV_ERR_TIMEOUT and winds down instead of hanging.  Pipeline waits
// take their bound from the launch arguments (pnkv_set_wait_limit_ns); the
// waits of a wind-down -- for bulk copies or MMAs already issued, which always
// complete -- keep this bound, so that no CTA exits with work in flight.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

// -------------------------------------------------------------- mbarrier --
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbarrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("{ .reg .b64 st; mbarrier.arrive.shared::cta.b64 st, [%0]; }" ::"r"(smem_addr(bar))
               : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile(
      "{ .reg .b64 st; mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1; }" ::"r"(
          smem_addr(bar)),
      "r"(bytes)
      : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait until the phase with the given parity has completed.  Returns false
// (and the caller flags a timeout) if that takes longer than limit_ns.  Each
// test may suspend the thread for the hardware's own time limit (a few
// microseconds); between tests the thread sleeps 20 ns and reads the clock, so
// the bound is kept to within one test.  (Tests with an explicit suspend-time
// hint measured a few percent slower in the tensor-core tiles.)
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    __nanosleep(20);
    if (mbar_try_wait(bar, parity)) return true;
    if (globaltimer_ns() - t0 > limit_ns) return false;
  }
}

// ------------------------------------------------------------------- TMA --
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// 2-D tiled tensor load: box at (x, y) -> dst (shared), completion counted
// on `bar` in bytes.  x must be a multiple of 16 bytes' worth of elements.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int32_t x, int32_t y,
                                            uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

// ------------------------------------------- programmatic dependent launch --
// A kernel launched with programmatic stream serialisation may start before
// the previous kernel in the stream has finished; it must wait here before
// its first global memory access.  Without the launch attribute these are
// no-ops.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ------------------------------------------------------- named barriers --
__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ----------------------------------------------------------- conversions --
// Two E2M1 codes (one byte: element 2k low nibble, 2k+1 high nibble) ->
// f16x2 (low half = low nibble).  Exact.
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t byte) {
  uint32_t out;
  asm("{ .reg .b8 t; .reg .b16 w; cvt.u16.u32 w, %1; cvt.u8.u16 t, w; cvt.rn.f16x2.e2m1x2 %0, t; }"
      : "=r"(out)
      : "r"(byte));
  return out;
}

// Two E4M3 bytes (low byte -> low half) -> f16x2.  Exact.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_bytes) {
  uint32_t out;
  asm("{ .reg .b16 w; cvt.u16.u32 w, %1; cvt.rn.f16x2.e4m3x2 %0, w; }" : "=r"(out) : "r"(two_bytes));
  return out;
}

// Four E4M3 bytes as two fp16x2 (bytes 0, 1 -> lo; bytes 2, 3 -> hi; the
// lower byte of each pair in the lower half).  Exact: every E4M3 value is an
// fp16 value.
__device__ __forceinline__ void e4m3x4_to_f16x2x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
  asm("{ .reg .b16 l, h; mov.b32 {l, h}, %2; cvt.rn.f16x2.e4m3x2 %0, l; cvt.rn.f16x2.e4m3x2 %1, h; }"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
}

// Four int8 as two fp16x2 (bytes 0, 1 -> lo; bytes 2, 3 -> hi), exactly: a
// byte b biased to u = b ^ 0x80 becomes the fp16 1024 + u (its bits 0x6400 |
// u), and subtracting 1152 leaves the signed value.
__device__ __forceinline__ void s8x4_to_f16x2x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t t = w ^ 0x80808080u;
  uint32_t a, b;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(a) : "r"(t), "r"(0x64646464u), "r"(0x5150u));
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(b) : "r"(t), "r"(0x64646464u), "r"(0x5352u));
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(lo) : "r"(a), "r"(0x64806480u));
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(hi) : "r"(b), "r"(0x64806480u));
}

// fp32 -> E4M3 byte, round to nearest even, saturating to +-448.
__device__ __forceinline__ uint32_t f32_to_e4m3_satfinite(float x) {
  uint16_t out;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(out) : "f"(0.0f), "f"(x));
  return out & 0xFFu;  // second source lands in the low byte
}

// (lo, hi) fp32 -> f16x2 with round to nearest even.
__device__ __forceinline__ uint32_t f32x2_to_f16x2(float lo, float hi) {
  uint32_t out;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(out) : "f"(hi), "f"(lo));
  return out;
}

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  uint32_t out;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(out) : "r"(a), "r"(b));
  return out;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t out;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(out) : "r"(a), "r"(b), "r"(sel));
  return out;
}

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t bits16) {
  return __uint_as_float(bits16 << 16);
}

// fp32 -> bf16 bits, round to nearest even.
__device__ __forceinline__ uint32_t f32_to_bf16_bits(float x) {
  return static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(x)));
}

// ---------------------------------------------------------------- mma ----
// D = A(16x16, row) * B(16x8, col) + D, fp16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                              uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Same with bf16 inputs.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Transpose an 8x8 matrix of 16-bit elements held one 32-bit register per
// lane (row lane/4, columns 2*(lane%4) and +1).
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t out;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(out) : "r"(x));
  return out;
}

// max(a, b, c) in one instruction (a NaN operand is ignored, as by fmaxf).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

__device__ __forceinline__ uint32_t lds8(uint32_t addr) {
  uint16_t v;
  asm volatile("ld.shared.u8 %0, [%1];" : "=h"(v) : "r"(addr));
  return v;
}

__device__ __forceinline__ uint32_t lds16(uint32_t addr) {
  uint16_t v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
  return v;
}

// ------------------------------------------------------- NVFP4 encoding --
// The two-level NVFP4 encoder of the cache ("262,144 Tokens on One RTX 5090",
// section "Why NVFP4 KV changes the math": E2M1 codes with an E4M3 scale per
// 16 elements and one fp32 decode scale g per tensor), shared by the cache
// writer and the FP4-query prefill tile so that both round identically.

// E2M1 code of a binary32 value: round to nearest, ties to the even code,
// saturate at 6; the sign bit is the value's (so -0 and tiny negatives give
// code 8).  Thresholds are the midpoints of {0, .5, 1, 1.5, 2, 3, 4, 6}; at a
// midpoint the even code wins (codes 0, 2, 4, 6 hold 0, 1, 2, 4).
__device__ __forceinline__ uint32_t e2m1_code(float y) {
  const float m = fabsf(y);
  uint32_t c = (m > 0.25f) + (m >= 0.75f) + (m > 1.25f) + (m >= 1.75f) + (m > 2.5f) + (m >= 3.5f) +
               (m > 5.0f);
  return c | ((__float_as_uint(y) >> 31) << 3);
}

// Scale byte of a 16-element block whose largest magnitude is amax, for the
// decode scale g and enc = fp32(1 / (6 g)): S = E4M3_rn_satfinite(fp32(amax *
// enc)); 0 when E4M3(S) is zero (the block's codes are then all zero).
// Otherwise *r = fp32(1 / fp32(E4M3(S) * g)), the factor the codes are
// rounded from: code_i = E2M1(fp32(x_i * r)).
__device__ __forceinline__ uint32_t nvfp4_block_scale(float amax, float g, float enc, float* r) {
  const uint32_t s = f32_to_e4m3_satfinite(__fmul_rn(amax, enc));
  const float sdec = __half2float(__ushort_as_half(static_cast<unsigned short>(e4m3x2_to_f16x2(s) & 0xFFFFu)));
  if (sdec == 0.f) {
    *r = 0.f;
    return 0u;
  }
  *r = __frcp_rn(__fmul_rn(sdec, g));
  return s;
}

// Byte offset of (row, byte) inside a tile written by a 2-D TMA load with
// 128-byte swizzling and 128-byte rows, the tile starting 1024-byte aligned:
// 16-byte chunk c of row r sits at chunk position c ^ (r % 8).
__device__ __forceinline__ uint32_t swz128(uint32_t row, uint32_t byte) {
  return row * 128u + ((((byte >> 4) ^ row) & 7u) << 4) + (byte & 15u);
}


// Four E2M1 codes (the low 16 bits of w, element 2k in the low nibble of byte
// k) -> two f16x2 values, o[k] = (element 2k, element 2k+1) of byte k.  Exact.
__device__ __forceinline__ void e2m1x4_unpack(uint32_t w, uint32_t (&o)[2]) {
  asm("{ .reg .b8 b0, b1, b2, b3; mov.b32 {b0, b1, b2, b3}, %2;"
      " cvt.rn.f16x2.e2m1x2 %0, b0; cvt.rn.f16x2.e2m1x2 %1, b1; }"
      : "=r"(o[0]), "=r"(o[1]) : "r"(w));
}

// Eight E2M1 codes (one 32-bit word, element 2k in the low nibble of byte k)
// -> four f16x2 values, o[k] = (element 2k, element 2k+1) of byte k.  Exact.
__device__ __forceinline__ void e2m1x8_unpack(uint32_t w, uint32_t (&o)[4]) {
  asm("{ .reg .b8 b0, b1, b2, b3; mov.b32 {b0, b1, b2, b3}, %4;"
      " cvt.rn.f16x2.e2m1x2 %0, b0; cvt.rn.f16x2.e2m1x2 %1, b1;"
      " cvt.rn.f16x2.e2m1x2 %2, b2; cvt.rn.f16x2.e2m1x2 %3, b3; }"
      : "=r"(o[0]), "=r"(o[1]), "=r"(o[2]), "=r"(o[3]) : "r"(w));
}
}  // namespace pnkv
