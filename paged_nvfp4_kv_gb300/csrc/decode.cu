// paged_decode_attention: split-KV GQA decode over the paged pool.
//
// The attention is the plain softmax(q k^T * sm_scale) v of every new query
// row over the keys of its sequence (causal inside the new rows), evaluated
// in key splits whose partials are merged by split_kv_combine ("NInfer --
// Windows 11 TP2 fork" README, section "Limitations": the decode key range
// is split; "A 1,048,576-token context on two RTX 5090s", section "Things
// that bit me": no compile-time ceiling on the number of keys -- nothing here
// is sized by the context length).
//
// Work decomposition (stream-K).  The unit of work is one (sequence b, KV
// head h, page) triple: 16 tokens of one head, 4,608 bytes NVFP4 or 16 KiB
// bf16, read exactly once per call and shared by all the head's query rows
// (GQA).  Units are ordered (b, h, page) and the whole list is cut into
// gridDim.x equal contiguous ranges, one per CTA, gridDim.x = SM count; a
// CTA's range meets at most a few (b, h) segments and writes one partial per
// segment piece into slot (segment + CTA index), which is injective.
//
// Inside a CTA: warp 8 produces, warps 0..7 consume.  The producer walks the
// CTA's units, reads their page ids from the page table and issues one 2-D
// TMA load per unit (the head record as 36 or 128 rows of 128 bytes, 128-byte
// swizzle) into a ring of shared-memory stages guarded by full/empty
// mbarriers.  Consumer warp w takes every (8/RG)-th unit; for RG > 1 the RG
// warps of a group split the query rows of the same unit.  Per unit a warp
// computes S^T = K Q^T with m16n8k16 tensor-core MMAs (16 tokens of the page
// are the M dimension, query rows the N dimension, so GQA rows pad only to
// 8), keeps an online softmax per query row, and accumulates O^T += V^T P^T
// (head dims as M).  NVFP4 codes are widened in registers: E2M1 -> fp16 and
// times the E4M3 block scale, both exact in fp16; the per-tensor scales fold
// into the logit scale (K) and the output (V).  P is rounded to fp16 for the
// P.V product.  At the end of each segment piece the consumer warps merge
// their (m, l, O) in shared memory in a fixed order (deterministic) and write
// the normalised partial and its natural-log LSE.
#include <cmath>

#include <cudaTypedefs.h>

#include "decode_common.cuh"
#include "device_common.cuh"
#include "host_common.h"

namespace pnkv {

int launch_prefill(const pnkv_cache* cache, const uint16_t* q_roped, const int32_t* qo_indptr,
                   const int32_t* page_table, int64_t pt_stride, const int32_t* seq_lens, int32_t batch,
                   int64_t total_q, int32_t num_q_heads, int32_t max_qlen, float sm_scale, int32_t causal,
                   float q_scale, float* o_part, float* lse_part, int64_t part_slots, int32_t* work_meta,
                   int32_t* dev_err, cudaStream_t stream);
int prefill_splits(int32_t batch, int32_t num_kv_heads, int32_t group, int32_t max_qlen, int sms);
int launch_verify(const CUtensorMap& map, const DecodeArgs& a, int grid, cudaStream_t stream);

namespace {

// A CTA has NW warps: the last one produces, the consumers are the largest
// multiple of RG below it.  Register allocation is per 4-warp group, so up
// to 8 warps (256 threads) keep 255 registers per thread and 12 warps (384)
// keep 168: the single-n-tile NVFP4 path fits 168 and runs 11 consumers; the
// other paths need the larger budget and run with at most 8 warps.
#ifndef PNKV_ISSUE_LANES
#define PNKV_ISSUE_LANES 8
#endif
constexpr int kIssueLanes = PNKV_ISSUE_LANES;  // producer lanes that issue TMA loads together
template <int NW, int RG>
struct Consumers {
  static constexpr int kWarps = ((NW - 1) / RG) * RG;
  static constexpr int kThreads = kWarps * 32;
};
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;


template <int KVDT>
struct Geometry;
template <>
struct Geometry<PNKV_KV_NVFP4> {
  static constexpr int kBoxRows = 36;      // 4,608 B head record
  static constexpr int kStageBytes = 5120; // next multiple of 1,024
  static constexpr uint32_t kTxBytes = 4608;
};
template <>
struct Geometry<PNKV_KV_FP8> {
  static constexpr int kBoxRows = 64;      // 8,192 B head record
  static constexpr int kStageBytes = 8192;
  static constexpr uint32_t kTxBytes = 8192;
};
template <>
struct Geometry<PNKV_KV_INT8> {
  static constexpr int kBoxRows = 66;      // 8,448 B head record
  static constexpr int kStageBytes = 9216; // next multiple of 1,024
  static constexpr uint32_t kTxBytes = 8448;
};
template <>
struct Geometry<PNKV_KV_BF16> {
  static constexpr int kBoxRows = 128;     // 16,384 B head record
  static constexpr int kStageBytes = 16384;
  static constexpr uint32_t kTxBytes = 16384;
};

// ---------------------------------------------------------------------------
// Shared memory plan.

// The stage count is a multiple of the number of consumer streams, so unit
// i always lands in a stage that only stream i % kStreams reads: a consumer
// then waits on a stage whose previous round it consumed itself, i.e. never
// more than one barrier phase ahead (a parity wait cannot tell phase k from
// phase k + 2, so a wait two phases ahead would pass on stale data).
template <int KVDT, int NTW, int RG, int NW, int QS>
struct Plan {
  static constexpr int kStreams = Consumers<NW, RG>::kWarps / RG;   // warps that split the units
  static constexpr int kRows = 8 * NTW * RG;             // query rows per KV head handled
  static constexpr int kMergeBytes = kRows * 256 * 4;
  static constexpr int kMlBytes = kStreams * kRows * 2 * 4;
  static constexpr int kQBytes = QS ? NTW * RG * 16 * 32 * 8 : 0;  // Q fragments in shared memory
  // per stage: its bytes plus two mbarriers and two int32 (valid, armed)
  static constexpr int kFixed = kMergeBytes + kMlBytes + kQBytes + 1024 /*align*/ + 64 /*flags, padding*/;
  static constexpr int kMaxSmem = 232448;
  static constexpr int kStagesFit = (kMaxSmem - kFixed) / (Geometry<KVDT>::kStageBytes + 24);
#ifndef PNKV_MAX_STAGES
#define PNKV_MAX_STAGES 48
#endif
  static constexpr int kStagesCap = kStagesFit < PNKV_MAX_STAGES ? kStagesFit : PNKV_MAX_STAGES;
  static constexpr int kStages = (kStagesCap / kStreams) * kStreams;
  static constexpr int kStageRegion = kStages * Geometry<KVDT>::kStageBytes;
  static constexpr int kBarOff = kStageRegion;                 // full[S], empty[S]
  static constexpr int kMetaOff = kBarOff + 2 * 8 * kStages;   // int32 valid[S]
  static constexpr int kArmOff = kMetaOff + 4 * kStages;       // int32 armed[S]: unit that armed the stage
  static constexpr int kAbortOff = kArmOff + 4 * kStages;      // int32 abort flag
  static constexpr int kPieceAbortOff = kAbortOff + 4;         // the flag as seen at a piece's end
  static constexpr int kMlOff = (kPieceAbortOff + 4 + 15) & ~15;
  static constexpr int kMergeOff = (kMlOff + kMlBytes + 15) & ~15;
  static constexpr int kQOff = kMergeOff + kMergeBytes;
  static constexpr int kTotal = kQOff + kQBytes;
  static constexpr int kDynamicBytes = kTotal + 1024;          // room to align the base
  static_assert(kStages >= 2 * kStreams, "every consumer stream needs two stages");
  static_assert(kStages % kStreams == 0, "stages must split evenly over the streams");
  // producer lanes that issue together (they need distinct stages)
  static constexpr int kIssue = kIssueLanes <= kStages ? kIssueLanes : 8;
  static_assert(kStages >= kIssue && 32 % kIssue == 0, "lanes that issue together need distinct stages");
  static_assert(kDynamicBytes <= kMaxSmem, "shared memory plan too large");
};

// Position of (row, dim) in the merge buffer: 32-dim chunks stay in place,
// inside a chunk the float pairs rotate with the chunk index and the row so
// that the consumers' fragment stores hit distinct banks.
__device__ __forceinline__ int merge_pos(int row, int d) {
  return row * 256 + (d & ~31) + (((d & 31) + 8 * ((d >> 5) & 3) + 2 * ((row & 7) >> 1)) & 31);
}

// ---------------------------------------------------------------------------
// Per-warp consumer state.

template <int NTW>
struct WarpState {
  float o[16][NTW][4];  // O^T fragments: [m-tile of dims][n-tile of rows]
  float m[NTW][2];      // running max (log2 domain) of the thread's 2 columns
  float l[NTW][2];      // running partial sum of p (this thread's tokens)
  int32_t lim[NTW][2];  // keys visible to each column (absolute count)

  __device__ void reset() {
#pragma unroll
    for (int mt = 0; mt < 16; ++mt)
#pragma unroll
      for (int nt = 0; nt < NTW; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) o[mt][nt][e] = 0.f;
#pragma unroll
    for (int nt = 0; nt < NTW; ++nt) {
      m[nt][0] = m[nt][1] = -INFINITY;
      l[nt][0] = l[nt][1] = 0.f;
    }
  }
};

// Query B-fragments, held in registers (QS = 0) or in shared memory (QS = 1,
// fragment order [n-tile][k-step][lane] x 8 bytes, read with one 64-bit load
// per k-step; frees 32 registers per n-tile for more resident warps).
template <int NTW, int QS>
struct QFrag;
template <int NTW>
struct QFrag<NTW, 0> {
  uint32_t r[NTW][16][2];
  __device__ __forceinline__ uint2 get(int nt, int kk) const { return make_uint2(r[nt][kk][0], r[nt][kk][1]); }
};
template <int NTW>
struct QFrag<NTW, 1> {
  uint32_t base;  // shared address of this warp's first n-tile, lane offset included
  __device__ __forceinline__ uint2 get(int nt, int kk) const {
    uint2 v;
    asm volatile("ld.shared.v2.b32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(base + (nt * 16 + kk) * 256));
    return v;
  }
};

// Query B-fragments of the warp's rows: for k-step kk the thread holds
// (Q[row][64*tig + 4*kk + 0..1]) and (Q[row][64*tig + 4*kk + 2..3]), row =
// 8*nt + gid of the warp's row block; fp16 for the NVFP4 path (the K tile is
// fp16), bf16 bits for the bf16 path.
template <int KVDT, int NTW>
__device__ __forceinline__ void load_q(const DecodeArgs& a, const Piece& pc, int row_base, int lane,
                                       uint32_t (&qb)[NTW][16][2]) {
  const int gid = lane >> 2, tig = lane & 3;
#pragma unroll
  for (int nt = 0; nt < NTW; ++nt) {
    const int n = row_base + 8 * nt + gid;
    const int rows = a.group * pc.s.qlen;
    if (KVDT == PNKV_KV_INT8 && n < rows) {
      // INT8 k order: k-step kk holds dims 16*kk + 4*tig + 0..3 (one 64-dim
      // scale group per four k-steps)
      const int t = pc.s.q0 + n / a.group;
      const int hq = pc.h * a.group + n % a.group;
      const uint2* src = reinterpret_cast<const uint2*>(a.q + (static_cast<int64_t>(t) * a.hq + hq) * 256 + 4 * tig);
#pragma unroll
      for (int kk = 0; kk < 16; ++kk) {
        const uint2 w = __ldg(src + 4 * kk);
        qb[nt][kk][0] = f32x2_to_f16x2(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xFFFF0000u));
        qb[nt][kk][1] = f32x2_to_f16x2(__uint_as_float(w.y << 16), __uint_as_float(w.y & 0xFFFF0000u));
      }
    } else if (n < rows) {
      const int t = pc.s.q0 + n / a.group;
      const int hq = pc.h * a.group + n % a.group;
      const uint4* src = reinterpret_cast<const uint4*>(a.q + (static_cast<int64_t>(t) * a.hq + hq) * 256 +
                                                        64 * tig);
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const uint4 w = __ldg(src + c);
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int word = 4 * c + e;  // dims 64*tig + 2*word, +1
          uint32_t v = ws[e];
          if (KVDT != PNKV_KV_BF16)
            v = f32x2_to_f16x2(__uint_as_float(v << 16), __uint_as_float(v & 0xFFFF0000u));
          qb[nt][word >> 1][word & 1] = v;
        }
      }
    } else {
#pragma unroll
      for (int kk = 0; kk < 16; ++kk) qb[nt][kk][0] = qb[nt][kk][1] = 0u;
    }
  }
}

template <int NTW>
__device__ __forceinline__ void set_qfrag_base(QFrag<NTW, 1>& q, uint32_t base) { q.base = base; }
template <int NTW>
__device__ __forceinline__ void set_qfrag_base(QFrag<NTW, 0>&, uint32_t) {}
template <int KVDT, int NTW>
__device__ __forceinline__ void load_q_regs(const DecodeArgs& a, const Piece& pc, int row_base, int lane,
                                            QFrag<NTW, 0>& q) {
  load_q<KVDT, NTW>(a, pc, row_base, lane, q.r);
}
template <int KVDT, int NTW>
__device__ __forceinline__ void load_q_regs(const DecodeArgs&, const Piece&, int, int, QFrag<NTW, 1>&) {}

// S^T (16 tokens x 8 rows per n-tile) for one page: NVFP4.  The 16 k-steps
// feed NA independent accumulator sets (k-step mod NA), summed at the end.
// For NVFP4 one set measured fastest (2 % over two on the million-token
// decode: the warp's widening work hides the MMA latency, and fewer
// registers and adds are live); the FP8 path keeps two.
#ifndef PNKV_QK_ACC_NVFP4
#define PNKV_QK_ACC_NVFP4 1
#endif
#ifndef PNKV_QK_ACC
#define PNKV_QK_ACC 2
#endif
template <int NTW, typename Q>
__device__ __forceinline__ void qk_nvfp4(uint32_t sb, int lane, const Q& qf, float (&s)[NTW][4]) {
  const int gid = lane >> 2, tig = lane & 3;
  constexpr int NA = PNKV_QK_ACC_NVFP4;  // independent accumulator sets (k-step mod NA)
  float acc[4][NTW][4];
#pragma unroll
  for (int j = 0; j < 4; ++j)
#pragma unroll
    for (int nt = 0; nt < NTW; ++nt) acc[j][nt][0] = acc[j][nt][1] = acc[j][nt][2] = acc[j][nt][3] = 0.f;
  // scales of blocks 4*tig .. 4*tig+3 for tokens gid and gid+8
  const uint32_t sc_lo = lds32(sb + swz128(16, gid * 16 + 4 * tig));
  const uint32_t sc_hi = lds32(sb + swz128(17, gid * 16 + 4 * tig));
  const uint32_t slo01 = e4m3x2_to_f16x2(sc_lo & 0xFFFFu), slo23 = e4m3x2_to_f16x2(sc_lo >> 16);
  const uint32_t shi01 = e4m3x2_to_f16x2(sc_hi & 0xFFFFu), shi23 = e4m3x2_to_f16x2(sc_hi >> 16);
#pragma unroll
  for (int h = 0; h < 2; ++h) {  // 16-byte chunk 2*tig + h: k-steps 8h .. 8h+7
    const uint4 klo = lds128(sb + swz128(gid, 16 * (2 * tig + h)));
    const uint4 khi = lds128(sb + swz128(gid + 8, 16 * (2 * tig + h)));
    const uint32_t wl[4] = {klo.x, klo.y, klo.z, klo.w};
    const uint32_t wh[4] = {khi.x, khi.y, khi.z, khi.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {  // word q: k-steps 8h + 2q, 8h + 2q + 1
      const int blk = 2 * h + (q >> 1);  // block 4*tig + blk
      const uint32_t sl = (blk < 2) ? slo01 : slo23;
      const uint32_t sh = (blk < 2) ? shi01 : shi23;
      const uint32_t sel = (blk & 1) ? 0x3232u : 0x1010u;
      const uint32_t scl = prmt(sl, sl, sel), sch = prmt(sh, sh, sel);
      uint32_t cl[4], ch[4];
      e2m1x8_unpack(wl[q], cl);
      e2m1x8_unpack(wh[q], ch);
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int kk = 8 * h + 2 * q + half;
        uint32_t af[4];
        af[0] = hmul2(cl[2 * half], scl);
        af[1] = hmul2(ch[2 * half], sch);
        af[2] = hmul2(cl[2 * half + 1], scl);
        af[3] = hmul2(ch[2 * half + 1], sch);
#pragma unroll
        for (int nt = 0; nt < NTW; ++nt) {
          const uint2 qv = qf.get(nt, kk);
          mma_f16_16816(acc[kk % NA][nt], af, qv.x, qv.y);
        }
      }
    }
  }
#pragma unroll
  for (int nt = 0; nt < NTW; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      // only the NA sets in use (adding a zero set is not free: x + 0 is not x for x = -0)
      float v = acc[0][nt][e];
#pragma unroll
      for (int j = 1; j < NA; ++j) v += acc[j][nt][e];
      s[nt][e] = v;
    }
}

// S^T for one page: bf16 cache (four independent accumulator sets).
template <int NTW, typename Q>
__device__ __forceinline__ void qk_bf16(uint32_t sb, int lane, const Q& qf, float (&s)[NTW][4]) {
  const int gid = lane >> 2, tig = lane & 3;
  float acc[4][NTW][4];
#pragma unroll
  for (int j = 0; j < 4; ++j)
#pragma unroll
    for (int nt = 0; nt < NTW; ++nt) acc[j][nt][0] = acc[j][nt][1] = acc[j][nt][2] = acc[j][nt][3] = 0.f;
  const uint32_t rlo = 4 * gid + tig, rhi = 4 * (gid + 8) + tig;  // box rows
#pragma unroll
  for (int c = 0; c < 8; ++c) {  // chunk c: words 4c..4c+3 -> k-steps 2c, 2c+1
    const uint4 klo = lds128(sb + swz128(rlo, 16 * c));
    const uint4 khi = lds128(sb + swz128(rhi, 16 * c));
    {
      const uint32_t af[4] = {klo.x, khi.x, klo.y, khi.y};
#pragma unroll
      for (int nt = 0; nt < NTW; ++nt) {
        const uint2 qv = qf.get(nt, 2 * c);
        mma_bf16_16816(acc[(2 * c) & 3][nt], af, qv.x, qv.y);
      }
    }
    {
      const uint32_t af[4] = {klo.z, khi.z, klo.w, khi.w};
#pragma unroll
      for (int nt = 0; nt < NTW; ++nt) {
        const uint2 qv = qf.get(nt, 2 * c + 1);
        mma_bf16_16816(acc[(2 * c + 1) & 3][nt], af, qv.x, qv.y);
      }
    }
  }
#pragma unroll
  for (int nt = 0; nt < NTW; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) s[nt][e] = (acc[0][nt][e] + acc[1][nt][e]) + (acc[2][nt][e] + acc[3][nt][e]);
}

// Online softmax over the logits of NP pages at once (one max reduction and
// one accumulator rescale per call); returns the P^T B-fragments per page.
template <int NTW, int NP>
__device__ __forceinline__ void softmax_pages(WarpState<NTW>& st, float (&s)[NP][NTW][4], float scale,
                                              const int32_t (&key0)[NP], const int32_t (&page_lim)[NP],
                                              const bool (&masked)[NP], int lane,
                                              uint32_t (&pb)[NP][NTW][2]) {
  const int gid = lane >> 2;
#pragma unroll
  for (int nt = 0; nt < NTW; ++nt) {
    // maxima of the raw logits (masked keys -inf); the logit scale is
    // positive, so the scaled maximum is the maximum of the scaled logits
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int pg = 0; pg < NP; ++pg) {
      if (masked[pg]) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int tok = gid + ((e & 2) ? 8 : 0);
          if (tok >= page_lim[pg] || key0[pg] + tok >= st.lim[nt][e & 1]) s[pg][nt][e] = -INFINITY;
        }
      }
      mx0 = fmaxf(mx0, fmaxf(s[pg][nt][0], s[pg][nt][2]));
      mx1 = fmaxf(mx1, fmaxf(s[pg][nt][1], s[pg][nt][3]));
    }
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
    }
    const float mn0 = fmaxf(st.m[nt][0], mx0 * scale), mn1 = fmaxf(st.m[nt][1], mx1 * scale);
    const float base0 = (mn0 == -INFINITY) ? 0.f : mn0;
    const float base1 = (mn1 == -INFINITY) ? 0.f : mn1;
    const float al0 = fast_exp2(st.m[nt][0] - base0), al1 = fast_exp2(st.m[nt][1] - base1);
    st.m[nt][0] = mn0;
    st.m[nt][1] = mn1;
    // p = 2^(s * scale - base): P V takes p in fp16, l sums p in fp32
    float add0 = 0.f, add1 = 0.f;
#pragma unroll
    for (int pg = 0; pg < NP; ++pg) {
      const float p0 = fast_exp2(fmaf(s[pg][nt][0], scale, -base0));
      const float p1 = fast_exp2(fmaf(s[pg][nt][1], scale, -base1));
      const float p2 = fast_exp2(fmaf(s[pg][nt][2], scale, -base0));
      const float p3 = fast_exp2(fmaf(s[pg][nt][3], scale, -base1));
      const uint32_t x0 = f32x2_to_f16x2(p0, p1);
      const uint32_t x1 = f32x2_to_f16x2(p2, p3);
      add0 += p0 + p2;
      add1 += p1 + p3;
      pb[pg][nt][0] = movmatrix_trans(x0);
      pb[pg][nt][1] = movmatrix_trans(x1);
    }
    st.l[nt][0] = st.l[nt][0] * al0 + add0;
    st.l[nt][1] = st.l[nt][1] * al1 + add1;
    // rescale the accumulators only when some column's running max moved
    if (__any_sync(0xffffffffu, al0 != 1.f || al1 != 1.f)) {
#pragma unroll
      for (int mt = 0; mt < 16; ++mt) {
        st.o[mt][nt][0] *= al0;
        st.o[mt][nt][2] *= al0;
        st.o[mt][nt][1] *= al1;
        st.o[mt][nt][3] *= al1;
      }
    }
  }
}

// O^T += V^T P^T for one page: NVFP4.  V codes are stored slot-pair
// interleaved (byte d of pair i holds element d of slots 2i and 2i+1), so one
// byte widens to the (token 2i, token 2i+1) pair an A-fragment register holds.
// Thread (gid, tig) covers dims 16*gid + mt (rows gid of m-tile mt, block gid)
// and 128 + 16*gid + mt (rows gid+8, block 8+gid), tokens 2tig, 2tig+1 (pair
// tig) and 2tig+8, 2tig+9 (pair tig+4).
template <int NTW>
__device__ __forceinline__ void pv_nvfp4(uint32_t sb, int lane, WarpState<NTW>& st,
                                         const uint32_t (&pb)[NTW][2], int page_lim) {
  const int gid = lane >> 2, tig = lane & 3;
  // scale pairs (token 2p, token 2p+1) of a block; tokens past page_lim
  // scale to 0 (their codes and scales may be stale)
  const int t0 = 2 * tig, t2 = 2 * tig + 8;
  auto sbyte = [&](int t, int blk) -> uint32_t { return lds8(sb + swz128(34 + (t >> 3), (t & 7) * 16 + blk)); };
  uint32_t b[8] = {sbyte(t0, gid), sbyte(t0 + 1, gid), sbyte(t0, 8 + gid), sbyte(t0 + 1, 8 + gid),
                   sbyte(t2, gid), sbyte(t2 + 1, gid), sbyte(t2, 8 + gid), sbyte(t2 + 1, 8 + gid)};
  if (page_lim < 16) {  // a partial or missing page (uniform over the warp)
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int t = (i < 4 ? t0 : t2) + (i & 1);
      if (t >= page_lim) b[i] = 0u;
    }
  }
  const uint32_t s_a_lo = e4m3x2_to_f16x2(prmt(b[0], b[1], 0x0040u));
  const uint32_t s_a_hi = e4m3x2_to_f16x2(prmt(b[2], b[3], 0x0040u));
  const uint32_t s_b_lo = e4m3x2_to_f16x2(prmt(b[4], b[5], 0x0040u));
  const uint32_t s_b_hi = e4m3x2_to_f16x2(prmt(b[6], b[7], 0x0040u));
  // pair row p = box rows 18 + 2p (dims 0..127) and 19 + 2p (dims 128..255)
  const uint4 a_lo = lds128(sb + swz128(18 + 2 * tig, 16 * gid));
  const uint4 a_hi = lds128(sb + swz128(19 + 2 * tig, 16 * gid));
  const uint4 b_lo = lds128(sb + swz128(26 + 2 * tig, 16 * gid));
  const uint4 b_hi = lds128(sb + swz128(27 + 2 * tig, 16 * gid));
  const uint32_t wal[4] = {a_lo.x, a_lo.y, a_lo.z, a_lo.w}, wah[4] = {a_hi.x, a_hi.y, a_hi.z, a_hi.w};
  const uint32_t wbl[4] = {b_lo.x, b_lo.y, b_lo.z, b_lo.w}, wbh[4] = {b_hi.x, b_hi.y, b_hi.z, b_hi.w};
#pragma unroll
  for (int wi = 0; wi < 4; ++wi) {
    uint32_t c0[4], c1[4], c2[4], c3[4];
    e2m1x8_unpack(wal[wi], c0);
    e2m1x8_unpack(wah[wi], c1);
    e2m1x8_unpack(wbl[wi], c2);
    e2m1x8_unpack(wbh[wi], c3);
#pragma unroll
    for (int bi = 0; bi < 4; ++bi) {
      const int mt = 4 * wi + bi;  // byte mt of each chunk
      uint32_t af[4];
      af[0] = hmul2(c0[bi], s_a_lo);  // dim 16*gid + mt,       tokens 2tig, 2tig+1
      af[1] = hmul2(c1[bi], s_a_hi);  // dim 128 + 16*gid + mt
      af[2] = hmul2(c2[bi], s_b_lo);  // tokens 2tig+8, 2tig+9
      af[3] = hmul2(c3[bi], s_b_hi);
#pragma unroll
      for (int nt = 0; nt < NTW; ++nt) mma_f16_16816(st.o[mt][nt], af, pb[nt][0], pb[nt][1]);
    }
  }
}

// S^T for one page: FP8 cache.  Token t's codes are box rows 2t, 2t+1; for
// k-step kk lane (gid, tig) takes dims 64*tig + 4*kk .. +3 of tokens gid and
// gid+8 (the NVFP4 path's k order, so the same Q fragments serve), i.e. bytes
// 64*(tig & 1) + 4*kk of box row 2*token + tig/2: four 16-byte loads per
// token.  E4M3 widens exactly to fp16; the per-tensor scale folds into the
// logit scale.
template <int NTW, typename Q>
__device__ __forceinline__ void qk_fp8(uint32_t sb, int lane, const Q& qf, float (&s)[NTW][4]) {
  const int gid = lane >> 2, tig = lane & 3;
  constexpr int NA = PNKV_QK_ACC;
  float acc[4][NTW][4];
#pragma unroll
  for (int j = 0; j < NA; ++j)
#pragma unroll
    for (int nt = 0; nt < NTW; ++nt) acc[j][nt][0] = acc[j][nt][1] = acc[j][nt][2] = acc[j][nt][3] = 0.f;
  const int rlo = 2 * gid + (tig >> 1), rhi = 2 * (gid + 8) + (tig >> 1);
#pragma unroll
  for (int c = 0; c < 4; ++c) {  // 16-byte chunk 4*(tig & 1) + c: k-steps 4c .. 4c+3
    const uint4 klo = lds128(sb + swz128(rlo, 16 * (4 * (tig & 1) + c)));
    const uint4 khi = lds128(sb + swz128(rhi, 16 * (4 * (tig & 1) + c)));
    const uint32_t wl[4] = {klo.x, klo.y, klo.z, klo.w};
    const uint32_t wh[4] = {khi.x, khi.y, khi.z, khi.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int kk = 4 * c + q;
      uint32_t af[4];
      e4m3x4_to_f16x2x2(wl[q], af[0], af[2]);  // token gid: dims +0,+1 and +2,+3
      e4m3x4_to_f16x2x2(wh[q], af[1], af[3]);  // token gid+8
#pragma unroll
      for (int nt = 0; nt < NTW; ++nt) {
        const uint2 qv = qf.get(nt, kk);
        mma_f16_16816(acc[kk % NA][nt], af, qv.x, qv.y);
      }
    }
  }
#pragma unroll
  for (int nt = 0; nt < NTW; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      float v = acc[0][nt][e];
#pragma unroll
      for (int j = 1; j < NA; ++j) v += acc[j][nt][e];
      s[nt][e] = v;
    }
}

// O^T += V^T P^T for one page: FP8 cache.  Pair row p (slots 2p, 2p+1) is
// [256 dims][2 bytes] at box rows 32 + 4p .. 32 + 4p + 3; two bytes are the
// (token 2p, token 2p+1) pair an A register holds.  Thread (gid, tig) covers
// dims 16*gid + mt (rows gid of m-tile mt) and 128 + 16*gid + mt (rows
// gid+8), pairs tig and tig+4, as in the NVFP4 path.  Tokens at or past
// page_lim (a partial or missing page) are zeroed, so stale codes cannot
// reach the product.
template <int NTW>
__device__ __forceinline__ void pv_fp8(uint32_t sb, int lane, WarpState<NTW>& st,
                                       const uint32_t (&pb)[NTW][2], int page_lim) {
  const int gid = lane >> 2, tig = lane & 3;
  auto keep = [&](int t) -> uint32_t {
    return (t < page_lim ? 0x0000FFFFu : 0u) | (t + 1 < page_lim ? 0xFFFF0000u : 0u);
  };
  const uint32_t ma = keep(2 * tig), mb = keep(2 * tig + 8);
  // dims 16*gid .. +15 of pair p, low half (dims 0..127) and high half
  auto ld2 = [&](int p, int hi, uint4& x0, uint4& x1) {
    const int row = 32 + 4 * p + 2 * hi + (gid >> 2);
    x0 = lds128(sb + swz128(row, 32 * (gid & 3)));
    x1 = lds128(sb + swz128(row, 32 * (gid & 3) + 16));
  };
  uint4 al0, al1, ah0, ah1, bl0, bl1, bh0, bh1;
  ld2(tig, 0, al0, al1);
  ld2(tig, 1, ah0, ah1);
  ld2(tig + 4, 0, bl0, bl1);
  ld2(tig + 4, 1, bh0, bh1);
  const uint32_t wal[8] = {al0.x, al0.y, al0.z, al0.w, al1.x, al1.y, al1.z, al1.w};
  const uint32_t wah[8] = {ah0.x, ah0.y, ah0.z, ah0.w, ah1.x, ah1.y, ah1.z, ah1.w};
  const uint32_t wbl[8] = {bl0.x, bl0.y, bl0.z, bl0.w, bl1.x, bl1.y, bl1.z, bl1.w};
  const uint32_t wbh[8] = {bh0.x, bh0.y, bh0.z, bh0.w, bh1.x, bh1.y, bh1.z, bh1.w};
#pragma unroll
  for (int wi = 0; wi < 8; ++wi) {  // word wi: dims 16*gid + 2wi, +1
    uint32_t a0[2], a1[2], a2[2], a3[2];
    e4m3x4_to_f16x2x2(wal[wi], a0[0], a0[1]);
    e4m3x4_to_f16x2x2(wah[wi], a1[0], a1[1]);
    e4m3x4_to_f16x2x2(wbl[wi], a2[0], a2[1]);
    e4m3x4_to_f16x2x2(wbh[wi], a3[0], a3[1]);
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int mt = 2 * wi + u;
      const uint32_t af[4] = {a0[u] & ma, a1[u] & ma, a2[u] & mb, a3[u] & mb};
#pragma unroll
      for (int nt = 0; nt < NTW; ++nt) mma_f16_16816(st.o[mt][nt], af, pb[nt][0], pb[nt][1]);
    }
  }
}

// S^T for one page: INT8 group-64 cache.  Token t's codes are box rows 2t,
// 2t+1 with dims permuted so that lane (gid, tig) reads its 16 k-steps
// (dims 16*kk + 4*tig .. +3) as 64 contiguous bytes: chunk c of them is scale
// group c.  Each group's four MMAs go to a fresh accumulator that is then
// scaled by the two tokens' group scales (fp32 FFMA), so the int8 codes enter
// the product exactly.
template <int NTW, typename Q>
__device__ __forceinline__ void qk_int8(uint32_t sb, int lane, const Q& qf, float (&s)[NTW][4]) {
  const int gid = lane >> 2, tig = lane & 3;
  const int rlo = 2 * gid + (tig >> 1), rhi = 2 * (gid + 8) + (tig >> 1);
  // group scales of tokens gid and gid+8 (row 32: [16 tokens][4] fp16)
  uint2 sl, sh;
  asm volatile("ld.shared.v2.b32 {%0,%1}, [%2];" : "=r"(sl.x), "=r"(sl.y) : "r"(sb + swz128(32, 8 * gid)));
  asm volatile("ld.shared.v2.b32 {%0,%1}, [%2];" : "=r"(sh.x), "=r"(sh.y) : "r"(sb + swz128(32, 8 * (gid + 8))));
  const float2 sl01 = __half22float2(*reinterpret_cast<const __half2*>(&sl.x));
  const float2 sl23 = __half22float2(*reinterpret_cast<const __half2*>(&sl.y));
  const float2 sh01 = __half22float2(*reinterpret_cast<const __half2*>(&sh.x));
  const float2 sh23 = __half22float2(*reinterpret_cast<const __half2*>(&sh.y));
  const float slo[4] = {sl01.x, sl01.y, sl23.x, sl23.y}, shi[4] = {sh01.x, sh01.y, sh23.x, sh23.y};
#pragma unroll
  for (int nt = 0; nt < NTW; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
  for (int c = 0; c < 4; ++c) {  // chunk 4*(tig & 1) + c: group c, k-steps 4c .. 4c+3
    const uint4 klo = lds128(sb + swz128(rlo, 16 * (4 * (tig & 1) + c)));
    const uint4 khi = lds128(sb + swz128(rhi, 16 * (4 * (tig & 1) + c)));
    const uint32_t wl[4] = {klo.x, klo.y, klo.z, klo.w};
    const uint32_t wh[4] = {khi.x, khi.y, khi.z, khi.w};
    float acc[NTW][4];
#pragma unroll
    for (int nt = 0; nt < NTW; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int kk = 4 * c + q;
      uint32_t af[4];
      s8x4_to_f16x2x2(wl[q], af[0], af[2]);  // token gid: dims +0,+1 and +2,+3
      s8x4_to_f16x2x2(wh[q], af[1], af[3]);  // token gid+8
#pragma unroll
      for (int nt = 0; nt < NTW; ++nt) {
        const uint2 qv = qf.get(nt, kk);
        mma_f16_16816(acc[nt], af, qv.x, qv.y);
      }
    }
#pragma unroll
    for (int nt = 0; nt < NTW; ++nt) {
      s[nt][0] = fmaf(acc[nt][0], slo[c], s[nt][0]);
      s[nt][1] = fmaf(acc[nt][1], slo[c], s[nt][1]);
      s[nt][2] = fmaf(acc[nt][2], shi[c], s[nt][2]);
      s[nt][3] = fmaf(acc[nt][3], shi[c], s[nt][3]);
    }
  }
}

// O^T += V^T P^T for one page: INT8 group-64 cache.  Pair row p (slots 2p,
// 2p+1) holds 256 positions x 2 bytes at box rows 33 + 4p .. +3, position
// 32*(d%8) + d/8 holding dim d, so lane (gid, tig) reads dims 8j + gid (j =
// 0..31) of pairs tig and tig+4 as 64 contiguous bytes each: word w gives
// m-tile w's rows gid (dim 16w + gid) and gid+8 (dim 16w + 8 + gid).  The
// m-tiles of a 64-dim scale group share one scale per token, which scales
// the P^T fragment (fp16) instead of the codes; tokens at or past page_lim
// get a zero scale.
template <int NTW>
__device__ __forceinline__ void pv_int8(uint32_t sb, int lane, WarpState<NTW>& st,
                                        const uint32_t (&pb)[NTW][2], int page_lim) {
  const int gid = lane >> 2, tig = lane & 3;
  // group scales of tokens 2tig, 2tig+1, 2tig+8, 2tig+9 (row 65: [16][4] fp16)
  auto ldsc = [&](int t) -> uint2 {
    uint2 v;
    asm volatile("ld.shared.v2.b32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(sb + swz128(65, 8 * t)));
    return v;
  };
  const uint2 s0 = ldsc(2 * tig), s1 = ldsc(2 * tig + 1), s2 = ldsc(2 * tig + 8), s3 = ldsc(2 * tig + 9);
  auto keep = [&](int t) -> uint32_t {
    return (t < page_lim ? 0x0000FFFFu : 0u) | (t + 1 < page_lim ? 0xFFFF0000u : 0u);
  };
  const uint32_t ma = keep(2 * tig), mb = keep(2 * tig + 8);
  uint32_t pg[4][NTW][2];  // P^T fragments scaled by group g's token scales
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    const uint32_t sel = (g & 1) ? 0x7632u : 0x5410u;
    const uint32_t sa = prmt(g < 2 ? s0.x : s0.y, g < 2 ? s1.x : s1.y, sel) & ma;
    const uint32_t sbb = prmt(g < 2 ? s2.x : s2.y, g < 2 ? s3.x : s3.y, sel) & mb;
#pragma unroll
    for (int nt = 0; nt < NTW; ++nt) {
      pg[g][nt][0] = hmul2(pb[nt][0], sa);
      pg[g][nt][1] = hmul2(pb[nt][1], sbb);
    }
  }
  const int rbase = 33 + (gid >> 1);
#pragma unroll
  for (int c = 0; c < 4; ++c) {  // chunk c: words 4c .. 4c+3 -> m-tiles 4c .. 4c+3 = group c
    const uint4 va = lds128(sb + swz128(rbase + 4 * tig, 16 * (4 * (gid & 1) + c)));
    const uint4 vb = lds128(sb + swz128(rbase + 4 * (tig + 4), 16 * (4 * (gid & 1) + c)));
    const uint32_t wa[4] = {va.x, va.y, va.z, va.w}, wb[4] = {vb.x, vb.y, vb.z, vb.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int mt = 4 * c + q;
      uint32_t af[4];
      s8x4_to_f16x2x2(wa[q], af[0], af[1]);  // pair tig: rows gid, gid+8
      s8x4_to_f16x2x2(wb[q], af[2], af[3]);  // pair tig+4
#pragma unroll
      for (int nt = 0; nt < NTW; ++nt) mma_f16_16816(st.o[mt][nt], af, pg[c][nt][0], pg[c][nt][1]);
    }
  }
}

// O^T += V^T P^T for one page: bf16 cache (V widened to fp16).
template <int NTW>
__device__ __forceinline__ void pv_bf16(uint32_t sb, int lane, WarpState<NTW>& st,
                                        const uint32_t (&pb)[NTW][2], int page_lim) {
  const int gid = lane >> 2, tig = lane & 3;
  const int toks[4] = {2 * tig, 2 * tig + 1, 2 * tig + 8, 2 * tig + 9};
#pragma unroll
  for (int c = 0; c < 4; ++c) {  // chunk c: words 16*gid + 4*c .. +3
    uint32_t w[4][4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int t = toks[k];
      const uint4 v = lds128(sb + swz128(64 + 4 * t + (gid >> 1), 64 * (gid & 1) + 16 * c));
      const bool ok = t < page_lim;
      w[k][0] = ok ? v.x : 0u;
      w[k][1] = ok ? v.y : 0u;
      w[k][2] = ok ? v.z : 0u;
      w[k][3] = ok ? v.w : 0u;
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int mt = 4 * c + e;  // word 16*gid + mt of each token
      uint32_t af[4];
      af[0] = f32x2_to_f16x2(__uint_as_float(w[0][e] << 16), __uint_as_float(w[1][e] << 16));
      af[1] = f32x2_to_f16x2(__uint_as_float(w[0][e] & 0xFFFF0000u), __uint_as_float(w[1][e] & 0xFFFF0000u));
      af[2] = f32x2_to_f16x2(__uint_as_float(w[2][e] << 16), __uint_as_float(w[3][e] << 16));
      af[3] = f32x2_to_f16x2(__uint_as_float(w[2][e] & 0xFFFF0000u), __uint_as_float(w[3][e] & 0xFFFF0000u));
#pragma unroll
      for (int nt = 0; nt < NTW; ++nt) mma_f16_16816(st.o[mt][nt], af, pb[nt][0], pb[nt][1]);
    }
  }
}

// ---------------------------------------------------------------------------

template <int KVDT, int NTW, int RG, int NW, int QS, int NP>
__global__ void __launch_bounds__(NW * 32, 1)
    paged_decode_kernel(const __grid_constant__ CUtensorMap tmap, const DecodeArgs a) {
  using P = Plan<KVDT, NTW, RG, NW, QS>;
  using C = Consumers<NW, RG>;
  constexpr int kProducerWarp = NW - 1;
  using Geo = Geometry<KVDT>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + P::kBarOff);
  uint64_t* empty = full + P::kStages;
  int32_t* stage_valid = reinterpret_cast<int32_t*>(smem + P::kMetaOff);
  int32_t* stage_armed = reinterpret_cast<int32_t*>(smem + P::kArmOff);
  volatile int32_t* abort_flag = reinterpret_cast<int32_t*>(smem + P::kAbortOff);
  volatile int32_t* piece_abort = reinterpret_cast<int32_t*>(smem + P::kPieceAbortOff);
  float* ml = reinterpret_cast<float*>(smem + P::kMlOff);
  float* mbuf = reinterpret_cast<float*>(smem + P::kMergeOff);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < P::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], RG);
      stage_armed[s] = -1;
    }
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == kProducerWarp && lane == 0) tma_prefetch_desc(&tmap);
  __syncthreads();
  griddep_wait();  // the previous kernel's writes (pool, queries) are visible from here
  griddep_launch_dependents();

  // this CTA's unit range
  const int64_t total = total_units<1>(a, lane);
  const int64_t chunk = (total + gridDim.x - 1) / gridDim.x;
  const int64_t u_begin = min(total, static_cast<int64_t>(blockIdx.x) * chunk);
  const int64_t u_end = min(total, u_begin + chunk);

  if (blockIdx.x == 0 && warp == 0) {
    if (lane == 0) {
      a.work_meta[0] = a.hkv;
      a.work_meta[1] = a.group;
      a.work_meta[2] = a.rows_per_slot;
      a.work_meta[3] = a.batch;
    }
    // segments without units get an empty slot range here; every other
    // segment's range is written by the CTA that holds its first unit
    for (int b = lane; b < a.batch; b += 32)
      if (load_seq<1>(a, b, false).units == 0)
        for (int h = 0; h < a.hkv; ++h) {
          a.work_meta[4 + 2 * (static_cast<int64_t>(b) * a.hkv + h)] = 0;
          a.work_meta[4 + 2 * (static_cast<int64_t>(b) * a.hkv + h) + 1] = 0;
        }
  }

  Walker<1> walk;
  walk.init(a, u_begin, u_end, lane);
  Piece pc;

  // the CTA holding a segment's first unit records where the segment's slots
  // are, before any work (so the record exists even if the call winds down
  // after a timeout)
  if (threadIdx.x == 0) {
    Walker<1> w0 = walk;
    while (w0.next(a, &pc)) {
      if (pc.p0 != 0) continue;
      const int64_t seg = pc.b * static_cast<int64_t>(a.hkv) + pc.h;
      const int64_t first_cta = pc.seg_start / chunk;
      const int64_t last_cta = (pc.seg_start + pc.s.units - 1) / chunk;
      a.work_meta[4 + 2 * seg] = static_cast<int32_t>(seg + first_cta);
      a.work_meta[4 + 2 * seg + 1] = static_cast<int32_t>(last_cta - first_cta + 1);
    }
  }

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    const uint64_t policy = l2_policy_evict_first();
    int64_t issued = 0;
    bool ok = true;
    while (ok && walk.next(a, &pc)) {
      const int32_t* row = a.page_table + static_cast<int64_t>(pc.b) * a.pt_stride + pc.p0;
      // the next group's page ids are read while this group issues
      int32_t next_page = lane < pc.n ? __ldg(row + lane) : 0;
      for (int j0 = 0; j0 < pc.n && ok; j0 += 32) {
        // lane j handles unit j0 + j: its own page id, stage and barrier;
        // lanes issue in groups of kIssueLanes so the ring refills steadily
        const bool mine = j0 + lane < pc.n;
        const int32_t page = next_page;
        next_page = j0 + 32 + lane < pc.n ? __ldg(row + j0 + 32 + lane) : 0;
        bool lane_ok = true;
#pragma unroll 1
        for (int g = 0; g < 32 / P::kIssue; ++g) {
          if (mine && lane / P::kIssue == g) {
            const int64_t i = issued + lane;
            const int s = static_cast<int>(i % P::kStages);
            const uint32_t par = static_cast<uint32_t>((i / P::kStages) & 1) ^ 1u;
            if (*abort_flag || !mbar_wait(&empty[s], par, a.wait_ns)) {
              lane_ok = false;  // nothing armed: the drain skips this unit
            } else if (page < 0 || page >= a.num_pages) {
              flag_error(a.dev_err, PNKV_DEV_ERR_PAGE_ID);
              stage_valid[s] = 0;
              stage_armed[s] = static_cast<int32_t>(i);
              mbar_arrive(&full[s]);
            } else {
              stage_valid[s] = 1;
              stage_armed[s] = static_cast<int32_t>(i);
              mbar_arrive_expect_tx(&full[s], Geo::kTxBytes);
              const int32_t y = (page * a.hkv + pc.h) * Geo::kBoxRows;
              tma_load_2d(smem + s * Geo::kStageBytes, &tmap, 0, y, &full[s], policy);
            }
          }
          __syncwarp();
        }
        if (!__all_sync(0xffffffffu, lane_ok)) {
          if (lane == 0) {
            flag_error(a.dev_err, PNKV_DEV_ERR_TIMEOUT);
            *abort_flag = 1;
          }
          ok = false;
        }
        issued += min(32, pc.n - j0);
      }
    }
    if (!ok && lane == 0) {
      // drain: wait (with the fixed bound) for the loads that may still be in
      // flight, so the CTA never exits with a bulk copy landing; a unit whose
      // stage was never armed (its lane gave up first) has nothing to wait for
      const int64_t first = issued > P::kStages ? issued - P::kStages : 0;
      for (int64_t i = first; i < issued; ++i)
        if (stage_armed[i % P::kStages] == static_cast<int32_t>(i))
          mbar_wait(&full[i % P::kStages], static_cast<uint32_t>((i / P::kStages) & 1));
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  if (warp >= C::kWarps) return;  // spare warp when RG does not divide 7
  const int rg = warp % RG;
  const int stream = warp / RG;
  const int row_base = rg * 8 * NTW;
  const int gid = lane >> 2, tig = lane & 3;
  WarpState<NTW> st;
  QFrag<NTW, QS> qf;

  while (walk.next(a, &pc)) {
    const int rows = a.group * pc.s.qlen;
    if (QS) {
      // one warp per row group stages the fragments; the others wait for it
      if (stream == 0) {
        uint32_t tmp[NTW][16][2];
        load_q<KVDT, NTW>(a, pc, row_base, lane, tmp);
#pragma unroll
        for (int nt = 0; nt < NTW; ++nt)
#pragma unroll
          for (int kk = 0; kk < 16; ++kk)
            *reinterpret_cast<uint2*>(smem + P::kQOff + (((rg * NTW + nt) * 16 + kk) * 32 + lane) * 8) =
                make_uint2(tmp[nt][kk][0], tmp[nt][kk][1]);
      }
      named_bar_sync(1, C::kThreads);
      set_qfrag_base(qf, smem_addr(smem + P::kQOff + (rg * NTW * 16 * 32 + lane) * 8));
    } else {
      load_q_regs<KVDT, NTW>(a, pc, row_base, lane, qf);
    }
    st.reset();
#pragma unroll
    for (int nt = 0; nt < NTW; ++nt)
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int n = row_base + 8 * nt + 2 * tig + c;
        st.lim[nt][c] = a.causal ? pc.s.len - pc.s.qlen + n / a.group + 1 : pc.s.len;
      }
    const int32_t mask_from = a.causal ? pc.s.len - pc.s.qlen + 1 : pc.s.len;  // first key some row cannot see
    // units of this piece owned by this warp, NP per iteration: i, i + S, ...
    // (missing trailing units are stand-ins for unit i, fully masked)
    // (32-bit: i0 counts the CTA's own units)
    constexpr int32_t S = P::kStreams;
    const int32_t i0 = static_cast<int32_t>(pc.i0);
    const int32_t end = i0 + pc.n;
    int32_t i = i0 + ((stream - i0 % S) % S + S) % S;
    // stage and phase parity of unit i, advanced with 32-bit arithmetic
    // (NP * S <= kStages, so one step wraps the ring at most once)
    static_assert(NP * S <= P::kStages, "one iteration wraps the stage ring at most once");
    int i_stage = i % P::kStages;
    uint32_t i_par = static_cast<uint32_t>((i / P::kStages) & 1);
    for (; i < end; i += NP * S) {
      int32_t u[NP];
      bool here[NP];
      int st_idx[NP];
      bool okw = !*abort_flag;
#pragma unroll
      for (int pg = 0; pg < NP; ++pg) {
        here[pg] = i + pg * S < end;
        u[pg] = here[pg] ? i + pg * S : i;
        int idx = i_stage + (here[pg] ? pg * S : 0);
        uint32_t par = i_par;
        if (idx >= P::kStages) {
          idx -= P::kStages;
          par ^= 1u;
        }
        st_idx[pg] = idx;
        if (okw && here[pg]) okw = mbar_wait(&full[idx], par, a.wait_ns);
      }
      // one outcome per warp: the MMAs below need every lane
      okw = __all_sync(0xffffffffu, okw);
      i_stage += NP * S;
      if (i_stage >= P::kStages) {
        i_stage -= P::kStages;
        i_par ^= 1u;
      }
      if (!okw) {
        if (lane == 0) flag_error(a.dev_err, PNKV_DEV_ERR_TIMEOUT);
        *abort_flag = 1;
        break;
      }
      int32_t key0[NP], page_lim[NP];
      bool masked[NP];
      uint32_t sb[NP];
#pragma unroll
      for (int pg = 0; pg < NP; ++pg) {
        const int32_t page_idx = pc.p0 + (u[pg] - i0);
        key0[pg] = page_idx * 16;
        const bool live = here[pg] && stage_valid[st_idx[pg]];
        page_lim[pg] = live ? pc.s.len - key0[pg] : 0;  // valid tokens in the page
        masked[pg] = !live || key0[pg] + 16 > mask_from;
        sb[pg] = smem_addr(smem + st_idx[pg] * Geo::kStageBytes);
      }
      float sacc[NP][NTW][4];
      uint32_t pb[NP][NTW][2];
#pragma unroll
      for (int pg = 0; pg < NP; ++pg) {
        if constexpr (KVDT == PNKV_KV_NVFP4) qk_nvfp4<NTW>(sb[pg], lane, qf, sacc[pg]);
        else if constexpr (KVDT == PNKV_KV_FP8) qk_fp8<NTW>(sb[pg], lane, qf, sacc[pg]);
        else if constexpr (KVDT == PNKV_KV_INT8) qk_int8<NTW>(sb[pg], lane, qf, sacc[pg]);
        else qk_bf16<NTW>(sb[pg], lane, qf, sacc[pg]);
      }
      softmax_pages<NTW, NP>(st, sacc, a.qk_scale_log2, key0, page_lim, masked, lane, pb);
#pragma unroll
      for (int pg = 0; pg < NP; ++pg) {
        if constexpr (KVDT == PNKV_KV_NVFP4) pv_nvfp4<NTW>(sb[pg], lane, st, pb[pg], page_lim[pg]);
        else if constexpr (KVDT == PNKV_KV_FP8) pv_fp8<NTW>(sb[pg], lane, st, pb[pg], page_lim[pg]);
        else if constexpr (KVDT == PNKV_KV_INT8) pv_int8<NTW>(sb[pg], lane, st, pb[pg], page_lim[pg]);
        else pv_bf16<NTW>(sb[pg], lane, st, pb[pg], page_lim[pg]);
      }
      __syncwarp();
      if (lane == 0)
#pragma unroll
        for (int pg = 0; pg < NP; ++pg)
          if (here[pg]) mbar_arrive(&empty[st_idx[pg]]);
    }

    // ---- merge the warps' partial states (fixed order) and write the slot
    // 1. full l per column; m is already uniform across the column's lanes
#pragma unroll
    for (int nt = 0; nt < NTW; ++nt)
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        float l = st.l[nt][c];
        l += __shfl_xor_sync(0xffffffffu, l, 4);
        l += __shfl_xor_sync(0xffffffffu, l, 8);
        l += __shfl_xor_sync(0xffffffffu, l, 16);
        st.l[nt][c] = l;
        if (gid == 0) {
          const int row = row_base + 8 * nt + 2 * tig + c;
          ml[(stream * P::kRows + row) * 2 + 0] = st.m[nt][c];
          ml[(stream * P::kRows + row) * 2 + 1] = l;
        }
      }
    named_bar_sync(1, C::kThreads);
    // 2. this warp's weight per column: 2^(m_w - M)
    float wgt[NTW][2];
#pragma unroll
    for (int nt = 0; nt < NTW; ++nt)
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int row = row_base + 8 * nt + 2 * tig + c;
        float M = -INFINITY;
        for (int k = 0; k < P::kStreams; ++k) M = fmaxf(M, ml[(k * P::kRows + row) * 2]);
        wgt[nt][c] = (M == -INFINITY) ? 0.f : fast_exp2(st.m[nt][c] - M);
      }
    // 3. ordered accumulation into the merge buffer, one stream per round
    for (int k = 0; k < P::kStreams; ++k) {
      if (stream == k) {
#pragma unroll
        for (int nt = 0; nt < NTW; ++nt)
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            const int row = row_base + 8 * nt + 2 * tig + c;
            // pairs of adjacent dims: bf16 m-tile mt holds dims 32*gid + 2*mt
            // (c) and +1 (c + 2); NVFP4/FP8 m-tiles mt, mt+1 hold dims
            // 16*gid + mt, +1 (c) and 128 + 16*gid + mt, +1 (c + 2); INT8
            // m-tile mt holds dims 16*mt + gid (c) and 16*mt + 8 + gid (c + 2)
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const float w = wgt[nt][c];
              if constexpr (KVDT == PNKV_KV_INT8) {
                float* d0 = mbuf + merge_pos(row, 16 * j + gid);
                float* d1 = mbuf + merge_pos(row, 16 * j + 8 + gid);
                *d0 = (k == 0 ? 0.f : *d0) + st.o[j][nt][c] * w;
                *d1 = (k == 0 ? 0.f : *d1) + st.o[j][nt][c + 2] * w;
              } else {
                int d;
                float2 v;
                if constexpr (KVDT != PNKV_KV_BF16) {
                  const int mt = j & ~1;
                  const int e = (j & 1) ? c + 2 : c;
                  d = ((j & 1) ? 128 : 0) + 16 * gid + mt;
                  v = make_float2(st.o[mt][nt][e] * w, st.o[mt + 1][nt][e] * w);
                } else {
                  d = 32 * gid + 2 * j;
                  v = make_float2(st.o[j][nt][c] * w, st.o[j][nt][c + 2] * w);
                }
                float2* dst = reinterpret_cast<float2*>(mbuf + merge_pos(row, d));
                if (k == 0) {
                  *dst = v;
                } else {
                  float2 acc = *dst;
                  acc.x += v.x;
                  acc.y += v.y;
                  *dst = acc;
                }
              }
            }
          }
      }
      named_bar_sync(1, C::kThreads);
    }
    // 4. normalise and write the partial (all consumer threads, coalesced)
    const int64_t slot = pc.b * static_cast<int64_t>(a.hkv) + pc.h + blockIdx.x;
    const int nrows = min(rows, P::kRows);
    for (int idx = threadIdx.x; idx < nrows * 64; idx += C::kThreads) {
      const int row = idx >> 6;
      const int d4 = (idx & 63) * 4;
      float M = -INFINITY;
      for (int k = 0; k < P::kStreams; ++k) M = fmaxf(M, ml[(k * P::kRows + row) * 2]);
      float L = 0.f;
      if (M != -INFINITY)
        for (int k = 0; k < P::kStreams; ++k)
          L += ml[(k * P::kRows + row) * 2 + 1] * fast_exp2(ml[(k * P::kRows + row) * 2] - M);
      const float inv = (L > 0.f) ? a.out_scale / L : 0.f;
      float4 o;
      o.x = mbuf[merge_pos(row, d4 + 0)] * inv;
      o.y = mbuf[merge_pos(row, d4 + 1)] * inv;
      o.z = mbuf[merge_pos(row, d4 + 2)] * inv;
      o.w = mbuf[merge_pos(row, d4 + 3)] * inv;
      if (slot < a.part_slots) {
        reinterpret_cast<float4*>(a.o_part + (slot * a.rows_per_slot + row) * 256)[d4 >> 2] = o;
        if (d4 == 0) a.lse_part[slot * a.rows_per_slot + row] = (L > 0.f) ? (M + __log2f(L)) * kLn2 : -INFINITY;
      }
    }
    // every consumer warp takes the same decision: the flag (which the
    // producer may set at any time) is sampled once, before the barrier, and
    // read after it (the next sample comes after further barriers)
    if (threadIdx.x == 0) *piece_abort = *abort_flag;
    named_bar_sync(1, C::kThreads);
    if (*piece_abort) break;
  }
}

// ---------------------------------------------------------------------------
// Host side.

// NP = pages per consumer iteration: 2 amortises the softmax reduction and
// gives more independent work, but needs registers the 168-register
// single-n-tile configuration does not have.
template <int KVDT, int NTW, int RG, int NW, int QS = 0, int NP = (NTW > 1 ? 2 : 1)>
int launch_decode(const CUtensorMap& map, const DecodeArgs& a, int grid, cudaStream_t stream) {
  using P = Plan<KVDT, NTW, RG, NW, QS>;
  auto kern = paged_decode_kernel<KVDT, NTW, RG, NW, QS, NP>;
  static std::atomic<uint64_t> configured{0};  // devices whose attribute is set
  const int st = set_smem_limit_once(configured, reinterpret_cast<const void*>(kern), P::kDynamicBytes);
  if (st != PNKV_OK) return st;
  return launch_pdl(kern, dim3(grid), dim3(NW * 32), P::kDynamicBytes, stream, map, a);
}

template <int KVDT>
int dispatch_rows(const CUtensorMap& map, const DecodeArgs& a, int grid, cudaStream_t stream) {
  const int rows = a.rows_per_slot;
  // warps per CTA: NVFP4 stages are small, so many consumer streams each keep
  // two or more stages; bf16 stages are 16 KiB, so fewer streams share the
  // 13 that fit and each still double-buffers.
  constexpr bool fp4 = KVDT != PNKV_KV_BF16;  // coded pools (NVFP4, FP8): small stages
#ifndef PNKV_NVFP4_NW
#define PNKV_NVFP4_NW 12
#define PNKV_NVFP4_QS 0
#endif
// two n-tiles (9 .. 64 rows per KV head): Q fragments staged in shared
// memory or held in registers, pages per consumer iteration
#ifndef PNKV_WIDE_QS
#define PNKV_WIDE_QS 1
#endif
#ifndef PNKV_WIDE_NP
#define PNKV_WIDE_NP 2
#endif
#ifndef PNKV_NVFP4_NP
#define PNKV_NVFP4_NP 1
#endif
  if (rows <= 8)
    return launch_decode<KVDT, 1, 1, fp4 ? PNKV_NVFP4_NW : 7, fp4 ? PNKV_NVFP4_QS : 0, fp4 ? PNKV_NVFP4_NP : 1>(
        map, a, grid, stream);
  // 9 .. 32 rows on an NVFP4 pool (speculative verify): the tensor-core tile
  // with the keys as the M dimension, K and V widened once per page-head
  if (KVDT == PNKV_KV_NVFP4 && rows <= 32) return launch_verify(map, a, grid, stream);
  if (rows <= 16) return launch_decode<KVDT, 2, 1, 7, PNKV_WIDE_QS, PNKV_WIDE_NP>(map, a, grid, stream);
  if (rows <= 32) return launch_decode<KVDT, 2, 2, 7, PNKV_WIDE_QS, PNKV_WIDE_NP>(map, a, grid, stream);
  if (rows <= 64) return launch_decode<KVDT, 2, 4, 5, PNKV_WIDE_QS, PNKV_WIDE_NP>(map, a, grid, stream);
  return PNKV_ERR_UNSUPPORTED;
}

int decode_grid(int* grid) { return device_sm_count(grid); }

}  // namespace
}  // namespace pnkv

extern "C" int64_t pnkv_decode_slots(const pnkv_cache* cache, int32_t batch, int32_t num_q_heads,
                                     int32_t max_qlen) {
  using namespace pnkv;
  int st = check_cache(cache);
  if (st != PNKV_OK) return st;
  if (batch < 1 || max_qlen < 1 || num_q_heads < 1 || num_q_heads % cache->num_kv_heads != 0)
    return PNKV_ERR_INVALID_ARG;
  int grid = 0;
  if ((st = decode_grid(&grid)) != PNKV_OK) return st;
  // the tensor-core tile path (more than 64 rows per KV head) writes one slot
  // per (sequence, KV head, key split); the split-KV path one per piece
  const int32_t group = num_q_heads / cache->num_kv_heads;
  if (static_cast<int64_t>(group) * max_qlen > 64)
    return static_cast<int64_t>(batch) * cache->num_kv_heads *
           prefill_splits(batch, cache->num_kv_heads, group, max_qlen, grid);
  return static_cast<int64_t>(batch) * cache->num_kv_heads + grid;
}

extern "C" int64_t pnkv_work_meta_ints(int32_t batch, int32_t num_kv_heads) {
  if (batch < 1 || num_kv_heads < 1) return PNKV_ERR_INVALID_ARG;
  return 4 + 2 * static_cast<int64_t>(batch) * num_kv_heads;
}

extern "C" int paged_decode_attention(const pnkv_cache* cache, const uint16_t* q_roped,
                                      const int32_t* qo_indptr, const int32_t* page_table,
                                      int64_t pt_stride, const int32_t* seq_lens, int32_t batch,
                                      int64_t total_q, int32_t num_q_heads, int32_t max_qlen, float sm_scale,
                                      int32_t causal, float* o_part, float* lse_part, int64_t part_slots,
                                      int32_t* work_meta, int32_t* dev_err, void* stream) {
  using namespace pnkv;
  int st = check_cache(cache);
  if (st != PNKV_OK) return st;
  if (!q_roped || !qo_indptr || !page_table || !seq_lens || !o_part || !lse_part || !work_meta || !dev_err)
    return PNKV_ERR_INVALID_ARG;
  if (batch < 1 || pt_stride < 1 || max_qlen < 1 || max_qlen > 8192 || num_q_heads < 1 ||
      num_q_heads % cache->num_kv_heads != 0 || total_q < 0)
    return PNKV_ERR_INVALID_ARG;
  if (!std::isfinite(sm_scale) || !(sm_scale > 0.f)) return PNKV_ERR_INVALID_ARG;
  if (!aligned(q_roped, 16) || !aligned(o_part, 16) || !aligned(lse_part, 4)) return PNKV_ERR_INVALID_ARG;
  const int group = num_q_heads / cache->num_kv_heads;
  if (group > 8) return PNKV_ERR_UNSUPPORTED;
  const int64_t rows_per_slot = static_cast<int64_t>(group) * max_qlen;
  if (rows_per_slot > 64)  // many query rows per KV head: the tensor-core tile path
    return launch_prefill(cache, q_roped, qo_indptr, page_table, pt_stride, seq_lens, batch, total_q,
                          num_q_heads, max_qlen, sm_scale, causal, 0.f, o_part, lse_part, part_slots,
                          work_meta, dev_err, as_stream(stream));
  int grid = 0;
  if ((st = decode_grid(&grid)) != PNKV_OK) return st;
  if (part_slots < static_cast<int64_t>(batch) * cache->num_kv_heads + grid) return PNKV_ERR_INVALID_ARG;

  DecodeArgs a;
  a.num_pages = cache->num_pages;
  a.hkv = cache->num_kv_heads;
  a.group = group;
  const bool tensor_scaled = cache->dtype == PNKV_KV_NVFP4 || cache->dtype == PNKV_KV_FP8;
  const float kscale = tensor_scaled ? cache->k_scale : 1.0f;
  a.qk_scale_log2 = sm_scale * kscale * kLog2e;
  a.out_scale = tensor_scaled ? cache->v_scale : 1.0f;
  a.q = q_roped;
  a.qo_indptr = qo_indptr;
  a.page_table = page_table;
  a.pt_stride = pt_stride;
  a.seq_lens = seq_lens;
  a.batch = batch;
  a.total_q = total_q;
  a.hq = num_q_heads;
  a.max_qlen = max_qlen;
  a.rows_per_slot = static_cast<int32_t>(rows_per_slot);
  a.causal = causal ? 1 : 0;
  a.wait_ns = pipeline_wait_ns();
  a.o_part = o_part;
  a.lse_part = lse_part;
  a.part_slots = part_slots;
  a.work_meta = work_meta;
  a.dev_err = dev_err;

  CUtensorMap map;
  const int box_rows = cache->dtype == PNKV_KV_NVFP4 ? Geometry<PNKV_KV_NVFP4>::kBoxRows
                       : cache->dtype == PNKV_KV_FP8 ? Geometry<PNKV_KV_FP8>::kBoxRows
                       : cache->dtype == PNKV_KV_INT8 ? Geometry<PNKV_KV_INT8>::kBoxRows
                                                     : Geometry<PNKV_KV_BF16>::kBoxRows;
  if ((st = make_pool_map(cache, box_rows, &map)) != PNKV_OK) return st;
  cudaStream_t s = as_stream(stream);
  if (cache->dtype == PNKV_KV_NVFP4) return dispatch_rows<PNKV_KV_NVFP4>(map, a, grid, s);
  if (cache->dtype == PNKV_KV_FP8) return dispatch_rows<PNKV_KV_FP8>(map, a, grid, s);
  if (cache->dtype == PNKV_KV_INT8) return dispatch_rows<PNKV_KV_INT8>(map, a, grid, s);
  return dispatch_rows<PNKV_KV_BF16>(map, a, grid, s);
}

extern "C" int paged_prefill_attention_fp4q(const pnkv_cache* cache, const uint16_t* q_roped,
                                           const int32_t* qo_indptr, const int32_t* page_table,
                                           int64_t pt_stride, const int32_t* seq_lens, int32_t batch,
                                           int64_t total_q, int32_t num_q_heads, int32_t max_qlen,
                                           float sm_scale, int32_t causal, float q_scale, float* o_part,
                                           float* lse_part, int64_t part_slots, int32_t* work_meta,
                                           int32_t* dev_err, void* stream) {
  using namespace pnkv;
  int st = check_cache(cache);
  if (st != PNKV_OK) return st;
  if (!q_roped || !qo_indptr || !page_table || !seq_lens || !o_part || !lse_part || !work_meta || !dev_err)
    return PNKV_ERR_INVALID_ARG;
  if (batch < 1 || pt_stride < 1 || max_qlen < 1 || max_qlen > 8192 || num_q_heads < 1 ||
      num_q_heads % cache->num_kv_heads != 0 || total_q < 0)
    return PNKV_ERR_INVALID_ARG;
  if (!std::isfinite(sm_scale) || !(sm_scale > 0.f)) return PNKV_ERR_INVALID_ARG;
  // the query encoder's scales must stay normal in binary32, as the cache's do
  if (!std::isfinite(q_scale) || !(q_scale >= 0x1p-100f) || !(q_scale <= 0x1p100f)) return PNKV_ERR_INVALID_ARG;
  if (!aligned(q_roped, 16) || !aligned(o_part, 16) || !aligned(lse_part, 4)) return PNKV_ERR_INVALID_ARG;
  const int group = num_q_heads / cache->num_kv_heads;
  if (group > 8) return PNKV_ERR_UNSUPPORTED;
  // the block-scaled product is the tile path's: at most 64 rows per KV head
  // (a decode step) stay with paged_decode_attention
  if (static_cast<int64_t>(group) * max_qlen <= 64) return PNKV_ERR_UNSUPPORTED;
  return launch_prefill(cache, q_roped, qo_indptr, page_table, pt_stride, seq_lens, batch, total_q, num_q_heads,
                        max_qlen, sm_scale, causal, q_scale, o_part, lse_part, part_slots, work_meta, dev_err,
                        as_stream(stream));
}
