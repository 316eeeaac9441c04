// Split-KV GQA attention on the 5th-generation tensor cores for KV heads with
// 9 .. 32 query rows per step: speculative-decoding verify, a few new tokens
// per sequence times the GQA group ("Ten Cards, Over 100 tok/s": four draft
// tokens need five query columns per session), over a paged NVFP4 cache
// ("262,144 Tokens on One RTX 5090", section "Why NVFP4 KV changes the
// math").
//
// The attention and its numerics are those of the register-tile decode path
// (q k^T * sm_scale with K, V widened exactly to fp16 from E2M1 x E4M3, fp32
// logits, fp16 probabilities in P.V, fp32 accumulation).  What changes is the
// orientation.  With 30 rows per KV head a row-major tensor-core tile would
// be mostly padding, and mma.sync would need 128 m16n8k16 per page and head,
// more tensor time than the page's bytes take to arrive.  Here the keys are
// the M dimension: a unit is 128 keys (8 pages) of one (sequence, KV head),
//   S^T [128 keys x 32 rows]  = K [128 x 256] . Q^T      (16 MMAs, M128 N32 K16)
//   O^T [256 dims x 32 rows] += V^T [256 x 128] . P^T    (2 x 8 MMAs)
// with K and V^T widened once per unit straight into TMEM as the A operands
// (lane = key for K; lane L = dims 2L and 2L + 1, one per half, for V^T; two
// fp16 per column), Q^T and P^T as the B operands in shared memory, S^T and
// O^T accumulating in TMEM.
// Each page-head's codes are read from HBM once and widened once, whatever
// the number of query rows.
//
// Roles (15 warps):
//   softmax warps 0-3   one key per thread (TMEM lane), 32 rows per thread:
//                       tcgen05.ld of S^T, mask, exponentials against a per-
//                       row reference maximum that moves only when a row's
//                       logits pass it by more than 2^8 (then the exact block
//                       maxima are reduced and O^T and the row sums rescaled),
//                       P^T (fp16, rows contiguous) to shared memory, per-
//                       thread row sums
//   K warps 4-7         K codes x block scales -> fp16 K rows in TMEM
//   V warps 8-11        V codes x block scales -> fp16 V^T rows in TMEM (the
//                       pool stores V slot-pair interleaved, so one code byte
//                       widens to the key pair one TMEM column holds)
//   producer warp 12    one 2-D TMA load per page (the head record) into a
//                       4-stage ring
//   warp 13             allocates TMEM, issues the QK products
//   warp 14             issues the P.V products (both warps run their loops
//                       warp-uniform; one elected thread issues)
// Work is split stream-K over (sequence, KV head, unit) exactly as the decode
// path splits its pages, with the same partial slots, so split_kv_combine
// merges the pieces.
#include <algorithm>
#include <atomic>
#include <cmath>

#include <cudaTypedefs.h>

#include "decode_common.cuh"
#include "device_common.cuh"
#include "host_common.h"
#include "tcgen05.cuh"

namespace pnkv {
namespace {

constexpr int kThreadsV = 480;
constexpr int kKWarp0 = 4, kVWarp0 = 8, kProdWarp = 12, kQkWarp = 13, kPvWarp = 14;
constexpr int kUnitPages = 8;
constexpr int kUnitKeys = 16 * kUnitPages;  // 128: the M of the products
constexpr int kRowsN = 32;                  // query rows per KV head covered (N)
constexpr int kRawStages = 4;
constexpr int kRawPage = 5120;              // 4,608-byte record in a 1,024-aligned slot
constexpr int kRawStage = kUnitPages * kRawPage;
constexpr uint32_t kRecBytesV = 4608;
constexpr int kPStages = 2;
// TMEM slots (128 columns each) of widened K and of widened V^T.  K's slot is
// freed by the QK that read it, so one slot keeps the K widening one QK
// behind; V^T's are freed by the P.V, which waits for the softmax, so V^T
// gets two.
constexpr int kKSlots = 1, kVSlots = 2;
constexpr float kLn2V = 0.6931471805599453f;
constexpr float kMoveThreshold = 8.f;       // log2 units

// shared memory (from a 1,024-aligned base)
constexpr int kRawOff = 0;
constexpr int kQOff = kRawOff + kRawStages * kRawStage;  // Q^T: fp16 [32 rows][256 dims], core matrices
constexpr int kQBytes = kRowsN * 256 * 2;
// P^T: fp16 [128 keys][32 rows], the B of P.V stored MN-major (rows
// contiguous): each 8-key group is four core matrices of 8 keys x 16 bytes
// (rows 8c .. 8c + 7), 128 bytes apart, and the groups are 512 bytes apart.
// A key's 32 probabilities are four 16-byte stores, and a warp's 32 keys
// write each of them as 512 contiguous bytes.
constexpr int kPRowChunk = 128, kPKeyGroup = 512;
constexpr int kPOff = kQOff + kQBytes;
constexpr int kPBytes = (kUnitKeys / 8) * kPKeyGroup;
// per V warp: fp16x2 block scales [page][4 blocks][8 slot pairs]
constexpr int kScrOff = kPOff + kPStages * kPBytes;
constexpr int kScrWarp = kUnitPages * 4 * 8 * 4;
constexpr int kMrefOff = kScrOff + 4 * kScrWarp;         // float [32]: per-row reference maximum (log2)
constexpr int kBaseOff = kMrefOff + kRowsN * 4;          // float [32]: exponent base (reference, 0 if none)
constexpr int kLimOff = kBaseOff + kRowsN * 4;           // int [32]: keys row r may see
constexpr int kAlphaOff = kLimOff + kRowsN * 4;          // float [32]: rescale factors
constexpr int kXchgOff = kAlphaOff + kRowsN * 4;         // float [4 warps][32]: reductions
constexpr int kFlagOff = kXchgOff + 4 * kRowsN * 4;      // uint [2][4]: softmax warps' flags, two rounds
constexpr int kBarOffV = (kFlagOff + 32 + 7) & ~7;
enum {
  V_RAW_FULL = 0,
  V_RAW_EMPTY = V_RAW_FULL + kRawStages,
  // K and V^T slots: widened into the slot; the QK or P.V that read it
  // completed
  V_FULL_K = V_RAW_EMPTY + kRawStages,
  V_FULL_V = V_FULL_K + kKSlots,
  V_FREE_K = V_FULL_V + kVSlots,
  V_FREE_V = V_FREE_K + kKSlots,
  V_S_FULL = V_FREE_V + kVSlots,
  V_S_FREE = V_S_FULL + 2,
  V_P_FULL = V_S_FREE + 2,
  V_PV_DONE = V_P_FULL + kPStages,
  V_Q_FULL = V_PV_DONE + kPStages,
  V_FINAL = V_Q_FULL + 1,
  kNumBarsV = V_FINAL + 1
};
constexpr int kMiscOffV = kBarOffV + kNumBarsV * 8;  // tmem base, abort flag, raw valid[4], armed[4]
constexpr int kSmemV = kMiscOffV + 64 + 1024;
static_assert(kSmemV <= 232448, "verify tile shared memory plan too large");
static_assert(kQOff % 1024 == 0, "raw ring slots need 1,024-byte alignment");

// TMEM columns: the K slots, the V^T slots (halves at +0 and +64), then S^T
// (two stages of 32) and O^T (halves of 32).
constexpr uint32_t kTmemColsV = 512;
constexpr uint32_t kTK = 0, kTV = 128 * kKSlots, kTS = 384, kTO = 448;
static_assert(kTV + 128 * kVSlots <= kTS, "TMEM plan: K and V^T slots overlap S^T");

// Two fp32 lanes per instruction (packed f32x2 on the FMA pipe); each lane
// is the IEEE operation of its scalar form, so results are bitwise the same.
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{ .reg .b64 ra, rb, rc, rd; mov.b64 ra, {%2, %3}; mov.b64 rb, {%4, %5}; mov.b64 rc, {%6, %7};"
      " fma.rn.f32x2 rd, ra, rb, rc; mov.b64 {%0, %1}, rd; }"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}
__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
  float2 d;
  asm("{ .reg .b64 ra, rb, rd; mov.b64 ra, {%2, %3}; mov.b64 rb, {%4, %5};"
      " add.rn.f32x2 rd, ra, rb; mov.b64 {%0, %1}, rd; }"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}

__device__ __forceinline__ uint64_t* vbar(uint8_t* smem, int i) {
  return reinterpret_cast<uint64_t*>(smem + kBarOffV) + i;
}

__device__ __forceinline__ uint32_t par(int64_t g, int n) { return static_cast<uint32_t>((g / n) & 1); }

// The 32-bit TMEM word of a warp's lane quarter: lane 32 * quarter, column c.
__device__ __forceinline__ uint32_t lane_base(uint32_t tmem, int quarter) {
  return tmem + (static_cast<uint32_t>(quarter * 32) << 16);
}

__global__ void __launch_bounds__(kThreadsV, 1)
    verify_tile_kernel(const __grid_constant__ CUtensorMap tmap, const DecodeArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + kMiscOffV);
  volatile uint32_t* abort_flag = misc + 1;
  uint32_t* raw_valid = misc + 2;            // [kRawStages] bit j: page j of the unit loaded
  int32_t* raw_armed = reinterpret_cast<int32_t*>(misc + 6);  // [kRawStages] unit that armed the stage
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  auto bar = [&](int i) { return vbar(smem, i); };

  if (threadIdx.x == 0) {
    for (int i = 0; i < kRawStages; ++i) {
      mbar_init(bar(V_RAW_FULL + i), 1);
      mbar_init(bar(V_RAW_EMPTY + i), 8);  // the K and the V warps
      raw_armed[i] = -1;
    }
    for (int i = 0; i < kKSlots; ++i) {
      mbar_init(bar(V_FULL_K + i), 4);
      mbar_init(bar(V_FREE_K + i), 1);
    }
    for (int i = 0; i < kVSlots; ++i) {
      mbar_init(bar(V_FULL_V + i), 4);
      mbar_init(bar(V_FREE_V + i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(V_S_FULL + i), 1);
      mbar_init(bar(V_S_FREE + i), 4);
    }
    for (int i = 0; i < kPStages; ++i) {
      mbar_init(bar(V_P_FULL + i), 4);
      mbar_init(bar(V_PV_DONE + i), 1);
    }
    mbar_init(bar(V_Q_FULL), 4);
    mbar_init(bar(V_FINAL), 2);
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == kQkWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(misc)),
                 "r"(kTmemColsV)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    tc_fence_before();
  }
  if (warp == kProdWarp && lane == 0) tma_prefetch_desc(&tmap);
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc[0];
  griddep_wait();
  griddep_launch_dependents();

  // this CTA's unit range, as in the decode path
  const int64_t total = total_units<kUnitPages>(a, lane);
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
    for (int b = lane; b < a.batch; b += 32)
      if (load_seq<kUnitPages>(a, b, false).units == 0)
        for (int h = 0; h < a.hkv; ++h) {
          a.work_meta[4 + 2 * (static_cast<int64_t>(b) * a.hkv + h)] = 0;
          a.work_meta[4 + 2 * (static_cast<int64_t>(b) * a.hkv + h) + 1] = 0;
        }
  }
  Walker<kUnitPages> walk;
  walk.init(a, u_begin, u_end, lane);
  Piece pc;
  if (threadIdx.x == 0) {  // slot ranges of the segments that start here, before any work
    Walker<kUnitPages> w0 = walk;
    while (w0.next(a, &pc)) {
      if (pc.p0 != 0) continue;
      const int64_t seg = pc.b * static_cast<int64_t>(a.hkv) + pc.h;
      const int64_t first_cta = pc.seg_start / chunk;
      const int64_t last_cta = (pc.seg_start + pc.s.units - 1) / chunk;
      a.work_meta[4 + 2 * seg] = static_cast<int32_t>(seg + first_cta);
      a.work_meta[4 + 2 * seg + 1] = static_cast<int32_t>(last_cta - first_cta + 1);
    }
  }

  auto fail = [&]() {
    flag_error(a.dev_err, PNKV_DEV_ERR_TIMEOUT);
    *abort_flag = 1;
  };
  auto wait1 = [&](int b, uint32_t parity) -> bool {  // one thread
    if (mbar_try_wait(bar(b), parity)) return true;
    if (*abort_flag) return false;
    if (!mbar_wait(bar(b), parity, a.wait_ns)) {
      fail();
      return false;
    }
    return true;
  };
  auto waitw = [&](int b, uint32_t parity) -> bool {  // warp-uniform
    bool ok = !*abort_flag && mbar_wait(bar(b), parity, a.wait_ns);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok && lane == 0) fail();
    return ok;
  };

  if (warp == kProdWarp) {
    // ---------------------------------------------------------- producer
    const uint64_t policy = l2_policy_evict_first();
    int64_t g = 0;
    bool ok = true;
    while (ok && walk.next(a, &pc)) {
      const int32_t* row = a.page_table + static_cast<int64_t>(pc.b) * a.pt_stride;
      // page ids four units at a time (lane l: unit k0 + l / 8, page l % 8),
      // loaded a group ahead, so that no table read sits between a free
      // slot and its loads
      auto load_ids = [&](int k0) -> int32_t {
        const int u = k0 + (lane >> 3);
        const int pi = (pc.p0 + u) * kUnitPages + (lane & 7);
        return (u < pc.n && pi < pc.s.pages) ? __ldg(row + pi) : -1;
      };
      int32_t ids = load_ids(0), ids_next = load_ids(4);
      for (int k = 0; k < pc.n && ok; ++k, ++g) {
        if (k > 0 && (k & 3) == 0) {
          ids = ids_next;
          ids_next = load_ids(k + 4);
        }
        int32_t page = __shfl_sync(0xffffffffu, ids, ((k & 3) << 3) | (lane & 7));
        const int rs = static_cast<int>(g % kRawStages);
        if (lane == 0) ok = wait1(V_RAW_EMPTY + rs, par(g, kRawStages) ^ 1u);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        if (lane < kUnitPages && (pc.p0 + k) * kUnitPages + lane < pc.s.pages) {
          if (page < 0 || page >= a.num_pages) {
            flag_error(a.dev_err, PNKV_DEV_ERR_PAGE_ID);
            page = -1;
          }
        } else {
          page = -1;
        }
        const unsigned load = __ballot_sync(0xffffffffu, lane < kUnitPages && page >= 0);
        if (lane == 0) {
          raw_valid[rs] = load;
          raw_armed[rs] = static_cast<int32_t>(g);
          mbar_arrive_expect_tx(bar(V_RAW_FULL + rs), __popc(load) * kRecBytesV);
        }
        __syncwarp();
        if (lane < kUnitPages && page >= 0)
          tma_load_2d(smem + kRawOff + rs * kRawStage + lane * kRawPage, &tmap, 0, (page * a.hkv + pc.h) * 36,
                      bar(V_RAW_FULL + rs), policy);
      }
    }
    if (!ok && lane == 0) {
      // loads still landing complete before the CTA exits (fixed bound)
      const int64_t first = g > kRawStages ? g - kRawStages : 0;
      for (int64_t i = first; i <= g; ++i)
        if (raw_armed[i % kRawStages] == static_cast<int32_t>(i))
          mbar_wait(bar(V_RAW_FULL + static_cast<int>(i % kRawStages)), par(i, kRawStages));
    }
  } else if (warp >= kKWarp0 && warp < kKWarp0 + 4) {
    // -------------------------------------------------------- K widening
    // thread = key 32 q + lane of the unit (page key / 16, slot key % 16):
    // its 256 dims, two fp16 per TMEM column, into lane 32 q + lane of the K
    // stage; keys past the sequence or in a page that was not loaded are 0
    const int q = warp - kKWarp0;
    const int key = 32 * q + lane, pg = key >> 4, slot = key & 15;
    const uint32_t krow = pg * kRawPage + slot * 128;  // the slot's code row (chunks swizzled by slot % 8)
    const uint32_t kscale = pg * kRawPage + swz128(16 + (slot >> 3), (slot & 7) * 16);
    // 16 code bytes (32 dims, blocks b and b + 1) and the two blocks' scale
    // bytes -> 16 TMEM columns of fp16 pairs
    auto widen = [](const uint4 w, uint32_t sb, uint32_t (&h)[16]) {
      const uint32_t s2 = e4m3x2_to_f16x2(sb);
      const uint32_t s_lo = prmt(s2, s2, 0x1010u), s_hi = prmt(s2, s2, 0x3232u);
      const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        uint32_t o4[4];
        e2m1x8_unpack(ws[e], o4);
        const uint32_t s = e < 2 ? s_lo : s_hi;
#pragma unroll
        for (int f = 0; f < 4; ++f) h[4 * e + f] = hmul2(o4[f], s);
      }
    };
    int64_t g = 0;
    bool ok = true;
    while (ok && walk.next(a, &pc)) {
      for (int k = 0; k < pc.n && ok; ++k, ++g) {
        const int rs = static_cast<int>(g % kRawStages);
        const int ks = static_cast<int>(g % kKSlots);
        // the slot's previous user is the QK of unit g - kKSlots
        ok = waitw(V_RAW_FULL + rs, par(g, kRawStages)) &&
             (g < kKSlots || waitw(V_FREE_K + ks, par(g - kKSlots, kKSlots)));
        if (!ok) break;
        // a dead key's scales are zeroed, which zeroes its row whatever the codes
        const bool live = ((raw_valid[rs] >> pg) & 1) && (pc.p0 + k) * kUnitKeys + key < pc.s.len;
        const uint32_t smask = live ? 0xFFFFFFFFu : 0u;
        const uint32_t rawb = smem_addr(smem + kRawOff + rs * kRawStage);
        const uint32_t taddr = lane_base(tmem, q) + kTK + 128 * ks;
        // a runtime loop keeps the code small (the tile's roles share each
        // SM sub-partition's instruction cache); two operand sets in turn, so
        // that each step's loads are issued before the previous step is
        // converted (the last look-ahead wraps to step 0: in bounds, unused)
        const uint32_t kr = rawb + krow;
        struct KOps {
          uint4 w0, w1;
          uint32_t sw;
        };
        auto kload = [&](int c2, KOps& o) {  // chunks 2 c2, 2 c2 + 1: dims 64 c2 .. + 63, blocks 4 c2 .. + 3
          o.w0 = lds128(kr + ((((2 * c2) ^ slot) & 7) << 4));
          o.w1 = lds128(kr + ((((2 * c2 + 1) ^ slot) & 7) << 4));
          o.sw = lds32(rawb + kscale + 4 * c2);
        };
        auto kwiden = [&](int c2, const KOps& o) {
          const uint32_t sw = o.sw & smask;
          uint32_t h[16];
          widen(o.w0, sw & 0xFFFFu, h);
          tmem_st16(taddr + 32 * c2, h);
          widen(o.w1, sw >> 16, h);
          tmem_st16(taddr + 32 * c2 + 16, h);
        };
        KOps ka, kb;
        kload(0, ka);
#pragma unroll 1
        for (int c2 = 0; c2 < 4; c2 += 2) {
          kload(c2 + 1, kb);
          kwiden(c2, ka);
          kload((c2 + 2) & 3, ka);
          kwiden(c2 + 1, kb);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(bar(V_FULL_K + ks));
          mbar_arrive(bar(V_RAW_EMPTY + rs));
        }
      }
    }
  } else if (warp >= kVWarp0 && warp < kVWarp0 + 4) {
    // -------------------------------------------------------- V widening
    // thread = TMEM lane L = 32 q + lane of the V^T halves, dims 2L (half 0)
    // and 2L + 1 (half 1): the V^T accumulator's lane L, half h is dim
    // 2L + h (the product does not care how dims map to lanes, only the
    // epilogue does).  Dims 2L, 2L + 1 are adjacent bytes of one slot-pair
    // row (rows 18 .. 25 + 2 pr hold dims 0 .. 127 of pair pr, the next rows
    // dims 128 .. 255), so one 16-bit load gives both, and both lie in block
    // L / 8, whose scales the 8 lanes of that block share.  The warp first
    // converts the block scales of its four blocks (4q .. 4q + 3) over the
    // unit's 8 pages into a scratch of fp16 pairs [page][block][slot pair];
    // slots past the sequence or in a page that was not loaded scale to 0,
    // which zeroes their values whatever the stale codes (E2M1 has no
    // infinities).
    const int q = warp - kVWarp0;
    const uint32_t scr = smem_addr(smem + kScrOff + q * kScrWarp);
    const int L = 32 * q + lane;
    const uint32_t hrow = 18 + (L >> 6);   // slot-pair row of pair 0 for this lane's dims
    const uint32_t col = (2 * L) & 127;    // their byte in that row
    // swizzled offsets of pairs 0 .. 3 (pairs 4 .. 7 are 8 rows = 1,024 bytes
    // further, with the same residues mod 8)
    uint32_t cofs[4];
#pragma unroll
    for (int m = 0; m < 4; ++m) cofs[m] = swz128(hrow + 2 * m, col);
    // scratch fill: lane -> block 4q + lane / 8, slot pair fp = lane % 8;
    // one word per page.  The scale of (slot s, block b) is byte 16 (s % 8)
    // + b of raw row 34 + s / 8.
    const int fp = lane & 7;
    const int fblk = 4 * q + (lane >> 3);
    const uint32_t fo0 = swz128(34 + (fp >> 2), ((2 * fp) & 7) * 16 + fblk);
    const uint32_t fo1 = swz128(34 + (fp >> 2), ((2 * fp + 1) & 7) * 16 + fblk);
    uint32_t* fdst = reinterpret_cast<uint32_t*>(smem + kScrOff + q * kScrWarp) + lane;  // + 32 j
    const uint32_t sread = scr + (lane >> 3) * 32;  // + 128 j: the 8 pairs of the lane's block
    int64_t g = 0;
    bool ok = true;
    while (ok && walk.next(a, &pc)) {
      for (int k = 0; k < pc.n && ok; ++k, ++g) {
        const int rs = static_cast<int>(g % kRawStages);
        ok = waitw(V_RAW_FULL + rs, par(g, kRawStages));
        if (!ok) break;
        const uint32_t valid = raw_valid[rs];
        const uint32_t raw = smem_addr(smem + kRawOff + rs * kRawStage);
        const int keys_left = pc.s.len - (pc.p0 + k) * kUnitKeys;  // keys of the unit in the sequence
        {
          uint32_t b0[kUnitPages], b1[kUnitPages];
#pragma unroll
          for (int j = 0; j < kUnitPages; ++j) {
            b0[j] = lds8(raw + j * kRawPage + fo0);
            b1[j] = lds8(raw + j * kRawPage + fo1);
          }
          if (valid == (1u << kUnitPages) - 1 && keys_left >= kUnitKeys) {  // every slot live (uniform)
#pragma unroll
            for (int j = 0; j < kUnitPages; ++j) fdst[32 * j] = e4m3x2_to_f16x2(prmt(b0[j], b1[j], 0x0040u));
          } else {
#pragma unroll
            for (int j = 0; j < kUnitPages; ++j) {
              const int s0 = 16 * j + 2 * fp;  // the pair's first key in the unit
              const bool pv = (valid >> j) & 1;
              const uint32_t m =
                  (pv && s0 < keys_left ? 0x0000FFFFu : 0u) | (pv && s0 + 1 < keys_left ? 0xFFFF0000u : 0u);
              fdst[32 * j] = e4m3x2_to_f16x2(prmt(b0[j], b1[j], 0x0040u)) & m;
            }
          }
        }
        __syncwarp();
        // the V^T slot's previous user is the P.V of unit g - kVSlots
        const int vs = static_cast<int>(g % kVSlots);
        if (g >= kVSlots) ok = waitw(V_FREE_V + vs, par(g - kVSlots, kVSlots));
        if (!ok) break;
        const uint32_t taddr = lane_base(tmem, q) + kTV + 128 * vs;
        // operands of page j: its 8 pair scales and 8 code pairs
        struct VOps {
          uint4 s0, s1;
          uint32_t code[8];
        };
        auto vload = [&](int j, VOps& o) {
          const uint32_t pg = raw + j * kRawPage;
          o.s0 = lds128(sread + j * 128);
          o.s1 = lds128(sread + j * 128 + 16);
#pragma unroll
          for (int pr = 0; pr < 8; ++pr) o.code[pr] = lds16(pg + cofs[pr & 3] + (pr >> 2) * 1024);
        };
        auto vwiden = [&](int j, const VOps& o) {  // page j = 8 columns of each half
          const uint32_t sf[8] = {o.s0.x, o.s0.y, o.s0.z, o.s0.w, o.s1.x, o.s1.y, o.s1.z, o.s1.w};
          uint32_t h0[8], h1[8];
#pragma unroll
          for (int pr = 0; pr < 8; ++pr) {
            uint32_t o2[2];
            e2m1x4_unpack(o.code[pr], o2);  // byte 0: dim 2L, byte 1: dim 2L + 1
            h0[pr] = hmul2(o2[0], sf[pr]);
            h1[pr] = hmul2(o2[1], sf[pr]);
          }
          tmem_st8(taddr + 8 * j, h0);
          tmem_st8(taddr + 64 + 8 * j, h1);
        };
        // two operand sets in turn: each page's loads are issued before the
        // previous page is converted (the last look-ahead wraps to page 0:
        // in bounds, unused)
        VOps va, vb;
        vload(0, va);
#pragma unroll 1
        for (int j = 0; j < kUnitPages; j += 2) {
          vload(j + 1, vb);
          vwiden(j, va);
          vload((j + 2) & (kUnitPages - 1), va);
          vwiden(j + 1, vb);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(bar(V_FULL_V + vs));
          mbar_arrive(bar(V_RAW_EMPTY + rs));
        }
      }
    }
  } else if (warp == kQkWarp || warp == kPvWarp) {
    // --------------------------------------------------------------- MMA
    // QK and P.V from different warps, so a wait of one never stalls the
    // other's queue of products.  The whole warp runs the loop and waits;
    // one elected thread issues.  The shared-memory descriptors advance by
    // their encoded address field (16-byte units) per product.
    const bool qk = warp == kQkWarp;
    const uint32_t idesc = idesc_f16(128, kRowsN), idesc_pv = idesc_f16_bmn(128, kRowsN);
    const uint64_t qdesc = smem_desc(smem_addr(smem + kQOff), 128, 4096);
    const uint64_t pdesc0 = smem_desc(smem_addr(smem + kPOff), kPKeyGroup, kPRowChunk);
    int64_t g = 0, npiece = 0;
    bool ok = true, issued = false;
    while (ok && walk.next(a, &pc)) {
      if (qk) ok = waitw(V_Q_FULL, static_cast<uint32_t>(npiece & 1));
      for (int k = 0; ok && k < pc.n; ++k, ++g) {
        if (qk) {
          const int sb = static_cast<int>(g & 1);
          const int ks = static_cast<int>(g % kKSlots);
          ok = waitw(V_FULL_K + ks, par(g, kKSlots)) && (g < 2 || waitw(V_S_FREE + sb, par(g - 2, 2)));
          if (!ok) break;
          tc_fence_after();
          const uint32_t d = tmem + kTS + 32 * sb, a0 = tmem + kTK + 128 * ks;
          if (elect_one()) {
#pragma unroll
            for (int kk = 0; kk < 16; ++kk)  // 16 dims: 8 TMEM columns of K, 2 core matrices (256 B) of Q^T
              umma_f16_ta(d, a0 + 8 * kk, qdesc + 16 * kk, idesc, kk > 0);
            umma_commit(bar(V_S_FULL + sb));
            umma_commit(bar(V_FREE_K + ks));
          }
          __syncwarp();
        } else {
          const int pb = static_cast<int>(g % kPStages);
          const int vs = static_cast<int>(g % kVSlots);
          ok = waitw(V_FULL_V + vs, par(g, kVSlots)) && waitw(V_P_FULL + pb, par(g, kPStages));
          if (!ok) break;
          tc_fence_after();
          const uint64_t pdesc = pdesc0 + static_cast<uint64_t>(pb * (kPBytes >> 4));
          const uint32_t a0 = tmem + kTV + 128 * vs;
          const uint32_t acc = k > 0 ? 1u : 0u;
          if (elect_one()) {
            // the two halves' products interleaved: two independent
            // accumulation chains for the tensor core
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)  // 16 keys: 8 TMEM columns of V^T, 2 key groups (1 KB) of P^T
#pragma unroll
              for (int hh = 0; hh < 2; ++hh)
                umma_f16_ta(tmem + kTO + 32 * hh, a0 + 64 * hh + 8 * kk, pdesc + 64 * kk, idesc_pv,
                            kk > 0 ? 1u : acc);
            umma_commit(bar(V_FREE_V + vs));
            umma_commit(bar(V_PV_DONE + pb));
          }
          __syncwarp();
        }
        issued = true;
      }
      ++npiece;
    }
    // every issued product completes before TMEM is released (fixed bound)
    if (elect_one()) {
      if (issued)
        umma_commit(bar(V_FINAL));
      else
        mbar_arrive(bar(V_FINAL));
    }
    __syncwarp();
    mbar_wait(bar(V_FINAL), 0);
  } else {
    // ----------------------------------------------------------- softmax
    // thread = key 32 q + lane of the unit (TMEM lane); columns = rows.  The
    // four warps meet at named barrier 1 at fixed points, exchanging their
    // state there, so that all of them take the same branch and stop
    // together (a warp whose wait gave up carries on to the next meeting).
    const int q = warp;
    const int key = 32 * q + lane;
    float* mref = reinterpret_cast<float*>(smem + kMrefOff);
    float* basev = reinterpret_cast<float*>(smem + kBaseOff);
    int* lim = reinterpret_cast<int*>(smem + kLimOff);
    float* alpha = reinterpret_cast<float*>(smem + kAlphaOff);
    float* xchg = reinterpret_cast<float*>(smem + kXchgOff);
    volatile uint32_t* flags = reinterpret_cast<uint32_t*>(smem + kFlagOff);
    const uint32_t lb = lane_base(tmem, q);
    // meeting: every warp posts bits, all read the OR and the AND.  The
    // posts alternate between two flag sets, so one barrier suffices: a
    // warp posts into a set again only two meetings later, after every warp
    // has passed the meeting in between (and so has read that set).
    uint32_t meets = 0;
    auto meet = [&](uint32_t bits, uint32_t* all_and, uint32_t* any_or) {
      volatile uint32_t* f = flags + 4 * (meets & 1);
      ++meets;
      if (lane == 0) f[q] = bits;
      named_bar_sync(1, 128);
      const uint32_t f0 = f[0], f1 = f[1], f2 = f[2], f3 = f[3];
      *all_and = f0 & f1 & f2 & f3;
      *any_or = f0 | f1 | f2 | f3;
    };
    int64_t g = 0;
    bool ok = true;
    uint32_t all_and, any_or;
    while (walk.next(a, &pc)) {
      meet(ok ? 1u : 0u, &all_and, &any_or);
      if (!(all_and & 1u)) break;
      const int rows = a.group * pc.s.qlen;
      // Q^T of the piece (B of QK): thread t: row t / 4, dims 64 (t % 4) ..
      // + 63, fp16, core-matrix layout [32 rows][256 dims]; rows past the
      // piece's are zero.  (Every QK of the previous piece has completed: its
      // S were all read.)
      {
        const int t = threadIdx.x, r = t >> 2, d0 = 64 * (t & 3);
        const bool live = r < rows;
        const uint4* src = live ? reinterpret_cast<const uint4*>(
                                      a.q + (static_cast<int64_t>(pc.s.q0 + r / a.group) * a.hq + pc.h * a.group +
                                             r % a.group) * 256 + d0)
                                : nullptr;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint4 w = live ? __ldg(src + c) : make_uint4(0, 0, 0, 0);
          const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
          uint32_t h[4];
#pragma unroll
          for (int e = 0; e < 4; ++e)
            h[e] = f32x2_to_f16x2(__uint_as_float(ws[e] << 16), __uint_as_float(ws[e] & 0xFFFF0000u));
          *reinterpret_cast<uint4*>(smem + kQOff + core_off(r, d0 + 8 * c, 256)) = make_uint4(h[0], h[1], h[2], h[3]);
        }
        fence_proxy_async();
      }
      if (threadIdx.x < kRowsN) {
        const int r = threadIdx.x;
        mref[r] = -INFINITY;
        basev[r] = 0.f;
        lim[r] = r < rows ? (a.causal ? pc.s.len - pc.s.qlen + r / a.group + 1 : pc.s.len) : 0;
      }
      // keys every query row of the piece sees: a unit below this needs no
      // mask (its rows past the piece's carry harmless values, never written)
      const int vis_all = a.causal ? pc.s.len - pc.s.qlen + 1 : pc.s.len;
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(V_Q_FULL));
      named_bar_sync(1, 128);  // mref and lim written
      float l[kRowsN];
#pragma unroll
      for (int r = 0; r < kRowsN; ++r) l[r] = 0.f;

      for (int k = 0; k < pc.n; ++k, ++g) {
        const int sb = static_cast<int>(g & 1), pb = static_cast<int>(g % kPStages);
        float x[kRowsN];
        bool viol = false;
        const int kg = (pc.p0 + k) * kUnitKeys + key;
        // S^T column r of this key -> masked logits relative to the row's
        // exponent base, x = s * scale - base (log2 units, one FFMA); the S
        // slot is released once no reduction can read it again
        const bool unmasked = (pc.p0 + k + 1) * kUnitKeys <= vis_all;  // uniform over the CTA
        auto load_x = [&]() {
          uint32_t sr[kRowsN];
          tmem_ld32(lb + kTS + 32 * sb, sr);
          float4 b4[kRowsN / 4];  // the bases, read while the TMEM load is in flight
#pragma unroll
          for (int r4 = 0; r4 < kRowsN / 4; ++r4) b4[r4] = reinterpret_cast<const float4*>(basev)[r4];
          tmem_wait_ld();
          const float2 sc2 = make_float2(a.qk_scale_log2, a.qk_scale_log2);
#pragma unroll
          for (int r4 = 0; r4 < kRowsN / 4; ++r4) {
            const float2 lo = ffma2(make_float2(__uint_as_float(sr[4 * r4]), __uint_as_float(sr[4 * r4 + 1])), sc2,
                                    make_float2(-b4[r4].x, -b4[r4].y));
            const float2 hi = ffma2(make_float2(__uint_as_float(sr[4 * r4 + 2]), __uint_as_float(sr[4 * r4 + 3])),
                                    sc2, make_float2(-b4[r4].z, -b4[r4].w));
            x[4 * r4] = lo.x;
            x[4 * r4 + 1] = lo.y;
            x[4 * r4 + 2] = hi.x;
            x[4 * r4 + 3] = hi.y;
          }
          if (!unmasked) {
#pragma unroll
            for (int r4 = 0; r4 < kRowsN; r4 += 4) {
              const int4 l4 = *reinterpret_cast<const int4*>(lim + r4);
              const int lv[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
              for (int e = 0; e < 4; ++e)
                if (kg >= lv[e]) x[r4 + e] = -INFINITY;
            }
          }
        };
        if (ok) ok = waitw(V_S_FULL + sb, par(g, 2));
        if (ok) tc_fence_after();
        // one or two passes: x from S^T; after a reduction (which moves the
        // bases) x is read again.  (One copy of the load keeps the code small.)
        for (bool second = false;; second = true) {
          if (ok) load_x();
          if (second) break;
          if (ok) {
            // a row's reference moves when its logits pass it by more than
            // the threshold.  The first unit of a piece always reduces (it
            // sets the references); after it every row either has a finite
            // reference or sees no key of the piece at all (a row's visible
            // keys are a prefix of the sequence, and the piece's first unit
            // holds its first key), so the test is on x alone.
            float o0 = x[0], o1 = x[1];
#pragma unroll
            for (int r = 2; r + 3 < kRowsN; r += 4) {  // rows 2 .. 29 in two chains
              o0 = fmax3(o0, x[r], x[r + 1]);
              o1 = fmax3(o1, x[r + 2], x[r + 3]);
            }
            viol = fmax3(fmaxf(o0, o1), x[kRowsN - 2], x[kRowsN - 1]) > kMoveThreshold;
          }
          meet((ok ? 1u : 0u) | (__any_sync(0xffffffffu, viol) ? 2u : 0u), &all_and, &any_or);
          if (!(all_and & 1u) || !(k == 0 || (any_or & 2u))) break;
          // the unit's exact row maxima (warp transpose-reduction, then over
          // the four warps, relative to the old bases) move the references
          // that grew by more than the threshold; x is then recomputed
          // against the new bases
#pragma unroll
          for (int s = 16; s >= 1; s >>= 1) {
            const bool up = lane & s;
#pragma unroll
            for (int i = 0; i < s; ++i) {
              const float send = up ? x[i] : x[i + s];
              const float recv = __shfl_xor_sync(0xffffffffu, send, s);
              x[i] = fmaxf(up ? x[i + s] : x[i], recv);
            }
          }
          xchg[q * 32 + lane] = x[0];  // the warp's maximum of row `lane`
          named_bar_sync(1, 128);
          if (threadIdx.x < kRowsN) {
            const int r = threadIdx.x;
            const float bm = fmaxf(fmaxf(xchg[r], xchg[32 + r]), fmaxf(xchg[64 + r], xchg[96 + r])) + basev[r];
            const float m0 = mref[r];
            const bool move = bm > m0 + kMoveThreshold || (m0 == -INFINITY && bm > -INFINITY);
            const float mn = move ? bm : m0;
            alpha[r] = (move && m0 != -INFINITY) ? fast_exp2(m0 - mn) : 1.f;
            mref[r] = mn;
            basev[r] = mn == -INFINITY ? 0.f : mn;
          }
          named_bar_sync(1, 128);
#pragma unroll
          for (int r = 0; r < kRowsN; ++r) l[r] *= alpha[r];
          if (k > 0) {
            // O^T (lane = dim, column = row) holds this piece's products up to
            // unit g - 1: rescale its columns once that P.V has completed
            ok = waitw(V_PV_DONE + static_cast<int>((g - 1) % kPStages), par(g - 1, kPStages));
            if (ok) {
              tc_fence_after();
#pragma unroll 1
              for (int c = 0; c < 2 * kRowsN; c += 16) {  // both halves, 16 columns at a time
                uint32_t o[16];
                tmem_ld16(lb + kTO + c, o);
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 16; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha[(c + e) & 31]);
                tmem_st16(lb + kTO + c, o);
              }
              tmem_wait_st();
              tc_fence_before();
            }
          }
        }
        if (!(all_and & 1u)) {
          ok = false;
          break;
        }
        if (!ok) continue;  // reported at the next meeting
        // S^T of this unit has been read for the last time: free its slot
        // for the QK two units on
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(V_S_FREE + sb));
        // p = 2^x (at most 2^threshold; 0 for masked keys)
#pragma unroll
        for (int r = 0; r < kRowsN; r += 2) {
          x[r] = fast_exp2(x[r]);
          x[r + 1] = fast_exp2(x[r + 1]);
          const float2 s2 = fadd2(make_float2(l[r], l[r + 1]), make_float2(x[r], x[r + 1]));
          l[r] = s2.x;
          l[r + 1] = s2.y;
        }
        // P^T slot pb was last read by the P.V of unit g - kPStages
        if (g >= kPStages) ok = waitw(V_PV_DONE + pb, par(g - kPStages, kPStages));
        if (!ok) continue;
        // this key's 32 probabilities as fp16, four 16-byte pieces (rows
        // 8c .. 8c + 7) of the MN-major P^T
        {
          uint8_t* pt = smem + kPOff + pb * kPBytes + (key >> 3) * kPKeyGroup + (key & 7) * 16;
#pragma unroll
          for (int c = 0; c < 4; ++c)
            *reinterpret_cast<uint4*>(pt + c * kPRowChunk) =
                make_uint4(f32x2_to_f16x2(x[8 * c], x[8 * c + 1]), f32x2_to_f16x2(x[8 * c + 2], x[8 * c + 3]),
                           f32x2_to_f16x2(x[8 * c + 4], x[8 * c + 5]), f32x2_to_f16x2(x[8 * c + 6], x[8 * c + 7]));
          fence_proxy_async();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(V_P_FULL + pb));
        }
      }
      if (!(all_and & 1u)) break;
      // ---- end of the piece: the last P.V, the row sums, the partial
      if (ok) ok = waitw(V_PV_DONE + static_cast<int>((g - 1) % kPStages), par(g - 1, kPStages));
      {
#pragma unroll
        for (int s = 16; s >= 1; s >>= 1) {
          const bool up = lane & s;
#pragma unroll
          for (int i = 0; i < s; ++i) {
            const float send = up ? l[i] : l[i + s];
            const float recv = __shfl_xor_sync(0xffffffffu, send, s);
            l[i] = (up ? l[i + s] : l[i]) + recv;
          }
        }
        xchg[q * 32 + lane] = l[0];  // the warp's sum of row `lane`
      }
      meet(ok ? 1u : 0u, &all_and, &any_or);
      if (!(all_and & 1u)) break;
      if (threadIdx.x < kRowsN) {
        const int r = threadIdx.x;
        alpha[r] = (xchg[r] + xchg[32 + r]) + (xchg[64 + r] + xchg[96 + r]);  // the row's sum L
      }
      named_bar_sync(1, 128);
      const int64_t slot = pc.b * static_cast<int64_t>(a.hkv) + pc.h + blockIdx.x;
      tc_fence_after();
#pragma unroll 1
      for (int c = 0; c < kRowsN; c += 8) {  // 8 rows at a time: O^T lane `key`, half h = dim 2 key + h
        uint32_t o0[8], o1[8];
        tmem_ld8(lb + kTO + c, o0);
        tmem_ld8(lb + kTO + 32 + c, o1);
        tmem_wait_ld();
        if (slot < a.part_slots) {
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int r = c + e;
            if (r < rows) {
              const float L = alpha[r];
              const float f = L > 0.f ? a.out_scale / L : 0.f;
              *reinterpret_cast<float2*>(a.o_part + (slot * a.rows_per_slot + r) * 256 + 2 * key) =
                  make_float2(__uint_as_float(o0[e]) * f, __uint_as_float(o1[e]) * f);
            }
          }
        }
      }
      tc_fence_before();
      if (threadIdx.x < kRowsN && threadIdx.x < rows && slot < a.part_slots) {
        const int r = threadIdx.x;
        const float L = alpha[r];
        a.lse_part[slot * a.rows_per_slot + r] = L > 0.f ? (mref[r] + __log2f(L)) * kLn2V : -INFINITY;
      }
      // (alpha and mref are rewritten only after the next piece's meeting)
    }
  }

  __syncthreads();
  if (warp == kQkWarp) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemColsV) : "memory");
  }
}

}  // namespace

// Launch the tensor-core verify tile (NVFP4 pools, 9 .. 32 query rows per KV
// head); `map` is the pool's whole-record tensor map.
int launch_verify(const CUtensorMap& map, const DecodeArgs& a, int grid, cudaStream_t stream) {
  static std::atomic<uint64_t> configured{0};  // devices whose attribute is set
  const int st = set_smem_limit_once(configured, reinterpret_cast<const void*>(verify_tile_kernel), kSmemV);
  if (st != PNKV_OK) return st;
  return launch_pdl(verify_tile_kernel, dim3(grid), dim3(kThreadsV), kSmemV, stream, map, a);
}

}  // namespace pnkv
