// Chunked-prefill attention tile on the 5th-generation tensor cores
// (tcgen05 MMAs with TMEM accumulators), used by paged_decode_attention when a
// KV head has more query rows than the register-tile decode path handles.
//
// Same attention as the decode path: for every query row, softmax(q k^T *
// sm_scale) v over its visible keys (causal inside the chunk: query token t
// of a chunk of qlen tokens at the end of a sequence of len keys sees keys
// 0 .. len - qlen + t).  The chunk is prefilled against the paged NVFP4 cache
// ("A 1,048,576-token context on two RTX 5090s", section "Against vLLM:
// prefill loses, decode wins, and one surprise": prompts are ingested in
// chunks, 1,024 tokens in one engine and 16,768 batched tokens in the other).
//
// A CTA tile is 128 TMEM lanes = 128 query rows of one KV head: T = 128 / G
// consecutive query tokens times the G query heads that share the KV head
// (GQA), so every KV byte read serves all G heads.  Keys are swept in
// blocks of 64 (four 16-token pages):
//   producer warp   TMA-loads the four pages' NVFP4 head records (raw ring)
//   dequant warps   widen K to fp16 [64 keys][256 dims] and V to fp16
//                   V^T [256 dims][64 keys] (E2M1 x E4M3 is exact in fp16),
//                   both in the no-swizzle K-major core-matrix layout
//   MMA thread      S = Q K^T   (M 128, N 64, K 256)  -> TMEM ring, with Q
//                               (fp16) held in TMEM as the A operand, so
//                               shared memory feeds only K
//                   O += P V    (M 128, N 256, K 64)  -> TMEM
//   softmax warps   one row per thread: tcgen05.ld of S, online softmax,
//                   P (fp16) -> shared memory; O is rescaled in TMEM only when
//                   a row's running maximum grows by more than 2^8, so the
//                   exponentials stay below 256 and most blocks need no
//                   rescale (the row sum adds the fp32 exponentials; P V
//                   takes them rounded to fp16, a relative difference of at
//                   most 2^-11 per term)
// Per-tensor K/V scales fold into the logit scale and the output, as in the
// decode path.  The CTA writes one normalised partial (with its natural-log
// LSE) per row into the (sequence, KV head) slot, which split_kv_combine
// passes through.
#include <algorithm>
#include <cmath>

#include <cudaTypedefs.h>

#include "device_common.cuh"
#include "host_common.h"

namespace pnkv {
namespace {

constexpr int kThreads = 480;         // 15 warps
// warps 0-3 run the softmax, one TMEM lane quarter (32 rows) each
constexpr int kDequantWarp0 = 4;      // warps 4-11
constexpr int kDequantWarps = 8;
constexpr int kProducerWarp = 12;
constexpr int kMmaWarp = 13;          // issues P V; allocates TMEM
constexpr int kQkWarp = 14;           // issues QK
constexpr int kBlockKeys = 64;        // keys per KV block (four pages)
constexpr int kBlockPages = kBlockKeys / 16;
// ring depths.  The QK of block g waits for the softmax of block g - kSStages
// to have loaded its S slot, so QK runs up to kSStages blocks ahead of the
// softmax, and the softmax of a block overlaps the P V of the one before.
constexpr int kRawStages = 3;
constexpr int kKStages = 2;
constexpr int kVStages = 2;
constexpr int kSStages = 2;
constexpr int kPStages = 2;
constexpr int kRawPageBytes = 5120;   // 4,608-byte record, 1,024-aligned slot
constexpr int kRawStageBytes = kBlockPages * kRawPageBytes;
constexpr uint32_t kRecBytes = 4608;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.f;  // log2 units

// Shared memory plan (offsets from a 1,024-byte aligned base).  Q lives in
// TMEM (the A operand of S = Q K^T), so shared memory holds only the streamed
// operands.
constexpr int kKOff = 0;                                  // ring of [64 x 256] fp16
constexpr int kKBytes = kBlockKeys * 256 * 2;
constexpr int kVOff = kKOff + kKStages * kKBytes;         // ring of [256 x 64] fp16
constexpr int kVBytes = 256 * kBlockKeys * 2;
constexpr int kPOff = kVOff + kVStages * kVBytes;         // ring of [128 x 64] fp16
constexpr int kPBytes = 128 * kBlockKeys * 2;
constexpr int kRawOff = kPOff + kPStages * kPBytes;       // raw NVFP4 records
constexpr int kScrOff = kRawOff + kRawStages * kRawStageBytes;  // per dequant warp: V scales
constexpr int kScrWarpBytes = kBlockPages * 32;                 // [page][2 blocks][16 slots]
constexpr int kBarOff = kScrOff + kDequantWarps * kScrWarpBytes;
enum {
  B_RAW_FULL = 0,
  B_RAW_EMPTY = B_RAW_FULL + kRawStages,
  B_K_FULL = B_RAW_EMPTY + kRawStages,
  B_K_FREE = B_K_FULL + kKStages,
  B_V_FULL = B_K_FREE + kKStages,
  B_V_FREE = B_V_FULL + kVStages,
  B_S_FULL = B_V_FREE + kVStages,
  B_S_FREE = B_S_FULL + kSStages,
  B_P_FULL = B_S_FREE + kSStages,
  B_PV_DONE = B_P_FULL + kPStages,
  B_Q_FULL = B_PV_DONE + kPStages,
  B_FINAL = B_Q_FULL + 1,
  kNumBars = B_FINAL + 1
};
constexpr int kMiscOff = kBarOff + kNumBars * 8;          // tmem base, abort, raw valid[]
constexpr int kSmemBytes = kMiscOff + 64 + 1024;
static_assert(kSmemBytes <= 232448, "prefill shared memory plan too large");

// TMEM columns: the S ring at 0 and 64; O at 128 .. 383; Q (fp16, two per
// 32-bit column) at 384 .. 511.
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemS = 0;
constexpr uint32_t kTmemO = kSStages * kBlockKeys;
constexpr uint32_t kTmemQ = kTmemO + 256;
static_assert(kTmemQ + 128 <= kTmemCols, "TMEM plan too large");

struct PrefillArgs {
  int64_t num_pages;
  int32_t hkv, group, tpt;  // tpt: query tokens per tile (128 / group)
  float qk_scale_log2, out_scale;
  const uint16_t* q;
  const int32_t* qo_indptr;
  const int32_t* page_table;
  int64_t pt_stride;
  const int32_t* seq_lens;
  int32_t batch, hq, max_qlen, rows_per_slot, causal;
  int32_t splits;  // key-range splits per tile (slots per (sequence, KV head))
  float* o_part;
  float* lse_part;
  int64_t part_slots;
  int32_t* work_meta;
  int32_t* dev_err;
};

// ------------------------------------------------------------ tcgen05 --
// Byte offset of element (r, k) in a no-swizzle K-major tile whose rows hold
// kdim 16-bit elements: 8 x 8 core matrices of 128 contiguous bytes, the core
// matrices of a row group consecutive along K.
__device__ __forceinline__ uint32_t core_off(uint32_t r, uint32_t k, uint32_t kdim) {
  return (((r >> 3) * (kdim >> 3) + (k >> 3)) << 7) + ((r & 7) << 4) + ((k & 7) << 1);
}

// Shared-memory matrix descriptor: start address, leading-dimension byte
// offset (between core matrices along K), stride-dimension byte offset
// (between 8-row groups), descriptor version 1, no swizzle.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  return d;
}

// Instruction descriptor, kind::f16: fp16 A and B, fp32 D, both K-major.
__host__ __device__ constexpr uint32_t idesc_f16(int m, int n) {
  return (1u << 4) | (static_cast<uint32_t>(n >> 3) << 17) | (static_cast<uint32_t>(m >> 4) << 24);
}

__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{ .reg .pred p; setp.ne.b32 p, %4, 0; tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p; }" ::"r"(
          d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Same with the A operand in TMEM (row i in lane i, two fp16 per column).
__device__ __forceinline__ void umma_f16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{ .reg .pred p; setp.ne.b32 p, %4, 0; tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p; }" ::"r"(
          d_tmem),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_addr(bar))
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// 16 consecutive TMEM columns of this warp's 32 lanes (one row per thread).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
// 32 consecutive TMEM columns of this warp's 32 lanes into r[0 .. 31].
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// --------------------------------------------------------------- tiles --
// Work items enumerate (sequence, KV head, token tile, key split); every role
// of a CTA walks the same list: item = blockIdx.x + k * gridDim.x.  When
// there are too few token tiles to fill the GPU, each tile's key blocks are
// cut into `splits` ranges whose partials split_kv_combine merges.
struct Tile {
  int b, h;
  int t0, ntok;      // first query token (within the chunk) and tokens in tile
  int q0, qlen, len; // qo_indptr[b], chunk length, keys of the sequence
  int split;         // key range of the item: blocks kb0 .. kb0 + nblocks - 1
  int kb0;
  int nblocks;
  int keys;          // keys the last row of the tile may see
};

__device__ __forceinline__ bool seq_ok(const PrefillArgs& a, int b, int* q0, int* qlen, int* len) {
  *len = __ldg(a.seq_lens + b);
  *q0 = __ldg(a.qo_indptr + b);
  *qlen = __ldg(a.qo_indptr + b + 1) - *q0;
  return *qlen > 0 && *qlen <= a.max_qlen && *qlen <= *len && *q0 >= 0 &&
         static_cast<int64_t>((*len + 15) >> 4) <= a.pt_stride;
}

// The idx-th tile, or false if there is none.
__device__ bool find_tile(const PrefillArgs& a, int64_t idx, Tile* t) {
  int64_t base = 0;
  for (int b = 0; b < a.batch; ++b) {
    int q0, qlen, len;
    if (!seq_ok(a, b, &q0, &qlen, &len)) continue;
    const int per_head = (qlen + a.tpt - 1) / a.tpt;
    const int64_t per_h = static_cast<int64_t>(per_head) * a.splits;
    const int64_t n = per_h * a.hkv;
    if (idx < base + n) {
      const int64_t r = idx - base;
      t->b = b;
      t->h = static_cast<int>(r / per_h);
      const int64_t rem = r % per_h;
      const int tt = static_cast<int>(rem / a.splits);
      t->split = static_cast<int>(rem % a.splits);
      t->t0 = tt * a.tpt;
      t->ntok = min(a.tpt, qlen - t->t0);
      t->q0 = q0;
      t->qlen = qlen;
      t->len = len;
      t->keys = a.causal ? len - qlen + t->t0 + t->ntok : len;
      const int nb = (t->keys + kBlockKeys - 1) / kBlockKeys;
      t->kb0 = static_cast<int>(static_cast<int64_t>(t->split) * nb / a.splits);
      t->nblocks = static_cast<int>(static_cast<int64_t>(t->split + 1) * nb / a.splits) - t->kb0;
      return true;
    }
    base += n;
  }
  return false;
}

// Parity of the phase in which item g of a ring of n slots lands in its slot.
__device__ __forceinline__ uint32_t ring_parity(int64_t g, int n) { return static_cast<uint32_t>((g / n) & 1); }

__device__ __forceinline__ uint64_t* bar_at(uint8_t* smem, int i) {
  return reinterpret_cast<uint64_t*>(smem + kBarOff) + i;
}
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tile_kernel(const __grid_constant__ CUtensorMap tmap, const PrefillArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + kMiscOff);
  volatile uint32_t* abort_flag = misc + 1;
  uint32_t* raw_valid = misc + 2;  // [kRawStages] bit p: page p of the block loaded
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kRawStages; ++i) {
      mbar_init(bar_at(smem, B_RAW_FULL + i), 1);
      mbar_init(bar_at(smem, B_RAW_EMPTY + i), kDequantWarps);
    }
    for (int i = 0; i < kKStages; ++i) {
      mbar_init(bar_at(smem, B_K_FULL + i), kDequantWarps);
      mbar_init(bar_at(smem, B_K_FREE + i), 1);
    }
    for (int i = 0; i < kVStages; ++i) {
      mbar_init(bar_at(smem, B_V_FULL + i), kDequantWarps);
      mbar_init(bar_at(smem, B_V_FREE + i), 1);
    }
    for (int i = 0; i < kSStages; ++i) {
      mbar_init(bar_at(smem, B_S_FULL + i), 1);
      mbar_init(bar_at(smem, B_S_FREE + i), 4);
    }
    for (int i = 0; i < kPStages; ++i) {
      mbar_init(bar_at(smem, B_P_FULL + i), 4);
      mbar_init(bar_at(smem, B_PV_DONE + i), 1);
    }
    mbar_init(bar_at(smem, B_Q_FULL), 4);
    mbar_init(bar_at(smem, B_FINAL), 2);  // one arrival per MMA-issuing thread
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == kMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(misc)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    tc_fence_before();
  }
  if (warp == kProducerWarp && lane == 0) tma_prefetch_desc(&tmap);
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc[0];
  griddep_wait();
  griddep_launch_dependents();

  auto fail = [&]() {
    flag_error(a.dev_err, PNKV_DEV_ERR_TIMEOUT);
    *abort_flag = 1;
  };
  // single-thread wait (the MMA issuer, producer lane 0); a completed phase
  // returns at once, without reading the abort flag
  auto wait = [&](int bar, uint32_t parity) -> bool {
    if (mbar_try_wait(bar_at(smem, bar), parity)) return true;
    if (*abort_flag) return false;
    if (!mbar_wait(bar_at(smem, bar), parity)) {
      fail();
      return false;
    }
    return true;
  };
  // warp-uniform wait: every lane waits, the warp agrees on the outcome, so
  // an abort never splits a warp before a collective operation
  auto wait_warp = [&](int bar, uint32_t parity) -> bool {
    bool ok = !*abort_flag && mbar_wait(bar_at(smem, bar), parity);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok && lane == 0) fail();
    return ok;
  };

  if (warp == kProducerWarp) {
    // ---------------------------------------------------------- producer
    const uint64_t policy = l2_policy_evict_first();
    int64_t gb = 0;
    bool ok = true;
    Tile t;
    for (int64_t ti = blockIdx.x; ok && find_tile(a, ti, &t); ti += gridDim.x) {
      const int32_t* row = a.page_table + static_cast<int64_t>(t.b) * a.pt_stride;
      const int pages = (t.len + 15) >> 4;
      for (int j = 0; j < t.nblocks && ok; ++j, ++gb) {
        const int rs = static_cast<int>(gb % kRawStages);
        if (lane == 0) ok = wait(B_RAW_EMPTY + rs, ring_parity(gb, kRawStages) ^ 1u);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        // lanes 0 .. kBlockPages - 1: the block's pages
        int32_t page = -1;
        bool in_seq = false;
        if (lane < kBlockPages) {
          const int pi = kBlockPages * (t.kb0 + j) + lane;
          in_seq = pi < pages;
          if (in_seq) {
            page = __ldg(row + pi);
            if (page < 0 || page >= a.num_pages) {
              flag_error(a.dev_err, PNKV_DEV_ERR_PAGE_ID);
              page = -1;
            }
          }
        }
        const unsigned load = __ballot_sync(0xffffffffu, lane < kBlockPages && page >= 0);
        if (lane == 0) {
          raw_valid[rs] = load;
          mbar_arrive_expect_tx(bar_at(smem, B_RAW_FULL + rs), __popc(load) * kRecBytes);
        }
        __syncwarp();
        if (lane < kBlockPages && page >= 0) {
          const int32_t y = (page * a.hkv + t.h) * 36;
          tma_load_2d(smem + kRawOff + rs * kRawStageBytes + lane * kRawPageBytes, &tmap, 0, y,
                      bar_at(smem, B_RAW_FULL + rs), policy);
        }
      }
    }
    if (!ok && lane == 0) {
      // bounded drain of the loads that may still be landing
      const int64_t first = gb > kRawStages ? gb - kRawStages : 0;
      for (int64_t i = first; i < gb; ++i)
        mbar_wait(bar_at(smem, B_RAW_FULL + static_cast<int>(i % kRawStages)), ring_parity(i, kRawStages));
    }
  } else if (warp >= kDequantWarp0 && warp < kDequantWarp0 + kDequantWarps) {
    // ----------------------------------------------------------- dequant
    const int dt = threadIdx.x - kDequantWarp0 * 32;  // 0 .. 32 * kDequantWarps - 1
    int64_t gb = 0;
    bool ok = true;
    Tile t;
    for (int64_t ti = blockIdx.x; ok && find_tile(a, ti, &t); ti += gridDim.x) {
      for (int j = 0; j < t.nblocks && ok; ++j, ++gb) {
        const int rs = static_cast<int>(gb % kRawStages);
        const int ks = static_cast<int>(gb % kKStages), vs = static_cast<int>(gb % kVStages);
        ok = wait_warp(B_RAW_FULL + rs, ring_parity(gb, kRawStages));
        // K slot: free once the QK of block gb - kKStages completed
        if (ok && gb >= kKStages) ok = wait_warp(B_K_FREE + ks, ring_parity(gb - kKStages, kKStages));
        if (!ok) break;
        const uint32_t valid = raw_valid[rs];
        const uint32_t raw = smem_addr(smem + kRawOff + rs * kRawStageBytes);
        uint8_t* ktile = smem + kKOff + ks * kKBytes;
        uint8_t* vtile = smem + kVOff + vs * kVBytes;
        // K: 1,024 units (key, 16-dim block); the lanes of a warp take 32
        // consecutive keys, so each quarter-warp stores one contiguous
        // 128-byte core matrix (8 keys x 8 dims)
        static_assert(kDequantWarps * 32 == 256, "unit mapping assumes 256 dequant threads");
        // all loads first: a load may not pass an earlier shared-memory store
        uint2 kw[4];
        uint32_t ksb[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int key = (dt & 31) + 32 * (i & 1), blk = (dt >> 5) + 8 * (i >> 1);
          const int pg = key >> 4, slot = key & 15;
          kw[i] = make_uint2(0, 0);
          ksb[i] = 0;
          if ((valid >> pg) & 1) {
            const uint32_t rec = raw + pg * kRawPageBytes;
            asm volatile("ld.shared.v2.b32 {%0,%1}, [%2];" : "=r"(kw[i].x), "=r"(kw[i].y) : "r"(rec + swz128(slot, 8 * blk)));
            ksb[i] = lds8(rec + swz128(16 + (slot >> 3), (slot & 7) * 16 + blk));
          }
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int key = (dt & 31) + 32 * (i & 1), blk = (dt >> 5) + 8 * (i >> 1);
          // a missing page has zero codes and a zero scale: fp16 zeros
          uint32_t s2 = e4m3x2_to_f16x2(ksb[i]);
          s2 = prmt(s2, s2, 0x1010u);
          uint32_t c0[4], c1[4];
          e2m1x8_unpack(kw[i].x, c0);
          e2m1x8_unpack(kw[i].y, c1);
          *reinterpret_cast<uint4*>(ktile + core_off(key, 16 * blk, 256)) =
              make_uint4(hmul2(c0[0], s2), hmul2(c0[1], s2), hmul2(c0[2], s2), hmul2(c0[3], s2));
          *reinterpret_cast<uint4*>(ktile + core_off(key, 16 * blk + 8, 256)) =
              make_uint4(hmul2(c1[0], s2), hmul2(c1[1], s2), hmul2(c1[2], s2), hmul2(c1[3], s2));
        }
        fence_proxy_async();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_at(smem, B_K_FULL + ks));
        // V slot: free once the P V of block gb - kVStages completed
        if (gb >= kVStages) ok = wait_warp(B_V_FREE + vs, ring_parity(gb - kVStages, kVStages));
        if (!ok) break;
        // V^T: thread dt owns dim d = dt over the block's 64 keys.  The
        // lanes of a warp read consecutive code bytes of a slot-pair row, and
        // each quarter-warp stores one contiguous core matrix (8 dims x 8
        // keys).  The block scales of the warp's two 16-dim blocks are first
        // transposed through a per-warp scratch ([page][block][slot]), so a
        // thread reads the 16 slot scales of its block with one 16-byte load.
        {
          const int d = dt;
          const int wq = dt >> 5;
          const uint32_t scr = smem_addr(smem + kScrOff + wq * kScrWarpBytes);
          {
            const int slot = lane & 15, bsel = lane >> 4, blk = 2 * wq + bsel;
#pragma unroll
            for (int pg = 0; pg < kBlockPages; ++pg) {
              const uint32_t b = ((valid >> pg) & 1)
                                     ? lds8(raw + pg * kRawPageBytes + swz128(34 + (slot >> 3), (slot & 7) * 16 + blk))
                                     : 0u;
              asm volatile("st.shared.u8 [%0], %1;" ::"r"(scr + pg * 32 + bsel * 16 + slot), "h"(static_cast<uint16_t>(b)));
            }
          }
          __syncwarp();
          const uint32_t code_row = 18 + (d >> 7), code_col = d & 127;
          // all loads first (codes of the four pages, then their scales)
          uint32_t code[kBlockPages][8];
          uint4 sc[kBlockPages];
#pragma unroll
          for (int pg = 0; pg < kBlockPages; ++pg) {
            const uint32_t rec = raw + pg * kRawPageBytes;
#pragma unroll
            for (int pr = 0; pr < 8; ++pr) code[pg][pr] = lds8(rec + swz128(code_row + 2 * pr, code_col));
            sc[pg] = lds128(scr + pg * 32 + ((d >> 4) & 1) * 16);
          }
#pragma unroll
          for (int pg = 0; pg < kBlockPages; ++pg) {
            // a missing page: its scales in the scratch are zero
            uint32_t sf[8];  // fp16x2 scales of slot pairs 0 .. 7
            e4m3x4_to_f16x2x2(sc[pg].x, sf[0], sf[1]);
            e4m3x4_to_f16x2x2(sc[pg].y, sf[2], sf[3]);
            e4m3x4_to_f16x2x2(sc[pg].z, sf[4], sf[5]);
            e4m3x4_to_f16x2x2(sc[pg].w, sf[6], sf[7]);
            uint32_t o[8];
#pragma unroll
            for (int pr = 0; pr < 8; ++pr) o[pr] = hmul2(e2m1x2_to_f16x2(code[pg][pr]), sf[pr]);
            *reinterpret_cast<uint4*>(vtile + core_off(d, 16 * pg, kBlockKeys)) = make_uint4(o[0], o[1], o[2], o[3]);
            *reinterpret_cast<uint4*>(vtile + core_off(d, 16 * pg + 8, kBlockKeys)) = make_uint4(o[4], o[5], o[6], o[7]);
          }
        }
        fence_proxy_async();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(bar_at(smem, B_V_FULL + vs));
          mbar_arrive(bar_at(smem, B_RAW_EMPTY + rs));
        }
      }
    }
  } else if (warp == kMmaWarp || warp == kQkWarp) {
    // --------------------------------------------------------------- MMA
    // Two issuing threads in different warps: a shared-memory access of a
    // thread (an mbarrier wait included) waits until the tensor core has
    // taken the MMAs that thread issued before it, so the QK thread's waits
    // never stall the P V stream and the other way round.
    if (lane == 0) {
      const bool qk_role = warp == kQkWarp;
      const uint32_t idesc = qk_role ? idesc_f16(128, kBlockKeys) : idesc_f16(128, 256);
      int64_t gb = 0;  // first block of the current tile
      int64_t tcount = 0;
      bool ok = true, issued_any = false;
      Tile t;
      for (int64_t ti = blockIdx.x; ok && find_tile(a, ti, &t); ti += gridDim.x, ++tcount) {
        const int64_t g0 = gb;
        if (qk_role) {
          // Q of this tile is in TMEM (written by the softmax warps)
          ok = wait(B_Q_FULL, static_cast<uint32_t>(tcount & 1));
          for (int j = 0; ok && j < t.nblocks; ++j) {
            const int64_t g = g0 + j;
            const int ks = static_cast<int>(g % kKStages), ss = static_cast<int>(g % kSStages);
            ok = wait(B_K_FULL + ks, ring_parity(g, kKStages)) &&
                 (g < kSStages || wait(B_S_FREE + ss, ring_parity(g - kSStages, kSStages)));
            if (!ok) break;
            tc_fence_after();
            const uint32_t k_base = smem_addr(smem + kKOff + ks * kKBytes);
#pragma unroll
            for (int kk = 0; kk < 16; ++kk)  // 16 dims = 8 TMEM columns of Q per k-step
              umma_f16_ta(tmem + kTmemS + ss * kBlockKeys, tmem + kTmemQ + kk * 8,
                          smem_desc(k_base + kk * 256, 128, 4096), idesc, kk > 0);
            umma_commit(bar_at(smem, B_S_FULL + ss));
            umma_commit(bar_at(smem, B_K_FREE + ks));
            issued_any = true;
          }
        } else {
          for (int j = 0; ok && j < t.nblocks; ++j) {
            const int64_t g = g0 + j;
            const int ps = static_cast<int>(g % kPStages), vs = static_cast<int>(g % kVStages);
            ok = wait(B_P_FULL + ps, ring_parity(g, kPStages)) && wait(B_V_FULL + vs, ring_parity(g, kVStages));
            if (!ok) break;
            tc_fence_after();
            const uint32_t p_base = smem_addr(smem + kPOff + ps * kPBytes);
            const uint32_t v_base = smem_addr(smem + kVOff + vs * kVBytes);
#pragma unroll
            for (int kk = 0; kk < kBlockKeys / 16; ++kk)
              umma_f16(tmem + kTmemO, smem_desc(p_base + kk * 256, 128, kBlockKeys * 16),
                       smem_desc(v_base + kk * 256, 128, kBlockKeys * 16), idesc, (j > 0 || kk > 0) ? 1u : 0u);
            umma_commit(bar_at(smem, B_V_FREE + vs));
            umma_commit(bar_at(smem, B_PV_DONE + ps));
            issued_any = true;
          }
        }
        gb = g0 + t.nblocks;
      }
      // every issued MMA completes before TMEM is released
      if (issued_any)
        umma_commit(bar_at(smem, B_FINAL));
      else
        mbar_arrive(bar_at(smem, B_FINAL));
      mbar_wait(bar_at(smem, B_FINAL), 0);
    }
    __syncwarp();
  } else {
    // ----------------------------------------------------------- softmax
    const int r = threadIdx.x;  // row = TMEM lane (warps 0-3)
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    int64_t gb = 0;
    int64_t tcount = 0;
    bool ok = true;
    Tile t;
    for (int64_t ti = blockIdx.x; ok && find_tile(a, ti, &t); ti += gridDim.x, ++tcount) {
      const int tok = t.t0 + r / a.group;
      const int head = r % a.group;
      const bool row_live = r < a.tpt * a.group && r / a.group < t.ntok;
      const int lim = !row_live ? 0 : (a.causal ? t.len - t.qlen + tok + 1 : t.len);
      // Q row -> fp16 into this thread's TMEM lane (the previous tile's MMAs
      // are done: its epilogue waited for the last P V)
      {
        const uint4* src = row_live ? reinterpret_cast<const uint4*>(
                                          a.q + (static_cast<int64_t>(t.q0 + tok) * a.hq + t.h * a.group + head) * 256)
                                    : nullptr;
#pragma unroll 1
        for (int c = 0; c < 8; ++c) {  // 32 dims = 16 columns per store
          uint32_t h[16];
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            uint4 w = make_uint4(0, 0, 0, 0);
            if (row_live) w = __ldg(src + 4 * c + v);
            const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int e = 0; e < 4; ++e)
              h[4 * v + e] = f32x2_to_f16x2(__uint_as_float(ws[e] << 16), __uint_as_float(ws[e] & 0xFFFF0000u));
          }
          tmem_st16(lane_addr + kTmemQ + 16 * c, h);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_at(smem, B_Q_FULL));
      }
      float m_used = -INFINITY, l = 0.f;
      const int64_t g0 = gb;
      for (int j = 0; j < t.nblocks; ++j) {
        const int64_t g = g0 + j;
        const int ss = static_cast<int>(g % kSStages), ps = static_cast<int>(g % kPStages);
        ok = wait_warp(B_S_FULL + ss, ring_parity(g, kSStages));
        if (!ok) break;
        tc_fence_after();
        uint32_t sr[kBlockKeys];
        tmem_ld32(lane_addr + kTmemS + ss * kBlockKeys, sr);
        tmem_ld32(lane_addr + kTmemS + ss * kBlockKeys + 32, sr + 32);
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_at(smem, B_S_FREE + ss));
        // the row maximum of the raw logits over the visible keys (masked
        // keys become -inf); the logit scale is positive, so the maximum of
        // the scaled logits is the scaled maximum
        const int key0 = (t.kb0 + j) * kBlockKeys;
        float mraw = -INFINITY;
        if (__all_sync(0xffffffffu, key0 + kBlockKeys <= lim)) {
#pragma unroll
          for (int k = 0; k < kBlockKeys; ++k) mraw = fmaxf(mraw, __uint_as_float(sr[k]));
        } else {
#pragma unroll
          for (int k = 0; k < kBlockKeys; ++k) {
            if (key0 + k >= lim) sr[k] = __float_as_uint(-INFINITY);
            mraw = fmaxf(mraw, __uint_as_float(sr[k]));
          }
        }
        const float mb = mraw * a.qk_scale_log2;
        // lazy rescale: move the exponent base only when the row max grows
        // by more than the threshold (or for the first finite max)
        float alpha = 1.f;
        const bool move = mb > m_used + kRescaleThreshold || (m_used == -INFINITY && mb > -INFINITY);
        const float base_new = move ? mb : m_used;
        if (move && m_used != -INFINITY) alpha = fast_exp2(m_used - base_new);
        // O holds this row's sum so far only after at least one P V
        const bool need = move && m_used != -INFINITY && j > 0;
        if (__any_sync(0xffffffffu, need)) {
          ok = wait_warp(B_PV_DONE + static_cast<int>((g - 1) % kPStages), ring_parity(g - 1, kPStages));
          if (!ok) break;
          tc_fence_after();
          const float f = need ? alpha : 1.f;
#pragma unroll 1
          for (int c = 0; c < 256; c += 16) {
            uint32_t x[16];
            tmem_ld16(lane_addr + kTmemO + c, x);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 16; ++e) x[e] = __float_as_uint(__uint_as_float(x[e]) * f);
            tmem_st16(lane_addr + kTmemO + c, x);
          }
          tmem_wait_st();
          tc_fence_before();
        }
        l *= alpha;
        m_used = base_new;
        // p = 2^(s * scale - base) (at most 2^threshold), P V takes p in fp16
        // and l sums p in fp32
        const float nbse = (m_used == -INFINITY) ? 0.f : -m_used;
        uint32_t ph[kBlockKeys / 2];
        float add0 = 0.f, add1 = 0.f;
#pragma unroll
        for (int k = 0; k < kBlockKeys / 2; ++k) {
          const float p0 = fast_exp2(fmaf(__uint_as_float(sr[2 * k]), a.qk_scale_log2, nbse));
          const float p1 = fast_exp2(fmaf(__uint_as_float(sr[2 * k + 1]), a.qk_scale_log2, nbse));
          ph[k] = f32x2_to_f16x2(p0, p1);
          add0 += p0;
          add1 += p1;
        }
        l += add0 + add1;
        // P slot ps was last read by the P V of block g - kPStages
        if (g >= kPStages) {
          ok = wait_warp(B_PV_DONE + ps, ring_parity(g - kPStages, kPStages));
          if (!ok) break;
        }
        uint8_t* pt = smem + kPOff + ps * kPBytes;
#pragma unroll
        for (int c = 0; c < kBlockKeys / 8; ++c)
          *reinterpret_cast<uint4*>(pt + core_off(r, 8 * c, kBlockKeys)) =
              make_uint4(ph[4 * c], ph[4 * c + 1], ph[4 * c + 2], ph[4 * c + 3]);
        fence_proxy_async();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_at(smem, B_P_FULL + ps));
      }
      if (!ok) break;
      gb = g0 + t.nblocks;
      // epilogue: final O row, normalised, into the (sequence, KV head,
      // split) slot (an item with no key block writes zeros and LSE -inf)
      if (t.nblocks > 0) {
        const int64_t gl = gb - 1;
        ok = wait_warp(B_PV_DONE + static_cast<int>(gl % kPStages), ring_parity(gl, kPStages));
        if (!ok) break;
        tc_fence_after();
      }
      const int64_t seg = static_cast<int64_t>(t.b) * a.hkv + t.h;
      const int64_t slot = seg * a.splits + t.split;
      const int64_t n = static_cast<int64_t>(tok) * a.group + head;
      const bool have = l > 0.f;
      const float inv = have ? a.out_scale / l : 0.f;
      float* dst = a.o_part + (slot * a.rows_per_slot + n) * 256;
      const bool write = row_live && slot < a.part_slots && n < a.rows_per_slot;
#pragma unroll 1
      for (int c = 0; c < 256; c += 16) {
        uint32_t x[16];
        tmem_ld16(lane_addr + kTmemO + c, x);
        tmem_wait_ld();
        if (write) {
#pragma unroll
          for (int e = 0; e < 16; e += 4)
            *reinterpret_cast<float4*>(dst + c + e) =
                have ? make_float4(__uint_as_float(x[e]) * inv, __uint_as_float(x[e + 1]) * inv,
                                   __uint_as_float(x[e + 2]) * inv, __uint_as_float(x[e + 3]) * inv)
                     : make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
      tc_fence_before();
      if (write) a.lse_part[slot * a.rows_per_slot + n] = have ? (m_used + __log2f(l)) * kLn2 : -INFINITY;
      if (r == 0 && t.t0 == 0 && t.split == 0) {
        a.work_meta[4 + 2 * seg] = static_cast<int32_t>(seg * a.splits);
        a.work_meta[4 + 2 * seg + 1] = a.splits;
      }
    }
  }

  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
  }
}

// Work metadata header and empty segments (sequences without query rows).
__global__ void prefill_meta_kernel(const PrefillArgs a) {
  griddep_wait();
  griddep_launch_dependents();
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    a.work_meta[0] = a.hkv;
    a.work_meta[1] = a.group;
    a.work_meta[2] = a.rows_per_slot;
    a.work_meta[3] = a.batch;
  }
  for (int b = blockIdx.x * blockDim.x + threadIdx.x; b < a.batch; b += gridDim.x * blockDim.x) {
    int q0, qlen, len;
    if (!seq_ok(a, b, &q0, &qlen, &len)) {
      if (__ldg(a.qo_indptr + b + 1) - __ldg(a.qo_indptr + b) != 0)
        flag_error(a.dev_err, PNKV_DEV_ERR_QO_INDPTR);
      for (int h = 0; h < a.hkv; ++h) {
        a.work_meta[4 + 2 * (static_cast<int64_t>(b) * a.hkv + h)] = 0;
        a.work_meta[4 + 2 * (static_cast<int64_t>(b) * a.hkv + h) + 1] = 0;
      }
    }
  }
}

}  // namespace

// Key-range splits per tile, chosen so that the work items fill the SMs'
// last wave: with T tiles and S SMs, s splits make T*s items in ceil(T*s/S)
// waves, a fraction (T*s/S) / ceil(T*s/S) of the GPU busy.  The smallest s
// (at most 8) within 1 % of the best fraction wins.  Host only; T is the
// bound batch * KV heads * ceil(max_qlen / tokens per tile).
int prefill_splits(int32_t batch, int32_t num_kv_heads, int32_t group, int32_t max_qlen, int sms) {
  const int tpt = 128 / group;
  const int64_t tiles = static_cast<int64_t>(batch) * num_kv_heads * ((max_qlen + tpt - 1) / tpt);
  if (tiles <= 0 || sms <= 0) return 1;
  double busy[9] = {0.0};
  double best = 0.0;
  for (int s = 1; s <= 8; ++s) {
    const int64_t items = tiles * s;
    const int64_t waves = (items + sms - 1) / sms;
    busy[s] = static_cast<double>(items) / static_cast<double>(waves * sms);
    best = std::max(best, busy[s]);
  }
  for (int s = 1; s <= 8; ++s)
    if (busy[s] >= best - 0.01) return s;
  return 1;
}

// Launch the tensor-core tile path (called by paged_decode_attention when a KV
// head has more than 64 query rows).
int launch_prefill(const pnkv_cache* cache, const uint16_t* q_roped, const int32_t* qo_indptr,
                   const int32_t* page_table, int64_t pt_stride, const int32_t* seq_lens, int32_t batch,
                   int32_t num_q_heads, int32_t max_qlen, float sm_scale, int32_t causal, float* o_part,
                   float* lse_part, int64_t part_slots, int32_t* work_meta, int32_t* dev_err,
                   cudaStream_t stream) {
  if (cache->dtype != PNKV_KV_NVFP4) return PNKV_ERR_UNSUPPORTED;
  PrefillArgs a;
  a.num_pages = cache->num_pages;
  a.hkv = cache->num_kv_heads;
  a.group = num_q_heads / cache->num_kv_heads;
  a.tpt = 128 / a.group;
  a.qk_scale_log2 = sm_scale * cache->k_scale * kLog2e;
  a.out_scale = cache->v_scale;
  a.q = q_roped;
  a.qo_indptr = qo_indptr;
  a.page_table = page_table;
  a.pt_stride = pt_stride;
  a.seq_lens = seq_lens;
  a.batch = batch;
  a.hq = num_q_heads;
  a.max_qlen = max_qlen;
  a.rows_per_slot = a.group * max_qlen;
  a.causal = causal ? 1 : 0;
  a.o_part = o_part;
  a.lse_part = lse_part;
  a.part_slots = part_slots;
  a.work_meta = work_meta;
  a.dev_err = dev_err;
  CUtensorMap map;
  int st = make_pool_map(cache, 36, &map);
  if (st != PNKV_OK) return st;
  int sms = 0;
  if ((st = device_sm_count(&sms)) != PNKV_OK) return st;
  a.splits = prefill_splits(batch, a.hkv, a.group, max_qlen, sms);
  if (part_slots < static_cast<int64_t>(batch) * a.hkv * a.splits) return PNKV_ERR_INVALID_ARG;
  static bool configured = false;
  if (!configured) {
    if (cudaFuncSetAttribute(prefill_tile_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) !=
        cudaSuccess)
      return PNKV_ERR_CUDA;
    configured = true;
  }
  st = launch_pdl(prefill_meta_kernel, dim3((batch + 255) / 256), dim3(256), 0, stream, a);
  if (st != PNKV_OK) return st;
  return launch_pdl(prefill_tile_kernel, dim3(sms), dim3(kThreads), kSmemBytes, stream, map, a);
}

}  // namespace pnkv
