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
//   MMA warps       S = Q K^T   (M 128, N 64, K 256)  -> TMEM ring, with Q
//                               (fp16) held in TMEM as the A operand, so
//                               shared memory feeds only K
//                   O += P V    (M 128, N 256, K 64)  -> TMEM, with P the A
//                               operand in TMEM
//   softmax warps   one row per thread: tcgen05.ld of S, online softmax,
//                   P (fp16) -> TMEM (tcgen05.st into the S slot it came
//                   from, or with FP4 queries into columns of its own); O is
//                   rescaled in TMEM only when
//                   a row's running maximum grows by more than 2^8, so the
//                   exponentials stay below 256 and most blocks need no
//                   rescale (the row sum adds the fp32 exponentials; P V
//                   takes them rounded to fp16, a relative difference of at
//                   most 2^-11 per term)
// Per-tensor K/V scales fold into the logit scale and the output, as in the
// decode path.  The CTA writes one normalised partial (with its natural-log
// LSE) per row into the (sequence, KV head) slot, which split_kv_combine
// passes through.
//
// FP4-query variant (paged_prefill_attention_fp4q).  The cache's K codes are
// E2M1 with an E4M3 scale per 16 elements ("262,144 Tokens on One RTX 5090",
// section "Why NVFP4 KV changes the math"), which is the operand format of
// the block-scaled FP4 tensor-core product.  With the queries encoded the
// same way (the cache's own encoder, a caller-given per-tensor decode scale
// g_Q), S = Q K^T runs as tcgen05.mma kind::mxf4nvf4 (K 64 per instruction,
// E4M3 scales per 16 elements applied inside the product) straight on the
// codes: each page's 16 rows of K codes are TMA-loaded into a contiguous
// 128-byte-swizzled B tile, the K scales go to TMEM, and nothing of K is
// widened.  The logits are then (q_hat . k_hat) * sm_scale with q_hat the
// queries' NVFP4 round trip; P V is unchanged.
#include <algorithm>
#include <atomic>
#include <cmath>

#include <cudaTypedefs.h>

#include "device_common.cuh"
#include "host_common.h"
#include "tcgen05.cuh"

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
constexpr uint32_t kRecBytes = 4608;  // one NVFP4 head record (36 rows of 128 B)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.f;  // log2 units

// Shared-memory and TMEM plan of each variant (offsets from a 1,024-byte
// aligned base).  Ring depths: the QK of block g waits for its S slot to be
// free -- with NVFP4 queries once the softmax of block g - kSStages has
// loaded it, with bf16 queries (whose P overwrites the slot) once the P V of
// that block has completed -- so QK runs up to kSStages blocks ahead, and the
// softmax of a block overlaps the P V of the one before.
template <bool FP4Q>
struct Plan;

// fp16 QK: the raw ring holds whole head records (one 36-row TMA box per
// page); K is widened into an fp16 ring; Q (fp16) lives in TMEM.
template <>
struct Plan<false> {
  static constexpr int kRawStages = 4, kKStages = 2, kVStages = 2, kSStages = 2, kPStages = 2;
  static constexpr int kRawRows = 36;                    // record rows in a raw page slot
  static constexpr int kRawRow0 = 0;                     // record row of raw row 0
  static constexpr int kRawPageBytes = 5120;             // 4,608-byte record, 1,024-aligned slot
  static constexpr uint32_t kRawTx = kRecBytes;
  static constexpr int kKBytes = kBlockKeys * 256 * 2;   // fp16 [64 keys][256 dims]
  static constexpr int kQBytes = 0, kSfaXBytes = 0;
  static constexpr uint32_t kTmemQ = 384;                // fp16 Q, two per column: 384 .. 511
  static constexpr uint32_t kTmemSfb = 0;
  // P (fp16, two per column) overwrites the first 32 columns of the S slot
  // it was computed from (TMEM has no other room); that slot then waits for
  // the P V of its block, not for the softmax's read, before the next QK
  static constexpr uint32_t kTmemP = 0, kPStrideCols = kBlockKeys;
};

// FP4 QK: K codes go straight from the pool into an FP4 ring (one 16-row TMA
// box per page); the raw ring holds the records' other 20 rows (K scales, V
// codes, V scales); Q codes live in shared memory, the scale factors in TMEM.
template <>
struct Plan<true> {
  static constexpr int kRawStages = 4, kKStages = 3, kVStages = 3, kSStages = 2, kPStages = 2;
  static constexpr int kRawRows = 20;
  static constexpr int kRawRow0 = 16;
  static constexpr int kRawPageBytes = 3072;             // 2,560 bytes, 1,024-aligned slot
  static constexpr uint32_t kRawTx = 20 * 128;
  static constexpr int kKBytes = kBlockKeys * 128;       // E2M1 codes [64 keys][128 B], SW128
  static constexpr int kQBytes = 128 * 128;              // E2M1 codes [128 rows][128 B], SW128
  static constexpr int kSfaXBytes = 128 * 16;            // Q scale bytes [128 rows][16]
  static constexpr uint32_t kTmemQ = 0;
  // scale factors: 16 columns per operand (4 K-chunks x 4 columns), the K
  // ones per K stage
  static constexpr uint32_t kTmemSfa = 384;
  static constexpr uint32_t kTmemSfb = 400;
  // P (fp16, two per column, 32 columns per stage) in its own columns
  static constexpr uint32_t kTmemP = 448, kPStrideCols = 32;
};

template <bool FP4Q>
struct Layout {
  using P = Plan<FP4Q>;
  static constexpr int kRawStageBytes = kBlockPages * P::kRawPageBytes;
  static constexpr int kVBytes = 256 * kBlockKeys * 2;   // fp16 V^T [256 dims][64 keys]
  static constexpr int kKOff = 0;
  static constexpr int kVOff = kKOff + P::kKStages * P::kKBytes;
  static constexpr int kRawOff = kVOff + P::kVStages * kVBytes;  // (P is the A operand of P V in TMEM)
  static constexpr int kQOff = kRawOff + P::kRawStages * kRawStageBytes;  // FP4 Q codes
  static constexpr int kSfaXOff = kQOff + P::kQBytes;
  static constexpr int kScrOff = kSfaXOff + P::kSfaXBytes;  // per dequant warp: V scales
  static constexpr int kScrWarpBytes = kBlockPages * 2 * 8 * 4;  // fp16x2 [page][2 blocks][8 slot pairs]
  static constexpr int kBarOff = kScrOff + kDequantWarps * kScrWarpBytes;
  // barriers, in this order
  static constexpr int B_RAW_FULL = 0;
  static constexpr int B_RAW_EMPTY = B_RAW_FULL + P::kRawStages;
  static constexpr int B_K_FULL = B_RAW_EMPTY + P::kRawStages;
  static constexpr int B_K_FREE = B_K_FULL + P::kKStages;
  static constexpr int B_KC_FULL = B_K_FREE + P::kKStages;  // FP4: K codes landed (TMA bytes)
  static constexpr int B_V_FULL = B_KC_FULL + P::kKStages;
  static constexpr int B_V_FREE = B_V_FULL + P::kVStages;
  static constexpr int B_S_FULL = B_V_FREE + P::kVStages;
  static constexpr int B_S_FREE = B_S_FULL + P::kSStages;
  static constexpr int B_P_FULL = B_S_FREE + P::kSStages;
  static constexpr int B_PV_DONE = B_P_FULL + P::kPStages;
  static constexpr int B_Q_FULL = B_PV_DONE + P::kPStages;
  static constexpr int B_FINAL = B_Q_FULL + 1;
  static constexpr int kNumBars = B_FINAL + 1;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;  // tmem base, abort, raw valid[], softmax ok[]
  static constexpr int kSmemBytes = kMiscOff + 64 + 1024;
  static_assert(kSmemBytes <= 232448, "prefill shared memory plan too large");
  static_assert(kQOff % 1024 == 0 && P::kKBytes % 1024 == 0 && P::kRawPageBytes % 1024 == 0,
                "128-byte-swizzled tiles need 1,024-byte alignment");
  static_assert(P::kRawStages >= 2 && P::kRawStages <= 8, "raw valid words live in misc[2 .. 9], softmax ok in misc[12 .. 15]");
  // TMEM: the S ring at 0 and 64, O at 128 .. 383, then Q (fp16) or the scale factors
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kTmemS = 0;
  static constexpr uint32_t kTmemO = P::kSStages * kBlockKeys;
  static_assert(kTmemO + 256 <= 384, "TMEM plan: S ring and O");
  static_assert(FP4Q ? P::kTmemSfb + 16 * P::kKStages <= P::kTmemP && P::kTmemP + 32 * P::kPStages <= kTmemCols
                     : P::kTmemQ + 128 <= kTmemCols && P::kTmemP == kTmemS && P::kPStages == P::kSStages,
                "TMEM plan too large (or P not aliasing the S ring)");
};

struct PrefillArgs {
  int64_t num_pages;
  int32_t hkv, group, tpt;  // tpt: query tokens per tile (128 / group)
  float qk_scale_log2, out_scale;
  float q_scale, q_enc;     // FP4 queries: decode scale g_Q and fp32(1 / (6 g_Q))
  const uint16_t* q;
  const int32_t* qo_indptr;
  const int32_t* page_table;
  int64_t pt_stride;
  const int32_t* seq_lens;
  int32_t batch, hq, max_qlen, rows_per_slot, causal;
  int64_t total_q;  // rows of q (qo_indptr[batch] must not exceed it)
  int32_t splits;   // key-range splits per tile (slots per (sequence, KV head))
  uint64_t wait_ns; // bound of a pipeline wait
  float* o_part;
  float* lse_part;
  int64_t part_slots;
  int32_t* work_meta;
  int32_t* dev_err;
};

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

// Error bits of a sequence's row range and length (0 when both are valid).
__device__ __forceinline__ int seq_errors(const PrefillArgs& a, int q0, int qlen, int len) {
  int e = 0;
  if (qlen < 0 || qlen > a.max_qlen || qlen > len || q0 < 0 || static_cast<int64_t>(q0) + qlen > a.total_q)
    e |= PNKV_DEV_ERR_QO_INDPTR;
  if (len < 0 || static_cast<int64_t>((len + 15) >> 4) > a.pt_stride) e |= PNKV_DEV_ERR_SEQ_LEN;
  return e;
}

// Sequence b has query rows and valid geometry.
__device__ __forceinline__ bool seq_ok(const PrefillArgs& a, int b, int* q0, int* qlen, int* len) {
  *len = __ldg(a.seq_lens + b);
  *q0 = __ldg(a.qo_indptr + b);
  *qlen = __ldg(a.qo_indptr + b + 1) - *q0;
  return *qlen > 0 && seq_errors(a, *q0, *qlen, *len) == 0;
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

template <bool FP4Q>
__device__ __forceinline__ uint64_t* bar_at(uint8_t* smem, int i) {
  return reinterpret_cast<uint64_t*>(smem + Layout<FP4Q>::kBarOff) + i;
}

// tmap: the pool as 128-byte rows with a box of Plan::kRawRows rows (whole
// records for the fp16 variant, the 20 rows after the K codes for the FP4
// one); tmap_k (FP4 only): the same rows with a box of the 16 K-code rows.
template <bool FP4Q>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tile_kernel(const __grid_constant__ CUtensorMap tmap, const __grid_constant__ CUtensorMap tmap_k,
                        const PrefillArgs a) {
  using P = Plan<FP4Q>;
  using L = Layout<FP4Q>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);
  volatile uint32_t* abort_flag = misc + 1;
  uint32_t* raw_valid = misc + 2;  // [kRawStages] bit p: page p of the block loaded
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  auto bar = [&](int i) { return bar_at<FP4Q>(smem, i); };

  if (threadIdx.x == 0) {
    for (int i = 0; i < P::kRawStages; ++i) {
      mbar_init(bar(L::B_RAW_FULL + i), 1);
      mbar_init(bar(L::B_RAW_EMPTY + i), kDequantWarps);
    }
    for (int i = 0; i < P::kKStages; ++i) {
      // fp16: the dequant warps (K widened); FP4: the four warps that write
      // the K scale factors, with the codes' bytes counted on B_KC_FULL
      mbar_init(bar(L::B_K_FULL + i), FP4Q ? 4 : kDequantWarps);
      mbar_init(bar(L::B_K_FREE + i), 1);
      mbar_init(bar(L::B_KC_FULL + i), 1);
    }
    for (int i = 0; i < P::kVStages; ++i) {
      mbar_init(bar(L::B_V_FULL + i), kDequantWarps);
      mbar_init(bar(L::B_V_FREE + i), 1);
    }
    for (int i = 0; i < P::kSStages; ++i) {
      mbar_init(bar(L::B_S_FULL + i), 1);
      mbar_init(bar(L::B_S_FREE + i), 4);
    }
    for (int i = 0; i < P::kPStages; ++i) {
      mbar_init(bar(L::B_P_FULL + i), 4);
      mbar_init(bar(L::B_PV_DONE + i), 1);
    }
    mbar_init(bar(L::B_Q_FULL), 4);
    mbar_init(bar(L::B_FINAL), 2);  // one arrival per MMA-issuing thread
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == kMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(misc)),
                 "r"(L::kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    tc_fence_before();
  }
  if (warp == kProducerWarp && lane == 0) {
    tma_prefetch_desc(&tmap);
    if (FP4Q) tma_prefetch_desc(&tmap_k);
  }
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
  auto wait = [&](int b, uint32_t parity) -> bool {
    if (mbar_try_wait(bar(b), parity)) return true;
    if (*abort_flag) return false;
    if (!mbar_wait(bar(b), parity, a.wait_ns)) {
      fail();
      return false;
    }
    return true;
  };
  // warp-uniform wait: every lane waits, the warp agrees on the outcome, so
  // an abort never splits a warp before a collective operation
  auto wait_warp = [&](int b, uint32_t parity) -> bool {
    bool ok = !*abort_flag && mbar_wait(bar(b), parity, a.wait_ns);
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
      // page ids eight blocks at a time (lane l: block j0 + l / 4, page
      // l % 4), loaded a group ahead, so that no table read sits between a
      // free slot and its loads
      auto load_ids = [&](int j0) -> int32_t {
        const int jb = j0 + (lane >> 2);
        const int pi = kBlockPages * (t.kb0 + jb) + (lane & 3);
        return (jb < t.nblocks && pi < pages) ? __ldg(row + pi) : -1;
      };
      static_assert(kBlockPages == 4, "the id groups assume four pages per block");
      int32_t ids = load_ids(0), ids_next = load_ids(8);
      for (int j = 0; j < t.nblocks && ok; ++j, ++gb) {
        if (j > 0 && (j & 7) == 0) {
          ids = ids_next;
          ids_next = load_ids(j + 8);
        }
        int32_t page = __shfl_sync(0xffffffffu, ids, ((j & 7) << 2) | (lane & 3));
        const int rs = static_cast<int>(gb % P::kRawStages);
        const int ks = static_cast<int>(gb % P::kKStages);
        if (lane == 0) {
          ok = wait(L::B_RAW_EMPTY + rs, ring_parity(gb, P::kRawStages) ^ 1u);
          // FP4: the K-code slot is free once the QK of block gb - kKStages completed
          if (FP4Q && ok && gb >= P::kKStages) ok = wait(L::B_K_FREE + ks, ring_parity(gb - P::kKStages, P::kKStages));
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        // lanes 0 .. kBlockPages - 1: the block's pages
        if (lane < kBlockPages && kBlockPages * (t.kb0 + j) + lane < pages) {
          if (page < 0 || page >= a.num_pages) {
            flag_error(a.dev_err, PNKV_DEV_ERR_PAGE_ID);
            page = -1;
          }
        } else {
          page = -1;
        }
        const unsigned load = __ballot_sync(0xffffffffu, lane < kBlockPages && page >= 0);
        if (lane == 0) {
          raw_valid[rs] = load;
          mbar_arrive_expect_tx(bar(L::B_RAW_FULL + rs), __popc(load) * P::kRawTx);
          if (FP4Q) mbar_arrive_expect_tx(bar(L::B_KC_FULL + ks), __popc(load) * (16 * 128));
        }
        __syncwarp();
        if (lane < kBlockPages && page >= 0) {
          const int32_t y = (page * a.hkv + t.h) * 36;
          tma_load_2d(smem + L::kRawOff + rs * L::kRawStageBytes + lane * P::kRawPageBytes, &tmap, 0,
                      y + P::kRawRow0, bar(L::B_RAW_FULL + rs), policy);
          if (FP4Q)
            tma_load_2d(smem + L::kKOff + ks * P::kKBytes + lane * (16 * 128), &tmap_k, 0, y,
                        bar(L::B_KC_FULL + ks), policy);
        }
      }
    }
    if (!ok && lane == 0) {
      // drain of the loads that may still be landing (fixed bound: a CTA must
      // not exit with a bulk copy in flight); every block below gb was armed
      const int64_t first = gb > P::kRawStages ? gb - P::kRawStages : 0;
      for (int64_t i = first; i < gb; ++i)
        mbar_wait(bar(L::B_RAW_FULL + static_cast<int>(i % P::kRawStages)), ring_parity(i, P::kRawStages));
      if (FP4Q) {
        const int64_t fk = gb > P::kKStages ? gb - P::kKStages : 0;
        for (int64_t i = fk; i < gb; ++i)
          mbar_wait(bar(L::B_KC_FULL + static_cast<int>(i % P::kKStages)), ring_parity(i, P::kKStages));
      }
    }
  } else if (warp >= kDequantWarp0 && warp < kDequantWarp0 + kDequantWarps) {
    // ----------------------------------------------------------- dequant
    const int dt = threadIdx.x - kDequantWarp0 * 32;  // 0 .. 32 * kDequantWarps - 1
    int64_t gb = 0;
    bool ok = true;
    Tile t;
    for (int64_t ti = blockIdx.x; ok && find_tile(a, ti, &t); ti += gridDim.x) {
      for (int j = 0; j < t.nblocks && ok; ++j, ++gb) {
        const int rs = static_cast<int>(gb % P::kRawStages);
        const int ks = static_cast<int>(gb % P::kKStages), vs = static_cast<int>(gb % P::kVStages);
        ok = wait_warp(L::B_RAW_FULL + rs, ring_parity(gb, P::kRawStages));
        // K slot: free once the QK of block gb - kKStages completed
        if (ok && gb >= P::kKStages && (!FP4Q || warp < kDequantWarp0 + 4))
          ok = wait_warp(L::B_K_FREE + ks, ring_parity(gb - P::kKStages, P::kKStages));
        if (!ok) break;
        const uint32_t valid = raw_valid[rs];
        const uint32_t raw = smem_addr(smem + L::kRawOff + rs * L::kRawStageBytes);
        if constexpr (FP4Q) {
          // the K scales of the block's 64 keys as the B operand's scale
          // factors, one copy per TMEM lane quarter (warps 4-7 hold quarters
          // 0-3); key n = page n / 16, slot n % 16, whose 16 scale bytes are
          // raw row slot / 8 (record row 16 + slot / 8), bytes 16 (slot % 8) ..
          if (warp < kDequantWarp0 + 4) {
            const uint32_t taddr = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16) + P::kTmemSfb + ks * 16;
            // lane l reads the whole 16-byte chunks of keys l and l + 32 (each
            // quarter-warp then reads 128 distinct bytes) and stores them in
            // the layout store_scale_factors describes
            uint4 kc[2];
#pragma unroll
            for (int j = 0; j < 2; ++j) {
              const int n = lane + 32 * j, pg = n >> 4, slot = n & 15;
              kc[j] = lds128(raw + pg * P::kRawPageBytes + swz128(slot >> 3, (slot & 7) * 16));
              if (!((valid >> pg) & 1)) kc[j] = make_uint4(0, 0, 0, 0);  // a missing page scales to zero
            }
            // column 4c + j of this lane = the scale word of row lane + 32 j,
            // K-chunk c (rows 64 .. 127 are not keys of the block: zero)
            const uint32_t cw[2][4] = {{kc[0].x, kc[0].y, kc[0].z, kc[0].w}, {kc[1].x, kc[1].y, kc[1].z, kc[1].w}};
            uint32_t r[16];
#pragma unroll
            for (int c = 0; c < 4; ++c)
#pragma unroll
              for (int j = 0; j < 4; ++j) r[4 * c + j] = j < 2 ? cw[j][c] : 0u;
            tmem_st16(taddr, r);
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(L::B_K_FULL + ks));
          }
        } else {
          uint8_t* ktile = smem + L::kKOff + ks * P::kKBytes;
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
              const uint32_t rec = raw + pg * P::kRawPageBytes;
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
          if (lane == 0) mbar_arrive(bar(L::B_K_FULL + ks));
        }
        // V slot: free once the P V of block gb - kVStages completed
        if (gb >= P::kVStages) ok = wait_warp(L::B_V_FREE + vs, ring_parity(gb - P::kVStages, P::kVStages));
        if (!ok) break;
        uint8_t* vtile = smem + L::kVOff + vs * L::kVBytes;
        // V^T: thread dt owns dim d = dt over the block's 64 keys.  The
        // lanes of a warp read consecutive code bytes of a slot-pair row, and
        // each quarter-warp stores one contiguous core matrix (8 dims x 8
        // keys).  The block scales of the warp's two 16-dim blocks (each
        // shared by 16 of its lanes) are first converted into a per-warp
        // scratch of fp16 pairs [page][block][slot pair], so a thread reads
        // the 8 pair scales of its block with two 16-byte loads.  Slots past
        // the sequence and pages that were not loaded scale to 0, which
        // zeroes their values whatever the stale codes.  (Raw rows are record
        // rows minus kRawRow0: V codes at record rows 18 .. 33, V scales at
        // 34 and 35, slot s's 16 block scales at byte 16 (s % 8) of row
        // 34 + s / 8.)
        {
          const int d = dt;
          const int wq = dt >> 5;
          const uint32_t scr = smem_addr(smem + L::kScrOff + wq * L::kScrWarpBytes);
          {
            const int bsel = (lane >> 3) & 1, fp = lane & 7, blk = 2 * wq + bsel;
            const uint32_t o0 = swz128(34 - P::kRawRow0 + (fp >> 2), ((2 * fp) & 7) * 16 + blk);
            const uint32_t o1 = swz128(34 - P::kRawRow0 + (fp >> 2), ((2 * fp + 1) & 7) * 16 + blk);
            const int keys_left = t.len - (t.kb0 + j) * kBlockKeys;  // keys of the block in the sequence
            uint32_t* fdst = reinterpret_cast<uint32_t*>(smem + L::kScrOff + wq * L::kScrWarpBytes) + lane;
#pragma unroll
            for (int i = 0; i < kBlockPages / 2; ++i) {
              const int pg = 2 * i + (lane >> 4);  // word lane + 32 i = (pg, bsel, fp)
              const uint32_t b0 = lds8(raw + pg * P::kRawPageBytes + o0);
              const uint32_t b1 = lds8(raw + pg * P::kRawPageBytes + o1);
              const int s0 = 16 * pg + 2 * fp;
              const bool pv = (valid >> pg) & 1;
              const uint32_t m = (pv && s0 < keys_left ? 0x0000FFFFu : 0u) | (pv && s0 + 1 < keys_left ? 0xFFFF0000u : 0u);
              fdst[32 * i] = e4m3x2_to_f16x2(b0 | (b1 << 8)) & m;
            }
          }
          __syncwarp();
          // all loads first (codes of the four pages, then their scales); the
          // code rows 18 - kRawRow0 + d / 128 + 2 pr have residues mod 8 that
          // repeat every 4 pairs, so 4 swizzled column offsets make each byte
          // load one instruction
          const uint32_t code_row = 18 - P::kRawRow0 + (d >> 7), code_col = d & 127;
          uint32_t cbase[4];
#pragma unroll
          for (int m = 0; m < 4; ++m) cbase[m] = raw + swz128(code_row + 2 * m, code_col);
          uint32_t code[kBlockPages][8];
          uint4 sc[kBlockPages][2];
#pragma unroll
          for (int pg = 0; pg < kBlockPages; ++pg) {
#pragma unroll
            for (int pr = 0; pr < 8; ++pr)
              code[pg][pr] = lds8(cbase[pr & 3] + pg * P::kRawPageBytes + (pr >> 2) * 8 * 128);
            sc[pg][0] = lds128(scr + (2 * pg + ((d >> 4) & 1)) * 32);
            sc[pg][1] = lds128(scr + (2 * pg + ((d >> 4) & 1)) * 32 + 16);
          }
#pragma unroll
          for (int pg = 0; pg < kBlockPages; ++pg) {
            // fp16x2 scales of slot pairs 0 .. 7
            const uint32_t sf[8] = {sc[pg][0].x, sc[pg][0].y, sc[pg][0].z, sc[pg][0].w,
                                    sc[pg][1].x, sc[pg][1].y, sc[pg][1].z, sc[pg][1].w};
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
          mbar_arrive(bar(L::B_V_FULL + vs));
          mbar_arrive(bar(L::B_RAW_EMPTY + rs));
        }
      }
    }
  } else if (warp == kMmaWarp || warp == kQkWarp) {
    // --------------------------------------------------------------- MMA
    // QK and P V from different warps: a shared-memory access of a thread
    // (an mbarrier wait included) waits until the tensor core has taken the
    // MMAs that thread issued before it, so the QK warp's waits never stall
    // the P V stream and the other way round.  The whole warp runs the loop
    // and waits, one elected thread issues (the operands stay in uniform
    // registers), and the shared-memory descriptors advance by their encoded
    // address field (16-byte units).
    const bool qk_role = warp == kQkWarp;
    const uint32_t idesc = qk_role ? (FP4Q ? idesc_mxf4nvf4(128, kBlockKeys) : idesc_f16(128, kBlockKeys))
                                   : idesc_f16(128, 256);
    const uint64_t kdesc0 =
        FP4Q ? smem_desc_sw128(smem_addr(smem + L::kKOff)) : smem_desc(smem_addr(smem + L::kKOff), 128, 4096);
    const uint64_t qdesc0 = FP4Q ? smem_desc_sw128(smem_addr(smem + L::kQOff)) : 0;
    const uint64_t vdesc0 = smem_desc(smem_addr(smem + L::kVOff), 128, kBlockKeys * 16);
    int64_t gb = 0;  // first block of the current tile
    int64_t tcount = 0;
    bool ok = true, issued_any = false;
    Tile t;
    for (int64_t ti = blockIdx.x; ok && find_tile(a, ti, &t); ti += gridDim.x, ++tcount) {
      const int64_t g0 = gb;
      if (qk_role) {
        // Q of this tile is ready (fp16 in TMEM, or FP4 codes in shared
        // memory with their scale factors in TMEM), written by the softmax warps
        ok = wait_warp(L::B_Q_FULL, static_cast<uint32_t>(tcount & 1));
        for (int j = 0; ok && j < t.nblocks; ++j) {
          const int64_t g = g0 + j;
          const int ks = static_cast<int>(g % P::kKStages), ss = static_cast<int>(g % P::kSStages);
          ok = wait_warp(L::B_K_FULL + ks, ring_parity(g, P::kKStages)) &&
               (!FP4Q || wait_warp(L::B_KC_FULL + ks, ring_parity(g, P::kKStages))) &&
               (g < P::kSStages ||
                (FP4Q ? wait_warp(L::B_S_FREE + ss, ring_parity(g - P::kSStages, P::kSStages))
                      // P of block g - 2 sits in this S slot: wait for its P V
                      : wait_warp(L::B_PV_DONE + ss, ring_parity(g - P::kSStages, P::kPStages))));
          if (!ok) break;
          tc_fence_after();
          const uint64_t kdesc = kdesc0 + static_cast<uint64_t>(ks * (P::kKBytes >> 4));
          const uint32_t d = tmem + L::kTmemS + ss * kBlockKeys;
          if (elect_one()) {
            if constexpr (FP4Q) {
#pragma unroll
              for (int c = 0; c < 4; ++c)  // 64 FP4 elements = 32 bytes of every row per K-chunk
                umma_fp4(d, qdesc0 + 2 * c, kdesc + 2 * c, idesc, tmem + P::kTmemSfa + 4 * c,
                         tmem + P::kTmemSfb + ks * 16 + 4 * c, c > 0);
            } else {
#pragma unroll
              for (int kk = 0; kk < 16; ++kk)  // 16 dims = 8 TMEM columns of Q, 2 core matrices (256 B) of K
                umma_f16_ta(d, tmem + P::kTmemQ + kk * 8, kdesc + 16 * kk, idesc, kk > 0);
            }
            umma_commit(bar(L::B_S_FULL + ss));
            umma_commit(bar(L::B_K_FREE + ks));
          }
          __syncwarp();
          issued_any = true;
        }
      } else {
        for (int j = 0; ok && j < t.nblocks; ++j) {
          const int64_t g = g0 + j;
          const int ps = static_cast<int>(g % P::kPStages), vs = static_cast<int>(g % P::kVStages);
          ok = wait_warp(L::B_P_FULL + ps, ring_parity(g, P::kPStages)) &&
               wait_warp(L::B_V_FULL + vs, ring_parity(g, P::kVStages));
          if (!ok) break;
          tc_fence_after();
          const uint64_t vdesc = vdesc0 + static_cast<uint64_t>(vs * (L::kVBytes >> 4));
          const uint32_t acc = j > 0 ? 1u : 0u;
          if (elect_one()) {
#pragma unroll
            for (int kk = 0; kk < kBlockKeys / 16; ++kk) {  // 16 keys = 2 core matrices (256 B) of P and of V^T
              // P from TMEM: 8 columns per 16 keys
              umma_f16_ta(tmem + L::kTmemO, tmem + P::kTmemP + P::kPStrideCols * ps + 8 * kk, vdesc + 16 * kk,
                          idesc, kk > 0 ? 1u : acc);
            }
            umma_commit(bar(L::B_V_FREE + vs));
            umma_commit(bar(L::B_PV_DONE + ps));
          }
          __syncwarp();
          issued_any = true;
        }
      }
      gb = g0 + t.nblocks;
    }
    // every issued MMA completes before TMEM is released (fixed bound)
    if (elect_one()) {
      if (issued_any)
        umma_commit(bar(L::B_FINAL));
      else
        mbar_arrive(bar(L::B_FINAL));
    }
    __syncwarp();
    mbar_wait(bar(L::B_FINAL), 0);
  } else {
    // ----------------------------------------------------------- softmax
    const int r = threadIdx.x;  // row = TMEM lane (warps 0-3)
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    int64_t gb = 0;
    int64_t tcount = 0;
    bool ok = true;
    Tile t;
    volatile uint32_t* sm_ok = misc + 12;  // [4] each softmax warp's state at a tile start
    for (int64_t ti = blockIdx.x; find_tile(a, ti, &t); ti += gridDim.x, ++tcount) {
      const int tok = t.t0 + r / a.group;
      const int head = r % a.group;
      const bool row_live = r < a.tpt * a.group && r / a.group < t.ntok;
      const int lim = !row_live ? 0 : (a.causal ? t.len - t.qlen + tok + 1 : t.len);
      // the four softmax warps enter a tile together, so each arrives on
      // B_Q_FULL once per tile even when tiles without key blocks follow
      // each other (and the FP4 scale exchange below is not overwritten
      // while another warp still reads it).  They also stop together: a
      // warp whose wait gave up comes on to this barrier rather than leaving
      // the loop, and all four leave here if any of them failed.
      if (lane == 0) sm_ok[warp] = ok ? 1u : 0u;
      named_bar_sync(1, 128);
      if (!(sm_ok[0] & sm_ok[1] & sm_ok[2] & sm_ok[3])) break;
      // Q row into its operand (the previous tile's MMAs are done: its
      // epilogue waited for the last P V, and every QK before that was read)
      {
        const uint4* src = row_live ? reinterpret_cast<const uint4*>(
                                          a.q + (static_cast<int64_t>(t.q0 + tok) * a.hq + t.h * a.group + head) * 256)
                                    : nullptr;
        if constexpr (FP4Q) {
          // NVFP4 codes of the row (the cache's encoder, decode scale g_Q)
          // into row r of the 128-byte-swizzled A tile; the 16 scale bytes
          // through shared memory into the A scale factors in TMEM
          uint8_t* qt = smem + L::kQOff + r * 128;
          uint32_t* sfx = reinterpret_cast<uint32_t*>(smem + L::kSfaXOff);  // [128 rows][4 words]
#pragma unroll 1
          for (int ch = 0; ch < 8; ++ch) {  // 16-byte chunk ch: blocks 2ch, 2ch + 1
            uint32_t cw[4];
#pragma unroll
            for (int hb = 0; hb < 2; ++hb) {
              const int blk = 2 * ch + hb;
              float x[16];
#pragma unroll
              for (int v = 0; v < 2; ++v) {
                uint4 w = make_uint4(0, 0, 0, 0);
                if (row_live) w = __ldg(src + 2 * blk + v);
                const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  x[8 * v + 2 * e] = __uint_as_float(ws[e] << 16);
                  x[8 * v + 2 * e + 1] = __uint_as_float(ws[e] & 0xFFFF0000u);
                }
              }
              float amax = 0.f;
#pragma unroll
              for (int e = 0; e < 16; ++e) amax = fmaxf(amax, fabsf(x[e]));
              float rcp;
              const uint32_t sb = nvfp4_block_scale(amax, a.q_scale, a.q_enc, &rcp);
              uint32_t lo = 0u, hi = 0u;
              if (sb != 0u) {
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                  lo |= e2m1_code(__fmul_rn(x[e], rcp)) << (4 * e);
                  hi |= e2m1_code(__fmul_rn(x[8 + e], rcp)) << (4 * e);
                }
              }
              cw[2 * hb] = lo;
              cw[2 * hb + 1] = hi;
              // scale byte of block blk: byte blk % 4 of word blk / 4
              reinterpret_cast<uint8_t*>(sfx + 4 * r)[blk] = static_cast<uint8_t>(sb);
            }
            *reinterpret_cast<uint4*>(qt + ((ch ^ (r & 7)) << 4)) = make_uint4(cw[0], cw[1], cw[2], cw[3]);
          }
          named_bar_sync(1, 128);
          store_scale_factors(lane_addr + P::kTmemSfa, lane,
                              [&](int n, int c) -> uint32_t { return sfx[4 * n + c]; });
          fence_proxy_async();  // the A tile's generic stores, before the MMA reads them
        } else {
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
            tmem_st16(lane_addr + P::kTmemQ + 16 * c, h);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(L::B_Q_FULL));
      }
      float m_used = -INFINITY, l = 0.f;
      const int64_t g0 = gb;
      for (int j = 0; j < t.nblocks; ++j) {
        const int64_t g = g0 + j;
        const int ss = static_cast<int>(g % P::kSStages), ps = static_cast<int>(g % P::kPStages);
        ok = wait_warp(L::B_S_FULL + ss, ring_parity(g, P::kSStages));
        if (!ok) break;
        tc_fence_after();
        uint32_t sr[kBlockKeys];
        tmem_ld32(lane_addr + L::kTmemS + ss * kBlockKeys, sr);
        tmem_ld32(lane_addr + L::kTmemS + ss * kBlockKeys + 32, sr + 32);
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (FP4Q && lane == 0) mbar_arrive(bar(L::B_S_FREE + ss));
        // the row maximum of the raw logits over the visible keys (masked
        // keys become -inf); the logit scale is positive, so the maximum of
        // the scaled logits is the scaled maximum
        const int key0 = (t.kb0 + j) * kBlockKeys;
        if (!__all_sync(0xffffffffu, key0 + kBlockKeys <= lim)) {
#pragma unroll
          for (int k = 0; k < kBlockKeys; ++k)
            if (key0 + k >= lim) sr[k] = __float_as_uint(-INFINITY);
        }
        float mraw;
        {
          // two chains of three-input maxima over keys 0 .. 61, then 62, 63
          float m0 = __uint_as_float(sr[0]), m1 = __uint_as_float(sr[1]);
#pragma unroll
          for (int k = 2; k + 3 < kBlockKeys; k += 4) {
            m0 = fmax3(m0, __uint_as_float(sr[k]), __uint_as_float(sr[k + 1]));
            m1 = fmax3(m1, __uint_as_float(sr[k + 2]), __uint_as_float(sr[k + 3]));
          }
          mraw = fmax3(fmaxf(m0, m1), __uint_as_float(sr[kBlockKeys - 2]), __uint_as_float(sr[kBlockKeys - 1]));
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
          ok = wait_warp(L::B_PV_DONE + static_cast<int>((g - 1) % P::kPStages), ring_parity(g - 1, P::kPStages));
          if (!ok) break;
          tc_fence_after();
          const float f = need ? alpha : 1.f;
#pragma unroll 1
          for (int c = 0; c < 256; c += 16) {
            uint32_t x[16];
            tmem_ld16(lane_addr + L::kTmemO + c, x);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 16; ++e) x[e] = __float_as_uint(__uint_as_float(x[e]) * f);
            tmem_st16(lane_addr + L::kTmemO + c, x);
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
        if (g >= P::kPStages) {
          ok = wait_warp(L::B_PV_DONE + ps, ring_parity(g - P::kPStages, P::kPStages));
          if (!ok) break;
        }
        {
          // the row's 64 fp16 probabilities into its TMEM lane
          uint32_t h0[16], h1[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            h0[i] = ph[i];
            h1[i] = ph[16 + i];
          }
          tmem_st16(lane_addr + P::kTmemP + P::kPStrideCols * ps, h0);
          tmem_st16(lane_addr + P::kTmemP + P::kPStrideCols * ps + 16, h1);
          tmem_wait_st();
          tc_fence_before();
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(L::B_P_FULL + ps));
      }
      if (!ok) continue;  // on to the next tile start, where all four warps stop
      gb = g0 + t.nblocks;
      // epilogue: final O row, normalised, into the (sequence, KV head,
      // split) slot (an item with no key block writes zeros and LSE -inf)
      if (t.nblocks > 0) {
        const int64_t gl = gb - 1;
        ok = wait_warp(L::B_PV_DONE + static_cast<int>(gl % P::kPStages), ring_parity(gl, P::kPStages));
        if (!ok) continue;
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
        tmem_ld16(lane_addr + L::kTmemO + c, x);
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
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(L::kTmemCols) : "memory");
  }
}

// Work metadata header and empty segments (sequences without query rows, or
// flagged ones).
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
      const int e = seq_errors(a, q0, qlen, len);
      if (e) flag_error(a.dev_err, e);
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

// Launch the tensor-core tile path: called by paged_decode_attention when a KV
// head has more than 64 query rows (q_scale = 0: fp16 queries), and by
// paged_prefill_attention_fp4q (q_scale = g_Q > 0: NVFP4 queries, block-scaled
// FP4 QK^T).
int launch_prefill(const pnkv_cache* cache, const uint16_t* q_roped, const int32_t* qo_indptr,
                   const int32_t* page_table, int64_t pt_stride, const int32_t* seq_lens, int32_t batch,
                   int64_t total_q, int32_t num_q_heads, int32_t max_qlen, float sm_scale, int32_t causal,
                   float q_scale, float* o_part, float* lse_part, int64_t part_slots, int32_t* work_meta,
                   int32_t* dev_err, cudaStream_t stream) {
  if (cache->dtype != PNKV_KV_NVFP4) return PNKV_ERR_UNSUPPORTED;
  const bool fp4q = q_scale > 0.f;
  PrefillArgs a;
  a.num_pages = cache->num_pages;
  a.hkv = cache->num_kv_heads;
  a.group = num_q_heads / cache->num_kv_heads;
  a.tpt = 128 / a.group;
  // logit = (q . k) * sm_scale; the products run on codes times block scales,
  // so the per-tensor decode scales of K (and of Q for FP4 queries) multiply here
  a.qk_scale_log2 = sm_scale * cache->k_scale * (fp4q ? q_scale : 1.f) * kLog2e;
  a.out_scale = cache->v_scale;
  a.q_scale = fp4q ? q_scale : 0.f;
  a.q_enc = fp4q ? static_cast<float>(1.0 / (6.0 * static_cast<double>(q_scale))) : 0.f;
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
  a.total_q = total_q;
  a.wait_ns = pipeline_wait_ns();
  a.o_part = o_part;
  a.lse_part = lse_part;
  a.part_slots = part_slots;
  a.work_meta = work_meta;
  a.dev_err = dev_err;
  // the pool as 128-byte rows, 36 per head record: whole-record boxes for the
  // fp16 tile; for the FP4 tile a box of the 20 rows after the K codes and a
  // box of the 16 K-code rows
  CUtensorMap map, map_k;
  int st = make_pool_map_box(cache, 36, fp4q ? Plan<true>::kRawRows : Plan<false>::kRawRows, &map);
  if (st != PNKV_OK) return st;
  if (fp4q) {
    if ((st = make_pool_map_box(cache, 36, 16, &map_k)) != PNKV_OK) return st;
  } else {
    map_k = map;
  }
  int sms = 0;
  if ((st = device_sm_count(&sms)) != PNKV_OK) return st;
  a.splits = prefill_splits(batch, a.hkv, a.group, max_qlen, sms);
  if (part_slots < static_cast<int64_t>(batch) * a.hkv * a.splits) return PNKV_ERR_INVALID_ARG;
  static std::atomic<uint64_t> configured_f16{0}, configured_fp4{0};  // devices whose attribute is set
  const void* kern = fp4q ? reinterpret_cast<const void*>(prefill_tile_kernel<true>)
                          : reinterpret_cast<const void*>(prefill_tile_kernel<false>);
  const int smem = fp4q ? Layout<true>::kSmemBytes : Layout<false>::kSmemBytes;
  if ((st = set_smem_limit_once(fp4q ? configured_fp4 : configured_f16, kern, smem)) != PNKV_OK) return st;
  st = launch_pdl(prefill_meta_kernel, dim3((batch + 255) / 256), dim3(256), 0, stream, a);
  if (st != PNKV_OK) return st;
  if (fp4q) return launch_pdl(prefill_tile_kernel<true>, dim3(sms), dim3(kThreads), smem, stream, map, map_k, a);
  return launch_pdl(prefill_tile_kernel<false>, dim3(sms), dim3(kThreads), smem, stream, map, map_k, a);
}

}  // namespace pnkv
