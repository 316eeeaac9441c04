// Work decomposition shared by the split-KV decode kernels: the launch
// arguments, and the stream-K walk over (sequence b, KV head h, unit) triples,
// a unit being UP consecutive 16-token pages of one head (UP = 1 for the
// register-tile decode, 8 for the tensor-core verify tile).  Units are ordered
// (b, h, unit) and the list is cut into gridDim.x equal contiguous ranges, one
// per CTA; a CTA's range meets a few (b, h) segments, and each maximal run
// inside one segment is a piece with its own partial result.
#pragma once

#include <cstdint>

#include "device_common.cuh"

namespace pnkv {

struct DecodeArgs {
  int64_t num_pages;
  int32_t hkv;
  int32_t group;          // query heads per KV head
  float qk_scale_log2;    // sm_scale * log2(e) (* k_scale for NVFP4 and FP8)
  float out_scale;        // v_scale for NVFP4 and FP8, 1 for INT8 and bf16
  const uint16_t* q;      // roped bf16 queries [total_q, hq, 256]
  const int32_t* qo_indptr;
  const int32_t* page_table;
  int64_t pt_stride;
  const int32_t* seq_lens;
  int32_t batch;
  int64_t total_q;        // rows of q (qo_indptr[batch] must not exceed it)
  int32_t hq;
  int32_t max_qlen;
  int32_t rows_per_slot;  // group * max_qlen
  int32_t causal;
  uint64_t wait_ns;       // bound of a pipeline wait
  float* o_part;
  float* lse_part;
  int64_t part_slots;
  int32_t* work_meta;
  int32_t* dev_err;
};

// ---------------------------------------------------------------------------
// Sequence walk: unit counts per sequence and the segment containing a unit.
// Every thread of a CTA runs the same walk, so all agree on the pieces.

struct SeqInfo {
  int32_t len;    // keys
  int32_t qlen;   // new query rows (tokens)
  int32_t q0;     // qo_indptr[b]
  int32_t pages;  // pages of the sequence
  int32_t units;  // units per (b, h): UP pages each; 0 if the sequence has no valid work
};

// Sequence b with units of UP pages (16 UP keys).
template <int UP>
__device__ __forceinline__ SeqInfo load_seq(const DecodeArgs& a, int b, bool flag) {
  SeqInfo s;
  s.len = __ldg(a.seq_lens + b);
  s.q0 = __ldg(a.qo_indptr + b);
  s.qlen = __ldg(a.qo_indptr + b + 1) - s.q0;
  s.pages = (s.len + 15) >> 4;
  bool ok = true;
  if (s.qlen < 0 || s.qlen > a.max_qlen || s.qlen > s.len || s.q0 < 0 ||
      static_cast<int64_t>(s.q0) + s.qlen > a.total_q) {
    if (flag) flag_error(a.dev_err, PNKV_DEV_ERR_QO_INDPTR);
    ok = false;
  }
  if (s.len < 0 || static_cast<int64_t>(s.pages) > a.pt_stride) {
    if (flag) flag_error(a.dev_err, PNKV_DEV_ERR_SEQ_LEN);
    ok = false;
  }
  s.units = (!ok || s.qlen == 0) ? 0 : (s.pages + UP - 1) / UP;
  return s;
}

// Total units over all sequences (warp-cooperative; every lane gets it).
template <int UP>
__device__ __forceinline__ int64_t total_units(const DecodeArgs& a, int lane) {
  int64_t tot = 0;
  for (int b0 = 0; b0 < a.batch; b0 += 32) {
    const int b = b0 + lane;
    int64_t u = 0;
    if (b < a.batch) u = static_cast<int64_t>(load_seq<UP>(a, b, true).units) * a.hkv;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) u += __shfl_xor_sync(0xffffffffu, u, o);
    tot += u;
  }
  return tot;
}

// Find the sequence b whose unit range [base, base + hkv * units) contains
// `u` (warp-cooperative).  Returns b and its base.
template <int UP>
__device__ __forceinline__ void find_seq(const DecodeArgs& a, int64_t u, int lane, int* b_out,
                                         int64_t* base_out) {
  int64_t base = 0;
  for (int b0 = 0; b0 < a.batch; b0 += 32) {
    const int b = b0 + lane;
    int64_t cnt = 0;
    if (b < a.batch) cnt = static_cast<int64_t>(load_seq<UP>(a, b, false).units) * a.hkv;
    // inclusive scan
    int64_t inc = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t t = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += t;
    }
    const unsigned hit = __ballot_sync(0xffffffffu, b < a.batch && base + inc > u);
    if (hit) {
      const int first = __ffs(hit) - 1;
      const int64_t excl = __shfl_sync(0xffffffffu, inc - cnt, first);
      *b_out = b0 + first;
      *base_out = base + excl;
      return;
    }
    base += __shfl_sync(0xffffffffu, inc, 31);
  }
  *b_out = a.batch;
  *base_out = base;
}

// A maximal run of this CTA's units inside one (b, h) segment.
struct Piece {
  int b, h;
  SeqInfo s;
  int64_t seg_start;  // flattened unit index of the segment's first unit
  int32_t p0;         // first unit (index within the segment)
  int32_t n;          // units in this piece
  int64_t i0;         // CTA-local index of the piece's first unit
};

template <int UP>
struct Walker {
  int b, h;
  SeqInfo s;
  int64_t seg_start;
  int64_t u, u_end, u_begin;
  bool valid;

  __device__ void init(const DecodeArgs& a, int64_t begin, int64_t end, int lane) {
    u_begin = u = begin;
    u_end = end;
    valid = begin < end;
    if (!valid) return;
    int64_t base;
    find_seq<UP>(a, begin, lane, &b, &base);
    s = load_seq<UP>(a, b, false);
    h = static_cast<int>((begin - base) / s.units);
    seg_start = base + static_cast<int64_t>(h) * s.units;
  }

  // Next piece; false when the CTA's range is done.
  __device__ bool next(const DecodeArgs& a, Piece* pc) {
    if (!valid || u >= u_end) return false;
    while (u >= seg_start + s.units) {  // advance to the segment holding u
      seg_start += s.units;
      if (++h == a.hkv) {
        h = 0;
        ++b;
        s = load_seq<UP>(a, b, false);
      }
    }
    pc->b = b;
    pc->h = h;
    pc->s = s;
    pc->seg_start = seg_start;
    pc->p0 = static_cast<int32_t>(u - seg_start);
    const int64_t stop = min(u_end, seg_start + s.units);
    pc->n = static_cast<int32_t>(stop - u);
    pc->i0 = u - u_begin;
    u = stop;
    return true;
  }
};

}  // namespace pnkv
