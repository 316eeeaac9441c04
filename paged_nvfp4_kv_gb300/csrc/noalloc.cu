// paged_decode_attention_noalloc: decode + combine for callers that cannot
// allocate device memory.
//
// The regular path asks the caller for the split-KV partial buffers (o_part,
// lse_part, work_meta).  Some callers cannot provide them: an engine whose
// device memory is reserved up front by its own allocator and which forbids
// libraries from calling cudaMalloc, a latency-critical loop where
// cudaMalloc would synchronise the device, or plain C code without a tensor
// library.  This entry point keeps the partials in a fixed scratch array
// that lives in the library's own device memory (every GPU that loads the
// library holds it until the process exits) and otherwise runs exactly the
// regular decode and combine kernels.
#include <mutex>

#include "host_common.h"

namespace pnkv {
namespace {

// The scratch: work metadata, then LSE partials, then output partials.
static __device__ __align__(256) unsigned char g_scratch[PNKV_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of the scratch on the current device.  In host code the
// array's name is only a host-side stand-in, so the address is looked up once
// per device (with that device current) and then reused; the lock makes the
// first calls of several host threads safe.
int scratch_for_current_device(unsigned char** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PNKV_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p) return PNKV_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = static_cast<unsigned char*>(g_scratch_ptr[dev]);
  return PNKV_OK;
}

inline int64_t round256(int64_t x) { return (x + 255) & ~int64_t(255); }

}  // namespace
}  // namespace pnkv

extern "C" int paged_decode_attention_noalloc(const pnkv_cache* cache, const uint16_t* q_roped,
                                              const int32_t* qo_indptr, const int32_t* page_table,
                                              int64_t pt_stride, const int32_t* seq_lens,
                                              int32_t batch, int32_t num_q_heads, int32_t max_qlen,
                                              float sm_scale, int32_t causal, int64_t total_q,
                                              void* out, int32_t out_is_fp32, float* lse_out,
                                              int32_t* dev_err, void* stream) {
  using namespace pnkv;
  int st = check_cache(cache);
  if (st != PNKV_OK) return st;
  if (batch < 1 || max_qlen < 1 || max_qlen > 8192 || num_q_heads < 1 ||
      num_q_heads % cache->num_kv_heads != 0 || total_q < 0 || !out)
    return PNKV_ERR_INVALID_ARG;
  const int64_t slots = pnkv_decode_slots(cache, batch, num_q_heads, max_qlen);
  if (slots < 0) return static_cast<int>(slots);
  const int64_t meta_ints = pnkv_work_meta_ints(batch, cache->num_kv_heads);
  if (meta_ints < 0) return static_cast<int>(meta_ints);
  const int64_t rows = static_cast<int64_t>(num_q_heads / cache->num_kv_heads) * max_qlen;
  const int64_t meta_bytes = round256(meta_ints * 4);
  const int64_t lse_bytes = round256(slots * rows * 4);
  const int64_t o_bytes = slots * rows * 256 * 4;
  if (meta_bytes + lse_bytes + o_bytes > static_cast<int64_t>(PNKV_NOALLOC_SCRATCH_BYTES))
    return PNKV_ERR_INVALID_ARG;  // the request does not fit the fixed scratch
  unsigned char* base = nullptr;
  if ((st = scratch_for_current_device(&base)) != PNKV_OK) return st;
  int32_t* meta = reinterpret_cast<int32_t*>(base);
  float* lse_part = reinterpret_cast<float*>(base + meta_bytes);
  float* o_part = reinterpret_cast<float*>(base + meta_bytes + lse_bytes);
  st = paged_decode_attention(cache, q_roped, qo_indptr, page_table, pt_stride, seq_lens, batch,
                              total_q, num_q_heads, max_qlen, sm_scale, causal, o_part, lse_part, slots,
                              meta, dev_err, stream);
  if (st != PNKV_OK) return st;
  return split_kv_combine(o_part, lse_part, meta, qo_indptr, batch, total_q, num_q_heads,
                          cache->num_kv_heads, 256, max_qlen, out, out_is_fp32, lse_out, stream);
}
