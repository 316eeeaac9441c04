// libpnkv: small host-only entry points (status text, version, page sizes)
// and the per-device SM count cache.
#include <atomic>
#include <mutex>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "host_common.h"

namespace pnkv {

int device_sm_count(int* out_sms) {
  static std::mutex mu;
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PNKV_ERR_CUDA;
  if (dev >= 0 && dev < 64) {
    std::lock_guard<std::mutex> lock(mu);
    if (cached[dev] == 0) {
      int sms = 0;
      if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return PNKV_ERR_CUDA;
      cached[dev] = sms;
    }
    *out_sms = cached[dev];
    return PNKV_OK;
  }
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return PNKV_ERR_CUDA;
  *out_sms = sms;
  return PNKV_OK;
}


namespace {
std::atomic<uint64_t> g_wait_ns{2000000000ull};
}

uint64_t pipeline_wait_ns() { return g_wait_ns.load(std::memory_order_relaxed); }

// The driver's tensor-map encoder, looked up once (thread-safe static).
PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = []() -> PFN_cuTensorMapEncodeTiled_v12000 {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    return nullptr;
  }();
  return fn;
}

// The pool seen as a 2-D byte tensor [num_pages * hkv * record_rows][128]
// read in boxes of box_rows rows.
int make_pool_map_box(const pnkv_cache* c, int record_rows, int box_rows, void* map_out) {
  CUtensorMap* map = static_cast<CUtensorMap*>(map_out);
  if (box_rows < 1 || box_rows > record_rows || box_rows > 256) return PNKV_ERR_INVALID_ARG;
  const cuuint64_t rows = static_cast<cuuint64_t>(c->num_pages) * c->num_kv_heads * record_rows;
  if (rows >= (1ull << 31)) return PNKV_ERR_INVALID_ARG;  // TMA row coordinates are int32
  PFN_cuTensorMapEncodeTiled_v12000 enc = get_encode_fn();
  if (!enc) return PNKV_ERR_CUDA;
  const cuuint64_t dims[2] = {128, rows};
  const cuuint64_t strides[1] = {128};
  const cuuint32_t box[2] = {128, static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, c->pool, dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PNKV_OK : PNKV_ERR_CUDA;
}

int make_pool_map(const pnkv_cache* c, int box_rows, void* map_out) {
  return make_pool_map_box(c, box_rows, box_rows, map_out);
}

}  // namespace pnkv

extern "C" const char* pnkv_status_string(int status) {
  switch (status) {
    case PNKV_OK: return "ok";
    case PNKV_ERR_INVALID_ARG: return "invalid argument";
    case PNKV_ERR_UNSUPPORTED: return "unsupported";
    case PNKV_ERR_CUDA: return "CUDA error";
    default: return "unknown status";
  }
}

extern "C" int pnkv_version(void) { return 200; }

extern "C" int64_t pnkv_set_wait_limit_ns(int64_t ns) {
  if (ns < 1000 || ns > 60000000000LL) return PNKV_ERR_INVALID_ARG;
  return static_cast<int64_t>(pnkv::g_wait_ns.exchange(static_cast<uint64_t>(ns)));
}

extern "C" int pnkv_page_bytes(const pnkv_cache* cache, int64_t* out) {
  int st = pnkv::check_cache(cache);
  if (st != PNKV_OK) return st;
  if (!out) return PNKV_ERR_INVALID_ARG;
  *out = pnkv::head_record_bytes(cache->dtype) * cache->num_kv_heads;
  return PNKV_OK;
}
