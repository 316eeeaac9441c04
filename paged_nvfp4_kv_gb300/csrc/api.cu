// libpnkv: small host-only entry points (status text, version, page sizes)
// and the per-device SM count cache.
#include <mutex>

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

extern "C" int pnkv_version(void) { return 100; }

extern "C" int pnkv_page_bytes(const pnkv_cache* cache, int64_t* out) {
  int st = pnkv::check_cache(cache);
  if (st != PNKV_OK) return st;
  if (!out) return PNKV_ERR_INVALID_ARG;
  *out = pnkv::head_record_bytes(cache->dtype) * cache->num_kv_heads;
  return PNKV_OK;
}
