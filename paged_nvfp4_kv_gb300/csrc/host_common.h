// Host-side helpers shared by the libpnkv entry points: argument checks,
// launch-error mapping and the per-device SM count.
#pragma once

#include <atomic>
#include <cmath>
#include <cstdint>
#include <utility>
#include <cuda_runtime.h>

#include "pnkv.h"

namespace pnkv {

inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

inline bool aligned(const void* p, uintptr_t a) {
  return (reinterpret_cast<uintptr_t>(p) % a) == 0;
}

// Status of the most recent launch on this thread.
inline int launch_status() {
  return cudaGetLastError() == cudaSuccess ? PNKV_OK : PNKV_ERR_CUDA;
}

// Launch `kernel` with programmatic stream serialisation, so that its
// launch and prologue overlap the tail of the previous kernel in the stream
// (the kernel waits with griddepcontrol.wait before touching global memory).
template <typename... KArgs, typename... Args>
int launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
               Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...) == cudaSuccess ? PNKV_OK
                                                                                       : PNKV_ERR_CUDA;
}

// SM count of the current device (cached per device id).
int device_sm_count(int* out_sms);

// Bound, in nanoseconds, that kernels launched from now on give their
// pipeline waits (pnkv_set_wait_limit_ns).
uint64_t pipeline_wait_ns();

// Raise `kernel`'s dynamic shared-memory limit to `bytes` on the current
// device.  The attribute belongs to the device that is current when it is
// set, so it is set once per device; `done` (one static per kernel) records
// the devices (ids below 64; higher ids set it on every call).  Two threads
// racing on a device's first call both set it, which is harmless.
inline int set_smem_limit_once(std::atomic<uint64_t>& done, const void* kernel, int bytes) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PNKV_ERR_CUDA;
  const uint64_t bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0ull;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return PNKV_OK;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess)
    return PNKV_ERR_CUDA;
  if (bit) done.fetch_or(bit, std::memory_order_acq_rel);
  return PNKV_OK;
}

// The pool as a 2-D byte tensor [num_pages * num_kv_heads * box_rows][128]
// with a box of box_rows x 128 bytes and 128-byte swizzling (one head record
// of a page per box); written to *map (a CUtensorMap).
int make_pool_map(const pnkv_cache* c, int box_rows, void* map);

// Same with records of record_rows rows read in boxes of box_rows rows.
int make_pool_map_box(const pnkv_cache* c, int record_rows, int box_rows, void* map);

// Pool geometry checks shared by every call that touches the pool.
inline int check_cache(const pnkv_cache* c) {
  if (!c || !c->pool || c->num_pages <= 0 || c->page_size != 16 || c->head_dim != 256 ||
      c->num_kv_heads < 1 || c->num_kv_heads > 16)
    return PNKV_ERR_INVALID_ARG;
  if (c->dtype != PNKV_KV_BF16 && c->dtype != PNKV_KV_NVFP4 && c->dtype != PNKV_KV_FP8 &&
      c->dtype != PNKV_KV_INT8)
    return PNKV_ERR_INVALID_ARG;
  if (!aligned(c->pool, 128)) return PNKV_ERR_INVALID_ARG;
  if (c->dtype == PNKV_KV_NVFP4 || c->dtype == PNKV_KV_FP8) {
    if (!(c->k_scale > 0.f) || !(c->v_scale > 0.f) || !std::isfinite(c->k_scale) ||
        !std::isfinite(c->v_scale))
      return PNKV_ERR_INVALID_ARG;
  }
  return PNKV_OK;
}

// Bytes of one KV head's record inside a page (head_dim 256, 16 slots).
inline int64_t head_record_bytes(int dtype) {
  if (dtype == PNKV_KV_NVFP4) return 2 * 16 * (128 + 16);
  if (dtype == PNKV_KV_FP8) return 2 * 16 * 256;
  if (dtype == PNKV_KV_INT8) return 2 * 16 * (256 + 8);
  return 2 * 16 * 256 * 2;
}

}  // namespace pnkv
