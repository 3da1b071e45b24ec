// kvq_host.cuh -- host-side argument checks and launch helpers shared by the
// libkvq entry points.  Checks run before anything is enqueued.
#pragma once

#include <cuda_runtime.h>

#include <atomic>
#include <stdint.h>

#include "../../include/kvq.h"

namespace kvq {

inline bool is_pow2_page(int32_t p) { return p == 16 || p == 32 || p == 64 || p == 128 || p == 256; }

inline bool aligned_to(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Validates a cache description for `batch` sequences.
inline bool is_fp4_layout(const kvq_cache* c) {
  return c->format == KVQ_FORMAT_FP4_E2M1_E4M3_G16 || c->format == KVQ_FORMAT_NVFP4;
}

inline kvq_status check_cache(const kvq_cache* c, int32_t batch) {
  if (c == nullptr || c->reserved != 0 || c->num_kv_heads < 1 || c->data == nullptr) return KVQ_ERR_INVALID_ARGUMENT;
  if (!aligned_to(c->data, 16)) return KVQ_ERR_INVALID_ARGUMENT;
  if (c->format == KVQ_FORMAT_FP4_E2M1_E4M3_G16 || c->format == KVQ_FORMAT_NVFP4) {
    if (c->head_dim != 64 && c->head_dim != 128 && c->head_dim != 256) return KVQ_ERR_INVALID_ARGUMENT;
    if (!is_pow2_page(c->page_size) || c->num_pages < 1 || c->max_pages_per_seq < 1)
      return KVQ_ERR_INVALID_ARGUMENT;
    if (c->v_data != nullptr) return KVQ_ERR_INVALID_ARGUMENT;
    if (c->format == KVQ_FORMAT_NVFP4) {  // second-level scales: float [Hkv] each
      if (c->k_scale == nullptr || c->v_scale == nullptr || !aligned_to(c->k_scale, 4) || !aligned_to(c->v_scale, 4))
        return KVQ_ERR_INVALID_ARGUMENT;
    } else if (c->k_scale != nullptr || c->v_scale != nullptr) {
      return KVQ_ERR_INVALID_ARGUMENT;
    }
    if (c->page_table == nullptr && (int64_t)batch * c->max_pages_per_seq > c->num_pages)
      return KVQ_ERR_INVALID_ARGUMENT;
    if (c->num_pages * (int64_t)c->num_kv_heads > (int64_t)INT32_MAX) return KVQ_ERR_UNSUPPORTED;
    return KVQ_OK;
  }
  if (c->format == KVQ_FORMAT_FP8_E4M3_HEAD) {
    if (c->head_dim < 16 || c->head_dim > 512 || (c->head_dim % 16) != 0) return KVQ_ERR_INVALID_ARGUMENT;
    if (c->v_data == nullptr || c->k_scale == nullptr || c->v_scale == nullptr) return KVQ_ERR_INVALID_ARGUMENT;
    if (!aligned_to(c->v_data, 16)) return KVQ_ERR_INVALID_ARGUMENT;
    if (c->page_size < 1 || c->page_size > 1024 || c->page_table != nullptr) return KVQ_ERR_INVALID_ARGUMENT;
    if (c->num_pages < batch) return KVQ_ERR_INVALID_ARGUMENT;
    if (!aligned_to(c->k_scale, 4) || !aligned_to(c->v_scale, 4)) return KVQ_ERR_INVALID_ARGUMENT;
    return KVQ_OK;
  }
  return KVQ_ERR_INVALID_ARGUMENT;
}

constexpr int kMaxDevices = 256;

// SM count of the current device, queried once per device.
inline int device_sm_count() {
  static std::atomic<int> cache[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < kMaxDevices) {
    const int c = cache[dev].load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < kMaxDevices) cache[dev].store(sms, std::memory_order_relaxed);
  return sms;
}

// Per-device once-only flag for one-time host setup (a kernel's attributes).
struct DeviceOnce {
  std::atomic<bool> done[kMaxDevices];
  // true when the setup for the current device still has to run
  bool pending(int dev) const { return dev < 0 || dev >= kMaxDevices || !done[dev].load(std::memory_order_acquire); }
  void mark(int dev) {
    if (dev >= 0 && dev < kMaxDevices) done[dev].store(true, std::memory_order_release);
  }
};

inline unsigned grid_for(int64_t work_items, int threads) {
  int64_t g = (work_items + threads - 1) / threads;
  if (g < 1) g = 1;
  if (g > 0x7FFFFFFF) g = 0x7FFFFFFF;
  return (unsigned)g;
}

inline kvq_status launch_status() {
  return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

// kvq_append's FP4 / NVFP4 launches (kvq_append.cu): n_new tokens per
// sequence from position start_pos[b] + sp_offset; sp_offset -1 reads the
// lengths of a decode step (a zero length appends nothing).
kvq_status launch_fp4_append(const kvq_cache* cache, int32_t batch, int32_t n_new, const int32_t* d_start_pos,
                             int32_t sp_offset, const uint16_t* k16, const uint16_t* v16, int32_t* d_err_flag,
                             cudaStream_t s);

}  // namespace kvq
