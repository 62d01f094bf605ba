// Host-side pool state shared by the translation units of the library (not part of the ABI).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>
#include <vector>

#include "lazy_attn.h"

struct lazy_pool {
  void *k = nullptr;
  void *v = nullptr;
  int32_t num_blocks = 0, page_size = 0, hkv = 0, d = 0, dtype = 0;
  double base = 0.0;

  std::mutex mu;                    // guards the allocator and lazy device set-up
  std::vector<int32_t> free_list;   // stack of free block ids (top = back)
  std::vector<int32_t> refcount;    // per block
  std::vector<uint64_t> turn;       // frac(theta_i / 2pi) * 2^64, i < d/2

  bool dev_ready = false;
  int device = -1;
  int num_sms = 0;
  int32_t *d_err = nullptr;         // device error word
  uint64_t *d_turn = nullptr;       // device copy of `turn`
  uint64_t wait_limit_ns = 2000000000ull;

  // ALiBi mode (lazy_pool_set_alibi): K is stored unrotated and attention adds
  // slope[head] * (n - m); page-word offsets are page start positions.
  int32_t decode_kernel = 0;        // LAZY_DECODE_* (lazy_pool_set_decode_kernel)
  int32_t schedule_sms = 0;         // SMs the prefill schedule assumes; 0 = num_sms
  bool alibi = false;
  bool encoded = false;             // something was written: the mode can no longer change
  std::vector<float> slopes;        // per query head
  float *d_slopes = nullptr;

  // Pinned host staging of kv_pool_materialise_batch's page list (grown on demand, guarded by
  // mu); stage_done marks the end of the last upload from it, which the next call waits for
  // before refilling it.
  void *h_stage = nullptr;
  size_t h_stage_bytes = 0;
  cudaEvent_t stage_done = nullptr;

  // Tensor maps of the page buffers for the tensor-core prefill (built lazily).
  bool tmaps_ready = false;
  alignas(64) unsigned char tmap_k[128];   // 2-D view: 16-row page boxes
  alignas(64) unsigned char tmap_v[128];
  alignas(64) unsigned char tmap_k8[128];  // 4-D view: 8 consecutive blocks of one kv head
  alignas(64) unsigned char tmap_v8[128];
  alignas(64) unsigned char tmap_k3[128];  // 3-D view: one whole page per box
  alignas(64) unsigned char tmap_v3[128];
};

namespace lazy {
int record_cuda(cudaError_t e, const char *what);
void record_msg(const char *msg);
int ensure_device(lazy_pool *p);
// TMA tensor maps of the page buffers (bf16, head_dim 128, 128-byte swizzle), built once:
//   tmap_k / tmap_v    2-D, rows (block * Hkv + h) * 16 + slot, box 16 rows x 64 dims
//   tmap_k8 / tmap_v8  4-D [block][kv head][slot][dim], box 8 blocks x 1 head x 16 x 64
//   tmap_k3 / tmap_v3  3-D (64 dims, rows, 2 halves of 128 B), box 64 x 16 x 2: one page in one
//                      copy, landing as the two 16 x 64 boxes of the 2-D view, half-major
// LAZY_ERR_UNSUPPORTED for other pools.
int ensure_pool_tmaps(lazy_pool *p);
inline size_t elem_bytes(int32_t dtype) { return dtype == LAZY_DTYPE_BF16 ? 2 : 4; }
inline size_t pool_bytes(const lazy_pool *p) {
  return (size_t)p->num_blocks * p->hkv * p->page_size * p->d * elem_bytes(p->dtype);
}
}  // namespace lazy

#define LAZY_CUDA_TRY(call)                                      \
  do {                                                           \
    cudaError_t e_ = (call);                                     \
    if (e_ != cudaSuccess) return lazy::record_cuda(e_, #call);  \
  } while (0)
