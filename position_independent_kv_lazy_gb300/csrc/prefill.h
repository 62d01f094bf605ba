// Parameters shared by the prefill kernels (internal).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "pool_internal.h"

namespace lazy {

struct PrefillParams {
  const void *q;
  const void *k_new;
  const void *v_new;
  const int32_t *cu_q;
  const int32_t *q_pos0;
  const uint64_t *words;
  const int32_t *cu_pages;
  const void *k_pool;
  const void *v_pool;
  const uint64_t *turn;
  void *out;
  float *lse;
  int32_t *err;
  int32_t batch, hkv, hq, num_blocks, G, TQ, total_q;
  float scale_log2;
  uint64_t wait_ns;
  const float *slopes;  // ALiBi pools: per query head (device); nullptr for RoPE pools
  void *workspace;      // caller's scratch (tensor-core path: partial results of split units)
  size_t workspace_bytes;
  int32_t qside;        // CUDA-core path: query-side rotation per document offset
  int32_t absolute;     // tensor-core path: reference position 0 (LAZY_PREFILL_ABSOLUTE_KEYS)
  int32_t tc_qside;     // tensor-core path: query-side rotation, reference per document
};

int prefill_simt(lazy_pool *p, const PrefillParams &pp, int32_t max_q_len, cudaStream_t s);
// Tensor-core path; LAZY_ERR_UNSUPPORTED when the shape is not built.
int prefill_tc_supported(const lazy_pool *p, int32_t hq);
int prefill_tc(lazy_pool *p, const PrefillParams &pp, int32_t max_q_len, cudaStream_t s);
// Scratch the tensor-core path can use for this call shape (0 when it would not split).
int prefill_tc_workspace_bytes(lazy_pool *p, int32_t batch, int32_t max_q_len, int32_t hq,
                               size_t *bytes);

}  // namespace lazy
