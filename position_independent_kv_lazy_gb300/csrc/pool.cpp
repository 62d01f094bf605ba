// Pool handle, block allocator, page-word packing, error reporting (host side of the C ABI).
#include <math.h>
#include <stdio.h>
#include <string.h>

#include <unordered_map>

#include "pool_internal.h"

namespace {
thread_local char g_msg[512] = "no error";

uint64_t turn_fraction(double theta) {
  // frac(theta / 2pi) as a 64-bit fixed-point fraction of one turn.
  long double f = (long double)theta / (2.0L * 3.141592653589793238462643383279502884L);
  f -= floorl(f);
  long double scaled = ldexpl(f, 64);
  if (!(scaled < 18446744073709551616.0L)) return 0;  // rounds up to a full turn
  return (uint64_t)scaled;
}
}  // namespace

namespace lazy {
int record_cuda(cudaError_t e, const char *what) {
  snprintf(g_msg, sizeof(g_msg), "%s: %s", what, cudaGetErrorString(e));
  return LAZY_ERR_CUDA;
}
void record_msg(const char *msg) { snprintf(g_msg, sizeof(g_msg), "%s", msg); }

int ensure_device(lazy_pool *p) {
  std::lock_guard<std::mutex> g(p->mu);
  if (p->dev_ready) return LAZY_OK;
  LAZY_CUDA_TRY(cudaGetDevice(&p->device));
  LAZY_CUDA_TRY(cudaDeviceGetAttribute(&p->num_sms, cudaDevAttrMultiProcessorCount, p->device));
  LAZY_CUDA_TRY(cudaMalloc((void **)&p->d_err, 256));
  LAZY_CUDA_TRY(cudaMalloc((void **)&p->d_turn, sizeof(uint64_t) * p->turn.size()));
  LAZY_CUDA_TRY(cudaMemcpy(p->d_turn, p->turn.data(), sizeof(uint64_t) * p->turn.size(),
                           cudaMemcpyHostToDevice));
  LAZY_CUDA_TRY(cudaMemset(p->d_err, 0, 256));
  if (p->alibi) {
    LAZY_CUDA_TRY(cudaMalloc((void **)&p->d_slopes, sizeof(float) * p->slopes.size()));
    LAZY_CUDA_TRY(cudaMemcpy(p->d_slopes, p->slopes.data(), sizeof(float) * p->slopes.size(),
                             cudaMemcpyHostToDevice));
  }
  LAZY_CUDA_TRY(cudaMemset(p->k, 0, pool_bytes(p)));
  LAZY_CUDA_TRY(cudaMemset(p->v, 0, pool_bytes(p)));
  LAZY_CUDA_TRY(cudaDeviceSynchronize());
  p->dev_ready = true;
  return LAZY_OK;
}
}  // namespace lazy

extern "C" {

int lazy_version(void) { return 100; }

const char *lazy_status_string(int s) {
  switch (s) {
    case LAZY_OK: return "ok";
    case LAZY_ERR_INVALID_ARG: return "invalid argument";
    case LAZY_ERR_OUT_OF_BLOCKS: return "out of pool blocks";
    case LAZY_ERR_UNSUPPORTED: return "unsupported configuration";
    case LAZY_ERR_CUDA: return "CUDA error";
    case LAZY_ERR_BAD_PAGE: return "page word outside the pool";
    case LAZY_ERR_TIMEOUT: return "bounded wait expired";
    case LAZY_ERR_SCRATCH_LIMIT: return "call exceeds the fixed scratch of the allocation-free decode";
    default: return "unknown status";
  }
}

const char *lazy_last_error(void) { return g_msg; }

int lazy_pool_create(lazy_pool **out, void *d_k_pages, void *d_v_pages, int32_t num_blocks,
                     int32_t page_size, int32_t num_kv_heads, int32_t head_dim, int32_t dtype,
                     double rope_base) {
  if (!out || !d_k_pages || !d_v_pages || num_blocks <= 0 || num_kv_heads <= 0)
    return LAZY_ERR_INVALID_ARG;
  if (!(rope_base > 0.0) || !isfinite(rope_base)) return LAZY_ERR_INVALID_ARG;
  if (((uintptr_t)d_k_pages & 15) || ((uintptr_t)d_v_pages & 15)) return LAZY_ERR_INVALID_ARG;
  if (dtype != LAZY_DTYPE_BF16 && dtype != LAZY_DTYPE_FP32) return LAZY_ERR_UNSUPPORTED;
  if (page_size != 16) return LAZY_ERR_UNSUPPORTED;
  if (head_dim != 64 && head_dim != 128) return LAZY_ERR_UNSUPPORTED;
  lazy_pool *p = new (std::nothrow) lazy_pool();
  if (!p) return LAZY_ERR_INVALID_ARG;
  p->k = d_k_pages;
  p->v = d_v_pages;
  p->num_blocks = num_blocks;
  p->page_size = page_size;
  p->hkv = num_kv_heads;
  p->d = head_dim;
  p->dtype = dtype;
  p->base = rope_base;
  p->refcount.assign(num_blocks, 0);
  p->free_list.resize(num_blocks);
  for (int32_t i = 0; i < num_blocks; ++i) p->free_list[i] = num_blocks - 1 - i;
  p->turn.resize(head_dim / 2);
  for (int i = 0; i < head_dim / 2; ++i)
    p->turn[i] = turn_fraction(pow(rope_base, -2.0 * (double)i / (double)head_dim));
  *out = p;
  return LAZY_OK;
}

int lazy_pool_destroy(lazy_pool *p) {
  if (!p) return LAZY_ERR_INVALID_ARG;
  if (p->dev_ready) {
    cudaFree(p->d_err);
    cudaFree(p->d_turn);
    if (p->d_slopes) cudaFree(p->d_slopes);
  }
  if (p->stage_done) {
    cudaEventSynchronize(p->stage_done);
    cudaEventDestroy(p->stage_done);
  }
  if (p->h_stage) cudaFreeHost(p->h_stage);
  delete p;
  return LAZY_OK;
}

int lazy_pool_set_alibi(lazy_pool *p, const float *slopes, int32_t num_q_heads) {
  if (!p || !slopes || num_q_heads <= 0 || num_q_heads % p->hkv) return LAZY_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> g(p->mu);
  if (p->encoded || p->dev_ready) {
    lazy::record_msg("lazy_pool_set_alibi: the pool has already been used");
    return LAZY_ERR_INVALID_ARG;
  }
  for (int32_t h = 0; h < num_q_heads; ++h)
    if (!(slopes[h] >= 0.f) || slopes[h] > 64.f) return LAZY_ERR_INVALID_ARG;  // finite, >= 0
  p->slopes.assign(slopes, slopes + num_q_heads);
  p->alibi = true;
  return LAZY_OK;
}

int lazy_pool_set_decode_kernel(lazy_pool *p, int32_t kind) {
  if (!p || kind < LAZY_DECODE_AUTO || kind > LAZY_DECODE_SIMT) return LAZY_ERR_INVALID_ARG;
  p->decode_kernel = kind;
  return LAZY_OK;
}

int lazy_pool_set_schedule_sms(lazy_pool *p, int32_t sms) {
  if (!p || sms < 0) return LAZY_ERR_INVALID_ARG;
  p->schedule_sms = sms;
  return LAZY_OK;
}

int lazy_pool_position_mode(lazy_pool *p, int32_t *mode, int32_t *num_q_heads) {
  if (!p || !mode) return LAZY_ERR_INVALID_ARG;
  *mode = p->alibi ? LAZY_POS_ALIBI : LAZY_POS_ROPE;
  if (num_q_heads) *num_q_heads = (int32_t)p->slopes.size();
  return LAZY_OK;
}

int lazy_pool_set_wait_limit(lazy_pool *p, uint64_t ns) {
  if (!p || ns == 0) return LAZY_ERR_INVALID_ARG;
  p->wait_limit_ns = ns;
  return LAZY_OK;
}

int kv_pool_alloc(lazy_pool *p, int32_t n, int32_t *ids) {
  if (!p || n < 0 || (n > 0 && !ids)) return LAZY_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> g(p->mu);
  if ((size_t)n > p->free_list.size()) return LAZY_ERR_OUT_OF_BLOCKS;
  for (int32_t i = 0; i < n; ++i) {
    int32_t b = p->free_list.back();
    p->free_list.pop_back();
    p->refcount[b] = 1;
    ids[i] = b;
  }
  return LAZY_OK;
}

int kv_pool_retain(lazy_pool *p, const int32_t *ids, int32_t n) {
  if (!p || n < 0 || (n > 0 && !ids)) return LAZY_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> g(p->mu);
  for (int32_t i = 0; i < n; ++i)
    if (ids[i] < 0 || ids[i] >= p->num_blocks || p->refcount[ids[i]] <= 0)
      return LAZY_ERR_INVALID_ARG;
  for (int32_t i = 0; i < n; ++i) ++p->refcount[ids[i]];
  return LAZY_OK;
}

int kv_pool_release(lazy_pool *p, const int32_t *ids, int32_t n) {
  if (!p || n < 0 || (n > 0 && !ids)) return LAZY_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> g(p->mu);
  std::unordered_map<int32_t, int32_t> drops;
  for (int32_t i = 0; i < n; ++i) {
    if (ids[i] < 0 || ids[i] >= p->num_blocks) return LAZY_ERR_INVALID_ARG;
    if (++drops[ids[i]] > p->refcount[ids[i]]) return LAZY_ERR_INVALID_ARG;
  }
  for (int32_t i = 0; i < n; ++i) {
    if (--p->refcount[ids[i]] == 0) p->free_list.push_back(ids[i]);
  }
  return LAZY_OK;
}

int kv_pool_num_free(lazy_pool *p, int32_t *n_free) {
  if (!p || !n_free) return LAZY_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> g(p->mu);
  *n_free = (int32_t)p->free_list.size();
  return LAZY_OK;
}

int kv_pool_refcount(lazy_pool *p, int32_t block, int32_t *rc) {
  if (!p || !rc || block < 0 || block >= p->num_blocks) return LAZY_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> g(p->mu);
  *rc = p->refcount[block];
  return LAZY_OK;
}

int lazy_pack_page(uint32_t block_id, uint32_t offset, uint32_t n_valid, uint64_t *word) {
  if (!word || offset >= (1u << 26) || n_valid < 1 || n_valid > 64) return LAZY_ERR_INVALID_ARG;
  *word = (uint64_t)block_id | ((uint64_t)offset << 32) | ((uint64_t)(n_valid - 1) << 58);
  return LAZY_OK;
}

int lazy_unpack_page(uint64_t word, uint32_t *block_id, uint32_t *offset, uint32_t *n_valid) {
  if (!block_id || !offset || !n_valid) return LAZY_ERR_INVALID_ARG;
  *block_id = (uint32_t)(word & 0xFFFFFFFFull);
  *offset = (uint32_t)((word >> 32) & 0x3FFFFFFull);
  *n_valid = (uint32_t)(word >> 58) + 1u;
  return LAZY_OK;
}

int lazy_pack_pages(int32_t n, const uint32_t *block_ids, const uint32_t *offsets,
                    const uint32_t *n_valid, uint64_t *words) {
  if (n < 0 || (n > 0 && (!block_ids || !offsets || !n_valid || !words)))
    return LAZY_ERR_INVALID_ARG;
  for (int32_t i = 0; i < n; ++i) {
    int rc = lazy_pack_page(block_ids[i], offsets[i], n_valid[i], &words[i]);
    if (rc != LAZY_OK) return rc;
  }
  return LAZY_OK;
}

int lazy_pack_segment(const uint32_t *block_ids, int32_t n_blocks, uint32_t offset,
                      int32_t length, int32_t page_size, int32_t page_positions,
                      uint64_t *words, int32_t max_words, int32_t *n_words) {
  if (!n_words || length < 0 || page_size < 1 || page_size > 64 ||
      (page_positions != 0 && page_positions != 1))
    return LAZY_ERR_INVALID_ARG;
  const int32_t n_pages = (int32_t)(((int64_t)length + page_size - 1) / page_size);
  if (n_pages > 0 && (!block_ids || !words)) return LAZY_ERR_INVALID_ARG;
  if (n_blocks < n_pages || max_words < n_pages) return LAZY_ERR_INVALID_ARG;
  for (int32_t i = 0; i < n_pages; ++i) {
    const uint64_t pos = (uint64_t)offset + (page_positions ? (uint64_t)i * page_size : 0);
    if (pos >= (1ull << 26)) return LAZY_ERR_INVALID_ARG;
    const int32_t nv = length - i * page_size < page_size ? length - i * page_size : page_size;
    int rc = lazy_pack_page(block_ids[i], (uint32_t)pos, (uint32_t)nv, &words[i]);
    if (rc != LAZY_OK) return rc;
  }
  *n_words = n_pages;
  return LAZY_OK;
}

int lazy_get_device_error(lazy_pool *p, int32_t *err, lazy_stream_t stream) {
  if (!p || !err) return LAZY_ERR_INVALID_ARG;
  int rc = lazy::ensure_device(p);
  if (rc != LAZY_OK) return rc;
  cudaStream_t s = (cudaStream_t)stream;
  int32_t h = 0;
  LAZY_CUDA_TRY(cudaMemcpyAsync(&h, p->d_err, sizeof(int32_t), cudaMemcpyDeviceToHost, s));
  LAZY_CUDA_TRY(cudaStreamSynchronize(s));
  LAZY_CUDA_TRY(cudaMemsetAsync(p->d_err, 0, sizeof(int32_t), s));
  LAZY_CUDA_TRY(cudaStreamSynchronize(s));
  *err = h;
  return LAZY_OK;
}

}  // extern "C"
