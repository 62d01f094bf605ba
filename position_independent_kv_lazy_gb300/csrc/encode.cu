// Doc-KV encode: K page row = R(j) k_raw (document-local position j), V copied; scattered into
// the paged pool. The cache thereby holds position-free content ("keys and values purely based on
// content", LazyAttention summaries, core concept) and one copy serves every logical offset.
//
// Also: lazy_debug_gather, a test hook that reads pages through the same device unpack and
// address arithmetic the attention kernels use.
#include <algorithm>
#include <vector>

#include "lazy_common.cuh"
#include "pool_internal.h"

namespace lazy {
namespace {

// A document insert passes its block ids in the launch's parameters: up to 4096 pages (65,536
// tokens, 16 KB of the 32 KB parameter space) per launch, so a long document is one launch.
// Inserts of up to 512 pages take a 2 KB list (a 16 KB parameter block costs a short launch
// about 1 us), and the scattered append (a decode step's tokens, located by a slot map) a
// one-entry list.
constexpr int kMaxIdsPerLaunch = 4096;
constexpr int kSmallIds = 512;

template <int N>
struct BlockList {
  int32_t first_page;  // page index (within the segment) of ids[0]
  int32_t n;
  int32_t ids[N];
};

// One thread = (token, group of hpt kv heads, 16-byte chunk of the lower half): it also handles
// the matching chunk of the upper half, which holds the rotation partners (pairs (i, i + D/2)).
// The angles depend only on the position and the frequency, so a thread evaluates them once
// for its hpt heads (large inserts: several heads per thread; a decode step's few tokens: one).
template <typename T, int D, int NIDS>
__global__ void __launch_bounds__(256) encode_kernel(
    const T *__restrict__ k_raw, const T *__restrict__ v, int32_t n_tokens, int32_t hkv,
    int32_t hpt, T *__restrict__ k_pool, T *__restrict__ v_pool, const uint64_t *__restrict__ turn,
    int32_t tok0, int32_t local_pos0, const __grid_constant__ BlockList<NIDS> blocks,
    const int32_t *__restrict__ slot_map,
    const int32_t *__restrict__ local_pos, int32_t num_blocks, int32_t *err, int32_t rope) {
  constexpr int EPL = 16 / (int)sizeof(T);
  constexpr int CH = (D / 2) / EPL;
  // A decode launched right after this append may start its launch early; it waits for this
  // grid to finish before reading anything (programmatic dependent launch).
  cudaTriggerProgrammaticLaunchCompletion();
  const int32_t groups = hkv / hpt;
  const int64_t total = (int64_t)n_tokens * groups * CH;
  for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int c = (int)(idx % CH);
    const int64_t rest = idx / CH;
    const int h0 = (int)(rest % groups) * hpt;
    const int32_t t = tok0 + (int32_t)(rest / groups);
    int32_t j, blk, slot;
    if (slot_map) {
      const int32_t s = slot_map[t];
      if (s < 0) continue;
      j = local_pos[t];
      blk = s / kPage;
      slot = s % kPage;
      if (blk >= num_blocks) {  // a slot outside the pool: flag it, write nothing
        if (c == 0 && h0 == 0) set_error(err, LAZY_DEVERR_BAD_PAGE);
        continue;
      }
    } else {
      j = local_pos0 + t;
      blk = blocks.ids[j / kPage - blocks.first_page];
      slot = j % kPage;
    }
    float cs[EPL], sn[EPL];
    if (rope) {  // ALiBi pools keep K as given
#pragma unroll
      for (int e = 0; e < EPL; ++e) rope_cos_sin((int64_t)j, turn[c * EPL + e], cs[e], sn[e]);
    }
#pragma unroll 2
    for (int h = h0; h < h0 + hpt; ++h) {
      const size_t src = ((size_t)t * hkv + h) * D;
      const size_t dst = (((size_t)blk * hkv + h) * kPage + slot) * D;
      const uint4 ka = *reinterpret_cast<const uint4 *>(k_raw + src + c * EPL);
      const uint4 kb = *reinterpret_cast<const uint4 *>(k_raw + src + D / 2 + c * EPL);
      const uint4 va = *reinterpret_cast<const uint4 *>(v + src + c * EPL);
      const uint4 vb = *reinterpret_cast<const uint4 *>(v + src + D / 2 + c * EPL);
      float lo[EPL], hi[EPL];
      unpack16<T>(ka, lo);
      unpack16<T>(kb, hi);
      if (rope) {
#pragma unroll
        for (int e = 0; e < EPL; ++e) {
          const float x = lo[e], y = hi[e];
          lo[e] = x * cs[e] - y * sn[e];
          hi[e] = x * sn[e] + y * cs[e];
        }
      }
      *reinterpret_cast<uint4 *>(k_pool + dst + c * EPL) = pack16<T>(lo);
      *reinterpret_cast<uint4 *>(k_pool + dst + D / 2 + c * EPL) = pack16<T>(hi);
      *reinterpret_cast<uint4 *>(v_pool + dst + c * EPL) = va;
      *reinterpret_cast<uint4 *>(v_pool + dst + D / 2 + c * EPL) = vb;
    }
  }
}

// kv heads per thread: the largest of 8, 4, 2, 1 dividing Hkv that still leaves two 256-thread
// CTAs per SM (fewer, longer threads would expose the memory latency of short launches).
int heads_per_thread(const lazy_pool *p, int64_t rows) {
  for (int hpt = 8; hpt > 1; hpt >>= 1)
    if (p->hkv % hpt == 0 && rows * (p->hkv / hpt) >= (int64_t)p->num_sms * 512) return hpt;
  return 1;
}

template <typename T, int D, int NIDS>
int launch_encode(lazy_pool *p, const void *k_raw, const void *v, int32_t n_tokens, int32_t tok0,
                  int32_t local_pos0, const BlockList<NIDS> &bl, const int32_t *slot_map,
                  const int32_t *local_pos, cudaStream_t s) {
  constexpr int EPL = 16 / (int)sizeof(T);
  const int64_t rows = (int64_t)n_tokens * ((D / 2) / EPL);
  const int hpt = heads_per_thread(p, rows);
  const int64_t total = rows * (p->hkv / hpt);
  const int threads = 256;
  const int64_t want = (total + threads - 1) / threads;
  const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(want, (int64_t)p->num_sms * 16));
  encode_kernel<T, D, NIDS><<<grid, threads, 0, s>>>(
      (const T *)k_raw, (const T *)v, n_tokens, p->hkv, hpt, (T *)p->k, (T *)p->v, p->d_turn, tok0,
      local_pos0, bl, slot_map, local_pos, p->num_blocks, p->d_err, p->alibi ? 0 : 1);
  LAZY_CUDA_TRY(cudaGetLastError());
  return LAZY_OK;
}

template <int NIDS>
int dispatch_encode(lazy_pool *p, const void *k_raw, const void *v, int32_t n_tokens,
                    int32_t tok0, int32_t local_pos0, const BlockList<NIDS> &bl,
                    const int32_t *slot_map, const int32_t *local_pos, cudaStream_t s) {
  if (p->dtype == LAZY_DTYPE_BF16) {
    if (p->d == 128)
      return launch_encode<__nv_bfloat16, 128, NIDS>(p, k_raw, v, n_tokens, tok0, local_pos0, bl,
                                               slot_map, local_pos, s);
    return launch_encode<__nv_bfloat16, 64, NIDS>(p, k_raw, v, n_tokens, tok0, local_pos0, bl,
                                            slot_map, local_pos, s);
  }
  if (p->d == 128)
    return launch_encode<float, 128, NIDS>(p, k_raw, v, n_tokens, tok0, local_pos0, bl, slot_map,
                                     local_pos, s);
  return launch_encode<float, 64, NIDS>(p, k_raw, v, n_tokens, tok0, local_pos0, bl, slot_map,
                                  local_pos, s);
}

// ----------------------------------------------------------------------------------------------
// Materialised copy (the position-aware baseline the summaries compare against, "Problem
// statement" and the prefill part: a cached block re-encoded for one target position by two
// rotations, one resetting it to position 0 and one to the target). Token j of a cached segment
// (K row R(j) k) becomes K row R(offset + j) R(-j) (R(j) k) in the copy; V is copied. The two
// rotations compose to R(offset) exactly (the angle arithmetic is exact modulo a full turn), so
// the copy applies that one rotation in fp32 with one rounding to the pool type, and its angles
// depend only on the offset. One thread = (token, kv heads h0 .. h0 + hpt - 1, 16-byte chunk of
// the lower half) and the matching chunk of the upper half, as in the encode.
// ----------------------------------------------------------------------------------------------
constexpr int kMaxMatIds = 256;
struct MatBlocks {
  int32_t first_page;
  int32_t n;
  int32_t src[kMaxMatIds];
  int32_t dst[kMaxMatIds];
};

// Rotate one (token, chunk) of hpt consecutive kv heads from src to dst (element offsets of head
// h0), the next head's loads issued before this head's arithmetic; the first head's loads go out
// before the angles are evaluated.
template <typename T, int D>
__device__ __forceinline__ void copy_rotate_heads(T *__restrict__ k_pool, T *__restrict__ v_pool,
                                                  const uint64_t *__restrict__ turn, int c,
                                                  int32_t offset, int hpt, size_t src,
                                                  size_t dst) {
  constexpr int EPL = 16 / (int)sizeof(T);
  constexpr size_t kHead = (size_t)kPage * D;  // elements between heads of one block
  uint4 ka = *reinterpret_cast<const uint4 *>(k_pool + src);
  uint4 kb = *reinterpret_cast<const uint4 *>(k_pool + src + D / 2);
  uint4 va = *reinterpret_cast<const uint4 *>(v_pool + src);
  uint4 vb = *reinterpret_cast<const uint4 *>(v_pool + src + D / 2);
  float cs[EPL], sn[EPL];
#pragma unroll
  for (int e = 0; e < EPL; ++e) rope_cos_sin((int64_t)offset, turn[c * EPL + e], cs[e], sn[e]);
  for (int hh = 0; hh < hpt; ++hh) {
    uint4 nka = ka, nkb = kb, nva = va, nvb = vb;
    if (hh + 1 < hpt) {
      const size_t ns = src + kHead;
      nka = *reinterpret_cast<const uint4 *>(k_pool + ns);
      nkb = *reinterpret_cast<const uint4 *>(k_pool + ns + D / 2);
      nva = *reinterpret_cast<const uint4 *>(v_pool + ns);
      nvb = *reinterpret_cast<const uint4 *>(v_pool + ns + D / 2);
    }
    float lo[EPL], hi[EPL];
    unpack16<T>(ka, lo);
    unpack16<T>(kb, hi);
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
      const float x = lo[e], y = hi[e];
      lo[e] = x * cs[e] - y * sn[e];
      hi[e] = x * sn[e] + y * cs[e];
    }
    *reinterpret_cast<uint4 *>(k_pool + dst) = pack16<T>(lo);
    *reinterpret_cast<uint4 *>(k_pool + dst + D / 2) = pack16<T>(hi);
    *reinterpret_cast<uint4 *>(v_pool + dst) = va;
    *reinterpret_cast<uint4 *>(v_pool + dst + D / 2) = vb;
    ka = nka, kb = nkb, va = nva, vb = nvb;
    src += kHead;
    dst += kHead;
  }
}

template <typename T, int D>
__global__ void __launch_bounds__(256) materialise_kernel(
    T *__restrict__ k_pool, T *__restrict__ v_pool, const uint64_t *__restrict__ turn,
    int32_t hkv, int32_t hpt, int32_t tok_lo, int32_t n_tokens, int32_t offset, MatBlocks mb) {
  constexpr int EPL = 16 / (int)sizeof(T);
  constexpr int CH = (D / 2) / EPL;
  const int32_t groups = hkv / hpt;
  const int64_t total = (int64_t)n_tokens * groups * CH;
  for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int c = (int)(idx % CH);
    const int64_t rest = idx / CH;
    const int h0 = (int)(rest % groups) * hpt;
    const int32_t j = tok_lo + (int32_t)(rest / groups);
    const int pg = j / kPage - mb.first_page, slot = j % kPage;
    copy_rotate_heads<T, D>(k_pool, v_pool, turn, c, offset, hpt,
                            (((size_t)mb.src[pg] * hkv + h0) * kPage + slot) * D + c * EPL,
                            (((size_t)mb.dst[pg] * hkv + h0) * kPage + slot) * D + c * EPL);
  }
}

// Many copies in one launch: one item = (page of the batch, slot, head group, chunk). The
// page's entry gives its copy, its page index within the copy and its two blocks; the copy's
// entry its token count and offset.
template <typename T, int D>
__global__ void __launch_bounds__(256) materialise_batch_kernel(
    T *__restrict__ k_pool, T *__restrict__ v_pool, const uint64_t *__restrict__ turn,
    int32_t hkv, int32_t hpt, const int4 *__restrict__ pages, const int2 *__restrict__ copies,
    int32_t total_pages) {
  constexpr int EPL = 16 / (int)sizeof(T);
  constexpr int CH = (D / 2) / EPL;
  const int32_t groups = hkv / hpt;
  const int64_t total = (int64_t)total_pages * kPage * groups * CH;
  for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int c = (int)(idx % CH);
    int64_t rest = idx / CH;
    const int h0 = (int)(rest % groups) * hpt;
    rest /= groups;
    const int slot = (int)(rest % kPage);
    const int4 pe = pages[rest / kPage];  // (copy, page within the copy, source, destination)
    const int2 ce = copies[pe.x];         // (tokens, offset)
    if (pe.y * kPage + slot >= ce.x) continue;
    copy_rotate_heads<T, D>(k_pool, v_pool, turn, c, ce.y, hpt,
                            (((size_t)pe.z * hkv + h0) * kPage + slot) * D + c * EPL,
                            (((size_t)pe.w * hkv + h0) * kPage + slot) * D + c * EPL);
  }
}

template <typename T, int D>
int launch_materialise_batch(lazy_pool *p, const int4 *pages, const int2 *copies,
                             int32_t total_pages, cudaStream_t s) {
  constexpr int EPL = 16 / (int)sizeof(T);
  const int64_t rows = (int64_t)total_pages * kPage * ((D / 2) / EPL);
  const int hpt = heads_per_thread(p, rows);
  const int64_t total = rows * (p->hkv / hpt);
  const int threads = 256;
  const int64_t want = (total + threads - 1) / threads;
  const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(want, (int64_t)p->num_sms * 16));
  materialise_batch_kernel<T, D><<<grid, threads, 0, s>>>((T *)p->k, (T *)p->v, p->d_turn,
                                                         p->hkv, hpt, pages, copies,
                                                         total_pages);
  LAZY_CUDA_TRY(cudaGetLastError());
  return LAZY_OK;
}

template <typename T, int D>
int launch_materialise(lazy_pool *p, int32_t tok_lo, int32_t n_tokens, int32_t offset,
                       const MatBlocks &mb, cudaStream_t s) {
  constexpr int EPL = 16 / (int)sizeof(T);
  const int64_t rows = (int64_t)n_tokens * ((D / 2) / EPL);
  const int hpt = heads_per_thread(p, rows);
  const int64_t total = rows * (p->hkv / hpt);
  const int threads = 256;
  const int64_t want = (total + threads - 1) / threads;
  const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(want, (int64_t)p->num_sms * 16));
  materialise_kernel<T, D><<<grid, threads, 0, s>>>((T *)p->k, (T *)p->v, p->d_turn, p->hkv,
                                                   hpt, tok_lo, n_tokens, offset, mb);
  LAZY_CUDA_TRY(cudaGetLastError());
  return LAZY_OK;
}

// ----------------------------------------------------------------------------------------------
// Debug gather: same unpack (word_block / word_offset / word_nvalid) and page addressing as the
// attention kernels.
// ----------------------------------------------------------------------------------------------
__global__ void gather_kernel(const uint64_t *__restrict__ words, int32_t n_words, int32_t hkv,
                              int32_t num_blocks, size_t page_bytes, const uint8_t *k_pool,
                              const uint8_t *v_pool, uint8_t *k_out, uint8_t *v_out,
                              uint32_t *fields, int32_t *err) {
  const int32_t w = blockIdx.x;
  if (w >= n_words) return;
  const uint64_t word = words[w];
  uint32_t blk = word_block(word);
  if (threadIdx.x == 0) {
    fields[3 * w + 0] = blk;
    fields[3 * w + 1] = word_offset(word);
    fields[3 * w + 2] = word_nvalid(word);
  }
  if (blk >= (uint32_t)num_blocks) {
    if (threadIdx.x == 0) set_error(err, LAZY_DEVERR_BAD_PAGE);
    blk = 0;
  }
  const size_t per_word = page_bytes * hkv;
  const uint4 *ks = reinterpret_cast<const uint4 *>(k_pool + (size_t)blk * per_word);
  const uint4 *vs = reinterpret_cast<const uint4 *>(v_pool + (size_t)blk * per_word);
  uint4 *kd = reinterpret_cast<uint4 *>(k_out + (size_t)w * per_word);
  uint4 *vd = reinterpret_cast<uint4 *>(v_out + (size_t)w * per_word);
  for (size_t i = threadIdx.x; i < per_word / 16; i += blockDim.x) {
    kd[i] = ks[i];
    vd[i] = vs[i];
  }
}

// Waits on a barrier that nothing arrives at; gives up after limit_ns (bounded wait).
__global__ void wait_timeout_kernel(uint64_t limit_ns, int32_t *err) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
  }
  __syncwarp();
  const bool ok = mbar_wait(&bar, 0, limit_ns);
  if (!ok && threadIdx.x == 0) set_error(err, LAZY_DEVERR_TIMEOUT);
}

}  // namespace
}  // namespace lazy

using namespace lazy;

extern "C" int lazy_debug_wait_timeout(lazy_pool *p, uint64_t limit_ns, lazy_stream_t stream) {
  if (!p || limit_ns == 0 || limit_ns > 10000000000ull) return LAZY_ERR_INVALID_ARG;
  int rc = ensure_device(p);
  if (rc != LAZY_OK) return rc;
  wait_timeout_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(limit_ns, p->d_err);
  LAZY_CUDA_TRY(cudaGetLastError());
  return LAZY_OK;
}

extern "C" int kv_pool_insert_doc(lazy_pool *p, const void *k_raw, const void *v,
                                  int32_t n_tokens, int32_t local_pos0, int32_t *block_ids,
                                  int32_t *n_blocks, int32_t max_blocks, lazy_stream_t stream) {
  if (!p || n_tokens < 0 || local_pos0 < 0 || !n_blocks || *n_blocks < 0 || max_blocks < 0)
    return LAZY_ERR_INVALID_ARG;
  if (n_tokens > 0 && (!k_raw || !v || !block_ids)) return LAZY_ERR_INVALID_ARG;
  if (((uintptr_t)k_raw & 15) || ((uintptr_t)v & 15)) return LAZY_ERR_INVALID_ARG;
  if (n_tokens == 0) return LAZY_OK;
  p->encoded = true;
  const int64_t end = (int64_t)local_pos0 + n_tokens;
  if (end > (1ll << 26)) return LAZY_ERR_INVALID_ARG;
  const int32_t need = (int32_t)((end + kPage - 1) / kPage);
  if (need > max_blocks || *n_blocks > max_blocks) return LAZY_ERR_INVALID_ARG;
  int rc = ensure_device(p);
  if (rc != LAZY_OK) return rc;
  for (int32_t i = 0; i < std::min(*n_blocks, need); ++i)
    if (block_ids[i] < 0 || block_ids[i] >= p->num_blocks) return LAZY_ERR_INVALID_ARG;
  if (need > *n_blocks) {
    rc = kv_pool_alloc(p, need - *n_blocks, block_ids + *n_blocks);
    if (rc != LAZY_OK) return rc;
    *n_blocks = need;
  }
  cudaStream_t s = (cudaStream_t)stream;
  const int32_t first_page = local_pos0 / kPage, last_page = (int32_t)((end - 1) / kPage);
  // one parameter block per call (kept off the stack of the caller's thread)
  const int32_t pages = last_page - first_page + 1;
  auto run = [&](auto &bl, int32_t max_ids) -> int {
    for (int32_t pg = first_page; pg <= last_page; pg += max_ids) {
      bl.first_page = pg;
      bl.n = std::min(max_ids, last_page - pg + 1);
      for (int i = 0; i < bl.n; ++i) bl.ids[i] = block_ids[pg + i];
      const int64_t pos_lo = std::max<int64_t>(local_pos0, (int64_t)pg * kPage);
      const int64_t pos_hi = std::min<int64_t>(end, (int64_t)(pg + bl.n) * kPage);
      const int rc2 = dispatch_encode(p, k_raw, v, (int32_t)(pos_hi - pos_lo),
                                      (int32_t)(pos_lo - local_pos0), local_pos0, bl, nullptr,
                                      nullptr, s);
      if (rc2 != LAZY_OK) return rc2;
    }
    return LAZY_OK;
  };
  if (pages <= kSmallIds) {
    static thread_local BlockList<kSmallIds> small;
    rc = run(small, kSmallIds);
  } else {
    static thread_local BlockList<kMaxIdsPerLaunch> large;
    rc = run(large, kMaxIdsPerLaunch);
  }
  return rc;
}

// Scattered encode: token t goes to slot_mapping[t] with local position local_pos[t].
extern "C" int kv_pool_write_tokens(lazy_pool *p, const void *k_raw, const void *v,
                                    int32_t n_tokens, const int32_t *slot_mapping,
                                    const int32_t *local_pos, lazy_stream_t stream) {
  if (!p || n_tokens < 0) return LAZY_ERR_INVALID_ARG;
  if (n_tokens == 0) return LAZY_OK;
  if (!k_raw || !v || !slot_mapping || !local_pos) return LAZY_ERR_INVALID_ARG;
  if (((uintptr_t)k_raw & 15) || ((uintptr_t)v & 15)) return LAZY_ERR_INVALID_ARG;
  int rc = ensure_device(p);
  if (rc != LAZY_OK) return rc;
  p->encoded = true;
  BlockList<1> bl;  // unused: the slot map locates every token
  bl.first_page = 0;
  bl.n = 0;
  bl.ids[0] = 0;
  return dispatch_encode(p, k_raw, v, n_tokens, 0, 0, bl, slot_mapping, local_pos,
                         (cudaStream_t)stream);
}

extern "C" int kv_pool_materialise(lazy_pool *p, const int32_t *src_block_ids,
                                   const int32_t *dst_block_ids, int32_t n_tokens,
                                   int32_t offset, lazy_stream_t stream) {
  if (!p || n_tokens < 0 || offset < 0) return LAZY_ERR_INVALID_ARG;
  if (n_tokens == 0) return LAZY_OK;
  if (!src_block_ids || !dst_block_ids) return LAZY_ERR_INVALID_ARG;
  if (p->alibi) return LAZY_ERR_UNSUPPORTED;  // ALiBi pools cache K unrotated
  if ((int64_t)offset + n_tokens > (1ll << 26)) return LAZY_ERR_INVALID_ARG;
  const int32_t n_pages = (n_tokens + kPage - 1) / kPage;
  std::vector<int32_t> src_sorted(src_block_ids, src_block_ids + n_pages);
  std::sort(src_sorted.begin(), src_sorted.end());
  for (int32_t i = 0; i < n_pages; ++i) {
    if (src_block_ids[i] < 0 || src_block_ids[i] >= p->num_blocks || dst_block_ids[i] < 0 ||
        dst_block_ids[i] >= p->num_blocks)
      return LAZY_ERR_INVALID_ARG;
    // the copy must not overwrite the pages it reads
    if (std::binary_search(src_sorted.begin(), src_sorted.end(), dst_block_ids[i]))
      return LAZY_ERR_INVALID_ARG;
  }
  int rc = ensure_device(p);
  if (rc != LAZY_OK) return rc;
  p->encoded = true;
  cudaStream_t s = (cudaStream_t)stream;
  for (int32_t pg = 0; pg < n_pages; pg += kMaxMatIds) {
    MatBlocks mb;
    mb.first_page = pg;
    mb.n = std::min(kMaxMatIds, n_pages - pg);
    for (int i = 0; i < mb.n; ++i) {
      mb.src[i] = src_block_ids[pg + i];
      mb.dst[i] = dst_block_ids[pg + i];
    }
    const int32_t lo = pg * kPage, hi = std::min(n_tokens, (pg + mb.n) * kPage);
    if (p->dtype == LAZY_DTYPE_BF16)
      rc = p->d == 128 ? launch_materialise<__nv_bfloat16, 128>(p, lo, hi - lo, offset, mb, s)
                       : launch_materialise<__nv_bfloat16, 64>(p, lo, hi - lo, offset, mb, s);
    else
      rc = p->d == 128 ? launch_materialise<float, 128>(p, lo, hi - lo, offset, mb, s)
                       : launch_materialise<float, 64>(p, lo, hi - lo, offset, mb, s);
    if (rc != LAZY_OK) return rc;
  }
  return LAZY_OK;
}

extern "C" int kv_pool_materialise_batch(lazy_pool *p, int32_t n_copies, const int32_t *cu_pages,
                                         const int32_t *src_block_ids,
                                         const int32_t *dst_block_ids, const int32_t *n_tokens,
                                         const int32_t *offsets, lazy_stream_t stream) {
  if (!p || n_copies < 0) return LAZY_ERR_INVALID_ARG;
  if (n_copies == 0) return LAZY_OK;
  if (!cu_pages || !n_tokens || !offsets || cu_pages[0] != 0) return LAZY_ERR_INVALID_ARG;
  if (p->alibi) return LAZY_ERR_UNSUPPORTED;  // ALiBi pools cache K unrotated
  for (int32_t c = 0; c < n_copies; ++c) {
    if (n_tokens[c] < 0 || offsets[c] < 0 || (int64_t)offsets[c] + n_tokens[c] > (1ll << 26))
      return LAZY_ERR_INVALID_ARG;
    if ((int64_t)cu_pages[c + 1] - cu_pages[c] != (n_tokens[c] + kPage - 1) / kPage)
      return LAZY_ERR_INVALID_ARG;
  }
  const int32_t total_pages = cu_pages[n_copies];
  if (total_pages == 0) return LAZY_OK;
  if (!src_block_ids || !dst_block_ids) return LAZY_ERR_INVALID_ARG;
  // no copy may overwrite pages that any copy reads, and no two may write one block: one byte
  // per pool block (1 = read by a copy, 2 = written by one)
  std::vector<uint8_t> use(p->num_blocks, 0);
  for (int32_t i = 0; i < total_pages; ++i) {
    if (src_block_ids[i] < 0 || src_block_ids[i] >= p->num_blocks) return LAZY_ERR_INVALID_ARG;
    use[src_block_ids[i]] = 1;
  }
  for (int32_t i = 0; i < total_pages; ++i) {
    const int32_t b = dst_block_ids[i];
    if (b < 0 || b >= p->num_blocks || use[b] != 0) return LAZY_ERR_INVALID_ARG;
    use[b] = 2;
  }
  int rc = ensure_device(p);
  if (rc != LAZY_OK) return rc;
  p->encoded = true;
  cudaStream_t s = (cudaStream_t)stream;
  const size_t pages_bytes = sizeof(int4) * (size_t)total_pages;
  const size_t bytes = pages_bytes + sizeof(int2) * (size_t)n_copies;
  // The page list is written into the pool's pinned staging buffer and uploaded from there in
  // one asynchronous copy (a pageable source would go through the driver's staging, which cost
  // more than the copy kernel itself). The previous call's upload from the buffer ends first.
  std::lock_guard<std::mutex> g(p->mu);
  if (p->stage_done) LAZY_CUDA_TRY(cudaEventSynchronize(p->stage_done));
  else LAZY_CUDA_TRY(cudaEventCreateWithFlags(&p->stage_done, cudaEventDisableTiming));
  if (p->h_stage_bytes < bytes) {
    if (p->h_stage) LAZY_CUDA_TRY(cudaFreeHost(p->h_stage));
    p->h_stage = nullptr;
    p->h_stage_bytes = 0;
    size_t cap = (size_t)1 << 20;
    while (cap < bytes) cap <<= 1;
    LAZY_CUDA_TRY(cudaHostAlloc(&p->h_stage, cap, cudaHostAllocDefault));
    p->h_stage_bytes = cap;
  }
  // the page list: (copy, page within the copy, source, destination) per page, then
  // (tokens, offset) per copy
  int4 *pages = reinterpret_cast<int4 *>(p->h_stage);
  int2 *copies = reinterpret_cast<int2 *>(reinterpret_cast<uint8_t *>(p->h_stage) + pages_bytes);
  for (int32_t c = 0; c < n_copies; ++c) {
    copies[c] = make_int2(n_tokens[c], offsets[c]);
    for (int32_t pg = cu_pages[c]; pg < cu_pages[c + 1]; ++pg)
      pages[pg] = make_int4(c, pg - cu_pages[c], src_block_ids[pg], dst_block_ids[pg]);
  }
  void *buf = nullptr;
  LAZY_CUDA_TRY(cudaMallocAsync(&buf, bytes, s));
  cudaError_t e = cudaMemcpyAsync(buf, p->h_stage, bytes, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaEventRecord(p->stage_done, s);
  if (e != cudaSuccess) {
    cudaFreeAsync(buf, s);
    return record_cuda(e, "kv_pool_materialise_batch page list");
  }
  const int4 *d_pages = reinterpret_cast<const int4 *>(buf);
  const int2 *d_copies = reinterpret_cast<const int2 *>((uint8_t *)buf + pages_bytes);
  if (p->dtype == LAZY_DTYPE_BF16)
    rc = p->d == 128
             ? launch_materialise_batch<__nv_bfloat16, 128>(p, d_pages, d_copies, total_pages, s)
             : launch_materialise_batch<__nv_bfloat16, 64>(p, d_pages, d_copies, total_pages, s);
  else
    rc = p->d == 128 ? launch_materialise_batch<float, 128>(p, d_pages, d_copies, total_pages, s)
                     : launch_materialise_batch<float, 64>(p, d_pages, d_copies, total_pages, s);
  const cudaError_t ef = cudaFreeAsync(buf, s);
  if (rc != LAZY_OK) return rc;
  LAZY_CUDA_TRY(ef);
  return LAZY_OK;
}

extern "C" int lazy_debug_gather(lazy_pool *p, const uint64_t *words, int32_t n_words,
                                 void *k_out, void *v_out, uint32_t *fields,
                                 lazy_stream_t stream) {
  if (!p || n_words < 0) return LAZY_ERR_INVALID_ARG;
  if (n_words == 0) return LAZY_OK;
  if (!words || !k_out || !v_out || !fields) return LAZY_ERR_INVALID_ARG;
  if (((uintptr_t)k_out & 15) || ((uintptr_t)v_out & 15)) return LAZY_ERR_INVALID_ARG;
  int rc = ensure_device(p);
  if (rc != LAZY_OK) return rc;
  const size_t page_bytes = (size_t)p->page_size * p->d * elem_bytes(p->dtype);
  gather_kernel<<<n_words, 256, 0, (cudaStream_t)stream>>>(
      words, n_words, p->hkv, p->num_blocks, page_bytes, (const uint8_t *)p->k,
      (const uint8_t *)p->v, (uint8_t *)k_out, (uint8_t *)v_out, fields, p->d_err);
  LAZY_CUDA_TRY(cudaGetLastError());
  return LAZY_OK;
}
