// Split-KV GQA decode with deferred RoPE (LazyAttention summaries, decoding part: M = 1, the
// rotation fused into the inner loop, the query re-rotated only when the offset changes at a
// document boundary, (block id, offset) read from one packed word, memory traffic = K and V).
//
// Work partition. Every (request b, virtual head hv) is a "unit" whose pages are the request's
// page words; a virtual head is one kv head and a chunk of at most 8 of its query heads. All
// units' pages are flattened in (b, hv, page) order and cut into equal contiguous ranges, one per
// warp of a single persistent wave (grid = SMs x resident CTAs). A warp streams its range through
// its own two-stage ring of shared-memory stages filled by 1-D bulk async copies (one 4 KB K page
// and one 4 KB V page per stage for bf16, D = 128), so the pipeline never drains at unit
// boundaries and
// every SM moves the same number of bytes. Each (unit, warp) piece leaves a partial
// (o / l, log2-sum-exp) in the workspace at slot (unit + warp); combine_kernel merges the pieces
// of a unit (log-sum-exp combine).
//
// Per page, lane (group gq, row chunk r) holds 16 bytes of a key row: the QK partial dot products
// of the GC query heads are reduced across the row's lanes with a reduce-scatter of shuffles,
// the page's per-head max with a butterfly, probabilities go through 256 B of shared memory, and
// PV accumulates in registers (GC x 16 bytes worth of fp32 per lane).
#include <cuda.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <mutex>
#include <type_traits>

#include "lazy_common.cuh"
#include "pool_internal.h"

namespace lazy {
namespace {

struct DecodeParams {
  const void *q;
  const int32_t *q_pos;
  const uint64_t *words;
  const int32_t *cu_pages;
  const void *k_pool;
  const void *v_pool;
  const uint64_t *turn;
  float *ws_o;    // [slots][GC][D]
  float *ws_lse;  // [slots][GC]  log2-domain
  int32_t *err;
  int32_t batch, hkv, hq, num_blocks;
  int32_t hv;      // virtual heads = hkv * chunks
  int32_t chunks;  // query-head chunks per kv head
  float scale_log2;
  uint64_t wait_ns;
  const float *slopes;  // ALiBi pools: per query head; nullptr for RoPE pools
};

// KV head of virtual head hv. Most shapes have one chunk per kv head; the division is kept off
// their per-page path (a 32-bit division is about 20 instructions).
__device__ __forceinline__ int32_t kv_head_of(int32_t hv, int32_t chunks) {
  return chunks == 1 ? hv : hv / chunks;
}

// Walks the flattened (request, virtual head, page) sequence.
struct Walker {
  int32_t b, hv, pg, npages, wbase;
  __device__ __forceinline__ void init(int64_t x, const int32_t *cu, int32_t batch,
                                       int32_t hvt) {
    int lo = 0, hi = batch;  // hvt*cu[lo] <= x < hvt*cu[hi]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if ((int64_t)hvt * cu[mid] <= x) lo = mid; else hi = mid;
    }
    b = lo;
    wbase = cu[b];
    npages = cu[b + 1] - wbase;
    const int64_t rem = x - (int64_t)hvt * wbase;
    hv = (int32_t)(rem / npages);
    pg = (int32_t)(rem % npages);
  }
  __device__ __forceinline__ void advance(const int32_t *cu, int32_t batch, int32_t hvt) {
    if (++pg < npages) return;
    pg = 0;
    if (++hv < hvt) return;
    hv = 0;
    do { ++b; } while (b < batch && cu[b + 1] == cu[b]);
    if (b < batch) {
      wbase = cu[b];
      npages = cu[b + 1] - wbase;
    }
  }
};

// Reduce-scatter of N values across lane groups of size 2*M (masks M, M/2, ..., 1). While more
// than one value is left, each step keeps half of them (lanes with the mask bit set keep the upper
// half, `base` tracks which flat index slot 0 now holds); single values are all-reduced.
template <int N, int M>
__device__ __forceinline__ void reduce_scatter(float *v, int lane, int &base) {
  if constexpr (M >= 1) {
    if constexpr (N >= 2) {
      const bool upper = (lane & M) != 0;
#pragma unroll
      for (int i = 0; i < N / 2; ++i) {
        const float send = upper ? v[i] : v[i + N / 2];
        const float keep = upper ? v[i + N / 2] : v[i];
        v[i] = keep + __shfl_xor_sync(0xffffffffu, send, M);
      }
      if (upper) base += N / 2;
      reduce_scatter<N / 2, M / 2>(v, lane, base);
    } else {
      v[0] += __shfl_xor_sync(0xffffffffu, v[0], M);
      reduce_scatter<1, M / 2>(v, lane, base);
    }
  }
}

template <typename T, int D, int GC, int STAGES>
struct DecodeSmem {
  static constexpr int kPageBytes = kPage * D * (int)sizeof(T);
  static constexpr int kK = 0;
  static constexpr int kV = kK + STAGES * kPageBytes;
  static constexpr int kP = kV + STAGES * kPageBytes;          // float [kPage][GC]
  static constexpr int kQ = kP + kPage * GC * 4;               // float [GC][D]
  static constexpr int kBar = kQ + GC * D * 4;                 // uint64 [STAGES]
  static constexpr int kWord = kBar + STAGES * 8;              // uint64 [STAGES]
  static constexpr int kUnit = kWord + STAGES * 8;             // int32 [STAGES]
  static constexpr int kBytes = ((kUnit + STAGES * 4) + 127) / 128 * 128;  // per warp
};

template <typename T, int D, int GC, int WARPS, int STAGES>
__global__ void __launch_bounds__(WARPS * 32) decode_split_kernel(const DecodeParams p) {
  using S = DecodeSmem<T, D, GC, STAGES>;
  constexpr int EPL = 16 / (int)sizeof(T);  // elements per 16-byte load
  constexpr int EP2 = EPL / 2;              // float2 pairs per 16-byte load
  constexpr int LPR = D / EPL;              // lanes per key row
  constexpr int KPI = 32 / LPR;             // keys per load instruction
  constexpr int NIT = kPage / KPI;          // load iterations per page
  constexpr int NV0 = NIT * GC;             // partial dots per lane per page
  constexpr int NF = NV0 / LPR > 0 ? NV0 / LPR : 1;  // fully reduced values per lane
  static_assert(LPR <= 32 && KPI <= kPage, "shape");

  extern __shared__ __align__(128) uint8_t smem_split[];  // the other kernels align theirs to 1 KB
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint8_t *ws = smem_split + warp * S::kBytes;
  T *kbuf = reinterpret_cast<T *>(ws + S::kK);
  T *vbuf = reinterpret_cast<T *>(ws + S::kV);
  float *psm = reinterpret_cast<float *>(ws + S::kP);
  float *qraw = reinterpret_cast<float *>(ws + S::kQ);
  uint64_t *bars = reinterpret_cast<uint64_t *>(ws + S::kBar);
  uint64_t *meta_w = reinterpret_cast<uint64_t *>(ws + S::kWord);
  int32_t *meta_u = reinterpret_cast<int32_t *>(ws + S::kUnit);

  // Everything this kernel reads may come from the preceding kernel in the stream (a token
  // append launched ahead of it); wait for it (no-op without programmatic dependent launch).
  cudaGridDependencySynchronize();
  const int32_t B = p.batch, HV = p.hv;
  const int64_t N = (int64_t)HV * p.cu_pages[B];
  const int64_t WT = (int64_t)gridDim.x * WARPS;
  const int64_t wg = (int64_t)blockIdx.x * WARPS + warp;
  const int64_t x0 = wg * N / WT, x1 = (wg + 1) * N / WT;
  if (x0 >= x1) {
    cudaTriggerProgrammaticLaunchCompletion();
    return;
  }
  const int64_t n_mine = x1 - x0;

  if (lane == 0) {
    for (int s = 0; s < STAGES; ++s) mbar_init(&bars[s], 1);
    fence_barrier_init();
  }
  __syncwarp();

  const T *kpool = reinterpret_cast<const T *>(p.k_pool);
  const T *vpool = reinterpret_cast<const T *>(p.v_pool);

  // Producer (lane 0): fill stage s with the page the walker points at. The word of the next
  // page to issue is loaded one issue ahead, so its latency never stalls the warp.
  Walker prod;
  prod.init(x0, p.cu_pages, B, HV);
  uint64_t w_next = 0;
  if (lane == 0) w_next = p.words[prod.wbase + prod.pg];
  auto issue = [&](int s) {
    const uint64_t w = w_next;
    uint32_t blk = word_block(w);
    if (blk >= (uint32_t)p.num_blocks || word_nvalid(w) > (uint32_t)kPage) {
      set_error(p.err, LAZY_DEVERR_BAD_PAGE);
      blk = 0;
    }
    meta_w[s] = w;
    meta_u[s] = prod.b * HV + prod.hv;
    const size_t page =
        ((size_t)blk * p.hkv + kv_head_of(prod.hv, p.chunks)) * (size_t)(kPage * D);
    mbar_arrive_expect_tx(&bars[s], 2u * S::kPageBytes);
    bulk_g2s(kbuf + s * kPage * D, kpool + page, S::kPageBytes, &bars[s]);
    bulk_g2s(vbuf + s * kPage * D, vpool + page, S::kPageBytes, &bars[s]);
  };
  int64_t issued = 0;
  auto issue_next = [&](int s) {
    if (lane == 0) issue(s);
    prod.advance(p.cu_pages, B, HV);
    ++issued;
    if (lane == 0 && issued < n_mine) w_next = p.words[prod.wbase + prod.pg];
  };
  for (int s = 0; s < STAGES && s < n_mine; ++s) issue_next(s);

  const int gq = lane / LPR, r = lane % LPR;
  float2 qr[GC][EP2];    // rotated query slice, pre-scaled by sm_scale * log2(e)
  float2 acc[GC][EP2];   // unnormalised output slice
  float m_run[GC], lsum[GC];
  float sl2[GC];         // ALiBi: the unit's query-head slopes, times log2(e)
  const bool alibi = p.slopes != nullptr;
  int32_t cur_unit = -1, cur_b = 0;
  uint32_t cur_off = 0xFFFFFFFFu;
  int32_t m_pos = 0;
  bool timed_out = false;

  auto flush = [&](int32_t unit) {
    // Sum the KPI key groups, then lanes of group 0 write this piece's partial.
#pragma unroll
    for (int mk = LPR; mk < 32; mk <<= 1) {
#pragma unroll
      for (int g = 0; g < GC; ++g) {
        lsum[g] += __shfl_xor_sync(0xffffffffu, lsum[g], mk);
#pragma unroll
        for (int e = 0; e < EP2; ++e) {
          acc[g][e].x += __shfl_xor_sync(0xffffffffu, acc[g][e].x, mk);
          acc[g][e].y += __shfl_xor_sync(0xffffffffu, acc[g][e].y, mk);
        }
      }
    }
    const int64_t slot = (int64_t)unit + wg;
    if (gq == 0) {
#pragma unroll
      for (int g = 0; g < GC; ++g) {
        const float inv = lsum[g] > 0.f ? 1.f / lsum[g] : 0.f;
        float *dst = p.ws_o + ((size_t)slot * GC + g) * D + r * EPL;
#pragma unroll
        for (int e = 0; e < EP2; e += 2)
          *reinterpret_cast<float4 *>(dst + 2 * e) =
              make_float4(acc[g][e].x * inv, acc[g][e].y * inv, acc[g][e + 1].x * inv,
                          acc[g][e + 1].y * inv);
      }
    }
    if (lane == 0) {
#pragma unroll
      for (int g = 0; g < GC; ++g)
        p.ws_lse[(size_t)slot * GC + g] = lsum[g] > 0.f ? m_run[g] + log2f(lsum[g]) : -INFINITY;
    }
  };

  for (int64_t i = 0; i < n_mine; ++i) {
    const int s = (int)(i % STAGES);
    const uint32_t par = (uint32_t)((i / STAGES) & 1);
    if (!mbar_wait(&bars[s], par, p.wait_ns)) {
      if (lane == 0) set_error(p.err, LAZY_DEVERR_TIMEOUT);
      timed_out = true;
      // Drain the copies still in flight into this warp's stages (bounded), then stop.
      const int64_t last = (i + STAGES < n_mine) ? i + STAGES : n_mine;
      for (int64_t k = i; k < last; ++k)
        mbar_wait(&bars[k % STAGES], (uint32_t)((k / STAGES) & 1), p.wait_ns);
      break;
    }
    const uint64_t word = meta_w[s];
    const int32_t unit = meta_u[s];
    if (unit != cur_unit) {
      if (cur_unit >= 0) flush(cur_unit);
      cur_unit = unit;
      cur_b = unit / HV;
      const int32_t hv = unit % HV;
      m_pos = p.q_pos[cur_b];
      const T *qsrc = reinterpret_cast<const T *>(p.q) + ((size_t)cur_b * p.hq + hv * GC) * D;
      __syncwarp();
      for (int idx = lane; idx < GC * D; idx += 32) qraw[idx] = Elem<T>::to_f(qsrc[idx]);
      __syncwarp();
#pragma unroll
      for (int g = 0; g < GC; ++g) {
        sl2[g] = alibi ? p.slopes[hv * GC + g] * 1.4426950408889634f : 0.f;
        m_run[g] = -INFINITY;
        lsum[g] = 0.f;
#pragma unroll
        for (int e = 0; e < EP2; ++e) acc[g][e] = make_float2(0.f, 0.f);
      }
      cur_off = 0xFFFFFFFFu;
    }
    const uint32_t nv = word_nvalid(word);
    const bool bad = word_block(word) >= (uint32_t)p.num_blocks || nv > (uint32_t)kPage;
    const uint32_t off = word_offset(word);
    // ALiBi pools rotate nothing: q is only scaled, once per unit (delta 0 is the identity).
    const uint32_t rot_off = alibi ? 0u : off;
    if (!bad) {
      if (rot_off != cur_off) {
        // q <- R(m - o) q: the one rotation per document boundary.
        cur_off = rot_off;
        const int64_t delta = alibi ? 0 : (int64_t)m_pos - (int64_t)off;
#pragma unroll
        for (int e = 0; e < EPL; ++e) {
          const int d = r * EPL + e;
          const int i2 = d % (D / 2);
          const int pd = d < D / 2 ? d + D / 2 : d - D / 2;
          float cs, sn;
          rope_cos_sin(delta, p.turn[i2], cs, sn);
#pragma unroll
          for (int g = 0; g < GC; ++g) {
            const float x = qraw[g * D + d], y = qraw[g * D + pd];
            const float rot = (d < D / 2 ? x * cs - y * sn : y * sn + x * cs) * p.scale_log2;
            if (e & 1) qr[g][e / 2].y = rot; else qr[g][e / 2].x = rot;
          }
        }
      }
      const T *K = kbuf + s * kPage * D;
      const T *V = vbuf + s * kPage * D;
      // ---- scores: partial dots over this lane's 16 bytes of each key row (packed f32x2 FMA)
      float part[NV0];
#pragma unroll
      for (int it = 0; it < NIT; ++it) {
        float kf[EPL];
        unpack16<T>(*reinterpret_cast<const uint4 *>(K + (it * KPI + gq) * D + r * EPL), kf);
#pragma unroll
        for (int g = 0; g < GC; ++g) {
          float2 a = make_float2(0.f, 0.f);
#pragma unroll
          for (int e = 0; e < EP2; ++e)
            a = __ffma2_rn(qr[g][e], make_float2(kf[2 * e], kf[2 * e + 1]), a);
          part[it * GC + g] = a.x + a.y;
        }
      }
      int base = 0;
      reduce_scatter<NV0, LPR / 2>(part, lane, base);
      // part[0..NF) hold full (log2-domain) scores of flat indices base .. base+NF-1,
      // index = it * GC + g  ->  key it * KPI + gq, head g.
      if (alibi) {
        // bias slope * (n - m); the word's offset is the page's first position, n - m exact
#pragma unroll
        for (int j = 0; j < NF; ++j) {
          const int idx = base + j;
          const int g = idx % GC;
          float sg = 0.f;
#pragma unroll
          for (int gg = 0; gg < GC; ++gg)
            if (gg == g) sg = sl2[gg];
          part[j] = fmaf(sg, (float)((int32_t)off + (idx / GC) * KPI + gq - m_pos), part[j]);
        }
      }
      if (nv < (uint32_t)kPage) {
#pragma unroll
        for (int j = 0; j < NF; ++j)
          if (((base + j) / GC) * KPI + gq >= (int)nv) part[j] = -INFINITY;
      }
      // The running max only moves when some score exceeds it (rare after the first pages):
      // a warp vote skips the butterfly otherwise.
      bool above = false;
#pragma unroll
      for (int j = 0; j < NF; ++j) {
        const int g = (base + j) % GC;
#pragma unroll
        for (int gg = 0; gg < GC; ++gg)
          if (gg == g) above |= part[j] > m_run[gg];
      }
      if (__any_sync(0xffffffffu, above)) {
        float pmax[GC];
#pragma unroll
        for (int g = 0; g < GC; ++g) pmax[g] = -INFINITY;
#pragma unroll
        for (int j = 0; j < NF; ++j) {
          const int g = (base + j) % GC;
#pragma unroll
          for (int gg = 0; gg < GC; ++gg)
            if (gg == g) pmax[gg] = fmaxf(pmax[gg], part[j]);
        }
#pragma unroll
        for (int mk = 16; mk >= 1; mk >>= 1)
#pragma unroll
          for (int g = 0; g < GC; ++g)
            pmax[g] = fmaxf(pmax[g], __shfl_xor_sync(0xffffffffu, pmax[g], mk));
#pragma unroll
        for (int g = 0; g < GC; ++g) {
          const float m_new = fmaxf(m_run[g], pmax[g]);
          if (m_new > m_run[g]) {  // identical in every lane
            const float alpha = m_run[g] == -INFINITY ? 0.f : exp2f(m_run[g] - m_new);
            lsum[g] *= alpha;
#pragma unroll
            for (int e = 0; e < EP2; ++e) {
              acc[g][e].x *= alpha;
              acc[g][e].y *= alpha;
            }
            m_run[g] = m_new;
          }
        }
      }
#pragma unroll
      for (int j = 0; j < NF; ++j) {
        const int idx = base + j;
        const int key = (idx / GC) * KPI + gq;
        const int g = idx % GC;
        float mg = 0.f;
#pragma unroll
        for (int gg = 0; gg < GC; ++gg)
          if (gg == g) mg = m_run[gg];
        psm[key * GC + g] = part[j] == -INFINITY ? 0.f : exp2f(part[j] - mg);
      }
      __syncwarp();
      // ---- PV (packed f32x2 FMA); masked keys of a partial page contribute exactly zero
      const bool partial = nv < (uint32_t)kPage;
#pragma unroll
      for (int it = 0; it < NIT; ++it) {
        const int key = it * KPI + gq;
        float vf[EPL];
        unpack16<T>(*reinterpret_cast<const uint4 *>(V + key * D + r * EPL), vf);
        if (partial && key >= (int)nv) {
#pragma unroll
          for (int e = 0; e < EPL; ++e) vf[e] = 0.f;
        }
        float pk[GC];
        if constexpr (GC % 4 == 0) {
#pragma unroll
          for (int g = 0; g < GC; g += 4) {
            const float4 t4 = *reinterpret_cast<const float4 *>(psm + key * GC + g);
            pk[g] = t4.x; pk[g + 1] = t4.y; pk[g + 2] = t4.z; pk[g + 3] = t4.w;
          }
        } else {
#pragma unroll
          for (int g = 0; g < GC; ++g) pk[g] = psm[key * GC + g];
        }
#pragma unroll
        for (int g = 0; g < GC; ++g) {
          lsum[g] += pk[g];
          const float2 pp = make_float2(pk[g], pk[g]);
#pragma unroll
          for (int e = 0; e < EP2; ++e)
            acc[g][e] = __ffma2_rn(pp, make_float2(vf[2 * e], vf[2 * e + 1]), acc[g][e]);
        }
      }
    }
    __syncwarp();
    if (issued < n_mine) issue_next(s);
  }
  cudaTriggerProgrammaticLaunchCompletion();
  if (!timed_out && cur_unit >= 0) flush(cur_unit);
}


// ------------------------------------------------------------------ tensor-core decode (bf16)
// The same flattened warp-granular partition, page ring, partial slots and combine as
// decode_split_kernel, but each page's two small contractions run on the tensor cores with
// warp-level mma.sync (m16n8k16, bf16 operands, fp32 accumulate) instead of ~1000 FMA/shuffle
// instructions per page, which made that kernel issue-bound rather than HBM-bound:
//   S[16 x 16] = Q[16 x 128] . K_page^T   A = the query fragment held in registers,
//                                          B = K page rows via ldmatrix (8 k-steps x 2 n-tiles)
//   O^T[128 x 8] += V_page^T[128 x 16] . P^T[16 x 8]
//                                          A = V page via ldmatrix.trans (8 m-tiles of 16 dims),
//                                          B = P^T, re-packed from the S accumulator registers
//                                          (its layout is already the B fragment's)
// A-operand rows of S: row g < GC holds bf16(q_g), row g + 8 holds bf16(q_g - bf16(q_g)), so
// the S accumulator's rows g and g + 8 - registers of the same thread - add up to the score of
// a query with ~16 mantissa bits, as accurate as the fp32 path. Rows >= GC are zero; their P
// columns feed O^T columns that are never written out. Pages arrive by TMA (one copy each for K and V; in shared memory two 16 x 64
// boxes with 128-byte swizzle), so the ldmatrix row reads are bank-conflict free. One copy per
// page rather than one per box: the issuing warp is latency-bound at three warps per scheduler,
// and fewer copy instructions shorten its per-page chain (on decode_b64 -6% instructions,
// -4.6% time against four 2-D boxes).
struct MmaDecodeParams {
  DecodeParams d;
  CUtensorMap tm_k, tm_v;  // 3-D page views (64 dims, pool rows, 2 halves), box 64 x 16 x 2
};

constexpr int kMmaStageBytes = 8192;  // K page (2 x 2 KB boxes) + V page (2 x 2 KB boxes)

template <int STAGES>
struct MmaSmem {
  static constexpr int kStage = 0;                                  // STAGES x 8 KB, 1024-aligned
  static constexpr int kBar = kStage + STAGES * kMmaStageBytes;     // uint64 [STAGES]
  static constexpr int kWord = kBar + STAGES * 8;                   // uint64 [STAGES]
  static constexpr int kUnit = kWord + STAGES * 8;                  // int32 [STAGES]
  static constexpr int kBytes = ((kUnit + STAGES * 4) + 1023) / 1024 * 1024;  // per warp
};

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4],
                                               uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                        uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                          uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
// One whole page (pool rows y .. y + 15, both 64-dim halves) through a 3-D page view.
__device__ __forceinline__ void tma_page_g2s(void *dst, const CUtensorMap *m, int y,
                                             uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, "
      "{%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
      "l"((uint64_t)m), "r"(0), "r"(y), "r"(0), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&h);
}
// Shared-memory address of 16-byte chunk `chunk` (0..15 over the 128 dims) of page row `row`
// (0..15) in a page stored as two 16 x 64 boxes with 128-byte swizzle.
__device__ __forceinline__ uint32_t page_chunk(uint32_t page, int row, int chunk) {
  return page + (chunk >> 3) * 2048 + row * 128 + (((chunk & 7) ^ (row & 7)) << 4);
}

// 2^x in one MUFU instruction (arguments <= 0 here; the weights are rounded to bf16 next).
__device__ __forceinline__ float ex2_fast(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Per-warp attention state of the tensor-core decode over one unit (request, virtual head), or
// in the shared-segment decode over one (segment unit, kv head) whose fragment rows 0-3 and
// 4-7 belong to two requests. Everything but the page words is per row, so each thread keeps
// its own row's position, rotation offset and softmax state. `word` in mma_attend_page is the
// thread's row's page word (the same block for every live row).
template <int GC>
struct MmaWarpState {
  uint32_t qa[8][4];  // A fragments of the rotated, scaled query (hi rows g, lo rows g + 8)
  // This thread's raw query pairs (dims 16ks + 2t + {0,1} and {8,9} at words 8ks and 8ks + 4);
  // null for a dead row. Read from global memory at each rotation rather than kept in 16
  // registers for the whole page loop: the loop runs at the register limit, and those 16
  // registers made long decode 6% slower.
  const uint32_t *qsrc;
  // O transposed, O^T = V^T P^T (dims x heads): o[mt] holds dims 16 mt + g and 16 mt + g + 8
  // of heads 2t and 2t + 1 (registers 0, 1: dim 16 mt + g; 2, 3: dim 16 mt + g + 8)
  float o[8][4];
  float m_run, l_run, sl2;
  int32_t m_pos;
  uint32_t cur_off;
  bool live;  // this thread's fragment row is a real query head
};

// Start unit (request b, virtual head hv): raw query rows, ALiBi slopes, empty accumulators.
template <int GC>
__device__ __forceinline__ void mma_begin_unit(MmaWarpState<GC> &st, const DecodeParams &p,
                                               int32_t b, int32_t hv, int lane) {
  constexpr int D = 128;
  const int g = lane >> 2, t = lane & 3;
  const bool live = g < GC;
  st.live = live;
  st.m_pos = p.q_pos[b];
  const __nv_bfloat16 *q = reinterpret_cast<const __nv_bfloat16 *>(p.q) +
                           ((size_t)b * p.hq + hv * GC + (live ? g : 0)) * D + 2 * t;
  st.qsrc = live ? reinterpret_cast<const uint32_t *>(q) : nullptr;
  st.sl2 = (p.slopes != nullptr && live) ? p.slopes[hv * GC + g] * 1.4426950408889634f : 0.f;
  st.m_run = -INFINITY;
  st.l_run = 0.f;
#pragma unroll
  for (int mt = 0; mt < 8; ++mt)
#pragma unroll
    for (int e = 0; e < 4; ++e) st.o[mt][e] = 0.f;
  st.cur_off = 0xFFFFFFFFu;
}

// One 16-key page (K at page_smem, V 4 KB after it): S = Q K^T, online softmax,
// O^T += V^T P^T.
// kSameDelta: every row of the warp has the same query position and page word (one request per
// warp), so the 64 angles of a query rotation are evaluated once per warp rather than per row.
template <int GC, bool kSameDelta = false>
__device__ __forceinline__ void mma_attend_page(MmaWarpState<GC> &st, const DecodeParams &p,
                                                uint64_t word, uint32_t page_smem, int lane) {
  const int t = lane & 3;  // fragment column pair
  const bool alibi = p.slopes != nullptr;
  const uint32_t nv = word_nvalid(word);
  // The page's MMAs are warp-collective: a bad word in any row skips the page for the warp,
  // and is reported (the producer also reports the word it loads).
  const bool bad = __any_sync(0xffffffffu, word_block(word) >= (uint32_t)p.num_blocks ||
                                               nv > (uint32_t)kPage);
  if (bad && lane == 0) set_error(p.err, LAZY_DEVERR_BAD_PAGE);
  const uint32_t off = word_offset(word);
  const uint32_t rot_off = alibi ? 0u : off;
  if (!bad) {
    if (rot_off != st.cur_off) {
      // q <- R(m - o) q (identity for ALiBi), scaled into the log2 domain, split hi + lo
      st.cur_off = rot_off;
      const int64_t delta = alibi ? 0 : (int64_t)st.m_pos - (int64_t)off;
      // kSameDelta: lane l evaluates rotation pairs l and l + 32; each thread then fetches its
      // 16 pairs from the lanes that own them
      uint32_t qraw[16];
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        qraw[2 * ks] = st.qsrc ? st.qsrc[8 * ks] : 0u;
        qraw[2 * ks + 1] = st.qsrc ? st.qsrc[8 * ks + 4] : 0u;
      }
      float c_lo = 0.f, s_lo = 0.f, c_hi = 0.f, s_hi = 0.f;
      if constexpr (kSameDelta) {
        rope_cos_sin(delta, p.turn[lane], c_lo, s_lo);
        rope_cos_sin(delta, p.turn[lane + 32], c_hi, s_hi);
      }
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {  // dims d < 64 pair with d + 64 (k-step ks + 4)
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          const uint32_t lo_raw = qraw[2 * ks + h2], hi_raw = qraw[2 * (ks + 4) + h2];
          float x[2], y[2];
          x[0] = __uint_as_float(lo_raw << 16);
          x[1] = __uint_as_float(lo_raw & 0xFFFF0000u);
          y[0] = __uint_as_float(hi_raw << 16);
          y[1] = __uint_as_float(hi_raw & 0xFFFF0000u);
          float rx[2], ry[2];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int d = 16 * ks + 8 * h2 + 2 * t + e;
            float cs, sn;
            if constexpr (kSameDelta) {
              cs = __shfl_sync(0xffffffffu, ks >= 2 ? c_hi : c_lo, d & 31);
              sn = __shfl_sync(0xffffffffu, ks >= 2 ? s_hi : s_lo, d & 31);
            } else {
              rope_cos_sin(delta, p.turn[d], cs, sn);
            }
            rx[e] = (x[e] * cs - y[e] * sn) * p.scale_log2;
            ry[e] = (x[e] * sn + y[e] * cs) * p.scale_log2;
          }
          const uint32_t xh = pack_bf16x2(rx[0], rx[1]), yh = pack_bf16x2(ry[0], ry[1]);
          const uint32_t xl = pack_bf16x2(rx[0] - __uint_as_float(xh << 16),
                                          rx[1] - __uint_as_float(xh & 0xFFFF0000u));
          const uint32_t yl = pack_bf16x2(ry[0] - __uint_as_float(yh << 16),
                                          ry[1] - __uint_as_float(yh & 0xFFFF0000u));
          // fragment registers: [0] row g cols 2t.., [1] row g+8, [2] row g cols 2t+8..,
          // [3] row g+8 cols 2t+8.. (a dead row's raw query is 0, so its fragments are 0)
          st.qa[ks][2 * h2] = xh;
          st.qa[ks][2 * h2 + 1] = xl;
          st.qa[ks + 4][2 * h2] = yh;
          st.qa[ks + 4][2 * h2 + 1] = yl;
        }
      }
    }
    const uint32_t kpg = page_smem;
    const uint32_t vpg = kpg + 4096;
    // ---- S = Q K^T: ldmatrix matrix j = lane / 8 covers keys 8 (j >> 1) .. +7 and
    // dims 16 ks + 8 (j & 1) .. +7; row = lane % 8
    float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    const int lrow = ((lane >> 4) << 3) + (lane & 7), lhalf = (lane >> 3) & 1;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      uint32_t b0, b1, b2, b3;
      ldsm_x4(page_chunk(kpg, lrow, 2 * ks + lhalf), b0, b1, b2, b3);
      mma_bf16_16816(sc[0], st.qa[ks], b0, b1);
      mma_bf16_16816(sc[1], st.qa[ks], b2, b3);
    }
    // scores of keys 2t, 2t+1 (n-tile 0) and 8+2t, 9+2t (n-tile 1): hi row + lo row
    float sv[4] = {sc[0][0] + sc[0][2], sc[0][1] + sc[0][3], sc[1][0] + sc[1][2],
                   sc[1][1] + sc[1][3]};
    if (alibi) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int key = (e >> 1) * 8 + 2 * t + (e & 1);
        sv[e] = fmaf(st.sl2, (float)((int32_t)off + key - st.m_pos), sv[e]);
      }
    }
    // Keys past the page's valid count are masked. Dead rows (q = 0) are left unmasked: their
    // scores stay finite and their results are never written out.
    if (nv < (uint32_t)kPage) {
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if ((e >> 1) * 8 + 2 * t + (e & 1) >= (int)nv) sv[e] = -INFINITY;
    }
    float pm = fmaxf(fmaxf(sv[0], sv[1]), fmaxf(sv[2], sv[3]));
    pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, 1));
    pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, 2));
    float alpha = 1.f;  // the same in the 4 lanes of a row
    if (pm > st.m_run) {
      alpha = st.m_run == -INFINITY ? 0.f : ex2_fast(st.m_run - pm);
      st.l_run *= alpha;
      st.m_run = pm;
    }
    // O^T's columns are heads 2t and 2t + 1: their factors come from the lanes of those rows
    if (__any_sync(0xffffffffu, alpha != 1.f)) {
      const float a0 = __shfl_sync(0xffffffffu, alpha, 8 * t);
      const float a1 = __shfl_sync(0xffffffffu, alpha, 8 * t + 4);
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        st.o[mt][0] *= a0;
        st.o[mt][1] *= a1;
        st.o[mt][2] *= a0;
        st.o[mt][3] *= a1;
      }
    }
    float pv[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      pv[e] = ex2_fast(sv[e] - st.m_run);  // m_run is finite (key 0 is valid): exp2(-inf) = 0
      st.l_run += pv[e];
    }
    // ---- O^T += V^T P^T (M = 16 dims, N = 8 heads, K = 16 keys). P^T as the B operand is the
    // S accumulator's layout as it stands: keys 2t, 2t+1 and 2t+8, 2t+9 of head g. A = V^T:
    // ldmatrix.trans matrix j covers keys 8 (j >> 1) .. +7 and dims 16 mt + 8 (j & 1) .. +7.
    // 8 MMAs per page, against 16 for O = P V with its 8 idle rows.
    const uint32_t pb0 = pack_bf16x2(pv[0], pv[1]), pb1 = pack_bf16x2(pv[2], pv[3]);
    const int vrow = ((lane >> 4) << 3) + (lane & 7), vhalf = (lane >> 3) & 1;
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      uint32_t va[4];
      ldsm_x4_t(page_chunk(vpg, vrow, 2 * mt + vhalf), va[0], va[1], va[2], va[3]);
      mma_bf16_16816(st.o[mt], va, pb0, pb1);
    }
  }
}

// The unit's partial (o / l, log2-sum-exp) to workspace slot `slot`.
template <int GC>
__device__ __forceinline__ void mma_flush(MmaWarpState<GC> &st, const DecodeParams &p,
                                          int64_t slot, int lane) {
  constexpr int D = 128;
  const int g = lane >> 2, t = lane & 3;
  float l = st.l_run;
  l += __shfl_xor_sync(0xffffffffu, l, 1);
  l += __shfl_xor_sync(0xffffffffu, l, 2);
  // this thread's O^T columns are heads h0 = 2t and h0 + 1: their sums and liveness come from
  // the lanes of those rows (nobody reads a dead row's slot)
  const int h0 = 2 * t;
  const float l0 = __shfl_sync(0xffffffffu, l, 8 * t), l1 = __shfl_sync(0xffffffffu, l, 8 * t + 4);
  const bool live0 = __shfl_sync(0xffffffffu, (int)st.live, 8 * t) != 0 && h0 < GC;
  const bool live1 = __shfl_sync(0xffffffffu, (int)st.live, 8 * t + 4) != 0 && h0 + 1 < GC;
  const float inv0 = l0 > 0.f ? 1.f / l0 : 0.f, inv1 = l1 > 0.f ? 1.f / l1 : 0.f;
  float *dst0 = p.ws_o + ((size_t)slot * GC + h0) * D + g;
  float *dst1 = dst0 + D;
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) {
    if (live0) {
      dst0[16 * mt] = st.o[mt][0] * inv0;
      dst0[16 * mt + 8] = st.o[mt][2] * inv0;
    }
    if (live1) {
      dst1[16 * mt] = st.o[mt][1] * inv1;
      dst1[16 * mt + 8] = st.o[mt][3] * inv1;
    }
  }
  if (g < GC && st.live && t == 0)
    p.ws_lse[(size_t)slot * GC + g] = l > 0.f ? st.m_run + log2f(l) : -INFINITY;
}

// Loads page word w of the tensor-core kernels into stage `st` (K and V, one page-view copy
// each, landing as two 16 x 64 boxes). A word whose block is out of range loads block 0; the
// consumer's warp vote on the same word skips that page and reports it.
__device__ __forceinline__ void mma_issue_page(const MmaDecodeParams &mp, uint64_t w,
                                               int32_t kv_head, uint8_t *st, uint64_t *bar) {
  const DecodeParams &p = mp.d;
  const uint32_t blk = word_block(w) < (uint32_t)p.num_blocks ? word_block(w) : 0u;
  const int row = (int)((blk * (uint32_t)p.hkv + (uint32_t)kv_head) * kPage);
  mbar_arrive_expect_tx(bar, kMmaStageBytes);
  tma_page_g2s(st, &mp.tm_k, row, bar);
  tma_page_g2s(st + 4096, &mp.tm_v, row, bar);
}

template <int GC, int WARPS, int STAGES>
__global__ void __launch_bounds__(WARPS * 32)
    decode_mma_kernel(const __grid_constant__ MmaDecodeParams mp) {
  using S = MmaSmem<STAGES>;
  static_assert(GC >= 1 && GC <= 8, "a 16-row fragment holds up to 8 heads (hi and lo rows)");
  const DecodeParams &p = mp.d;

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint8_t *base = reinterpret_cast<uint8_t *>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t *ws = base + warp * S::kBytes;
  uint8_t *stage = ws + S::kStage;
  uint64_t *bars = reinterpret_cast<uint64_t *>(ws + S::kBar);
  uint64_t *meta_w = reinterpret_cast<uint64_t *>(ws + S::kWord);
  int32_t *meta_u = reinterpret_cast<int32_t *>(ws + S::kUnit);

  cudaGridDependencySynchronize();
  const int32_t B = p.batch, HV = p.hv;
  const int64_t N = (int64_t)HV * p.cu_pages[B];
  const int64_t WT = (int64_t)gridDim.x * WARPS;
  const int64_t wg = (int64_t)blockIdx.x * WARPS + warp;
  const int64_t x0 = wg * N / WT, x1 = (wg + 1) * N / WT;
  if (x0 >= x1) {
    cudaTriggerProgrammaticLaunchCompletion();
    return;
  }
  if (lane == 0) {
    for (int s = 0; s < STAGES; ++s) mbar_init(&bars[s], 1);
    fence_barrier_init();
  }
  __syncwarp();

  Walker prod;
  prod.init(x0, p.cu_pages, B, HV);
  uint64_t w_next = 0;
  if (lane == 0) w_next = p.words[prod.wbase + prod.pg];
  // 32-bit page counters (64-bit ones cost ~3% here): decode_grid gives every launch at least
  // as many warps as virtual heads, so a warp's range is shorter than the page table (< 2^31)
  const int32_t n_mine = (int32_t)(x1 - x0);
  int32_t issued = 0;
  auto issue_next = [&](int s) {
    if (lane == 0) {
      meta_w[s] = w_next;
      meta_u[s] = prod.b * HV + prod.hv;
      mma_issue_page(mp, w_next, kv_head_of(prod.hv, p.chunks), stage + s * kMmaStageBytes,
                     &bars[s]);
    }
    prod.advance(p.cu_pages, B, HV);
    ++issued;
    if (lane == 0 && issued < n_mine) w_next = p.words[prod.wbase + prod.pg];
  };
  for (int s = 0; s < STAGES && s < n_mine; ++s) issue_next(s);

  MmaWarpState<GC> st;
  int32_t cur_unit = -1;
  bool timed_out = false;
  for (int32_t i = 0; i < n_mine; ++i) {
    const int s = i % STAGES;
    const uint32_t par = (uint32_t)((i / STAGES) & 1);
    if (!mbar_wait(&bars[s], par, p.wait_ns)) {
      if (lane == 0) set_error(p.err, LAZY_DEVERR_TIMEOUT);
      timed_out = true;
      const int32_t last = (i + STAGES < n_mine) ? i + STAGES : n_mine;
      for (int32_t k = i; k < last; ++k)
        mbar_wait(&bars[k % STAGES], (uint32_t)((k / STAGES) & 1), p.wait_ns);
      break;
    }
    const uint64_t word = meta_w[s];
    const int32_t unit = meta_u[s];
    if (unit != cur_unit) {
      if (cur_unit >= 0) mma_flush(st, p, (int64_t)cur_unit + wg, lane);
      cur_unit = unit;
      mma_begin_unit(st, p, unit / HV, unit % HV, lane);
    }
    mma_attend_page<GC, true>(st, p, word, smem_u32(stage + s * kMmaStageBytes), lane);
    __syncwarp();
    if (issued < n_mine) issue_next(s);
  }
  cudaTriggerProgrammaticLaunchCompletion();
  if (!timed_out && cur_unit >= 0) mma_flush(st, p, (int64_t)cur_unit + wg, lane);
}

// Groups of more than 8 query heads per kv head (chunks == WARPS, e.g. MQA 32/1): the CTA's
// warps are the chunks of one kv head and share one page ring, so each K/V page is loaded into
// shared memory once for all of them instead of once per chunk. Units are (request, kv head);
// the flattened (request, kv head, page) sequence is cut into equal ranges, one per CTA. Warp 0
// lane 0 issues; a stage is refilled once every warp has arrived on its empty barrier. Warp w
// leaves its partial of virtual head kv head * WARPS + w at slot (unit + CTA) * WARPS + w.
template <int STAGES>
struct MmaGroupSmem {
  static constexpr int kStage = 0;                                  // STAGES x 8 KB
  static constexpr int kFull = kStage + STAGES * kMmaStageBytes;    // uint64 [STAGES]
  static constexpr int kEmpty = kFull + STAGES * 8;                 // uint64 [STAGES]
  static constexpr int kWord = kEmpty + STAGES * 8;                 // uint64 [STAGES]
  static constexpr int kUnit = kWord + STAGES * 8;                  // int32 [STAGES]
  static constexpr int kBytes = kUnit + STAGES * 4 + 1024;          // + alignment slack
};

template <int GC, int WARPS, int STAGES>
__global__ void __launch_bounds__(WARPS * 32)
    decode_mma_group_kernel(const __grid_constant__ MmaDecodeParams mp) {
  using S = MmaGroupSmem<STAGES>;
  const DecodeParams &p = mp.d;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint8_t *base = reinterpret_cast<uint8_t *>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t *stage = base + S::kStage;
  uint64_t *full = reinterpret_cast<uint64_t *>(base + S::kFull);
  uint64_t *empty = reinterpret_cast<uint64_t *>(base + S::kEmpty);
  uint64_t *meta_w = reinterpret_cast<uint64_t *>(base + S::kWord);
  int32_t *meta_u = reinterpret_cast<int32_t *>(base + S::kUnit);

  cudaGridDependencySynchronize();
  const int32_t B = p.batch, HU = p.hkv;  // units: (request, kv head)
  const int64_t N = (int64_t)HU * p.cu_pages[B];
  const int64_t CT = gridDim.x, cg = blockIdx.x;
  const int64_t x0 = cg * N / CT, x1 = (cg + 1) * N / CT;
  if (x0 >= x1) {  // the whole CTA has no pages
    cudaTriggerProgrammaticLaunchCompletion();
    return;
  }
  const int64_t n_mine = x1 - x0;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], WARPS);
    }
    fence_barrier_init();
  }
  __syncthreads();

  // producer state (warp 0)
  Walker prod;
  uint64_t w_next = 0;
  int64_t issued = 0;
  if (warp == 0) {
    prod.init(x0, p.cu_pages, B, HU);
    if (lane == 0) w_next = p.words[prod.wbase + prod.pg];
  }
  auto issue_next = [&](int s) {
    if (lane == 0) {
      meta_w[s] = w_next;
      meta_u[s] = prod.b * HU + prod.hv;
      mma_issue_page(mp, w_next, prod.hv, stage + s * kMmaStageBytes, &full[s]);
    }
    prod.advance(p.cu_pages, B, HU);
    ++issued;
    if (lane == 0 && issued < n_mine) w_next = p.words[prod.wbase + prod.pg];
  };
  if (warp == 0)
    for (int s = 0; s < STAGES && s < n_mine; ++s) issue_next(s);

  MmaWarpState<GC> st;
  int32_t cur_unit = -1;
  bool timed_out = false;
  for (int64_t i = 0; i < n_mine; ++i) {
    const int s = (int)(i % STAGES);
    const uint32_t par = (uint32_t)((i / STAGES) & 1);
    if (!mbar_wait(&full[s], par, p.wait_ns)) {
      if (lane == 0) set_error(p.err, LAZY_DEVERR_TIMEOUT);
      timed_out = true;
      break;
    }
    const uint64_t word = meta_w[s];
    const int32_t unit = meta_u[s];
    if (unit != cur_unit) {
      if (cur_unit >= 0) mma_flush(st, p, ((int64_t)cur_unit + cg) * WARPS + warp, lane);
      cur_unit = unit;
      mma_begin_unit(st, p, unit / HU, (unit % HU) * WARPS + warp, lane);
    }
    mma_attend_page<GC, true>(st, p, word, smem_u32(stage + s * kMmaStageBytes), lane);
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
    if (warp == 0 && issued < n_mine) {
      // every warp is done with this stage before it is refilled
      if (!mbar_wait(&empty[s], par, p.wait_ns)) {
        if (lane == 0) set_error(p.err, LAZY_DEVERR_TIMEOUT);
        timed_out = true;
        break;
      }
      issue_next(s);
    }
  }
  if (warp == 0) {
    // copies still in flight land before the CTA may exit
    for (int64_t k = issued - STAGES; k < issued; ++k)
      if (k >= 0) mbar_wait(&full[k % STAGES], (uint32_t)((k / STAGES) & 1), p.wait_ns);
  }
  cudaTriggerProgrammaticLaunchCompletion();
  if (!timed_out && cur_unit >= 0)
    mma_flush(st, p, ((int64_t)cur_unit + cg) * WARPS + warp, lane);
}

struct CombineParams {
  const float *ws_o;
  const float *ws_lse;
  const int32_t *cu_pages;
  void *out;
  float *lse;
  int32_t batch, hq, hv;
  int64_t warps;  // ranges of the decode launch: its warps, or its CTAs for the group kernel
  int32_t ch;     // virtual heads sharing one range (the group kernel's warps), else 1
};

// One CTA per unit: merges the unit's pieces (slots unit + w for the warps w whose ranges
// intersect it) with a log-sum-exp combine and writes the final rows. One thread per (head,
// 4-dim group) of the unit (combine_threads), so that each thread makes one pass: with 8 heads
// per unit (MQA's chunks) two passes on 128 threads took 8 us of a 47 us call.
template <int GC, int D>
constexpr int combine_threads() {
  return GC * (D / 4) < 32 ? 32 : (GC * (D / 4) > 256 ? 256 : GC * (D / 4));
}
template <typename T, int D, int GC>
__global__ void __launch_bounds__(combine_threads<GC, D>()) combine_kernel(const CombineParams p) {
  // The piece range comes from the page table, an input of the decode step: it is read while
  // the decode kernel launched just before still runs, and only the partials wait for it.
  const int32_t u = blockIdx.x;
  const int32_t b = u / p.hv, hv = u % p.hv;
  // the partition's units: (request, virtual head), or (request, kv head) shared by ch chunks
  const int32_t hu = p.hv / p.ch, kv = hv / p.ch, chunk = hv % p.ch;
  const int32_t ub = b * hu + kv;
  const int32_t wbase = p.cu_pages[b], np = p.cu_pages[b + 1] - wbase;
  const int64_t N = (int64_t)hu * p.cu_pages[p.batch];
  const int64_t W = p.warps;
  T *out = reinterpret_cast<T *>(p.out);
  // The unit's pieces. With at least one page per warp (N >= W) every warp range is non-empty
  // and the pieces are the warps wf..wl whose ranges meet the unit. With fewer pages than warps
  // each non-empty range holds exactly one page, so the pieces are the unit's np pages, page x
  // (flattened index) in the range of warp ceil((x + 1) W / N) - 1: walking the pages instead of
  // the warps skips the empty ranges without testing them.
  const bool dense = N >= W;
  int64_t wf = 0, S = 0;
  int64_t n_pieces = 0;
  if (np > 0) {
    S = (int64_t)hu * wbase + (int64_t)kv * np;
    const int64_t E = S + np;
    wf = ((S + 1) * W + N - 1) / N - 1;
    n_pieces = dense ? (E * W + N - 1) / N - 1 - wf + 1 : np;
  }
  cudaGridDependencySynchronize();  // the decode kernel's partials
  for (int idx = threadIdx.x; idx < GC * (D / 4); idx += blockDim.x) {
    const int g = idx / (D / 4), d4 = idx % (D / 4);
    // one online pass over the unit's slots, eight at a time with their loads issued together
    float mx = -INFINITY, sum = 0.f;
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int64_t k0 = 0; k0 < n_pieces; k0 += 8) {
      float lv[8];
      float4 ov[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const bool use = k0 + k < n_pieces;
        const int64_t w = dense ? wf + k0 + k : ((S + k0 + k + 1) * W + N - 1) / N - 1;
        const size_t slot = (size_t)(ub + w) * p.ch + chunk;
        lv[k] = use ? p.ws_lse[slot * GC + g] : -INFINITY;
        ov[k] = use ? *reinterpret_cast<const float4 *>(p.ws_o + (slot * GC + g) * D + d4 * 4)
                    : make_float4(0.f, 0.f, 0.f, 0.f);
      }
      float bm = lv[0];
#pragma unroll
      for (int k = 1; k < 8; ++k) bm = fmaxf(bm, lv[k]);
      if (bm == -INFINITY) continue;
      const float nm = fmaxf(mx, bm);
      const float sc = mx == -INFINITY ? 0.f : exp2f(mx - nm);
      sum *= sc;
      a.x *= sc; a.y *= sc; a.z *= sc; a.w *= sc;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const float wt = lv[k] == -INFINITY ? 0.f : exp2f(lv[k] - nm);
        sum += wt;
        a.x = fmaf(wt, ov[k].x, a.x); a.y = fmaf(wt, ov[k].y, a.y);
        a.z = fmaf(wt, ov[k].z, a.z); a.w = fmaf(wt, ov[k].w, a.w);
      }
      mx = nm;
    }
    const float inv = sum > 0.f ? 1.f / sum : 0.f;
    const int qh = hv * GC + g;
    T *dst = out + ((size_t)b * p.hq + qh) * D + d4 * 4;
    dst[0] = Elem<T>::from_f(a.x * inv);
    dst[1] = Elem<T>::from_f(a.y * inv);
    dst[2] = Elem<T>::from_f(a.z * inv);
    dst[3] = Elem<T>::from_f(a.w * inv);
    if (d4 == 0)
      p.lse[(size_t)b * p.hq + qh] = sum > 0.f ? (mx + __log2f(sum)) * 0.69314718055994531f
                                               : -INFINITY;
  }
}

// ------------------------------------------------------------------------------------------------
// Shared-segment decode. A document cached once sits in many requests' contexts at different
// logical offsets; in the position-agnostic pool its pages are the same blocks for all of them,
// and only the query rotation R(m - o) differs per request. A host plan cuts every request's
// page list into segments (runs of pages with one offset), finds identical segments (the same
// block and valid-count sequence) across requests and pairs them: a pair unit streams the
// segment's pages once, with request A's query heads in fragment rows 0-3 and request B's in
// rows 4-7 (rows the GC = 4 kernel leaves empty), so one page load and one set of MMAs serve both.
// Unpaired segments (and private ones) are single units with rows 4-7 dead.
//   entries      uint64 [2 * n_entries]: (word of A, word of B) per page of a unit; B's word is
//                only read when the unit has a second request
//   cu_entries   int32 [n_units + 1]
//   unit_req     int32 [2 * n_units]: requests A and B (-1: none)
//   cu_members   int32 [batch + 1], members int32: the units of request r as unit * 2 + half
//   member_entries int32 [2 * n_members]: each membership's unit (first entry, entry count)
// ------------------------------------------------------------------------------------------------
struct MmaSharedParams {
  MmaDecodeParams m;
  const uint64_t *entries;
  const int32_t *cu_entries;
  const int32_t *unit_req;
  int32_t n_units;
  int32_t G;  // query heads per kv head (1, 2 or 4)
};

template <int STAGES>
struct MmaSharedSmem {
  static constexpr int kStage = 0;                                  // STAGES x 8 KB, 1024-aligned
  static constexpr int kBar = kStage + STAGES * kMmaStageBytes;     // uint64 [STAGES]
  static constexpr int kWord = kBar + STAGES * 8;                   // uint64 [2 * STAGES]
  static constexpr int kUnit = kWord + STAGES * 16;                 // int32 [STAGES]
  static constexpr int kBytes = ((kUnit + STAGES * 4) + 1023) / 1024 * 1024;  // per warp
};

// Start (segment unit u, kv head h): rows 0-3 take request A's heads h G + r (r < G), rows 4-7
// request B's.
__device__ __forceinline__ void mma_begin_shared_unit(MmaWarpState<8> &st,
                                                      const MmaSharedParams &sp, int32_t u,
                                                      int32_t h, int lane) {
  constexpr int D = 128;
  const DecodeParams &p = sp.m.d;
  const int g = lane >> 2, t = lane & 3;
  const int half = g >> 2, r = g & 3;
  const int32_t req = sp.unit_req[2 * u + half];
  const bool live = r < sp.G && req >= 0;
  st.live = live;
  st.m_pos = live ? p.q_pos[req] : 0;
  const __nv_bfloat16 *q = reinterpret_cast<const __nv_bfloat16 *>(p.q) +
                           ((size_t)(live ? req : 0) * p.hq + h * sp.G + (live ? r : 0)) * D +
                           2 * t;
  st.qsrc = live ? reinterpret_cast<const uint32_t *>(q) : nullptr;
  st.sl2 = (p.slopes != nullptr && live) ? p.slopes[h * sp.G + r] * 1.4426950408889634f : 0.f;
  st.m_run = -INFINITY;
  st.l_run = 0.f;
#pragma unroll
  for (int mt = 0; mt < 8; ++mt)
#pragma unroll
    for (int e = 0; e < 4; ++e) st.o[mt][e] = 0.f;
  st.cur_off = 0xFFFFFFFFu;
}

// The decode_mma_kernel partition over the flattened (unit, kv head, entry) sequence; the
// partial of (unit, kv head) at warp w goes to slot (unit * Hkv + kv head) + w, 8 rows.
template <int WARPS, int STAGES>
__global__ void __launch_bounds__(WARPS * 32)
    decode_shared_kernel(const __grid_constant__ MmaSharedParams sp) {
  using S = MmaSharedSmem<STAGES>;
  const DecodeParams &p = sp.m.d;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint8_t *base = reinterpret_cast<uint8_t *>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t *ws = base + warp * S::kBytes;
  uint8_t *stage = ws + S::kStage;
  uint64_t *bars = reinterpret_cast<uint64_t *>(ws + S::kBar);
  uint64_t *meta_w = reinterpret_cast<uint64_t *>(ws + S::kWord);
  int32_t *meta_u = reinterpret_cast<int32_t *>(ws + S::kUnit);

  cudaGridDependencySynchronize();
  const int32_t NU = sp.n_units, HV = p.hv;
  const int64_t N = (int64_t)HV * sp.cu_entries[NU];
  const int64_t WT = (int64_t)gridDim.x * WARPS;
  const int64_t wg = (int64_t)blockIdx.x * WARPS + warp;
  const int64_t x0 = wg * N / WT, x1 = (wg + 1) * N / WT;
  if (x0 >= x1) {
    cudaTriggerProgrammaticLaunchCompletion();
    return;
  }
  const int64_t n_mine = x1 - x0;
  if (lane == 0) {
    for (int s = 0; s < STAGES; ++s) mbar_init(&bars[s], 1);
    fence_barrier_init();
  }
  __syncwarp();

  Walker prod;
  prod.init(x0, sp.cu_entries, NU, HV);
  uint64_t wa_next = 0, wb_next = 0;
  auto load_entry = [&]() {
    const size_t e = (size_t)prod.wbase + prod.pg;
    wa_next = sp.entries[2 * e];
    wb_next = sp.entries[2 * e + 1];
  };
  if (lane == 0) load_entry();
  int64_t issued = 0;
  auto issue_next = [&](int s) {
    if (lane == 0) {
      meta_w[2 * s] = wa_next;
      meta_w[2 * s + 1] = wb_next;
      meta_u[s] = prod.b * HV + prod.hv;
      mma_issue_page(sp.m, wa_next, prod.hv, stage + s * kMmaStageBytes, &bars[s]);
    }
    prod.advance(sp.cu_entries, NU, HV);
    ++issued;
    if (lane == 0 && issued < n_mine) load_entry();
  };
  for (int s = 0; s < STAGES && s < n_mine; ++s) issue_next(s);

  MmaWarpState<8> st;
  int32_t cur_unit = -1;
  bool timed_out = false;
  const int half = (lane >> 2) >> 2;
  for (int64_t i = 0; i < n_mine; ++i) {
    const int s = (int)(i % STAGES);
    const uint32_t par = (uint32_t)((i / STAGES) & 1);
    if (!mbar_wait(&bars[s], par, p.wait_ns)) {
      if (lane == 0) set_error(p.err, LAZY_DEVERR_TIMEOUT);
      timed_out = true;
      const int64_t last = (i + STAGES < n_mine) ? i + STAGES : n_mine;
      for (int64_t k = i; k < last; ++k)
        mbar_wait(&bars[k % STAGES], (uint32_t)((k / STAGES) & 1), p.wait_ns);
      break;
    }
    const int32_t unit = meta_u[s];
    if (unit != cur_unit) {
      if (cur_unit >= 0) mma_flush(st, p, (int64_t)cur_unit + wg, lane);
      cur_unit = unit;
      mma_begin_shared_unit(st, sp, unit / HV, unit % HV, lane);
    }
    // a dead row's word only feeds the warp-wide bad-page vote and the dead row's own (unused)
    // scores: give it row A's word so that an absent B cannot veto the page. B's word must name
    // the block that was loaded (A's); a plan that pairs different blocks makes it a bad word.
    const uint64_t wa = meta_w[2 * s];
    uint64_t word = wa;
    if (half && st.live) {
      const uint64_t wb = meta_w[2 * s + 1];
      word = word_block(wb) == word_block(wa) ? wb : ~0ull;
    }
    mma_attend_page(st, p, word, smem_u32(stage + s * kMmaStageBytes), lane);
    __syncwarp();
    if (issued < n_mine) issue_next(s);
  }
  cudaTriggerProgrammaticLaunchCompletion();
  if (!timed_out && cur_unit >= 0) mma_flush(st, p, (int64_t)cur_unit + wg, lane);
}

struct SharedCombineParams {
  const float *ws_o;
  const float *ws_lse;
  const int32_t *cu_entries;
  const int32_t *cu_members;
  const int32_t *members;
  const int32_t *member_entries;  // per membership: its unit's (first entry, entry count)
  void *out;
  float *lse;
  int32_t batch, hq, hkv, G, n_units;
  int64_t warps;
};

// One CTA per (request, kv head): one online log-sum-exp pass over the slots of every unit the
// request belongs to (rows half * 4 + r of each), then the final rows. The request's units are
// taken kChunk at a time: their slot ranges are worked out by the CTA's threads in parallel into
// shared memory, and the pass then loads eight slots at a time across unit boundaries.
__global__ void __launch_bounds__(128) combine_shared_kernel(const SharedCombineParams p) {
  constexpr int D = 128, kChunk = 128, kBatch = 16;
  __shared__ int64_t s_first[kChunk];  // dense: slot of the first piece; sparse: first page index
  __shared__ int64_t s_base[kChunk];   // sparse: slot of warp 0 for the unit (unit * hkv + h)
  __shared__ int32_t s_count[kChunk];  // pieces of the unit (0: none)
  __shared__ int32_t s_row[kChunk];
  cudaGridDependencySynchronize();
  const int32_t b = blockIdx.x / p.hkv, h = blockIdx.x % p.hkv;
  const int64_t N = (int64_t)p.hkv * p.cu_entries[p.n_units];
  const int64_t W = p.warps;
  const bool dense = N >= W;
  const int32_t m0 = p.cu_members[b], m1 = p.cu_members[b + 1];
  __nv_bfloat16 *out = reinterpret_cast<__nv_bfloat16 *>(p.out);
  const bool mine = threadIdx.x < p.G * (D / 4);
  const int r = threadIdx.x / (D / 4), d4 = threadIdx.x % (D / 4);
  float mx = -INFINITY, sum = 0.f;
  float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int32_t c0 = m0; c0 < m1; c0 += kChunk) {
    const int32_t nc = min(kChunk, m1 - c0);
    __syncthreads();  // the previous chunk's ranges are no longer read
    for (int i = threadIdx.x; i < nc; i += blockDim.x) {
      const int32_t mem = p.members[c0 + i];
      const int32_t unit = mem >> 1;
      // the unit's entry range, stored with the membership (no dependent load of cu_entries)
      const int32_t ebase = p.member_entries[2 * (c0 + i)];
      const int32_t ne = p.member_entries[2 * (c0 + i) + 1];
      // Pieces as in combine_kernel: the warps meeting the unit's entries (dense), or, with
      // fewer entries than warps, the entries themselves, entry x in warp ceil((x+1) W / N) - 1.
      const int64_t S = (int64_t)p.hkv * ebase + (int64_t)h * ne;
      s_base[i] = (int64_t)unit * p.hkv + h;
      s_row[i] = (mem & 1) * 4;
      if (ne <= 0) {
        s_first[i] = 0;
        s_count[i] = 0;
      } else if (dense) {
        const int64_t wf = ((S + 1) * W + N - 1) / N - 1, wl = ((S + ne) * W + N - 1) / N - 1;
        s_first[i] = s_base[i] + wf;
        s_count[i] = (int32_t)(wl - wf + 1);
      } else {
        s_first[i] = S;
        s_count[i] = ne;
      }
    }
    __syncthreads();
    if (!mine) continue;
    int ci = 0, cw = 0;  // cursor: chunk unit, piece within it
    while (ci < nc) {
      float lv[kBatch];
      float4 ov[kBatch];
#pragma unroll
      for (int k = 0; k < kBatch; ++k) {
        while (ci < nc && cw >= s_count[ci]) {
          ++ci;
          cw = 0;
        }
        const bool use = ci < nc;
        size_t slot = 0;
        int row = 0;
        if (use) {
          slot = dense ? (size_t)(s_first[ci] + cw)
                       : (size_t)(s_base[ci] + ((s_first[ci] + cw + 1) * W + N - 1) / N - 1);
          row = s_row[ci] + r;
          ++cw;
        }
        lv[k] = use ? p.ws_lse[slot * 8 + row] : -INFINITY;
        ov[k] = use ? *reinterpret_cast<const float4 *>(p.ws_o + (slot * 8 + row) * D + d4 * 4)
                    : make_float4(0.f, 0.f, 0.f, 0.f);
      }
      float bm = lv[0];
#pragma unroll
      for (int k = 1; k < kBatch; ++k) bm = fmaxf(bm, lv[k]);
      if (bm == -INFINITY) continue;
      const float nm = fmaxf(mx, bm);
      const float sc = mx == -INFINITY ? 0.f : exp2f(mx - nm);
      sum *= sc;
      a.x *= sc; a.y *= sc; a.z *= sc; a.w *= sc;
#pragma unroll
      for (int k = 0; k < kBatch; ++k) {
        const float wt = lv[k] == -INFINITY ? 0.f : exp2f(lv[k] - nm);
        sum += wt;
        a.x = fmaf(wt, ov[k].x, a.x); a.y = fmaf(wt, ov[k].y, a.y);
        a.z = fmaf(wt, ov[k].z, a.z); a.w = fmaf(wt, ov[k].w, a.w);
      }
      mx = nm;
    }
  }
  if (!mine) return;
  const float inv = sum > 0.f ? 1.f / sum : 0.f;
  const int qh = h * p.G + r;
  __nv_bfloat16 *dst = out + ((size_t)b * p.hq + qh) * D + d4 * 4;
  __nv_bfloat162 v0 = __floats2bfloat162_rn(a.x * inv, a.y * inv);
  __nv_bfloat162 v1 = __floats2bfloat162_rn(a.z * inv, a.w * inv);
  uint2 pk;
  pk.x = *reinterpret_cast<uint32_t *>(&v0);
  pk.y = *reinterpret_cast<uint32_t *>(&v1);
  *reinterpret_cast<uint2 *>(dst) = pk;
  if (d4 == 0)
    p.lse[(size_t)b * p.hq + qh] = sum > 0.f ? (mx + __log2f(sum)) * 0.69314718055994531f
                                             : -INFINITY;
}

constexpr int kWarps = 4;  // warps per CTA of every decode variant

// Two stages (one page in flight while the other is consumed) keep a warp's ring at 16 KB, so
// three 4-warp CTAs fit per SM: 12 warps per SM hide the fixed-latency chains better than
// deeper rings with fewer warps (measured on GB300: 86% vs 75% of copy bandwidth).
constexpr int kStages = 2;

template <typename K, typename... Args>
cudaError_t launch_pdl(K kernel, int grid, int block, int smem, cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// The tensor-core kernel serves bf16 pools with head_dim 128 unless the pool asks for the
// CUDA-core kernel (lazy_pool_set_decode_kernel).
bool use_mma(const lazy_pool *p) {
  return p->decode_kernel != LAZY_DECODE_SIMT && p->dtype == LAZY_DTYPE_BF16 && p->d == 128;
}

constexpr int kGroupStages = 4;  // page ring of the group kernel
constexpr int kGroupSmem = MmaGroupSmem<kGroupStages>::kBytes;

template <int GC, int STAGES>
struct MmaLaunch {
  static constexpr int kSmem = MmaSmem<STAGES>::kBytes * kWarps + 1024;  // + alignment slack
  // groups of 4 chunks of 8 query heads (e.g. MQA 32/1) share one page ring per CTA
  static bool grouped(int32_t chunks) { return GC == 8 && chunks == kWarps; }
  // Occupancy, queried once. The cache is atomic: calls from several threads may run the
  // (idempotent) query concurrently, and each then stores the same value.
  template <typename F>
  static int occupancy(F fn, int smem, std::atomic<int> *cached) {
    int c = cached->load(std::memory_order_acquire);
    if (c < 0) {
      if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
          cudaSuccess)
        return -1;
      int n = 0;
      if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, kWarps * 32, smem) !=
          cudaSuccess)
        return -1;
      c = std::max(1, n);
      cached->store(c, std::memory_order_release);
    }
    return c;
  }
  static int ctas_per_sm(int32_t chunks) {
    static std::atomic<int> cached{-1}, cached_group{-1};
    if constexpr (GC == 8) {
      if (grouped(chunks))
        return occupancy(decode_mma_group_kernel<GC, kWarps, kGroupStages>, kGroupSmem,
                         &cached_group);
    }
    return occupancy(decode_mma_kernel<GC, kWarps, STAGES>, kSmem, &cached);
  }
  static int run(lazy_pool *pl, const DecodeParams &dp, const CombineParams &cp, int grid,
                 cudaStream_t s) {
    int rc = ensure_pool_tmaps(pl);
    if (rc != LAZY_OK) return rc;
    if (ctas_per_sm(dp.chunks) < 0)
      return record_cuda(cudaGetLastError(), "decode_mma_kernel set-up");
    MmaDecodeParams mp;
    mp.d = dp;
    {
      std::lock_guard<std::mutex> g(pl->mu);
      memcpy(&mp.tm_k, pl->tmap_k3, sizeof(CUtensorMap));
      memcpy(&mp.tm_v, pl->tmap_v3, sizeof(CUtensorMap));
    }
    CombineParams c2 = cp;
    bool launched = false;
    if constexpr (GC == 8) {
      if (grouped(dp.chunks)) {
        LAZY_CUDA_TRY(launch_pdl(decode_mma_group_kernel<GC, kWarps, kGroupStages>, grid,
                                 kWarps * 32, kGroupSmem, s, mp));
        c2.warps = grid;  // one range per CTA, shared by its kWarps chunks
        c2.ch = kWarps;
        launched = true;
      }
    }
    if (!launched)
      LAZY_CUDA_TRY(launch_pdl(decode_mma_kernel<GC, kWarps, STAGES>, grid, kWarps * 32, kSmem,
                               s, mp));
    LAZY_CUDA_TRY(launch_pdl(combine_kernel<__nv_bfloat16, 128, GC>, dp.batch * dp.hv,
                             combine_threads<GC, 128>(), 0, s, c2));
    return LAZY_OK;
  }
};

template <typename T, int D, int GC, int STAGES>
struct DecodeLaunch {
  using S = DecodeSmem<T, D, GC, STAGES>;
  static constexpr int kSmem = S::kBytes * kWarps;
  static constexpr bool kHasMma = std::is_same<T, __nv_bfloat16>::value && D == 128;
  static int ctas_per_sm(const lazy_pool *pl, int32_t chunks) {
    if constexpr (kHasMma) {
      if (use_mma(pl)) return MmaLaunch<GC, STAGES>::ctas_per_sm(chunks);
    }
    return simt_ctas_per_sm();
  }
  static int simt_ctas_per_sm() {
    static std::atomic<int> cached{-1};
    return MmaLaunch<GC, STAGES>::occupancy(decode_split_kernel<T, D, GC, kWarps, STAGES>, kSmem,
                                            &cached);
  }
  static int run(lazy_pool *pl, const DecodeParams &dp, const CombineParams &cp, int grid,
                 cudaStream_t s) {
    if constexpr (kHasMma) {
      if (use_mma(pl)) return MmaLaunch<GC, STAGES>::run(pl, dp, cp, grid, s);
    }
    LAZY_CUDA_TRY(launch_pdl(decode_split_kernel<T, D, GC, kWarps, STAGES>, grid, kWarps * 32,
                             kSmem, s, dp));
    LAZY_CUDA_TRY(launch_pdl(combine_kernel<T, D, GC>, dp.batch * dp.hv, combine_threads<GC, D>(),
                             0, s, cp));
    return LAZY_OK;
  }
};

template <typename F>
int with_decode_shape(int32_t dtype, int32_t d, int32_t gc, F &&f) {
#define LAZY_GC_CASES(T, DD)                                        \
  switch (gc) {                                                     \
    case 1: return f(DecodeLaunch<T, DD, 1, kStages>{});            \
    case 2: return f(DecodeLaunch<T, DD, 2, kStages>{});            \
    case 4: return f(DecodeLaunch<T, DD, 4, kStages>{});            \
    case 8: return f(DecodeLaunch<T, DD, 8, kStages>{});            \
    default: return LAZY_ERR_UNSUPPORTED;                           \
  }
  if (dtype == LAZY_DTYPE_BF16) {
    if (d == 128) { LAZY_GC_CASES(__nv_bfloat16, 128) }
    if (d == 64) { LAZY_GC_CASES(__nv_bfloat16, 64) }
  } else {
    if (d == 128) { LAZY_GC_CASES(float, 128) }
    if (d == 64) { LAZY_GC_CASES(float, 64) }
  }
#undef LAZY_GC_CASES
  return LAZY_ERR_UNSUPPORTED;
}

// Query-head chunking: a group of G query heads per kv head runs as ceil(G/8) virtual heads of
// GC = G / chunks heads each (G must split evenly).
int plan_groups(int32_t hq, int32_t hkv, int32_t *gc, int32_t *chunks) {
  if (hq <= 0 || hkv <= 0 || hq % hkv) return LAZY_ERR_INVALID_ARG;
  const int32_t g = hq / hkv;
  int32_t c = 1;
  while (g / c > 8 || g % c) ++c;
  const int32_t per = g / c;
  if (per != 1 && per != 2 && per != 4 && per != 8) return LAZY_ERR_UNSUPPORTED;
  *gc = per;
  *chunks = c;
  return LAZY_OK;
}

// The decode grid: grid_ctas, or one persistent wave, raised to at least one warp per virtual
// head. The tensor-core decode counts a warp's pages in 32 bits: N = virtual heads x pages
// (< 2^31) split over at least virtual-heads warps leaves every range below 2^31.
int decode_grid(lazy_pool *p, int32_t gc, int32_t chunks, int32_t grid_ctas, int *grid) {
  const int min_grid = (p->hkv * chunks + kWarps - 1) / kWarps;
  if (grid_ctas > 0) {
    *grid = std::max<int>(grid_ctas, min_grid);
    return LAZY_OK;
  }
  const int per_sm = with_decode_shape(
      p->dtype, p->d, gc, [&](auto L) { return decltype(L)::ctas_per_sm(p, chunks); });
  if (per_sm <= 0) {
    record_msg("decode kernel occupancy query failed");
    return LAZY_ERR_CUDA;
  }
  *grid = std::max<int>(p->num_sms * per_sm, min_grid);
  return LAZY_OK;
}

constexpr int kSharedSmem = MmaSharedSmem<kStages>::kBytes * kWarps + 1024;  // + alignment slack

// CTAs per SM of the shared-segment decode (occupancy query, once).
int shared_ctas_per_sm() {
  static std::atomic<int> cached{-1};
  return MmaLaunch<4, kStages>::occupancy(decode_shared_kernel<kWarps, kStages>, kSharedSmem,
                                          &cached);
}

// The shared-segment decode serves bf16 pools with head_dim 128 and 1, 2 or 4 query heads per
// kv head (two requests' groups fill the 8 rows of one fragment half each).
int shared_supported(const lazy_pool *p, int32_t hq) {
  if (p->dtype != LAZY_DTYPE_BF16 || p->d != 128 || p->page_size != kPage)
    return LAZY_ERR_UNSUPPORTED;
  if (hq <= 0 || hq % p->hkv) return LAZY_ERR_INVALID_ARG;
  const int32_t g = hq / p->hkv;
  return (g == 1 || g == 2 || g == 4) ? LAZY_OK : LAZY_ERR_UNSUPPORTED;
}

int shared_grid(lazy_pool *p, int32_t grid_ctas, int *grid) {
  if (grid_ctas > 0) {
    *grid = grid_ctas;
    return LAZY_OK;
  }
  const int per_sm = shared_ctas_per_sm();
  if (per_sm <= 0) return record_cuda(cudaGetLastError(), "decode_shared_kernel set-up");
  *grid = p->num_sms * per_sm;
  return LAZY_OK;
}

}  // namespace
}  // namespace lazy

using namespace lazy;

extern "C" int lazy_decode_shared_workspace_bytes(lazy_pool *p, int32_t n_units,
                                                  int32_t num_q_heads, int32_t grid_ctas,
                                                  size_t *bytes) {
  if (!p || !bytes || n_units < 0 || grid_ctas < 0) return LAZY_ERR_INVALID_ARG;
  int rc = shared_supported(p, num_q_heads);
  if (rc != LAZY_OK) return rc;
  rc = ensure_device(p);
  if (rc != LAZY_OK) return rc;
  int grid;
  rc = shared_grid(p, grid_ctas, &grid);
  if (rc != LAZY_OK) return rc;
  const size_t slots = (size_t)n_units * p->hkv + (size_t)grid * kWarps;
  *bytes = slots * 8 * ((size_t)p->d + 1) * sizeof(float) + 256;
  return LAZY_OK;
}

extern "C" int lazy_attn_decode_shared(lazy_pool *p, const void *q, const int32_t *q_pos,
                                       const uint64_t *entries, const int32_t *cu_entries,
                                       const int32_t *unit_req, int32_t n_units,
                                       const int32_t *cu_members, const int32_t *members,
                                       const int32_t *member_entries, int32_t batch, int32_t num_q_heads, float sm_scale,
                                       int32_t grid_ctas, void *out, float *lse, void *workspace,
                                       size_t workspace_bytes, lazy_stream_t stream) {
  if (!p || batch < 0 || n_units < 0 || grid_ctas < 0 || !(sm_scale > 0.f))
    return LAZY_ERR_INVALID_ARG;
  if (batch == 0) return LAZY_OK;
  if (!q || !q_pos || !cu_entries || !cu_members || !out || !lse || !workspace)
    return LAZY_ERR_INVALID_ARG;
  if (n_units > 0 && (!entries || !unit_req || !members || !member_entries))
    return LAZY_ERR_INVALID_ARG;
  if (((uintptr_t)q & 15) || ((uintptr_t)out & 15) || ((uintptr_t)workspace & 15) ||
      ((uintptr_t)entries & 7))
    return LAZY_ERR_INVALID_ARG;
  if (p->alibi && num_q_heads != (int32_t)p->slopes.size()) return LAZY_ERR_INVALID_ARG;
  size_t need = 0;
  int rc = lazy_decode_shared_workspace_bytes(p, n_units, num_q_heads, grid_ctas, &need);
  if (rc != LAZY_OK) return rc;
  if (workspace_bytes < need) return LAZY_ERR_INVALID_ARG;
  rc = ensure_pool_tmaps(p);
  if (rc != LAZY_OK) return rc;
  int grid;
  rc = shared_grid(p, grid_ctas, &grid);
  if (rc != LAZY_OK) return rc;
  const size_t slots = (size_t)n_units * p->hkv + (size_t)grid * kWarps;
  MmaSharedParams sp;
  DecodeParams &dp = sp.m.d;
  memset(&dp, 0, sizeof(dp));
  dp.q = q;
  dp.q_pos = q_pos;
  dp.k_pool = p->k;
  dp.v_pool = p->v;
  dp.turn = p->d_turn;
  dp.ws_o = reinterpret_cast<float *>(workspace);
  dp.ws_lse = dp.ws_o + slots * 8 * p->d;
  dp.err = p->d_err;
  dp.batch = batch;
  dp.hkv = p->hkv;
  dp.hq = num_q_heads;
  dp.num_blocks = p->num_blocks;
  dp.hv = p->hkv;
  dp.chunks = 1;
  dp.scale_log2 = sm_scale * 1.4426950408889634f;
  dp.wait_ns = p->wait_limit_ns;
  dp.slopes = p->alibi ? p->d_slopes : nullptr;
  {
    std::lock_guard<std::mutex> g(p->mu);
    memcpy(&sp.m.tm_k, p->tmap_k3, sizeof(CUtensorMap));
    memcpy(&sp.m.tm_v, p->tmap_v3, sizeof(CUtensorMap));
  }
  sp.entries = entries;
  sp.cu_entries = cu_entries;
  sp.unit_req = unit_req;
  sp.n_units = n_units;
  sp.G = num_q_heads / p->hkv;
  SharedCombineParams cp;
  cp.ws_o = dp.ws_o;
  cp.ws_lse = dp.ws_lse;
  cp.cu_entries = cu_entries;
  cp.cu_members = cu_members;
  cp.members = members;
  cp.member_entries = member_entries;
  cp.out = out;
  cp.lse = lse;
  cp.batch = batch;
  cp.hq = num_q_heads;
  cp.hkv = p->hkv;
  cp.G = sp.G;
  cp.n_units = n_units;
  cp.warps = (int64_t)grid * kWarps;
  cudaStream_t s = (cudaStream_t)stream;
  if (n_units > 0)
    LAZY_CUDA_TRY(launch_pdl(decode_shared_kernel<kWarps, kStages>, grid, kWarps * 32,
                             kSharedSmem, s, sp));
  LAZY_CUDA_TRY(launch_pdl(combine_shared_kernel, batch * p->hkv, 128, 0, s, cp));
  return LAZY_OK;
}

extern "C" int lazy_decode_workspace_bytes(lazy_pool *p, int32_t batch, int32_t num_q_heads,
                                           int32_t grid_ctas, size_t *bytes) {
  if (!p || !bytes || batch < 0 || grid_ctas < 0) return LAZY_ERR_INVALID_ARG;
  if (p->alibi && num_q_heads != (int32_t)p->slopes.size()) return LAZY_ERR_INVALID_ARG;
  int32_t gc, chunks;
  int rc = plan_groups(num_q_heads, p->hkv, &gc, &chunks);
  if (rc != LAZY_OK) return rc;
  rc = ensure_device(p);
  if (rc != LAZY_OK) return rc;
  int grid;
  rc = decode_grid(p, gc, chunks, grid_ctas, &grid);
  if (rc != LAZY_OK) return rc;
  const size_t slots = (size_t)batch * p->hkv * chunks + (size_t)grid * kWarps;
  *bytes = slots * gc * ((size_t)p->d + 1) * sizeof(float) + 256;
  return LAZY_OK;
}

extern "C" int lazy_decode_partition(lazy_pool *p, int32_t num_q_heads, int32_t grid_ctas,
                                     int32_t *units_per_request, int64_t *ranges) {
  if (!p || !units_per_request || !ranges || grid_ctas < 0) return LAZY_ERR_INVALID_ARG;
  int32_t gc, chunks;
  int rc = plan_groups(num_q_heads, p->hkv, &gc, &chunks);
  if (rc != LAZY_OK) return rc;
  rc = ensure_device(p);
  if (rc != LAZY_OK) return rc;
  int grid;
  rc = decode_grid(p, gc, chunks, grid_ctas, &grid);
  if (rc != LAZY_OK) return rc;
  // the group kernel (chunks of 8 heads sharing a CTA's page ring) cuts (request, kv head)
  // units into one range per CTA; every other decode kernel cuts (request, virtual head) units
  // into one range per warp
  const bool grouped = use_mma(p) && gc == 8 && chunks == kWarps;
  *units_per_request = grouped ? p->hkv : p->hkv * chunks;
  *ranges = grouped ? (int64_t)grid : (int64_t)grid * kWarps;
  return LAZY_OK;
}

extern "C" int lazy_attn_decode(lazy_pool *p, const void *q, const int32_t *q_pos,
                                const uint64_t *words, const int32_t *cu_pages, int32_t batch,
                                int32_t num_q_heads, float sm_scale, int32_t grid_ctas, void *out,
                                float *lse, void *workspace, size_t workspace_bytes,
                                lazy_stream_t stream) {
  if (!p || batch < 0 || grid_ctas < 0 || !(sm_scale > 0.f)) return LAZY_ERR_INVALID_ARG;
  if (batch == 0) return LAZY_OK;
  if (!q || !q_pos || !cu_pages || !out || !lse || !workspace) return LAZY_ERR_INVALID_ARG;
  if (((uintptr_t)q & 15) || ((uintptr_t)out & 15) || ((uintptr_t)workspace & 15) ||
      ((uintptr_t)words & 7))
    return LAZY_ERR_INVALID_ARG;
  if (p->alibi && num_q_heads != (int32_t)p->slopes.size()) return LAZY_ERR_INVALID_ARG;
  int32_t gc, chunks;
  int rc = plan_groups(num_q_heads, p->hkv, &gc, &chunks);
  if (rc != LAZY_OK) return rc;
  size_t need = 0;
  rc = lazy_decode_workspace_bytes(p, batch, num_q_heads, grid_ctas, &need);
  if (rc != LAZY_OK) return rc;
  if (workspace_bytes < need) return LAZY_ERR_INVALID_ARG;
  int grid;
  rc = decode_grid(p, gc, chunks, grid_ctas, &grid);
  if (rc != LAZY_OK) return rc;
  const int32_t hv = p->hkv * chunks;
  const size_t slots = (size_t)batch * hv + (size_t)grid * kWarps;
  DecodeParams dp;
  dp.q = q;
  dp.q_pos = q_pos;
  dp.words = words;
  dp.cu_pages = cu_pages;
  dp.k_pool = p->k;
  dp.v_pool = p->v;
  dp.turn = p->d_turn;
  dp.ws_o = reinterpret_cast<float *>(workspace);
  dp.ws_lse = dp.ws_o + slots * gc * p->d;
  dp.err = p->d_err;
  dp.batch = batch;
  dp.hkv = p->hkv;
  dp.hq = num_q_heads;
  dp.num_blocks = p->num_blocks;
  dp.hv = hv;
  dp.chunks = chunks;
  dp.scale_log2 = sm_scale * 1.4426950408889634f;
  dp.wait_ns = p->wait_limit_ns;
  dp.slopes = p->alibi ? p->d_slopes : nullptr;
  CombineParams cp;
  cp.ws_o = dp.ws_o;
  cp.ws_lse = dp.ws_lse;
  cp.cu_pages = cu_pages;
  cp.out = out;
  cp.lse = lse;
  cp.batch = batch;
  cp.hq = num_q_heads;
  cp.hv = hv;
  cp.warps = (int64_t)grid * kWarps;
  cp.ch = 1;
  cudaStream_t s = (cudaStream_t)stream;
  return with_decode_shape(p->dtype, p->d, gc,
                           [&](auto L) { return decltype(L)::run(p, dp, cp, grid, s); });
}

// ------------------------------------------------------------------------------------------------
// Allocation-free decode: the same kernels, with their partial results in a fixed array compiled
// into the library instead of a caller workspace (for callers that may not allocate).
// ------------------------------------------------------------------------------------------------

// Scratch for lazy_attn_decode_noalloc. In host code this name is only a stand-in for the
// symbol; the device address comes from cudaGetSymbolAddress (noalloc_scratch below).
static __device__ __align__(256) unsigned char lazy_noalloc_scratch[LAZY_NOALLOC_SCRATCH_BYTES];

namespace {
// Device address of the scratch array in the current context. Looked up on every call rather
// than cached: after a device reset the module is loaded again and the array may move.
int noalloc_scratch(void **out) {
  void *ptr = nullptr;
  LAZY_CUDA_TRY(cudaGetSymbolAddress(&ptr, lazy_noalloc_scratch));
  *out = ptr;
  return LAZY_OK;
}
}  // namespace

extern "C" int lazy_attn_decode_noalloc(lazy_pool *p, const void *q, const int32_t *q_pos,
                                        const uint64_t *words, const int32_t *cu_pages,
                                        int32_t batch, int32_t num_q_heads, float sm_scale,
                                        int32_t grid_ctas, void *out, float *lse,
                                        lazy_stream_t stream) {
  if (!p || batch < 0 || grid_ctas < 0 || !(sm_scale > 0.f)) return LAZY_ERR_INVALID_ARG;
  if (batch == 0) return LAZY_OK;
  if (!q || !q_pos || !cu_pages || !out || !lse) return LAZY_ERR_INVALID_ARG;
  if (((uintptr_t)q & 15) || ((uintptr_t)out & 15) || ((uintptr_t)words & 7))
    return LAZY_ERR_INVALID_ARG;
  {
    std::lock_guard<std::mutex> g(p->mu);
    if (!p->dev_ready) {
      record_msg("pool has no device state yet: insert or write tokens before this call");
      return LAZY_ERR_INVALID_ARG;
    }
  }
  int dev = -1;
  LAZY_CUDA_TRY(cudaGetDevice(&dev));
  if (dev != p->device) {
    record_msg("the current device is not the pool's device");
    return LAZY_ERR_INVALID_ARG;
  }
  if (p->alibi && num_q_heads != (int32_t)p->slopes.size()) return LAZY_ERR_INVALID_ARG;
  int32_t gc, chunks;
  int rc = plan_groups(num_q_heads, p->hkv, &gc, &chunks);
  if (rc != LAZY_OK) return rc;
  int grid;
  rc = decode_grid(p, gc, chunks, grid_ctas, &grid);
  if (rc != LAZY_OK) return rc;
  const int32_t hv = p->hkv * chunks;
  const size_t slots = (size_t)batch * hv + (size_t)grid * kWarps;
  const size_t need = slots * gc * ((size_t)p->d + 1) * sizeof(float);
  if (need > (size_t)LAZY_NOALLOC_SCRATCH_BYTES) {
    record_msg("allocation-free decode: the batch needs more scratch than the fixed array");
    return LAZY_ERR_SCRATCH_LIMIT;
  }
  void *scratch = nullptr;
  rc = noalloc_scratch(&scratch);
  if (rc != LAZY_OK) return rc;
  DecodeParams dp;
  dp.q = q;
  dp.q_pos = q_pos;
  dp.words = words;
  dp.cu_pages = cu_pages;
  dp.k_pool = p->k;
  dp.v_pool = p->v;
  dp.turn = p->d_turn;
  dp.ws_o = reinterpret_cast<float *>(scratch);
  dp.ws_lse = dp.ws_o + slots * gc * p->d;
  dp.err = p->d_err;
  dp.batch = batch;
  dp.hkv = p->hkv;
  dp.hq = num_q_heads;
  dp.num_blocks = p->num_blocks;
  dp.hv = hv;
  dp.chunks = chunks;
  dp.scale_log2 = sm_scale * 1.4426950408889634f;
  dp.wait_ns = p->wait_limit_ns;
  dp.slopes = p->alibi ? p->d_slopes : nullptr;
  CombineParams cp;
  cp.ws_o = dp.ws_o;
  cp.ws_lse = dp.ws_lse;
  cp.cu_pages = cu_pages;
  cp.out = out;
  cp.lse = lse;
  cp.batch = batch;
  cp.hq = num_q_heads;
  cp.hv = hv;
  cp.warps = (int64_t)grid * kWarps;
  cp.ch = 1;
  cudaStream_t s = (cudaStream_t)stream;
  return with_decode_shape(p->dtype, p->d, gc,
                           [&](auto L) { return decltype(L)::run(p, dp, cp, grid, s); });
}
