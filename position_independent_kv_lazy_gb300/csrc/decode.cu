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
#include <algorithm>

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

  extern __shared__ __align__(128) uint8_t smem_raw[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint8_t *ws = smem_raw + warp * S::kBytes;
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
    const size_t page = ((size_t)blk * p.hkv + prod.hv / p.chunks) * (size_t)(kPage * D);
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

struct CombineParams {
  const float *ws_o;
  const float *ws_lse;
  const int32_t *cu_pages;
  void *out;
  float *lse;
  int32_t batch, hq, hv;
  int64_t warps;  // total warps of the decode launch
};

// One CTA per unit: merges the unit's pieces (slots unit + w for the warps w whose ranges
// intersect it) with a log-sum-exp combine and writes the final rows.
template <typename T, int D, int GC>
__global__ void __launch_bounds__(128) combine_kernel(const CombineParams p) {
  cudaGridDependencySynchronize();  // partials of the decode kernel launched just before
  const int32_t u = blockIdx.x;
  const int32_t b = u / p.hv, hv = u % p.hv;
  const int32_t wbase = p.cu_pages[b], np = p.cu_pages[b + 1] - wbase;
  const int64_t N = (int64_t)p.hv * p.cu_pages[p.batch];
  const int64_t W = p.warps;
  T *out = reinterpret_cast<T *>(p.out);
  int64_t wf = 0, wl = -1;
  if (np > 0) {
    const int64_t S = (int64_t)p.hv * wbase + (int64_t)hv * np, E = S + np;
    wf = ((S + 1) * W + N - 1) / N - 1;
    wl = (E * W + N - 1) / N - 1;
  }
  for (int idx = threadIdx.x; idx < GC * (D / 4); idx += blockDim.x) {
    const int g = idx / (D / 4), d4 = idx % (D / 4);
    float mx = -INFINITY;
    for (int64_t w = wf; w <= wl; ++w) {
      if (w * N / W == (w + 1) * N / W) continue;  // empty range
      mx = fmaxf(mx, p.ws_lse[(size_t)(u + w) * GC + g]);
    }
    float sum = 0.f;
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
    if (mx != -INFINITY) {
      for (int64_t w = wf; w <= wl; ++w) {
        if (w * N / W == (w + 1) * N / W) continue;
        const float l = p.ws_lse[(size_t)(u + w) * GC + g];
        if (l == -INFINITY) continue;
        const float wt = exp2f(l - mx);
        const float4 o = *reinterpret_cast<const float4 *>(p.ws_o + ((size_t)(u + w) * GC + g) * D +
                                                           d4 * 4);
        sum += wt;
        a.x = fmaf(wt, o.x, a.x); a.y = fmaf(wt, o.y, a.y);
        a.z = fmaf(wt, o.z, a.z); a.w = fmaf(wt, o.w, a.w);
      }
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

template <typename T, int D, int GC, int STAGES>
struct DecodeLaunch {
  using S = DecodeSmem<T, D, GC, STAGES>;
  static constexpr int kSmem = S::kBytes * kWarps;
  static int ctas_per_sm() {
    static int cached = -1;
    if (cached < 0) {
      auto fn = decode_split_kernel<T, D, GC, kWarps, STAGES>;
      if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem) !=
          cudaSuccess)
        return -1;
      int n = 0;
      if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, kWarps * 32, kSmem) !=
          cudaSuccess)
        return -1;
      cached = std::max(1, n);
    }
    return cached;
  }
  static int run(lazy_pool *pl, const DecodeParams &dp, const CombineParams &cp, int grid,
                 cudaStream_t s) {
    (void)pl;
    LAZY_CUDA_TRY(launch_pdl(decode_split_kernel<T, D, GC, kWarps, STAGES>, grid, kWarps * 32,
                             kSmem, s, dp));
    LAZY_CUDA_TRY(launch_pdl(combine_kernel<T, D, GC>, dp.batch * dp.hv, 128, 0, s, cp));
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

int decode_grid(lazy_pool *p, int32_t gc, int32_t grid_ctas, int *grid) {
  if (grid_ctas > 0) {
    *grid = grid_ctas;
    return LAZY_OK;
  }
  const int per_sm =
      with_decode_shape(p->dtype, p->d, gc, [](auto L) { return decltype(L)::ctas_per_sm(); });
  if (per_sm <= 0) {
    record_msg("decode kernel occupancy query failed");
    return LAZY_ERR_CUDA;
  }
  *grid = p->num_sms * per_sm;
  return LAZY_OK;
}

}  // namespace
}  // namespace lazy

using namespace lazy;

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
  rc = decode_grid(p, gc, grid_ctas, &grid);
  if (rc != LAZY_OK) return rc;
  const size_t slots = (size_t)batch * p->hkv * chunks + (size_t)grid * kWarps;
  *bytes = slots * gc * ((size_t)p->d + 1) * sizeof(float) + 256;
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
  rc = decode_grid(p, gc, grid_ctas, &grid);
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
  cudaStream_t s = (cudaStream_t)stream;
  return with_decode_shape(p->dtype, p->d, gc,
                           [&](auto L) { return decltype(L)::run(p, dp, cp, grid, s); });
}

// ------------------------------------------------------------------------------------------------
// Allocation-free decode: the same kernels, with their partial results in a fixed array compiled
// into the library instead of a caller workspace (for callers that may not allocate).
// ------------------------------------------------------------------------------------------------
#include <mutex>

// Scratch for lazy_attn_decode_noalloc. In host code this name is only a stand-in for the
// symbol; the device address comes from cudaGetSymbolAddress (noalloc_scratch below).
static __device__ __align__(256) unsigned char lazy_noalloc_scratch[LAZY_NOALLOC_SCRATCH_BYTES];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void *g_noalloc_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once per device.
int noalloc_scratch(void **out) {
  int dev = -1;
  LAZY_CUDA_TRY(cudaGetDevice(&dev));
  if (dev < 0 || dev >= kMaxDevices) {
    record_msg("allocation-free decode supports device ordinals below 64");
    return LAZY_ERR_UNSUPPORTED;
  }
  std::lock_guard<std::mutex> g(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void *ptr = nullptr;
    LAZY_CUDA_TRY(cudaGetSymbolAddress(&ptr, lazy_noalloc_scratch));
    g_noalloc_ptr[dev] = ptr;
  }
  *out = g_noalloc_ptr[dev];
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
  rc = decode_grid(p, gc, grid_ctas, &grid);
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
  cudaStream_t s = (cudaStream_t)stream;
  return with_decode_shape(p->dtype, p->d, gc,
                           [&](auto L) { return decltype(L)::run(p, dp, cp, grid, s); });
}
