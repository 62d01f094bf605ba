// CUDA-core prefill with deferred RoPE, fp32 arithmetic for any pool dtype. Serves the fp32
// pool (a tolerance of 1e-5 rules out reduced-precision tensor cores) and every shape the
// tensor-core kernel is not built for.
//
// One CTA = (request b, kv head h, TQ question tokens) and all G query heads of h: 64 rows.
// Rotations follow the LazyAttention summaries' prefill part: queries are rotated once to
// positions relative to the tile start m0 (R(m - m0)), and every cached key page gets ONE
// relative rotation R(o - m0) (its rows already carry R(j) from the encode), instead of an
// un-rotate to 0 followed by a re-rotate to the target position. The question's own keys (raw)
// are rotated by R(p - m0) and attended causally.
//
// Query-side variant (QS, LAZY_PREFILL_SIMT_QSIDE; the summaries' prefill part allows rotating
// either side): cached key pages are used as stored, R(j) k, and the query buffer holds
// R(m - o) q for the current document offset o, reloaded from the raw queries when o changes
// (and R(m - m0) q again for the question's own keys). A document of L_d keys then costs one
// rotation of the 64 query rows instead of L_d key rotations:
// (R(m - o) q) . (R(j) k) = (R(m) q) . (R(o + j) k).
#include <algorithm>

#include "lazy_common.cuh"
#include "pool_internal.h"
#include "prefill.h"

namespace lazy {
namespace {

constexpr int kRows = 64;
constexpr int kThreads = 128;

template <int D, bool QS>
struct SimtSmem {
  static constexpr int kQ = 0;                          // float [kRows][D+1]
  static constexpr int kK = kQ + kRows * (D + 1) * 4;   // float [kPage][D+1]
  static constexpr int kV = kK + kPage * (D + 1) * 4;   // float [kPage][D]
  static constexpr int kP = kV + kPage * D * 4;         // float [kRows][kPage+1]
  static constexpr int kKt = kP + kRows * (kPage + 1) * 4;  // int32 [kPage] key token (-1 = doc)
  static constexpr int kKp = kKt + kPage * 4;               // int32 [kPage] key logical position
  static constexpr int kBytes = kKp + kPage * 4;
};

template <typename T, int D, bool QS>
__global__ void __launch_bounds__(kThreads) prefill_simt_kernel(const PrefillParams p) {
  using S = SimtSmem<D, QS>;
  extern __shared__ __align__(16) uint8_t smem_raw[];
  float *Qs = reinterpret_cast<float *>(smem_raw + S::kQ);
  float *Ks = reinterpret_cast<float *>(smem_raw + S::kK);
  float *Vs = reinterpret_cast<float *>(smem_raw + S::kV);
  float *Ps = reinterpret_cast<float *>(smem_raw + S::kP);
  int32_t *Kt = reinterpret_cast<int32_t *>(smem_raw + S::kKt);
  int32_t *Kp = reinterpret_cast<int32_t *>(smem_raw + S::kKp);
  // ALiBi pools: no rotation anywhere; scores get slope * (n - m) instead
  const bool alibi = p.slopes != nullptr;
  const bool qside = QS && !alibi;

  const int b = blockIdx.z, h = blockIdx.y;
  const int G = p.G, TQ = p.TQ;
  const int t0 = blockIdx.x * TQ;
  const int32_t qbeg = p.cu_q[b];
  const int32_t Tb = p.cu_q[b + 1] - qbeg;
  if (t0 >= Tb) return;
  const int nt = min(TQ, Tb - t0);
  const int nrows = nt * G;
  const int32_t m0 = p.q_pos0[b] + t0;
  const int tid = threadIdx.x;
  const T *q = reinterpret_cast<const T *>(p.q);

  // ---- queries R(m - target) q, pre-scaled (log2 domain); target m0 = relative to the tile
  // start. The QS variant reloads them whenever the target (a document offset) changes.
  auto load_q = [&](int64_t target) {
    for (int idx = tid; idx < kRows * (D / 2); idx += kThreads) {
      const int row = idx / (D / 2), i = idx % (D / 2);
      float x = 0.f, y = 0.f;
      if (row < nrows) {
        const int t = t0 + row / G, qh = h * G + row % G;
        const T *src = q + ((size_t)(qbeg + t) * p.hq + qh) * D;
        float cs = 1.f, sn = 0.f;
        if (!alibi) rope_cos_sin((int64_t)(m0 + (t - t0)) - target, p.turn[i], cs, sn);
        const float a = Elem<T>::to_f(src[i]), c = Elem<T>::to_f(src[i + D / 2]);
        x = (a * cs - c * sn) * p.scale_log2;
        y = (a * sn + c * cs) * p.scale_log2;
      }
      Qs[row * (D + 1) + i] = x;
      Qs[row * (D + 1) + i + D / 2] = y;
    }
  };
  load_q(m0);
  int64_t q_target = m0;  // what the query buffer is rotated relative to

  const int row = tid >> 1, half = tid & 1;
  const int t_row = t0 + row / G;
  const int32_t m_row = p.q_pos0[b] + t_row;  // the row's logical position (ALiBi bias)
  const float slope2 = alibi ? p.slopes[h * G + row % G] * 1.4426950408889634f : 0.f;
  float acc[D / 2];
#pragma unroll
  for (int d = 0; d < D / 2; ++d) acc[d] = 0.f;
  float m_run = -INFINITY, l_run = 0.f;

  const T *kpool = reinterpret_cast<const T *>(p.k_pool);
  const T *vpool = reinterpret_cast<const T *>(p.v_pool);
  const T *knew = reinterpret_cast<const T *>(p.k_new);
  const T *vnew = reinterpret_cast<const T *>(p.v_new);
  const int32_t pg0 = p.cu_pages[b], npg = p.cu_pages[b + 1] - pg0;
  const int n_new_tiles = knew ? (t0 + nt + kPage - 1) / kPage : 0;

  for (int tile = 0; tile < npg + n_new_tiles; ++tile) {
    __syncthreads();
    const bool doc = tile < npg;
    int nvalid = kPage;
    bool skip = false;
    if (doc) {
      const uint64_t w = p.words[pg0 + tile];
      const uint32_t blk = word_block(w);
      nvalid = (int)word_nvalid(w);
      if (blk >= (uint32_t)p.num_blocks || nvalid > kPage) {
        if (tid == 0) set_error(p.err, LAZY_DEVERR_BAD_PAGE);
        skip = true;
      } else if (qside) {
        // keys as stored; the query rows follow the document offset (the same word for every
        // thread, so the reload is CTA-uniform)
        const uint32_t off = word_offset(w);
        const size_t page = ((size_t)blk * p.hkv + h) * (size_t)(kPage * D);
        for (int idx = tid; idx < kPage * D; idx += kThreads) {
          const int k = idx / D, i = idx % D;
          Ks[k * (D + 1) + i] = Elem<T>::to_f(kpool[page + idx]);
          Vs[idx] = Elem<T>::to_f(vpool[page + idx]);
        }
        if (tid < kPage) {
          Kt[tid] = -1;
          Kp[tid] = (int32_t)off + tid;
        }
        if ((int64_t)off != q_target) {
          q_target = off;
          load_q(off);
        }
      } else {
        const int64_t delta = (int64_t)word_offset(w) - m0;  // the one relative rotation
        const size_t page = ((size_t)blk * p.hkv + h) * (size_t)(kPage * D);
        for (int idx = tid; idx < kPage * (D / 2); idx += kThreads) {
          const int k = idx / (D / 2), i = idx % (D / 2);
          float cs = 1.f, sn = 0.f;
          if (!alibi) rope_cos_sin(delta, p.turn[i], cs, sn);
          const float a = Elem<T>::to_f(kpool[page + k * D + i]);
          const float c = Elem<T>::to_f(kpool[page + k * D + i + D / 2]);
          Ks[k * (D + 1) + i] = a * cs - c * sn;
          Ks[k * (D + 1) + i + D / 2] = a * sn + c * cs;
          Vs[k * D + i] = Elem<T>::to_f(vpool[page + k * D + i]);
          Vs[k * D + i + D / 2] = Elem<T>::to_f(vpool[page + k * D + i + D / 2]);
        }
        if (tid < kPage) {
          Kt[tid] = -1;
          Kp[tid] = (int32_t)word_offset(w) + tid;  // ALiBi: the word holds the page start
        }
      }
    } else {
      if (qside && q_target != m0) {  // the question's own keys: queries relative to m0 again
        q_target = m0;
        load_q(m0);
      }
      const int c0 = (tile - npg) * kPage;
      for (int idx = tid; idx < kPage * (D / 2); idx += kThreads) {
        const int k = idx / (D / 2), i = idx % (D / 2);
        const int kt = c0 + k;
        float a = 0.f, c = 0.f, va = 0.f, vc = 0.f, cs = 1.f, sn = 0.f;
        if (kt < Tb) {
          const size_t src = ((size_t)(qbeg + kt) * p.hkv + h) * D;
          a = Elem<T>::to_f(knew[src + i]);
          c = Elem<T>::to_f(knew[src + i + D / 2]);
          va = Elem<T>::to_f(vnew[src + i]);
          vc = Elem<T>::to_f(vnew[src + i + D / 2]);
          if (!alibi) rope_cos_sin((int64_t)(kt - t0), p.turn[i], cs, sn);
        }
        Ks[k * (D + 1) + i] = a * cs - c * sn;
        Ks[k * (D + 1) + i + D / 2] = a * sn + c * cs;
        Vs[k * D + i] = va;
        Vs[k * D + i + D / 2] = vc;
      }
      if (tid < kPage) {
        Kt[tid] = (c0 + tid < Tb) ? c0 + tid : 0x7FFFFFFF;
        Kp[tid] = p.q_pos0[b] + c0 + tid;
      }
    }
    __syncthreads();
    if (skip) continue;

    // ---- scores for (row, 8 keys), online softmax per row (two threads share a row)
    float s[8];
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) s[kk] = 0.f;
    for (int d = 0; d < D; ++d) {
      const float qv = Qs[row * (D + 1) + d];
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) s[kk] = fmaf(qv, Ks[(half * 8 + kk) * (D + 1) + d], s[kk]);
    }
    float mx = -INFINITY;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      const int k = half * 8 + kk;
      bool vis = k < nvalid;
      if (!doc) vis = Kt[k] <= t_row;
      if (alibi) s[kk] = fmaf(slope2, (float)(Kp[k] - m_row), s[kk]);
      if (!vis) s[kk] = -INFINITY;
      mx = fmaxf(mx, s[kk]);
    }
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    const float m_new = fmaxf(m_run, mx);
    const float alpha = (m_run == -INFINITY) ? 0.f : exp2f(m_run - m_new);
    float ls = 0.f;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      const float pr = s[kk] == -INFINITY ? 0.f : exp2f(s[kk] - m_new);
      ls += pr;
      Ps[row * (kPage + 1) + half * 8 + kk] = pr;
    }
    ls += __shfl_xor_sync(0xffffffffu, ls, 1);
    l_run = l_run * alpha + ls;
    m_run = m_new;
    __syncthreads();
#pragma unroll
    for (int d = 0; d < D / 2; ++d) acc[d] *= alpha;
    for (int k = 0; k < kPage; ++k) {
      const float pr = Ps[row * (kPage + 1) + k];
#pragma unroll
      for (int d = 0; d < D / 2; ++d) acc[d] = fmaf(pr, Vs[k * D + half * (D / 2) + d], acc[d]);
    }
  }

  if (row < nrows) {
    const int t = t0 + row / G, qh = h * G + row % G;
    T *dst = reinterpret_cast<T *>(p.out) + ((size_t)(qbeg + t) * p.hq + qh) * D + half * (D / 2);
    const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
#pragma unroll
    for (int d = 0; d < D / 2; ++d) dst[d] = Elem<T>::from_f(acc[d] * inv);
    if (half == 0)
      p.lse[(size_t)(qbeg + t) * p.hq + qh] =
          l_run > 0.f ? (m_run + log2f(l_run)) * 0.69314718055994531f : -INFINITY;
  }
}

template <typename T, int D, bool QS>
int launch_simt_variant(const PrefillParams &pp, int32_t max_q_len, cudaStream_t s) {
  constexpr int smem = SimtSmem<D, QS>::kBytes;
  static bool attr = false;
  if (!attr) {
    LAZY_CUDA_TRY(cudaFuncSetAttribute(prefill_simt_kernel<T, D, QS>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem));
    attr = true;
  }
  dim3 grid((max_q_len + pp.TQ - 1) / pp.TQ, pp.hkv, pp.batch);
  prefill_simt_kernel<T, D, QS><<<grid, kThreads, smem, s>>>(pp);
  LAZY_CUDA_TRY(cudaGetLastError());
  return LAZY_OK;
}

template <typename T, int D>
int launch_simt(const PrefillParams &pp, int32_t max_q_len, cudaStream_t s) {
  return pp.qside ? launch_simt_variant<T, D, true>(pp, max_q_len, s)
                  : launch_simt_variant<T, D, false>(pp, max_q_len, s);
}

}  // namespace

int prefill_simt(lazy_pool *p, const PrefillParams &pp, int32_t max_q_len, cudaStream_t s) {
  if (pp.G > kRows) return LAZY_ERR_UNSUPPORTED;
  if (p->dtype == LAZY_DTYPE_BF16)
    return p->d == 128 ? launch_simt<__nv_bfloat16, 128>(pp, max_q_len, s)
                       : launch_simt<__nv_bfloat16, 64>(pp, max_q_len, s);
  return p->d == 128 ? launch_simt<float, 128>(pp, max_q_len, s)
                     : launch_simt<float, 64>(pp, max_q_len, s);
}

}  // namespace lazy
