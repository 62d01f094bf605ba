// lazy_attn_prefill: argument checks and kernel choice; lazy_attn_prefill_append: the same
// call followed by the question's own K/V going into the pool as a private segment.
#include "prefill.h"

using namespace lazy;

extern "C" int lazy_prefill_workspace_bytes(lazy_pool *p, int32_t batch, int32_t total_q,
                                            int32_t max_q_len, int32_t num_q_heads,
                                            int32_t flags, size_t *bytes) {
  if (!p || !bytes || batch < 0 || total_q < 0 || max_q_len < 0 || num_q_heads <= 0)
    return LAZY_ERR_INVALID_ARG;
  if (flags & ~(15 | LAZY_PREFILL_ABSOLUTE_KEYS)) return LAZY_ERR_INVALID_ARG;
  flags &= 15;
  if (flags < LAZY_PREFILL_AUTO || flags > LAZY_PREFILL_TC_QSIDE) return LAZY_ERR_INVALID_ARG;
  *bytes = 0;  // the SIMT kernel needs no scratch; the tensor-core one may split its last wave
  if (flags == LAZY_PREFILL_SIMT || flags == LAZY_PREFILL_SIMT_QSIDE || batch == 0 ||
      total_q == 0 || max_q_len == 0)
    return LAZY_OK;
  if (num_q_heads % p->hkv || prefill_tc_supported(p, num_q_heads) != LAZY_OK) return LAZY_OK;
  int rc = ensure_device(p);
  if (rc != LAZY_OK) return rc;
  return prefill_tc_workspace_bytes(p, batch, max_q_len, num_q_heads, bytes);
}

extern "C" int lazy_attn_prefill(lazy_pool *p, const void *q, const void *k_new,
                                 const void *v_new, const int32_t *cu_q, const int32_t *q_pos0,
                                 const uint64_t *words, const int32_t *cu_pages, int32_t batch,
                                 int32_t total_q, int32_t max_q_len, int32_t num_q_heads,
                                 float sm_scale, void *out, float *lse, void *workspace,
                                 size_t workspace_bytes, int32_t flags, lazy_stream_t stream) {
  if (!p || batch < 0 || total_q < 0 || max_q_len < 0 || !(sm_scale > 0.f))
    return LAZY_ERR_INVALID_ARG;
  if (num_q_heads <= 0 || num_q_heads % p->hkv) return LAZY_ERR_INVALID_ARG;
  if (p->alibi && num_q_heads != (int32_t)p->slopes.size()) return LAZY_ERR_INVALID_ARG;
  if (flags & ~(15 | LAZY_PREFILL_ABSOLUTE_KEYS)) return LAZY_ERR_INVALID_ARG;
  const int32_t absolute = (flags & LAZY_PREFILL_ABSOLUTE_KEYS) ? 1 : 0;
  flags &= 15;
  if (flags < LAZY_PREFILL_AUTO || flags > LAZY_PREFILL_TC_QSIDE) return LAZY_ERR_INVALID_ARG;
  if (batch == 0 || total_q == 0 || max_q_len == 0) return LAZY_OK;
  if (!q || !cu_q || !q_pos0 || !cu_pages || !out || !lse) return LAZY_ERR_INVALID_ARG;
  if ((k_new == nullptr) != (v_new == nullptr)) return LAZY_ERR_INVALID_ARG;
  if (((uintptr_t)q & 15) || ((uintptr_t)out & 15) || ((uintptr_t)k_new & 15) ||
      ((uintptr_t)v_new & 15) || ((uintptr_t)words & 7))
    return LAZY_ERR_INVALID_ARG;
  int rc = ensure_device(p);
  if (rc != LAZY_OK) return rc;
  PrefillParams pp;
  pp.q = q;
  pp.k_new = k_new;
  pp.v_new = v_new;
  pp.cu_q = cu_q;
  pp.q_pos0 = q_pos0;
  pp.words = words;
  pp.cu_pages = cu_pages;
  pp.k_pool = p->k;
  pp.v_pool = p->v;
  pp.turn = p->d_turn;
  pp.out = out;
  pp.lse = lse;
  pp.err = p->d_err;
  pp.batch = batch;
  pp.hkv = p->hkv;
  pp.hq = num_q_heads;
  pp.num_blocks = p->num_blocks;
  pp.G = num_q_heads / p->hkv;
  pp.TQ = pp.G >= 64 ? 1 : 64 / pp.G;
  pp.total_q = total_q;
  pp.scale_log2 = sm_scale * 1.4426950408889634f;
  pp.wait_ns = p->wait_limit_ns;
  pp.slopes = p->alibi ? p->d_slopes : nullptr;
  pp.workspace = workspace;
  pp.workspace_bytes = workspace ? workspace_bytes : 0;
  pp.qside = flags == LAZY_PREFILL_SIMT_QSIDE ? 1 : 0;
  pp.absolute = absolute && !p->alibi;
  pp.tc_qside = flags == LAZY_PREFILL_TC_QSIDE && !p->alibi;
  cudaStream_t s = (cudaStream_t)stream;
  const bool tc_ok = prefill_tc_supported(p, num_q_heads) == LAZY_OK;
  if (flags == LAZY_PREFILL_TC || flags == LAZY_PREFILL_TC_QSIDE) {
    if (!tc_ok) return LAZY_ERR_UNSUPPORTED;
    return prefill_tc(p, pp, max_q_len, s);
  }
  if (flags == LAZY_PREFILL_AUTO && tc_ok) return prefill_tc(p, pp, max_q_len, s);
  return prefill_simt(p, pp, max_q_len, s);
}

extern "C" int lazy_attn_prefill_append(lazy_pool *p, const void *q, const void *k_new,
                                        const void *v_new, const int32_t *cu_q,
                                        const int32_t *q_pos0, const uint64_t *words,
                                        const int32_t *cu_pages, int32_t batch, int32_t total_q,
                                        int32_t max_q_len, int32_t num_q_heads, float sm_scale,
                                        void *out, float *lse, void *workspace,
                                        size_t workspace_bytes, int32_t flags,
                                        const int32_t *append_slots,
                                        const int32_t *append_local_pos, lazy_stream_t stream) {
  // Every argument of both steps is checked before anything is launched.
  if (!p || total_q < 0) return LAZY_ERR_INVALID_ARG;
  if (total_q > 0 && (!k_new || !v_new || !append_slots || !append_local_pos))
    return LAZY_ERR_INVALID_ARG;
  int rc = lazy_attn_prefill(p, q, k_new, v_new, cu_q, q_pos0, words, cu_pages, batch, total_q,
                             max_q_len, num_q_heads, sm_scale, out, lse, workspace,
                             workspace_bytes, flags, stream);
  if (rc != LAZY_OK || batch == 0 || total_q == 0 || max_q_len == 0) return rc;
  // Both steps only read k_new / v_new, so the encode needs no ordering after the attention
  // beyond the stream's.
  return kv_pool_write_tokens(p, k_new, v_new, total_q, append_slots, append_local_pos, stream);
}
