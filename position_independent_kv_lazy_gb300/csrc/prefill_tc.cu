// Tensor-core (tcgen05/TMEM/TMA) prefill: not built yet.
#include "prefill.h"

namespace lazy {
int prefill_tc_supported(const lazy_pool *p, int32_t hq) {
  (void)p;
  (void)hq;
  return LAZY_ERR_UNSUPPORTED;
}
int prefill_tc(lazy_pool *p, const PrefillParams &pp, int32_t max_q_len, cudaStream_t s) {
  (void)p; (void)pp; (void)max_q_len; (void)s;
  return LAZY_ERR_UNSUPPORTED;
}
}  // namespace lazy
