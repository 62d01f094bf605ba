// Device-side helpers shared by the kernels of the deferred-RoPE attention library.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "lazy_attn.h"

namespace lazy {

constexpr int kPage = 16;  // tokens per page (the only page size the kernels are built for)

// ------------------------------------------------------------------------------------------
// Page word: bits 0-31 block id, 32-57 logical offset, 58-63 n_valid-1 ("block ID, offset"
// bit-packed in one register, LazyAttention summaries, decoding part). One 8-byte load.
// ------------------------------------------------------------------------------------------
__host__ __device__ __forceinline__ uint32_t word_block(uint64_t w) { return (uint32_t)w; }
__host__ __device__ __forceinline__ uint32_t word_offset(uint64_t w) {
  return (uint32_t)(w >> 32) & 0x3FFFFFFu;
}
__host__ __device__ __forceinline__ uint32_t word_nvalid(uint64_t w) {
  return (uint32_t)(w >> 58) + 1u;
}

// ------------------------------------------------------------------------------------------
// RoPE angle for an integer position difference, reduced exactly.
// turn_frac[i] = frac(theta_i / 2pi) as a 64-bit fixed-point fraction of a turn, so
// delta * turn_frac[i] (mod 2^64, i.e. two's-complement wrap) is the angle delta*theta_i in
// turns modulo 1, with no floating-point range reduction and an error of ~|delta| * 2^-53 turns.
// The nearest quarter turn q is taken off in fixed point; the remainder x, |x| <= pi/4, goes
// through the Taylor series of sin (to x^9) and cos (to x^10), whose truncation errors at pi/4
// are 1.8e-9 and 1.2e-10; with the fp32 rounding of x (<= 4.7e-8 rad) and of the Horner steps
// the result is within 2e-7 of the exact value (largest error seen: 8e-8). The quadrant then
// swaps and negates (cos, sin) of x. No library call, about 25 instructions and no branch.
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ void rope_cos_sin(int64_t delta, uint64_t turn_frac, float &c,
                                             float &s) {
  const uint64_t t = (uint64_t)delta * turn_frac;
  const uint32_t q = (uint32_t)((t + (1ull << 61)) >> 62);     // nearest quarter turn, 0..3
  const int64_t r = (int64_t)(t - ((uint64_t)q << 62));          // [-2^61, 2^61): +-1/8 turn
  const float x = (float)(int32_t)(r >> 32) * 1.46291807926715968e-9f;  // * 2 pi / 2^32
  const float x2 = x * x;
  float sp = fmaf(x2, 2.75573192e-6f, -1.98412698e-4f);  // 1/9!, -1/7!
  sp = fmaf(x2, sp, 8.33333333e-3f);                        // 1/5!
  sp = fmaf(x2, sp, -1.66666667e-1f);                       // -1/3!
  const float sx = fmaf(x * x2, sp, x);
  float cp = fmaf(x2, -2.75573192e-7f, 2.48015873e-5f);  // -1/10!, 1/8!
  cp = fmaf(x2, cp, -1.38888889e-3f);                       // -1/6!
  cp = fmaf(x2, cp, 4.16666667e-2f);                        // 1/4!
  cp = fmaf(x2, cp, -0.5f);                                 // -1/2!
  const float cx = fmaf(x2, cp, 1.0f);
  const float cc = (q & 1) ? sx : cx, ss = (q & 1) ? cx : sx;
  c = (q == 1 || q == 2) ? -cc : cc;  // cos(q pi/2 + x): cos x, -sin x, -cos x, sin x
  s = (q >= 2) ? -ss : ss;            // sin(q pi/2 + x): sin x, cos x, -sin x, -cos x
}

// Element conversion helpers.
template <typename T>
struct Elem;
template <>
struct Elem<__nv_bfloat16> {
  static constexpr int kBytes = 2;
  __device__ __forceinline__ static float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
  __device__ __forceinline__ static __nv_bfloat16 from_f(float x) { return __float2bfloat16_rn(x); }
};
template <>
struct Elem<float> {
  static constexpr int kBytes = 4;
  __device__ __forceinline__ static float to_f(float x) { return x; }
  __device__ __forceinline__ static float from_f(float x) { return x; }
};

// Unpack 16 bytes into EPL floats.
template <typename T>
__device__ __forceinline__ void unpack16(const uint4 &u, float *f);
template <>
__device__ __forceinline__ void unpack16<__nv_bfloat16>(const uint4 &u, float *f) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}
template <>
__device__ __forceinline__ void unpack16<float>(const uint4 &u, float *f) {
  f[0] = __uint_as_float(u.x);
  f[1] = __uint_as_float(u.y);
  f[2] = __uint_as_float(u.z);
  f[3] = __uint_as_float(u.w);
}

template <typename T>
__device__ __forceinline__ uint4 pack16(const float *f);
template <>
__device__ __forceinline__ uint4 pack16<__nv_bfloat16>(const float *f) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
    w[i] = *reinterpret_cast<uint32_t *>(&h);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}
template <>
__device__ __forceinline__ uint4 pack16<float>(const float *f) {
  return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                    __float_as_uint(f[3]));
}

// ------------------------------------------------------------------------------------------
// Shared-memory barriers, bulk async copies, bounded waits.
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Wait for the phase with the given parity to complete; false if `limit_ns` passed first.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, uint64_t limit_ns) {
  const uint32_t a = smem_u32(bar);
  if (mbar_try_wait(a, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(a, parity)) {
    if (global_timer_ns() - t0 > limit_ns) return false;
  }
  return true;
}

// 1-D bulk copy global -> shared, completion counted in bytes on `bar`.
// Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes,
                                         uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void set_error(int32_t *err, int32_t bits) {
  if (err) atomicOr(err, bits);
}

}  // namespace lazy
