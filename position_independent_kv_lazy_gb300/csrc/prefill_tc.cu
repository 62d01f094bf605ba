// Tensor-core prefill with deferred RoPE for bf16 pools, head_dim 128 (tcgen05 + TMEM + TMA).
//
// Follows the LazyAttention summaries' prefill part: KV blocks are loaded from the cache and each
// key tile receives ONE relative rotation, by the offset between its document and the query
// tile, instead of an un-rotate followed by a re-rotate. Here the query tile's reference position
// is m0 = the CTA's first question token: queries are rotated by R(m - m0), a cached page of a
// segment at offset o (rows already carry R(j)) by R(o - m0), a question key at p by R(p - m0).
//
// CTA = (request b, kv head h, 2 x TQ question tokens): two 128-row Q tiles, rows ordered
// (token, query head of the group), TQ = 128 / G. 12 warps:
//   warp 0      TMA producer: Q tiles once, then per 128-key tile K into a 3-stage ring and V
//               into a 2-stage ring (K one tile ahead of V); 8 consecutive full blocks go as one
//               box, otherwise 8 page boxes (16 rows x 64 dims, 128B swizzle); question keys by
//               128-token boxes.
//   warp 1      TMEM owner (512 columns) and single-thread tcgen05.mma issuer:
//               S_i = Q_i K^T (SS; fp16 operands written by the rotation passes, bf16 in the
//               ALiBi mode), then O_i += P_i V (bf16; P from TMEM, V MN-major).
//   warps 4-7   softmax of Q tile 0, warps 8-11 of Q tile 1 (TMEM lane quadrant = warp % 4):
//               each thread holds its row's 128 scores, online softmax in the log2 domain with
//               a lazy rescale (the running max only moves when the tile max exceeds it by more
//               than 8), P written back into S's TMEM columns as bf16 pairs. The same 256 threads
//               rotate their Q rows once and each K tile in shared memory, in place (the pair
//               (i, i+64) sits at the same swizzled offset of the two 64-dim boxes), two tiles
//               ahead of the scores that need it: fp32 arithmetic, rounded once to fp16.
// The softmax loop is kept compact (one shared angle routine, one code path for masked and full
// tiles): with per-site copies the kernel was instruction-fetch bound.
// TMEM: S_0 [0,128) S_1 [128,256) O_0 [256,384) O_1 [384,512) fp32 columns.
// Every wait is bounded; a timeout sets LAZY_DEVERR_TIMEOUT, raises a CTA abort flag that
// releases the other roles, drains outstanding copies and MMAs, frees TMEM and returns.
#include <cuda.h>
#include <cuda_fp16.h>
#include <string.h>

#include <algorithm>
#include <cmath>
#include <mutex>

#include "lazy_common.cuh"
#include "prefill.h"

namespace lazy {
namespace {

constexpr int kTile = 128;
constexpr int kNK = 3;  // K ring: a K tile is free again as soon as both QK products read it
constexpr int kNV = 2;  // V ring: freed after both PV products
constexpr int kThreads = 384;
constexpr int kTileBytes = kTile * 128 * 2;  // 32 KB: 128 rows x 128 bf16
constexpr int kHalfBytes = kTileBytes / 2;   // one 64-dim box column

// Shared-memory map (offsets from a 1024-aligned base).
constexpr int kOffQ = 0;                               // 2 Q tiles
constexpr int kOffK = kOffQ + 2 * kTileBytes;          // kNK K stages
constexpr int kOffV = kOffK + kNK * kTileBytes;        // kNV V stages
constexpr int kMaxSplit = 8;  // most key-range chunks of a split unit
constexpr int kNM = 4;  // softmax metadata ring (see SMeta)
constexpr int kOffMetaK = kOffV + kNV * kTileBytes;    // KMeta [kNK]
constexpr int kOffMetaS = kOffMetaK + kNK * 48;        // SMeta [kNM]
constexpr int kOffBar = kOffMetaS + kNM * 80 + 16;     // barriers (8-byte aligned)
constexpr int kOffTurn = kOffBar + 256;                // the 64 turn fractions (uint64)
constexpr int kSmemBytes = kOffTurn + 64 * 8 + 1024;   // + alignment slack
static_assert(kSmemBytes <= 232448, "shared memory per block");

// Read by the rotation group (valid until the K stage is refilled, after QK of this tile).
struct KMeta {
  int32_t kind;   // 0 = document pages, 1 = question keys
  int32_t c0;     // question tile: first key token
  int32_t off[8]; // document tile: logical offset of each page
  int32_t ref;    // query-side mode: the tile's reference position r (Q tiles hold R(m - r) q)
  int32_t pad;
};
// Read by the softmax groups. Written when tile j's K copy is issued, which precedes S_j; the
// slot is rewritten for tile j + 4, whose K copy waits for QK of tile j + 1, which the MMA
// issuer only starts after both softmax groups released tile j.
struct SMeta {
  int32_t kind;
  int32_t c0;
  int32_t full;    // document tile: every page present and full
  int32_t pad;
  int32_t nv[8];   // document tile: valid tokens per page (0 = absent / bad)
  int32_t pos0[8]; // ALiBi: logical position of the first key of each 16-key group
};
static_assert(sizeof(SMeta) == 80, "SMeta layout");

struct TcParams {
  CUtensorMap tm_q, tm_knew, tm_vnew, tm_k, tm_v, tm_k8, tm_v8;
  CUtensorMap tm_out;   // out, the same boxes as tm_q (one Q tile per 64-dim half)
  CUtensorMap tm_part;  // part_o as [items * 256 rows][128] fp32, box 32 dims x 128 rows
  const int32_t *cu_q;
  const int32_t *q_pos0;
  const uint64_t *words;
  const int32_t *cu_pages;
  const uint64_t *turn;
  __nv_bfloat16 *out;
  float *lse;
  int32_t *err;
  int32_t batch, hkv, hq, num_blocks, G, TQ, has_new;
  float scale_log2;
  uint64_t wait_ns;
  const float *slopes;  // ALiBi: per query head
  // Schedule (1-D grid). Unit u = (request b, kv head h, token block x) with x fastest; blocks
  // [0, n_full) take whole units. With ksplit > 1 the n_split units from n_full on are cut into
  // ksplit key-range chunks each (split_item): split units go in groups of X, and a group's
  // items run chunk by chunk, so blocks side by side read the same keys and share them through
  // L2. Chunk results go to part_o / part_lse (item index, 256 rows: Q tile i row r at
  // i * 128 + r) for prefill_combine_kernel.
  int32_t X, n_full, n_split, ksplit;
  float *part_o;    // [items][256][128] O / l
  float *part_lse;  // [items][256] log2-domain lse (m + log2 l), -inf when no key was visible
};

// ---------------------------------------------------------------- PTX helpers
__device__ __forceinline__ void tma2d(void *dst, const CUtensorMap *m, int x, int y,
                                      uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, "
      "{%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"((uint64_t)m), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void tma3d(void *dst, const CUtensorMap *m, int x, int y, int z,
                                      uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, "
      "{%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
      "l"((uint64_t)m), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void tma4d(void *dst, const CUtensorMap *m, int x, int y, int z, int w,
                                      uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, "
      "{%2, %3, %4, %5}], [%6];" ::"r"(smem_u32(dst)),
      "l"((uint64_t)m), "r"(x), "r"(y), "r"(z), "r"(w), "r"(smem_u32(bar))
      : "memory");
}
// Shared-memory matrix descriptor: 128B swizzle, version 1.
__device__ __forceinline__ uint64_t sdesc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((addr & 0x3FFFF) >> 4) | ((uint64_t)(lbo >> 4) << 16) |
         ((uint64_t)(sbo >> 4) << 32) | (1ull << 46) | (2ull << 61);
}
__device__ __forceinline__ void mma_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                       int acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc));
}
__device__ __forceinline__ void mma_ts(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                       int acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc));
}
__device__ __forceinline__ void mma_commit(uint64_t *bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// TMA stores (shared -> global, bulk-group completion) and their wait. The wait is for the
// writes themselves, not only for the reads of the source: the issuing thread leaves the kernel
// with its stores complete, as it does with plain stores.
__device__ __forceinline__ void tma_store2d(const CUtensorMap *m, const void *src, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
          (uint64_t)m),
      "r"(smem_u32(src)), "r"(x), "r"(y)
      : "memory");
}
__device__ __forceinline__ void tma_store3d(const CUtensorMap *m, const void *src, int x, int y,
                                            int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
          (uint64_t)m),
      "r"(smem_u32(src)), "r"(x), "r"(y), "r"(z)
      : "memory");
}
__device__ __forceinline__ void bulk_commit_and_wait() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
// Named barrier 1 + i over the 128 threads of softmax group i (immediate ids, so that only
// barriers 0-2 are reserved).
__device__ __forceinline__ void group_bar(int i) {
  if (i == 0)
    asm volatile("bar.sync 1, 128;" ::: "memory");
  else
    asm volatile("bar.sync 2, 128;" ::: "memory");
}

#define LAZY_R32(r)                                                                          \
  "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),        \
      "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), \
      "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),           \
      "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),           \
      "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
#define LAZY_W32(r)                                                                          \
  "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),    \
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),       \
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),     \
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),     \
      "r"(r[29]), "r"(r[30]), "r"(r[31])

// 32 consecutive fp32 TMEM columns of this thread's lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : LAZY_R32(r)
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
// All 128 fp32 TMEM columns of this thread's lane. Load and wait are one statement, so no use
// of the registers can be scheduled before the wait.
__device__ __forceinline__ void tmem_ld128(uint32_t taddr, uint32_t (&r)[128]) {
  asm volatile(
      "{\n"
      "tcgen05.ld.sync.aligned.32x32b.x128.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,"
      "%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,"
      "%58,%59,%60,%61,%62,%63,%64,%65,%66,%67,%68,%69,%70,%71,%72,%73,%74,%75,%76,%77,%78,%79,"
      "%80,%81,%82,%83,%84,%85,%86,%87,%88,%89,%90,%91,%92,%93,%94,%95,%96,%97,%98,%99,%100,"
      "%101,%102,%103,%104,%105,%106,%107,%108,%109,%110,%111,%112,%113,%114,%115,%116,%117,"
      "%118,%119,%120,%121,%122,%123,%124,%125,%126,%127}, [%128];\n"
      "tcgen05.wait::ld.sync.aligned;\n"
      "}"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]),
        "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]),
        "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]),
        "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]),
        "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]),
        "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]),
        "=r"(r[62]), "=r"(r[63]), "=r"(r[64]), "=r"(r[65]), "=r"(r[66]), "=r"(r[67]),
        "=r"(r[68]), "=r"(r[69]), "=r"(r[70]), "=r"(r[71]), "=r"(r[72]), "=r"(r[73]),
        "=r"(r[74]), "=r"(r[75]), "=r"(r[76]), "=r"(r[77]), "=r"(r[78]), "=r"(r[79]),
        "=r"(r[80]), "=r"(r[81]), "=r"(r[82]), "=r"(r[83]), "=r"(r[84]), "=r"(r[85]),
        "=r"(r[86]), "=r"(r[87]), "=r"(r[88]), "=r"(r[89]), "=r"(r[90]), "=r"(r[91]),
        "=r"(r[92]), "=r"(r[93]), "=r"(r[94]), "=r"(r[95]), "=r"(r[96]), "=r"(r[97]),
        "=r"(r[98]), "=r"(r[99]), "=r"(r[100]), "=r"(r[101]), "=r"(r[102]), "=r"(r[103]),
        "=r"(r[104]), "=r"(r[105]), "=r"(r[106]), "=r"(r[107]), "=r"(r[108]), "=r"(r[109]),
        "=r"(r[110]), "=r"(r[111]), "=r"(r[112]), "=r"(r[113]), "=r"(r[114]), "=r"(r[115]),
        "=r"(r[116]), "=r"(r[117]), "=r"(r[118]), "=r"(r[119]), "=r"(r[120]), "=r"(r[121]),
        "=r"(r[122]), "=r"(r[123]), "=r"(r[124]), "=r"(r[125]), "=r"(r[126]), "=r"(r[127])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
      "%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
      "%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(
          taddr),
      LAZY_W32(r)
      : "memory");
}

// max(a, b, c) in one instruction.
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// 2^x with one MUFU instruction (inputs here are <= 8, results in (0, 256]; -inf gives 0).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf2(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t *>(&h);
}

// (cos, sin) of the 8 frequencies of one 16-byte chunk c (dims 8c .. 8c+7 of each 64-dim half)
// as fp32 pairs: co[k] = (cos, cos') of frequencies 8c+2k, 8c+2k+1, matching the (low, high)
// halves of the chunk's 32-bit word k.
struct RotF {
  float2 co[4], si[4];
};

__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&h);
}

// The relative rotation of one row chunk, x_i <- x_i cos - x_{i+64} sin and
// x_{i+64} <- x_i sin + x_{i+64} cos for i = 8c .. 8c+7: bf16 in (as loaded), out in the operand
// type of the QK product (kF16: fp16, else bf16), fp32 arithmetic with a single rounding at the
// end. fp16 keeps 11 significant bits against bf16's 8, so the rotated query row, whose rounding
// error is the same for every key it meets and does not average out, costs 8x less in the
// log-sum-exp.
template <bool kF16>
__device__ __forceinline__ void rot_words(uint4 &a, uint4 &b, const RotF &rf) {
  uint32_t *x = reinterpret_cast<uint32_t *>(&a);
  uint32_t *y = reinterpret_cast<uint32_t *>(&b);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 xf = make_float2(__uint_as_float(x[k] << 16), __uint_as_float(x[k] & 0xFFFF0000u));
    const float2 yf = make_float2(__uint_as_float(y[k] << 16), __uint_as_float(y[k] & 0xFFFF0000u));
    const float2 ys = __fmul2_rn(yf, rf.si[k]);
    const float2 xo = __ffma2_rn(xf, rf.co[k], make_float2(-ys.x, -ys.y));
    const float2 yo = __ffma2_rn(xf, rf.si[k], __fmul2_rn(yf, rf.co[k]));
    x[k] = kF16 ? pack_h2(xo.x, xo.y) : pack_bf2(xo.x, xo.y);
    y[k] = kF16 ? pack_h2(yo.x, yo.y) : pack_bf2(yo.x, yo.y);
  }
}

// Rotate, in place, one row of a 128-row swizzled tile at 16-byte chunk c of both 64-dim boxes
// (the pair (i, i+64) of a row sits at the same swizzled offset of the two boxes).
template <bool kF16>
__device__ __forceinline__ void rotate_row_chunk(uint8_t *tile, int row, int c, const RotF &rf) {
  const int phys = (c ^ (row & 7)) * 16;
  uint4 *lo = reinterpret_cast<uint4 *>(tile + row * 128 + phys);
  uint4 *hi = reinterpret_cast<uint4 *>(tile + kHalfBytes + row * 128 + phys);
  uint4 a = *lo, b = *hi;
  rot_words<kF16>(a, b, rf);
  *lo = a;
  *hi = b;
}

// The same rotation for 4 consecutive rows of one page (one angle set): all loads first, then
// the math, then the stores.
template <bool kF16>
__device__ __forceinline__ void rotate_4rows_chunk(uint8_t *tile, int row0, int c, const RotF &rf) {
  uint4 a[4], b[4];
#pragma unroll
  for (int rr = 0; rr < 4; ++rr) {
    const int row = row0 + rr;
    const int phys = (c ^ (row & 7)) * 16;
    a[rr] = *reinterpret_cast<const uint4 *>(tile + row * 128 + phys);
    b[rr] = *reinterpret_cast<const uint4 *>(tile + kHalfBytes + row * 128 + phys);
  }
#pragma unroll
  for (int rr = 0; rr < 4; ++rr) rot_words<kF16>(a[rr], b[rr], rf);
#pragma unroll
  for (int rr = 0; rr < 4; ++rr) {
    const int row = row0 + rr;
    const int phys = (c ^ (row & 7)) * 16;
    *reinterpret_cast<uint4 *>(tile + row * 128 + phys) = a[rr];
    *reinterpret_cast<uint4 *>(tile + kHalfBytes + row * 128 + phys) = b[rr];
  }
}

// The identity on 4 rows of one page at chunk c: bf16 in, fp16 out (the absolute-keys mode's
// pages listed at offset 0 need no rotation, only the operand type of the QK product).
__device__ __forceinline__ void convert_4rows_chunk(uint8_t *tile, int row0, int c) {
#pragma unroll
  for (int rr = 0; rr < 4; ++rr) {
    const int row = row0 + rr;
    const int phys = (c ^ (row & 7)) * 16;
#pragma unroll
    for (int hb = 0; hb < 2; ++hb) {
      uint4 *ptr = reinterpret_cast<uint4 *>(tile + hb * kHalfBytes + row * 128 + phys);
      uint4 a = *ptr;
      uint32_t *x = reinterpret_cast<uint32_t *>(&a);
#pragma unroll
      for (int k = 0; k < 4; ++k)
        x[k] = pack_h2(__uint_as_float(x[k] << 16), __uint_as_float(x[k] & 0xFFFF0000u));
      *ptr = a;
    }
  }
}

// (cos, sin) of delta * theta for two frequencies (turn fractions ta, tb), as two independent
// chains. Not inlined: inside the tile loop the angles are needed only when a page offset
// changes, and one shared copy keeps the loop's code compact (inlining the eight angles of a
// chunk there was measured slower); two per call halve the latency-bound chain of one per call.
__device__ __noinline__ float4 angle_cs2(int64_t delta, uint64_t ta, uint64_t tb) {
  float c0, s0, c1, s1;
  rope_cos_sin(delta, ta, c0, s0);
  rope_cos_sin(delta, tb, c1, s1);
  return make_float4(c0, s0, c1, s1);
}

// The same angles with the turn fractions in shared memory and the eight evaluations inlined,
// so that they run as independent chains (one after another they are latency-bound: about
// 300 cycles per angle with two warps per scheduler). Used for the query rows, 64 angles per
// thread before the first product; inside the tile loop the inlined copy costs more in code
// size than it saves (measured), so a page offset change takes chunk_angles.
__device__ __forceinline__ void chunk_angles_ilp(int64_t delta, const uint64_t *turn_s, int c,
                                                 RotF &rf) {
  uint64_t tf[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) tf[e] = turn_s[c * 8 + e];
  float co[8], si[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) rope_cos_sin(delta, tf[e], co[e], si[e]);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    rf.co[k] = make_float2(co[2 * k], co[2 * k + 1]);
    rf.si[k] = make_float2(si[2 * k], si[2 * k + 1]);
  }
}

// Query-side mode: this thread's query row, raw bf16 as loaded, replaced in place by
// R(delta) q in fp16 (delta = m - r for the tile's reference position r). A row's 64 angles
// depend only on its token. With 4 or more query heads per kv head, each aligned group of 4
// lanes holds rows of one token: then every lane evaluates 2 of a chunk's 8 angles and the group
// exchanges them by shuffles (4x fewer evaluations); otherwise each lane evaluates all 64. Two
// chunks per step keep 4 angle chains in flight. Warp-collective when share4 is set. Not
// inlined: the call sits in the softmax loop but runs once per document, and an inlined copy
// there made the whole loop slower (instruction fetch), with no document change at all.
__device__ __noinline__ void qside_rotate_row(uint8_t *tile, int row, int64_t delta,
                                              const uint64_t *turn_s, bool share4, int lane) {
  if (!share4) {
#pragma unroll 1
    for (int c = 0; c < 8; ++c) {
      RotF rq;
      chunk_angles_ilp(delta, turn_s, c, rq);
      rotate_row_chunk<true>(tile, row, c, rq);
    }
    return;
  }
  const int g4 = lane & 3, src0 = lane & ~3;
#pragma unroll 1
  for (int c = 0; c < 8; c += 2) {
    float ca[2], sa[2], cb[2], sb[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      rope_cos_sin(delta, turn_s[(c + u) * 8 + g4], ca[u], sa[u]);
      rope_cos_sin(delta, turn_s[(c + u) * 8 + 4 + g4], cb[u], sb[u]);
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      float co[8], si[8];  // frequency 8(c + u) + e, held by lane src0 + e % 4
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        co[e] = __shfl_sync(0xffffffffu, e < 4 ? ca[u] : cb[u], src0 | (e & 3));
        si[e] = __shfl_sync(0xffffffffu, e < 4 ? sa[u] : sb[u], src0 | (e & 3));
      }
      RotF rq;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        rq.co[k] = make_float2(co[2 * k], co[2 * k + 1]);
        rq.si[k] = make_float2(si[2 * k], si[2 * k + 1]);
      }
      rotate_row_chunk<true>(tile, row, c + u, rq);
    }
  }
}

// (cos, sin) of delta * theta_i for i = 8c .. 8c+7 (exact fp32 angles).
__device__ __forceinline__ void chunk_angles(int64_t delta, const uint64_t *turn, int c, RotF &rf) {
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float4 ab = angle_cs2(delta, turn[c * 8 + 2 * k], turn[c * 8 + 2 * k + 1]);
    rf.co[k] = make_float2(ab.x, ab.z);
    rf.si[k] = make_float2(ab.y, ab.w);
  }
}

// The same angle set held compactly between tiles (a page offset usually spans several tiles):
// fp16 pairs, 8 registers instead of 16 (the kernel runs at its register limit), widened to fp32
// once per rotated tile. cos and sin are within 2^-12 of the fp32 values, the same order as the
// fp16 rounding of the rotated element itself.
struct RotH {
  __half2 co[4], si[4];
};
__device__ __forceinline__ void chunk_angles_h(int64_t delta, const uint64_t *turn, int c,
                                               RotH &rh) {
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float4 ab = angle_cs2(delta, turn[c * 8 + 2 * k], turn[c * 8 + 2 * k + 1]);
    rh.co[k] = __floats2half2_rn(ab.x, ab.z);
    rh.si[k] = __floats2half2_rn(ab.y, ab.w);
  }
}
__device__ __forceinline__ RotF widen(const RotH &rh) {
  RotF rf;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    rf.co[k] = __half22float2(rh.co[k]);
    rf.si[k] = __half22float2(rh.si[k]);
  }
  return rf;
}

// Work that runs on few key tiles (masks on partial pages and question tiles, the question
// keys' per-row rotation, the O rescale when a row's max moves) sits out of line: the softmax
// loop is bound by instruction fetch, and the same blocks inlined there slowed every tile
// (measured with them removed: +6.5% for the mask block, +2.7% for the question rotation).

// Hidden keys of this thread's score row get -inf in TMEM, before the row is loaded for the
// softmax. A document tile hides the slots past each page's valid count (nv[page]); a question
// tile (c0 >= 0, first key token c0) hides the key tokens after the row's own token t_row and
// from the request's end Tb on. Warp-collective.
__device__ __noinline__ void mask_scores_tmem(uint32_t s_col, const int32_t *nv, int c0,
                                              int t_row, int Tb) {
  uint32_t vm[4];  // bit c of vm[c / 32] set = column c visible
  if (c0 < 0) {
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const uint32_t lo = (uint32_t)min(nv[2 * w], 16), hi = (uint32_t)min(nv[2 * w + 1], 16);
      vm[w] = (lo >= 16 ? 0xFFFFu : ((1u << lo) - 1u)) |
              ((hi >= 16 ? 0xFFFFu : ((1u << hi) - 1u)) << 16);
    }
  } else {
    const int lim_tok = min(t_row, Tb - 1) - c0;  // last visible column
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const int h = lim_tok - 32 * w;  // columns 32w .. 32w + h visible
      vm[w] = h < 0 ? 0u : (h >= 31 ? 0xFFFFFFFFu : ((2u << h) - 1u));
    }
  }
#pragma unroll 1
  for (int c = 0; c < 4; ++c) {
    const uint32_t m = c == 0 ? vm[0] : c == 1 ? vm[1] : c == 2 ? vm[2] : vm[3];
    uint32_t r[32];
    tmem_ld32(s_col + c * 32, r);
#pragma unroll
    for (int e = 0; e < 32; ++e)
      if (!((m >> e) & 1u)) r[e] = 0xFF800000u;
    tmem_st32(s_col + c * 32, r);
  }
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// O *= alpha for this thread's row (128 fp32 columns). Warp-collective.
__device__ __noinline__ void rescale_o_tmem(uint32_t o_col, float alpha) {
#pragma unroll 1
  for (int c = 0; c < 4; ++c) {
    uint32_t r[32];
    tmem_ld32(o_col + c * 32, r);
#pragma unroll
    for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * alpha);
    tmem_st32(o_col + c * 32, r);
  }
}

// Question keys (raw): rows row0 .. row0 + 3 of the tile at chunk c, row row0 + rr rotated by
// R(d0 + rr), in place, fp16 out.
__device__ __noinline__ void rotate_question_rows(uint8_t *tile, int row0, int c, int64_t d0,
                                                  const uint64_t *turn) {
#pragma unroll 1
  for (int rr = 0; rr < 4; ++rr) {
    RotF rk;
    chunk_angles(d0 + rr, turn, c, rk);
    rotate_row_chunk<true>(tile, row0 + rr, c, rk);
  }
}

// Bounded wait that also gives up when another role raised the CTA abort flag.
__device__ __forceinline__ bool cta_wait(uint64_t *bar, uint32_t par, volatile int *abort,
                                         uint64_t limit, int32_t *err) {
  const uint32_t a = smem_u32(bar);
  if (mbar_try_wait(a, par)) return true;
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(a, par)) {
    if (*abort) return false;
    if (global_timer_ns() - t0 > limit) {
      *abort = 1;
      set_error(err, LAZY_DEVERR_TIMEOUT);
      return false;
    }
  }
  return true;
}

// Item order of the split units: group g holds split units [g X, g X + gsz), gsz = X except in
// a short last group, and its gsz * ksplit items run chunk-major.
__device__ __forceinline__ int split_item(const TcParams &p, int su, int chunk) {
  const int g = su / p.X, gsz = min(p.X, p.n_split - g * p.X);
  return g * p.X * p.ksplit + chunk * gsz + (su - g * p.X);
}
__device__ __forceinline__ void split_unit(const TcParams &p, int item, int *su, int *chunk) {
  const int g = item / (p.X * p.ksplit), gsz = min(p.X, p.n_split - g * p.X);
  const int w = item - g * p.X * p.ksplit;
  *chunk = w / gsz;
  *su = g * p.X + w % gsz;
}

// The unit of this block and, for a split unit, its chunk and item (item -1 for a whole unit).
// The block index is read through asm volatile, so every call decodes it again: the softmax warps
// call it in their epilogue instead of keeping these values in registers through the tile loop.
struct TcUnit {
  int b, h, t0, chunk, item;
};
__device__ __forceinline__ TcUnit tc_unit(const TcParams &p) {
  int u;
  asm volatile("mov.u32 %0, %%ctaid.x;" : "=r"(u));
  TcUnit t;
  t.chunk = 0;
  t.item = -1;
  if (p.ksplit > 1 && u >= p.n_full) {
    t.item = u - p.n_full;
    int su;
    split_unit(p, t.item, &su, &t.chunk);
    u = p.n_full + su;
  }
  t.b = u / (p.X * p.hkv);
  t.h = (u / p.X) % p.hkv;
  t.t0 = (u % p.X) * 2 * p.TQ;
  return t;
}

// Modes. kRelative: RoPE pools, reference position m0 = the CTA's first question token, QK in
// fp16 from the rotation passes. kAbsolute (LAZY_PREFILL_ABSOLUTE_KEYS): reference position 0,
// so pages listed at offset 0 (keys materialised at absolute positions) need no rotation, only
// a conversion to fp16; everything else as kRelative. kAlibi: the pool's ALiBi mode; nothing
// is rotated (the barriers keep their order), QK in bf16 as loaded, and every score gets
// slope * (n - m) before the row max. kQuerySide (LAZY_PREFILL_TC_QSIDE): the reference moves
// with the documents. Each key tile takes r = the offset of its first page; when r changes the
// raw Q tiles are reloaded and rotated to R(m - r) q, so the pages of that document are only
// converted to fp16, and only pages of another offset in the same tile (a document boundary
// inside the tile) or question keys (R(p - r)) are rotated.
enum { kRelative = 0, kAbsolute = 1, kAlibiMode = 2, kQuerySide = 3 };

template <int kMode>
__global__ void __launch_bounds__(kThreads, 1) prefill_tc_kernel(const __grid_constant__ TcParams p) {
  constexpr bool kAlibi = kMode == kAlibiMode;
  constexpr bool kAbs = kMode == kAbsolute;
  constexpr bool kQS = kMode == kQuerySide;
  constexpr bool kF16 = kMode != kAlibiMode;  // operand type of the QK product
  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = reinterpret_cast<uint8_t *>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t *Qs = sm + kOffQ;
  uint8_t *Ks = sm + kOffK;
  uint8_t *Vs = sm + kOffV;
  KMeta *meta_k = reinterpret_cast<KMeta *>(sm + kOffMetaK);
  SMeta *meta_s = reinterpret_cast<SMeta *>(sm + kOffMetaS);
  uint64_t *bars = reinterpret_cast<uint64_t *>(sm + kOffBar);
  uint64_t *q_full = bars + 0, *q_rot = bars + 1;
  uint64_t *k_full = bars + 2, *k_rot = bars + 5, *k_empty = bars + 8;     // [kNK]
  uint64_t *v_full = bars + 11, *v_empty = bars + 13;                     // [kNV]
  uint64_t *s_full = bars + 15, *p_ready = bars + 17, *o_final = bars + 19;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 20);
  uint64_t *turn_s = reinterpret_cast<uint64_t *>(sm + kOffTurn);
  volatile int *abort = reinterpret_cast<volatile int *>(bars + 21);
  uint64_t *q_ld = bars + 22, *q_rdy = bars + 24;  // [2] query-side mode: Q reloads, re-rotations

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const TcUnit unit = tc_unit(p);
  const int b = unit.b, h = unit.h, t0 = unit.t0;
  const int G = p.G, TQ = p.TQ;
  const int32_t qbeg = p.cu_q[b];
  const int32_t Tb = p.cu_q[b + 1] - qbeg;
  if (t0 >= Tb) return;
  const int32_t q_pos0_b = p.q_pos0[b];
  const int32_t m0 = kAbs ? 0 : q_pos0_b + t0;  // reference position of the rotations
  const int32_t pg0 = p.cu_pages[b], npg = p.cu_pages[b + 1] - pg0;
  const int n_doc = (npg + 7) / 8;
  const int t_end = min(t0 + 2 * TQ, Tb);
  const int n_new = p.has_new ? (t_end + kTile - 1) / kTile : 0;
  // key tiles [lo, lo + n_tiles) of the n_doc + n_new: all of them, or this block's chunk
  int lo = 0, n_tiles = n_doc + n_new;
  if (unit.item >= 0) {
    const int n_all = n_tiles;
    lo = (int)((int64_t)unit.chunk * n_all / p.ksplit);
    n_tiles = (int)((int64_t)(unit.chunk + 1) * n_all / p.ksplit) - lo;
  }

  if (tid == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_rot, 256);
    for (int s = 0; s < kNK; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_rot[s], 256);
      mbar_init(&k_empty[s], 1);
    }
    for (int s = 0; s < kNV; ++s) {
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_ready[i], 128);
    }
    mbar_init(o_final, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&q_ld[i], 1);
      mbar_init(&q_rdy[i], 128);
    }
    *abort = 0;
    fence_barrier_init();
  }
  if (tid >= 64 && tid < 128) turn_s[tid - 64] = p.turn[tid - 64];  // warps 2-3, else idle
  if (warp == 1) {
    asm volatile(
        "tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(
            smem_u32(tmem_slot)));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint64_t lim = p.wait_ns;

  if (warp == 0) {
    // ============================== producer: K runs one tile ahead of V
    if (lane == 0) {
      mbar_arrive_expect_tx(q_full, 2 * kTileBytes);
      for (int i = 0; i < 2; ++i)
        for (int cb = 0; cb < 2; ++cb)
          tma3d(Qs + i * kTileBytes + cb * kHalfBytes, &p.tm_q, cb * 64, h * G,
                qbeg + t0 + i * TQ, q_full);
      // page words of the next document tile, loaded one tile ahead
      uint64_t wnext[8];
      auto load_words = [&](int j) {
#pragma unroll
        for (int pp = 0; pp < 8; ++pp) wnext[pp] = p.words[pg0 + min(j * 8 + pp, npg - 1)];
      };
      if (lo < n_doc) load_words(lo);
      int32_t rows[kNK][8];
      int32_t run8[kNK];  // first block id when the tile's 8 blocks are consecutive, else -1
      int k_issued[kNK] = {0, 0, 0}, v_issued[kNV] = {0, 0};
      int32_t ref_cur = q_pos0_b + t0;  // query-side mode: the reference of the last tile
      bool ok = true;
      for (int e = 0; ok && e <= n_tiles; ++e) {
        if (e < n_tiles) {  // ---- K of tile e (content tile jc = lo + e)
          const int j = e, s = j % kNK, jc = lo + j;
          if (j >= kNK && !cta_wait(&k_empty[s], ((j / kNK) - 1) & 1, abort, lim, p.err)) {
            ok = false;
            break;
          }
          KMeta &mk = meta_k[s];
          SMeta &ms = meta_s[j % kNM];
          uint8_t *kd = Ks + s * kTileBytes;
          if (jc < n_doc) {
            int full = 1;
            uint64_t w[8];
#pragma unroll
            for (int pp = 0; pp < 8; ++pp) w[pp] = wnext[pp];
            if (jc + 1 < n_doc) load_words(jc + 1);
            mk.kind = 0;
#pragma unroll
            for (int pp = 0; pp < 8; ++pp) {
              uint32_t blk = word_block(w[pp]);
              int nv = (int)word_nvalid(w[pp]);
              if (blk >= (uint32_t)p.num_blocks || nv > kPage) {
                set_error(p.err, LAZY_DEVERR_BAD_PAGE);
                blk = 0;
                nv = 0;
              }
              if (jc * 8 + pp >= npg) nv = 0;  // absent page: the last one is loaded again, masked
              ms.nv[pp] = nv;
              ms.pos0[pp] = (int32_t)word_offset(w[pp]);  // ALiBi pools: the page start
              full &= (nv == kPage);
              mk.off[pp] = (int32_t)word_offset(w[pp]);
              rows[s][pp] = (int32_t)((blk * (uint32_t)p.hkv + (uint32_t)h) * kPage);
            }
            ms.kind = 0;
            ms.full = full;
            if (kQS) {
              ref_cur = mk.off[0];
              mk.ref = ref_cur;
            }
            // Documents are encoded into freshly allocated, usually consecutive blocks: then one
            // 8-block box per 64-dim half replaces 8 page boxes.
            bool consec = full != 0;
#pragma unroll
            for (int pp = 1; pp < 8; ++pp)
              consec &= (rows[s][pp] == rows[s][0] + pp * p.hkv * kPage);
            run8[s] = consec ? (rows[s][0] / kPage - h) / p.hkv : -1;
            mbar_arrive_expect_tx(&k_full[s], kTileBytes);
            if (consec) {
              for (int cb = 0; cb < 2; ++cb)
                tma4d(kd + cb * kHalfBytes, &p.tm_k8, cb * 64, 0, h, run8[s], &k_full[s]);
            } else {
#pragma unroll
              for (int pp = 0; pp < 8; ++pp)
                for (int cb = 0; cb < 2; ++cb)
                  tma2d(kd + cb * kHalfBytes + pp * 2048, &p.tm_k, cb * 64, rows[s][pp],
                        &k_full[s]);
            }
          } else {
            const int c0 = (jc - n_doc) * kTile;
            mk.kind = 1;
            mk.c0 = c0;
            if (kQS) mk.ref = ref_cur;  // question keys take R(p - r) for the current r
            ms.kind = 1;
            ms.c0 = c0;
            ms.full = 0;
#pragma unroll
            for (int pp = 0; pp < 8; ++pp) ms.pos0[pp] = q_pos0_b + c0 + pp * kPage;
            mbar_arrive_expect_tx(&k_full[s], kTileBytes);
            for (int cb = 0; cb < 2; ++cb)
              tma3d(kd + cb * kHalfBytes, &p.tm_knew, cb * 64, h, qbeg + c0, &k_full[s]);
          }
          ++k_issued[s];
        }
        if (e >= 1) {  // ---- V of tile e - 1
          const int j = e - 1, s = j % kNV, sk = j % kNK, jc = lo + j;
          if (j >= kNV && !cta_wait(&v_empty[s], ((j / kNV) - 1) & 1, abort, lim, p.err)) {
            ok = false;
            break;
          }
          uint8_t *vd = Vs + s * kTileBytes;
          mbar_arrive_expect_tx(&v_full[s], kTileBytes);
          if (jc < n_doc) {
            if (run8[sk] >= 0) {
              for (int cb = 0; cb < 2; ++cb)
                tma4d(vd + cb * kHalfBytes, &p.tm_v8, cb * 64, 0, h, run8[sk], &v_full[s]);
            } else {
#pragma unroll
              for (int pp = 0; pp < 8; ++pp)
                for (int cb = 0; cb < 2; ++cb)
                  tma2d(vd + cb * kHalfBytes + pp * 2048, &p.tm_v, cb * 64, rows[sk][pp],
                        &v_full[s]);
            }
          } else {
            const int c0 = (jc - n_doc) * kTile;
            for (int cb = 0; cb < 2; ++cb)
              tma3d(vd + cb * kHalfBytes, &p.tm_vnew, cb * 64, h, qbeg + c0, &v_full[s]);
          }
          ++v_issued[s];
        }
      }
      // Drain: every copy issued into a stage has landed before the CTA may exit.
      mbar_wait(q_full, 0, lim);
      for (int s = 0; s < kNK; ++s)
        if (k_issued[s] > 0) mbar_wait(&k_full[s], (k_issued[s] - 1) & 1, lim);
      for (int s = 0; s < kNV; ++s)
        if (v_issued[s] > 0) mbar_wait(&v_full[s], (v_issued[s] - 1) & 1, lim);
    }
  } else if (warp == 1) {
    // ============================== MMA issuer
    if (lane == 0) {
      // Instruction descriptors: fp32 accumulator (bit 4), N = 128 (bits 17-22), M = 128
      // (bits 24-28); A type bits 7-9 and B type bits 10-12 are 0 = fp16, 1 = bf16. QK takes
      // fp16 operands when the rotation passes wrote them (RoPE) and bf16 as loaded (ALiBi,
      // nothing rotated); PV multiplies bf16 weights by bf16 values, V MN-major (bit 16).
      const uint32_t idesc_base = (1u << 4) | ((128u >> 3) << 17) | ((128u >> 4) << 24);
      const uint32_t idesc_bf16 = idesc_base | (1u << 7) | (1u << 10);
      const uint32_t idesc_qk = kF16 ? idesc_base : idesc_bf16;
      const uint32_t idesc_pv = idesc_bf16 | (1u << 16);
      const uint32_t q_addr = smem_u32(Qs), k_addr = smem_u32(Ks), v_addr = smem_u32(Vs);
      // Issue order keeps both softmax groups busy: QK for Q tile 0 of the next key tile is
      // issued as soon as P_0 of this tile is consumed, while group 1 still works on S_1.
      // Descriptors of the tiles' first rows. Shared-memory addresses stay below 2^18 and every
      // offset is a multiple of 16 bytes, so the descriptor of address + off is the base
      // descriptor + off / 16 (the start-address field never carries into the others).
      const uint64_t dq0 = sdesc(q_addr, 16, 1024), dk0 = sdesc(k_addr, 16, 1024);
      const uint64_t dv0 = sdesc(v_addr, kHalfBytes, 1024);
      auto qk = [&](int j, int i) {
        const uint64_t a0 = dq0 + (uint64_t)((i * kTileBytes) >> 4);
        const uint64_t b0 = dk0 + (uint64_t)(((j % kNK) * kTileBytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint64_t off = (uint64_t)(((kk >> 2) * kHalfBytes + (kk & 3) * 32) >> 4);
          mma_ss(tmem + i * 128, a0 + off, b0 + off, idesc_qk, kk > 0);
        }
        mma_commit(&s_full[i]);
      };
      auto pv = [&](int j, int i) {
        const uint64_t b0 = dv0 + (uint64_t)(((j % kNV) * kTileBytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ts(tmem + 256 + i * 128, tmem + i * 128 + kk * 8, b0 + (uint64_t)(kk * (2048 >> 4)),
                 idesc_pv, (j > 0 || kk > 0) ? 1 : 0);
      };
      // Query-side mode: the reference of the last QK; when tile j + 1 has another, QK of each Q
      // tile waits for that tile's re-rotation (q_rdy, phase = re-rotations so far).
      int32_t ref_prev = 0;
      int n_rerot = 0;
      bool ok = cta_wait(q_rot, 0, abort, lim, p.err);
      tc_fence_after();
      if (ok && n_tiles > 0) {
        ok = cta_wait(&k_rot[0], 0, abort, lim, p.err);
        if (ok) {
          if (kQS) ref_prev = meta_k[0].ref;
          tc_fence_after();
          qk(0, 0);
          qk(0, 1);
          mma_commit(&k_empty[0]);
        }
      }
      for (int j = 0; ok && j < n_tiles; ++j) {
        const bool more = j + 1 < n_tiles;
        const int sn = (j + 1) % kNK;
        if (!cta_wait(&v_full[j % kNV], (j / kNV) & 1, abort, lim, p.err)) break;
        if (!cta_wait(&p_ready[0], j & 1, abort, lim, p.err)) break;
        tc_fence_after();
        pv(j, 0);
        bool rerot = false;
        if (more) {
          if (!cta_wait(&k_rot[sn], ((j + 1) / kNK) & 1, abort, lim, p.err)) break;
          if (kQS) {
            const int32_t ref_next = meta_k[sn].ref;
            rerot = ref_next != ref_prev;
            ref_prev = ref_next;
            if (rerot && !cta_wait(&q_rdy[0], n_rerot & 1, abort, lim, p.err)) break;
          }
          tc_fence_after();
          qk(j + 1, 0);
        }
        if (!cta_wait(&p_ready[1], j & 1, abort, lim, p.err)) break;
        tc_fence_after();
        pv(j, 1);
        mma_commit(&v_empty[j % kNV]);
        if (more) {
          if (kQS && rerot) {
            if (!cta_wait(&q_rdy[1], n_rerot & 1, abort, lim, p.err)) break;
            ++n_rerot;
            tc_fence_after();
          }
          qk(j + 1, 1);
          mma_commit(&k_empty[sn]);
        }
      }
      mma_commit(o_final);
      // MMAs still in flight must finish before TMEM is released.
      mbar_wait(o_final, 0, lim);
    }
  } else if (warp >= 4) {
    // ============================== softmax (Q tile i, TMEM lane quadrant warp % 4) + rotation
    // The 256 softmax threads also apply the relative rotation to the key tiles, in the gap
    // between finishing the softmax of tile j and the scores of tile j+1: right after tile j
    // they rotate their share of tile j+2 (the K ring holds 3 tiles, so it has landed, and the
    // MMA issuer needs it only after tile j+1). Share of a thread: 16-byte chunk c of 4
    // consecutive rows of one page; group 0 takes rows 0-63, group 1 rows 64-127. Each thread
    // keeps the (cos, sin) of its page's offset in registers until the offset changes.
    const int i = (warp - 4) >> 2;
    const int row = (warp & 3) * 32 + lane;
    const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const uint32_t s_col = lane_base + i * 128, o_col = lane_base + 256 + i * 128;
    const int t_off = i * TQ + row / G;  // the row's token within the unit (t_row - t0)
    const int t_row = t0 + t_off;
    const float sl2 = p.scale_log2;
    const float slope2 = kAlibi ? p.slopes[h * G + row % G] * 1.4426950408889634f : 0.f;
    const int32_t m_row = q_pos0_b + t_row;  // the row's logical position
    const uint64_t *turn = p.turn;
    const int st = tid - 128;               // 0..255
    const int rc = st & 7, rrow0 = (st >> 3) * 4;  // rotation share: chunk rc, rows rrow0..+3
    float m_run = -INFINITY, l_run = 0.f;
    int32_t cur_ref = 0;  // query-side mode: r of the rows now in this group's Q tile
    int n_reload = 0;     // query-side mode: raw Q reloads of this tile so far
    bool reload_open = false;
    bool ok = cta_wait(q_full, 0, abort, lim, p.err);
    if (kQS) {
      // the first tile's reference, then this thread's row rotated to R(m - r)
      cur_ref = q_pos0_b + t0;
      if (ok && n_tiles > 0) {
        ok = cta_wait(&k_full[0], 0, abort, lim, p.err);
        if (ok) cur_ref = meta_k[0].ref;
      }
      if (__all_sync(0xffffffffu, ok)) {  // the row rotation exchanges angles between lanes
        qside_rotate_row(Qs + i * kTileBytes, row, (int64_t)m_row - cur_ref, turn_s, G >= 4,
                         lane);
        fence_async_smem();
      }
    } else if (ok && !kAlibi) {
      // this thread's own query row of Q tile i, rotated to R(m - m0)
#pragma unroll 1
      for (int c = 0; c < 8; ++c) {
        RotF rq;
        chunk_angles_ilp(kAbs ? (int64_t)(q_pos0_b + t_row) : (int64_t)(i * TQ + row / G),
                         turn_s, c, rq);
        rotate_row_chunk<kF16>(Qs + i * kTileBytes, row, c, rq);
      }
      fence_async_smem();
    }
    mbar_arrive(q_rot);
    int64_t cached = INT64_MIN;
    RotH rp;
    auto rotate_tile = [&](int jj) -> bool {
      const int s = jj % kNK;
      if (!cta_wait(&k_full[s], (jj / kNK) & 1, abort, lim, p.err)) return false;
      const KMeta &mt = meta_k[s];
      uint8_t *kt = Ks + s * kTileBytes;
      if (kAlibi) {
        // no rotation: the tile is used as loaded
      } else if (mt.kind == 0) {
        // one relative rotation R(o - m0) per page (query-side mode: R(o - r))
        const int64_t d = (int64_t)mt.off[rrow0 >> 4] - (kQS ? (int64_t)mt.ref : (int64_t)m0);
        if ((kAbs || kQS) && d == 0) {  // offset at the reference: only the operand type
          convert_4rows_chunk(kt, rrow0, rc);
        } else {
          if (d != cached) {
            cached = d;
            chunk_angles_h(d, turn, rc, rp);
          }
          rotate_4rows_chunk<kF16>(kt, rrow0, rc, widen(rp));
        }
      } else {
        // question keys: raw, rotated by R(p - m0) row by row (the absolute mode re-reads the
        // request's first position here rather than keeping it in a register)
        const int64_t q0 = (kAbs || kQS) ? (int64_t)p.q_pos0[tc_unit(p).b] : 0;
        rotate_question_rows(kt, rrow0, rc,
                             kAbs  ? q0 + mt.c0 + rrow0
                             : kQS ? q0 + mt.c0 + rrow0 - mt.ref
                                   : (int64_t)(mt.c0 + rrow0 - t_row + t_off),
                             turn);
      }
      if (!kAlibi) fence_async_smem();
      mbar_arrive(&k_rot[s]);
      return true;
    };
    for (int jj = 0; ok && jj < 2 && jj < n_tiles; ++jj) ok = rotate_tile(jj);
    for (int j = 0; ok && j < n_tiles; ++j) {
      if (!cta_wait(&s_full[i], j & 1, abort, lim, p.err)) {
        ok = false;
        break;
      }
      tc_fence_after();
      // Query-side mode: a new reference at tile j + 1 (its K metadata stays until QK of that
      // tile). QK of tile j, the last product that reads this Q tile before then, is complete, so
      // the raw rows are reloaded now and rotated after this tile's softmax.
      int32_t ref_next = cur_ref;
      if (kQS && j + 1 < n_tiles) {
        ref_next = meta_k[(j + 1) % kNK].ref;
        if (ref_next != cur_ref && row == 0) {
          mbar_arrive_expect_tx(&q_ld[i], kTileBytes);
          for (int cb = 0; cb < 2; ++cb)
            tma3d(Qs + i * kTileBytes + cb * kHalfBytes, &p.tm_q, cb * 64, h * G,
                  qbeg + t0 + i * TQ, &q_ld[i]);
          reload_open = true;
        }
      }
      const SMeta &mt = meta_s[j % kNM];
      const bool doc = mt.kind == 0;
      const bool need_mask = !(doc && mt.full);
      // The whole score row is loaded at once; the running max m_use only moves when the
      // tile's max exceeds it by more than 8 (log2 domain, so weights stay <= 2^8), and then
      // this row's sum and (below) O are scaled by alpha = 2^(m_old - m_new).
      float m_use = m_run, alpha = 1.f;
      // hidden keys get -inf: they drop out of the max and ex2(-inf) = 0
      if (need_mask) mask_scores_tmem(s_col, mt.nv, doc ? -1 : mt.c0, t_row, Tb);
      uint32_t r[128];
      tmem_ld128(s_col, r);
      if (kAlibi) {
        // log2-domain scores with the bias: slope * (n - m), n = pos0 of the 16-key group + e
#pragma unroll
        for (int pg = 0; pg < 8; ++pg) {
          const float base = slope2 * (float)(mt.pos0[pg] - m_row);
#pragma unroll
          for (int e = 0; e < 16; e += 2) {
            const float2 bias = __ffma2_rn(make_float2(slope2, slope2),
                                           make_float2((float)e, (float)(e + 1)),
                                           make_float2(base, base));
            const float2 t = __ffma2_rn(
                make_float2(__uint_as_float(r[pg * 16 + e]), __uint_as_float(r[pg * 16 + e + 1])),
                make_float2(sl2, sl2), bias);
            r[pg * 16 + e] = __float_as_uint(t.x);
            r[pg * 16 + e + 1] = __float_as_uint(t.y);
          }
        }
      }
      // max with eight independent chains of three-input maxima (one running max would be a
      // 128-long chain)
      float cmk[8];
#pragma unroll
      for (int k = 0; k < 8; ++k)
        cmk[k] = fmaxf(__uint_as_float(r[2 * k]), __uint_as_float(r[2 * k + 1]));
#pragma unroll
      for (int e = 16; e < 128; e += 16) {
#pragma unroll
        for (int k = 0; k < 8; ++k)
          cmk[k] = fmax3(cmk[k], __uint_as_float(r[e + 2 * k]), __uint_as_float(r[e + 2 * k + 1]));
      }
      const float cm = fmax3(fmax3(cmk[0], cmk[1], cmk[2]), fmax3(cmk[3], cmk[4], cmk[5]),
                             fmaxf(cmk[6], cmk[7]));
      const float cm2 = kAlibi ? cm : cm * sl2;
      const float sle = kAlibi ? 1.f : sl2;  // scale still to apply in the exponent
      if (cm2 > m_use + 8.f) {  // includes the first finite max (m_use = -inf)
        alpha = (m_use == -INFINITY) ? 0.f : ex2(m_use - cm2);
        m_use = cm2;
      }
      const float neg_m = (m_use == -INFINITY) ? 0.f : -m_use;
      float2 lp2[4];  // row-sum partials, four independent chains
#pragma unroll
      for (int k = 0; k < 4; ++k) lp2[k] = make_float2(0.f, 0.f);
      // weights as bf16 pairs into S's first 64 columns (all of S is in registers by now)
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        uint32_t pw[16];
#pragma unroll
        for (int e2 = 0; e2 < 32; e2 += 2) {
          const int e = q4 * 32 + e2;
          const float2 t = __ffma2_rn(make_float2(__uint_as_float(r[e]), __uint_as_float(r[e + 1])),
                                      make_float2(sle, sle), make_float2(neg_m, neg_m));
          const float s0 = ex2(t.x), s1 = ex2(t.y);
          lp2[(e2 >> 1) & 3] = __fadd2_rn(lp2[(e2 >> 1) & 3], make_float2(s0, s1));
          pw[e2 / 2] = pack_bf2(s0, s1);
        }
        tmem_st16(s_col + q4 * 16, pw);
      }
      // O *= alpha for rows whose max moved (warp-collective TMEM access); O holds data only
      // after the first tile's PV.
      if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) rescale_o_tmem(o_col, alpha);
      const float2 lps = __fadd2_rn(__fadd2_rn(lp2[0], lp2[1]), __fadd2_rn(lp2[2], lp2[3]));
      const float lp = lps.x + lps.y;
      asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      l_run = l_run * alpha + lp;
      m_run = m_use;
      tc_fence_before();
      mbar_arrive(&p_ready[i]);
      if (kQS && ref_next != cur_ref) {
        const bool landed = cta_wait(&q_ld[i], n_reload & 1, abort, lim, p.err);
        if (landed) reload_open = false;
        if (!__all_sync(0xffffffffu, landed)) {  // the row rotation is warp-collective
          ok = false;
          break;
        }
        ++n_reload;
        qside_rotate_row(Qs + i * kTileBytes, row, (int64_t)m_row - ref_next, turn_s, G >= 4,
                         lane);
        fence_async_smem();
        mbar_arrive(&q_rdy[i]);
        cur_ref = ref_next;
      }
      if (j + 2 < n_tiles && !rotate_tile(j + 2)) {
        ok = false;
        break;
      }
    }
    // a reload still in flight after an abort lands before the CTA exits
    if (kQS && reload_open) mbar_wait(&q_ld[i], n_reload & 1, lim);
    // epilogue: O / l -> bf16 rows, lse
    ok = ok && cta_wait(o_final, 0, abort, lim, p.err);
    // Each thread holds one row of its group's O tile. The rows are staged in shared memory in
    // the 128-byte-swizzled layout of a TMA box (chunk q of row r at 16 (q ^ (r & 7)), so a
    // warp's 32 rows spread over all banks) and leave in a few TMA stores: one store per lane
    // and row would be 32 separate segments per instruction. The Q tiles and the K/V rings are
    // free once o_final has arrived (every MMA, hence every copy it read, is done).
    const TcUnit ue = tc_unit(p);  // decoded again (see tc_unit)
    if (ue.item >= 0) {
      // chunk of a split unit: fp32 O / l (zeros when the chunk saw no key of the row) for the
      // combine, staged as four 16 KB boxes of 32 dims x 128 rows in the K/V rings
      uint8_t *stg = Ks + i * 65536;
      if (ok) {
        tc_fence_after();
        const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t r[32];
          tmem_ld32(o_col + c * 32, r);
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            float f[4];
#pragma unroll
            for (int k = 0; k < 4; ++k)
              f[k] = l_run > 0.f ? __uint_as_float(r[4 * q + k]) * inv : 0.f;
            *reinterpret_cast<float4 *>(stg + c * 16384 + row * 128 + ((q ^ (row & 7)) << 4)) =
                make_float4(f[0], f[1], f[2], f[3]);
          }
        }
        fence_async_smem();
        if (t_row < Tb)
          p.part_lse[(size_t)ue.item * 256 + i * 128 + row] =
              l_run > 0.f ? m_run + log2f(l_run) : -INFINITY;
      }
      group_bar(i);
      if (ok && row == 0) {
        for (int c = 0; c < 4; ++c)
          tma_store2d(&p.tm_part, stg + c * 16384, c * 32, ue.item * 256 + i * 128);
        bulk_commit_and_wait();
      }
    } else {
      // whole unit: bf16 O / l. A Q tile whose TQ tokens all belong to the request goes out as
      // two TMA boxes (one per 64-dim half) staged in its own Q slot; a ragged last tile keeps
      // per-row stores, since its box would reach into the next request's rows.
      const bool full_tile = ue.t0 + (i + 1) * TQ <= Tb;
      const int qh = ue.h * G + row % G;
      const int32_t qb = p.cu_q[ue.b];
      uint8_t *stg = Qs + i * kTileBytes;
      if (ok) {
        tc_fence_after();
        const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
        const bool valid_row = t_row < Tb;
        __nv_bfloat16 *dst = p.out + ((size_t)(qb + t_row) * p.hq + qh) * 128;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t r[32];
          tmem_ld32(o_col + c * 32, r);
#pragma unroll
          for (int e = 0; e < 32; e += 8) {
            float f[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) f[k] = l_run > 0.f ? __uint_as_float(r[e + k]) * inv : 0.f;
            const uint4 v = pack16<__nv_bfloat16>(f);
            if (full_tile) {
              const int q = (c & 1) * 4 + e / 8;  // 16-byte chunk within the 64-dim half
              *reinterpret_cast<uint4 *>(stg + (c >> 1) * kHalfBytes + row * 128 +
                                         ((q ^ (row & 7)) << 4)) = v;
            } else if (valid_row) {
              *reinterpret_cast<uint4 *>(dst + c * 32 + e) = v;
            }
          }
        }
        if (full_tile) fence_async_smem();
        if (valid_row)
          p.lse[(size_t)(qb + t_row) * p.hq + qh] =
              l_run > 0.f ? (m_run + log2f(l_run)) * 0.69314718055994531f : -INFINITY;
      }
      if (full_tile) {
        group_bar(i);
        if (ok && row == 0) {
          for (int hb = 0; hb < 2; ++hb)
            tma_store3d(&p.tm_out, stg + hb * kHalfBytes, hb * 64, ue.h * G,
                        qb + ue.t0 + i * TQ);
          bulk_commit_and_wait();
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem));
  }
}

// Merges the K = ksplit chunk results of every row of the split units: each warp takes R rows,
// lane l holding dims 4l .. 4l + 3. With lse_c the chunks' log2-domain lse and M their max, a
// row is sum_c 2^(lse_c - M) o_c / W, W = sum_c 2^(lse_c - M), and its lse (M + log2 W) ln 2.
// Every chunk wrote every valid row (zeros and -inf when it saw no key), so all R K loads of a
// warp are issued before any weight or row validity is known: one memory round trip per warp.
template <int K, int R>
__global__ void __launch_bounds__(256) prefill_combine_kernel(const __grid_constant__ TcParams p) {
  const int gw = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  const int n_rows = p.n_split * 256;
  float lse[R][K];
  float4 o[R][K];
  bool valid[R];
  size_t dst[R];
  // The partial loads do not wait for the row's validity (which needs cu_q): every item's 256
  // rows exist in the workspace, and a row past its request is loaded but not used.
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const int gr = min(gw * R + r, n_rows - 1);  // global row: split unit gr / 256, row gr % 256
    const int su = gr >> 8, r256 = gr & 255;
#pragma unroll
    for (int c = 0; c < K; ++c) {
      const size_t it = (size_t)split_item(p, su, c) * 256 + r256;
      lse[r][c] = p.part_lse[it];
      o[r][c] = *reinterpret_cast<const float4 *>(p.part_o + it * 128 + lane * 4);
    }
  }
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const int gr = gw * R + r;
    valid[r] = false;
    dst[r] = 0;
    if (gr < n_rows) {
      const int su = gr >> 8, r256 = gr & 255;
      const int u = p.n_full + su;
      const int b = u / (p.X * p.hkv), h = (u / p.X) % p.hkv;
      const int t0 = (u % p.X) * 2 * p.TQ;
      const int32_t qbeg = p.cu_q[b], Tb = p.cu_q[b + 1] - qbeg;
      const int i = r256 >> 7, row = r256 & 127;
      const int t_row = t0 + i * p.TQ + row / p.G;
      valid[r] = t_row < Tb;
      dst[r] = (size_t)(qbeg + t_row) * p.hq + h * p.G + row % p.G;
    }
  }
#pragma unroll
  for (int r = 0; r < R; ++r) {
    if (!valid[r]) continue;
    float M = -INFINITY;
#pragma unroll
    for (int c = 0; c < K; ++c) M = fmaxf(M, lse[r][c]);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float W = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int c = 0; c < K; ++c) {
        const float w = lse[r][c] == -INFINITY ? 0.f : exp2f(lse[r][c] - M);
        W += w;
        acc.x += w * o[r][c].x;
        acc.y += w * o[r][c].y;
        acc.z += w * o[r][c].z;
        acc.w += w * o[r][c].w;
      }
    }
    const float inv = W > 0.f ? 1.f / W : 0.f;
    __nv_bfloat162 v0 = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
    __nv_bfloat162 v1 = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
    uint2 pk;
    pk.x = *reinterpret_cast<uint32_t *>(&v0);
    pk.y = *reinterpret_cast<uint32_t *>(&v1);
    *reinterpret_cast<uint2 *>(p.out + dst[r] * 128 + lane * 4) = pk;
    if (lane == 0) p.lse[dst[r]] = W > 0.f ? (M + log2f(W)) * 0.69314718055994531f : -INFINITY;
  }
}

// Launch of the combine for K chunks: R = 16 / K rows per warp keeps 16 loads in flight.
template <int K>
void launch_combine(const TcParams &tp, cudaStream_t s) {
  constexpr int R = (16 / K) > 0 ? 16 / K : 1;
  const int rows = tp.n_split * 256, warps = (rows + R - 1) / R;
  prefill_combine_kernel<K, R><<<(warps + 7) / 8, 256, 0, s>>>(tp);
}

// ---------------------------------------------------------------- host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  }
  return fn;
}

// Tensor [dims[rank-1]]...[dims[0]] (dims innermost first; bf16 unless dt says otherwise),
// 128B swizzle, zero OOB fill.
int make_map(CUtensorMap *m, void *base, int rank, const cuuint64_t *dims,
             const cuuint64_t *strides_bytes, const cuuint32_t *box,
             CUtensorMapDataType dt = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) {
    record_msg("cuTensorMapEncodeTiled is unavailable");
    return LAZY_ERR_CUDA;
  }
  cuuint32_t es[4] = {1, 1, 1, 1};
  CUresult r = enc(m, dt, rank, base, dims, strides_bytes, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    record_msg("cuTensorMapEncodeTiled rejected a tensor map");
    return LAZY_ERR_CUDA;
  }
  return LAZY_OK;
}

}  // namespace

int ensure_pool_tmaps(lazy_pool *p) {
  if (p->dtype != LAZY_DTYPE_BF16 || p->d != 128 || p->page_size != kPage)
    return LAZY_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> g(p->mu);
  if (p->tmaps_ready) return LAZY_OK;
  // rows (block * Hkv + h) * 16 + slot, 128 dims; box 16 rows x 64 dims
  const cuuint64_t dims[2] = {128, (cuuint64_t)p->num_blocks * p->hkv * kPage};
  const cuuint64_t strides[1] = {256};
  const cuuint32_t box[2] = {64, 16};
  int rc = make_map(reinterpret_cast<CUtensorMap *>(p->tmap_k), p->k, 2, dims, strides, box);
  if (rc != LAZY_OK) return rc;
  rc = make_map(reinterpret_cast<CUtensorMap *>(p->tmap_v), p->v, 2, dims, strides, box);
  if (rc != LAZY_OK) return rc;
  // [block][kv head][slot][dim]; box = 64 dims x 16 slots x 1 head x 8 blocks
  const cuuint64_t dims4[4] = {128, (cuuint64_t)kPage, (cuuint64_t)p->hkv,
                               (cuuint64_t)p->num_blocks};
  const cuuint64_t strides4[3] = {256, 256 * kPage, (cuuint64_t)256 * kPage * p->hkv};
  const cuuint32_t box4[4] = {64, (cuuint32_t)kPage, 1, 8};
  rc = make_map(reinterpret_cast<CUtensorMap *>(p->tmap_k8), p->k, 4, dims4, strides4, box4);
  if (rc != LAZY_OK) return rc;
  rc = make_map(reinterpret_cast<CUtensorMap *>(p->tmap_v8), p->v, 4, dims4, strides4, box4);
  if (rc != LAZY_OK) return rc;
  // one page per box: the halves (dims 0-63, 64-127) are an outer dimension of stride 128 B, so
  // the box lands half-major, exactly as two boxes of the 2-D view would
  const cuuint64_t dims3[3] = {64, (cuuint64_t)p->num_blocks * p->hkv * kPage, 2};
  const cuuint64_t strides3[2] = {256, 128};
  const cuuint32_t box3[3] = {64, (cuuint32_t)kPage, 2};
  rc = make_map(reinterpret_cast<CUtensorMap *>(p->tmap_k3), p->k, 3, dims3, strides3, box3);
  if (rc != LAZY_OK) return rc;
  rc = make_map(reinterpret_cast<CUtensorMap *>(p->tmap_v3), p->v, 3, dims3, strides3, box3);
  if (rc != LAZY_OK) return rc;
  p->tmaps_ready = true;
  return LAZY_OK;
}

int prefill_tc_supported(const lazy_pool *p, int32_t hq) {
  if (p->dtype != LAZY_DTYPE_BF16 || p->d != 128 || p->page_size != kPage)
    return LAZY_ERR_UNSUPPORTED;
  if (hq % p->hkv) return LAZY_ERR_INVALID_ARG;
  // a 128-row Q tile holds 128 / g whole tokens of the group; groups up to 32 (MQA with 32
  // query heads) are the parity-tested range
  const int g = hq / p->hkv;
  if (g < 1 || g > 32 || (g & (g - 1))) return LAZY_ERR_UNSUPPORTED;
  return LAZY_OK;
}

namespace {
// Last-wave split. A whole unit takes one unit-time T on its SM; a chunk of a unit cut into k
// takes T / k plus a fixed cost (Q load and rotation, pipeline fill, epilogue) taken as 3% of T.
// The units beyond the last full wave of `sms` blocks are cut into the k in 2..kMaxSplit that
// minimises (full waves) + ceil(split units * k / sms) * (1 / k + 0.03); the split is planned
// only when that beats ceil(units / sms) waves by 3%.
struct TcPlan {
  int X = 0, units = 0, n_full = 0, n_split = 0, ksplit = 1, grid = 0;
  size_t ws_bytes = 0;  // partial results: [items][256][128] O plus [items][256] lse, fp32
};

TcPlan plan_tc(int32_t batch, int32_t hkv, int32_t TQ, int32_t max_q_len, int sms) {
  TcPlan pl;
  pl.X = (max_q_len + 2 * TQ - 1) / (2 * TQ);
  pl.units = pl.X * hkv * batch;
  pl.n_full = pl.grid = pl.units;
  if (sms <= 0 || pl.units == 0) return pl;
  const int waves = pl.units / sms;
  const int n_full = waves * sms, r = pl.units - n_full;
  if (r == 0) return pl;
  const double whole = (double)waves + 1.0;
  double best = 0.97 * whole;
  int best_k = 1;
  for (int k = 2; k <= kMaxSplit; ++k) {
    const double t = waves + std::ceil((double)r * k / sms) * (1.0 / k + 0.03);
    if (t < best) {
      best = t;
      best_k = k;
    }
  }
  if (best_k == 1) return pl;
  pl.n_full = n_full;
  pl.n_split = r;
  pl.ksplit = best_k;
  pl.grid = n_full + r * best_k;
  pl.ws_bytes = (size_t)r * best_k * 256 * (128 + 1) * sizeof(float);
  return pl;
}

int schedule_sms(const lazy_pool *p) { return p->schedule_sms > 0 ? p->schedule_sms : p->num_sms; }
}  // namespace

int prefill_tc_workspace_bytes(lazy_pool *p, int32_t batch, int32_t max_q_len, int32_t hq,
                               size_t *bytes) {
  const int G = hq / p->hkv;
  *bytes = plan_tc(batch, p->hkv, 128 / G, max_q_len, schedule_sms(p)).ws_bytes;
  return LAZY_OK;
}

int prefill_tc(lazy_pool *p, const PrefillParams &pp, int32_t max_q_len, cudaStream_t s) {
  TcParams tp;
  memset(&tp, 0, sizeof(tp));
  int rc;
  rc = ensure_pool_tmaps(p);
  if (rc != LAZY_OK) return rc;
  {
    std::lock_guard<std::mutex> g(p->mu);
    memcpy(&tp.tm_k, p->tmap_k, sizeof(CUtensorMap));
    memcpy(&tp.tm_v, p->tmap_v, sizeof(CUtensorMap));
    memcpy(&tp.tm_k8, p->tmap_k8, sizeof(CUtensorMap));
    memcpy(&tp.tm_v8, p->tmap_v8, sizeof(CUtensorMap));
  }
  const int G = pp.G, TQ = 128 / G;
  {
    const cuuint64_t dims[3] = {128, (cuuint64_t)pp.hq, (cuuint64_t)pp.total_q};
    const cuuint64_t strides[2] = {256, (cuuint64_t)pp.hq * 256};
    const cuuint32_t box[3] = {64, (cuuint32_t)G, (cuuint32_t)TQ};
    rc = make_map(&tp.tm_q, const_cast<void *>(pp.q), 3, dims, strides, box);
    if (rc != LAZY_OK) return rc;
    rc = make_map(&tp.tm_out, pp.out, 3, dims, strides, box);
    if (rc != LAZY_OK) return rc;
  }
  if (pp.k_new) {
    const cuuint64_t dims[3] = {128, (cuuint64_t)pp.hkv, (cuuint64_t)pp.total_q};
    const cuuint64_t strides[2] = {256, (cuuint64_t)pp.hkv * 256};
    const cuuint32_t box[3] = {64, 1, 128};
    rc = make_map(&tp.tm_knew, const_cast<void *>(pp.k_new), 3, dims, strides, box);
    if (rc != LAZY_OK) return rc;
    rc = make_map(&tp.tm_vnew, const_cast<void *>(pp.v_new), 3, dims, strides, box);
    if (rc != LAZY_OK) return rc;
  }
  tp.cu_q = pp.cu_q;
  tp.q_pos0 = pp.q_pos0;
  tp.words = pp.words;
  tp.cu_pages = pp.cu_pages;
  tp.turn = pp.turn;
  tp.out = reinterpret_cast<__nv_bfloat16 *>(pp.out);
  tp.lse = pp.lse;
  tp.err = pp.err;
  tp.batch = pp.batch;
  tp.hkv = pp.hkv;
  tp.hq = pp.hq;
  tp.num_blocks = pp.num_blocks;
  tp.G = G;
  tp.TQ = TQ;
  tp.has_new = pp.k_new != nullptr;
  tp.scale_log2 = pp.scale_log2;
  tp.wait_ns = pp.wait_ns;
  tp.slopes = pp.slopes;
  static std::once_flag attr_once;
  static cudaError_t attr_rc = cudaSuccess;
  std::call_once(attr_once, [] {
    for (auto fn : {prefill_tc_kernel<kRelative>, prefill_tc_kernel<kAbsolute>,
                    prefill_tc_kernel<kAlibiMode>, prefill_tc_kernel<kQuerySide>}) {
      const cudaError_t e = cudaFuncSetAttribute(
          fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
      if (e != cudaSuccess && attr_rc == cudaSuccess) attr_rc = e;
    }
  });
  LAZY_CUDA_TRY(attr_rc);
  // The split runs only when the caller's workspace holds its partial results.
  TcPlan pl = plan_tc(pp.batch, pp.hkv, TQ, max_q_len, schedule_sms(p));
  if (pl.ksplit > 1 && (!pp.workspace || pp.workspace_bytes < pl.ws_bytes ||
                        ((uintptr_t)pp.workspace & 15))) {
    pl.n_full = pl.grid = pl.units;
    pl.n_split = 0;
    pl.ksplit = 1;
  }
  tp.X = pl.X;
  tp.n_full = pl.n_full;
  tp.n_split = pl.n_split;
  tp.ksplit = pl.ksplit;
  if (pl.ksplit > 1) {
    const size_t rows = (size_t)pl.n_split * pl.ksplit * 256;
    tp.part_o = reinterpret_cast<float *>(pp.workspace);
    tp.part_lse = tp.part_o + rows * 128;
    const cuuint64_t dims[2] = {128, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {128 * sizeof(float)};
    const cuuint32_t box[2] = {32, 128};
    rc = make_map(&tp.tm_part, tp.part_o, 2, dims, strides, box, CU_TENSOR_MAP_DATA_TYPE_FLOAT32);
    if (rc != LAZY_OK) return rc;
  }
  if (pp.slopes)
    prefill_tc_kernel<kAlibiMode><<<pl.grid, kThreads, kSmemBytes, s>>>(tp);
  else if (pp.tc_qside)
    prefill_tc_kernel<kQuerySide><<<pl.grid, kThreads, kSmemBytes, s>>>(tp);
  else if (pp.absolute)
    prefill_tc_kernel<kAbsolute><<<pl.grid, kThreads, kSmemBytes, s>>>(tp);
  else
    prefill_tc_kernel<kRelative><<<pl.grid, kThreads, kSmemBytes, s>>>(tp);
  LAZY_CUDA_TRY(cudaGetLastError());
  if (pl.ksplit > 1) {
    switch (pl.ksplit) {
      case 2: launch_combine<2>(tp, s); break;
      case 3: launch_combine<3>(tp, s); break;
      case 4: launch_combine<4>(tp, s); break;
      case 5: launch_combine<5>(tp, s); break;
      case 6: launch_combine<6>(tp, s); break;
      case 7: launch_combine<7>(tp, s); break;
      default: launch_combine<8>(tp, s); break;
    }
    LAZY_CUDA_TRY(cudaGetLastError());
  }
  return LAZY_OK;
}

}  // namespace lazy
