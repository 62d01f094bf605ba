/*
 * lazy_attn.h — C ABI of the deferred-RoPE ("lazy") attention library for GB300 (sm_103a).
 *
 * The operation: attention in which RoPE is not baked into the cached keys. Each retrieved
 * document's K/V is stored once, rotated only at its document-local positions 0..L-1, in a paged
 * pool; a request attends that single copy at any logical offset o. Source: "LazyAttention:
 * Efficient Retrieval-Augmented Generation with Deferred Positional Encoding" (technical
 * summaries: "Core concept: deferred positional encoding", "Technical implementation" with its
 * prefill and decode parts, "Mathematical equivalence").
 *
 * Conventions (fixed for the whole library):
 *   RoPE     R(p) rotates the pair (x_i, x_{i+D/2}) by p * theta_i, theta_i = base^(-2i/D)
 *            (half-split pairing, as in Llama-3.x, the summaries' evaluation models).
 *   Scores   s = sm_scale * (R(m) q) . (R(o + j) k) = sm_scale * (R(m - o) q) . (R(j) k);
 *            the pool stores R(j) k, so a page attended at offset o needs only R(m - o) on q
 *            (decode) or one relative rotation of the key tile (prefill).
 *   lse      natural log of sum_k exp(s_k) over the visible keys (s already scaled).
 *   GQA      query head qh reads kv head qh / (num_q_heads / num_kv_heads).
 *   Layout   pool pages K_pool, V_pool: [num_blocks][num_kv_heads][page_size][head_dim],
 *            row-major, pool dtype; one (block, kv head) page is contiguous.
 *            q: [tokens][num_q_heads][head_dim]; k/v inputs: [tokens][num_kv_heads][head_dim].
 *   Page word (one uint64 per page of a request's page table; see lazy_pack_page):
 *            bits 0-31 block id, bits 32-57 logical offset o of the segment the page belongs to
 *            (26 bits), bits 58-63 n_valid - 1 (tokens valid in the page, 1..64).
 *   Pointers Arguments named d_* or documented "device" are device pointers; the rest are
 *            host pointers. All device buffers are owned by the caller. The pool handle owns
 *            only host metadata and a few bytes of device state (error word, angle table).
 *   Streams  Every device operation is enqueued on the given stream and returns without
 *            waiting. Argument errors are returned synchronously; faults the kernels detect
 *            (a corrupt page word, an expired bounded wait) set bits in the pool's device error
 *            word, read by lazy_get_device_error. Kernels never trap.
 *   Status   Every function returns LAZY_OK (0) or a negative LAZY_ERR_* code.
 */
#ifndef LAZY_ATTN_H
#define LAZY_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct lazy_pool lazy_pool;
/* Same type as cudaStream_t; 0 is the legacy default stream. */
typedef struct CUstream_st *lazy_stream_t;

enum {
    LAZY_OK = 0,
    LAZY_ERR_INVALID_ARG = -1,   /* null pointer, bad size, inconsistent shapes */
    LAZY_ERR_OUT_OF_BLOCKS = -2, /* the pool's free list cannot satisfy the request */
    LAZY_ERR_UNSUPPORTED = -3,   /* dtype / head_dim / page_size / group size not built */
    LAZY_ERR_CUDA = -4,          /* a CUDA runtime call failed (message: lazy_last_error) */
    LAZY_ERR_BAD_PAGE = -5,      /* device error word: a page word pointed outside the pool */
    LAZY_ERR_TIMEOUT = -6,       /* device error word: a bounded wait inside a kernel expired */
    LAZY_ERR_SCRATCH_LIMIT = -7  /* lazy_attn_decode_noalloc: the call needs more scratch than
                                    the library's fixed array holds */
};

enum { LAZY_DTYPE_BF16 = 0, LAZY_DTYPE_FP32 = 1 };

/* Bits of the device error word. */
enum { LAZY_DEVERR_BAD_PAGE = 1, LAZY_DEVERR_TIMEOUT = 2 };

/* Prefill kernel choice (lazy_attn_prefill `flags`). */
enum {
    LAZY_PREFILL_AUTO = 0,  /* tensor-core kernel when bf16, head_dim 128 and the group size
                               (num_q_heads / num_kv_heads) is a power of two <= 32; else
                               CUDA-core. On RoPE pools the tensor-core kernel multiplies the
                               rotated query rows and key tiles as fp16 (11 significant bits,
                               rotated in fp32 and rounded once); query and key elements must
                               then stay below 65504 in magnitude (use LAZY_PREFILL_SIMT for
                               larger ones). P.V and the ALiBi mode's Q.K use bf16 operands. */
    LAZY_PREFILL_SIMT = 1,  /* CUDA-core kernel, fp32 arithmetic, group size <= 64 */
    LAZY_PREFILL_TC = 2,    /* tcgen05/TMEM kernel; LAZY_ERR_UNSUPPORTED if the shape is not */
    LAZY_PREFILL_SIMT_QSIDE = 3, /* the CUDA-core kernel with the query-side variant of the
                                    relative rotation: cached key pages are used as stored
                                    (R(j) k) and the queries take R(m - o) once per document
                                    offset o, instead of every key page taking R(o - m0) */
    LAZY_PREFILL_TC_QSIDE = 4, /* the tensor-core kernel with the query-side variant: each
                                  128-key tile takes the offset r of its first page as its
                                  reference; when r changes the query tiles are reloaded and
                                  rotated to R(m - r) q, pages at offset r are only converted to
                                  the fp16 operand type, and pages of another offset in the same
                                  tile and the question's own keys take R(o - r) and R(p - r).
                                  Same shapes and LAZY_ERR_UNSUPPORTED rule as LAZY_PREFILL_TC;
                                  on ALiBi pools it is LAZY_PREFILL_TC. ([ES] "1. Prefilling") */
    /* Added to one of the above: the cached pages hold keys at absolute positions (copies
       written by kv_pool_materialise) and are listed with offset 0. The attention is the same;
       the tensor-core kernel then takes position 0 as its reference (queries rotated by R(m),
       question keys by R(p)) and gives offset-0 pages no rotation, only their conversion to
       the fp16 operand type of its Q.K product. The CUDA-core kernels ignore it. */
    LAZY_PREFILL_ABSOLUTE_KEYS = 16
};

/* ---------------------------------------------------------------------------------------
 * Library information
 * --------------------------------------------------------------------------------------- */
/* Version as 10000*major + 100*minor + patch. */
int lazy_version(void);
/* Static string for a status code. */
const char *lazy_status_string(int status);
/* Message of the last failing CUDA call made by this thread (static buffer, never null). */
const char *lazy_last_error(void);

/* ---------------------------------------------------------------------------------------
 * Paged KV pool ("cache stores purely content-based keys and values", summaries' core concept)
 * --------------------------------------------------------------------------------------- */
/*
 * Create a pool over caller-owned device buffers d_k_pages / d_v_pages, each
 * num_blocks * num_kv_heads * page_size * head_dim elements of `dtype`, 16-byte aligned.
 * page_size must be 16; head_dim 64 or 128; rope_base > 0. No device memory is touched here:
 * on the first device call the pool allocates its device state (error word, angle table) on
 * the current device and zero-fills both page buffers (synchronously), so that never-written
 * slots hold finite values. *out receives the handle. Not thread-safe against destroy.
 */
int lazy_pool_create(lazy_pool **out, void *d_k_pages, void *d_v_pages, int32_t num_blocks,
                     int32_t page_size, int32_t num_kv_heads, int32_t head_dim, int32_t dtype,
                     double rope_base);
/* Free the pool's host metadata and device state (not the page buffers). */
int lazy_pool_destroy(lazy_pool *pool);
/* Bound, in nanoseconds, on every spin wait inside the kernels (default 2e9). After it
 * expires the kernel sets LAZY_DEVERR_TIMEOUT, drains its own copies and returns. */
int lazy_pool_set_wait_limit(lazy_pool *pool, uint64_t ns);

/*
 * Position encodings. The summaries state that the mechanism is not tied to RoPE and also
 * serves ALiBi ("Main contributions" item 4, generalisability). A pool is in one mode for its
 * whole life:
 *   LAZY_POS_ROPE   (default) as described above.
 *   LAZY_POS_ALIBI  K is cached as given (no rotation at all), and every score gets the bias
 *                   slope[qh] * (n - m), with n the key's and m the query's logical position:
 *                       s = sm_scale * q . k + slope[qh] * (n - m).
 *                   A page word's offset field then holds the logical position of the page's
 *                   FIRST token (segment offset + page_size * page index within the segment),
 *                   so key slot j of the page sits at n = offset + j. Decode and prefill rotate
 *                   nothing.
 */
enum { LAZY_POS_ROPE = 0, LAZY_POS_ALIBI = 1 };
/*
 * Switch a fresh pool to LAZY_POS_ALIBI with per-query-head slopes:
 *   h_slopes      host float [num_q_heads], copied (finite, 0 <= slope <= 64)
 *   num_q_heads   must be a multiple of num_kv_heads, and every later decode / prefill call on
 *                 the pool must pass the same num_q_heads (else LAZY_ERR_INVALID_ARG).
 * Only before the pool's first device use (insert, write, attention); LAZY_ERR_INVALID_ARG
 * afterwards, with nothing changed.
 */
int lazy_pool_set_alibi(lazy_pool *pool, const float *h_slopes, int32_t num_q_heads);
/*
 * Decode kernel choice for a pool (lazy_attn_decode / lazy_attn_decode_noalloc):
 *   LAZY_DECODE_AUTO  (default) the tensor-core kernel (warp-level mma.sync on each page, pages
 *                     by TMA) for bf16 pools with head_dim 128, else the CUDA-core kernel
 *   LAZY_DECODE_SIMT  always the CUDA-core kernel (fp32 arithmetic throughout)
 * Both give results within the library's tolerances; the setting exists for comparison. It
 * applies to calls made after it, and the workspace size depends on it (query
 * lazy_decode_workspace_bytes after setting it).
 */
enum { LAZY_DECODE_AUTO = 0, LAZY_DECODE_SIMT = 1 };
int lazy_pool_set_decode_kernel(lazy_pool *pool, int32_t kind);
/* The pool's mode (LAZY_POS_*) and, in ALiBi mode, its number of query heads (else 0). */
int lazy_pool_position_mode(lazy_pool *pool, int32_t *mode, int32_t *num_q_heads);
/*
 * The number of SMs the tensor-core prefill plans its last wave for (0, the default, = the
 * device's). When a call's units (request, kv head, 2 x 128 question rows) overflow the last wave,
 * the units of that wave are cut into key-range chunks and merged afterwards, if the caller's
 * workspace holds the partial results (lazy_prefill_workspace_bytes). Setting a smaller count
 * makes small calls take that path (tests), or leaves SMs to other work. Applies to calls made
 * after it; query lazy_prefill_workspace_bytes after setting it.
 */
int lazy_pool_set_schedule_sms(lazy_pool *pool, int32_t sms);

/* Block allocator (host-side free list with reference counts; thread-safe).
 * kv_pool_alloc pops n blocks (refcount 1) into block_ids; LAZY_ERR_OUT_OF_BLOCKS leaves the
 * pool unchanged. retain adds a reference (a second request sharing a cached document);
 * release drops one and returns the block to the free list at zero. Releasing a free block is
 * LAZY_ERR_INVALID_ARG and changes nothing. */
int kv_pool_alloc(lazy_pool *pool, int32_t n, int32_t *block_ids);
int kv_pool_retain(lazy_pool *pool, const int32_t *block_ids, int32_t n);
int kv_pool_release(lazy_pool *pool, const int32_t *block_ids, int32_t n);
int kv_pool_num_free(lazy_pool *pool, int32_t *n_free);
int kv_pool_refcount(lazy_pool *pool, int32_t block_id, int32_t *refcount);

/*
 * Encode one segment's tokens into the pool (the doc-KV encode step; the cache keeps
 * position-free content, summaries' core concept): for the tokens at document-local positions
 * j = local_pos0 .. local_pos0 + n_tokens - 1,
 *     K page row  = R(j) k_raw[t]   (fp32 arithmetic, rounded to the pool dtype, RNE)
 *     V page row  = v[t]
 * written to block block_ids[j / page_size], slot j % page_size, every kv head.
 *   d_k_raw, d_v : device [n_tokens][num_kv_heads][head_dim], pool dtype.
 *   block_ids    : host, in/out. On entry the first *n_blocks entries are blocks the segment
 *                  already owns (appending to a segment); blocks still missing for
 *                  positions < local_pos0 + n_tokens are allocated and appended, and
 *                  *n_blocks is updated. max_blocks is the capacity of block_ids.
 * On LAZY_ERR_OUT_OF_BLOCKS nothing is allocated or written.
 */
int kv_pool_insert_doc(lazy_pool *pool, const void *d_k_raw, const void *d_v, int32_t n_tokens,
                       int32_t local_pos0, int32_t *block_ids, int32_t *n_blocks,
                       int32_t max_blocks, lazy_stream_t stream);
/*
 * Scattered form of the same encode for batches of appended tokens (one decode step adds one
 * token to each request's private segment): token t goes to slot d_slot_mapping[t]
 * (= block * page_size + slot) with local position d_local_pos[t]. Device arrays, n_tokens
 * entries; entries < 0 are skipped. Blocks must already be allocated. A slot whose block lies
 * outside the pool is not written and sets LAZY_DEVERR_BAD_PAGE (read by
 * lazy_get_device_error).
 */
int kv_pool_write_tokens(lazy_pool *pool, const void *d_k_raw, const void *d_v, int32_t n_tokens,
                         const int32_t *d_slot_mapping, const int32_t *d_local_pos,
                         lazy_stream_t stream);

/*
 * Materialised copy: the position-aware alternative the summaries compare the method against
 * ("Problem statement": a cached document re-encoded for each position it is used at; the
 * prefill part describes that re-encoding as two rotations, one back to position 0 and one to
 * the target). For the n_tokens tokens of a cached segment held in src_block_ids (K rows
 * R(j) k at local positions j), writes to dst_block_ids:
 *     K row = R(offset + j) R(-j) (cached K row) = R(offset) (cached K row)
 *             (the two rotations compose exactly, the angles being exact modulo a full turn;
 *             applied as the one rotation R(offset), fp32 arithmetic, one rounding to the pool
 *             type)
 *     V row = cached V row
 * src_block_ids, dst_block_ids: host int32 [ceil(n_tokens / page_size)], blocks the caller
 * owns (kv_pool_alloc); no destination block may be one of the source blocks. The copy's keys
 * sit at absolute positions: attend its pages with page words of offset 0 (decode), and, for
 * the tensor-core prefill, with LAZY_PREFILL_ABSOLUTE_KEYS. RoPE pools only
 * (LAZY_ERR_UNSUPPORTED on ALiBi pools, whose keys carry no rotation); offset + n_tokens must
 * stay below 2^26. Exists to measure the method against the copy-per-offset baseline.
 */
int kv_pool_materialise(lazy_pool *pool, const int32_t *src_block_ids,
                        const int32_t *dst_block_ids, int32_t n_tokens, int32_t offset,
                        lazy_stream_t stream);
/*
 * The same copies for many (segment, offset) pairs in one launch (the baseline's set-up cost
 * without a launch per copy). Copy c re-encodes n_tokens[c] tokens held in
 * src_block_ids[cu_pages[c] .. cu_pages[c+1]) for offset offsets[c] into the blocks
 * dst_block_ids[cu_pages[c] .. cu_pages[c+1]), with the arithmetic of kv_pool_materialise.
 *   cu_pages      host int32 [n_copies + 1], cu_pages[0] = 0 and
 *                 cu_pages[c+1] - cu_pages[c] = ceil(n_tokens[c] / page_size)
 *   src_block_ids, dst_block_ids  host int32 [cu_pages[n_copies]]
 *   n_tokens, offsets             host int32 [n_copies]; offsets[c] + n_tokens[c] < 2^26
 * No destination block may be a source block of any copy, nor appear twice (copies run in
 * parallel). The page list is built in a pinned host buffer the pool keeps (grown on demand; a
 * call first waits until the previous call's upload from it has ended), uploaded in one
 * asynchronous copy to device memory taken from the stream-ordered allocator, and that memory
 * is returned after the launch. LAZY_ERR_INVALID_ARG for any violation (nothing launched);
 * LAZY_ERR_UNSUPPORTED on ALiBi pools.
 */
int kv_pool_materialise_batch(lazy_pool *pool, int32_t n_copies, const int32_t *cu_pages,
                              const int32_t *src_block_ids, const int32_t *dst_block_ids,
                              const int32_t *n_tokens, const int32_t *offsets,
                              lazy_stream_t stream);

/* ---------------------------------------------------------------------------------------
 * Page words ("(block ID, offset) bit-packed in a single register", summaries' decoding part)
 * --------------------------------------------------------------------------------------- */
/* Pack (block_id < 2^32, offset < 2^26, 1 <= n_valid <= 64) into *word; host only. */
int lazy_pack_page(uint32_t block_id, uint32_t offset, uint32_t n_valid, uint64_t *word);
int lazy_unpack_page(uint64_t word, uint32_t *block_id, uint32_t *offset, uint32_t *n_valid);
/* Pack n words from host arrays; stops at the first invalid entry and returns
 * LAZY_ERR_INVALID_ARG (words before it are written). */
int lazy_pack_pages(int32_t n, const uint32_t *block_ids, const uint32_t *offsets,
                    const uint32_t *n_valid, uint64_t *words);
/*
 * The page words of one segment: `length` tokens held in blocks block_ids[0 .. n_pages-1],
 * n_pages = ceil(length / page_size), attended at logical offset `offset`. Word i is
 * (block_ids[i], position, min(page_size, length - i * page_size)) with position = offset for
 * RoPE pools (page_positions = 0: every page of a segment carries the segment's offset) or
 * offset + i * page_size for ALiBi pools (page_positions = 1: each page carries its first
 * token's position). Host arrays; words has room for max_words; *n_words receives n_pages.
 * LAZY_ERR_INVALID_ARG if n_blocks or max_words < n_pages, a position reaches 2^26, or
 * page_size is outside 1..64 (words before the failing page are written).
 */
int lazy_pack_segment(const uint32_t *block_ids, int32_t n_blocks, uint32_t offset,
                      int32_t length, int32_t page_size, int32_t page_positions,
                      uint64_t *words, int32_t max_words, int32_t *n_words);

/* ---------------------------------------------------------------------------------------
 * Decode (summaries' decoding part: M = 1, rotation fused in the inner loop, q re-rotated only
 * when the offset changes at a document boundary; here a split-KV GQA decode streaming
 * pages, warp-shuffle reductions, log-sum-exp combine)
 * --------------------------------------------------------------------------------------- */
/*
 * One query token per request attends exactly the keys its page words list:
 *   d_q          device [batch][num_q_heads][head_dim], pool dtype, RAW (unrotated)
 *   d_q_pos      device int32 [batch]: logical position m of each query
 *   d_page_words device uint64 [d_cu_pages[batch]]; request b owns
 *                words d_cu_pages[b] .. d_cu_pages[b+1]-1 (CSR; d_cu_pages device int32
 *                [batch+1], nondecreasing, d_cu_pages[0] = 0). Word order within a request
 *                does not change the result, only how often q is re-rotated.
 *   sm_scale     score scale (1/sqrt(head_dim) for standard attention)
 *   grid_ctas    0 = one persistent wave sized to the GPU; otherwise that many CTAs. Either is
 *                raised to at least ceil(virtual heads / 4) CTAs (virtual heads = num_kv_heads x
 *                ceil(G / 8)), so that no warp's share of the pages reaches 2^31.
 *   d_out        device [batch][num_q_heads][head_dim], pool dtype, 16-byte aligned
 *   d_lse        device float [batch][num_q_heads]; -inf (and out = 0) for a request with no keys
 *                d_out and d_lse are written once, by the final merge kernel, and may also be
 *                pinned host memory (which the GPU addresses directly): the result then reaches
 *                the host without a separate copy.
 *   d_workspace  device scratch of at least lazy_decode_workspace_bytes(...) bytes, 16-byte
 *                aligned; holds partial (o, lse) per split. Not read before it is written.
 * Requires num_q_heads % num_kv_heads == 0; group sizes 1, 2, 4, 8 run natively, larger groups
 * (MQA) in chunks of 8 query heads (K/V then streamed once per chunk).
 */
int lazy_decode_workspace_bytes(lazy_pool *pool, int32_t batch, int32_t num_q_heads,
                                int32_t grid_ctas, size_t *bytes);
int lazy_attn_decode(lazy_pool *pool, const void *d_q, const int32_t *d_q_pos,
                     const uint64_t *d_page_words, const int32_t *d_cu_pages, int32_t batch,
                     int32_t num_q_heads, float sm_scale, int32_t grid_ctas, void *d_out,
                     float *d_lse, void *d_workspace, size_t workspace_bytes,
                     lazy_stream_t stream);


/*
 * Allocation-free decode. The paper has no counterpart to this entry point; it exists for
 * callers that cannot provide the workspace lazy_attn_decode needs. Examples: a plugin running
 * inside a serving process whose memory manager has already reserved the GPU's memory and
 * does not let libraries allocate more, or a latency-critical loop where a cudaMalloc /
 * cudaFree pair would stall the device.
 *
 * Same arguments and results as lazy_attn_decode, minus the workspace: the partial results go
 * to a scratch array of LAZY_NOALLOC_SCRATCH_BYTES (8 MiB) compiled into the library. Every
 * GPU that loads the library holds that array until the process exits. The call allocates
 * nothing. Rules:
 *   - The pool must already have done its one-time device set-up on the current device (any
 *     earlier kv_pool_insert_doc, kv_pool_write_tokens or lazy_attn_decode call does it);
 *     otherwise LAZY_ERR_INVALID_ARG.
 *   - Each call looks up the array's device address in the current context (a driver query,
 *     not an allocation), so the address stays right across a cudaDeviceReset. The first call
 *     on a device may load the array; make it before any stream capture.
 *   - If (batch * num_kv_heads * chunks + 4 * CTAs) * group * (head_dim + 1) * 4 bytes exceeds
 *     the array (chunks = ceil(group / 8), group = num_q_heads / num_kv_heads, CTAs = the grid,
 *     by default SMs x resident CTAs), the call returns LAZY_ERR_SCRATCH_LIMIT and launches
 *     nothing. With 32/8/128 heads on a 152-SM GPU running 3 decode CTAs per SM (456 CTAs,
 *     the tensor-core decode's occupancy) that allows up to 280 requests.
 *   - All calls share the one array, and it keeps whatever the last call left there. Each call
 *     writes every scratch entry before reading it, so nothing has to start at zero. Calls
 *     whose kernels overlap on the GPU (other streams, other threads) race on the array:
 *     serialise them.
 */
enum { LAZY_NOALLOC_SCRATCH_BYTES = 8 * 1024 * 1024 };
int lazy_attn_decode_noalloc(lazy_pool *pool, const void *d_q, const int32_t *d_q_pos,
                             const uint64_t *d_page_words, const int32_t *d_cu_pages,
                             int32_t batch, int32_t num_q_heads, float sm_scale,
                             int32_t grid_ctas, void *d_out, float *d_lse, lazy_stream_t stream);

/*
 * How lazy_attn_decode (and lazy_attn_decode_noalloc) partitions its work for this pool, head
 * count and grid_ctas (0 = the default grid): the flattened (request, unit, page) sequence, with
 * *units_per_request units per request (kv heads, or virtual heads of up to 8 query heads), is
 * cut into *ranges equal contiguous ranges that run side by side. For lazy_order_segments.
 */
int lazy_decode_partition(lazy_pool *pool, int32_t num_q_heads, int32_t grid_ctas,
                          int32_t *units_per_request, int64_t *ranges);
/*
 * Host scheduling helper: an order of each request's segments under which the decode reads a
 * document shared by several requests at nearly the same time, so that its pages come from DRAM
 * once and from L2 for the other requests (the result does not depend on the order; only the
 * DRAM traffic does). Page x of the flattened sequence is read at about step x mod R of its
 * range, R = units_per_request * (all pages) / ranges; the helper places each shared segment,
 * most used first, in the slot of every request holding it whose step is closest to a common
 * target, summed over the request's units.
 *   cu_segs      host int32 [batch + 1]: request b's segments are cu_segs[b] .. cu_segs[b+1]-1
 *   seg_key      host int64 [n]: equal keys = the same cached segment (e.g. its first block id)
 *   seg_pages    host int32 [n]: pages of each segment (its page words)
 *   pinned       host uint8 [n]: 1 = keep after the movable segments (a private tail)
 *   units_per_request, ranges: from lazy_decode_partition
 *   perm         host int32 [n] out: for each request, the segment index (within the request)
 *                placed at each position
 * Requests whose movable segments have different page counts keep their order (pinned
 * segments still go last). LAZY_ERR_INVALID_ARG on a null pointer, a decreasing cu_segs or a
 * negative page count.
 */
int lazy_order_segments(int32_t batch, const int32_t *cu_segs, const int64_t *seg_key,
                        const int32_t *seg_pages, const uint8_t *pinned,
                        int32_t units_per_request, int64_t ranges, int32_t *perm);

/* ---------------------------------------------------------------------------------------
 * Shared-segment decode (the summaries' core concept carried into decode: one cached copy of a
 * document serves every request at its own offset, so requests holding the same document can
 * read its pages once between them; only the query rotation R(m - o) is per request)
 * --------------------------------------------------------------------------------------- */
/*
 * Host planner. From the host copy of a decode batch's page tables (words, cu_pages as for
 * lazy_attn_decode, host memory), cuts every request's pages into segments, groups identical
 * segments (same block and valid-count sequence) across requests and pairs each group's members
 * in order; a leftover member, and every unshared segment, is a single unit. A segment is a
 * maximal run of pages with one offset field (page_positions = 0: RoPE pools, whose words carry
 * the segment's offset) or whose offset advances by the previous page's valid count while the
 * block id advances by one (page_positions = 1: ALiBi pools, whose words carry each page's
 * first position). Any cut gives the same attention; the cut only decides what is shared.
 * With P = cu_pages[batch] - cu_pages[0] pages, the caller provides (host):
 *   entries     uint64 [2 * P]: per page of each unit, (word of request A, word of request B);
 *               B's word is 0 in single units
 *   cu_entries  int32 [P + 1]: unit u's entries are cu_entries[u] .. cu_entries[u+1]-1
 *   unit_req    int32 [2 * P]: unit u's requests A and B (B = -1 in single units)
 *   cu_members  int32 [batch + 1], members int32 [P]: request r's units, as unit * 2 + half
 *               (half 0 = A, 1 = B)
 *   member_entries int32 [2 * P]: per member, its unit's (first entry, entry count)
 * and receives the unit and entry counts. Copy the six arrays to the device unchanged for
 * lazy_attn_decode_shared. LAZY_ERR_INVALID_ARG on a null pointer or a decreasing cu_pages.
 */
int lazy_decode_shared_plan(const uint64_t *h_words, const int32_t *h_cu_pages, int32_t batch,
                            int32_t page_positions, uint64_t *h_entries, int32_t *h_cu_entries,
                            int32_t *h_unit_req, int32_t *h_cu_members, int32_t *h_members,
                            int32_t *h_member_entries, int32_t *n_units, int32_t *n_entries);
/*
 * Device scratch for lazy_attn_decode_shared: per (unit, kv head) piece of a warp's range, 8
 * rows of fp32 O and lse. grid_ctas as for lazy_attn_decode (0 = one persistent wave).
 */
int lazy_decode_shared_workspace_bytes(lazy_pool *pool, int32_t n_units, int32_t num_q_heads,
                                       int32_t grid_ctas, size_t *bytes);
/*
 * The same attention as lazy_attn_decode over the plan's units. A pair unit streams its pages
 * once with request A's query heads in the first four rows of the tensor-core fragment and
 * request B's in the other four, each rotated by its own R(m - o). Arguments:
 *   d_q, d_q_pos, batch, num_q_heads, sm_scale, grid_ctas, d_out, d_lse: as lazy_attn_decode
 *               (d_out / d_lse on the device)
 *   d_entries, d_cu_entries, d_unit_req, n_units, d_cu_members, d_members,
 *   d_member_entries: the plan, on the device (entries 8-byte aligned)
 *   d_workspace device scratch of lazy_decode_shared_workspace_bytes(...) bytes, 16-byte aligned
 * bf16 pools with head_dim 128 and 1, 2 or 4 query heads per kv head; LAZY_ERR_UNSUPPORTED
 * otherwise. Device errors (bad page words, wait timeouts) as for lazy_attn_decode.
 */
int lazy_attn_decode_shared(lazy_pool *pool, const void *d_q, const int32_t *d_q_pos,
                            const uint64_t *d_entries, const int32_t *d_cu_entries,
                            const int32_t *d_unit_req, int32_t n_units,
                            const int32_t *d_cu_members, const int32_t *d_members,
                            const int32_t *d_member_entries, int32_t batch,
                            int32_t num_q_heads, float sm_scale, int32_t grid_ctas, void *d_out,
                            float *d_lse, void *d_workspace, size_t workspace_bytes,
                            lazy_stream_t stream);

/* ---------------------------------------------------------------------------------------
 * Prefill (summaries' prefill part: compute-bound, KV blocks loaded from the cache, one
 * relative rotation of each key tile by the offset between query tile and document instead
 * of an un-rotate plus re-rotate)
 * --------------------------------------------------------------------------------------- */
/*
 * Question tokens of each request attend (a) every key of the pages listed by its page words
 * (fully visible) and (b) the question's own keys causally (key position <= query position):
 *   d_q          device [total_q][num_q_heads][head_dim], RAW; request b owns rows
 *                d_cu_q[b] .. d_cu_q[b+1]-1 (device int32 [batch+1])
 *   d_k_new,
 *   d_v_new      device [total_q][num_kv_heads][head_dim], RAW question keys/values, or both
 *                null for no question keys. They are not written to the pool (insert them with
 *                kv_pool_insert_doc / kv_pool_write_tokens if a decode follows).
 *   d_q_pos0     device int32 [batch]: logical position of request b's first question token;
 *                token t of the request sits at d_q_pos0[b] + t.
 *   d_page_words,
 *   d_cu_pages   as for decode.
 *   total_q      host: d_cu_q[batch]; max_q_len host: max_b (d_cu_q[b+1]-d_cu_q[b]).
 *   d_out        device [total_q][num_q_heads][head_dim] pool dtype; d_lse float [total_q][Hq].
 *   d_workspace  device scratch of lazy_prefill_workspace_bytes(...) bytes (may be 0).
 *   flags        LAZY_PREFILL_AUTO / _SIMT / _TC / _SIMT_QSIDE / _TC_QSIDE, optionally
 *                + LAZY_PREFILL_ABSOLUTE_KEYS.
 */
int lazy_prefill_workspace_bytes(lazy_pool *pool, int32_t batch, int32_t total_q,
                                 int32_t max_q_len, int32_t num_q_heads, int32_t flags,
                                 size_t *bytes);
int lazy_attn_prefill(lazy_pool *pool, const void *d_q, const void *d_k_new, const void *d_v_new,
                      const int32_t *d_cu_q, const int32_t *d_q_pos0,
                      const uint64_t *d_page_words, const int32_t *d_cu_pages, int32_t batch,
                      int32_t total_q, int32_t max_q_len, int32_t num_q_heads, float sm_scale,
                      void *d_out, float *d_lse, void *d_workspace, size_t workspace_bytes,
                      int32_t flags, lazy_stream_t stream);

/*
 * Prefill followed by the question's own K/V entering the pool, in one call (the summaries'
 * prefill and decoding parts chained: after prefill the question is a cached segment that
 * decode steps read by page word like any document). Arguments as lazy_attn_prefill, plus
 *   d_append_slots      device int32 [total_q]: slot (block * page_size + slot) that question
 *                       token t (row t of d_k_new / d_v_new) goes to; < 0 skips the token
 *   d_append_local_pos  device int32 [total_q]: its local position j within the private
 *                       segment; the pool receives R(j) k_new[t] and v_new[t], exactly as
 *                       kv_pool_write_tokens writes them
 * The caller owns the private segment's blocks (kv_pool_alloc) and lists them, with the
 * segment's logical offset (normally d_q_pos0[b]), in later decode page words.
 * d_k_new and d_v_new must be given. All arguments are checked before anything is launched;
 * both steps are queued on `stream`.
 */
int lazy_attn_prefill_append(lazy_pool *pool, const void *d_q, const void *d_k_new,
                             const void *d_v_new, const int32_t *d_cu_q, const int32_t *d_q_pos0,
                             const uint64_t *d_page_words, const int32_t *d_cu_pages,
                             int32_t batch, int32_t total_q, int32_t max_q_len,
                             int32_t num_q_heads, float sm_scale, void *d_out, float *d_lse,
                             void *d_workspace, size_t workspace_bytes, int32_t flags,
                             const int32_t *d_append_slots, const int32_t *d_append_local_pos,
                             lazy_stream_t stream);

/* ---------------------------------------------------------------------------------------
 * Errors and test hooks
 * --------------------------------------------------------------------------------------- */
/* Wait for `stream`, return the device error word's bits in *err and clear it. */
int lazy_get_device_error(lazy_pool *pool, int32_t *err, lazy_stream_t stream);

/*
 * Upload of a step's inputs: copies `bytes` from pinned host memory to device memory with a
 * kernel whose threads read the host buffer directly over the host link (many 16-byte loads in
 * flight), instead of a copy-engine transfer, whose start-up dominates at the size of one
 * decode step's inputs (about a megabyte). Not an operation of the method: the serving loop's
 * host-to-device step, for measuring a decode step end to end.
 *   d_dst   device memory of the current device, 16-byte aligned.
 *   h_src   pinned host memory mapped for the device (cudaHostAlloc / cudaMallocHost /
 *           cudaHostRegister), 16-byte aligned. The caller keeps it unchanged until the copy
 *           has completed on `stream`.
 *   bytes   a multiple of 16; 0 is a no-op.
 * Stream-ordered and asynchronous. LAZY_ERR_INVALID_ARG for null or misaligned pointers, a
 * size that is not a multiple of 16, a source that is not pinned host memory, or a destination
 * that is not memory of the current device; nothing is launched then.
 */
int lazy_copy_to_device(void *d_dst, const void *h_src, size_t bytes, lazy_stream_t stream);
/*
 * Test hook: gather the pages the words address using the kernels' own device unpack and
 * address arithmetic. d_k_out, d_v_out: device [n_words][num_kv_heads][page_size][head_dim];
 * d_fields: device uint32 [n_words][3] = (block id, offset, n_valid) as unpacked on the device.
 * Words whose block id is outside the pool set LAZY_DEVERR_BAD_PAGE and gather block 0.
 */
int lazy_debug_gather(lazy_pool *pool, const uint64_t *d_page_words, int32_t n_words,
                      void *d_k_out, void *d_v_out, uint32_t *d_fields, lazy_stream_t stream);

/*
 * Test hook for the bounded-wait path: one warp waits on a shared-memory barrier that nothing
 * arrives at, with the same bounded wait the kernels use and a limit of limit_ns; when it gives
 * up it sets LAZY_DEVERR_TIMEOUT and returns. The context stays usable.
 */
int lazy_debug_wait_timeout(lazy_pool *pool, uint64_t limit_ns, lazy_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* LAZY_ATTN_H */
