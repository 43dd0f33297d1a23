/*
 * pfkv.h -- C ABI of libpfkv: a paged FP8 (e4m3) KV cache for decode
 * attention on GB300 (sm_103a).
 *
 * What the operations are, from "Smaller, faster, safer: running Kimi and GLM
 * at scale" (Cloudflare):
 *  - section "Quantizing the KV cache": the decode pool keeps K and V in
 *    8-bit floating point (FP8, e4m3) instead of BF16, halving the cache, and
 *    the FP8 attention kernel converts the values as it reads them.  Both
 *    cache precisions exist (BF16 is the default and the prefill pool's).
 *  - the cache-protection passage: many concurrent requests read and write
 *    one shared physical cache; each page carries a tag that changes whenever
 *    the page is reallocated; before a read the mapping's tag is compared
 *    with the page's, and on a mismatch the request is aborted instead of
 *    returning wrong data; the check is off by default.
 *
 * Conventions for every entry point:
 *  - Ownership: the caller owns every buffer.  The library never allocates,
 *    never frees and never synchronises; it only enqueues work on `stream`
 *    (a cudaStream_t passed as void*; NULL = the legacy default stream).
 *  - Pointers are DEVICE pointers unless marked "host".  The cache descriptor
 *    itself is host memory, read during the call only.
 *  - Return value: 0 (PFKV_OK) or a negative PFKV_ERR_* code for errors that
 *    the host can see (bad argument, unsupported shape, small workspace,
 *    launch failure).  Nothing is enqueued when an error is returned.
 *  - Per-request data faults (stale tag, page id outside the pool, bad
 *    length) are reported in status[batch] (uint32 bit set, PFKV_ST_*), which
 *    every call overwrites.  They never trap on the device.
 *  - The attention output rows of a request with a data fault (STALE_TAG,
 *    PAGE_OOB, BAD_LEN) are all zero; under TIMEOUT the output of the call
 *    is not valid.
 *  - Results are deterministic for identical inputs.
 */
#ifndef PFKV_H
#define PFKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Cache element type. */
enum { PFKV_DTYPE_BF16 = 0, PFKV_DTYPE_FP8_E4M3 = 1 };

/* FP8 scale granularity.  PER_HEAD: one fp32 scale per KV head for the whole
 * pool (calibrated, see pfkv_calibrate_scales).  PER_TOKEN: one fp32 scale
 * per cached (token, KV head) row, computed by the append from that row. */
enum { PFKV_SCALE_PER_HEAD = 0, PFKV_SCALE_PER_TOKEN = 1 };

/* Call flags.  TAG_CHECK enables the page-tag comparison; it is off unless
 * set, as in the post.  TEST_WITHHOLD is a test hook for the decode
 * kernels, never set in normal use: the first CTA's page loader withholds
 * its first work item from the other warps, whose bounded wait then runs
 * out (about 2 s); every request of the call reports PFKV_ST_TIMEOUT and the
 * context stays usable.  It exercises the abort path without a fault. */
enum { PFKV_FLAG_TAG_CHECK = 1u, PFKV_FLAG_TEST_WITHHOLD = 0x80000000u };

/* Per-request status bits. */
enum {
  PFKV_ST_STALE_TAG = 1u, /* a page's tag differs from the mapping's tag  */
  PFKV_ST_PAGE_OOB = 2u,  /* a page id is outside [0, num_pages)          */
  PFKV_ST_BAD_LEN = 4u,   /* length < 1 or beyond max_pages * page_size,
                             or an append position outside the table      */
  PFKV_ST_TIMEOUT = 8u,   /* a pipeline wait inside the kernel gave up;
                             the output of the call is not valid          */
  PFKV_ST_NO_PAGES = 16u, /* page allocator: fewer free pages than asked  */
  PFKV_ST_NOT_HELD = 32u, /* page allocator: the page is not handed out   */
  PFKV_ST_DUPLICATE = 64u /* page allocator: id listed twice in one call  */
};

/* Return codes. */
enum {
  PFKV_OK = 0,
  PFKV_ERR_NULL = -1,        /* a required pointer is NULL                  */
  PFKV_ERR_SHAPE = -2,       /* inconsistent or out-of-range sizes          */
  PFKV_ERR_UNSUPPORTED = -3, /* valid but not implemented (head dim, group) */
  PFKV_ERR_DTYPE = -4,       /* cache dtype does not match the entry point  */
  PFKV_ERR_WORKSPACE = -5,   /* workspace NULL or smaller than required     */
  PFKV_ERR_ALIGN = -6,       /* a buffer is not 16-byte aligned             */
  PFKV_ERR_CUDA = -7         /* a CUDA runtime/driver call failed           */
};

/*
 * Paged cache descriptor (host struct; the arrays it points to are device
 * memory).  Layout (this library's choice; the post gives none):
 *   k_pool : [num_pages][num_kv_heads][page_size][head_dim]   elements
 *   v_pool : [num_pages][num_kv_heads][page_size][v_head_dim] elements
 *   element = 1 byte e4m3 code (FP8) or 2 byte bf16 (BF16).
 *   k_scale/v_scale (FP8 only): PER_HEAD [num_kv_heads];
 *                               PER_TOKEN [num_pages][num_kv_heads][page_size].
 *   page_tags : [num_pages] uint32, the page's current generation tag.
 * Logical token t of a request lives in page block_table[b][t / page_size],
 * slot t % page_size.
 * Latent (shared) stream: kv_shared = 1, num_kv_heads = 1, v_pool = NULL,
 * v_scale = NULL; V is the first v_head_dim values of each K row.
 * Every pool base must be 16-byte aligned.
 */
typedef struct pfkv_cache {
  int32_t num_pages;
  int32_t page_size;
  int32_t num_kv_heads;
  int32_t head_dim;
  int32_t v_head_dim;
  int32_t kv_shared;
  int32_t dtype;      /* PFKV_DTYPE_*      */
  int32_t scale_mode; /* PFKV_SCALE_*      */
  void *k_pool;
  void *v_pool;
  float *k_scale;
  float *v_scale;
  const uint32_t *page_tags;
} pfkv_cache;

/*
 * kv_append_quantize -- write new K/V rows into the paged cache ("Quantizing
 * the KV cache": the cache is stored in FP8 e4m3).
 *
 * num_rows new tokens.  Row i belongs to request row_req[i] (row_req may be
 * NULL: row i belongs to request i, the one-token-per-request decode case)
 * and goes to logical position positions[i]:
 *   page = block_table[b][positions[i] / page_size], slot = positions[i] % page_size.
 *   k_new : bf16 [num_rows][num_kv_heads][head_dim]
 *   v_new : bf16 [num_rows][num_kv_heads][v_head_dim] (ignored when kv_shared)
 *   block_table, block_tags : [batch][max_pages] int32 / uint32
 * FP8: code = e4m3(fp32(x) / s), IEEE fp32 division, round to nearest even,
 * saturating to +-448.  PER_HEAD uses k_scale[h] / v_scale[h] as given.
 * PER_TOKEN computes s = amax(|row|)/448 (1 when the row is all zero) for each
 * (token, head) row, stores it in the scale array and quantizes with it.
 * BF16: the bits are copied.
 * A row is refused -- nothing of it is written -- when its position is
 * outside [0, max_pages*page_size) (BAD_LEN), its page id is outside the pool
 * (PAGE_OOB), or TAG_CHECK is set and page_tags[page] differs from
 * block_tags[b][positions[i] / page_size] (STALE_TAG).  status[batch] is
 * cleared and then gets the bits of every refused row of each request.
 * Rows of one call must not target the same slot.
 */
int pfkv_kv_append_quantize(const pfkv_cache *cache, const void *k_new, const void *v_new, int32_t num_rows,
                            const int32_t *row_req, const int32_t *positions, const int32_t *block_table,
                            const uint32_t *block_tags, int32_t batch, int32_t max_pages, uint32_t flags,
                            uint32_t *status, void *stream);

/*
 * Bytes of device workspace a decode call needs for these sizes (split-KV
 * partial results and the split plan).  Host-only, no CUDA call.
 */
size_t pfkv_decode_workspace_bytes(const pfkv_cache *cache, int32_t batch, int32_t num_q_heads,
                                   int32_t max_splits);

/*
 * paged_decode_attention -- single-token decode attention over the paged
 * cache, converting FP8 codes as they are read ("Quantizing the KV cache")
 * and, when TAG_CHECK is set, comparing every page's tag with the mapping's
 * before its data may be returned (cache-protection passage).
 *
 *   q          : bf16 [batch][num_q_heads][head_dim]
 *   seq_lens   : int32 [batch], tokens of context per request (>= 1)
 *   block_table: int32 [batch][max_pages]; block_tags: uint32 [batch][max_pages]
 *   out        : fp32 [batch][num_q_heads][v_head_dim]
 *   status     : uint32 [batch]
 * For query head h (KV head g = h / (num_q_heads / num_kv_heads)):
 *   z_t = softmax_scale * q[b][h] . k^[g][t],  p = softmax(z over t < L_b),
 *   out[b][h] = sum_t p_t v^[g][t],  where k^, v^ are the dequantized rows
 *   (code value * scale for FP8).
 * Only logical pages i < ceil(L_b / page_size) are inspected.  A request
 * with a data-fault bit gets zero output.  batch * max_pages may not exceed
 * 2^40 (PFKV_ERR_SHAPE).  max_splits (1..256) bounds how many
 * pieces one request's context is split into (flash-decoding); the pieces
 * are merged with the log-sum-exp rule.  workspace must hold
 * pfkv_decode_workspace_bytes(cache, batch, num_q_heads, max_splits) bytes;
 * its contents need no initialisation and are scratch between calls.
 * Supported: head_dim 64 or 128 with any group size num_q_heads /
 * num_kv_heads (page_size a multiple of 16, at most 256; a group of more
 * than 8 query heads is run as ceil(G / 8) groups of at most 8 that each
 * read the KV head, and num_kv_heads * ceil(G / 8) may not exceed 4096, else
 * PFKV_ERR_UNSUPPORTED); the latent stream head_dim 576 / v_head_dim 512
 * with 64 query heads (FP8, PER_TOKEN, page_size 64).  num_q_heads must be a
 * multiple of num_kv_heads (PFKV_ERR_SHAPE).
 * pfkv_paged_decode_attention_fp8 requires an FP8 cache, _bf16 a BF16 cache.
 */
int pfkv_paged_decode_attention_fp8(const pfkv_cache *cache, const void *q, int32_t num_q_heads,
                                    const int32_t *seq_lens, const int32_t *block_table,
                                    const uint32_t *block_tags, int32_t batch, int32_t max_pages,
                                    float softmax_scale, uint32_t flags, int32_t max_splits, void *workspace,
                                    size_t workspace_bytes, float *out, uint32_t *status, void *stream);

int pfkv_paged_decode_attention_bf16(const pfkv_cache *cache, const void *q, int32_t num_q_heads,
                                     const int32_t *seq_lens, const int32_t *block_table,
                                     const uint32_t *block_tags, int32_t batch, int32_t max_pages,
                                     float softmax_scale, uint32_t flags, int32_t max_splits, void *workspace,
                                     size_t workspace_bytes, float *out, uint32_t *status, void *stream);

/*
 * paged_decode_attention_fp8_noalloc -- the FP8 decode above for callers
 * that cannot allocate device memory.  (The post has no counterpart; this is
 * an interface convenience of this library.)
 *
 * Some callers have no way to hand the library a workspace: code embedded in
 * a host framework that owns every device allocation and passes in only its
 * input and output buffers, plugins that must not bypass their host's
 * allocator, or serving paths where a cudaMalloc would synchronise the
 * device.  This entry point takes no workspace; it uses a scratch buffer of
 * PFKV_NOALLOC_SCRATCH_BYTES that lives in the library as a file-scope device
 * array (every GPU that loads the library holds it until the process exits)
 * and otherwise behaves exactly like pfkv_paged_decode_attention_fp8 with the
 * same arguments.  It calls no cudaMalloc, cudaFree or allocating routine.
 *  - Returns PFKV_ERR_WORKSPACE, before any device work, when
 *    pfkv_decode_workspace_bytes(cache, batch, num_q_heads, max_splits) is
 *    larger than PFKV_NOALLOC_SCRATCH_BYTES (lower max_splits or split the
 *    batch).
 *  - The first call on each device looks up the buffer's device address
 *    (cudaGetSymbolAddress, with that device current); make that first call
 *    before any stream capture.
 *  - Every call shares the one buffer, which keeps the last call's
 *    contents; every word a call reads back is written earlier in the same
 *    call.  Calls that overlap on the GPU (different streams, or different
 *    host threads, at the same time) race on the buffer and give wrong
 *    results.
 */
#define PFKV_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)

int pfkv_paged_decode_attention_fp8_noalloc(const pfkv_cache *cache, const void *q, int32_t num_q_heads,
                                            const int32_t *seq_lens, const int32_t *block_table,
                                            const uint32_t *block_tags, int32_t batch, int32_t max_pages,
                                            float softmax_scale, uint32_t flags, int32_t max_splits, float *out,
                                            uint32_t *status, void *stream);

/*
 * paged_decode_step -- one decode step of the paged cache: every request's
 * new token is written into the cache (as pfkv_kv_append_quantize would,
 * quantized on the way in for an FP8 cache) and then attended over, together
 * with the rest of its context, as pfkv_paged_decode_attention_* does.  The
 * post's two halves of the decode pool ("Quantizing the KV cache": rows are
 * stored as FP8 and converted as they are read) in one call: the attention
 * kernel's page loader writes each (request, KV head) row itself before it
 * copies the destination page (grouped-query layouts and the latent
 * stream alike).
 *   k_new, v_new : bf16 [batch][num_kv_heads][head_dim]; row b goes to
 *                  logical position seq_lens[b] - 1 (seq_lens counts the new
 *                  token); v_new is ignored (may be NULL) for a kv_shared
 *                  cache.  16-byte aligned.
 *   The other arguments, the workspace and the outputs are those of
 *   pfkv_paged_decode_attention_fp8 / _bf16; the cache's dtype selects the
 *   variant, with the same supported shapes.
 * status[b] is the attention's status.  It covers every refusal of the
 * write: the write targets logical page (seq_lens[b] - 1) / page_size,
 * which the attention inspects under the same rules, and a refused row
 * writes nothing.  Distinct requests must not share a destination slot, and
 * a request's destination page must not be read by another request of the
 * same call (a page being appended to belongs to one request).
 */
int pfkv_paged_decode_step(const pfkv_cache *cache, const void *k_new, const void *v_new, const void *q,
                           int32_t num_q_heads, const int32_t *seq_lens, const int32_t *block_table,
                           const uint32_t *block_tags, int32_t batch, int32_t max_pages, float softmax_scale,
                           uint32_t flags, int32_t max_splits, void *workspace, size_t workspace_bytes, float *out,
                           uint32_t *status, void *stream);

/*
 * handoff_bf16_to_fp8 -- quantize whole pages of a BF16 cache into an FP8
 * cache ("Quantizing the KV cache": prefill keeps BF16 because it is
 * compute-bound, the decode pool stores FP8 e4m3; a request moving between
 * the two has its pages converted).
 *   src : BF16 cache; dst : FP8 cache with the same num_kv_heads, page_size,
 *         head_dim, v_head_dim and kv_shared.
 *   src_pages, dst_pages : int32 [n_pages]; page src_pages[i] of src becomes
 *         page dst_pages[i] of dst (every head, every slot, K and V).
 *   page_status : uint32 [n_pages]; PFKV_ST_PAGE_OOB when either id is outside
 *         its pool (that pair is skipped), else 0.
 * Codes as in kv_append_quantize: e4m3(fp32(x)/s), s = dst's per-head scale,
 * or (PER_TOKEN) amax/448 of each (token, head) row, stored in dst's scales.
 * Destination pages must be distinct.
 */
int pfkv_handoff_bf16_to_fp8(const pfkv_cache *src, const pfkv_cache *dst, const int32_t *src_pages,
                             const int32_t *dst_pages, int32_t n_pages, uint32_t *page_status, void *stream);

/*
 * Page allocator -- the producer side of the page tags (cache-protection
 * passage: each page's tag changes whenever the page is reallocated, so a
 * request that still holds the old mapping fails the tag check).  A free
 * list that lives in device memory, so a step can take and return pages
 * without a host round trip.  Every hand-out of a page to an owner (alloc,
 * realloc) advances page_tags[p] by one, modulo 2^32; freeing leaves it.
 *
 * State (caller-owned device memory, pfkv_page_allocator_bytes(num_pages)
 * bytes, 256-byte aligned):
 *   bytes [0, 4)     int32 num_pages
 *   bytes [4, 8)     int32 free_count
 *   bytes [256, ...) int32 stack[num_pages]: stack[0 .. free_count) are the
 *                    free ids, the last one is handed out first
 *   followed by per-page bookkeeping (a held flag and a scratch word).
 * A fresh state hands out pages in increasing id order; freed pages are
 * reused last-in first-out.  Calls on one state must be ordered (one stream,
 * or events): each call is one kernel that owns the state while it runs.
 * Lists are processed as if in order (first occurrence wins); results are
 * deterministic.
 */
size_t pfkv_page_allocator_bytes(int32_t num_pages);

/* Make every page free except held_pages[0 .. n_held) (ids outside the pool
 * and repeats are ignored; held_pages may be NULL when n_held == 0).
 * Returns PFKV_ERR_WORKSPACE when state_bytes is too small. */
int pfkv_page_allocator_init(void *state, size_t state_bytes, int32_t num_pages, const int32_t *held_pages,
                             int32_t n_held, void *stream);

/* Take n pages: pages_out[i], their new tags tags_out[i] (to be stored in
 * the owner's block_tags).  All or nothing: with fewer than n free pages
 * nothing is taken, pages_out = -1, tags_out = 0 and *status = NO_PAGES;
 * else *status = 0.  page_tags: the cache's tag array [num_pages]. */
int pfkv_page_alloc(void *state, uint32_t *page_tags, int32_t n, int32_t *pages_out, uint32_t *tags_out,
                    uint32_t *status, void *stream);

/* Give pages back.  page_status[i]: 0, PAGE_OOB (id outside the pool) or
 * NOT_HELD (not handed out, or already given back earlier in the list);
 * flagged entries are skipped. */
int pfkv_page_free(void *state, const int32_t *pages, int32_t n, uint32_t *page_status, void *stream);

/* Move held pages to new owners without a trip through the free list: each
 * listed page's tag advances once and is returned in tags_out[i].
 * page_status[i]: 0, PAGE_OOB, NOT_HELD, or DUPLICATE for a repeat of an
 * earlier entry; flagged entries get tags_out 0 and change nothing. */
int pfkv_page_realloc(void *state, uint32_t *page_tags, const int32_t *pages, int32_t n, uint32_t *tags_out,
                      uint32_t *page_status, void *stream);

/*
 * calibrate_scales -- per-head FP8 scales s[h] = fp32(amax/448) over
 * rows[n_rows][num_heads][head_dim] (bf16); s[h] = 1 when the head's rows
 * are all zero.  This is the "scale = amax / 448" convention of an e4m3 cache
 * whose largest finite value is 448.  scale: fp32 [num_heads], overwritten.
 */
int pfkv_calibrate_scales(const void *rows, int64_t n_rows, int32_t num_heads, int32_t head_dim, float *scale,
                          void *stream);

/*
 * e4m3_encode -- codes[i] = e4m3(x[i]) for fp32 x: round to nearest even,
 * saturate finite overflow to +-448, sign kept on zero, NaN -> NaN code.
 * The same conversion the append uses (exposed for the codec tests).
 */
int pfkv_e4m3_encode(const float *x, uint8_t *codes, int64_t n, void *stream);

/* Human-readable text for a PFKV_ERR_* code. */
const char *pfkv_strerror(int code);

/* Text of the CUDA error behind the calling thread's most recent
 * PFKV_ERR_CUDA return (which call failed and the runtime's message); empty
 * if there was none.  The string is owned by the library. */
const char *pfkv_last_error_detail(void);

/* ABI version of this header (bumped when a signature changes). */
int pfkv_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PFKV_H */
