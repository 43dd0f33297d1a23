// api.cu -- the extern "C" entry points of libpfkv: argument checks on the
// host, workspace layout, and dispatch to the kernels on the caller's stream.
#include <math.h>
#include <stdio.h>

#include <mutex>

#include "pfkv_internal.h"

namespace pfkv {

static thread_local char g_last_error[256] = "";

int cuda_fail(cudaError_t e, const char *where) {
  snprintf(g_last_error, sizeof(g_last_error), "%s: %s (%d)", where, cudaGetErrorString(e), (int)e);
  return PFKV_ERR_CUDA;
}

EncodeTiledFn encode_tiled_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

int num_sms() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 1;
}

static size_t up256(size_t x) { return (x + 255) & ~size_t(255); }

// Every size here is bounded by the callers (batch < 2^31, max_splits <= 256,
// q_heads <= kMaxQHeads, v_dim <= kMaxHeadDim), so the products below stay
// far inside size_t.
WsLayout ws_layout(int batch, int q_heads, int v_dim, int max_splits, bool latent) {
  WsLayout w;
  const size_t slots = (size_t)batch * max_splits * q_heads;
  w.split_first = 0;
  w.split_count = w.split_first + up256(sizeof(int) * ((size_t)batch + 1));
  w.part_ml = w.split_count + up256(sizeof(int) * (size_t)batch);
  w.part_o = w.part_ml + up256(sizeof(float2) * slots);
  w.part_st = w.part_o + up256(sizeof(float) * slots * v_dim);
  // a status word per piece and head group (at most q_heads head groups)
  w.cta_abort = w.part_st + up256(sizeof(uint32_t) * (size_t)batch * max_splits * q_heads);
  w.qterms = w.cta_abort + up256(sizeof(int) * (size_t)kMaxCtas);
  w.qfac = w.qterms + (latent ? up256(kLatentQTermBytes * (size_t)batch) : 0);
  w.total = w.qfac + (latent ? up256(sizeof(float) * (size_t)batch * q_heads) : 0);
  return w;
}

static bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Largest query-head count and head width a decode call accepts (far above
// any model's; they bound the workspace arithmetic).
constexpr int kMaxQHeads = 65536;
constexpr int kMaxHeadDim = 4096;

static bool is_latent(const pfkv_cache *c) {
  return c->kv_shared && c->num_kv_heads == 1 && c->head_dim == 576 && c->v_head_dim == 512;
}

// Checks shared by every call that takes a cache descriptor.
static int check_cache(const pfkv_cache *c) {
  if (!c) return PFKV_ERR_NULL;
  if (c->num_pages < 1 || c->page_size < 1 || c->num_kv_heads < 1 || c->head_dim < 1 || c->v_head_dim < 1)
    return PFKV_ERR_SHAPE;
  if (c->head_dim > kMaxHeadDim || c->v_head_dim > kMaxHeadDim || c->num_kv_heads > kMaxQHeads) return PFKV_ERR_SHAPE;
  if (c->dtype != PFKV_DTYPE_BF16 && c->dtype != PFKV_DTYPE_FP8_E4M3) return PFKV_ERR_DTYPE;
  if (c->scale_mode != PFKV_SCALE_PER_HEAD && c->scale_mode != PFKV_SCALE_PER_TOKEN) return PFKV_ERR_SHAPE;
  if (!c->k_pool) return PFKV_ERR_NULL;
  if (c->kv_shared) {
    if (c->num_kv_heads != 1 || c->v_head_dim > c->head_dim) return PFKV_ERR_SHAPE;
  } else {
    if (!c->v_pool) return PFKV_ERR_NULL;
    if (c->v_head_dim != c->head_dim) return PFKV_ERR_UNSUPPORTED;
  }
  if (c->dtype == PFKV_DTYPE_FP8_E4M3 && (!c->k_scale || (!c->kv_shared && !c->v_scale))) return PFKV_ERR_NULL;
  if (c->head_dim % 8 || c->v_head_dim % 8) return PFKV_ERR_UNSUPPORTED;
  if (!aligned16(c->k_pool) || (c->v_pool && !aligned16(c->v_pool))) return PFKV_ERR_ALIGN;
  if (c->scale_mode == PFKV_SCALE_PER_TOKEN &&
      (!aligned16(c->k_scale) || (c->v_scale && !aligned16(c->v_scale))))
    return PFKV_ERR_ALIGN;
  return PFKV_OK;
}

// The checks a decode call makes before it looks at the workspace (shared
// with the no-allocation entry point, so that both return the same code for
// the same bad arguments).
int decode_precheck(int want_dtype, const pfkv_cache *c, int32_t Hq, int32_t batch, int32_t max_pages,
                    int32_t max_splits) {
  int rc = check_cache(c);
  if (rc) return rc;
  if (c->dtype != want_dtype) return PFKV_ERR_DTYPE;
  if (batch < 0 || max_pages < 1 || Hq < 1 || Hq > kMaxQHeads || max_splits < 1 || max_splits > 256)
    return PFKV_ERR_SHAPE;
  return PFKV_OK;
}

static int decode_common(int want_dtype, const pfkv_cache *c, const void *q, int32_t Hq, const int32_t *seq_lens,
                         const int32_t *block_table, const uint32_t *block_tags, int32_t batch, int32_t max_pages,
                         float softmax_scale, uint32_t flags, int32_t max_splits, void *ws, size_t ws_bytes,
                         float *out, uint32_t *status, void *stream, const void *k_new = nullptr,
                         const void *v_new = nullptr) {
  const int rc = decode_precheck(want_dtype, c, Hq, batch, max_pages, max_splits);
  if (rc) return rc;
  // the kernels' page arithmetic assumes at most 2^40 pages in one call
  if ((uint64_t)batch * (uint64_t)max_pages > (1ull << 40)) return PFKV_ERR_SHAPE;
  if (!isfinite(softmax_scale)) return PFKV_ERR_SHAPE;
  if (batch == 0) return PFKV_OK;
  if (!q || !seq_lens || !block_table || !out || !status || !ws) return PFKV_ERR_NULL;
  if ((flags & PFKV_FLAG_TAG_CHECK) && (!c->page_tags || !block_tags)) return PFKV_ERR_NULL;
  if (Hq % c->num_kv_heads) return PFKV_ERR_SHAPE;
  if (!aligned16(q) || !aligned16(out)) return PFKV_ERR_ALIGN;
  if (c->page_size % 16 || c->page_size > 256) return PFKV_ERR_UNSUPPORTED;
  const WsLayout L = ws_layout(batch, Hq, c->v_head_dim, max_splits, is_latent(c));
  if (ws_bytes < L.total) return PFKV_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return PFKV_ERR_ALIGN;

  DecodeArgs a;
  a.P = c->num_pages; a.S = c->page_size; a.Hkv = c->num_kv_heads; a.D = c->head_dim; a.Dv = c->v_head_dim;
  a.scale_mode = c->scale_mode; a.dtype = c->dtype; a.kv_shared = c->kv_shared;
  a.k_pool = c->k_pool; a.v_pool = c->v_pool; a.k_scale = c->k_scale; a.v_scale = c->v_scale;
  a.page_tags = c->page_tags;
  a.q = q; a.Hq = Hq; a.G = Hq / c->num_kv_heads;
  a.kv_sub = 1; a.Gs = a.G;
  a.seq_lens = seq_lens; a.block_table = block_table; a.block_tags = block_tags;
  a.B = batch; a.MP = max_pages;
  a.sm_scale_log2 = softmax_scale * 1.4426950408889634f;
  a.flags = flags; a.max_splits = max_splits;
  uint8_t *w = static_cast<uint8_t *>(ws);
  a.split_first = reinterpret_cast<int *>(w + L.split_first);
  a.split_count = reinterpret_cast<int *>(w + L.split_count);
  a.part_ml = reinterpret_cast<float2 *>(w + L.part_ml);
  a.part_o = reinterpret_cast<float *>(w + L.part_o);
  a.out = out; a.status = status;
  a.append = k_new != nullptr;
  a.k_new = static_cast<const uint16_t *>(k_new);
  a.v_new = static_cast<const uint16_t *>(v_new);
  a.cache = *c;
  a.ranges = 0;
  a.target_items = 0;
  a.min_chunk_pages = 1;
  a.n_ctas = 0;
  a.st_groups = 1;
  a.piece_cost = 0;
  a.part_st = reinterpret_cast<uint32_t *>(w + L.part_st);
  a.cta_abort = reinterpret_cast<int *>(w + L.cta_abort);
  a.qterms = w + L.qterms;
  a.qfac = reinterpret_cast<float *>(w + L.qfac);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (c->kv_shared) {
    if (!is_latent(c) || Hq != 64 || c->dtype != PFKV_DTYPE_FP8_E4M3 || c->scale_mode != PFKV_SCALE_PER_TOKEN ||
        c->page_size != 64)
      return PFKV_ERR_UNSUPPORTED;
    return launch_latent_decode(a, s);
  }
  if (c->head_dim != 64 && c->head_dim != 128) return PFKV_ERR_UNSUPPORTED;
  if (c->dtype == PFKV_DTYPE_BF16 && c->scale_mode != PFKV_SCALE_PER_HEAD) return PFKV_ERR_SHAPE;
  return launch_gqa_decode(a, s);
}

}  // namespace pfkv

using namespace pfkv;

extern "C" {

int pfkv_abi_version(void) { return 1; }

const char *pfkv_last_error_detail(void) { return g_last_error; }

const char *pfkv_strerror(int code) {
  switch (code) {
    case PFKV_OK: return "ok";
    case PFKV_ERR_NULL: return "a required pointer is NULL";
    case PFKV_ERR_SHAPE: return "inconsistent or out-of-range sizes";
    case PFKV_ERR_UNSUPPORTED: return "shape or mode not implemented";
    case PFKV_ERR_DTYPE: return "cache dtype does not match the entry point";
    case PFKV_ERR_WORKSPACE: return "workspace missing or too small";
    case PFKV_ERR_ALIGN: return "buffer not aligned (16 bytes; workspace 256 bytes)";
    case PFKV_ERR_CUDA: return "CUDA runtime or driver call failed";
    default: return "unknown error";
  }
}

int pfkv_kv_append_quantize(const pfkv_cache *cache, const void *k_new, const void *v_new, int32_t num_rows,
                            const int32_t *row_req, const int32_t *positions, const int32_t *block_table,
                            const uint32_t *block_tags, int32_t batch, int32_t max_pages, uint32_t flags,
                            uint32_t *status, void *stream) {
  int rc = check_cache(cache);
  if (rc) return rc;
  if (num_rows < 0 || batch < 0 || max_pages < 1) return PFKV_ERR_SHAPE;
  if (!row_req && num_rows > batch) return PFKV_ERR_SHAPE;
  if (batch == 0) return PFKV_OK;
  if (!status) return PFKV_ERR_NULL;
  if (num_rows > 0) {
    if (!k_new || !positions || !block_table || (!cache->kv_shared && !v_new)) return PFKV_ERR_NULL;
    if ((flags & PFKV_FLAG_TAG_CHECK) && (!cache->page_tags || !block_tags)) return PFKV_ERR_NULL;
    if (!aligned16(k_new) || (v_new && !cache->kv_shared && !aligned16(v_new))) return PFKV_ERR_ALIGN;
  }
  if (cache->dtype == PFKV_DTYPE_BF16 && cache->scale_mode != PFKV_SCALE_PER_HEAD) return PFKV_ERR_SHAPE;
  return launch_append(*cache, k_new, v_new, num_rows, row_req, positions, block_table, block_tags, batch,
                       max_pages, flags, status, static_cast<cudaStream_t>(stream));
}

size_t pfkv_decode_workspace_bytes(const pfkv_cache *cache, int32_t batch, int32_t num_q_heads, int32_t max_splits) {
  if (!cache || batch < 0 || num_q_heads < 1 || max_splits < 1) return 0;
  // sizes a decode call would refuse: no workspace fits them
  if (num_q_heads > kMaxQHeads || max_splits > 256 || cache->v_head_dim < 1 || cache->v_head_dim > kMaxHeadDim)
    return SIZE_MAX;
  return ws_layout(batch, num_q_heads, cache->v_head_dim, max_splits, is_latent(cache)).total;
}



int pfkv_paged_decode_attention_fp8(const pfkv_cache *cache, const void *q, int32_t num_q_heads,
                                    const int32_t *seq_lens, const int32_t *block_table,
                                    const uint32_t *block_tags, int32_t batch, int32_t max_pages,
                                    float softmax_scale, uint32_t flags, int32_t max_splits, void *workspace,
                                    size_t workspace_bytes, float *out, uint32_t *status, void *stream) {
  return decode_common(PFKV_DTYPE_FP8_E4M3, cache, q, num_q_heads, seq_lens, block_table, block_tags, batch,
                       max_pages, softmax_scale, flags, max_splits, workspace, workspace_bytes, out, status, stream);
}

int pfkv_paged_decode_attention_bf16(const pfkv_cache *cache, const void *q, int32_t num_q_heads,
                                     const int32_t *seq_lens, const int32_t *block_table,
                                     const uint32_t *block_tags, int32_t batch, int32_t max_pages,
                                     float softmax_scale, uint32_t flags, int32_t max_splits, void *workspace,
                                     size_t workspace_bytes, float *out, uint32_t *status, void *stream) {
  return decode_common(PFKV_DTYPE_BF16, cache, q, num_q_heads, seq_lens, block_table, block_tags, batch, max_pages,
                       softmax_scale, flags, max_splits, workspace, workspace_bytes, out, status, stream);
}

int pfkv_paged_decode_step(const pfkv_cache *cache, const void *k_new, const void *v_new, const void *q,
                           int32_t num_q_heads, const int32_t *seq_lens, const int32_t *block_table,
                           const uint32_t *block_tags, int32_t batch, int32_t max_pages, float softmax_scale,
                           uint32_t flags, int32_t max_splits, void *workspace, size_t workspace_bytes, float *out,
                           uint32_t *status, void *stream) {
  if (!cache) return PFKV_ERR_NULL;
  if (batch > 0) {
    if (!k_new || (!cache->kv_shared && !v_new)) return PFKV_ERR_NULL;
    if (!aligned16(k_new) || (!cache->kv_shared && !aligned16(v_new))) return PFKV_ERR_ALIGN;
  }
  return decode_common(cache->dtype, cache, q, num_q_heads, seq_lens, block_table, block_tags, batch, max_pages,
                       softmax_scale, flags, max_splits, workspace, workspace_bytes, out, status, stream,
                       batch > 0 ? k_new : nullptr, cache->kv_shared ? nullptr : v_new);
}

int pfkv_handoff_bf16_to_fp8(const pfkv_cache *src, const pfkv_cache *dst, const int32_t *src_pages,
                             const int32_t *dst_pages, int32_t n_pages, uint32_t *page_status, void *stream) {
  int rc = check_cache(src);
  if (rc) return rc;
  rc = check_cache(dst);
  if (rc) return rc;
  if (src->dtype != PFKV_DTYPE_BF16 || dst->dtype != PFKV_DTYPE_FP8_E4M3) return PFKV_ERR_DTYPE;
  if (src->num_kv_heads != dst->num_kv_heads || src->page_size != dst->page_size ||
      src->head_dim != dst->head_dim || src->v_head_dim != dst->v_head_dim || src->kv_shared != dst->kv_shared)
    return PFKV_ERR_SHAPE;
  if (n_pages < 0) return PFKV_ERR_SHAPE;
  if (n_pages == 0) return PFKV_OK;
  if (!src_pages || !dst_pages || !page_status) return PFKV_ERR_NULL;
  return launch_handoff(*src, *dst, src_pages, dst_pages, n_pages, page_status, static_cast<cudaStream_t>(stream));
}

size_t pfkv_page_allocator_bytes(int32_t num_pages) { return alloc_state_bytes(num_pages); }

static bool aligned256(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 255u) == 0; }

int pfkv_page_allocator_init(void *state, size_t state_bytes, int32_t num_pages, const int32_t *held_pages,
                             int32_t n_held, void *stream) {
  if (!state) return PFKV_ERR_NULL;
  if (num_pages < 1 || n_held < 0) return PFKV_ERR_SHAPE;
  if (n_held > 0 && !held_pages) return PFKV_ERR_NULL;
  if (state_bytes < alloc_state_bytes(num_pages)) return PFKV_ERR_WORKSPACE;
  if (!aligned256(state)) return PFKV_ERR_ALIGN;
  return launch_alloc_init(state, num_pages, held_pages, n_held, static_cast<cudaStream_t>(stream));
}

int pfkv_page_alloc(void *state, uint32_t *page_tags, int32_t n, int32_t *pages_out, uint32_t *tags_out,
                    uint32_t *status, void *stream) {
  if (!state || !page_tags || !status) return PFKV_ERR_NULL;
  if (n < 0) return PFKV_ERR_SHAPE;
  if (n > 0 && (!pages_out || !tags_out)) return PFKV_ERR_NULL;
  if (!aligned256(state)) return PFKV_ERR_ALIGN;
  return launch_page_alloc(state, page_tags, n, pages_out, tags_out, status, static_cast<cudaStream_t>(stream));
}

int pfkv_page_free(void *state, const int32_t *pages, int32_t n, uint32_t *page_status, void *stream) {
  if (!state) return PFKV_ERR_NULL;
  if (n < 0) return PFKV_ERR_SHAPE;
  if (n == 0) return PFKV_OK;
  if (!pages || !page_status) return PFKV_ERR_NULL;
  if (!aligned256(state)) return PFKV_ERR_ALIGN;
  return launch_page_free(state, pages, n, page_status, static_cast<cudaStream_t>(stream));
}

int pfkv_page_realloc(void *state, uint32_t *page_tags, const int32_t *pages, int32_t n, uint32_t *tags_out,
                      uint32_t *page_status, void *stream) {
  if (!state || !page_tags) return PFKV_ERR_NULL;
  if (n < 0) return PFKV_ERR_SHAPE;
  if (n == 0) return PFKV_OK;
  if (!pages || !tags_out || !page_status) return PFKV_ERR_NULL;
  if (!aligned256(state)) return PFKV_ERR_ALIGN;
  return launch_page_realloc(state, page_tags, pages, n, tags_out, page_status, static_cast<cudaStream_t>(stream));
}

int pfkv_calibrate_scales(const void *rows, int64_t n_rows, int32_t num_heads, int32_t head_dim, float *scale,
                          void *stream) {
  if (n_rows < 0 || num_heads < 1 || head_dim < 1 || num_heads > 65535) return PFKV_ERR_SHAPE;
  if (!scale || (n_rows > 0 && !rows)) return PFKV_ERR_NULL;
  return launch_calibrate(rows, n_rows, num_heads, head_dim, scale, static_cast<cudaStream_t>(stream));
}

int pfkv_e4m3_encode(const float *x, uint8_t *codes, int64_t n, void *stream) {
  if (n < 0) return PFKV_ERR_SHAPE;
  if (n > 0 && (!x || !codes)) return PFKV_ERR_NULL;
  if (!aligned16(x) || (reinterpret_cast<uintptr_t>(codes) & 3u)) return PFKV_ERR_ALIGN;
  return launch_encode(x, codes, n, static_cast<cudaStream_t>(stream));
}

}  // extern "C"
