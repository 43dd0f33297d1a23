// pfkv_internal.h -- declarations shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/pfkv.h"

namespace pfkv {

// Decode workspace carve-up.
struct WsLayout {
  size_t split_first, split_count, part_ml, part_o, part_st, cta_abort, qterms, qfac, total;
};
constexpr int kMaxCtas = 4096;  // decode split grid: at most this many CTAs (one abort word each)
// latent: the latent-stream path also keeps each request's query as two e4m3
// terms in the operand image its kernel loads (qterms, 72 KB per request)
// and one factor per head (qfac), written by its query-term kernel.
WsLayout ws_layout(int batch, int q_heads, int v_dim, int max_splits, bool latent);
constexpr size_t kLatentQTermBytes = 128 * 576;  // 128 operand rows (two terms x 64 heads) x 576 codes

struct DecodeArgs {
  // cache
  int P, S, Hkv, D, Dv, scale_mode, dtype, kv_shared;
  const void *k_pool, *v_pool;
  const float *k_scale, *v_scale;
  const uint32_t *page_tags;
  // request batch
  const void *q;
  int Hq, G;  // query heads; query heads per KV head
  // Head groups (grouped-query path): the G query heads of a KV head are cut
  // into kv_sub groups of up to Gs heads, each run as a "virtual" KV head by
  // its own CTAs; Hkv then counts virtual heads (num_kv_heads * kv_sub).
  // Virtual head v reads KV head v / kv_sub for query heads
  // (v / kv_sub) G + (v % kv_sub) Gs .. + min(Gs, G - (v % kv_sub) Gs) - 1.
  int kv_sub, Gs;
  const int *seq_lens, *block_table;
  const uint32_t *block_tags;
  int B, MP;
  float sm_scale_log2;  // softmax_scale * log2(e)
  uint32_t flags;
  int max_splits;
  // workspace and outputs
  int *split_first, *split_count;  // per request: number of its first piece, number of pieces
  float2 *part_ml;
  float *part_o;
  float *out;
  uint32_t *status;
  // decode step only (append == 1): the new rows k_new / v_new [B][Hkv][D]
  // bf16 go to position seq_lens[b] - 1 of each request; the split kernel's
  // page loader writes each (request, KV head)'s row through `cache` (the same
  // pools, writable) just before it copies that page.
  int append;
  const uint16_t *k_new, *v_new;
  pfkv_cache cache;
  // Work split (no plan kernel): every split CTA works out its own pieces
  // from seq_lens.  ranges = CTA groups (one CTA per KV head each); the chunk
  // rule of small or lopsided batches takes pieces of at least
  // min_chunk_pages pages, about target_items of them over all KV heads.
  // Written per call: split_first / split_count of every request with a
  // valid length (by the head-0 CTA holding its first piece),
  // part_st[piece * st_groups + group] (status bits found by each head
  // group's item of the piece) and cta_abort[0 .. n_ctas) (1: a
  // wait of that CTA gave up).  The merge turns them into status[] and zeroes
  // the rows of faulted requests.
  int ranges, target_items, min_chunk_pages, n_ctas;
  int st_groups;  // status words per piece in part_st (grouped-query path: one per head group)
  // latent-stream path: the query terms and per-head factors (see ws_layout)
  uint8_t *qterms;
  float *qfac;
  int piece_cost;  // cut rule: pages' worth of time one piece costs beyond its pages
  uint32_t *part_st;
  int *cta_abort;
};

// Tensor-map encoder obtained from the driver without linking libcuda.
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_tiled_fn();

int num_sms();

// launchers (return PFKV_* codes)
int launch_gqa_decode(const DecodeArgs &a, cudaStream_t s);
int launch_latent_decode(const DecodeArgs &a, cudaStream_t s);
int launch_append(const pfkv_cache &c, const void *k_new, const void *v_new, int n_rows, const int *row_req,
                  const int *positions, const int *block_table, const uint32_t *block_tags, int batch,
                  int max_pages, uint32_t flags, uint32_t *status, cudaStream_t s);
int launch_handoff(const pfkv_cache &src, const pfkv_cache &dst, const int *src_pages, const int *dst_pages,
                   int n_pages, uint32_t *page_status, cudaStream_t s);
size_t alloc_state_bytes(int num_pages);
int launch_alloc_init(void *state, int num_pages, const int *held_pages, int n_held, cudaStream_t s);
int launch_page_alloc(void *state, uint32_t *page_tags, int n, int *pages_out, uint32_t *tags_out, uint32_t *status,
                      cudaStream_t s);
int launch_page_free(void *state, const int *pages, int n, uint32_t *page_status, cudaStream_t s);
int launch_page_realloc(void *state, uint32_t *page_tags, const int *pages, int n, uint32_t *tags_out,
                        uint32_t *page_status, cudaStream_t s);
int launch_calibrate(const void *rows, int64_t n_rows, int heads, int dim, float *scale, cudaStream_t s);
int launch_encode(const float *x, uint8_t *codes, int64_t n, cudaStream_t s);

// The argument checks a decode call makes before it looks at the workspace.
int decode_precheck(int want_dtype, const pfkv_cache *c, int32_t Hq, int32_t batch, int32_t max_pages,
                    int32_t max_splits);

// Records the CUDA error behind a PFKV_ERR_CUDA return (per host thread).
int cuda_fail(cudaError_t e, const char *where);
inline int cuda_ok(cudaError_t e, const char *where = "kernel launch") {
  return e == cudaSuccess ? PFKV_OK : cuda_fail(e, where);
}

}  // namespace pfkv
