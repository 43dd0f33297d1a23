/*
 * pfkv_oracle.c -- plain, slow, fp64 CPU oracle for the paged FP8 KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the tests, the smoke check and the benchmark's CPU
 * baseline leg do.  It shares no code, header, table or constant generator
 * with the CUDA library; the few numbers that are an interface (status bits,
 * flag bits, layout order) are restated here by hand.
 *
 * What it computes, and where that comes from:
 *
 *  - "Smaller, faster, safer: running Kimi and GLM at scale" (Cloudflare),
 *    section "Quantizing the KV cache": the decode pool stores K and V as
 *    FP8 e4m3 instead of BF16, and the FP8 attention kernel converts the
 *    values as it reads them.  The e4m3 format itself is the OCP 8-bit
 *    floating point E4M3 ("FN") encoding: 1 sign, 4 exponent (bias 7),
 *    3 mantissa bits, no infinities, S.1111.111 is NaN, max finite 448.
 *  - same post, the cache-protection passage: every page of the shared
 *    physical cache carries a tag that changes on each reallocation; the
 *    mapping's tag is compared with the page's before a read, and a
 *    mismatch aborts the request instead of returning wrong data.  The
 *    check is off by default.
 *  - Attention is the plain definition: z = tau * q.k, softmax over the
 *    request's tokens, o = sum p v, evaluated in fp64 on the dequantized
 *    cache.
 *
 * Readings where the pages are silent (the plainest one the rest supports):
 *  R1  encode saturates: |y| > 448 encodes as +-448 (E4M3FN has no inf).
 *  R2  the sign survives rounding to zero: -tiny -> 0x80.
 *  R3  quantize divides: code = e4m3(fp32(x) / s), an IEEE fp32 division.
 *  R4  per-head scale s = fp32(amax / 448) with amax over the calibration
 *      rows; R5: amax == 0 gives s = 1.
 *  R6  layout: pool[page][kv_head][slot][dim], K and V in separate pools;
 *      per-token scales at [page][kv_head][slot].
 *  R7  the append also checks its destination page and writes nothing on
 *      a bad page.
 *  R8  attention output is fp32 [batch][q_heads][v_dim] (here fp64).
 *  R13 a page's tag advances by one (mod 2^32) each time the page is handed
 *      to an owner: at allocation and at a move to a new owner; freeing
 *      leaves it.  A fresh allocator hands out pages in increasing id order
 *      and reuses the most recently freed page first (a stack).
 *  NaN input encodes as 0x7F; +-inf saturates like any large value.
 *
 * Build: gcc -O2 -std=c11 -fPIC -shared -pthread pfkv_oracle.c -lm
 */
#define _GNU_SOURCE
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Interface numbers (restated by hand; they must equal the library's). */
#define ORC_DTYPE_BF16 0
#define ORC_DTYPE_FP8 1
#define ORC_SCALE_PER_HEAD 0
#define ORC_SCALE_PER_TOKEN 1
#define ORC_FLAG_TAG_CHECK 1u
#define ORC_ST_STALE_TAG 1u
#define ORC_ST_PAGE_OOB 2u
#define ORC_ST_BAD_LEN 4u
#define ORC_ST_NO_PAGES 16u
#define ORC_ST_NOT_HELD 32u
#define ORC_ST_DUPLICATE 64u

typedef struct {
  int32_t num_pages, page_size, num_kv_heads, head_dim, v_head_dim;
  int32_t kv_shared, dtype, scale_mode;
  void *k_pool, *v_pool;      /* uint8 codes (fp8) or uint16 bits (bf16) */
  float *k_scale, *v_scale;   /* per head [Hkv] or per token [P][Hkv][S] */
  const uint32_t *page_tags;  /* [P] */
} orc_cache;

/* ------------------------------------------------------------------ */
/* Scalars                                                              */
/* ------------------------------------------------------------------ */

/* bfloat16 is the top half of an IEEE binary32. */
double orc_bf16_to_double(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* E4M3 decode straight from the bit-field definition. */
double orc_e4m3_decode(uint8_t c) {
  int sign = (c >> 7) & 1;
  int e = (c >> 3) & 0xF;
  int m = c & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    v = ldexp((double)m / 8.0, -6);          /* subnormal: 0.m * 2^-6 */
  else
    v = ldexp(1.0 + (double)m / 8.0, e - 7); /* normal: 1.m * 2^(e-7) */
  return sign ? -v : v;
}

/*
 * E4M3 encode of an fp32 value: round to nearest, ties to even, saturate
 * to the largest finite magnitude (R1), keep the sign of zero (R2).
 *
 * Within the binade [2^e, 2^(e+1)) the representable step is 2^(e-3); the
 * subnormal range [0, 2^-6) uses the step of the lowest binade, 2^-9.  So
 * with e clamped below at -6, n = |y| / 2^(e-3) is an exact dyadic number,
 * its nearest-even integer r is the rounded significand, and the codes are
 * consecutive integers: code = 8*(e+6) + r.  r == 16 carries into the next
 * binade by the same formula.
 */
uint8_t orc_e4m3_encode(float y) {
  uint8_t sign = signbit(y) ? 0x80 : 0x00;
  double a = fabs((double)y);
  int e;
  double r;
  int code;
  if (isnan(y)) return 0x7F;
  if (a >= 448.0) return sign | 0x7E;
  if (a == 0.0) return sign;
  e = ilogb(a);
  if (e < -6) e = -6;
  r = nearbyint(ldexp(a, 3 - e)); /* default rounding mode: ties to even */
  code = 8 * (e + 6) + (int)r;
  if (code > 0x7E) code = 0x7E; /* rounds past 448: saturate (R1) */
  return sign | (uint8_t)code;
}

/*
 * Independent encoder used only to pin orc_e4m3_encode: look the magnitude
 * up among the 127 non-negative finite code values (binary search over the
 * decoded table), take the nearer neighbour, and on an exact tie the code
 * with an even mantissa (even code).  Values past 448 saturate.
 */
static double g_nearest_tab[127];
static int g_nearest_ready = 0;
static pthread_once_t g_nearest_once = PTHREAD_ONCE_INIT;
static void nearest_init(void) {
  for (int c = 0; c < 127; ++c) g_nearest_tab[c] = orc_e4m3_decode((uint8_t)c);
  g_nearest_ready = 1;
}
uint8_t orc_e4m3_encode_nearest(float y) {
  uint8_t sign = signbit(y) ? 0x80 : 0x00;
  double a = fabs((double)y);
  int lo = 0, hi = 126;
  pthread_once(&g_nearest_once, nearest_init);
  if (isnan(y)) return 0x7F;
  if (a >= g_nearest_tab[126]) return sign | 126;
  /* invariant: tab[lo] <= a < tab[hi] */
  while (hi - lo > 1) {
    int mid = (lo + hi) / 2;
    if (g_nearest_tab[mid] <= a) lo = mid; else hi = mid;
  }
  {
    double dl = a - g_nearest_tab[lo], dh = g_nearest_tab[hi] - a;
    int c;
    if (dl < dh) c = lo;
    else if (dh < dl) c = hi;
    else c = (lo % 2 == 0) ? lo : hi;
    return sign | (uint8_t)c;
  }
}

/* fp32 division y = fp32(x) / s, correctly rounded (R3).  The quotient is
 * formed in double and rounded once to float; for +,-,*,/ of two binary32
 * operands this double rounding always equals the correctly rounded binary32
 * result because 53 >= 2*24 + 2. */
static float fp32_div(float x, float s) { return (float)((double)x / (double)s); }

uint8_t orc_quantize(uint16_t x_bf16, float s) {
  return orc_e4m3_encode(fp32_div((float)orc_bf16_to_double(x_bf16), s));
}

/* s = fp32(amax / 448), amax == 0 -> 1 (R4, R5).  amax is a bf16 value, so
 * the fp64 quotient rounded once to fp32 is the correctly rounded fp32
 * quotient (same argument as above). */
float orc_scale_from_amax(double amax) {
  if (!(amax > 0.0)) return 1.0f;
  return (float)(amax / 448.0);
}

/* ------------------------------------------------------------------ */
/* Bulk codec helpers (used by the tests)                               */
/* ------------------------------------------------------------------ */

void orc_e4m3_encode_array(const float *y, uint8_t *out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_e4m3_encode(y[i]);
}

void orc_e4m3_encode_nearest_array(const float *y, uint8_t *out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_e4m3_encode_nearest(y[i]);
}

void orc_e4m3_encode_bits(const uint32_t *bits, uint8_t *out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) {
    float f;
    memcpy(&f, &bits[i], 4);
    out[i] = orc_e4m3_encode(f);
  }
}

typedef struct {
  uint64_t lo, hi;
  uint64_t mismatches;
  uint64_t first_bad;
} sweep_job;

static void *sweep_worker(void *arg) {
  sweep_job *j = (sweep_job *)arg;
  for (uint64_t u = j->lo; u < j->hi; ++u) {
    uint32_t b = (uint32_t)u;
    float f;
    memcpy(&f, &b, 4);
    if (orc_e4m3_encode(f) != orc_e4m3_encode_nearest(f)) {
      if (j->mismatches == 0) j->first_bad = u;
      j->mismatches++;
    }
  }
  return NULL;
}

/* Compare the two encoders on every fp32 bit pattern in [lo, hi).  Returns
 * the number of disagreements; *first_bad gets the first one (if any). */
uint64_t orc_e4m3_sweep(uint64_t lo, uint64_t hi, int threads, uint64_t *first_bad) {
  pthread_t th[256];
  sweep_job jobs[256];
  uint64_t total = 0, span;
  if (threads < 1) threads = 1;
  if (threads > 256) threads = 256;
  pthread_once(&g_nearest_once, nearest_init);
  span = (hi - lo + (uint64_t)threads - 1) / (uint64_t)threads;
  for (int t = 0; t < threads; ++t) {
    jobs[t].lo = lo + span * (uint64_t)t;
    jobs[t].hi = jobs[t].lo + span > hi ? hi : jobs[t].lo + span;
    if (jobs[t].lo > hi) jobs[t].lo = hi;
    jobs[t].mismatches = 0;
    jobs[t].first_bad = 0;
    pthread_create(&th[t], NULL, sweep_worker, &jobs[t]);
  }
  *first_bad = UINT64_MAX;
  for (int t = 0; t < threads; ++t) {
    pthread_join(th[t], NULL);
    total += jobs[t].mismatches;
    if (jobs[t].mismatches && jobs[t].first_bad < *first_bad) *first_bad = jobs[t].first_bad;
  }
  return total;
}

/* ------------------------------------------------------------------ */
/* Calibration (per-head scales)                                        */
/* ------------------------------------------------------------------ */

/* x: bf16 rows [n_rows][H][D]; scale[h] = fp32(max |x[:, h, :]| / 448). */
void orc_calibrate_per_head(const uint16_t *x, int64_t n_rows, int32_t H, int32_t D, float *scale) {
  for (int32_t h = 0; h < H; ++h) {
    double amax = 0.0;
    for (int64_t r = 0; r < n_rows; ++r)
      for (int32_t d = 0; d < D; ++d) {
        double v = fabs(orc_bf16_to_double(x[(r * H + h) * D + d]));
        if (v > amax) amax = v;
      }
    scale[h] = orc_scale_from_amax(amax);
  }
}

/* ------------------------------------------------------------------ */
/* Page addressing                                                      */
/* ------------------------------------------------------------------ */

static int64_t row_index(const orc_cache *c, int64_t page, int32_t h, int32_t slot) {
  return (page * c->num_kv_heads + h) * (int64_t)c->page_size + slot;
}

/* Status bits for one logical page i of request b (tag compare only when the
 * flag is on). */
static uint32_t page_status(const orc_cache *c, const int32_t *block_table, const uint32_t *block_tags,
                            int32_t max_pages, int32_t b, int32_t i, uint32_t flags, int32_t *page_out) {
  int32_t p = block_table[(int64_t)b * max_pages + i];
  *page_out = p;
  if (p < 0 || p >= c->num_pages) return ORC_ST_PAGE_OOB;
  if ((flags & ORC_FLAG_TAG_CHECK) && c->page_tags[p] != block_tags[(int64_t)b * max_pages + i])
    return ORC_ST_STALE_TAG;
  return 0;
}

/* ------------------------------------------------------------------ */
/* Append / quantize                                                    */
/* ------------------------------------------------------------------ */

/* Write one (token, head) row of D values into a pool. */
static void put_row(const orc_cache *c, void *pool, float *scale_arr, const uint16_t *x, int32_t D,
                    int64_t page, int32_t h, int32_t slot) {
  int64_t r = row_index(c, page, h, slot);
  if (c->dtype == ORC_DTYPE_BF16) {
    memcpy((uint16_t *)pool + r * D, x, (size_t)D * 2);
    return;
  }
  {
    uint8_t *dst = (uint8_t *)pool + r * D;
    float s;
    if (c->scale_mode == ORC_SCALE_PER_TOKEN) {
      double amax = 0.0;
      for (int32_t d = 0; d < D; ++d) {
        double v = fabs(orc_bf16_to_double(x[d]));
        if (v > amax) amax = v;
      }
      s = orc_scale_from_amax(amax);
      scale_arr[r] = s;
    } else {
      s = scale_arr[h];
    }
    for (int32_t d = 0; d < D; ++d) dst[d] = orc_quantize(x[d], s);
  }
}

/*
 * Append n_rows new tokens.  Row i belongs to request row_req[i] (or i when
 * row_req is NULL) at logical position positions[i]; its K row is
 * k_new[i][Hkv][D] and V row v_new[i][Hkv][Dv].  status[batch] is cleared
 * and then collects, per request, the bits of every refused row (R7).
 */
void orc_append(const orc_cache *c, const uint16_t *k_new, const uint16_t *v_new, int32_t n_rows,
                const int32_t *row_req, const int32_t *positions, const int32_t *block_table,
                const uint32_t *block_tags, int32_t batch, int32_t max_pages, uint32_t flags,
                uint32_t *status) {
  const int32_t H = c->num_kv_heads, D = c->head_dim, Dv = c->v_head_dim, S = c->page_size;
  for (int32_t b = 0; b < batch; ++b) status[b] = 0;
  for (int32_t i = 0; i < n_rows; ++i) {
    int32_t b = row_req ? row_req[i] : i;
    int32_t pos = positions[i];
    int32_t page = -1;
    uint32_t st;
    if (b < 0 || b >= batch) continue; /* not a request of this call */
    if (pos < 0 || (int64_t)pos >= (int64_t)max_pages * S) {
      status[b] |= ORC_ST_BAD_LEN;
      continue;
    }
    st = page_status(c, block_table, block_tags, max_pages, b, pos / S, flags, &page);
    if (st) {
      status[b] |= st;
      continue;
    }
    for (int32_t h = 0; h < H; ++h) {
      put_row(c, c->k_pool, c->k_scale, k_new + ((int64_t)i * H + h) * D, D, page, h, pos % S);
      if (!c->kv_shared)
        put_row(c, c->v_pool, c->v_scale, v_new + ((int64_t)i * H + h) * Dv, Dv, page, h, pos % S);
    }
  }
}

/*
 * Hand-off of whole pages from a BF16 cache to an FP8 cache ("Quantizing the
 * KV cache": prefill keeps BF16, decode stores FP8).  Page src_pages[i] of
 * src becomes page dst_pages[i] of dst, each (head, slot) row quantized as an
 * appended row would be.  page_status[i] gets PAGE_OOB for an id outside its
 * pool (nothing written for that pair).
 */
void orc_handoff(const orc_cache *src, const orc_cache *dst, const int32_t *src_pages, const int32_t *dst_pages,
                 int32_t n_pages, uint32_t *page_status) {
  const int32_t H = dst->num_kv_heads, S = dst->page_size, D = dst->head_dim, Dv = dst->v_head_dim;
  for (int32_t i = 0; i < n_pages; ++i) {
    const int32_t sp = src_pages[i], dp = dst_pages[i];
    if (sp < 0 || sp >= src->num_pages || dp < 0 || dp >= dst->num_pages) {
      page_status[i] = ORC_ST_PAGE_OOB;
      continue;
    }
    page_status[i] = 0;
    for (int32_t h = 0; h < H; ++h)
      for (int32_t slot = 0; slot < S; ++slot) {
        const int64_t r = row_index(src, sp, h, slot);
        put_row(dst, dst->k_pool, dst->k_scale, (const uint16_t *)src->k_pool + r * D, D, dp, h, slot);
        if (!dst->kv_shared)
          put_row(dst, dst->v_pool, dst->v_scale, (const uint16_t *)src->v_pool + r * Dv, Dv, dp, h, slot);
      }
  }
}

/* ------------------------------------------------------------------ */
/* Page allocator (the producer side of the tags)                      */
/* ------------------------------------------------------------------ */

/*
 * Same post, cache-protection passage: the tag of a page changes each time
 * the page is reallocated, so a request still holding the old mapping (and
 * the old tag) fails the check.  The allocator below is the plain sequential
 * model: a stack of free page ids, a held flag per page, the tag bumped when
 * a page is given to an owner (R13).  Every call is all-or-nothing per
 * element and processes its list in order.
 *   stack[0 .. *free_count) : free ids; the top (the end) is popped first.
 */
void orc_alloc_init(int32_t *stack, uint8_t *held, int32_t *free_count, int32_t num_pages,
                    const int32_t *held_pages, int32_t n_held) {
  memset(held, 0, (size_t)num_pages);
  for (int32_t i = 0; i < n_held; ++i)
    if (held_pages[i] >= 0 && held_pages[i] < num_pages) held[held_pages[i]] = 1;
  int32_t n = 0;
  for (int32_t p = num_pages - 1; p >= 0; --p) /* smallest free id on top */
    if (!held[p]) stack[n++] = p;
  *free_count = n;
}

/* Take n pages.  Not enough free pages: nothing is taken, pages_out = -1,
 * tags_out = 0, *status = NO_PAGES. */
void orc_page_alloc(int32_t *stack, uint8_t *held, int32_t *free_count, uint32_t *page_tags, int32_t n,
                    int32_t *pages_out, uint32_t *tags_out, uint32_t *status) {
  if (n > *free_count) {
    for (int32_t i = 0; i < n; ++i) {
      pages_out[i] = -1;
      tags_out[i] = 0;
    }
    *status = ORC_ST_NO_PAGES;
    return;
  }
  for (int32_t i = 0; i < n; ++i) {
    const int32_t p = stack[--*free_count];
    held[p] = 1;
    page_tags[p] += 1u;
    pages_out[i] = p;
    tags_out[i] = page_tags[p];
  }
  *status = 0;
}

/* Give pages back.  An id outside the pool: PAGE_OOB; a page that is not
 * held (never taken, or already given back, earlier in this list too):
 * NOT_HELD.  Either way that entry is skipped. */
void orc_page_free(int32_t *stack, uint8_t *held, int32_t *free_count, int32_t num_pages, const int32_t *pages,
                   int32_t n, uint32_t *page_status) {
  for (int32_t i = 0; i < n; ++i) {
    const int32_t p = pages[i];
    if (p < 0 || p >= num_pages) {
      page_status[i] = ORC_ST_PAGE_OOB;
    } else if (!held[p]) {
      page_status[i] = ORC_ST_NOT_HELD;
    } else {
      held[p] = 0;
      stack[(*free_count)++] = p;
      page_status[i] = 0;
    }
  }
}

/* Move held pages to new owners without a trip through the free list: each
 * listed page's tag advances by one and the new tag is returned.  A page
 * listed twice is moved once; the later entries get DUPLICATE (tag_out 0),
 * as do entries that are OOB or NOT_HELD. */
void orc_page_realloc(const uint8_t *held, int32_t num_pages, uint32_t *page_tags, const int32_t *pages, int32_t n,
                      uint32_t *tags_out, uint32_t *page_status) {
  for (int32_t i = 0; i < n; ++i) {
    const int32_t p = pages[i];
    tags_out[i] = 0;
    if (p < 0 || p >= num_pages) {
      page_status[i] = ORC_ST_PAGE_OOB;
      continue;
    }
    if (!held[p]) {
      page_status[i] = ORC_ST_NOT_HELD;
      continue;
    }
    int seen = 0;
    for (int32_t j = 0; j < i && !seen; ++j) seen = pages[j] == p;
    if (seen) {
      page_status[i] = ORC_ST_DUPLICATE;
      continue;
    }
    page_tags[p] += 1u;
    tags_out[i] = page_tags[p];
    page_status[i] = 0;
  }
}

/* ------------------------------------------------------------------ */
/* Decode attention                                                     */
/* ------------------------------------------------------------------ */

/* Dequantized value of element d of the (page, h, slot) row. */
static double load_k(const orc_cache *c, int64_t page, int32_t h, int32_t slot, int32_t d) {
  int64_t r = row_index(c, page, h, slot);
  if (c->dtype == ORC_DTYPE_BF16) return orc_bf16_to_double(((const uint16_t *)c->k_pool)[r * c->head_dim + d]);
  {
    double s = c->scale_mode == ORC_SCALE_PER_TOKEN ? c->k_scale[r] : c->k_scale[h];
    return orc_e4m3_decode(((const uint8_t *)c->k_pool)[r * c->head_dim + d]) * s;
  }
}

static double load_v(const orc_cache *c, int64_t page, int32_t h, int32_t slot, int32_t d) {
  int64_t r;
  if (c->kv_shared) return load_k(c, page, h, slot, d); /* V = leading dims of the K row */
  r = row_index(c, page, h, slot);
  if (c->dtype == ORC_DTYPE_BF16) return orc_bf16_to_double(((const uint16_t *)c->v_pool)[r * c->v_head_dim + d]);
  {
    double s = c->scale_mode == ORC_SCALE_PER_TOKEN ? c->v_scale[r] : c->v_scale[h];
    return orc_e4m3_decode(((const uint8_t *)c->v_pool)[r * c->v_head_dim + d]) * s;
  }
}

/* Status of request b for a decode call: length check, then every logical
 * page i < ceil(L/S) is inspected.  A bad length inspects nothing. */
static uint32_t request_status(const orc_cache *c, const int32_t *seq_lens, const int32_t *block_table,
                               const uint32_t *block_tags, int32_t max_pages, int32_t b, uint32_t flags) {
  int32_t L = seq_lens[b], S = c->page_size, p;
  uint32_t st = 0;
  if (L < 1 || (int64_t)L > (int64_t)max_pages * S) return ORC_ST_BAD_LEN;
  for (int32_t i = 0; i < (L + S - 1) / S; ++i) st |= page_status(c, block_table, block_tags, max_pages, b, i, flags, &p);
  return st;
}

/* One (request, query head): out[Dv] = softmax(tau q.K^T) V in fp64. */
static void attend_one(const orc_cache *c, const uint16_t *q_bh, int32_t g, int32_t L, const int32_t *table_b,
                       double tau, double *z, double *out) {
  const int32_t D = c->head_dim, Dv = c->v_head_dim, S = c->page_size;
  double zmax = -INFINITY, denom = 0.0;
  for (int32_t t = 0; t < L; ++t) {
    int64_t page = table_b[t / S];
    double acc = 0.0;
    for (int32_t d = 0; d < D; ++d) acc += orc_bf16_to_double(q_bh[d]) * load_k(c, page, g, t % S, d);
    z[t] = tau * acc;
    if (z[t] > zmax) zmax = z[t];
  }
  for (int32_t t = 0; t < L; ++t) {
    z[t] = exp(z[t] - zmax);
    denom += z[t];
  }
  for (int32_t d = 0; d < Dv; ++d) out[d] = 0.0;
  for (int32_t t = 0; t < L; ++t) {
    int64_t page = table_b[t / S];
    double p = z[t] / denom;
    for (int32_t d = 0; d < Dv; ++d) out[d] += p * load_v(c, page, g, t % S, d);
  }
}

typedef struct {
  const orc_cache *c;
  const uint16_t *q;
  int32_t Hq;
  const int32_t *seq_lens, *block_table;
  int32_t batch, max_pages;
  double tau;
  const uint32_t *status;
  double *out;
  int32_t next; /* work counter over (b, h) */
  pthread_mutex_t mu;
} decode_ctx;

static void *decode_worker(void *arg) {
  decode_ctx *x = (decode_ctx *)arg;
  const orc_cache *c = x->c;
  double *z = NULL;
  int32_t zcap = 0;
  for (;;) {
    int32_t w, b, h, L;
    pthread_mutex_lock(&x->mu);
    w = x->next++;
    pthread_mutex_unlock(&x->mu);
    if (w >= x->batch * x->Hq) break;
    b = w / x->Hq;
    h = w % x->Hq;
    L = x->seq_lens[b];
    if (x->status[b]) continue; /* aborted: output stays zero */
    if (L > zcap) {
      free(z);
      zcap = L;
      z = (double *)malloc(sizeof(double) * (size_t)zcap);
    }
    attend_one(c, x->q + ((int64_t)b * x->Hq + h) * c->head_dim, h / (x->Hq / c->num_kv_heads), L,
               x->block_table + (int64_t)b * x->max_pages, x->tau, z,
               x->out + ((int64_t)b * x->Hq + h) * c->v_head_dim);
  }
  free(z);
  return NULL;
}

/*
 * Paged decode attention.  q: bf16 [batch][Hq][D]; out: [batch][Hq][Dv]
 * (zero for an aborted request); status[batch] as described above.
 * threads > 1 splits the (request, head) pairs over POSIX threads; the
 * arithmetic of each pair is the same either way.
 */
void orc_decode(const orc_cache *c, const uint16_t *q, int32_t Hq, const int32_t *seq_lens,
                const int32_t *block_table, const uint32_t *block_tags, int32_t batch, int32_t max_pages,
                double softmax_scale, uint32_t flags, double *out, uint32_t *status, int32_t threads) {
  decode_ctx x;
  pthread_t th[256];
  for (int32_t b = 0; b < batch; ++b)
    status[b] = request_status(c, seq_lens, block_table, block_tags, max_pages, b, flags);
  memset(out, 0, sizeof(double) * (size_t)batch * Hq * c->v_head_dim);
  x.c = c;
  x.q = q;
  x.Hq = Hq;
  x.seq_lens = seq_lens;
  x.block_table = block_table;
  x.batch = batch;
  x.max_pages = max_pages;
  x.tau = softmax_scale;
  x.status = status;
  x.out = out;
  x.next = 0;
  pthread_mutex_init(&x.mu, NULL);
  if (threads <= 1) {
    decode_worker(&x);
  } else {
    if (threads > 256) threads = 256;
    for (int t = 0; t < threads; ++t) pthread_create(&th[t], NULL, decode_worker, &x);
    for (int t = 0; t < threads; ++t) pthread_join(th[t], NULL);
  }
  pthread_mutex_destroy(&x.mu);
}
