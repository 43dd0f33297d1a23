// append_device.cuh -- one warp writes one (row, K|V, head) of a new token
// into the paged cache.  Used by the stand-alone append kernel and by the
// decode step's page loaders (which write a request's new row into its page
// just before copying that page).
//
// "Smaller, faster, safer: running Kimi and GLM at scale", section
// "Quantizing the KV cache": the decode pool stores K and V as FP8 e4m3.
// A new row x (bf16) becomes codes e4m3(fp32(x) / s): IEEE fp32 division,
// round to nearest even, saturating at +-448; s is the head's calibrated
// scale amax/448, or, in per-token mode, the row's own amax/448 (1 for an
// all-zero row).  A BF16 cache takes the bits as they are.  The destination
// page is bounds- and (optionally) tag-checked first, as the post's
// cache-protection passage does before a read; a refused row writes nothing.
#pragma once

#include "pfkv_device.cuh"
#include "pfkv_internal.h"

namespace pfkv {

// Destination check of an append at logical position pos of request b.
// Returns 0 or the PFKV_ST_* bit; *page gets the physical page when 0.
__device__ __forceinline__ uint32_t append_target(const pfkv_cache &c, int b, int pos, const int *block_table,
                                                  const uint32_t *block_tags, int max_pages, uint32_t flags,
                                                  int *page) {
  const int S = c.page_size;
  if (pos < 0 || (long long)pos >= (long long)max_pages * S) return PFKV_ST_BAD_LEN;
  const int i = pos / S;
  const int p = block_table[(size_t)b * max_pages + i];
  if (p < 0 || p >= c.num_pages) return PFKV_ST_PAGE_OOB;
  if ((flags & PFKV_FLAG_TAG_CHECK) && c.page_tags[p] != block_tags[(size_t)b * max_pages + i])
    return PFKV_ST_STALE_TAG;
  *page = p;
  return 0u;
}

// max(m, |x|) over the 8 bf16 values of v.
__device__ __forceinline__ float amax8(uint4 v, float m) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    m = fmaxf(m, fabsf(__uint_as_float(w[q] << 16)));
    m = fmaxf(m, fabsf(__uint_as_float(w[q] & 0xffff0000u)));
  }
  return m;
}

// e4m3 codes of x / s for the 8 bf16 values of v (IEEE division, RNE, satfinite).
__device__ __forceinline__ uint2 e4m3x8(uint4 v, float s) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t out[2];
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const uint32_t lo = f32x2_to_e4m3x2(__fdiv_rn(__uint_as_float(w[2 * q] << 16), s),
                                        __fdiv_rn(__uint_as_float(w[2 * q] & 0xffff0000u), s));
    const uint32_t hi = f32x2_to_e4m3x2(__fdiv_rn(__uint_as_float(w[2 * q + 1] << 16), s),
                                        __fdiv_rn(__uint_as_float(w[2 * q + 1] & 0xffff0000u), s));
    out[q] = lo | (hi << 16);
  }
  return make_uint2(out[0], out[1]);
}

// Per-token scale of a row from the warp's partial maxima; lane 0 stores it.
__device__ __forceinline__ float token_scale(float amax, float *dst, int lane) {
  for (int off = 16; off; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  const float s = amax > 0.f ? __fdiv_rn(amax, 448.0f) : 1.0f;
  if (lane == 0) *dst = s;
  return s;
}

// A new row as one warp holds it: lane l has values 8l + 256j (j <
// kAppendRegs) of the row, plus the head's scale in per-head FP8 mode.
// Loaded before the destination is looked up, so that these loads overlap
// the page-table and tag reads.
constexpr int kAppendRegs = 3;  // rows of up to 768 values

struct AppendRow {
  uint4 v[kAppendRegs];
  float s;
};

// True when the register form carries whole rows of this cache.
__device__ __forceinline__ bool append_row_fits(const pfkv_cache &c) {
  return c.head_dim <= 256 * kAppendRegs && c.v_head_dim <= 256 * kAppendRegs;
}

// Loads row `row` of k_new / v_new ([rows][num_kv_heads][dim] bf16), part
// (0 = K, 1 = V) and head h.  Whole warp.
template <bool kFp8>
__device__ __forceinline__ AppendRow append_row_load(const pfkv_cache &c, const uint16_t *k_new,
                                                     const uint16_t *v_new, int row, int part, int h, int lane) {
  const int D = part ? c.v_head_dim : c.head_dim;
  const uint16_t *src = (part ? v_new : k_new) + ((size_t)row * c.num_kv_heads + h) * D;
  AppendRow r;
#pragma unroll
  for (int j = 0; j < kAppendRegs; ++j) {
    const int k = lane * 8 + 256 * j;
    r.v[j] = k < D ? *reinterpret_cast<const uint4 *>(src + k) : make_uint4(0u, 0u, 0u, 0u);
  }
  r.s = 0.f;
  if (kFp8 && c.scale_mode != PFKV_SCALE_PER_TOKEN) r.s = (part ? c.v_scale : c.k_scale)[h];
  return r;
}

// Writes a loaded row to slot pos % S of `page`: BF16 bits as they are, or
// e4m3 codes of x / s (per-token mode: s = the row's amax / 448 or 1 for an
// all-zero row, stored beside the row).  Whole warp.
template <bool kFp8>
__device__ __forceinline__ void append_row_store(const pfkv_cache &c, const AppendRow &r, int part, int h, int page,
                                                 int pos, int lane) {
  const int D = part ? c.v_head_dim : c.head_dim;
  const size_t dst_row = ((size_t)page * c.num_kv_heads + h) * c.page_size + (pos % c.page_size);
  if constexpr (!kFp8) {
    uint16_t *dst = reinterpret_cast<uint16_t *>(part ? c.v_pool : c.k_pool) + dst_row * D;
#pragma unroll
    for (int j = 0; j < kAppendRegs; ++j)
      if (lane * 8 + 256 * j < D) *reinterpret_cast<uint4 *>(dst + lane * 8 + 256 * j) = r.v[j];
  } else {
    uint8_t *dst = reinterpret_cast<uint8_t *>(part ? c.v_pool : c.k_pool) + dst_row * D;
    float s = r.s;
    if (c.scale_mode == PFKV_SCALE_PER_TOKEN) {
      float amax = 0.f;  // the zero-filled values beyond D leave it as it is
#pragma unroll
      for (int j = 0; j < kAppendRegs; ++j) amax = amax8(r.v[j], amax);
      s = token_scale(amax, (part ? c.v_scale : c.k_scale) + dst_row, lane);
    }
#pragma unroll
    for (int j = 0; j < kAppendRegs; ++j)
      if (lane * 8 + 256 * j < D) *reinterpret_cast<uint2 *>(dst + lane * 8 + 256 * j) = e4m3x8(r.v[j], s);
  }
}

// Rows wider than the register form: the same arithmetic, read as it goes.
template <bool kFp8>
__device__ __forceinline__ void append_row_wide(const pfkv_cache &c, const uint16_t *k_new, const uint16_t *v_new,
                                                int row, int part, int h, int page, int pos, int lane) {
  const int D = part ? c.v_head_dim : c.head_dim;
  const uint16_t *src = (part ? v_new : k_new) + ((size_t)row * c.num_kv_heads + h) * D;
  const size_t dst_row = ((size_t)page * c.num_kv_heads + h) * c.page_size + (pos % c.page_size);
  if constexpr (!kFp8) {
    uint16_t *dst = reinterpret_cast<uint16_t *>(part ? c.v_pool : c.k_pool) + dst_row * D;
    for (int k = lane * 8; k < D; k += 256)
      *reinterpret_cast<uint4 *>(dst + k) = *reinterpret_cast<const uint4 *>(src + k);
  } else {
    uint8_t *dst = reinterpret_cast<uint8_t *>(part ? c.v_pool : c.k_pool) + dst_row * D;
    float *scale_arr = part ? c.v_scale : c.k_scale;
    float s;
    if (c.scale_mode == PFKV_SCALE_PER_TOKEN) {
      float amax = 0.f;
      for (int k = lane * 8; k < D; k += 256) amax = amax8(*reinterpret_cast<const uint4 *>(src + k), amax);
      s = token_scale(amax, scale_arr + dst_row, lane);
    } else {
      s = scale_arr[h];
    }
    for (int k = lane * 8; k < D; k += 256)
      *reinterpret_cast<uint2 *>(dst + k) = e4m3x8(*reinterpret_cast<const uint4 *>(src + k), s);
  }
}

}  // namespace pfkv
