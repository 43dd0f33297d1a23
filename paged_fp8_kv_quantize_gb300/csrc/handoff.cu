// handoff.cu -- bulk hand-off of whole pages from a BF16 cache to an FP8
// e4m3 cache.
//
// "Smaller, faster, safer: running Kimi and GLM at scale", section
// "Quantizing the KV cache": prefill is compute-bound and keeps its cache in
// BF16, while the decode pool stores FP8 e4m3.  Moving a request from the
// prefill pool to the decode pool therefore quantizes whole pages:
// code = e4m3(fp32(x) / s) per element (IEEE division, round to nearest
// even, saturating at +-448), s the destination's per-head scale or, in
// per-token mode, amax/448 of each (token, head) row (1 for an all-zero row).
// One CTA per (page, head, K|V) slice, up to 8 lanes per row, 16-byte
// loads; the kernel streams src once and writes dst once (HBM-bound).
#include "pfkv_device.cuh"
#include "pfkv_internal.h"

namespace pfkv {

namespace {

__global__ void __launch_bounds__(256) handoff_kernel(pfkv_cache src, pfkv_cache dst, const int *src_pages,
                                                      const int *dst_pages, int n_pages, uint32_t *page_status) {
  const int parts = dst.kv_shared ? 1 : 2;
  const int H = dst.num_kv_heads, S = dst.page_size;
  const int slice = blockIdx.x;  // (page index, head, part)
  const int part = slice % parts, h = (slice / parts) % H, i = slice / (parts * H);
  if (i >= n_pages) return;
  const int sp = src_pages[i], dp = dst_pages[i];
  const bool bad = sp < 0 || sp >= src.num_pages || dp < 0 || dp >= dst.num_pages;
  if (bad) {
    if (part == 0 && h == 0 && threadIdx.x == 0) page_status[i] = PFKV_ST_PAGE_OOB;
    return;
  }
  if (part == 0 && h == 0 && threadIdx.x == 0) page_status[i] = 0u;
  const int D = part ? dst.v_head_dim : dst.head_dim;
  const uint16_t *in = reinterpret_cast<const uint16_t *>(part ? src.v_pool : src.k_pool) +
                       ((size_t)sp * H + h) * S * D;
  uint8_t *out = reinterpret_cast<uint8_t *>(part ? dst.v_pool : dst.k_pool) + ((size_t)dp * H + h) * S * D;
  float *scale_arr = part ? dst.v_scale : dst.k_scale;
  const bool per_token = dst.scale_mode == PFKV_SCALE_PER_TOKEN;
  const float head_scale = per_token ? 1.f : scale_arr[h];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // lanes per row (a power of two, so the amax shuffles stay inside a row),
  // each reading 16-byte chunks of 8 elements
  const int lpr = D >= 64 ? 8 : D >= 32 ? 4 : D >= 16 ? 2 : 1;
  const int rows_per_warp_step = 32 / lpr;
  for (int r0 = warp * rows_per_warp_step; r0 < S; r0 += 8 * rows_per_warp_step) {
    const int r = r0 + lane / lpr, sub = lane % lpr;
    const bool row_ok = r < S && lane < rows_per_warp_step * lpr;
    float amax = 0.f;
    if (per_token) {
      if (row_ok)
        for (int k = sub * 8; k < D; k += lpr * 8) {
          const uint4 v = *reinterpret_cast<const uint4 *>(in + (size_t)r * D + k);
          const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            amax = fmaxf(amax, fabsf(__uint_as_float(w[j] << 16)));
            amax = fmaxf(amax, fabsf(__uint_as_float(w[j] & 0xffff0000u)));
          }
        }
      for (int o = 1; o < lpr; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    }
    if (!row_ok) continue;
    const float s = per_token ? (amax > 0.f ? __fdiv_rn(amax, 448.0f) : 1.0f) : head_scale;
    if (per_token && sub == 0) scale_arr[((size_t)dp * H + h) * S + r] = s;
    for (int k = sub * 8; k < D; k += lpr * 8) {
      const uint4 v = *reinterpret_cast<const uint4 *>(in + (size_t)r * D + k);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
      uint32_t o2[2];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const uint32_t lo = f32x2_to_e4m3x2(__fdiv_rn(__uint_as_float(w[2 * j] << 16), s),
                                            __fdiv_rn(__uint_as_float(w[2 * j] & 0xffff0000u), s));
        const uint32_t hi = f32x2_to_e4m3x2(__fdiv_rn(__uint_as_float(w[2 * j + 1] << 16), s),
                                            __fdiv_rn(__uint_as_float(w[2 * j + 1] & 0xffff0000u), s));
        o2[j] = lo | (hi << 16);
      }
      *reinterpret_cast<uint2 *>(out + (size_t)r * D + k) = make_uint2(o2[0], o2[1]);
    }
  }
}

}  // namespace

int launch_handoff(const pfkv_cache &src, const pfkv_cache &dst, const int *src_pages, const int *dst_pages,
                   int n_pages, uint32_t *page_status, cudaStream_t s) {
  if (n_pages == 0) return PFKV_OK;
  const long long slices = (long long)n_pages * dst.num_kv_heads * (dst.kv_shared ? 1 : 2);
  if (slices > 0x7fffffffLL) return PFKV_ERR_SHAPE;
  handoff_kernel<<<(unsigned)slices, 256, 0, s>>>(src, dst, src_pages, dst_pages, n_pages, page_status);
  return cuda_ok(cudaGetLastError(), "handoff kernel launch");
}

}  // namespace pfkv
