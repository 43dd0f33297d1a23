// append.cu -- quantize-on-append into the paged cache, per-head scale
// calibration and a bulk e4m3 encoder.
//
// "Smaller, faster, safer: running Kimi and GLM at scale", section
// "Quantizing the KV cache": the decode pool stores K and V as FP8 e4m3.
// A new row x (bf16) becomes codes e4m3(fp32(x) / s): IEEE fp32 division,
// round to nearest even, saturating at +-448; s is the head's calibrated
// scale amax/448, or, in per-token mode, the row's own amax/448.  The
// destination page is bounds- and (optionally) tag-checked first, as the
// post's cache-protection passage does before a read; a refused row writes
// nothing.
#include "pfkv_device.cuh"
#include "pfkv_internal.h"

namespace pfkv {

namespace {

// One warp per (row, part, head); part 0 = K, 1 = V.  blockDim = 128.
template <bool kFp8>
__global__ void __launch_bounds__(128) append_kernel(pfkv_cache c, const uint16_t *k_new, const uint16_t *v_new,
                                                     int n_rows, const int *row_req, const int *positions,
                                                     const int *block_table, const uint32_t *block_tags,
                                                     int batch, int max_pages, uint32_t flags, uint32_t *status) {
  const int row = blockIdx.x;
  const int lane = threadIdx.x & 31;
  const int unit = blockIdx.y * 4 + (threadIdx.x >> 5);  // (part, head)
  const int parts = c.kv_shared ? 1 : 2;
  if (row >= n_rows) return;
  const int b = row_req ? row_req[row] : row;
  if (b < 0 || b >= batch) return;
  const int pos = positions[row];
  const int S = c.page_size;
  uint32_t bad = 0;
  int page = -1;
  if (pos < 0 || (long long)pos >= (long long)max_pages * S) {
    bad = PFKV_ST_BAD_LEN;
  } else {
    const int i = pos / S;
    page = block_table[(size_t)b * max_pages + i];
    if (page < 0 || page >= c.num_pages) bad = PFKV_ST_PAGE_OOB;
    else if ((flags & PFKV_FLAG_TAG_CHECK) && c.page_tags[page] != block_tags[(size_t)b * max_pages + i])
      bad = PFKV_ST_STALE_TAG;
  }
  if (bad) {
    if (unit == 0 && lane == 0) atomicOr(&status[b], bad);
    return;
  }
  if (unit >= parts * c.num_kv_heads) return;
  const int part = unit / c.num_kv_heads, h = unit - part * c.num_kv_heads;
  const int D = part ? c.v_head_dim : c.head_dim;
  const uint16_t *src = (part ? v_new : k_new) + ((size_t)row * c.num_kv_heads + h) * D;
  const size_t dst_row = ((size_t)page * c.num_kv_heads + h) * S + (pos % S);
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
      for (int k = lane * 8; k < D; k += 256) {
        const uint4 v = *reinterpret_cast<const uint4 *>(src + k);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          amax = fmaxf(amax, fabsf(__uint_as_float(w[j] << 16)));
          amax = fmaxf(amax, fabsf(__uint_as_float(w[j] & 0xffff0000u)));
        }
      }
      for (int off = 16; off; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
      s = amax > 0.f ? __fdiv_rn(amax, 448.0f) : 1.0f;
      if (lane == 0) scale_arr[dst_row] = s;
    } else {
      s = scale_arr[h];
    }
    for (int k = lane * 8; k < D; k += 256) {
      const uint4 v = *reinterpret_cast<const uint4 *>(src + k);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
      uint32_t out[2];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const uint32_t lo = f32x2_to_e4m3x2(__fdiv_rn(__uint_as_float(w[2 * j] << 16), s),
                                            __fdiv_rn(__uint_as_float(w[2 * j] & 0xffff0000u), s));
        const uint32_t hi = f32x2_to_e4m3x2(__fdiv_rn(__uint_as_float(w[2 * j + 1] << 16), s),
                                            __fdiv_rn(__uint_as_float(w[2 * j + 1] & 0xffff0000u), s));
        out[j] = lo | (hi << 16);
      }
      *reinterpret_cast<uint2 *>(dst + k) = make_uint2(out[0], out[1]);
    }
  }
}

// amax per head into scale[] (as fp32 bits, non-negative floats order like uints)
__global__ void __launch_bounds__(256) amax_kernel(const uint16_t *rows, int64_t n_rows, int heads, int dim,
                                                   unsigned *amax_bits) {
  const int h = blockIdx.y;
  float m = 0.f;
  const int64_t per_row = dim;
  for (int64_t r = blockIdx.x; r < n_rows; r += gridDim.x) {
    const uint16_t *x = rows + ((size_t)r * heads + h) * per_row;
    for (int k = threadIdx.x; k < dim; k += blockDim.x) m = fmaxf(m, fabsf(__uint_as_float((uint32_t)x[k] << 16)));
  }
  for (int off = 16; off; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  if ((threadIdx.x & 31) == 0 && m > 0.f) atomicMax(&amax_bits[h], __float_as_uint(m));
}

__global__ void amax_to_scale_kernel(float *scale, int heads) {
  const int h = blockIdx.x * blockDim.x + threadIdx.x;
  if (h < heads) {
    const float amax = __uint_as_float(reinterpret_cast<unsigned *>(scale)[h]);
    scale[h] = amax > 0.f ? __fdiv_rn(amax, 448.0f) : 1.0f;
  }
}

__global__ void encode_kernel(const float *x, uint8_t *codes, int64_t n) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 4; i < n; i += stride * 4) {
    if (i + 4 <= n) {
      const float4 v = *reinterpret_cast<const float4 *>(x + i);
      const uint32_t c = f32x2_to_e4m3x2(v.x, v.y) | (f32x2_to_e4m3x2(v.z, v.w) << 16);
      *reinterpret_cast<uint32_t *>(codes + i) = c;
    } else {
      for (int64_t j = i; j < n; ++j) codes[j] = (uint8_t)f32x2_to_e4m3x2(x[j], 0.f);
    }
  }
}

}  // namespace

int launch_append(const pfkv_cache &c, const void *k_new, const void *v_new, int n_rows, const int *row_req,
                  const int *positions, const int *block_table, const uint32_t *block_tags, int batch,
                  int max_pages, uint32_t flags, uint32_t *status, cudaStream_t s) {
  int rc = cuda_ok(cudaMemsetAsync(status, 0, sizeof(uint32_t) * (size_t)batch, s), "status memset");
  if (rc) return rc;
  if (n_rows == 0) return PFKV_OK;
  const int units = (c.kv_shared ? 1 : 2) * c.num_kv_heads;
  const dim3 grid(n_rows, (units + 3) / 4);
  if (c.dtype == PFKV_DTYPE_FP8_E4M3)
    append_kernel<true><<<grid, 128, 0, s>>>(c, (const uint16_t *)k_new, (const uint16_t *)v_new, n_rows, row_req,
                                             positions, block_table, block_tags, batch, max_pages, flags, status);
  else
    append_kernel<false><<<grid, 128, 0, s>>>(c, (const uint16_t *)k_new, (const uint16_t *)v_new, n_rows, row_req,
                                              positions, block_table, block_tags, batch, max_pages, flags, status);
  return cuda_ok(cudaGetLastError());
}

int launch_calibrate(const void *rows, int64_t n_rows, int heads, int dim, float *scale, cudaStream_t s) {
  int rc = cuda_ok(cudaMemsetAsync(scale, 0, sizeof(float) * (size_t)heads, s), "scale memset");
  if (rc) return rc;
  if (n_rows > 0) {
    const int gx = (int)(n_rows < 4096 ? n_rows : 4096);
    amax_kernel<<<dim3(gx, heads), 256, 0, s>>>((const uint16_t *)rows, n_rows, heads, dim, (unsigned *)scale);
  }
  amax_to_scale_kernel<<<(heads + 127) / 128, 128, 0, s>>>(scale, heads);
  return cuda_ok(cudaGetLastError());
}

int launch_encode(const float *x, uint8_t *codes, int64_t n, cudaStream_t s) {
  if (n == 0) return PFKV_OK;
  int64_t blocks = (n / 4 + 255) / 256 + 1;
  if (blocks > 65536) blocks = 65536;
  encode_kernel<<<(int)blocks, 256, 0, s>>>(x, codes, n);
  return cuda_ok(cudaGetLastError());
}

}  // namespace pfkv
