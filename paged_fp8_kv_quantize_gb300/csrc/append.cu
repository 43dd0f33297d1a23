// append.cu -- quantize-on-append into the paged cache, per-head scale
// calibration and a bulk e4m3 encoder.
//
// "Smaller, faster, safer: running Kimi and GLM at scale", section
// "Quantizing the KV cache": the decode pool stores K and V as FP8 e4m3;
// a new row is quantized as it is written (append_device.cuh holds the
// per-row work and the destination check).
#include "append_device.cuh"

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
  const bool mine = unit < parts * c.num_kv_heads;  // this warp writes a (part, head) of the row
  const int part = unit / c.num_kv_heads, h = unit - part * c.num_kv_heads;
  const bool regs = append_row_fits(c);
  AppendRow r;
  if (mine && regs) r = append_row_load<kFp8>(c, k_new, v_new, row, part, h, lane);  // overlaps the lookups
  const int b = row_req ? row_req[row] : row;
  if (b < 0 || b >= batch) return;
  const int pos = positions[row];
  int page = -1;
  const uint32_t bad = append_target(c, b, pos, block_table, block_tags, max_pages, flags, &page);
  if (bad) {
    if (unit == 0 && lane == 0) atomicOr(&status[b], bad);
    return;
  }
  if (!mine) return;
  if (regs)
    append_row_store<kFp8>(c, r, part, h, page, pos, lane);
  else
    append_row_wide<kFp8>(c, k_new, v_new, row, part, h, page, pos, lane);
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
