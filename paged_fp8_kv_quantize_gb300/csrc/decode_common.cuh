// decode_common.cuh -- pieces shared by the decode kernels: the split plan
// (flash-decoding work list) and the log-sum-exp merge of split partials.
// Included by each decode translation unit; everything here has internal
// linkage.
#pragma once

#include <math.h>

#include "append_device.cuh"
#include "pfkv_device.cuh"
#include "pfkv_internal.h"

namespace pfkv {
namespace {

constexpr float kNegInf = -INFINITY;
constexpr int kNIQ = 4;  // item descriptors in flight per CTA

struct ItemDesc {
  int b, cg, g, p0, p1, L;
  uint32_t ring;
  int nb;  // splits of request b
};

// ---------------------------------------------------------------- plan

constexpr int kSortMax = 2048;  // requests ordered by length when the batch is at most this

// Blocks after the first (decode step only): one warp per (request, K|V,
// head) writes the step's new token at position seq_lens[b] - 1.  The split
// kernel's grid-dependency wait covers this whole grid, so its page reads
// see the new rows.  Status is the planning block's: the attention inspects
// the same destination page under the same rules, so every refusal here is
// also a status bit there.
__device__ __forceinline__ void plan_append(const DecodeArgs &a) {
  // heads of the cache itself (a work-item view such as the latent kernel's
  // head groups may use another Hkv in the rest of DecodeArgs)
  const int H = a.cache.num_kv_heads;
  const int units = (a.cache.kv_shared ? 1 : 2) * H;
  const int gw = (int)(blockIdx.x - 1) * (int)(blockDim.x >> 5) + (int)(threadIdx.x >> 5);
  const int b = gw / units, unit = gw - b * units;
  if (b >= a.B) return;
  const int pos = a.seq_lens[b] - 1;
  int page = -1;
  if (append_target(a.cache, b, pos, a.block_table, a.block_tags, a.MP, a.flags, &page)) return;
  const int part = unit / H, h = unit - part * H;
  if (a.cache.dtype == PFKV_DTYPE_FP8_E4M3)
    append_row_warp<true>(a.cache, a.k_new, a.v_new, b, part, h, page, pos, threadIdx.x & 31);
  else
    append_row_warp<false>(a.cache, a.k_new, a.v_new, b, part, h, page, pos, threadIdx.x & 31);
}

// Number of plan-grid blocks: the planning block plus the append blocks.
inline int plan_blocks(const DecodeArgs &a) {
  if (!a.append) return 1;
  const long long warps = (long long)a.B * (a.cache.kv_shared ? 1 : 2) * a.cache.num_kv_heads;
  return 1 + (int)((warps + 31) / 32);
}

__global__ void __launch_bounds__(1024) plan_kernel(DecodeArgs a, int target_items, int min_chunk_pages) {
  pdl_launch_dependents();  // the split kernel waits for this grid's results before reading them
  if (blockIdx.x > 0) {
    plan_append(a);
    return;
  }
  __shared__ long long s_red[32];
  __shared__ int s_scan[32];
  __shared__ int s_carry;
  __shared__ int s_order[kSortMax];  // position -> request, longest first
  __shared__ int s_pages[kSortMax];  // request -> pages (0 for a bad length)
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int S = a.S;
  const long long max_len = (long long)a.MP * S;
  const bool sorted = a.B <= kSortMax;
  auto pages_of = [&](int b) -> int {
    if (sorted) return s_pages[b];
    const int L = a.seq_lens[b];
    return (L < 1 || (long long)L > max_len) ? 0 : (L + S - 1) / S;
  };
  // status (bad lengths) and total pages, which sets the split size
  long long tot = 0;
  for (int b = tid; b < a.B; b += blockDim.x) {
    const int L = a.seq_lens[b];
    const bool bad = L < 1 || (long long)L > max_len;
    a.status[b] = bad ? PFKV_ST_BAD_LEN : 0u;
    if (!bad) tot += (L + S - 1) / S;
    if (sorted) s_pages[b] = bad ? 0 : (L + S - 1) / S;
  }
  for (int o = 16; o; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
  if (lane == 0) s_red[wid] = tot;
  __syncthreads();
  if (wid == 0) {
    long long v = lane < (int)(blockDim.x >> 5) ? s_red[lane] : 0;
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0) s_red[0] = v;
  }
  __syncthreads();
  const long long total_units = s_red[0] * a.Hkv;
  long long cp = (total_units + target_items - 1) / target_items;
  if (cp < min_chunk_pages) cp = min_chunk_pages;
  if (sorted)  // rank by (pages descending, index ascending)
    for (int b = tid; b < a.B; b += blockDim.x) {
      const int pb = pages_of(b);
      int rank = 0;
      for (int o = 0; o < a.B; ++o) {
        const int po = pages_of(o);
        rank += (po > pb) || (po == pb && o < b);
      }
      s_order[rank] = b;
    }
  if (tid == 0) s_carry = 0;
  __syncthreads();
  // split counts and their exclusive prefix in processing order, 1024 per pass
  for (int base = 0; base < a.B; base += blockDim.x) {
    const int r = base + tid;
    const int b = r < a.B ? (sorted ? s_order[r] : r) : -1;
    int n = 0, ppc = 0, pages = 0;
    if (b >= 0) {
      pages = pages_of(b);
      if (pages) {
        long long nn = (pages + cp - 1) / cp;
        if (nn > a.max_splits) nn = a.max_splits;
        ppc = (int)((pages + nn - 1) / nn);
        n = (pages + ppc - 1) / ppc;
      }
    }
    int x = n;
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) s_scan[wid] = x;
    __syncthreads();
    if (wid == 0) {
      int v = lane < (int)(blockDim.x >> 5) ? s_scan[lane] : 0;
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += y;
      }
      s_scan[lane] = v;  // inclusive prefix of warp totals
    }
    __syncthreads();
    const int warp_off = wid ? s_scan[wid - 1] : 0;
    const int excl = s_carry + warp_off + x - n;
    if (b >= 0) {
      a.split_first[b] = excl;
      a.split_count[b] = n;
      const int L = a.seq_lens[b];
      for (int c = 0; c < n; ++c) {
        a.chunk_info[2 * (excl + c)] = make_int4(b, c * ppc, min((c + 1) * ppc, pages), L);
        a.chunk_info[2 * (excl + c) + 1] = make_int4(n, c, 0, 0);
      }
      if (n == 0)  // bad length: no split writes this request's rows
        for (size_t k = 0; k < (size_t)a.Hq * a.Dv; ++k) a.out[(size_t)b * a.Hq * a.Dv + k] = 0.f;
    }
    __syncthreads();
    if (tid == blockDim.x - 1) s_carry = excl + n;
    __syncthreads();
  }
  if (tid == 0) {
    a.hdr->n_chunks = s_carry;
    a.hdr->n_items = s_carry * a.Hkv;
    a.hdr->work = 0u;
    a.hdr->err = 0u;
    a.hdr->chunk_pages = (int)cp;
  }
}

// ---------------------------------------------------------------- merge

template <int kD, int kG>
__global__ void __launch_bounds__(256) merge_kernel(const DecodeArgs a) {
  __shared__ float s_w[256 * kG];  // per (split, head): m, then the split's weight (splits <= 256)
  __shared__ float s_l[256 * kG];
  __shared__ float s_M[kG], s_W[kG];
  __shared__ float4 s_acc[256];
  pdl_wait();  // partials and status of the split kernel are visible from here on
  const int b = blockIdx.x / a.Hkv, g = blockIdx.x - b * a.Hkv;
  const int nb = a.split_count[b];
  if (nb <= 1) return;  // finished by the split kernel (or zeroed by the plan kernel)
  const int t = threadIdx.x, c0 = a.split_first[b];
  float *out_bg = a.out + ((size_t)b * a.Hq + g * kG) * kD;
  if (__ldcg(&a.status[b]) != 0u) {
    for (int i = t; i < kG * kD; i += 256) out_bg[i] = 0.f;
    return;
  }
  for (int i = t; i < nb * kG; i += 256) {
    const float2 ml = __ldcg(&a.part_ml[(size_t)(c0 + i / kG) * a.Hq + g * kG + i % kG]);
    s_w[i] = ml.x;
    s_l[i] = ml.y;
  }
  __syncthreads();
  const int warp = t >> 5, lane = t & 31;
  for (int hh = warp; hh < kG; hh += 8) {  // 8 warps cover the group's heads
    float M = -INFINITY;
    for (int c = lane; c < nb; c += 32) M = fmaxf(M, s_w[c * kG + hh]);
    for (int o = 16; o; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float W = 0.f;
    for (int c = lane; c < nb; c += 32) W += s_l[c * kG + hh] * fast_exp2(s_w[c * kG + hh] - M);
    for (int o = 16; o; o >>= 1) W += __shfl_xor_sync(0xffffffffu, W, o);
    if (lane == 0) {
      s_M[hh] = M;
      s_W[hh] = W;
    }
  }
  __syncthreads();
  for (int i = t; i < nb * kG; i += 256) s_w[i] = fast_exp2(s_w[i] - s_M[i % kG]);
  __syncthreads();
  // thread = (float4 column, group of splits); wide rows loop over columns
  constexpr int kCols = kG * kD / 4;
  constexpr int kGroups = kCols >= 256 ? 1 : 256 / kCols;
  const size_t cstride = (size_t)a.Hq * kD / 4;
  const float4 *pbase = reinterpret_cast<const float4 *>(a.part_o + ((size_t)c0 * a.Hq + g * kG) * kD);
  for (int col0 = 0; col0 < kCols; col0 += 256) {
    const int col = col0 + t % (kCols < 256 ? kCols : 256), grp = kCols < 256 ? t / kCols : 0;
    const int jh = (col * 4) / kD;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (grp < kGroups && col < kCols) {
      const float4 *po = pbase + col;
#pragma unroll 8
      for (int c = grp; c < nb; c += kGroups) {
        const float w = s_w[c * kG + jh];
        const float4 v = __ldcg(po + (size_t)c * cstride);
        acc.x += w * v.x; acc.y += w * v.y; acc.z += w * v.z; acc.w += w * v.w;
      }
    }
    if (kGroups > 1) {
      s_acc[t] = acc;
      __syncthreads();
    }
    if (t < (kCols < 256 ? kCols : 256) && col < kCols) {
      for (int k = 1; k < kGroups; ++k) {
        const float4 v = s_acc[t + k * kCols];
        acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
      }
      const float inv = 1.f / s_W[jh];
      reinterpret_cast<float4 *>(out_bg)[col] = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
    }
  }
}

}  // namespace
}  // namespace pfkv
