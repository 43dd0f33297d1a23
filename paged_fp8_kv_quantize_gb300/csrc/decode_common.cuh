// decode_common.cuh -- pieces shared by the decode kernels: the split plan
// (flash-decoding work list) and the log-sum-exp merge of split partials.
// Included by each decode translation unit; everything here has internal
// linkage.
#pragma once

#include <cuda_fp16.h>
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
  const int part = unit / H, h = unit - part * H, lane = threadIdx.x & 31;
  const bool fp8 = a.cache.dtype == PFKV_DTYPE_FP8_E4M3;
  const bool regs = append_row_fits(a.cache);
  AppendRow r;
  if (regs)  // the row and its scale load while the destination is looked up
    r = fp8 ? append_row_load<true>(a.cache, a.k_new, a.v_new, b, part, h, lane)
            : append_row_load<false>(a.cache, a.k_new, a.v_new, b, part, h, lane);
  const int pos = a.seq_lens[b] - 1;
  int page = -1;
  if (append_target(a.cache, b, pos, a.block_table, a.block_tags, a.MP, a.flags, &page)) return;
  if (regs) {
    if (fp8) append_row_store<true>(a.cache, r, part, h, page, pos, lane);
    else append_row_store<false>(a.cache, r, part, h, page, pos, lane);
  } else {
    if (fp8) append_row_wide<true>(a.cache, a.k_new, a.v_new, b, part, h, page, pos, lane);
    else append_row_wide<false>(a.cache, a.k_new, a.v_new, b, part, h, page, pos, lane);
  }
}

// Append blocks of the plan grid (decode step only).
__host__ __device__ inline int plan_append_blocks(const DecodeArgs &a) {
  if (!a.append) return 0;
  const long long warps = (long long)a.B * (a.cache.kv_shared ? 1 : 2) * a.cache.num_kv_heads;
  return (int)((warps + 31) / 32);
}

// Number of plan-grid blocks: the planning block, the append blocks, and
// (latent stream) one query-term block per request.
__host__ __device__ inline int plan_blocks(const DecodeArgs &a) { return 1 + plan_append_blocks(a) + (a.qprep ? a.B : 0); }

// Query terms of request b for the latent-stream kernel.  Head h's bf16 row
// q (576 values) is scaled by 2^-e_h, e_h = the exponent that puts max|q| in
// [128, 256), and written as T1 = e4m3(q 2^-e_h), T2 = e4m3(q 2^-e_h - T1):
// T1 + T2 equals the scaled row exactly for every element of magnitude at
// least 2^-2 (a bf16 significand has 8 bits, each term carries 4), the
// rest to within 2^-10.  The terms form one 128-row operand: row
// R = 32 (h / 16) + 16 t + h % 16 holds term t of head h.  Columns 0-511 of
// row R are stored as 512 plain bytes at R * 512 (loaded into tensor memory
// by the kernel), columns 512-575 as the 64-byte-swizzled shared-memory
// image at 65536: 16-byte chunk j of row R at 65536 + R * 64 +
// 16 (j ^ ((R >> 1) & 3)).  qfac[h] = softmax scale * log2(e) * 2^e_h.
__device__ __forceinline__ void plan_qprep(const DecodeArgs &a, int b) {
  __shared__ float s_qinv[64];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint16_t *q = static_cast<const uint16_t *>(a.q) + (size_t)b * 64 * 576;
  for (int h = warp; h < 64; h += (int)(blockDim.x >> 5)) {
    float m = 0.f;
    for (int k = lane; k < 576; k += 32) m = fmaxf(m, fabsf(__uint_as_float((uint32_t)q[h * 576 + k] << 16)));
    for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane == 0) {
      int e = 8;
      if (m > 0.f) frexpf(m, &e);  // m = f 2^e, f in [0.5, 1)
      s_qinv[h] = ldexpf(1.f, 8 - e);
      a.qfac[(size_t)b * 64 + h] = a.sm_scale_log2 * ldexpf(1.f, e - 8);
    }
  }
  __syncthreads();
  uint8_t *dst = a.qterms + (size_t)b * kLatentQTermBytes;
  for (int u = tid; u < 64 * 36; u += (int)blockDim.x) {
    const int h = u / 36, r = u % 36;
    const int k0 = 16 * r;  // 16 columns starting here (r < 36 covers all 576)
    const int R1 = 32 * (h >> 4) + (h & 15), R2 = R1 + 16;  // rows of T1 and T2 of head h
    size_t off1, off2;
    if (r < 32) {
      off1 = (size_t)R1 * 512 + 16 * r;
      off2 = (size_t)R2 * 512 + 16 * r;
    } else {
      const int j = r - 32;
      off1 = (size_t)65536 + R1 * 64 + 16 * (j ^ ((R1 >> 1) & 3));
      off2 = (size_t)65536 + R2 * 64 + 16 * (j ^ ((R2 >> 1) & 3));
    }
    uint32_t t1[4], t2[4];
    {
      const uint4 *src = reinterpret_cast<const uint4 *>(q + h * 576 + k0);
      const uint4 v0 = src[0], v1 = src[1];
      const uint32_t wv[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
      const float inv = s_qinv[h];
#pragma unroll
      for (int i = 0; i < 8; i += 2) {
        const float x0 = __uint_as_float(wv[i] << 16) * inv, x1 = __uint_as_float(wv[i] & 0xffff0000u) * inv;
        const float x2 = __uint_as_float(wv[i + 1] << 16) * inv, x3 = __uint_as_float(wv[i + 1] & 0xffff0000u) * inv;
        const uint32_t a01 = f32x2_to_e4m3x2(x0, x1), a23 = f32x2_to_e4m3x2(x2, x3);
        const uint32_t h01 = e4m3x2_to_f16x2(a01), h23 = e4m3x2_to_f16x2(a23);
        const float2 f01 = __half22float2(*reinterpret_cast<const __half2 *>(&h01));
        const float2 f23 = __half22float2(*reinterpret_cast<const __half2 *>(&h23));
        t1[i / 2] = a01 | (a23 << 16);
        t2[i / 2] = f32x2_to_e4m3x2(x0 - f01.x, x1 - f01.y) | (f32x2_to_e4m3x2(x2 - f23.x, x3 - f23.y) << 16);
      }
    }
    *reinterpret_cast<uint4 *>(dst + off1) = make_uint4(t1[0], t1[1], t1[2], t1[3]);
    *reinterpret_cast<uint4 *>(dst + off2) = make_uint4(t2[0], t2[1], t2[2], t2[3]);
  }
}

// Exclusive prefix over the block (1024 threads) of one int64 per thread;
// returns this thread's prefix, the block total in *total.  s_w: 33 entries.
__device__ __forceinline__ long long block_excl_scan(long long v, long long *s_w, long long *total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  long long x = v;
  for (int o = 1; o < 32; o <<= 1) {
    const long long y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_w[wid] = x;
  __syncthreads();
  if (wid == 0) {
    long long w = lane < (int)(blockDim.x >> 5) ? s_w[lane] : 0;
    for (int o = 1; o < 32; o <<= 1) {
      const long long y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    s_w[lane] = w;  // inclusive prefix of warp totals
  }
  __syncthreads();
  const long long r = (wid ? s_w[wid - 1] : 0) + x - v;
  *total = s_w[(blockDim.x >> 5) - 1];
  __syncthreads();
  return r;
}

// Balanced plan: the requests' pages, concatenated in request order (T in
// all), are cut into R ranges [floor(kT/R), floor((k+1)T/R)), one per CTA;
// an item is the part of one request inside one range.  Every CTA gets the
// same number of pages to within one, and at most R + B - 1 partial results
// are written.  R <= ranges, R <= T, and R is small enough that no request
// is cut into more than max_splits pieces (a request of p pages meets at
// most ceil(p R / T) + 1 ranges).  Returns false, having written nothing
// but status, when those caps leave fewer than 3/4 of `ranges`.
__device__ bool plan_balanced(const DecodeArgs &a, int ranges) {
  __shared__ long long s_w[33];
  __shared__ long long s_tot, s_max, s_pcarry, s_icarry;
  // one pass of up to 1024 requests, handed from the thread that sized a
  // request to the warp that writes its chunks (one chunk per lane)
  __shared__ long long s_off[1024];
  __shared__ int s_np[1024], s_kf[1024], s_n[1024], s_first[1024];
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int S = a.S;
  const long long max_len = (long long)a.MP * S;
  long long tot = 0, mx = 0;
  for (int b = tid; b < a.B; b += blockDim.x) {
    const int L = a.seq_lens[b];
    const bool bad = L < 1 || (long long)L > max_len;
    a.status[b] = bad ? PFKV_ST_BAD_LEN : 0u;
    const long long p = bad ? 0 : (L + S - 1) / S;
    tot += p;
    mx = p > mx ? p : mx;
  }
  for (int o = 16; o; o >>= 1) {
    tot += __shfl_xor_sync(0xffffffffu, tot, o);
    const long long y = __shfl_xor_sync(0xffffffffu, mx, o);
    mx = y > mx ? y : mx;
  }
  if (tid == 0) { s_tot = 0; s_max = 0; s_pcarry = 0; s_icarry = 0; }
  __syncthreads();
  if ((tid & 31) == 0) {
    atomicAdd(reinterpret_cast<unsigned long long *>(&s_tot), (unsigned long long)tot);
    atomicMax(reinterpret_cast<unsigned long long *>(&s_max), (unsigned long long)mx);
  }
  __syncthreads();
  const long long T = s_tot, pmax = s_max;
  long long R = ranges;
  if (R > T) R = T;
  if (pmax > 0) {
    const long long cap = (long long)(a.max_splits - 2) * T / pmax;
    if (R > cap) R = cap;
  }
  if (R > kMaxRanges) R = kMaxRanges;
  if (R < 1) R = 1;
  if (T > 0 && 4 * R < 3 * (long long)ranges) return false;
  if (tid == 0 && T == 0) a.cta_first[0] = 0;
  for (int base = 0; base < a.B; base += blockDim.x) {
    const int b = base + tid;
    long long pages = 0;
    int L = 0;
    if (b < a.B) {
      L = a.seq_lens[b];
      pages = (L < 1 || (long long)L > max_len) ? 0 : (L + S - 1) / S;
    }
    long long ptot;
    const long long off = s_pcarry + block_excl_scan(pages, s_w, &ptot);
    long long kf = 0, kl = -1;
    if (pages > 0) {
      kf = ((off + 1) * R - 1) / T;          // range holding the first page
      kl = ((off + pages) * R - 1) / T;      // range holding the last page
    }
    const long long n = pages > 0 ? kl - kf + 1 : 0;
    long long itot;
    const long long first = s_icarry + block_excl_scan(n, s_w, &itot);
    if (b < a.B) {
      a.split_first[b] = (int)first;
      a.split_count[b] = (int)n;
    }
    s_off[tid] = off;
    s_np[tid] = (int)pages;
    s_kf[tid] = (int)kf;
    s_n[tid] = b < a.B ? (int)n : 0;
    s_first[tid] = (int)first;
    __syncthreads();
    // chunk descriptors: warp per request, lane per chunk
    const int in_pass = min((int)blockDim.x, a.B - base);
    for (int i = wid; i < in_pass; i += (int)(blockDim.x >> 5)) {
      const int bi = base + i, ni = s_n[i], fi = s_first[i];
      const long long oi = s_off[i], pi = s_np[i];
      if (ni == 0) {  // bad length: no item writes this request's rows
        for (size_t k = lane; k < (size_t)a.Hq * a.Dv; k += 32) a.out[(size_t)bi * a.Hq * a.Dv + k] = 0.f;
        continue;
      }
      const int Li = a.seq_lens[bi];
      for (int j = lane; j < ni; j += 32) {
        const long long k = s_kf[i] + j;
        const long long r0 = k * T / R, r1 = (k + 1) * T / R;
        const long long p0 = (r0 > oi ? r0 : oi) - oi, p1 = (r1 < oi + pi ? r1 : oi + pi) - oi;
        a.chunk_info[2 * (fi + j)] = make_int4(bi, (int)p0, (int)p1, Li);
        a.chunk_info[2 * (fi + j) + 1] = make_int4(ni, j, (int)k, 0);
        if (j > 0 || oi == r0) a.cta_first[k] = fi + j;  // first item of range k
      }
    }
    __syncthreads();
    if (tid == 0) {
      s_pcarry += ptot;
      s_icarry += itot;
    }
    __syncthreads();
  }
  if (tid == 0) {
    a.cta_first[R] = (int)s_icarry;
    a.hdr->n_chunks = (int)s_icarry;
    a.hdr->n_items = (int)s_icarry * a.Hkv;
    a.hdr->work = 0u;
    a.hdr->err = 0u;
    a.hdr->chunk_pages = (int)R;
    a.hdr->n_ranges = (int)R;
  }
  return true;
}

__global__ void __launch_bounds__(1024) plan_kernel(DecodeArgs a, int target_items, int min_chunk_pages) {
  // Launched as a programmatic dependent: the stream's earlier work is
  // complete from here.  Only then may the split kernel launch (it waits for
  // this grid's results before reading them): its CTAs must not take SMs
  // while the previous call's merge still runs.
  pdl_wait();
  pdl_launch_dependents();
  if (blockIdx.x > 0) {
    const int nab = plan_append_blocks(a);
    if ((int)blockIdx.x <= nab) plan_append(a);
    else plan_qprep(a, (int)blockIdx.x - 1 - nab);
    return;
  }
  if (a.balanced > 0 && plan_balanced(a, a.balanced)) return;
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
    a.hdr->n_ranges = 0;
  }
}

// The plan grid, launched as a programmatic dependent of the stream's
// previous kernel: its launch overlaps that kernel's tail, and it waits for
// it (griddepcontrol.wait) before touching memory.
inline cudaError_t launch_plan(const DecodeArgs &a, cudaStream_t s, int target_items, int min_chunk_pages) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(plan_blocks(a));
  cfg.blockDim = dim3(1024);
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, plan_kernel, a, target_items, min_chunk_pages);
}

// ---------------------------------------------------------------- merge

// Merge launch shape: a block takes kW float4 columns of one (request, KV
// head)'s group rows (kG heads x kD values) and spreads the splits over
// 256 / kW thread groups; gridDim.y = kBlocks.
template <int kD, int kG>
struct MergeShape {
  static constexpr int kCols = kG * kD / 4;               // float4 columns of the group
  // float4 columns per block: 64, so that the splits of a column spread
  // over 4 thread groups; very wide groups (the latent stream's 16 x 512)
  // take 256 per block, which keeps the block count down
  static constexpr int kW = kCols < 64 ? kCols : (kCols >= 1024 ? 256 : 64);
  static constexpr int kGroups = 256 / kW;                // split groups per column
  static constexpr int kBlocks = kCols / kW;
  static constexpr int kNH = kW * 4 / kD > 0 ? kW * 4 / kD : 1;  // heads a block touches
  static_assert(kCols % kW == 0 && 256 % kW == 0, "merge columns");
};

template <int kD, int kG>
constexpr int merge_col_blocks() { return MergeShape<kD, kG>::kBlocks; }

template <int kD, int kG>
__global__ void __launch_bounds__(256) merge_kernel(const DecodeArgs a) {
  using M = MergeShape<kD, kG>;
  __shared__ float s_w[256 * M::kNH];  // per (split, head of this block): m, then the split's weight (splits <= 256)
  __shared__ float s_l[256 * M::kNH];
  __shared__ float s_M[M::kNH], s_W[M::kNH];
  __shared__ float4 s_acc[256];
  __shared__ unsigned s_or[8];  // status bits per warp
  // Latent stream: the next call's plan grid (one CTA that waits for this
  // grid) may launch at once.  Grouped-query path: the next call's split
  // grid launches only when this grid has finished.  Measured on the ragged
  // batch of 64: letting it launch at this grid's start made the back-to-back
  // call 165 us instead of 120 us, and at the end of this grid's wait 148 us
  // (146 us with both kernels asking for the largest shared-memory carveout).
  if (!a.self_plan) pdl_launch_dependents();
  pdl_wait();  // partials and status of the split kernel are visible from here on
  const int b = blockIdx.x / a.Hkv, g = blockIdx.x - b * a.Hkv;
  const int t = threadIdx.x;
  float *out_bg = a.out + ((size_t)b * a.Hq + g * kG) * kD;
  const int col_lo = (int)blockIdx.y * M::kW;
  const int h_lo = col_lo * 4 / kD;  // first head of this block's columns
  int nb, c0;
  // each split's (m, l) for the heads of this block's columns
  auto load_ml = [&]() {
    for (int i = t; i < nb * M::kNH; i += 256) {
      const float2 ml = __ldcg(&a.part_ml[(size_t)(c0 + i / M::kNH) * a.Hq + g * kG + h_lo + i % M::kNH]);
      s_w[i] = ml.x;
      s_l[i] = ml.y;
    }
  };
  if (a.self_plan) {
    // Grouped-query path: this kernel writes status[b].  The block of
    // (request, head 0, first columns) gathers the bits its pieces found
    // and whether any split CTA gave up; every block zeroes its columns of
    // a faulted request.  The pieces' (m, l) are loaded beside their status
    // words.
    const bool lead = g == 0 && blockIdx.y == 0;
    const int L = a.seq_lens[b];
    if (L < 1 || (long long)L > (long long)a.MP * a.S) {
      for (int i = 4 * col_lo + t; i < 4 * (col_lo + M::kW); i += 256) out_bg[i] = 0.f;
      if (lead && t == 0) a.status[b] = PFKV_ST_BAD_LEN;
      return;
    }
    nb = a.split_count[b];
    c0 = a.split_first[b];
    // written by this call's split kernel unless one of its CTAs gave up
    // first; checked so that no read leaves the workspace
    const bool sane = nb >= 1 && nb <= a.max_splits && c0 >= 0 && c0 <= a.B * a.max_splits - nb;
    uint32_t st = 0u;
    if (sane) {
      for (int i = t; i < nb; i += 256) st |= __ldcg(&a.part_st[c0 + i]);
      if (nb > 1) load_ml();
    }
    int any = 0;
    if (lead)
      for (int i = t; i < a.n_ctas; i += 256) any |= __ldcg(&a.cta_abort[i]);
    st = __reduce_or_sync(0xffffffffu, st);
    if ((t & 31) == 0) s_or[t >> 5] = st;
    const bool gave_up = __syncthreads_or(any) != 0;
    st = 0u;
#pragma unroll
    for (int w = 0; w < 8; ++w) st |= s_or[w];
    if (lead && t == 0) a.status[b] = st | (gave_up || !sane ? (uint32_t)PFKV_ST_TIMEOUT : 0u);
    if (!sane || nb == 1) return;  // a one-piece request's rows come from the split kernel
    if (st) {
      for (int i = 4 * col_lo + t; i < 4 * (col_lo + M::kW); i += 256) out_bg[i] = 0.f;
      return;
    }
  } else {
    nb = a.split_count[b];
    if (nb <= 1) return;  // finished by the split kernel (or zeroed by the plan kernel)
    c0 = a.split_first[b];
    if (__ldcg(&a.status[b]) != 0u) {
      for (int i = 4 * col_lo + t; i < 4 * (col_lo + M::kW); i += 256) out_bg[i] = 0.f;
      return;
    }
    load_ml();
  }
  __syncthreads();
  const int warp = t >> 5, lane = t & 31;
  if (warp < M::kNH) {
    const int hh = warp;
    float Mx = -INFINITY;
    for (int c = lane; c < nb; c += 32) Mx = fmaxf(Mx, s_w[c * M::kNH + hh]);
    for (int o = 16; o; o >>= 1) Mx = fmaxf(Mx, __shfl_xor_sync(0xffffffffu, Mx, o));
    float W = 0.f;
    for (int c = lane; c < nb; c += 32) W += s_l[c * M::kNH + hh] * fast_exp2(s_w[c * M::kNH + hh] - Mx);
    for (int o = 16; o; o >>= 1) W += __shfl_xor_sync(0xffffffffu, W, o);
    if (lane == 0) {
      s_M[hh] = Mx;
      s_W[hh] = W;
    }
  }
  __syncthreads();
  for (int i = t; i < nb * M::kNH; i += 256) s_w[i] = fast_exp2(s_w[i] - s_M[i % M::kNH]);
  __syncthreads();
  // thread = (float4 column, group of splits)
  const size_t cstride = (size_t)a.Hq * kD / 4;
  const int col = col_lo + t % M::kW, grp = t / M::kW;
  const int jh = col * 4 / kD - h_lo;
  const float4 *po = reinterpret_cast<const float4 *>(a.part_o + ((size_t)c0 * a.Hq + g * kG) * kD) + col;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
  for (int c = grp; c < nb; c += M::kGroups) {
    const float w = s_w[c * M::kNH + jh];
    const float4 v = __ldcg(po + (size_t)c * cstride);
    acc.x += w * v.x; acc.y += w * v.y; acc.z += w * v.z; acc.w += w * v.w;
  }
  s_acc[t] = acc;
  __syncthreads();
  if (t < M::kW) {
    for (int k = 1; k < M::kGroups; ++k) {
      const float4 v = s_acc[t + k * M::kW];
      acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
    }
    const float inv = 1.f / s_W[jh];
    reinterpret_cast<float4 *>(out_bg)[col] = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
  }
}

}  // namespace
}  // namespace pfkv
