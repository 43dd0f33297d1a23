// merge.cuh -- the log-sum-exp merge of split partials, shared by the decode
// paths (the second kernel of a grouped-query call, the third of a latent
// one).  Included by each decode translation unit after decode_common.cuh;
// everything here has internal linkage.
#pragma once

#include "decode_common.cuh"

namespace pfkv {
namespace {

// ---------------------------------------------------------------- merge

// Merge launch shape: a block takes kW float4 columns of one (request, KV
// head)'s group rows (kG heads x kD values) and spreads the splits over
// 256 / kW thread groups; gridDim.y = kBlocks.
template <int kD, int kG, int kWide = 1>
struct MergeShape {
  static constexpr int kCols = kG * kD / 4;               // float4 columns of the group
  // float4 columns per block: 64, so that the splits of a column spread
  // over 4 thread groups; very wide groups (the latent stream's 16 x 512)
  // take 256 per block, which keeps the block count down.  The narrow shape
  // (kWide = 0, for grids that would leave most SMs idle: a few requests
  // with many pieces each) takes 16 columns and spreads a column's splits
  // over 16 thread groups, so that each thread reads a few pieces at once
  // and the block count grows fourfold.
  static constexpr int kW = kWide ? (kCols < 64 ? kCols : (kCols >= 1024 ? 256 : 64)) : (kCols < 16 ? kCols : 16);
  static constexpr int kGroups = 256 / kW;                // split groups per column
  static constexpr int kBlocks = kCols / kW;
  static constexpr int kNH = kW * 4 / kD > 0 ? kW * 4 / kD : 1;  // heads a block touches
  static_assert(kCols % kW == 0 && 256 % kW == 0, "merge columns");
};

template <int kD, int kG, int kWide = 1>
constexpr int merge_col_blocks() { return MergeShape<kD, kG, kWide>::kBlocks; }

template <int kD, int kG, int kWide = 1>
__global__ void __launch_bounds__(256) merge_kernel(const DecodeArgs a) {
  using M = MergeShape<kD, kG, kWide>;
  __shared__ float s_w[256 * M::kNH];  // per (split, head of this block): m, then the split's weight (splits <= 256)
  __shared__ float s_l[256 * M::kNH];
  __shared__ float s_M[M::kNH], s_W[M::kNH];
  __shared__ float4 s_acc[256];
  __shared__ unsigned s_or[8];  // status bits per warp
  // The next call's split grid launches only when this grid has finished.
  // Measured on the ragged batch of 64 (grouped-query path): letting it
  // launch at this grid's start made the back-to-back call 165 us instead of
  // 120 us, and at the end of this grid's wait 148 us (146 us with both
  // kernels asking for the largest shared-memory carveout).
  pdl_wait();  // partials and status of the split kernel are visible from here on
  const int b = blockIdx.x / a.Hkv, g = blockIdx.x - b * a.Hkv;
  const HeadGroup hg = head_group(a, g);
  const int t = threadIdx.x;
  float *out_bg = a.out + ((size_t)b * a.Hq + hg.first) * kD;
  const int col_lo = (int)blockIdx.y * M::kW;
  const int h_lo = col_lo * 4 / kD;  // first head of this block's columns
  // float4 columns of this block that belong to real heads of the group
  const int col_hi = min(col_lo + M::kW, hg.count * kD / 4);
  // This kernel writes status[b].  The block of (request, head group 0, first
  // columns) gathers the bits the request's pieces found and whether any
  // split CTA gave up; every block zeroes its columns of a faulted request.
  // The pieces' (m, l) are loaded beside their status words.
  const bool lead = g == 0 && blockIdx.y == 0;
  const int L = a.seq_lens[b];
  if (L < 1 || (long long)L > (long long)a.MP * a.S) {
    for (int i = 4 * col_lo + t; i < 4 * col_hi; i += 256) out_bg[i] = 0.f;
    if (lead && t == 0) a.status[b] = PFKV_ST_BAD_LEN;
    return;
  }
  const int nb = a.split_count[b];
  const int c0 = a.split_first[b];
  // written by this call's split kernel unless one of its CTAs gave up
  // first; checked so that no read leaves the workspace
  const bool sane = nb >= 1 && nb <= a.max_splits && c0 >= 0 && c0 <= a.B * a.max_splits - nb;
  // The partial O rows this thread will weigh (thread = float4 column, group
  // of pieces), the first kPre of them loaded now beside the status words
  // and (m, l), so that their latency overlaps those loads: in the narrow
  // shape (a few requests, many pieces each, where the merge's round trips
  // are the whole of its time; long-context batch 58.7 -> 57.7 us per call).
  // The wide shape keeps its registers (the ragged batch was 0.7 us slower
  // with it).
  constexpr int kPre = kWide ? 0 : 4;
  const size_t cstride = (size_t)a.Hq * kD / 4;
  const int col = col_lo + t % M::kW, grp = t / M::kW;
  const bool real = col < col_hi;
  const float4 *po =
      reinterpret_cast<const float4 *>(a.part_o + ((size_t)(sane ? c0 : 0) * a.Hq + hg.first) * kD) + col;
  float4 pre[kPre > 0 ? kPre : 1];
#pragma unroll
  for (int k = 0; k < kPre; ++k) {
    const int c = grp + k * M::kGroups;
    pre[k] = sane && nb > 1 && real && c < nb ? __ldcg(po + (size_t)c * cstride) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  uint32_t st = 0u;
  if (sane) {  // every piece's status word, one per head group of the pieces' kernel
    for (int i = t; i < nb * a.st_groups; i += 256) st |= __ldcg(&a.part_st[(size_t)c0 * a.st_groups + i]);
    if (nb > 1)  // each piece's (m, l) for the heads of this block's columns
      for (int i = t; i < nb * M::kNH; i += 256) {
        if (h_lo + i % M::kNH >= hg.count) continue;  // a padding slot of the group
        const float2 ml = __ldcg(&a.part_ml[(size_t)(c0 + i / M::kNH) * a.Hq + hg.first + h_lo + i % M::kNH]);
        s_w[i] = ml.x;
        s_l[i] = ml.y;
      }
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
  if (!sane) return;
  // A faulted request's rows are zeroed here, one-piece requests included:
  // the split kernel writes a one-piece request's rows itself, but only head
  // group 0's walk checks tags, so the other groups' CTAs do not know of a
  // stale page.
  if (st) {
    for (int i = 4 * col_lo + t; i < 4 * col_hi; i += 256) out_bg[i] = 0.f;
    return;
  }
  if (nb == 1) return;  // a one-piece request's rows come from the split kernel
  if (col_hi <= col_lo) return;  // only padding slots in this block
  __syncthreads();
  const int warp = t >> 5, lane = t & 31;
  if (warp < M::kNH && h_lo + warp < hg.count) {
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
  const int jh = col * 4 / kD - h_lo;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int k = 0; k < kPre; ++k) {
    const int c = grp + k * M::kGroups;
    if (real && c < nb) {
      const float w = s_w[c * M::kNH + jh];
      acc.x += w * pre[k].x; acc.y += w * pre[k].y; acc.z += w * pre[k].z; acc.w += w * pre[k].w;
    }
  }
#pragma unroll 4
  for (int c = grp + kPre * M::kGroups; real && c < nb; c += M::kGroups) {
    const float w = s_w[c * M::kNH + jh];
    const float4 v = __ldcg(po + (size_t)c * cstride);
    acc.x += w * v.x; acc.y += w * v.y; acc.z += w * v.z; acc.w += w * v.w;
  }
  s_acc[t] = acc;
  __syncthreads();
  if (t < M::kW && real) {
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
