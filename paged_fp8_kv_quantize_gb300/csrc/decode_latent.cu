// decode_latent.cu -- decode attention over a latent-shared FP8 stream:
// 64 query heads read one 576-wide stream per token (512 latent + 64 rotary
// values); V is the first 512 values of the same row; one fp32 scale per
// cached token; pages of 64 tokens.
//
// "Smaller, faster, safer: running Kimi and GLM at scale", section
// "Quantizing the KV cache": the cache is FP8 e4m3 and is converted as it is
// read.  Here the conversion is folded into the tensor cores: both
// contractions run on FP8 (e4m3 x e4m3 -> fp32) register-operand MMA, with
// the higher-precision operand written as a sum of e4m3 terms that share one
// scale and are stacked along the contraction:
//   QK^T: a bf16 query row q/2^e = T1 + T2 + T3 (three e4m3 terms; a bf16
//         significand has 8 bits, each term carries 4, so the sum is exact
//         except far below the row's largest element), contracted against the
//         cached codes as they arrived in shared memory -- no conversion.
//   PV:   the probabilities, with the per-token scale folded in through a
//         second running maximum (log2 s_t is added to the score), are
//         written as P1 + P2 (two e4m3 terms, about 8 bits), contracted
//         against the cached codes of the first 512 values.
// The softmax normaliser l is summed from the exact fp32 probabilities.
//
// Work item = (split of a request, group of 16 heads).  A CTA has one
// producer warp (bulk copies of whole pages plus their scales into a ring,
// page ids bounds-checked and tags compared beside the copies, as in the
// grouped kernel) and four consumer warps.  Per pair of pages (128 tokens):
// warp w computes S for the 16 heads x 32 tokens of k-block w; the four
// warps agree on the running maxima through shared memory; each writes its
// block's P terms as MMA operand fragments; then warp w accumulates
// O[16 heads x 128 values] for its quarter of V over all 128 tokens.  The
// QK^T accumulator layout is, token for token, the layout of the PV operand,
// so no shuffles are needed between the two.  Partials are merged by the
// shared log-sum-exp merge kernel.
#include <mutex>

#include "decode_common.cuh"

namespace pfkv {

namespace {

constexpr int kLD = 576;                         // stream width
constexpr int kLDv = 512;                        // V = leading values
constexpr int kLS = 64;                          // tokens per page
constexpr int kLHG = 16;                         // heads per work item
constexpr int kLGroups = 4;                      // head groups of 64 heads
constexpr int kLNCW = 4;                         // consumer warps
constexpr int kQT = 3;                           // e4m3 terms of the query
constexpr int kPT = 2;                           // e4m3 terms of the probabilities
constexpr int kDSteps = kLD / 32;                // 18 contraction steps of 32
constexpr uint32_t kPageBytes = kLS * kLD;       // 36864
constexpr uint32_t kStageBytes = kPageBytes + kLS * 4;  // + per-token scales
constexpr int kLThreads = (kLNCW + 1) * 32;
constexpr float kPScaleL = 256.f;                // probabilities in [0, 1] -> [0, 256]

struct LatSmem {
  uint32_t stages_off, qfrag_off, pfrag_off, exch_off, bars_off, items_off, total;
};

__host__ __device__ inline LatSmem lat_smem(int nst) {
  LatSmem p;
  p.stages_off = 0;
  p.qfrag_off = p.stages_off + kStageBytes * nst;                  // [term][step][lane] x 16 B
  p.pfrag_off = p.qfrag_off + kQT * kDSteps * 32 * 16;             // [kblock][term][lane] x 16 B
  p.exch_off = p.pfrag_off + kLNCW * kPT * 32 * 16;                // maxima, sums, query scales
  p.bars_off = p.exch_off + 4 * (2 * kLNCW * kLHG + kLNCW * kLHG + kLHG + 16);
  p.bars_off = (p.bars_off + 15u) & ~15u;
  p.items_off = p.bars_off + 8u * (2 * nst + 3 * kNIQ) + 16u;
  p.total = p.items_off + (sizeof(ItemDesc) + 4u) * kNIQ + 128u;
  return p;
}

// Physical column of the stream for contraction step s, logical index k
// (0..31) of thread quad position tq: each thread's bytes for steps 2s',
// 2s'+1 are 16 contiguous bytes at 64 s' + 16 tq.
__device__ __forceinline__ int qk_col(int s, int tq, int half, int j) {
  return 64 * (s >> 1) + 16 * tq + 8 * (s & 1) + 4 * half + j;
}

__device__ __forceinline__ uint32_t pack4_e4m3(float a, float b, float c, float d) {
  return f32x2_to_e4m3x2(a, b) | (f32x2_to_e4m3x2(c, d) << 16);
}

// 4x4 byte transpose: out[x] = byte x of r0..r3.
__device__ __forceinline__ void transpose4x4(uint32_t r0, uint32_t r1, uint32_t r2, uint32_t r3, uint32_t (&o)[4]) {
  const uint32_t t0 = prmt(r0, r1, 0x5140u), t1 = prmt(r0, r1, 0x7362u);
  const uint32_t t2 = prmt(r2, r3, 0x5140u), t3 = prmt(r2, r3, 0x7362u);
  o[0] = prmt(t0, t2, 0x5410u);
  o[1] = prmt(t0, t2, 0x7632u);
  o[2] = prmt(t1, t3, 0x5410u);
  o[3] = prmt(t1, t3, 0x7632u);
}

__global__ void __launch_bounds__(kLThreads, 2) latent_split_kernel(const DecodeArgs a, const int nst) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  const LatSmem sp = lat_smem(nst);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + sp.bars_off);
  uint64_t *empty = full + nst;
  uint64_t *item_full = empty + nst;
  uint64_t *item_empty = item_full + kNIQ;
  uint64_t *item_done = item_empty + kNIQ;
  volatile int *abort_flag = reinterpret_cast<volatile int *>(item_done + kNIQ);
  ItemDesc *items = reinterpret_cast<ItemDesc *>(smem + sp.items_off);
  uint32_t *item_status = reinterpret_cast<uint32_t *>(items + kNIQ);
  float *ex_m = reinterpret_cast<float *>(smem + sp.exch_off);  // [warp][head] score maxima
  float *ex_mv = ex_m + kLNCW * kLHG;                            // [warp][head] value-weight maxima
  float *ex_l = ex_mv + kLNCW * kLHG;                            // [warp][head] sums
  float *sq_scale = ex_l + kLNCW * kLHG;                         // [head] query scale 2^e
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < nst; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kLNCW);
    }
    for (int i = 0; i < kNIQ; ++i) {
      mbar_init(&item_full[i], 1);
      mbar_init(&item_empty[i], 1);
      mbar_init(&item_done[i], 1);
    }
    *abort_flag = 0;
    mbar_init_fence();
  }
  __syncthreads();
  pdl_wait();
  pdl_launch_dependents();

  if (warp == kLNCW) {
    // ------------------------------------------------------------ producer
    const int n_items = a.hdr->n_items;
    const bool tag_check = (a.flags & PFKV_FLAG_TAG_CHECK) != 0u;
    const int batch_pages = min(32, nst);
    uint32_t ring = 0;
    int item = 0, item_next = 0;
    if (lane == 0) item = (int)atomicAdd(&a.hdr->work, 1u);
    item = __shfl_sync(0xffffffffu, item, 0);
    int4 info = make_int4(0, 0, 0, 0), info2 = make_int4(0, 0, 0, 0);
    if (item < n_items) {
      info = a.chunk_info[2 * (item / kLGroups)];
      info2 = a.chunk_info[2 * (item / kLGroups) + 1];
    }
    for (uint32_t iq = 0;; ++iq) {
      if (lane == 0) item_next = (int)atomicAdd(&a.hdr->work, 1u);
      const uint32_t slot = iq % kNIQ;
      bool ok = true;
      if (lane == 0) ok = mbar_wait(&item_empty[slot], ((iq / kNIQ) & 1u) ^ 1u, abort_flag);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      if (item >= n_items) {
        if (lane == 0) {
          items[slot].b = -1;
          mbar_arrive(&item_full[slot]);
        }
        break;
      }
      const int cg = item / kLGroups, g = item - cg * kLGroups;
      const int b = info.x, p0 = info.y, p1 = info.z, L = info.w;
      if (lane == 0) {
        ItemDesc d;
        d.b = b; d.cg = cg; d.g = g; d.p0 = p0; d.p1 = p1; d.L = L; d.ring = ring; d.nb = info2.x;
        items[slot] = d;
        mbar_arrive(&item_full[slot]);
      }
      item_next = __shfl_sync(0xffffffffu, item_next, 0);
      int4 info_next = make_int4(0, 0, 0, 0), info2_next = make_int4(0, 0, 0, 0);
      if (item_next < n_items) {
        info_next = a.chunk_info[2 * (item_next / kLGroups)];
        info2_next = a.chunk_info[2 * (item_next / kLGroups) + 1];
      }
      const int *trow = a.block_table + (size_t)b * a.MP;
      const uint32_t *tagrow = a.block_tags + (size_t)b * a.MP;
      uint32_t st_bits = 0;
      for (int i0 = p0; i0 < p1 && ok; i0 += batch_pages) {
        const int i = i0 + lane;
        const bool valid = lane < batch_pages && i < p1;
        const int pid = valid ? __ldg(&trow[i]) : 0;
        const bool oob = valid && (pid < 0 || pid >= a.P);
        uint32_t page_tag = 0, want_tag = 0;
        if (tag_check && valid && !oob) {
          page_tag = __ldg(&a.page_tags[pid]);
          want_tag = __ldg(&tagrow[i]);
        }
        bool lane_ok = true;
        if (valid) {
          const uint32_t r = ring + (uint32_t)lane;
          const uint32_t st = r % (uint32_t)nst;
          lane_ok = mbar_wait(&empty[st], ((r / (uint32_t)nst) & 1u) ^ 1u, abort_flag);
          if (lane_ok) {
            uint8_t *stage = smem + sp.stages_off + (size_t)st * kStageBytes;
            if (oob) {
              mbar_arrive(&full[st]);  // never fetched; the request is aborted
            } else {
              mbar_arrive_expect_tx(&full[st], kStageBytes);
              bulk_load(stage, reinterpret_cast<const uint8_t *>(a.k_pool) + (size_t)pid * kPageBytes, kPageBytes,
                        &full[st]);
              bulk_load(stage + kPageBytes, a.k_scale + (size_t)pid * kLS, kLS * 4u, &full[st]);
            }
          }
        }
        ring += (uint32_t)min(batch_pages, p1 - i0);
        ok = __all_sync(0xffffffffu, lane_ok);
        if (__any_sync(0xffffffffu, oob)) st_bits |= PFKV_ST_PAGE_OOB;
        if (__any_sync(0xffffffffu, page_tag != want_tag)) st_bits |= PFKV_ST_STALE_TAG;
      }
      if (lane == 0) {
        item_status[slot] = st_bits;
        mbar_arrive(&item_done[slot]);
      }
      if (!ok) break;
      item = item_next;
      info = info_next;
      info2 = info2_next;
    }
  } else {
    // ------------------------------------------------------------ consumers
    const int gid = lane >> 2, tq = lane & 3, t = threadIdx.x;
    constexpr int kCT = kLNCW * 32;
    const uint32_t s_base = smem_addr(smem + sp.stages_off);
    const uint32_t q_base = smem_addr(smem + sp.qfrag_off);
    const uint32_t p_base = smem_addr(smem + sp.pfrag_off);
    uint32_t *qfrag = reinterpret_cast<uint32_t *>(smem + sp.qfrag_off);
    uint32_t *pfrag = reinterpret_cast<uint32_t *>(smem + sp.pfrag_off);
    for (uint32_t iq = 0;; ++iq) {
      const uint32_t slot = iq % kNIQ;
      if (!mbar_wait(&item_full[slot], (iq / kNIQ) & 1u, abort_flag)) break;
      const ItemDesc d = items[slot];
      if (d.b < 0) break;
      const __nv_bfloat16 *qrow = reinterpret_cast<const __nv_bfloat16 *>(a.q) +
                                  ((size_t)d.b * a.Hq + d.g * kLHG) * kLD;
      // ---- query terms: per head scale 2^e with max|q| / 2^e in [128, 256)
      for (int h = warp * 4; h < warp * 4 + 4; ++h) {
        float mx = 0.f;
        for (int k = lane; k < kLD; k += 32) mx = fmaxf(mx, fabsf(__bfloat162float(qrow[h * kLD + k])));
        for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        if (lane == 0) {
          int k2 = 0;
          if (mx > 0.f) frexpf(mx, &k2);
          sq_scale[h] = mx > 0.f ? ldexpf(1.f, k2 - 8) : 1.f;
        }
      }
      named_bar_sync(1, kCT);
      // fragment word (term i, step s, lane ln, register r): 4 consecutive columns
      for (int wd = t; wd < kQT * kDSteps * 32 * 4; wd += kCT) {
        const int r = wd & 3, ln = (wd >> 2) & 31, rest = wd >> 7;
        const int s = rest % kDSteps, i = rest / kDSteps;
        const int row = (ln >> 2) + 8 * (r & 1), c0 = qk_col(s, ln & 3, r >> 1, 0);
        const float inv = 1.f / sq_scale[row];
        float v[4], term[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) v[j] = __bfloat162float(qrow[row * kLD + c0 + j]) * inv;  // exact (power of 2)
        for (int k = 0; k <= i; ++k) {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            term[j] = e4m3_to_f32(f32x2_to_e4m3x2(v[j], 0.f));
            v[j] -= term[j];  // exact: the residual of a round to nearest
          }
        }
        qfrag[wd] = pack4_e4m3(term[0], term[1], term[2], term[3]);
      }
      named_bar_sync(1, kCT);
      const float rs0 = sq_scale[gid] * a.sm_scale_log2, rs1 = sq_scale[gid + 8] * a.sm_scale_log2;

      float m[2] = {kNegInf, kNegInf}, mv[2] = {kNegInf, kNegInf}, l[2] = {0.f, 0.f};
      float o[16][4];
#pragma unroll
      for (int i = 0; i < 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
      const int n_pages = d.p1 - d.p0;
      bool alive = true;
      for (int pr = 0; 2 * pr < n_pages; ++pr) {
        const bool has2 = 2 * pr + 1 < n_pages;
        uint32_t stg[2];
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const uint32_t rp = d.ring + (uint32_t)(2 * pr + k);
          stg[k] = rp % (uint32_t)nst;
          if ((k == 0 || has2) && !mbar_wait(&full[stg[k]], (rp / (uint32_t)nst) & 1u, abort_flag)) alive = false;
        }
        if (!alive) break;
        const int tok_pair = (d.p0 + 2 * pr) * kLS;  // token index of the pair's first row
        // ---- S = Q K^T for k-block `warp` (32 tokens)
        const int kpage = warp >> 1;
        const int tok0 = tok_pair + warp * 32;
        const bool live = (kpage == 0 || has2) && tok0 < d.L;
        const uint32_t kst = s_base + stg[kpage] * kStageBytes;
        const uint32_t krow = kst + (uint32_t)((warp & 1) * 32) * kLD;
        float acc[4][4];
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
        if (live) {
#pragma unroll 1
          for (int s2 = 0; s2 < kDSteps / 2; ++s2) {
            uint4 kb[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) kb[j] = lds128(krow + (uint32_t)(8 * j + gid) * kLD + 64 * s2 + 16 * tq);
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
              const int s = 2 * s2 + h2;
#pragma unroll
              for (int i = 0; i < kQT; ++i) {
                const uint4 av = lds128(q_base + (uint32_t)(((i * kDSteps + s) * 32 + lane) * 16));
                const uint32_t af[4] = {av.x, av.y, av.z, av.w};
#pragma unroll
                for (int j = 0; j < 4; ++j) mma_e4m3(acc[j], af, h2 ? kb[j].z : kb[j].x, h2 ? kb[j].w : kb[j].y);
              }
            }
          }
        }
        // ---- scores (log2 domain); value weights carry log2 of the token scale
        const uint32_t scl = kst + kPageBytes + (uint32_t)((warp & 1) * 32) * 4;
        float z[4][4], zv[4][4];
        float mz0 = kNegInf, mz1 = kNegInf, mzv0 = kNegInf, mzv1 = kNegInf;
        float tsc[4][2], tlg[4][2];  // this thread's 8 tokens: scale and its log2
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint2 v = live ? lds64(scl + 4 * (8 * j + 2 * tq)) : make_uint2(0x3f800000u, 0x3f800000u);
          tsc[j][0] = __uint_as_float(v.x);
          tsc[j][1] = __uint_as_float(v.y);
          tlg[j][0] = fast_log2(tsc[j][0]);
          tlg[j][1] = fast_log2(tsc[j][1]);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const int tk = 8 * j + 2 * tq + (c & 1);
            const bool ok_tok = live && tok0 + tk < d.L;
            const float zz = ok_tok ? acc[j][c] * ((c < 2) ? rs0 : rs1) * tsc[j][c & 1] : kNegInf;
            z[j][c] = zz;
            zv[j][c] = ok_tok ? zz + tlg[j][c & 1] : kNegInf;
            if (c < 2) { mz0 = fmaxf(mz0, zz); mzv0 = fmaxf(mzv0, zv[j][c]); }
            else { mz1 = fmaxf(mz1, zz); mzv1 = fmaxf(mzv1, zv[j][c]); }
          }
#pragma unroll
        for (int off = 1; off < 4; off <<= 1) {
          mz0 = fmaxf(mz0, __shfl_xor_sync(0xffffffffu, mz0, off));
          mz1 = fmaxf(mz1, __shfl_xor_sync(0xffffffffu, mz1, off));
          mzv0 = fmaxf(mzv0, __shfl_xor_sync(0xffffffffu, mzv0, off));
          mzv1 = fmaxf(mzv1, __shfl_xor_sync(0xffffffffu, mzv1, off));
        }
        if (tq == 0) {
          ex_m[warp * kLHG + gid] = mz0;
          ex_m[warp * kLHG + gid + 8] = mz1;
          ex_mv[warp * kLHG + gid] = mzv0;
          ex_mv[warp * kLHG + gid + 8] = mzv1;
        }
        named_bar_sync(1, kCT);
        float M0 = m[0], M1 = m[1], MV0 = mv[0], MV1 = mv[1];
#pragma unroll
        for (int w = 0; w < kLNCW; ++w) {
          M0 = fmaxf(M0, ex_m[w * kLHG + gid]);
          M1 = fmaxf(M1, ex_m[w * kLHG + gid + 8]);
          MV0 = fmaxf(MV0, ex_mv[w * kLHG + gid]);
          MV1 = fmaxf(MV1, ex_mv[w * kLHG + gid + 8]);
        }
        const float al0 = fast_exp2(m[0] - M0), al1 = fast_exp2(m[1] - M1);
        const float av0 = fast_exp2(mv[0] - MV0), av1 = fast_exp2(mv[1] - MV1);
        m[0] = M0; m[1] = M1; mv[0] = MV0; mv[1] = MV1;
        float ls0 = 0.f, ls1 = 0.f;
        float pv[4][4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const float p = fast_exp2(z[j][c] - ((c < 2) ? M0 : M1));
            if (c < 2) ls0 += p; else ls1 += p;
            pv[j][c] = fast_exp2(zv[j][c] - ((c < 2) ? MV0 : MV1)) * kPScaleL;
          }
        l[0] = l[0] * al0 + ls0;
        l[1] = l[1] * al1 + ls1;
        if (av0 != 1.f || av1 != 1.f) {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            o[i][0] *= av0; o[i][1] *= av0; o[i][2] *= av1; o[i][3] *= av1;
          }
        }
        // ---- this k-block's P as PV operand fragments: term 1 then the residual term
        {
          uint32_t fr[kPT][4];
          // register r: row (gid | gid+8) = r & 1, k half = r >> 1 -> n-tiles 2*(r>>1), 2*(r>>1)+1
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            const int cc = (r & 1) * 2, ja = 2 * (r >> 1);
            float v4[4] = {pv[ja][cc], pv[ja][cc + 1], pv[ja + 1][cc], pv[ja + 1][cc + 1]};
#pragma unroll
            for (int i = 0; i < kPT; ++i) {
              float tm[4];
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                tm[j] = (i + 1 < kPT) ? e4m3_to_f32(f32x2_to_e4m3x2(v4[j], 0.f)) : v4[j];
                v4[j] -= tm[j];
              }
              fr[i][r] = pack4_e4m3(tm[0], tm[1], tm[2], tm[3]);
            }
          }
#pragma unroll
          for (int i = 0; i < kPT; ++i)
            *reinterpret_cast<uint4 *>(pfrag + ((warp * kPT + i) * 32 + lane) * 4) =
                make_uint4(fr[i][0], fr[i][1], fr[i][2], fr[i][3]);
        }
        named_bar_sync(1, kCT);
        // ---- O[16 heads x 128 values of quarter `warp`] += P V over the pair's k-blocks
#pragma unroll 1
        for (int kbk = 0; kbk < kLNCW; ++kbk) {
          const int vpage = kbk >> 1;
          if (!((vpage == 0 || has2) && tok_pair + kbk * 32 < d.L)) continue;
          uint32_t af[kPT][4];
#pragma unroll
          for (int i = 0; i < kPT; ++i) {
            const uint4 v = lds128(p_base + (uint32_t)(((kbk * kPT + i) * 32 + lane) * 16));
            af[i][0] = v.x; af[i][1] = v.y; af[i][2] = v.z; af[i][3] = v.w;
          }
          const uint32_t vrow = s_base + stg[vpage] * kStageBytes + (uint32_t)((kbk & 1) * 32) * kLD + warp * 128 +
                                16 * gid;
          uint32_t bq[2][16];  // [b0|b1][n-tile]
#pragma unroll
          for (int hb = 0; hb < 2; ++hb) {
            uint4 rv[4];
            const int tks[4] = {16 * hb + 2 * tq, 16 * hb + 2 * tq + 1, 16 * hb + 8 + 2 * tq, 16 * hb + 9 + 2 * tq};
#pragma unroll
            for (int x = 0; x < 4; ++x) rv[x] = lds128(vrow + (uint32_t)tks[x] * kLD);
            const uint32_t w0[4] = {rv[0].x, rv[0].y, rv[0].z, rv[0].w}, w1[4] = {rv[1].x, rv[1].y, rv[1].z, rv[1].w};
            const uint32_t w2[4] = {rv[2].x, rv[2].y, rv[2].z, rv[2].w}, w3[4] = {rv[3].x, rv[3].y, rv[3].z, rv[3].w};
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              uint32_t tr[4];
              transpose4x4(w0[u], w1[u], w2[u], w3[u], tr);
#pragma unroll
              for (int x = 0; x < 4; ++x) bq[hb][4 * u + x] = tr[x];
            }
          }
#pragma unroll
          for (int nt = 0; nt < 16; ++nt)
#pragma unroll
            for (int i = 0; i < kPT; ++i) mma_e4m3(o[nt], af[i], bq[0][nt], bq[1][nt]);
        }
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&empty[stg[0]]);
          if (has2) mbar_arrive(&empty[stg[1]]);
        }
      }
      // ---- item epilogue: total l over the warps, then this warp's quarter of O
#pragma unroll
      for (int off = 1; off < 4; off <<= 1) {
        l[0] += __shfl_xor_sync(0xffffffffu, l[0], off);
        l[1] += __shfl_xor_sync(0xffffffffu, l[1], off);
      }
      if (tq == 0) {
        ex_l[warp * kLHG + gid] = l[0];
        ex_l[warp * kLHG + gid + 8] = l[1];
      }
      if (t == 0) {
        uint32_t stv = PFKV_ST_TIMEOUT;
        if (mbar_wait(&item_done[slot], (iq / kNIQ) & 1u, abort_flag)) stv = item_status[slot];
        ex_l[kLNCW * kLHG + kLHG] = __uint_as_float(stv);  // broadcast word after sq_scale
      }
      named_bar_sync(1, kCT);
      const uint32_t item_st = __float_as_uint(ex_l[kLNCW * kLHG + kLHG]);
      float L0 = 0.f, L1 = 0.f;
#pragma unroll
      for (int w = 0; w < kLNCW; ++w) {
        L0 += ex_l[w * kLHG + gid];
        L1 += ex_l[w * kLHG + gid + 8];
      }
      // O holds 256 * sum p' v with p' relative to mv; rebase to m
      const float f0 = fast_exp2(mv[0] - m[0]) / kPScaleL, f1 = fast_exp2(mv[1] - m[1]) / kPScaleL;
      const int h0 = d.g * kLHG + gid;
      const int dbase = warp * 128 + 32 * tq;  // this thread's 32 output values (n-tile nt -> dbase + nt, +16)
      if (d.nb == 1) {
        float *o0 = a.out + ((size_t)d.b * a.Hq + h0) * kLDv + dbase;
        float *o1 = o0 + 8 * kLDv;
        // an aborted request's rows are zero, whatever the never-fetched pages held
        const float g0 = f0 / L0, g1 = f1 / L1;
        const float4 zero4 = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int e = 0; e < 2; ++e)
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            const int nt = 4 * q4;
            *reinterpret_cast<float4 *>(o0 + 16 * e + nt) =
                item_st ? zero4 : make_float4(o[nt][e] * g0, o[nt + 1][e] * g0, o[nt + 2][e] * g0, o[nt + 3][e] * g0);
            *reinterpret_cast<float4 *>(o1 + 16 * e + nt) =
                item_st ? zero4
                        : make_float4(o[nt][2 + e] * g1, o[nt + 1][2 + e] * g1, o[nt + 2][2 + e] * g1,
                                      o[nt + 3][2 + e] * g1);
          }
        if (t == 0 && item_st) atomicOr(&a.status[d.b], item_st);
      } else {
        float *o0 = a.part_o + ((size_t)d.cg * a.Hq + h0) * kLDv + dbase;
        float *o1 = o0 + 8 * kLDv;
#pragma unroll
        for (int e = 0; e < 2; ++e)
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            const int nt = 4 * q4;
            *reinterpret_cast<float4 *>(o0 + 16 * e + nt) =
                make_float4(o[nt][e] * f0, o[nt + 1][e] * f0, o[nt + 2][e] * f0, o[nt + 3][e] * f0);
            *reinterpret_cast<float4 *>(o1 + 16 * e + nt) =
                make_float4(o[nt][2 + e] * f1, o[nt + 1][2 + e] * f1, o[nt + 2][2 + e] * f1, o[nt + 3][2 + e] * f1);
          }
        if (warp == 0 && tq == 0) {
          a.part_ml[(size_t)d.cg * a.Hq + h0] = make_float2(m[0], L0);
          a.part_ml[(size_t)d.cg * a.Hq + h0 + 8] = make_float2(m[1], L1);
        }
        if (t == 0 && item_st) atomicOr(&a.status[d.b], item_st);
      }
      named_bar_sync(1, kCT);
      if (t == 0) mbar_arrive(&item_empty[slot]);
      if (!alive) break;
    }
  }
  if (lane == 0 && *abort_flag)
    for (int b = 0; b < a.B; ++b) atomicOr(&a.status[b], PFKV_ST_TIMEOUT);
}

}  // namespace

int launch_latent_decode(const DecodeArgs &a0, cudaStream_t s) {
  // head groups play the role of KV heads for the split plan and the merge
  DecodeArgs a = a0;
  a.Hkv = kLGroups;
  a.G = kLHG;
  static int nst = 2;  // one pair of pages: two CTAs share an SM and hide each other's copies
  static uint32_t smem = 0;
  static int grid = 0;
  static std::mutex mu;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!smem) {
      smem = lat_smem(nst).total;
      cudaError_t e = cudaFuncSetAttribute(latent_split_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(latent kernel)");
      int per_sm = 0;
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, latent_split_kernel, kLThreads, smem);
      if (e != cudaSuccess) return cuda_fail(e, "occupancy query (latent kernel)");
      if (per_sm < 1) return cuda_fail(cudaErrorInvalidConfiguration, "latent kernel does not fit on an SM");
      grid = num_sms() * per_sm;
    }
  }
  plan_kernel<<<plan_blocks(a), 1024, 0, s>>>(a, grid * 8, (1024 + kLS - 1) / kLS);
  int rc = cuda_ok(cudaGetLastError(), "plan kernel launch");
  if (rc) return rc;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kLThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  rc = cuda_ok(cudaLaunchKernelEx(&cfg, latent_split_kernel, a, nst), "latent kernel launch");
  if (rc) return rc;
  cudaLaunchConfig_t mcfg = {};
  mcfg.gridDim = dim3(a.B * kLGroups);
  mcfg.blockDim = dim3(256);
  mcfg.stream = s;
  mcfg.attrs = attr;
  mcfg.numAttrs = 1;
  return cuda_ok(cudaLaunchKernelEx(&mcfg, merge_kernel<kLDv, kLHG>, a), "merge kernel launch (latent)");
}

}  // namespace pfkv
