// decode_latent.cu -- decode attention over a latent-shared FP8 stream on the
// fifth-generation tensor cores: 64 query heads read one 576-wide stream per
// token (512 latent + 64 rotary values); V is the first 512 values of the
// same row; one fp32 scale per cached token; pages of 64 tokens.
//
// "Smaller, faster, safer: running Kimi and GLM at scale", section
// "Quantizing the KV cache": the cache is FP8 e4m3 and is converted as it is
// read.  With 64 heads on one stream the step is a dense contraction
// (about 240 flop per cached byte), so both products run as tcgen05 MMAs of
// kind f8f6f4 (e4m3 x e4m3 -> fp32 in tensor memory), straight from the
// codes the TMA engine landed in shared memory:
//   S^T = K . Q^T   M = 64 tokens (one page), N = 64 heads, K = 576.  The
//        bf16 query of head h is q_h = 2^e_h (T1 + T2), two e4m3 terms with
//        one power-of-two scale; T1 + T2 is exact for every element within
//        2^10 of the row's largest, so the term split adds no error that
//        matters.  Terms are prepared once per request by the plan grid.
//   O^T += V^T . P^T   M = 128 values (four chunks of the 512), N = 64
//        heads, K = 64 tokens.  V^T is the page itself read MN-major.  The
//        probabilities, with the token's scale folded in relative to a
//        running reference scale, are written as P1 + P2 + P3 (three e4m3
//        terms, about 12 significant bits) by the softmax warps.
// The softmax normaliser l is summed from the fp32 probabilities.
//
// One CTA per SM, persistent, work item = (request, split of its pages),
// all 64 heads.  Warp 0 loads pages (TMA, 128-byte swizzle, bounds and tag
// checks beside the copies) and the query terms; warp 1 owns tensor memory
// and issues the MMAs (one thread); warps 2-5 read S^T from tensor memory,
// run the online softmax (running maxima move only when they grow by more
// than 2x, and only then is O^T rescaled in tensor memory), write P^T, and
// write the item's partial or final output.  Partials are merged by the
// shared log-sum-exp merge kernel.
#include <cuda_fp16.h>

#include <mutex>

#include "decode_common.cuh"

namespace pfkv {

namespace {

constexpr int kTD = 576;                      // stream width
constexpr int kTDv = 512;                     // V = leading values
constexpr int kTS = 64;                       // tokens per page
constexpr int kTH = 64;                       // query heads
constexpr int kTBlocks = 5;                   // 128-byte column blocks of a row (the last one half used)
constexpr uint32_t kBlk = kTS * 128;          // 8192: one column block of a page or of a query term
constexpr uint32_t kPageSm = kTBlocks * kBlk;  // 40960
// Query terms: blocks 0-3 of T1, blocks 0-3 of T2, then one block whose
// rows hold the last 64 columns of T1 (bytes 0-63) and of T2 (64-127).
constexpr uint32_t kQBytes = 9 * kBlk;        // 73728
constexpr uint32_t kQTail = 8 * kBlk;
constexpr int kPT = 3;                        // e4m3 terms of the probabilities
constexpr uint32_t kPTerm = kTS * kTH;        // 4096: one P^T term of one page
constexpr uint32_t kPBuf = kPT * kPTerm;      // 12288
constexpr int kNst = 3;                       // pages in flight per CTA
constexpr int kTThreads = 192;                // producer, MMA, four softmax warps
constexpr uint32_t kTmemCols = 512;           // S^T x2 (64 columns each), O^T (4 x 64)
constexpr uint32_t kColS = 0, kColO = 128;
constexpr float kPExp = 6.75f;                // P'' = p (s_t / s_ref) 2^kPExp <= 2 * 2 * 2^6.75 < 448
constexpr float kTheta = 1.f;                 // log2 growth of a running max that triggers a rescale
constexpr uint32_t kIdQK = umma_idesc_e4m3(64, 64, 0, 0);
constexpr uint32_t kIdPV = umma_idesc_e4m3(128, 64, 1, 1);

struct TcSmem {
  uint32_t ring, q, p, scales, wg, bars, items, total;
};

__host__ __device__ constexpr TcSmem tc_smem() {
  TcSmem s{};
  s.ring = 0;                                  // kNst pages, each 5 column blocks (1024-aligned)
  s.q = s.ring + kNst * kPageSm;               // 2 query terms x 5 blocks
  s.p = s.q + kQBytes;                         // 2 buffers x kPT P^T terms
  s.scales = s.p + 2 * kPBuf;                  // kNst x 64 per-token scales
  s.wg = s.scales + kNst * kTS * 4;            // softmax-warp scratch (see below)
  s.bars = s.wg + 4 * (64 * 4 + 4 * 64 + 8);   // cq, m, alpha, beta | ex[4][64] | ex_s[4], misc
  s.items = s.bars + 8 * (2 * kNst + 12 + 3 * kNIQ);
  s.total = s.items + (sizeof(ItemDesc) + 4) * kNIQ + 16;
  return s;
}
static_assert(tc_smem().total + 1024 <= 232448, "shared memory plan exceeds one SM");

// Softmax-warp scratch, floats: cq[64] | m[64] | alpha[64] | beta[64] | ex[4][64] | ex_s[4] | pad
constexpr int kWgCq = 0, kWgM = 64, kWgAlpha = 128, kWgBeta = 192, kWgEx = 256, kWgExS = 512;

// Bounded wait that ignores the abort flag: used on the way out, so that a
// block that gave up still lets its own copies and MMAs land before it exits.
__device__ __forceinline__ void drain_wait(uint64_t *bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity))
    if (global_timer_ns() - t0 > kWaitLimitNs) return;
}

struct Bars {
  uint64_t *full, *empty, *s_full, *s_empty, *p_full, *p_empty, *q_full, *q_empty, *o_empty, *drain;
  uint64_t *item_full, *item_empty, *item_done;
};

__device__ __forceinline__ Bars bars_at(uint8_t *base) {
  uint64_t *b = reinterpret_cast<uint64_t *>(base);
  Bars r;
  r.full = b; b += kNst;
  r.empty = b; b += kNst;
  r.s_full = b; b += 2;
  r.s_empty = b; b += 2;
  r.p_full = b; b += 2;
  r.p_empty = b; b += 2;
  r.q_full = b; b += 1;
  r.q_empty = b; b += 1;
  r.o_empty = b; b += 1;
  r.drain = b; b += 1;
  r.item_full = b; b += kNIQ;
  r.item_empty = b; b += kNIQ;
  r.item_done = b;
  return r;
}

// ---------------------------------------------------------------- producer (warp 0)

__device__ __forceinline__ void tc_producer(const DecodeArgs &a, const CUtensorMap &map, uint8_t *smem,
                                            const Bars &B, ItemDesc *items, uint32_t *item_status,
                                            volatile int *abort_flag) {
  const TcSmem sp = tc_smem();
  const int lane = threadIdx.x & 31;
  const int n_items = a.hdr->n_items;
  const bool tag_check = (a.flags & PFKV_FLAG_TAG_CHECK) != 0u;
  uint32_t g = 0;  // pages issued by this CTA
  uint32_t it = 0, q_loads = 0;
  bool ok = true;
  for (;; ++it) {
    int item = 0;
    if (lane == 0) item = (int)atomicAdd(&a.hdr->work, 1u);
    item = __shfl_sync(0xffffffffu, item, 0);
    const uint32_t slot = it % kNIQ;
    bool w = true;
    if (lane == 0) w = mbar_wait(&B.item_empty[slot], ((it / kNIQ) & 1u) ^ 1u, abort_flag);
    if (!__shfl_sync(0xffffffffu, w, 0)) { ok = false; break; }
    if (item >= n_items) {
      if (lane == 0) {
        items[slot].b = -1;
        mbar_arrive(&B.item_full[slot]);
      }
      break;
    }
    const int4 info = a.chunk_info[2 * item], info2 = a.chunk_info[2 * item + 1];
    const int b = info.x, p0 = info.y, p1 = info.z;
    if (lane == 0) {
      ItemDesc d;
      d.b = b; d.cg = item; d.g = 0; d.p0 = p0; d.p1 = p1; d.L = info.w; d.ring = g; d.nb = info2.x;
      items[slot] = d;
      mbar_arrive(&B.item_full[slot]);
      // the request's query terms, once the previous item's last QK^T is done
      if (mbar_wait(B.q_empty, (it & 1u) ^ 1u, abort_flag)) {
        mbar_arrive_expect_tx(B.q_full, kQBytes);
        const uint8_t *src = a.qterms + (size_t)b * kQBytes;
        for (uint32_t o = 0; o < kQBytes; o += kBlk) bulk_load(smem + sp.q + o, src + o, kBlk, B.q_full);
        ++q_loads;
      }
    }
    const int *trow = a.block_table + (size_t)b * a.MP;
    const uint32_t *tagrow = a.block_tags + (size_t)b * a.MP;
    uint32_t st_bits = 0;
    for (int i0 = p0; i0 < p1 && ok; i0 += kNst) {
      const int i = i0 + lane;
      const bool valid = lane < kNst && i < p1;
      const int pid = valid ? __ldg(&trow[i]) : 0;
      const bool oob = valid && (pid < 0 || pid >= a.P);
      uint32_t page_tag = 0, want_tag = 0;
      if (tag_check && valid && !oob) {  // loads issued now, compared after the copies
        page_tag = __ldg(&a.page_tags[pid]);
        want_tag = __ldg(&tagrow[i]);
      }
      bool lane_ok = true;
      if (valid) {
        const uint32_t r = g + (uint32_t)lane;
        const uint32_t st = r % kNst;
        lane_ok = mbar_wait(&B.empty[st], ((r / kNst) & 1u) ^ 1u, abort_flag);
        if (lane_ok) {
          if (oob) {
            mbar_arrive(&B.full[st]);  // never fetched; the request is aborted
          } else {
            mbar_arrive_expect_tx(&B.full[st], kPageSm + kTS * 4);
            uint8_t *stage = smem + sp.ring + st * kPageSm;
#pragma unroll
            for (int c = 0; c < kTBlocks; ++c) tma_load_3d(stage + c * kBlk, &map, &B.full[st], 128 * c, 0, pid);
            bulk_load(smem + sp.scales + st * (kTS * 4), a.k_scale + (size_t)pid * kTS, kTS * 4, &B.full[st]);
          }
        }
      }
      g += (uint32_t)min(kNst, p1 - i0);
      ok = __all_sync(0xffffffffu, lane_ok);
      if (__any_sync(0xffffffffu, oob)) st_bits |= PFKV_ST_PAGE_OOB;
      if (__any_sync(0xffffffffu, page_tag != want_tag)) st_bits |= PFKV_ST_STALE_TAG;
    }
    if (lane == 0) {
      item_status[slot] = st_bits;
      if (st_bits) atomicOr(&a.status[b], st_bits);
      mbar_arrive(&B.item_done[slot]);
    }
    if (!ok) break;
  }
  // Copies still in flight land before the block may exit: the last pages
  // issued and the last query load.
  if (lane == 0) {
    for (uint32_t k = g > kNst ? g - kNst : 0; k < g; ++k) drain_wait(&B.full[k % kNst], (k / kNst) & 1u);
    if (q_loads) drain_wait(B.q_full, (q_loads - 1) & 1u);
  }
}

// ---------------------------------------------------------------- MMA issuer (warp 1, one thread)

__device__ __forceinline__ void tc_mma(const DecodeArgs &a, uint8_t *smem, const Bars &B, const ItemDesc *items,
                                       uint32_t tmem, volatile int *abort_flag) {
  const TcSmem sp = tc_smem();
  const uint32_t s_ring = smem_addr(smem + sp.ring), s_q = smem_addr(smem + sp.q), s_p = smem_addr(smem + sp.p);
  uint32_t g = 0;   // pages consumed
  uint32_t it = 0;  // items
  bool ok = true;
  // PV of page gp (j-th page of its item): O^T[c] (+)= V^T_c . (P1 + P2)^T
  auto pv = [&](uint32_t gp, bool first) -> bool {
    const uint32_t pb = gp & 1u;
    if (!mbar_wait(&B.p_full[pb], (gp >> 1) & 1u, abort_flag)) return false;
    tc_fence_after();
    const uint32_t st = gp % kNst;
#pragma unroll
    for (int c = 0; c < 4; ++c)
#pragma unroll
      for (int t = 0; t < kPT; ++t)
#pragma unroll
        for (int ks = 0; ks < 2; ++ks) {
          const uint64_t da = umma_sdesc(s_ring + st * kPageSm + c * kBlk + ks * 4096, 8192, 1024, 2);
          const uint64_t db = umma_sdesc(s_p + pb * kPBuf + t * kPTerm + ks * 512, 128, 1024, 0);
          umma_e4m3(tmem + kColO + 64 * c, da, db, kIdPV, (first && t == 0 && ks == 0) ? 0u : 1u);
        }
    umma_commit(&B.empty[st]);
    umma_commit(&B.p_empty[pb]);
    return true;
  };
  for (;; ++it) {
    const uint32_t slot = it % kNIQ;
    if (!mbar_wait(&B.item_full[slot], (it / kNIQ) & 1u, abort_flag)) break;
    const ItemDesc d = items[slot];
    mbar_arrive(&B.item_empty[slot]);
    if (d.b < 0) break;
    const uint32_t n = (uint32_t)(d.p1 - d.p0);
    if (!mbar_wait(B.q_full, it & 1u, abort_flag)) break;
    for (uint32_t j = 0; j < n && ok; ++j) {
      const uint32_t gp = g + j, st = gp % kNst, sb = gp & 1u;
      if (!mbar_wait(&B.full[st], (gp / kNst) & 1u, abort_flag) ||
          !mbar_wait(&B.s_empty[sb], ((gp >> 1) & 1u) ^ 1u, abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
      // S^T[sb] = K_page . (T1 + T2)^T over the 576 columns (18 steps of 32 per term)
      uint32_t acc = 0;
#pragma unroll
      for (int t = 0; t < 2; ++t)
#pragma unroll
        for (int c = 0; c < kTBlocks; ++c)
#pragma unroll
          for (int kk = 0; kk < (c < 4 ? 4 : 2); ++kk) {
            const uint64_t da = umma_sdesc(s_ring + st * kPageSm + c * kBlk + kk * 32, 16, 1024, 2);
            const uint32_t qb = c < 4 ? (uint32_t)(4 * t + c) * kBlk + kk * 32 : kQTail + (uint32_t)(2 * t + kk) * 32;
            const uint64_t db = umma_sdesc(s_q + qb, 16, 1024, 2);
            umma_e4m3(tmem + kColS + 64 * sb, da, db, kIdQK, acc);
            acc = 1u;
          }
      umma_commit(&B.s_full[sb]);
      if (j + 1 == n) umma_commit(B.q_empty);  // the query terms may be replaced
      if (j > 0) {
        if (j == 1 && !mbar_wait(B.o_empty, (it & 1u) ^ 1u, abort_flag)) { ok = false; break; }
        if (!pv(gp - 1, j == 1)) { ok = false; break; }
      }
    }
    if (!ok) break;
    if (n == 1 && !mbar_wait(B.o_empty, (it & 1u) ^ 1u, abort_flag)) break;
    if (!pv(g + n - 1, n == 1)) break;
    g += n;
  }
  // every MMA issued above has completed before tensor memory is released
  umma_commit(B.drain);
  drain_wait(B.drain, 0);
}


// ---------------------------------------------------------------- softmax warps (warps 2-5)

// Barrier of the four softmax warps that also ORs a flag over them.
__device__ __forceinline__ bool wg_bar_or(bool v) {
  uint32_t r;
  asm volatile(
      "{\n.reg .pred p, q;\nsetp.ne.u32 p, %1, 0;\nbar.red.or.pred q, 1, 128, p;\nselp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)v)
      : "memory");
  return r != 0u;
}

// e4m3 pair of x and the exact fp32 values the two codes stand for.
__device__ __forceinline__ uint32_t e4m3_pair(float x0, float x1, float &v0, float &v1) {
  const uint32_t c = f32x2_to_e4m3x2(x0, x1);
  const uint32_t hv = e4m3x2_to_f16x2(c);
  const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&hv));
  v0 = f.x;
  v1 = f.y;
  return c;
}

// Three e4m3 terms of four non-negative floats: t1 = e4m3(x), t2 = e4m3(x -
// t1), t3 = e4m3(x - t1 - t2) (each difference is exact in fp32).
__device__ __forceinline__ void three_terms4(float x0, float x1, float x2, float x3, uint32_t &t1, uint32_t &t2,
                                             uint32_t &t3) {
  float a0, a1, a2, a3;
  t1 = e4m3_pair(x0, x1, a0, a1) | (e4m3_pair(x2, x3, a2, a3) << 16);
  x0 -= a0; x1 -= a1; x2 -= a2; x3 -= a3;
  t2 = e4m3_pair(x0, x1, a0, a1) | (e4m3_pair(x2, x3, a2, a3) << 16);
  t3 = f32x2_to_e4m3x2(x0 - a0, x1 - a1) | (f32x2_to_e4m3x2(x2 - a2, x3 - a3) << 16);
}

__device__ __forceinline__ void tc_softmax(const DecodeArgs &a, uint8_t *smem, const Bars &B, const ItemDesc *items,
                                           const uint32_t *item_status, uint32_t tmem, volatile int *abort_flag) {
  const TcSmem sp = tc_smem();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int wq = warp - 2;          // 0..3 among the softmax warps
  const int gq = warp & 3;          // tensor-memory lane quarter this warp may access
  const int wt = threadIdx.x - 64;  // 0..127
  float *wg = reinterpret_cast<float *>(smem + sp.wg);
  float *s_cq = wg + kWgCq, *s_m = wg + kWgM, *s_alpha = wg + kWgAlpha, *s_beta = wg + kWgBeta;
  float *s_ex = wg + kWgEx, *s_exs = wg + kWgExS;
  const float *scales = reinterpret_cast<const float *>(smem + sp.scales);
  uint8_t *pbase = smem + sp.p;
  const uint32_t tq = tmem + ((uint32_t)(32 * gq) << 16);  // this warp's lanes
  // S^T row i (token i of the page) sits in lane 32 (i / 16) + i % 16: this
  // warp holds tokens 16 gq .. 16 gq + 15 in its lanes 0-15.
  const int t = 16 * gq + (lane & 15);
  const bool tok_lane = lane < 16;
  uint32_t g = 0;
  for (uint32_t it = 0;; ++it) {
    const uint32_t slot = it % kNIQ;
    bool fail = !mbar_wait(&B.item_full[slot], (it / kNIQ) & 1u, abort_flag);
    if (wg_bar_or(fail)) break;
    const ItemDesc d = items[slot];
    if (d.b < 0) break;
    const uint32_t n = (uint32_t)(d.p1 - d.p0);
    if (wt < kTH) {
      s_cq[wt] = __ldg(&a.qfac[(size_t)d.b * kTH + wt]);
      s_m[wt] = kNegInf;
    }
    float s_ref = 0.f;
    float lp[kTH];
#pragma unroll
    for (int h = 0; h < kTH; ++h) lp[h] = 0.f;
    named_bar_sync(1, 128);
    bool dead = false;
    for (uint32_t j = 0; j < n; ++j) {
      const uint32_t gp = g + j, sb = gp & 1u, st = gp % kNst;
      fail = fail || !mbar_wait(&B.s_full[sb], (gp >> 1) & 1u, abort_flag) ||
             !mbar_wait(&B.full[st], (gp / kNst) & 1u, abort_flag) ||
             !mbar_wait(&B.p_empty[sb], ((gp >> 1) & 1u) ^ 1u, abort_flag);
      float y[kTH];
      {
        tc_fence_after();
        uint32_t r[32];
        tmem_ld32(tq + kColS + 64 * sb, r);
#pragma unroll
        for (int i = 0; i < 32; ++i) y[i] = __uint_as_float(r[i]);
        tmem_ld32(tq + kColS + 64 * sb + 32, r);
#pragma unroll
        for (int i = 0; i < 32; ++i) y[32 + i] = __uint_as_float(r[i]);
        tc_fence_before();
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&B.s_empty[sb]);
      const bool valid = tok_lane && (d.p0 + (int)j) * kTS + t < d.L;
      const float s_t = valid ? scales[st * kTS + t] : 0.f;
      // z (log2 units) = S * (tau log2(e) 2^e_h) * s_t; padding and spare lanes -> -inf
#pragma unroll
      for (int h = 0; h < kTH; h += 4) {
        const float4 c4 = *reinterpret_cast<const float4 *>(&s_cq[h]);
        y[h] = valid ? y[h] * c4.x * s_t : kNegInf;
        y[h + 1] = valid ? y[h + 1] * c4.y * s_t : kNegInf;
        y[h + 2] = valid ? y[h + 2] * c4.z * s_t : kNegInf;
        y[h + 3] = valid ? y[h + 3] * c4.w * s_t : kNegInf;
      }
      // per-head maxima over the page: warp maxima, then over the four warps
      float mine0 = kNegInf, mine1 = kNegInf;
#pragma unroll
      for (int h = 0; h < kTH; ++h) {
        const float r = warp_max_f32(y[h]);
        if (lane == (h & 31)) {
          if (h < 32) mine0 = r;
          else mine1 = r;
        }
      }
      const float smx = warp_max_f32(s_t);
      s_ex[wq * kTH + lane] = mine0;
      s_ex[wq * kTH + 32 + lane] = mine1;
      if (lane == 0) s_exs[wq] = smx;
      if (wg_bar_or(fail)) {
        dead = true;
        break;
      }
      const float sm = fmaxf(fmaxf(s_exs[0], s_exs[1]), fmaxf(s_exs[2], s_exs[3]));
      const float s_old = s_ref;
      const float s_new = sm > 2.f * s_old ? sm : s_old;
      bool resc = s_new != s_old;
      if (wt < kTH) {
        const float tm = fmaxf(fmaxf(s_ex[wt], s_ex[kTH + wt]), fmaxf(s_ex[2 * kTH + wt], s_ex[3 * kTH + wt]));
        const float m_old = s_m[wt];
        const float m_new = tm > m_old + kTheta ? tm : m_old;
        const float alpha = fast_exp2(m_old - m_new);
        s_m[wt] = m_new;
        s_alpha[wt] = alpha;
        s_beta[wt] = alpha * (s_old / s_new);
        resc = resc || m_new != m_old;
      }
      s_ref = s_new;
      resc = wg_bar_or(resc) && j > 0;
      if (resc) {
        // O^T so far holds the earlier pages: every head column h scaled by beta_h
        // once the previous page's PV has landed; l by alpha_h.
        fail = fail || !mbar_wait(&B.p_empty[(gp - 1) & 1u], ((gp - 1) >> 1) & 1u, abort_flag);
        if (!fail) {
          tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < 8; ++c) {
            uint32_t r[32];
            const uint32_t ta = tq + kColO + 32 * c;
            tmem_ld32(ta, r);
            const float *bt = s_beta + 32 * (c & 1);
#pragma unroll
            for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * bt[i]);
            tmem_st32(ta, r);
          }
          tmem_wait_st();
        }
#pragma unroll
        for (int h = 0; h < kTH; ++h) lp[h] *= s_alpha[h];
      }
      // P'' = p (s_t / s_ref) 2^kPExp as three e4m3 terms; p = 2^(z - m) summed into l
      const float kt = valid ? fast_log2(s_t / s_ref) + kPExp : 0.f;
      const float rt = fast_exp2(-kt);
      // P^T, MN-major without swizzle: head chunks of 16 bytes, token rows 16 bytes apart
      uint8_t *pt = pbase + sb * kPBuf + (t & 7) * 16 + (t >> 3) * 128;
#pragma unroll
      for (int hc = 0; hc < 4; ++hc) {
        uint32_t w1[4], w2[4], w3[4];
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          const int h = 16 * hc + 4 * q4;
          const float4 m4 = *reinterpret_cast<const float4 *>(&s_m[h]);
          const float p0 = fast_exp2(y[h] - m4.x + kt), p1 = fast_exp2(y[h + 1] - m4.y + kt);
          const float p2 = fast_exp2(y[h + 2] - m4.z + kt), p3 = fast_exp2(y[h + 3] - m4.w + kt);
          lp[h] += p0 * rt;
          lp[h + 1] += p1 * rt;
          lp[h + 2] += p2 * rt;
          lp[h + 3] += p3 * rt;
          three_terms4(p0, p1, p2, p3, w1[q4], w2[q4], w3[q4]);
        }
        if (tok_lane && !fail) {
          *reinterpret_cast<uint4 *>(pt + hc * 1024) = make_uint4(w1[0], w1[1], w1[2], w1[3]);
          *reinterpret_cast<uint4 *>(pt + kPTerm + hc * 1024) = make_uint4(w2[0], w2[1], w2[2], w2[3]);
          *reinterpret_cast<uint4 *>(pt + 2 * kPTerm + hc * 1024) = make_uint4(w3[0], w3[1], w3[2], w3[3]);
        }
      }
      fence_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&B.p_full[sb]);
    }
    if (dead) break;
    // ---- the item's result: wait for its last PV and its status
    const uint32_t gl = g + n - 1;
    fail = fail || !mbar_wait(&B.p_empty[gl & 1u], (gl >> 1) & 1u, abort_flag) ||
           !mbar_wait(&B.item_done[slot], (it / kNIQ) & 1u, abort_flag);
    // l per head: over the 16 token lanes, then over the four warps
#pragma unroll
    for (int h = 0; h < kTH; ++h) {
      float v = lp[h];
      v += __shfl_xor_sync(0xffffffffu, v, 1);
      v += __shfl_xor_sync(0xffffffffu, v, 2);
      v += __shfl_xor_sync(0xffffffffu, v, 4);
      v += __shfl_xor_sync(0xffffffffu, v, 8);
      if (lane == (h & 15)) s_ex[wq * kTH + h] = v;
    }
    if (wg_bar_or(fail)) break;
    if (wt < kTH) s_alpha[wt] = s_ex[wt] + s_ex[kTH + wt] + s_ex[2 * kTH + wt] + s_ex[3 * kTH + wt];
    named_bar_sync(1, 128);
    tc_fence_after();
    const uint32_t stv = item_status[slot];
    const float oscale = s_ref * exp2f(-kPExp);  // O^T accumulates p (s_t / s_ref) 2^kPExp * code
#pragma unroll 1
    for (int c = 0; c < 8; ++c) {
      uint32_t r[32];
      tmem_ld32(tq + kColO + 32 * c, r);
      const int dd = 128 * (c >> 1) + 32 * gq + lane;  // value index of this thread's row
      const int h0 = 32 * (c & 1);
      if (d.nb == 1) {
        float *o = a.out + (size_t)d.b * kTH * kTDv + dd;
#pragma unroll
        for (int i = 0; i < 32; ++i)
          o[(size_t)(h0 + i) * kTDv] = stv ? 0.f : __uint_as_float(r[i]) * oscale / s_alpha[h0 + i];
      } else {
        float *o = a.part_o + (size_t)d.cg * kTH * kTDv + dd;
#pragma unroll
        for (int i = 0; i < 32; ++i) o[(size_t)(h0 + i) * kTDv] = __uint_as_float(r[i]) * oscale;
      }
    }
    if (d.nb != 1 && wt < kTH) a.part_ml[(size_t)d.cg * kTH + wt] = make_float2(s_m[wt], s_alpha[wt]);
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(B.o_empty);
    named_bar_sync(1, 128);  // the scratch is reused by the next item
    if (wt == 0) mbar_arrive(&B.item_empty[slot]);
    g += n;
  }
}


__global__ void __launch_bounds__(kTThreads, 1) latent_tc_kernel(const __grid_constant__ CUtensorMap map,
                                                                 const DecodeArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const TcSmem sp = tc_smem();
  const Bars B = bars_at(smem + sp.bars);
  ItemDesc *items = reinterpret_cast<ItemDesc *>(smem + sp.items);
  uint32_t *item_status = reinterpret_cast<uint32_t *>(items + kNIQ);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(item_status + kNIQ);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(item_status + kNIQ + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kNst; ++i) {
      mbar_init(&B.full[i], 1);
      mbar_init(&B.empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&B.s_full[i], 1);
      mbar_init(&B.s_empty[i], 4);
      mbar_init(&B.p_full[i], 4);
      mbar_init(&B.p_empty[i], 1);
    }
    mbar_init(B.q_full, 1);
    mbar_init(B.q_empty, 1);
    mbar_init(B.o_empty, 4);
    mbar_init(B.drain, 1);
    for (int i = 0; i < kNIQ; ++i) {
      mbar_init(&B.item_full[i], 1);
      mbar_init(&B.item_empty[i], 2);  // the MMA thread and the softmax warps
      mbar_init(&B.item_done[i], 1);
    }
    *abort_flag = 0;
    mbar_init_fence();
  }
  if (warp == 1) tmem_alloc(tmem_slot, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();
  pdl_launch_dependents();
  if (warp == 0) {
    if (lane == 0) tma_prefetch_desc(&map);
    tc_producer(a, map, smem, B, items, item_status, abort_flag);
  } else if (warp == 1) {
    if (lane == 0) tc_mma(a, smem, B, items, tmem, abort_flag);
    __syncwarp();
  } else {
    tc_softmax(a, smem, B, items, item_status, tmem, abort_flag);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  // A wait gave up somewhere in this block: every request of the call is
  // reported as timed out (its output is not valid).
  if (threadIdx.x == 0 && *abort_flag)
    for (int b = 0; b < a.B; ++b) atomicOr(&a.status[b], PFKV_ST_TIMEOUT);
}

}  // namespace

// Tensor map over the stream pool viewed as [page][slot][576 bytes]; a box
// is one 128-byte column block of a page (the fifth box reads 64 bytes past
// the row end, which the copy fills with zeros).
static int make_stream_map(CUtensorMap *map, const void *pool, int P) {
  EncodeTiledFn enc = encode_tiled_fn();
  if (!enc) return cuda_fail(cudaErrorNotSupported, "cuTensorMapEncodeTiled entry point");
  cuuint64_t dims[3] = {(cuuint64_t)kTD, (cuuint64_t)kTS, (cuuint64_t)P};
  cuuint64_t strides[2] = {(cuuint64_t)kTD, (cuuint64_t)kTD * kTS};
  cuuint32_t box[3] = {128, (cuuint32_t)kTS, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(pool), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cuda_fail(cudaErrorInvalidValue, "cuTensorMapEncodeTiled (stream)");
  return PFKV_OK;
}

int launch_latent_decode(const DecodeArgs &a0, cudaStream_t s) {
  // Work items are splits of a request, all 64 heads each.
  DecodeArgs a = a0;
  a.Hkv = 1;
  a.G = kTH;
  a.qprep = 1;
  CUtensorMap map;
  int rc = make_stream_map(&map, a.k_pool, a.P);
  if (rc) return rc;
  const uint32_t smem = tc_smem().total + 1024;
  static std::mutex mu;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  {
    std::lock_guard<std::mutex> lock(mu);
    if (dev >= 64 || !attr_set[dev]) {
      const cudaError_t e =
          cudaFuncSetAttribute(latent_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(latent kernel)");
      if (dev < 64) attr_set[dev] = true;
    }
  }
  const int grid = num_sms();
  plan_kernel<<<plan_blocks(a), 1024, 0, s>>>(a, grid * 2, 8);
  rc = cuda_ok(cudaGetLastError(), "plan kernel launch");
  if (rc) return rc;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kTThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  rc = cuda_ok(cudaLaunchKernelEx(&cfg, latent_tc_kernel, map, a), "latent kernel launch");
  if (rc) return rc;
  // merge in blocks of 16 heads
  DecodeArgs m = a;
  m.Hkv = kTH / 16;
  m.G = 16;
  cudaLaunchConfig_t mcfg = {};
  mcfg.gridDim = dim3(a.B * m.Hkv);
  mcfg.blockDim = dim3(256);
  mcfg.stream = s;
  mcfg.attrs = attr;
  mcfg.numAttrs = 1;
  return cuda_ok(cudaLaunchKernelEx(&mcfg, merge_kernel<kTDv, 16>, m), "merge kernel launch");
}

}  // namespace pfkv
