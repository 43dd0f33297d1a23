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
// and issues the MMAs (one thread); warps 2-9, two groups of four with 32
// heads each, read S^T from tensor memory (every lane holds two tokens x
// eight heads), run the online softmax (running maxima move only when they
// grow by more than 8x, and only then is the group's part of O^T rescaled
// in tensor memory), write P^T, and write the item's partial or final
// output.  Partials are merged by the shared log-sum-exp merge kernel.
#include <cuda_fp16.h>

#include <mutex>

#include "decode_common.cuh"

namespace pfkv {

namespace {

constexpr int kTD = 576;                      // stream width
constexpr int kTDv = 512;                     // V = leading values
constexpr int kTS = 64;                       // tokens per page
constexpr int kTH = 64;                       // query heads
constexpr uint32_t kBlk = kTS * 128;          // 8192: one 128-byte column block of a page
// A page in shared memory: columns 0-511 as four 128-byte blocks (128-byte
// swizzle), columns 512-575 as one 64-byte block (64-byte swizzle).
constexpr uint32_t kPageTail = 4 * kBlk;      // 32768
constexpr uint32_t kPageSm = kPageTail + kTS * 64;  // 36864
// Query terms as one 128-row operand (rows 0-63: T1 of heads 0-63, rows
// 64-127: T2): four 128-byte column blocks of 16 KB, then the 64-byte tail.
constexpr uint32_t kQBlk = 2 * kBlk;          // 16384
constexpr uint32_t kQTail = 4 * kQBlk;        // 65536
constexpr uint32_t kQBytes = kQTail + 2 * kTH * 64;  // 73728
constexpr int kPT = 3;                        // e4m3 terms of the probabilities
constexpr uint32_t kPTerm = kTS * kTH;        // 4096: one P^T term of one page
constexpr uint32_t kPBuf = kPT * kPTerm;      // 12288
constexpr int kNst = 3;                       // pages in flight per CTA
constexpr int kPrefetch = 6;                  // pages pulled into L2 ahead of their copy
constexpr int kTThreads = 320;                // producer, MMA, two groups of four softmax warps
constexpr uint32_t kTmemCols = 512;           // S^T x2 (128 columns each: T1 | T2 parts), O^T (4 x 64)
constexpr uint32_t kColS = 0, kColO = 256;
constexpr float kTheta = 3.f;                 // log2 growth of a running max that triggers a rescale
constexpr float kPExp = 4.75f;                // P'' = p (s_t / s_ref) 2^kPExp <= 2^kTheta * 2 * 2^4.75 < 448
constexpr uint32_t kIdQK = umma_idesc_e4m3(64, 128, 0, 0);
constexpr uint32_t kIdPV = umma_idesc_e4m3(128, 64, 1, 1);

struct TcSmem {
  uint32_t ring, q, p, scales, wg, bars, items, total;
};

__host__ __device__ constexpr TcSmem tc_smem() {
  TcSmem s{};
  s.ring = 0;                                  // kNst pages, each 5 column blocks (1024-aligned)
  s.q = s.ring + kNst * kPageSm;               // query terms (kQBytes)
  s.p = s.q + kQBytes;                         // 2 buffers x kPT P^T terms
  s.scales = s.p + 2 * kPBuf;                  // kNst x 64 per-token scales
  s.wg = s.scales + kNst * kTS * 4;            // softmax-warp scratch (see below)
  s.bars = s.wg + 4 * (64 * 4 + 2 * 4 * 32 + 2 * 4);  // cq, m, alpha, beta | ex[2][4][32] | ex_s[2][4]
  s.items = s.bars + 8 * (2 * kNst + 12 + 3 * kNIQ);
  s.total = s.items + (sizeof(ItemDesc) + 4) * kNIQ + 16;
  return s;
}
static_assert(tc_smem().total + 1024 <= 232448, "shared memory plan exceeds one SM");

// Softmax-warp scratch, floats: cq[64] | m[64] | alpha[64] | beta[64] | ex[group][warp][32] | ex_s[group][warp]
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

__device__ __forceinline__ void tc_producer(const DecodeArgs &a, const CUtensorMap &map, const CUtensorMap &map_tail,
                                            uint8_t *smem,
                                            const Bars &B, ItemDesc *items, uint32_t *item_status,
                                            volatile int *abort_flag) {
  const TcSmem sp = tc_smem();
  const int lane = threadIdx.x & 31;
  const int n_items = a.hdr->n_items;
  const bool tag_check = (a.flags & PFKV_FLAG_TAG_CHECK) != 0u;
  uint32_t g = 0;  // pages issued by this CTA
  uint32_t it = 0, q_loads = 0;
  bool ok = true;
  // balanced plan: this CTA's items are a fixed run; otherwise items are
  // taken from a shared counter
  int next = 0, last = 0;
  if (a.balanced > 0 && (int)blockIdx.x < a.hdr->chunk_pages) {
    next = a.cta_first[blockIdx.x];
    last = a.cta_first[blockIdx.x + 1];
  }
  for (;; ++it) {
    int item = 0;
    if (a.balanced > 0) {
      item = next < last ? next++ : n_items;
    } else {
      if (lane == 0) item = (int)atomicAdd(&a.hdr->work, 1u);
      item = __shfl_sync(0xffffffffu, item, 0);
    }
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
        static_assert(kQBytes % kBlk == 0, "query image is copied in 8 KB pieces");
        ++q_loads;
      }
    }
    const int *trow = a.block_table + (size_t)b * a.MP;
    const uint32_t *tagrow = a.block_tags + (size_t)b * a.MP;
    uint32_t st_bits = 0;
    // Table entries 32 at a time (one round trip per 32 pages, hidden behind
    // the pages in flight); pages issued one by one as ring slots free up.
    for (int i0 = p0; i0 < p1 && ok; i0 += 32) {
      const int i = i0 + lane;
      const bool valid = i < p1;
      const int pid = valid ? __ldg(&trow[i]) : 0;
      const bool oob = valid && (pid < 0 || pid >= a.P);
      uint32_t page_tag = 0, want_tag = 0;
      if (tag_check && valid && !oob) {  // loads issued now, compared after the copies
        page_tag = __ldg(&a.page_tags[pid]);
        want_tag = __ldg(&tagrow[i]);
      }
      const int cnt = min(32, p1 - i0);
      // pages kPrefetch ahead of the copies are pulled into L2, so that a copy
      // issued when a ring slot frees up finds its page there
      auto prefetch = [&](int k) {
        const int pk = __shfl_sync(0xffffffffu, pid, k);
        const bool bad = __shfl_sync(0xffffffffu, oob, k);
        if (lane == 0 && !bad) {
#pragma unroll
          for (int c = 0; c < 4; ++c) tma_prefetch_l2_3d(&map, 128 * c, 0, pk);
          tma_prefetch_l2_3d(&map_tail, 512, 0, pk);
          bulk_prefetch_l2(a.k_scale + (size_t)pk * kTS, kTS * 4);
        }
      };
      for (int k = 0; k < min(kPrefetch, cnt); ++k) prefetch(k);
      for (int k = 0; k < cnt; ++k) {
        if (k + kPrefetch < cnt) prefetch(k + kPrefetch);
        const int pk = __shfl_sync(0xffffffffu, pid, k);
        const bool ok_k = __shfl_sync(0xffffffffu, oob, k);
        bool w = true;
        if (lane == 0) {
          const uint32_t r = g + (uint32_t)k, st = r % kNst;
          w = mbar_wait(&B.empty[st], ((r / kNst) & 1u) ^ 1u, abort_flag);
          if (w) {
            if (ok_k) {
              mbar_arrive(&B.full[st]);  // never fetched; the request is aborted
            } else {
              mbar_arrive_expect_tx(&B.full[st], kPageSm + kTS * 4);
              uint8_t *stage = smem + sp.ring + st * kPageSm;
#pragma unroll
              for (int c = 0; c < 4; ++c) tma_load_3d(stage + c * kBlk, &map, &B.full[st], 128 * c, 0, pk);
              tma_load_3d(stage + kPageTail, &map_tail, &B.full[st], 512, 0, pk);
              bulk_load(smem + sp.scales + st * (kTS * 4), a.k_scale + (size_t)pk * kTS, kTS * 4, &B.full[st]);
            }
          }
        }
        if (!__shfl_sync(0xffffffffu, w, 0)) {
          ok = false;
          g += (uint32_t)k;  // pages issued so far in this batch
          break;
        }
      }
      if (ok) g += (uint32_t)cnt;
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
  uint32_t g = 0;  // pages consumed before the current item
  bool ok = true;
  for (uint32_t it = 0; ok; ++it) {
    const uint32_t slot = it % kNIQ;
    if (!mbar_wait(&B.item_full[slot], (it / kNIQ) & 1u, abort_flag)) break;
    const ItemDesc d = items[slot];
    mbar_arrive(&B.item_empty[slot]);
    if (d.b < 0) break;
    const uint32_t n = (uint32_t)(d.p1 - d.p0);
    if (!mbar_wait(B.q_full, it & 1u, abort_flag)) break;
    // Issue each MMA group as soon as its inputs are ready: QK^T of page nq
    // (page landed, its S^T buffer read by the softmax warps) or PV of page
    // np (P^T written; for the item's first page, O^T read out).  A PV never
    // waits behind the next page's copy.
    uint32_t nq = 0, np = 0;
    bool o_free = false;
    uint64_t t_last = 0;  // start of the current stretch without progress
    while (np < n) {
      bool did = false;
      if (nq < n) {
        const uint32_t gp = g + nq, st = gp % kNst, sb = gp & 1u;
        if (mbar_test(&B.full[st], (gp / kNst) & 1u) && mbar_test(&B.s_empty[sb], ((gp >> 1) & 1u) ^ 1u)) {
          tc_fence_after();
          // S^T[sb] = K_page . [T1; T2]^T: 64 tokens x 128 columns (heads of T1,
          // then of T2) over the 576 columns, 18 steps of 32
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t da = umma_sdesc(s_ring + st * kPageSm + c * kBlk + kk * 32, 16, 1024, 2);
              const uint64_t db = umma_sdesc(s_q + c * kQBlk + kk * 32, 16, 1024, 2);
              umma_e4m3(tmem + kColS + 128 * sb, da, db, kIdQK, (c | kk) ? 1u : 0u);
            }
#pragma unroll
          for (int kk = 0; kk < 2; ++kk) {
            const uint64_t da = umma_sdesc(s_ring + st * kPageSm + kPageTail + kk * 32, 16, 512, 4);
            const uint64_t db = umma_sdesc(s_q + kQTail + kk * 32, 16, 512, 4);
            umma_e4m3(tmem + kColS + 128 * sb, da, db, kIdQK, 1u);
          }
          umma_commit(&B.s_full[sb]);
          if (nq + 1 == n) umma_commit(B.q_empty);  // the query terms may be replaced
          ++nq;
          did = true;
        }
      }
      if (np < nq) {
        const uint32_t gp = g + np, st = gp % kNst, pb = gp & 1u;
        if (np == 0 && !o_free) o_free = mbar_test(B.o_empty, (it & 1u) ^ 1u);
        if ((np > 0 || o_free) && mbar_test(&B.p_full[pb], (gp >> 1) & 1u)) {
          tc_fence_after();
          // O^T[c] (+)= V^T_c . (P1 + P2 + P3)^T
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int t = 0; t < kPT; ++t)
#pragma unroll
              for (int ks = 0; ks < 2; ++ks) {
                const uint64_t da = umma_sdesc(s_ring + st * kPageSm + c * kBlk + ks * 4096, 8192, 1024, 2);
                const uint64_t db = umma_sdesc(s_p + pb * kPBuf + t * kPTerm + ks * 512, 128, 1024, 0);
                umma_e4m3(tmem + kColO + 64 * c, da, db, kIdPV, (np == 0 && t == 0 && ks == 0) ? 0u : 1u);
              }
          umma_commit(&B.empty[st]);
          umma_commit(&B.p_empty[pb]);
          ++np;
          did = true;
        }
      }
      if (did) {
        t_last = 0;
      } else {
        const uint64_t now = global_timer_ns();
        if (t_last == 0) t_last = now;
        if (*abort_flag || now - t_last > kWaitLimitNs) {
          *abort_flag = 1;
          ok = false;
          break;
        }
      }
    }
    g += n;
  }
  // every MMA issued above has completed before tensor memory is released
  umma_commit(B.drain);
  drain_wait(B.drain, 0);
}

// ---------------------------------------------------------------- softmax warps (warps 2-9)

// Barrier of one softmax warpgroup (id 1 + wg, 128 threads) that also ORs a
// flag over it.
__device__ __forceinline__ bool wg_bar_or(int id, bool v) {
  uint32_t r;
  asm volatile(
      "{\n.reg .pred p, q;\nsetp.ne.u32 p, %1, 0;\nbar.red.or.pred q, %2, 128, p;\nselp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)v), "r"(id)
      : "memory");
  return r != 0u;
}

// Whole warp: 16 lanes from taddr's lane, 32 columns, in the register-MMA
// accumulator layout: thread t gets rows t/4 and t/4 + 8; for column group k
// (8 columns) r[4k..4k+3] = (row t/4, col 8k + 2(t%4)), (.., +1),
// (row t/4 + 8, 8k + 2(t%4)), (.., +1).
__device__ __forceinline__ void tmem_ld16x256_x4(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.16x256b.x4.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ uint32_t f16x2_to_e4m3x2(uint32_t h2) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(r) : "r"(h2));
  return r;
}

// Three e4m3 terms of a pair of non-negative floats (lo -> low byte), split
// in f16: x = f16(x), t1 = e4m3(x), t2 = e4m3(x - t1), t3 = e4m3(x - t1 - t2);
// each difference is exact in f16.
__device__ __forceinline__ void three_terms2(float lo, float hi, uint32_t &t1, uint32_t &t2, uint32_t &t3) {
  const __half2 x = __floats2half2_rn(lo, hi);
  const uint32_t xb = *reinterpret_cast<const uint32_t *>(&x);
  t1 = f16x2_to_e4m3x2(xb);
  const uint32_t b1 = e4m3x2_to_f16x2(t1);
  const __half2 r1 = __hsub2(x, *reinterpret_cast<const __half2 *>(&b1));
  const uint32_t r1b = *reinterpret_cast<const uint32_t *>(&r1);
  t2 = f16x2_to_e4m3x2(r1b);
  const uint32_t b2 = e4m3x2_to_f16x2(t2);
  const __half2 r2 = __hsub2(r1, *reinterpret_cast<const __half2 *>(&b2));
  t3 = f16x2_to_e4m3x2(*reinterpret_cast<const uint32_t *>(&r2));
}

// Softmax warpgroup wg (heads 32 wg .. 32 wg + 31).  Warp w of the group
// reads the S^T rows of tensor-memory quarter w % 4: tokens 16 q .. 16 q + 15
// of the page (the M = 64 accumulator keeps row i in lane 32 (i / 16) + i % 16).
__device__ __forceinline__ void tc_softmax(const DecodeArgs &a, uint8_t *smem, const Bars &B, const ItemDesc *items,
                                           const uint32_t *item_status, uint32_t tmem, volatile int *abort_flag) {
  const TcSmem sp = tc_smem();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int wg = (warp - 2) >> 2;          // warpgroup: 0 or 1
  const int wq = (warp - 2) & 3;           // warp within the group
  const int gq = warp & 3;                 // tensor-memory lane quarter
  const int wt = threadIdx.x - 64 - 128 * wg;  // 0..127 within the group
  const int bar_id = 1 + wg;
  const int gid = lane >> 2, tig = lane & 3;
  const int hb = 32 * wg;                  // first head of the group
  float *wsc = reinterpret_cast<float *>(smem + sp.wg);
  float *s_cq = wsc + kWgCq, *s_m = wsc + kWgM, *s_alpha = wsc + kWgAlpha, *s_beta = wsc + kWgBeta;
  float *s_ex = wsc + kWgEx + wg * 128;     // [warp][32 heads]
  float *s_exs = wsc + kWgExS + wg * 4;     // [warp]
  const float *scales = reinterpret_cast<const float *>(smem + sp.scales);
  uint8_t *pbase = smem + sp.p;
  const uint32_t tq = tmem + ((uint32_t)(32 * gq) << 16);
  const int t0 = 16 * gq + gid, t1 = t0 + 8;  // this thread's two tokens of the page
  uint32_t g = 0;
  for (uint32_t it = 0;; ++it) {
    const uint32_t slot = it % kNIQ;
    bool fail = !mbar_wait(&B.item_full[slot], (it / kNIQ) & 1u, abort_flag);
    if (wg_bar_or(bar_id, fail)) break;
    const ItemDesc d = items[slot];
    if (d.b < 0) break;
    const uint32_t n = (uint32_t)(d.p1 - d.p0);
    if (wt < 32) {
      s_cq[hb + wt] = __ldg(&a.qfac[(size_t)d.b * kTH + hb + wt]);
      s_m[hb + wt] = kNegInf;
    }
    float s_ref = 0.f;
    float lp[8];  // l of heads hb + 8k + 2 tig + e, index 2k + e
#pragma unroll
    for (int i = 0; i < 8; ++i) lp[i] = 0.f;
    named_bar_sync(bar_id, 128);
    float cq[8];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 c2 = *reinterpret_cast<const float2 *>(&s_cq[hb + 8 * k + 2 * tig]);
      cq[2 * k] = c2.x;
      cq[2 * k + 1] = c2.y;
    }
    bool dead = false;
    for (uint32_t j = 0; j < n; ++j) {
      const uint32_t gp = g + j, sb = gp & 1u, st = gp % kNst;
      fail = fail || !mbar_wait(&B.s_full[sb], (gp >> 1) & 1u, abort_flag) ||
             !mbar_wait(&B.full[st], (gp / kNst) & 1u, abort_flag) ||
             !mbar_wait(&B.p_empty[sb], ((gp >> 1) & 1u) ^ 1u, abort_flag);
      float y[16];  // [k][row][e] -> 4k + 2 row + e
      {
        tc_fence_after();
        uint32_t r[16], r2[16];
        tmem_ld16x256_x4(tq + kColS + 128 * sb + hb, r);        // K . T1
        tmem_ld16x256_x4(tq + kColS + 128 * sb + 64 + hb, r2);  // K . T2
#pragma unroll
        for (int i = 0; i < 16; ++i) y[i] = __uint_as_float(r[i]) + __uint_as_float(r2[i]);
        tc_fence_before();
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&B.s_empty[sb]);
      const int tok0 = (d.p0 + (int)j) * kTS;
      const bool v0 = tok0 + t0 < d.L, v1 = tok0 + t1 < d.L;
      const float s0 = v0 ? scales[st * kTS + t0] : 0.f, s1 = v1 ? scales[st * kTS + t1] : 0.f;
      float mx[8];
#pragma unroll
      for (int k = 0; k < 4; ++k)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          float &ya = y[4 * k + e], &yb = y[4 * k + 2 + e];
          ya = v0 ? ya * cq[2 * k + e] * s0 : kNegInf;
          yb = v1 ? yb * cq[2 * k + e] * s1 : kNegInf;
          float m = fmaxf(ya, yb);
          m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
          m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 8));
          m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 16));
          mx[2 * k + e] = m;
        }
      const float smx = warp_max_f32(fmaxf(s0, s1));
      if (gid == 0) {
#pragma unroll
        for (int k = 0; k < 4; ++k)
          *reinterpret_cast<float2 *>(&s_ex[wq * 32 + 8 * k + 2 * tig]) = make_float2(mx[2 * k], mx[2 * k + 1]);
      }
      if (lane == 0) s_exs[wq] = smx;
      if (wg_bar_or(bar_id, fail)) {
        dead = true;
        break;
      }
      const float sm = fmaxf(fmaxf(s_exs[0], s_exs[1]), fmaxf(s_exs[2], s_exs[3]));
      const float s_old = s_ref;
      const float s_new = sm > 2.f * s_old ? sm : s_old;
      bool resc = s_new != s_old;
      if (wt < 32) {
        const int h = hb + wt;
        const float tm = fmaxf(fmaxf(s_ex[wt], s_ex[32 + wt]), fmaxf(s_ex[64 + wt], s_ex[96 + wt]));
        const float m_old = s_m[h];
        const float m_new = tm > m_old + kTheta ? tm : m_old;
        const float alpha = fast_exp2(m_old - m_new);
        s_m[h] = m_new;
        s_alpha[h] = alpha;
        s_beta[h] = alpha * (s_old / s_new);
        resc = resc || m_new != m_old;
      }
      s_ref = s_new;
      resc = wg_bar_or(bar_id, resc) && j > 0;
      if (resc) {
        // this group's columns of O^T hold the earlier pages: scale head h by
        // beta_h once the previous page's PV has landed; l by alpha_h
        fail = fail || !mbar_wait(&B.p_empty[(gp - 1) & 1u], ((gp - 1) >> 1) & 1u, abort_flag);
        if (!fail) {
          tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < 4; ++c) {
            uint32_t r[32];
            const uint32_t ta = tq + kColO + 64 * c + hb;
            tmem_ld32(ta, r);
#pragma unroll
            for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * s_beta[hb + i]);
            tmem_st32(ta, r);
          }
          tmem_wait_st();
        }
#pragma unroll
        for (int k = 0; k < 4; ++k)
#pragma unroll
          for (int e = 0; e < 2; ++e) lp[2 * k + e] *= s_alpha[hb + 8 * k + 2 * tig + e];
      }
      // P'' = p (s_t / s_ref) 2^kPExp as three e4m3 terms; p = 2^(z - m) summed into l
      const float kt0 = v0 ? fast_log2(s0 / s_ref) + kPExp : 0.f;
      const float kt1 = v1 ? fast_log2(s1 / s_ref) + kPExp : 0.f;
      const float rt0 = fast_exp2(-kt0), rt1 = fast_exp2(-kt1);
      // P^T, MN-major without swizzle: byte (head h, token t) at
      // (h % 16) + (h / 16) * 1024 + (t % 8) * 16 + (t / 8) * 128
      uint8_t *pt = pbase + sb * kPBuf;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int h = hb + 8 * k + 2 * tig;
        const float2 m2 = *reinterpret_cast<const float2 *>(&s_m[h]);
        const float pa0 = fast_exp2(y[4 * k] - m2.x + kt0), pa1 = fast_exp2(y[4 * k + 1] - m2.y + kt0);
        const float pb0 = fast_exp2(y[4 * k + 2] - m2.x + kt1), pb1 = fast_exp2(y[4 * k + 3] - m2.y + kt1);
        lp[2 * k] += pa0 * rt0 + pb0 * rt1;
        lp[2 * k + 1] += pa1 * rt0 + pb1 * rt1;
        uint32_t a1, a2, a3, b1, b2, b3;
        three_terms2(pa0, pa1, a1, a2, a3);
        three_terms2(pb0, pb1, b1, b2, b3);
        if (!fail) {
          const int hoff = (h & 15) + (h >> 4) * 1024;
          uint8_t *q0 = pt + hoff + (t0 & 7) * 16 + (t0 >> 3) * 128;
          uint8_t *q1 = pt + hoff + (t1 & 7) * 16 + (t1 >> 3) * 128;
          *reinterpret_cast<uint16_t *>(q0) = (uint16_t)a1;
          *reinterpret_cast<uint16_t *>(q0 + kPTerm) = (uint16_t)a2;
          *reinterpret_cast<uint16_t *>(q0 + 2 * kPTerm) = (uint16_t)a3;
          *reinterpret_cast<uint16_t *>(q1) = (uint16_t)b1;
          *reinterpret_cast<uint16_t *>(q1 + kPTerm) = (uint16_t)b2;
          *reinterpret_cast<uint16_t *>(q1 + 2 * kPTerm) = (uint16_t)b3;
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
    // l per head: over the eight threads that share a head, then the four warps
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      float v = lp[i];
      v += __shfl_xor_sync(0xffffffffu, v, 4);
      v += __shfl_xor_sync(0xffffffffu, v, 8);
      v += __shfl_xor_sync(0xffffffffu, v, 16);
      lp[i] = v;
    }
    if (gid == 0) {
#pragma unroll
      for (int k = 0; k < 4; ++k)
        *reinterpret_cast<float2 *>(&s_ex[wq * 32 + 8 * k + 2 * tig]) = make_float2(lp[2 * k], lp[2 * k + 1]);
    }
    if (wg_bar_or(bar_id, fail)) break;
    if (wt < 32) s_alpha[hb + wt] = s_ex[wt] + s_ex[32 + wt] + s_ex[64 + wt] + s_ex[96 + wt];
    named_bar_sync(bar_id, 128);
    tc_fence_after();
    const uint32_t stv = item_status[slot];
    const float oscale = s_ref * exp2f(-kPExp);  // O^T accumulates p (s_t / s_ref) 2^kPExp * code
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
      uint32_t r[32];
      tmem_ld32(tq + kColO + 64 * c + hb, r);
      const int dd = 128 * c + 32 * gq + lane;  // value index of this thread's row
      if (d.nb == 1) {
        float *o = a.out + ((size_t)d.b * kTH + hb) * kTDv + dd;
#pragma unroll
        for (int i = 0; i < 32; ++i)
          o[(size_t)i * kTDv] = stv ? 0.f : __uint_as_float(r[i]) * oscale / s_alpha[hb + i];
      } else {
        float *o = a.part_o + ((size_t)d.cg * kTH + hb) * kTDv + dd;
#pragma unroll
        for (int i = 0; i < 32; ++i) o[(size_t)i * kTDv] = __uint_as_float(r[i]) * oscale;
      }
    }
    if (d.nb != 1 && wt < 32)
      a.part_ml[(size_t)d.cg * kTH + hb + wt] = make_float2(s_m[hb + wt], s_alpha[hb + wt]);
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(B.o_empty);
    named_bar_sync(bar_id, 128);  // the scratch is reused by the next item
    if (wt == 0) mbar_arrive(&B.item_empty[slot]);
    g += n;
  }
}

__global__ void __launch_bounds__(kTThreads, 1) latent_tc_kernel(const __grid_constant__ CUtensorMap map,
                                                                 const __grid_constant__ CUtensorMap map_tail,
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
      mbar_init(&B.s_empty[i], 8);
      mbar_init(&B.p_full[i], 8);
      mbar_init(&B.p_empty[i], 1);
    }
    mbar_init(B.q_full, 1);
    mbar_init(B.q_empty, 1);
    mbar_init(B.o_empty, 8);
    mbar_init(B.drain, 1);
    for (int i = 0; i < kNIQ; ++i) {
      mbar_init(&B.item_full[i], 1);
      mbar_init(&B.item_empty[i], 3);  // the MMA thread and the two softmax groups
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
    if (lane == 0) {
      tma_prefetch_desc(&map);
      tma_prefetch_desc(&map_tail);
    }
    tc_producer(a, map, map_tail, smem, B, items, item_status, abort_flag);
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

// Tensor maps over the stream pool viewed as [page][slot][576 bytes]: boxes
// of one page x 128 bytes (128-byte swizzle) for columns 0-511, and one page
// x 64 bytes (64-byte swizzle) for columns 512-575.
static int make_stream_map(CUtensorMap *map, const void *pool, int P, uint32_t box_bytes, CUtensorMapSwizzle swz) {
  EncodeTiledFn enc = encode_tiled_fn();
  if (!enc) return cuda_fail(cudaErrorNotSupported, "cuTensorMapEncodeTiled entry point");
  cuuint64_t dims[3] = {(cuuint64_t)kTD, (cuuint64_t)kTS, (cuuint64_t)P};
  cuuint64_t strides[2] = {(cuuint64_t)kTD, (cuuint64_t)kTD * kTS};
  cuuint32_t box[3] = {box_bytes, (cuuint32_t)kTS, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(pool), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cuda_fail(cudaErrorInvalidValue, "cuTensorMapEncodeTiled (stream)");
  return PFKV_OK;
}

int launch_latent_decode(const DecodeArgs &a0, cudaStream_t s) {
  // Work items are splits of a request, all 64 heads each.
  DecodeArgs a = a0;
  a.Hkv = 1;
  a.G = kTH;
  a.qprep = 1;
  CUtensorMap map, map_tail;
  int rc = make_stream_map(&map, a.k_pool, a.P, 128, CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc) return rc;
  rc = make_stream_map(&map_tail, a.k_pool, a.P, 64, CU_TENSOR_MAP_SWIZZLE_64B);
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
  // one equal page range per CTA when requests may be cut into 3 or more
  // pieces; otherwise longest-first items from a shared counter
  a.balanced = a.max_splits >= 3 ? (grid < kMaxRanges ? grid : kMaxRanges) : 0;
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
  rc = cuda_ok(cudaLaunchKernelEx(&cfg, latent_tc_kernel, map, map_tail, a), "latent kernel launch");
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
