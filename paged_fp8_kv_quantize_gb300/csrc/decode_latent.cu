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
//   S = Q . K^T   M = 128 query rows, N = 64 tokens (one page), K = 576.
//        The bf16 query of head h is q_h = 2^e_h (T1 + T2), two e4m3 terms
//        with one power-of-two scale (exact for every element within 2^10
//        of the row's largest); both terms are rows of A, so one MMA per K
//        step gives T1.k and T2.k, which the softmax warps add.  A lives in
//        tensor memory (columns 0-511 of the query) and, for the last 64
//        columns, in shared memory; the softmax warps move it there from
//        the page ring once per work item.
//   O^T += V^T . P^T   M = 128 values (four chunks of the 512), N = 64
//        heads, K = 64 tokens.  V^T is the page itself read MN-major.  The
//        probabilities, with the token's scale folded in relative to a
//        running reference scale, are written by the softmax warps as three
//        8-bit terms (e4m3, e4m3, e5m2: 11 significant bits) or, on pages
//        with large values, four (e4m3 x 3, e5m2: about 15 bits).
// The softmax normaliser l sums the weights as the terms carry them.
//
// A small kernel first writes every request's query terms into the
// workspace (one block per request and 16 heads).  The decode kernel: one
// CTA per SM, persistent.  There is no plan kernel: every CTA works out
// its pieces from the lengths (the shared work split: the requests' pages,
// plus a small per-piece overhead, cut into one equal range per CTA); a
// piece is a request's part of the range, all 64 heads.  Warp 0 loads each
// piece's query image (two ring entries) and then its pages into a
// five-entry ring (TMA, bounds and tag checks beside the copies; in a
// decode step it writes the request's new row into its page just before
// copying that page); warp 1
// owns tensor memory and issues the QK^T MMAs and warps 6 and 7 the PV MMAs
// of two value chunks each (one thread each, so that the instruction
// streams overlap on the tensor pipe); warps 2-5 and 8-11 run the softmax:
// warp w reads tensor-memory quarter w % 4, i.e. heads 16 q .. 16 q + 15,
// and one half of the page's tokens, each lane one head and 16 tokens; the
// two warps of a quarter agree on each page's maximum through shared
// memory, so the running maxima are identical in both and the sums are per
// thread.  The softmax warps also load each piece's query terms (tensor
// memory and the shared-memory tail), the next piece's as soon as the last
// QK^T of the current one has read the operand, before the current piece's
// result is read out, so that the next piece's QK^T overlaps that read-out.
// A running maximum moves only when it grows by more than 8x; O^T, whose
// columns are heads and whose lanes are values, is then rescaled by the
// softmax warps before the page's PV, a hand-off that costs nothing on the
// pages that need none.  Partials of a request cut into several pieces are
// merged by the shared log-sum-exp merge kernel, which also writes status.
#include <cuda_fp16.h>

#include <mutex>

#include "decode_common.cuh"
#include "merge.cuh"

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
// Query operand: 128 rows, row R = 32 (h / 16) + 16 t + h % 16 holds term t
// of head h; columns 0-511 live in tensor memory, columns 512-575 in shared
// memory as a 128 x 64 image with the 64-byte swizzle.
constexpr uint32_t kQTailBytes = 128 * 64;    // 8192
constexpr int kPieceCostLatent = 4;           // pages' worth of time a piece costs beyond its pages (swept 0-12: 4 fastest)
constexpr int kPT = 4;                        // 8-bit terms of the probabilities (at most)
constexpr uint32_t kPTerm = kTS * kTH;        // 4096: one P^T term of one page
constexpr uint32_t kPBuf = kPT * kPTerm;      // 16384
// A page whose largest value (its largest per-token scale x 448) exceeds this
// carries its probabilities in four terms instead of three: the output's
// error grows with the values' magnitude, and three terms (about 12
// significant bits) keep it within 2e-3 only for values up to about this.
constexpr float kFourTermAt = 8.f;
constexpr int kNst = 5;                       // pages in flight per CTA
constexpr int kPrefetch = 1;                  // pages pulled into L2 ahead of their copy (swept 0-10: 1 fastest)
constexpr int kTThreads = 384;                // producer, QK issuer, softmax x4, two PV issuers, softmax x4
constexpr int kSmxThreads = 256;              // the eight softmax warps (2-5 and 8-11)
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColQ = 0, kColS = 128, kColO = 256;  // Q (128) | S x2 (64 each) | O^T (4 x 64)
constexpr float kTheta = 3.f;                 // log2 growth of a running max that triggers a rescale
constexpr float kPExp = 4.75f;                // P'' = p (s_t / s_ref) 2^kPExp <= 2^kTheta * 2 * 2^4.75 < 448
constexpr uint32_t kIdQK = umma_idesc_e4m3(128, 64, 0, 0);
constexpr uint32_t kIdPV = umma_idesc_e4m3(128, 64, 1, 0);
constexpr uint32_t kIdPV5 = kIdPV | (1u << 10);  // B (the last probability term) in e5m2

// Softmax-warp scratch, floats: beta[2][64] | l[2 halves][64] | m[64] | resc_tag[2] (uint32) |
// four-term flag per P buffer [2] (uint32) | pad |
// page maxima exchanged by the two warps of a lane quarter: scores [2 pages][2 halves][64] and
// per-token scales [2 pages][2 halves][4 quarters] | per softmax warp, the reciprocal scales of
// its 32 tokens of the current page [8][32]
constexpr int kWgBeta = 0, kWgL = 128, kWgM = 256, kWgTag = 320, kWgFour = 322, kWgX = 328,
              kWgSmx = kWgX + 2 * 2 * 64, kWgInv = kWgSmx + 2 * 2 * 4, kWgFloats = kWgInv + 8 * 32;
static_assert(kWgInv % 4 == 0, "the reciprocal scales are read as float4");

struct TcSmem {
  uint32_t ring, qtail, p, scales, wg, bars, items, ws, total;
};

__host__ __device__ constexpr TcSmem tc_smem() {
  TcSmem s{};
  s.ring = 0;                                  // kNst pages (1024-aligned)
  s.qtail = s.ring + kNst * kPageSm;           // query tail (A of the last two QK^T steps)
  s.p = s.qtail + kQTailBytes;                 // 2 buffers x kPT P^T terms
  s.scales = s.p + 2 * kPBuf;                  // kNst x 64 per-token scales
  s.wg = s.scales + kNst * kTS * 4;            // softmax-warp scratch (layout above)
  s.bars = s.wg + 4 * kWgFloats;
  s.items = s.bars + 8 * (2 * kNst + 14 + 3 * kNIQ);
  s.ws = (s.items + (sizeof(ItemDesc) + 4) * kNIQ + 16 + 15) & ~15u;  // the page loader's work-split state
  s.total = s.ws + sizeof(WorkSplit);
  return s;
}
static_assert(tc_smem().total + 1024 <= 232448, "shared memory plan exceeds one SM");
static_assert(kLatentQTermBytes == 2 * kPageSm && kQTailBytes == kSmxThreads * 32 && kTH <= kTS,
              "the query image fills two ring entries; each softmax thread copies 32 bytes of its tail");

// Bounded wait that ignores the abort flag: used on the way out, so that a
// block that gave up still lets its own copies and MMAs land before it exits.
__device__ __forceinline__ void drain_wait(uint64_t *bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity))
    if (global_timer_ns() - t0 > kWaitLimitNs) return;
}

struct Bars {
  uint64_t *full, *empty, *s_full, *s_empty, *p_full, *p_empty, *q_ready, *q_empty, *o_empty, *r_done, *drain;
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
  r.q_ready = b; b += 1;
  r.q_empty = b; b += 1;
  r.o_empty = b; b += 1;
  r.r_done = b; b += 1;
  r.drain = b; b += 1;
  r.item_full = b; b += kNIQ;
  r.item_empty = b; b += kNIQ;
  r.item_done = b;
  return r;
}

// ---------------------------------------------------------------- producer (warp 0)

// Decode step: the request's new token goes to slot `pos` % 64 of the page
// that lane `src` of the batch looked up, unless that page is outside the
// pool or (tag check on) its tag does not match; the walk reports those cases
// in the request's status as for any page.  Quantized exactly as the append
// does (per-token scale amax / 448, or 1 for an all-zero row; x / s with
// IEEE division, round to nearest even, saturating).  The stores are made
// visible to the tensor-copy engine before the page is copied.
__device__ __forceinline__ void write_new_row(const DecodeArgs &a, const AppendRow &r, int src, int pid_lane,
                                              bool bad_lane, int pos, int lane) {
  const int pid = __shfl_sync(0xffffffffu, pid_lane, src);
  if (__shfl_sync(0xffffffffu, bad_lane, src)) return;
  append_row_store<true>(a.cache, r, 0, 0, pid, pos, lane);
  asm volatile("fence.proxy.async.global;" ::: "memory");
  __syncwarp();
}

__device__ __forceinline__ void tc_producer(const DecodeArgs &a, const CUtensorMap &map, const CUtensorMap &map_tail,
                                            uint8_t *smem, const Bars &B, ItemDesc *items, uint32_t *item_status,
                                            volatile int *abort_flag) {
  const TcSmem sp = tc_smem();
  const int lane = threadIdx.x & 31;
  const bool tag_check = (a.flags & PFKV_FLAG_TAG_CHECK) != 0u;
  const uint64_t stream_pol = l2_evict_first_policy();
  uint32_t g = 0;  // ring entries (query images and pages) issued by this CTA
  bool ok = true;
  // This CTA's pieces, worked out from the lengths; the next one is found
  // once the current one's pages have gone out.
  WorkSplit &s_ws = *reinterpret_cast<WorkSplit *>(smem + sp.ws);
  const WsArgs wa = ws_args(a);
  {
    WorkSplit w;
    ws_init(w, wa, lane);
    if (lane == 0) s_ws = w;
    __syncwarp();
  }
  Piece cur;
  bool have = ws_next_shared(s_ws, wa, cur, lane);
  for (uint32_t it = 0;; ++it) {
    const uint32_t slot = it % kNIQ;
    bool w = true;
    if (lane == 0) w = mbar_wait(&B.item_empty[slot], ((it / kNIQ) & 1u) ^ 1u, abort_flag);
    if (!__shfl_sync(0xffffffffu, w, 0)) { ok = false; break; }
    // test hook (PFKV_FLAG_TEST_WITHHOLD): the first CTA never hands its
    // first item (or its end marker) to the other warps, whose bounded waits
    // then give up
    const bool withhold = (a.flags & PFKV_FLAG_TEST_WITHHOLD) && blockIdx.x == 0 && it == 0;
    if (!have) {
      if (lane == 0) {
        items[slot].b = -1;
        if (!withhold) mbar_arrive(&B.item_full[slot]);
      }
      break;
    }
    const int b = cur.b, p0 = cur.p0, p1 = cur.p1, L = cur.L;
    if (lane == 0) {
      // ring entries g, g + 1: the query image; g + 2 + j: page p0 + j
      ItemDesc d;
      d.b = b; d.cg = cur.cg; d.g = 0; d.p0 = p0; d.p1 = p1; d.L = L; d.ring = g; d.nb = cur.nb;
      items[slot] = d;
      if (!withhold) mbar_arrive(&B.item_full[slot]);
      if (cur.lead) {  // the merge's view of the numbering
        a.split_first[b] = cur.cg;
        a.split_count[b] = cur.nb;
      }
    }
    // The item's query image in two ring entries ahead of its pages, with
    // its score factors in the first entry's scale slot: copied with the
    // page stream, so that reaching them costs the consumers no memory round
    // trip at the item change.
    {
      uint32_t nq = 0;
      if (lane == 0)
        for (; nq < 2; ++nq) {
          const uint32_t r = g + nq, st = r % kNst;
          if (!mbar_wait(&B.empty[st], ((r / kNst) & 1u) ^ 1u, abort_flag)) break;
          mbar_arrive_expect_tx(&B.full[st], kPageSm + (nq == 0 ? kTH * 4 : 0));
          bulk_load_stream(smem + sp.ring + st * kPageSm, a.qterms + (size_t)b * kLatentQTermBytes + nq * kPageSm,
                           kPageSm, &B.full[st], stream_pol);
          if (nq == 0)
            bulk_load_stream(smem + sp.scales + st * (kTS * 4), a.qfac + (size_t)b * kTH, kTH * 4, &B.full[st],
                             stream_pol);
        }
      nq = __shfl_sync(0xffffffffu, nq, 0);
      g += nq;
      ok = nq == 2;
    }
    // Decode step: the piece holding the request's last page writes the new
    // token's row into that page before copying it; the row is loaded now so
    // that its latency hides behind the walk.
    const int i_new = (L - 1) / kTS;
    const bool has_new = a.append && p0 <= i_new && i_new < p1;
    AppendRow nrow;
    if (has_new) nrow = append_row_load<true>(a.cache, a.k_new, nullptr, b, 0, 0, lane);
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
      // a decode step's destination page (the request's last) gets the new
      // row just before its own copy, the pages before it already in flight
      const int dest_k = has_new && i0 <= i_new && i_new < i0 + 32 ? i_new - i0 : -1;
      const int cnt = min(32, p1 - i0);
      // pages kPrefetch ahead of the copies are pulled into L2, so that a copy
      // issued when a ring slot frees up finds its page there
      auto prefetch = [&](int k) {
        const int pk = __shfl_sync(0xffffffffu, pid, k);
        const bool bad = __shfl_sync(0xffffffffu, oob, k);
        if (lane == 0 && !bad) {
#pragma unroll
          for (int c = 0; c < 4; ++c) tma_prefetch_l2_3d_stream(&map, 128 * c, 0, pk, stream_pol);
          tma_prefetch_l2_3d_stream(&map_tail, 512, 0, pk, stream_pol);
          bulk_prefetch_l2_stream(a.k_scale + (size_t)pk * kTS, kTS * 4, stream_pol);
        }
      };
      // (the CTA's first kNst pages go straight into an empty ring: no prefetch)
      for (int k = 0; k < min(kPrefetch, cnt); ++k)
        if (g + (uint32_t)k >= (uint32_t)kNst) prefetch(k);
      for (int k = 0; k < cnt; ++k) {
        if (k + kPrefetch < cnt) prefetch(k + kPrefetch);
        if (k == dest_k) write_new_row(a, nrow, k, pid, oob || page_tag != want_tag, L - 1, lane);
        const int pk = __shfl_sync(0xffffffffu, pid, k);
        const bool bad_k = __shfl_sync(0xffffffffu, oob, k);
        bool w = true;
        if (lane == 0) {
          const uint32_t r = g + (uint32_t)k, st = r % kNst;
          w = mbar_wait(&B.empty[st], ((r / kNst) & 1u) ^ 1u, abort_flag);
          if (w) {
            if (bad_k) {
              mbar_arrive(&B.full[st]);  // never fetched; the request is aborted
            } else {
              mbar_arrive_expect_tx(&B.full[st], kPageSm + kTS * 4);
              uint8_t *stage = smem + sp.ring + st * kPageSm;
#pragma unroll
              for (int c = 0; c < 4; ++c)
                tma_load_3d_stream(stage + c * kBlk, &map, &B.full[st], 128 * c, 0, pk, stream_pol);
              tma_load_3d_stream(stage + kPageTail, &map_tail, &B.full[st], 512, 0, pk, stream_pol);
              bulk_load_stream(smem + sp.scales + st * (kTS * 4), a.k_scale + (size_t)pk * kTS, kTS * 4, &B.full[st],
                               stream_pol);
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
      mbar_arrive(&B.item_done[slot]);
    }
    if (!ok) break;
    have = ws_next_shared(s_ws, wa, cur, lane);
  }
  // Copies still in flight land before the block may exit.
  if (lane == 0)
    for (uint32_t k = g > kNst ? g - kNst : 0; k < g; ++k) drain_wait(&B.full[k % kNst], (k / kNst) & 1u);
}

// ---------------------------------------------------------------- MMA issuers (warps 1 and 6, one thread each)

// Shared-memory descriptors, built once; an MMA adds its operand's byte
// offset / 16 to the start-address field (addresses stay below 256 KB, so
// the 14-bit field never carries).
struct TcDesc {
  uint64_t page, page_tail, qtail, vt, pt;
};

__device__ __forceinline__ TcDesc tc_desc(uint8_t *smem) {
  const TcSmem sp = tc_smem();
  const uint32_t s_ring = smem_addr(smem + sp.ring), s_qt = smem_addr(smem + sp.qtail), s_p = smem_addr(smem + sp.p);
  TcDesc d;
  d.page = umma_sdesc(s_ring, 16, 1024, 2);                // B of QK^T: page rows, 128-byte swizzle
  d.page_tail = umma_sdesc(s_ring + kPageTail, 16, 512, 4);  // B of the tail steps
  d.qtail = umma_sdesc(s_qt, 16, 512, 4);                   // A of the tail steps
  d.vt = umma_sdesc(s_ring, 8192, 1024, 2);                 // A of PV: V^T, MN-major
  d.pt = umma_sdesc(s_p, 128, 512, 0);                      // B of PV: P^T, K-major
  return d;
}

// QK^T issuer (warp 1): S[sb] = [T1; T2 rows] . K_page^T for every page in
// order (page j of an item in ring entry ring + 2 + j), as soon as the page
// has landed and the softmax warps have read the S buffer's previous page.
// After an item's last page it commits q_empty: the query operand may then be
// replaced by the next item's.
__device__ __forceinline__ void tc_mma_qk(uint8_t *smem, const Bars &B, const ItemDesc *items, uint32_t tmem,
                                          volatile int *abort_flag) {
  const TcDesc dd = tc_desc(smem);
  uint32_t g = 0;  // pages consumed before the current item
  for (uint32_t it = 0;; ++it) {
    const uint32_t slot = it % kNIQ;
    if (!mbar_wait(&B.item_full[slot], (it / kNIQ) & 1u, abort_flag)) break;
    const ItemDesc d = items[slot];
    mbar_arrive(&B.item_empty[slot]);
    if (d.b < 0) break;
    const uint32_t n = (uint32_t)(d.p1 - d.p0);
    if (!mbar_wait(B.q_ready, it & 1u, abort_flag)) break;  // the item's query operand is in place
    bool ok = true;
    for (uint32_t j = 0; j < n; ++j) {
      const uint32_t gp = g + j, sb = gp & 1u, rr = d.ring + 2 + j, st = rr % kNst;
      if (!mbar_wait(&B.full[st], (rr / kNst) & 1u, abort_flag) ||
          !mbar_wait(&B.s_empty[sb], ((gp >> 1) & 1u) ^ 1u, abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
      // 128 x 64, K = 576 in 18 steps of 32
      const uint64_t pg = (uint64_t)((st * kPageSm) >> 4);
      const uint32_t d_s = tmem + kColS + 64 * sb;
#pragma unroll
      for (int kk = 0; kk < 16; ++kk)
        umma_e4m3_ts(d_s, tmem + kColQ + 8 * kk, dd.page + pg + (uint64_t)(((kk >> 2) * kBlk + (kk & 3) * 32) >> 4),
                     kIdQK, kk ? 1u : 0u);
#pragma unroll
      for (int kk = 0; kk < 2; ++kk)
        umma_e4m3(d_s, dd.qtail + (uint64_t)(2 * kk), dd.page_tail + pg + (uint64_t)(2 * kk), kIdQK, 1u);
      umma_commit(&B.s_full[sb]);
    }
    if (!ok) break;
    umma_commit(B.q_empty);  // the query operand may be replaced
    g += n;
  }
  // every MMA issued here has completed before tensor memory is released
  umma_commit(B.drain);
  drain_wait(B.drain, 0);
}

// PV issuers (warps 6 and 7, value chunks 2 h and 2 h + 1 for h = warp - 6):
// O^T[c] (+)= V^T_c . (P1 + P2 + P3)^T for every page in order, once its
// P^T is written (and, for an item's first page, the
// previous item's O^T has been read out; after a rescale hand-off, once the
// softmax warps have scaled O^T).  Frees the page's ring slot and P buffer.
__device__ __forceinline__ void tc_mma_pv(uint8_t *smem, const Bars &B, const ItemDesc *items, uint32_t tmem,
                                          volatile int *abort_flag, int half) {
  const TcSmem sp = tc_smem();
  const TcDesc dd = tc_desc(smem);
  const volatile uint32_t *resc_tag = reinterpret_cast<const uint32_t *>(smem + sp.wg) + kWgTag;
  const volatile uint32_t *four_flag = reinterpret_cast<const uint32_t *>(smem + sp.wg) + kWgFour;
  uint32_t g = 0, n_resc = 0;
  for (uint32_t it = 0;; ++it) {
    const uint32_t slot = it % kNIQ;
    if (!mbar_wait(&B.item_full[slot], (it / kNIQ) & 1u, abort_flag)) break;
    const ItemDesc d = items[slot];
    mbar_arrive(&B.item_empty[slot]);
    if (d.b < 0) break;
    const uint32_t n = (uint32_t)(d.p1 - d.p0);
    if (!mbar_wait(B.o_empty, (it & 1u) ^ 1u, abort_flag)) break;
    bool ok = true;
    for (uint32_t j = 0; j < n; ++j) {
      const uint32_t gp = g + j, st = (d.ring + 2 + j) % kNst, pb = gp & 1u;
      if (!mbar_wait(&B.p_full[pb], (gp >> 1) & 1u, abort_flag)) {
        ok = false;
        break;
      }
      if (j > 0 && resc_tag[pb] == gp + 1u) {
        if (!mbar_wait(B.r_done, n_resc & 1u, abort_flag)) {
          ok = false;
          break;
        }
        ++n_resc;
      }
      tc_fence_after();
      const uint64_t pg = (uint64_t)((st * kPageSm) >> 4), pp = (uint64_t)((pb * kPBuf) >> 4);
      const uint32_t first = j == 0 ? 0u : 1u;
      // three terms (e4m3, e4m3, e5m2) or four (e4m3 x 3, e5m2), as the softmax warps chose for the page
      const bool four = four_flag[pb] != 0u;
#pragma unroll
      for (int c = 2 * half; c < 2 * half + 2; ++c)
#pragma unroll
        for (int t = 0; t < kPT; ++t) {
          if (t == kPT - 1 && !four) continue;
          const uint32_t id = (t == kPT - 1 || (t == kPT - 2 && !four)) ? kIdPV5 : kIdPV;
#pragma unroll
          for (int ks = 0; ks < 2; ++ks)
            umma_e4m3(tmem + kColO + 64 * c, dd.vt + pg + (uint64_t)((c * kBlk + ks * 4096) >> 4),
                      dd.pt + pp + (uint64_t)((t * kPTerm + ks * 256) >> 4), id, (t == 0 && ks == 0) ? first : 1u);
        }
      umma_commit(&B.empty[st]);
      umma_commit(&B.p_empty[pb]);
    }
    if (!ok) break;
    g += n;
  }
  umma_commit(B.drain);
  drain_wait(B.drain, 0);
}

// ---------------------------------------------------------------- softmax warps (warps 2-5 and 8-11)

// Barrier `id` of `nthreads` threads that also ORs a flag over them.
__device__ __forceinline__ bool bar_or(int id, int nthreads, bool v) {
  uint32_t r;
  asm volatile(
      "{\n.reg .pred p, q;\nsetp.ne.u32 p, %3, 0;\nbar.red.or.pred q, %1, %2, p;\nselp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"(id), "r"(nthreads), "r"((uint32_t)v)
      : "memory");
  return r != 0u;
}

// All softmax warps (barrier 1).
__device__ __forceinline__ bool wg_bar_or(bool v) { return bar_or(1, kSmxThreads, v); }

__device__ __forceinline__ uint32_t f16x2_to_e4m3x2(uint32_t h2) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(r) : "r"(h2));
  return r;
}
__device__ __forceinline__ uint32_t f16x2_to_e5m2x2(uint32_t h2) {
  uint16_t r;
  asm("cvt.rn.satfinite.e5m2x2.f16x2 %0, %1;" : "=h"(r) : "r"(h2));
  return r;
}

// The 8-bit terms of a pair of non-negative floats (lo -> low byte), each
// rounded to nearest even.  Three terms (pages of small values): x is
// rounded to f16 and split as t1 = e4m3(x), t2 = e4m3(x - t1),
// t3 = e5m2(x - t1 - t2), every difference exact in f16 (about 11
// significant bits, packed f16 arithmetic).  Four terms (pages with large
// values, whose output needs more): split from fp32 as t1 = e4m3(x),
// t2 = e4m3(x - t1), t3 = e4m3(x - t1 - t2), t4 = e5m2(x - t1 - t2 - t3),
// every difference exact in fp32 (about 15 bits).  The last term is e5m2 for
// its range (down to 2^-16, against 2^-9 for e4m3): it keeps the share of
// the many small weights far below the running maximum, which e4m3 alone
// would flush to zero.  Returns the pair the terms represent, exactly.
__device__ __forceinline__ float2 p_terms2(float lo, float hi, bool four, uint32_t &t1, uint32_t &t2, uint32_t &t3,
                                           uint32_t &t4) {
  if (!four) {
    const __half2 x = __floats2half2_rn(lo, hi);
    t1 = f16x2_to_e4m3x2(*reinterpret_cast<const uint32_t *>(&x));
    const uint32_t b1 = e4m3x2_to_f16x2(t1);
    const __half2 r1 = __hsub2(x, *reinterpret_cast<const __half2 *>(&b1));
    t2 = f16x2_to_e4m3x2(*reinterpret_cast<const uint32_t *>(&r1));
    const uint32_t b2 = e4m3x2_to_f16x2(t2);
    const __half2 r2 = __hsub2(r1, *reinterpret_cast<const __half2 *>(&b2));
    t3 = f16x2_to_e5m2x2(*reinterpret_cast<const uint32_t *>(&r2));
    const uint32_t b3 = e5m2x2_to_f16x2(t3);
    const __half2 r3 = __hsub2(r2, *reinterpret_cast<const __half2 *>(&b3));
    t4 = 0u;
    return __half22float2(__hsub2(x, r3));
  }
  t1 = f32x2_to_e4m3x2(lo, hi);
  const uint32_t b1 = e4m3x2_to_f16x2(t1);
  const float2 d1 = __half22float2(*reinterpret_cast<const __half2 *>(&b1));
  const float r1x = lo - d1.x, r1y = hi - d1.y;
  t2 = f32x2_to_e4m3x2(r1x, r1y);
  const uint32_t b2 = e4m3x2_to_f16x2(t2);
  const float2 d2 = __half22float2(*reinterpret_cast<const __half2 *>(&b2));
  const float r2x = r1x - d2.x, r2y = r1y - d2.y;
  t3 = f32x2_to_e4m3x2(r2x, r2y);
  const uint32_t b3 = e4m3x2_to_f16x2(t3);
  const float2 d3 = __half22float2(*reinterpret_cast<const __half2 *>(&b3));
  t4 = f32x2_to_e5m2x2(r2x - d3.x, r2y - d3.y);
  const uint32_t b4 = e5m2x2_to_f16x2(t4);
  const float2 d4 = __half22float2(*reinterpret_cast<const __half2 *>(&b4));
  return make_float2(((d1.x + d2.x) + d3.x) + d4.x, ((d1.y + d2.y) + d3.y) + d4.y);
}

// Query terms of the latent stream, one block per (request, 16 heads),
// before the decode kernel.  Head h's bf16 row (576 values) is scaled by
// 2^-e_h, e_h the exponent that puts max|q| in [128, 256), and written as
// T1 = e4m3(q 2^-e_h) and T2 = e4m3(q 2^-e_h - T1), both rounded to nearest
// even: T1 + T2 equals the scaled row exactly for every element of magnitude
// at least 2^-2 (a bf16 significand has 8 bits, each term carries 4), the
// rest to within 2^-10.  The terms form one 128-row operand: row
// R = 32 (h / 16) + 16 t + h % 16 holds term t of head h.  Columns 0-511
// are laid out as sixteen blocks of 128 rows x 32 bytes: block k (columns
// 32 k .. 32 k + 31) at 4096 k, inside it units of 8 rows x 16 bytes, the 16
// bytes of row R, columns 32 k + 16 c .. + 15 at 4096 k + 256 (R / 8) +
// 128 c + 16 (R % 8), so that eight consecutive rows' bytes are contiguous.
// Columns 512-575 follow as the 64-byte-swizzled shared-memory image at
// 65536 (16-byte chunk j of row R at 65536 + R * 64 + 16 (j ^ ((R >> 1) & 3))).
// The decode kernel copies the whole image into two ring slots (bytes
// 0-36863: blocks 0-8; 36864-73727: blocks 9-15 and the tail).
// qfac[b][h] = softmax scale * log2(e) * 2^e_h.
__global__ void __launch_bounds__(256) qterm_kernel(const DecodeArgs a) {
  constexpr int kRowV = kTD / 8 + 1;  // uint4 per staged row: 72 + 1 of padding (spreads the rows over the banks)
  __shared__ uint4 s_q[16 * kRowV];
  __shared__ float s_inv[16];
  __shared__ uint64_t s_bar;
  __shared__ int s_abort;
  pdl_wait();  // the stream's earlier work is complete from here on
  pdl_launch_dependents();
  const int b = blockIdx.x >> 2, hq = blockIdx.x & 3;  // request, group of 16 heads
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint16_t *q = static_cast<const uint16_t *>(a.q) + ((size_t)b * kTH + 16 * hq) * kTD;
  // the 16 query rows into shared memory with one bulk copy each (one
  // memory round trip for the block)
  if (tid == 0) {
    s_abort = 0;
    mbar_init(&s_bar, 1);
    mbar_init_fence();
  }
  __syncthreads();
  if (tid == 0) {
    mbar_arrive_expect_tx(&s_bar, 16 * kTD * 2);
    for (int hh = 0; hh < 16; ++hh) bulk_load(&s_q[hh * kRowV], q + hh * kTD, kTD * 2, &s_bar);
  }
  const bool landed = mbar_wait(&s_bar, 0, &s_abort);  // bounded
  if (__syncthreads_or(!landed))  // the copies did not land: read the rows directly
    for (int i = tid; i < 16 * (kTD / 8); i += (int)blockDim.x)
      s_q[(i / (kTD / 8)) * kRowV + i % (kTD / 8)] = reinterpret_cast<const uint4 *>(q)[i];
  __syncthreads();
  for (int hh = warp; hh < 16; hh += 8) {
    float m = 0.f;
    for (int k = lane; k < kTD / 8; k += 32) m = amax8(s_q[hh * kRowV + k], m);
    for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane == 0) {
      int e = 8;
      if (m > 0.f) frexpf(m, &e);  // m = f 2^e, f in [0.5, 1)
      s_inv[hh] = ldexpf(1.f, 8 - e);
      a.qfac[(size_t)b * kTH + 16 * hq + hh] = a.sm_scale_log2 * ldexpf(1.f, e - 8);
    }
  }
  __syncthreads();
  uint8_t *dst = a.qterms + (size_t)b * kLatentQTermBytes;
  for (int u = tid; u < 16 * 36; u += (int)blockDim.x) {
    // 16-value chunk r of head hh's row: neighbouring threads take
    // neighbouring heads, whose rows are neighbours in the image
    const int r = u >> 4, hh = u & 15;
    const int R1 = 32 * hq + hh, R2 = R1 + 16;  // rows of T1 and T2
    size_t off1, off2;
    if (r < 32) {
      const size_t blk = (size_t)(r >> 1) * 4096 + (size_t)(r & 1) * 128;
      off1 = blk + (size_t)(R1 >> 3) * 256 + (R1 & 7) * 16;
      off2 = blk + (size_t)(R2 >> 3) * 256 + (R2 & 7) * 16;
    } else {
      const int j = r - 32;
      off1 = (size_t)65536 + R1 * 64 + 16 * (j ^ ((R1 >> 1) & 3));
      off2 = (size_t)65536 + R2 * 64 + 16 * (j ^ ((R2 >> 1) & 3));
    }
    const uint4 v0 = s_q[hh * kRowV + 2 * r], v1 = s_q[hh * kRowV + 2 * r + 1];
    const uint32_t wv[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
    const float inv = s_inv[hh];
    uint32_t t1[4], t2[4];
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
    *reinterpret_cast<uint4 *>(dst + off1) = make_uint4(t1[0], t1[1], t1[2], t1[3]);
    *reinterpret_cast<uint4 *>(dst + off2) = make_uint4(t2[0], t2[1], t2[2], t2[3]);
  }
}

// The query operand of the item whose image sits in ring entries `ring`
// (bytes 0-36863 of the image, the score factors in its scale slot) and
// ring + 1 (the rest; the 8 KB tail image at 28672), once both have landed.
// Softmax thread (q, x, lane) moves row R = 32 q + lane, columns
// 256 x .. 256 x + 255, into tensor-memory columns 64 x .. 64 x + 63 of its
// lane (the image's 8-row x 16-byte blocks put the rows a phase of 8 lanes
// reads in distinct banks), and bytes 32 wt .. 32 wt + 31 of the tail image
// into the query-tail buffer.  Returns the score factor of head h, or sets
// fail (warp-uniform) if a wait gave up.  Whole warp; arrives on q_ready.
// The caller frees the two entries once every softmax warp is past this.
// One compiled copy for both call sites (first item, next item).
__device__ __noinline__ float q_take(uint8_t *smem, uint32_t ring, uint64_t *full, uint64_t *q_ready, uint32_t tq,
                                     int wt, int h, volatile int *abort_flag, bool &fail) {
  const TcSmem sp = tc_smem();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, q = warp & 3, x = warp >= 8 ? 1 : 0;
  const uint32_t qa = ring % kNst, qb = (ring + 1) % kNst;
  fail = __any_sync(0xffffffffu, !mbar_wait(&full[qa], (ring / kNst) & 1u, abort_flag) ||
                                     !mbar_wait(&full[qb], ((ring + 1) / kNst) & 1u, abort_flag));
  if (fail) return 0.f;
  const int R = 32 * q + lane;
  uint32_t r[2][32];
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    const int k = 8 * x + kk;  // 32-byte column block of the row
    const uint8_t *src = smem + sp.ring + (k < 9 ? qa * kPageSm + 4096 * k : qb * kPageSm + 4096 * (k - 9)) +
                         (R >> 3) * 256 + (R & 7) * 16;
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const uint4 v = *reinterpret_cast<const uint4 *>(src + 128 * c);
      const int o = (kk & 3) * 8 + c * 4;
      r[kk >> 2][o] = v.x; r[kk >> 2][o + 1] = v.y; r[kk >> 2][o + 2] = v.z; r[kk >> 2][o + 3] = v.w;
    }
  }
  tmem_st32(tq + kColQ + 64 * x, r[0]);
  tmem_st32(tq + kColQ + 64 * x + 32, r[1]);
  const uint4 *tsrc = reinterpret_cast<const uint4 *>(smem + sp.ring + qb * kPageSm +
                                                      (kLatentQTermBytes - kPageSm - kQTailBytes));
  uint4 *tdst = reinterpret_cast<uint4 *>(smem + sp.qtail);
  const uint4 v0 = tsrc[2 * wt], v1 = tsrc[2 * wt + 1];
  tdst[2 * wt] = v0;
  tdst[2 * wt + 1] = v1;
  const float qf = reinterpret_cast<const float *>(smem + sp.scales)[qa * kTS + h];
  fence_async_smem();
  tmem_wait_st();
  tc_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive(q_ready);
  return qf;
}

// Frees the two ring entries of a query image (two arrivals each, from two
// softmax warps), once every softmax warp is past q_take.
__device__ __forceinline__ void q_release(const Bars &B, uint32_t ring, int wt) {
  if (wt == 0 || wt == 32) {
    mbar_arrive(&B.empty[ring % kNst]);
    mbar_arrive(&B.empty[(ring + 1) % kNst]);
  }
}

// Softmax warp w (2-5 and 8-11) reads tensor-memory quarter q = w % 4, i.e.
// rows 32 q .. 32 q + 31 of S: T1 (lanes 0-15) and T2 (lanes 16-31) of heads
// 16 q .. 16 q + 15, and takes half x = (w >= 8) of the page's tokens.  After
// adding the two terms, lane l holds head 16 q + l % 16 and tokens
// 32 x + 16 (l / 16) .. + 15.  The two warps of a quarter agree on each
// page's maximum through shared memory (barrier 2 + q, which also ORs their
// failure flags, so both leave the page loop together).
__device__ __forceinline__ void tc_softmax(const DecodeArgs &a, uint8_t *smem, const Bars &B, const ItemDesc *items,
                                           const uint32_t *item_status, uint32_t tmem, volatile int *abort_flag) {
  const TcSmem sp = tc_smem();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int q = warp & 3;                       // tensor-memory lane quarter
  const int x = warp >= 8 ? 1 : 0;              // token half of the page (and half of the O^T columns)
  const int wt = (4 * x + (warp - 2 - 6 * x)) * 32 + lane;  // 0..255 over the softmax warps
  const int half = lane >> 4;                   // term of this lane's S row; then the 16-token chunk
  const int h = 16 * q + (lane & 15);           // head of this thread
  const int tb = 32 * x + 16 * half;            // first token of the page this thread owns
  float *wsc = reinterpret_cast<float *>(smem + sp.wg);
  float *s_beta = wsc + kWgBeta, *s_l = wsc + kWgL, *s_m = wsc + kWgM;
  float *s_x = wsc + kWgX, *s_smx = wsc + kWgSmx;
  float *s_inv = wsc + kWgInv + 32 * (wt >> 5);  // this warp's 32 tokens
  volatile uint32_t *resc_tag = reinterpret_cast<uint32_t *>(wsc + kWgTag);
  volatile uint32_t *four_flag = reinterpret_cast<uint32_t *>(wsc + kWgFour);
  const float *scales = reinterpret_cast<const float *>(smem + sp.scales);
  uint8_t *pbase = smem + sp.p;
  const uint32_t tq = tmem + ((uint32_t)(32 * q) << 16);
  // P^T (K-major, no swizzle): byte (head, token) at (head % 8) * 16 + (head / 8) * 512 +
  // (token / 16) * 128 + token % 16; this thread writes the 16-token chunk tb / 16
  const uint32_t p_off = (h & 7) * 16 + (h >> 3) * 512 + (tb / 16) * 128;
  uint32_t g = 0, n_resc = 0;
  float cq = 0.f;  // score factor of this lane's head for the current item
  {
    // the first item's query (the operand starts out free)
    bool fail = !mbar_wait(&B.item_full[0], 0, abort_flag);
    fail = wg_bar_or(fail);
    const int b0 = fail ? -1 : items[0].b;
    const uint32_t ring0 = items[0].ring;
    if (b0 >= 0) cq = q_take(smem, ring0, B.full, B.q_ready, tq, wt, h, abort_flag, fail);
    if (wg_bar_or(fail)) return;
    if (b0 >= 0) q_release(B, ring0, wt);
  }
  for (uint32_t it = 0;; ++it) {
    const uint32_t slot = it % kNIQ;
    bool fail = !mbar_wait(&B.item_full[slot], (it / kNIQ) & 1u, abort_flag);
    if (wg_bar_or(fail)) break;
    const ItemDesc d = items[slot];
    if (d.b < 0) break;
    const uint32_t n = (uint32_t)(d.p1 - d.p0);
    float cq_next = cq;
    float m = kNegInf, l = 0.f, s_ref = 0.f;
    // Rescale hand-off for page gq (not an item's first page): once every
    // warp's P^T and scale factors for it are in, if any head asked for it,
    // scale this warp's share of O^T (its quarter's lanes, columns 128 x ..
    // 128 x + 127) by beta_h per head column, after the previous page's PV
    // and before this page's.  Checked one page late, so that the softmax
    // warps need not wait for one another on every page: the PV of a page
    // that needs it waits for this hand-off, and the buffers it reads are
    // reused only after that PV.
    auto rescale_check = [&](uint32_t gq, bool &fl) {
      const uint32_t sq = gq & 1u;
      if (fl) return;
      fl = __any_sync(0xffffffffu, !mbar_wait(&B.p_full[sq], (gq >> 1) & 1u, abort_flag));
      if (fl || resc_tag[sq] != gq + 1u) return;
      fl = __any_sync(0xffffffffu, !mbar_wait(&B.p_empty[(gq - 1) & 1u], ((gq - 1) >> 1) & 1u, abort_flag));
      if (!fl) {
        tc_fence_after();
#pragma unroll 1
        for (int c = 4 * x; c < 4 * x + 4; ++c) {
          uint32_t r[32];
          const uint32_t ta = tq + kColO + 32 * c;
          tmem_ld32(ta, r);
          const float *bt = s_beta + sq * kTH + 32 * (c & 1);
#pragma unroll
          for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * bt[i]);
          tmem_st32(ta, r);
        }
        tmem_wait_st();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(B.r_done);
      ++n_resc;
    };
    for (uint32_t j = 0; j < n; ++j) {
      const uint32_t gp = g + j, sb = gp & 1u, rr = d.ring + 2 + j, st = rr % kNst;
      if (!fail)
        fail = !mbar_wait(&B.s_full[sb], (gp >> 1) & 1u, abort_flag) ||
               !mbar_wait(&B.full[st], (rr / kNst) & 1u, abort_flag) ||
               !mbar_wait(&B.p_empty[sb], ((gp >> 1) & 1u) ^ 1u, abort_flag);
      fail = __any_sync(0xffffffffu, fail);  // the warp-wide tensor-memory load below needs every lane
      float v[16], sv[16];
      float mt = kNegInf, smx = 0.f;
      if (!fail) {
        {
          tc_fence_after();
          uint32_t r[32];
          // T1 (rows 0-15 of the quarter) and T2 (rows 16-31) of head h, tokens tb .. tb + 15
          tmem_ld_pair16(tq + kColS + 64 * sb + 32 * x, r);
          tc_fence_before();
#pragma unroll
          for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]) + __uint_as_float(r[16 + i]);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&B.s_empty[sb]);
        const int tok0 = (d.p0 + (int)j) * kTS + tb;
#pragma unroll
        for (int i = 0; i < 16; i += 4) {
          const float4 s4 = *reinterpret_cast<const float4 *>(&scales[st * kTS + tb + i]);
          sv[i] = s4.x; sv[i + 1] = s4.y; sv[i + 2] = s4.z; sv[i + 3] = s4.w;
        }
        {
          // 1 / s_t of token 32 x + lane (0 past the end), for the normaliser below
          const float s_me = scales[st * kTS + 32 * x + lane];
          s_inv[lane] = (d.p0 + (int)j) * kTS + 32 * x + lane < d.L && s_me > 0.f ? fast_rcp(s_me) : 0.f;
        }
        const bool all_valid = tok0 + 16 <= d.L;  // (warp-uniform per lane half) no token past the end
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const bool valid = all_valid || tok0 + i < d.L;
          if (!valid) sv[i] = 0.f;
          v[i] = valid ? v[i] * cq * sv[i] : kNegInf;  // z in log2 units
          mt = fmaxf(mt, v[i]);
          smx = fmaxf(smx, sv[i]);
        }
        mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 16));
        smx = fmaxf(smx, __shfl_xor_sync(0xffffffffu, smx, 16));
        if (lane < 16) s_x[(sb * 2 + x) * kTH + h] = mt;
        if (lane == 0) s_smx[(sb * 2 + x) * 4 + q] = smx;  // the same for every head
      }
      if (bar_or(2 + q, 64, fail)) {
        fail = true;
        break;
      }
      {
        // the other half of the page
        mt = fmaxf(mt, s_x[(sb * 2 + (x ^ 1)) * kTH + h]);
        smx = fmaxf(smx, s_smx[(sb * 2 + (x ^ 1)) * 4 + q]);
      }
      // the previous page's rescale hand-off, before this page's
      // probabilities, so that a page held back by it waits as little as
      // possible (every warp of this page's lane quarter is past page j - 1)
      if (j > 1) rescale_check(g + j - 1, fail);
      const float s_new = smx > 2.f * s_ref ? smx : s_ref;
      const float m_new = mt > m + kTheta ? mt : m;
      const float alpha = fast_exp2(m - m_new);
      const bool resc = j > 0 && (m_new != m || s_new != s_ref);
      if (j > 0 && x == 0 && lane < 16) s_beta[sb * kTH + h] = alpha * (s_ref / s_new);
      if (__any_sync(0xffffffffu, resc) && x == 0 && lane == 0) resc_tag[sb] = gp + 1u;
      l *= alpha;
      m = m_new;
      s_ref = s_new;
      // P'' = 2^(z - m) (s_t / s_ref) 2^kPExp as three or four 8-bit terms
      // (four when the page holds large values: smx is the same in every
      // softmax warp, so they all choose alike).  l sums the weights exactly
      // as the terms carry them (the represented P'' divided by
      // (s_t / s_ref) 2^kPExp), so that the output is a weighted mean of the
      // value rows with the weights the PV product used: a dominant token's
      // rounding cancels against its own share of l, and a weight too small
      // for the terms drops out of both.
      const bool four = smx * 448.f > kFourTermAt;
      if (wt == 0) four_flag[sb] = four ? 1u : 0u;  // read by the PV issuers after p_full
      const float w = exp2f(kPExp) / s_ref;
      __syncwarp();  // s_inv
      float inv[16];
#pragma unroll
      for (int i = 0; i < 16; i += 4) {
        const float4 r4 = *reinterpret_cast<const float4 *>(&s_inv[16 * half + i]);
        inv[i] = r4.x; inv[i + 1] = r4.y; inv[i + 2] = r4.z; inv[i + 3] = r4.w;
      }
      uint32_t t1[8], t2[8], t3[8], t4[8];
      float lp = 0.f;  // this page's share of l, times w
#pragma unroll
      for (int i = 0; i < 16; i += 2) {
        const float2 rep = p_terms2(fast_exp2(v[i] - m) * (sv[i] * w), fast_exp2(v[i + 1] - m) * (sv[i + 1] * w),
                                    four, t1[i / 2], t2[i / 2], t3[i / 2], t4[i / 2]);
        lp = fmaf(rep.x, inv[i], fmaf(rep.y, inv[i + 1], lp));
      }
      l = fmaf(lp, s_ref * exp2f(-kPExp), l);
      uint8_t *pt = pbase + sb * kPBuf + p_off;
      *reinterpret_cast<uint4 *>(pt) =
          make_uint4(t1[0] | (t1[1] << 16), t1[2] | (t1[3] << 16), t1[4] | (t1[5] << 16), t1[6] | (t1[7] << 16));
      *reinterpret_cast<uint4 *>(pt + kPTerm) =
          make_uint4(t2[0] | (t2[1] << 16), t2[2] | (t2[3] << 16), t2[4] | (t2[5] << 16), t2[6] | (t2[7] << 16));
      *reinterpret_cast<uint4 *>(pt + 2 * kPTerm) =
          make_uint4(t3[0] | (t3[1] << 16), t3[2] | (t3[3] << 16), t3[4] | (t3[5] << 16), t3[6] | (t3[7] << 16));
      if (four)
        *reinterpret_cast<uint4 *>(pt + 3 * kPTerm) =
            make_uint4(t4[0] | (t4[1] << 16), t4[2] | (t4[3] << 16), t4[4] | (t4[5] << 16), t4[6] | (t4[7] << 16));
      fence_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&B.p_full[sb]);
    }
    if (n > 1) rescale_check(g + n - 1, fail);  // the item's last page
    if (wg_bar_or(fail)) break;
    // ---- the next item's query, as soon as this item's last QK^T has read
    // the operand, so that the next item's first QK^T overlaps the read-out
    // below
    {
      const uint32_t nslot = (it + 1) % kNIQ;
      fail = !mbar_wait(&B.item_full[nslot], ((it + 1) / kNIQ) & 1u, abort_flag);
      if (wg_bar_or(fail)) break;
      const int b_next = items[nslot].b;
      if (b_next >= 0) {
        const uint32_t ring_next = items[nslot].ring;
        fail = __any_sync(0xffffffffu, !mbar_wait(B.q_empty, it & 1u, abort_flag));  // warp-uniform
        if (!fail) cq_next = q_take(smem, ring_next, B.full, B.q_ready, tq, wt, h, abort_flag, fail);
        if (wg_bar_or(fail)) break;
        q_release(B, ring_next, wt);
      }
    }
    // ---- the item's result: wait for its last PV and its status
    const uint32_t gl = g + n - 1;
    fail = !mbar_wait(&B.p_empty[gl & 1u], (gl >> 1) & 1u, abort_flag) ||
           !mbar_wait(&B.item_done[slot], (it / kNIQ) & 1u, abort_flag);
    const float l_half = l + __shfl_xor_sync(0xffffffffu, l, 16);
    if (lane < 16) {
      s_l[x * kTH + h] = l_half;
      if (x == 0) s_m[h] = m;
    }
    if (wg_bar_or(fail)) break;
    tc_fence_after();
    const uint32_t stv = item_status[slot];
    const float oscale = s_ref * exp2f(-kPExp);  // O^T accumulates 2^(z - m) (s_t / s_ref) 2^kPExp * code
#pragma unroll 1
    for (int c = 4 * x; c < 4 * x + 4; ++c) {
      uint32_t r[32];
      tmem_ld32(tq + kColO + 32 * c, r);
      const int dd = 128 * (c >> 1) + 32 * q + lane;  // value index of this thread's row
      const int h0 = 32 * (c & 1);
      if (d.nb == 1) {
        float *o = a.out + ((size_t)d.b * kTH + h0) * kTDv + dd;
#pragma unroll
        for (int i = 0; i < 32; ++i)
          o[(size_t)i * kTDv] = stv ? 0.f : __uint_as_float(r[i]) * oscale / (s_l[h0 + i] + s_l[kTH + h0 + i]);
      } else {
        float *o = a.part_o + ((size_t)d.cg * kTH + h0) * kTDv + dd;
#pragma unroll
        for (int i = 0; i < 32; ++i) o[(size_t)i * kTDv] = __uint_as_float(r[i]) * oscale;
      }
    }
    if (d.nb != 1 && wt < kTH) a.part_ml[(size_t)d.cg * kTH + wt] = make_float2(s_m[wt], s_l[wt] + s_l[kTH + wt]);
    if (wt == 0) a.part_st[d.cg] = stv;  // the merge ORs the pieces' bits into the request's status
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(B.o_empty);
    named_bar_sync(1, kSmxThreads);  // the scratch is reused by the next item
    if (wt == 0) mbar_arrive(&B.item_empty[slot]);
    cq = cq_next;
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
      mbar_init(&B.empty[i], 2);  // a commit from each PV issuer
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&B.s_full[i], 1);
      mbar_init(&B.s_empty[i], kSmxThreads / 32);
      mbar_init(&B.p_full[i], kSmxThreads / 32);
      mbar_init(&B.p_empty[i], 2);  // a commit from each PV issuer
    }
    mbar_init(B.q_ready, kSmxThreads / 32);
    mbar_init(B.q_empty, 1);
    mbar_init(B.o_empty, kSmxThreads / 32);
    mbar_init(B.r_done, kSmxThreads / 32);
    mbar_init(B.drain, 3);  // one commit from each MMA issuer
    for (int i = 0; i < kNIQ; ++i) {
      mbar_init(&B.item_full[i], 1);
      mbar_init(&B.item_empty[i], 4);  // the three MMA threads and the softmax warps
      mbar_init(&B.item_done[i], 1);
    }
    uint32_t *tag = reinterpret_cast<uint32_t *>(smem + sp.wg) + kWgTag;
    tag[0] = tag[1] = 0u;
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
    if (lane == 0) tc_mma_qk(smem, B, items, tmem, abort_flag);
    __syncwarp();
  } else if (warp == 6 || warp == 7) {
    if (lane == 0) tc_mma_pv(smem, B, items, tmem, abort_flag, warp - 6);
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
  // Whether a wait gave up somewhere in this block; the merge then reports
  // every request of the call as timed out (its output is not valid).
  if (threadIdx.x == 0) a.cta_abort[blockIdx.x] = *abort_flag != 0;
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
  // Work items are pieces of a request, all 64 heads each.
  DecodeArgs a = a0;
  a.Hkv = 1;
  a.G = kTH;
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
  // One CTA per SM, each taking one range of the requests' pages (no plan
  // kernel); small or lopsided batches fall back to chunks of at least 8
  // pages, about two per CTA.
  const int grid = min(num_sms(), kMaxCtas);
  a.ranges = grid;
  a.n_ctas = grid;
  a.target_items = 2 * grid;
  a.min_chunk_pages = 8;
  a.piece_cost = kPieceCostLatent;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  // the query terms of every request (one block per request and 16 heads)
  cudaLaunchConfig_t qcfg = {};
  qcfg.gridDim = dim3(a.B * 4);
  qcfg.blockDim = dim3(256);
  qcfg.stream = s;
  qcfg.attrs = attr;
  qcfg.numAttrs = 1;
  rc = cuda_ok(cudaLaunchKernelEx(&qcfg, qterm_kernel, a), "query-term kernel launch");
  if (rc) return rc;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kTThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  rc = cuda_ok(cudaLaunchKernelEx(&cfg, latent_tc_kernel, map, map_tail, a), "latent kernel launch");
  if (rc) return rc;
  // status of every request, and the merge of requests cut into several
  // pieces, in blocks of 16 heads
  DecodeArgs m = a;
  m.Hkv = kTH / 16;  // four groups of 16 query heads, all on the one stream
  m.kv_sub = kTH / 16;
  m.G = kTH;
  m.Gs = 16;
  cudaLaunchConfig_t mcfg = {};
  mcfg.gridDim = dim3(a.B * m.Hkv, merge_col_blocks<kTDv, 16>());
  mcfg.blockDim = dim3(256);
  mcfg.stream = s;
  mcfg.attrs = attr;
  mcfg.numAttrs = 1;
  return cuda_ok(cudaLaunchKernelEx(&mcfg, merge_kernel<kTDv, 16>, m), "merge kernel launch");
}

}  // namespace pfkv
