// decode_gqa.cu -- split-KV paged decode attention for grouped-query heads
// (head_dim 64/128, any group size: groups above 8 heads run as head groups
// of up to 8) over an FP8 e4m3 or a BF16 paged cache.
//
// "Smaller, faster, safer: running Kimi and GLM at scale", section
// "Quantizing the KV cache": the cache is FP8 e4m3 and the attention kernel
// converts the values as it reads them.  Cache-protection passage: each
// page's tag is compared with the mapping's tag before its data may be
// returned; a mismatch aborts the request.
//
// Kernels (both on the caller's stream; no plan kernel):
//   1. split  -- persistent CTAs, one producer warp + NCW consumer warps.
//                Each CTA works out its own pieces from the lengths (see
//                "work split" below): CTA k * Hkv + h takes page range k of
//                the requests' concatenated pages for KV head h.  The
//                producer walks a piece's page-table entries 32 at a time,
//                bounds-checks every page id before any fetch, compares tags
//                off the critical path (the tag load is issued next to the
//                page copy; a mismatch only sets the piece's status bits),
//                and stages whole (page, head) K and V slices into a
//                shared-memory ring with TMA tensor copies (128-byte
//                swizzle).  Consumer warps take 16-token tiles: e4m3 -> f16
//                in registers (exact), QK^T and PV on register-operand
//                tensor-core MMA, online softmax in fp32.  A piece that
//                covers a whole request writes its output directly;
//                otherwise it leaves an unnormalised partial (m, l, O).
//   2. merge  -- one CTA per (request, head group, block of 64 -- or, for
//                small grids, 16 -- float4 columns; merge.cuh): writes
//                each request's status (the bits its pieces found, a bad
//                length, or a timeout anywhere in the split grid), zeroes
//                the rows of a faulted request, and
//                merges the partials of a request cut into several pieces
//                by the log-sum-exp rule, split weights staged in shared
//                memory and splits spread over thread groups.
//   A request with a data-fault bit gets zero output.  The merge is a
//   programmatic dependent of the split kernel, so its launch and prologue
//   overlap the split's tail.  The split kernel is launched the same way,
//   but a previous call's merge releases it only when it has finished:
//   split CTAs placed beside running merge CTAs slowed back-to-back calls.
#include <math.h>

#include <mutex>

#include "decode_common.cuh"
#include "merge.cuh"

namespace pfkv {

namespace {

// ---------------------------------------------------------------- split

template <bool kFp8, int kD, int kG, int kNCW>
struct Cfg {
  static constexpr int kEsz = kFp8 ? 1 : 2;
  static constexpr int kRowBytes = kD * kEsz;       // 64, 128 or 256
  static constexpr bool kSwz = kRowBytes >= 128;    // 64-byte rows are read conflict-free unswizzled
  static constexpr int kKsteps = kD / 16;           // QK^T k-steps; also PV m-tiles
  static constexpr int kSegK = kD / 4 * kEsz;       // bytes of a K row held by one thread
  static constexpr int kSegV = kD / 8 * kEsz;       // bytes of a V row held by one thread
  static constexpr int kNP = (2 * kG + 7) / 8;      // PV n-tiles (hi and lo columns)
  static constexpr int kThreads = (kNCW + 1) * 32;
  static constexpr int kMinBlocks = (kG == 8 && kD == 128) ? 2 : 3;  // register budget per thread
  static constexpr float kPScale = kFp8 ? 16384.0f : 1.0f;  // keeps f16 P away from subnormals
};

struct SmemPlan {
  uint32_t stage_bytes, page_bytes, stages_off, bars_off, items_off, merge_off, total;
};

__host__ __device__ inline SmemPlan smem_plan(int S, int row_bytes, bool per_token, int nst, int ncw, int G, int D) {
  SmemPlan p;
  p.page_bytes = 2u * S * row_bytes + (per_token ? 8u * S : 0u);
  p.stage_bytes = (p.page_bytes + 1023u) & ~1023u;
  p.stages_off = 0;
  p.bars_off = p.stages_off + p.stage_bytes * nst;
  p.items_off = p.bars_off + 8u * (2 * nst + 3 * kNIQ) + 16u;  // + abort flag
  p.merge_off = (p.items_off + (sizeof(ItemDesc) + 4u) * kNIQ + 15u) & ~15u;
  p.total = p.merge_off + 4u * ncw * (2 * G + G * D) + 4u * (2 * G + 4) + 1024u;  // + alignment slack
  return p;
}

template <bool kFp8>
__device__ __forceinline__ void mma_t(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  if constexpr (kFp8) mma_f16(d, a, b0, b1);
  else mma_bf16(d, a, b0, b1);
}

template <bool kFp8>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  if constexpr (kFp8) return pack_f16x2(lo, hi);
  else return pack_bf16x2(lo, hi);
}

template <bool kFp8>
__device__ __forceinline__ float round16(float x) {
  if constexpr (kFp8) return __half2float(__float2half_rn(x));
  else return __bfloat162float(__float2bfloat16_rn(x));
}

// Decode step, producer warp: the new token of (request, KV head g) goes to
// slot `slot` of page `pid`, unless that page is out of range or (tag check
// on) its tag does not match (`refused`, the same on every lane); the walk
// reports those cases in the request's status as for any page.  Quantized
// as the append does (x / s, RNE, satfinite; per-token s = amax / 448, or 1
// for an all-zero row).  Whole warp.  The caller fences the stores for the
// tensor-copy engine (proxy fence) before it copies the page.
template <bool kFp8, int kD>
__device__ __forceinline__ void store_new_row(const DecodeArgs &a, uint4 v, float s, bool has, int part, int k, int pid,
                                              bool refused, int g, int slot, bool per_token) {
  if (refused) return;
  const size_t row = ((size_t)pid * a.cache.num_kv_heads + g) * a.S + slot;
  if constexpr (kFp8) {
    if (per_token) {
      float amax = amax8(v, 0.f);  // lanes without values hold zeros
#pragma unroll
      for (int o = 8; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
      s = amax > 0.f ? __fdiv_rn(amax, 448.0f) : 1.0f;
      if (has && k == 0) (part ? a.cache.v_scale : a.cache.k_scale)[row] = s;
    }
    if (has)
      *reinterpret_cast<uint2 *>(reinterpret_cast<uint8_t *>(part ? a.cache.v_pool : a.cache.k_pool) + row * kD + k) =
          e4m3x8(v, s);
  } else {
    if (has) *reinterpret_cast<uint4 *>(reinterpret_cast<uint16_t *>(part ? a.cache.v_pool : a.cache.k_pool) + row * kD + k) = v;
  }
}

// Bounded wait that ignores the abort flag: the page loader's way out, so
// that a block that gave up still lets its own copies land before it exits.
__device__ __forceinline__ void drain_wait_full(uint64_t *bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity))
    if (global_timer_ns() - t0 > kWaitLimitNs) return;
}

template <bool kFp8, int kD, int kG, int kNCW>
__global__ void __launch_bounds__(Cfg<kFp8, kD, kG, kNCW>::kThreads, Cfg<kFp8, kD, kG, kNCW>::kMinBlocks)
    gqa_split_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                     const DecodeArgs a, const int nst) {
  using C = Cfg<kFp8, kD, kG, kNCW>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const bool per_token = kFp8 && a.scale_mode == PFKV_SCALE_PER_TOKEN;
  const SmemPlan sp = smem_plan(a.S, C::kRowBytes, per_token, nst, kNCW, kG, kD);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + sp.bars_off);
  uint64_t *empty = full + nst;
  uint64_t *item_full = empty + nst;
  uint64_t *item_empty = item_full + kNIQ;
  uint64_t *item_done = item_empty + kNIQ;  // the producer finished the item's page walk
  volatile int *abort_flag = reinterpret_cast<volatile int *>(item_done + kNIQ);
  ItemDesc *items = reinterpret_cast<ItemDesc *>(smem + sp.items_off);
  uint32_t *item_status = reinterpret_cast<uint32_t *>(items + kNIQ);  // status bits found by the walk
  float *sm_m = reinterpret_cast<float *>(smem + sp.merge_off);  // [NCW][G]
  float *sm_l = sm_m + kNCW * kG;                                 // [NCW][G]
  float *sm_o = sm_l + kNCW * kG;                                 // [NCW][G][D]
  float *sm_fin = sm_o + kNCW * kG * kD;                          // [G] (m, l) of the item
  volatile int *sm_ctl = reinterpret_cast<volatile int *>(sm_fin + 2 * kG);  // [4] broadcast words

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = a.S, mpp = S / 16;  // 16-token tiles per page

  if (threadIdx.x == 0) {
    for (int i = 0; i < nst; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], mpp);
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
  pdl_wait();  // the kernel before this one (the previous call's merge) is complete from here on
  pdl_launch_dependents();  // the merge kernel may be scheduled; it waits for this grid to finish

  if (warp == kNCW) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
    }
    const bool tag_check = (a.flags & PFKV_FLAG_TAG_CHECK) != 0u;
    const uint64_t stream_pol = l2_evict_first_policy();
    // Pages of one batch are issued by separate lanes at once.  A batch never
    // holds more pages than the ring has stages, so no two lanes of a batch
    // share a stage and every empty-barrier wait is for the stage's previous
    // use only (no parity aliasing).
    const int batch_pages = min(32, nst);
    uint32_t ring = 0;
    // This CTA's pieces for KV head g, worked out from the lengths; the next
    // piece is found once the current one's pages have gone out.
    // this CTA's head group: virtual KV head vg, which reads KV head g (a KV
    // head whose query heads are cut into several groups is read by one CTA
    // of each group; every one of them writes a decode step's new row, the
    // same bytes, before its own copy of the page)
    const int vg = (int)blockIdx.x % a.Hkv;
    const int g = vg / a.kv_sub;
    __shared__ WorkSplit s_ws;
    const WsArgs wa = ws_args(a);
    {
      WorkSplit w;
      ws_init(w, wa, lane);
      if (lane == 0) s_ws = w;
      __syncwarp();
    }
    Piece cur;
    bool have = ws_next_shared(s_ws, wa, cur, lane);
    // the last batch's first ring position, and whether this lane's page of
    // it was issued (every page of earlier batches was)
    uint32_t last_first = 0;
    bool last_issued = false;
    for (uint32_t iq = 0;; ++iq) {
      const uint32_t slot = iq % kNIQ;
      bool ok = true;
      if (lane == 0) ok = mbar_wait(&item_empty[slot], ((iq / kNIQ) & 1u) ^ 1u, abort_flag);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      // test hook (PFKV_FLAG_TEST_WITHHOLD): the first CTA never hands its
      // first item (or its end marker) to the consumers, whose bounded wait
      // then gives up
      const bool withhold = (a.flags & PFKV_FLAG_TEST_WITHHOLD) && blockIdx.x == 0 && iq == 0;
      if (!have) {
        if (lane == 0) {
          items[slot].b = -1;
          if (!withhold) mbar_arrive(&item_full[slot]);
        }
        break;
      }
      const int b = cur.b, p0 = cur.p0, p1 = cur.p1, L = cur.L;
      if (lane == 0) {
        ItemDesc d;
        d.b = b; d.cg = cur.cg; d.g = vg; d.p0 = p0; d.p1 = p1; d.L = L; d.ring = ring; d.nb = cur.nb;
        items[slot] = d;
        if (!withhold) mbar_arrive(&item_full[slot]);
        if (vg == 0 && cur.lead) {  // the merge's view of the numbering
          a.split_first[b] = cur.cg;
          a.split_count[b] = cur.nb;
        }
      }
      const int *trow = a.block_table + (size_t)b * a.MP;
      const uint32_t *tagrow = a.block_tags + (size_t)b * a.MP;
      uint32_t st_bits = 0;
      // Decode step: the item holding the request's last page writes the new
      // token's K and V rows of head g into that page before copying it.
      // Lanes 0-15 hold 8 values each of the K row, lanes 16-31 of the V row,
      // loaded now so that their latency hides behind the walk.
      const int i_new = (L - 1) / S;
      const bool has_new = a.append && p0 <= i_new && i_new < p1;
      const int nv_part = lane >> 4, nv_k = (lane & 15) * 8;
      const bool nv_lane = has_new && nv_k < kD;
      uint4 nv = make_uint4(0u, 0u, 0u, 0u);
      float nv_scale = 1.f;
      if (nv_lane) {
        nv = *reinterpret_cast<const uint4 *>((nv_part ? a.v_new : a.k_new) +
                                              ((size_t)b * a.cache.num_kv_heads + g) * kD + nv_k);
        if (kFp8 && !per_token) nv_scale = __ldg(&(nv_part ? a.v_scale : a.k_scale)[g]);
      }
      // ... and the destination page's id, loaded now as well: the row is
      // stored as soon as the first batch's copies are out (before them if
      // the destination is in that batch), off the path of the destination
      // batch, which only fences the stores before its copies
      const int pid_new = has_new ? __ldg(&trow[i_new]) : 0;
      bool row_stored = !has_new;
      auto store_row = [&]() {  // whole warp
        bool bad = pid_new < 0 || pid_new >= a.P;
        if (tag_check && !bad) bad = __ldg(&a.page_tags[pid_new]) != __ldg(&tagrow[i_new]);
        store_new_row<kFp8, kD>(a, nv, nv_scale, nv_lane, nv_part, nv_k, pid_new, bad, g, (L - 1) % S, per_token);
        row_stored = true;
      };
      int kb = 0;  // batch number within the piece
      for (int i0 = p0; i0 < p1 && ok; i0 += batch_pages, ++kb) {
        last_first = ring;
        const int i = i0 + lane;
        const bool valid = lane < batch_pages && i < p1;
        const int pid = valid ? __ldg(&trow[i]) : 0;
        const bool oob = valid && (pid < 0 || pid >= a.P);
        uint32_t page_tag = 0, want_tag = 0;
        // Tags: every head group of a page range walks the same pages, so each
        // batch's tags are checked by one of them, in turn (batch kb of piece
        // cg by head group (cg + kb) mod Hkv); each group reports what it
        // found in its own status word of the piece, and the merge ORs them.
        // A decode step's destination page is checked by every group (each
        // decides the refusal of its own rows).
        const bool dest_batch = has_new && i0 <= i_new && i_new < i0 + batch_pages;
        const bool my_batch = (int)(((unsigned)cur.cg + (unsigned)kb) % (unsigned)a.Hkv) == vg;
        if (tag_check && (my_batch || dest_batch) && valid && !oob) {  // issued now, compared after the copies
          page_tag = __ldg(&a.page_tags[pid]);
          want_tag = __ldg(&tagrow[i]);
        }
        if (dest_batch) {
          if (!row_stored) store_row();
          asm volatile("fence.proxy.async.global;" ::: "memory");
          __syncwarp();
        }
        bool lane_ok = true;
        if (valid) {
          const uint32_t r = ring + (uint32_t)lane;
          const uint32_t st = r % (uint32_t)nst;
          lane_ok = mbar_wait(&empty[st], ((r / (uint32_t)nst) & 1u) ^ 1u, abort_flag);
          if (lane_ok) {
            uint8_t *stage = smem + sp.stages_off + (size_t)st * sp.stage_bytes;
            if (oob) {
              mbar_arrive(&full[st]);  // never fetched; the request is aborted
            } else {
              mbar_arrive_expect_tx(&full[st], sp.page_bytes);
              if constexpr (C::kRowBytes == 256) {
                tma_load_5d_stream(stage, &tmK, &full[st], 0, 0, 0, g, pid, stream_pol);
                tma_load_5d_stream(stage + S * C::kRowBytes, &tmV, &full[st], 0, 0, 0, g, pid, stream_pol);
              } else {
                tma_load_4d_stream(stage, &tmK, &full[st], 0, 0, g, pid, stream_pol);
                tma_load_4d_stream(stage + S * C::kRowBytes, &tmV, &full[st], 0, 0, g, pid, stream_pol);
              }
              if (per_token) {
                const size_t rr = ((size_t)pid * a.cache.num_kv_heads + g) * S;
                bulk_load_stream(stage + 2 * S * C::kRowBytes, a.k_scale + rr, 4u * S, &full[st], stream_pol);
                bulk_load_stream(stage + 2 * S * C::kRowBytes + 4 * S, a.v_scale + rr, 4u * S, &full[st], stream_pol);
              }
            }
          }
        }
        if (!row_stored) store_row();  // the first batch's copies are out
        ring += (uint32_t)min(batch_pages, p1 - i0);
        last_issued = valid && lane_ok;
        ok = __all_sync(0xffffffffu, lane_ok);
        if (__any_sync(0xffffffffu, oob)) st_bits |= PFKV_ST_PAGE_OOB;
        if (__any_sync(0xffffffffu, page_tag != want_tag)) st_bits |= PFKV_ST_STALE_TAG;
      }
      if (lane == 0) {
        item_status[slot] = st_bits;  // read by the consumers when they finish the item
        mbar_arrive(&item_done[slot]);
      }
      if (!ok) break;
      have = ws_next_shared(s_ws, wa, cur, lane);
    }
    // Copies still in flight land before the block may exit (the consumers
    // wait for every page they use, but on the abort path they leave early):
    // lane k waits for the k-th of the last nst pages issued.
    if (__shfl_sync(0xffffffffu, (int)(*abort_flag != 0), 0)) {
      const bool have = lane < nst && ring >= (uint32_t)(nst - lane);
      const uint32_t r = ring - (uint32_t)nst + (uint32_t)lane;  // meaningful when have
      const bool in_last = have && r >= last_first;            // then r - last_first < batch_pages
      const bool src_issued = __shfl_sync(0xffffffffu, last_issued, in_last ? (int)(r - last_first) : 0);
      if (have && (!in_last || src_issued)) drain_wait_full(&full[r % (uint32_t)nst], (r / (uint32_t)nst) & 1u);
    }
  } else {
    // ------------------------------------------------------------ consumers
    const int gid = lane >> 2, tq = lane & 3;
    constexpr int kSrcMask = (kG == 4) ? 1 : 0;  // PV column -> QK column owner
    const int src_lane = (lane & ~3) | (tq & kSrcMask);
    // Shared-memory offsets of this thread's fragments inside a 16-row tile.
    // Tiles start at multiples of 16 rows, which leaves the 128-byte swizzle
    // pattern unchanged, so the offsets are computed once.
    constexpr int kKC = C::kSegK / 16;                 // 16-byte chunks of a K row segment
    constexpr int kVC = C::kSegV >= 16 ? C::kSegV / 16 : 1;
    uint32_t koff[2][kKC], voff[4][kVC];
#pragma unroll
    for (int r = 0; r < 2; ++r)
#pragma unroll
      for (int c = 0; c < kKC; ++c) {
        const uint32_t off = (uint32_t)(gid + 8 * r) * C::kRowBytes + tq * C::kSegK + 16 * c;
        koff[r][c] = C::kSwz ? swz128(off) : off;
      }
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int trow = 2 * tq + (r & 1) + 8 * (r >> 1);
#pragma unroll
      for (int c = 0; c < kVC; ++c) {
        const uint32_t off = (uint32_t)trow * C::kRowBytes + gid * C::kSegV + 16 * c;
        voff[r][c] = C::kSwz ? swz128(off) : off;
      }
    }
    const uint32_t smem_base = smem_addr(smem + sp.stages_off);

    for (uint32_t iq = 0;; ++iq) {
      const uint32_t slot = iq % kNIQ;
      if (!__all_sync(0xffffffffu, mbar_wait(&item_full[slot], (iq / kNIQ) & 1u, abort_flag))) break;
      const ItemDesc d = items[slot];
      if (d.b < 0) break;

      // query fragments of the group's heads (row gid of the B operand; rows
      // past the group's heads are padding, zero)
      const HeadGroup hg = head_group(a, d.g);
      uint32_t qf[C::kKsteps][2];
      float mult[2];
      {
        const int h = hg.first + gid;
        float qv[kD / 4];
        if (gid < hg.count) {
          const uint4 *src = reinterpret_cast<const uint4 *>(reinterpret_cast<const __nv_bfloat16 *>(a.q) +
                                                              ((size_t)d.b * a.Hq + h) * kD + tq * (kD / 4));
#pragma unroll
          for (int c = 0; c < kD / 32; ++c) {
            const uint4 v = __ldg(&src[c]);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              qv[c * 8 + 2 * k] = __uint_as_float(w[k] << 16);
              qv[c * 8 + 2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
            }
          }
        } else {
#pragma unroll
          for (int k = 0; k < kD / 4; ++k) qv[k] = 0.f;
        }
        int e = 0;
        if constexpr (kFp8) {
          // exact bf16 -> f16: scale the head by 2^e so that max|q| lands in [2^14, 2^15)
          float mx = 0.f;
#pragma unroll
          for (int k = 0; k < kD / 4; ++k) mx = fmaxf(mx, fabsf(qv[k]));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
          if (mx > 0.f) {
            int k2;
            frexpf(mx, &k2);
            e = 15 - k2;
          }
        }
#pragma unroll
        for (int s = 0; s < C::kKsteps; ++s) {
          if constexpr (kFp8) {
            qf[s][0] = pack_f16x2(ldexpf(qv[4 * s], e), ldexpf(qv[4 * s + 1], e));
            qf[s][1] = pack_f16x2(ldexpf(qv[4 * s + 2], e), ldexpf(qv[4 * s + 3], e));
          } else {
            qf[s][0] = pack_bf16x2(qv[4 * s], qv[4 * s + 1]);
            qf[s][1] = pack_bf16x2(qv[4 * s + 2], qv[4 * s + 3]);
          }
        }
        float base = a.sm_scale_log2;
        if (kFp8 && !per_token) base *= __ldg(&a.k_scale[hg.kv]);
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int ec = __shfl_sync(0xffffffffu, e, ((2 * tq + c) & 7) * 4);
          mult[c] = ldexpf(base, -ec);
        }
      }

      float m[2] = {kNegInf, kNegInf}, l[2] = {0.f, 0.f};
      float o[C::kKsteps][C::kNP][4];
#pragma unroll
      for (int i = 0; i < C::kKsteps; ++i)
#pragma unroll
        for (int j = 0; j < C::kNP; ++j)
#pragma unroll
          for (int k = 0; k < 4; ++k) o[i][j][k] = 0.f;

      const int n_mt = (d.p1 - d.p0) * mpp;
      bool alive = true;
      // Each iteration takes two consecutive 16-token tiles of the item.
      for (int jp = warp; 2 * jp < n_mt; jp += kNCW) {
        uint32_t stg[2], tbase[2];
        bool valid[2], live[2];
        int tok_base[2];
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          const int j = 2 * jp + t;
          valid[t] = j < n_mt;
          const int page_local = j / mpp, mt_in_page = j - page_local * mpp;
          const uint32_t rp = d.ring + (uint32_t)page_local;
          stg[t] = rp % (uint32_t)nst;
          if (valid[t] && !mbar_wait(&full[stg[t]], (rp / (uint32_t)nst) & 1u, abort_flag)) alive = false;
          tok_base[t] = (d.p0 + page_local) * S + mt_in_page * 16;
          live[t] = valid[t] && tok_base[t] < d.L;
          tbase[t] = smem_base + stg[t] * sp.stage_bytes + (uint32_t)(mt_in_page * 16 * C::kRowBytes);
        }
        alive = __all_sync(0xffffffffu, alive);  // the whole warp leaves together
        if (!alive) break;
        // ---- S = K q^T for both tiles
        float z[2][4];
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          float sacc[4] = {0.f, 0.f, 0.f, 0.f};
          if (live[t]) {
            uint32_t wk[2][C::kSegK / 4];
#pragma unroll
            for (int r = 0; r < 2; ++r)
#pragma unroll
              for (int c = 0; c < kKC; ++c) {
                const uint4 v = lds128(tbase[t] + koff[r][c]);
                wk[r][4 * c] = v.x; wk[r][4 * c + 1] = v.y; wk[r][4 * c + 2] = v.z; wk[r][4 * c + 3] = v.w;
              }
#pragma unroll
            for (int s = 0; s < C::kKsteps; ++s) {
              uint32_t af[4];
              if constexpr (kFp8) {
                e4m3x4_to_f16x4(wk[0][s], af[0], af[2]);
                e4m3x4_to_f16x4(wk[1][s], af[1], af[3]);
              } else {
                af[0] = wk[0][2 * s];
                af[1] = wk[1][2 * s];
                af[2] = wk[0][2 * s + 1];
                af[3] = wk[1][2 * s + 1];
              }
              mma_t<kFp8>(sacc, af, qf[s][0], qf[s][1]);
            }
          }
          z[t][0] = sacc[0] * mult[0]; z[t][1] = sacc[1] * mult[1];
          z[t][2] = sacc[2] * mult[0]; z[t][3] = sacc[3] * mult[1];
          if (per_token && live[t]) {
            const uint32_t sks = smem_base + stg[t] * sp.stage_bytes + 2 * S * C::kRowBytes +
                                 4 * ((tok_base[t] - (tok_base[t] / S) * S) + gid);
            const float k0 = lds_f32(sks), k1 = lds_f32(sks + 32);
            z[t][0] *= k0; z[t][1] *= k0; z[t][2] *= k1; z[t][3] *= k1;
          }
          if (!live[t] || tok_base[t] + gid >= d.L) z[t][0] = z[t][1] = kNegInf;
          if (!live[t] || tok_base[t] + gid + 8 >= d.L) z[t][2] = z[t][3] = kNegInf;
        }
        // ---- online softmax over the 32 tokens (log2 domain)
        float mx0 = fmaxf(fmaxf(z[0][0], z[0][2]), fmaxf(z[1][0], z[1][2]));
        float mx1 = fmaxf(fmaxf(z[0][1], z[0][3]), fmaxf(z[1][1], z[1][3]));
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
          mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
          mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
        }
        const float mn0 = fmaxf(m[0], mx0), mn1 = fmaxf(m[1], mx1);
        const float al0 = fast_exp2(m[0] - mn0), al1 = fast_exp2(m[1] - mn1);
        const bool moved = __any_sync(0xffffffffu, (mn0 != m[0]) | (mn1 != m[1]));
        m[0] = mn0;
        m[1] = mn1;
        float p[2][4];
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          p[t][0] = fast_exp2(z[t][0] - mn0); p[t][1] = fast_exp2(z[t][1] - mn1);
          p[t][2] = fast_exp2(z[t][2] - mn0); p[t][3] = fast_exp2(z[t][3] - mn1);
        }
        l[0] = l[0] * al0 + (p[0][0] + p[0][2]) + (p[1][0] + p[1][2]);
        l[1] = l[1] * al1 + (p[0][1] + p[0][3]) + (p[1][1] + p[1][3]);
        if (moved) {  // rescale the accumulators only when some running max moved
          float apv0 = al0, apv1 = al1;
          if constexpr (kG == 1) {
            apv0 = apv1 = __shfl_sync(0xffffffffu, al0, lane & ~3);
          } else if constexpr (kG < 8) {
            apv0 = __shfl_sync(0xffffffffu, al0, src_lane);
            apv1 = __shfl_sync(0xffffffffu, al1, src_lane);
          }
#pragma unroll
          for (int i = 0; i < C::kKsteps; ++i)
#pragma unroll
            for (int nt = 0; nt < C::kNP; ++nt) {
              o[i][nt][0] *= apv0; o[i][nt][1] *= apv1; o[i][nt][2] *= apv0; o[i][nt][3] *= apv1;
            }
        }
        // ---- O^T += V^T P^T, one 16-token k-step per tile
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          if (!live[t]) continue;
          // PV columns: v = 8*nt + 2*tq + e -> head v % G; hi part for v < G, lo part for G <= v < 2G
          float pv[4] = {p[t][0], p[t][1], p[t][2], p[t][3]};
          if constexpr (kG == 1) {
            pv[0] = pv[1] = __shfl_sync(0xffffffffu, p[t][0], lane & ~3);
            pv[2] = pv[3] = __shfl_sync(0xffffffffu, p[t][2], lane & ~3);
          } else if constexpr (kG < 8) {
#pragma unroll
            for (int k = 0; k < 4; ++k) pv[k] = __shfl_sync(0xffffffffu, p[t][k], src_lane);
          }
          float vs0 = 1.f, vs1 = 1.f;
          if (per_token) {
            const uint32_t svs = smem_base + stg[t] * sp.stage_bytes + 2 * S * C::kRowBytes + 4 * S +
                                 4 * ((tok_base[t] - (tok_base[t] / S) * S) + gid);
            vs0 = lds_f32(svs);
            vs1 = lds_f32(svs + 32);
          }
          uint32_t pb[C::kNP][2];
#pragma unroll
          for (int nt = 0; nt < C::kNP; ++nt) {
            float val[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const int e = k & 1;
              const int v = 8 * nt + 2 * tq + e;
              const float pp = pv[k] * C::kPScale * ((k < 2) ? vs0 : vs1);
              const float hi = round16<kFp8>(pp);
              const bool lo_part = (kG == 1) ? (e == 1) : (v >= kG);
              val[k] = (v < 2 * kG) ? (lo_part ? pp - hi : hi) : 0.f;
            }
            pb[nt][0] = movmatrix_trans(pack2<kFp8>(val[0], val[1]));
            pb[nt][1] = movmatrix_trans(pack2<kFp8>(val[2], val[3]));
          }
          uint32_t wv[4][C::kSegV / 4];
          const uint32_t vbase = tbase[t] + S * C::kRowBytes;  // V tile follows the K tile in the stage
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            if constexpr (C::kSegV == 8) {
              const uint2 v = lds64(vbase + voff[r][0]);
              wv[r][0] = v.x; wv[r][1] = v.y;
            } else {
#pragma unroll
              for (int c = 0; c < kVC; ++c) {
                const uint4 v = lds128(vbase + voff[r][c]);
                wv[r][4 * c] = v.x; wv[r][4 * c + 1] = v.y; wv[r][4 * c + 2] = v.z; wv[r][4 * c + 3] = v.w;
              }
            }
          }
#pragma unroll
          for (int mt = 0; mt < C::kKsteps; ++mt) {
            uint32_t af[4];
            if constexpr (kFp8) {
              const uint32_t sel = (mt & 1) ? 0x7362u : 0x5140u;
              e4m3x4_to_f16x4(prmt(wv[0][mt >> 1], wv[1][mt >> 1], sel), af[0], af[1]);
              e4m3x4_to_f16x4(prmt(wv[2][mt >> 1], wv[3][mt >> 1], sel), af[2], af[3]);
            } else {
              af[0] = prmt(wv[0][mt], wv[1][mt], 0x5410u);
              af[1] = prmt(wv[0][mt], wv[1][mt], 0x7632u);
              af[2] = prmt(wv[2][mt], wv[3][mt], 0x5410u);
              af[3] = prmt(wv[2][mt], wv[3][mt], 0x7632u);
            }
#pragma unroll
            for (int nt = 0; nt < C::kNP; ++nt) mma_t<kFp8>(o[mt][nt], af, pb[nt][0], pb[nt][1]);
          }
        }
        __syncwarp();
        if (lane == 0) {
          if (valid[0]) mbar_arrive(&empty[stg[0]]);
          if (valid[1]) mbar_arrive(&empty[stg[1]]);
        }
      }
      // ---- per-warp state -> shared memory
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        l[0] += __shfl_xor_sync(0xffffffffu, l[0], off);
        l[1] += __shfl_xor_sync(0xffffffffu, l[1], off);
      }
      if (gid == 0) {
#pragma unroll
        for (int e = 0; e < 2; ++e)
          if (2 * tq + e < kG) {
            sm_m[warp * kG + 2 * tq + e] = m[e];
            sm_l[warp * kG + 2 * tq + e] = l[e];
          }
      }
#pragma unroll
      for (int mt = 0; mt < C::kKsteps; ++mt) {
        float hv[4];
        if constexpr (kG == 8) {
#pragma unroll
          for (int k = 0; k < 4; ++k) hv[k] = o[mt][0][k] + o[mt][1][k];
        } else if constexpr (kG == 1) {
          hv[0] = o[mt][0][0] + o[mt][0][1];
          hv[2] = o[mt][0][2] + o[mt][0][3];
          hv[1] = hv[3] = 0.f;
        } else {
          constexpr int kX = kG / 2;  // lane distance from a lo column to its hi column
#pragma unroll
          for (int k = 0; k < 4; ++k) hv[k] = o[mt][0][k] + __shfl_xor_sync(0xffffffffu, o[mt][0][k], kX);
        }
        const int d0 = gid * (kD / 8) + 2 * mt;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int hh = 2 * tq + e;
          if (hh < kG && !(kG == 1 && e == 1)) {
            sm_o[(warp * kG + hh) * kD + d0] = hv[e];
            sm_o[(warp * kG + hh) * kD + d0 + 1] = hv[2 + e];
          }
        }
      }
      named_bar_sync(1, kNCW * 32);
      // ---- merge the consumer warps' states
      const int t = threadIdx.x;
      constexpr int kCT = kNCW * 32;
      if (t == 0) {
        uint32_t stv = PFKV_ST_TIMEOUT;
        if (mbar_wait(&item_done[slot], (iq / kNIQ) & 1u, abort_flag)) stv = item_status[slot];
        sm_ctl[0] = (int)stv;
      }
      if (t < kG) {
        float M = kNegInf;
#pragma unroll
        for (int w = 0; w < kNCW; ++w) M = fmaxf(M, sm_m[w * kG + t]);
        float ls = 0.f;
#pragma unroll
        for (int w = 0; w < kNCW; ++w) {
          const float mw = sm_m[w * kG + t];
          if (mw != kNegInf) ls += sm_l[w * kG + t] * fast_exp2(mw - M);
        }
        sm_fin[2 * t] = M;
        sm_fin[2 * t + 1] = ls;
      }
      named_bar_sync(1, kCT);
      const uint32_t item_st = (uint32_t)sm_ctl[0];
      float ofac = 1.f;
      if constexpr (kFp8) ofac = (per_token ? 1.f : __ldg(&a.v_scale[hg.kv])) / C::kPScale;
      float *out_bg = a.out + ((size_t)d.b * a.Hq + hg.first) * kD;  // rows of this (request, head group)
      if (d.nb == 1) {
        // the item covers the whole request: finish it here
        for (int idx = t; idx < hg.count * kD; idx += kCT) {
          const int jh = idx / kD, dd = idx - jh * kD;
          const float M = sm_fin[2 * jh];
          float acc = 0.f;
#pragma unroll
          for (int w = 0; w < kNCW; ++w) {
            const float mw = sm_m[w * kG + jh];
            if (mw != kNegInf) acc += sm_o[(w * kG + jh) * kD + dd] * fast_exp2(mw - M);
          }
          out_bg[idx] = item_st ? 0.f : acc * ofac / sm_fin[2 * jh + 1];
        }
      } else {
        for (int idx = t; idx < hg.count * kD; idx += kCT) {
          const int jh = idx / kD, dd = idx - jh * kD;
          const float M = sm_fin[2 * jh];
          float acc = 0.f;
#pragma unroll
          for (int w = 0; w < kNCW; ++w) {
            const float mw = sm_m[w * kG + jh];
            if (mw != kNegInf) acc += sm_o[(w * kG + jh) * kD + dd] * fast_exp2(mw - M);
          }
          a.part_o[((size_t)d.cg * a.Hq + hg.first) * kD + idx] = acc * ofac;
        }
        if (t < hg.count) a.part_ml[(size_t)d.cg * a.Hq + hg.first + t] = make_float2(sm_fin[2 * t], sm_fin[2 * t + 1]);
      }
      // this head group's share of the walk's bits (the merge ORs the groups')
      if (t == 0) a.part_st[(size_t)d.cg * a.Hkv + d.g] = item_st;
      named_bar_sync(1, kCT);
      if (threadIdx.x == 0) mbar_arrive(&item_empty[slot]);
      if (!alive) break;
    }
  }
  // Whether a wait gave up somewhere in this block; the merge then reports
  // every request of the call as timed out (its output is not valid).
  __syncthreads();
  if (threadIdx.x == 0) a.cta_abort[blockIdx.x] = *abort_flag != 0;
}

// ---------------------------------------------------------------- host side

int make_pool_map(CUtensorMap *map, const void *pool, int dtype, int D, int S, int Hkv, int P) {
  EncodeTiledFn enc = encode_tiled_fn();
  if (!enc) return cuda_fail(cudaErrorNotSupported, "cuTensorMapEncodeTiled entry point");
  const int esz = dtype == PFKV_DTYPE_FP8_E4M3 ? 1 : 2;
  const CUtensorMapDataType dt = esz == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const uint64_t row = (uint64_t)D * esz;
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  CUresult r;
  if (row == 256) {  // two 128-byte halves per row
    cuuint64_t dims[5] = {64, 2, (cuuint64_t)S, (cuuint64_t)Hkv, (cuuint64_t)P};
    cuuint64_t strides[4] = {128, 256, 256ull * S, 256ull * S * Hkv};
    cuuint32_t box[5] = {64, 2, (cuuint32_t)S, 1, 1};
    r = enc(map, dt, 5, const_cast<void *>(pool), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  } else {
    cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)S, (cuuint64_t)Hkv, (cuuint64_t)P};
    cuuint64_t strides[3] = {row, row * S, row * S * Hkv};
    cuuint32_t box[4] = {(cuuint32_t)D, (cuuint32_t)S, 1, 1};
    r = enc(map, dt, 4, const_cast<void *>(pool), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            row >= 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  }
  if (r != CUDA_SUCCESS) return cuda_fail(cudaErrorInvalidValue, "cuTensorMapEncodeTiled");
  return PFKV_OK;
}

constexpr int kNCW = 4;
// Cut rule: each request's segment of the cut line starts with this many
// pages' worth of overhead, so that a range holding many short requests
// (many pieces, each with its own set-up and finish) gets fewer pages.
constexpr int kPieceCost = 16;

// Launch shape of one split-kernel instantiation for one (page size, scale
// mode), worked out on its first use and reused afterwards, so that later
// calls -- including calls under stream capture -- only enqueue kernels.
struct SplitShape {
  int S = 0, per_token = -1, dev = -1, nst = 0, grid = 0;
  uint32_t smem = 0;
};

template <bool kFp8, int kD, int kG>
int run_split(const DecodeArgs &a_in, cudaStream_t s, const CUtensorMap &mk, const CUtensorMap &mv) {
  using C = Cfg<kFp8, kD, kG, kNCW>;
  DecodeArgs a = a_in;
  const bool per_token = kFp8 && a.scale_mode == PFKV_SCALE_PER_TOKEN;
  auto kern = gqa_split_kernel<kFp8, kD, kG, kNCW>;
  static SplitShape cache[4];
  static std::mutex mu;
  int dev = 0;
  cudaGetDevice(&dev);
  SplitShape sh;
  {
    std::lock_guard<std::mutex> lock(mu);
    bool found = false;
    for (auto &e : cache)
      if (e.S == a.S && e.per_token == (int)per_token && e.dev == dev) {
        sh = e;
        found = true;
        break;
      }
    if (!found) {
      // stage ring of roughly 64 KB (at least 4 pages) so that two or three CTAs share an SM
      const SmemPlan one = smem_plan(a.S, C::kRowBytes, per_token, 1, kNCW, kG, kD);
      int nst = (int)(65536u / one.stage_bytes);
      if (nst < 4) nst = 4;
      if (nst > 32) nst = 32;
      SmemPlan sp = smem_plan(a.S, C::kRowBytes, per_token, nst, kNCW, kG, kD);
      while (sp.total > 200u * 1024u && nst > 2) sp = smem_plan(a.S, C::kRowBytes, per_token, --nst, kNCW, kG, kD);
      // The attribute is a per-kernel cap on the device: only ever raise it, so
      // that a shape with a larger ring, cached earlier, keeps launching.
      static uint32_t attr_set[64] = {};
      if (dev < 64 && sp.total > attr_set[dev]) {
        const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sp.total);
        if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(split kernel)");
        attr_set[dev] = sp.total;
      }
      int per_sm = 0;
      const cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, C::kThreads, sp.total);
      if (e != cudaSuccess) return cuda_fail(e, "occupancy query (split kernel)");
      if (per_sm < 1) return cuda_fail(cudaErrorInvalidConfiguration, "split kernel does not fit on an SM");
      sh.S = a.S; sh.per_token = (int)per_token; sh.dev = dev; sh.nst = nst; sh.smem = sp.total;
      sh.grid = num_sms() * per_sm;
      int slot = 0;
      for (int i = 0; i < 4; ++i)
        if (cache[i].S == 0) { slot = i; break; }
      cache[slot] = sh;
    }
  }
  // No plan kernel: the split CTAs work out their pieces themselves (one CTA
  // group of Hkv CTAs per page range), and the merge kernel writes status.
  a.ranges = max(1, min(sh.grid, kMaxCtas) / a.Hkv);
  a.n_ctas = a.ranges * a.Hkv;
  a.st_groups = a.Hkv;
  a.target_items = a.n_ctas * 8;
  a.min_chunk_pages = (1024 + a.S - 1) / a.S;
  a.piece_cost = kPieceCost;
  if (a.n_ctas > kMaxCtas) return PFKV_ERR_UNSUPPORTED;  // more KV heads than abort words
  // The split kernel is a programmatic dependent of the stream's previous
  // kernel: its CTAs take SMs as that kernel's blocks drain and wait for it
  // to finish (griddepcontrol.wait) before touching memory.
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.n_ctas);
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = sh.smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int rc = cuda_ok(cudaLaunchKernelEx(&cfg, kern, mk, mv, a, sh.nst), "split kernel launch");
  if (rc) return rc;
  // the narrow merge shape when the wide one would give fewer than two
  // blocks per SM (a few requests, many pieces each)
  const bool narrow = (long long)a.B * a.Hkv * merge_col_blocks<kD, kG>() < 2LL * num_sms();
  cudaLaunchConfig_t mcfg = {};
  mcfg.gridDim = dim3(a.B * a.Hkv, narrow ? merge_col_blocks<kD, kG, 0>() : merge_col_blocks<kD, kG>());
  mcfg.blockDim = dim3(256);
  mcfg.stream = s;
  mcfg.attrs = attr;
  mcfg.numAttrs = 1;
  return cuda_ok(narrow ? cudaLaunchKernelEx(&mcfg, merge_kernel<kD, kG, 0>, a)
                        : cudaLaunchKernelEx(&mcfg, merge_kernel<kD, kG>, a),
                 "merge kernel launch");
}

// Any group size: up to 8 query heads per CTA group (the register-operand
// MMA's N dimension); a larger group is cut into kv_sub head groups of Gs
// heads each, run as virtual KV heads (every group reads the KV head's
// pages: the groups of one KV head are neighbouring CTAs, whose copies of a
// page mostly meet in L2).  The kernel is instantiated for 1, 2, 4 or 8
// head slots; a group of Gs heads takes the next of these and leaves the
// other slots as zero-query padding whose results are never written.
template <bool kFp8, int kD>
int dispatch_g(const DecodeArgs &a_in, cudaStream_t s, const CUtensorMap &mk, const CUtensorMap &mv) {
  DecodeArgs a = a_in;
  a.kv_sub = (a.G + 7) / 8;
  a.Gs = (a.G + a.kv_sub - 1) / a.kv_sub;
  if ((long long)a.Hkv * a.kv_sub > kMaxCtas) return PFKV_ERR_UNSUPPORTED;
  a.Hkv *= a.kv_sub;
  const int slots = a.Gs <= 1 ? 1 : a.Gs <= 2 ? 2 : a.Gs <= 4 ? 4 : 8;
  switch (slots) {
    case 1: return run_split<kFp8, kD, 1>(a, s, mk, mv);
    case 2: return run_split<kFp8, kD, 2>(a, s, mk, mv);
    case 4: return run_split<kFp8, kD, 4>(a, s, mk, mv);
    default: return run_split<kFp8, kD, 8>(a, s, mk, mv);
  }
}

}  // namespace

int launch_gqa_decode(const DecodeArgs &a, cudaStream_t s) {
  CUtensorMap mk, mv;
  int rc = make_pool_map(&mk, a.k_pool, a.dtype, a.D, a.S, a.Hkv, a.P);
  if (rc) return rc;
  rc = make_pool_map(&mv, a.v_pool, a.dtype, a.D, a.S, a.Hkv, a.P);
  if (rc) return rc;
  const bool fp8 = a.dtype == PFKV_DTYPE_FP8_E4M3;
  if (a.D == 128) return fp8 ? dispatch_g<true, 128>(a, s, mk, mv) : dispatch_g<false, 128>(a, s, mk, mv);
  if (a.D == 64) return fp8 ? dispatch_g<true, 64>(a, s, mk, mv) : dispatch_g<false, 64>(a, s, mk, mv);
  return PFKV_ERR_UNSUPPORTED;
}

}  // namespace pfkv
