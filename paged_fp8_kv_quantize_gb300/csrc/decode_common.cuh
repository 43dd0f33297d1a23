// decode_common.cuh -- pieces shared by the decode kernels: the work split
// (flash-decoding pieces, worked out by every CTA from the lengths).  The
// log-sum-exp merge of split partials is in merge.cuh.  Included by each
// decode translation unit; everything here has internal linkage.
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

// One virtual KV head's KV head and query heads (see DecodeArgs::kv_sub).
struct HeadGroup {
  int kv, first, count;
};

__device__ __forceinline__ HeadGroup head_group(const DecodeArgs &a, int v) {
  HeadGroup r;
  r.kv = v / a.kv_sub;
  const int sub = v - r.kv * a.kv_sub;
  r.first = r.kv * a.G + sub * a.Gs;
  r.count = min(a.Gs, a.G - sub * a.Gs);
  return r;
}

struct ItemDesc {
  int b, cg, g, p0, p1, L;
  uint32_t ring;
  int nb;  // splits of request b
};

// ---------------------------------------------------------------- work split
//
// There is no plan kernel: every CTA works out its own share from the
// lengths, and all CTAs reach the same answer.  The requests, in
// request order (a request with a bad length counting nothing), lie on a
// line of T units that is cut into R ranges [floor(kT/R), floor((k+1)T/R));
// CTA k * Hkv + h takes range k for KV head h (the latent stream: Hkv = 1).  Piece j of request b
// is numbered b * max_splits + j (j < max_splits under both rules), so that
// no CTA needs the piece counts of the requests before its own; the merge
// finds a request's pieces at split_first[b] = b * max_splits ..
// + split_count[b].  Two rules:
//  - cut: a request's segment of the line is c0 units of overhead followed
//    by its pages (c0 = piece_cost: a piece's set-up and finish, and the
//    consumer warps a short piece leaves idle, cost about that many pages'
//    time); a piece is the part of one request's pages inside one range, so
//    every CTA gets the same pages + overhead to within one.  R is capped so
//    that no request is cut into more than max_splits pieces (a segment of
//    s units meets at most ceil(s R / T) + 1 ranges); the rule is used when
//    max_splits >= 3 and the caps leave at least 3/4 of the CTA groups.
//  - chunk: the line is the bare pages (c0 = 0); each request is first cut
//    into at most max_splits chunks of about cp pages, and a range takes the
//    chunks that start inside it.  Used
//    for small batches (T below the number of CTA groups) and batches whose
//    longest request the split cap would otherwise leave on few CTAs.
struct WorkSplit {
  long long T, R, r0, r1, cp, max_len;
  int k, chunks;
  int c0;  // cut rule: overhead length placed before each request's pages on the cut line
  // walk: next request to look at, its first unit on the line, and (chunk
  // rule) its next chunk
  int b;
  long long off, c;
};

// The fields of DecodeArgs the work split reads, passed on their own so that
// the split's functions (compiled once, not inlined) never take the kernel
// parameter's address, which would move all of it to local memory.
struct WsArgs {
  const int *seq_lens;
  int B, S, MP, max_splits, ranges, piece_cost, target_items, min_chunk_pages, Hkv;
};

__device__ __forceinline__ WsArgs ws_args(const DecodeArgs &a) {
  WsArgs w;
  w.seq_lens = a.seq_lens;
  w.B = a.B; w.S = a.S; w.MP = a.MP; w.max_splits = a.max_splits; w.ranges = a.ranges; w.piece_cost = a.piece_cost;
  w.target_items = a.target_items; w.min_chunk_pages = a.min_chunk_pages; w.Hkv = a.Hkv;
  return w;
}

struct Piece {
  int b, cg, p0, p1, L, nb;
  bool lead;  // the request's first piece: its CTA of head 0 records the numbering
};

// The work split runs at the start of every CTA and once per piece.  Its
// walk is inlined into the page loaders and keeps its state in registers:
// as separately compiled functions taking the state by reference, the state
// lived in local memory and each call paid the calling convention's register
// saves (measured, grouped-query kernel: the first page copy ~1 us later and
// the ragged decode call 1.5 us longer).  The rarely needed divisions stay
// compiled once (noinline, all operands by value).
//
// floor(x / y) for x >= 0 and y >= 1 (the entry points bound batch *
// max_pages by 2^40, and every dividend here is at most 2^12 times a page
// count, so x < 2^53).  Operands that fit 32 bits -- every practical batch --
// take the 32-bit unsigned division; larger ones a bitwise long division.
// No floating point: double precision is slow on this part (an earlier
// reciprocal-estimate form in fp64 cost 0.3-0.6 us per call).
__device__ __forceinline__ unsigned long long div_floor_wide(unsigned long long x, unsigned long long y) {
  unsigned long long q = 0, r = 0;
  for (int i = 63; i >= 0; --i) {
    r = (r << 1) | ((x >> i) & 1ull);
    if (r >= y) {
      r -= y;
      q |= 1ull << i;
    }
  }
  return q;
}

__device__ __noinline__ long long div_floor(long long x, long long y) {
  const unsigned long long ux = (unsigned long long)x, uy = (unsigned long long)y;
  if (((ux | uy) >> 32) == 0ull) return (long long)((uint32_t)ux / (uint32_t)uy);
  return (long long)div_floor_wide(ux, uy);
}

__device__ __forceinline__ int ws_pages(const WorkSplit &w, int L, int S) {
  return (L < 1 || (long long)L > w.max_len) ? 0 : (int)(((unsigned)L + (unsigned)S - 1u) / (unsigned)S);
}

// Pieces of a request of p > 0 pages whose segment of the cut line starts
// at `off` (its pages start at off + c0), and the chunk length (chunk rule;
// 1 under the cut rule).  Every operand by value: the split's state stays
// in registers (a reference would put it in local memory, and every field
// access would become a memory round trip).
__device__ __noinline__ int2 ws_count(bool chunks, int c0, long long R, long long T, long long cp, long long off,
                                      int p, int max_splits) {
  if (!chunks) {
    const long long s0 = off + c0;
    return make_int2((int)(div_floor((s0 + p) * R - 1, T) - div_floor((s0 + 1) * R - 1, T) + 1), 1);
  }
  int nn = cp >= p ? 1 : (int)(((unsigned)p + (unsigned)cp - 1u) / (unsigned)cp);
  if (nn > max_splits) nn = max_splits;
  const int q = (int)(((unsigned)p + (unsigned)nn - 1u) / (unsigned)nn);
  return make_int2((int)(((unsigned)p + (unsigned)q - 1u) / (unsigned)q), q);
}

__device__ __forceinline__ void ws_init_regs(WorkSplit &w, const WsArgs &a, int lane) {
  const int S = a.S;
  w.max_len = (long long)a.MP * S;
  long long tot = 0;
  int mx = 0, nv = 0;
  for (int b = lane; b < a.B; b += 32) {
    const int p = ws_pages(w, __ldg(&a.seq_lens[b]), S);
    tot += p;
    mx = p > mx ? p : mx;
    nv += p > 0;
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    tot += __shfl_xor_sync(0xffffffffu, tot, o);
    mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    nv += __shfl_xor_sync(0xffffffffu, nv, o);
  }
  long long T = tot;
  const long long ranges = a.ranges, c = a.piece_cost;
  const long long Tc = T + c * nv;  // the cut rule's line: pages plus c before each request
  long long R = ranges < Tc ? ranges : Tc;
  if (mx > 0 && a.max_splits >= 3) {
    const long long cap = div_floor((long long)(a.max_splits - 2) * Tc, mx + c);
    if (R > cap) R = cap;
  }
  w.chunks = !(a.max_splits >= 3 && T > 0 && R >= 1 && 4 * R >= 3 * ranges);
  if (w.chunks) {
    R = ranges < T ? ranges : T;
    const long long cp = div_floor(T * a.Hkv + a.target_items - 1, a.target_items);
    w.cp = cp < a.min_chunk_pages ? a.min_chunk_pages : cp;
    w.c0 = 0;
  } else {
    w.cp = 0;
    w.c0 = (int)c;
    T = Tc;
  }
  w.T = T;
  w.R = R < 1 ? 1 : R;
  w.k = (int)blockIdx.x / a.Hkv;
  w.b = a.B;  // no pieces unless found below
  w.off = w.c = 0;
  if (T == 0 || w.k >= w.R) return;
  w.r0 = div_floor((long long)w.k * T, w.R);
  w.r1 = div_floor((long long)(w.k + 1) * T, w.R);
  long long off_c = 0;  // line units of earlier passes
  for (int base = 0; base < a.B; base += 32) {
    const int b = base + lane;
    const int p = b < a.B ? ws_pages(w, __ldg(&a.seq_lens[b]), S) : 0;
    const long long seg = p > 0 ? p + w.c0 : 0;  // the request's segment of the line
    long long xp = seg;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long y = __shfl_up_sync(0xffffffffu, xp, o);
      if (lane >= o) xp += y;
    }
    const long long off = off_c + xp - seg;
    bool has = false;
    int c_lo = 0;
    if (p > 0 && off + w.c0 < w.r1 && off + w.c0 + p > w.r0) {
      if (!w.chunks) {
        has = true;
      } else {
        const int2 np = ws_count(w.chunks, w.c0, w.R, w.T, w.cp, off, p, a.max_splits);
        const int n = np.x, ppc = np.y;
        // r0 - off < p here, so the chunk index fits an int
        c_lo = off >= w.r0 ? 0 : (int)((unsigned)(w.r0 - off + ppc - 1) / (unsigned)ppc);
        has = c_lo < n && off + (long long)c_lo * ppc < w.r1;
      }
    }
    const unsigned m = __ballot_sync(0xffffffffu, has);
    if (m) {
      const int src = __ffs(m) - 1;
      w.b = base + src;
      w.off = __shfl_sync(0xffffffffu, off, src);
      w.c = __shfl_sync(0xffffffffu, c_lo, src);
      return;
    }
    off_c += __shfl_sync(0xffffffffu, xp, 31);
  }
}

// Warp-wide (all 32 lanes, same result in each): the rule, R and this CTA's
// range, then the first request with a piece in it.  Works on register
// copies of its arguments and writes the state once at the end.
__device__ __forceinline__ void ws_init(WorkSplit &w_out, const WsArgs &a_in, int lane) {
  const WsArgs a = a_in;
  WorkSplit w{};
  ws_init_regs(w, a, lane);
  w_out = w;
}

// The CTA's next piece, in request order (uniform across the warp); false
// when the range has none left.  A piece that would break the workspace
// bounds ends the walk instead of being used (it cannot occur when the
// rules above hold).
__device__ __forceinline__ bool ws_next_regs(WorkSplit &w, const WsArgs &a, Piece &pc) {
  while (w.b < a.B) {
    const int L = __ldg(&a.seq_lens[w.b]);
    const int p = ws_pages(w, L, a.S);
    if (p == 0) {
      ++w.b;
      continue;
    }
    if (w.off + w.c0 >= w.r1) return false;
    const int2 np = ws_count(w.chunks, w.c0, w.R, w.T, w.cp, w.off, p, a.max_splits);
    const int n = np.x, ppc = np.y;
    long long j, p0, p1;
    if (!w.chunks) {
      const long long s0 = w.off + w.c0;  // the request's first page on the cut line
      j = (long long)w.k - div_floor((s0 + 1) * w.R - 1, w.T);
      p0 = (w.r0 > s0 ? w.r0 : s0) - s0;
      p1 = (w.r1 < s0 + p ? w.r1 : s0 + p) - s0;
    } else {
      if (w.c >= n) {
        w.off += p;
        ++w.b;
        w.c = 0;
        continue;
      }
      if (w.off + w.c * ppc >= w.r1) return false;
      j = w.c++;
      p0 = j * ppc;
      p1 = p0 + ppc < p ? p0 + ppc : p;
    }
    if (j < 0 || j >= n || n > a.max_splits || p0 < 0 || p0 >= p1 || p1 > p) return false;
    const long long cg = (long long)w.b * a.max_splits + j;
    pc.b = w.b;
    pc.cg = (int)cg;
    pc.p0 = (int)p0;
    pc.p1 = (int)p1;
    pc.L = L;
    pc.nb = n;
    pc.lead = j == 0;
    if (!w.chunks) {
      w.off += p + w.c0;
      ++w.b;
    }
    return true;
  }
  return false;
}

// ws_next_regs on register copies of the state and the arguments; the state
// and the piece are written back once.
__device__ __forceinline__ bool ws_next(WorkSplit &w_io, const WsArgs &a_in, Piece &pc_out) {
  const WsArgs a = a_in;
  WorkSplit w = w_io;
  Piece pc{};
  const bool r = ws_next_regs(w, a, pc);
  w_io = w;
  pc_out = pc;
  return r;
}

// ws_next on a state kept in shared memory (one copy per warp), so that it
// holds no registers while the pages go out.
__device__ __forceinline__ bool ws_next_shared(WorkSplit &s, const WsArgs &a, Piece &pc, int lane) {
  WorkSplit w = s;
  __syncwarp();
  const bool r = ws_next(w, a, pc);
  if (lane == 0) s = w;
  __syncwarp();
  return r;
}

}  // namespace
}  // namespace pfkv
