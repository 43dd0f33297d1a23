// alloc.cu -- device-resident page allocator; every hand-out of a page moves
// its tag.
//
// "Smaller, faster, safer: running Kimi and GLM at scale", cache-protection
// passage: each page of the shared cache carries a tag that changes whenever
// the page is reallocated, and a read through a mapping with the old tag
// aborts.  This file is the side that changes the tags.  The free list is a
// stack in device memory, so a decode step can take and return pages on its
// stream without a host round trip.
//
// alloc / free / realloc are one CTA of 1024 threads each: the lists a step
// hands over are short (at most a few thousand ids), and one CTA gives
// list-order semantics with a block scan and no inter-CTA protocol.
// Duplicates inside one list are resolved with an atomicMin on a per-page
// scratch word (the lowest index wins), which every call leaves reset.
// init is grid-wide (pools reach millions of pages): count free ids per
// 1024-page chunk, scan the counts, scatter.
#include <climits>

#include "pfkv_internal.h"

namespace pfkv {

namespace {

constexpr int kAT = 1024;  // threads of the single-CTA kernels; also init's chunk

struct AllocHdr {
  int num_pages;
  int free_count;
  int pad[62];
};

__host__ __device__ inline size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

struct AllocLayout {
  size_t stack, mark, held, counts, total;
};

__host__ __device__ inline AllocLayout alloc_layout(int P) {
  AllocLayout L;
  L.stack = 256;
  L.mark = L.stack + round256(size_t(P) * 4);
  L.held = L.mark + round256(size_t(P) * 4);
  L.counts = L.held + round256(size_t(P));
  L.total = L.counts + round256((size_t((P + kAT - 1) / kAT) + 1) * 4);
  return L;
}

struct AllocView {
  AllocHdr *hdr;
  int *stack, *mark;
  uint8_t *held;
  int *counts;
};

__device__ inline AllocView view(void *state) {
  uint8_t *base = static_cast<uint8_t *>(state);
  AllocView v;
  v.hdr = reinterpret_cast<AllocHdr *>(base);
  const AllocLayout L = alloc_layout(v.hdr->num_pages);
  v.stack = reinterpret_cast<int *>(base + L.stack);
  v.mark = reinterpret_cast<int *>(base + L.mark);
  v.held = base + L.held;
  v.counts = reinterpret_cast<int *>(base + L.counts);
  return v;
}

// Exclusive scan of one flag per thread over the block (1024 threads);
// returns this thread's rank, total in *total.  Uses s_warp[32].
__device__ inline int block_rank(bool flag, int *s_warp, int *total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const unsigned bal = __ballot_sync(0xffffffffu, flag);
  const int in_warp = __popc(bal & ((1u << lane) - 1u));
  if (lane == 0) s_warp[warp] = __popc(bal);
  __syncthreads();
  if (warp == 0) {
    const int c = s_warp[lane];
    int incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    s_warp[lane] = incl - c;
    if (lane == 31) s_warp[32] = incl;
  }
  __syncthreads();
  const int r = s_warp[warp] + in_warp;
  *total = s_warp[32];
  __syncthreads();  // s_warp is reused by the next call
  return r;
}

// ---------------------------------------------------------------- init

__global__ void init_clear_kernel(void *state, int P) {
  uint8_t *base = static_cast<uint8_t *>(state);
  const AllocLayout L = alloc_layout(P);
  int *mark = reinterpret_cast<int *>(base + L.mark);
  uint8_t *held = base + L.held;
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    AllocHdr *h = reinterpret_cast<AllocHdr *>(base);
    h->num_pages = P;
    h->free_count = 0;
  }
  for (long long p = blockIdx.x * (long long)blockDim.x + threadIdx.x; p < P; p += (long long)gridDim.x * blockDim.x) {
    mark[p] = INT_MAX;
    held[p] = 0;
  }
}

__global__ void init_mark_held_kernel(void *state, const int *held_pages, int n_held) {
  AllocView v = view(state);
  const int P = v.hdr->num_pages;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n_held;
       i += (long long)gridDim.x * blockDim.x) {
    const int p = held_pages[i];
    if (p >= 0 && p < P) v.held[p] = 1;
  }
}

// Chunk c covers stack order positions q in [c*1024, (c+1)*1024), page p = P-1-q
// (the stack holds free ids in decreasing order, so the smallest is on top).
__global__ void __launch_bounds__(kAT) init_count_kernel(void *state) {
  AllocView v = view(state);
  const int P = v.hdr->num_pages;
  const long long q = (long long)blockIdx.x * kAT + threadIdx.x;
  const bool is_free = q < P && !v.held[P - 1 - q];
  const int n = __syncthreads_count(is_free);
  if (threadIdx.x == 0) v.counts[blockIdx.x] = n;
}

__global__ void __launch_bounds__(kAT) init_scan_kernel(void *state, int n_chunks) {
  __shared__ int s_warp[33];
  AllocView v = view(state);
  int carry = 0;
  for (int base = 0; base < n_chunks; base += kAT) {
    const int c = base + (int)threadIdx.x;
    const int cnt = c < n_chunks ? v.counts[c] : 0;
    // exclusive scan of counts (not flags): warp scan of values
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      const int wsum = s_warp[lane];
      int wincl = wsum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, wincl, o);
        if (lane >= o) wincl += t;
      }
      s_warp[lane] = wincl - wsum;
      if (lane == 31) s_warp[32] = wincl;
    }
    __syncthreads();
    if (c < n_chunks) v.counts[c] = carry + s_warp[warp] + incl - cnt;
    carry += s_warp[32];
    __syncthreads();
  }
  if (threadIdx.x == 0) v.hdr->free_count = carry;
}

__global__ void __launch_bounds__(kAT) init_scatter_kernel(void *state) {
  __shared__ int s_warp[33];
  AllocView v = view(state);
  const int P = v.hdr->num_pages;
  const long long q = (long long)blockIdx.x * kAT + threadIdx.x;
  const bool is_free = q < P && !v.held[P - 1 - q];
  int total;
  const int r = block_rank(is_free, s_warp, &total);
  if (is_free) v.stack[v.counts[blockIdx.x] + r] = (int)(P - 1 - q);
}

// ---------------------------------------------------------------- alloc / free / realloc

__global__ void __launch_bounds__(kAT) alloc_kernel(void *state, uint32_t *page_tags, int n, int *pages_out,
                                                    uint32_t *tags_out, uint32_t *status) {
  AllocView v = view(state);
  const int fc = v.hdr->free_count;
  if (n > fc) {
    for (int i = threadIdx.x; i < n; i += kAT) {
      pages_out[i] = -1;
      tags_out[i] = 0u;
    }
    if (threadIdx.x == 0) *status = PFKV_ST_NO_PAGES;
    return;
  }
  for (int i = threadIdx.x; i < n; i += kAT) {
    const int p = v.stack[fc - 1 - i];
    v.held[p] = 1;
    const uint32_t t = page_tags[p] + 1u;
    page_tags[p] = t;
    pages_out[i] = p;
    tags_out[i] = t;
  }
  __syncthreads();  // every thread has read free_count
  if (threadIdx.x == 0) {
    v.hdr->free_count = fc - n;
    *status = 0u;
  }
}

// First occurrence of each held page in the list claims the page's scratch word.
__device__ inline void claim_first(const AllocView &v, int P, const int *pages, int n) {
  for (int i = threadIdx.x; i < n; i += kAT) {
    const int p = pages[i];
    if (p >= 0 && p < P && v.held[p]) atomicMin(&v.mark[p], i);
  }
  __syncthreads();
}

__global__ void __launch_bounds__(kAT) free_kernel(void *state, const int *pages, int n, uint32_t *page_status) {
  __shared__ int s_warp[33];
  AllocView v = view(state);
  const int P = v.hdr->num_pages;
  const int fc = v.hdr->free_count;
  claim_first(v, P, pages, n);
  int pushed = 0;
  for (int base = 0; base < n; base += kAT) {
    const int i = base + (int)threadIdx.x;
    int p = -1;
    bool in_range = false, win = false;
    if (i < n) {
      p = pages[i];
      in_range = p >= 0 && p < P;
      win = in_range && v.mark[p] == i;
    }
    int total;
    const int r = block_rank(win, s_warp, &total);
    if (i < n) page_status[i] = !in_range ? PFKV_ST_PAGE_OOB : win ? 0u : PFKV_ST_NOT_HELD;
    if (win) {
      v.stack[fc + pushed + r] = p;
      v.held[p] = 0;
      v.mark[p] = INT_MAX;
    }
    pushed += total;
  }
  if (threadIdx.x == 0) v.hdr->free_count = fc + pushed;
}

__global__ void __launch_bounds__(kAT) realloc_kernel(void *state, uint32_t *page_tags, const int *pages, int n,
                                                      uint32_t *tags_out, uint32_t *page_status) {
  AllocView v = view(state);
  const int P = v.hdr->num_pages;
  claim_first(v, P, pages, n);
  for (int i = threadIdx.x; i < n; i += kAT) {
    const int p = pages[i];
    uint32_t st, t = 0u;
    if (p < 0 || p >= P) {
      st = PFKV_ST_PAGE_OOB;
    } else if (!v.held[p]) {
      st = PFKV_ST_NOT_HELD;
    } else if (v.mark[p] != i) {
      st = PFKV_ST_DUPLICATE;
    } else {
      st = 0u;
      t = page_tags[p] + 1u;
      page_tags[p] = t;
    }
    tags_out[i] = t;
    page_status[i] = st;
  }
  __syncthreads();  // every comparison with the scratch words is done
  for (int i = threadIdx.x; i < n; i += kAT) {
    const int p = pages[i];
    if (p >= 0 && p < P) v.mark[p] = INT_MAX;
  }
}

}  // namespace

size_t alloc_state_bytes(int num_pages) { return num_pages < 1 ? 0 : alloc_layout(num_pages).total; }

int launch_alloc_init(void *state, int P, const int *held_pages, int n_held, cudaStream_t s) {
  const int sms = num_sms();
  const int n_chunks = (P + kAT - 1) / kAT;
  const int grid = n_chunks < 8 * sms ? n_chunks : 8 * sms;
  init_clear_kernel<<<grid, kAT, 0, s>>>(state, P);
  if (n_held > 0) {
    const int g2 = (n_held + kAT - 1) / kAT < 8 * sms ? (n_held + kAT - 1) / kAT : 8 * sms;
    init_mark_held_kernel<<<g2, kAT, 0, s>>>(state, held_pages, n_held);
  }
  init_count_kernel<<<n_chunks, kAT, 0, s>>>(state);
  init_scan_kernel<<<1, kAT, 0, s>>>(state, n_chunks);
  init_scatter_kernel<<<n_chunks, kAT, 0, s>>>(state);
  return cuda_ok(cudaGetLastError(), "allocator init launch");
}

int launch_page_alloc(void *state, uint32_t *page_tags, int n, int *pages_out, uint32_t *tags_out, uint32_t *status,
                      cudaStream_t s) {
  alloc_kernel<<<1, kAT, 0, s>>>(state, page_tags, n, pages_out, tags_out, status);
  return cuda_ok(cudaGetLastError(), "page alloc launch");
}

int launch_page_free(void *state, const int *pages, int n, uint32_t *page_status, cudaStream_t s) {
  free_kernel<<<1, kAT, 0, s>>>(state, pages, n, page_status);
  return cuda_ok(cudaGetLastError(), "page free launch");
}

int launch_page_realloc(void *state, uint32_t *page_tags, const int *pages, int n, uint32_t *tags_out,
                        uint32_t *page_status, cudaStream_t s) {
  realloc_kernel<<<1, kAT, 0, s>>>(state, page_tags, pages, n, tags_out, page_status);
  return cuda_ok(cudaGetLastError(), "page realloc launch");
}

}  // namespace pfkv
