// decode_noalloc.cu -- FP8 paged decode attention for callers that cannot
// allocate device memory.
//
// The regular entry point takes its split-KV scratch (the "workspace") from
// the caller.  Some callers have no way to provide it: code running inside a
// host framework that owns every device allocation and hands out only input
// and output buffers, plugins loaded into a process whose allocator must not
// be bypassed, or paths where a cudaMalloc would synchronise the device in the
// middle of serving.  For them this file keeps a fixed scratch buffer in the
// library itself, as a file-scope __device__ array, and forwards to the
// regular FP8 entry point with that buffer as the workspace.  Nothing here
// allocates: no cudaMalloc, no cudaFree, no allocating library call.
#include <mutex>

#include "pfkv_internal.h"

namespace {

// Every GPU that loads the library holds this buffer until the process exits.
static __device__ __align__(256) uint8_t g_noalloc_scratch[PFKV_NOALLOC_SCRATCH_BYTES];

// Device address of g_noalloc_scratch, looked up once per device.  In host
// code the array's name is only a host-side stand-in, so it is never passed
// to a kernel directly.
constexpr int kMaxDevices = 64;
void *g_scratch_ptr[kMaxDevices] = {};
std::mutex g_scratch_mu;

int scratch_for_current_device(void **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return pfkv::cuda_fail(e, "cudaGetDevice (no-alloc decode)");
  if (dev < 0 || dev >= kMaxDevices) return pfkv::cuda_fail(cudaErrorInvalidDevice, "device index (no-alloc decode)");
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);  // this device is current
    if (e != cudaSuccess) return pfkv::cuda_fail(e, "cudaGetSymbolAddress (no-alloc decode scratch)");
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return PFKV_OK;
}

}  // namespace

extern "C" int pfkv_paged_decode_attention_fp8_noalloc(const pfkv_cache *cache, const void *q, int32_t num_q_heads,
                                                       const int32_t *seq_lens, const int32_t *block_table,
                                                       const uint32_t *block_tags, int32_t batch, int32_t max_pages,
                                                       float softmax_scale, uint32_t flags, int32_t max_splits,
                                                       float *out, uint32_t *status, void *stream) {
  // The regular entry point's own checks first, so that a bad descriptor or
  // size gives the same code here as there; then, before touching the
  // device, any call whose scratch would not fit is rejected.
  const int pre = pfkv::decode_precheck(PFKV_DTYPE_FP8_E4M3, cache, num_q_heads, batch, max_pages, max_splits);
  if (pre) return pre;
  if (pfkv_decode_workspace_bytes(cache, batch, num_q_heads, max_splits) > (size_t)PFKV_NOALLOC_SCRATCH_BYTES)
    return PFKV_ERR_WORKSPACE;
  void *scratch = nullptr;
  const int rc = scratch_for_current_device(&scratch);
  if (rc) return rc;
  // The regular path rewrites, on every call, every workspace word it reads
  // back, so the buffer needs no clearing between calls.
  return pfkv_paged_decode_attention_fp8(cache, q, num_q_heads, seq_lens, block_table, block_tags, batch, max_pages,
                                         softmax_scale, flags, max_splits, scratch,
                                         (size_t)PFKV_NOALLOC_SCRATCH_BYTES, out, status, stream);
}
