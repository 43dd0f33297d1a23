// decode_latent.cu -- decode attention over a latent-shared FP8 stream
// (576 values per token: 512 latent + 64 rotary; V = the first 512).
#include "pfkv_device.cuh"
#include "pfkv_internal.h"

namespace pfkv {

int launch_latent_decode(const DecodeArgs &, cudaStream_t) { return PFKV_ERR_UNSUPPORTED; }

}  // namespace pfkv
