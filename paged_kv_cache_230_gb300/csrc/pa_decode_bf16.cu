// Decode kernels for bf16 caches (one translation unit per cache dtype so the
// instantiations compile in parallel).
#include "pa_decode.cuh"

namespace pa {

cudaError_t launch_decode_bf16(const DecodeParams& p, const CUtensorMap& tmK, const CUtensorMap& tmV,
                              int head_dim, cudaStream_t st) {
  return launch_decode_kv<kBF16>(p, tmK, tmV, head_dim, st);
}

}  // namespace pa
