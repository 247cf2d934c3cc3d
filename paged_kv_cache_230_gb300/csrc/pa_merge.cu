// Log-sum-exp merge of split-decode partials.
#include "pa_decode.cuh"

namespace pa {

cudaError_t launch_lse_merge(const DecodeParams& p, int head_dim, cudaStream_t st) {
  const unsigned grid = static_cast<unsigned>(static_cast<long long>(p.S) * p.qlen * p.Hq);
  if (head_dim == 64)
    lse_merge_kernel<64><<<grid, kMergeThreads, 0, st>>>(p);
  else
    lse_merge_kernel<128><<<grid, kMergeThreads, 0, st>>>(p);
  return cudaGetLastError();
}

}  // namespace pa
