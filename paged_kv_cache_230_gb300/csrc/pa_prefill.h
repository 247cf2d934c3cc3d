// Internal interface of the paged prefill kernel (tcgen05 path).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace pa {

constexpr int kPfRows = 128;     // query rows per CTA (MMA M, TMEM lanes)
constexpr int kPfTile = 128;     // KV tokens per tile (MMA N of S, K of P.V)
constexpr int kPfStages = 2;     // K/V tiles in flight
constexpr int kPfThreads = 384;  // softmax, epilogue and TMA/MMA warpgroups

struct PrefillParams {
  void* out;                    // [S, C, Hq, D] of the cache dtype
  const int32_t* block_tables;  // [S, maxB]
  const int32_t* context_lens;  // [S] (includes the C new tokens)
  int* err;                     // device error word
  int64_t num_blocks;
  int S, C, Hq, Hkv, G, bs, maxB;
  int D;                        // head_dim: 128 (both kernels) or 64 (two-head kernel)
  int bf16;                     // 1: bf16 operands, 0: f16
  float scale_log2;             // softmax scale * log2(e)
  float vscale;                 // output factor (the E4M3 per-tensor scale; 1 for 16-bit caches)
  int cluster;                  // two-head kernel, head_dim 128, G % 4 == 0: clusters of two CTAs
                                // sharing each K/V tile by TMA multicast
};

// tmQ: 3-D map over q {D channels, Hq, S*C tokens}, box {64, 1, 128};
// tmK/tmV: the caches' 4-D maps (box {64, bs, 1, 1}), 128-byte swizzle.
cudaError_t launch_prefill(const PrefillParams& p, const CUtensorMap& tmQ, const CUtensorMap& tmK,
                           const CUtensorMap& tmV, cudaStream_t st);

// The same with two query heads of one kv head per work item (an even group
// size G; head_dim 64 or 128): their query tiles share each K/V tile
// (pa_prefill_pair.cu).  Same maps and parameters.
cudaError_t launch_prefill_pair(const PrefillParams& p, const CUtensorMap& tmQ, const CUtensorMap& tmK,
                                const CUtensorMap& tmV, cudaStream_t st);

}  // namespace pa
