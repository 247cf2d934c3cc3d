// Internal interface of the E4M3 -> 16-bit widening of a batch's K/V blocks
// (pa_widen.cu), used by prefill over FP8 caches.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace pa {

struct WidenParams {
  const uint8_t* k_src;          // E4M3 pool [num_blocks, Hkv, bs, D]
  const uint8_t* v_src;
  uint16_t* k_dst;               // compact pool [S * maxB, Hkv, bs, D] of the 16-bit type
  uint16_t* v_dst;
  int32_t* tab;                  // [S, maxB]: entry (s, j) = s * maxB + j
  const int32_t* block_tables;   // [S, maxB]
  const int32_t* context_lens;   // [S]
  int* err;                      // device error word (block ids out of range)
  int64_t num_blocks;
  int S, maxB, Hkv, bs, D;
  int bf16;                      // 1: widen to bf16, 0: to f16
};

// Block j < ceil(L_s / bs) of sequence s (all kv heads, K and V) to compact
// block s * maxB + j; every table entry written.  Stream-ordered.
cudaError_t launch_widen_kv(const WidenParams& p, cudaStream_t st);

}  // namespace pa
