// Whole-block data movement on the paged KV pool:
//  - copy_blocks: pool block dst <- pool block src, for copy-on-write of a
//    shared, partially filled last block (review §6: blocks are shared via
//    copy-on-write; §9: the block table makes COW sharing possible);
//  - gather_blocks / scatter_blocks: pool blocks <-> a contiguous buffer,
//    for swapping a preempted sequence's blocks to host memory and back
//    (review §9: preemptive scheduling swaps blocks to CPU; KV offload).
// A block of one cache is Hkv * bs * D * eb contiguous bytes; every kernel
// moves 16-byte words with a grid-stride loop over (item, K/V, word).  Block
// ids outside the pool are skipped and recorded in the device error word.
#include "pagedattn.h"
#include "pa_internal.h"

namespace pa {

namespace {

constexpr int kErrBlockId = 0x1;

__device__ __forceinline__ bool in_pool(int64_t b, int64_t nb) { return b >= 0 && b < nb; }

__global__ void __launch_bounds__(256) copy_blocks_kernel(uint4* k_cache, uint4* v_cache, const int64_t* pairs,
                                                          int n, int64_t words_per_block, int64_t nb, int* err) {
  const int64_t total = static_cast<int64_t>(n) * 2 * words_per_block;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t w = i % words_per_block;
    const int64_t rest = i / words_per_block;
    const int which = static_cast<int>(rest & 1);
    const int64_t item = rest >> 1;
    const int64_t src = pairs[2 * item], dst = pairs[2 * item + 1];
    if (!in_pool(src, nb) || !in_pool(dst, nb)) {
      if (w == 0 && which == 0) atomicOr(err, kErrBlockId);
      continue;
    }
    uint4* c = which ? v_cache : k_cache;
    c[dst * words_per_block + w] = c[src * words_per_block + w];
  }
}

// buffer layout: [n][2 (K, V)][words_per_block]
__global__ void __launch_bounds__(256) gather_blocks_kernel(uint4* buf, const uint4* k_cache, const uint4* v_cache,
                                                            const int64_t* ids, int n, int64_t words_per_block,
                                                            int64_t nb, int* err) {
  const int64_t total = static_cast<int64_t>(n) * 2 * words_per_block;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t w = i % words_per_block;
    const int64_t rest = i / words_per_block;
    const int which = static_cast<int>(rest & 1);
    const int64_t item = rest >> 1;
    const int64_t b = ids[item];
    if (!in_pool(b, nb)) {
      if (w == 0 && which == 0) atomicOr(err, kErrBlockId);
      continue;
    }
    const uint4* c = which ? v_cache : k_cache;
    buf[i] = c[b * words_per_block + w];
  }
}

__global__ void __launch_bounds__(256) scatter_blocks_kernel(uint4* k_cache, uint4* v_cache, const uint4* buf,
                                                             const int64_t* ids, int n, int64_t words_per_block,
                                                             int64_t nb, int* err) {
  const int64_t total = static_cast<int64_t>(n) * 2 * words_per_block;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t w = i % words_per_block;
    const int64_t rest = i / words_per_block;
    const int which = static_cast<int>(rest & 1);
    const int64_t item = rest >> 1;
    const int64_t b = ids[item];
    if (!in_pool(b, nb)) {
      if (w == 0 && which == 0) atomicOr(err, kErrBlockId);
      continue;
    }
    uint4* c = which ? v_cache : k_cache;
    c[b * words_per_block + w] = buf[i];
  }
}

unsigned grid_for(int64_t total) {
  // enough CTAs to fill every SM several times; the loops are grid-stride
  int64_t g = (total + 255) / 256;
  if (g > 152 * 16) g = 152 * 16;
  return static_cast<unsigned>(g < 1 ? 1 : g);
}

}  // namespace

cudaError_t launch_block_op(int op, void* buf, void* k_cache, void* v_cache, const int64_t* ids, int n,
                            int64_t block_bytes, int64_t num_blocks, int* err, cudaStream_t st) {
  const int64_t wpb = block_bytes / 16;
  const int64_t total = static_cast<int64_t>(n) * 2 * wpb;
  if (total == 0) return cudaSuccess;
  const unsigned grid = grid_for(total);
  uint4* kc = static_cast<uint4*>(k_cache);
  uint4* vc = static_cast<uint4*>(v_cache);
  if (op == 0)
    copy_blocks_kernel<<<grid, 256, 0, st>>>(kc, vc, ids, n, wpb, num_blocks, err);
  else if (op == 1)
    gather_blocks_kernel<<<grid, 256, 0, st>>>(static_cast<uint4*>(buf), kc, vc, ids, n, wpb, num_blocks, err);
  else
    scatter_blocks_kernel<<<grid, 256, 0, st>>>(kc, vc, static_cast<const uint4*>(buf), ids, n, wpb, num_blocks,
                                                err);
  return cudaGetLastError();
}

}  // namespace pa
