// reshape_and_cache: scatter of this step's new K/V rows into their cache
// slots (blocks are extended by one token per sequence per decode step:
// vLLM review, §6 "KV Cache Block Tables").
//
// One thread moves 8 consecutive channels (one 16-byte load) of one
// (token, kv head, K-or-V) row, so a warp covers whole rows with coalesced
// loads and 16-byte (16-bit cache) or 8-byte (FP8 cache) stores.  Every slot
// is bounds-checked: a slot outside the pool is skipped and recorded.
#include "pa_cache_row.cuh"
#include "pa_internal.h"

namespace pa {

namespace {

constexpr int kErrSlot = 0x4;

template <bool TO_FP8>
__global__ void __launch_bounds__(256) reshape_and_cache_kernel(const CacheParams p) {
  const int chunks = p.D / 8;
  const int64_t total = static_cast<int64_t>(p.T) * p.Hkv * 2 * chunks;
  const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= total) return;
  const int chunk = static_cast<int>(idx % chunks);
  int64_t rest = idx / chunks;
  const int which = static_cast<int>(rest & 1);  // 0 = key, 1 = value
  rest >>= 1;
  const int h = static_cast<int>(rest % p.Hkv);
  const int64_t t = rest / p.Hkv;

  const int64_t slot = p.slot_mapping[t];
  if (slot < 0) return;  // padding token
  if (slot >= p.num_blocks * p.bs) {
    if (which == 0 && h == 0 && chunk == 0) atomicOr(p.err, kErrSlot);
    return;
  }
  const int64_t blk = slot / p.bs, off = slot % p.bs;
  const int64_t src = (t * p.Hkv + h) * p.D + chunk * 8;
  const int64_t dst = ((blk * p.Hkv + h) * p.bs + off) * p.D + chunk * 8;
  const uint16_t* in = static_cast<const uint16_t*>(which ? p.value : p.key);
  const uint4 u = *reinterpret_cast<const uint4*>(in + src);
  store_row_piece<TO_FP8>(u, which ? p.v_cache : p.k_cache, dst, p.in_dtype, p.kv_scale);
}

// Check mode of the fused cache write: the new row of token (s, j) goes to
// block slot / bs, which must be private to sequence s (copy-on-write gives a
// sequence its own copy of a shared block before it appends).  One CTA per
// new token scans the live table entries of every other sequence; a match
// means another sequence's CTA may read that block while it is written, and
// sets the slot error bit.
__global__ void __launch_bounds__(256)
    shared_slot_check_kernel(const int64_t* __restrict__ slots, const int32_t* __restrict__ block_tables,
                             const int32_t* __restrict__ context_lens, int S, int qlen, int maxB, int bs,
                             int64_t num_blocks, int* err) {
  const int64_t tok = blockIdx.x;
  const int s = static_cast<int>(tok / qlen);
  const int64_t slot = slots[tok];
  if (slot < 0 || slot >= num_blocks * bs) return;  // padding, or reported by the write itself
  const int blk = static_cast<int>(slot / bs);
  for (int t = 0; t < S; ++t) {
    if (t == s) continue;
    const int L = min(max(context_lens[t], 0), maxB * bs);
    const int nblk = (L + bs - 1) / bs;
    const int32_t* row = block_tables + static_cast<int64_t>(t) * maxB;
    bool hit = false;
    for (int j = threadIdx.x; j < nblk; j += blockDim.x) hit |= __ldg(row + j) == blk;
    if (__syncthreads_or(hit)) {
      if (threadIdx.x == 0) atomicOr(err, kErrSlot);
      return;
    }
  }
}

}  // namespace

cudaError_t launch_shared_slot_check(const int64_t* slots, const int32_t* block_tables, const int32_t* context_lens,
                                     int S, int qlen, int maxB, int bs, int64_t num_blocks, int* err,
                                     cudaStream_t st) {
  const int64_t tokens = static_cast<int64_t>(S) * qlen;
  if (tokens == 0) return cudaSuccess;
  shared_slot_check_kernel<<<static_cast<unsigned>(tokens), 256, 0, st>>>(slots, block_tables, context_lens, S,
                                                                          qlen, maxB, bs, num_blocks, err);
  return cudaGetLastError();
}

cudaError_t launch_reshape_and_cache(const CacheParams& p, cudaStream_t st) {
  const int64_t total = static_cast<int64_t>(p.T) * p.Hkv * 2 * (p.D / 8);
  if (total == 0) return cudaSuccess;
  const unsigned blocks = static_cast<unsigned>((total + 255) / 256);
  if (p.cache_dtype == kE4M3)
    reshape_and_cache_kernel<true><<<blocks, 256, 0, st>>>(p);
  else
    reshape_and_cache_kernel<false><<<blocks, 256, 0, st>>>(p);
  return cudaGetLastError();
}

}  // namespace pa
