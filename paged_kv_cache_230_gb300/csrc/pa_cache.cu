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

}  // namespace

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
