// reshape_and_cache: scatter of this step's new K/V rows into their cache
// slots (blocks are extended by one token per sequence per decode step:
// vLLM review, §6 "KV Cache Block Tables").
//
// One thread moves 8 consecutive channels (one 16-byte load) of one
// (token, kv head, K-or-V) row, so a warp covers whole rows with coalesced
// loads and 16-byte (16-bit cache) or 8-byte (FP8 cache) stores.  Every slot
// is bounds-checked: a slot outside the pool is skipped and recorded.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "pa_internal.h"

namespace pa {

namespace {

constexpr int kErrSlot = 0x4;

__device__ __forceinline__ float widen16(uint32_t bits, int dtype) {
  return dtype == kF16 ? __half2float(__ushort_as_half(static_cast<uint16_t>(bits)))
                       : __uint_as_float(bits << 16);
}

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

  if constexpr (!TO_FP8) {
    uint16_t* cache = static_cast<uint16_t*>(which ? p.v_cache : p.k_cache);
    *reinterpret_cast<uint4*>(cache + dst) = u;
  } else {
    uint8_t* cache = static_cast<uint8_t*>(which ? p.v_cache : p.k_cache);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
    uint32_t packed[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      uint32_t word = 0;
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const uint32_t src2 = w[2 * i + j];
        // float32 widening is exact; the division is IEEE round-to-nearest
        const float lo = __fdiv_rn(widen16(src2 & 0xFFFFu, p.in_dtype), p.kv_scale);
        const float hi = __fdiv_rn(widen16(src2 >> 16, p.in_dtype), p.kv_scale);
        const __nv_fp8x2_storage_t two =
            __nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3);
        word |= static_cast<uint32_t>(two) << (16 * j);
      }
      packed[i] = word;
    }
    *reinterpret_cast<uint2*>(cache + dst) = make_uint2(packed[0], packed[1]);
  }
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
