// Storing one 16-byte piece (8 channels, 16-bit input) of a new K or V row
// into its cache slot, shared by the scatter kernel and the decode kernel's
// fused cache write.  16-bit caches take the bits as they are; FP8 caches
// store round-to-nearest-even(x / kv_scale) with saturation to the largest
// finite E4M3 value (x widened exactly to float32, IEEE division).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <stdint.h>

#include "pa_internal.h"

namespace pa {

__device__ __forceinline__ float widen16(uint32_t bits, int dtype) {
  return dtype == kF16 ? __half2float(__ushort_as_half(static_cast<uint16_t>(bits)))
                       : __uint_as_float(bits << 16);
}

// `dst` indexes elements of the cache (bytes for FP8, 16-bit words otherwise).
template <bool TO_FP8>
__device__ __forceinline__ void store_row_piece(const uint4 u, void* cache, int64_t dst, int in_dtype,
                                                float kv_scale) {
  if constexpr (!TO_FP8) {
    *reinterpret_cast<uint4*>(static_cast<uint16_t*>(cache) + dst) = u;
  } else {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
    uint32_t packed[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      uint32_t word = 0;
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const uint32_t src2 = w[2 * i + j];
        const float lo = __fdiv_rn(widen16(src2 & 0xFFFFu, in_dtype), kv_scale);
        const float hi = __fdiv_rn(widen16(src2 >> 16, in_dtype), kv_scale);
        const __nv_fp8x2_storage_t two = __nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3);
        word |= static_cast<uint32_t>(two) << (16 * j);
      }
      packed[i] = word;
    }
    *reinterpret_cast<uint2*>(static_cast<uint8_t*>(cache) + dst) = make_uint2(packed[0], packed[1]);
  }
}

}  // namespace pa
