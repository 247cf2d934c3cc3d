// Widening of a batch's E4M3 K/V blocks to the query's 16-bit type, for the
// prefill path over FP8 caches: every E4M3 code (1 sign, 4 exponent, 3
// mantissa bits, bias 7; quantization, review §10 table) is exactly
// representable in f16 and in bf16, so the widened blocks hold the same
// values and the tensor-core kernels for 16-bit caches run on them unchanged
// (the per-tensor scale is applied to the scores and the output instead).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "pa_widen.h"

namespace pa {

namespace {

constexpr int kWidenThreads = 256;
constexpr int kErrBlockId = 0x1;

// 16 E4M3 codes -> 16 values of 16 bits (32 bytes), in order.
template <bool BF16>
__device__ __forceinline__ void widen16(const uint4 w, uint4& o0, uint4& o1) {
  const uint32_t in[4] = {w.x, w.y, w.z, w.w};
  uint32_t out[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t lo, hi;
    asm("{\n\t.reg .b16 c0, c1;\n\t"
        "mov.b32 {c0, c1}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, c0;\n\t"
        "cvt.rn.f16x2.e4m3x2 %1, c1;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(in[i]));
    if constexpr (BF16) {
      // f16 -> f32 -> bf16: exact, an E4M3 value has at most 4 significant bits
      const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&lo));
      const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&hi));
      const __nv_bfloat162 ba = __floats2bfloat162_rn(a.x, a.y);
      const __nv_bfloat162 bb = __floats2bfloat162_rn(b.x, b.y);
      lo = *reinterpret_cast<const uint32_t*>(&ba);
      hi = *reinterpret_cast<const uint32_t*>(&bb);
    }
    out[2 * i] = lo;
    out[2 * i + 1] = hi;
  }
  o0 = make_uint4(out[0], out[1], out[2], out[3]);
  o1 = make_uint4(out[4], out[5], out[6], out[7]);
}

// CTA = (sequence s, table column j): block j of sequence s, all kv heads, K
// and V, to compact block s * maxB + j; also writes that index into the
// compact table.  Columns past the context only write the table.
template <bool BF16>
__global__ void __launch_bounds__(kWidenThreads) widen_kv_kernel(const WidenParams p) {
  const int64_t slot = blockIdx.x;  // s * maxB + j
  const int s = static_cast<int>(slot / p.maxB), j = static_cast<int>(slot % p.maxB);
  if (threadIdx.x == 0) p.tab[slot] = static_cast<int32_t>(slot);
  const int lmax = p.maxB * p.bs;
  const int L = min(max(__ldg(p.context_lens + s), 0), lmax);
  if (j >= (L + p.bs - 1) / p.bs) return;
  const int phys = __ldg(p.block_tables + slot);
  const bool ok = phys >= 0 && static_cast<int64_t>(phys) < p.num_blocks;
  if (!ok && threadIdx.x == 0) atomicOr(p.err, kErrBlockId);  // read as zeros
  const int64_t bytes = static_cast<int64_t>(p.Hkv) * p.bs * p.D;  // one block of K (or V), E4M3
  const int n16 = static_cast<int>(bytes / 16);
  // four 16-byte loads in flight per thread before any store
  for (int i0 = threadIdx.x; i0 < 2 * n16; i0 += 4 * kWidenThreads) {
    uint4 w[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = i0 + u * kWidenThreads;
      const bool v = i >= n16;
      const int k = v ? i - n16 : i;
      w[u] = (ok && i < 2 * n16) ? __ldg(reinterpret_cast<const uint4*>((v ? p.v_src : p.k_src) + phys * bytes) + k)
                                 : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int i = i0 + u * kWidenThreads;
      if (i >= 2 * n16) break;
      const bool v = i >= n16;
      const int k = v ? i - n16 : i;
      uint4 o0, o1;
      widen16<BF16>(w[u], o0, o1);
      uint4* dst = reinterpret_cast<uint4*>((v ? p.v_dst : p.k_dst) + slot * bytes) + 2 * k;
      dst[0] = o0;
      dst[1] = o1;
    }
  }
}

}  // namespace

cudaError_t launch_widen_kv(const WidenParams& p, cudaStream_t st) {
  const int64_t grid = static_cast<int64_t>(p.S) * p.maxB;
  if (grid <= 0 || grid > INT32_MAX || (static_cast<int64_t>(p.Hkv) * p.bs * p.D) % 16) return cudaErrorInvalidValue;
  if (p.bf16)
    widen_kv_kernel<true><<<static_cast<unsigned>(grid), kWidenThreads, 0, st>>>(p);
  else
    widen_kv_kernel<false><<<static_cast<unsigned>(grid), kWidenThreads, 0, st>>>(p);
  return cudaGetLastError();
}

}  // namespace pa
