// Measurement utility: the rate at which the SMs can read a buffer that sits
// in L2, the bound of a kernel whose bytes come from L2 rather than HBM (a
// pool whose blocks many sequences share, or K/V tiles that several CTAs
// read).  Not part of the attention path.  Two forms of the read:
//   mode 0  plain 16-byte loads cached in L2 only (ld.global.cg), 4 CTAs of
//           512 threads per SM, eight independent loads in flight per thread,
//           each load instruction of a warp covering 512 contiguous bytes;
//   mode 1  TMA boxes of 16 rows x 128 bytes (2 KB, 128-byte swizzle: the box
//           the decode and tensor-core kernels load K/V with), one CTA per
//           SM whose 8 warps issue 2 boxes each per 32 KB stage of a 4-stage
//           ring.
// Mode 0 reads the whole buffer once per pass, each pass starting at another
// offset so that the lines a thread reads change from pass to pass; mode 1's
// CTAs sweep the buffer box by box, stage use u of CTA c taking the 16 boxes
// from (c + u * grid) * 16 on (modulo the buffer).  The checksum of what was
// read is stored only when it equals a fixed pattern, which keeps every load
// without writing anything for a zero-filled buffer.
#include "pa_internal.h"
#include "pa_ptx.cuh"
#include "pagedattn.h"

namespace pa {

namespace {

constexpr uint32_t kSinkPattern = 0x5EED1234u;

__global__ void __launch_bounds__(512) l2_read_plain_kernel(const uint4* __restrict__ buf, int64_t n16, int iters,
                                                             uint32_t* sink) {
  const int64_t nthr = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int64_t me = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  uint32_t acc[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
  for (int it = 0; it < iters; ++it) {
    // pass `it` starts it * 7919 * 64 vectors further in (modulo the buffer)
    const int64_t shift = (static_cast<int64_t>(it) * 7919 * 64) % n16;
    int64_t i0 = 0;
    for (; i0 + 8 * nthr <= n16; i0 += 8 * nthr) {
      uint4 v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        int64_t j = i0 + u * nthr + me + shift;
        if (j >= n16) j -= n16;
        v[u] = __ldcg(buf + j);
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) acc[u] ^= v[u].x ^ v[u].y ^ v[u].z ^ v[u].w;
    }
    for (int64_t i = i0 + me; i < n16; i += nthr) {  // the rest of the pass
      int64_t j = i + shift;
      if (j >= n16) j -= n16;
      const uint4 v = __ldcg(buf + j);
      acc[0] ^= v.x ^ v.y ^ v.z ^ v.w;
    }
  }
  uint32_t a = 0;
#pragma unroll
  for (int u = 0; u < 8; ++u) a ^= acc[u];
  if (a == kSinkPattern) *sink = a;
}

constexpr int kBoxRows = 16, kBoxBytes = kBoxRows * 128, kStageBytes = 32768, kStages = 4;
constexpr int kTmaWarps = 8;  // x 2 lanes = the 16 boxes of a stage

// 2-D tiled TMA load of one box into shared memory, completion as
// transaction bytes on `bar`.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* m, uint32_t bar, int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}

__global__ void __launch_bounds__(kTmaWarps * 32, 1) l2_read_tma_kernel(const __grid_constant__ CUtensorMap map,
                                                                         int nrows, int iters, uint32_t* sink,
                                                                         int* err) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t base = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (base & 1023u) {
    if (threadIdx.x == 0) atomicOr(err, PA_DEVERR_LAYOUT);
    return;
  }
  const uint32_t bars = base + kStages * kStageBytes;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(bars + 8 * s, 1);
    fence_mbar_init();
  }
  __syncthreads();
  // box b of this CTA's stage use u: 128-byte rows from
  // ((cta + u * grid) * 16 + b) * 16 on, modulo the buffer's row count
  const int boxes = kStageBytes / kBoxBytes;  // 16 per stage
  const int nbox_rows = nrows / kBoxRows;
  bool ok = true;
  int u = 0;
  for (; u < iters; ++u) {
    const int st = u % kStages;
    if (u >= kStages && !__all_sync(0xFFFFFFFFu, mbar_wait(bars + 8 * st, ((u / kStages) - 1) & 1))) {
      ok = false;
      break;
    }
    if (warp == 0 && lane == 0) mbar_arrive_expect_tx(bars + 8 * st, kStageBytes);
    __syncwarp();
    if (lane < 2) {
      const int b = warp * 2 + lane;  // 0..15
      const int64_t unit = (static_cast<int64_t>(blockIdx.x) + static_cast<int64_t>(u) * gridDim.x) * boxes + b;
      const int row = static_cast<int>(unit % nbox_rows) * kBoxRows;
      tma_load_2d(base + st * kStageBytes + b * kBoxBytes, &map, bars + 8 * st, 0, row);
    }
  }
  // every box issued lands before the CTA exits
  for (int v = max(0, u - kStages); v < u; ++v) mbar_wait(bars + 8 * (v % kStages), (v / kStages) & 1);
  __syncthreads();
  if (!ok && threadIdx.x == 0) atomicOr(err, PA_DEVERR_TIMEOUT);
  if (threadIdx.x == 0) {
    const uint32_t a = *reinterpret_cast<const volatile uint32_t*>(smem);
    if (a == kSinkPattern) *sink = a;
  }
}

}  // namespace

cudaError_t launch_l2_read_plain(const void* buf, size_t bytes, int iters, void* sink, int nsm, cudaStream_t st) {
  l2_read_plain_kernel<<<4 * nsm, 512, 0, st>>>(static_cast<const uint4*>(buf), static_cast<int64_t>(bytes / 16),
                                                iters, static_cast<uint32_t*>(sink));
  return cudaGetLastError();
}

cudaError_t launch_l2_read_tma(const CUtensorMap& map, int nrows, int iters, void* sink, int* err, int nsm,
                               cudaStream_t st) {
  const int smem = kStages * kStageBytes + 8 * kStages;
  cudaError_t e = cudaFuncSetAttribute(l2_read_tma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  l2_read_tma_kernel<<<nsm, kTmaWarps * 32, smem, st>>>(map, nrows, iters, static_cast<uint32_t*>(sink), err);
  return cudaGetLastError();
}

}  // namespace pa
