// Log-sum-exp merge of split-decode partials (the second kernel of
// pa_decode_split and pa_decode_multi_split).
#include "pa_decode.cuh"
#include "pa_pdl.cuh"

namespace pa {

// Log-sum-exp merge of the split partials of one (sequence, query head) per
// CTA of 256 threads (one partial per run of partitions):  M = max_p m_p,  w_p = 2^(m_p - M),  L = sum_p l_p w_p,
// out = sum_p w_p o_p / L.  The partials are spread over the threads, each
// read with 16-byte loads, and every sum is reduced in a fixed order, so the
// result is deterministic.
constexpr int kMergeThreads = 256;
constexpr int kMergeMaxParts = 4096;  // weights kept in shared memory; beyond, recomputed

__device__ __forceinline__ float block_reduce(float v, float* red, bool is_max) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float u = __shfl_xor_sync(0xFFFFFFFFu, v, o);
    v = is_max ? fmaxf(v, u) : v + u;
  }
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float r = red[0];
#pragma unroll
  for (int w = 1; w < kMergeThreads / 32; ++w) r = is_max ? fmaxf(r, red[w]) : r + red[w];
  __syncthreads();
  return r;
}

template <int D>
__global__ void __launch_bounds__(kMergeThreads) lse_merge_kernel(const DecodeParams p) {
  // A partial's D floats are read by D / 4 threads with one 16-byte load
  // each, so a pass of the block reads NGRP partials at once.
  constexpr int TPG = D / 4;
  constexpr int NGRP = kMergeThreads / TPG;
  __shared__ float wsh[kMergeMaxParts];
  __shared__ float red[kMergeThreads / 32];
  __shared__ float4 acc_sh[NGRP][TPG];
  // launched to start while the split kernel ends: its partials are read only
  // after that kernel has completed
  pdl_wait();
  const int row = blockIdx.x;  // (s * qlen + new token) * Hq + query head
  const int s = row / (p.Hq * p.qlen);
  const int lmax = min(p.maxB * p.bs, p.Pmax * p.partition_size);
  const int L = min(max(p.context_lens[s], 0), lmax);
  const int nparts = (L + p.partition_size - 1) / p.partition_size;
  const int np = (nparts + p.parts_per_cta - 1) / p.parts_per_cta;  // runs, one partial each
  if (np <= 1) return;  // written directly by the CTA that held every partition
  const int tid = threadIdx.x;
  const float* ml = p.ws_ml + static_cast<int64_t>(row) * p.Pmax * 2;
  const float4* o = reinterpret_cast<const float4*>(p.ws_o + static_cast<int64_t>(row) * p.Pmax * D);
  float mx = -CUDART_INF_F;
  for (int i = tid; i < np; i += kMergeThreads) mx = fmaxf(mx, ml[2 * i]);
  const float M = block_reduce(mx, red, true);
  float lpart = 0.f;
  for (int i = tid; i < np; i += kMergeThreads) {
    const float w = ex2(ml[2 * i] - M);
    if (i < kMergeMaxParts) wsh[i] = w;
    lpart += ml[2 * i + 1] * w;
  }
  const float lsum = block_reduce(lpart, red, false);  // ends with a barrier: wsh is visible
  const int grp = tid / TPG, q = tid % TPG;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
  for (int i = grp; i < np; i += NGRP) {
    const float w = i < kMergeMaxParts ? wsh[i] : ex2(ml[2 * i] - M);
    const float4 v = __ldg(o + static_cast<int64_t>(i) * TPG + q);
    acc.x += v.x * w;
    acc.y += v.y * w;
    acc.z += v.z * w;
    acc.w += v.w * w;
  }
  acc_sh[grp][q] = acc;
  __syncthreads();
  if (tid < TPG) {
    float4 t = acc_sh[0][tid];
#pragma unroll
    for (int g = 1; g < NGRP; ++g) {
      const float4 u = acc_sh[g][tid];
      t.x += u.x;
      t.y += u.y;
      t.z += u.z;
      t.w += u.w;
    }
    const int64_t o0 = static_cast<int64_t>(row) * D + 4 * tid;
    const bool any = lsum > 0.f;
    store_out(p.out, o0 + 0, p.q_dtype, any ? t.x / lsum : 0.f);
    store_out(p.out, o0 + 1, p.q_dtype, any ? t.y / lsum : 0.f);
    store_out(p.out, o0 + 2, p.q_dtype, any ? t.z / lsum : 0.f);
    store_out(p.out, o0 + 3, p.q_dtype, any ? t.w / lsum : 0.f);
  }
}


cudaError_t launch_lse_merge(const DecodeParams& p, int head_dim, cudaStream_t st) {
  const unsigned grid = static_cast<unsigned>(static_cast<long long>(p.S) * p.qlen * p.Hq);
  // programmatic dependent launch: the merge's CTAs are set up while the split
  // kernel before it on the stream finishes, and wait for its partials
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kMergeThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return head_dim == 64 ? cudaLaunchKernelEx(&cfg, lse_merge_kernel<64>, p)
                        : cudaLaunchKernelEx(&cfg, lse_merge_kernel<128>, p);
}

}  // namespace pa
