// Log-sum-exp merge of split-decode partials (the second kernel of
// pa_decode_split and pa_decode_multi_split).
#include "pa_decode.cuh"
#include "pa_pdl.cuh"

namespace pa {

// Log-sum-exp merge of the split partials of one (sequence, query head) per
// CTA of 256 threads (one partial (o_p, m_p, l_p) per run of partitions):
// M = max_p m_p,  w_p = 2^(m_p - M),  L = sum_p l_p w_p,  out = sum_p w_p o_p / L.
// The block's threads form groups of D / 4, each thread of a group reading 4
// of a partial's D floats with one 16-byte load; group g folds partials g,
// g + NGRP, ... in that order with a running max (one pass over the partials,
// the loads independent of the max), then the groups are combined in group
// order.  Every sum has a fixed order, so the result is deterministic.
constexpr int kMergeThreads = 256;

template <int D>
__global__ void __launch_bounds__(kMergeThreads) lse_merge_kernel(const DecodeParams p) {
  constexpr int TPG = D / 4;
  constexpr int NGRP = kMergeThreads / TPG;
  __shared__ float4 acc_sh[NGRP][TPG];
  __shared__ float2 ml_sh[NGRP];
  // launched to start while the split kernel ends: its partials are read only
  // after that kernel has completed
  pdl_wait();
  const int row = blockIdx.x;  // (s * qlen + new token) * Hq + query head
  const int s = row / (p.Hq * p.qlen);
  const int lmax = min(p.maxB * p.bs, p.Pmax * p.partition_size);
  const int L = min(max(p.context_lens[s], 0), lmax);
  const int nparts = (L + p.partition_size - 1) / p.partition_size;
  const int np = split_runs(nparts, p.fringe, p.parts_per_cta);  // runs, one partial each
  if (np <= 1) return;  // written directly by the CTA that held every partition
  const int tid = threadIdx.x, grp = tid / TPG, q = tid % TPG;
  const float2* ml = reinterpret_cast<const float2*>(p.ws_ml + static_cast<int64_t>(row) * p.Pmax * 2);
  const float4* o = reinterpret_cast<const float4*>(p.ws_o + static_cast<int64_t>(row) * p.Pmax * D);
  float m = -CUDART_INF_F, l = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
  for (int i = grp; i < np; i += NGRP) {
    const float2 mli = __ldg(ml + i);
    const float4 v = __ldg(o + static_cast<int64_t>(i) * TPG + q);
    const float mn = fmaxf(m, mli.x);
    const float a = m == -CUDART_INF_F ? 0.f : ex2(m - mn);
    const float b = mli.x == -CUDART_INF_F ? 0.f : ex2(mli.x - mn);
    acc.x = acc.x * a + v.x * b;
    acc.y = acc.y * a + v.y * b;
    acc.z = acc.z * a + v.z * b;
    acc.w = acc.w * a + v.w * b;
    l = l * a + mli.y * b;
    m = mn;
  }
  acc_sh[grp][q] = acc;
  if (q == 0) ml_sh[grp] = make_float2(m, l);
  __syncthreads();
  if (tid < TPG) {
    float M = -CUDART_INF_F;
#pragma unroll
    for (int g = 0; g < NGRP; ++g) M = fmaxf(M, ml_sh[g].x);
    float4 t = make_float4(0.f, 0.f, 0.f, 0.f);
    float lsum = 0.f;
#pragma unroll
    for (int g = 0; g < NGRP; ++g) {
      const float w = ml_sh[g].x == -CUDART_INF_F ? 0.f : ex2(ml_sh[g].x - M);
      const float4 u = acc_sh[g][tid];
      t.x += u.x * w;
      t.y += u.y * w;
      t.z += u.z * w;
      t.w += u.w * w;
      lsum += ml_sh[g].y * w;
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
