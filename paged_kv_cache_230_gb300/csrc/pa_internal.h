// Internal interface between the C-ABI front end (pa_api.cu) and the kernel
// translation units.  Not installed; not part of the ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace pa {

// Pipeline shape (compile-time; the defaults are the measured best on GB300).
#ifndef PA_CONSUMER_WARPS
#define PA_CONSUMER_WARPS 4
#endif
#ifndef PA_MIN_CTAS_PER_SM
#define PA_MIN_CTAS_PER_SM 3
#endif
constexpr int kConsumerWarps = PA_CONSUMER_WARPS;    // warps that compute
constexpr int kThreads = (kConsumerWarps + 1) * 32;  // + one producer warp
constexpr int kTileTokens = 16 * kConsumerWarps;     // tokens per pipeline stage
constexpr int kMinCtasPerSm = PA_MIN_CTAS_PER_SM;
constexpr int kMaxGroup = 16;                     // largest query group G

enum : int { kF16 = 0, kBF16 = 1, kE4M3 = 2 };

struct DecodeParams {
  void* out;                  // [S, qlen, Hq, D] of q_dtype
  const void* q;              // [S, qlen, Hq, D] of q_dtype
  const int32_t* block_tables;  // [S, maxB]
  const int32_t* context_lens;  // [S]
  float* ws_ml;               // split: [S, qlen, Hq, Pmax, 2] (m, l); nullptr without split
  float* ws_o;                // split: [S, qlen, Hq, Pmax, D]
  int* err;                   // device error word (PA_DEVERR_* bits)
  int64_t num_blocks;
  int S, Hq, Hkv, G, bs, maxB;
  int qlen;                   // new query tokens per sequence (1 = one-token decode)
  int q_dtype;
  int partition_size;         // tokens per partition; 0 = whole context per CTA
  int Pmax;                   // partitions per sequence (1 without split)
  int parts_per_cta;          // split: consecutive partitions streamed by one CTA
  int fringe;                 // split: a context's last partitions run one per CTA
  int nst;                    // ring stages (set by the launcher)
  float scale_log2;           // scale * log2(e)
  float kv_scale;             // FP8 dequantisation scale (1 for 16-bit caches)
  // fused cache write (pa_cache_and_decode); new_key == nullptr: none
  const void* new_key;        // [S * qlen, Hkv, D] of q_dtype
  const void* new_value;
  const int64_t* slot_mapping;  // [S * qlen]
  void* k_cache;              // the pool, written through plain stores
  void* v_cache;
};

// Runs of a split context of P partitions: its first max(P - F, 0)
// partitions in runs of ppc consecutive ones, its last min(P, F) one per run
// (the fringe); an empty context is one empty run.  Run r's partial is
// workspace slot r of each of the context's query rows.
__host__ __device__ inline int split_runs(int P, int F, int ppc) {
  const int bulk = P > F ? P - F : 0;
  const int n = (bulk + ppc - 1) / ppc + (P < F ? P : F);
  return n > 1 ? n : 1;
}
// Split CTAs per (sequence, kv head) in the grid: the bulk runs of the
// longest context, then F fringe runs.
__host__ __device__ inline int split_bulk_ctas(int Pmax, int F, int ppc) {
  return ((Pmax > F ? Pmax - F : 0) + ppc - 1) / ppc;
}

// Launches the decode (or split-partition) kernel for one cache dtype.
// tmK/tmV: 4-D tensor maps over [NB, Hkv, bs, D] with the box and swizzle that
// make_cache_tensor_map (pa_api.cu) chose for this cache dtype and head_dim.
cudaError_t launch_decode_f16(const DecodeParams& p, const CUtensorMap& tmK, const CUtensorMap& tmV,
                              int head_dim, cudaStream_t st);
cudaError_t launch_decode_bf16(const DecodeParams& p, const CUtensorMap& tmK, const CUtensorMap& tmV,
                               int head_dim, cudaStream_t st);
cudaError_t launch_decode_fp8(const DecodeParams& p, const CUtensorMap& tmK, const CUtensorMap& tmV,
                              int head_dim, cudaStream_t st);

// Log-sum-exp merge of split partials into out.
cudaError_t launch_lse_merge(const DecodeParams& p, int head_dim, cudaStream_t st);

struct CacheParams {
  const void* key;
  const void* value;
  void* k_cache;
  void* v_cache;
  const int64_t* slot_mapping;
  int* err;
  int64_t num_blocks;
  int T, Hkv, D, bs;
  int in_dtype, cache_dtype;
  float kv_scale;
};

cudaError_t launch_reshape_and_cache(const CacheParams& p, cudaStream_t st);

// Check mode of pa_cache_and_decode: flags (PA_DEVERR_SLOT) a new row whose
// block is also named by a live table entry of another sequence of the batch.
cudaError_t launch_shared_slot_check(const int64_t* slots, const int32_t* block_tables, const int32_t* context_lens,
                                     int S, int qlen, int maxB, int bs, int64_t num_blocks, int* err,
                                     cudaStream_t st);

// Whole-block moves: op 0 copy (ids = [n][2] pairs), 1 gather into buf,
// 2 scatter from buf.  block_bytes is one block of one cache (a multiple of 16).
cudaError_t launch_block_op(int op, void* buf, void* k_cache, void* v_cache, const int64_t* ids, int n,
                            int64_t block_bytes, int64_t num_blocks, int* err, cudaStream_t st);

}  // namespace pa
