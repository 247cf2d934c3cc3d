// Internal interface of the tensor-core paged attention kernel (tcgen05
// path): chunked prefill, and multi-token decode whose query group is too
// wide for the warp-MMA decode kernel.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace pa {

constexpr int kTcRows = 128;        // query rows per tile (MMA M, TMEM lanes)
constexpr int kTcTok = 128;         // KV tokens per tile (N of Q.K^T, K of P.V)
constexpr int kTcThreads = 512;     // two softmax, one epilogue, one load/MMA warpgroup
constexpr int kTcMaxSlots = 8;      // K/V ring slots at most
constexpr int kTcMaxRanked = 128;   // work items per CTA ordered longest-first at most
constexpr int kTcMaxGroup = 128;    // query heads per kv head at most (one head per row)

// One work item: (sequence, kv head, query tile, run of partitions).  A
// query tile holds T consecutive new tokens x the G query heads of the kv
// head, packed as row = token * G + head (T * G <= 128 rows), so every K/V
// tile a CTA loads serves all of them.
struct TcParams {
  void* out;                    // [S, C, Hq, D] of the q dtype
  const int32_t* block_tables;  // [S, maxB]
  const int32_t* context_lens;  // [S] (counts the C new tokens)
  float* ws_o;                  // split: partial outputs [S * C * Hq, Pmax, D]
  float* ws_ml;                 // split: (m, l) [S * C * Hq, Pmax, 2]
  int* err;                     // device error word
  int64_t num_blocks;
  int S, C, Hq, Hkv, G, bs, maxB, D;
  int T;               // new tokens per query tile
  int n_qt;            // query tiles per (sequence, kv head)
  int R;               // runs per sequence (1 without split)
  int partition_size;  // split: tokens per partition (0: whole context per item)
  int Pmax;            // split: partitions per sequence at most
  int ppc;             // split: partitions per run
  int nslot;           // K/V ring slots
  int nqb;             // query tile buffers in shared memory (1 or 2)
  int rank_seqs;       // 1: items ordered by context length, longest first
  int bf16;            // MMA operands (q, K, V, P): 1 bf16, 0 f16
  int out_bf16;        // output (and q) dtype: 1 bf16, 0 f16
  int fp8;             // 1: E4M3 caches, widened to f16 in shared memory
  int q_scale_rows;    // 1: bf16 q rounded to f16 per row after scaling by 2^e (FP8 caches)
  int total;           // work items
  float scale_log2;    // softmax scale * log2(e) (* kv_scale for FP8 caches)
  float vscale;        // kv_scale for FP8 caches, 1 otherwise
};

// Ring slots and dynamic shared memory for a launch with head_dim D,
// 16-bit (fp8 = 0) or E4M3 (fp8 = 1) caches and nqb query tile buffers.
int tc_ring_slots(int D, int fp8, int nqb);
int tc_smem_bytes(int D, int nslot, int fp8, int nqb);

// tmQ: 3-D map over q {D, Hq, S * C}, box {64, G, T}, 128-byte swizzle;
// tmK / tmV: the caches' 4-D maps (16-bit: box {64, bs, 1, 1}, 128-byte
// swizzle; E4M3: box {D, bs, 1, 1}, 128-byte swizzle for D = 128, 64-byte
// for D = 64).
cudaError_t launch_attn_tc(const TcParams& p, const CUtensorMap& tmQ, const CUtensorMap& tmK,
                           const CUtensorMap& tmV, cudaStream_t st);

}  // namespace pa
