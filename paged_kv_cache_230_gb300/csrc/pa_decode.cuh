// Paged decode attention kernels for sm_103a.
//
// Work unit: one CTA per (sequence s, kv head h) — or per (s, h, partition)
// in the split variant.  The CTA streams the K and V rows of its token range
// through a ring of shared-memory stages exactly once and serves all G query
// heads that read kv head h (decode reads the full KV cache once per step and
// is bandwidth bound: vLLM review, §7).
//
//   warp 4 (producer): walks the block table (logical block j -> physical
//     block id, review §6 "KV Cache Block Tables"), 32 entries per coalesced
//     load, and issues one 4-D TMA tile load per (block, 128-byte segment) for
//     K and for V into the next free stage.  TMA writes the tile with the
//     128-byte (or 64-byte) swizzle so the consumers' row reads are free of
//     bank conflicts.  A block id outside the pool is a TMA out-of-bounds box
//     and reads zeros.
//   warps 0-3 (consumers): each owns 16 consecutive tokens of every stage and
//     keeps its own running max m, running sum l and output accumulator for
//     the G query heads (online softmax, base 2: scores are pre-scaled by
//     log2 e).  After the last stage the four partial states are merged in a
//     fixed order, so the result depends only on logical token positions —
//     never on where blocks sit in the pool or on timing.
//
// Group product.  For G >= 4 the per-warp work is two warp MMAs per 16 tokens
// (m16n8k16, fp32 accumulate):  S^T[16 tok x 8 heads] = K[16 x D] Q^T and
// O^T[D x 8 heads] += V^T[D x 16 tok] P^T, with the query group padded to 8
// (or 16) columns.  For G <= 3 (too narrow to be a dense contraction) each
// token row is split over 8 lanes that form dot products with warp shuffles.
//
// FP8 E4M3 caches: codes are widened exactly to f16 in registers and the MMA
// runs in f16.  q is scaled by a power of two 2^e chosen per CTA so that
// max|q| * 2^e lies in [2^14, 2^15) before its f16 rounding, which keeps the
// f16 copy exact except for entries below 2^-29 max|q|; 2^-e and kv_scale are
// folded into the score multiplier and kv_scale into the output.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <math_constants.h>

#include "pa_cache_row.cuh"
#include "pa_internal.h"
#include "pa_ptx.cuh"

namespace pa {

constexpr int kErrBlockId = 0x1;
constexpr int kErrContextLen = 0x2;
constexpr int kErrSlot = 0x4;
constexpr int kErrTimeout = 0x8;

template <int KV, int D>
struct Geom {
  static constexpr int EB = (KV == kE4M3) ? 1 : 2;         // bytes per element
  static constexpr int ROWB = D * EB;                       // bytes per token row
  static constexpr int BOXB = ROWB < 128 ? ROWB : 128;      // bytes per TMA box row
  static constexpr int BOXE = BOXB / EB;                    // elements per box row
  static constexpr int NSEG = ROWB / BOXB;                  // boxes per token row
  static constexpr int SWZ = (BOXB == 128) ? 0x70 : 0x30;   // swizzle XOR mask (bits 4-6 / 4-5)
  static constexpr int SEG_BYTES = kTileTokens * BOXB;
  static constexpr int HALF_BYTES = NSEG * SEG_BYTES;       // K (or V) bytes per stage
  static constexpr int STAGE_BYTES = 2 * HALF_BYTES;
  static_assert(SEG_BYTES % 1024 == 0, "segments must keep the swizzle atom alignment");
};

// Byte offset inside a swizzled segment: the 16-byte chunk index (bits 4-6,
// or 4-5) is XORed with the row index bits (7-9, or 7-8), as TMA writes it.
template <class Gm>
__device__ __forceinline__ uint32_t swz(uint32_t off) {
  return off ^ ((off >> 3) & Gm::SWZ);
}

// Dynamic shared memory of one CTA: alignment slack, the ring of `nst`
// stages, the [NG][D] output area (q staging at start-up), the ring's
// mbarriers, the warps' (m, l), the run's (m, l) and, in the split variant
// only, the run accumulator [NG][D] (last, so one-pass launches omit it).
template <int NG, int D>
__host__ __device__ constexpr int decode_smem_bytes_for(int ring, int nst, bool split) {
  return 1024 + ring + NG * D * 4 + 4 * nst * 8 + kConsumerWarps * NG * 2 * 4 + 2 * NG * 2 * 4 +
         (split ? NG * D * 4 : 0);
}

__device__ __forceinline__ float load_q(const void* q, int64_t idx, int q_dtype) {
  const uint16_t bits = static_cast<const uint16_t*>(q)[idx];
  return q_dtype == kF16 ? __half2float(__ushort_as_half(bits)) : __uint_as_float(uint32_t(bits) << 16);
}

__device__ __forceinline__ void store_out(void* out, int64_t idx, int q_dtype, float v) {
  uint16_t bits = q_dtype == kF16 ? __half_as_ushort(__float2half_rn(v))
                                  : __bfloat16_as_ushort(__float2bfloat16_rn(v));
  static_cast<uint16_t*>(out)[idx] = bits;
}

template <bool IS_BF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  if constexpr (IS_BF16) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  } else {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  }
}

// Four E4M3 codes (low byte = first element) widened exactly to two f16x2
// words: codes 0, 1 to `lo`, codes 2, 3 to `hi`.  The conversion instruction
// reads each 16-bit half directly; masking and shifting the word for a
// conversion helper cost as much as the conversions.
__device__ __forceinline__ void e4m3x4_to_f16x2x2(uint32_t four, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b16 c0, c1;\n\t"
      "mov.b32 {c0, c1}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, c0;\n\t"
      "cvt.rn.f16x2.e4m3x2 %1, c1;\n\t}"
      : "=r"(lo), "=r"(hi) : "r"(four));
}

// Zero the halves of an A fragment whose token index (k) is >= n_valid.
// a[0], a[1] hold tokens 2c, 2c+1; a[2], a[3] hold tokens 8+2c, 9+2c (c = lane % 4).
__device__ __forceinline__ void mask_tokens(uint32_t (&a)[4], int lane, int n_valid) {
  const int t0 = 2 * (lane & 3);
  const uint32_t m_lo = (t0 < n_valid ? 0x0000FFFFu : 0u) | (t0 + 1 < n_valid ? 0xFFFF0000u : 0u);
  const uint32_t m_hi = (t0 + 8 < n_valid ? 0x0000FFFFu : 0u) | (t0 + 9 < n_valid ? 0xFFFF0000u : 0u);
  a[0] &= m_lo;
  a[1] &= m_lo;
  a[2] &= m_hi;
  a[3] &= m_hi;
}

// Two 16x16 matrices of bytes, transposed: lanes 0-15 give the 16-byte row
// addresses of the first, lanes 16-31 those of the second; lane (g = lane / 4,
// c = lane % 4) receives, per matrix, column g then column g + 8 of the stored
// rows 4c .. 4c+3 (lowest byte = row 4c).
__device__ __forceinline__ void ldsm_b8_x2_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                             uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m16n16.x2.trans.shared.b8 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// FP8 sub-tiles order their 16 tokens so that the transposing byte load of V
// lines up with the f16 MMA: S^T row (= k index of P) r holds token
// tok_perm(r), which puts tokens 4c .. 4c+3 at k = 2c, 2c+1, 2c+8, 2c+9.
__device__ __forceinline__ int tok_perm(int r) { return 4 * ((r & 7) >> 1) + (r & 1) + 2 * (r >> 3); }

// Zero the E4M3 codes of tokens >= n_valid in a word holding tokens 4c .. 4c+3
// (lowest byte first, c = lane % 4); a zero code is +0.
__device__ __forceinline__ uint32_t token_byte_mask(int lane, int n_valid) {
  const int nv = n_valid - 4 * (lane & 3);
  return nv >= 4 ? 0xFFFFFFFFu : (nv <= 0 ? 0u : (1u << (8 * nv)) - 1u);
}

// Widen one lane's piece of a token row (PB bytes at a 16- or 8-byte aligned
// shared address) to floats.
template <int KV, int PB>
__device__ __forceinline__ void load_piece(const uint8_t* src, float* f) {
  if constexpr (PB == 16) {
    const uint4 u = *reinterpret_cast<const uint4*>(src);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
    if constexpr (KV == kF16) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 v = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
        f[2 * i] = v.x;
        f[2 * i + 1] = v.y;
      }
    } else if constexpr (KV == kBF16) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
      }
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        uint32_t h2[2];
        e4m3x4_to_f16x2x2(w[i], h2[0], h2[1]);
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const float2 v = __half22float2(*reinterpret_cast<const __half2*>(&h2[j]));
          f[4 * i + 2 * j] = v.x;
          f[4 * i + 2 * j + 1] = v.y;
        }
      }
    }
  } else {
    static_assert(KV == kE4M3, "8-byte pieces only occur for FP8 rows of 64 bytes");
    const uint2 u = *reinterpret_cast<const uint2*>(src);
    const uint32_t w[2] = {u.x, u.y};
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      uint32_t h2[2];
      e4m3x4_to_f16x2x2(w[i], h2[0], h2[1]);
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const float2 v = __half22float2(*reinterpret_cast<const __half2*>(&h2[j]));
        f[4 * i + 2 * j] = v.x;
        f[4 * i + 2 * j + 1] = v.y;
      }
    }
  }
}

// Dispatch order.  CTAs start roughly in blockIdx order, so handing the
// longest contexts to the first CTAs gives longest-first list scheduling and
// removes the tail where a long sequence starts late.  Lengths are ranked by
// a 128-bucket key (4 buckets per power of two), descending, ties by sequence
// index; CTA rank r processes the sequence of rank r.  Computed by every CTA
// from context_lens with one histogram and one block-wide scan (no scratch
// memory), identically in all CTAs, so the mapping is a permutation.
constexpr int kOrderBuckets = 128;

__device__ __forceinline__ int length_bucket_desc(int L) {
  if (L <= 0) return kOrderBuckets - 1;
  const int msb = 31 - __clz(L);
  const int frac = msb >= 2 ? (L >> (msb - 2)) & 3 : (L << (2 - msb)) & 3;
  return kOrderBuckets - 1 - min(msb * 4 + frac, kOrderBuckets - 1);
}

// All kThreads threads call this; returns the sequence of rank r.
__device__ __noinline__ static int seq_of_rank(const int32_t* __restrict__ context_lens, int S, int r) {
  __shared__ int hist[kOrderBuckets];
  __shared__ int warp_tot[kThreads / 32];
  __shared__ int sel[3];  // bucket, index inside the bucket, chosen sequence
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int i = tid; i < kOrderBuckets; i += kThreads) hist[i] = 0;
  if (tid == 0) sel[2] = min(r, S - 1);
  __syncthreads();
  const int per = (S + kThreads - 1) / kThreads;  // contiguous chunk of sequences per thread
  const int s0 = min(S, tid * per), s1 = min(S, s0 + per);
  for (int i = 0; i < per; ++i) {  // same trip count in every lane: one atomic per distinct bucket
    const int s = s0 + i;
    const int b = s < s1 ? length_bucket_desc(__ldg(context_lens + s)) : -1;
    const unsigned same = __match_any_sync(0xFFFFFFFFu, b);
    if (b >= 0 && lane == __ffs(same) - 1) atomicAdd(&hist[b], __popc(same));
  }
  __syncthreads();
  if (warp == 0) {
    // exclusive scan of the histogram (4 buckets per lane), then locate r
    int c[4], run = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      c[k] = hist[lane * 4 + k];
      run += c[k];
    }
    int incl = run;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += v;
    }
    int base = incl - run;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      if (r >= base && r < base + c[k]) {
        sel[0] = lane * 4 + k;
        sel[1] = r - base;
      }
      base += c[k];
    }
  }
  __syncthreads();
  const int bucket = sel[0], want = sel[1];
  int mine = 0;
  for (int s = s0; s < s1; ++s) mine += length_bucket_desc(__ldg(context_lens + s)) == bucket;
  int incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  int before = incl - mine;
  for (int w = 0; w < warp; ++w) before += warp_tot[w];
  if (want >= before && want < before + mine) {
    int k = want - before;
    for (int s = s0; s < s1; ++s) {
      if (length_bucket_desc(__ldg(context_lens + s)) == bucket) {
        if (k == 0) {
          sel[2] = s;
          break;
        }
        --k;
      }
    }
  }
  __syncthreads();
  return min(max(sel[2], 0), S - 1);
}

// Query columns of a CTA: column n is query token n / G (of qlen new tokens)
// and query head h * G + n % G; its row in q / out [S, qlen, Hq, D].
__device__ __forceinline__ int64_t query_row(const DecodeParams& p, int s, int h, int n) {
  return (static_cast<int64_t>(s) * p.qlen + n / p.G) * p.Hq + h * p.G + n % p.G;
}

// Combination of the consumer warps' partial states for one segment (the
// whole token range, or one 512-token partition in the split variant).
// Every warp has written its (m, l) per head to ml[w][g]; the warps then add
// their rescaled outputs 2^(m_w - M) o_w into `area` ([NG][D] floats) one
// after the other in warp order (`add_mine` is called by warp w on its turn).
// Then, per output element:
//  - one-pass decode, or a context whose partitions all belong to this CTA:
//    the partition partials are folded into the run accumulator (`carea`,
//    `cml`) by log-sum-exp, and the last segment writes o / l;
//  - otherwise the run's log-sum-exp of its partitions is written to the
//    workspace as one partial (slot = this CTA's run), merged later by
//    lse_merge_kernel.  The two levels together are the log-sum-exp merge of
//    all 512-token partitions, in a fixed order.
struct SegInfo {
  int seg;        // segment index inside this CTA's run
  bool last;      // last segment of the run
  bool split;     // split variant
  bool final_out; // this CTA writes the normalised output
  int chunk;      // the run's index (workspace slot)
};

template <int D, int NG, class AddMine>
__device__ __forceinline__ void segment_epilogue(const DecodeParams& p, int cw, int ctid, float* area,
                                                 float* carea, float* cml, const float* ml, int s, int h,
                                                 const SegInfo& si, float vscale, AddMine add_mine) {
  constexpr int NCW = kConsumerWarps;
  named_bar_sync(1, NCW * 32);  // every warp's (m, l) is visible
#pragma unroll 1
  for (int w = 0; w < NCW; ++w) {
    if (cw == w) add_mine(w == 0);
    named_bar_sync(1, NCW * 32);
  }
  const float* cml_in = cml + ((si.seg + 1) & 1) * NG * 2;  // run state before this segment
  float* cml_out = cml + (si.seg & 1) * NG * 2;
  for (int idx = ctid; idx < p.G * p.qlen * D; idx += NCW * 32) {
    const int g = idx / D, d = idx % D;
    float M = -CUDART_INF_F;
#pragma unroll
    for (int w = 0; w < NCW; ++w) M = fmaxf(M, ml[(w * NG + g) * 2]);
    float lsum = 0.f;
    if (M != -CUDART_INF_F) {
#pragma unroll
      for (int w = 0; w < NCW; ++w) lsum += ml[(w * NG + g) * 2 + 1] * ex2(ml[(w * NG + g) * 2] - M);
    }
    float acc = area[g * D + d] * vscale;
    const int64_t row = query_row(p, s, h, g);
    if (si.split) {
      // fold this partition into the run: log-sum-exp of (run so far, partition)
      if (si.seg > 0) {
        const float Mc = cml_in[2 * g], Lc = cml_in[2 * g + 1];
        const float M2 = fmaxf(Mc, M);
        const float fa = Mc == -CUDART_INF_F ? 0.f : ex2(Mc - M2);
        const float fb = M == -CUDART_INF_F ? 0.f : ex2(M - M2);
        acc = carea[g * D + d] * fa + acc * fb;
        lsum = Lc * fa + lsum * fb;
        M = M2;
      }
      if (!si.last) {
        carea[g * D + d] = acc;
        if (d == 0) {
          cml_out[2 * g] = M;
          cml_out[2 * g + 1] = lsum;
        }
        continue;
      }
    }
    if (si.final_out) {
      store_out(p.out, row * D + d, p.q_dtype, lsum > 0.f ? acc / lsum : 0.f);
    } else {
      const int64_t slot = row * p.Pmax + si.chunk;
      p.ws_o[slot * D + d] = acc;
      if (d == 0) {
        p.ws_ml[2 * slot] = M;
        p.ws_ml[2 * slot + 1] = lsum;
      }
    }
  }
  named_bar_sync(1, NCW * 32);  // area, carea and ml may be reused
}

// Scale factor of warp w's state for head g: 2^(m_w - M), M = max over warps.
template <int NG>
__device__ __forceinline__ float warp_factor(const float* ml, int w, int g) {
  float M = -CUDART_INF_F;
#pragma unroll
  for (int v = 0; v < kConsumerWarps; ++v) M = fmaxf(M, ml[(v * NG + g) * 2]);
  return M == -CUDART_INF_F ? 0.f : ex2(ml[(w * NG + g) * 2] - M);
}

// CTAs per SM the register budget is sized for: the 3-head shuffle variant
// with 128 channels holds too many accumulators for three (the 16-column MMA
// variant splits its columns over warp pairs instead).  The E4M3 MMA variants
// with 128 channels run four: their consumer warps, not the loads, bound them
// (conversions and MMAs per byte are twice bf16's), an E4M3 stage is half the
// bytes, so four rings fit, and the fourth CTA's warps hide more of the
// dependent conversion -> MMA chains than the registers it costs (at most
// 102 per thread) lose.
template <int KV, int D, bool USE_MMA, int NG>
constexpr int decode_min_ctas() {
  if (KV == kE4M3 && USE_MMA && D == 128) return kMinCtasPerSm < 4 ? kMinCtasPerSm + 1 : kMinCtasPerSm;
  return (!USE_MMA && NG > 1 && D > 64) ? (kMinCtasPerSm < 2 ? kMinCtasPerSm : 2) : kMinCtasPerSm;
}

template <int KV, int D, bool USE_MMA, int NG>
__global__ void __launch_bounds__(kThreads, (decode_min_ctas<KV, D, USE_MMA, NG>()))
    decode_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                  const DecodeParams p) {
  using Gm = Geom<KV, D>;
  const int NST = p.nst;  // ring stages, chosen per launch from the shared-memory budget
  const int RING = NST * Gm::STAGE_BYTES;
  constexpr int NCW = kConsumerWarps;
  constexpr int TILE = kTileTokens;
  // K and V halves of a stage released separately: the 16-column MMA variant
  // on 16-bit caches, whose consumers take longest per stage (the other
  // variants measured faster with one barrier pair per stage)
  constexpr bool SPLITKV = USE_MMA && NG == 16 && KV != kE4M3;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_u32 & 1023u)) & 1023u);
  const uint32_t ring_u32 = smem_u32(smem);
  // q staging at start-up, then the epilogue's output area: [NG][D] floats
  float* qbuf = reinterpret_cast<float*>(smem + RING);
  float* area = qbuf;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + RING + NG * D * 4);
  float* ml = reinterpret_cast<float*>(bars + 4 * NST);  // [NCW][NG][2]
  float* cml = ml + NCW * NG * 2;                         // [2][NG][2] run (m, l), double-buffered
  // [NG][D] run accumulator: split variant only (not allocated otherwise)
  float* carea = reinterpret_cast<float*>(smem + RING + NG * D * 4 + 4 * NST * 8 + (NCW + 2) * NG * 2 * 4);
  // per stage: K (or K and V) landed, V landed, K (or K and V) free, V free.
  // With SPLITKV the K half is released as soon as the scores are formed, so
  // the next K streams in during the softmax and P.V of the stage
  const uint32_t fullk0 = smem_u32(bars), fullv0 = fullk0 + NST * 8;
  const uint32_t emptyk0 = fullv0 + NST * 8, emptyv0 = emptyk0 + NST * 8;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // ---- which (sequence, kv head, run of partitions) ----
  // Split variant: the grid's first S * Hkv * nb CTAs take the bulk runs (CTA
  // c of a (sequence, kv head) streams partitions [c * ppc, (c + 1) * ppc) of
  // the context's first P - F back to back), the last S * Hkv * F CTAs the
  // fringe: each of a context's last F partitions alone.  CTAs start roughly
  // in index order, so the runs that end the launch are single partitions.
  const bool split = p.partition_size > 0;
  const int F = split ? p.fringe : 0;
  const int nb = split ? split_bulk_ctas(p.Pmax, F, p.parts_per_cta) : 1;
  int bid = blockIdx.x;
  const bool fringe = bid >= p.S * p.Hkv * nb;
  int chunk;  // bulk run index, or fringe index j in [0, F)
  if (!fringe) {
    chunk = bid % nb;
    bid /= nb;
  } else {
    bid -= p.S * p.Hkv * nb;
    chunk = bid % F;
    bid /= F;
  }
  const int h = bid % p.Hkv;
  const int s = p.S > 1 ? seq_of_rank(p.context_lens, p.S, bid / p.Hkv) : 0;
  int lmax = p.maxB * p.bs;
  if (split) lmax = min(lmax, p.Pmax * p.partition_size);
  int L = p.context_lens[s];
  // the first CTA of the (sequence, kv head 0): bulk run 0, or the last fringe
  // CTA when there is no bulk
  const bool lead = h == 0 && (nb > 0 ? !fringe && chunk == 0 : chunk == F - 1);
  if (L < 0 || L > lmax) {
    if (tid == 0 && lead) atomicOr(p.err, kErrContextLen);
    L = min(max(L, 0), lmax);
  }
  int tok_begin = 0, tok_end = L, run = 0, nruns = 1;
  if (split) {
    const int ps = p.partition_size, ppc = p.parts_per_cta;
    const int P = (L + ps - 1) / ps;
    const int bulk_end = max(P - F, 0);
    nruns = split_runs(P, F, ppc);
    // an empty context is one empty run: bulk run 0, or the last fringe CTA
    // without a fringe
    const bool empty_owner = P == 0 && (F == 0 ? !fringe && chunk == 0 : fringe && chunk == F - 1);
    int first = 0, last = 0;  // partitions [first, last)
    if (!empty_owner) {
      if (!fringe) {
        first = chunk * ppc;
        if (first >= bulk_end) return;  // past this context's bulk
        last = min(first + ppc, bulk_end);
        run = chunk;
      } else {
        first = P - F + chunk;
        if (first < 0) return;  // the context has fewer than F partitions
        last = first + 1;
        run = (bulk_end + ppc - 1) / ppc + (first - bulk_end);
      }
    }
    tok_begin = first * ps;
    tok_end = min(L, last * ps);
  }
  // this CTA holds every partition of the context: it writes the final output
  const bool final_out = !split || nruns == 1;
  const int ntiles = tok_end > tok_begin ? (tok_end - tok_begin + TILE - 1) / TILE : 0;
  const int tiles_per_seg = split ? p.partition_size / TILE : max(ntiles, 1);

  if (tid == 0) {
    for (int i = 0; i < NST; ++i) {
      mbar_init(fullk0 + 8 * i, 1);
      mbar_init(fullv0 + 8 * i, 1);
      mbar_init(emptyk0 + 8 * i, NCW);
      mbar_init(emptyv0 + 8 * i, NCW);
    }
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == NCW) {
    // ======================= producer warp =======================
    if (ntiles == 0) return;
    if (lane == 0) {
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
    }
    const int bs = p.bs;
    const int* bt_row = p.block_tables + static_cast<int64_t>(s) * p.maxB;
    const int blk_begin = tok_begin / bs;
    const int blk_end = (tok_end + bs - 1) / bs;
    const int bpt = TILE / bs;  // blocks per stage
    const uint32_t tx = static_cast<uint32_t>(bs * Gm::ROWB);  // one block of K (or V)
    int base = blk_begin;
    int cur = (base + lane < blk_end) ? __ldg(bt_row + base + lane) : -1;
    int nxt = (base + 32 + lane < blk_end) ? __ldg(bt_row + base + 32 + lane) : -1;
    if (p.new_key != nullptr) {
      // fused cache write: this CTA's own new rows (position L - qlen + j of
      // sequence s, kv head h, inside its token range) go to their slots
      // before any tile load reads the pool.  A slot that is not that
      // position's slot in the sequence's own table is written as given and
      // flagged (the tile loads would not see it).
      constexpr int kPieces = D / 8;  // 16-byte pieces of a 16-bit row
      for (int i = lane; i < p.qlen * 2 * kPieces; i += 32) {
        const int piece = i % kPieces, which = (i / kPieces) & 1, j = i / (2 * kPieces);
        const int pos = L - p.qlen + j;
        if (pos < tok_begin || pos >= tok_end) continue;  // before the context, or another run's part
        const int64_t tok = static_cast<int64_t>(s) * p.qlen + j;
        const int64_t slot = p.slot_mapping[tok];
        if (slot < 0) continue;  // padding token
        const bool first = piece == 0 && which == 0;
        if (slot >= p.num_blocks * bs) {
          if (first) atomicOr(p.err, kErrSlot);
          continue;
        }
        if (first && slot != static_cast<int64_t>(__ldg(bt_row + pos / bs)) * bs + pos % bs) atomicOr(p.err, kErrSlot);
        const int64_t blk = slot / bs, off = slot % bs;
        const uint16_t* in = static_cast<const uint16_t*>(which ? p.new_value : p.new_key);
        const uint4 u = *reinterpret_cast<const uint4*>(in + (tok * p.Hkv + h) * D + piece * 8);
        store_row_piece<KV == kE4M3>(u, which ? p.v_cache : p.k_cache, ((blk * p.Hkv + h) * bs + off) * D + piece * 8,
                                     p.q_dtype, p.kv_scale);
      }
      // the plain stores are visible to the tile loads (async proxy) issued next
      asm volatile("fence.proxy.async.global;" ::: "memory");
      __syncwarp();
    }
    int t = 0, nk = 0, nv = 0;  // tiles started; K and V halves issued
    bool ok = true;
    for (; t < ntiles; ++t) {
      const int stage = t % NST;
      if (t >= NST && !mbar_wait(emptyk0 + 8 * stage, ((t / NST) - 1) & 1)) {
        ok = false;
        break;
      }
      const int b0 = blk_begin + t * bpt;
      const int nb = min(bpt, blk_end - b0);
      const uint32_t kdst0 = ring_u32 + stage * Gm::STAGE_BYTES;
      // one lane per block of the stage (at most 64 / 8), so the warp issues
      // every block's tile loads together; issuing them from one lane after
      // another capped the rate at which a CTA could stream
      while (b0 >= base + 32) {
        base += 32;
        cur = nxt;
        nxt = (base + 32 + lane < blk_end) ? __ldg(bt_row + base + 32 + lane) : -1;
      }
      const int rel = b0 + lane - base;  // table window index, below 64 for lane < nb
      const int pc = __shfl_sync(0xFFFFFFFFu, cur, rel & 31);
      const int pn = __shfl_sync(0xFFFFFFFFu, nxt, rel & 31);
      const int phys = rel < 32 ? pc : pn;
      const uint32_t kdst = kdst0 + lane * bs * Gm::BOXB;
      const uint32_t fk = fullk0 + 8 * stage;
      if (lane == 0) mbar_arrive_expect_tx(fk, (SPLITKV ? tx : 2 * tx) * nb);
      if (lane < nb) {
        if (phys < 0 || static_cast<int64_t>(phys) >= p.num_blocks) atomicOr(p.err, kErrBlockId);
#pragma unroll
        for (int sg = 0; sg < Gm::NSEG; ++sg) {
          tma_load_4d(kdst + sg * Gm::SEG_BYTES, &tmK, fk, sg * Gm::BOXE, 0, h, phys);
          if constexpr (!SPLITKV)
            tma_load_4d(kdst + Gm::HALF_BYTES + sg * Gm::SEG_BYTES, &tmV, fk, sg * Gm::BOXE, 0, h, phys);
        }
      }
      nk = t + 1;
      if constexpr (SPLITKV) {
        // V half: free once the consumers have finished tile t - NST
        if (t >= NST && !mbar_wait(emptyv0 + 8 * stage, ((t / NST) - 1) & 1)) {
          ok = false;
          break;
        }
        const uint32_t fv = fullv0 + 8 * stage;
        if (lane == 0) mbar_arrive_expect_tx(fv, tx * nb);
        if (lane < nb) {
#pragma unroll
          for (int sg = 0; sg < Gm::NSEG; ++sg)
            tma_load_4d(kdst + Gm::HALF_BYTES + sg * Gm::SEG_BYTES, &tmV, fv, sg * Gm::BOXE, 0, h, phys);
        }
        nv = t + 1;
      }
    }
    if (!ok) {
      if (lane == 0) atomicOr(p.err, kErrTimeout);
      // let the copies already issued land before the CTA can exit
      for (int u = max(0, nk - NST); u < nk; ++u) mbar_wait(fullk0 + 8 * (u % NST), (u / NST) & 1);
      for (int u = max(0, nv - NST); u < nv; ++u) mbar_wait(fullv0 + 8 * (u % NST), (u / NST) & 1);
    }
    return;
  }

  // ========================= consumer warps =========================
  const int cw = warp;
  const int ctid = tid;  // 0..NCW*32-1
  const int ncol = p.G * p.qlen;  // query columns (heads x new tokens)
  float qmax = 0.f;
  for (int idx = ctid; idx < NG * D; idx += NCW * 32) {
    const int g = idx / D, d = idx % D;
    float v = 0.f;
    if (g < ncol) v = load_q(p.q, query_row(p, s, h, g) * D + d, p.q_dtype);
    qbuf[idx] = v;
    qmax = fmaxf(qmax, fabsf(v));
  }
  float qk_mult = p.scale_log2 * p.kv_scale;
  float qmul = 1.f;
  if constexpr (KV == kE4M3 && USE_MMA) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) qmax = fmaxf(qmax, __shfl_xor_sync(0xFFFFFFFFu, qmax, o));
    if (lane == 0) ml[cw] = qmax;
  }
  named_bar_sync(1, NCW * 32);
  if constexpr (KV == kE4M3 && USE_MMA) {
    qmax = ml[0];
#pragma unroll
    for (int w = 1; w < NCW; ++w) qmax = fmaxf(qmax, ml[w]);
    int e = 0;
    if (qmax > 0.f) {
      int ex;
      frexpf(qmax, &ex);  // qmax = f * 2^ex, f in [0.5, 1)
      e = min(15 - ex, 126);
    }
    qmul = ldexpf(1.f, e);
    qk_mult = ldexpf(qk_mult, -e);
  }
  const float vscale = (KV == kE4M3) ? p.kv_scale : 1.f;
  const int qr = lane >> 2, qc = lane & 3;
  const int row0 = cw * 16;

  if constexpr (USE_MMA) {
    constexpr int NT = NG / 8;   // head tiles of 8
    constexpr int KS = D / 16;   // 16-wide k-steps (and 16-row output tiles)
    constexpr bool BF = (KV == kBF16);
    // 16 columns: the warps split them, warp cw taking column tile cw & 1 for
    // the 32 tokens (cw >> 1) * 32 .. +31 of every stage, which halves its
    // accumulators and q fragments so that three CTAs fit per SM.  8 columns:
    // warp cw takes all of them for tokens cw * 16 .. +15.
    constexpr bool CSPLIT = NT == 2;
    constexpr int NTW = CSPLIT ? 1 : NT;   // column tiles per warp
    constexpr int NSUB = CSPLIT ? 2 : 1;   // 16-token sub-tiles per warp and stage
    static_assert(!CSPLIT || NCW % 2 == 0, "column split pairs the consumer warps");
    const int ct = CSPLIT ? (cw & 1) : 0;  // this warp's first column tile
    const int rowbase = CSPLIT ? (cw >> 1) * 32 : cw * 16;
    uint32_t qf[KS][NTW][2];
#pragma unroll
    for (int j = 0; j < KS; ++j) {
#pragma unroll
      for (int nt = 0; nt < NTW; ++nt) {
        const float* qg = qbuf + ((ct + nt) * 8 + qr) * D;
        if constexpr (KV == kE4M3) {
          const int d = 16 * j + 4 * qc;  // k order of the widened FP8 fragments
          qf[j][nt][0] = pack2<false>(qg[d] * qmul, qg[d + 1] * qmul);
          qf[j][nt][1] = pack2<false>(qg[d + 2] * qmul, qg[d + 3] * qmul);
        } else {
          const int d = 16 * j + 2 * qc;
          qf[j][nt][0] = pack2<BF>(qg[d], qg[d + 1]);
          qf[j][nt][1] = pack2<BF>(qg[d + 8], qg[d + 9]);
        }
      }
    }
    named_bar_sync(1, NCW * 32);  // qbuf is free: it becomes the epilogue area
    float m_run[NTW][2], l_run[NTW][2], oacc[KS][NTW][4];
    auto reset = [&]() {
#pragma unroll
      for (int nt = 0; nt < NTW; ++nt) {
        m_run[nt][0] = m_run[nt][1] = -CUDART_INF_F;
        l_run[nt][0] = l_run[nt][1] = 0.f;
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) oacc[mt][nt][0] = oacc[mt][nt][1] = oacc[mt][nt][2] = oacc[mt][nt][3] = 0.f;
      }
    };
    // (m, l) of this warp to ml[], then its rescaled output into `area` on its turn
    auto epilogue = [&](int seg, bool last) {
#pragma unroll
      for (int nt = 0; nt < NTW; ++nt) {
#pragma unroll
        for (int c2 = 0; c2 < 2; ++c2) {
          float l = l_run[nt][c2];
          l += __shfl_xor_sync(0xFFFFFFFFu, l, 4);
          l += __shfl_xor_sync(0xFFFFFFFFu, l, 8);
          l += __shfl_xor_sync(0xFFFFFFFFu, l, 16);
          if (qr == 0) {
            const int g = (ct + nt) * 8 + 2 * qc + c2;
            ml[(cw * NG + g) * 2] = m_run[nt][c2];
            ml[(cw * NG + g) * 2 + 1] = l;
            if constexpr (CSPLIT) {  // the other tile's columns: nothing from this warp
              const int go = ((ct ^ 1) + nt) * 8 + 2 * qc + c2;
              ml[(cw * NG + go) * 2] = -CUDART_INF_F;
              ml[(cw * NG + go) * 2 + 1] = 0.f;
            }
          }
        }
      }
      segment_epilogue<D, NG>(p, cw, ctid, area, carea, cml, ml, s, h, SegInfo{seg, last, split, final_out, run},
                              vscale, [&](bool first) {
        // with split columns, the first warp in order that owns a column
        // (cw 0 or 1) initialises it and the other (cw 2 or 3) adds
        const bool fst = CSPLIT ? (cw < 2) : first;
#pragma unroll
        for (int nt = 0; nt < NTW; ++nt) {
          const float f0 = warp_factor<NG>(ml, cw, (ct + nt) * 8 + 2 * qc);
          const float f1 = warp_factor<NG>(ml, cw, (ct + nt) * 8 + 2 * qc + 1);
#pragma unroll
          for (int mt = 0; mt < KS; ++mt) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int g = (ct + nt) * 8 + 2 * qc + (e & 1);
              const int d = 16 * mt + qr + (e >= 2 ? 8 : 0);
              const float v = oacc[mt][nt][e] * ((e & 1) ? f1 : f0);
              area[g * D + d] = fst ? v : area[g * D + d] + v;
            }
          }
        }
      });
    };
    // token limit of each of this lane's query columns: new token j of qlen
    // sits at position L - qlen + j and attends to positions up to itself
    int lim[NTW][2];
#pragma unroll
    for (int nt = 0; nt < NTW; ++nt)
#pragma unroll
      for (int c2 = 0; c2 < 2; ++c2) {
        const int n = (ct + nt) * 8 + 2 * qc + c2;
        lim[nt][c2] = n < ncol ? min(tok_end, L - p.qlen + n / p.G + 1) : tok_end;
      }
    reset();
    int seg_t = 0;  // tiles done in the current segment
    for (int t = 0; t < ntiles; ++t) {
      const int stage = t % NST;
      if (!mbar_wait(fullk0 + 8 * stage, (t / NST) & 1)) {
        if (lane == 0) atomicOr(p.err, kErrTimeout);
        break;
      }
      const int slice0 = tok_begin + t * TILE + rowbase;  // first token of this warp's rows
      int n_valid[NSUB];
#pragma unroll
      for (int u = 0; u < NSUB; ++u) n_valid[u] = min(16, tok_end - (slice0 + 16 * u));
      bool vok = true;
      if (n_valid[0] > 0) {
        const uint32_t kst = ring_u32 + stage * Gm::STAGE_BYTES;
        const uint32_t vst = kst + Gm::HALF_BYTES;
        float sacc[NSUB][NTW][4];
#pragma unroll
        for (int u = 0; u < NSUB; ++u)
#pragma unroll
          for (int nt = 0; nt < NTW; ++nt) sacc[u][nt][0] = sacc[u][nt][1] = sacc[u][nt][2] = sacc[u][nt][3] = 0.f;
        // ---- S^T = K Q^T, per 16-token sub-tile ----
#pragma unroll
        for (int u = 0; u < NSUB; ++u) {
          if (u > 0 && n_valid[u] <= 0) continue;
          const int row0 = rowbase + 16 * u;
          if constexpr (KV != kE4M3) {
            const int r = row0 + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
            for (int j = 0; j < KS; ++j) {
              const int cb = 32 * j;
              const int sg = cb / Gm::BOXB, c = (cb % Gm::BOXB) / 16 + (lane >> 4);
              uint32_t a[4];
              ldsm_x4(kst + sg * Gm::SEG_BYTES + swz<Gm>(r * Gm::BOXB + c * 16), a[0], a[1], a[2], a[3]);
#pragma unroll
              for (int nt = 0; nt < NTW; ++nt) mma16816<BF>(sacc[u][nt], a, qf[j][nt][0], qf[j][nt][1]);
            }
          } else {
            const int r = row0 + tok_perm((lane & 7) + ((lane >> 3) & 1) * 8);
#pragma unroll
            for (int j = 0; j < KS; j += 2) {
              const int c = j + (lane >> 4);
              uint32_t R[4];
              ldsm_x4(kst + swz<Gm>(r * Gm::BOXB + c * 16), R[0], R[1], R[2], R[3]);
#pragma unroll
              for (int kk = 0; kk < 2; ++kk) {
                uint32_t a[4];
                e4m3x4_to_f16x2x2(R[2 * kk], a[0], a[2]);
                e4m3x4_to_f16x2x2(R[2 * kk + 1], a[1], a[3]);
#pragma unroll
                for (int nt = 0; nt < NTW; ++nt)
                  mma16816<false>(sacc[u][nt], a, qf[j + kk][nt][0], qf[j + kk][nt][1]);
              }
            }
          }
        }
        if constexpr (SPLITKV) {
          __syncwarp();
          if (lane == 0) mbar_arrive(emptyk0 + 8 * stage);  // K read: its half may refill
        }
        // ---- online softmax over this warp's NSUB x 16 tokens ----
        uint32_t pb[NSUB][NTW][2];
#pragma unroll
        for (int nt = 0; nt < NTW; ++nt) {
          float sv[NSUB][4], alpha[2];
#pragma unroll
          for (int u = 0; u < NSUB; ++u)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int row = 16 * u + (KV == kE4M3 ? tok_perm(qr + (e >= 2 ? 8 : 0)) : qr + (e >= 2 ? 8 : 0));
              sv[u][e] = slice0 + row < lim[nt][e & 1] ? sacc[u][nt][e] * qk_mult : -CUDART_INF_F;
            }
#pragma unroll
          for (int c2 = 0; c2 < 2; ++c2) {
            float mx = fmaxf(sv[0][c2], sv[0][c2 + 2]);
#pragma unroll
            for (int u = 1; u < NSUB; ++u) mx = fmaxf(mx, fmaxf(sv[u][c2], sv[u][c2 + 2]));
            mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 4));
            mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 8));
            mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 16));
            const float m_new = fmaxf(m_run[nt][c2], mx);
            const float m_use = m_new == -CUDART_INF_F ? 0.f : m_new;
            alpha[c2] = ex2(m_run[nt][c2] - m_use);
            float add = 0.f;
#pragma unroll
            for (int u = 0; u < NSUB; ++u) {
              sv[u][c2] = ex2(sv[u][c2] - m_use);
              sv[u][c2 + 2] = ex2(sv[u][c2 + 2] - m_use);
              add += sv[u][c2] + sv[u][c2 + 2];
            }
            l_run[nt][c2] = l_run[nt][c2] * alpha[c2] + add;
            m_run[nt][c2] = m_new;
          }
#pragma unroll
          for (int mt = 0; mt < KS; ++mt) {
            oacc[mt][nt][0] *= alpha[0];
            oacc[mt][nt][1] *= alpha[1];
            oacc[mt][nt][2] *= alpha[0];
            oacc[mt][nt][3] *= alpha[1];
          }
          // P^T fragment (rows = tokens) -> transposed into the B operand of the PV product
#pragma unroll
          for (int u = 0; u < NSUB; ++u) {
            pb[u][nt][0] = movm_t(pack2<BF>(sv[u][0], sv[u][1]));
            pb[u][nt][1] = movm_t(pack2<BF>(sv[u][2], sv[u][3]));
          }
        }
        // ---- O^T += V^T P^T, per 16-token sub-tile ----
        if constexpr (SPLITKV) vok = __all_sync(0xFFFFFFFFu, mbar_wait(fullv0 + 8 * stage, (t / NST) & 1));
#pragma unroll
        for (int u = 0; u < NSUB; ++u) {
          if (!vok) break;
          if (u > 0 && n_valid[u] <= 0) continue;
          const int row0 = rowbase + 16 * u;
          if constexpr (KV != kE4M3) {
            const int r = row0 + (lane & 7) + (lane >> 4) * 8;
#pragma unroll
            for (int mt = 0; mt < KS; ++mt) {
              const int cb = 32 * mt;
              const int sg = cb / Gm::BOXB, c = (cb % Gm::BOXB) / 16 + ((lane >> 3) & 1);
              uint32_t a[4];
              ldsm_x4_t(vst + sg * Gm::SEG_BYTES + swz<Gm>(r * Gm::BOXB + c * 16), a[0], a[1], a[2], a[3]);
              if (n_valid[u] < 16) mask_tokens(a, lane, n_valid[u]);
#pragma unroll
              for (int nt = 0; nt < NTW; ++nt) mma16816<BF>(oacc[mt][nt], a, pb[u][nt][0], pb[u][nt][1]);
            }
          } else {
            // rows = tokens, columns = channels: the transposing byte load gives
            // lane (g, c) channels g and g + 8 of each 16-channel block at tokens
            // 4c .. 4c+3, i.e. k = 2c, 2c+1 (low) and 2c+8, 2c+9 (high) in the
            // sub-tile's token order
            const int r = row0 + (lane & 15);
            const uint32_t keep = n_valid[u] < 16 ? token_byte_mask(lane, n_valid[u]) : 0xFFFFFFFFu;
#pragma unroll
            for (int j = 0; j < KS; j += 2) {
              const int c = j + (lane >> 4);
              uint32_t R[4];
              ldsm_b8_x2_t(vst + swz<Gm>(r * Gm::BOXB + c * 16), R[0], R[1], R[2], R[3]);
#pragma unroll
              for (int kk = 0; kk < 2; ++kk) {
                uint32_t a[4];
                e4m3x4_to_f16x2x2(R[2 * kk] & keep, a[0], a[2]);
                e4m3x4_to_f16x2x2(R[2 * kk + 1] & keep, a[1], a[3]);
#pragma unroll
                for (int nt = 0; nt < NTW; ++nt) mma16816<false>(oacc[j + kk][nt], a, pb[u][nt][0], pb[u][nt][1]);
              }
            }
          }
        }
      } else if (SPLITKV && lane == 0) {
        mbar_arrive(emptyk0 + 8 * stage);  // no rows of this warp in the tile
      }
      if (!vok) {
        if (lane == 0) atomicOr(p.err, kErrTimeout);
        break;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(SPLITKV ? emptyv0 + 8 * stage : emptyk0 + 8 * stage);
      if (++seg_t == tiles_per_seg && t + 1 < ntiles) {  // a partition ends inside this CTA's run
        epilogue(t / tiles_per_seg, false);
        reset();
        seg_t = 0;
      }
    }
    epilogue(ntiles > 0 ? (ntiles - 1) / tiles_per_seg : 0, true);
  } else {
    // ================= warp-shuffle path (G <= 3) =================
    constexpr int EPL = D / 8;              // elements per lane per row
    constexpr int PB = Gm::BOXB / 8;        // bytes per lane per segment
    constexpr int EPS = PB / Gm::EB;        // elements per lane per segment
    const int grp = lane >> 3, sub = lane & 7;
    float qv[NG][EPL];
#pragma unroll
    for (int g = 0; g < NG; ++g)
#pragma unroll
      for (int sg = 0; sg < Gm::NSEG; ++sg)
#pragma unroll
        for (int e = 0; e < EPS; ++e) qv[g][sg * EPS + e] = qbuf[g * D + sg * Gm::BOXE + sub * EPS + e];
    named_bar_sync(1, NCW * 32);  // qbuf is free: it becomes the epilogue area
    float m_run[NG], l_run[NG], o[NG][EPL];
    auto reset = [&]() {
#pragma unroll
      for (int g = 0; g < NG; ++g) {
        m_run[g] = -CUDART_INF_F;
        l_run[g] = 0.f;
#pragma unroll
        for (int e = 0; e < EPL; ++e) o[g][e] = 0.f;
      }
    };
    auto epilogue = [&](int seg, bool last) {
      // merge the four 8-lane groups (commutative, so every lane gets the same bits)
#pragma unroll
      for (int off = 8; off <= 16; off <<= 1) {
#pragma unroll
        for (int g = 0; g < NG; ++g) {
          const float m_o = __shfl_xor_sync(0xFFFFFFFFu, m_run[g], off);
          const float l_o = __shfl_xor_sync(0xFFFFFFFFu, l_run[g], off);
          const float M = fmaxf(m_run[g], m_o);
          const float M_use = M == -CUDART_INF_F ? 0.f : M;
          const float a = ex2(m_run[g] - M_use), b = ex2(m_o - M_use);
          l_run[g] = l_run[g] * a + l_o * b;
#pragma unroll
          for (int e = 0; e < EPL; ++e) {
            const float o_o = __shfl_xor_sync(0xFFFFFFFFu, o[g][e], off);
            o[g][e] = o[g][e] * a + o_o * b;
          }
          m_run[g] = M;
        }
      }
      if (lane == 0) {
#pragma unroll
        for (int g = 0; g < NG; ++g) {
          ml[(cw * NG + g) * 2] = m_run[g];
          ml[(cw * NG + g) * 2 + 1] = l_run[g];
        }
      }
      segment_epilogue<D, NG>(p, cw, ctid, area, carea, cml, ml, s, h, SegInfo{seg, last, split, final_out, run},
                              vscale, [&](bool first) {
        if (grp == 0) {
#pragma unroll
          for (int g = 0; g < NG; ++g) {
            const float f = warp_factor<NG>(ml, cw, g);
#pragma unroll
            for (int sg = 0; sg < Gm::NSEG; ++sg)
#pragma unroll
              for (int e = 0; e < EPS; ++e) {
                const int d = sg * Gm::BOXE + sub * EPS + e;
                const float v = o[g][sg * EPS + e] * f;
                area[g * D + d] = first ? v : area[g * D + d] + v;
              }
          }
        }
      });
    };
    reset();
    int seg_t = 0;
    for (int t = 0; t < ntiles; ++t) {
      const int stage = t % NST;
      if (!mbar_wait(fullk0 + 8 * stage, (t / NST) & 1)) {
        if (lane == 0) atomicOr(p.err, kErrTimeout);
        break;
      }
      const int n_valid = min(16, tok_end - (tok_begin + t * TILE + row0));
      if (n_valid > 0) {
        const uint8_t* kst = smem + stage * Gm::STAGE_BYTES;
        const uint8_t* vst = kst + Gm::HALF_BYTES;
        float sc[4][NG];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int rr = 4 * i + grp, r = row0 + rr;
          float kf[EPL];
#pragma unroll
          for (int sg = 0; sg < Gm::NSEG; ++sg)
            load_piece<KV, PB>(kst + sg * Gm::SEG_BYTES + swz<Gm>(r * Gm::BOXB + sub * PB), kf + sg * EPS);
#pragma unroll
          for (int g = 0; g < NG; ++g) {
            float dot = 0.f;
#pragma unroll
            for (int e = 0; e < EPL; ++e) dot = fmaf(qv[g][e], kf[e], dot);
            dot += __shfl_xor_sync(0xFFFFFFFFu, dot, 1);
            dot += __shfl_xor_sync(0xFFFFFFFFu, dot, 2);
            dot += __shfl_xor_sync(0xFFFFFFFFu, dot, 4);
            sc[i][g] = rr < n_valid ? dot * qk_mult : -CUDART_INF_F;
          }
        }
#pragma unroll
        for (int g = 0; g < NG; ++g) {
          const float mx = fmaxf(fmaxf(sc[0][g], sc[1][g]), fmaxf(sc[2][g], sc[3][g]));
          const float m_new = fmaxf(m_run[g], mx);
          const float m_use = m_new == -CUDART_INF_F ? 0.f : m_new;
          const float alpha = ex2(m_run[g] - m_use);
          float lsum = 0.f;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            sc[i][g] = ex2(sc[i][g] - m_use);
            lsum += sc[i][g];
          }
          l_run[g] = l_run[g] * alpha + lsum;
          m_run[g] = m_new;
#pragma unroll
          for (int e = 0; e < EPL; ++e) o[g][e] *= alpha;
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int rr = 4 * i + grp, r = row0 + rr;
          if (rr < n_valid) {
            float vf[EPL];
#pragma unroll
            for (int sg = 0; sg < Gm::NSEG; ++sg)
              load_piece<KV, PB>(vst + sg * Gm::SEG_BYTES + swz<Gm>(r * Gm::BOXB + sub * PB), vf + sg * EPS);
#pragma unroll
            for (int g = 0; g < NG; ++g)
#pragma unroll
              for (int e = 0; e < EPL; ++e) o[g][e] = fmaf(sc[i][g], vf[e], o[g][e]);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(emptyk0 + 8 * stage);
      if (++seg_t == tiles_per_seg && t + 1 < ntiles) {
        epilogue(t / tiles_per_seg, false);
        reset();
        seg_t = 0;
      }
    }
    epilogue(ntiles > 0 ? (ntiles - 1) / tiles_per_seg : 0, true);
  }
}

// Ring stages: as many as fit when the variant's CTAs per SM (its register
// budget) share the SM's shared memory, between 2 and 8.  More stages keep
// more loads in flight per SM, which the two-CTA variants need to stay near
// the HBM rate.
template <int KV, int D, bool USE_MMA, int NG>
int ring_stages(bool split) {
  constexpr int kSmemPerSm = 228 * 1024, kReservedPerCta = 1024;
  constexpr int ctas = decode_min_ctas<KV, D, USE_MMA, NG>();
  const int budget = kSmemPerSm / ctas - kReservedPerCta;
  const int fixed = decode_smem_bytes_for<NG, D>(0, 0, split);
  int nst = (budget - fixed) / (Geom<KV, D>::STAGE_BYTES + 32);
  return nst < 2 ? 2 : (nst > 8 ? 8 : nst);
}

template <int KV, int D, bool USE_MMA, int NG>
cudaError_t launch_one(const DecodeParams& p0, const CUtensorMap& tmK, const CUtensorMap& tmV,
                       cudaStream_t st) {
  DecodeParams p = p0;
  const bool split = p.partition_size > 0;
  p.nst = ring_stages<KV, D, USE_MMA, NG>(split);
  const int smem = decode_smem_bytes_for<NG, D>(p.nst * Geom<KV, D>::STAGE_BYTES, p.nst, split);
  auto kern = decode_kernel<KV, D, USE_MMA, NG>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int nchunk = split ? split_bulk_ctas(p.Pmax, p.fringe, p.parts_per_cta) + p.fringe : 1;
  const long long grid = static_cast<long long>(p.S) * p.Hkv * nchunk;
  kern<<<static_cast<unsigned>(grid), kThreads, smem, st>>>(tmK, tmV, p);
  return cudaGetLastError();
}

template <int KV, int D>
cudaError_t launch_for_d(const DecodeParams& p, const CUtensorMap& tmK, const CUtensorMap& tmV,
                         cudaStream_t st) {
  const int ncol = p.G * p.qlen;
  if (p.qlen == 1 && p.G == 1) return launch_one<KV, D, false, 1>(p, tmK, tmV, st);
  if (p.qlen == 1 && p.G <= 3) return launch_one<KV, D, false, 3>(p, tmK, tmV, st);
  if (ncol <= 8) return launch_one<KV, D, true, 8>(p, tmK, tmV, st);
  return launch_one<KV, D, true, 16>(p, tmK, tmV, st);
}

template <int KV>
cudaError_t launch_decode_kv(const DecodeParams& p, const CUtensorMap& tmK, const CUtensorMap& tmV,
                             int head_dim, cudaStream_t st) {
  if (head_dim == 64) return launch_for_d<KV, 64>(p, tmK, tmV, st);
  return launch_for_d<KV, 128>(p, tmK, tmV, st);
}

}  // namespace pa
