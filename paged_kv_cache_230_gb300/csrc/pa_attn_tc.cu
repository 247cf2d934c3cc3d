// Paged attention on the 5th-generation tensor cores: chunked prefill (C new
// tokens per sequence attend causally through the block table; prefill is
// the compute-bound phase of the review's §7, chunked prefill its §10 table)
// and multi-token decode with more query columns than the warp-MMA decode
// kernel serves (speculative verification of k draft tokens, web page
// "vLLM", speculative decoding paragraph).
//
// Rows.  The queries of one (sequence, kv head) are the pairs (new token j,
// query head g of the kv head's group of G), packed as row = j * G + g, so a
// 128-row query tile holds T = floor(128 / G) tokens of every head of the
// group and each K/V tile loaded serves all of them (GQA reuse).
//
// Pipeline of one CTA (persistent: one per SM, walking the work items c,
// c + grid, ...; items ordered by context length, longest first, then kv
// head, last query tiles first, then runs of partitions in the split
// variant).  Tensor memory holds two score buffers S (128 columns each), two
// probability buffers P (64 columns each: 16-bit pairs) and the output O.
// Two threads issue the MMAs: one runs S(j) = Q K(j)^T as soon as K(j) has
// landed and the softmax has read S(j - 2) out of its buffer, the other
// O += P(j) V(j) once the softmax has written P(j); their MMAs meet on the
// tensor core in alternation, two accumulators in flight (a chain of MMAs
// into one accumulator waits on itself), and each thread's waits overlap
// the other's MMAs.  P.V takes its A operand from tensor memory, so shared
// memory only feeds Q, K and V.  16 warps:
//   warps 0-3, 4-7  softmax: one thread per (row, column half): tcgen05.ld of
//       64 scores, causal mask where a tile crosses the row's position, the
//       row max combined with the other half's through shared memory, online
//       softmax in base 2 with a reference max that moves only by more than
//       2^8 (O rescaled in TMEM then), P written to TMEM with tcgen05.st;
//   warps 8-11  epilogue, one thread per row: O / l to the output (or the
//       unnormalised partial and its (m, l) to the split workspace); with
//       E4M3 caches also the converter that widens each 8-bit K/V tile to
//       16 bits in shared memory (and rounds bf16 q to f16);
//   warp 13     TMA: each item's query tile (two buffers) and the 128-token K
//       tiles, block by block through the block table, into the K ring;
//   warp 15     TMA: the V tiles into the V ring;
//   warp 12     the Q.K^T issuer; warp 14 the P.V issuer.
// Every mbarrier wait gives up after about one second (error bit); a warp
// that gives up raises a shared abort flag that stops the others, and
// in-flight MMAs and TMA loads are drained (bounded) before the tensor
// memory is released.
#include <atomic>

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math_constants.h>

#include "pa_attn_tc.h"
#include "pa_ptx.cuh"
#include "pa_tcgen05.cuh"

namespace pa {

namespace {

constexpr int kErrBlockId = 0x1;
constexpr int kErrContextLen = 0x2;
constexpr int kErrTimeout = 0x8;
constexpr int kErrLayout = 0x10;

constexpr int kHalfBytes = kTcRows * 128;  // 64 channels (128 bytes) of 128 rows
constexpr int kStageOff = kHalfBytes;      // E4M3 tile inside a ring slot (see slot_bytes)
// the K producer sits on its own sub-partition (warp % 4 = 1) rather than on
// the one of the first softmax rows, which are the only live ones of a
// narrow decode group
constexpr int kKProdWarp = 13, kSWarp = 12, kPvWarp = 14, kVProdWarp = 15;
// tensor memory columns
constexpr uint32_t kTmS = 0, kTmP = 256, kTmO = 384;
// mbarriers (8 bytes each): q full / empty / converted per q buffer; S full
// / free, P full, P.V done and max exchange per score buffer; O full / free
// and l ready; full / empty / converted per K slot and per V slot; one drain
// barrier per issuer
constexpr int kBarQFull = 0, kBarQEmpty = 2, kBarQConv = 4, kBarSFull = 6, kBarSFree = 8, kBarPFull = 10,
              kBarPvDone = 12, kBarXchg = 14, kBarOFull = 16, kBarOFree = 17, kBarLReady = 18,
              kBarKFull = 19, kBarKEmpty = kBarKFull + kTcMaxSlots, kBarKConv = kBarKEmpty + kTcMaxSlots,
              kBarVFull = kBarKConv + kTcMaxSlots, kBarVEmpty = kBarVFull + kTcMaxSlots,
              kBarVConv = kBarVEmpty + kTcMaxSlots, kBarDrain = kBarVConv + kTcMaxSlots, kNumBars = kBarDrain + 2;
// after the barriers: abort flag, TMEM address, this CTA's item -> sequence
// and context-length tables, the row-max exchange [2][2][128], the row sums
// [2][128] and reference maxima [128] handed to the epilogue, and the rows' q
// scales [2][128]
constexpr int kAbortOff = kNumBars * 8, kTmemOff = kAbortOff + 4, kSeqTabOff = kTmemOff + 4;
constexpr int kLenTabOff = kSeqTabOff + kTcMaxRanked * 4;
constexpr int kXchgOff = kLenTabOff + kTcMaxRanked * 4;
constexpr int kLOff = kXchgOff + 2 * 2 * kTcRows * 4;
constexpr int kMOff = kLOff + 2 * kTcRows * 4;
constexpr int kQscOff = kMOff + kTcRows * 4;
constexpr int kTailBytes = (kQscOff + 2 * kTcRows * 4 + 15) / 16 * 16;
constexpr int kSmemLimit = 227 * 1024;
// A row's reference max moves only when a tile exceeds it by more than this
// (base 2): probabilities stay below 2^8 and O is rescaled rarely.
constexpr float kRescaleThreshold = 8.f;

__host__ __device__ constexpr int tile_bytes(int D) { return kTcRows * D * 2; }

// A ring slot holds one 16-bit K or V tile in the MMA's operand layout.
// With E4M3 caches the TMA lands the 8-bit tile at kStageOff and the
// converter widens it there: for head_dim 128 in place (the 8-bit row r sits
// where the second channel half of 16-bit row r goes, and only the thread
// that owns row r touches either), for head_dim 64 in an extra 8 KB behind
// the 16-bit tile.
__host__ __device__ constexpr int slot_bytes(int D, int fp8) {
  return (fp8 && D == 64) ? tile_bytes(D) + kTcRows * 64 : tile_bytes(D);
}

struct Layout {
  int q, kring, vring, slot, nks, nvs, tail, total;
};

// nqb q buffers (items alternate between two, or share one), the K ring
// (the first half of the slots, rounded up), the V ring, the tail
__host__ __device__ inline Layout layout_of(int D, int nslot, int fp8, int nqb) {
  Layout L;
  L.q = 0;
  L.slot = slot_bytes(D, fp8);
  L.nks = (nslot + 1) / 2;
  L.nvs = nslot / 2;
  L.kring = nqb * tile_bytes(D);
  L.vring = L.kring + L.nks * L.slot;
  L.tail = L.vring + L.nvs * L.slot;
  L.total = L.tail + kTailBytes;
  return L;
}

__device__ __forceinline__ uint64_t f2pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2unpack(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t fadd2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
__device__ __forceinline__ uint32_t pack16(float a, float b, int bf16) {
  if (bf16) {
    __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&v);
  }
  __half2 v = __floats2half2_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
               : "memory");
}
__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr)
               : "memory");
  return v;
}
// Four E4M3 codes (first element in the low byte) widened exactly to two
// f16x2 words: codes 0, 1 to `lo`, codes 2, 3 to `hi` (the conversion
// instruction reads each 16-bit half of the word).
__device__ __forceinline__ void e4m3x4_to_f16(uint32_t four, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b16 c0, c1;\n\t"
      "mov.b32 {c0, c1}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, c0;\n\t"
      "cvt.rn.f16x2.e4m3x2 %1, c1;\n\t}"
      : "=r"(lo), "=r"(hi) : "r"(four));
}
// L2 prefetch of a 3-D tensor box (the next item's query tile).
__device__ __forceinline__ void tma_prefetch_3d(const void* map, int c0, int c1, int c2) {
  asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(c0), "r"(c1), "r"(c2)
               : "memory");
}
// The MMAs with no memory clobber: the issuing thread's ordering with the
// other warps goes through mbarriers and tcgen05 fences, not through C++
// memory, so the compiler may keep its operands in registers around them.
__device__ __forceinline__ void mma_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc));
}
__device__ __forceinline__ void mma_ts(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
      "r"(a), "l"(b), "r"(idesc), "r"(acc));
}

// Length key of the longest-first order: 128 buckets, 4 per power of two,
// descending (bucket 0 = longest).
__device__ __forceinline__ int length_bucket(int L) {
  if (L <= 0) return 127;
  const int msb = 31 - __clz(L);
  const int frac = msb >= 2 ? (L >> (msb - 2)) & 3 : (L << (2 - msb)) & 3;
  return 127 - min(msb * 4 + frac, 127);
}

// Global index of this CTA's k-th work item.  Round k of the grid covers
// indices k * grid .. k * grid + grid - 1; CTA c takes the c-th of them, and
// without split runs the (grid - 1 - c)-th in odd rounds (a snake: the long
// items at the head of the longest-first list spread evenly over the CTAs).
// The split form keeps c-th in every round, its runs rotated per sequence
// instead (item_of).
__device__ __forceinline__ int item_index(const TcParams& p, int k) {
  const int grid = static_cast<int>(gridDim.x), c = static_cast<int>(blockIdx.x);
  return k * grid + ((p.R == 1 && (k & 1)) ? grid - 1 - c : c);
}

struct Item {
  int s, h, qt, run, L;
  int j0, ntok;        // first new token of the query tile and how many it holds
  int kv_lo, kv_hi;    // KV tokens the item reads
  int ntiles;          // 128-token KV tiles
  bool valid;          // false: a run past the end of its context (nothing to write)
  bool final_out;      // the item writes normalised outputs (not a split partial)
};

// Work item k of this CTA (global index item_index(p, k)).  With
// at most kTcMaxRanked items per CTA their sequences and context lengths
// come from the tables built at start-up (shared memory, no global load on
// the pipeline's path).  Out of line: every warp role looks items up at its
// item boundaries, and one copy of this code instead of one per role leaves
// more of the instruction caches to the loops (E4M3 prefill 702 -> 823
// TFLOP/s, k = 8 decode 324 -> 315 us).
__device__ __noinline__ Item item_of(const TcParams& p, const int* seq_tab, const int* len_tab, bool tabs, int k) {
  Item it;
  const int idx = item_index(p, k);
  const int per_h = p.n_qt * p.R;
  const int per_seq = p.Hkv * per_h;
  const int rank = idx / per_seq;
  int rem = idx - rank * per_seq;
  // split: the items of one sequence are rotated by rank * delta (delta about
  // 0.38 R), so that a CTA whose index keeps landing on the same run (the grid
  // a multiple of the items per sequence) meets runs spread over the whole
  // range instead of always the first (which every context has) or always
  // the last (which few have)
  if (p.R > 1) {
    const int64_t delta = max(1, (p.R * 5 + 6) / 13);
    rem = static_cast<int>((rem + (static_cast<int64_t>(rank) * delta) % per_seq) % per_seq);
  }
  it.h = rem / per_h;
  rem -= it.h * per_h;
  it.qt = p.n_qt - 1 - rem / p.R;
  it.run = rem % p.R;
  it.s = tabs ? seq_tab[k] : rank;
  int lmax = p.maxB * p.bs;
  if (p.partition_size > 0) lmax = min(lmax, p.Pmax * p.partition_size);
  const int L = min(max(tabs ? len_tab[k] : __ldg(p.context_lens + it.s), 0), lmax);
  it.L = L;
  it.j0 = it.qt * p.T;
  it.ntok = min(p.C - it.j0, p.T);
  int lo = 0, hi = min(L, L - p.C + it.j0 + it.ntok);  // the last row attends to tokens < hi
  it.valid = true;
  it.final_out = true;
  if (p.partition_size > 0) {
    const int run_tok = p.ppc * p.partition_size;
    const int np = ((L + p.partition_size - 1) / p.partition_size + p.ppc - 1) / p.ppc;
    it.valid = it.run == 0 || it.run < np;
    it.final_out = np <= 1;
    lo = it.run * run_tok;
    hi = min(hi, lo + run_tok);
  }
  it.kv_lo = lo;
  it.kv_hi = max(hi, lo);
  it.ntiles = hi > lo ? (hi - lo + kTcTok - 1) / kTcTok : 0;
  return it;
}

// Position in the stream of K/V tiles of this CTA's items that have any:
// item k (its ordinal among such items) and tile t.
struct Cursor {
  int k, ord, t;
  Item it;
};

// KIND: 0 f16 q and caches, 1 bf16 q and caches, 2 f16 q with E4M3 caches,
// 3 bf16 q with E4M3 caches (an instantiation per kind keeps each one's
// code to its own path: the warps of six roles share an SM's instruction
// caches).  NARROW: a launch whose query tiles hold at most 96 rows (a decode
// group), whose softmax warps without a live row skip the arithmetic.
// Row r of an E4M3 tile landed at s16 + kStageOff, widened exactly to f16 in
// the 128-byte-swizzled operand layout of the 16-bit tile at s16 (rows at or
// past `valid` become zeros, so that 0 * junk cannot make NaN in P.V).  For
// head_dim 128 in place: the 8-bit row r sits where the second channel half
// of 16-bit row r goes, and it is read whole before any of it is written.
// Out of line: one copy serves the K and the V tiles.
template <int D>
__device__ __noinline__ void widen_row(uint32_t s16, int r, int valid) {
  const uint32_t s8 = s16 + kStageOff;
  const int rsw = r & 7;
  if constexpr (D == 128) {
    uint4 in[8];
#pragma unroll
    for (int cc = 0; cc < 8; ++cc)
      in[cc] = r < valid ? ld_shared_v4(s8 + r * 128 + ((cc ^ rsw) << 4)) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int cc = 0; cc < 8; ++cc) {  // 16 channels: 16-bit chunks 2 cc, 2 cc + 1 of the row
      uint32_t h[8];
      e4m3x4_to_f16(in[cc].x, h[0], h[1]);
      e4m3x4_to_f16(in[cc].y, h[2], h[3]);
      e4m3x4_to_f16(in[cc].z, h[4], h[5]);
      e4m3x4_to_f16(in[cc].w, h[6], h[7]);
      const uint32_t rowa = s16 + (cc >> 2) * kHalfBytes + r * 128;
      const int jj = 2 * (cc & 3);
      st_shared_v4(rowa + ((jj ^ rsw) << 4), h[0], h[1], h[2], h[3]);
      st_shared_v4(rowa + (((jj + 1) ^ rsw) << 4), h[4], h[5], h[6], h[7]);
    }
  } else {
    uint4 in[4];
    const int rsw64 = (r >> 1) & 3;  // 64-byte swizzle of the 8-bit rows
#pragma unroll
    for (int cc = 0; cc < 4; ++cc)
      in[cc] = r < valid ? ld_shared_v4(s8 + r * 64 + ((cc ^ rsw64) << 4)) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int cc = 0; cc < 4; ++cc) {
      uint32_t h[8];
      e4m3x4_to_f16(in[cc].x, h[0], h[1]);
      e4m3x4_to_f16(in[cc].y, h[2], h[3]);
      e4m3x4_to_f16(in[cc].z, h[4], h[5]);
      e4m3x4_to_f16(in[cc].w, h[6], h[7]);
      const uint32_t rowa = s16 + r * 128;
      st_shared_v4(rowa + (((2 * cc) ^ rsw) << 4), h[0], h[1], h[2], h[3]);
      st_shared_v4(rowa + (((2 * cc + 1) ^ rsw) << 4), h[4], h[5], h[6], h[7]);
    }
  }
}

// The outputs of item `it` (or its split partials) from the epilogue thread
// of row r: the context-length check (once per sequence), then, once the
// item's last P.V has completed (O full) and the softmax has handed over the
// row's (l, m), O / l from tensor memory to the output in the q dtype, or the
// unnormalised partial and its (m, l) to the split workspace; O and the
// (l, m) slots are released to the next item after the last tensor-memory
// read.  ord: the item's ordinal among those with tiles (the phase parity of
// O full and l ready).  False on a failed wait.  (Kept inline: out of line it
// measured slower.)
template <int D, bool kOutBf16>
__device__ __forceinline__ bool write_item_out(const TcParams& p, const Item& it, int r, uint32_t tO, uint32_t bar0,
                                            volatile int* abort_flag, const float* l_buf, const float* m_buf,
                                            int ord) {
  auto bar = [&](int k) -> uint32_t { return bar0 + 8u * k; };
  if (r == 0 && it.h == 0 && it.run == 0 && it.qt == p.n_qt - 1) {  // once per sequence
    const int L = __ldg(p.context_lens + it.s);
    if (L != it.L) atomicOr(p.err, kErrContextLen);  // negative, or past the table (or partitions)
  }
  if (!it.valid) return true;
  const bool live = r < it.ntok * p.G;
  const int j = it.j0 + r / p.G;
  const int64_t row = (static_cast<int64_t>(it.s) * p.C + j) * p.Hq + it.h * p.G + r % p.G;
  const bool have = it.ntiles > 0;
  float l = 0.f, m = -CUDART_INF_F;
  if (have) {
    // the epilogue idles through most of an item: poll with a pause (at most
    // about 50 ms) so that it takes few issue slots from the softmax warps,
    // then the usual bounded wait
    for (int spin = 0; spin < 400000 && !mbar_try_wait(bar(kBarOFull), ord & 1); ++spin) __nanosleep(128);
    const bool got = !*abort_flag && __all_sync(0xFFFFFFFFu, mbar_wait(bar(kBarOFull), ord & 1)) &&
                     __all_sync(0xFFFFFFFFu, mbar_wait(bar(kBarLReady), ord & 1));
    if (!got) return false;
    tc_fence_after();
    l = l_buf[r] + l_buf[kTcRows + r];
    m = m_buf[r];
  }
  const float inv = l > 0.f ? p.vscale / l : 0.f;
#pragma unroll 1
  for (int c = 0; c < D / 32; ++c) {
    float o[32];
    if (have) {
      tmem_ld32(tO + 32 * c, o);
      tmem_wait_ld();
    } else {
#pragma unroll
      for (int e = 0; e < 32; ++e) o[e] = 0.f;
    }
    if (c == D / 32 - 1 && have) {
      // O and the (l, m) slots may take the next item's
      tc_fence_before();
      mbar_arrive(bar(kBarOFree));
    }
    if (!live) continue;
    if (it.final_out) {
      uint16_t* orow = static_cast<uint16_t*>(p.out) + row * D + c * 32;
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        uint4 w;
        w.x = pack16(o[8 * q4 + 0] * inv, o[8 * q4 + 1] * inv, kOutBf16);
        w.y = pack16(o[8 * q4 + 2] * inv, o[8 * q4 + 3] * inv, kOutBf16);
        w.z = pack16(o[8 * q4 + 4] * inv, o[8 * q4 + 5] * inv, kOutBf16);
        w.w = pack16(o[8 * q4 + 6] * inv, o[8 * q4 + 7] * inv, kOutBf16);
        *reinterpret_cast<uint4*>(orow + q4 * 8) = w;
      }
    } else {
      float4* dst = reinterpret_cast<float4*>(p.ws_o + (row * p.Pmax + it.run) * D + c * 32);
      const float vs = p.vscale;
#pragma unroll
      for (int q4 = 0; q4 < 8; ++q4)
        dst[q4] = make_float4(o[4 * q4] * vs, o[4 * q4 + 1] * vs, o[4 * q4 + 2] * vs, o[4 * q4 + 3] * vs);
    }
  }
  if (live && !it.final_out) {
    const int64_t slot = row * p.Pmax + it.run;
    p.ws_ml[2 * slot] = l > 0.f ? m : -CUDART_INF_F;
    p.ws_ml[2 * slot + 1] = l;
  }
  return true;
}

template <int D, int KIND, bool NARROW>
__global__ void __launch_bounds__(kTcThreads, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const TcParams p) {
  constexpr int TB = tile_bytes(D);
  constexpr int HALVES = D / 64;
  constexpr bool kFp8 = KIND >= 2;                         // E4M3 caches, widened to f16
  constexpr bool kBf16 = KIND == 1;                        // MMA operands and P in bf16 (else f16)
  constexpr bool kOutBf16 = KIND == 1 || KIND == 3;        // q and output dtype
  constexpr bool kQScale = KIND == 3;                      // bf16 q rounded to f16 per row
  extern __shared__ __align__(1024) uint8_t smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t base = smem_u32(smem);
  // The swizzled operand tiles need 1024-byte alignment; the dynamic area
  // starts there when the kernel declares no static shared memory.
  if (base & 1023u) {
    if (tid == 0) atomicOr(p.err, kErrLayout);
    return;
  }
  const Layout Ly = layout_of(D, p.nslot, kFp8, p.nqb);
  const uint32_t bar0 = base + Ly.tail;
  auto bar = [&](int k) -> uint32_t { return bar0 + 8u * k; };
  uint8_t* tail = smem + Ly.tail;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tail + kAbortOff);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tail + kTmemOff);
  int* seq_tab = reinterpret_cast<int*>(tail + kSeqTabOff);
  int* len_tab = reinterpret_cast<int*>(tail + kLenTabOff);
  float* xchg = reinterpret_cast<float*>(tail + kXchgOff);  // [2 buffers][2 halves][128]
  float* l_buf = reinterpret_cast<float*>(tail + kLOff);    // [2 halves][128]
  float* m_buf = reinterpret_cast<float*>(tail + kMOff);    // [128]
  float* qsc = reinterpret_cast<float*>(tail + kQscOff);    // [2 q buffers][128]
  const uint32_t q_base = base + Ly.q, kring = base + Ly.kring, vring = base + Ly.vring;
  const int slot_b = Ly.slot;
  // this CTA's work items: every full round, and the last partial one if its
  // place in that round is below the items left over
  const int rounds = p.total / static_cast<int>(gridDim.x);
  const int nk = rounds + (item_index(p, rounds) < p.total ? 1 : 0);
  const bool tabs = nk <= kTcMaxRanked;
  // the q buffer of the item with ordinal o among those with tiles, and the
  // parity of that buffer's phase for it
  const bool q2 = p.nqb == 2;
  auto q_buf = [q2](int o) { return q2 ? (o & 1) : 0; };
  auto q_par = [q2](int o) { return (q2 ? o >> 1 : o) & 1; };

  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(kBarQFull + i), 1);
      mbar_init(bar(kBarQEmpty + i), kQScale ? 1 + 2 * kTcRows : 1);
      mbar_init(bar(kBarQConv + i), kTcRows);
      mbar_init(bar(kBarSFull + i), 1);
      mbar_init(bar(kBarSFree + i), 2 * kTcRows);
      mbar_init(bar(kBarPFull + i), 2 * kTcRows);
      mbar_init(bar(kBarPvDone + i), 1);
      mbar_init(bar(kBarXchg + i), 2 * kTcRows);
      mbar_init(bar(kBarDrain + i), 1);
    }
    mbar_init(bar(kBarOFull), 1);
    mbar_init(bar(kBarOFree), kTcRows);
    mbar_init(bar(kBarLReady), 2 * kTcRows);
    for (int k = 0; k < kTcMaxSlots; ++k) {
      mbar_init(bar(kBarKFull + k), 1);
      mbar_init(bar(kBarKEmpty + k), 1);
      mbar_init(bar(kBarKConv + k), kTcRows);
      mbar_init(bar(kBarVFull + k), 1);
      mbar_init(bar(kBarVEmpty + k), 1);
      mbar_init(bar(kBarVConv + k), kTcRows);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  // Longest-first order: the sequence of each of this CTA's items, from a
  // histogram of context-length buckets built in the (not yet used) K ring;
  // then the items' context lengths.
  if (tabs && p.rank_seqs) {
    int* hist = reinterpret_cast<int*>(smem + Ly.kring);  // [128] counts, then [128] offsets
    int* offs = hist + 128;
    if (tid < 128) hist[tid] = 0;
    __syncthreads();
    for (int s = tid; s < p.S; s += kTcThreads) atomicAdd(&hist[length_bucket(__ldg(p.context_lens + s))], 1);
    __syncthreads();
    if (warp == 0) {
      int c[4], run = 0;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        c[k] = hist[4 * lane + k];
        run += c[k];
      }
      int incl = run;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += v;
      }
      int b = incl - run;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        offs[4 * lane + k] = b;
        b += c[k];
      }
    }
    __syncthreads();
    const int per_seq = p.Hkv * p.n_qt * p.R;
    for (int k = warp; k < nk; k += kTcThreads / 32) {
      const int rank = item_index(p, k) / per_seq;
      // the bucket holding rank, then the rank's place among that bucket's
      // sequences in index order
      int mine = -1;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int bk = 4 * lane + j;
        if (rank >= offs[bk] && rank < offs[bk] + hist[bk]) mine = bk;
      }
      const unsigned who = __ballot_sync(0xFFFFFFFFu, mine >= 0);
      const int bucket = __shfl_sync(0xFFFFFFFFu, mine, who ? __ffs(who) - 1 : 0);
      int want = rank - offs[max(bucket, 0)];
      int found = min(rank, p.S - 1);
      if (who) {
        for (int s0 = 0; s0 < p.S; s0 += 32) {
          const int s = s0 + lane;
          const unsigned m = __ballot_sync(0xFFFFFFFFu, s < p.S && length_bucket(__ldg(p.context_lens + s)) == bucket);
          const int cnt = __popc(m);
          if (want < cnt) {
            unsigned mm = m;
            for (int q = 0; q < want; ++q) mm &= mm - 1;
            found = s0 + __ffs(mm) - 1;
            break;
          }
          want -= cnt;
        }
      }
      if (lane == 0) seq_tab[k] = found;
    }
  } else if (tabs) {
    const int per_seq = p.Hkv * p.n_qt * p.R;
    for (int k = tid; k < nk; k += kTcThreads) seq_tab[k] = item_index(p, k) / per_seq;
  }
  if (tabs) {
    __syncthreads();
    for (int k = tid; k < nk; k += kTcThreads) len_tab[k] = __ldg(p.context_lens + seq_tab[k]);
  }
  if (warp == kSWarp) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  auto fail = [&]() {
    if (lane == 0) {
      atomicOr(p.err, kErrTimeout);
      *abort_flag = 1;
    }
  };
  // the next item with K/V tiles to process, at or after item k
  auto next_active = [&](int k, Item& it) -> int {
    for (; k < nk; ++k) {
      it = item_of(p, seq_tab, len_tab, tabs, k);
      if (it.valid && it.ntiles > 0) return k;
    }
    return nk;
  };
  auto cur_start = [&](Cursor& c) {
    c.k = next_active(0, c.it);
    c.ord = 0;
    c.t = 0;
  };
  auto cur_next = [&](Cursor& c) {
    if (++c.t < c.it.ntiles) return;
    c.k = next_active(c.k + 1, c.it);
    ++c.ord;
    c.t = 0;
  };
  // tokens of KV tile t of an item that lie in its range
  auto valid_tokens = [](const Item& it, int t) { return min(kTcTok, it.kv_hi - (it.kv_lo + t * kTcTok)); };

  if (warp == kKProdWarp || warp == kVProdWarp) {
    // ============================ TMA producers ============================
    // warp 13: the query tiles and the K tiles; warp 15: the V tiles.  Lane i
    // issues box i of a tile: 64-channel half i % HALVES of block i / HALVES
    // (one box of D bytes per block for E4M3); a tile has at most
    // 128 / 8 blocks x 2 halves = 32 boxes.
    const bool is_k = warp == kKProdWarp;
    const CUtensorMap* map = is_k ? &tmK : &tmV;
    const int bpb = kFp8 ? 1 : HALVES;  // boxes per block
    const int my_blk = lane / bpb, my_half = lane % bpb;
    const int nslots = is_k ? Ly.nks : Ly.nvs;
    const uint32_t ring = is_k ? kring : vring;
    const int full_bar = is_k ? kBarKFull : kBarVFull, empty_bar = is_k ? kBarKEmpty : kBarVEmpty;
    if (lane == 0) {
      tma_prefetch_desc(map);
      if (is_k) tma_prefetch_desc(&tmQ);
    }
    // blocks of a tile: at most 128 / 8 = 16
    auto tile_blocks = [&](const Cursor& c, int& b0) -> int {
      const int tok0 = c.it.kv_lo + c.t * kTcTok;
      b0 = tok0 / p.bs;
      return (tok0 + valid_tokens(c.it, c.t) - 1) / p.bs - b0 + 1;
    };
    // the block id of this lane's box, read one tile ahead of the load that
    // needs it (the block-table read is a dependent global load)
    auto tile_id = [&](const Cursor& c) -> int {
      if (c.k >= nk) return -1;
      int b0;
      const int nb = tile_blocks(c, b0);
      return my_blk < nb ? __ldg(p.block_tables + static_cast<int64_t>(c.it.s) * p.maxB + b0 + my_blk) : -1;
    };
    int rslot = 0, rphase = 0, n = 0, nq = 0;  // ring step n: its slot and phase parity; q tiles loaded
    bool ok = true;
    Cursor c;
    cur_start(c);
    int pre = tile_id(c);
    while (c.k < nk) {
      if (*abort_flag) {
        ok = false;
        break;
      }
      if (is_k && c.t == 0) {
        // the item's query tile (G heads x T tokens per 64-channel half) into
        // its q buffer, once the item that used the buffer before has finished
        // with it
        const int qb = q_buf(c.ord);
        if (c.ord >= p.nqb &&
            !(ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar(kBarQEmpty + qb), q_par(c.ord - p.nqb)))))
          break;
        if (lane == 0) {
          const uint32_t full = bar(kBarQFull + qb);
          mbar_arrive_expect_tx(full, static_cast<uint32_t>(p.G * p.T * 128 * HALVES));
#pragma unroll
          for (int hf = 0; hf < HALVES; ++hf)
            tma_load_3d(q_base + qb * TB + hf * kHalfBytes, &tmQ, full, 64 * hf, c.it.h * p.G, c.it.s * p.C + c.it.j0);
          // the next item's query tile into L2 ahead of time
          Item nx;
          if (next_active(c.k + 1, nx) < nk)
            for (int hf = 0; hf < HALVES; ++hf) tma_prefetch_3d(&tmQ, 64 * hf, nx.h * p.G, nx.s * p.C + nx.j0);
        }
        ++nq;
        __syncwarp();
      }
      if (n >= nslots && !(ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar(empty_bar + rslot), rphase ^ 1)))) break;
      const uint32_t full = bar(full_bar + rslot), dst = ring + rslot * slot_b;
      int b0;
      const int nb = tile_blocks(c, b0);
      if (lane == 0) mbar_arrive_expect_tx(full, static_cast<uint32_t>(nb * p.bs * D * (kFp8 ? 1 : 2)));
      __syncwarp();
      if (my_blk < nb) {
        const int phys = pre;
        if (is_k && my_half == 0 && (phys < 0 || static_cast<int64_t>(phys) >= p.num_blocks))
          atomicOr(p.err, kErrBlockId);
        if (kFp8)  // the 8-bit tile, widened later
          tma_load_4d(dst + kStageOff + my_blk * p.bs * D, map, full, 0, 0, c.it.h, phys);
        else
          tma_load_4d(dst + my_blk * p.bs * 128 + my_half * kHalfBytes, map, full, 64 * my_half, 0, c.it.h, phys);
      }
      ++n;
      if (++rslot == nslots) {
        rslot = 0;
        rphase ^= 1;
      }
      cur_next(c);
      pre = tile_id(c);
    }
    if (!ok) fail();
    // every load issued lands before the CTA can exit
    for (int u = max(0, n - nslots); u < n; ++u) mbar_wait(bar(full_bar + u % nslots), (u / nslots) & 1);
    if (is_k)
      for (int u = max(0, nq - p.nqb); u < nq; ++u) mbar_wait(bar(kBarQFull + q_buf(u)), q_par(u));
  } else if (warp == kSWarp) {
    // ======================== Q.K^T issuer (one thread) ========================
    if (lane == 0) {
      constexpr int KS = D / 16;  // k-steps of Q.K^T
      const uint32_t id_qk = tc_idesc_f16(kBf16, false, kTcRows, kTcTok);
      const int k_ready = kFp8 ? kBarKConv : kBarKFull;  // the slot holds a 16-bit tile
      const int q_bar = kQScale ? kBarQConv : kBarQFull;
      int rslot = 0, rphase = 0, j = 0;  // K ring slot and phase parity; score tiles issued
      bool ok = true;
      Cursor c;
      cur_start(c);
      while (c.k < nk) {
        if (*abort_flag) {
          ok = false;
          break;
        }
        // S(j) into score buffer j & 1 once the item's query tile and K(j)
        // have landed and the softmax has read S(j - 2) out of the buffer
        const int qb = q_buf(c.ord);
        if (c.t == 0 && !(ok = mbar_wait(bar(q_bar + qb), q_par(c.ord)))) break;
        if (!(ok = mbar_wait(bar(k_ready + rslot), rphase))) break;
        if (j >= 2 && !(ok = mbar_wait(bar(kBarSFree + (j & 1)), ((j - 2) >> 1) & 1))) break;
        tc_fence_after();
        const uint64_t qd = tc_desc_sw128(q_base + qb * TB, 16, 1024);
        const uint64_t kd = tc_desc_sw128(kring + rslot * slot_b, 16, 1024);
        const uint32_t dS = tmem + kTmS + 128u * (j & 1);
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) {
          const uint32_t off = ((kk >> 2) * kHalfBytes + (kk & 3) * 32) >> 4;
          mma_ss(dS, qd + off, kd + off, id_qk, kk > 0);
        }
        tc_commit(bar(kBarSFull + (j & 1)));
        tc_commit(bar(kBarKEmpty + rslot));
        if (c.t == c.it.ntiles - 1) tc_commit(bar(kBarQEmpty + qb));
        ++j;
        if (++rslot == Ly.nks) {
          rslot = 0;
          rphase ^= 1;
        }
        cur_next(c);
      }
      if (!ok) fail();
      // every MMA issued has completed before tensor memory is released
      if (j > 0) {
        tc_commit(bar(kBarDrain));
        mbar_wait(bar(kBarDrain), 0);
      }
    }
    __syncwarp();
  } else if (warp == kPvWarp) {
    // ========================== P.V issuer (one warp) ==========================
    const uint32_t id_pv = tc_idesc_f16(kBf16, true, kTcRows, D);
    const int v_ready = kFp8 ? kBarVConv : kBarVFull;
    int rslot = 0, rphase = 0, j = 0;  // V ring slot and phase parity; P.V tiles issued
    bool ok = true;
    Cursor c;
    cur_start(c);
    while (c.k < nk) {
      if (*abort_flag) {
        ok = false;
        break;
      }
      // O += P(j) V(j) once V(j) has landed, the softmax has written P(j), and
      // at an item's first tile the epilogue has read the previous item's O
      if (!(ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar(v_ready + rslot), rphase)))) break;
      const int valid = valid_tokens(c.it, c.t);
      const int nks = (valid + 15) / 16;
      const uint32_t vb = vring + rslot * slot_b;
      if (valid < nks * 16 && !kFp8) {
        // rows past the context in the last k-step hold pool bytes past the
        // context or stale tiles: zero them so that 0 * junk cannot make NaN
        // (the E4M3 converter zeroes them itself)
        const int rows = nks * 16 - valid;
        for (int w = lane; w < rows * 8 * HALVES; w += 32) {
          const int row = valid + w / (8 * HALVES), rest = w % (8 * HALVES);
          st_shared_v4(vb + (rest / 8) * kHalfBytes + row * 128 + (rest % 8) * 16, 0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();
        __syncwarp();
      }
      if (!(ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar(kBarPFull + (j & 1)), (j >> 1) & 1)))) break;
      if (c.t == 0 && c.ord >= 1 && !(ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar(kBarOFree), (c.ord - 1) & 1))))
        break;
      tc_fence_after();
      if (lane == 0) {
        const uint32_t dO = tmem + kTmO, aP = tmem + kTmP + 64u * (j & 1);
        const uint64_t vd = tc_desc_sw128(vb, kHalfBytes, 1024);
        const uint32_t acc0 = c.t > 0 ? 1u : 0u;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          if (kk < nks) mma_ts(dO, aP + 8 * kk, vd + ((kk * 2048) >> 4), id_pv, kk > 0 ? 1u : acc0);
        tc_commit(bar(kBarPvDone + (j & 1)));
        tc_commit(bar(kBarVEmpty + rslot));
        if (c.t == c.it.ntiles - 1) tc_commit(bar(kBarOFull));
      }
      __syncwarp();
      ++j;
      if (++rslot == Ly.nvs) {
        rslot = 0;
        rphase ^= 1;
      }
      cur_next(c);
    }
    if (!ok) fail();
    if (j > 0) {
      if (lane == 0) tc_commit(bar(kBarDrain + 1));
      __syncwarp();
      mbar_wait(bar(kBarDrain + 1), 0);
    }
  } else if (warp < 8) {
    // ============ softmax: one thread per (row, half of the columns) ============
    const int hh = warp >> 2;  // column half of every tile: tokens 64 hh .. 64 hh + 63
    const int r = tid & 127;   // row = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + kTmS + lane_off + 64u * hh;
    const uint32_t tP = tmem + kTmP + lane_off + 32u * hh;
    const uint32_t tO = tmem + kTmO + lane_off + (D / 2) * hh;
    int g = 0, ord = 0;
    bool ok = true;
    for (int k = 0; ok && k < nk; ++k) {
      const Item it = item_of(p, seq_tab, len_tab, tabs, k);
      if (!it.valid || it.ntiles == 0) continue;
      const bool live = r < it.ntok * p.G;
      const bool dead = NARROW && (warp & 3) * 32 >= it.ntok * p.G;  // all 32 rows past the item's rows
      const int pos = live ? it.L - p.C + it.j0 + r / p.G : -1;
      const int last = min(pos, it.kv_hi - 1);  // last token this row attends to
      float sl2 = p.scale_log2;                 // this row's score multiplier (base 2)
      const int qb = q_buf(ord);
      if (kQScale) {
        // the converter rounded this row of q to f16 after scaling it by 2^e:
        // 2^-e goes into the row's score multiplier; the q buffer (and its
        // scales) may take another item once every row has read its scale
        if (!(ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar(kBarQConv + qb), q_par(ord))))) break;
        sl2 *= qsc[qb * kTcRows + r];
        mbar_arrive(bar(kBarQEmpty + qb));
      }
      float m = -CUDART_INF_F, l = 0.f;  // reference max (base 2) and this half's row sum
      for (int t = 0; t < it.ntiles; ++t, ++g) {
        if (*abort_flag) {
          ok = false;
          break;
        }
        const int b = g & 1, ph = (g >> 1) & 1;
        if (!(ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar(kBarSFull + b), ph)))) break;
        if (dead) {
          // no row of this warp is a query of the item (a decode group of
          // fewer than 128 rows): only the arrivals, in the same order, and
          // the waits that keep them to one phase at a time; P and O of these
          // rows are never read into an output
          mbar_arrive(bar(kBarSFree + b));
          xchg[b * 2 * kTcRows + hh * kTcRows + r] = -CUDART_INF_F;
          mbar_arrive(bar(kBarXchg + b));
          if (!(ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar(kBarXchg + b), ph)))) break;
          mbar_arrive(bar(kBarPFull + b));
          continue;
        }
        tc_fence_after();
        float sv[64];
        tmem_ld32(tS + 128u * b, *reinterpret_cast<float(*)[32]>(sv));
        tmem_ld32(tS + 128u * b + 32, *reinterpret_cast<float(*)[32]>(sv + 32));
        tmem_wait_ld();
        // the score buffer may take S(g + 2)
        tc_fence_before();
        mbar_arrive(bar(kBarSFree + b));
        const int lim = last - (it.kv_lo + t * kTcTok + 64 * hh);  // last visible column of this half
        if (!__all_sync(0xFFFFFFFFu, lim >= 63)) {
#pragma unroll
          for (int c = 0; c < 64; ++c) sv[c] = (c <= lim) ? sv[c] : -CUDART_INF_F;
        }
        float mx8[8];
#pragma unroll
        for (int a = 0; a < 8; ++a) mx8[a] = -CUDART_INF_F;
#pragma unroll
        for (int c = 0; c < 64; c += 2) mx8[(c >> 1) & 7] = fmax3(mx8[(c >> 1) & 7], sv[c], sv[c + 1]);
        // the row max over both halves: exchange through shared memory
        float* xs = xchg + b * 2 * kTcRows;
        xs[hh * kTcRows + r] = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                                     fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
        mbar_arrive(bar(kBarXchg + b));
        if (!(ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar(kBarXchg + b), ph)))) break;
        // P buffer b is free once P.V(g - 2) has completed
        if (g >= 2 && !(ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar(kBarPvDone + b), ((g - 2) >> 1) & 1)))) break;
        const float mx = sl2 * fmaxf(xs[r], xs[kTcRows + r]);
        const bool bump = mx > m + kRescaleThreshold;  // false while both are -inf
        float alpha = 1.f;
        if (bump) {
          alpha = m == -CUDART_INF_F ? 0.f : ex2(m - mx);
          m = mx;
        }
        const float m_use = m == -CUDART_INF_F ? 0.f : m;
        const uint64_t sc2 = f2pack(sl2, sl2), nm2 = f2pack(-m_use, -m_use);
        uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
        for (int c = 0; c < 64; c += 2) {
          float lo, hi;
          f2unpack(ffma2(f2pack(sv[c], sv[c + 1]), sc2, nm2), lo, hi);
          sv[c] = ex2(lo);
          sv[c + 1] = ex2(hi);
          acc[(c >> 1) & 3] = fadd2(acc[(c >> 1) & 3], f2pack(sv[c], sv[c + 1]));
        }
        float sum8[8];
#pragma unroll
        for (int a = 0; a < 4; ++a) f2unpack(acc[a], sum8[2 * a], sum8[2 * a + 1]);
        l = l * alpha + (((sum8[0] + sum8[1]) + (sum8[2] + sum8[3])) + ((sum8[4] + sum8[5]) + (sum8[6] + sum8[7])));
        uint32_t pw[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) pw[c] = pack16(sv[2 * c], sv[2 * c + 1], kBf16);
        if (t > 0 && __any_sync(0xFFFFFFFFu, bump)) {
          // rows whose reference moved rescale their half of the O row once
          // P.V(g - 1) has landed (the others multiply by 1)
          if (!(ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar(kBarPvDone + (b ^ 1)), ((g - 1) >> 1) & 1)))) break;
          tc_fence_after();
#pragma unroll 1  // rare: rolled, so that it takes little of the instruction caches
          for (int c = 0; c < D / 64; ++c) {
            float o[32];
            tmem_ld32(tO + 32 * c, o);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] *= alpha;
            tmem_st32(tO + 32 * c, o);
          }
        } else {
          tc_fence_after();
        }
        tmem_st32(tP + 64u * b, pw);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar(kBarPFull + b));
      }
      if (!ok) break;
      // hand (l, m) to the epilogue; the slots were read by the previous item's
      if (ord >= 1 && !(ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar(kBarOFree), (ord - 1) & 1)))) break;
      l_buf[hh * kTcRows + r] = l;
      if (hh == 0) m_buf[r] = m;
      mbar_arrive(bar(kBarLReady));
      ++ord;
    }
    if (!ok) fail();
  } else {
    // ============ epilogue (and E4M3 converter): one thread per row ============
    const int r = tid & 127;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tO = tmem + kTmO + lane_off;
    int ord = 0;
    bool ok = true;
    // the outputs of item k (or its split partials)
    auto epilogue = [&](int k) -> bool {
      const Item it = item_of(p, seq_tab, len_tab, tabs, k);
      if (!write_item_out<D, kOutBf16>(p, it, r, tO, bar0, abort_flag, l_buf, m_buf, ord)) return false;
      if (it.valid && it.ntiles > 0) ++ord;
      return true;
    };
    if (!kFp8) {
      for (int k = 0; ok && k < nk; ++k) ok = epilogue(k);
    } else {
      // E4M3 caches: every ring load, in the order the producer issues them,
      // is widened row by row (this thread: row r) from the 8-bit tile to the
      // slot's 16-bit operand tile; rows past the tile's valid tokens become
      // zeros (so 0 * junk cannot make NaN in P.V).  An item's outputs are
      // written once the ring step holding its last V tile is widened.
      // bf16 q with E4M3 caches: the MMA runs in f16, so row r of an item's
      // query tile is scaled by 2^e with max|q| 2^e in [2^14, 2^15) and
      // rounded to f16 in place (exact but for entries below 2^-29 max|q|);
      // 2^-e goes to the softmax through qsc.  Done before the item's first K
      // tile, in the producer's order, so it never waits on the softmax.
      auto convert_q = [&](const Cursor& c) -> bool {
        const int qb = q_buf(c.ord);
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(bar(kBarQFull + qb), q_par(c.ord)))) return false;
        float mul_inv = 1.f;
        if (r < c.it.ntok * p.G) {
          const uint32_t qrow = q_base + qb * TB + r * 128;
          const int rsw = r & 7;
          float qmax = 0.f;
#pragma unroll
          for (int cc = 0; cc < D / 8; ++cc) {
            const uint4 u = ld_shared_v4(qrow + (cc >> 3) * kHalfBytes + (((cc & 7) ^ rsw) << 4));
            const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int e = 0; e < 4; ++e)
              qmax = fmaxf(qmax, fmaxf(fabsf(__uint_as_float(w[e] << 16)), fabsf(__uint_as_float(w[e] & 0xFFFF0000u))));
          }
          int ex = 0, e2 = 0;
          if (qmax > 0.f) {
            frexpf(qmax, &ex);  // qmax = f 2^ex, f in [0.5, 1)
            e2 = min(15 - ex, 126);
          }
          const float mul = ldexpf(1.f, e2);
#pragma unroll
          for (int cc = 0; cc < D / 8; ++cc) {
            const uint32_t a = qrow + (cc >> 3) * kHalfBytes + (((cc & 7) ^ rsw) << 4);
            const uint4 u = ld_shared_v4(a);
            const uint32_t w[4] = {u.x, u.y, u.z, u.w};
            uint32_t hw[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
              hw[e] = pack16(__uint_as_float(w[e] << 16) * mul, __uint_as_float(w[e] & 0xFFFF0000u) * mul, 0);
            st_shared_v4(a, hw[0], hw[1], hw[2], hw[3]);
          }
          mul_inv = ldexpf(1.f, -e2);
        }
        qsc[qb * kTcRows + r] = mul_inv;
        fence_proxy_async_smem();
        mbar_arrive(bar(kBarQConv + qb));
        return true;
      };
      // one landed tile, widened in place (its 16-bit tile at s16)
      auto convert = [&](const Cursor& c, uint32_t s16) { widen_row<D>(s16, r, valid_tokens(c.it, c.t)); };
      // the tiles in the order K(0), K(1), then V(j), K(j + 2) for j = 0, 1,
      // ...; an item's outputs once its last V tile is widened
      Cursor kc, vc;
      cur_start(kc);
      vc = kc;
      int ks = 0, kph = 0, vs = 0, vph = 0;  // K and V ring slots and phase parities
      int ke = 0;                            // first item whose outputs are not yet written
      auto conv_k = [&]() -> bool {
        if (kc.t == 0 && kQScale && !convert_q(kc)) return false;
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(bar(kBarKFull + ks), kph))) return false;
        convert(kc, kring + ks * slot_b);
        fence_proxy_async_smem();
        mbar_arrive(bar(kBarKConv + ks));
        if (++ks == Ly.nks) {
          ks = 0;
          kph ^= 1;
        }
        cur_next(kc);
        return true;
      };
      auto conv_v = [&]() -> bool {
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(bar(kBarVFull + vs), vph))) return false;
        convert(vc, vring + vs * slot_b);
        fence_proxy_async_smem();
        mbar_arrive(bar(kBarVConv + vs));
        if (++vs == Ly.nvs) {
          vs = 0;
          vph ^= 1;
        }
        cur_next(vc);
        return true;
      };
      for (int i = 0; ok && i < 2 && kc.k < nk; ++i) ok = conv_k();
      while (ok && vc.k < nk) {
        if (*abort_flag) {
          ok = false;
          break;
        }
        const int vk = vc.k;
        const bool item_done = vc.t == vc.it.ntiles - 1;
        ok = conv_v();
        if (ok && kc.k < nk) ok = conv_k();
        if (item_done)
          for (; ok && ke <= vk; ++ke) ok = epilogue(ke);
      }
      for (; ok && ke < nk; ++ke) ok = epilogue(ke);
    }
    if (!ok) fail();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kSWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, int KIND>
cudaError_t launch_d(const TcParams& p, const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                     int grid, int smem, cudaStream_t st) {
  // every warp role fits in the 128 registers a thread of the 512 gets
  auto kern = p.n_qt == 1 && p.C * p.G <= 96 ? attn_tc_kernel<D, KIND, true> : attn_tc_kernel<D, KIND, false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  kern<<<grid, kTcThreads, smem, st>>>(tmQ, tmK, tmV, p);
  return cudaGetLastError();
}

}  // namespace

int tc_ring_slots(int D, int fp8, int nqb) {
  const Layout L0 = layout_of(D, 0, fp8, nqb);
  const int n = (kSmemLimit - L0.total) / L0.slot;
  return n < kTcMaxSlots ? n : kTcMaxSlots;
}

int tc_smem_bytes(int D, int nslot, int fp8, int nqb) { return layout_of(D, nslot, fp8, nqb).total; }

cudaError_t launch_attn_tc(const TcParams& p, const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                           cudaStream_t st) {
  if (p.nslot < 2 || p.nslot > kTcMaxSlots || (p.D != 64 && p.D != 128) || (p.nqb != 1 && p.nqb != 2))
    return cudaErrorInvalidValue;
  const int smem = tc_smem_bytes(p.D, p.nslot, p.fp8, p.nqb);
  if (smem > kSmemLimit) return cudaErrorInvalidValue;
  static std::atomic<int> sms[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
  int nsm = sms[dev].load(std::memory_order_relaxed);
  if (nsm == 0) {
    if (cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || nsm <= 0) nsm = 148;
    sms[dev].store(nsm, std::memory_order_relaxed);
  }
  if (p.total <= 0) return cudaSuccess;
  // persistent: one CTA per SM (the kernel holds all of an SM's tensor memory,
  // and its shared memory keeps a second CTA off the SM)
  const int grid = p.total < nsm ? p.total : nsm;
  TcParams q = p;
  // items per CTA beyond the table are not ordered
  if ((p.total + grid - 1) / grid > kTcMaxRanked) q.rank_seqs = 0;
  // the kind of the launch: the operand dtype (bf16, or f16 for E4M3 caches),
  // the q and output dtype, whether bf16 q is rounded to f16 per row
  if (p.fp8 ? (p.bf16 != 0 || p.q_scale_rows != p.out_bf16) : (p.bf16 != p.out_bf16 || p.q_scale_rows != 0))
    return cudaErrorInvalidValue;
  const int kind = p.fp8 ? (p.out_bf16 ? 3 : 2) : (p.bf16 ? 1 : 0);
  switch (kind + 4 * (p.D == 64 ? 0 : 1)) {
    case 0: return launch_d<64, 0>(q, tmQ, tmK, tmV, grid, smem, st);
    case 1: return launch_d<64, 1>(q, tmQ, tmK, tmV, grid, smem, st);
    case 2: return launch_d<64, 2>(q, tmQ, tmK, tmV, grid, smem, st);
    case 3: return launch_d<64, 3>(q, tmQ, tmK, tmV, grid, smem, st);
    case 4: return launch_d<128, 0>(q, tmQ, tmK, tmV, grid, smem, st);
    case 5: return launch_d<128, 1>(q, tmQ, tmK, tmV, grid, smem, st);
    case 6: return launch_d<128, 2>(q, tmQ, tmK, tmV, grid, smem, st);
    default: return launch_d<128, 3>(q, tmQ, tmK, tmV, grid, smem, st);
  }
}

}  // namespace pa
