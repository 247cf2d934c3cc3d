// Paged chunked prefill on the 5th-generation tensor cores with two query
// heads per work item: C new tokens per sequence attend causally through the
// block table (prefill is the compute-bound phase of the review's §7, chunked
// prefill its §10 table).  Work item = (sequence, kv head, pair of query heads
// of that kv head's group, 128 new tokens): the two heads' 128-row query tiles
// (a and b) have the same positions, so they share every K/V tile loaded and
// the same causal mask.  Each tile is a chain S_x(j) -> softmax -> P_x(j).V(j)
// -> S_x(j + 1); the two chains are synchronised only through the shared K/V
// ring, so they settle half a step apart and the tensor core runs one tile's
// MMAs while the other tile's softmax runs.
//
// With head_dim 128 on 16-bit caches and a group of four or more heads, the
// CTAs run in clusters of two on two SMs taking the same (sequence, kv head,
// query tile) for different head pairs: each loads every other block of a
// K/V tile into both CTAs by TMA multicast, and each tile is released once
// both CTAs' MMAs are done with it (commits to both), so a K/V tile crosses
// L2 -> SM once per four query heads.
//
// A template on head_dim D (64 or 128).  Tensor memory: the score tiles S_a,
// S_b (128 columns each) and the accumulators O_a, O_b (D columns each).  P
// of a tile is written as 16-bit pairs over the upper 64 columns of its own S
// buffer (the A operand of P.V), so those columns of S_x(j + 1) are issued
// only after P_x(j).V has completed (with D = 64 its other 64 columns go out
// as soon as the softmax has read S_x(j)).  16 warps:
//   warps 0-3, 4-7  softmax of tile a, of tile b: one thread per row (TMEM
//       lane), the row's 128 scores held in registers (176 a thread, by
//       setmaxnreg), causal mask on the tiles that cross a row's position,
//       online softmax in base 2 with a reference max that moves only by
//       more than 2^8 (then the O row is rescaled in TMEM, where no P.V into
//       it is in flight); the per-tensor E4M3 scale, when the blocks were
//       widened from E4M3, is folded into the score scale and the output;
//   warps 8-11  epilogue, one thread per row: O / l of both tiles to the output;
//   warp 12     issues S_a(j) = Q_a K(j)^T, then S_b(j), each once the tile's
//       previous P.V has completed;
//   warp 13     TMA: the item's two query tiles and the 128-token K tiles,
//       block by block through the block table, into a 2-slot ring;
//   warp 14     issues O_a += P_a(j) V(j), then O_b += P_b(j) V(j), the MMAs
//       of each half of the keys once the softmax has stored that half of P
//       (so P.V runs while the softmax finishes the row);
//   warp 15     TMA: the V tiles into a 2-slot ring.
// Every mbarrier wait gives up after about one second (error bit); a warp that
// gives up raises a shared abort flag that stops the others, and in-flight
// MMAs and TMA loads are drained (bounded) before the tensor memory is
// released.
#include <atomic>

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math_constants.h>

#include "pa_prefill.h"
#include "pa_ptx.cuh"
#include "pa_tcgen05.cuh"

namespace pa {

namespace {

constexpr int kErrBlockId = 0x1;
constexpr int kErrContextLen = 0x2;
constexpr int kErrTimeout = 0x8;
constexpr int kErrLayout = 0x10;

constexpr int kRows = 128, kTok = 128, kThreads = 512;
constexpr int kHalf = kRows * 128;  // 64 channels (128 bytes) of 128 rows
// Per head_dim D: a tile (128 rows x D channels of 16 bits) is D / 64
// segments of kHalf; shared memory holds the query tiles a and b, two K
// slots, two V slots, then the tail.
template <int D>
struct Geo {
  static constexpr int kHalves = D / 64;
  static constexpr int kTileB = kHalves * kHalf;
  static constexpr int kQOff = 0, kKOff = 2 * kTileB, kVOff = kKOff + 2 * kTileB, kTailOff = kVOff + 2 * kTileB;
};
// mbarriers: q full / empty; S full of a and of b; P full of each half of
// the keys of a and of b (head_dim 64: the first of each pair only); P.V done
// of a and of b; O full / free; l ready; full / empty per K slot and per V
// slot; one drain barrier per issuer; S read by the softmax, of a and of b
// (head_dim 64)
constexpr int kBarQFull = 0, kBarQEmpty = 1, kBarSFull = 2, kBarPFull = 4, kBarPvDone = 8, kBarOFull = 10,
              kBarOFree = 11, kBarLReady = 12, kBarKFull = 13, kBarKEmpty = 15, kBarVFull = 17, kBarVEmpty = 19,
              kBarDrain = 21, kBarSRead = 23, kNumBars = 25;
constexpr int kAbortOff = kNumBars * 8, kTmemOff = kAbortOff + 4, kLOff = kTmemOff + 4;
template <int D>
constexpr int smem_bytes() { return Geo<D>::kTailOff + kLOff + 2 * kRows * 4; }
static_assert(smem_bytes<128>() <= 227 * 1024, "shared memory budget");
// tensor memory columns of S and O of tile x (0: a, 1: b)
__host__ __device__ constexpr uint32_t tm_s(int x) { return x ? 128u : 0u; }
template <int D>
__host__ __device__ constexpr uint32_t tm_o(int x) { return 256u + static_cast<uint32_t>(x * D); }
// A row's reference max moves only when a tile exceeds it by more than this
// (base 2): probabilities stay below 2^8 and O is rescaled rarely.
constexpr float kRescaleThreshold = 8.f;
// registers a thread of each warpgroup holds after setmaxnreg: two softmax
// warpgroups, the epilogue, the TMA/MMA warps (128 x 512 = 65536 of the
// 512 x 128 the CTA is launched with); head_dim 64's S issue in two halves
// needs more in the TMA/MMA warps
template <int D>
struct Regs {
  static constexpr int kSoftmax = 176, kEpilogue = D == 64 ? 64 : 88, kTmaMma = D == 64 ? 96 : 72;
  static_assert(2 * kSoftmax + kEpilogue + kTmaMma <= 512, "register shares");
};

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
template <bool BF16>
__device__ __forceinline__ uint32_t pack16(float a, float b) {
  if constexpr (BF16) {
    __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&v);
  } else {
    __half2 v = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&v);
  }
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
               : "memory");
}
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

// 16 columns of 32-bit words from registers to tensor memory (one per lane)
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
      "%14, %15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

// Cluster-of-two forms (two CTAs on two SMs, sharing each K/V tile through
// TMA multicast): this CTA's rank; a K/V box loaded into the same shared
// memory offset of both CTAs, completing on the same-offset mbarrier of
// each; an MMA commit arriving on the same-offset mbarrier of both CTAs;
// both CTAs of the cluster meeting (release / acquire).
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void tma_load_4d_both(uint32_t dst, const CUtensorMap* m, uint32_t bar, int c0, int c1,
                                                 int c2, int c3) {
  const uint16_t mask = 3;
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.multicast::cluster"
      " [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar), "h"(mask)
      : "memory");
}
__device__ __forceinline__ void tc_commit_both(uint32_t bar) {
  const uint16_t mask = 3;
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::
                   "r"(bar), "h"(mask)
               : "memory");
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// One work item.
struct PairItem {
  int s, h, hp, qt;  // sequence, kv head, head pair of its group, query tile
  int L;             // context length (clamped to the table)
  int i0, rows;      // first new token of the tile and how many of its 128 rows are live
  int pos0;          // position of row 0 (may be negative)
  int kv_len;        // tokens a live row attends to at most
  int ntiles;        // 128-token K/V tiles
};

// Items run over sequences, then kv heads, then head pairs, then query tiles
// (the last, which attends to the most tokens, first): the items that read one
// (sequence, kv head)'s K/V are adjacent, so the CTAs running at one time share
// a few contexts' K/V in L2.  A cluster of two (CL) takes the head pairs two
// at a time, CTA rank hp_off the second of them.  Out of line: every warp
// role looks items up.
template <bool CL>
__device__ __noinline__ PairItem pair_item(const PrefillParams& p, int idx, int nqt, int hp_off) {
  PairItem it;
  constexpr int hp_per = CL ? 2 : 1;
  const int per_h = (p.G / 2 / hp_per) * nqt;
  const int per_seq = p.Hkv * per_h;
  it.s = idx / per_seq;
  int rem = idx - it.s * per_seq;
  it.h = rem / per_h;
  rem -= it.h * per_h;
  const int hq = rem / nqt;
  it.hp = CL ? hq * hp_per + hp_off : hq;
  it.qt = nqt - 1 - (rem - hq * nqt);
  const int lmax = p.maxB * p.bs;
  it.L = min(max(__ldg(p.context_lens + it.s), 0), lmax);
  it.i0 = it.qt * kRows;
  it.rows = min(kRows, p.C - it.i0);
  it.pos0 = it.L - p.C + it.i0;
  it.kv_len = max(0, min(it.L, it.pos0 + it.rows));
  it.ntiles = (it.kv_len + kTok - 1) / kTok;
  return it;
}

template <int D, bool BF16, bool CL>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_pair_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV, const __grid_constant__ PrefillParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  using Gm = Geo<D>;
  constexpr int kTileB = Gm::kTileB, kQOff = Gm::kQOff, kKOff = Gm::kKOff, kVOff = Gm::kVOff,
                kTailOff = Gm::kTailOff;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t base = smem_u32(smem);
  if (base & 1023u) {  // the swizzled operand tiles need 1024-byte alignment
    if (tid == 0) atomicOr(p.err, kErrLayout);
    return;
  }
  const uint32_t bar0 = base + kTailOff;
  auto bar = [&](int k) -> uint32_t { return bar0 + 8u * k; };
  uint8_t* tail = smem + kTailOff;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tail + kAbortOff);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tail + kTmemOff);
  float* l_buf = reinterpret_cast<float*>(tail + kLOff);  // [2 tiles][128]
  const int nqt = (p.C + kRows - 1) / kRows;
  // cluster form: both CTAs of cluster c take the same (sequence, kv head,
  // query tile) items, CTA rank r head pair 2 j + r of the j-th pair of pairs
  const int rank = CL ? static_cast<int>(cluster_rank()) : 0;
  constexpr int hp_per = CL ? 2 : 1;
  const int total = p.S * p.Hkv * (p.G / 2 / hp_per) * nqt;
  // round k of the grid: CTA (cluster) c takes the c-th item, the
  // (grid - 1 - c)-th in odd rounds (a snake, which spreads the longest items)
  const int grid = static_cast<int>(gridDim.x) / hp_per, cta = static_cast<int>(blockIdx.x) / hp_per;
  auto item_index = [&](int k) { return k * grid + ((k & 1) ? grid - 1 - cta : cta); };
  const int rounds = total / grid;
  const int nk = rounds + (item_index(rounds) < total ? 1 : 0);

  if (tid == 0) {
    mbar_init(bar(kBarQFull), 1);
    mbar_init(bar(kBarQEmpty), 1);
    for (int x = 0; x < 2; ++x) {
      mbar_init(bar(kBarSFull + x), 1);
      mbar_init(bar(kBarPFull + 2 * x), kRows);
      mbar_init(bar(kBarPFull + 2 * x + 1), kRows);
      mbar_init(bar(kBarPvDone + x), 1);
      if constexpr (D == 64) mbar_init(bar(kBarSRead + x), kRows);
    }
    mbar_init(bar(kBarOFull), 1);
    mbar_init(bar(kBarOFree), kRows);
    mbar_init(bar(kBarLReady), 2 * kRows);
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(kBarKFull + i), 1);
      mbar_init(bar(kBarKEmpty + i), CL ? 2 : 1);  // cluster form: both CTAs' issuers
      mbar_init(bar(kBarVFull + i), 1);
      mbar_init(bar(kBarVEmpty + i), CL ? 2 : 1);
      mbar_init(bar(kBarDrain + i), 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 12) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  // cluster form: the peer multicasts into this CTA's rings and arrives on
  // its barriers only once they are initialised
  if constexpr (CL) cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  auto fail = [&]() {
    if (lane == 0) {
      atomicOr(p.err, kErrTimeout);
      *abort_flag = 1;
    }
  };
  // the next item with K/V tiles at or after item k of this CTA (nk if none)
  auto next_active = [&](int k, PairItem& it) -> int {
    for (; k < nk; ++k) {
      it = pair_item<CL>(p, item_index(k), nqt, rank);
      if (it.ntiles > 0) return k;
    }
    return nk;
  };

  // Each warpgroup's branch opens with its register share (all four warps of
  // a warpgroup execute the same setmaxnreg; the shares sum to at most the
  // launch's total, which the launcher checks, so the increases are granted).
  if (warp >= 12) {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;\n" ::"n"(Regs<D>::kTmaMma) : "memory");
  if (warp == 13 || warp == 15) {
    // ============================ TMA producers ============================
    // warp 13: the query tiles and the K tiles; warp 15: the V tiles.  Lane i
    // issues box i of a tile: 64-channel segment i % (D / 64) of block
    // i / (D / 64) (at most 128 / 8 blocks x 2 segments = 32 boxes).
    const bool is_k = warp == 13;
    const CUtensorMap* map = is_k ? &tmK : &tmV;
    // cluster form: this CTA loads every other block (rank r: blocks r, r + 2,
    // ...) into both CTAs
    const int my_blk = (lane / Gm::kHalves) * hp_per + rank, my_half = lane % Gm::kHalves;
    const uint32_t ring = base + (is_k ? kKOff : kVOff);
    const int full_bar = is_k ? kBarKFull : kBarVFull, empty_bar = is_k ? kBarKEmpty : kBarVEmpty;
    if (lane == 0) {
      tma_prefetch_desc(map);
      if (is_k) tma_prefetch_desc(&tmQ);
    }
    int n = 0, ord = 0;  // K/V tiles and items with tiles issued
    bool ok = true;
    PairItem it;
    for (int k = next_active(0, it); ok && k < nk; k = next_active(k + 1, it), ++ord) {
      if (is_k) {
        // the item's two query tiles (head 2 hp and 2 hp + 1 of the group,
        // 128 new tokens each) once the item before has issued its last S
        if (ord >= 1 && !(ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar(kBarQEmpty), (ord - 1) & 1)))) break;
        if (lane == 0) {
          const uint32_t full = bar(kBarQFull);
          mbar_arrive_expect_tx(full, static_cast<uint32_t>(2 * kTileB));
          const int head = it.h * p.G + 2 * it.hp;
          const int row = it.s * p.C + it.i0;
#pragma unroll
          for (int x = 0; x < 2; ++x)
#pragma unroll
            for (int hf = 0; hf < Gm::kHalves; ++hf)
              tma_load_3d(base + kQOff + x * kTileB + hf * kHalf, &tmQ, full, 64 * hf, head + x, row);
        }
        __syncwarp();
      }
      const int* bt_row = p.block_tables + static_cast<int64_t>(it.s) * p.maxB;
      const int bpt = kTok / p.bs;
      const int nblk = (it.kv_len + p.bs - 1) / p.bs;
      int pre = my_blk < min(bpt, nblk) ? __ldg(bt_row + my_blk) : -1;  // tile 0's block id
      for (int t = 0; t < it.ntiles; ++t, ++n) {
        if (*abort_flag) {
          ok = false;
          break;
        }
        const int slot = n & 1;
        if (n >= 2 && !(ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar(empty_bar + slot), ((n >> 1) - 1) & 1)))) break;
        const int b0 = t * bpt;
        const int nb = min(bpt, nblk - b0);
        const uint32_t full = bar(full_bar + slot);
        if (lane == 0) mbar_arrive_expect_tx(full, static_cast<uint32_t>(nb * p.bs * D * 2));
        __syncwarp();
        const int phys = pre;
        if (t + 1 < it.ntiles) pre = my_blk < min(bpt, nblk - b0 - bpt) ? __ldg(bt_row + b0 + bpt + my_blk) : -1;
        if (my_blk < nb) {
          if (is_k && my_half == 0 && (phys < 0 || static_cast<int64_t>(phys) >= p.num_blocks))
            atomicOr(p.err, kErrBlockId);
          if constexpr (CL)
            tma_load_4d_both(ring + slot * kTileB + my_blk * p.bs * 128 + my_half * kHalf, map, full, 64 * my_half, 0,
                             it.h, phys);
          else
            tma_load_4d(ring + slot * kTileB + my_blk * p.bs * 128 + my_half * kHalf, map, full, 64 * my_half, 0,
                        it.h, phys);
        }
      }
    }
    if (!ok) fail();
    // every load issued lands before the CTA can exit
    for (int u = max(0, n - 2); u < n; ++u) mbar_wait(bar(full_bar + (u & 1)), (u >> 1) & 1);
    if (is_k && ord >= 1) mbar_wait(bar(kBarQFull), (ord - 1) & 1);
  } else if (warp == 12) {
    // ================== Q.K^T issuer (one thread), a and b alternating ==================
    if (lane == 0) {
      // head_dim 64 issues S in two halves of the keys (below), head_dim 128 whole
      constexpr bool kSplitS = D == 64;
      const uint32_t idesc = tc_idesc_f16(BF16, false, kRows, kSplitS ? kTok / 2 : kTok);
      int g = 0, ord = 0;  // tiles and items with tiles issued
      bool ok = true;
      PairItem it;
      for (int k = next_active(0, it); ok && k < nk; k = next_active(k + 1, it), ++ord) {
        for (int t = 0; t < it.ntiles; ++t, ++g) {
          if (*abort_flag) {
            ok = false;
            break;
          }
          const int slot = g & 1;
          if (t == 0 && !(ok = mbar_wait(bar(kBarQFull), ord & 1))) break;
          if (!(ok = mbar_wait(bar(kBarKFull + slot), (g >> 1) & 1))) break;
          const uint64_t kd = tc_desc_sw128(base + kKOff + slot * kTileB, 16, 1024);
          for (int x = 0; x < 2; ++x) {
            const uint64_t qd = tc_desc_sw128(base + kQOff + x * kTileB, 16, 1024);
            if constexpr (kSplitS) {
              // keys 0..63 of S_x(g) go to columns 0..63, free once the
              // softmax has read S_x(g - 1); keys 64..127 overwrite P_x(g - 1)
              // (columns 64..127): after its P.V
              if (g >= 1 && !(ok = mbar_wait(bar(kBarSRead + x), (g - 1) & 1))) break;
              tc_fence_after();
#pragma unroll
              for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t off = ((kk >> 2) * kHalf + (kk & 3) * 32) >> 4;
                mma_ss(tmem + tm_s(x), qd + off, kd + off, idesc, kk > 0);
              }
              if (g >= 1 && !(ok = mbar_wait(bar(kBarPvDone + x), (g - 1) & 1))) break;
              tc_fence_after();
#pragma unroll
              for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t off = ((kk >> 2) * kHalf + (kk & 3) * 32) >> 4;
                mma_ss(tmem + tm_s(x) + 64, qd + off, kd + ((64 * 128) >> 4) + off, idesc, kk > 0);
              }
            } else {
              // S_x(g) overwrites P_x(g - 1): after its P.V
              if (g >= 1 && !(ok = mbar_wait(bar(kBarPvDone + x), (g - 1) & 1))) break;
              tc_fence_after();
#pragma unroll
              for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t off = ((kk >> 2) * kHalf + (kk & 3) * 32) >> 4;
                mma_ss(tmem + tm_s(x), qd + off, kd + off, idesc, kk > 0);
              }
            }
            tc_commit(bar(kBarSFull + x));
          }
          if (!ok) break;
          if constexpr (CL)
            tc_commit_both(bar(kBarKEmpty + slot));
          else
            tc_commit(bar(kBarKEmpty + slot));
          if (t == it.ntiles - 1) tc_commit(bar(kBarQEmpty));
        }
      }
      if (!ok) fail();
      if (g > 0) {  // every MMA issued has completed before tensor memory is released
        tc_commit(bar(kBarDrain));
        mbar_wait(bar(kBarDrain), 0);
      }
    }
    __syncwarp();
  } else if (warp == 14) {
    // ================== P.V issuer (one warp), a and b alternating ==================
    const uint32_t idesc = tc_idesc_f16(BF16, true, kRows, D);
    int g = 0, ord = 0;
    bool ok = true;
    PairItem it;
    for (int k = next_active(0, it); ok && k < nk; k = next_active(k + 1, it), ++ord) {
      for (int t = 0; t < it.ntiles; ++t, ++g) {
        if (*abort_flag) {
          ok = false;
          break;
        }
        const int slot = g & 1;
        if (!(ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar(kBarVFull + slot), (g >> 1) & 1)))) break;
        const int valid = min(kTok, it.kv_len - t * kTok);
        const int nks = (valid + 15) / 16;
        const uint32_t vb = base + kVOff + slot * kTileB;
        if (valid < nks * 16) {
          // rows past the context in the last k-step hold pool bytes past the
          // context or stale tiles: zero them so that 0 * junk cannot make NaN
          const int rows = nks * 16 - valid;
          constexpr int kPieces = D / 8;  // 16-byte pieces of a row
          for (int w = lane; w < rows * kPieces; w += 32) {
            const int row = valid + w / kPieces, rest = w % kPieces;
            st_shared_v4(vb + (rest / 8) * kHalf + row * 128 + (rest % 8) * 16, 0u, 0u, 0u, 0u);
          }
          fence_proxy_async_smem();
          __syncwarp();
        }
        // an item's first P.V overwrites O, which the epilogue reads for the item before
        if (t == 0 && ord >= 1 && !(ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar(kBarOFree), (ord - 1) & 1)))) break;
        const uint64_t vd = tc_desc_sw128(vb, kHalf, 1024);
        const uint32_t acc0 = t > 0 ? 1u : 0u;
        for (int x = 0; x < 2 && ok; ++x) {
          // head_dim 128: P_x(g) arrives in two halves of the keys, and the
          // MMAs of a half go out as soon as it is stored; head_dim 64: all at once
          constexpr int kParts = D == 128 ? 2 : 1;
          for (int h = 0; h < kParts; ++h) {
            if (!(ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar(kBarPFull + 2 * x + h), g & 1)))) break;
            tc_fence_after();
            if (lane == 0) {
#pragma unroll
              for (int k = 0; k < 8 / kParts; ++k) {
                const int kk = (8 / kParts) * h + k;
                if (kk < nks)
                  mma_ts(tmem + tm_o<D>(x), tmem + tm_s(x) + 64 + 8 * kk, vd + ((kk * 2048) >> 4), idesc,
                         kk > 0 ? 1u : acc0);
              }
              if (h == kParts - 1) tc_commit(bar(kBarPvDone + x));
            }
            __syncwarp();
          }
        }
        if (!ok) break;
        if (lane == 0) {
          if constexpr (CL)
            tc_commit_both(bar(kBarVEmpty + slot));
          else
            tc_commit(bar(kBarVEmpty + slot));
          if (t == it.ntiles - 1) tc_commit(bar(kBarOFull));
        }
        __syncwarp();
      }
    }
    if (!ok) fail();
    if (g > 0) {
      if (lane == 0) tc_commit(bar(kBarDrain + 1));
      __syncwarp();
      mbar_wait(bar(kBarDrain + 1), 0);
    }
  }
  } else if (warp < 8) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;\n" ::"n"(Regs<D>::kSoftmax) : "memory");
    // ============ softmax: one thread per (tile, row) ============
    const int x = warp >> 2;   // 0: tile a, 1: tile b
    const int r = tid & 127;   // row = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + tm_s(x) + lane_off;
    const uint32_t tO = tmem + tm_o<D>(x) + lane_off;
    const float sl2 = p.scale_log2;
    int g = 0, ord = 0;
    bool ok = true;
    PairItem it;
    for (int k = next_active(0, it); ok && k < nk; k = next_active(k + 1, it), ++ord) {
      const int last = r < it.rows ? it.pos0 + r : -1;  // last token this row attends to
      float m = -CUDART_INF_F, l = 0.f;                  // reference max (base 2) and row sum
      for (int t = 0; t < it.ntiles; ++t, ++g) {
        if (*abort_flag) {
          ok = false;
          break;
        }
        if (!(ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar(kBarSFull + x), g & 1)))) break;
        tc_fence_after();
        // the row's 128 scores stay in registers through both passes
        float sv[128];
        const int lim0 = last - t * kTok;  // last visible column
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(tS + 32 * c, *reinterpret_cast<float(*)[32]>(sv + 32 * c));
        tmem_wait_ld();
        if constexpr (D == 64) {
          // S_x(g) is in registers: keys 0..63 of S_x(g + 1) may overwrite columns 0..63
          tc_fence_before();
          mbar_arrive(bar(kBarSRead + x));
        }
        if (!__all_sync(0xFFFFFFFFu, lim0 >= 127)) {
#pragma unroll
          for (int c = 0; c < 128; ++c) sv[c] = (c <= lim0) ? sv[c] : -CUDART_INF_F;
        }
        float mx8[8];
#pragma unroll
        for (int a = 0; a < 8; ++a) mx8[a] = -CUDART_INF_F;
#pragma unroll
        for (int c = 0; c < 128; c += 2) mx8[(c >> 1) & 7] = fmax3(mx8[(c >> 1) & 7], sv[c], sv[c + 1]);
        const float mx = sl2 * fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                                     fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
        const bool bump = mx > m + kRescaleThreshold;  // false while both are -inf
        float alpha = 1.f;
        if (bump) {
          alpha = m == -CUDART_INF_F ? 0.f : ex2(m - mx);
          m = mx;
        }
        const float m_use = m == -CUDART_INF_F ? 0.f : m;
        const uint64_t sc2 = f2pack(sl2, sl2), nm2 = f2pack(-m_use, -m_use);
        uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
        // P as 16-bit pairs, 16 words (32 columns) at a time, over S columns
        // 64..127 (all read above), then the row sum
        auto exps_store = [&](int c) {
          uint32_t pw[16];
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            float lo, hi;
            f2unpack(ffma2(f2pack(sv[32 * c + e], sv[32 * c + e + 1]), sc2, nm2), lo, hi);
            const float e0 = ex2(lo), e1 = ex2(hi);
            acc[(e >> 1) & 3] = fadd2(acc[(e >> 1) & 3], f2pack(e0, e1));
            pw[e >> 1] = pack16<BF16>(e0, e1);
          }
          tmem_st16(tS + 64 + 16 * c, pw);
        };
        // rows whose reference moved rescale their O row (no P.V into it is
        // in flight: S_x(g) was issued after P_x(g - 1).V completed, and
        // P_x(g).V starts at the first arrival on P full below)
        auto rescale_o = [&]() {
          if (t > 0 && __any_sync(0xFFFFFFFFu, bump)) {
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
              float o[32];
              tmem_ld32(tO + 32 * c, o);
              tmem_wait_ld();
#pragma unroll
              for (int e = 0; e < 32; ++e) o[e] *= alpha;
              tmem_st32(tO + 32 * c, o);
            }
          }
        };
        if constexpr (D == 128) {
          // each half of the keys released to the P.V issuer once stored, so
          // P.V runs while the softmax finishes the row
          rescale_o();
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            exps_store(c);
            if (c & 1) {
              tmem_wait_st();
              tc_fence_before();
              mbar_arrive(bar(kBarPFull + 2 * x + (c >> 1)));
            }
          }
        } else {
          // head_dim 64 (half the P.V work): all of P at once, which measured
          // faster there
#pragma unroll
          for (int c = 0; c < 4; ++c) exps_store(c);
          rescale_o();
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(bar(kBarPFull + 2 * x));
        }
        float sum8[8];
#pragma unroll
        for (int a = 0; a < 4; ++a) f2unpack(acc[a], sum8[2 * a], sum8[2 * a + 1]);
        l = l * alpha + (((sum8[0] + sum8[1]) + (sum8[2] + sum8[3])) + ((sum8[4] + sum8[5]) + (sum8[6] + sum8[7])));
      }
      if (!ok) break;
      // hand l to the epilogue; the slots were read by the previous item's
      if (ord >= 1 && !(ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar(kBarOFree), (ord - 1) & 1)))) break;
      l_buf[x * kRows + r] = l;
      mbar_arrive(bar(kBarLReady));
    }
    if (!ok) fail();
  } else {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;\n" ::"n"(Regs<D>::kEpilogue) : "memory");
    // ============ epilogue: one thread per row, both tiles ============
    const int r = tid & 127;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    int ord = 0;
    bool ok = true;
    for (int k = 0; ok && k < nk; ++k) {
      const PairItem it = pair_item<CL>(p, item_index(k), nqt, rank);
      if (r == 0 && it.h == 0 && it.hp == 0 && it.qt == nqt - 1) {  // once per sequence
        const int L = __ldg(p.context_lens + it.s);
        if (L != it.L) atomicOr(p.err, kErrContextLen);  // negative, or past the table
      }
      const bool have = it.ntiles > 0;
      if (have) {
        // the epilogue idles through most of an item: poll with a pause (at
        // most about 50 ms), then the usual bounded wait
        for (int spin = 0; spin < 400000 && !mbar_try_wait(bar(kBarOFull), ord & 1); ++spin) __nanosleep(128);
        ok = !*abort_flag && __all_sync(0xFFFFFFFFu, mbar_wait(bar(kBarOFull), ord & 1)) &&
             __all_sync(0xFFFFFFFFu, mbar_wait(bar(kBarLReady), ord & 1));
        if (!ok) break;
        tc_fence_after();
      }
      const bool live = r < it.rows;
#pragma unroll 1
      for (int x = 0; x < 2; ++x) {
        const float l = have ? l_buf[x * kRows + r] : 0.f;
        const float inv = l > 0.f ? p.vscale / l : 0.f;
        const int head = it.h * p.G + 2 * it.hp + x;
        uint16_t* orow = static_cast<uint16_t*>(p.out) +
                         ((static_cast<int64_t>(it.s) * p.C + it.i0 + r) * p.Hq + head) * D;
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          float o[32];
          if (have) {
            tmem_ld32(tmem + tm_o<D>(x) + lane_off + 32 * c, o);
            tmem_wait_ld();
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = 0.f;
          }
          if (x == 1 && c == D / 32 - 1 && have) {
            // O and the l slots may take the next item's
            tc_fence_before();
            mbar_arrive(bar(kBarOFree));
          }
          if (!live) continue;
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            uint4 w;
            w.x = pack16<BF16>(o[8 * q4 + 0] * inv, o[8 * q4 + 1] * inv);
            w.y = pack16<BF16>(o[8 * q4 + 2] * inv, o[8 * q4 + 3] * inv);
            w.z = pack16<BF16>(o[8 * q4 + 4] * inv, o[8 * q4 + 5] * inv);
            w.w = pack16<BF16>(o[8 * q4 + 6] * inv, o[8 * q4 + 7] * inv);
            *reinterpret_cast<uint4*>(orow + 32 * c + q4 * 8) = w;
          }
        }
      }
      if (have) ++ord;
    }
    if (!ok) fail();
  }

  tc_fence_before();
  __syncthreads();
  // cluster form: neither CTA leaves while the other may still load into it
  if constexpr (CL) cluster_sync_all();
  if (warp == 12) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, bool BF16, bool CL>
cudaError_t launch_pair_t(const PrefillParams& p, const CUtensorMap& tmQ, const CUtensorMap& tmK,
                          const CUtensorMap& tmV, int64_t items, int nsm, cudaStream_t st) {
  auto kern = prefill_pair_kernel<D, BF16, CL>;
  // at least half an SM's shared memory, so that no two CTAs share an SM
  // (each allocates all 512 TMEM columns; a second one would wait for them)
  constexpr int kSmemBytes = smem_bytes<D>() > 116 * 1024 ? smem_bytes<D>() : 116 * 1024;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  // the warpgroups' setmaxnreg shares must fit in the registers the CTA is
  // launched with, or a softmax warpgroup's increase would never be granted
  static std::atomic<int> launch_regs{0};
  int regs = launch_regs.load(std::memory_order_relaxed);
  if (regs == 0) {
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, kern);
    if (e != cudaSuccess) return e;
    regs = fa.numRegs;
    launch_regs.store(regs, std::memory_order_relaxed);
  }
  if (128 * (2 * Regs<D>::kSoftmax + Regs<D>::kEpilogue + Regs<D>::kTmaMma) > regs * kThreads)
    return cudaErrorInvalidConfiguration;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  if constexpr (CL) {
    // persistent clusters of two: as many as can be resident at once (an SM
    // left over in a GPC holds none), each taking its items in turn
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cfg.gridDim = dim3(2);
    static std::atomic<int> max_clusters[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
    int mc = max_clusters[dev].load(std::memory_order_relaxed);
    if (mc == 0) {
      e = cudaOccupancyMaxActiveClusters(&mc, kern, &cfg);
      if (e != cudaSuccess) return e;
      if (mc <= 0) return cudaErrorInvalidConfiguration;
      max_clusters[dev].store(mc, std::memory_order_relaxed);
    }
    const int64_t nc = items < mc ? items : mc;
    cfg.gridDim = dim3(static_cast<unsigned>(2 * nc));
  } else {
    // persistent: one CTA per SM (all of its tensor memory)
    cfg.gridDim = dim3(static_cast<unsigned>(items < nsm ? items : nsm));
    cfg.numAttrs = 0;
  }
  return cudaLaunchKernelEx(&cfg, kern, tmQ, tmK, tmV, p);
}

template <int D, bool BF16>
cudaError_t launch_pair_d(const PrefillParams& p, const CUtensorMap& tmQ, const CUtensorMap& tmK,
                          const CUtensorMap& tmV, int64_t nqt, int nsm, cudaStream_t st) {
  // a group of four or more heads in pairs of pairs: clusters of two CTAs,
  // each K/V tile loaded once for both (TMA multicast; head_dim 128 on
  // 16-bit caches, where it measured level or ahead at the power cap and
  // halves the L2 -> SM bytes)
  if constexpr (D == 128) {
    if (p.cluster && p.G % 4 == 0)
      return launch_pair_t<D, BF16, true>(p, tmQ, tmK, tmV, static_cast<int64_t>(p.S) * p.Hkv * (p.G / 4) * nqt,
                                          nsm, st);
  }
  return launch_pair_t<D, BF16, false>(p, tmQ, tmK, tmV, static_cast<int64_t>(p.S) * p.Hkv * (p.G / 2) * nqt, nsm,
                                       st);
}

}  // namespace

cudaError_t launch_prefill_pair(const PrefillParams& p, const CUtensorMap& tmQ, const CUtensorMap& tmK,
                                const CUtensorMap& tmV, cudaStream_t st) {
  if (p.G < 2 || (p.G & 1) || p.S <= 0 || p.C <= 0 || (p.D != 64 && p.D != 128)) return cudaErrorInvalidValue;
  static std::atomic<int> sms[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
  int nsm = sms[dev].load(std::memory_order_relaxed);
  if (nsm == 0) {
    if (cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || nsm <= 0) nsm = 148;
    sms[dev].store(nsm, std::memory_order_relaxed);
  }
  const int64_t nqt = (p.C + kRows - 1) / kRows;
  if (static_cast<int64_t>(p.S) * p.Hkv * (p.G / 2) * nqt > INT32_MAX) return cudaErrorInvalidValue;
  if (p.D == 64)
    return p.bf16 ? launch_pair_d<64, true>(p, tmQ, tmK, tmV, nqt, nsm, st)
                  : launch_pair_d<64, false>(p, tmQ, tmK, tmV, nqt, nsm, st);
  return p.bf16 ? launch_pair_d<128, true>(p, tmQ, tmK, tmV, nqt, nsm, st)
                : launch_pair_d<128, false>(p, tmQ, tmK, tmV, nqt, nsm, st);
}

}  // namespace pa
