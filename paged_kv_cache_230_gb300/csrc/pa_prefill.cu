// Paged prefill (chunked prefill) attention on the 5th-generation tensor
// cores.  C new query tokens per sequence sit at positions L - C .. L - 1 and
// attend causally to every cached token up to their own position, through
// the block table (prefill is the compute-bound phase of the review's §7;
// chunked prefill interleaves such chunks with decode, §10 table).
//
// Work item = (sequence, query head, 128 query rows).  The kernel is
// persistent: one CTA per SM walks the items c, c + grid, c + 2 grid, ...,
// ordered so that the items reading one (sequence, kv head)'s K/V are
// adjacent.  The loads of the next item stream in while this one computes,
// and a separate warpgroup writes each item's output while the softmax warps
// already work on the next item, so the tensor core does not wait for
// epilogues.  12 warps in three warpgroups:
//   warps 8 and 10  TMA: the q tile of each item (warp 8, two buffers), then
//           128-token K (warp 8) and V (warp 10) tiles, block by block through
//           the block table, each into its own 2-stage ring (128-byte
//           swizzle, the canonical K-major layout of the MMA operands); K
//           buffers are released when QK^T completes, V buffers when P.V
//           completes, q buffers after the item's last QK^T;
//   warp 9  one thread issues tcgen05.mma: S = Q K^T (M = 128 rows, N = 128
//           tokens, K = 128 channels) into one of two TMEM score buffers
//           (the next tile's scores, of this item or the next, are computed
//           while this tile's softmax runs), then, once the probabilities are
//           ready, O += P V (N = 128 channels, K = 128 tokens, V read
//           channel-major) into the item's O buffer (two, alternating);
//   warps 0-3  one thread per query row (= TMEM lane): reads its S row with
//           tcgen05.ld, applies the causal mask and the online softmax in
//           base 2 (no cross-thread reduction), writes P as 16-bit pairs
//           over the first 64 columns of its own S buffer in TMEM (the A
//           operand of P.V comes from TMEM, so shared memory only feeds K, V
//           and Q to the tensor core), rescales its O row in TMEM when its
//           reference max moved by more than 2^8, and at the end of the item
//           hands its row sum l to the epilogue warps;
//   warps 4-7  epilogue, one thread per row: once the item's last P.V is
//           done, O / l from TMEM to the output, then the O buffer is free.
// The softmax warpgroup takes 240 registers a thread, the epilogue 112 and
// the TMA/MMA warpgroup 80 (setmaxnreg; 128 x 432 = 55296 of the 384 x 168 =
// 64512 the CTA is launched with, which the launcher checks).
// Every mbarrier wait gives up after about one second (error bit set); a
// warp that gives up raises a shared abort flag that stops the others after
// their current wait, and in-flight MMAs and TMA loads are drained (bounded)
// before the CTA releases its tensor memory and exits.
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

constexpr int kSegBytes = kPfTile * 128;  // 64 channels (128 B) of 128 rows
constexpr int kTileBytes = 2 * kSegBytes;  // 128 rows x 128 channels x 2 B
constexpr int kQOff = 0;                                      // two q buffers
constexpr int kKVOff = kQOff + 2 * kTileBytes;                // stage st: K at +2*st*tile, V after it
constexpr int kBarOff = kKVOff + kPfStages * 2 * kTileBytes;
// mbarriers: q full/empty per q buffer, K full/empty and V full/empty per
// stage, S full, P full and O done per score buffer, O free, O full and l
// ready per O buffer, a drain barrier; then the abort flag and the TMEM
// address slot; then the row sums handed to the epilogue ([2][128] floats)
constexpr int kBarBytes = 32 + 32 * kPfStages + 48 + 16 + 16 + 16 + 8 + 8 + 8;
constexpr int kLOff = (kBarOff + kBarBytes + 15) / 16 * 16;
constexpr int kSmemBytes = 1024 + kLOff + 2 * kPfRows * 4;
constexpr int kKWarp = 8, kMmaWarp = 9, kVWarp = 10;  // warps 0-3 softmax, 4-7 epilogue, 11 idle
// S buffers in columns [0, 128) and [128, 256), O buffers in [256, 384) and [384, 512)
constexpr uint32_t kTmemCols = 512;
// A row's reference max moves only when the tile max exceeds it by more than
// this (base 2): probabilities then stay below 2^8 and O is rescaled rarely.
constexpr float kRescaleThreshold = 8.f;

static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
// registers a thread of each warpgroup holds after setmaxnreg
constexpr int kRegsSoftmax = 240, kRegsEpilogue = 112, kRegsTmaMma = 80;

// Paired fp32 arithmetic: two lanes of one 64-bit register per FMA/ADD issue,
// and a three-input max, halve the instruction count of the row softmax.
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

// One work item of the persistent loop.
struct Item {
  int s, h, hkv;
  int i0, rows;  // first query row of the item and how many of its 128 are live
  int pos0;      // position of row 0 (may be negative)
  int kv_len;    // tokens any live row attends to
  int ntiles;    // 128-token K/V tiles
};

// Item idx: the items that read one (sequence, kv head)'s K/V are adjacent
// (its G query heads x its query tiles, the last query tile, which attends to
// the most tokens, first), so the CTAs running at one time share a few
// contexts' K/V in L2 instead of each streaming its own.
__device__ __forceinline__ Item item_of(const PrefillParams& p, int idx, int nqt, bool report) {
  Item it;
  const int per = p.G * nqt;  // items of one (sequence, kv head)
  const int grp = idx / per, w = idx % per;
  const int qt = nqt - 1 - w / p.G;
  it.s = grp / p.Hkv;
  it.hkv = grp % p.Hkv;
  it.h = it.hkv * p.G + w % p.G;
  const int lmax = p.maxB * p.bs;
  int L = p.context_lens[it.s];
  if (L < 0 || L > lmax) {
    if (report && qt == 0 && it.h == 0) atomicOr(p.err, kErrContextLen);
    L = min(max(L, 0), lmax);
  }
  it.i0 = qt * kPfRows;
  it.rows = min(kPfRows, p.C - it.i0);
  it.pos0 = L - p.C + it.i0;
  it.kv_len = max(0, min(L, it.pos0 + it.rows));
  it.ntiles = (it.kv_len + kPfTile - 1) / kPfTile;
  return it;
}

__global__ void __launch_bounds__(kPfThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const PrefillParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
  const uint32_t base = smem_u32(smem);
  const uint32_t q_s0 = base + kQOff;
  const uint32_t bar0 = base + kBarOff;
  // per-buffer barriers, so no wait is on an ambiguous phase: q buffers by
  // item parity, K/V stages by tile, score buffers by tile parity, O buffers
  // by item parity
  const uint32_t q_full0 = bar0, q_empty0 = bar0 + 16;
  const uint32_t k_full0 = bar0 + 32, k_empty0 = k_full0 + 8 * kPfStages;
  const uint32_t v_full0 = k_empty0 + 8 * kPfStages, v_empty0 = v_full0 + 8 * kPfStages;
  const uint32_t s_full0 = v_empty0 + 8 * kPfStages, p_full0 = s_full0 + 16, o_done0 = p_full0 + 16;
  const uint32_t o_free0 = o_done0 + 16, o_full0 = o_free0 + 16, l_ready0 = o_full0 + 16, drain = l_ready0 + 16;
  float* l_buf = reinterpret_cast<float*>(smem + kLOff);  // [2][128]
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kBarOff + kBarBytes - 16);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kBarOff + kBarBytes - 8);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nqt = (p.C + kPfRows - 1) / kPfRows;
  const int total = nqt * p.S * p.Hq;

  if (tid == 0) {
    for (int b = 0; b < 2; ++b) {
      mbar_init(q_full0 + 8 * b, 1);
      mbar_init(q_empty0 + 8 * b, 1);
      mbar_init(s_full0 + 8 * b, 1);
      mbar_init(p_full0 + 8 * b, 128);
      mbar_init(o_done0 + 8 * b, 1);
      mbar_init(o_free0 + 8 * b, 128);
      mbar_init(o_full0 + 8 * b, 1);
      mbar_init(l_ready0 + 8 * b, 128);
    }
    for (int st = 0; st < kPfStages; ++st) {
      mbar_init(k_full0 + 8 * st, 1);
      mbar_init(k_empty0 + 8 * st, 1);
      mbar_init(v_full0 + 8 * st, 1);
      mbar_init(v_empty0 + 8 * st, 1);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tS0 = tmem, tO0 = tmem + 256;
  // a failed wait stops this warp and, through the flag, the others
  auto fail = [&]() {
    if (lane == 0) {
      atomicOr(p.err, kErrTimeout);
      *abort_flag = 1;
    }
  };

  // Each warpgroup's branch opens with its register share (every warp of a
  // warpgroup executes the same setmaxnreg; the three shares sum to less than
  // the launch's total, so the increase never waits).
  if (warp >= 8) {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;\n" :: "n"(kRegsTmaMma) : "memory");
  if (warp == kKWarp || warp == kVWarp) {
    // ===================== TMA producers: q + K, V =====================
    const bool is_k = warp == kKWarp;
    if (lane == 0) {
      tma_prefetch_desc(is_k ? &tmK : &tmV);
      if (is_k) tma_prefetch_desc(&tmQ);
    }
    const CUtensorMap* map = is_k ? &tmK : &tmV;
    const uint32_t full0 = is_k ? k_full0 : v_full0, empty0 = is_k ? k_empty0 : v_empty0;
    const uint32_t dst0 = base + kKVOff + (is_k ? 0 : kTileBytes);
    const int bpt = kPfTile / p.bs;
    const uint32_t tx_block = static_cast<uint32_t>(p.bs * 256);
    int g = 0, k = 0, nq = 0;  // tiles, active items and q tiles issued
    bool ok = true;
    for (int idx = blockIdx.x; ok && idx < total; idx += gridDim.x) {
      const Item it = item_of(p, idx, nqt, is_k && lane == 0);
      if (it.ntiles == 0) continue;
      if (is_k) {
        const int qb = k & 1;
        if (k >= 2 && !(ok = mbar_wait(q_empty0 + 8 * qb, ((k >> 1) - 1) & 1))) break;
        if (lane == 0) {
          mbar_arrive_expect_tx(q_full0 + 8 * qb, kTileBytes);
          const int row = it.s * p.C + it.i0;
          tma_load_3d(q_s0 + qb * kTileBytes, &tmQ, q_full0 + 8 * qb, 0, it.h, row);
          tma_load_3d(q_s0 + qb * kTileBytes + kSegBytes, &tmQ, q_full0 + 8 * qb, 64, it.h, row);
        }
        ++nq;
      }
      const int* bt_row = p.block_tables + static_cast<int64_t>(it.s) * p.maxB;
      const int nblk = (it.kv_len + p.bs - 1) / p.bs;
      for (int t = 0; t < it.ntiles; ++t, ++g) {
        if (*abort_flag) {
          ok = false;
          break;
        }
        const int st = g % kPfStages;
        if (g >= kPfStages && !(ok = mbar_wait(empty0 + 8 * st, ((g / kPfStages) - 1) & 1))) break;
        const int b0 = t * bpt;
        const int nb = min(bpt, nblk - b0);
        const uint32_t full = full0 + 8 * st;
        if (lane == 0) mbar_arrive_expect_tx(full, tx_block * nb);
        __syncwarp();
        if (lane < nb) {  // one block per lane, issued together
          const int phys = __ldg(bt_row + b0 + lane);
          if (is_k && (phys < 0 || static_cast<int64_t>(phys) >= p.num_blocks)) atomicOr(p.err, kErrBlockId);
          const uint32_t dst = dst0 + st * 2 * kTileBytes + lane * p.bs * 128;
          tma_load_4d(dst, map, full, 0, 0, it.hkv, phys);
          tma_load_4d(dst + kSegBytes, map, full, 64, 0, it.hkv, phys);
        }
        __syncwarp();
      }
      ++k;
    }
    if (!ok) fail();
    // let every load already issued land before the CTA can exit
    for (int u = max(0, g - kPfStages); u < g; ++u) mbar_wait(full0 + 8 * (u % kPfStages), (u / kPfStages) & 1);
    if (is_k)
      for (int u = max(0, nq - 2); u < nq; ++u) mbar_wait(q_full0 + 8 * (u & 1), (u >> 1) & 1);
  } else if (warp == kMmaWarp) {
    // ============================ MMA issuer ============================
    if (lane == 0) {
      const uint32_t id_qk = tc_idesc_f16(p.bf16 != 0, false, kPfRows, kPfTile);
      const uint32_t id_pv = tc_idesc_f16(p.bf16 != 0, true, kPfRows, 128);
      // S(g) = Q K(g)^T into score buffer g % 2, both operands K-major
      // (channels contiguous), 16 channels per step; `last` releases the
      // item's q buffer once this QK^T completes
      auto issue_qk = [&](int g, int qb, bool last) -> bool {
        const int st = g % kPfStages;
        if (!mbar_wait(k_full0 + 8 * st, (g / kPfStages) & 1)) return false;
        tc_fence_after();
        const uint32_t k_s = base + kKVOff + st * 2 * kTileBytes;
        const uint32_t q_s = q_s0 + qb * kTileBytes;
        const uint32_t tS = tS0 + (g & 1) * 128;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint32_t off = (j >> 2) * kSegBytes + (j & 3) * 32;
          tc_mma_f16(tS, tc_desc_sw128(q_s + off, 16, 1024), tc_desc_sw128(k_s + off, 16, 1024), id_qk, j > 0);
        }
        tc_commit(s_full0 + 8 * (g & 1));
        tc_commit(k_empty0 + 8 * st);
        if (last) tc_commit(q_empty0 + 8 * qb);
        return true;
      };
      // the next active item at or after idx
      auto next_active = [&](int idx, Item& it) -> int {
        for (; idx < total; idx += gridDim.x) {
          it = item_of(p, idx, nqt, false);
          if (it.ntiles > 0) return idx;
        }
        return total;
      };
      bool ok = true;
      Item cur;
      int idx = next_active(blockIdx.x, cur);
      const bool any = idx < total;
      int g = 0, k = 0;
      if (idx < total) {
        ok = mbar_wait(q_full0, 0);
        if (ok) {
          tc_fence_after();
          ok = issue_qk(0, 0, cur.ntiles == 1);
        }
      }
      while (ok && idx < total) {
        Item nxt;
        const int nidx = next_active(idx + gridDim.x, nxt);
        const int ob = k & 1;
        for (int t = 0; t < cur.ntiles; ++t, ++g) {
          if (*abort_flag) {
            ok = false;
            break;
          }
          // the next tile's scores (this item's, or the next item's first)
          // overlap this tile's softmax; its score buffer was released when
          // the softmax of tile g - 1 arrived on p_full
          if (t + 1 < cur.ntiles) {
            if (!(ok = issue_qk(g + 1, k & 1, t + 2 == cur.ntiles))) break;
          } else if (nidx < total) {
            const int qn = (k + 1) & 1;
            if (!(ok = mbar_wait(q_full0 + 8 * qn, ((k + 1) >> 1) & 1))) break;
            tc_fence_after();
            if (!(ok = issue_qk(g + 1, qn, nxt.ntiles == 1))) break;
          }
          if (!(ok = mbar_wait(p_full0 + 8 * (g & 1), (g >> 1) & 1))) break;
          const int st = g % kPfStages;
          if (!(ok = mbar_wait(v_full0 + 8 * st, (g / kPfStages) & 1))) break;
          // O buffer ob was last read by the epilogue of item k - 2
          if (t == 0 && k >= 2 && !(ok = mbar_wait(o_free0 + 8 * ob, ((k >> 1) - 1) & 1))) break;
          tc_fence_after();
          // O += P V: P from TMEM (16 tokens = 8 columns per step); V
          // channel-major: 64-channel halves 16 KB apart, 8-token groups 1 KB apart
          const uint32_t v_s = base + kKVOff + st * 2 * kTileBytes + kTileBytes;
          const uint32_t p_t = tS0 + (g & 1) * 128;
          const uint32_t tO = tO0 + ob * 128;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const uint64_t b = tc_desc_sw128(v_s + j * 2048, kSegBytes, 1024);
            tc_mma_f16_ts(tO, p_t + j * 8, b, id_pv, (t > 0 || j > 0) ? 1u : 0u);
          }
          tc_commit(o_done0 + 8 * (g & 1));
          tc_commit(v_empty0 + 8 * st);
          if (t + 1 == cur.ntiles) tc_commit(o_full0 + 8 * ob);  // the item's O is complete
        }
        if (!ok) break;
        idx = nidx;
        cur = nxt;
        ++k;
      }
      if (!ok) fail();
      // every MMA issued has completed before tensor memory is released
      if (any) {
        tc_commit(drain);
        mbar_wait(drain, 0);
      }
    }
  }  // warp 11: idle
  } else if (warp < 4) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;\n" :: "n"(kRegsSoftmax) : "memory");
    // ====================== softmax: one thread per row ======================
    const int r = tid;  // query row = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    int g = 0, k = 0;
    bool ok = true;
    for (int idx = blockIdx.x; idx < total; idx += gridDim.x) {
      const Item it = item_of(p, idx, nqt, false);
      const int pos = it.pos0 + r;  // this row's position; it attends to tokens 0..pos
      const int ntiles = ok ? it.ntiles : 0;
      const uint32_t tO = tO0 + (k & 1) * 128;
      float m = -CUDART_INF_F, l = 0.f;  // m: this row's reference max (base 2)
      int t = 0;
      for (; t < ntiles; ++t, ++g) {
        if (*abort_flag) {
          ok = false;
          break;
        }
        const int st = g % kPfStages;
        const int buf = g & 1;
        if (!(ok = __all_sync(0xFFFFFFFFu, mbar_wait(s_full0 + 8 * buf, (g >> 1) & 1)))) break;
        tc_fence_after();
        float sv[128];
#pragma unroll
        for (int c = 0; c < 4; ++c)
          tmem_ld32(tS0 + buf * 128 + lane_off + c * 32, *reinterpret_cast<float(*)[32]>(sv + 32 * c));
        tmem_wait_ld();
        const int tok0 = t * kPfTile;
        const int lim = pos - tok0;  // last visible column of this tile
        // the causal mask only matters on tiles that reach past some row's
        // position (warp-uniform test); elsewhere every column is visible
        if (!__all_sync(0xFFFFFFFFu, lim >= kPfTile - 1)) {
#pragma unroll
          for (int c = 0; c < 128; ++c) sv[c] = (c <= lim) ? sv[c] : -CUDART_INF_F;
        }
        // max of the raw scores (the scale is positive), 8 independent chains
        float mx8[8];
#pragma unroll
        for (int a = 0; a < 8; ++a) mx8[a] = -CUDART_INF_F;
#pragma unroll
        for (int c = 0; c < 128; c += 2) mx8[(c >> 1) & 7] = fmax3(mx8[(c >> 1) & 7], sv[c], sv[c + 1]);
        const float mx = p.scale_log2 * fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                                              fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
        // the reference max moves only when this tile exceeds it by more than
        // the threshold; O and l are then scaled by alpha = 2^(m_old - m_new)
        const bool bump = mx > m + kRescaleThreshold;  // false while both are -inf
        float alpha = 1.f;
        if (bump) {
          alpha = m == -CUDART_INF_F ? 0.f : ex2(m - mx);
          m = mx;
        }
        const float m_use = m == -CUDART_INF_F ? 0.f : m;
        // p = 2^(scale log2e s - m) two columns per FMA, row sum in 4 paired chains
        const uint64_t sc2 = f2pack(p.scale_log2, p.scale_log2), nm2 = f2pack(-m_use, -m_use);
        uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};  // (+0, +0) pairs
#pragma unroll
        for (int c = 0; c < 128; c += 2) {
          float lo, hi;
          f2unpack(ffma2(f2pack(sv[c], sv[c + 1]), sc2, nm2), lo, hi);
          sv[c] = ex2(lo);
          sv[c + 1] = ex2(hi);
          acc[(c >> 1) & 3] = fadd2(acc[(c >> 1) & 3], f2pack(sv[c], sv[c + 1]));
        }
        float sum8[8];
#pragma unroll
        for (int a = 0; a < 4; ++a) f2unpack(acc[a], sum8[2 * a], sum8[2 * a + 1]);
        const float sum = ((sum8[0] + sum8[1]) + (sum8[2] + sum8[3])) + ((sum8[4] + sum8[5]) + (sum8[6] + sum8[7]));
        l = l * alpha + sum;
        // P(g) over the first 64 columns of score buffer `buf`: S(g) was
        // issued after P.V of tile g - 2, so that MMA has finished reading P(g - 2)
        {
          uint32_t pw[64];
#pragma unroll
          for (int c = 0; c < 64; ++c) pw[c] = pack16(sv[2 * c], sv[2 * c + 1], p.bf16);
          tmem_st32(tS0 + buf * 128 + lane_off, pw);
          tmem_st32(tS0 + buf * 128 + lane_off + 32, pw + 32);
        }
        if (t == ntiles - 1) {
          // rows of the last V tile past the context hold whatever the pool had:
          // once V has landed, zero them so that 0 * value cannot make NaN in P.V
          if (!(ok = __all_sync(0xFFFFFFFFu, mbar_wait(v_full0 + 8 * st, (g / kPfStages) & 1)))) break;
          if (r >= it.kv_len - tok0) {
            uint8_t* vrow = smem + kKVOff + st * 2 * kTileBytes + kTileBytes + r * 128;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              *reinterpret_cast<uint4*>(vrow + c * 16) = make_uint4(0, 0, 0, 0);
              *reinterpret_cast<uint4*>(vrow + kSegBytes + c * 16) = make_uint4(0, 0, 0, 0);
            }
          }
        }
        // rescale O rows whose reference moved, once P.V of tile g - 1 (of
        // this item) is done (warp-uniform: the TMEM moves are warp-wide;
        // other rows multiply by 1)
        if (t > 0 && __any_sync(0xFFFFFFFFu, bump)) {
          if (!(ok = __all_sync(0xFFFFFFFFu, mbar_wait(o_done0 + 8 * (buf ^ 1), ((g - 1) >> 1) & 1)))) break;
          tc_fence_after();
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            float o[32];
            tmem_ld32(tO + lane_off + c * 32, o);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] *= alpha;
            tmem_st32(tO + lane_off + c * 32, o);
          }
        }
        tmem_wait_st();
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(p_full0 + 8 * buf);
      }
      if (it.ntiles > 0) {
        // hand l to the epilogue warps; its slot was read by item k - 2's epilogue
        if (ok && k >= 2) ok = __all_sync(0xFFFFFFFFu, mbar_wait(o_free0 + 8 * (k & 1), ((k >> 1) - 1) & 1));
        l_buf[(k & 1) * kPfRows + r] = l;
        mbar_arrive(l_ready0 + 8 * (k & 1));
        ++k;
      }
      if (!ok) break;
    }
    if (!ok) fail();
  } else {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;\n" :: "n"(kRegsEpilogue) : "memory");
    // ====================== epilogue: one thread per row ======================
    const int qq = warp & 3;
    const int r = qq * 32 + lane;  // query row = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(qq * 32) << 16;
    int k = 0;
    bool ok = true;
    for (int idx = blockIdx.x; idx < total; idx += gridDim.x) {
      const Item it = item_of(p, idx, nqt, false);
      const uint32_t tO = tO0 + (k & 1) * 128;
      bool have = false;
      float inv = 0.f;
      if (it.ntiles > 0 && ok) {
        // the item's last P.V has completed and its softmax has handed over l
        // the epilogue warps idle through most of an item: poll with a pause
        // (at most about 50 ms) so that they take few issue slots from the
        // softmax warps, then the usual bounded wait
        for (int spin = 0; spin < 200000 && !mbar_try_wait(o_full0 + 8 * (k & 1), (k >> 1) & 1); ++spin)
          __nanosleep(256);
        ok = !*abort_flag && __all_sync(0xFFFFFFFFu, mbar_wait(o_full0 + 8 * (k & 1), (k >> 1) & 1)) &&
             __all_sync(0xFFFFFFFFu, mbar_wait(l_ready0 + 8 * (k & 1), (k >> 1) & 1));
        if (ok) {
          tc_fence_after();
          const float l = l_buf[(k & 1) * kPfRows + r];
          inv = l > 0.f ? p.vscale / l : 0.f;
          have = true;
        }
      }
      uint16_t* orow = static_cast<uint16_t*>(p.out) +
                       ((static_cast<int64_t>(it.s) * p.C + it.i0 + r) * p.Hq + it.h) * 128;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        float o[32];
        if (have) {
          tmem_ld32(tO + lane_off + c * 32, o);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = 0.f;
        }
        if (r < it.rows) {
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            uint4 w;
            w.x = pack16(o[8 * q4 + 0] * inv, o[8 * q4 + 1] * inv, p.bf16);
            w.y = pack16(o[8 * q4 + 2] * inv, o[8 * q4 + 3] * inv, p.bf16);
            w.z = pack16(o[8 * q4 + 4] * inv, o[8 * q4 + 5] * inv, p.bf16);
            w.w = pack16(o[8 * q4 + 6] * inv, o[8 * q4 + 7] * inv, p.bf16);
            *reinterpret_cast<uint4*>(orow + c * 32 + q4 * 8) = w;
          }
        }
      }
      if (it.ntiles > 0) {
        // O buffer and l slot k & 1 may take item k + 2's
        tc_fence_before();
        mbar_arrive(o_free0 + 8 * (k & 1));
        ++k;
      }
      if (!ok) break;
    }
    if (!ok) fail();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

cudaError_t launch_prefill(const PrefillParams& p, const CUtensorMap& tmQ, const CUtensorMap& tmK,
                           const CUtensorMap& tmV, cudaStream_t st) {
  cudaError_t e = cudaFuncSetAttribute(prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  // the warpgroups' setmaxnreg shares must fit in the registers the CTA is
  // launched with, or the softmax warps' increase would never be granted
  static std::atomic<int> launch_regs{0};
  int regs = launch_regs.load(std::memory_order_relaxed);
  if (regs == 0) {
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, prefill_kernel);
    if (e != cudaSuccess) return e;
    regs = fa.numRegs;
    launch_regs.store(regs, std::memory_order_relaxed);
  }
  if (128 * (kRegsSoftmax + kRegsEpilogue + kRegsTmaMma) > regs * kPfThreads)
    return cudaErrorInvalidConfiguration;
  // persistent: one CTA per SM (the kernel holds all of an SM's tensor
  // memory), each walking the work items with a stride of the grid
  static std::atomic<int> sms[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
  int nsm = sms[dev].load(std::memory_order_relaxed);
  if (nsm == 0) {
    if (cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || nsm <= 0) nsm = 148;
    sms[dev].store(nsm, std::memory_order_relaxed);
  }
  const long long nqt = (p.C + kPfRows - 1) / kPfRows;
  const long long items = nqt * p.Hq * p.S;
  const long long grid = items < nsm ? items : nsm;
  prefill_kernel<<<static_cast<unsigned>(grid), kPfThreads, kSmemBytes, st>>>(tmQ, tmK, tmV, p);
  return cudaGetLastError();
}

}  // namespace pa
