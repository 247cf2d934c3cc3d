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
// group and each K/V tile loaded serves all of them (GQA reuse).  A work
// item holds NQ = 2 consecutive query tiles when there are two (one
// otherwise): both read the same K/V tiles, and their MMAs alternate
// accumulators instruction by instruction, which is what keeps the tensor
// core at full rate (a chain of MMAs into one accumulator waits on itself).
//
// Persistent: one CTA per SM walks the work items c, c + grid, ...; the
// items are ordered by context length, longest first, then by kv head, last
// query tiles first (they attend to the most tokens), and runs of partitions
// in the split variant.  16 warps in four warpgroups:
//   warps 0-3, 4-7  softmax of query tile 0 and 1, one thread per row (=
//       TMEM lane): tcgen05.ld of the 128 scores, causal mask where a tile
//       crosses the row's position, online softmax in base 2 with a
//       reference max that moves only by more than 2^8 (O rescaled in TMEM
//       then), P written as 16-bit pairs to shared memory (the A operand of
//       P.V);
//   warps 8-11  epilogue, one thread per row: O / l from TMEM to the output
//       (or the unnormalised partial and its (m, l) to the split workspace);
//   warp 12     TMA: each item's query tiles, then its 128-token K and V
//       tiles block by block through the block table into a ring of slots,
//       in the order the tensor core consumes them;
//   warp 13     one thread issues tcgen05.mma: S_i = Q_i K^T (both operands
//       in shared memory) into TMEM, then O_i += P_i V once the softmax has
//       written P_i.  The scores of tile t + 1 are computed while the
//       softmax works on tile t: a score buffer is free as soon as its
//       softmax has loaded it into registers.
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

constexpr int kHalfBytes = kTcRows * 128;      // 64 channels (128 bytes) of 128 rows
constexpr int kPBytes = kTcRows * kTcTok * 2;  // one P tile, 16-bit
constexpr int kProdWarp = 12, kMmaWarp = 13;
// mbarriers (8 bytes each): q full / empty, S full / free, P full, P.V done,
// O full / free and l ready per query tile; full / empty per ring slot; drain
constexpr int kBarQFull = 0, kBarQEmpty = 2, kBarSFull = 4, kBarSFree = 6, kBarPFull = 8, kBarPvDone = 10,
              kBarOFull = 12, kBarOFree = 14, kBarLReady = 16, kBarSlotFull = 18,
              kBarSlotEmpty = kBarSlotFull + kTcMaxSlots, kBarDrain = kBarSlotEmpty + kTcMaxSlots,
              kNumBars = kBarDrain + 1;
// after the barriers: abort flag, TMEM address, item -> sequence table, then
// the row sums and reference maxima handed to the epilogue ([2][128] each)
constexpr int kAbortOff = kNumBars * 8, kTmemOff = kAbortOff + 4, kSeqTabOff = kTmemOff + 4;
constexpr int kLmOff = kSeqTabOff + kTcMaxRanked * 4;
constexpr int kTailBytes = kLmOff + 2 * 2 * kTcRows * 4;
constexpr int kSmemLimit = 227 * 1024;
// A row's reference max moves only when a tile exceeds it by more than this
// (base 2): probabilities stay below 2^8 and O is rescaled rarely.
constexpr float kRescaleThreshold = 8.f;
// registers a thread of each warpgroup holds after setmaxnreg (x128 threads:
// 2 x 184 + 72 + 72 = 512 = the 128 a thread of the 512 is launched with)
constexpr int kRegsSoftmax = 184, kRegsEpilogue = 72, kRegsAux = 72;

__host__ __device__ constexpr int tile_bytes(int D) { return kTcRows * D * 2; }

struct Layout {
  int q, p, ring, tail, total;
};

__host__ __device__ inline Layout layout_of(int D, int NQ, int nslot) {
  Layout L;
  L.q = 0;
  L.p = NQ * tile_bytes(D);
  L.ring = L.p + NQ * kPBytes;
  L.tail = L.ring + nslot * tile_bytes(D);
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
// L2 prefetch of a 3-D tensor box (the next item's query tile).
__device__ __forceinline__ void tma_prefetch_3d(const void* map, int c0, int c1, int c2) {
  asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(c0), "r"(c1), "r"(c2)
               : "memory");
}

// Length key of the longest-first order: 128 buckets, 4 per power of two,
// descending (bucket 0 = longest).
__device__ __forceinline__ int length_bucket(int L) {
  if (L <= 0) return 127;
  const int msb = 31 - __clz(L);
  const int frac = msb >= 2 ? (L >> (msb - 2)) & 3 : (L << (2 - msb)) & 3;
  return 127 - min(msb * 4 + frac, 127);
}

struct Item {
  int s, h, qp, run, L;
  int j0[2], ntok[2];  // first new token and token count of each query tile (0: no tile)
  int kv_lo, kv_hi;    // KV tokens the item reads
  int ntiles;          // 128-token KV tiles
  bool valid;          // false: a run past the end of its context (nothing to write)
  bool final_out;      // the item writes normalised outputs (not a split partial)
};

// Work item k of this CTA (global index blockIdx.x + k * gridDim.x).
__device__ Item item_of(const TcParams& p, const int* seq_tab, int k) {
  Item it;
  const int idx = blockIdx.x + k * gridDim.x;
  const int per_h = p.n_qp * p.R;
  const int per_seq = p.Hkv * per_h;
  const int rank = idx / per_seq;
  int rem = idx - rank * per_seq;
  it.h = rem / per_h;
  rem -= it.h * per_h;
  const int qp = p.n_qp - 1 - rem / p.R;
  it.qp = qp;
  it.run = rem % p.R;
  it.s = p.rank_seqs ? seq_tab[k] : rank;
  int lmax = p.maxB * p.bs;
  if (p.partition_size > 0) lmax = min(lmax, p.Pmax * p.partition_size);
  const int L = min(max(__ldg(p.context_lens + it.s), 0), lmax);
  it.L = L;
  int jl = -1;
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int j0 = (qp * p.NQ + i) * p.T;
    const int n = i < p.NQ ? min(max(p.C - j0, 0), p.T) : 0;
    it.j0[i] = j0;
    it.ntok[i] = n;
    if (n > 0) jl = j0 + n - 1;
  }
  int lo = 0, hi = min(L, L - p.C + jl + 1);  // the last live row attends to tokens < hi
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

__global__ void __launch_bounds__(kTcThreads, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const TcParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t base = smem_u32(smem);
  // The swizzled operand tiles need 1024-byte alignment; the dynamic area
  // starts there when the kernel declares no static shared memory.
  if (base & 1023u) {
    if (tid == 0) atomicOr(p.err, kErrLayout);
    return;
  }
  const Layout Ly = layout_of(p.D, p.NQ, p.nslot);
  const int TB = tile_bytes(p.D);
  const uint32_t bar0 = base + Ly.tail;
  auto bar = [&](int k) -> uint32_t { return bar0 + 8u * k; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Ly.tail + kAbortOff);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Ly.tail + kTmemOff);
  int* seq_tab = reinterpret_cast<int*>(smem + Ly.tail + kSeqTabOff);
  float* l_buf = reinterpret_cast<float*>(smem + Ly.tail + kLmOff);  // [2][128]
  float* m_buf = l_buf + 2 * kTcRows;                                 // [2][128]
  auto q_smem = [&](int i) -> uint32_t { return base + Ly.q + i * TB; };
  auto p_smem = [&](int i) -> uint32_t { return base + Ly.p + i * kPBytes; };
  auto slot_smem = [&](int k) -> uint32_t { return base + Ly.ring + k * TB; };
  const int nk = (p.total - static_cast<int>(blockIdx.x) + static_cast<int>(gridDim.x) - 1) /
                 static_cast<int>(gridDim.x);  // this CTA's work items

  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(kBarQFull + i), 1);
      mbar_init(bar(kBarQEmpty + i), 1);
      mbar_init(bar(kBarSFull + i), 1);
      mbar_init(bar(kBarSFree + i), kTcRows);
      mbar_init(bar(kBarPFull + i), kTcRows);
      mbar_init(bar(kBarPvDone + i), 1);
      mbar_init(bar(kBarOFull + i), 1);
      mbar_init(bar(kBarOFree + i), kTcRows);
      mbar_init(bar(kBarLReady + i), kTcRows);
    }
    for (int k = 0; k < p.nslot; ++k) {
      mbar_init(bar(kBarSlotFull + k), 1);
      mbar_init(bar(kBarSlotEmpty + k), 1);
    }
    mbar_init(bar(kBarDrain), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  // Longest-first order: the sequence of each of this CTA's items, from a
  // histogram of context-length buckets built in the (not yet used) P area.
  if (p.rank_seqs) {
    int* hist = reinterpret_cast<int*>(smem + Ly.p);  // [128] counts, then [128] offsets
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
    const int per_seq = p.Hkv * p.n_qp * p.R;
    for (int k = warp; k < nk; k += kTcThreads / 32) {
      const int rank = (static_cast<int>(blockIdx.x) + k * static_cast<int>(gridDim.x)) / per_seq;
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
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  auto tS = [&](int i) -> uint32_t { return tmem + 128u * i; };
  auto tO = [&](int i) -> uint32_t { return tmem + 256u + 128u * i; };
  auto fail = [&]() {
    if (lane == 0) {
      atomicOr(p.err, kErrTimeout);
      *abort_flag = 1;
    }
  };
  // the next item with K/V tiles to process, at or after item k
  auto next_active = [&](int k, Item& it) -> int {
    for (; k < nk; ++k) {
      it = item_of(p, seq_tab, k);
      if (it.valid && it.ntiles > 0) return k;
    }
    return nk;
  };

  if (warp >= 12) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;\n" ::"n"(kRegsAux) : "memory");
    if (warp == kProdWarp) {
      // ============================ TMA producer ============================
      if (lane == 0) {
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
      }
      const int halves = p.D / 64;
      int n = 0, ql[2] = {0, 0};
      bool ok = true;
      // K or V tile t of item `it` into the next ring slot
      auto load_kv = [&](const Item& it, int t, bool is_v) -> bool {
        const int slot = n % p.nslot;
        if (n >= p.nslot && !mbar_wait(bar(kBarSlotEmpty + slot), ((n / p.nslot) - 1) & 1)) return false;
        const int tok0 = it.kv_lo + t * kTcTok;
        const int tok1 = min(tok0 + kTcTok, it.kv_hi);
        const int b0 = tok0 / p.bs;
        const int nb = (tok1 - 1) / p.bs - b0 + 1;
        const uint32_t full = bar(kBarSlotFull + slot);
        if (lane == 0) mbar_arrive_expect_tx(full, static_cast<uint32_t>(nb * p.bs * p.D * 2));
        __syncwarp();
        const int* bt_row = p.block_tables + static_cast<int64_t>(it.s) * p.maxB;
        for (int b = lane; b < nb; b += 32) {
          const int phys = __ldg(bt_row + b0 + b);
          if (!is_v && (phys < 0 || static_cast<int64_t>(phys) >= p.num_blocks)) atomicOr(p.err, kErrBlockId);
          const uint32_t dst = slot_smem(slot) + b * p.bs * 128;
          for (int hf = 0; hf < halves; ++hf)
            tma_load_4d(dst + hf * kHalfBytes, is_v ? &tmV : &tmK, full, 64 * hf, 0, it.h, phys);
        }
        __syncwarp();
        ++n;
        return true;
      };
      // the item's query tiles (one TMA box per 64-channel half: G heads x T tokens)
      auto load_q = [&](const Item& it) -> bool {
        for (int i = 0; i < 2; ++i) {
          if (it.ntok[i] == 0) continue;
          if (ql[i] >= 1 && !mbar_wait(bar(kBarQEmpty + i), (ql[i] - 1) & 1)) return false;
          if (lane == 0) {
            const uint32_t full = bar(kBarQFull + i);
            mbar_arrive_expect_tx(full, static_cast<uint32_t>(p.G * p.T * 128 * halves));
            for (int hf = 0; hf < halves; ++hf)
              tma_load_3d(q_smem(i) + hf * kHalfBytes, &tmQ, full, 64 * hf, it.h * p.G, it.s * p.C + it.j0[i]);
          }
          __syncwarp();
          ++ql[i];
        }
        return true;
      };
      Item cur;
      int k = next_active(0, cur);
      if (k < nk) ok = load_q(cur) && load_kv(cur, 0, false);
      while (ok && k < nk) {
        Item nxt;
        const int kn = next_active(k + 1, nxt);
        if (kn < nk && lane == 0) {  // the next item's query tiles into L2 ahead of time
          for (int i = 0; i < 2; ++i)
            if (nxt.ntok[i] > 0)
              for (int hf = 0; hf < halves; ++hf)
                tma_prefetch_3d(&tmQ, 64 * hf, nxt.h * p.G, nxt.s * p.C + nxt.j0[i]);
        }
        for (int t = 0; ok && t < cur.ntiles; ++t) {
          if (*abort_flag) {
            ok = false;
            break;
          }
          // consumption order of the tensor core: K of the next tile (this
          // item's, or the next item's first after its query tiles), then V
          if (t + 1 < cur.ntiles)
            ok = load_kv(cur, t + 1, false);
          else if (kn < nk)
            ok = load_q(nxt) && load_kv(nxt, 0, false);
          if (ok) ok = load_kv(cur, t, true);
        }
        k = kn;
        cur = nxt;
      }
      if (!ok) fail();
      // every load issued lands before the CTA can exit
      for (int u = max(0, n - p.nslot); u < n; ++u) mbar_wait(bar(kBarSlotFull + u % p.nslot), (u / p.nslot) & 1);
      for (int i = 0; i < 2; ++i)
        if (ql[i] > 0) mbar_wait(bar(kBarQFull + i), (ql[i] - 1) & 1);
    } else if (warp == kMmaWarp) {
      // ============================= MMA issuer =============================
      const uint32_t id_qk = tc_idesc_f16(p.bf16 != 0, false, kTcRows, kTcTok);
      const uint32_t id_pv = tc_idesc_f16(p.bf16 != 0, true, kTcRows, p.D);
      const int KS = p.D / 16;
      int n = 0, qc[2] = {0, 0}, sc[2] = {0, 0}, pc[2] = {0, 0}, oc[2] = {0, 0};
      bool ok = true, issued = false;
      auto wait_q = [&](const Item& it) -> bool {
        for (int i = 0; i < 2; ++i) {
          if (it.ntok[i] == 0) continue;
          if (!mbar_wait(bar(kBarQFull + i), qc[i] & 1)) return false;
          ++qc[i];
        }
        return true;
      };
      // S_i = Q_i K^T for the item's query tiles, MMA by MMA alternating tiles
      auto s_phase = [&](const Item& it, int t) -> bool {
        const int slot = n % p.nslot;
        if (!mbar_wait(bar(kBarSlotFull + slot), (n / p.nslot) & 1)) return false;
        for (int i = 0; i < 2; ++i)
          if (it.ntok[i] > 0 && sc[i] >= 1 && !mbar_wait(bar(kBarSFree + i), (sc[i] - 1) & 1)) return false;
        tc_fence_after();
        if (lane == 0) {
          const uint32_t kb = slot_smem(slot);
          for (int kk = 0; kk < KS; ++kk) {
            const uint32_t off = (kk >> 2) * kHalfBytes + (kk & 3) * 32;
            const uint64_t bdesc = tc_desc_sw128(kb + off, 16, 1024);
            for (int i = 0; i < 2; ++i)
              if (it.ntok[i] > 0) tc_mma_f16(tS(i), tc_desc_sw128(q_smem(i) + off, 16, 1024), bdesc, id_qk, kk > 0);
          }
          for (int i = 0; i < 2; ++i)
            if (it.ntok[i] > 0) tc_commit(bar(kBarSFull + i));
          tc_commit(bar(kBarSlotEmpty + slot));
          if (t == it.ntiles - 1)
            for (int i = 0; i < 2; ++i)
              if (it.ntok[i] > 0) tc_commit(bar(kBarQEmpty + i));
        }
        __syncwarp();
        for (int i = 0; i < 2; ++i) sc[i] += it.ntok[i] > 0;
        ++n;
        issued = true;
        return true;
      };
      // O_i += P_i V over the tile's valid tokens
      auto pv_phase = [&](const Item& it, int t) -> bool {
        const int slot = n % p.nslot;
        if (!mbar_wait(bar(kBarSlotFull + slot), (n / p.nslot) & 1)) return false;
        const int valid = min(kTcTok, it.kv_hi - (it.kv_lo + t * kTcTok));
        const int nks = (valid + 15) / 16;
        const uint32_t vb = slot_smem(slot);
        if (valid < nks * 16) {
          // rows past the context in the last k-step hold pool bytes past the
          // context or stale tiles: zero them so that 0 * junk cannot make NaN
          const int rows = nks * 16 - valid, halves = p.D / 64;
          for (int w = lane; w < rows * 8 * halves; w += 32) {
            const int row = valid + w / (8 * halves), rest = w % (8 * halves);
            st_shared_v4(vb + (rest / 8) * kHalfBytes + row * 128 + (rest % 8) * 16, 0u, 0u, 0u, 0u);
          }
          fence_proxy_async_smem();
          __syncwarp();
        }
        for (int i = 0; i < 2; ++i) {
          if (it.ntok[i] == 0) continue;
          if (!mbar_wait(bar(kBarPFull + i), pc[i] & 1)) return false;
          // O_i was last read by the epilogue of the previous item using tile i
          if (t == 0 && oc[i] >= 1 && !mbar_wait(bar(kBarOFree + i), (oc[i] - 1) & 1)) return false;
        }
        tc_fence_after();
        if (lane == 0) {
          for (int kk = 0; kk < nks; ++kk) {
            const uint64_t bdesc = tc_desc_sw128(vb + kk * 2048, kHalfBytes, 1024);
            const uint32_t aoff = (kk >> 2) * kHalfBytes + (kk & 3) * 32;
            for (int i = 0; i < 2; ++i)
              if (it.ntok[i] > 0)
                tc_mma_f16(tO(i), tc_desc_sw128(p_smem(i) + aoff, 16, 1024), bdesc, id_pv, (t > 0 || kk > 0));
          }
          for (int i = 0; i < 2; ++i)
            if (it.ntok[i] > 0) tc_commit(bar(kBarPvDone + i));
          tc_commit(bar(kBarSlotEmpty + slot));
          if (t == it.ntiles - 1)
            for (int i = 0; i < 2; ++i)
              if (it.ntok[i] > 0) tc_commit(bar(kBarOFull + i));
        }
        __syncwarp();
        for (int i = 0; i < 2; ++i) {
          pc[i] += it.ntok[i] > 0;
          if (t == it.ntiles - 1) oc[i] += it.ntok[i] > 0;
        }
        ++n;
        return true;
      };
      Item cur;
      int k = next_active(0, cur);
      if (k < nk) ok = wait_q(cur) && s_phase(cur, 0);
      while (ok && k < nk) {
        Item nxt;
        const int kn = next_active(k + 1, nxt);
        for (int t = 0; t < cur.ntiles; ++t) {
          if (*abort_flag) {
            ok = false;
            break;
          }
          // the next tile's scores overlap this tile's softmax
          if (t + 1 < cur.ntiles)
            ok = s_phase(cur, t + 1);
          else if (kn < nk)
            ok = wait_q(nxt) && s_phase(nxt, 0);
          if (!ok || !(ok = pv_phase(cur, t))) break;
        }
        k = kn;
        cur = nxt;
      }
      if (!ok) fail();
      // every MMA issued has completed before tensor memory is released
      if (issued) {
        if (lane == 0) tc_commit(bar(kBarDrain));
        __syncwarp();
        mbar_wait(bar(kBarDrain), 0);
      }
    }  // warps 14, 15: idle
  } else if (warp < 8) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;\n" ::"n"(kRegsSoftmax) : "memory");
    // ===================== softmax: one thread per row =====================
    const int i = warp >> 2;  // query tile
    const int r = tid & 127;  // row = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t prow = p_smem(i) + r * 128;
    const int rsw = r & 7;
    int sc = 0, pcnt = 0, oc = 0;
    bool ok = true;
    for (int k = 0; ok && k < nk; ++k) {
      const Item it = item_of(p, seq_tab, k);
      if (!it.valid || it.ntiles == 0 || it.ntok[i] == 0) continue;
      const bool live = r < it.ntok[i] * p.G;
      const int pos = live ? it.L - p.C + it.j0[i] + r / p.G : -1;
      const int last = min(pos, it.kv_hi - 1);  // last token this row attends to
      float m = -CUDART_INF_F, l = 0.f;         // reference max (base 2) and row sum
      for (int t = 0; t < it.ntiles; ++t) {
        if (*abort_flag) {
          ok = false;
          break;
        }
        if (!(ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar(kBarSFull + i), sc & 1)))) break;
        tc_fence_after();
        float sv[128];
#pragma unroll
        for (int c = 0; c < 4; ++c)
          tmem_ld32(tS(i) + lane_off + c * 32, *reinterpret_cast<float(*)[32]>(sv + 32 * c));
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(bar(kBarSFree + i));  // the next scores may overwrite the buffer
        ++sc;
        const int lim = last - (it.kv_lo + t * kTcTok);  // last visible column of this tile
        if (!__all_sync(0xFFFFFFFFu, lim >= kTcTok - 1)) {
#pragma unroll
          for (int c = 0; c < 128; ++c) sv[c] = (c <= lim) ? sv[c] : -CUDART_INF_F;
        }
        float mx8[8];
#pragma unroll
        for (int a = 0; a < 8; ++a) mx8[a] = -CUDART_INF_F;
#pragma unroll
        for (int c = 0; c < 128; c += 2) mx8[(c >> 1) & 7] = fmax3(mx8[(c >> 1) & 7], sv[c], sv[c + 1]);
        const float mx = p.scale_log2 * fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                                              fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
        const bool bump = mx > m + kRescaleThreshold;  // false while both are -inf
        float alpha = 1.f;
        if (bump) {
          alpha = m == -CUDART_INF_F ? 0.f : ex2(m - mx);
          m = mx;
        }
        const float m_use = m == -CUDART_INF_F ? 0.f : m;
        const uint64_t sc2 = f2pack(p.scale_log2, p.scale_log2), nm2 = f2pack(-m_use, -m_use);
        uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
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
        l = l * alpha + (((sum8[0] + sum8[1]) + (sum8[2] + sum8[3])) + ((sum8[4] + sum8[5]) + (sum8[6] + sum8[7])));
        uint32_t pw[64];
#pragma unroll
        for (int c = 0; c < 64; ++c) pw[c] = pack16(sv[2 * c], sv[2 * c + 1], p.bf16);
        // P_i and O_i are free once the previous P.V of this tile slot has completed
        if (pcnt >= 1 && !(ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar(kBarPvDone + i), (pcnt - 1) & 1)))) break;
        if (t > 0 && __any_sync(0xFFFFFFFFu, bump)) {
          // rows whose reference moved rescale their O row (others multiply by 1)
          tc_fence_after();
          for (int c = 0; c < p.D / 32; ++c) {
            float o[32];
            tmem_ld32(tO(i) + lane_off + c * 32, o);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] *= alpha;
            tmem_st32(tO(i) + lane_off + c * 32, o);
          }
          tmem_wait_st();
        }
#pragma unroll
        for (int c = 0; c < 16; ++c)
          st_shared_v4(prow + (c >> 3) * kHalfBytes + (((c & 7) ^ rsw) << 4), pw[4 * c], pw[4 * c + 1],
                       pw[4 * c + 2], pw[4 * c + 3]);
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(bar(kBarPFull + i));
        ++pcnt;
      }
      if (!ok) break;
      // hand (l, m) to the epilogue; the slot was read by the previous item's epilogue
      if (oc >= 1 && !(ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar(kBarOFree + i), (oc - 1) & 1)))) break;
      l_buf[i * kTcRows + r] = l;
      m_buf[i * kTcRows + r] = m;
      mbar_arrive(bar(kBarLReady + i));
      ++oc;
    }
    if (!ok) fail();
  } else {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;\n" ::"n"(kRegsEpilogue) : "memory");
    // ====================== epilogue: one thread per row ======================
    const int r = tid & 127;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    int oc[2] = {0, 0};
    bool ok = true;
    for (int k = 0; ok && k < nk; ++k) {
      const Item it = item_of(p, seq_tab, k);
      if (r == 0 && it.h == 0 && it.run == 0 && it.qp == p.n_qp - 1) {  // once per sequence
        const int L = __ldg(p.context_lens + it.s);
        if (L != it.L) atomicOr(p.err, kErrContextLen);  // negative, or past the table (or partitions)
      }
      if (!it.valid) continue;
      for (int i = 0; i < 2; ++i) {
        if (it.ntok[i] == 0) continue;
        const bool live = r < it.ntok[i] * p.G;
        const int j = it.j0[i] + r / p.G;
        const int64_t row = (static_cast<int64_t>(it.s) * p.C + j) * p.Hq + it.h * p.G + r % p.G;
        const bool have = it.ntiles > 0;
        float l = 0.f, m = -CUDART_INF_F;
        if (have) {
          // the epilogue idles through most of an item: poll with a pause (at
          // most about 50 ms) so that it takes few issue slots from the
          // softmax warps, then the usual bounded wait
          for (int spin = 0; spin < 200000 && !mbar_try_wait(bar(kBarOFull + i), oc[i] & 1); ++spin)
            __nanosleep(256);
          ok = !*abort_flag && __all_sync(0xFFFFFFFFu, mbar_wait(bar(kBarOFull + i), oc[i] & 1)) &&
               __all_sync(0xFFFFFFFFu, mbar_wait(bar(kBarLReady + i), oc[i] & 1));
          if (!ok) break;
          tc_fence_after();
          l = l_buf[i * kTcRows + r];
          m = m_buf[i * kTcRows + r];
        }
        const bool final_out = it.final_out;
        const float inv = l > 0.f ? 1.f / l : 0.f;
        for (int c = 0; c < p.D / 32; ++c) {
          float o[32];
          if (have) {
            tmem_ld32(tO(i) + lane_off + c * 32, o);
            tmem_wait_ld();
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = 0.f;
          }
          if (!live) continue;
          if (final_out) {
            uint16_t* orow = static_cast<uint16_t*>(p.out) + row * p.D + c * 32;
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
              uint4 w;
              w.x = pack16(o[8 * q4 + 0] * inv, o[8 * q4 + 1] * inv, p.bf16);
              w.y = pack16(o[8 * q4 + 2] * inv, o[8 * q4 + 3] * inv, p.bf16);
              w.z = pack16(o[8 * q4 + 4] * inv, o[8 * q4 + 5] * inv, p.bf16);
              w.w = pack16(o[8 * q4 + 6] * inv, o[8 * q4 + 7] * inv, p.bf16);
              *reinterpret_cast<uint4*>(orow + q4 * 8) = w;
            }
          } else {
            float4* dst = reinterpret_cast<float4*>(p.ws_o + (row * p.Pmax + it.run) * p.D + c * 32);
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4)
              dst[q4] = make_float4(o[4 * q4], o[4 * q4 + 1], o[4 * q4 + 2], o[4 * q4 + 3]);
          }
        }
        if (live && !final_out) {
          const int64_t slot = row * p.Pmax + it.run;
          p.ws_ml[2 * slot] = l > 0.f ? m : -CUDART_INF_F;
          p.ws_ml[2 * slot + 1] = l;
        }
        if (have) {
          // O_i and the (l, m) slot may take the next item's
          tc_fence_before();
          mbar_arrive(bar(kBarOFree + i));
          ++oc[i];
        }
      }
    }
    if (!ok) fail();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

int tc_ring_slots(int D, int NQ) {
  const Layout L0 = layout_of(D, NQ, 0);
  const int n = (kSmemLimit - L0.total) / tile_bytes(D);
  return n < kTcMaxSlots ? n : kTcMaxSlots;
}

int tc_smem_bytes(int D, int NQ, int nslot) { return layout_of(D, NQ, nslot).total; }

cudaError_t launch_attn_tc(const TcParams& p, const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                           cudaStream_t st) {
  if (p.nslot < 3 || p.nslot > kTcMaxSlots) return cudaErrorInvalidValue;
  const int smem = tc_smem_bytes(p.D, p.NQ, p.nslot);
  if (smem > kSmemLimit) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  // the warpgroups' setmaxnreg shares must fit in the registers the CTA is
  // launched with, or the softmax warps' increase would never be granted
  static std::atomic<int> launch_regs{0};
  int regs = launch_regs.load(std::memory_order_relaxed);
  if (regs == 0) {
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, attn_tc_kernel);
    if (e != cudaSuccess) return e;
    regs = fa.numRegs;
    launch_regs.store(regs, std::memory_order_relaxed);
  }
  if (128 * (2 * kRegsSoftmax + kRegsEpilogue + kRegsAux) > regs * kTcThreads) return cudaErrorInvalidConfiguration;
  static std::atomic<int> sms[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
  int nsm = sms[dev].load(std::memory_order_relaxed);
  if (nsm == 0) {
    if (cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || nsm <= 0) nsm = 148;
    sms[dev].store(nsm, std::memory_order_relaxed);
  }
  if (p.total <= 0) return cudaSuccess;
  // persistent: one CTA per SM (the kernel holds all of an SM's tensor memory)
  const int grid = p.total < nsm ? p.total : nsm;
  TcParams q = p;
  // items per CTA beyond the table are not ordered
  if ((p.total + grid - 1) / grid > kTcMaxRanked) q.rank_seqs = 0;
  attn_tc_kernel<<<grid, kTcThreads, smem, st>>>(tmQ, tmK, tmV, q);
  return cudaGetLastError();
}

}  // namespace pa
