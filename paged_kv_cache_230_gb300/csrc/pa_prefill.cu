// Paged prefill (chunked prefill) attention on the 5th-generation tensor
// cores.  C new query tokens per sequence sit at positions L - C .. L - 1 and
// attend causally to every cached token up to their own position, through
// the block table (prefill is the compute-bound phase of the review's §7;
// chunked prefill interleaves such chunks with decode, §10 table).
//
// CTA = (sequence, query head, 128 query rows); 7 warps:
//   warps 4 and 6  TMA: the q tile once, then 128-token K (warp 4) and V
//           (warp 6) tiles, block by block through the block table, each
//           into its own 2-stage ring (128-byte swizzle, the canonical
//           K-major layout of the MMA operands); K buffers are released when
//           QK^T completes, V buffers when P.V completes;
//   warp 5  one thread issues tcgen05.mma: S = Q K^T (M = 128 rows, N = 128
//           tokens, K = 128 channels) into one of two TMEM score buffers
//           (the next tile's scores are computed while this tile's softmax
//           runs), then, once the probabilities are ready, O += P V (N = 128
//           channels, K = 128 tokens, V read channel-major) into a third;
//   warps 0-3  one thread per query row (= TMEM lane): reads its S row with
//           tcgen05.ld, applies the causal mask and the online softmax in
//           base 2 (no cross-thread reduction), writes P as 16-bit pairs
//           over the first 64 columns of its own S buffer in TMEM (the A
//           operand of P.V comes from TMEM, so shared memory only feeds K, V
//           and Q to the tensor core), rescales its O row in TMEM when its
//           reference max moved by more than 2^8, and at the end writes O / l.
// Every mbarrier wait gives up after about one second (error bit set).
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
constexpr int kQOff = 0;
constexpr int kKVOff = kQOff + kTileBytes;                    // stage st: K at +2*st*tile, V after it
constexpr int kBarOff = kKVOff + kPfStages * 2 * kTileBytes;
// mbarriers: q, K full/empty and V full/empty per stage, S full, P full and
// O done per TMEM buffer; then the TMEM address slot
constexpr int kBarBytes = 8 + 32 * kPfStages + 48 + 8;
constexpr int kSmemBytes = 1024 + kBarOff + kBarBytes;
constexpr uint32_t kTmemCols = 512;  // S buffers in columns [0, 128) and [128, 256), O in [256, 384)
// A row's reference max moves only when the tile max exceeds it by more than
// this (base 2): probabilities then stay below 2^8 and O is rescaled rarely.
constexpr float kRescaleThreshold = 8.f;

static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");

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

__global__ void __launch_bounds__(kPfThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const PrefillParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
  const uint32_t base = smem_u32(smem);
  const uint32_t q_s = base + kQOff;
  const uint32_t bar0 = base + kBarOff;
  // per-buffer barriers (index = tile parity), so no wait is on an ambiguous
  // phase; K and V have their own buffers: K of a tile is released as soon as
  // its QK^T completes, V only after its P.V
  const uint32_t q_full = bar0, k_full0 = bar0 + 8, k_empty0 = k_full0 + 8 * kPfStages;
  const uint32_t v_full0 = k_empty0 + 8 * kPfStages, v_empty0 = v_full0 + 8 * kPfStages;
  const uint32_t s_full0 = v_empty0 + 8 * kPfStages, p_full0 = s_full0 + 16, o_done0 = p_full0 + 16;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kBarOff + kBarBytes - 8);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nqt = (p.C + kPfRows - 1) / kPfRows;
  const int qt = blockIdx.x % nqt;
  const int sh = blockIdx.x / nqt;
  const int h = sh % p.Hq, s = sh / p.Hq;
  const int hkv = h / p.G;
  const int lmax = p.maxB * p.bs;
  int L = p.context_lens[s];
  if (L < 0 || L > lmax) {
    if (tid == 0 && qt == 0 && h == 0) atomicOr(p.err, kErrContextLen);
    L = min(max(L, 0), lmax);
  }
  const int i0 = qt * kPfRows;                      // first query row of this CTA
  const int rows = min(kPfRows, p.C - i0);           // live rows
  const int pos0 = L - p.C + i0;                     // position of row 0 (may be negative)
  const int kv_len = max(0, min(L, pos0 + rows));    // tokens any live row attends to
  const int ntiles = (kv_len + kPfTile - 1) / kPfTile;

  if (tid == 0) {
    mbar_init(q_full, 1);
    for (int st = 0; st < kPfStages; ++st) {
      mbar_init(k_full0 + 8 * st, 1);
      mbar_init(k_empty0 + 8 * st, 1);
      mbar_init(v_full0 + 8 * st, 1);
      mbar_init(v_empty0 + 8 * st, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(s_full0 + 8 * b, 1);
      mbar_init(p_full0 + 8 * b, 128);
      mbar_init(o_done0 + 8 * b, 1);
    }
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tS0 = tmem, tO = tmem + 256;

  if (warp == 4 || warp == 6) {
    // ===================== TMA producers: warp 4 K, warp 6 V =====================
    const bool is_k = warp == 4;
    if (ntiles > 0) {
      if (lane == 0 && is_k) {
        tma_prefetch_desc(&tmK);
        mbar_arrive_expect_tx(q_full, kTileBytes);
        const int row = s * p.C + i0;
        tma_load_3d(q_s, &tmQ, q_full, 0, h, row);
        tma_load_3d(q_s + kSegBytes, &tmQ, q_full, 64, h, row);
      }
      if (lane == 0 && !is_k) tma_prefetch_desc(&tmV);
      const CUtensorMap* map = is_k ? &tmK : &tmV;
      const uint32_t full0 = is_k ? k_full0 : v_full0, empty0 = is_k ? k_empty0 : v_empty0;
      const uint32_t dst0 = base + kKVOff + (is_k ? 0 : kTileBytes);
      const int* bt_row = p.block_tables + static_cast<int64_t>(s) * p.maxB;
      const int bpt = kPfTile / p.bs;
      const int nblk = (kv_len + p.bs - 1) / p.bs;
      const uint32_t tx_block = static_cast<uint32_t>(p.bs * 256);
      for (int t = 0; t < ntiles; ++t) {
        const int st = t % kPfStages;
        bool ok = true;
        if (t >= kPfStages) ok = mbar_wait(empty0 + 8 * st, ((t / kPfStages) - 1) & 1);
        if (!ok) {
          if (lane == 0) atomicOr(p.err, kErrTimeout);
          break;
        }
        const int b0 = t * bpt;
        const int nb = min(bpt, nblk - b0);
        const uint32_t full = full0 + 8 * st;
        if (lane == 0) mbar_arrive_expect_tx(full, tx_block * nb);
        __syncwarp();
        if (lane < nb) {  // one block per lane, issued together
          const int phys = __ldg(bt_row + b0 + lane);
          if (is_k && (phys < 0 || static_cast<int64_t>(phys) >= p.num_blocks)) atomicOr(p.err, kErrBlockId);
          const uint32_t dst = dst0 + st * 2 * kTileBytes + lane * p.bs * 128;
          tma_load_4d(dst, map, full, 0, 0, hkv, phys);
          tma_load_4d(dst + kSegBytes, map, full, 64, 0, hkv, phys);
        }
        __syncwarp();
      }
    }
  } else if (warp == 5) {
    // ============================ MMA issuer ============================
    if (ntiles > 0 && lane == 0) {
      const uint32_t id_qk = tc_idesc_f16(p.bf16 != 0, false, kPfRows, kPfTile);
      const uint32_t id_pv = tc_idesc_f16(p.bf16 != 0, true, kPfRows, 128);
      bool ok = mbar_wait(q_full, 0);
      // S(t) = Q K(t)^T into S buffer t % 2, both operands K-major (channels
      // contiguous), 16 channels per step
      auto issue_qk = [&](int t) -> bool {
        const int st = t % kPfStages;
        if (!mbar_wait(k_full0 + 8 * st, (t / kPfStages) & 1)) return false;
        tc_fence_after();
        const uint32_t k_s = base + kKVOff + st * 2 * kTileBytes;
        const uint32_t tS = tS0 + (t & 1) * 128;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint32_t off = (j >> 2) * kSegBytes + (j & 3) * 32;
          tc_mma_f16(tS, tc_desc_sw128(q_s + off, 16, 1024), tc_desc_sw128(k_s + off, 16, 1024), id_qk, j > 0);
        }
        tc_commit(s_full0 + 8 * (t & 1));
        tc_commit(k_empty0 + 8 * st);
        return true;
      };
      if (ok) ok = issue_qk(0);
      for (int t = 0; ok && t < ntiles; ++t) {
        // the next tile's scores overlap this tile's softmax; its S buffer was
        // released when the softmax of tile t - 1 arrived on p_full
        if (t + 1 < ntiles && !(ok = issue_qk(t + 1))) break;
        if (!(ok = mbar_wait(p_full0 + 8 * (t & 1), (t >> 1) & 1))) break;
        const int st = t % kPfStages;
        if (!(ok = mbar_wait(v_full0 + 8 * st, (t / kPfStages) & 1))) break;
        tc_fence_after();
        // O += P V: P from TMEM (16 tokens = 8 columns per step); V
        // channel-major: 64-channel halves 16 KB apart, 8-token groups 1 KB apart
        const uint32_t v_s = base + kKVOff + st * 2 * kTileBytes + kTileBytes;
        const uint32_t p_t = tS0 + (t & 1) * 128;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint64_t b = tc_desc_sw128(v_s + j * 2048, kSegBytes, 1024);
          tc_mma_f16_ts(tO, p_t + j * 8, b, id_pv, (t > 0 || j > 0) ? 1u : 0u);
        }
        tc_commit(o_done0 + 8 * (t & 1));
        tc_commit(v_empty0 + 8 * st);
      }
      if (!ok) atomicOr(p.err, kErrTimeout);
    }
  } else {
    // ====================== softmax: one thread per row ======================
    const int r = tid;                 // query row = TMEM lane
    const int pos = pos0 + r;          // its position; it attends to tokens 0..pos
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    float m = -CUDART_INF_F, l = 0.f;  // m: this row's reference max (base 2)
    bool ok = true;
    for (int t = 0; t < ntiles; ++t) {
      const int st = t % kPfStages;
      const int buf = t & 1;
      if (!(ok = __all_sync(0xFFFFFFFFu, mbar_wait(s_full0 + 8 * buf, (t >> 1) & 1)))) break;
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
        for (int k = 0; k < 128; ++k) sv[k] = (k <= lim) ? sv[k] : -CUDART_INF_F;
      }
      // max of the raw scores (the scale is positive), 8 independent chains:
      // one softmax warp per SM sub-partition has nothing else to hide the
      // latency of long dependent chains with
      float mx8[8];
#pragma unroll
      for (int a = 0; a < 8; ++a) mx8[a] = -CUDART_INF_F;
#pragma unroll
      for (int k = 0; k < 128; k += 2) mx8[(k >> 1) & 7] = fmax3(mx8[(k >> 1) & 7], sv[k], sv[k + 1]);
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
      for (int k = 0; k < 128; k += 2) {
        float lo, hi;
        f2unpack(ffma2(f2pack(sv[k], sv[k + 1]), sc2, nm2), lo, hi);
        sv[k] = ex2(lo);
        sv[k + 1] = ex2(hi);
        acc[(k >> 1) & 3] = fadd2(acc[(k >> 1) & 3], f2pack(sv[k], sv[k + 1]));
      }
      float sum8[8];
#pragma unroll
      for (int a = 0; a < 4; ++a) f2unpack(acc[a], sum8[2 * a], sum8[2 * a + 1]);
      const float sum = ((sum8[0] + sum8[1]) + (sum8[2] + sum8[3])) + ((sum8[4] + sum8[5]) + (sum8[6] + sum8[7]));
      l = l * alpha + sum;
      // P(t) over the first 64 columns of S buffer `buf`: S(t) was issued
      // after P.V of tile t - 2, so that MMA has finished reading P(t - 2)
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
        if (!(ok = __all_sync(0xFFFFFFFFu, mbar_wait(v_full0 + 8 * st, (t / kPfStages) & 1)))) break;
        if (r >= kv_len - tok0) {
          uint8_t* vrow = smem + kKVOff + st * 2 * kTileBytes + kTileBytes + r * 128;
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            *reinterpret_cast<uint4*>(vrow + c * 16) = make_uint4(0, 0, 0, 0);
            *reinterpret_cast<uint4*>(vrow + kSegBytes + c * 16) = make_uint4(0, 0, 0, 0);
          }
        }
      }
      // rescale O rows whose reference moved, once P.V of tile t - 1 is done
      // (warp-uniform: the TMEM moves are warp-wide; other rows multiply by 1)
      if (t > 0 && __any_sync(0xFFFFFFFFu, bump)) {
        if (!(ok = __all_sync(0xFFFFFFFFu, mbar_wait(o_done0 + 8 * (buf ^ 1), ((t - 1) >> 1) & 1)))) break;
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          float o[32];
          tmem_ld32(tO + lane_off + c * 32, o);
          tmem_wait_ld();
#pragma unroll
          for (int k = 0; k < 32; ++k) o[k] *= alpha;
          tmem_st32(tO + lane_off + c * 32, o);
        }
      }
      tmem_wait_st();
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(p_full0 + 8 * buf);
    }
    if (ok && ntiles > 0)
      ok = __all_sync(0xFFFFFFFFu, mbar_wait(o_done0 + 8 * ((ntiles - 1) & 1), ((ntiles - 1) >> 1) & 1));
    if (!ok && lane == 0) atomicOr(p.err, kErrTimeout);
    tc_fence_after();
    const float inv = l > 0.f ? 1.f / l : 0.f;
    uint16_t* orow = static_cast<uint16_t*>(p.out) + ((static_cast<int64_t>(s) * p.C + i0 + r) * p.Hq + h) * 128;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      float o[32];
      if (ntiles > 0 && ok) {
        tmem_ld32(tO + lane_off + c * 32, o);
        tmem_wait_ld();
      } else {
#pragma unroll
        for (int k = 0; k < 32; ++k) o[k] = 0.f;
      }
      if (r < rows) {
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
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

cudaError_t launch_prefill(const PrefillParams& p, const CUtensorMap& tmQ, const CUtensorMap& tmK,
                           const CUtensorMap& tmV, cudaStream_t st) {
  cudaError_t e = cudaFuncSetAttribute(prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  const long long nqt = (p.C + kPfRows - 1) / kPfRows;
  const long long grid = nqt * p.Hq * p.S;
  prefill_kernel<<<static_cast<unsigned>(grid), kPfThreads, kSmemBytes, st>>>(tmQ, tmK, tmV, p);
  return cudaGetLastError();
}

}  // namespace pa
