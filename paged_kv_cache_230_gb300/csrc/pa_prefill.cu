// Paged prefill (chunked prefill) attention on the 5th-generation tensor
// cores.  C new query tokens per sequence sit at positions L - C .. L - 1 and
// attend causally to every cached token up to their own position, through
// the block table (prefill is the compute-bound phase of the review's §7;
// chunked prefill interleaves such chunks with decode, §10 table).
//
// CTA = (sequence, query head, 128 query rows); 6 warps:
//   warp 4  TMA: the q tile once, then 128-token K and V tiles, block by
//           block through the block table, into a 2-stage ring (128-byte
//           swizzle, the canonical K-major layout of the MMA operands);
//   warp 5  one thread issues tcgen05.mma: S = Q K^T (M = 128 rows, N = 128
//           tokens, K = 128 channels) into tensor memory, then, once the
//           probabilities are ready, O += P V (N = 128 channels, K = 128
//           tokens, V read channel-major) into a second TMEM region;
//   warps 0-3  one thread per query row (= TMEM lane): reads its S row with
//           tcgen05.ld, applies the causal mask and the online softmax in
//           base 2 (no cross-thread reduction), writes P as 16-bit values to
//           shared memory in the A-operand layout, rescales its O row in TMEM
//           when the running max moved, and at the end writes O / l.
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
constexpr int kPOff = kKVOff + kPfStages * 2 * kTileBytes;   // probabilities, A operand of P.V
constexpr int kBarOff = kPOff + kTileBytes;                   // 8 mbarriers + TMEM address slot
constexpr int kSmemBytes = 1024 + kBarOff + 128;
constexpr uint32_t kTmemCols = 256;  // S in columns [0, 128), O in [128, 256)

static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");

__device__ __forceinline__ uint32_t swz128(uint32_t off) { return off ^ ((off >> 3) & 0x70); }

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
  const uint32_t q_s = base + kQOff, p_s = base + kPOff;
  const uint32_t bar0 = base + kBarOff;
  const uint32_t q_full = bar0, kv_full0 = bar0 + 8, kv_empty0 = bar0 + 24;
  const uint32_t s_full = bar0 + 40, p_full = bar0 + 48, o_done = bar0 + 56;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kBarOff + 64);

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
      mbar_init(kv_full0 + 8 * st, 1);
      mbar_init(kv_empty0 + 8 * st, 1);
    }
    mbar_init(s_full, 1);
    mbar_init(p_full, 128);
    mbar_init(o_done, 1);
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
  const uint32_t tS = tmem, tO = tmem + 128;

  if (warp == 4) {
    // ============================ TMA producer ============================
    if (ntiles > 0) {
      if (lane == 0) {
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        mbar_arrive_expect_tx(q_full, kTileBytes);
        const int row = s * p.C + i0;
        tma_load_3d(q_s, &tmQ, q_full, 0, h, row);
        tma_load_3d(q_s + kSegBytes, &tmQ, q_full, 64, h, row);
      }
      const int* bt_row = p.block_tables + static_cast<int64_t>(s) * p.maxB;
      const int bpt = kPfTile / p.bs;
      const int nblk = (kv_len + p.bs - 1) / p.bs;
      const uint32_t tx_block = static_cast<uint32_t>(2 * p.bs * 256);
      for (int t = 0; t < ntiles; ++t) {
        const int st = t % kPfStages;
        bool ok = true;
        if (t >= kPfStages) ok = mbar_wait(kv_empty0 + 8 * st, ((t / kPfStages) - 1) & 1);
        if (!ok) {
          if (lane == 0) atomicOr(p.err, kErrTimeout);
          break;
        }
        const int b0 = t * bpt;
        const int nb = min(bpt, nblk - b0);
        const uint32_t full = kv_full0 + 8 * st;
        if (lane == 0) mbar_arrive_expect_tx(full, tx_block * nb);
        __syncwarp();
        if (lane < nb) {  // one block per lane, issued together
          const int phys = __ldg(bt_row + b0 + lane);
          if (phys < 0 || static_cast<int64_t>(phys) >= p.num_blocks) atomicOr(p.err, kErrBlockId);
          const uint32_t kdst = base + kKVOff + st * 2 * kTileBytes + lane * p.bs * 128;
          const uint32_t vdst = kdst + kTileBytes;
          tma_load_4d(kdst, &tmK, full, 0, 0, hkv, phys);
          tma_load_4d(kdst + kSegBytes, &tmK, full, 64, 0, hkv, phys);
          tma_load_4d(vdst, &tmV, full, 0, 0, hkv, phys);
          tma_load_4d(vdst + kSegBytes, &tmV, full, 64, 0, hkv, phys);
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
      for (int t = 0; ok && t < ntiles; ++t) {
        const int st = t % kPfStages;
        if (!(ok = mbar_wait(kv_full0 + 8 * st, (t / kPfStages) & 1))) break;
        tc_fence_after();
        const uint32_t k_s = base + kKVOff + st * 2 * kTileBytes, v_s = k_s + kTileBytes;
        // S = Q K^T: both operands K-major (channels contiguous), 16 channels per step
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint32_t off = (j >> 2) * kSegBytes + (j & 3) * 32;
          tc_mma_f16(tS, tc_desc_sw128(q_s + off, 16, 1024), tc_desc_sw128(k_s + off, 16, 1024), id_qk, j > 0);
        }
        tc_commit(s_full);
        if (!(ok = mbar_wait(p_full, t & 1))) break;
        tc_fence_after();
        // O += P V: P K-major (tokens contiguous); V channel-major: 64-channel
        // halves 16 KB apart, 8-token groups 1 KB apart, 16 tokens per step
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint64_t a = tc_desc_sw128(p_s + (j >> 2) * kSegBytes + (j & 3) * 32, 16, 1024);
          const uint64_t b = tc_desc_sw128(v_s + j * 2048, kSegBytes, 1024);
          tc_mma_f16(tO, a, b, id_pv, (t > 0 || j > 0) ? 1u : 0u);
        }
        tc_commit(o_done);
        tc_commit(kv_empty0 + 8 * st);
      }
      if (!ok) atomicOr(p.err, kErrTimeout);
    }
  } else {
    // ====================== softmax: one thread per row ======================
    const int r = tid;                 // query row = TMEM lane
    const int pos = pos0 + r;          // its position; it attends to tokens 0..pos
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    float m = -CUDART_INF_F, l = 0.f;
    bool ok = true;
    for (int t = 0; t < ntiles; ++t) {
      const int st = t % kPfStages;
      if (!(ok = __all_sync(0xFFFFFFFFu, mbar_wait(s_full, t & 1)))) break;
      tc_fence_after();
      float sv[128];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(tS + lane_off + c * 32, *reinterpret_cast<float(*)[32]>(sv + 32 * c));
      tmem_wait_ld();
      const int tok0 = t * kPfTile;
      float mx = -CUDART_INF_F;
#pragma unroll
      for (int k = 0; k < 128; ++k) {
        const float x = (tok0 + k <= pos) ? sv[k] * p.scale_log2 : -CUDART_INF_F;
        sv[k] = x;
        mx = fmaxf(mx, x);
      }
      const float m_new = fmaxf(m, mx);
      const float m_use = m_new == -CUDART_INF_F ? 0.f : m_new;
      float alpha = ex2(m - m_use);
      float sum = 0.f;
#pragma unroll
      for (int k = 0; k < 128; ++k) {
        sv[k] = ex2(sv[k] - m_use);
        sum += sv[k];
      }
      l = l * alpha + sum;
      m = m_new;
      // P.V of the previous tile must be done before P and O are touched again
      if (t > 0 && !(ok = __all_sync(0xFFFFFFFFu, mbar_wait(o_done, (t - 1) & 1)))) break;
      tc_fence_after();
      uint8_t* prow = smem + kPOff + r * 128;
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        uint4 w;
        w.x = pack16(sv[8 * c + 0], sv[8 * c + 1], p.bf16);
        w.y = pack16(sv[8 * c + 2], sv[8 * c + 3], p.bf16);
        w.z = pack16(sv[8 * c + 4], sv[8 * c + 5], p.bf16);
        w.w = pack16(sv[8 * c + 6], sv[8 * c + 7], p.bf16);
        const uint32_t off = swz128(static_cast<uint32_t>(r * 128 + (c & 7) * 16)) - r * 128;
        *reinterpret_cast<uint4*>(prow + (c >> 3) * kSegBytes + off) = w;
      }
      if (t == ntiles - 1 && r >= kv_len - tok0) {
        // rows of the last V tile past the context hold whatever the pool had:
        // zero them so that 0 * value cannot produce NaN in P.V
        uint8_t* vrow = smem + kKVOff + st * 2 * kTileBytes + kTileBytes + r * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          *reinterpret_cast<uint4*>(vrow + c * 16) = make_uint4(0, 0, 0, 0);
          *reinterpret_cast<uint4*>(vrow + kSegBytes + c * 16) = make_uint4(0, 0, 0, 0);
        }
      }
      // rescale this row of O when the running max moved (warp-uniform: the
      // TMEM moves are warp-wide; rows whose max did not move multiply by 1)
      if (t > 0 && __any_sync(0xFFFFFFFFu, alpha != 1.f)) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          float o[32];
          tmem_ld32(tO + lane_off + c * 32, o);
          tmem_wait_ld();
#pragma unroll
          for (int k = 0; k < 32; ++k) o[k] *= alpha;
          tmem_st32(tO + lane_off + c * 32, o);
        }
        tmem_wait_st();
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(p_full);
    }
    if (ok && ntiles > 0) ok = __all_sync(0xFFFFFFFFu, mbar_wait(o_done, (ntiles - 1) & 1));
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
