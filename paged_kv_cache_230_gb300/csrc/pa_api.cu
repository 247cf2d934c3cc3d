// C-ABI front end of libpagedattn.so: argument checks, TMA tensor-map
// encoding for the paged caches, launches, and the device error word.
#include <atomic>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "pagedattn.h"
#include "pa_attn_tc.h"
#include "pa_internal.h"
#include "pa_prefill.h"
#include "pa_widen.h"

namespace {

// Errors recorded by kernels (PA_DEVERR_* bits); one word per device.
__device__ int g_device_error;

constexpr int kMaxDevices = 64;
int* g_err_ptr[kMaxDevices];
std::mutex g_err_mu;

int* device_error_ptr() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_err_mu);
  if (!g_err_ptr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_device_error) != cudaSuccess) return nullptr;
    g_err_ptr[dev] = static_cast<int*>(ptr);
  }
  return g_err_ptr[dev];
}

std::atomic<int> g_check{-1};

bool check_mode() {
  int v = g_check.load();
  if (v < 0) {
    const char* e = std::getenv("PA_CHECK");
    v = (e && e[0] && e[0] != '0') ? 1 : 0;
    int expected = -1;
    g_check.compare_exchange_strong(expected, v);
    v = g_check.load();
  }
  return v != 0;
}

int read_and_clear_error(cudaStream_t st, bool whole_device) {
  cudaError_t e = whole_device ? cudaDeviceSynchronize() : cudaStreamSynchronize(st);
  if (e != cudaSuccess) return PA_ERR_CUDA;
  int bits = 0;
  if (cudaMemcpyFromSymbol(&bits, g_device_error, sizeof(int)) != cudaSuccess) return PA_ERR_CUDA;
  const int zero = 0;
  if (cudaMemcpyToSymbol(g_device_error, &zero, sizeof(int)) != cudaSuccess) return PA_ERR_CUDA;
  return bits;
}

// After a launch in check mode: wait for it and turn recorded errors into a status.
int finish(cudaError_t launch, cudaStream_t st) {
  if (launch != cudaSuccess) return PA_ERR_CUDA;
  if (!check_mode()) return PA_OK;
  const int bits = read_and_clear_error(st, false);
  if (bits < 0) return bits;
  if (bits & PA_DEVERR_LAYOUT) return PA_ERR_CUDA;
  if (bits & PA_DEVERR_TIMEOUT) return PA_ERR_TIMEOUT;
  if (bits) return PA_ERR_BAD_INDEX;
  return PA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int elem_bytes(int dt) { return dt == PA_FP8_E4M3 ? 1 : 2; }

int check_cache(const pa_cache_desc* c, const void* k, const void* v) {
  if (!c || !k || !v) return PA_ERR_INVALID_ARG;
  if (c->num_blocks <= 0 || c->num_blocks > (int64_t(1) << 32) || c->num_kv_heads <= 0 ||
      c->num_kv_heads > 65535)
    return PA_ERR_INVALID_ARG;
  if (c->kv_dtype != PA_F16 && c->kv_dtype != PA_BF16 && c->kv_dtype != PA_FP8_E4M3) return PA_ERR_UNSUPPORTED;
  if (c->head_dim != 64 && c->head_dim != 128) return PA_ERR_UNSUPPORTED;
  if (c->block_size != 8 && c->block_size != 16 && c->block_size != 32) return PA_ERR_UNSUPPORTED;
  if (!aligned16(k) || !aligned16(v)) return PA_ERR_INVALID_ARG;
  return PA_OK;
}

int check_kv_scale(int kv_dtype, float kv_scale) {
  if (kv_dtype == PA_FP8_E4M3) return (std::isfinite(kv_scale) && kv_scale > 0.f) ? PA_OK : PA_ERR_INVALID_ARG;
  return kv_scale == 1.0f ? PA_OK : PA_ERR_INVALID_ARG;
}

// ---- TMA tensor maps over [NB, Hkv, bs, D] --------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

// Box: one block's rows (bs) x one 128-byte (or 64-byte) slice of a row, for
// one kv head of one block.  Coordinates (channel, offset, head, block).
int make_cache_tensor_map(CUtensorMap* m, const void* base, const pa_cache_desc* c) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return PA_ERR_CUDA;
  const int eb = elem_bytes(c->kv_dtype);
  const int rowb = c->head_dim * eb;
  const int boxb = rowb < 128 ? rowb : 128;
  const cuuint64_t dims[4] = {cuuint64_t(c->head_dim), cuuint64_t(c->block_size), cuuint64_t(c->num_kv_heads),
                              cuuint64_t(c->num_blocks)};
  const cuuint64_t strides[3] = {cuuint64_t(rowb), cuuint64_t(rowb) * c->block_size,
                                 cuuint64_t(rowb) * c->block_size * c->num_kv_heads};
  const cuuint32_t box[4] = {cuuint32_t(boxb / eb), cuuint32_t(c->block_size), 1, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUresult r =
      fn(m, eb == 2 ? CU_TENSOR_MAP_DATA_TYPE_UINT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(base),
         dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
         boxb == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PA_OK : PA_ERR_CUDA;
}

struct DecodeArgs {
  void* out;
  const void* q;
  int32_t q_dtype, num_seqs, num_q_heads;
  int32_t qlen;
  const void* k_cache;
  const void* v_cache;
  const pa_cache_desc* cache;
  const int32_t* block_tables;
  int32_t max_blocks_per_seq;
  const int32_t* context_lens;
  float scale, kv_scale;
};

// The group product of a (sequence, kv head) has G * qlen query columns; up
// to kMaxGroup the warp-MMA decode kernel serves them, beyond that the
// tensor-core kernel (query rows packed as token x head).
bool use_tc(int G, int qlen) { return static_cast<int64_t>(G) * qlen > pa::kMaxGroup; }

int check_decode(const DecodeArgs& a) {
  int rc = check_cache(a.cache, a.k_cache, a.v_cache);
  if (rc) return rc;
  if (a.num_seqs < 0 || a.num_q_heads <= 0 || a.max_blocks_per_seq <= 0) return PA_ERR_INVALID_ARG;
  if (a.q_dtype != PA_F16 && a.q_dtype != PA_BF16) return PA_ERR_UNSUPPORTED;
  if (a.cache->kv_dtype != PA_FP8_E4M3 && a.cache->kv_dtype != a.q_dtype) return PA_ERR_UNSUPPORTED;
  if (a.num_q_heads % a.cache->num_kv_heads) return PA_ERR_INVALID_ARG;
  if (a.qlen < 1) return PA_ERR_INVALID_ARG;
  const int G = a.num_q_heads / a.cache->num_kv_heads;
  if (G > pa::kTcMaxGroup) return PA_ERR_UNSUPPORTED;
  if (!std::isfinite(a.scale)) return PA_ERR_INVALID_ARG;
  // the tensor-core path takes the row max of the raw scores
  if (use_tc(G, a.qlen) && !(a.scale > 0.f)) return PA_ERR_INVALID_ARG;
  rc = check_kv_scale(a.cache->kv_dtype, a.kv_scale);
  if (rc) return rc;
  if (static_cast<int64_t>(a.max_blocks_per_seq) * a.cache->block_size > INT32_MAX) return PA_ERR_INVALID_ARG;
  if (a.num_seqs == 0) return PA_OK;
  if (!a.out || !a.q || !a.block_tables || !a.context_lens) return PA_ERR_INVALID_ARG;
  if (!aligned16(a.out) || !aligned16(a.q)) return PA_ERR_INVALID_ARG;
  return PA_OK;
}

pa::DecodeParams make_params(const DecodeArgs& a, int* err) {
  pa::DecodeParams p{};
  p.out = a.out;
  p.q = a.q;
  p.block_tables = a.block_tables;
  p.context_lens = a.context_lens;
  p.err = err;
  p.num_blocks = a.cache->num_blocks;
  p.S = a.num_seqs;
  p.Hq = a.num_q_heads;
  p.Hkv = a.cache->num_kv_heads;
  p.G = a.num_q_heads / a.cache->num_kv_heads;
  p.bs = a.cache->block_size;
  p.maxB = a.max_blocks_per_seq;
  p.qlen = a.qlen;
  p.q_dtype = a.q_dtype;
  p.partition_size = 0;
  p.Pmax = 1;
  p.parts_per_cta = 1;
  p.scale_log2 = static_cast<float>(static_cast<double>(a.scale) * 1.4426950408889634);
  p.kv_scale = a.cache->kv_dtype == PA_FP8_E4M3 ? a.kv_scale : 1.0f;
  return p;
}

cudaError_t launch_decode(const pa::DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv, int kv_dtype,
                          int head_dim, cudaStream_t st) {
  switch (kv_dtype) {
    case PA_F16: return pa::launch_decode_f16(p, tk, tv, head_dim, st);
    case PA_BF16: return pa::launch_decode_bf16(p, tk, tv, head_dim, st);
    default: return pa::launch_decode_fp8(p, tk, tv, head_dim, st);
  }
}

// Consecutive partitions one split CTA streams: enough that the grid holds
// about PA_SPLIT_CTAS_PER_SLOT CTAs per resident slot when every sequence has
// Pmax partitions, so launch and pipeline ramp costs are paid per run, not
// per partition.
#ifndef PA_SPLIT_CTAS_PER_SLOT
#define PA_SPLIT_CTAS_PER_SLOT 8
#endif
// The last partitions of every context run one per CTA, after all the longer
// runs: the launch then ends on short runs instead of a partial wave of long
// ones.
#ifndef PA_SPLIT_FRINGE
#define PA_SPLIT_FRINGE 8
#endif
std::atomic<int> g_sm_count[kMaxDevices];

int sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) dev = 0;
  int n = g_sm_count[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    g_sm_count[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

int parts_per_cta(int S, int Hkv, int Pmax) {
  const int64_t target = int64_t(PA_SPLIT_CTAS_PER_SLOT) * sm_count() * pa::kMinCtasPerSm;
  const int64_t total = int64_t(S) * Hkv * Pmax;
  int64_t ppc = (total + target - 1) / target;
  if (ppc < 1) ppc = 1;
  if (ppc > Pmax) ppc = Pmax;
  return static_cast<int>(ppc);
}

int64_t split_partitions(int32_t max_context_len, int32_t partition_size) {
  if (max_context_len <= 0) return 1;
  return (static_cast<int64_t>(max_context_len) + partition_size - 1) / partition_size;
}

// The new rows a fused call writes into the pool (pa_cache_and_decode).
struct CacheWrite {
  const void* key;
  const void* value;
  const int64_t* slot_mapping;
  void* k_cache;
  void* v_cache;
};

void set_cache_write(pa::DecodeParams& p, const CacheWrite* w) {
  if (!w) return;
  p.new_key = w->key;
  p.new_value = w->value;
  p.slot_mapping = w->slot_mapping;
  p.k_cache = w->k_cache;
  p.v_cache = w->v_cache;
}

// Consecutive partitions per run of the tensor-core kernel: about eight
// work items per SM when every sequence has Pmax partitions (its CTAs are
// persistent, so more items only cost per-item pipeline ramps).
int tc_parts_per_run(int64_t units, int Pmax) {
  const int64_t target = int64_t(8) * sm_count();
  int64_t ppc = (units * Pmax + target - 1) / target;
  if (ppc < 1) ppc = 1;
  if (ppc > Pmax) ppc = Pmax;
  return static_cast<int>(ppc);
}

// Attention of a.qlen new tokens per sequence on the tensor cores (chunked
// prefill, and multi-token decode with a wide query group): causal among
// the new tokens; split into runs of partitions merged by log-sum-exp when
// partition_size > 0.  Arguments are checked by the caller.
int attn_tc_impl(const DecodeArgs& a, int32_t max_context_len, int32_t partition_size, void* workspace,
                 size_t workspace_bytes, pa_stream_t stream, const CacheWrite* write) {
  const pa_cache_desc* cache = a.cache;
  const int S = a.num_seqs, C = a.qlen, Hq = a.num_q_heads, Hkv = cache->num_kv_heads, D = cache->head_dim;
  const int G = Hq / Hkv;
  if (S == 0) return PA_OK;
  const int T = std::min(C, pa::kTcRows / G);  // new tokens per query tile
  const int64_t n_qt = (C + T - 1) / T;
  const int fp8 = cache->kv_dtype == PA_FP8_E4M3 ? 1 : 0;
  int64_t Pmax = 1, ppc = 1, R = 1;
  if (partition_size > 0) {
    Pmax = split_partitions(max_context_len, partition_size);
    if (Pmax > INT32_MAX) return PA_ERR_INVALID_ARG;
    ppc = tc_parts_per_run(int64_t(S) * Hkv * n_qt, static_cast<int>(Pmax));
    R = (Pmax + ppc - 1) / ppc;
  }
  const int64_t total = int64_t(S) * Hkv * n_qt * R;
  const int64_t rows = int64_t(S) * C;
  if (total > INT32_MAX || rows * Hq > INT32_MAX || rows > UINT32_MAX) return PA_ERR_INVALID_ARG;
  if (partition_size > 0) {
    const size_t need = pa_decode_multi_split_workspace_size(S, C, Hq, D, max_context_len, partition_size);
    if (!workspace || workspace_bytes < need || !aligned16(workspace)) return PA_ERR_WORKSPACE;
  }
  int* err = device_error_ptr();
  if (!err) return PA_ERR_CUDA;
  int rc;
  CUtensorMap tq, tk, tv;
  if ((rc = make_cache_tensor_map(&tk, a.k_cache, cache)) || (rc = make_cache_tensor_map(&tv, a.v_cache, cache)))
    return rc;
  EncodeTiledFn fn = encode_fn();
  if (!fn) return PA_ERR_CUDA;
  // q as {channels, heads, tokens}; box = 64 channels x the G heads of a kv
  // head x T tokens, landing as rows token * G + head of 128 bytes
  const cuuint64_t dims[3] = {cuuint64_t(D), cuuint64_t(Hq), cuuint64_t(rows)};
  const cuuint64_t strides[2] = {cuuint64_t(D) * 2, cuuint64_t(Hq) * D * 2};
  const cuuint32_t box[3] = {64, cuuint32_t(G), cuuint32_t(T)};
  const cuuint32_t estr[3] = {1, 1, 1};
  if (fn(&tq, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<void*>(a.q), dims, strides, box, estr,
         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return PA_ERR_CUDA;
  pa::TcParams p{};
  p.out = a.out;
  p.block_tables = a.block_tables;
  p.context_lens = a.context_lens;
  p.err = err;
  p.num_blocks = cache->num_blocks;
  p.S = S;
  p.C = C;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.G = G;
  p.bs = cache->block_size;
  p.maxB = a.max_blocks_per_seq;
  p.D = D;
  p.T = T;
  p.n_qt = static_cast<int>(n_qt);
  p.R = static_cast<int>(R);
  p.partition_size = partition_size > 0 ? partition_size : 0;
  p.Pmax = static_cast<int>(Pmax);
  p.ppc = static_cast<int>(ppc);
  p.nqb = 2;
  p.nslot = pa::tc_ring_slots(D, fp8, p.nqb);
  p.rank_seqs = 1;
  p.out_bf16 = a.q_dtype == PA_BF16 ? 1 : 0;
  // E4M3 caches are widened to f16 (exact), so the MMA runs in f16; bf16 q
  // is then scaled per row by a power of two and rounded to f16 in the kernel
  p.fp8 = fp8;
  p.bf16 = fp8 ? 0 : p.out_bf16;
  p.q_scale_rows = fp8 && p.out_bf16 ? 1 : 0;
  p.total = static_cast<int>(total);
  const double kvs = fp8 ? static_cast<double>(a.kv_scale) : 1.0;
  p.scale_log2 = static_cast<float>(static_cast<double>(a.scale) * kvs * 1.4426950408889634);
  p.vscale = static_cast<float>(kvs);
  if (partition_size > 0) {
    // partial outputs first (16-byte aligned rows for the merge), then (m, l)
    p.ws_o = static_cast<float*>(workspace);
    p.ws_ml = p.ws_o + static_cast<size_t>(rows) * Hq * Pmax * D;
  }
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  if (write) {
    // the new rows go to the pool first (the fused form of the warp-MMA path
    // writes them from inside its decode kernel)
    pa::CacheParams cp{};
    cp.key = write->key;
    cp.value = write->value;
    cp.k_cache = write->k_cache;
    cp.v_cache = write->v_cache;
    cp.slot_mapping = write->slot_mapping;
    cp.err = err;
    cp.num_blocks = cache->num_blocks;
    cp.T = static_cast<int>(rows);
    cp.Hkv = Hkv;
    cp.D = D;
    cp.bs = cache->block_size;
    cp.in_dtype = a.q_dtype;
    cp.cache_dtype = cache->kv_dtype;
    cp.kv_scale = fp8 ? a.kv_scale : 1.0f;
    e = pa::launch_reshape_and_cache(cp, st);
  }
  if (e == cudaSuccess) e = pa::launch_attn_tc(p, tq, tk, tv, st);
  if (e == cudaSuccess && partition_size > 0) {
    pa::DecodeParams mp = make_params(a, err);
    mp.partition_size = partition_size;
    mp.Pmax = p.Pmax;
    mp.parts_per_cta = p.ppc;
    mp.ws_o = p.ws_o;
    mp.ws_ml = p.ws_ml;
    e = pa::launch_lse_merge(mp, D, st);
  }
  return finish(e, st);
}

// Chunked prefill with 16-bit caches through a persistent kernel: work items
// (sequence, pair of query heads of one kv head, 128 new tokens) for an even
// group size and head_dim 64 or 128 (pa_prefill_pair.cu), else (sequence,
// query head, 128 new tokens) with head_dim 128 (pa_prefill.cu).  Arguments
// are checked by the caller.
int prefill_per_head_impl(const DecodeArgs& a, pa_stream_t stream, float vscale = 1.f, bool cluster = true) {
  const pa_cache_desc* cache = a.cache;
  const int64_t rows = static_cast<int64_t>(a.num_seqs) * a.qlen;
  const int64_t nqt = (a.qlen + pa::kPfRows - 1) / pa::kPfRows;
  if (rows > UINT32_MAX || nqt * a.num_q_heads * a.num_seqs > INT32_MAX) return PA_ERR_INVALID_ARG;
  int* err = device_error_ptr();
  if (!err) return PA_ERR_CUDA;
  int rc;
  CUtensorMap tq, tk, tv;
  if ((rc = make_cache_tensor_map(&tk, a.k_cache, cache)) || (rc = make_cache_tensor_map(&tv, a.v_cache, cache)))
    return rc;
  EncodeTiledFn fn = encode_fn();
  if (!fn) return PA_ERR_CUDA;
  // q as {D channels, heads, tokens}; box = 64 channels x 1 head x 128 tokens
  const int D = cache->head_dim;
  const cuuint64_t dims[3] = {cuuint64_t(D), cuuint64_t(a.num_q_heads), cuuint64_t(rows)};
  const cuuint64_t strides[2] = {cuuint64_t(D) * 2, cuuint64_t(a.num_q_heads) * D * 2};
  const cuuint32_t box[3] = {64, 1, cuuint32_t(pa::kPfRows)};
  const cuuint32_t estr[3] = {1, 1, 1};
  if (fn(&tq, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<void*>(a.q), dims, strides, box, estr,
         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return PA_ERR_CUDA;
  pa::PrefillParams p{};
  p.out = a.out;
  p.block_tables = a.block_tables;
  p.context_lens = a.context_lens;
  p.err = err;
  p.num_blocks = cache->num_blocks;
  p.S = a.num_seqs;
  p.C = a.qlen;
  p.Hq = a.num_q_heads;
  p.Hkv = cache->num_kv_heads;
  p.G = a.num_q_heads / cache->num_kv_heads;
  p.bs = cache->block_size;
  p.maxB = a.max_blocks_per_seq;
  p.D = D;
  p.bf16 = a.q_dtype == PA_BF16 ? 1 : 0;
  p.scale_log2 = static_cast<float>(static_cast<double>(a.scale) * 1.4426950408889634);
  p.vscale = vscale;
  p.cluster = cluster ? 1 : 0;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // an even group: two query heads per work item share each K/V tile
  const bool pair = p.G % 2 == 0;
  return finish(pair ? pa::launch_prefill_pair(p, tq, tk, tv, st) : pa::launch_prefill(p, tq, tk, tv, st), st);
}

// Bytes of the E4M3 prefill workspace: the widened K and V blocks (2-byte
// elements) of every block-table entry, then the compact table.
int64_t prefill_fp8_workspace_bytes(int64_t nslot, const pa_cache_desc* c) {
  const int64_t blk = static_cast<int64_t>(c->num_kv_heads) * c->block_size * c->head_dim;  // elements
  return nslot * blk * 2 * 2 + nslot * 4;
}

// Prefill over E4M3 caches with the caller's workspace: the batch's blocks are
// widened exactly to the query's 16-bit type into it (a compact pool with its
// own block table), then the 16-bit prefill kernels run on it with the
// per-tensor scale on the scores and the output.  Arguments are checked by
// the caller.
int prefill_fp8_widened_impl(const DecodeArgs& a, void* workspace, pa_stream_t stream) {
  const pa_cache_desc* cache = a.cache;
  const int64_t nslot = static_cast<int64_t>(a.num_seqs) * a.max_blocks_per_seq;
  if (nslot > INT32_MAX) return PA_ERR_INVALID_ARG;
  int* err = device_error_ptr();
  if (!err) return PA_ERR_CUDA;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const size_t kv_bytes = static_cast<size_t>(nslot) * cache->num_kv_heads * cache->block_size * cache->head_dim * 2;
  pa::WidenParams w{};
  w.k_src = static_cast<const uint8_t*>(a.k_cache);
  w.v_src = static_cast<const uint8_t*>(a.v_cache);
  w.k_dst = static_cast<uint16_t*>(workspace);
  w.v_dst = reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(workspace) + kv_bytes);
  w.tab = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(workspace) + 2 * kv_bytes);
  w.block_tables = a.block_tables;
  w.context_lens = a.context_lens;
  w.err = err;
  w.num_blocks = cache->num_blocks;
  w.S = a.num_seqs;
  w.maxB = a.max_blocks_per_seq;
  w.Hkv = cache->num_kv_heads;
  w.bs = cache->block_size;
  w.D = cache->head_dim;
  w.bf16 = a.q_dtype == PA_BF16 ? 1 : 0;
  const cudaError_t e = pa::launch_widen_kv(w, st);
  if (e != cudaSuccess) return finish(e, st);
  pa_cache_desc wide = *cache;
  wide.kv_dtype = a.q_dtype;
  wide.num_blocks = nslot;
  DecodeArgs b = a;
  b.k_cache = w.k_dst;
  b.v_cache = w.v_dst;
  b.cache = &wide;
  b.block_tables = w.tab;
  b.scale = a.scale * a.kv_scale;
  // the widened blocks run without the cluster form, which measured 1 % slower here
  return prefill_per_head_impl(b, stream, a.kv_scale, false);
}

}  // namespace

namespace pa {
// pa_selftest.cu: one kernel whose bounded wait runs out
cudaError_t launch_wait_timeout_selftest(int* err, cudaStream_t st);
cudaError_t launch_l2_read_plain(const void* buf, size_t bytes, int iters, void* sink, int nsm, cudaStream_t st);
cudaError_t launch_l2_read_tma(const CUtensorMap& map, int nrows, int iters, void* sink, int* err, int nsm,
                               cudaStream_t st);
}  // namespace pa

extern "C" {

int pa_reshape_and_cache(const void* key, const void* value, int32_t in_dtype, int32_t num_tokens, void* k_cache,
                         void* v_cache, const pa_cache_desc* cache, const int64_t* slot_mapping, float kv_scale,
                         pa_stream_t stream) {
  int rc = check_cache(cache, k_cache, v_cache);
  if (rc) return rc;
  if (in_dtype != PA_F16 && in_dtype != PA_BF16) return PA_ERR_UNSUPPORTED;
  if (cache->kv_dtype != PA_FP8_E4M3 && cache->kv_dtype != in_dtype) return PA_ERR_UNSUPPORTED;
  if (num_tokens < 0) return PA_ERR_INVALID_ARG;
  rc = check_kv_scale(cache->kv_dtype, kv_scale);
  if (rc) return rc;
  if (num_tokens == 0) return PA_OK;
  if (!key || !value || !slot_mapping || !aligned16(key) || !aligned16(value)) return PA_ERR_INVALID_ARG;
  int* err = device_error_ptr();
  if (!err) return PA_ERR_CUDA;
  pa::CacheParams p{};
  p.key = key;
  p.value = value;
  p.k_cache = k_cache;
  p.v_cache = v_cache;
  p.slot_mapping = slot_mapping;
  p.err = err;
  p.num_blocks = cache->num_blocks;
  p.T = num_tokens;
  p.Hkv = cache->num_kv_heads;
  p.D = cache->head_dim;
  p.bs = cache->block_size;
  p.in_dtype = in_dtype;
  p.cache_dtype = cache->kv_dtype;
  p.kv_scale = cache->kv_dtype == PA_FP8_E4M3 ? kv_scale : 1.0f;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  return finish(pa::launch_reshape_and_cache(p, st), st);
}

int pa_decode(void* out, const void* q, int32_t q_dtype, int32_t num_seqs, int32_t num_q_heads, const void* k_cache,
              const void* v_cache, const pa_cache_desc* cache, const int32_t* block_tables,
              int32_t max_blocks_per_seq, const int32_t* context_lens, float scale, float kv_scale,
              pa_stream_t stream) {
  const DecodeArgs a{out, q, q_dtype, num_seqs, num_q_heads, 1, k_cache, v_cache, cache, block_tables,
                     max_blocks_per_seq, context_lens, scale, kv_scale};
  int rc = check_decode(a);
  if (rc || num_seqs == 0) return rc;
  if (use_tc(num_q_heads / cache->num_kv_heads, 1)) return attn_tc_impl(a, 0, 0, nullptr, 0, stream, nullptr);
  if (static_cast<int64_t>(num_seqs) * cache->num_kv_heads > INT32_MAX) return PA_ERR_INVALID_ARG;
  int* err = device_error_ptr();
  if (!err) return PA_ERR_CUDA;
  CUtensorMap tk, tv;
  if ((rc = make_cache_tensor_map(&tk, k_cache, cache)) || (rc = make_cache_tensor_map(&tv, v_cache, cache)))
    return rc;
  const pa::DecodeParams p = make_params(a, err);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  return finish(launch_decode(p, tk, tv, cache->kv_dtype, cache->head_dim, st), st);
}

int pa_decode_multi(void* out, const void* q, int32_t q_dtype, int32_t num_seqs, int32_t num_q_tokens,
                    int32_t num_q_heads, const void* k_cache, const void* v_cache, const pa_cache_desc* cache,
                    const int32_t* block_tables, int32_t max_blocks_per_seq, const int32_t* context_lens,
                    float scale, float kv_scale, pa_stream_t stream) {
  const DecodeArgs a{out, q, q_dtype, num_seqs, num_q_heads, num_q_tokens, k_cache, v_cache, cache, block_tables,
                     max_blocks_per_seq, context_lens, scale, kv_scale};
  int rc = check_decode(a);
  if (rc || num_seqs == 0) return rc;
  if (use_tc(num_q_heads / cache->num_kv_heads, num_q_tokens))
    return attn_tc_impl(a, 0, 0, nullptr, 0, stream, nullptr);
  if (static_cast<int64_t>(num_seqs) * cache->num_kv_heads > INT32_MAX) return PA_ERR_INVALID_ARG;
  int* err = device_error_ptr();
  if (!err) return PA_ERR_CUDA;
  CUtensorMap tk, tv;
  if ((rc = make_cache_tensor_map(&tk, k_cache, cache)) || (rc = make_cache_tensor_map(&tv, v_cache, cache)))
    return rc;
  const pa::DecodeParams p = make_params(a, err);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  return finish(launch_decode(p, tk, tv, cache->kv_dtype, cache->head_dim, st), st);
}

size_t pa_prefill_workspace_size(int32_t num_seqs, int32_t max_blocks_per_seq, const pa_cache_desc* cache) {
  if (!cache || num_seqs < 0 || max_blocks_per_seq <= 0 || cache->kv_dtype != PA_FP8_E4M3 ||
      cache->num_kv_heads <= 0 || cache->block_size <= 0 || cache->head_dim <= 0)
    return 0;
  return static_cast<size_t>(
      prefill_fp8_workspace_bytes(static_cast<int64_t>(num_seqs) * max_blocks_per_seq, cache));
}

int pa_prefill(void* out, const void* q, int32_t q_dtype, int32_t num_seqs, int32_t num_q_tokens,
               int32_t num_q_heads, const void* k_cache, const void* v_cache, const pa_cache_desc* cache,
               const int32_t* block_tables, int32_t max_blocks_per_seq, const int32_t* context_lens, float scale,
               float kv_scale, void* workspace, size_t workspace_bytes, pa_stream_t stream) {
  int rc = check_cache(cache, k_cache, v_cache);
  if (rc) return rc;
  if (num_seqs < 0 || num_q_tokens < 1 || num_q_heads <= 0 || max_blocks_per_seq <= 0) return PA_ERR_INVALID_ARG;
  if (q_dtype != PA_F16 && q_dtype != PA_BF16) return PA_ERR_UNSUPPORTED;
  if (cache->kv_dtype != q_dtype && cache->kv_dtype != PA_FP8_E4M3) return PA_ERR_UNSUPPORTED;
  if (num_q_heads % cache->num_kv_heads) return PA_ERR_INVALID_ARG;
  if (num_q_heads / cache->num_kv_heads > pa::kTcMaxGroup) return PA_ERR_UNSUPPORTED;
  if (!std::isfinite(scale) || !(scale > 0.f)) return PA_ERR_INVALID_ARG;
  rc = check_kv_scale(cache->kv_dtype, kv_scale);
  if (rc) return rc;
  if (static_cast<int64_t>(max_blocks_per_seq) * cache->block_size > INT32_MAX) return PA_ERR_INVALID_ARG;
  const bool fp8 = cache->kv_dtype == PA_FP8_E4M3;
  if (fp8 && workspace &&
      (!aligned16(workspace) ||
       workspace_bytes < pa_prefill_workspace_size(num_seqs, max_blocks_per_seq, cache)))
    return PA_ERR_WORKSPACE;
  if (num_seqs == 0) return PA_OK;
  if (!out || !q || !block_tables || !context_lens || !aligned16(out) || !aligned16(q)) return PA_ERR_INVALID_ARG;
  const DecodeArgs a{out, q, q_dtype, num_seqs, num_q_heads, num_q_tokens, k_cache, v_cache, cache, block_tables,
                     max_blocks_per_seq, context_lens, scale, kv_scale};
  // the head-pair kernel for an even group (head_dim 64 or 128), the one-head
  // kernel for an odd group with head_dim 128; E4M3 caches reach them through
  // the widening pass into the caller's workspace
  const int G = num_q_heads / cache->num_kv_heads;
  if (G % 2 == 0 || cache->head_dim == 128) {
    if (!fp8) return prefill_per_head_impl(a, stream);
    if (workspace) return prefill_fp8_widened_impl(a, workspace, stream);
  }
  // otherwise the packed-group kernel (which widens E4M3 tiles in shared memory)
  return attn_tc_impl(a, 0, 0, nullptr, 0, stream, nullptr);
}

size_t pa_decode_multi_split_workspace_size(int32_t num_seqs, int32_t num_q_tokens, int32_t num_q_heads,
                                            int32_t head_dim, int32_t max_context_len, int32_t partition_size) {
  if (num_seqs < 0 || num_q_tokens < 1 || num_q_heads <= 0 || head_dim <= 0 || max_context_len < 0 ||
      partition_size <= 0)
    return 0;
  const int64_t np = split_partitions(max_context_len, partition_size);
  return static_cast<size_t>(num_seqs) * num_q_tokens * num_q_heads * np * (head_dim + 2) * sizeof(float);
}

size_t pa_decode_split_workspace_size(int32_t num_seqs, int32_t num_q_heads, int32_t head_dim,
                                      int32_t max_context_len, int32_t partition_size) {
  return pa_decode_multi_split_workspace_size(num_seqs, 1, num_q_heads, head_dim, max_context_len, partition_size);
}

}  // extern "C"

namespace {

// Split decode of one or several new tokens per sequence: the partition
// kernel, then the log-sum-exp merge of the runs, on one stream.
int decode_split_impl(const DecodeArgs& a, int32_t max_context_len, int32_t partition_size, void* workspace,
                      size_t workspace_bytes, pa_stream_t stream, const CacheWrite* write = nullptr) {
  int rc = check_decode(a);
  if (rc) return rc;
  if (partition_size <= 0 || partition_size % pa::kTileTokens || max_context_len < 0) return PA_ERR_INVALID_ARG;
  if (a.num_seqs == 0) return PA_OK;
  if (use_tc(a.num_q_heads / a.cache->num_kv_heads, a.qlen))
    return attn_tc_impl(a, max_context_len, partition_size, workspace, workspace_bytes, stream, write);
  const pa_cache_desc* cache = a.cache;
  const int64_t np = split_partitions(max_context_len, partition_size);
  if (static_cast<int64_t>(a.num_seqs) * cache->num_kv_heads * np > INT32_MAX) return PA_ERR_INVALID_ARG;
  if (static_cast<int64_t>(a.num_seqs) * a.qlen * a.num_q_heads > INT32_MAX) return PA_ERR_INVALID_ARG;
  const size_t need = pa_decode_multi_split_workspace_size(a.num_seqs, a.qlen, a.num_q_heads, cache->head_dim,
                                                           max_context_len, partition_size);
  if (!workspace || workspace_bytes < need || !aligned16(workspace)) return PA_ERR_WORKSPACE;
  int* err = device_error_ptr();
  if (!err) return PA_ERR_CUDA;
  CUtensorMap tk, tv;
  if ((rc = make_cache_tensor_map(&tk, a.k_cache, cache)) || (rc = make_cache_tensor_map(&tv, a.v_cache, cache)))
    return rc;
  pa::DecodeParams p = make_params(a, err);
  set_cache_write(p, write);
  p.partition_size = partition_size;
  p.Pmax = static_cast<int>(np);
  p.parts_per_cta = parts_per_cta(a.num_seqs, cache->num_kv_heads, p.Pmax);
  p.fringe = p.parts_per_cta > 1 ? static_cast<int>(std::min<int64_t>(PA_SPLIT_FRINGE, p.Pmax)) : 0;
  const size_t rows = static_cast<size_t>(a.num_seqs) * a.qlen * a.num_q_heads * np;
  // partial outputs first: their rows of head_dim floats keep the 16-byte
  // alignment of the workspace for the merge's vector loads
  p.ws_o = static_cast<float*>(workspace);
  p.ws_ml = p.ws_o + rows * cache->head_dim;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = launch_decode(p, tk, tv, cache->kv_dtype, cache->head_dim, st);
  if (e == cudaSuccess) e = pa::launch_lse_merge(p, cache->head_dim, st);
  return finish(e, st);
}

}  // namespace

extern "C" {

int pa_decode_split(void* out, const void* q, int32_t q_dtype, int32_t num_seqs, int32_t num_q_heads,
                    const void* k_cache, const void* v_cache, const pa_cache_desc* cache,
                    const int32_t* block_tables, int32_t max_blocks_per_seq, const int32_t* context_lens,
                    float scale, float kv_scale, int32_t max_context_len, int32_t partition_size, void* workspace,
                    size_t workspace_bytes, pa_stream_t stream) {
  const DecodeArgs a{out, q, q_dtype, num_seqs, num_q_heads, 1, k_cache, v_cache, cache, block_tables,
                     max_blocks_per_seq, context_lens, scale, kv_scale};
  return decode_split_impl(a, max_context_len, partition_size, workspace, workspace_bytes, stream);
}

int pa_cache_and_decode(void* out, const void* q, int32_t q_dtype, int32_t num_seqs, int32_t num_q_tokens,
                        int32_t num_q_heads, const void* key, const void* value, const int64_t* slot_mapping,
                        void* k_cache, void* v_cache, const pa_cache_desc* cache, const int32_t* block_tables,
                        int32_t max_blocks_per_seq, const int32_t* context_lens, float scale, float kv_scale,
                        int32_t max_context_len, int32_t partition_size, void* workspace, size_t workspace_bytes,
                        pa_stream_t stream) {
  const DecodeArgs a{out, q, q_dtype, num_seqs, num_q_heads, num_q_tokens, k_cache, v_cache, cache, block_tables,
                     max_blocks_per_seq, context_lens, scale, kv_scale};
  int rc = check_decode(a);
  if (rc) return rc;
  if (partition_size < 0) return PA_ERR_INVALID_ARG;
  if (num_seqs == 0) return PA_OK;
  if (!key || !value || !slot_mapping || !aligned16(key) || !aligned16(value)) return PA_ERR_INVALID_ARG;
  if (static_cast<int64_t>(num_seqs) * num_q_tokens > INT32_MAX) return PA_ERR_INVALID_ARG;
  if (check_mode()) {
    // a fused write into a block that another sequence's table also names
    // (copy-on-write skipped) would race with that sequence's tile loads
    int* err = device_error_ptr();
    if (!err) return PA_ERR_CUDA;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (pa::launch_shared_slot_check(slot_mapping, block_tables, context_lens, num_seqs, num_q_tokens,
                                     max_blocks_per_seq, cache->block_size, cache->num_blocks, err,
                                     st) != cudaSuccess)
      return PA_ERR_CUDA;
  }
  const CacheWrite w{key, value, slot_mapping, k_cache, v_cache};
  if (partition_size > 0)
    return decode_split_impl(a, max_context_len, partition_size, workspace, workspace_bytes, stream, &w);
  if (use_tc(num_q_heads / cache->num_kv_heads, num_q_tokens))
    return attn_tc_impl(a, 0, 0, nullptr, 0, stream, &w);
  if (static_cast<int64_t>(num_seqs) * cache->num_kv_heads > INT32_MAX) return PA_ERR_INVALID_ARG;
  int* err = device_error_ptr();
  if (!err) return PA_ERR_CUDA;
  CUtensorMap tk, tv;
  if ((rc = make_cache_tensor_map(&tk, k_cache, cache)) || (rc = make_cache_tensor_map(&tv, v_cache, cache)))
    return rc;
  pa::DecodeParams p = make_params(a, err);
  set_cache_write(p, &w);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  return finish(launch_decode(p, tk, tv, cache->kv_dtype, cache->head_dim, st), st);
}

int pa_decode_multi_split(void* out, const void* q, int32_t q_dtype, int32_t num_seqs, int32_t num_q_tokens,
                          int32_t num_q_heads, const void* k_cache, const void* v_cache, const pa_cache_desc* cache,
                          const int32_t* block_tables, int32_t max_blocks_per_seq, const int32_t* context_lens,
                          float scale, float kv_scale, int32_t max_context_len, int32_t partition_size,
                          void* workspace, size_t workspace_bytes, pa_stream_t stream) {
  const DecodeArgs a{out, q, q_dtype, num_seqs, num_q_heads, num_q_tokens, k_cache, v_cache, cache, block_tables,
                     max_blocks_per_seq, context_lens, scale, kv_scale};
  return decode_split_impl(a, max_context_len, partition_size, workspace, workspace_bytes, stream);
}

// Device address through which kernels may touch `p`: device or managed
// memory as is, pinned host memory through its mapping; false for anything
// else (for example pageable host memory), so nothing is launched on it.
static bool device_view(const void* p, void** dev) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) {
    *dev = const_cast<void*>(p);
    return true;
  }
  if (a.type == cudaMemoryTypeHost && a.devicePointer) {
    *dev = a.devicePointer;
    return true;
  }
  return false;
}

static int block_op(int op, void* buf, void* k_cache, void* v_cache, const pa_cache_desc* cache, const int64_t* ids,
                    int32_t n, pa_stream_t stream) {
  int rc = check_cache(cache, k_cache, v_cache);
  if (rc) return rc;
  if (n < 0) return PA_ERR_INVALID_ARG;
  if (n == 0) return PA_OK;
  if (!ids || (op != 0 && (!buf || !aligned16(buf)))) return PA_ERR_INVALID_ARG;
  void* ids_dev = nullptr;
  if (!device_view(ids, &ids_dev)) return PA_ERR_INVALID_ARG;
  ids = static_cast<const int64_t*>(ids_dev);
  if (op != 0) {
    void* buf_dev = nullptr;
    if (!device_view(buf, &buf_dev)) return PA_ERR_INVALID_ARG;
    buf = buf_dev;
  }
  int* err = device_error_ptr();
  if (!err) return PA_ERR_CUDA;
  const int64_t block_bytes = static_cast<int64_t>(cache->num_kv_heads) * cache->block_size * cache->head_dim *
                              elem_bytes(cache->kv_dtype);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  return finish(pa::launch_block_op(op, buf, k_cache, v_cache, ids, n, block_bytes, cache->num_blocks, err, st), st);
}

int pa_copy_blocks(void* k_cache, void* v_cache, const pa_cache_desc* cache, const int64_t* block_pairs,
                   int32_t num_pairs, pa_stream_t stream) {
  return block_op(0, nullptr, k_cache, v_cache, cache, block_pairs, num_pairs, stream);
}

int pa_gather_blocks(void* dst, const void* k_cache, const void* v_cache, const pa_cache_desc* cache,
                     const int64_t* block_ids, int32_t num, pa_stream_t stream) {
  return block_op(1, dst, const_cast<void*>(k_cache), const_cast<void*>(v_cache), cache, block_ids, num, stream);
}

int pa_scatter_blocks(void* k_cache, void* v_cache, const pa_cache_desc* cache, const void* src,
                      const int64_t* block_ids, int32_t num, pa_stream_t stream) {
  return block_op(2, const_cast<void*>(src), k_cache, v_cache, cache, block_ids, num, stream);
}

const char* pa_status_string(int status) {
  switch (status) {
    case PA_OK: return "ok";
    case PA_ERR_INVALID_ARG: return "invalid argument";
    case PA_ERR_UNSUPPORTED: return "unsupported configuration";
    case PA_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case PA_ERR_CUDA: return "CUDA error";
    case PA_ERR_BAD_INDEX: return "out-of-range index seen by a kernel";
    case PA_ERR_TIMEOUT: return "kernel pipeline wait timed out";
    case PA_ERR_OUT_OF_BLOCKS: return "not enough free blocks";
    case PA_ERR_NOT_FOUND: return "unknown or duplicate sequence id";
    default: return "unknown status";
  }
}

int pa_set_check_mode(int enable) {
  const int prev = check_mode() ? 1 : 0;
  g_check.store(enable ? 1 : 0);
  return prev;
}

int pa_get_device_error(void) { return read_and_clear_error(nullptr, true); }

int pa_selftest_wait_timeout(pa_stream_t stream) {
  int* err = device_error_ptr();
  if (!err) return PA_ERR_CUDA;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  return pa::launch_wait_timeout_selftest(err, st) == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

int pa_probe_l2_read(const void* buf, size_t bytes, int32_t mode, int32_t iters, void* sink,
                     unsigned long long* bytes_read, pa_stream_t stream) {
  if (!buf || !sink || !bytes_read || iters <= 0 || !aligned16(buf) || (mode != 0 && mode != 1))
    return PA_ERR_INVALID_ARG;
  if (mode == 0 && (bytes < 16 || bytes % 16)) return PA_ERR_INVALID_ARG;
  if (mode == 1 && (bytes < 2048 || bytes % 2048 || bytes / 128 > INT32_MAX)) return PA_ERR_INVALID_ARG;
  int* err = device_error_ptr();
  if (!err) return PA_ERR_CUDA;
  const int nsm = sm_count();
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (mode == 0) {
    *bytes_read = static_cast<unsigned long long>(bytes) * static_cast<unsigned long long>(iters);
    return pa::launch_l2_read_plain(buf, bytes, iters, sink, nsm, st) == cudaSuccess ? PA_OK : PA_ERR_CUDA;
  }
  // rows of 128 bytes, boxes of 16 rows with the 128-byte swizzle
  EncodeTiledFn fn = encode_fn();
  if (!fn) return PA_ERR_CUDA;
  CUtensorMap map;
  const cuuint64_t dims[2] = {64, cuuint64_t(bytes / 128)};
  const cuuint64_t strides[1] = {128};
  const cuuint32_t box[2] = {64, 16};
  const cuuint32_t estr[2] = {1, 1};
  if (fn(&map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void*>(buf), dims, strides, box, estr,
         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return PA_ERR_CUDA;
  *bytes_read = static_cast<unsigned long long>(nsm) * static_cast<unsigned long long>(iters) * 32768ull;
  return pa::launch_l2_read_tma(map, static_cast<int>(bytes / 128), iters, sink, err, nsm, st) == cudaSuccess
             ? PA_OK
             : PA_ERR_CUDA;
}

int pa_version(void) { return 100; }

}  // extern "C"
