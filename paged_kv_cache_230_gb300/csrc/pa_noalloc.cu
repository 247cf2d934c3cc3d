// pa_decode_split_noalloc: split-context decode whose partial results live in
// a scratch array compiled into the library, for callers that cannot
// allocate device memory when they call us.
//
// Who needs it: a serving process typically reserves almost all of HBM for
// its KV-cache pool at start-up and then forbids (or simply cannot satisfy)
// further device allocations; host frameworks that embed this library as a
// plug-in often own every device allocation themselves.  cudaMalloc in such a
// process fails or has to synchronise the device, so this entry point takes
// no workspace argument and allocates nothing.
//
// The scratch is a file-scope __device__ array of kScratchBytes.  Every GPU
// that loads this part of the library keeps it until the process exits.  Host
// code may not use the array's name as a device address, so the device
// address is looked up (cudaGetSymbolAddress, with that device current) by
// the first call made on a device, and again only if the device's context
// has changed since (a context torn down and created anew may load the
// module at another address); make that first call before any stream
// capture.  All calls on a device share the array: calls whose kernels may
// overlap on the GPU (different streams without ordering) race on it.
// Nothing in it needs to start at zero: every partial result the merge reads
// is written earlier by the same call.
#include <mutex>

#include "pagedattn.h"
#include "pa_internal.h"

namespace {

constexpr size_t kScratchBytes = size_t(32) << 20;  // 32 MiB
__device__ __align__(256) unsigned char g_split_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
struct ScratchSlot {
  CUcontext ctx;  // context the address was looked up in
  void* ptr;      // device address of g_split_scratch there
};
ScratchSlot g_scratch[kMaxDevices];
std::mutex g_scratch_mu;

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);

CtxGetCurrentFn ctx_get_current() {
  static CtxGetCurrentFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &ptr, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(ptr);
  });
  return fn;
}

// Device address of the scratch array in the current device's context.
int scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PA_ERR_CUDA;
  CtxGetCurrentFn get_ctx = ctx_get_current();
  if (!get_ctx) return PA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  CUcontext ctx = nullptr;
  if (get_ctx(&ctx) != CUDA_SUCCESS) return PA_ERR_CUDA;
  ScratchSlot& slot = g_scratch[dev];
  if (!slot.ptr || !ctx || ctx != slot.ctx) {
    // the lookup also makes the runtime bind the device's primary context
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_split_scratch) != cudaSuccess || !ptr) return PA_ERR_CUDA;
    if (get_ctx(&ctx) != CUDA_SUCCESS || !ctx) return PA_ERR_CUDA;
    slot.ctx = ctx;
    slot.ptr = ptr;
  }
  *out = slot.ptr;
  return PA_OK;
}

}  // namespace

extern "C" {

// Arguments, results and errors are those of pa_decode_split given a
// kScratchBytes workspace: argument errors first, then PA_ERR_WORKSPACE for
// a batch whose partials need more than the scratch holds; an empty batch
// launches nothing and returns PA_OK.
PA_API int pa_decode_split_noalloc(void* out, const void* q, int32_t q_dtype, int32_t num_seqs,
                                   int32_t num_q_heads, const void* k_cache, const void* v_cache,
                                   const pa_cache_desc* cache, const int32_t* block_tables,
                                   int32_t max_blocks_per_seq, const int32_t* context_lens, float scale,
                                   float kv_scale, int32_t max_context_len, int32_t partition_size,
                                   pa_stream_t stream) {
  void* scratch = nullptr;
  const int rc = scratch_for_current_device(&scratch);
  if (rc) return rc;
  return pa_decode_split(out, q, q_dtype, num_seqs, num_q_heads, k_cache, v_cache, cache, block_tables,
                         max_blocks_per_seq, context_lens, scale, kv_scale, max_context_len, partition_size,
                         scratch, kScratchBytes, stream);
}

}  // extern "C"
