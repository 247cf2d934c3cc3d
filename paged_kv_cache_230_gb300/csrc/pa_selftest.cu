// Self-test of the pipelines' bounded waits.  One thread waits on an
// mbarrier that nothing arrives at, through the same wait helper the decode
// and prefill pipelines use.  The helper gives up after about one second;
// the kernel then records PA_DEVERR_TIMEOUT in the device error word and
// returns, so the context stays usable and the host learns of the failure
// from the error word, as it would from a pipeline that lost a load.
#include "pa_internal.h"
#include "pa_ptx.cuh"
#include "pagedattn.h"

namespace pa {

namespace {

__global__ void wait_timeout_kernel(int* err) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    const uint32_t b = smem_u32(&bar);
    mbar_init(b, 1);
    fence_mbar_init();
    if (!mbar_wait(b, 0)) atomicOr(err, PA_DEVERR_TIMEOUT);
  }
}

}  // namespace

cudaError_t launch_wait_timeout_selftest(int* err, cudaStream_t st) {
  wait_timeout_kernel<<<1, 32, 0, st>>>(err);
  return cudaGetLastError();
}

}  // namespace pa
