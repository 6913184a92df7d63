// Self-test of the failure path shared by every kernel: a bounded mbarrier
// wait that runs out sets PKV_DEV_TIMEOUT in the device error word and
// returns, so the host learns of it and the context stays usable.  The pages
// have no counterpart; it exists so the timeout path can be exercised on a
// GPU without a fault or a hang (the barrier waited on simply never
// completes).
#include "common.cuh"

namespace pkv {

__global__ void selftest_wait_kernel(uint64_t limit_ns, unsigned* err) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(smem_addr(&bar), 1);
    fence_mbar_init();
    // Nothing ever arrives: the wait gives up after limit_ns.
    if (!mbar_wait(smem_addr(&bar), 0, limit_ns)) set_error(err, PKV_DEV_TIMEOUT);
  }
}

}  // namespace pkv

extern "C" int paged_selftest_wait_timeout(uint64_t limit_ns, cudaStream_t stream) {
  if (limit_ns == 0 || limit_ns > 1000000000ull) return PKV_ERR_ARG;
  unsigned* err = pkv_error_word();
  if (!err) return PKV_ERR_CUDA;
  pkv::selftest_wait_kernel<<<1, 32, 0, stream>>>(limit_ns, err);
  return cudaPeekAtLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}
