// Self-tests (the pages have no counterpart to either):
//
// * the failure path shared by every kernel: a bounded mbarrier wait that
//   runs out sets PKV_DEV_TIMEOUT in the device error word and returns, so
//   the host learns of it and the context stays usable.  It exists so the
//   timeout path can be exercised on a GPU without a fault or a hang (the
//   barrier waited on simply never completes);
// * a read-only streaming kernel, the measured read bandwidth that the
//   decode kernels (which only read the pool) are compared with.
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

// Read-only streaming: every 16-byte word of the buffer is loaded once
// (non-caching loads, four in flight per thread per iteration) and folded
// into an XOR per warp, so the loads cannot be elided; one atomic per warp.
__global__ void __launch_bounds__(512, 4) read_stream_kernel(const uint4* __restrict__ buf,
                                                          size_t n16, unsigned* sink) {
  auto ld = [](const uint4* q) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(q));
    return v.x ^ v.y ^ v.z ^ v.w;
  };
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  unsigned acc = 0;
  for (; i + 3 * stride < n16; i += 4 * stride) {
    const unsigned a = ld(buf + i), b = ld(buf + i + stride);
    const unsigned c = ld(buf + i + 2 * stride), d = ld(buf + i + 3 * stride);
    acc ^= a ^ b ^ c ^ d;
  }
  for (; i < n16; i += stride) acc ^= ld(buf + i);
  for (int o = 16; o > 0; o >>= 1) acc ^= __shfl_xor_sync(0xffffffffu, acc, o);
  if ((threadIdx.x & 31) == 0) atomicXor(sink, acc);
}

}  // namespace pkv

extern "C" int paged_selftest_read_stream(const void* buf, size_t bytes, uint32_t* sink,
                                          cudaStream_t stream) {
  if (!sink) return PKV_ERR_NULL;
  if (bytes == 0) return PKV_OK;  // nothing to read (buf may then be NULL)
  if (!buf) return PKV_ERR_NULL;
  if (((uintptr_t)buf & 15) || (bytes & 15)) return PKV_ERR_ALIGN;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) {
    (void)cudaGetLastError();
    return PKV_ERR_CUDA;
  }
  pkv::read_stream_kernel<<<(unsigned)sms * 4, 512, 0, stream>>>(
      static_cast<const uint4*>(buf), bytes / 16, sink);
  return cudaPeekAtLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

extern "C" int paged_selftest_wait_timeout(uint64_t limit_ns, cudaStream_t stream) {
  if (limit_ns == 0 || limit_ns > 1000000000ull) return PKV_ERR_ARG;
  unsigned* err = pkv_error_word();
  if (!err) return PKV_ERR_CUDA;
  pkv::selftest_wait_kernel<<<1, 32, 0, stream>>>(limit_ns, err);
  return cudaPeekAtLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}
