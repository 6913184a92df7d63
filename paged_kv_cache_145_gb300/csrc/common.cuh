// Device helpers shared by the paged KV cache kernels (sm_103a).
//
// Inline PTX for the Blackwell data movers used here: mbarrier
// initialisation / expect-tx / bounded parity waits, and 1-D bulk copies
// (cp.async.bulk, the TMA's non-tensor form) from global into shared memory.
// Element conversions for the three cache types, and 16-byte row loaders.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "../../include/pagedkv.h"

namespace pkv {

constexpr unsigned kFullMask = 0xffffffffu;
// Wall-clock bound on one mbarrier wait.  A bulk copy lands in about a
// microsecond; if one has not landed after this long, the kernel records
// PKV_DEV_TIMEOUT and stops waiting instead of hanging the GPU.
constexpr uint64_t kWaitLimitNs = 200ull * 1000 * 1000;

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Makes initialised barriers visible to the async (bulk-copy) proxy.
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Orders this thread's earlier generic shared-memory accesses before later
// async-proxy (bulk copy) accesses to the same memory.
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// One plain arrival (no transaction bytes).
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Named barrier `id` for `threads` threads (a multiple of 32): a subset of
// the block's warps waits for one another.
__device__ __forceinline__ void named_bar_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Non-blocking test of the same condition (never suspends the thread), for
// roles that poll several barriers.
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// Waits for the barrier phase with the given parity to complete; false if
// `limit_ns` of wall-clock time passed first.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity,
                                          uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (;;) {
#pragma unroll 1
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (global_ns() - t0 > limit_ns) return false;
  }
}

// Bulk copy of `bytes` (multiple of 16; both addresses 16-byte aligned)
// from global to this CTA's shared memory; completion is signalled on `bar`
// as transaction bytes.  The L2 policy marks the lines evict-first: every
// cache page is read once per decode step.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// 32-bit load through the non-coherent path, kept in program order with the
// other loads written this way (so independent loads issue back to back).
__device__ __forceinline__ int ld_nc(const int32_t* p) {
  int v;
  asm volatile("ld.global.nc.b32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}

__device__ __forceinline__ void set_error(unsigned* err, unsigned bits) {
  if (err) atomicOr(err, bits);
}

// ---------------------------------------------------------------------------
// Element types
// ---------------------------------------------------------------------------
template <typename T>
struct Elem;

template <>
struct Elem<float> {
  static __device__ __forceinline__ float from_f(float x) { return x; }
};

template <>
struct Elem<__half> {
  static __device__ __forceinline__ float2 pair(uint32_t w) {
    __half2 h = *reinterpret_cast<__half2*>(&w);
    return __half22float2(h);
  }
  static __device__ __forceinline__ __half from_f(float x) { return __float2half_rn(x); }
};

template <>
struct Elem<__nv_bfloat16> {
  // A bfloat16 is the upper half of an IEEE binary32: widening is a shift.
  static __device__ __forceinline__ float2 pair(uint32_t w) {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
  }
  static __device__ __forceinline__ __nv_bfloat16 from_f(float x) { return __float2bfloat16_rn(x); }
};

// Largest of three.
__device__ __forceinline__ float max3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// 2^x with the hardware approximation (flushes results below 2^-126 to 0).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <typename T>
__device__ __forceinline__ uint32_t pack_pair(float lo, float hi);
template <>
__device__ __forceinline__ uint32_t pack_pair<__half>(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}
template <>
__device__ __forceinline__ uint32_t pack_pair<__nv_bfloat16>(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// Loads N consecutive elements (N * sizeof(T) in {4, 8, 16} bytes, aligned to
// that size) and widens them to float.
template <typename T, int N>
struct RowLoad {
  static constexpr int kBytes = N * (int)sizeof(T);
  static_assert(kBytes == 4 || kBytes == 8 || kBytes == 16, "row fragment size");
  static __device__ __forceinline__ void load(const T* p, float (&f)[N]) {
    if constexpr (sizeof(T) == 4) {
      if constexpr (kBytes == 16) {
        float4 v = *reinterpret_cast<const float4*>(p);
        f[0] = v.x; f[1] = v.y; f[2] = v.z; f[3] = v.w;
      } else if constexpr (kBytes == 8) {
        float2 v = *reinterpret_cast<const float2*>(p);
        f[0] = v.x; f[1] = v.y;
      } else {
        f[0] = *reinterpret_cast<const float*>(p);
      }
    } else {
      constexpr int W = kBytes / 4;
      uint32_t w[W];
      if constexpr (W == 4) {
        uint4 v = *reinterpret_cast<const uint4*>(p);
        w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
      } else if constexpr (W == 2) {
        uint2 v = *reinterpret_cast<const uint2*>(p);
        w[0] = v.x; w[1] = v.y;
      } else {
        w[0] = *reinterpret_cast<const uint32_t*>(p);
      }
#pragma unroll
      for (int i = 0; i < W; ++i) {
        float2 x = Elem<T>::pair(w[i]);
        f[2 * i] = x.x;
        f[2 * i + 1] = x.y;
      }
    }
  }
};

// One row fragment of a cache page: N consecutive elements widened to float.
// 16- and 32-bit pools use RowLoad; FP8 E4M3 codes are widened two at a
// time through CUDA's e4m3x2 -> half2 conversion (exact: every E4M3 value
// is a half).
template <typename TC, int N>
struct CacheRow {
  static __device__ __forceinline__ void load(const TC* p, float (&f)[N]) { RowLoad<TC, N>::load(p, f); }
};

__device__ __forceinline__ float2 e4m3x2_to_float2(uint16_t x) {
  const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)x, __NV_E4M3);
  return __half22float2(*reinterpret_cast<const __half2*>(&h));
}

template <int N>
struct CacheRow<__nv_fp8_e4m3, N> {
  static_assert(N == 2 || N == 4, "FP8 row fragment size");
  static __device__ __forceinline__ void load(const __nv_fp8_e4m3* p, float (&f)[N]) {
    if constexpr (N == 4) {
      const uint32_t w = *reinterpret_cast<const uint32_t*>(p);
      const float2 a = e4m3x2_to_float2((uint16_t)(w & 0xffffu));
      const float2 b = e4m3x2_to_float2((uint16_t)(w >> 16));
      f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
    } else {
      const float2 a = e4m3x2_to_float2(*reinterpret_cast<const uint16_t*>(p));
      f[0] = a.x; f[1] = a.y;
    }
  }
};

}  // namespace pkv

// Host-side: address of the per-device error word (defined in api.cu).
unsigned* pkv_error_word();
