// paged_block_copy: whole-block copies, the copy half of copy-on-write.
//
// "Inside vLLM and TGI: Paging, Versioned Schedulers and Operations"
// ("Exact CPU block manager and copy-on-write"): appending to a shared,
// partially filled last block takes a fresh block and copies the old one
// into it; "vLLM and PagedAttention: Virtual Memory for LLM Serving"
// (sharing paragraph) calls this the private copy for the modified branch.
//
// With the [N][Hk][b][D] layout a block's keys for every head are one
// contiguous run of Hk * b * D elements, and likewise its values, so each
// pair is two contiguous copies.  Grid: (pair, key-or-value, slice); each
// thread moves kUnroll 16-byte vectors, issuing all loads before the stores.
#include "common.cuh"

namespace pkv {

constexpr int kCopyThreads = 256;
constexpr int kCopyUnroll = 4;
constexpr int kCopySlice = kCopyThreads * kCopyUnroll;  // vectors per CTA

__global__ void __launch_bounds__(kCopyThreads)
block_copy_kernel(const int64_t* __restrict__ pairs, uint4* __restrict__ kc,
                  uint4* __restrict__ vc, int64_t num_blocks, int64_t block_vecs,
                  unsigned* err) {
  const int64_t p = blockIdx.x;
  const int64_t src = pairs[2 * p];
  const int64_t dst = pairs[2 * p + 1];
  if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
    if (threadIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0) set_error(err, PKV_DEV_PAIR_RANGE);
    return;
  }
  if (src == dst) return;
  uint4* base = blockIdx.y == 0 ? kc : vc;
  const uint4* s = base + src * block_vecs;
  uint4* d = base + dst * block_vecs;
  const int64_t first = (int64_t)blockIdx.z * kCopySlice + threadIdx.x;
  uint4 buf[kCopyUnroll];
#pragma unroll
  for (int j = 0; j < kCopyUnroll; ++j) {
    const int64_t u = first + j * kCopyThreads;
    if (u < block_vecs) buf[j] = s[u];
  }
#pragma unroll
  for (int j = 0; j < kCopyUnroll; ++j) {
    const int64_t u = first + j * kCopyThreads;
    if (u < block_vecs) d[u] = buf[j];
  }
}

}  // namespace pkv

int pkv_launch_block_copy(const pkv_cache* c, const int64_t* pairs, int64_t num_pairs,
                          size_t elem_bytes, cudaStream_t stream) {
  const int64_t block_vecs =
      (int64_t)c->num_kv_heads * c->block_size * c->head_dim * (int64_t)elem_bytes / 16;
  const unsigned slices = (unsigned)((block_vecs + pkv::kCopySlice - 1) / pkv::kCopySlice);
  dim3 grid((unsigned)num_pairs, 2, slices);
  pkv::block_copy_kernel<<<grid, pkv::kCopyThreads, 0, stream>>>(
      pairs, static_cast<uint4*>(c->k_cache), static_cast<uint4*>(c->v_cache), c->num_blocks,
      block_vecs, pkv_error_word());
  return cudaPeekAtLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}
