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
// thread moves kCopyUnroll 16-byte vectors, issuing all loads before the
// stores.  The same mover serves host<->device swapping (paged_block_swap):
// "Inside vLLM and TGI: Paging, Versioned Schedulers and Operations" ("Read
// the vLLM 0.11.0 scheduler...": swapping costs cache bytes in both
// directions over the link) and "vLLM and PagedAttention: Virtual Memory
// for LLM Serving" (preemption paragraph: KV data swapped into CPU memory
// and restored later).
#include "common.cuh"

namespace pkv {

// 512 threads x 4 vectors = 32 KiB per CTA: one whole GQA block (8 heads x 16
// x 128 x 2 B) per CTA.  Measured (copy of half the pool): GQA 6161 -> 6686
// GB/s against 256 x 4, OPT-13B 6685 -> 6635.
constexpr int kCopyThreads = 512;
constexpr int kCopyUnroll = 4;
constexpr int kCopySlice = kCopyThreads * kCopyUnroll;  // vectors per CTA

// Moves whole blocks from one pool to another (or within one pool): for each
// pair, block dst of the destination := block src of the source, keys
// (blockIdx.y == 0) and values (== 1).  Either pool may be device memory or
// device-accessible pinned host memory.
__global__ void __launch_bounds__(kCopyThreads)
block_move_kernel(const int64_t* __restrict__ pairs, const uint4* src_k, const uint4* src_v,
                  int64_t src_blocks, uint4* dst_k, uint4* dst_v, int64_t dst_blocks,
                  int64_t block_vecs, bool same_pool, unsigned* err) {
  const int64_t p = blockIdx.x;
  const int64_t src = pairs[2 * p];
  const int64_t dst = pairs[2 * p + 1];
  if (src < 0 || src >= src_blocks || dst < 0 || dst >= dst_blocks) {
    if (threadIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0) set_error(err, PKV_DEV_PAIR_RANGE);
    return;
  }
  if (same_pool && src == dst) return;
  const uint4* s = (blockIdx.y == 0 ? src_k : src_v) + src * block_vecs;
  uint4* d = (blockIdx.y == 0 ? dst_k : dst_v) + dst * block_vecs;
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

static int64_t block_vecs_of(const pkv_cache* c, size_t elem_bytes) {
  return (int64_t)c->num_kv_heads * c->block_size * c->head_dim * (int64_t)elem_bytes / 16;
}

static int launch_move(const int64_t* pairs, int64_t num_pairs, const void* sk, const void* sv,
                       int64_t src_blocks, void* dk, void* dv, int64_t dst_blocks,
                       int64_t block_vecs, bool same_pool, cudaStream_t stream) {
  const unsigned slices = (unsigned)((block_vecs + pkv::kCopySlice - 1) / pkv::kCopySlice);
  dim3 grid((unsigned)num_pairs, 2, slices);
  pkv::block_move_kernel<<<grid, pkv::kCopyThreads, 0, stream>>>(
      pairs, static_cast<const uint4*>(sk), static_cast<const uint4*>(sv), src_blocks,
      static_cast<uint4*>(dk), static_cast<uint4*>(dv), dst_blocks, block_vecs, same_pool,
      pkv_error_word());
  return cudaPeekAtLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

int pkv_launch_block_copy(const pkv_cache* c, const int64_t* pairs, int64_t num_pairs,
                          size_t elem_bytes, cudaStream_t stream) {
  return launch_move(pairs, num_pairs, c->k_cache, c->v_cache, c->num_blocks, c->k_cache,
                     c->v_cache, c->num_blocks, block_vecs_of(c, elem_bytes), true, stream);
}

int pkv_launch_block_swap(const pkv_cache* c, void* host_k, void* host_v, int64_t host_blocks,
                          const int64_t* pairs, int64_t num_pairs, int direction,
                          size_t elem_bytes, cudaStream_t stream) {
  const int64_t bv = block_vecs_of(c, elem_bytes);
  if (direction == PKV_SWAP_OUT)
    return launch_move(pairs, num_pairs, c->k_cache, c->v_cache, c->num_blocks, host_k, host_v,
                       host_blocks, bv, false, stream);
  return launch_move(pairs, num_pairs, host_k, host_v, host_blocks, c->k_cache, c->v_cache,
                     c->num_blocks, bv, false, stream);
}
