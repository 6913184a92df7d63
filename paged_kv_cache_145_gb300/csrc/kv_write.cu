// paged_kv_write: slot-mapped store of each step's new keys and values
// ("reshape_and_cache").
//
// "vLLM and PagedAttention: Virtual Memory for LLM Serving" (paging
// paragraph) and "Inside vLLM and TGI: Paging, Versioned Schedulers and
// Operations" ("Exact CPU block manager and copy-on-write", append): a new
// token is stored at the next offset of its sequence's last block.  The host
// block manager turns that into a flat slot = block * b + offset; the kernel
// inverts it.
//
// Layout: k, v are [T][Hk][D]; each cache is [N][Hk][b][D].  One token's
// keys for all heads are one contiguous run of Hk * D elements in k; in the
// cache they land as Hk runs of D elements, one per (block, head) page.  The
// kernel is a byte mover over the flattened 16-byte vectors of all tokens:
// one thread per vector, keys and values loaded together, so a decode step's
// few hundred kilobytes spread over enough CTAs to finish in one round trip.
#include "common.cuh"

namespace pkv {

constexpr int kWriteThreads = 256;

__global__ void __launch_bounds__(kWriteThreads)
kv_write_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v,
                const int64_t* __restrict__ slots, uint4* __restrict__ kc,
                uint4* __restrict__ vc, int64_t num_blocks, int block_size,
                int kv_heads, int row_vecs, int64_t total, unsigned* err) {
  const int64_t u = (int64_t)blockIdx.x * kWriteThreads + threadIdx.x;
  if (u >= total) return;
  const int per_tok = kv_heads * row_vecs;
  const int64_t i = u / per_tok;
  const int rem = (int)(u - i * per_tok);
  const int64_t slot = slots[i];
  if (slot < 0) return;  // padding token
  const int64_t blk = slot / block_size;
  const int off = (int)(slot - blk * block_size);
  if (blk >= num_blocks) {
    if (rem == 0) set_error(err, PKV_DEV_SLOT_RANGE);
    return;
  }
  const int h = rem / row_vecs;
  const int r = rem - h * row_vecs;
  const int64_t dst = ((blk * kv_heads + h) * block_size + off) * row_vecs + r;
  const uint4 a = __ldg(k + u);
  const uint4 b = __ldg(v + u);
  kc[dst] = a;
  vc[dst] = b;
}

}  // namespace pkv

int pkv_launch_kv_write(const pkv_cache* c, const void* k, const void* v, const int64_t* slots,
                        int64_t num_tokens, size_t elem_bytes, cudaStream_t stream) {
  const int row_vecs = (int)(c->head_dim * elem_bytes / 16);
  const int64_t total = num_tokens * c->num_kv_heads * row_vecs;
  const int64_t blocks = (total + pkv::kWriteThreads - 1) / pkv::kWriteThreads;
  if (blocks > INT32_MAX) return PKV_ERR_ARG;
  pkv::kv_write_kernel<<<(unsigned)blocks, pkv::kWriteThreads, 0, stream>>>(
      static_cast<const uint4*>(k), static_cast<const uint4*>(v), slots,
      static_cast<uint4*>(c->k_cache), static_cast<uint4*>(c->v_cache), c->num_blocks,
      c->block_size, c->num_kv_heads, row_vecs, total, pkv_error_word());
  return cudaPeekAtLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}
