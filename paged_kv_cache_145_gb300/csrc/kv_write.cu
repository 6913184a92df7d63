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
// kernel is a byte mover: one CTA per token, 16-byte vectors, keys and
// values interleaved so each thread has two independent loads in flight.
#include "common.cuh"

namespace pkv {

__global__ void __launch_bounds__(128)
kv_write_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v,
                const int64_t* __restrict__ slots, uint4* __restrict__ kc,
                uint4* __restrict__ vc, int64_t num_blocks, int block_size,
                int kv_heads, int row_vecs, unsigned* err) {
  const int64_t i = blockIdx.x;
  const int64_t slot = slots[i];
  if (slot < 0) return;  // padding token
  const int64_t blk = slot / block_size;
  const int off = (int)(slot - blk * block_size);
  if (blk >= num_blocks) {
    if (threadIdx.x == 0) set_error(err, PKV_DEV_SLOT_RANGE);
    return;
  }
  const int total = kv_heads * row_vecs;  // 16-byte vectors per token
  const uint4* ks = k + i * total;
  const uint4* vs = v + i * total;
  const int64_t page0 = blk * kv_heads;
  for (int u = threadIdx.x; u < total; u += blockDim.x) {
    const int h = u / row_vecs;
    const int r = u - h * row_vecs;
    const int64_t dst = ((page0 + h) * block_size + off) * row_vecs + r;
    const uint4 a = __ldg(ks + u);
    const uint4 b = __ldg(vs + u);
    kc[dst] = a;
    vc[dst] = b;
  }
}

}  // namespace pkv

int pkv_launch_kv_write(const pkv_cache* c, const void* k, const void* v, const int64_t* slots,
                        int64_t num_tokens, size_t elem_bytes, cudaStream_t stream) {
  const int row_vecs = (int)(c->head_dim * elem_bytes / 16);
  pkv::kv_write_kernel<<<(unsigned)num_tokens, 128, 0, stream>>>(
      static_cast<const uint4*>(k), static_cast<const uint4*>(v), slots,
      static_cast<uint4*>(c->k_cache), static_cast<uint4*>(c->v_cache), c->num_blocks,
      c->block_size, c->num_kv_heads, row_vecs, pkv_error_word());
  return cudaPeekAtLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}
