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

// FP8 pools: one thread per 8 new elements (16 bytes of a 16-bit io type),
// each stored as e4m3(x / scale[h]) -- float32 division, round to nearest
// even, saturation to +-448 -- as 8 code bytes.
template <typename TI>
__global__ void __launch_bounds__(kWriteThreads)
kv_write_fp8_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v,
                    const int64_t* __restrict__ slots, uint2* __restrict__ kc,
                    uint2* __restrict__ vc, int64_t num_blocks, int block_size, int kv_heads,
                    int row_vecs, int64_t total, const float* __restrict__ k_scale,
                    const float* __restrict__ v_scale, unsigned* err) {
  const int64_t u = (int64_t)blockIdx.x * kWriteThreads + threadIdx.x;
  if (u >= total) return;
  const int per_tok = kv_heads * row_vecs;
  const int64_t i = u / per_tok;
  const int rem = (int)(u - i * per_tok);
  const int64_t slot = slots[i];
  if (slot < 0) return;
  const int64_t blk = slot / block_size;
  const int off = (int)(slot - blk * block_size);
  if (blk >= num_blocks) {
    if (rem == 0) set_error(err, PKV_DEV_SLOT_RANGE);
    return;
  }
  const int h = rem / row_vecs;
  const int r = rem - h * row_vecs;
  const int64_t dst = ((blk * kv_heads + h) * block_size + off) * row_vecs + r;
  const float ks = k_scale[h], vs = v_scale[h];
  const uint4 a = __ldg(k + u);
  const uint4 b = __ldg(v + u);
  auto quant = [](const uint4& w, float sc) {
    float f[8];
    RowLoad<TI, 8>::load(reinterpret_cast<const TI*>(&w), f);
    uint32_t lo = 0, hi = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t c = __nv_cvt_float2_to_fp8x2(make_float2(f[2 * j] / sc, f[2 * j + 1] / sc),
                                                  __NV_SATFINITE, __NV_E4M3);
      if (j < 2) lo |= c << (16 * j);
      else hi |= c << (16 * (j - 2));
    }
    return make_uint2(lo, hi);
  };
  kc[dst] = quant(a, ks);
  vc[dst] = quant(b, vs);
}

}  // namespace pkv

int pkv_launch_kv_write_fp8(const pkv_cache* c, const void* k, const void* v,
                            const int64_t* slots, int64_t num_tokens, cudaStream_t stream) {
  const int row_vecs = c->head_dim / 8;  // 8 elements per thread
  const int64_t total = num_tokens * c->num_kv_heads * row_vecs;
  const int64_t blocks = (total + pkv::kWriteThreads - 1) / pkv::kWriteThreads;
  if (blocks > INT32_MAX) return PKV_ERR_ARG;
  auto launch = [&](auto kern) {
    kern<<<(unsigned)blocks, pkv::kWriteThreads, 0, stream>>>(
        static_cast<const uint4*>(k), static_cast<const uint4*>(v), slots,
        static_cast<uint2*>(c->k_cache), static_cast<uint2*>(c->v_cache), c->num_blocks,
        c->block_size, c->num_kv_heads, row_vecs, total, c->k_scale, c->v_scale,
        pkv_error_word());
  };
  if (c->io_dtype == PKV_F16)
    launch(pkv::kv_write_fp8_kernel<__half>);
  else
    launch(pkv::kv_write_fp8_kernel<__nv_bfloat16>);
  return cudaPeekAtLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

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
