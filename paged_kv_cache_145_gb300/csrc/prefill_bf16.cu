// Prefill attention (mma.sync kernel) instantiations for one cache element type.
#include "prefill.cuh"

int pkv_launch_prefill_bf16(const pkv::PrefillParams& p, int num_seqs, int head_dim, int block_size,
                         int group, const CUtensorMap& mk, const CUtensorMap& mv,
                         cudaStream_t stream) {
  return pkv::launch_prefill<__nv_bfloat16>(p, num_seqs, head_dim, block_size, group, mk, mv, stream);
}
