// Prefill attention (tcgen05 kernel) instantiations for f16 pools.
#include "prefill_tc.cuh"

int pkv_launch_prefill_tc_f16(const pkv::PrefillParams& p, int num_seqs, int head_dim,
                            int block_size, int group, const CUtensorMap& mk,
                            const CUtensorMap& mv, cudaStream_t stream) {
  return pkv::launch_prefill_tc<__half>(p, num_seqs, head_dim, block_size, group, mk, mv, stream);
}
