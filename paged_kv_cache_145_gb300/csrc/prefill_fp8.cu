// Prefill attention over FP8 E4M3 pools (tcgen05 kernel), q and out in
// fp16 or bf16.
#include "prefill_tc.cuh"

int pkv_launch_prefill_tc_fp8(const pkv::PrefillParams& p, int io_dtype, int num_seqs,
                              int head_dim, int block_size, int group, const CUtensorMap& mk,
                              const CUtensorMap& mv, cudaStream_t stream) {
  if (io_dtype == PKV_F16)
    return pkv::launch_prefill_tc_fp8<__half>(p, num_seqs, head_dim, block_size, group, mk, mv,
                                              stream);
  return pkv::launch_prefill_tc_fp8<__nv_bfloat16>(p, num_seqs, head_dim, block_size, group, mk,
                                                   mv, stream);
}
