// Decode attention over FP8 E4M3 pools (q and out fp16 or bf16).
#include "decode_launch.cuh"

int pkv_launch_decode_fp8(const pkv::DecodeParams& p, int num_seqs, int head_dim, int block_size,
                          int group, int io_dtype, const pkv::DecodeMaps* maps, bool mma,
                          cudaStream_t stream) {
  if (io_dtype == PKV_F16)
    return pkv::launch_decode_fp8<__half>(p, num_seqs, head_dim, block_size, group, maps, mma,
                                          stream);
  return pkv::launch_decode_fp8<__nv_bfloat16>(p, num_seqs, head_dim, block_size, group, maps, mma,
                                               stream);
}
