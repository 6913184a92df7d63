// Decode attention instantiations for one cache element type (split per type
// so the three translation units compile in parallel).
#include "decode_launch.cuh"

int pkv_launch_decode_f16(const pkv::DecodeParams& p, int num_seqs, int head_dim, int block_size,
                        int group, const pkv::DecodeMaps* maps, cudaStream_t stream) {
  return pkv::launch_decode<__half>(p, num_seqs, head_dim, block_size, group, maps, stream);
}

int pkv_launch_decode_shared_f16(const pkv::DecodeParams& p, int num_seqs, int head_dim,
                               int block_size, int group, int max_group_size,
                               const pkv::DecodeMaps* maps, const pkv::DecodeMaps* part_maps,
                               cudaStream_t stream) {
  return pkv::launch_decode_shared<__half>(p, num_seqs, head_dim, block_size, group, max_group_size,
                                        maps, part_maps, stream);
}
