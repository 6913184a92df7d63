// Decode attention over FP8 E4M3 pools (q and out fp16 or bf16).
#include "decode_launch.cuh"

// One I/O type per translation unit (they compile in parallel).
#ifdef PKV_FP8_IO_BF16
int pkv_launch_decode_fp8_bf16(const pkv::DecodeParams& p, int S, int D, int BS, int G,
                               const pkv::DecodeMaps* maps, bool mma, cudaStream_t stream) {
  return pkv::launch_decode_fp8<__nv_bfloat16>(p, S, D, BS, G, maps, mma, stream);
}
#else
int pkv_launch_decode_fp8_f16(const pkv::DecodeParams& p, int S, int D, int BS, int G,
                              const pkv::DecodeMaps* maps, bool mma, cudaStream_t stream) {
  return pkv::launch_decode_fp8<__half>(p, S, D, BS, G, maps, mma, stream);
}

int pkv_launch_decode_fp8_bf16(const pkv::DecodeParams& p, int S, int D, int BS, int G,
                               const pkv::DecodeMaps* maps, bool mma, cudaStream_t stream);

int pkv_launch_decode_fp8(const pkv::DecodeParams& p, int S, int D, int BS, int G, int io_dtype,
                          const pkv::DecodeMaps* maps, bool mma, cudaStream_t stream) {
  if (io_dtype == PKV_F16) return pkv_launch_decode_fp8_f16(p, S, D, BS, G, maps, mma, stream);
  return pkv_launch_decode_fp8_bf16(p, S, D, BS, G, maps, mma, stream);
}
#endif
