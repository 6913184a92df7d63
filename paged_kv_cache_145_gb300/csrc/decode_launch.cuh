// Host launchers of the decode kernels: pick the kernel for the geometry,
// opt in to large dynamic shared memory once per device, launch the
// partition pass and, when sequences span several partitions, the merge.
#pragma once

#include <atomic>
#include <type_traits>

#include "decode.cuh"
#include "decode_mma.cuh"

namespace pkv {

// Tensor maps of the key and value pools, for the tensor-core kernel.
struct DecodeMaps {
  CUtensorMap k;
  CUtensorMap v;
};

template <typename T, int D, int BS, int G>
constexpr bool mma_eligible() {
  return !std::is_same<T, float>::value && G >= 2 && BS % 8 == 0;
}

// One flag word per kernel configuration (`Tag`): kernels of one signature
// share a function-pointer type, so the type of `kern` cannot key it.
template <typename Tag, typename K>
int allow_smem(K kern, int bytes) {
  static std::atomic<uint64_t> ready{0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ERR_CUDA;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(ready.load() & bit)) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) !=
        cudaSuccess)
      return PKV_ERR_CUDA;
    ready.fetch_or(bit);
  }
  return PKV_OK;
}

template <typename T, int D, int BS, int G>
int launch_decode_cfg(const DecodeParams& p, int num_seqs, const DecodeMaps* maps,
                      cudaStream_t stream) {
  dim3 grid((unsigned)p.kv_heads, (unsigned)num_seqs, (unsigned)p.num_parts);
  bool launched = false;
  if constexpr (mma_eligible<T, D, BS, G>()) {
    if (maps) {
      using Cfg = MmaCfg<T, D, BS, G>;
      auto kern = decode_partition_mma_kernel<T, D, BS, G>;
      if (allow_smem<Cfg>(kern, Cfg::kMaxSmem) != PKV_OK) return PKV_ERR_CUDA;
      kern<<<grid, Cfg::kThreads, Cfg::smem_bytes(p.part_size), stream>>>(p, maps->k, maps->v);
      launched = true;
    }
  }
  if (!launched) {
    using Cfg = DecodeCfg<T, D, BS, G>;
    auto kern = decode_partition_kernel<T, D, BS, G>;
    if (allow_smem<Cfg>(kern, Cfg::kMaxSmem) != PKV_OK) return PKV_ERR_CUDA;
    kern<<<grid, Cfg::kThreads, Cfg::smem_bytes(p.part_size), stream>>>(p);
  }
  if (p.num_parts > 1) {
    if (p.num_parts <= 8) {
      dim3 g2((unsigned)((p.num_heads + kReduceWarps - 1) / kReduceWarps), (unsigned)num_seqs);
      decode_reduce_kernel<T, D, 1><<<g2, kReduceWarps * 32, 0, stream>>>(p);
    } else {
      dim3 g2((unsigned)p.num_heads, (unsigned)num_seqs);
      decode_reduce_kernel<T, D, kReduceWarps><<<g2, kReduceWarps * 32, 0, stream>>>(p);
    }
  }
  return cudaPeekAtLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

template <typename T, int D, int BS>
int launch_decode_g(const DecodeParams& p, int num_seqs, int group, const DecodeMaps* maps,
                    cudaStream_t stream) {
  switch (group) {
    case 1: return launch_decode_cfg<T, D, BS, 1>(p, num_seqs, maps, stream);
    case 2: return launch_decode_cfg<T, D, BS, 2>(p, num_seqs, maps, stream);
    case 4: return launch_decode_cfg<T, D, BS, 4>(p, num_seqs, maps, stream);
    case 8: return launch_decode_cfg<T, D, BS, 8>(p, num_seqs, maps, stream);
  }
  return PKV_ERR_GEOMETRY;
}

template <typename T, int D>
int launch_decode_b(const DecodeParams& p, int num_seqs, int block_size, int group,
                    const DecodeMaps* maps, cudaStream_t stream) {
  switch (block_size) {
    case 8: return launch_decode_g<T, D, 8>(p, num_seqs, group, maps, stream);
    case 16: return launch_decode_g<T, D, 16>(p, num_seqs, group, maps, stream);
    case 32: return launch_decode_g<T, D, 32>(p, num_seqs, group, maps, stream);
    case 64: return launch_decode_g<T, D, 64>(p, num_seqs, group, maps, stream);
  }
  return PKV_ERR_GEOMETRY;
}

template <typename T>
int launch_decode(const DecodeParams& p, int num_seqs, int head_dim, int block_size, int group,
                  const DecodeMaps* maps, cudaStream_t stream) {
  switch (head_dim) {
    case 64: return launch_decode_b<T, 64>(p, num_seqs, block_size, group, maps, stream);
    case 128: return launch_decode_b<T, 128>(p, num_seqs, block_size, group, maps, stream);
  }
  return PKV_ERR_GEOMETRY;
}

}  // namespace pkv
