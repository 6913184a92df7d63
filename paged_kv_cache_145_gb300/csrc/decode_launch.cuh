// Host launchers of the decode kernels: pick the kernel for the geometry,
// opt in to large dynamic shared memory once per device, launch the
// partition pass and, when sequences span several partitions, the merge.
#pragma once

#include <atomic>
#include <type_traits>

#include "decode.cuh"
#include "decode_mma.cuh"
#include "decode_mma_fp8.cuh"
#include "decode_shared.cuh"

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

// The split-K merge, when any sequence spans several partitions.
template <typename T, int D>
void launch_reduce(const DecodeParams& p, int num_seqs, cudaStream_t stream) {
  if (p.num_parts <= 1) return;
  if (p.num_parts <= 8) {
    dim3 g2((unsigned)((p.num_heads + kReduceWarps - 1) / kReduceWarps), (unsigned)num_seqs);
    decode_reduce_kernel<T, D, 1><<<g2, kReduceWarps * 32, 0, stream>>>(p);
  } else {
    dim3 g2((unsigned)p.num_heads, (unsigned)num_seqs);
    decode_reduce_kernel<T, D, kReduceWarps><<<g2, kReduceWarps * 32, 0, stream>>>(p);
  }
}

template <typename T, int D, int BS, int G>
int launch_decode_cfg(const DecodeParams& p, int num_seqs, const DecodeMaps* maps,
                      cudaStream_t stream) {
  dim3 grid((unsigned)p.kv_heads, (unsigned)num_seqs,
            (unsigned)(p.tail_parts > 0 ? p.tail_parts : p.num_parts));
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
  launch_reduce<T, D>(p, num_seqs, stream);
  return cudaPeekAtLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

// Shared-prefix decode (16-bit pools): the groups' shared partitions, then
// the partition pass over the rest and the merge.
// `maps` feed the shared-prefix kernel; `part_maps` (null: CUDA-core
// kernel) the partition pass, as in the plain decode.
template <typename T, int D, int BS, int G, int DUP>
int launch_shared_dup(const DecodeParams& p, int max_group_size, const DecodeMaps* maps,
                      cudaStream_t stream) {
  using Cfg = SharedTcCfg<T, D, BS, G, DUP>;
  const int64_t row_blocks = ((int64_t)max_group_size * G + Cfg::kRows - 1) / Cfg::kRows;
  if ((int64_t)p.num_parts * row_blocks > 65535) return PKV_ERR_ARG;
  auto kern = decode_shared_prefix_kernel<T, D, BS, G, DUP>;
  if (allow_smem<Cfg>(kern, Cfg::kSmemBytes) != PKV_OK) return PKV_ERR_CUDA;
  dim3 grid((unsigned)p.kv_heads, (unsigned)p.num_groups, (unsigned)(p.num_parts * row_blocks));
  kern<<<grid, Cfg::kThreads, Cfg::kSmemBytes, stream>>>(p, (int)row_blocks, maps->k, maps->v);
  return cudaPeekAtLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

// Groups of at most 32 stacked rows (max_group_size x G) run with every row
// four times over the MMA's 128 rows, the copies splitting the softmax
// work; larger groups in blocks of 128 rows.
template <typename T, int D, int BS, int G>
int launch_shared_cfg(const DecodeParams& p, int num_seqs, int max_group_size,
                      const DecodeMaps* maps, const DecodeMaps* part_maps, cudaStream_t stream) {
  const int rc = (int64_t)max_group_size * G <= 32
                     ? launch_shared_dup<T, D, BS, G, 4>(p, max_group_size, maps, stream)
                     : launch_shared_dup<T, D, BS, G, 1>(p, max_group_size, maps, stream);
  if (rc != PKV_OK) return rc;
  if (p.tail_parts == 1) {  // every tail in one partition: tail and merge in one pass
    decode_tail_merge_kernel<T, D, BS, G>
        <<<dim3((unsigned)p.kv_heads, (unsigned)num_seqs), 128, 0, stream>>>(p);
    return cudaPeekAtLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
  }
  return launch_decode_cfg<T, D, BS, G>(p, num_seqs, part_maps, stream);
}

template <typename T>
int launch_decode_shared(const DecodeParams& p, int num_seqs, int head_dim, int block_size,
                         int group, int max_group_size, const DecodeMaps* maps,
                         const DecodeMaps* part_maps, cudaStream_t stream) {
#define PKV_SH_CASE(D_, B_, G_)                          \
  if (head_dim == D_ && block_size == B_ && group == G_) \
    return launch_shared_cfg<T, D_, B_, G_>(p, num_seqs, max_group_size, maps, part_maps, stream);
#define PKV_SH_G(D_, B_) PKV_SH_CASE(D_, B_, 1) PKV_SH_CASE(D_, B_, 2) \
  PKV_SH_CASE(D_, B_, 4) PKV_SH_CASE(D_, B_, 8)
  PKV_SH_G(64, 8) PKV_SH_G(64, 16) PKV_SH_G(64, 32) PKV_SH_G(64, 64)
  PKV_SH_G(128, 8) PKV_SH_G(128, 16) PKV_SH_G(128, 32) PKV_SH_G(128, 64)
#undef PKV_SH_G
#undef PKV_SH_CASE
  return PKV_ERR_GEOMETRY;
}

// FP8 pools (T is the 16-bit type of q and out): the tensor-core kernel
// that widens codes in shared memory, or the CUDA-core kernel.
template <typename T, int D, int BS, int G>
int launch_decode_fp8_cfg(const DecodeParams& p, int num_seqs, const DecodeMaps* maps,
                          bool mma, cudaStream_t stream) {
  dim3 grid((unsigned)p.kv_heads, (unsigned)num_seqs, (unsigned)p.num_parts);
  if (mma && D == 128) {
    if (!maps) return PKV_ERR_CUDA;
    if constexpr (D == 128) {
      using Cfg = Fp8MmaCfg<T, D, BS, G>;
      auto kern = decode_partition_mma_fp8_kernel<T, D, BS, G>;
      if (allow_smem<Cfg>(kern, Cfg::kMaxSmem) != PKV_OK) return PKV_ERR_CUDA;
      kern<<<grid, Cfg::kThreads, Cfg::smem_bytes(p.part_size), stream>>>(p, maps->k, maps->v);
    }
  } else if (mma) {
    using Cfg = Fp8WidenCfg<T, D, BS, G>;
    auto kern = decode_partition_mma_fp8_widen_kernel<T, D, BS, G>;
    if (allow_smem<Cfg>(kern, Cfg::kMaxSmem) != PKV_OK) return PKV_ERR_CUDA;
    kern<<<grid, Cfg::kThreads, Cfg::smem_bytes(p.part_size), stream>>>(p);
  } else {
    using Cfg = DecodeCfg<T, D, BS, G, __nv_fp8_e4m3>;
    auto kern = decode_partition_kernel<T, D, BS, G, __nv_fp8_e4m3>;
    if (allow_smem<Cfg>(kern, Cfg::kMaxSmem) != PKV_OK) return PKV_ERR_CUDA;
    kern<<<grid, Cfg::kThreads, Cfg::smem_bytes(p.part_size), stream>>>(p);
  }
  launch_reduce<T, D>(p, num_seqs, stream);
  return cudaPeekAtLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

template <typename T>
int launch_decode_fp8(const DecodeParams& p, int num_seqs, int head_dim, int block_size, int group,
                      const DecodeMaps* maps, bool mma, cudaStream_t stream) {
#define PKV_FP8_CASE(D_, B_, G_)                   \
  if (head_dim == D_ && block_size == B_ && group == G_) \
    return launch_decode_fp8_cfg<T, D_, B_, G_>(p, num_seqs, maps, mma, stream);
#define PKV_FP8_G(D_, B_) PKV_FP8_CASE(D_, B_, 1) PKV_FP8_CASE(D_, B_, 2) \
  PKV_FP8_CASE(D_, B_, 4) PKV_FP8_CASE(D_, B_, 8)
  PKV_FP8_G(64, 8) PKV_FP8_G(64, 16) PKV_FP8_G(64, 32) PKV_FP8_G(64, 64)
  PKV_FP8_G(128, 8) PKV_FP8_G(128, 16) PKV_FP8_G(128, 32) PKV_FP8_G(128, 64)
#undef PKV_FP8_G
#undef PKV_FP8_CASE
  return PKV_ERR_GEOMETRY;
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
