// C ABI entry points: host-side argument checks, dispatch, device error word.
// The semantics of each call are documented in include/pagedkv.h.
#include <cudaTypedefs.h>

#include <cmath>
#include <cstring>
#include <mutex>

#include "decode_launch.cuh"
#include "prefill.cuh"

int pkv_launch_kv_write(const pkv_cache* c, const void* k, const void* v, const int64_t* slots,
                        int64_t num_tokens, size_t elem_bytes, cudaStream_t stream);
int pkv_launch_kv_write_fp8(const pkv_cache* c, const void* k, const void* v,
                            const int64_t* slots, int64_t num_tokens, cudaStream_t stream);
int pkv_launch_decode_fp8(const pkv::DecodeParams& p, int num_seqs, int head_dim, int block_size,
                          int group, int io_dtype, const pkv::DecodeMaps* maps, bool mma,
                          cudaStream_t stream);
int pkv_launch_block_copy(const pkv_cache* c, const int64_t* pairs, int64_t num_pairs,
                          size_t elem_bytes, cudaStream_t stream);
int pkv_launch_block_swap(const pkv_cache* c, void* host_k, void* host_v, int64_t host_blocks,
                          const int64_t* pairs, int64_t num_pairs, int direction,
                          size_t elem_bytes, cudaStream_t stream);
int pkv_launch_prefill_f16(const pkv::PrefillParams&, int, int, int, int, const CUtensorMap&,
                           const CUtensorMap&, cudaStream_t);
int pkv_launch_prefill_bf16(const pkv::PrefillParams&, int, int, int, int, const CUtensorMap&,
                            const CUtensorMap&, cudaStream_t);
int pkv_launch_prefill_tc_f16(const pkv::PrefillParams&, int, int, int, int, const CUtensorMap&,
                              const CUtensorMap&, cudaStream_t);
int pkv_launch_prefill_tc_bf16(const pkv::PrefillParams&, int, int, int, int, const CUtensorMap&,
                               const CUtensorMap&, cudaStream_t);
int pkv_launch_prefill_tc_fp8(const pkv::PrefillParams&, int, int, int, int, int,
                              const CUtensorMap&, const CUtensorMap&, cudaStream_t);
int pkv_launch_decode_f32(const pkv::DecodeParams&, int, int, int, int, const pkv::DecodeMaps*,
                          cudaStream_t);
int pkv_launch_decode_f16(const pkv::DecodeParams&, int, int, int, int, const pkv::DecodeMaps*,
                          cudaStream_t);
int pkv_launch_decode_bf16(const pkv::DecodeParams&, int, int, int, int, const pkv::DecodeMaps*,
                           cudaStream_t);
int pkv_launch_decode_shared_f16(const pkv::DecodeParams&, int, int, int, int, int,
                                 const pkv::DecodeMaps*, const pkv::DecodeMaps*, cudaStream_t);
int pkv_launch_decode_shared_bf16(const pkv::DecodeParams&, int, int, int, int, int,
                                  const pkv::DecodeMaps*, const pkv::DecodeMaps*, cudaStream_t);

// One error word per device, OR-ed by the kernels (PKV_DEV_* bits).
static __device__ unsigned g_pkv_error;

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_err_mu;
unsigned* g_err_ptr[kMaxDevices] = {};

constexpr int kDefaultPartition = 512;

size_t elem_bytes(int dtype) {
  switch (dtype) {
    case PKV_F32: return 4;
    case PKV_F16: return 2;
    case PKV_BF16: return 2;
    case PKV_FP8_E4M3: return 1;
  }
  return 0;
}

// Pools whose elements the kernels must interpret (write, attention): an
// FP8 pool needs both scale arrays and a 16-bit io type.
int check_scales(const pkv_cache* c) {
  if (c->dtype != PKV_FP8_E4M3) return PKV_OK;
  if (c->io_dtype != PKV_F16 && c->io_dtype != PKV_BF16) return PKV_ERR_ARG;
  if (!c->k_scale || !c->v_scale) return PKV_ERR_NULL;
  if ((reinterpret_cast<uintptr_t>(c->k_scale) & 3u) || (reinterpret_cast<uintptr_t>(c->v_scale) & 3u))
    return PKV_ERR_ALIGN;
  return PKV_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Checks common to every call that touches the pool.
int check_cache(const pkv_cache* c) {
  if (!c || !c->k_cache || !c->v_cache) return PKV_ERR_NULL;
  if (elem_bytes(c->dtype) == 0) return PKV_ERR_ARG;
  if (c->num_blocks < 1 || c->num_blocks > INT32_MAX || c->block_size < 1 ||
      c->num_kv_heads < 1 || c->head_dim < 1)
    return PKV_ERR_ARG;
  if ((c->head_dim * elem_bytes(c->dtype)) % 16 != 0) return PKV_ERR_GEOMETRY;
  if (!aligned16(c->k_cache) || !aligned16(c->v_cache)) return PKV_ERR_ALIGN;
  return PKV_OK;
}

bool decode_geometry_ok(const pkv_cache* c, int num_heads) {
  if (c->head_dim != 64 && c->head_dim != 128) return false;
  if (c->block_size != 8 && c->block_size != 16 && c->block_size != 32 && c->block_size != 64)
    return false;
  if (num_heads < 1 || num_heads % c->num_kv_heads) return false;
  const int g = num_heads / c->num_kv_heads;
  return g == 1 || g == 2 || g == 4 || g == 8;
}

int resolve_max_len(const pkv_cache* c, int32_t max_blocks, int32_t max_seq_len) {
  const int64_t cap = (int64_t)max_blocks * c->block_size;
  if (max_seq_len == 0) return cap > INT32_MAX ? -1 : (int)cap;
  if (max_seq_len < 0 || max_seq_len > cap) return -1;
  return max_seq_len;
}

// Default partition length.  16-bit and 32-bit pools use 512 positions.
// An FP8 partition carries half the bytes per position, so its fixed costs
// (table staging, first-load latency, the split-K merge) weigh twice as
// much: FP8 pools take the longest of 2048, 1536, 1024 and 512 positions
// that still launches at least 8 thread blocks per SM (sequences x KV heads
// x partitions), so large batches skip the split while few long sequences
// keep every SM busy.  (Measured: 1536 beats 1024 by 2% on 8 sequences of
// 16k-32k positions, where 2048 leaves the last wave half empty.)
int default_partition(const pkv_cache* c, int64_t num_seqs, int64_t max_len) {
  if (c->dtype != PKV_FP8_E4M3 || num_seqs < 1 || max_len < 1) return kDefaultPartition;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1) {
    cudaGetLastError();
    return kDefaultPartition;
  }
  for (int part : {2048, 1536, 1024}) {
    const int64_t blocks = num_seqs * c->num_kv_heads * ((max_len + part - 1) / part);
    if (blocks >= 8LL * sms) return part;
  }
  return kDefaultPartition;
}

int resolve_partition(const pkv_cache* c, int32_t requested, int64_t num_seqs, int64_t max_len) {
  if (requested == 0) return default_partition(c, num_seqs, max_len);
  if (requested < c->block_size || requested % c->block_size || requested > pkv::kMaxPartSize)
    return PKV_ERR_ARG;
  return requested;
}

struct WsLayout {
  int parts;
  size_t ml_bytes;
  size_t o_offset;
  size_t total;
};

WsLayout workspace_layout(int num_seqs, int num_heads, int head_dim, int max_len, int part) {
  WsLayout w{};
  w.parts = (max_len + part - 1) / part;
  if (w.parts <= 1) {
    w.parts = 1;
    return w;
  }
  const size_t rows = (size_t)num_seqs * num_heads * w.parts;
  w.ml_bytes = rows * sizeof(float2);
  w.o_offset = (w.ml_bytes + 255) & ~size_t(255);
  w.total = w.o_offset + rows * head_dim * sizeof(float);
  return w;
}

// The tensor-core decode kernels serve fp16 / bf16 pools whose query heads
// come in groups of 2, 4 or 8, and every FP8 pool.  PKV_DECODE_KERNEL=simt in
// the environment selects the CUDA-core kernel instead (read on every call).
bool simt_forced() {
  const char* env = std::getenv("PKV_DECODE_KERNEL");
  return env && std::strcmp(env, "simt") == 0;
}

// Prefill runs on the tcgen05 kernel; PKV_PREFILL_KERNEL=mma in the
// environment selects the mma.sync kernel instead (read on every call).
bool prefill_mma_forced() {
  const char* env = std::getenv("PKV_PREFILL_KERNEL");
  return env && std::strcmp(env, "mma") == 0;
}

bool use_mma(const pkv_cache* c, int group) {
  if (c->dtype == PKV_FP8_E4M3) return !simt_forced();  // every grouping
  if (c->dtype == PKV_F32 || group < 2) return false;
  return !simt_forced();
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      f = nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }();
  return fn;
}

// Describes a [N][Hk][b][D] pool as a 4-D tensor (D fastest) read in boxes of
// min(b, 16) rows x 128 bytes (64 16-bit elements, or 128 FP8 codes) with the
// 128-byte shared-memory swizzle.
bool encode_pool_map(CUtensorMap* map, const pkv_cache* c, void* base) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint64_t elt = elem_bytes(c->dtype);
  const cuuint64_t dims[4] = {(cuuint64_t)c->head_dim, (cuuint64_t)c->block_size,
                              (cuuint64_t)c->num_kv_heads, (cuuint64_t)c->num_blocks};
  const cuuint64_t strides[3] = {c->head_dim * elt, c->block_size * c->head_dim * elt,
                                 (cuuint64_t)c->num_kv_heads * c->block_size * c->head_dim * elt};
  const cuuint32_t box[4] = {(cuuint32_t)(128 / elt),
                             (cuuint32_t)(c->block_size < 16 ? c->block_size : 16), 1, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUtensorMapDataType ty =
      c->dtype == PKV_FP8_E4M3 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
      : c->dtype == PKV_BF16   ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                               : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  return enc(map, ty, 4, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

unsigned* pkv_error_word() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_err_mu);
  if (!g_err_ptr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_pkv_error) != cudaSuccess) return nullptr;
    g_err_ptr[dev] = static_cast<unsigned*>(ptr);
  }
  return g_err_ptr[dev];
}

extern "C" {

int paged_kv_write(const pkv_cache* cache, const void* k, const void* v,
                   const int64_t* slot_mapping, int64_t num_tokens, cudaStream_t stream) {
  int rc = check_cache(cache);
  if (rc) return rc;
  rc = check_scales(cache);
  if (rc) return rc;
  if (num_tokens < 0 || num_tokens > INT32_MAX) return PKV_ERR_ARG;
  if (num_tokens == 0) return PKV_OK;
  if (!k || !v || !slot_mapping) return PKV_ERR_NULL;
  if (!aligned16(k) || !aligned16(v) || (reinterpret_cast<uintptr_t>(slot_mapping) & 7u))
    return PKV_ERR_ALIGN;
  if (!pkv_error_word()) return PKV_ERR_CUDA;
  if (cache->dtype == PKV_FP8_E4M3)
    return pkv_launch_kv_write_fp8(cache, k, v, slot_mapping, num_tokens, stream);
  return pkv_launch_kv_write(cache, k, v, slot_mapping, num_tokens, elem_bytes(cache->dtype),
                             stream);
}

int32_t paged_attention_partition_size(const pkv_cache* cache, int32_t num_seqs,
                                       int32_t num_heads, int32_t max_seq_len,
                                       int32_t requested) {
  if (!cache) return PKV_ERR_NULL;
  if (num_seqs < 0 || num_heads < 1 || max_seq_len < 0) return PKV_ERR_ARG;
  return resolve_partition(cache, requested, num_seqs, max_seq_len);
}

size_t paged_attention_workspace_bytes(const pkv_cache* cache, int32_t num_seqs,
                                       int32_t num_heads, int32_t max_seq_len,
                                       int32_t partition_size) {
  if (!cache || num_seqs < 1 || num_heads < 1 || max_seq_len < 1) return 0;
  const int part = resolve_partition(cache, partition_size, num_seqs, max_seq_len);
  if (part < 0) return 0;
  return workspace_layout(num_seqs, num_heads, cache->head_dim, max_seq_len, part).total;
}

namespace {

// Decode, plain (no groups) or with shared-prefix groups.
int decode_impl(const pkv_cache* cache, const void* q, const int32_t* block_tables,
                int32_t max_blocks_per_seq, const int32_t* seq_lens, int32_t num_seqs,
                int32_t num_heads, int32_t max_seq_len, float scale, void* out,
                const int32_t* group_starts, const int32_t* group_prefix, int32_t num_groups,
                int32_t max_group_size, int32_t tail_parts, void* workspace,
                size_t workspace_bytes, int32_t partition_size, cudaStream_t stream) {
  int rc = check_cache(cache);
  if (rc) return rc;
  rc = check_scales(cache);
  if (rc) return rc;
  if (num_seqs < 0 || num_seqs > 65535 || max_blocks_per_seq < 1 || num_heads < 1)
    return PKV_ERR_ARG;
  if (num_seqs == 0) return PKV_OK;
  if (!q || !out || !block_tables || !seq_lens) return PKV_ERR_NULL;
  if (!decode_geometry_ok(cache, num_heads)) return PKV_ERR_GEOMETRY;
  if (cache->num_kv_heads > 65535 || !std::isfinite(scale)) return PKV_ERR_ARG;
  if (!aligned16(q) || !aligned16(out) || (reinterpret_cast<uintptr_t>(block_tables) & 3u) ||
      (reinterpret_cast<uintptr_t>(seq_lens) & 3u))
    return PKV_ERR_ALIGN;
  const int max_len = resolve_max_len(cache, max_blocks_per_seq, max_seq_len);
  if (max_len < 1) return PKV_ERR_ARG;
  const int part = resolve_partition(cache, partition_size, num_seqs, max_len);
  if (part < 0) return part;
  const WsLayout ws = workspace_layout(num_seqs, num_heads, cache->head_dim, max_len, part);
  if (ws.parts > 65535) return PKV_ERR_ARG;  // partitions index the grid's z dimension
  if (ws.total > 0) {
    if (!workspace) return PKV_ERR_WORKSPACE;
    if (workspace_bytes < ws.total) return PKV_ERR_WORKSPACE;
    if (!aligned16(workspace)) return PKV_ERR_ALIGN;
  }
  unsigned* err = pkv_error_word();
  if (!err) return PKV_ERR_CUDA;

  pkv::DecodeParams p{};
  p.k_cache = cache->k_cache;
  p.v_cache = cache->v_cache;
  p.num_blocks = cache->num_blocks;
  p.kv_heads = cache->num_kv_heads;
  p.num_heads = num_heads;
  p.q = q;
  p.out = out;
  p.tables = block_tables;
  p.max_blocks = max_blocks_per_seq;
  p.seq_lens = seq_lens;
  p.max_len = max_len;
  p.qscale = scale * 1.4426950408889634f;  // log2(e): scores in base-2 units
  p.part_size = part;
  p.num_parts = ws.parts;
  p.ws_ml = ws.total ? static_cast<float2*>(workspace) : nullptr;
  p.ws_o = ws.total ? reinterpret_cast<float*>(static_cast<char*>(workspace) + ws.o_offset)
                    : nullptr;
  p.err = err;
  p.k_scale = cache->k_scale;
  p.v_scale = cache->v_scale;
  p.num_seqs = num_seqs;
  const int group = num_heads / cache->num_kv_heads;
  // Shared-prefix groups run on 16-bit pools (the grouped kernel's
  // tensor-core tiles); other pools decode every sequence in full, which
  // gives the same attention.
  const bool shared = group_starts && num_groups > 0 &&
                      (cache->dtype == PKV_F16 || cache->dtype == PKV_BF16);
  if (shared) {
    pkv::DecodeMaps maps;
    if (!encode_pool_map(&maps.k, cache, cache->k_cache) ||
        !encode_pool_map(&maps.v, cache, cache->v_cache))
      return PKV_ERR_CUDA;
    p.group_starts = group_starts;
    p.group_prefix = group_prefix;
    p.num_groups = num_groups;
    p.tail_parts = tail_parts < ws.parts ? tail_parts : 0;  // n >= the grid: the full grid
    const int D = cache->head_dim, B = cache->block_size;
    // The partition pass takes the tensor-core kernel only where the plain
    // decode would; the shared-prefix kernel always reads through the maps.
    const pkv::DecodeMaps* mp = use_mma(cache, group) ? &maps : nullptr;
    return cache->dtype == PKV_F16
               ? pkv_launch_decode_shared_f16(p, num_seqs, D, B, group, max_group_size, &maps, mp,
                                              stream)
               : pkv_launch_decode_shared_bf16(p, num_seqs, D, B, group, max_group_size, &maps,
                                               mp, stream);
  }
  if (cache->dtype == PKV_FP8_E4M3) {
    const bool mma = use_mma(cache, group);
    pkv::DecodeMaps fmaps;
    const pkv::DecodeMaps* fmp = nullptr;
    if (mma && cache->head_dim == 128) {  // direct key fragments read TMA-swizzled codes
      if (!encode_pool_map(&fmaps.k, cache, cache->k_cache) ||
          !encode_pool_map(&fmaps.v, cache, cache->v_cache))
        return PKV_ERR_CUDA;
      fmp = &fmaps;
    }
    return pkv_launch_decode_fp8(p, num_seqs, cache->head_dim, cache->block_size, group,
                                 cache->io_dtype, fmp, mma, stream);
  }
  pkv::DecodeMaps maps;
  const pkv::DecodeMaps* mp = nullptr;
  if (use_mma(cache, group)) {
    if (!encode_pool_map(&maps.k, cache, cache->k_cache) ||
        !encode_pool_map(&maps.v, cache, cache->v_cache))
      return PKV_ERR_CUDA;
    mp = &maps;
  }
  const int D = cache->head_dim, B = cache->block_size;
  switch (cache->dtype) {
    case PKV_F32: return pkv_launch_decode_f32(p, num_seqs, D, B, group, mp, stream);
    case PKV_F16: return pkv_launch_decode_f16(p, num_seqs, D, B, group, mp, stream);
    case PKV_BF16: return pkv_launch_decode_bf16(p, num_seqs, D, B, group, mp, stream);
  }
  return PKV_ERR_ARG;
}

}  // namespace

int paged_attention_decode(const pkv_cache* cache, const void* q, const int32_t* block_tables,
                           int32_t max_blocks_per_seq, const int32_t* seq_lens, int32_t num_seqs,
                           int32_t num_heads, int32_t max_seq_len, float scale, void* out,
                           void* workspace, size_t workspace_bytes, int32_t partition_size,
                           cudaStream_t stream) {
  return decode_impl(cache, q, block_tables, max_blocks_per_seq, seq_lens, num_seqs, num_heads,
                     max_seq_len, scale, out, nullptr, nullptr, 0, 0, 0, workspace,
                     workspace_bytes, partition_size, stream);
}

int paged_attention_decode_shared(const pkv_cache* cache, const void* q,
                                  const int32_t* block_tables, int32_t max_blocks_per_seq,
                                  const int32_t* seq_lens, int32_t num_seqs, int32_t num_heads,
                                  int32_t max_seq_len, float scale, void* out,
                                  const int32_t* group_starts, const int32_t* group_prefix,
                                  int32_t num_groups, int32_t max_group_size,
                                  int32_t tail_parts, void* workspace, size_t workspace_bytes,
                                  int32_t partition_size, cudaStream_t stream) {
  if (num_groups < 0 || num_groups > 65535 || tail_parts < 0 ||
      (num_groups > 0 && (max_group_size < 1 || max_group_size > num_seqs)))
    return PKV_ERR_ARG;
  if (num_groups > 0 && (!group_starts || !group_prefix)) return PKV_ERR_NULL;
  if ((reinterpret_cast<uintptr_t>(group_starts) & 3u) ||
      (reinterpret_cast<uintptr_t>(group_prefix) & 3u))
    return PKV_ERR_ALIGN;
  return decode_impl(cache, q, block_tables, max_blocks_per_seq, seq_lens, num_seqs, num_heads,
                     max_seq_len, scale, out, group_starts, group_prefix, num_groups,
                     max_group_size, tail_parts, workspace, workspace_bytes, partition_size,
                     stream);
}

int paged_attention_prefill(const pkv_cache* cache, const void* q, int64_t total_queries,
                            const int32_t* query_starts, int32_t num_seqs, int32_t max_queries,
                            const int32_t* block_tables, int32_t max_blocks_per_seq,
                            const int32_t* seq_lens, int32_t num_heads, float scale, void* out,
                            cudaStream_t stream) {
  int rc = check_cache(cache);
  if (rc) return rc;
  if (num_seqs < 0 || num_seqs > 65535 || max_blocks_per_seq < 1 || num_heads < 1 ||
      total_queries < 0 || total_queries > INT32_MAX || max_queries < 1 || !std::isfinite(scale))
    return PKV_ERR_ARG;
  if (num_seqs == 0 || total_queries == 0) return PKV_OK;
  if (!q || !out || !query_starts || !block_tables || !seq_lens) return PKV_ERR_NULL;
  // FP8 pools: the tcgen05 kernel only, head_dim 128.
  const bool fp8 = cache->dtype == PKV_FP8_E4M3;
  if (cache->dtype == PKV_F32 || !decode_geometry_ok(cache, num_heads) ||
      (fp8 && (cache->head_dim != 128 || prefill_mma_forced())))
    return PKV_ERR_GEOMETRY;
  rc = check_scales(cache);
  if (rc) return rc;
  if (cache->num_kv_heads > 65535 || (int64_t)max_blocks_per_seq * cache->block_size > INT32_MAX)
    return PKV_ERR_ARG;
  if (!aligned16(q) || !aligned16(out) || (reinterpret_cast<uintptr_t>(block_tables) & 3u) ||
      (reinterpret_cast<uintptr_t>(seq_lens) & 3u) ||
      (reinterpret_cast<uintptr_t>(query_starts) & 3u))
    return PKV_ERR_ALIGN;
  // The partition's table entries are staged in shared memory next to a
  // 64 KiB ring: bound the table width accordingly.
  if ((int64_t)max_blocks_per_seq * 4 > 150 * 1024) return PKV_ERR_ARG;
  unsigned* err = pkv_error_word();
  if (!err) return PKV_ERR_CUDA;
  CUtensorMap mk, mv;
  if (!encode_pool_map(&mk, cache, cache->k_cache) || !encode_pool_map(&mv, cache, cache->v_cache))
    return PKV_ERR_CUDA;
  pkv::PrefillParams p{};
  p.q = q;
  p.out = out;
  p.starts = query_starts;
  p.total_queries = total_queries;
  p.tables = block_tables;
  p.max_blocks = max_blocks_per_seq;
  p.seq_lens = seq_lens;
  p.num_blocks = cache->num_blocks;
  p.kv_heads = cache->num_kv_heads;
  p.num_heads = num_heads;
  p.max_queries = max_queries;
  p.qscale = scale * 1.4426950408889634f;
  p.err = err;
  p.k_scale = cache->k_scale;
  p.v_scale = cache->v_scale;
  const int group = num_heads / cache->num_kv_heads;
  const bool f16 = cache->dtype == PKV_F16;
  if (prefill_mma_forced())
    return (f16 ? pkv_launch_prefill_f16 : pkv_launch_prefill_bf16)(
        p, num_seqs, cache->head_dim, cache->block_size, group, mk, mv, stream);
  if (cache->num_blocks > INT32_MAX) return PKV_ERR_ARG;  // block coordinates are 32-bit
  if (fp8)
    return pkv_launch_prefill_tc_fp8(p, cache->io_dtype, num_seqs, cache->head_dim,
                                     cache->block_size, group, mk, mv, stream);
  return (f16 ? pkv_launch_prefill_tc_f16 : pkv_launch_prefill_tc_bf16)(
      p, num_seqs, cache->head_dim, cache->block_size, group, mk, mv, stream);
}

int paged_block_copy(const pkv_cache* cache, const int64_t* src_dst_pairs, int64_t num_pairs,
                     cudaStream_t stream) {
  int rc = check_cache(cache);
  if (rc) return rc;
  if (num_pairs < 0 || num_pairs > INT32_MAX) return PKV_ERR_ARG;
  if (num_pairs == 0) return PKV_OK;
  if (!src_dst_pairs) return PKV_ERR_NULL;
  if (reinterpret_cast<uintptr_t>(src_dst_pairs) & 7u) return PKV_ERR_ALIGN;
  if ((int64_t)cache->num_kv_heads * cache->block_size * cache->head_dim *
          (int64_t)elem_bytes(cache->dtype) % 16)
    return PKV_ERR_GEOMETRY;
  if (!pkv_error_word()) return PKV_ERR_CUDA;
  return pkv_launch_block_copy(cache, src_dst_pairs, num_pairs, elem_bytes(cache->dtype), stream);
}

// Device-side address of a host pool, or nullptr if the memory is neither
// page-locked nor managed (the kernel could not reach it).
static void* host_pool_address(void* p) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();  // clear the sticky-free error of the query
    return nullptr;
  }
  if (a.type == cudaMemoryTypeHost) return a.devicePointer;
  if (a.type == cudaMemoryTypeManaged) return p;
  return nullptr;
}

int paged_block_swap(const pkv_cache* cache, void* host_k, void* host_v, int64_t host_blocks,
                     const int64_t* src_dst_pairs, int64_t num_pairs, int32_t direction,
                     cudaStream_t stream) {
  int rc = check_cache(cache);
  if (rc) return rc;
  if (num_pairs < 0 || num_pairs > INT32_MAX || host_blocks < 1 ||
      (direction != PKV_SWAP_OUT && direction != PKV_SWAP_IN))
    return PKV_ERR_ARG;
  if (num_pairs == 0) return PKV_OK;
  if (!host_k || !host_v || !src_dst_pairs) return PKV_ERR_NULL;
  if (!aligned16(host_k) || !aligned16(host_v) ||
      (reinterpret_cast<uintptr_t>(src_dst_pairs) & 7u))
    return PKV_ERR_ALIGN;
  if ((int64_t)cache->num_kv_heads * cache->block_size * cache->head_dim *
          (int64_t)elem_bytes(cache->dtype) % 16)
    return PKV_ERR_GEOMETRY;
  void* dk = host_pool_address(host_k);
  void* dv = host_pool_address(host_v);
  if (!dk || !dv) return PKV_ERR_ARG;
  if (!pkv_error_word()) return PKV_ERR_CUDA;
  return pkv_launch_block_swap(cache, dk, dv, host_blocks, src_dst_pairs, num_pairs, direction,
                               elem_bytes(cache->dtype), stream);
}

int paged_get_device_error(cudaStream_t stream, uint32_t* bits) {
  if (!bits) return PKV_ERR_NULL;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return PKV_ERR_CUDA;
  unsigned v = 0;
  if (cudaMemcpyFromSymbol(&v, g_pkv_error, sizeof(v)) != cudaSuccess) return PKV_ERR_CUDA;
  const unsigned zero = 0;
  if (cudaMemcpyToSymbol(g_pkv_error, &zero, sizeof(zero)) != cudaSuccess) return PKV_ERR_CUDA;
  *bits = v;
  return PKV_OK;
}

const char* paged_strerror(int code) {
  switch (code) {
    case PKV_OK: return "ok";
    case PKV_ERR_NULL: return "a required pointer is NULL";
    case PKV_ERR_GEOMETRY: return "unsupported block size, head dim or head grouping";
    case PKV_ERR_ARG: return "invalid count, length bound or partition size";
    case PKV_ERR_ALIGN: return "buffer not aligned (16 bytes for data, element size for indices)";
    case PKV_ERR_WORKSPACE: return "workspace missing or too small";
    case PKV_ERR_CUDA: return "CUDA runtime call or kernel launch failed";
    case PKV_ERR_STATE: return "unknown or duplicate sequence id";
    case PKV_ERR_NOMEM: return "not enough free blocks (or host memory)";
    case PKV_ERR_CAPACITY: return "table wider than the output capacity";
  }
  return "unknown error code";
}

}  // extern "C"
