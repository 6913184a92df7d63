// paged_attention_decode_static_ws: decode attention whose split-K scratch is
// a fixed array inside this library, so the caller allocates nothing.
//
// Some callers cannot allocate device memory on their own: a plug-in running
// inside a host program that owns GPU memory and reserves nearly all of it up
// front (a serving engine that hands most of HBM to its KV pool leaves no
// headroom for ad-hoc buffers), code on a latency-critical path where
// cudaMalloc may synchronise the device, and plain C callers without a
// caching allocator.  For them this entry point takes the same inputs and
// output as paged_attention_decode but supplies the workspace itself.
#include <mutex>

#include "../../include/pagedkv.h"

// The scratch.  Every device that loads this part of the library holds these
// bytes until the process exits.  In host code the name is only a host-side
// stand-in for the symbol; the device address comes from
// cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_pkv_static_ws[PKV_STATIC_WS_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_static_mu;
void* g_static_ptr[kMaxDevices] = {};

// Device address of the scratch on the current device, looked up once per
// device (on that device's first call) and cached.
void* static_ws_address() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    (void)cudaGetLastError();
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_static_mu);
  if (!g_static_ptr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_pkv_static_ws) != cudaSuccess || !ptr) {
      // Clear the runtime's last error: the launchers judge their own
      // launches with cudaPeekAtLastError and must not see this one.
      (void)cudaGetLastError();
      return nullptr;
    }
    g_static_ptr[dev] = ptr;
  }
  return g_static_ptr[dev];
}

}  // namespace

extern "C" int paged_attention_decode_static_ws(const pkv_cache* cache, const void* q,
                                                const int32_t* block_tables,
                                                int32_t max_blocks_per_seq,
                                                const int32_t* seq_lens, int32_t num_seqs,
                                                int32_t num_heads, int32_t max_seq_len,
                                                float scale, void* out, int32_t partition_size,
                                                cudaStream_t stream) {
  if (!cache) return PKV_ERR_NULL;
  int64_t bound = max_seq_len;
  if (bound == 0) bound = (int64_t)max_blocks_per_seq * cache->block_size;
  size_t need = 0;
  if (bound >= 1 && bound <= INT32_MAX)
    need = paged_attention_workspace_bytes(cache, num_seqs, num_heads, (int32_t)bound,
                                           partition_size);
  // Requests whose split-K scratch exceeds the fixed array are refused
  // before anything is enqueued.
  if (need > (size_t)PKV_STATIC_WS_BYTES) return PKV_ERR_WORKSPACE;
  void* ws = nullptr;
  if (need > 0) {
    ws = static_ws_address();
    if (!ws) return PKV_ERR_CUDA;
  }
  // Every workspace entry the merge reads is written earlier in the same
  // call, so the previous call's contents never matter and nothing is
  // cleared.
  return paged_attention_decode(cache, q, block_tables, max_blocks_per_seq, seq_lens, num_seqs,
                                num_heads, max_seq_len, scale, out, ws,
                                ws ? (size_t)PKV_STATIC_WS_BYTES : 0, partition_size, stream);
}
