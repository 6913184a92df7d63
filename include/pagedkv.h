/*
 * pagedkv.h -- C ABI of a paged KV cache for single-query decode attention
 * on NVIDIA GB300 (sm_103a).
 *
 * Sources (web pages, cited by title and section):
 *   [vLLM-TGI] "Inside vLLM and TGI: Paging, Versioned Schedulers and
 *              Operations": sections "Block addresses and fragmentation
 *              arithmetic" and "Exact CPU block manager and copy-on-write".
 *   [VM-LLM]   "vLLM and PagedAttention: Virtual Memory for LLM Serving"
 *              (talk transcript, no headings: paragraphs on paging,
 *              sharing / copy-on-write and preemption).
 *   [CB-PA]    "Continuous Batching & PagedAttention: vLLM Memory
 *              Management Architecture": "Core PagedAttention Mechanics".
 *
 * Model.  Keys and values of all sequences live in one shared pool of
 * fixed-size physical blocks.  A sequence's block table lists, in logical
 * order, the physical block holding each run of b positions: position t is
 * in logical block t / b at offset t % b, and its physical block is
 * table[t / b] ([vLLM-TGI] "Block addresses ..."; [CB-PA]).  The flat slot
 * of a position is physical_block * b + offset.
 *
 * Cache layout (the pages leave it backend-specific; this library's choice):
 * two arrays, k_cache and v_cache, each [num_blocks][num_kv_heads][b][D],
 * row-major, element type pkv_cache.dtype.  One (block, KV head) page is a
 * contiguous b * D run, which the kernels move with 16-byte aligned bulk
 * copies.
 *
 * Ownership.  The caller owns every buffer.  All pointers in the GPU calls
 * below are DEVICE pointers unless stated; the library keeps them only for
 * the duration of the enqueued work and allocates no device memory.  Each
 * call enqueues its kernels on `stream` and returns without synchronising.
 * The only state the library keeps is one device error word per device
 * (see paged_get_device_error) and the small per-device set-up it does on
 * first use (kernel attributes, the error word's address).
 *
 * Errors.  Argument errors are found on the host, without synchronising:
 * the call returns a negative PKV_ERR_* code and enqueues nothing.  Errors
 * that depend on device-resident data (an out-of-range slot, table entry,
 * length or block pair) are found by the kernels, which never trap: the
 * offending item is skipped (attention rows are written as zeros) and a
 * PKV_DEV_* bit is OR-ed into the device error word.  After a device error
 * the caller should treat the pool as suspect.
 */
#ifndef PAGEDKV_H
#define PAGEDKV_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element type of the caches.  For PKV_F32 / PKV_F16 / PKV_BF16 pools, q,
 * out and the new keys/values have the same type.  PKV_FP8_E4M3 pools hold
 * 8-bit E4M3 codes (OCP FP8: bias 7, 3 mantissa bits, largest finite 448)
 * with one float scale per KV head for keys and one for values; q, out and
 * the new keys/values are then 16-bit (pkv_cache.io_dtype). */
typedef enum { PKV_F32 = 0, PKV_F16 = 1, PKV_BF16 = 2, PKV_FP8_E4M3 = 3 } pkv_dtype;

/* Host-side return codes. */
#define PKV_OK              0
#define PKV_ERR_NULL       -1  /* a required pointer is NULL                      */
#define PKV_ERR_GEOMETRY   -2  /* unsupported block size, head dim or group size  */
#define PKV_ERR_ARG        -3  /* bad count, length bound or partition size       */
#define PKV_ERR_ALIGN      -4  /* a buffer is not 16-byte aligned                 */
#define PKV_ERR_WORKSPACE  -5  /* workspace missing or too small                  */
#define PKV_ERR_CUDA       -6  /* a CUDA runtime call or launch failed            */
#define PKV_ERR_STATE      -7  /* block manager: unknown / duplicate sequence     */
#define PKV_ERR_NOMEM      -8  /* block manager: not enough free blocks, or host  */
                                   /* memory for its bookkeeping ran out              */
#define PKV_ERR_CAPACITY   -9  /* output table narrower than a sequence's table   */

/* Device error bits (paged_get_device_error). */
#define PKV_DEV_SLOT_RANGE   1u  /* paged_kv_write: slot >= num_blocks * b        */
#define PKV_DEV_TABLE_RANGE  2u  /* decode: a used table entry not in [0, N)      */
#define PKV_DEV_SEQ_LEN      4u  /* decode: length not in [1, max_seq_len]        */
#define PKV_DEV_PAIR_RANGE   8u  /* paged_block_copy: src or dst not in [0, N)    */
#define PKV_DEV_TIMEOUT     16u  /* a bounded wait for a bulk copy gave up        */
#define PKV_DEV_SHARING     32u  /* shared-prefix decode: a member's table or     */
                                 /* length disagrees with its group's prefix      */
#define PKV_DEV_LAUNCH      64u  /* a kernel found its shared memory not 1 KiB    */
                                 /* aligned and computed nothing                  */
/* After PKV_DEV_TIMEOUT the launch that set it may have ended with bulk
 * copies still in flight into its shared memory (the drain after a timeout
 * is itself bounded).  Treat the stream as failed: that launch's outputs,
 * and the results of any later launch on the same device, are suspect. */

/* The paged pool.  Supported geometry: block_size in {8, 16, 32, 64},
 * head_dim in {64, 128}.  k_cache / v_cache must be 16-byte aligned. */
typedef struct {
  void*   k_cache;       /* [num_blocks][num_kv_heads][block_size][head_dim] */
  void*   v_cache;       /* same shape and type as k_cache                   */
  int64_t num_blocks;    /* N: physical blocks in the pool                   */
  int32_t block_size;    /* b: token positions per block                     */
  int32_t num_kv_heads;  /* Hk                                               */
  int32_t head_dim;      /* D                                                */
  int32_t dtype;         /* a pkv_dtype                                      */
  /* FP8 pools only (ignored otherwise): */
  const float* k_scale;  /* device float[Hk]: key of head h = value(code) * k_scale[h] */
  const float* v_scale;  /* device float[Hk]: likewise for values            */
  int32_t io_dtype;      /* PKV_F16 or PKV_BF16: type of q, out, new k/v     */
} pkv_cache;

/*
 * paged_kv_write -- store each new token's key and value in its slot
 * (the "reshape_and_cache" step).
 *
 * Follows [VM-LLM] (paging paragraph: tokens fill the last block, a new
 * block is taken when it is full) and the append step of [vLLM-TGI]
 * "Exact CPU block manager and copy-on-write".  For every i in
 * [0, num_tokens) with slot = slot_mapping[i] >= 0:
 *     k_cache[slot / b][h][slot % b][:] = k[i][h][:]   for every KV head h
 *     v_cache[slot / b][h][slot % b][:] = v[i][h][:]
 * Elements are copied bit for bit.  For an FP8 pool the new elements (of
 * io_dtype, widened to float32) are stored as e4m3(x / scale[h]) with the
 * division in float32 (round to nearest), round-to-nearest-even and
 * saturation to +-448.  A negative slot marks padding and is
 * skipped silently; a slot >= num_blocks * b is skipped and sets
 * PKV_DEV_SLOT_RANGE.  Two tokens with the same slot race (last writer
 * undefined).
 *
 *   k, v          device, [num_tokens][num_kv_heads][head_dim], contiguous,
 *                 cache dtype (io_dtype for FP8 pools), 16-byte aligned
 *   slot_mapping  device, int64[num_tokens]
 */
int paged_kv_write(const pkv_cache* cache, const void* k, const void* v,
                   const int64_t* slot_mapping, int64_t num_tokens,
                   cudaStream_t stream);

/*
 * paged_attention_partition_size -- the partition length (in positions) a
 * decode call will use.  `requested` = 0 selects the library default:
 * 512 for 16- and 32-bit pools; for FP8 pools the longest of 2048, 1536,
 * 1024 and 512 for which num_seqs * num_kv_heads * ceil(max_seq_len /
 * length) reaches 8 thread blocks per SM of the current device.
 * Otherwise it must be a positive multiple of block_size no larger than
 * 8192 and is returned unchanged.  Returns a negative PKV_ERR_* on bad arguments.  The default
 * depends on (num_seqs, max_seq_len): size the workspace and call decode
 * with the same values.
 */
int32_t paged_attention_partition_size(const pkv_cache* cache, int32_t num_seqs,
                                       int32_t num_heads, int32_t max_seq_len,
                                       int32_t requested);

/*
 * paged_attention_workspace_bytes -- bytes of device workspace a decode
 * call with these arguments needs (0 when every sequence fits in one
 * partition).  Returns 0 and sets nothing on bad arguments; the decode
 * call itself reports them.
 *
 * Workspace layout (float32, P = ceil(max_seq_len / partition_size)):
 *   ml[num_seqs][num_heads][P]   as (m, l) float pairs: m = running maximum
 *                                of the partition's scores in base-2 units
 *                                (score * log2 e), l = sum of 2^(score - m)
 *   o [num_seqs][num_heads][P][head_dim], starting at the next 256-byte
 *                                boundary: the partition's normalised output
 */
size_t paged_attention_workspace_bytes(const pkv_cache* cache, int32_t num_seqs,
                                       int32_t num_heads, int32_t max_seq_len,
                                       int32_t partition_size);

/*
 * paged_attention_decode -- single-query attention of each sequence over
 * its cached keys and values, read through its block table.
 *
 * The method: [vLLM-TGI] opening section and "Block addresses ..." (kernels
 * read a sequence through its block table), [VM-LLM] paging paragraph (the
 * attention kernel reads through the mapping; token order is unchanged).
 * For sequence s, query head h and its KV head kh = h / (num_heads /
 * num_kv_heads) (query heads grouped contiguously), with L = seq_lens[s]
 * and K_t, V_t the rows of position t found through the table:
 *     z_t = scale * dot(q[s][h], K_t)                    t = 0 .. L-1
 *     out[s][h] = sum_t e^(z_t - max z) V_t / sum_t e^(z_t - max z)
 * accumulated in float32 and rounded once to the output type.  For FP8
 * pools K_t and V_t are the codes' values times the head's scales and q,
 * out are io_dtype.
 *
 * Long sequences are split into partitions of `partition_size` positions
 * processed by separate thread blocks; a second kernel merges them
 * (split-K).  Only the block-table entries covering positions < L are read.
 *
 *   q             device, [num_seqs][num_heads][head_dim], cache dtype
 *   block_tables  device, int32[num_seqs][max_blocks_per_seq]
 *   seq_lens      device, int32[num_seqs], positions to attend over
 *   max_seq_len   host bound on seq_lens (0 = max_blocks_per_seq * b); it
 *                 sizes the launch and the workspace
 *   scale         multiplies every score (typically 1 / sqrt(head_dim))
 *   out           device, [num_seqs][num_heads][head_dim], cache dtype
 *   workspace     device, >= paged_attention_workspace_bytes(...) bytes,
 *                 16-byte aligned; may be NULL when that is 0
 *   partition_size 0 = default, else a multiple of block_size <= 8192;
 *                 at most 65535 partitions (max_seq_len / partition_size)
 *   num_seqs      at most 65535
 *
 * num_heads must be num_kv_heads times 1, 2, 4 or 8.  A row whose length
 * is outside [1, max_seq_len] (PKV_DEV_SEQ_LEN) or whose used table
 * entries leave [0, num_blocks) (PKV_DEV_TABLE_RANGE) is written as zeros.
 */
int paged_attention_decode(const pkv_cache* cache, const void* q,
                           const int32_t* block_tables, int32_t max_blocks_per_seq,
                           const int32_t* seq_lens, int32_t num_seqs,
                           int32_t num_heads, int32_t max_seq_len, float scale,
                           void* out, void* workspace, size_t workspace_bytes,
                           int32_t partition_size, cudaStream_t stream);

/*
 * paged_attention_prefill -- causal attention of a chunk of new queries per
 * sequence through the block tables (prefill and chunked prefill).
 *
 * [VM-LLM] opening paragraph: in prefill all prompt tokens are known and
 * processed together; [vLLM-TGI] launch notes: chunked prefill splits long
 * prompts.  Sequence s holds L = seq_lens[s] positions, the last
 * Q = query_starts[s+1] - query_starts[s] of which are its new queries (their
 * keys and values already written, e.g. by paged_kv_write).  Query i of the
 * chunk sits at position L - Q + i and attends to positions 0 .. L - Q + i:
 *     out[query_starts[s] + i][h] = softmax-weighted mean, as in
 *     paged_attention_decode, over the first L - Q + i + 1 positions
 * accumulated in float32 on tensor cores.  fp16, bf16 and FP8 pools; FP8
 * pools with head_dim 128 only (others: PKV_ERR_GEOMETRY), their keys and
 * values being the codes' values times the head's scales, with q and out in
 * io_dtype.  PKV_PREFILL_KERNEL=mma in the environment selects the mma.sync
 * kernel (16-bit pools only).
 *
 *   q, out        device, [total_queries][num_heads][head_dim], cache dtype
 *                 (io_dtype for FP8 pools)
 *   query_starts  device, int32[num_seqs + 1], non-decreasing, last <=
 *                 total_queries
 *   max_queries   host bound on any sequence's Q (sizes the launch)
 *   block_tables, seq_lens, scale: as for paged_attention_decode
 *
 * A sequence whose Q exceeds its length or max_queries, or whose length
 * exceeds the table, gets zero rows and PKV_DEV_SEQ_LEN; one whose used
 * table entries leave [0, num_blocks) gets zero rows and
 * PKV_DEV_TABLE_RANGE.  max_blocks_per_seq is bounded by shared memory
 * (about 38k entries).
 */
int paged_attention_prefill(const pkv_cache* cache, const void* q, int64_t total_queries,
                            const int32_t* query_starts, int32_t num_seqs, int32_t max_queries,
                            const int32_t* block_tables, int32_t max_blocks_per_seq,
                            const int32_t* seq_lens, int32_t num_heads, float scale, void* out,
                            cudaStream_t stream);

/*
 * paged_attention_decode_shared -- paged_attention_decode for batches in
 * which groups of sequences share the first blocks of their tables (forks
 * of one prompt: parallel sampling, beam search).  [VM-LLM] sharing
 * paragraph: branches of one prompt share its KV blocks; [vLLM-TGI] "Exact
 * CPU block manager and copy-on-write": a fork shares every block of its
 * parent until a write needs a private copy.
 *
 * Same output as paged_attention_decode.  The partitions (of
 * partition_size positions) that lie wholly inside a group's shared prefix
 * are computed once per (group, KV head) for all members' queries
 * together, on the tensor cores, so each shared page is read once instead
 * of once per member; the rest of each sequence (its tail) is decoded by
 * the partition pass and merged with them.
 *
 *   group_starts   device int32[num_groups + 1]: group g is the sequences
 *                  group_starts[g] .. group_starts[g+1] - 1 (consecutive,
 *                  ascending).  Sequences outside every group are decoded
 *                  in full.
 *   group_prefix   device int32[num_groups]: positions 0 .. prefix - 1 of
 *                  every member are shared: each member's table names the
 *                  group's first member's blocks for them, and each
 *                  member's length is at least prefix.
 *   max_group_size host bound on group sizes (1 .. num_seqs).
 *   tail_parts     host hint for the partition pass.  0: its grid spans
 *                  every partition and the shared ones exit at once.
 *                  n > 0: its grid spans n partitions per sequence,
 *                  counted from the first partition after the sequence's
 *                  group's shared ones (from partition 0 for a sequence
 *                  outside every group); a sequence that needs more gets a
 *                  zero output row and sets PKV_DEV_SHARING.  With forks
 *                  whose tails fit in one partition, 1 computes each tail
 *                  and merges it with the shared partials in one small
 *                  pass per (sequence, KV head), in place of the partition
 *                  pass and the merge.
 *   workspace      as for paged_attention_decode (same size).
 *
 * A member whose table or length breaks its group's contract gets a zero
 * output row and sets PKV_DEV_SHARING.  Groups apply to fp16 and bf16
 * pools; other pools decode every sequence in full (the same attention).
 * num_groups = 0 is plain decode.  Host errors as for
 * paged_attention_decode, plus PKV_ERR_ARG for num_groups outside
 * [0, 65535], max_group_size outside [1, num_seqs] or tail_parts < 0,
 * PKV_ERR_NULL / PKV_ERR_ALIGN for the group arrays.
 */
int paged_attention_decode_shared(const pkv_cache* cache, const void* q,
                                  const int32_t* block_tables, int32_t max_blocks_per_seq,
                                  const int32_t* seq_lens, int32_t num_seqs, int32_t num_heads,
                                  int32_t max_seq_len, float scale, void* out,
                                  const int32_t* group_starts, const int32_t* group_prefix,
                                  int32_t num_groups, int32_t max_group_size,
                                  int32_t tail_parts, void* workspace, size_t workspace_bytes,
                                  int32_t partition_size, cudaStream_t stream);

/*
 * paged_attention_decode_static_ws -- paged_attention_decode without a
 * caller-supplied workspace.  The pages have no counterpart to this call; it
 * exists for callers that cannot allocate device memory themselves (a
 * plug-in inside a host program that owns and reserves GPU memory up front,
 * a latency-critical path where cudaMalloc may synchronise the device, a
 * plain C caller without a caching allocator).
 *
 * Same arguments, semantics and errors as paged_attention_decode, minus
 * `workspace` and `workspace_bytes`: the split-K scratch is one fixed device
 * array of PKV_STATIC_WS_BYTES bytes inside the library, held by every
 * device that loads it until the process exits.  The call allocates nothing
 * (no cudaMalloc, no cudaFree, no allocating library routine).
 *
 *   - A request whose scratch, as paged_attention_workspace_bytes would
 *     report it, exceeds PKV_STATIC_WS_BYTES returns PKV_ERR_WORKSPACE and
 *     enqueues nothing.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current) and caches it.  With
 *     lazy module loading that lookup is also when the 32 MiB are committed
 *     on the device, so make the first call before the host program reserves
 *     its device memory, and before any stream capture.  If the lookup
 *     fails the call returns PKV_ERR_CUDA and clears the runtime's error, so
 *     later calls are not affected.
 *   - All calls share the one array.  Calls whose kernels overlap on the GPU
 *     (different streams, no ordering between them) race on it and give
 *     wrong results; order them on one stream or with events.  Each call
 *     writes every scratch entry it reads, so nothing carries over between
 *     calls and nothing needs clearing.
 */
#define PKV_STATIC_WS_BYTES (32u << 20)
int paged_attention_decode_static_ws(const pkv_cache* cache, const void* q,
                                     const int32_t* block_tables, int32_t max_blocks_per_seq,
                                     const int32_t* seq_lens, int32_t num_seqs,
                                     int32_t num_heads, int32_t max_seq_len, float scale,
                                     void* out, int32_t partition_size, cudaStream_t stream);

/*
 * paged_block_copy -- copy whole blocks, keys and values, every KV head:
 *     block dst := block src   for each (src, dst) pair
 *
 * The copy half of copy-on-write: [vLLM-TGI] "Exact CPU block manager and
 * copy-on-write" (appending to a shared, partially filled last block takes
 * a fresh block and copies the old contents into it before the write) and
 * [VM-LLM] sharing paragraph (a private copy for the branch being
 * modified).  Enqueue it before the paged_kv_write that fills the new
 * block.  Pairs with src or dst outside [0, num_blocks) are skipped and set
 * PKV_DEV_PAIR_RANGE; src == dst is a no-op.  Destinations must be distinct
 * and must not appear as a source in the same call (the copies run
 * concurrently).
 *
 *   src_dst_pairs device, int64[num_pairs][2] as (src, dst)
 */
int paged_block_copy(const pkv_cache* cache, const int64_t* src_dst_pairs,
                     int64_t num_pairs, cudaStream_t stream);

/*
 * paged_block_swap -- move whole blocks between the device pool and a pool in
 * pinned host memory (keys and values, every KV head):
 *     PKV_SWAP_OUT:  host block dst := device block src
 *     PKV_SWAP_IN:   device block dst := host block src
 *
 * The swap alternative to recomputation when blocks run out: [VM-LLM]
 * preemption paragraph (KV data swapped into CPU memory and restored
 * later) and [vLLM-TGI] "Read the vLLM 0.11.0 scheduler..." (swapping costs
 * the cache bytes in both directions over the link).  Which sequences to
 * evict, and the tables that point at swapped-out blocks, are the caller's.
 *
 *   host_k, host_v  pinned (page-locked) or managed host memory,
 *                   [host_blocks][num_kv_heads][block_size][head_dim] of the
 *                   cache dtype, 16-byte aligned; the kernel reads or writes
 *                   them directly over the host link
 *   src_dst_pairs   device, int64[num_pairs][2] as (src, dst)
 *   direction       PKV_SWAP_OUT or PKV_SWAP_IN
 *
 * Pairs naming a block outside its pool are skipped and set
 * PKV_DEV_PAIR_RANGE.  Destinations must be distinct.  Host memory that is
 * neither page-locked nor managed returns PKV_ERR_ARG.  The host pool must
 * not be touched by the CPU until the stream has passed this call.
 */
#define PKV_SWAP_OUT 0
#define PKV_SWAP_IN  1
int paged_block_swap(const pkv_cache* cache, void* host_k, void* host_v, int64_t host_blocks,
                     const int64_t* src_dst_pairs, int64_t num_pairs, int32_t direction,
                     cudaStream_t stream);

/*
 * paged_get_device_error -- synchronise `stream`, then read and clear the
 * current device's error word (an OR of PKV_DEV_* bits; 0 = no error).
 * The word is shared by every stream on the device.
 */
int paged_get_device_error(cudaStream_t stream, uint32_t* bits);

/*
 * paged_selftest_wait_timeout -- exercises the failure path every kernel
 * shares.  The pages have no counterpart.  A one-warp kernel waits on a
 * barrier that nothing completes; after limit_ns nanoseconds of wall-clock
 * time (1 .. 10^9) the bounded wait gives up, sets PKV_DEV_TIMEOUT in the
 * device error word and returns, as any kernel's copy wait would.  Nothing
 * faults and the context stays usable.  PKV_ERR_ARG for a limit outside
 * the range.
 */
int paged_selftest_wait_timeout(uint64_t limit_ns, cudaStream_t stream);

/*
 * paged_selftest_read_stream -- reads every byte of a device buffer once
 * (16-byte non-caching loads over the whole GPU) and XOR-folds the words
 * into *sink.  The pages have no counterpart: it measures the read-only
 * streaming bandwidth that the decode kernels, which only read the pool,
 * are compared with.
 *
 *   buf    device, 16-byte aligned, `bytes` a multiple of 16 (else
 *          PKV_ERR_ALIGN); 0 bytes launches nothing (buf may be NULL)
 *   sink   device uint32; XOR-updated (its value has no meaning)
 */
int paged_selftest_read_stream(const void* buf, size_t bytes, uint32_t* sink, cudaStream_t stream);

/* Text for a PKV_ERR_* code. */
const char* paged_strerror(int code);

/* ---------------------------------------------------------------------
 * Host block manager: the allocator that decides block tables, slots and
 * copy-on-write pairs (host memory only; no GPU calls).
 *
 * It follows [vLLM-TGI] "Exact CPU block manager and copy-on-write":
 * admission takes ceil(len / b) blocks at once or fails with nothing
 * taken; fork shares every block of the parent and counts one more
 * reference; an append writes into the last block if it has room and is
 * not shared, takes a fresh block when the last is full, and when the last
 * is partial and shared takes a fresh block, records (old, fresh) for
 * paged_block_copy, drops one reference from the old block and repoints the
 * table; release drops one reference from every block and returns blocks
 * that reach zero to the free list.  Free-list policy (left open by the
 * pages): blocks are taken from the front of the list, the initial list is
 * `free_order` (NULL = 0..N-1), and freed blocks go back to the front.
 * Not thread-safe; sequences are named by caller-chosen int64 ids.  Every
 * call is all or nothing: one that fails (including for lack of host memory,
 * PKV_ERR_NOMEM) leaves the manager unchanged.
 * ------------------------------------------------------------------- */
typedef struct pkv_block_manager pkv_block_manager;

/* free_order: host, int64[num_blocks], a permutation of 0..num_blocks-1, or
 * NULL.  Returns NULL on bad arguments or host allocation failure. */
pkv_block_manager* pkv_bm_create(int64_t num_blocks, int32_t block_size,
                                 const int64_t* free_order);
void pkv_bm_destroy(pkv_block_manager* bm);

/* Admit sequence `seq` holding `num_tokens` (>= 1) positions. */
int pkv_bm_admit(pkv_block_manager* bm, int64_t seq, int64_t num_tokens);

/* Make `child` share every block of `parent`. */
int pkv_bm_fork(pkv_block_manager* bm, int64_t parent, int64_t child);

/* One decode step: append one position to each of seqs[0..n-1], in order.
 * Writes slot_mapping[i] (host, int64[n]) and the copy-on-write pairs the
 * step needs (host, int64[n][2] capacity) with their count.  All or
 * nothing: if the free list cannot cover every growth and copy of the step,
 * returns PKV_ERR_NOMEM and changes nothing. */
int pkv_bm_append(pkv_block_manager* bm, const int64_t* seqs, int64_t n,
                  int64_t* slot_mapping, int64_t* pairs, int64_t* num_pairs);

/* Drop the sequence and one reference from each of its blocks. */
int pkv_bm_release(pkv_block_manager* bm, int64_t seq);

/* Export tables (host, int32[n][max_blocks], padded with -1) and lengths
 * (host, int32[n]) of seqs[0..n-1].  PKV_ERR_CAPACITY if a table is wider
 * than max_blocks. */
int pkv_bm_tables(const pkv_block_manager* bm, const int64_t* seqs, int64_t n,
                  int32_t max_blocks, int32_t* tables, int32_t* seq_lens);

/* Slots of positions start .. start+count-1 of `seq` (host, int64[count]),
 * e.g. the slot mapping of a prefill chunk.  PKV_ERR_ARG if the range is not
 * inside the sequence. */
int pkv_bm_slots(const pkv_block_manager* bm, int64_t seq, int64_t start, int64_t count,
                 int64_t* slot_mapping);

int64_t pkv_bm_num_free(const pkv_block_manager* bm);
int64_t pkv_bm_seq_len(const pkv_block_manager* bm, int64_t seq);     /* -1 if unknown */
int64_t pkv_bm_num_seq_blocks(const pkv_block_manager* bm, int64_t seq); /* -1 if unknown */
int32_t pkv_bm_refcount(const pkv_block_manager* bm, int64_t block);   /* -1 if out of range */

/* Check the pool invariants: each count equals the table entries naming
 * the block, the free list is duplicate-free and equals the blocks with
 * count 0, every non-last block is full and the last holds 1..b positions.
 * PKV_OK or PKV_ERR_STATE. */
int pkv_bm_check(const pkv_block_manager* bm);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDKV_H */
