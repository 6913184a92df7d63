// Paged single-query decode attention for sm_103a: partition pass + merge.
//
// The method: "Inside vLLM and TGI: Paging, Versioned Schedulers and
// Operations" (opening section; "Block addresses and fragmentation
// arithmetic") -- a kernel reads each sequence through its block table,
// position t living at offset t % b of physical block table[t / b]; "vLLM
// and PagedAttention: Virtual Memory for LLM Serving" (paging paragraph) --
// the attention kernel reads through the mapping and token order is
// unchanged.  What is computed is ordinary softmax attention of one query
// over the sequence's cached keys and values.
//
// Work decomposition (this library's design):
//   grid = (partition, KV head, sequence), 4 warps per CTA.  A partition is
//   `part_size` consecutive positions (a multiple of b).  The CTA stages the
//   partition's table entries in shared memory, checks them, and processes
//   the G = H / Hk query heads that share the KV head, so each K/V page is
//   read from HBM once for the whole group.
//
//   The partition is cut into chunks of C = min(b, 8) positions; chunk j
//   goes to warp j % 4.  Each warp owns a ring of kStages shared-memory
//   stages; lane 0 fills a stage with two 1-D bulk copies (the chunk's keys
//   and values for this head: C * D contiguous elements each, because the
//   cache is [N][Hk][b][D]) that complete on the stage's mbarrier, and keeps
//   kStages chunks in flight ahead of the warp's computation.
//
//   Lane l owns elements [l * D/32, (l+1) * D/32) of every row.  For QK it
//   accumulates C partial dot products per query head; a butterfly
//   reduce-scatter over the warp turns them into full scores, one position
//   per group of 32 / C lanes.  The online softmax runs in base 2 (scores
//   pre-multiplied by scale * log2 e): running maximum m, running sum l,
//   unnormalised output acc, rescaled by 2^(m_old - m_new) when the maximum
//   grows.  For PV the probabilities are broadcast back (shuffle, or a small
//   shared buffer for G > 1) and each lane updates its own output elements.
//   Positions past the sequence end inside the last chunk get probability 0
//   and their value rows are never touched.
//
//   The four warps' (m, l, acc) are merged in shared memory.  A sequence
//   covered by one partition writes its output directly; otherwise each
//   partition writes (m, l) and its normalised output to the workspace and
//   decode_reduce_kernel merges them: M = max_p m_p, w_p = l_p 2^(m_p - M),
//   out = sum_p w_p o_p / sum_p w_p.
//
//   Every reduction order depends only on logical positions, never on
//   physical block ids, so relabelling the pool leaves results bit-identical.
#pragma once

#include <atomic>
#include <cmath>
#include <type_traits>

#include "common.cuh"

namespace pkv {

struct DecodeParams {
  const void* k_cache;
  const void* v_cache;
  int64_t num_blocks;
  int kv_heads;
  int num_heads;
  const void* q;
  void* out;
  const int32_t* tables;
  int max_blocks;
  const int32_t* seq_lens;
  int max_len;       // lengths above this (or above max_blocks * b) are invalid
  float qscale;      // scale * log2(e)
  int part_size;     // positions per partition, a multiple of b
  int num_parts;     // partitions per sequence in the grid (>= ceil(L / part_size))
  float2* ws_ml;     // [S][H][num_parts] (m, l), used when num_parts > 1
  float* ws_o;       // [S][H][num_parts][D]
  unsigned* err;
  const float* k_scale;  // FP8 pools: per-KV-head scales (else unused)
  const float* v_scale;
  // Shared-prefix decode (null otherwise): groups of consecutive sequences
  // [group_starts[g], group_starts[g+1]) whose first group_prefix[g]
  // positions are shared; the partitions inside that prefix are computed by
  // decode_shared_prefix_kernel, and the partition pass skips them.
  const int32_t* group_starts;
  const int32_t* group_prefix;
  int num_groups;
  int num_seqs;
  // Partition pass of the shared-prefix decode: 0, slice z is partition z
  // (the shared ones exit); tail_parts > 1, the grid has tail_parts slices
  // and slice z is the z-th partition after the sequence's shared ones;
  // 1, decode_tail_merge_kernel replaces the partition pass and the merge.
  int tail_parts;
};

// Group owning sequence s, or -1: the last g with group_starts[g] <= s
// (for a nondecreasing list, the group whose range holds s), provided
// s < group_starts[g+1].  The search is 32-way: each round issues its
// probes together, so a list of up to 32 groups costs one round of loads
// (a binary search would cost one dependent load per halving, and every
// CTA of the partition pass asks).  It is a fixed function of the list, and
// the shared-prefix kernel and the partition pass both call it, so a
// malformed list can leave a sequence without a group (decoded plainly) but
// never covered twice.
__device__ __forceinline__ int shared_owner(const DecodeParams& p, int s) {
  if (!p.group_starts || p.num_groups <= 0) return -1;
  const int32_t* gs = p.group_starts;
  int lo = 0, cnt = p.num_groups;  // candidates lo .. lo + cnt - 1; lo + cnt <= num_groups
  while (cnt > 32) {
    const int step = (cnt + 31) / 32;
    int best = 0;
#pragma unroll
    for (int i = 1; i < 32; ++i) {
      const int off = i * step;
      if (off < cnt && ld_nc(gs + lo + off) <= s) best = i;
    }
    lo += best * step;
    cnt = min(step, cnt - best * step);
  }
  // Last round: entries lo .. lo + cnt (each candidate's start and the end
  // of the last one).
  int v[33];
#pragma unroll
  for (int i = 0; i < 33; ++i) v[i] = i <= cnt ? ld_nc(gs + lo + i) : 0;
  int a = v[0], b = v[1], g = 0;
#pragma unroll
  for (int i = 1; i < 32; ++i)
    if (i < cnt && v[i] <= s) {
      g = i;
      a = v[i];
      b = v[i + 1];
    }
  return (a <= s && s < b) ? lo + g : -1;
}

// shared_owner for a sequence s that every lane of the warp asks about: the
// same function, with the last round's probes spread over the lanes (one
// load each, a ballot) when the list has at most 32 groups.
__device__ __forceinline__ int shared_owner_warp(const DecodeParams& p, int s) {
  if (!p.group_starts || p.num_groups <= 0) return -1;
  if (p.num_groups > 32) return shared_owner(p, s);
  const int lane = threadIdx.x & 31, n = p.num_groups;
  const int v = lane <= n ? ld_nc(p.group_starts + lane) : 0;  // entries 0 .. n (n <= 32)
  const int v32 = n == 32 ? ld_nc(p.group_starts + 32) : 0;
  const unsigned hit = __ballot_sync(kFullMask, lane >= 1 && lane < n && v <= s);
  const int g = hit ? 31 - __clz(hit) : 0;  // the last candidate with its start <= s
  const int a = __shfl_sync(kFullMask, v, g);
  const int b = g + 1 == 32 ? v32 : __shfl_sync(kFullMask, v, (g + 1) & 31);
  return (a <= s && s < b) ? g : -1;
}

// Partitions of sequence s that the shared-prefix kernel computes (at most
// the grid's partitions); s is the same for every lane of the warp.
__device__ __forceinline__ int shared_parts_of(const DecodeParams& p, int s) {
  const int g = shared_owner_warp(p, s);
  if (g < 0) return 0;
  const int pre = ld_nc(p.group_prefix + g);
  return pre > 0 ? min(pre / p.part_size, p.num_parts) : 0;
}

constexpr int kMaxPartSize = 8192;

constexpr int cmin(int a, int b) { return a < b ? a : b; }
constexpr int cmax(int a, int b) { return a > b ? a : b; }
constexpr int clog2(int x) { return x <= 1 ? 0 : 1 + clog2(x / 2); }

template <typename T, int D, int BS, int G, typename TC = T>
struct DecodeCfg {
  // Shape chosen by measurement on GB300: small rings (two 8-position stages
  // per warp, 32 KiB per CTA) let up to 7 CTAs share an SM, and the extra
  // resident warps hide each CTA's set-up latency; deeper rings with fewer
  // CTAs per SM stream less.
  static constexpr int kWarps = 4;
  static constexpr int kThreads = kWarps * 32;
  static constexpr int kChunk = cmin(BS, 8);                // positions per stage
  static constexpr int kChunksPerBlock = BS / kChunk;
  static constexpr int kLanesPerPos = 32 / kChunk;          // after the reduce-scatter
  static constexpr int kShift = clog2(kLanesPerPos);
  static constexpr int kDpl = D / 32;                       // elements per lane
  static constexpr int kChunkBytes = kChunk * D * (int)sizeof(TC);
  static constexpr int kStageBytes = 2 * kChunkBytes;       // keys + values
  static constexpr int kRingBudget = 32 * 1024;
  static constexpr int kStages = cmax(2, cmin(8, kRingBudget / (kWarps * kStageBytes)));
  static constexpr int kRingBytes = kWarps * kStages * kStageBytes;
  static constexpr int kBarOff = kRingBytes;
  static constexpr int kPbufOff = kBarOff + kWarps * kStages * 8;
  static constexpr int kTableOff = kPbufOff + kWarps * kChunk * G * 4;
  // Merge scratch (aliases the ring once every warp is done with it).
  static constexpr int kMergeBytes = (kWarps * G * D + 3 * kWarps * G + 2 * G) * 4;
  static_assert(kMergeBytes <= kRingBytes, "merge scratch must fit in the ring");
  static_assert(D % 32 == 0 && kChunkBytes % 16 == 0, "bulk copy granularity");
  static constexpr int smem_bytes(int part_size) { return kTableOff + (part_size / BS) * 4; }
  static constexpr int kMaxSmem = kTableOff + (kMaxPartSize / BS) * 4;
};

// Sums C per-lane partial values over the warp.  On return lane l holds the
// full sum of value number (l >> log2(32 / C)).  Each halving round trades
// half of the remaining values with the partner lane at distance `off`.
template <int C>
__device__ __forceinline__ float reduce_scatter(float (&v)[C], int lane) {
#pragma unroll
  for (int r = 0; (C >> r) > 1; ++r) {
    const int n = C >> r;
    const int off = 16 >> r;
    const bool upper = (lane & off) != 0;
#pragma unroll
    for (int i = 0; i < n / 2; ++i) {
      const float send = upper ? v[i] : v[i + n / 2];
      const float keep = upper ? v[i + n / 2] : v[i];
      v[i] = keep + __shfl_xor_sync(kFullMask, send, off);
    }
  }
  float x = v[0];
#pragma unroll
  for (int off = 16 / C; off >= 1; off >>= 1) x += __shfl_xor_sync(kFullMask, x, off);
  return x;
}

// T: type of q and out; TC: type of the cache elements (T itself, or FP8
// E4M3 codes whose per-head scales are folded into the query and the
// output).
template <typename T, int D, int BS, int G, typename TC = T>
__global__ void __launch_bounds__(DecodeCfg<T, D, BS, G, TC>::kThreads)
decode_partition_kernel(const DecodeParams p) {
  using Cfg = DecodeCfg<T, D, BS, G, TC>;
  constexpr bool kScaled = !std::is_same<T, TC>::value;
  constexpr int C = Cfg::kChunk;
  constexpr int NW = Cfg::kWarps;
  constexpr int NST = Cfg::kStages;
  constexpr int DPL = Cfg::kDpl;
  constexpr int CPB = Cfg::kChunksPerBlock;
  constexpr int SH = Cfg::kShift;
  extern __shared__ __align__(128) unsigned char smem[];

  // Partition is the slowest grid dimension: every sequence's first
  // partition is dispatched before any second one, so the CTAs of partitions
  // past a sequence's end (which exit at once) gather at the end of the grid.
  const int kvh = blockIdx.x;
  const int s = blockIdx.y;
  const int z = blockIdx.z;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int H = p.num_heads;
  T* out = static_cast<T*>(p.out);
  const int64_t out0 = ((int64_t)s * H + (int64_t)kvh * G) * D;  // out[s][kvh*G][0]
  const int PS = p.part_size;
  // The length, and with a tail grid (tail_parts > 0: slice z is the z-th
  // partition after the sequence's shared ones) the sequence's group, are
  // loaded first; otherwise slice z is partition z, and the length and this
  // partition's table entries are loaded together (the entries
  // speculatively, but never past the table row), so a CTA waits for one
  // global round trip before it can issue its first bulk copy.
  const int L = ld_nc(p.seq_lens + s);
  const bool tail_grid = p.tail_parts > 0;
  int shared_parts = tail_grid ? shared_parts_of(p, s) : 0;
  const int part = z + shared_parts;
  const int tok0 = part * PS;
  const int blk0 = tok0 / BS;
  const int32_t* trow = p.tables + (int64_t)s * p.max_blocks + blk0;
  const int span = min(PS / BS, p.max_blocks - blk0);
  const int e_first = (int)threadIdx.x < span ? ld_nc(trow + threadIdx.x) : -1;
  if (!tail_grid) shared_parts = shared_parts_of(p, s);  // loads issued with the two above

  if (L < 1 || L > p.max_len) {
    if (z == 0) {
      for (int e = threadIdx.x; e < G * D; e += Cfg::kThreads) out[out0 + e] = Elem<T>::from_f(0.f);
      if (threadIdx.x == 0) set_error(p.err, PKV_DEV_SEQ_LEN);
    }
    return;
  }
  if (tok0 >= L) return;
  // Partitions inside a shared prefix are the shared-prefix kernel's.
  if (part < shared_parts) return;
  const int ntok = min(L - tok0, PS);
  const int nparts = (L + PS - 1) / PS;
  if (tail_grid && z == p.tail_parts - 1 && part + 1 < nparts) {
    // The sequence needs partitions past the tail grid: their slots get the
    // invalid marker (nobody else writes them), so the merge zeroes its rows.
    if (threadIdx.x == 0) set_error(p.err, PKV_DEV_SHARING);
    for (int i = threadIdx.x; i < G * (nparts - part - 1); i += Cfg::kThreads)
      p.ws_ml[((int64_t)s * H + (int64_t)kvh * G + i % G) * p.num_parts + part + 1 + i / G] =
          make_float2(-INFINITY, -1.f);
  }
  const int nblk = (ntok + BS - 1) / BS;
  const int nchunks = (ntok + C - 1) / C;

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Cfg::kBarOff);
  float* pbuf = reinterpret_cast<float*>(smem + Cfg::kPbufOff);
  int* stable = reinterpret_cast<int*>(smem + Cfg::kTableOff);

  if (lane == 0) {
#pragma unroll
    for (int st = 0; st < NST; ++st) mbar_init(smem_addr(&bars[warp * NST + st]), 1);
    fence_mbar_init();
  }
  int bad = 0;
  if ((int)threadIdx.x < nblk) {
    bad = (e_first < 0 || (int64_t)e_first >= p.num_blocks);
    stable[threadIdx.x] = e_first;
  }
  for (int i = threadIdx.x + Cfg::kThreads; i < nblk; i += Cfg::kThreads) {
    const int e = trow[i];
    bad |= (e < 0 || (int64_t)e >= p.num_blocks);
    stable[i] = e;
  }
  bad = __syncthreads_or(bad);
  // Workspace row of (s, head kvh*G, this partition); head kvh*G+g adds g*P.
  const int64_t ws0 = ((int64_t)s * H + (int64_t)kvh * G) * p.num_parts + part;
  if (bad) {
    if (threadIdx.x == 0) set_error(p.err, PKV_DEV_TABLE_RANGE);
    if (nparts == 1) {
      for (int e = threadIdx.x; e < G * D; e += Cfg::kThreads) out[out0 + e] = Elem<T>::from_f(0.f);
    } else if (threadIdx.x < G) {
      p.ws_ml[ws0 + (int64_t)threadIdx.x * p.num_parts] = make_float2(-INFINITY, -1.f);
    }
    return;
  }

  const int count = warp < nchunks ? (nchunks - warp + NW - 1) / NW : 0;
  const char* kbase = static_cast<const char*>(p.k_cache);
  const char* vbase = static_cast<const char*>(p.v_cache);
  const uint32_t ring0 = smem_addr(smem) + warp * NST * Cfg::kStageBytes;
  const uint32_t bar0 = smem_addr(&bars[warp * NST]);
  const uint64_t policy = policy_evict_first();

  auto issue = [&](int j) {
    const int c = warp + j * NW;
    const int st = j % NST;
    const int pb = stable[c / CPB];
    const int64_t row = ((int64_t)pb * p.kv_heads + kvh) * BS + (c % CPB) * C;
    const int64_t off = row * D * (int64_t)sizeof(TC);  // bytes: cache element size
    const uint32_t bar = bar0 + st * 8;
    const uint32_t dst = ring0 + st * Cfg::kStageBytes;
    mbar_arrive_expect_tx(bar, Cfg::kStageBytes);
    bulk_g2s(dst, kbase + off, Cfg::kChunkBytes, bar, policy);
    bulk_g2s(dst + Cfg::kChunkBytes, vbase + off, Cfg::kChunkBytes, bar, policy);
  };
  if (lane == 0) {
    const int pre = count < NST ? count : NST;
    for (int j = 0; j < pre; ++j) issue(j);
  }

  // Query rows of the group, pre-scaled into base-2 score units (loaded while
  // the first copies are in flight); an FP8 key scale folds in here.
  float qv[G][DPL];
  {
    float qs = p.qscale;
    if constexpr (kScaled) qs *= p.k_scale[kvh];
    const T* qp = static_cast<const T*>(p.q) + out0 + lane * DPL;
#pragma unroll
    for (int g = 0; g < G; ++g) {
      RowLoad<T, DPL>::load(qp + g * D, qv[g]);
#pragma unroll
      for (int d = 0; d < DPL; ++d) qv[g][d] *= qs;
    }
  }

  float m[G], l[G], acc[G][DPL];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    m[g] = -INFINITY;
    l[g] = 0.f;
#pragma unroll
    for (int d = 0; d < DPL; ++d) acc[g][d] = 0.f;
  }
  bool timed_out = false;
  const int tok = lane >> SH;  // position (within the chunk) whose score this lane holds
  float* pw = pbuf + warp * C * G;

  int j = 0;
  for (; j < count; ++j) {
    const int st = j % NST;
    // Warp-uniform decision: every lane leaves together if any lane gave up.
    timed_out = __any_sync(kFullMask, !mbar_wait(bar0 + st * 8, (uint32_t)((j / NST) & 1)));
    if (timed_out) break;
    const int c = warp + j * NW;
    const int nvalid = min(C, ntok - c * C);
    const TC* ks = reinterpret_cast<const TC*>(smem + (warp * NST + st) * Cfg::kStageBytes);
    const TC* vs = ks + C * D;

    // ---- scores ------------------------------------------------------
    float sc[G];
    {
      float part_dot[G][C];
#pragma unroll
      for (int t = 0; t < C; ++t) {
        float kf[DPL];
        CacheRow<TC, DPL>::load(ks + t * D + lane * DPL, kf);
#pragma unroll
        for (int g = 0; g < G; ++g) {
          float a = 0.f;
#pragma unroll
          for (int d = 0; d < DPL; ++d) a = fmaf(qv[g][d], kf[d], a);
          part_dot[g][t] = a;
        }
      }
#pragma unroll
      for (int g = 0; g < G; ++g) sc[g] = reduce_scatter<C>(part_dot[g], lane);
    }

    // ---- online softmax ----------------------------------------------
    const bool valid = tok < nvalid;
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float x = valid ? sc[g] : -INFINITY;
      float cm = x;
#pragma unroll
      for (int off = 16; off >= (1 << SH); off >>= 1) cm = fmaxf(cm, __shfl_xor_sync(kFullMask, cm, off));
      const float mnew = fmaxf(m[g], cm);
      const float alpha = exp2f(m[g] - mnew);
      const float pe = valid ? exp2f(x - mnew) : 0.f;
      float cs = pe;
#pragma unroll
      for (int off = 16; off >= (1 << SH); off >>= 1) cs += __shfl_xor_sync(kFullMask, cs, off);
      l[g] = l[g] * alpha + cs;
      m[g] = mnew;
#pragma unroll
      for (int d = 0; d < DPL; ++d) acc[g][d] *= alpha;
      sc[g] = pe;
    }

    // ---- probabilities x values --------------------------------------
    if constexpr (G == 1) {
#pragma unroll
      for (int t = 0; t < C; ++t) {
        if (t < nvalid) {
          const float pt = __shfl_sync(kFullMask, sc[0], t << SH);
          float vf[DPL];
          CacheRow<TC, DPL>::load(vs + t * D + lane * DPL, vf);
#pragma unroll
          for (int d = 0; d < DPL; ++d) acc[0][d] = fmaf(pt, vf[d], acc[0][d]);
        }
      }
    } else {
      if ((lane & ((1 << SH) - 1)) == 0) {
#pragma unroll
        for (int g = 0; g < G; ++g) pw[tok * G + g] = sc[g];
      }
      __syncwarp();
#pragma unroll
      for (int t = 0; t < C; ++t) {
        if (t < nvalid) {
          float pt[G];
          if constexpr (G == 2) {
            const float2 v2 = *reinterpret_cast<const float2*>(pw + t * G);
            pt[0] = v2.x; pt[1] = v2.y;
          } else {
#pragma unroll
            for (int g = 0; g < G; g += 4) {  // G is 4 or 8: 16-byte broadcast reads
              const float4 v4 = *reinterpret_cast<const float4*>(pw + t * G + g);
              pt[g] = v4.x; pt[g + 1] = v4.y; pt[g + 2] = v4.z; pt[g + 3] = v4.w;
            }
          }
          float vf[DPL];
          CacheRow<TC, DPL>::load(vs + t * D + lane * DPL, vf);
#pragma unroll
          for (int g = 0; g < G; ++g)
#pragma unroll
            for (int d = 0; d < DPL; ++d) acc[g][d] = fmaf(pt[g], vf[d], acc[g][d]);
        }
      }
    }

    __syncwarp();
    if (lane == 0 && j + NST < count) {
      fence_proxy_async();
      issue(j + NST);
    }
  }
  if (timed_out) {
    // Give the copies already issued for later stages a short, bounded
    // chance to land before this CTA's shared memory is reused.
    const int last = count < j + NST ? count : j + NST;
    for (int jj = j + 1; jj < last; ++jj)
      mbar_wait(bar0 + (jj % NST) * 8, (uint32_t)((jj / NST) & 1), kWaitLimitNs / 8);
    if (lane == 0) set_error(p.err, PKV_DEV_TIMEOUT);
  }

  // ---- merge the four warps --------------------------------------------
  __syncthreads();
  float* red_acc = reinterpret_cast<float*>(smem);      // [NW][G][D]
  float* red_m = red_acc + NW * G * D;                  // [NW][G]
  float* red_l = red_m + NW * G;                        // [NW][G]
  float* fac = red_l + NW * G;                          // [NW][G]
  float* fin = fac + NW * G;                            // [G] max, [G] sum
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int d = 0; d < DPL; ++d) red_acc[(warp * G + g) * D + lane * DPL + d] = acc[g][d];
  if (lane == 0) {
#pragma unroll
    for (int g = 0; g < G; ++g) {
      red_m[warp * G + g] = m[g];
      red_l[warp * G + g] = l[g];
    }
  }
  __syncthreads();
  if (threadIdx.x < G) {
    const int g = threadIdx.x;
    float big = -INFINITY;
#pragma unroll
    for (int w = 0; w < NW; ++w) big = fmaxf(big, red_m[w * G + g]);
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const float f = exp2f(red_m[w * G + g] - big);  // 0 for a warp that saw no chunk
      fac[w * G + g] = f;
      tot += red_l[w * G + g] * f;
    }
    fin[g] = big;
    fin[G + g] = tot;
  }
  __syncthreads();
  float vscale = 1.f;
  if constexpr (kScaled) vscale = p.v_scale[kvh];  // FP8 value scale, applied once
  for (int e = threadIdx.x; e < G * D; e += Cfg::kThreads) {
    const int g = e / D;
    const int d = e - g * D;
    float o = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) o = fmaf(red_acc[(w * G + g) * D + d], fac[w * G + g], o);
    o = o / fin[G + g];
    if constexpr (kScaled) o *= vscale;
    if (nparts == 1)
      out[out0 + e] = Elem<T>::from_f(o);
    else
      p.ws_o[(ws0 + (int64_t)g * p.num_parts) * D + d] = o;
  }
  if (nparts > 1 && threadIdx.x < G)
    p.ws_ml[ws0 + (int64_t)threadIdx.x * p.num_parts] = make_float2(fin[threadIdx.x], fin[G + threadIdx.x]);
}

// Merges the partitions of every (sequence, query head) whose sequence needed
// more than one.  A CTA of 4 warps covers 4 / WPH heads of one sequence with
// WPH warps per head: every warp reads all (m, l) pairs of its head to find
// the common maximum M (they are few), then the head's warps accumulate its
// partitions round-robin with loads issued four at a time and their partial
// sums meet in shared memory.  WPH = 1 suits a handful of partitions, WPH = 4
// long contexts with dozens.
constexpr int kReduceWarps = 4;

template <typename T, int D, int WPH>
__global__ void __launch_bounds__(kReduceWarps * 32) decode_reduce_kernel(const DecodeParams p) {
  constexpr int DPL = D / 32;
  constexpr int NW = kReduceWarps;
  __shared__ float part_acc[NW][D];
  __shared__ float part_tot[NW];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int sub = warp % WPH;
  const int h = blockIdx.x * (NW / WPH) + warp / WPH;
  const int s = blockIdx.y;
  const int L = p.seq_lens[s];
  if (L < 1 || L > p.max_len) return;  // the partition pass wrote zeros
  const int nparts = (L + p.part_size - 1) / p.part_size;
  if (nparts <= 1) return;  // the partition pass wrote the output
  const bool live = h < p.num_heads;
  const int64_t row = ((int64_t)s * p.num_heads + (live ? h : 0)) * p.num_parts;
  const float2* ml = p.ws_ml + row;
  float big = -INFINITY;
  bool bad = false;
  for (int i = lane; live && i < nparts; i += 32) {
    const float2 v = ml[i];
    bad |= v.y < 0.f;
    big = fmaxf(big, v.x);
  }
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) big = fmaxf(big, __shfl_xor_sync(kFullMask, big, off));
  bad = __any_sync(kFullMask, bad);
  float acc[DPL];
#pragma unroll
  for (int d = 0; d < DPL; ++d) acc[d] = 0.f;
  float tot = 0.f;
  const float* o = p.ws_o + row * D + lane * DPL;
  int i = sub;
  for (; live && !bad && i + 3 * WPH < nparts; i += 4 * WPH) {
    float2 v[4];
    float of[4][DPL];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      v[u] = ml[i + u * WPH];
      RowLoad<float, DPL>::load(o + (int64_t)(i + u * WPH) * D, of[u]);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const float w = v[u].y * exp2f(v[u].x - big);
      tot += w;
#pragma unroll
      for (int d = 0; d < DPL; ++d) acc[d] = fmaf(w, of[u][d], acc[d]);
    }
  }
  for (; live && !bad && i < nparts; i += WPH) {
    const float2 v = ml[i];
    const float w = v.y * exp2f(v.x - big);
    tot += w;
    float of[DPL];
    RowLoad<float, DPL>::load(o + (int64_t)i * D, of);
#pragma unroll
    for (int d = 0; d < DPL; ++d) acc[d] = fmaf(w, of[d], acc[d]);
  }
  if constexpr (WPH > 1) {
#pragma unroll
    for (int d = 0; d < DPL; ++d) part_acc[warp][lane * DPL + d] = acc[d];
    if (lane == 0) part_tot[warp] = tot;
    __syncthreads();
    if (sub == 0) {
#pragma unroll
      for (int w = 1; w < WPH; ++w) tot += part_tot[warp + w];
#pragma unroll
      for (int d = 0; d < DPL; ++d)
#pragma unroll
        for (int w = 1; w < WPH; ++w) acc[d] += part_acc[warp + w][lane * DPL + d];
    }
  }
  if (!live || sub != 0) return;
  T* out = static_cast<T*>(p.out) + ((int64_t)s * p.num_heads + h) * D + lane * DPL;
#pragma unroll
  for (int d = 0; d < DPL; ++d)
    out[d] = Elem<T>::from_f(bad ? 0.f : acc[d] / tot);  // a bad partition zeroes the row
}

}  // namespace pkv
