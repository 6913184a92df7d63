// Paged causal prefill attention on the fifth-generation tensor cores
// (tcgen05, accumulators in tensor memory), fp16 / bf16 pools and FP8 E4M3
// pools (head_dim 128).
//
// Same operation as prefill_mma_kernel ("vLLM and PagedAttention: Virtual
// Memory for LLM Serving", opening paragraph; "Inside vLLM and TGI: Paging,
// Versioned Schedulers and Operations", launch notes on chunked prefill):
// sequence s holds L positions after its chunk of Q new queries was written;
// query i sits at position L - Q + i and attends to positions 0 .. L - Q + i
// through the block table.
//
// Work decomposition (this library's design): one work item per (query
// tile, KV head, sequence), on a 1-D grid: (KV head, sequence) pairs in
// groups whose K/V pages fit in a third of L2, the heaviest query tiles
// first within a group.  An item holds two Q tiles, A and B, of 128 rows each; a row is a
// (query, grouped head) pair, so the G query heads sharing a KV head share
// every K/V tile.  One CTA runs an item, except that when the last wave of
// CTAs would leave at least half the SMs idle, its items run as two CTAs of
// one Q tile each.  Keys stream in tiles of 64 positions.  Eleven warps
// with fixed roles:
//   warps 0-7  softmax: warp w serves Q tile w / 4; thread = one row = one
//              tensor-memory lane: loads its S row, releases S, masks keys
//              past its position, keeps the running maximum and sum, writes
//              P (16-bit; bf16 as high and low parts) into its own columns,
//              rescales its O row when needed, and finally normalises and
//              stores O;
//   warp 8     producer: 4-D TMA tile loads of K and V pages into a ring
//              (128-byte swizzle); allocates the tensor memory;
//   warps 9,10 MMA issuers, one thread each for Q tile A and B:
//              S_t = Q_t.K^T (A and B from shared memory, 128 x 64 x D) and
//              O_t += P_t.V (A = P_t from tensor memory, B = V from shared
//              memory in MN-major form, 128 x D x 64).  S_t(j+1) is issued as
//              soon as the softmax has read S_t(j), P.V_t(j) once P_t(j) is
//              written; each issuer zeroes the value rows past the last
//              needed key before its last P.V;
//   warps 11-14 (FP8 pools only) converters: widen the producer's raw code
//              tiles into the fp16 operand tiles (exact), writing zeros for
//              value rows past the last needed key.  Both products then run
//              in fp16; P is split into two fp16 parts only for heads whose
//              value scale needs it (fp8_split_p); bf16 queries enter as
//              fp16 with a per-row power-of-two shift.
// The running maximum is raised lazily: O and the sum are rescaled only
// when a row's maximum grows by more than 2^8, so P stays at or below 256
// and most tiles skip the tensor-memory round trip of O.
//
// Tensor memory (512 columns), per Q tile t at t * 256: S at +0 (64
// columns), P at +64 (64), O at +128 (D).  Every wait is bounded; on a
// timeout the roles stop, each MMA issuer waits for its MMAs to drain, and
// the tensor memory is released on every path.
#pragma once

#include <algorithm>
#include <type_traits>

#include "decode_mma_fp8.cuh"
#include "prefill.cuh"
#include "tcgen05.cuh"

namespace pkv {

// Q tiles per CTA: 2 (one CTA per SM, K/V tiles shared by 256 rows) or 1
// (two CTAs per SM, each one's set-up and tail overlapping the other's
// work).  Measured on the 2048-token prompt and chunked workloads: 649 / 759
// TFLOP/s with 2, 520 / 530 with 1 -- sharing each K/V tile between 256 rows
// outweighs the overlap.
constexpr int kPrefillQTiles = 2;

// KV8: the pool holds FP8 E4M3 codes (keys and values times per-KV-head
// scales); T is then the type of q and out.  Converter warps widen each K/V
// tile to fp16 (exact for every E4M3 value), so both products run in fp16.
template <typename T, int D, int BS, int G, int QT = kPrefillQTiles, bool KV8 = false>
struct PrefillTcCfg {
  static constexpr int kQTiles = QT;
  static constexpr bool kKv8 = KV8;
  static constexpr int kTileRows = 128;          // rows per Q tile = tensor-memory lanes
  static constexpr int kRows = QT * kTileRows;
  static constexpr int kQueries = kRows / G;     // queries per CTA
  static constexpr int kKeys = 64;               // keys per K/V tile
  static constexpr int kHalves = D / 64;         // 128-byte column blocks
  static constexpr int kHalfBytes = 128 * 128;   // 128 rows x 128 B
  static constexpr int kTileBytes = kHalves * kHalfBytes;     // one Q tile (128 rows)
  static constexpr int kKvHalfBytes = kKeys * 128;               // 64 key rows x 128 B
  static constexpr int kKvBytes = kHalves * kKvHalfBytes;        // one K or V tile
  // Operand (K/V) ring; FP8 pools add a raw-code ring.  FP8, measured on the
  // 2048-token prompt / chunked workloads (operand x raw stages, TFLOP/s):
  // 2 x 4 628 / 745, 3 x 2 701 / 874, 3 x 3 668 / 867, 4 x 2 665 / 861.
  static constexpr int kStages =
      KV8 ? 3 : (QT == 2 ? (D == 64 ? 6 : 4) : (D == 64 ? 4 : 2));
  static constexpr int kBoxRows = BS < 16 ? BS : 16;
  static constexpr int kBoxes = kKeys / kBoxRows;  // TMA boxes per tile per column block
  static constexpr int kSoftmaxWarps = 4 * QT;
  static constexpr int kProducerWarp = 4 * QT;
  static constexpr int kMmaWarp = 4 * QT + 1;    // one MMA issuer warp per Q tile
  static constexpr int kConvWarp = 5 * QT + 1;  // FP8 pools: converter warps
  static constexpr int kConvWarps = KV8 ? 4 : 0;
  static constexpr int kConvThreads = kConvWarps * 32;
  static constexpr int kThreads = (5 * QT + 1 + kConvWarps) * 32;
  static constexpr int kCtasPerSm = QT == 2 ? 1 : 2;
  static constexpr int kQOff = 0;                // Q tile t at t * kTileBytes
  static constexpr int kRingOff = QT * kTileBytes;
  static constexpr int kStageBytes = 2 * kKvBytes;  // K then V
  // FP8 pools: raw code tiles (64 rows x D codes, 128-byte swizzle), K then V.
  static constexpr int kRawStages = KV8 ? 2 : 0;
  static constexpr int kRawBytes = kKeys * D;
  static constexpr int kRawOff = kRingOff + kStages * kStageBytes;
  static constexpr int kBarOff = kRawOff + kRawStages * 2 * kRawBytes;
  static constexpr int kNumBars = 3 * kStages + 6 * QT + 2 * kRawStages + 1;
  static constexpr int kSlotOff = kBarOff + kNumBars * 8;
  static constexpr int kAlign = 1024;
  static constexpr int kSmemBytes = kAlign + kSlotOff + 16;
  // Tensor memory per Q tile t (base t * 256): S at +0 (64 columns), P at
  // +64 (keys 2c, 2c+1 in column c; bf16 low part in 32 + c), O at +128.
  static constexpr uint32_t kTmemCols = 256 * QT;
  static constexpr uint32_t kTileCols = 256;
  static constexpr uint32_t kPCol = 64, kOCol = 128;
  // MMA operand type: the pool's type, or fp16 for FP8 pools.
  using OpT = typename std::conditional<KV8, __half, T>::type;
  static constexpr uint32_t kFmt = std::is_same<OpT, __nv_bfloat16>::value ? 1u : 0u;
  static constexpr uint32_t kIdescS = idesc_f16(kFmt, 128, kKeys, false);
  static constexpr uint32_t kIdescPV = idesc_f16(kFmt, 128, D, true);
  // bf16 P keeps 8 significant bits; split into high and low bf16 parts
  // (two P.V MMAs) it keeps ~16, like the fp32 softmax it comes from.
  static constexpr bool kSplitP = !KV8 && std::is_same<T, __nv_bfloat16>::value;
  static_assert(kBoxes <= 32, "one producer lane per box");
  static_assert(kKeys == 64, "the softmax's P layout assumes 64-key tiles");
  // At most kCtasPerSm CTAs per SM, so that the tensor memory (512 columns
  // per SM) always covers every resident CTA's allocation.
  static_assert(kSmemBytes * (kCtasPerSm + 1) > 228 * 1024, "CTAs per SM vs tensor memory");
  static_assert(kOCol + D <= kTileCols, "tensor memory per Q tile");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory");
  static_assert(!KV8 || D == 128, "FP8 pools: 128-code rows");
};

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// Largest of three.
__device__ __forceinline__ float max3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// 2^x with the hardware approximation (flushes results below 2^-126 to 0).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <typename T>
__device__ __forceinline__ uint32_t pack_pair(float lo, float hi);
template <>
__device__ __forceinline__ uint32_t pack_pair<__half>(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}
template <>
__device__ __forceinline__ uint32_t pack_pair<__nv_bfloat16>(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

template <typename T, int D, int BS, int G, bool KV8>
__global__ void __launch_bounds__(PrefillTcCfg<T, D, BS, G, kPrefillQTiles, KV8>::kThreads,
                                  PrefillTcCfg<T, D, BS, G, kPrefillQTiles, KV8>::kCtasPerSm)
prefill_tc_kernel(const PrefillParams p, const __grid_constant__ CUtensorMap tmk,
                  const __grid_constant__ CUtensorMap tmv) {
  using Cfg = PrefillTcCfg<T, D, BS, G, kPrefillQTiles, KV8>;
  constexpr int NR = Cfg::kRawStages;
  constexpr int QT = Cfg::kQTiles;
  constexpr int NS = Cfg::kStages;
  constexpr int KT = Cfg::kKeys;
  constexpr int RB = Cfg::kBoxRows;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((Cfg::kAlign - (smem_addr(smem_raw) & (Cfg::kAlign - 1))) &
                                    (Cfg::kAlign - 1));
  const uint32_t sbase = smem_addr(smem);

  // Work item: the (KV head, sequence) pairs run in groups of group_pairs,
  // small enough that a group's K/V pages stay in L2 while its CTAs read
  // them; within a group, query tiles heaviest first over every pair.
  // Items from n_full on run as two CTAs, one per Q tile (half = 0 or 1),
  // so that the last wave of CTAs ends sooner.
  int item = blockIdx.x, half = -1;
  if (item >= p.n_full) {
    half = (item - p.n_full) & 1;
    item = p.n_full + ((item - p.n_full) >> 1);
  }
  const int pairs = p.kv_heads * p.num_seqs;
  const int group = item / (p.group_pairs * p.q_tiles);
  const int in_group = item % (p.group_pairs * p.q_tiles);
  const int gpairs = min(p.group_pairs, pairs - group * p.group_pairs);
  const int tile = p.q_tiles - 1 - in_group / gpairs;
  const int pair = group * p.group_pairs + in_group % gpairs;
  const int kvh = pair % p.kv_heads;
  const int s = pair / p.kv_heads;
  auto active = [&](int t) { return half < 0 || t == half; };
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int H = p.num_heads;
  T* out = static_cast<T*>(p.out);

  const int q0 = p.starts[s];
  const int q1 = p.starts[s + 1];
  const int L = p.seq_lens[s];
  if (q0 < 0 || q1 < q0 || q1 > p.total_queries) {  // cannot even locate the rows
    if (tile == 0 && kvh == 0 && threadIdx.x == 0) set_error(p.err, PKV_DEV_SEQ_LEN);
    return;
  }
  const int Q = q1 - q0;
  const int qa = tile * Cfg::kQueries;
  if (qa >= Q) return;
  const int qend = min(Q, qa + Cfg::kQueries);
  // Queries of the active rows: Q tile 0 holds rows 0..127 (queries
  // qa .. qa + kQueries / 2 - 1), tile 1 the rest.
  const int qlo = half == 1 ? qa + Cfg::kQueries / 2 : qa;
  const int qhi = half == 0 ? min(Q, qa + Cfg::kQueries / 2) : qend;
  if (qlo >= qhi) return;  // a second half with no real query
  auto zero_rows = [&]() {
    for (int e = threadIdx.x; e < (qend - qa) * G * D; e += Cfg::kThreads) {
      const int qi = qa + e / (G * D);
      const int rest = e % (G * D);
      out[((int64_t)(q0 + qi) * H + kvh * G) * D + rest] = Elem<T>::from_f(0.f);
    }
  };
  if (Q > L || Q > p.max_queries || L > p.max_blocks * BS) {
    if (threadIdx.x == 0) set_error(p.err, PKV_DEV_SEQ_LEN);
    zero_rows();
    return;
  }
  const int first = L - Q;         // position of query 0
  const int n_keys = first + qhi;  // keys 0 .. n_keys-1 are visible to some active row
  const int nblk = (n_keys + BS - 1) / BS;
  const int n_tiles = (n_keys + KT - 1) / KT;
  const int32_t* trow = p.tables + (int64_t)s * p.max_blocks;
  int bad = 0;
  for (int i = threadIdx.x; i < nblk; i += Cfg::kThreads) {
    const int e = trow[i];
    bad |= (e < 0 || (int64_t)e >= p.num_blocks);
  }
  if (__syncthreads_or(bad)) {
    if (threadIdx.x == 0) set_error(p.err, PKV_DEV_TABLE_RANGE);
    zero_rows();
    return;
  }

  // ---- barriers, tensor memory, Q tiles -------------------------------------
  const uint32_t bar0 = sbase + Cfg::kBarOff;
  auto k_full = [&](int st) { return bar0 + 8u * st; };
  auto v_full = [&](int st) { return bar0 + 8u * (NS + st); };
  auto kv_empty = [&](int st) { return bar0 + 8u * (2 * NS + st); };
  // Per Q tile t: S ready, S read (free), P written, P.V done (P free).
  auto s_full = [&](int t) { return bar0 + 8u * (3 * NS + t); };
  auto s_free = [&](int t) { return bar0 + 8u * (3 * NS + QT + t); };
  auto p_full = [&](int t) { return bar0 + 8u * (3 * NS + 2 * QT + t); };
  auto p_free = [&](int t) { return bar0 + 8u * (3 * NS + 3 * QT + t); };
  auto drain = [&](int t) { return bar0 + 8u * (3 * NS + 4 * QT + t); };
  auto o_last = [&](int t) { return bar0 + 8u * (3 * NS + 5 * QT + t); };  // last P.V (single use)
  // Tile A's first S done (single use): tile B's issuer starts after it.
  const uint32_t a_first = bar0 + 8u * (3 * NS + 6 * QT + 2 * NR);
  // FP8 pools: raw code tiles landed / converted.
  auto raw_full = [&](int rs) { return bar0 + 8u * (3 * NS + 6 * QT + rs); };
  auto raw_empty = [&](int rs) { return bar0 + 8u * (3 * NS + 6 * QT + NR + rs); };
  if (threadIdx.x == 0) {
    for (int st = 0; st < NS; ++st) {
      // Native pools: the producer's copy completes the stage; FP8 pools:
      // every converter thread arrives once it has widened its part.
      mbar_init(k_full(st), KV8 ? Cfg::kConvThreads : 1);
      mbar_init(v_full(st), KV8 ? Cfg::kConvThreads : 1);
      mbar_init(kv_empty(st), half < 0 ? QT : 1);  // every active Q tile's P.V
    }
    for (int t = 0; t < QT; ++t) {
      mbar_init(s_full(t), 1);
      mbar_init(s_free(t), Cfg::kTileRows);
      mbar_init(p_full(t), Cfg::kTileRows);
      mbar_init(p_free(t), 1);
      mbar_init(drain(t), 1);
      mbar_init(o_last(t), 1);
    }
    mbar_init(a_first, 1);
    for (int rs = 0; rs < NR; ++rs) {
      mbar_init(raw_full(rs), 1);
      mbar_init(raw_empty(rs), Cfg::kConvThreads);
    }
    fence_mbar_init();
  }
  uint32_t* slot = reinterpret_cast<uint32_t*>(smem + Cfg::kSlotOff);
  if (warp == Cfg::kProducerWarp) {
    tmem_alloc(smem_addr(slot), Cfg::kTmemCols);
    tmem_relinquish();
  }
  // Softmax thread: Q tile t = warp / 4, row rr = (warp % 4) * 32 + lane of
  // it (tensor-memory lane rr), CTA row R = t * 128 + rr: query
  // min(qa + R / G, Q - 1) (padding rows repeat the last query and are not
  // stored), head kvh * G + R % G.  It copies its Q row into the
  // 128-byte-swizzled operand layout.
  const int t = (warp >> 2) & (QT - 1);
  const int rr = (warp & 3) * 32 + lane;
  const int R = t * Cfg::kTileRows + rr;
  const int qi = min(qa + R / G, Q - 1);
  float row_scale = 1.f;  // FP8 pools: this row's factor on its scores
  if (warp < Cfg::kSoftmaxWarps && active(t)) {
    const uint4* qrow = reinterpret_cast<const uint4*>(static_cast<const T*>(p.q) +
                                                       ((int64_t)(q0 + qi) * H + kvh * G + R % G) * D);
    unsigned char* qt = smem + Cfg::kQOff + t * Cfg::kTileBytes;
    uint4 qv[D / 8];
#pragma unroll
    for (int c = 0; c < D / 8; ++c) qv[c] = qrow[c];
    if constexpr (KV8) {
      // The MMAs run in fp16.  A bf16 row whose largest magnitude reaches
      // 2^15 is first scaled by a power of two (exact; undone in the row's
      // score factor) so that it stays inside fp16's range.
      row_scale = p.k_scale[kvh];
      if constexpr (std::is_same<T, __nv_bfloat16>::value) {
        float amax = 0.f;
#pragma unroll
        for (int c = 0; c < D / 8; ++c) {
          const uint32_t* w = reinterpret_cast<const uint32_t*>(&qv[c]);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(w[i] << 16)),
                                     fabsf(__uint_as_float(w[i] & 0xFFFF0000u))));
        }
        float shrink = 1.f;
        if (amax >= 32768.f && amax <= 3.0e38f) {
          int e = 0;
          frexpf(amax, &e);  // amax = m * 2^e, m in [0.5, 1)
          shrink = ldexpf(1.f, 15 - e);
          row_scale = ldexpf(row_scale, e - 15);
        }
#pragma unroll
        for (int c = 0; c < D / 8; ++c) {
          uint32_t* w = reinterpret_cast<uint32_t*>(&qv[c]);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            w[i] = pack_pair<__half>(__uint_as_float(w[i] << 16) * shrink,
                                     __uint_as_float(w[i] & 0xFFFF0000u) * shrink);
        }
      }
    }
#pragma unroll
    for (int c = 0; c < D / 8; ++c) {
      const int half = c >> 3, cc = c & 7;
      *reinterpret_cast<uint4*>(qt + half * Cfg::kHalfBytes + rr * 128 + ((cc ^ (rr & 7)) << 4)) =
          qv[c];
    }
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *slot;
  bool failed = false;
  // P in two parts (a second P.V MMA): bf16 pools always; FP8 pools when
  // the head's value scale makes fp16 P too coarse (fp8_split_p, with the
  // FP8 decode kernels).
  bool split_p = Cfg::kSplitP;
  if constexpr (KV8) split_p = fp8_split_p<T>(p.v_scale[kvh]);

  if (warp == Cfg::kProducerWarp) {
    // ---- producer: K and V tiles ------------------------------------------
    // Native pools: straight into the operand ring.  FP8 pools: raw code
    // tiles into their own ring, for the converter warps.
    const uint64_t policy = policy_evict_last();
    const int oob_block = p.num_blocks > 0x7FFFFFFF ? 0x7FFFFFFF : (int)p.num_blocks;
    constexpr int RING = KV8 ? NR : NS;
    int issued = 0;
    for (int j = 0; j < n_tiles; ++j) {
      const int st = j % RING;
      if (j >= RING) {
        const uint32_t empty = KV8 ? raw_empty(st) : kv_empty(st);
        const bool ok = mbar_wait(empty, (uint32_t)(((j / RING) - 1) & 1));
        if (__any_sync(kFullMask, !ok)) {
          failed = true;
          break;
        }
      }
      uint32_t kdst, vdst, kbar, vbar;
      if constexpr (KV8) {
        kdst = sbase + Cfg::kRawOff + st * 2 * Cfg::kRawBytes;
        vdst = kdst + Cfg::kRawBytes;
        kbar = vbar = raw_full(st);
        if (lane == 0) mbar_arrive_expect_tx(kbar, 2 * Cfg::kRawBytes);
      } else {
        kdst = sbase + Cfg::kRingOff + st * Cfg::kStageBytes;
        vdst = kdst + Cfg::kKvBytes;
        kbar = k_full(st);
        vbar = v_full(st);
        if (lane == 0) {
          mbar_arrive_expect_tx(kbar, Cfg::kKvBytes);
          mbar_arrive_expect_tx(vbar, Cfg::kKvBytes);
        }
      }
      __syncwarp();
      if (lane < Cfg::kBoxes) {
        const int pos = j * KT + lane * RB;
        // Boxes wholly past the last needed key read an out-of-range block:
        // the copy fills them with zeros.
        int pb = oob_block, row = 0;
        if (pos < n_keys) {
          pb = trow[pos / BS];
          row = pos % BS;
        }
        if constexpr (KV8) {  // rows of 128 codes: one box per RB rows
          tma_load_4d(kdst + lane * RB * 128, &tmk, 0, row, kvh, pb, kbar, policy);
          tma_load_4d(vdst + lane * RB * 128, &tmv, 0, row, kvh, pb, vbar, policy);
        } else {
#pragma unroll
          for (int h = 0; h < Cfg::kHalves; ++h) {
            const uint32_t o = h * Cfg::kKvHalfBytes + lane * RB * 128;
            tma_load_4d(kdst + o, &tmk, h * 64, row, kvh, pb, kbar, policy);
            tma_load_4d(vdst + o, &tmv, h * 64, row, kvh, pb, vbar, policy);
          }
        }
      }
      issued = j + 1;
    }
    // Copies issued but possibly never consumed (another role stopped).
    for (int j = issued - RING < 0 ? 0 : issued - RING; j < issued; ++j) {
      if constexpr (KV8) {
        mbar_wait(raw_full(j % RING), (uint32_t)((j / RING) & 1), kWaitLimitNs / 8);
      } else {
        mbar_wait(k_full(j % RING), (uint32_t)((j / RING) & 1), kWaitLimitNs / 8);
        mbar_wait(v_full(j % RING), (uint32_t)((j / RING) & 1), kWaitLimitNs / 8);
      }
    }
  } else if (warp >= Cfg::kMmaWarp && warp < Cfg::kMmaWarp + QT &&
             !active(warp - Cfg::kMmaWarp)) {
    // The issuer of a Q tile this CTA does not run has nothing to do.
  } else if (warp >= Cfg::kMmaWarp && warp < Cfg::kMmaWarp + QT) {
    // ---- MMA issuers, one per Q tile t: S_t(0); then per K/V tile j:
    //      S_t(j+1) once the softmax has read S_t(j), and P.V_t(j) once
    //      P_t(j) is written.  The next S is computed while the softmax works
    //      on the current one; P has its own columns, so only the next P
    //      write waits for a P.V.  Separate issuers keep one tile's waits
    //      from holding up the other's MMAs (commits track each thread's
    //      own MMAs).
    auto wait_all = [&](uint32_t bar, int phase) {
      const bool o = mbar_wait(bar, (uint32_t)(phase & 1));
      return !__any_sync(kFullMask, !o);
    };
    auto issue_s = [&](int tt, int j) {
      if (lane == 0) {
        const uint32_t qb = sbase + Cfg::kQOff + tt * Cfg::kTileBytes;
        const uint32_t kb = sbase + Cfg::kRingOff + (j % NS) * Cfg::kStageBytes;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t qo = (kk >> 2) * Cfg::kHalfBytes + (kk & 3) * 32;
          const uint32_t ko = (kk >> 2) * Cfg::kKvHalfBytes + (kk & 3) * 32;
          tc_mma_ss(tmem + tt * Cfg::kTileCols, smem_desc_sw128(qb + qo, 16, 1024),
                    smem_desc_sw128(kb + ko, 16, 1024), Cfg::kIdescS, kk > 0 ? 1u : 0u);
        }
        tc_commit(s_full(tt));
      }
      __syncwarp();
    };
    auto issue_pv = [&](int tt, int j) {
      if (lane == 0) {
        const uint32_t vb = sbase + Cfg::kRingOff + (j % NS) * Cfg::kStageBytes + Cfg::kKvBytes;
        const uint32_t base = tmem + tt * Cfg::kTileCols;
#pragma unroll
        for (int kk = 0; kk < KT / 16; ++kk) {
          // MN-major V: 64-dim atoms kKvHalfBytes apart, 8-key groups 1024 B
          // apart.  With one atom (D = 64) the atom stride is unused; 1024
          // keeps every address inside the tile whichever field is read.
          const uint64_t bdesc = smem_desc_sw128(
              vb + kk * 2048, Cfg::kHalves > 1 ? Cfg::kKvHalfBytes : 1024, 1024);
          // P of keys 16kk .. 16kk+15: columns 8kk .. 8kk+7, low part 32 further.
          const uint32_t pa = base + Cfg::kPCol + 8 * kk;
          tc_mma_ts(base + Cfg::kOCol, pa, bdesc, Cfg::kIdescPV, (j > 0 || kk > 0) ? 1u : 0u);
          if (split_p) tc_mma_ts(base + Cfg::kOCol, pa + 32, bdesc, Cfg::kIdescPV, 1u);
        }
        tc_commit(p_free(tt));
      }
      __syncwarp();
    };
    const int tq = warp - Cfg::kMmaWarp;  // this issuer's Q tile
    bool ok = wait_all(k_full(0), 0);
    // Tile B starts once tile A's first S is done, so that the two tiles'
    // softmax passes are staggered rather than in step (1-2% faster on the
    // chunked and prompt workloads, 16-bit and FP8 pools).
    if (ok && tq == 1 && half < 0) ok = wait_all(a_first, 0);
    if (ok) {
      tc_fence_after();
      issue_s(tq, 0);
      if (tq == 0 && lane == 0) tc_commit(a_first);
    }
    for (int j = 0; j < n_tiles && ok; ++j) {
      const int st = j % NS;
      if (j + 1 < n_tiles) {
        ok = wait_all(k_full((j + 1) % NS), (j + 1) / NS) && wait_all(s_free(tq), j);
        if (!ok) break;
        tc_fence_after();
        issue_s(tq, j + 1);
      }
      ok = wait_all(p_full(tq), j) && wait_all(v_full(st), j / NS);
      if (!ok) break;
      if (!KV8 && j == n_tiles - 1 && n_keys - j * KT < KT) {
        // Value rows past the last needed key hold stale pool contents
        // (0 * NaN would poison O): zero them.  Both issuers do it, writing
        // the same zeros, each before its own last P.V.  (FP8 pools: the
        // converters write zeros there.)
        const int valid = n_keys - j * KT;
        unsigned char* vt = smem + Cfg::kRingOff + st * Cfg::kStageBytes + Cfg::kKvBytes;
        for (int e = lane; e < (KT - valid) * Cfg::kHalves * 8; e += 32) {
          const int row = valid + e / (Cfg::kHalves * 8);
          const int rest = e % (Cfg::kHalves * 8);
          *reinterpret_cast<uint4*>(vt + (rest >> 3) * Cfg::kKvHalfBytes + row * 128 +
                                    (rest & 7) * 16) = make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();
        __syncwarp();
      }
      tc_fence_after();
      issue_pv(tq, j);
      if (lane == 0) tc_commit(kv_empty(st));
    }
    if (ok && lane == 0) tc_commit(o_last(tq));
    failed = !ok;
    // Every MMA this thread issued has completed before the tensor memory
    // is released.
    if (lane == 0) tc_commit(drain(tq));
    __syncwarp();
    mbar_wait(drain(tq), 0);
  } else if (KV8 && warp >= Cfg::kConvWarp) {
    // ---- converters (FP8 pools): raw code tiles -> fp16 operand tiles ------
    // Thread ct widens 16-code chunks of K and then V: chunk ch of key row
    // r (swizzled in the raw tile) becomes dims 16ch .. 16ch+15, i.e. two
    // 16-byte chunks of the 128-byte-swizzled fp16 tile.  Value rows at or
    // past the last needed key are written as zeros (stale codes could be
    // NaN, and 0 * NaN would poison O).
    const int ct = threadIdx.x - Cfg::kConvWarp * 32;
    for (int j = 0; j < n_tiles; ++j) {
      const int rs = j % NR, st = j % NS;
      bool ok = mbar_wait(raw_full(rs), (uint32_t)((j / NR) & 1));
      if (ok && j >= NS) ok = mbar_wait(kv_empty(st), (uint32_t)(((j / NS) - 1) & 1));
      if (__any_sync(kFullMask, !ok)) {
        failed = true;
        break;
      }
      const unsigned char* raw = smem + Cfg::kRawOff + rs * 2 * Cfg::kRawBytes;
      unsigned char* wide = smem + Cfg::kRingOff + st * Cfg::kStageBytes;
      const int valid = n_keys - j * KT;
#pragma unroll
      for (int kv = 0; kv < 2; ++kv) {
        const unsigned char* src = raw + kv * Cfg::kRawBytes;
        unsigned char* dst = wide + kv * Cfg::kKvBytes;
#pragma unroll
        for (int i = 0; i < KT * 8 / Cfg::kConvThreads; ++i) {
          const int unit = ct + i * Cfg::kConvThreads;
          const int row = unit >> 3, ch = unit & 7;
          uint4 lo = make_uint4(0u, 0u, 0u, 0u), hi = lo;
          if (kv == 0 || row < valid) {
            const uint4 c =
                *reinterpret_cast<const uint4*>(src + row * 128 + ((ch ^ (row & 7)) << 4));
            e4m3x4_to_f16x4(c.x, lo.x, lo.y);
            e4m3x4_to_f16x4(c.y, lo.z, lo.w);
            e4m3x4_to_f16x4(c.z, hi.x, hi.y);
            e4m3x4_to_f16x4(c.w, hi.z, hi.w);
          }
          const int c2 = (ch & 3) * 2;
          unsigned char* drow = dst + (ch >> 2) * Cfg::kKvHalfBytes + row * 128;
          *reinterpret_cast<uint4*>(drow + ((c2 ^ (row & 7)) << 4)) = lo;
          *reinterpret_cast<uint4*>(drow + (((c2 + 1) ^ (row & 7)) << 4)) = hi;
        }
        fence_proxy_async_smem();
        mbar_arrive(kv == 0 ? k_full(st) : v_full(st));
      }
      mbar_arrive(raw_empty(rs));
    }
  } else if (!active(t)) {
    // Softmax warps of a Q tile this CTA does not run have nothing to do.
  } else {
    // ---- softmax, row rr of Q tile t ----------------------------------------
    const int pos = first + qi;
    const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const uint32_t scol = t * Cfg::kTileCols, pcol = scol + Cfg::kPCol, ocol = scol + Cfg::kOCol;
    // Scores are taken as s * |factor| with the sign folded into s, so the
    // row maximum can be found on the raw scores (a negative factor flips
    // every score's sign bit first).  FP8 pools: key scale and row shift.
    const float qfac = p.qscale * row_scale;
    const bool qneg = qfac < 0.f;
    const float qscale = fabsf(qfac);
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < n_tiles; ++j) {
      ok = mbar_wait(s_full(t), (uint32_t)(j & 1));
      if (__any_sync(kFullMask, !ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      // The S row (64 scores), then S is free for the next tile's MMA.
      uint32_t w[KT];
      tmem_ld64(lane_base + scol, w);
      tc_fence_before();
      mbar_arrive(s_free(t));
      if (qneg) {
#pragma unroll
        for (int c = 0; c < KT; ++c) w[c] ^= 0x80000000u;
      }
      // Keys past this row's position count as -inf (diagonal tiles only).
      const int lim = pos - j * KT;  // keys c <= lim are visible
      if (__any_sync(kFullMask, lim < KT - 1)) {
#pragma unroll
        for (int c = 0; c < KT; ++c)
          if (c > lim) w[c] = __float_as_uint(-INFINITY);
      }
      // Row maximum: four independent chains of three-input maxima.
      float mq[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int c = 0; c < KT; c += 8)
#pragma unroll
        for (int u = 0; u < 4; ++u)
          mq[u] = max3(mq[u], __uint_as_float(w[c + 2 * u]), __uint_as_float(w[c + 2 * u + 1]));
      const float mx = max3(mq[0], mq[1], fmaxf(mq[2], mq[3])) * qscale;
      // Lazy maximum: raise it (and rescale O and l) only when the tile's
      // maximum exceeds it by more than 8 (P <= 2^8 otherwise).  Every row
      // sees key 0 in tile 0, so m is finite from then on.
      bool rescale = false;
      float alpha = 1.f;
      if (j == 0) {
        m = mx;
      } else {
        const bool raise = mx > m + 8.f;
        rescale = __any_sync(kFullMask, raise);
        if (raise) {
          alpha = ex2(m - mx);
          l *= alpha;
          m = mx;
        }
      }
      // Pairs of scores through the packed fp32 pipe: 2^(s * scale - m) and
      // the running sum.
      const float2 qs2 = make_float2(qscale, qscale), nm2 = make_float2(-m, -m);
      float2 sum2[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                        make_float2(0.f, 0.f)};
#pragma unroll
      for (int c = 0; c < KT; c += 2) {
        const float2 a = __ffma2_rn(make_float2(__uint_as_float(w[c]), __uint_as_float(w[c + 1])),
                                    qs2, nm2);
        const float2 e = make_float2(ex2(a.x), ex2(a.y));
        w[c] = __float_as_uint(e.x);
        w[c + 1] = __float_as_uint(e.y);
        sum2[(c >> 1) & 3] = __fadd2_rn(sum2[(c >> 1) & 3], e);
      }
      const float2 s01 = __fadd2_rn(sum2[0], sum2[1]), s23 = __fadd2_rn(sum2[2], sum2[3]);
      const float2 sx = __fadd2_rn(s01, s23);
      l += sx.x + sx.y;
      // P: keys 2c, 2c+1 in column c (high part, or the only one); the bf16
      // low part of the same keys in column 32 + c.
      uint32_t pk[KT];
#pragma unroll
      for (int c = 0; c < KT / 2; ++c) {
        const uint32_t a = w[2 * c], b = w[2 * c + 1];
        if (Cfg::kSplitP) {
          pk[c] = __byte_perm(a, b, 0x7632);  // upper halves: truncated bf16
          // exact remainders p - trunc(p), rounded to bf16
          const float2 r = __ffma2_rn(
              make_float2(__uint_as_float(a & 0xFFFF0000u), __uint_as_float(b & 0xFFFF0000u)),
              make_float2(-1.f, -1.f), make_float2(__uint_as_float(a), __uint_as_float(b)));
          pk[KT / 2 + c] = pack_pair<typename Cfg::OpT>(r.x, r.y);
        } else if (KV8 && split_p) {
          // fp16 high part rounded to nearest, then the exact remainder
          // rounded to fp16
          const __half2 hi = __floats2half2_rn(__uint_as_float(a), __uint_as_float(b));
          const float2 hf = __half22float2(hi);
          pk[c] = *reinterpret_cast<const uint32_t*>(&hi);
          pk[KT / 2 + c] =
              pack_pair<__half>(__uint_as_float(a) - hf.x, __uint_as_float(b) - hf.y);
        } else {
          pk[c] = pack_pair<typename Cfg::OpT>(__uint_as_float(a), __uint_as_float(b));
          pk[KT / 2 + c] = 0u;
        }
      }
      // P.V of tile j-1 has read P and added into O before either changes.
      if (j > 0) {
        ok = mbar_wait(p_free(t), (uint32_t)((j - 1) & 1));
        if (__any_sync(kFullMask, !ok)) {
          ok = false;
          break;
        }
        tc_fence_after();
      }
      tmem_st64(lane_base + pcol, pk);
      if (rescale) {
#pragma unroll 1
        for (int c4 = 0; c4 < D / 32; ++c4) {
          uint32_t o[32];
          tmem_ld32(lane_base + ocol + c4 * 32, o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
          tmem_st32(lane_base + ocol + c4 * 32, o);
        }
      }
      tc_fence_before();
      mbar_arrive(p_full(t));
    }
    // ---- epilogue: O / l into the output rows that are real queries ---------
    if (ok) {
      ok = mbar_wait(o_last(t), 0);
      ok = !__any_sync(kFullMask, !ok);
    }
    failed = !ok;
    if (ok) {
      tc_fence_after();
      const bool real = qa + R / G < qend;
      const float inv = (KV8 ? p.v_scale[kvh] : 1.f) / l;
      uint4* orow = reinterpret_cast<uint4*>(out + ((int64_t)(q0 + qi) * H + kvh * G + R % G) * D);
#pragma unroll
      for (int c4 = 0; c4 < D / 32; ++c4) {
        uint32_t w[32];
        tmem_ld32(lane_base + ocol + c4 * 32, w);
        if (real) {
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            uint4 u;
            u.x = pack_pair<T>(__uint_as_float(w[8 * v + 0]) * inv, __uint_as_float(w[8 * v + 1]) * inv);
            u.y = pack_pair<T>(__uint_as_float(w[8 * v + 2]) * inv, __uint_as_float(w[8 * v + 3]) * inv);
            u.z = pack_pair<T>(__uint_as_float(w[8 * v + 4]) * inv, __uint_as_float(w[8 * v + 5]) * inv);
            u.w = pack_pair<T>(__uint_as_float(w[8 * v + 6]) * inv, __uint_as_float(w[8 * v + 7]) * inv);
            orow[c4 * 4 + v] = u;
          }
        }
      }
    }
  }

  // ---- release the tensor memory ------------------------------------------
  if (failed && lane == 0) set_error(p.err, PKV_DEV_TIMEOUT);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == Cfg::kProducerWarp) tmem_dealloc(tmem, Cfg::kTmemCols);
}

template <typename T, int D, int BS, int G, bool KV8>
int launch_prefill_tc_cfg(const PrefillParams& p, int num_seqs, const CUtensorMap& mk,
                          const CUtensorMap& mv, cudaStream_t stream) {
  using Cfg = PrefillTcCfg<T, D, BS, G, kPrefillQTiles, KV8>;
  auto kern = prefill_tc_kernel<T, D, BS, G, KV8>;
  static std::atomic<uint64_t> ready{0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ERR_CUDA;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(ready.load() & bit)) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Cfg::kSmemBytes) != cudaSuccess)
      return PKV_ERR_CUDA;
    ready.fetch_or(bit);
  }
  // One CTA per SM.  When the last wave would hold at most half the SMs'
  // worth of items, those items (the lightest: query tiles run heaviest
  // first) each run as two CTAs of one Q tile, which fill the idle SMs and
  // end the wave in about half the time.
  static std::atomic<int> sm_count[64];
  int sms = sm_count[dev & 63].load();
  if (sms == 0) {
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
      return PKV_ERR_CUDA;
    sm_count[dev & 63].store(sms);
  }
  PrefillParams q = p;
  q.q_tiles = (p.max_queries + Cfg::kQueries - 1) / Cfg::kQueries;
  q.num_seqs = num_seqs;
  // Pairs per group: about 48 MB of K/V pages (a third of L2) at the
  // longest possible sequence.
  const int64_t pair_bytes =
      (int64_t)p.max_blocks * BS * D * (KV8 ? 1 : (int64_t)sizeof(T)) * 2;
  const int64_t pairs_all = (int64_t)p.kv_heads * num_seqs;
  q.group_pairs = (int)std::max<int64_t>(1, std::min<int64_t>(pairs_all, (48ll << 20) / std::max<int64_t>(pair_bytes, 1)));
  const int64_t items = (int64_t)q.q_tiles * p.kv_heads * num_seqs;
  const int64_t rem = items % sms;
  const int64_t split = (rem > 0 && 2 * rem <= sms) ? rem : 0;
  if (items + split > 0x7FFFFFFF) return PKV_ERR_GEOMETRY;
  q.n_full = (int)(items - split);
  kern<<<(unsigned)(items + split), Cfg::kThreads, Cfg::kSmemBytes, stream>>>(q, mk, mv);
  return cudaPeekAtLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

template <typename T, int D, int BS, bool KV8>
int launch_prefill_tc_g(const PrefillParams& p, int num_seqs, int group, const CUtensorMap& mk,
                        const CUtensorMap& mv, cudaStream_t stream) {
  switch (group) {
    case 1: return launch_prefill_tc_cfg<T, D, BS, 1, KV8>(p, num_seqs, mk, mv, stream);
    case 2: return launch_prefill_tc_cfg<T, D, BS, 2, KV8>(p, num_seqs, mk, mv, stream);
    case 4: return launch_prefill_tc_cfg<T, D, BS, 4, KV8>(p, num_seqs, mk, mv, stream);
    case 8: return launch_prefill_tc_cfg<T, D, BS, 8, KV8>(p, num_seqs, mk, mv, stream);
  }
  return PKV_ERR_GEOMETRY;
}

// 16-bit pools: T is the cache and I/O type.
template <typename T>
int launch_prefill_tc(const PrefillParams& p, int num_seqs, int head_dim, int block_size,
                      int group, const CUtensorMap& mk, const CUtensorMap& mv,
                      cudaStream_t stream) {
  switch (head_dim * 1000 + block_size) {
    case 64008: return launch_prefill_tc_g<T, 64, 8, false>(p, num_seqs, group, mk, mv, stream);
    case 64016: return launch_prefill_tc_g<T, 64, 16, false>(p, num_seqs, group, mk, mv, stream);
    case 64032: return launch_prefill_tc_g<T, 64, 32, false>(p, num_seqs, group, mk, mv, stream);
    case 64064: return launch_prefill_tc_g<T, 64, 64, false>(p, num_seqs, group, mk, mv, stream);
    case 128008: return launch_prefill_tc_g<T, 128, 8, false>(p, num_seqs, group, mk, mv, stream);
    case 128016: return launch_prefill_tc_g<T, 128, 16, false>(p, num_seqs, group, mk, mv, stream);
    case 128032: return launch_prefill_tc_g<T, 128, 32, false>(p, num_seqs, group, mk, mv, stream);
    case 128064: return launch_prefill_tc_g<T, 128, 64, false>(p, num_seqs, group, mk, mv, stream);
  }
  return PKV_ERR_GEOMETRY;
}

// FP8 pools (head_dim 128): T is the I/O type of q and out.
template <typename T>
int launch_prefill_tc_fp8(const PrefillParams& p, int num_seqs, int head_dim, int block_size,
                          int group, const CUtensorMap& mk, const CUtensorMap& mv,
                          cudaStream_t stream) {
  if (head_dim != 128) return PKV_ERR_GEOMETRY;
  switch (block_size) {
    case 8: return launch_prefill_tc_g<T, 128, 8, true>(p, num_seqs, group, mk, mv, stream);
    case 16: return launch_prefill_tc_g<T, 128, 16, true>(p, num_seqs, group, mk, mv, stream);
    case 32: return launch_prefill_tc_g<T, 128, 32, true>(p, num_seqs, group, mk, mv, stream);
    case 64: return launch_prefill_tc_g<T, 128, 64, true>(p, num_seqs, group, mk, mv, stream);
  }
  return PKV_ERR_GEOMETRY;
}

}  // namespace pkv
