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
// first within a group.  An item holds two Q tiles, A and B, of 128 rows
// each; a row is a (query, grouped head) pair, so the G query heads sharing
// a KV head share every K/V tile.  One CTA runs an item, except that when
// the last wave of CTAs would leave at least half the SMs idle, its items
// run as two CTAs of one Q tile each.  Keys stream in tiles of 64 positions
// through two rings: key tiles (freed once both Q tiles' S has read them,
// so they can be fetched far ahead) and value tiles (freed after P.V).
// Fifteen warps with fixed roles:
//   warps 0-7  softmax: warp w serves Q tile w / 4; thread = one row = one
//              tensor-memory lane: loads its S row, releases S, masks keys
//              past its position, keeps the running maximum and sum, writes
//              P into its own columns, rescales its O row when needed, and
//              finally normalises and stores O;
//   warp 8     producer: 4-D TMA tile loads (128-byte swizzle) of key and
//              value pages, each into its ring as soon as a slot is free
//              (FP8 pools: raw code tiles into a third ring); allocates the
//              tensor memory;
//   warps 9,10 MMA issuers, one thread each for Q tile A and B:
//              S_t = Q_t.K^T (A and B from shared memory, 128 x 64 x D) and
//              O_t += P_t.V (A = P_t from tensor memory, 128 x D x 64).
//              S_t(j+1) is issued as soon as the softmax has read S_t(j),
//              P.V_t(j) once P_t(j) and the value operand are written.
//              Descriptors are built once and stepped by constants: the
//              issuing thread's own instruction chain sets how fast it can
//              feed the tensor pipe;
//   warps 11-14 converters.  16-bit pools: each value tile becomes V^T in
//              fp16 (ldmatrix.trans and stmatrix), the K-major operand of
//              P.V, with fp16 P; a bf16 tile whose largest value exceeds
//              kWideLimit instead runs P.V in bf16 with P as high and low
//              parts against the raw tile (MN-major).  FP8 pools: key and
//              value codes are widened to fp16 (exact) into K-major and
//              MN-major tiles; P is one fp16 part, or two for heads whose
//              value scale needs it (fp8_split_p); bf16 queries enter as
//              fp16 with a per-row power-of-two shift.  Value positions past
//              the last needed key are written as zeros.
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
// 16-bit pools: keys go straight from the TMA copy into the S product; the
// converter warps turn each value tile into its fp16 transpose.
template <typename T, int D, int BS, int G, int QT = kPrefillQTiles, bool KV8 = false>
struct PrefillTcCfg {
  static constexpr int kQTiles = QT;
  static constexpr bool kKv8 = KV8;
  static constexpr int kTileRows = 128;          // rows per Q tile = tensor-memory lanes
  static constexpr int kRows = QT * kTileRows;
  static constexpr int kQueries = kRows / G;     // queries per CTA
  static constexpr int kKeys = 64;               // keys per K/V tile
  static constexpr int kHalves = D / 64;         // 128-byte column blocks
  static constexpr int kKvHalfBytes = kKeys * 128;               // 64 key rows x 128 B
  static constexpr int kKvBytes = kHalves * kKvHalfBytes;        // one K or V tile
  // V^T: D rows (head dims) x 64 keys of fp16 (128 B), 128-byte swizzle: the
  // K-major B operand of P.V.
  static constexpr int kVtBytes = D * 128;
  // Two operand rings, so that key tiles can be fetched well ahead:
  //  * K ring: key tiles (16-bit pools: as copied; FP8 pools: widened),
  //    free once every active Q tile's S of that tile is done;
  //  * V ring: (16-bit pools) the raw value tile as copied, then V^T; free
  //    once every active Q tile's P.V of that tile is done.
  // FP8 pools keep their raw codes (keys and values) in a third ring.
  static constexpr int kKStages = KV8 ? 3 : (D == 64 ? 8 : 4);
  static constexpr int kVrawBytes = KV8 ? 0 : kKvBytes;
  static constexpr int kVStageBytes = kVrawBytes + kVtBytes;
  static constexpr int kVStages = D == 64 ? 6 : 3;
  // Q tiles, the A operand of S: 128 rows x D of 16-bit values in 128-byte
  // column blocks (128-byte swizzle).
  static constexpr int kHalfBytes = 128 * 128;               // 128 rows x 128 B
  static constexpr int kTileBytes = kHalves * kHalfBytes;    // one Q tile
  static constexpr int kBoxRows = BS < 16 ? BS : 16;
  static constexpr int kBoxes = kKeys / kBoxRows;  // TMA boxes per tile per column block
  static constexpr int kSoftmaxWarps = 4 * QT;
  static constexpr int kProducerWarp = 4 * QT;
  static constexpr int kMmaWarp = 4 * QT + 1;    // one MMA issuer warp per Q tile
  static constexpr int kConvWarp = 5 * QT + 1;   // converter warps
  static constexpr int kConvWarps = 4;
  static constexpr int kConvThreads = kConvWarps * 32;
  // All four converter warps turn values into V^T; on FP8 pools they widen
  // the key codes first.
  static constexpr int kConvKThreads = KV8 ? kConvThreads : 0;
  static constexpr int kConvVThreads = kConvThreads;
  static constexpr int kThreads = (5 * QT + 1 + kConvWarps) * 32;
  static constexpr int kCtasPerSm = QT == 2 ? 1 : 2;
  static constexpr int kQOff = 0;                          // Q tile t at t * kTileBytes
  static constexpr int kKRingOff = QT * kTileBytes;
  static constexpr int kVRingOff = kKRingOff + kKStages * kKvBytes;
  // FP8 pools: raw code tiles (64 rows x D codes, 128-byte swizzle), K then V.
  static constexpr int kRawStages = KV8 ? 2 : 0;
  static constexpr int kRawBytes = kKeys * D;
  static constexpr int kRawOff = kVRingOff + kVStages * kVStageBytes;
  static constexpr int kBarOff = kRawOff + kRawStages * 2 * kRawBytes;
  static constexpr int kNumBars = 2 * kKStages + 3 * kVStages + 6 * QT + 2 * kRawStages + 1;
  static constexpr int kFlagOff = kBarOff + kNumBars * 8;   // per V stage: 1 + last wide tile
  static constexpr int kSlotOff = kFlagOff + kVStages * 4;
  static constexpr int kAlign = 1024;
  static constexpr int kSmemBytes = kAlign + kSlotOff + 16;
  // Tensor memory per Q tile t (base t * 256): S at +0 (64 columns), P at
  // +64 (keys 2c, 2c+1 in column c; a low part in 32 + c), O at +128.
  static constexpr uint32_t kTmemCols = 256 * QT;
  static constexpr uint32_t kTileCols = 256;
  static constexpr uint32_t kSCol = 0, kPCol = 64, kOCol = 128;
  // S operand type: the pool's type, or fp16 for FP8 pools.  P.V runs in
  // fp16 against V^T; bf16 pools fall back to bf16 P.V (P as high and low
  // parts against the raw value tile) on tiles whose values are too large
  // for fp16 P (see kWideLimit).
  using OpT = typename std::conditional<KV8, __half, T>::type;
  static constexpr uint32_t kFmt = std::is_same<OpT, __nv_bfloat16>::value ? 1u : 0u;
  static constexpr uint32_t kIdescS = idesc_f16(kFmt, 128, kKeys, false);
  static constexpr uint32_t kIdescPV = idesc_f16(0u, 128, D, false);       // fp16, V^T K-major
  static constexpr uint32_t kIdescPVWide = idesc_f16(1u, 128, D, true);    // bf16, raw V MN-major
  static constexpr uint32_t kIdescPV8 = idesc_f16(0u, 128, D, true);       // fp16, widened V MN-major
  static constexpr bool kWideCheck = !KV8 && std::is_same<T, __nv_bfloat16>::value;
  // fp16 P rounds each weight by at most 2^-11 of itself, so it moves an
  // output by at most 2^-11 max |v|.  A bf16 value tile whose largest
  // magnitude exceeds 8.192 could push that past half of the bf16 error bar
  // for attention (max abs 8e-3); such tiles take the bf16 two-part P path
  // (about 16 bits of P), as do values beyond fp16's range.
  static constexpr float kWideLimit = 8.192f;
  static_assert(kBoxes <= 32, "one producer lane per box");
  static_assert(kKeys == 64, "the softmax's P layout assumes 64-key tiles");
  // At most kCtasPerSm CTAs per SM, so that the tensor memory (512 columns
  // per SM) always covers every resident CTA's allocation.
  static_assert(kSmemBytes * (kCtasPerSm + 1) > 228 * 1024, "CTAs per SM vs tensor memory");
  static_assert(kOCol + D <= kTileCols, "tensor memory per Q tile");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory");
  static_assert(!KV8 || D == 128, "FP8 pools: 128-code rows");
  static_assert(kKvBytes % 1024 == 0 && kVStageBytes % 1024 == 0 && kVrawBytes % 1024 == 0,
                "128-byte swizzle atoms");
};

__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

template <typename T, int D, int BS, int G, bool KV8>
__global__ void __launch_bounds__(PrefillTcCfg<T, D, BS, G, kPrefillQTiles, KV8>::kThreads,
                                  PrefillTcCfg<T, D, BS, G, kPrefillQTiles, KV8>::kCtasPerSm)
prefill_tc_kernel(const PrefillParams p, const __grid_constant__ CUtensorMap tmk,
                  const __grid_constant__ CUtensorMap tmv) {
  using Cfg = PrefillTcCfg<T, D, BS, G, kPrefillQTiles, KV8>;
  constexpr int NR = Cfg::kRawStages;
  constexpr int QT = Cfg::kQTiles;
  constexpr int NK = Cfg::kKStages;
  constexpr int NV = Cfg::kVStages;
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
  // K ring: key tile ready (the copy, or the FP8 key converters), free (every
  // active Q tile's S of it done).  V ring: raw values copied (16-bit pools),
  // V^T written by the converters, free (every active Q tile's P.V done).
  auto k_full = [&](int st) { return bar0 + 8u * st; };
  auto k_empty = [&](int st) { return bar0 + 8u * (NK + st); };
  auto vraw_full = [&](int st) { return bar0 + 8u * (2 * NK + st); };
  auto vt_full = [&](int st) { return bar0 + 8u * (2 * NK + NV + st); };
  auto v_empty = [&](int st) { return bar0 + 8u * (2 * NK + 2 * NV + st); };
  constexpr int B1 = 2 * NK + 3 * NV;
  // Per Q tile t: S ready, S read (free), P written, P.V done (P free).
  auto s_full = [&](int t) { return bar0 + 8u * (B1 + t); };
  auto s_free = [&](int t) { return bar0 + 8u * (B1 + QT + t); };
  auto p_full = [&](int t) { return bar0 + 8u * (B1 + 2 * QT + t); };
  auto p_free = [&](int t) { return bar0 + 8u * (B1 + 3 * QT + t); };
  auto drain = [&](int t) { return bar0 + 8u * (B1 + 4 * QT + t); };
  auto o_last = [&](int t) { return bar0 + 8u * (B1 + 5 * QT + t); };  // last P.V (single use)
  // FP8 pools: raw code tiles landed / converted.
  auto raw_full = [&](int rs) { return bar0 + 8u * (B1 + 6 * QT + rs); };
  auto raw_empty = [&](int rs) { return bar0 + 8u * (B1 + 6 * QT + NR + rs); };
  // Tile A's first S done (single use): tile B's issuer starts after it.
  const uint32_t a_first = bar0 + 8u * (B1 + 6 * QT + 2 * NR);
  // bf16 pools: per V stage, 1 + the last tile whose values need the bf16
  // two-part P path (written by the converters before they arrive on
  // vt_full; tile indices only grow, so nothing is ever cleared).
  volatile int* wide_tile = reinterpret_cast<volatile int*>(smem + Cfg::kFlagOff);
  const uint32_t users = half < 0 ? QT : 1;  // active Q tiles: S and P.V readers of a tile
  if (threadIdx.x == 0) {
    for (int st = 0; st < NK; ++st) {
      // 16-bit pools: the copy completes a key tile; FP8 pools: every key
      // converter thread arrives once it has widened its part.
      mbar_init(k_full(st), KV8 ? Cfg::kConvKThreads : 1);
      mbar_init(k_empty(st), users);
    }
    for (int st = 0; st < NV; ++st) {
      mbar_init(vraw_full(st), 1);
      mbar_init(vt_full(st), Cfg::kConvVThreads);
      mbar_init(v_empty(st), users);
      wide_tile[st] = 0;
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
      const int h = c >> 3, cc = c & 7;
      *reinterpret_cast<uint4*>(qt + h * Cfg::kHalfBytes + rr * 128 + ((cc ^ (rr & 7)) << 4)) =
          qv[c];
    }
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *slot;
  bool failed = false;
  // FP8 pools: fp16 P in two parts (a second P.V MMA) when the head's value
  // scale makes one part too coarse (fp8_split_p, shared with the FP8 decode
  // kernels).  bf16 pools decide per tile (wide_tile).
  bool split_p = false;
  if constexpr (KV8) split_p = fp8_split_p<T>(p.v_scale[kvh]);

  if (warp == Cfg::kProducerWarp) {
    // ---- producer: K and V tiles ------------------------------------------
    // 16-bit pools: key tiles into the K ring and raw value tiles into the V
    // ring, each as soon as its slot is free (keys first: they are needed a
    // step earlier).  FP8 pools: raw code tiles into their own ring, for the
    // converter warps.
    const uint64_t policy = policy_evict_last();
    const int oob_block = p.num_blocks > 0x7FFFFFFF ? 0x7FFFFFFF : (int)p.num_blocks;
    // One tensor's tile j (64 keys): boxes of RB rows; boxes wholly past the
    // last needed key read an out-of-range block, which the copy fills with
    // zeros.
    auto load_tile = [&](const CUtensorMap* map, uint32_t dst, int j, uint32_t bar) {
      if (lane < Cfg::kBoxes) {
        const int pos = j * KT + lane * RB;
        int pb = oob_block, row = 0;
        if (pos < n_keys) {
          pb = trow[pos / BS];
          row = pos % BS;
        }
        if constexpr (KV8) {  // rows of 128 codes: one box per RB rows
          tma_load_4d(dst + lane * RB * 128, map, 0, row, kvh, pb, bar, policy);
        } else {
#pragma unroll
          for (int h = 0; h < Cfg::kHalves; ++h)
            tma_load_4d(dst + h * Cfg::kKvHalfBytes + lane * RB * 128, map, h * 64, row, kvh, pb,
                        bar, policy);
        }
      }
    };
    if constexpr (KV8) {
      int issued = 0;
      for (int j = 0; j < n_tiles; ++j) {
        const int rs = j % NR;
        if (j >= NR) {
          const bool ok = mbar_wait(raw_empty(rs), (uint32_t)(((j / NR) - 1) & 1));
          if (__any_sync(kFullMask, !ok)) {
            failed = true;
            break;
          }
        }
        const uint32_t dst = sbase + Cfg::kRawOff + rs * 2 * Cfg::kRawBytes;
        if (lane == 0) mbar_arrive_expect_tx(raw_full(rs), 2 * Cfg::kRawBytes);
        __syncwarp();
        load_tile(&tmk, dst, j, raw_full(rs));
        load_tile(&tmv, dst + Cfg::kRawBytes, j, raw_full(rs));
        issued = j + 1;
      }
      // Copies issued but possibly never consumed (another role stopped).
      for (int j = issued - NR < 0 ? 0 : issued - NR; j < issued; ++j)
        mbar_wait(raw_full(j % NR), (uint32_t)((j / NR) & 1), kWaitLimitNs / 8);
    } else {
      int jk = 0, jv = 0;
      uint64_t idle_since = 0;
      while (jk < n_tiles || jv < n_tiles) {
        bool progress = false;
        if (jk < n_tiles) {
          bool ready = jk < NK;
          if (!ready && lane == 0)
            ready = mbar_test_wait(k_empty(jk % NK), (uint32_t)(((jk / NK) - 1) & 1));
          if (__shfl_sync(kFullMask, ready, 0)) {
            const int st = jk % NK;
            if (lane == 0) mbar_arrive_expect_tx(k_full(st), Cfg::kKvBytes);
            __syncwarp();
            load_tile(&tmk, sbase + Cfg::kKRingOff + st * Cfg::kKvBytes, jk, k_full(st));
            ++jk;
            progress = true;
          }
        }
        if (jv < jk) {
          bool ready = jv < NV;
          if (!ready && lane == 0)
            ready = mbar_test_wait(v_empty(jv % NV), (uint32_t)(((jv / NV) - 1) & 1));
          if (__shfl_sync(kFullMask, ready, 0)) {
            const int st = jv % NV;
            if (lane == 0) mbar_arrive_expect_tx(vraw_full(st), Cfg::kKvBytes);
            __syncwarp();
            load_tile(&tmv, sbase + Cfg::kVRingOff + st * Cfg::kVStageBytes, jv, vraw_full(st));
            ++jv;
            progress = true;
          }
        }
        // Bounded like every other wait: give up after kWaitLimitNs without
        // progress.
        if (progress) {
          idle_since = 0;
        } else {
          const uint64_t now = global_ns();
          if (idle_since == 0) idle_since = now;
          if (__shfl_sync(kFullMask, now - idle_since > kWaitLimitNs, 0)) {
            failed = true;
            break;
          }
        }
      }
      // Copies issued but possibly never consumed (another role stopped).
      for (int j = jk - NK < 0 ? 0 : jk - NK; j < jk; ++j)
        mbar_wait(k_full(j % NK), (uint32_t)((j / NK) & 1), kWaitLimitNs / 8);
      for (int j = jv - NV < 0 ? 0 : jv - NV; j < jv; ++j)
        mbar_wait(vraw_full(j % NV), (uint32_t)((j / NV) & 1), kWaitLimitNs / 8);
    }
  } else if (warp >= Cfg::kMmaWarp && warp < Cfg::kMmaWarp + QT &&
             !active(warp - Cfg::kMmaWarp)) {
    // The issuer of a Q tile this CTA does not run has nothing to do.
  } else if (warp >= Cfg::kMmaWarp && warp < Cfg::kMmaWarp + QT) {
    // ---- MMA issuers, one per Q tile t: S_t(0); then per K/V tile j:
    //      S_t(j+1) once the softmax has read S_t(j) and key tile j+1 is in,
    //      and P.V_t(j) once P_t(j) and V^T(j) are written.  The next S is
    //      computed while the softmax works on the current one.  Separate
    //      issuers keep one tile's waits from holding up the other's MMAs
    //      (commits track each thread's own MMAs), and two issuers keep the
    //      tensor pipe fed faster than one thread can issue.
    auto wait_all = [&](uint32_t bar, int phase) {
      const bool o = mbar_wait(bar, (uint32_t)(phase & 1));
      return !__any_sync(kFullMask, !o);
    };
    // The issuing thread's own instruction chain between two MMAs sets how
    // fast it can feed the tensor pipe, so descriptors are built once and
    // stepped by constants: a descriptor's start address is its low 14 bits
    // in 16-byte units, and every operand here lies below 256 KB, so adding
    // (bytes >> 4) moves the start without touching the other fields.
    const uint32_t tbase = tmem + (warp - Cfg::kMmaWarp) * Cfg::kTileCols;
    const uint64_t kdesc0 = smem_desc_sw128(sbase + Cfg::kKRingOff, 16, 1024);
    const uint64_t vtdesc0 = smem_desc_sw128(sbase + Cfg::kVRingOff + Cfg::kVrawBytes, 16, 1024);
    const uint64_t vrawdesc0 = smem_desc_sw128(
        sbase + Cfg::kVRingOff, Cfg::kHalves > 1 ? Cfg::kKvHalfBytes : 1024, 1024);
    const uint64_t qdesc =
        smem_desc_sw128(sbase + Cfg::kQOff + (warp - Cfg::kMmaWarp) * Cfg::kTileBytes, 16, 1024);
    // S = Q.K^T: A = the Q tile, B = the key tile (both K-major).
    auto issue_s = [&](int tt, int j) {
      if (lane == 0) {
        const uint64_t kb = kdesc0 + (uint64_t)(((j % NK) * Cfg::kKvBytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          tc_mma_ss(tbase + Cfg::kSCol,
                    qdesc + (uint64_t)((((kk >> 2) * Cfg::kHalfBytes) + (kk & 3) * 32) >> 4),
                    kb + (uint64_t)((((kk >> 2) * Cfg::kKvHalfBytes) + (kk & 3) * 32) >> 4),
                    Cfg::kIdescS, kk > 0 ? 1u : 0u);
        tc_commit(s_full(tt));
        tc_commit(k_empty(j % NK));
      }
      __syncwarp();
    };
    // P.V of K/V tile j, A = P_t in tensor memory (keys 16kk .. 16kk+15 in
    // columns 8kk .. 8kk+7, a low part 32 columns on): fp16 P against V^T
    // (K-major) or against the FP8 pool's widened values (MN-major), or, on
    // a bf16 tile whose values need it, bf16 P as high and low parts against
    // the raw value tile (MN-major: 64-dim atoms kKvHalfBytes apart, 8-key
    // groups 1024 B apart; with one atom (D = 64) the atom stride is unused).
    auto issue_pv = [&](int tt, int j, bool wide) {
      if (lane == 0) {
        const uint32_t dcol = tbase + Cfg::kOCol, pa = tbase + Cfg::kPCol;
        const uint64_t voff = (uint64_t)(((j % NV) * Cfg::kVStageBytes) >> 4);
        if constexpr (KV8) {
          const uint64_t vb = vrawdesc0 + voff;
          auto run = [&](auto split_tag) {
#pragma unroll
            for (int kk = 0; kk < KT / 16; ++kk) {
              tc_mma_ts(dcol, pa + 8 * kk, vb + 128 * kk, Cfg::kIdescPV8,
                        (j > 0 || kk > 0) ? 1u : 0u);
              if constexpr (decltype(split_tag)::value)
                tc_mma_ts(dcol, pa + 32 + 8 * kk, vb + 128 * kk, Cfg::kIdescPV8, 1u);
            }
          };
          if (split_p) run(std::true_type{});
          else run(std::false_type{});
        } else if (!wide) {
          const uint64_t vb = vtdesc0 + voff;
#pragma unroll
          for (int kk = 0; kk < KT / 16; ++kk)
            tc_mma_ts(dcol, pa + 8 * kk, vb + 2 * kk, Cfg::kIdescPV, (j > 0 || kk > 0) ? 1u : 0u);
        } else {
          const uint64_t vb = vrawdesc0 + voff;
#pragma unroll
          for (int kk = 0; kk < KT / 16; ++kk) {
            tc_mma_ts(dcol, pa + 8 * kk, vb + 128 * kk, Cfg::kIdescPVWide,
                      (j > 0 || kk > 0) ? 1u : 0u);
            tc_mma_ts(dcol, pa + 32 + 8 * kk, vb + 128 * kk, Cfg::kIdescPVWide, 1u);
          }
        }
        tc_commit(p_free(tt));
        tc_commit(v_empty(j % NV));
      }
      __syncwarp();
    };
    const int tq = warp - Cfg::kMmaWarp;  // this issuer's Q tile
    bool ok = wait_all(k_full(0), 0);
    // Tile B starts once tile A's first S is done, so that the two tiles'
    // softmax passes are staggered rather than in step.
    if (ok && tq == 1 && half < 0) ok = wait_all(a_first, 0);
    if (ok) {
      tc_fence_after();
      issue_s(tq, 0);
      if (tq == 0 && lane == 0) tc_commit(a_first);
    }
    for (int j = 0; j < n_tiles && ok; ++j) {
      if (j + 1 < n_tiles) {
        ok = wait_all(k_full((j + 1) % NK), (j + 1) / NK) && wait_all(s_free(tq), j);
        if (!ok) break;
        tc_fence_after();
        issue_s(tq, j + 1);
      }
      ok = wait_all(p_full(tq), j) && wait_all(vt_full(j % NV), j / NV);
      if (!ok) break;
      // (Value positions past the last needed key are zeros in V^T and, on
      // bf16 pools, in the raw tile: the converters write them.)
      const bool wide = Cfg::kWideCheck && wide_tile[j % NV] == j + 1;
      tc_fence_after();
      issue_pv(tq, j, wide);
    }
    if (ok && lane == 0) tc_commit(o_last(tq));
    failed = !ok;
    // Every MMA this thread issued has completed before the tensor memory
    // is released.
    if (lane == 0) tc_commit(drain(tq));
    __syncwarp();
    mbar_wait(drain(tq), 0);
  } else if (warp >= Cfg::kConvWarp) {
    // ---- converters: value tiles -> V^T (fp16, K-major); on FP8 pools the
    //      first two warps widen the key codes instead --------------------
    // V^T row d holds dimension d of the tile's 64 keys.  Key positions at
    // or past the last needed key are written as zeros (stale contents
    // could be NaN, and 0 * NaN would poison O).
    const int cw = warp - Cfg::kConvWarp;
    const int ct = threadIdx.x - Cfg::kConvWarp * 32;
    const int vw = cw;                     // value warp index
    constexpr int kVWarps = Cfg::kConvWarps;
    for (int j = 0; j < n_tiles; ++j) {
      const int sv = j % NV;
      const int valid = n_keys - j * KT;  // keys of this tile that are needed
      const uint32_t vstage = sbase + Cfg::kVRingOff + sv * Cfg::kVStageBytes;
      const uint32_t vt = vstage + Cfg::kVrawBytes;
      if constexpr (KV8) {
        const int rs = j % NR, sk = j % NK;
        bool ok = mbar_wait(raw_full(rs), (uint32_t)((j / NR) & 1));
        if (ok && j >= NK) ok = mbar_wait(k_empty(sk), (uint32_t)(((j / NK) - 1) & 1));
        if (__any_sync(kFullMask, !ok)) {
          failed = true;
          break;
        }
        const unsigned char* kraw = smem + Cfg::kRawOff + rs * 2 * Cfg::kRawBytes;
        {
          // Keys: 16-code chunk ch of key row r (swizzled in the raw tile)
          // becomes dims 16ch .. 16ch+15, two 16-byte chunks of the
          // 128-byte-swizzled fp16 K tile.
          unsigned char* kop = smem + Cfg::kKRingOff + sk * Cfg::kKvBytes;
#pragma unroll
          for (int i = 0; i < KT * 8 / Cfg::kConvThreads; ++i) {
            const int unit = ct + i * Cfg::kConvThreads;
            const int row = unit >> 3, ch = unit & 7;
            const uint4 c =
                *reinterpret_cast<const uint4*>(kraw + row * 128 + ((ch ^ (row & 7)) << 4));
            uint4 lo, hi;
            e4m3x4_to_f16x4(c.x, lo.x, lo.y);
            e4m3x4_to_f16x4(c.y, lo.z, lo.w);
            e4m3x4_to_f16x4(c.z, hi.x, hi.y);
            e4m3x4_to_f16x4(c.w, hi.z, hi.w);
            const int c2 = (ch & 3) * 2;
            unsigned char* drow = kop + (ch >> 2) * Cfg::kKvHalfBytes + row * 128;
            *reinterpret_cast<uint4*>(drow + ((c2 ^ (row & 7)) << 4)) = lo;
            *reinterpret_cast<uint4*>(drow + (((c2 + 1) ^ (row & 7)) << 4)) = hi;
          }
          fence_proxy_async_smem();
          mbar_arrive(k_full(sk));
        }
        ok = j < NV || mbar_wait(v_empty(sv), (uint32_t)(((j / NV) - 1) & 1));
        if (__any_sync(kFullMask, !ok)) {
          failed = true;
          break;
        }
        {
          // Values: widened the same way into an fp16 tile of 64 key rows
          // (MN-major for P.V: transposing 8-bit codes costs the converters
          // more than the MN-major operand costs the tensor pipe).  Rows at
          // or past the last needed key are zeros.
          const unsigned char* vraw = kraw + Cfg::kRawBytes;
          unsigned char* vop = smem + Cfg::kVRingOff + sv * Cfg::kVStageBytes;
#pragma unroll
          for (int i = 0; i < KT * 8 / Cfg::kConvThreads; ++i) {
            const int unit = ct + i * Cfg::kConvThreads;
            const int row = unit >> 3, ch = unit & 7;
            uint4 lo = make_uint4(0u, 0u, 0u, 0u), hi = lo;
            if (row < valid) {
              const uint4 c =
                  *reinterpret_cast<const uint4*>(vraw + row * 128 + ((ch ^ (row & 7)) << 4));
              e4m3x4_to_f16x4(c.x, lo.x, lo.y);
              e4m3x4_to_f16x4(c.y, lo.z, lo.w);
              e4m3x4_to_f16x4(c.z, hi.x, hi.y);
              e4m3x4_to_f16x4(c.w, hi.z, hi.w);
            }
            const int c2 = (ch & 3) * 2;
            unsigned char* drow = vop + (ch >> 2) * Cfg::kKvHalfBytes + row * 128;
            *reinterpret_cast<uint4*>(drow + ((c2 ^ (row & 7)) << 4)) = lo;
            *reinterpret_cast<uint4*>(drow + (((c2 + 1) ^ (row & 7)) << 4)) = hi;
          }
          fence_proxy_async_smem();
          mbar_arrive(vt_full(sv));
        }
        mbar_arrive(raw_empty(rs));
      } else {
        const bool ok = mbar_wait(vraw_full(sv), (uint32_t)((j / NV) & 1));
        if (__any_sync(kFullMask, !ok)) {
          failed = true;
          break;
        }
        // 8 x 8 blocks (8 keys x 8 dims) through ldmatrix.trans (lane t gets
        // keys 2 (t % 4), 2 (t % 4) + 1 of dim t / 4) and stmatrix into V^T
        // rows; four blocks of one 8-key group per instruction.
        const uint32_t vraw = vstage;
        constexpr int kOps = (KT / 8) * (D / 32);  // 4 blocks of 8 dims per op
        float amax = 0.f;
#pragma unroll
        for (int u = 0; u < kOps / kVWarps; ++u) {
          const int op = vw * (kOps / kVWarps) + u;
          const int kb = op / (D / 32), d32 = op % (D / 32);
          const int m = lane >> 3, r8 = lane & 7;
          const int db = 4 * d32 + m;            // this lane's block of 8 dims
          const int key = 8 * kb + r8;           // row it addresses (ldmatrix)
          uint32_t r[4];
          ldsm_x4_trans(r, vraw + (db >> 3) * Cfg::kKvHalfBytes + key * 128 +
                               (((db & 7) ^ (key & 7)) << 4));
          const int k0 = 8 * kb + 2 * (lane & 3);
          const bool v0 = k0 < valid, v1 = k0 + 1 < valid;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            float lo, hi;
            if constexpr (std::is_same<T, __nv_bfloat16>::value) {
              lo = __uint_as_float(r[q] << 16);
              hi = __uint_as_float(r[q] & 0xFFFF0000u);
            } else {
              const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&r[q]));
              lo = f.x;
              hi = f.y;
            }
            lo = v0 ? lo : 0.f;
            hi = v1 ? hi : 0.f;
            amax = fmaxf(amax, fmaxf(fabsf(lo), fabsf(hi)));
            r[q] = pack_pair<__half>(lo, hi);
          }
          const int drow = 8 * db + r8;          // V^T row this lane addresses (stmatrix)
          stsm_x4(vt + drow * 128 + ((kb ^ (drow & 7)) << 4), r);
        }
        if constexpr (Cfg::kWideCheck) {
          // Tiles with a value above kWideLimit (or beyond fp16's range) take
          // the bf16 path, which reads the raw tile: its rows past the last
          // needed key are zeroed too.
          const bool big = __any_sync(kFullMask, !(amax <= Cfg::kWideLimit));
          if (big && lane == 0) atomicMax(const_cast<int*>(wide_tile) + sv, j + 1);
          if (valid < KT) {
            unsigned char* raw = smem + Cfg::kVRingOff + sv * Cfg::kVStageBytes;
            for (int e = ct; e < (KT - valid) * Cfg::kHalves * 8; e += Cfg::kConvThreads) {
              const int row = valid + e / (Cfg::kHalves * 8);
              const int rest = e % (Cfg::kHalves * 8);
              *reinterpret_cast<uint4*>(raw + (rest >> 3) * Cfg::kKvHalfBytes + row * 128 +
                                        (rest & 7) * 16) = make_uint4(0u, 0u, 0u, 0u);
            }
          }
        }
        fence_proxy_async_smem();
        mbar_arrive(vt_full(sv));
      }
    }
  } else if (!active(t)) {
    // Softmax warps of a Q tile this CTA does not run have nothing to do.
  } else {
    // ---- softmax, row rr of Q tile t ----------------------------------------
    // FP8 pools compile this role twice, with and without two-part P, and
    // choose once per CTA: no per-tile test of the form stays in its loop.
    auto softmax_role = [&](auto split_tag) {
      constexpr bool SPLIT = decltype(split_tag)::value;
      const int pos = first + qi;
      const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
      const uint32_t scol = t * Cfg::kTileCols + Cfg::kSCol, pcol = t * Cfg::kTileCols + Cfg::kPCol,
                     ocol = t * Cfg::kTileCols + Cfg::kOCol;
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
        // P: keys 2c, 2c+1 in column c (high part, or the only one); a low
        // part of the same keys in column 32 + c.  fp16 unless this is a bf16
        // tile whose values need the bf16 two-part path (the converters'
        // decision on tile j, published before they arrive on vt_full).
        bool wide = false;
        if constexpr (Cfg::kWideCheck) {
          const bool got = mbar_wait(vt_full(j % NV), (uint32_t)((j / NV) & 1));
          if (__any_sync(kFullMask, !got)) {
            ok = false;
            break;
          }
          wide = wide_tile[j % NV] == j + 1;
        }
        // P: keys 2c, 2c+1 in column c, a low part in column 32 + c: one fp16
        // part; or, on a bf16 tile whose values need it, the truncated bf16
        // value and the remainder rounded to bf16; or, for FP8 heads whose
        // value scale needs it, the fp16 value and the remainder rounded to
        // fp16.  FP8 pools choose between their two forms once per CTA and
        // run a packing loop compiled for one form (fewer live registers);
        // bf16 pools decide per tile inside the loop, which measured faster
        // than two copies of it.
        uint32_t pk[KT];
        const bool two_parts = wide || SPLIT;
        if constexpr (KV8) {
          auto pack = [&](auto split_tag) {
  #pragma unroll
            for (int c = 0; c < KT / 2; ++c) {
              const float a = __uint_as_float(w[2 * c]), b = __uint_as_float(w[2 * c + 1]);
              const __half2 hi = __floats2half2_rn(a, b);
              pk[c] = *reinterpret_cast<const uint32_t*>(&hi);
              if constexpr (decltype(split_tag)::value) {
                const float2 hf = __half22float2(hi);
                pk[KT / 2 + c] = pack_pair<__half>(a - hf.x, b - hf.y);
              }
            }
          };
          pack(std::integral_constant<bool, SPLIT>{});
        } else {
  #pragma unroll
          for (int c = 0; c < KT / 2; ++c) {
            const uint32_t a = w[2 * c], b = w[2 * c + 1];
            if (wide) {
              pk[c] = __byte_perm(a, b, 0x7632);  // upper halves: truncated bf16
              // exact remainders p - trunc(p), rounded to bf16
              const float2 r = __ffma2_rn(
                  make_float2(__uint_as_float(a & 0xFFFF0000u), __uint_as_float(b & 0xFFFF0000u)),
                  make_float2(-1.f, -1.f), make_float2(__uint_as_float(a), __uint_as_float(b)));
              pk[KT / 2 + c] = pack_pair<__nv_bfloat16>(r.x, r.y);
            } else {
              pk[c] = pack_pair<__half>(__uint_as_float(a), __uint_as_float(b));
              pk[KT / 2 + c] = 0u;
            }
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
        if (two_parts) {
          tmem_st64(lane_base + pcol, pk);
        } else {
          tmem_st32(lane_base + pcol, *reinterpret_cast<const uint32_t(*)[32]>(pk));
        }
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
            auto o = [&](int d) { return __uint_as_float(w[d]) * inv; };
  #pragma unroll
            for (int v = 0; v < 4; ++v) {
              uint4 u;
              u.x = pack_pair<T>(o(8 * v + 0), o(8 * v + 1));
              u.y = pack_pair<T>(o(8 * v + 2), o(8 * v + 3));
              u.z = pack_pair<T>(o(8 * v + 4), o(8 * v + 5));
              u.w = pack_pair<T>(o(8 * v + 6), o(8 * v + 7));
              orow[c4 * 4 + v] = u;
            }
          }
        }
      }
    };
    if constexpr (KV8) {
      if (split_p) softmax_role(std::true_type{});
      else softmax_role(std::false_type{});
    } else {
      softmax_role(std::false_type{});
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
