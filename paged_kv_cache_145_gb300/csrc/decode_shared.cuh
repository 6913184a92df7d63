// Decode attention for groups of sequences that share a prefix of their
// block tables: forks of one prompt in parallel sampling or beam search
// ("vLLM and PagedAttention: Virtual Memory for LLM Serving", sharing
// paragraph: sequences that branch from one prompt share its blocks;
// "Inside vLLM and TGI: Paging, Versioned Schedulers and Operations",
// "Exact CPU block manager and copy-on-write": a fork shares every block of
// its parent until a write needs a private copy).
//
// A group is a run of consecutive sequences [group_starts[g],
// group_starts[g+1]) whose tables name the same physical blocks for their
// first group_prefix[g] positions.  The plain decode reads those pages once
// per sequence; here the partitions that lie wholly inside the shared
// prefix are computed once per (group, KV head) for all members' queries
// stacked together: with 8 forks and 4 query heads per KV head that is 32
// query rows against each K/V tile, a dense contraction.  Each member's
// partial (m, l, o) of such a partition goes to the same workspace slot the
// plain partition pass would have written; the plain partition pass skips
// those partitions, and the split-K merge combines them with the member's
// own tail unchanged (or, when every tail fits in one partition,
// decode_tail_merge_kernel below computes the tails and merges).
//
// Kernel (this library's design), on the fifth-generation tensor cores:
// grid (KV head, group, shared partition x row block).  The 128 rows of
// the MMAs (tensor-memory lanes) hold a row block's stacked rows (member
// r / G, query head r % G), each DUP times: 128 rows once, or, for groups
// of at most 32 stacked rows, every row four times, so that the four
// copies split each key tile's softmax work between them.  Keys stream in
// tiles of 64 positions, read through the group's first member's table.
// Six warps:
//   warps 0-3  softmax: thread = one copy of a row, lane = tensor-memory
//              lane: loads its S row, takes its 64 / DUP keys of it, keeps
//              the running maximum (shared by the copies; raised lazily,
//              only when a tile's maximum exceeds it by more than 2^8) and
//              its part of the sum, writes P for its keys (zeros for the
//              others) into its columns, rescales its O row when the
//              maximum moves; at the end the copies' O rows and sums add up
//              to the row's, which the copies write together; warps with no
//              real row idle;
//   warp 4     producer: 4-D TMA tile loads (128-byte swizzle) of key and
//              value tiles into two rings (values stay longer: three stages
//              against two for keys), reading the table one tile ahead;
//              allocates the tensor memory;
//   warp 5     MMA issuer (one thread): S = Q.K^T (A = the stacked query
//              rows, B = the key tile, both K-major in shared memory, 128 x
//              64 x D), and O += P.V (A = P in tensor memory, B = the value
//              tile as copied, read MN-major, 128 x D x 64).  bf16 pools
//              take P in two bf16 parts, the truncated weight and its
//              rounded remainder (about 16 bits of P); fp16 pools one fp16
//              part.  S of the next tile is issued while the softmax works
//              on the current one.
// Tensor memory (256 columns): S at 0 (64), P at 64 (64: keys 2c, 2c+1 in
// column c, a low part in 32 + c), O at 128 (D).  Shared memory: barriers
// and flags in the first KiB, then the query rows and the two rings, 1 KiB
// aligned (the dynamic base must be, else the kernel flags PKV_DEV_LAUNCH
// and computes nothing); two CTAs fit on an SM and a third does not, so
// their tensor-memory allocations always fit.  Every wait is bounded; on a
// timeout the roles stop, the issuer waits for its MMAs, the producer for
// its copies, and the tensor memory is released.
//
// Ownership.  Sequence s belongs to group shared_owner(s); this kernel and
// the partition pass both use that rule, so a malformed list can only leave
// sequences without a group (decoded plainly), never covered twice or not
// at all.  Checked per row: the length lies in [1, max_len] (else the row is
// left to the plain path's invalid-length handling), covers the partition,
// and the table names the leader's blocks for it; otherwise the row's
// partial is marked invalid (the merge writes zeros) and PKV_DEV_SHARING is
// set.
#pragma once

#include <type_traits>

#include "decode_mma.cuh"
#include "tcgen05.cuh"

namespace pkv {

template <typename T, int D, int BS, int G, int DUP>
struct SharedTcCfg {
  static constexpr int kLanes = 128;                       // MMA rows = tensor-memory lanes
  static constexpr int kDup = DUP;                         // copies of each stacked row
  static constexpr int kRowsPerWarp = 32 / DUP;            // stacked rows per softmax warp
  static constexpr int kRows = 4 * kRowsPerWarp;           // stacked rows per CTA
  static constexpr int kKeysPerCopy = 64 / DUP;
  static constexpr int kDimsPerCopy = 32 / DUP;            // of each 32-dim chunk of O
  static constexpr int kKeys = 64;                         // positions per K/V tile
  static constexpr int kHalves = D / 64;                   // 128-byte column blocks of a row
  static constexpr int kQHalfBytes = kLanes * 128;
  static constexpr int kQBytes = kHalves * kQHalfBytes;    // the stacked query rows
  static constexpr int kKvHalfBytes = kKeys * 128;
  static constexpr int kKvBytes = kHalves * kKvHalfBytes;  // one key (or value) tile
  static constexpr int kKStages = D == 64 ? 4 : 2;
  static constexpr int kVStages = D == 64 ? 6 : 3;
  static constexpr int kBoxRows = BS < 16 ? BS : 16;
  static constexpr int kBoxes = kKeys / kBoxRows;          // TMA boxes per tile per column block
  static constexpr int kProducerWarp = 4;
  static constexpr int kMmaWarp = 5;
  static constexpr int kThreads = 6 * 32;
  // First KiB: barriers, the tensor-memory slot, per-member flags.
  static constexpr int kNumBars = 2 * kKStages + 2 * kVStages + 6;
  static constexpr int kBarOff = 0;
  static constexpr int kSlotOff = 256;
  static constexpr int kMemberOff = 512;                   // per member of the row block: mismatch
  static constexpr int kQOff = 1024;
  static constexpr int kKRingOff = kQOff + kQBytes;
  static constexpr int kVRingOff = kKRingOff + kKStages * kKvBytes;
  static constexpr int kSmemBytes = kVRingOff + kVStages * kKvBytes;
  static constexpr uint32_t kTmemCols = 256;
  static constexpr uint32_t kSCol = 0, kPCol = 64, kOCol = 128;
  static constexpr bool kTwoPartP = std::is_same<T, __nv_bfloat16>::value;
  static constexpr uint32_t kFmt = kTwoPartP ? 1u : 0u;
  static constexpr uint32_t kIdescS = idesc_f16(kFmt, 128, kKeys, false);
  static constexpr uint32_t kIdescPV = idesc_f16(kFmt, 128, D, true);
  // An SM holds 228 KiB of shared memory, 1 KiB of it reserved per CTA.
  static_assert(2 * (kSmemBytes + 1024) <= 228 * 1024, "two CTAs per SM");
  static_assert(3 * (kSmemBytes + 1024) > 228 * 1024, "not three (tensor memory)");
  static_assert(kNumBars * 8 <= kSlotOff && kMemberOff + kRows * 4 <= kQOff, "header");
  static_assert(kOCol + D <= kTmemCols, "tensor memory");
  static_assert(kQBytes % 1024 == 0 && kKvBytes % 1024 == 0, "128-byte swizzle atoms");
  static_assert(kBoxes <= 32 && D % 64 == 0 && G <= 8, "geometry");
  static_assert(DUP == 1 || DUP == 2 || DUP == 4, "copies of a row: adjacent lanes");
};

template <typename T, int D, int BS, int G, int DUP>
__global__ void __launch_bounds__(SharedTcCfg<T, D, BS, G, DUP>::kThreads)
decode_shared_prefix_kernel(const DecodeParams p, int row_blocks,
                            const __grid_constant__ CUtensorMap tmk,
                            const __grid_constant__ CUtensorMap tmv) {
  using Cfg = SharedTcCfg<T, D, BS, G, DUP>;
  constexpr int NK = Cfg::kKStages;
  constexpr int NV = Cfg::kVStages;
  constexpr int KT = Cfg::kKeys;
  constexpr int KW = Cfg::kKeysPerCopy;
  constexpr int DW = Cfg::kDimsPerCopy;
  constexpr int RB = Cfg::kBoxRows;
  extern __shared__ __align__(1024) unsigned char smem[];
  const uint32_t sbase = smem_addr(smem);
  if (sbase & 1023u) {  // the swizzled tiles need a 1 KiB aligned base
    if (threadIdx.x == 0) set_error(p.err, PKV_DEV_LAUNCH);
    return;
  }

  const int kvh = blockIdx.x;
  const int g = blockIdx.y;
  const int part = blockIdx.z / row_blocks;
  const int rb = blockIdx.z % row_blocks;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int H = p.num_heads;
  const int PS = p.part_size;
  T* out = static_cast<T*>(p.out);

  const int s0 = ld_nc(p.group_starts + g);
  const int s1 = min(ld_nc(p.group_starts + g + 1), p.num_seqs);
  const int pre = ld_nc(p.group_prefix + g);
  if (s0 < 0 || s1 <= s0 || pre < PS || part >= pre / PS) return;
  const int gsize = s1 - s0;
  const int row0 = rb * Cfg::kRows;  // first stacked row of this CTA
  const int nrows = min(Cfg::kRows, gsize * G - row0);
  if (nrows <= 0) return;
  const int tok0 = part * PS;
  const int blk0 = tok0 / BS;
  const int span = PS / BS;  // blocks of the partition
  const int n_tiles = (PS + KT - 1) / KT;
  const bool fits = blk0 + span <= p.max_blocks;
  const int32_t* lrow = p.tables + (int64_t)s0 * p.max_blocks + blk0;
  const int m_first = row0 / G;  // first member with a row here

  int* member_bad = reinterpret_cast<int*>(smem + Cfg::kMemberOff);
  const uint32_t bar0 = sbase + Cfg::kBarOff;
  auto k_full = [&](int st) { return bar0 + 8u * st; };
  auto k_empty = [&](int st) { return bar0 + 8u * (NK + st); };
  auto v_full = [&](int st) { return bar0 + 8u * (2 * NK + st); };
  auto v_empty = [&](int st) { return bar0 + 8u * (2 * NK + NV + st); };
  const uint32_t s_full = bar0 + 8u * (2 * NK + 2 * NV);  // S written
  const uint32_t s_free = s_full + 8;                      // S read by every softmax thread
  const uint32_t p_full = s_full + 16;                     // P written (and O rescaled)
  const uint32_t p_free = s_full + 24;                     // P.V done
  const uint32_t o_last = s_full + 32;                     // the last P.V done (single use)
  const uint32_t drain = s_full + 40;                      // every MMA done (single use)
  const int nsw = (nrows + Cfg::kRowsPerWarp - 1) / Cfg::kRowsPerWarp;  // warps with real rows
  if (threadIdx.x == 0) {
    for (int st = 0; st < NK; ++st) {
      mbar_init(k_full(st), 1);
      mbar_init(k_empty(st), 1);
    }
    for (int st = 0; st < NV; ++st) {
      mbar_init(v_full(st), 1);
      mbar_init(v_empty(st), 1);
    }
    mbar_init(s_full, 1);
    mbar_init(s_free, nsw * 32);
    mbar_init(p_full, nsw * 32);
    mbar_init(p_free, 1);
    mbar_init(o_last, 1);
    mbar_init(drain, 1);
    fence_mbar_init();
  }
  for (int i = threadIdx.x; i < Cfg::kRows; i += Cfg::kThreads) member_bad[i] = 0;
  __syncthreads();

  // ---- producer: key tile j into K stage j % NK, value tile j into V stage
  //      j % NV.  Lane b < kBoxes copies box b (RB positions); a box past the
  //      partition's end reads an out-of-range block, which the copy fills
  //      with zeros.  Its table entry is read one tile ahead.  The producer
  //      allocates the tensor memory and issues the tiles whose stages are
  //      free from the start at once, while the other warps check the rows
  //      and stage the queries (entries are range-checked below; a copy at
  //      an out-of-range coordinate only reads fill values).
  uint32_t* slot = reinterpret_cast<uint32_t*>(smem + Cfg::kSlotOff);
  const uint64_t policy = policy_evict_first();
  const int oob_block = p.num_blocks > 0x7FFFFFFF ? 0x7FFFFFFF : (int)p.num_blocks;
  auto entry = [&](int j) {
    const int pos = j * KT + lane * RB;
    return (fits && lane < Cfg::kBoxes && j < n_tiles && pos < PS)
               ? make_int2(ld_nc(lrow + pos / BS), pos % BS)
               : make_int2(oob_block, 0);
  };
  auto load_tile = [&](const CUtensorMap* map, uint32_t dst, int2 e, uint32_t bar) {
    if (lane < Cfg::kBoxes) {
#pragma unroll
      for (int h = 0; h < Cfg::kHalves; ++h)
        tma_load_4d(dst + h * Cfg::kKvHalfBytes + lane * RB * 128, map, h * 64, e.y, kvh, e.x,
                    bar, policy);
    }
  };
  int jk = 0, jv = 0;  // tiles whose key / value copies were issued
  int2 cur = make_int2(oob_block, 0);
  // Tile j's copies once its stages are free; false if a wait gave up.
  auto issue_tile = [&](int j) {
    const int2 nxt = entry(j + 1);
    const int sk = j % NK, sv = j % NV;
    if (j >= NK &&
        __any_sync(kFullMask, !mbar_wait(k_empty(sk), (uint32_t)(((j / NK) - 1) & 1))))
      return false;
    if (lane == 0) mbar_arrive_expect_tx(k_full(sk), Cfg::kKvBytes);
    __syncwarp();
    load_tile(&tmk, sbase + Cfg::kKRingOff + sk * Cfg::kKvBytes, cur, k_full(sk));
    jk = j + 1;
    if (j >= NV &&
        __any_sync(kFullMask, !mbar_wait(v_empty(sv), (uint32_t)(((j / NV) - 1) & 1))))
      return false;
    if (lane == 0) mbar_arrive_expect_tx(v_full(sv), Cfg::kKvBytes);
    __syncwarp();
    load_tile(&tmv, sbase + Cfg::kVRingOff + sv * Cfg::kKvBytes, cur, v_full(sv));
    jv = j + 1;
    cur = nxt;
    return true;
  };
  // Copies issued but possibly never consumed (another role stopped).
  auto drain_copies = [&]() {
    for (int j = jk - NK < 0 ? 0 : jk - NK; j < jk; ++j)
      mbar_wait(k_full(j % NK), (uint32_t)((j / NK) & 1), kWaitLimitNs / 8);
    for (int j = jv - NV < 0 ? 0 : jv - NV; j < jv; ++j)
      mbar_wait(v_full(j % NV), (uint32_t)((j / NV) & 1), kWaitLimitNs / 8);
  };
  const int npre = fits ? min(n_tiles, min(NK, NV)) : 0;  // no waits before these
  if (warp == Cfg::kProducerWarp) {
    tmem_alloc(smem_addr(slot), Cfg::kTmemCols);
    tmem_relinquish();
    cur = entry(0);
    for (int j = 0; j < npre; ++j) issue_tile(j);
  }

  // ---- rows: lane `lane` of softmax warp `warp` (tensor-memory lane
  // 32 warp + lane) is copy `cp` of stacked row R = row0 + r_local.  Loads
  // issued together: its length, its group (shared_owner), its member's
  // table entries for the partition against the leader's (the member's
  // threads in this CTA split them), the leader's entries (range check, all
  // threads), and the query row.  Status: 1 usable, 0 skip (not owned, or
  // an invalid length: the plain path zeroes it), -1 sharing contract
  // broken.
  const int cp = lane % DUP;
  const int r_local = warp * Cfg::kRowsPerWarp + lane / DUP;
  const int R = row0 + r_local;
  const bool has_row = warp < 4 && r_local < nrows;
  const int head = kvh * G + R % G;
  int my_seq = -1, my_status = 0, my_len = 0;
  uint4 qv[D / 8];
  if (has_row) {
    const int mi = R / G;
    const int s = s0 + mi;
    const uint4* qrow =
        reinterpret_cast<const uint4*>(static_cast<const T*>(p.q) + ((int64_t)s * H + head) * D);
#pragma unroll
    for (int c = 0; c < D / 8; ++c) qv[c] = qrow[c];
    const int L = ld_nc(p.seq_lens + s);
    const int own = shared_owner(p, s);
    if (fits) {
      const int r_lo = max(row0, mi * G), r_hi = min(row0 + nrows, (mi + 1) * G);
      const int32_t* row = p.tables + (int64_t)s * p.max_blocks + blk0;
      int mismatch = 0;
#pragma unroll 4
      for (int i = (R - r_lo) * DUP + cp; i < span; i += (r_hi - r_lo) * DUP)
        mismatch |= ld_nc(row + i) != ld_nc(lrow + i);
      if (mismatch) atomicOr(member_bad + (mi - m_first), 1);
    }
    if (own == g) {
      my_seq = s;
      my_len = L;
      my_status = (L < 1 || L > p.max_len) ? 0 : 1;
    }
  } else {
#pragma unroll
    for (int c = 0; c < D / 8; ++c) qv[c] = make_uint4(0u, 0u, 0u, 0u);
  }
  int bad = !fits;
  for (int i = threadIdx.x; fits && i < span; i += Cfg::kThreads) {
    const int e = ld_nc(lrow + i);
    bad |= (e < 0 || (int64_t)e >= p.num_blocks);
  }
  // The stacked query rows go to shared memory as soon as they arrive (a row
  // whose checks fail is computed all the same and its result dropped;
  // lanes without a row hold zeros).
  if (warp < 4) {
    const int qr = warp * 32 + lane;  // this thread's MMA row
#pragma unroll
    for (int c = 0; c < D / 8; ++c) {
      const int h = c >> 3, cc = c & 7;
      *reinterpret_cast<uint4*>(smem + Cfg::kQOff + h * Cfg::kQHalfBytes + qr * 128 +
                                ((cc ^ (qr & 7)) << 4)) = qv[c];
    }
    fence_proxy_async_smem();
  }
  // The leader's entries are unusable: every member's row is marked invalid.
  tc_fence_before();
  bad = __syncthreads_or(bad);
  tc_fence_after();
  if (has_row && my_status == 1 &&
      (bad || my_len < tok0 + PS || member_bad[R / G - m_first] != 0))
    my_status = -1;

  // ---- this copy's DW dims of a row's partial, from dim d0 (v: the row's
  //      sums): o = O / l with (m, l), or the invalid marker ----------------
  auto store_row = [&](bool broken, float m, float l, const uint32_t(&v)[DW], int d0) {
    const int nparts = (my_len + PS - 1) / PS;
    const float inv = broken ? 0.f : 1.f / l;
    auto f = [&](int d) { return broken ? 0.f : __uint_as_float(v[d]) * inv; };
    if (nparts == 1) {  // the whole sequence is this partition: final output
      uint4* orow = reinterpret_cast<uint4*>(out + ((int64_t)my_seq * H + head) * D + d0);
#pragma unroll
      for (int u = 0; u < DW / 8; ++u) {
        uint4 w;
        w.x = pack_pair<T>(f(8 * u + 0), f(8 * u + 1));
        w.y = pack_pair<T>(f(8 * u + 2), f(8 * u + 3));
        w.z = pack_pair<T>(f(8 * u + 4), f(8 * u + 5));
        w.w = pack_pair<T>(f(8 * u + 6), f(8 * u + 7));
        orow[u] = w;
      }
    } else {
      const int64_t w = ((int64_t)my_seq * H + head) * p.num_parts + part;
      float4* orow = reinterpret_cast<float4*>(p.ws_o + w * D + d0);
#pragma unroll
      for (int u = 0; u < DW / 4; ++u)
        orow[u] = make_float4(f(4 * u), f(4 * u + 1), f(4 * u + 2), f(4 * u + 3));
      if (d0 == 0) p.ws_ml[w] = broken ? make_float2(-INFINITY, -1.f) : make_float2(m, l);
    }
  };
  // Rows whose partial is the invalid marker: status -1, and with `all`
  // (nothing computed, or a wait gave up) every usable row too.
  auto mark_broken_rows = [&](bool all) {
    if (!has_row || my_status == 0 || (!all && my_status == 1)) return;
    if (my_status < 0 && cp == 0) set_error(p.err, PKV_DEV_SHARING);
    const uint32_t zero[DW] = {};
    for (int c0 = 0; c0 < D; c0 += 32) store_row(true, 0.f, 0.f, zero, c0 + cp * DW);
  };
  if (bad) {  // no tensor-core work: every usable row is now broken
    if (warp == Cfg::kProducerWarp) {
      drain_copies();
      tc_fence_before();
      __syncwarp();
      tc_fence_after();
      tmem_dealloc(*slot, Cfg::kTmemCols);
    }
    mark_broken_rows(true);
    return;
  }

  const uint32_t tmem = *slot;
  bool failed = false;

  if (warp == Cfg::kProducerWarp) {
    // ---- producer, continued: the remaining tiles as their stages free up
    for (int j = npre; j < n_tiles; ++j) {
      if (!issue_tile(j)) {
        failed = true;
        break;
      }
    }
    drain_copies();
  } else if (warp == Cfg::kMmaWarp) {
    // ---- MMA issuer: S(0); per tile j, S(j+1) once its keys are in and the
    //      softmax has read S(j), then P.V(j) once P(j) and the values are in.
    // Descriptors are built once and stepped by constants (a descriptor's
    // start address is its low 14 bits in 16-byte units; every operand lies
    // below 256 KB).
    auto wait_all = [&](uint32_t bar, int phase) {
      const bool o = mbar_wait(bar, (uint32_t)(phase & 1));
      return !__any_sync(kFullMask, !o);
    };
    const uint64_t qdesc = smem_desc_sw128(sbase + Cfg::kQOff, 16, 1024);
    const uint64_t kdesc0 = smem_desc_sw128(sbase + Cfg::kKRingOff, 16, 1024);
    // Values as copied, MN-major: 64-dim atoms kKvHalfBytes apart, 8-key
    // groups 1024 B apart (with one atom, D = 64, the atom stride is unused).
    const uint64_t vdesc0 = smem_desc_sw128(sbase + Cfg::kVRingOff,
                                            Cfg::kHalves > 1 ? Cfg::kKvHalfBytes : 1024, 1024);
    auto issue_s = [&](int j) {
      if (lane == 0) {
        const uint64_t kb = kdesc0 + (uint64_t)(((j % NK) * Cfg::kKvBytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          tc_mma_ss(tmem + Cfg::kSCol,
                    qdesc + (uint64_t)((((kk >> 2) * Cfg::kQHalfBytes) + (kk & 3) * 32) >> 4),
                    kb + (uint64_t)((((kk >> 2) * Cfg::kKvHalfBytes) + (kk & 3) * 32) >> 4),
                    Cfg::kIdescS, kk > 0 ? 1u : 0u);
        tc_commit(s_full);
        tc_commit(k_empty(j % NK));
      }
      __syncwarp();
    };
    // P.V of tile j: keys 16kk .. 16kk+15 of P in columns 8kk .. 8kk+7 (a
    // low part 32 columns on), value rows 16kk .. 16kk+15 2048 B apart.
    auto issue_pv = [&](int j) {
      if (lane == 0) {
        const uint64_t vb = vdesc0 + (uint64_t)(((j % NV) * Cfg::kKvBytes) >> 4);
        const uint32_t dcol = tmem + Cfg::kOCol, pa = tmem + Cfg::kPCol;
#pragma unroll
        for (int kk = 0; kk < KT / 16; ++kk) {
          tc_mma_ts(dcol, pa + 8 * kk, vb + 128 * kk, Cfg::kIdescPV, (j > 0 || kk > 0) ? 1u : 0u);
          if constexpr (Cfg::kTwoPartP)
            tc_mma_ts(dcol, pa + 32 + 8 * kk, vb + 128 * kk, Cfg::kIdescPV, 1u);
        }
        tc_commit(p_free);
        tc_commit(v_empty(j % NV));
      }
      __syncwarp();
    };
    bool ok = wait_all(k_full(0), 0);
    if (ok) {
      tc_fence_after();
      issue_s(0);
    }
    for (int j = 0; j < n_tiles && ok; ++j) {
      if (j + 1 < n_tiles) {
        ok = wait_all(k_full((j + 1) % NK), (j + 1) / NK) && wait_all(s_free, j);
        if (!ok) break;
        tc_fence_after();
        issue_s(j + 1);
      }
      ok = wait_all(p_full, j) && wait_all(v_full(j % NV), j / NV);
      if (!ok) break;
      tc_fence_after();
      issue_pv(j);
    }
    if (ok && lane == 0) tc_commit(o_last);
    failed = !ok;
    // Every MMA this thread issued has completed before the tensor memory
    // is released.
    if (lane == 0) tc_commit(drain);
    __syncwarp();
    mbar_wait(drain, 0);
  } else if (warp < nsw) {
    // ---- softmax: copy cp of row r_local, keys cp * KW .. cp * KW + KW - 1 ---
    const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
    // Scores are taken as s * |factor| with the sign folded into s, so the
    // row maximum can be found on the raw scores.
    const bool qneg = p.qscale < 0.f;
    const float qscale = fabsf(p.qscale);
    float m = -INFINITY, l = 0.f;  // l: this copy's part of the row's sum
    bool ok = true;
    for (int j = 0; j < n_tiles; ++j) {
      ok = mbar_wait(s_full, (uint32_t)(j & 1));
      if (__any_sync(kFullMask, !ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t x[KW];
      {
        uint32_t w[KT];
        tmem_ld64(lane_base + Cfg::kSCol, w);
#pragma unroll
        for (int i = 0; i < KW; ++i) {
          uint32_t v = w[i];
#pragma unroll
          for (int cc = 1; cc < DUP; ++cc)
            if (cp == cc) v = w[cc * KW + i];
          x[i] = v;
        }
      }
      tc_fence_before();
      mbar_arrive(s_free);
      if (qneg) {
#pragma unroll
        for (int i = 0; i < KW; ++i) x[i] ^= 0x80000000u;
      }
      // Positions past the partition's end (a last tile of fewer than 64).
      const int lim = PS - j * KT - cp * KW;
      if (lim < KW) {
#pragma unroll
        for (int i = 0; i < KW; ++i)
          if (i >= lim) x[i] = __float_as_uint(-INFINITY);
      }
      float mq[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int i = 0; i < KW; i += 8)
#pragma unroll
        for (int u = 0; u < 4; ++u)
          mq[u] = max3(mq[u], __uint_as_float(x[i + 2 * u]), __uint_as_float(x[i + 2 * u + 1]));
      float mraw = max3(mq[0], mq[1], fmaxf(mq[2], mq[3]));
#pragma unroll
      for (int sh = 1; sh < DUP; sh <<= 1) mraw = fmaxf(mraw, __shfl_xor_sync(kFullMask, mraw, sh));
      const float mx = mraw * qscale;
      // Lazy maximum: raise it (and rescale O and l) only when the tile's
      // maximum exceeds it by more than 8 (P <= 2^8 otherwise).  Tile 0
      // always holds a position of the partition, so m is finite after it.
      // The copies of a row see the same maximum and decide alike.
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
      // Weights 2^(s * scale - m); positions past the partition's end get 0
      // (set after the exponential, so that a zero scale cannot make NaN).
      const float2 qs2 = make_float2(qscale, qscale), nm2 = make_float2(-m, -m);
      float2 sum2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
      for (int i = 0; i < KW; i += 2) {
        const float2 a =
            __ffma2_rn(make_float2(__uint_as_float(x[i]), __uint_as_float(x[i + 1])), qs2, nm2);
        const float2 e = make_float2(i < lim ? ex2(a.x) : 0.f, i + 1 < lim ? ex2(a.y) : 0.f);
        x[i] = __float_as_uint(e.x);
        x[i + 1] = __float_as_uint(e.y);
        sum2[(i >> 1) & 1] = __fadd2_rn(sum2[(i >> 1) & 1], e);
      }
      const float2 sx = __fadd2_rn(sum2[0], sum2[1]);
      l += sx.x + sx.y;
      // P: keys 2c, 2c+1 in column c, this copy's keys only (zeros for the
      // other copies' keys).  bf16: the truncated weights, and in column
      // 32 + c the exact remainders rounded to bf16; fp16: one part.
      uint32_t hi[KW / 2], lo[KW / 2];
#pragma unroll
      for (int c = 0; c < KW / 2; ++c) {
        const uint32_t a = x[2 * c], b = x[2 * c + 1];
        if constexpr (Cfg::kTwoPartP) {
          hi[c] = __byte_perm(a, b, 0x7632);
          const float2 r = __ffma2_rn(
              make_float2(__uint_as_float(a & 0xFFFF0000u), __uint_as_float(b & 0xFFFF0000u)),
              make_float2(-1.f, -1.f), make_float2(__uint_as_float(a), __uint_as_float(b)));
          lo[c] = pack_pair<__nv_bfloat16>(r.x, r.y);
        } else {
          hi[c] = pack_pair<__half>(__uint_as_float(a), __uint_as_float(b));
          lo[c] = 0u;
        }
      }
      uint32_t pk[KT];
#pragma unroll
      for (int c = 0; c < KT / 2; ++c) {
        const bool mine = c / (KW / 2) == cp;
        pk[c] = mine ? hi[c % (KW / 2)] : 0u;
        pk[KT / 2 + c] = mine ? lo[c % (KW / 2)] : 0u;
      }
      // P.V of tile j-1 has read P and added into O before either changes.
      if (j > 0) {
        ok = mbar_wait(p_free, (uint32_t)((j - 1) & 1));
        if (__any_sync(kFullMask, !ok)) {
          ok = false;
          break;
        }
        tc_fence_after();
      }
      if constexpr (Cfg::kTwoPartP) {
        tmem_st64(lane_base + Cfg::kPCol, pk);
      } else {
        tmem_st32(lane_base + Cfg::kPCol, *reinterpret_cast<const uint32_t(*)[32]>(pk));
      }
      if (rescale) {
#pragma unroll 1
        for (int c4 = 0; c4 < D / 32; ++c4) {
          uint32_t o[32];
          tmem_ld32(lane_base + Cfg::kOCol + c4 * 32, o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
          tmem_st32(lane_base + Cfg::kOCol + c4 * 32, o);
        }
      }
      tc_fence_before();
      mbar_arrive(p_full);
    }
    if (ok) ok = !__any_sync(kFullMask, !mbar_wait(o_last, 0));
    failed = !ok;
    if (ok) {
      tc_fence_after();
      // The row's sum and O: the copies' parts added together.  O is summed
      // by halving exchanges, after which copy cp holds dims cp * DW .. +
      // DW - 1 of each 32-dim chunk, the ones it writes.
#pragma unroll
      for (int sh = 1; sh < DUP; sh <<= 1) l += __shfl_xor_sync(kFullMask, l, sh);
#pragma unroll 1
      for (int c4 = 0; c4 < D / 32; ++c4) {
        uint32_t o[32];
        tmem_ld32(lane_base + Cfg::kOCol + c4 * 32, o);
        int n = 32;
#pragma unroll
        for (int sh = DUP / 2; sh >= 1; sh >>= 1) {
          const bool upper = (cp & sh) != 0;
          n >>= 1;
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            if (i < n) {
              const uint32_t keep = upper ? o[n + i] : o[i];
              const uint32_t give = upper ? o[i] : o[n + i];
              o[i] = __float_as_uint(__uint_as_float(keep) +
                                     __uint_as_float(__shfl_xor_sync(kFullMask, give, sh)));
            }
          }
        }
        uint32_t v[DW];
#pragma unroll
        for (int i = 0; i < DW; ++i) v[i] = o[i];
        if (has_row && my_status == 1) store_row(false, m, l, v, c4 * 32 + cp * DW);
      }
      mark_broken_rows(false);
    } else {
      mark_broken_rows(true);
    }
  }

  // ---- release the tensor memory ------------------------------------------
  if (failed && lane == 0) set_error(p.err, PKV_DEV_TIMEOUT);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == Cfg::kProducerWarp) tmem_dealloc(tmem, Cfg::kTmemCols);
}

// Tail and merge for a one-slice tail grid (tail_parts = 1): every
// sequence's positions past its group's shared partitions lie in one
// partition (for a sequence outside every group: the whole sequence in
// one partition).  One CTA per (KV head, sequence), four warps, warp w
// taking query heads kvh * G + h for h = w, w + 4: it computes the tail's
// partial on CUDA cores (a warp-wide dot product per position, eight
// positions' rows loaded at a time), merges it with the shared-prefix
// kernel's partials in the workspace (M = max m_p, w_p = l_p 2^(m_p - M),
// out = sum w_p o_p / sum w_p, partitions in order, then the tail), and
// writes the output.  This replaces the partition pass and the merge
// launch.  A sequence whose tail needs more than one partition, or whose
// length or tail table entries are invalid, gets zero rows and its error
// bit (PKV_DEV_SHARING, PKV_DEV_SEQ_LEN, PKV_DEV_TABLE_RANGE).
template <typename T, int D, int BS, int G>
__global__ void __launch_bounds__(128, (G > 4 ? 4 : 8)) decode_tail_merge_kernel(const DecodeParams p) {
  constexpr int DPL = D / 32;  // dims per lane
  constexpr int NB = 8;        // positions per batch of row loads
  constexpr int NPRE = 2;      // shared partials loaded ahead (the rest in the merge loop)
  constexpr int HPW = (G + 3) / 4;  // query heads per warp
  static_assert(sizeof(T) == 2 && DPL % 2 == 0, "16-bit pools");
  __shared__ int ent[kMaxPartSize / BS + 1];
  const int kvh = blockIdx.x;
  const int s = blockIdx.y;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int H = p.num_heads;
  const int PS = p.part_size;
  T* out = static_cast<T*>(p.out);
  const int64_t out0 = ((int64_t)s * H + (int64_t)kvh * G) * D;
  // Issued together: the length, the group search, this warp's query rows.
  const int L = ld_nc(p.seq_lens + s);
  float q[HPW][DPL];
#pragma unroll
  for (int hh = 0; hh < HPW; ++hh) {
    const int g = warp + 4 * hh;
    if (g < G)
      RowLoad<T, DPL>::load(static_cast<const T*>(p.q) + ((int64_t)s * H + kvh * G + g) * D +
                                lane * DPL, q[hh]);
  }
  // Partitions the shared-prefix kernel computed (shared_parts_of, with the
  // group lookup spread over each warp's lanes).
  const int g_own = shared_owner_warp(p, s);
  const int pre = g_own >= 0 ? ld_nc(p.group_prefix + g_own) : 0;
  const int first = pre > 0 ? min(pre / PS, p.num_parts) : 0;
  auto zero_rows = [&]() {
    for (int e = threadIdx.x; e < G * D; e += 128) out[out0 + e] = Elem<T>::from_f(0.f);
  };
  if (L < 1 || L > p.max_len) {
    zero_rows();
    if (threadIdx.x == 0) set_error(p.err, PKV_DEV_SEQ_LEN);
    return;
  }
  const int nparts = (L + PS - 1) / PS;
  const int tok0 = first * PS;
  if (nparts == 1 && first >= 1) return;  // the shared-prefix kernel wrote the output
  if (tok0 < L && first + 1 < nparts) {   // the tail needs more than one partition
    zero_rows();
    if (threadIdx.x == 0) set_error(p.err, PKV_DEV_SHARING);
    return;
  }
  const int nprev = min(first, nparts);  // partials in the workspace
  // Issued together: the tail's table entries (positions tok0 .. L - 1) and
  // the first shared partials of this warp's heads.
  const int tail = max(L - tok0, 0);
  const int blk0 = tok0 / BS;
  const int nblk = (tail + BS - 1) / BS;
  int bad = 0;
  for (int i = threadIdx.x; i < nblk; i += 128) {
    const int e = ld_nc(p.tables + (int64_t)s * p.max_blocks + blk0 + i);
    bad |= (e < 0 || (int64_t)e >= p.num_blocks);
    ent[i] = e;
  }
  float2 pml[HPW][NPRE];
  float po[HPW][NPRE][DPL];
#pragma unroll
  for (int hh = 0; hh < HPW; ++hh) {
    const int64_t row0 = ((int64_t)s * H + kvh * G + warp + 4 * hh) * p.num_parts;
#pragma unroll
    for (int k = 0; k < NPRE; ++k) {
      if (warp + 4 * hh < G && k < nprev) {
        pml[hh][k] = p.ws_ml[row0 + k];
        RowLoad<float, DPL>::load(p.ws_o + (row0 + k) * D + lane * DPL, po[hh][k]);
      }
    }
  }
  if (__syncthreads_or(bad)) {
    zero_rows();
    if (threadIdx.x == 0) set_error(p.err, PKV_DEV_TABLE_RANGE);
    return;
  }
  const T* kc = static_cast<const T*>(p.k_cache);
  const T* vc = static_cast<const T*>(p.v_cache);
#pragma unroll
  for (int hh = 0; hh < HPW; ++hh) {
    const int g = warp + 4 * hh;
    if (g >= G) break;
    const int head = kvh * G + g;
    // ---- the tail's partial (m, l, o) in base-2 units ----------------------
    float m = -INFINITY, l = 0.f, o[DPL];
#pragma unroll
    for (int i = 0; i < DPL; ++i) o[i] = 0.f;
    for (int t0 = 0; t0 < tail; t0 += NB) {
      // This lane's DPL elements of NB key and value rows, kept packed
      // (two 16-bit elements per word) until used.
      constexpr int W = DPL / 2;
      uint32_t kr[NB][W], vr[NB][W];
#pragma unroll
      for (int u = 0; u < NB; ++u) {
        const int t = min(t0 + u, tail - 1);  // past the tail: a repeat, weighted 0 below
        const int64_t row = ((int64_t)ent[t / BS] * p.kv_heads + kvh) * BS + (tok0 + t) % BS;
        const uint32_t* kp = reinterpret_cast<const uint32_t*>(kc + row * D + lane * DPL);
        const uint32_t* vp = reinterpret_cast<const uint32_t*>(vc + row * D + lane * DPL);
        if constexpr (W == 2) {
          const uint2 a = *reinterpret_cast<const uint2*>(kp), b = *reinterpret_cast<const uint2*>(vp);
          kr[u][0] = a.x; kr[u][1] = a.y; vr[u][0] = b.x; vr[u][1] = b.y;
        } else {
#pragma unroll
          for (int w = 0; w < W; ++w) {
            kr[u][w] = kp[w];
            vr[u][w] = vp[w];
          }
        }
      }
      float x[NB];
#pragma unroll
      for (int u = 0; u < NB; ++u) {
        float d = 0.f;
#pragma unroll
        for (int w = 0; w < W; ++w) {
          const float2 kf = Elem<T>::pair(kr[u][w]);
          d = fmaf(q[hh][2 * w], kf.x, d);
          d = fmaf(q[hh][2 * w + 1], kf.y, d);
        }
        x[u] = d;
      }
#pragma unroll
      for (int sh = 16; sh >= 1; sh >>= 1)
#pragma unroll
        for (int u = 0; u < NB; ++u) x[u] += __shfl_xor_sync(kFullMask, x[u], sh);
      float mb = -INFINITY;
#pragma unroll
      for (int u = 0; u < NB; ++u) {
        x[u] = t0 + u < tail ? x[u] * p.qscale : -INFINITY;
        mb = fmaxf(mb, x[u]);
      }
      const float mnew = fmaxf(m, mb);
      const float alpha = exp2f(m - mnew);  // 0 on the first batch (m = -inf)
      l *= alpha;
#pragma unroll
      for (int i = 0; i < DPL; ++i) o[i] *= alpha;
#pragma unroll
      for (int u = 0; u < NB; ++u) {
        const float pw = exp2f(x[u] - mnew);
        l += pw;
#pragma unroll
        for (int w = 0; w < W; ++w) {
          const float2 vf = Elem<T>::pair(vr[u][w]);
          o[2 * w] = fmaf(pw, vf.x, o[2 * w]);
          o[2 * w + 1] = fmaf(pw, vf.y, o[2 * w + 1]);
        }
      }
      m = mnew;
    }
    // ---- merge with the shared partials, in order, then the tail -----------
    // A partial's o is normalised (its weights sum to 1); the tail's is not.
    const int64_t row0 = ((int64_t)s * H + head) * p.num_parts;
    float big = m;
    bool broken = false;
#pragma unroll
    for (int k = 0; k < NPRE; ++k) {
      if (k < nprev) {
        broken |= pml[hh][k].y < 0.f;
        big = fmaxf(big, pml[hh][k].x);
      }
    }
    for (int k = NPRE; k < nprev; ++k) {
      const float2 v = p.ws_ml[row0 + k];
      broken |= v.y < 0.f;
      big = fmaxf(big, v.x);
    }
    float acc[DPL];
    float den = 0.f;
#pragma unroll
    for (int i = 0; i < DPL; ++i) acc[i] = 0.f;
#pragma unroll
    for (int k = 0; k < NPRE; ++k) {
      if (k < nprev) {
        const float wgt = pml[hh][k].y * exp2f(pml[hh][k].x - big);
        den += wgt;
#pragma unroll
        for (int i = 0; i < DPL; ++i) acc[i] = fmaf(po[hh][k][i], wgt, acc[i]);
      }
    }
    for (int k = NPRE; k < nprev; ++k) {
      const float2 v = p.ws_ml[row0 + k];
      const float wgt = v.y * exp2f(v.x - big);
      den += wgt;
      float ov[DPL];
      RowLoad<float, DPL>::load(p.ws_o + (row0 + k) * D + lane * DPL, ov);
#pragma unroll
      for (int i = 0; i < DPL; ++i) acc[i] = fmaf(ov[i], wgt, acc[i]);
    }
    if (tail > 0) {
      const float wt = exp2f(m - big);
      den += l * wt;
#pragma unroll
      for (int i = 0; i < DPL; ++i) acc[i] = fmaf(o[i], wt, acc[i]);
    }
#pragma unroll
    for (int i = 0; i < DPL; ++i)
      out[out0 + (int64_t)g * D + lane * DPL + i] = Elem<T>::from_f(broken ? 0.f : acc[i] / den);
  }
}

}  // namespace pkv
