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
// plain partition pass would have written, the plain partition pass skips
// those partitions, and the split-K merge combines them with the member's
// own tail unchanged.
//
// Kernel (this library's design): grid (KV head, group, shared partition x
// row block); one producer warp streams the partition's 16-position K/V
// chunks through a four-stage ring of TMA tile loads (128-byte swizzle),
// read through the first member's table; four compute warps each own 8 of
// the group's stacked rows (member r / G, query head r % G) and run every
// chunk with the grouped-head kernel's per-chunk steps (S^T = K.Q^T and
// O^T += V^T.P^T as mma.sync m16n8k16 tiles, online softmax per column,
// bf16 P in two parts).  Each warp writes its rows' partials directly; no
// cross-warp merge is needed.
//
// Ownership.  Sequence s belongs to group owner(s): the last g with
// group_starts[g] <= s, provided s < group_starts[g+1]; both this kernel and
// the partition pass use that rule, so a malformed list can only leave
// sequences without a group (decoded plainly), never covered twice or not
// at all.  Checked per row: the length lies in [1, max_len] (else the row is
// left to the plain path's invalid-length handling), covers the partition,
// and the table names the leader's blocks for it; otherwise the row's
// partial is marked invalid (the merge writes zeros) and PKV_DEV_SHARING is
// set.
#pragma once

#include "decode_mma.cuh"

namespace pkv {

template <typename T, int D, int BS, int G>
struct SharedCfg {
  static constexpr int kComputeWarps = 4;
  static constexpr int kRowsPerWarp = 8;                 // n of m16n8k16: query rows
  static constexpr int kRows = kComputeWarps * kRowsPerWarp;
  static constexpr int kThreads = (kComputeWarps + 1) * 32;  // + producer warp
  static constexpr int kChunk = 16;
  static constexpr int kBoxRows = BS < 16 ? BS : 16;
  static constexpr int kBoxesPerChunk = kChunk / kBoxRows;
  static constexpr int kCols = D / 64;                   // 128-byte column boxes per row
  static constexpr int kBoxBytes = kChunk * 128;
  static constexpr int kTileBytes = kCols * kBoxBytes;   // one chunk of K (or V)
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kStages = 4;
  static constexpr int kBarOff = kStages * kStageBytes;
  static constexpr int kPtOff = kBarOff + 2 * kStages * 8;
  static constexpr int kPtBytes = 2 * 8 * kChunk * 2;    // P^T high and low parts
  static constexpr int kTableOff = kPtOff + kComputeWarps * kPtBytes;
  static constexpr int kAlign = 1024;
  static constexpr int kSmemBytes = kAlign + kTableOff + (kMaxPartSize / BS) * 4;
  static_assert((BS % kChunk == 0 || kChunk % BS == 0) && D % 64 == 0 && G <= 8, "geometry");
};

template <typename T, int D, int BS, int G>
__global__ void __launch_bounds__(SharedCfg<T, D, BS, G>::kThreads)
decode_shared_prefix_kernel(const DecodeParams p, int row_blocks,
                            const __grid_constant__ CUtensorMap tmk,
                            const __grid_constant__ CUtensorMap tmv) {
  using Cfg = SharedCfg<T, D, BS, G>;
  using Op = MmaOp<T>;
  constexpr int C = Cfg::kChunk;
  constexpr int NW = Cfg::kComputeWarps;
  constexpr int NST = Cfg::kStages;
  constexpr int KSTEPS = D / 16;
  constexpr bool kSplitP = std::is_same<T, __nv_bfloat16>::value;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((Cfg::kAlign - (smem_addr(smem_raw) & (Cfg::kAlign - 1))) &
                                    (Cfg::kAlign - 1));

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
  if (rb * Cfg::kRows >= gsize * G) return;
  const int tok0 = part * PS;
  const int blk0 = tok0 / BS;
  const int span = PS / BS;  // blocks of the partition (<= max_blocks - blk0: checked below)
  const int nchunks = (PS + C - 1) / C;

  // ---- the leader's table entries for this partition ------------------------
  int* stable = reinterpret_cast<int*>(smem + Cfg::kTableOff);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + Cfg::kBarOff);
  uint64_t* empty = full + NST;
  if (threadIdx.x == 0) {
    for (int st = 0; st < NST; ++st) {
      mbar_init(smem_addr(&full[st]), 1);
      mbar_init(smem_addr(&empty[st]), NW);
    }
    fence_mbar_init();
  }
  const bool fits = blk0 + span <= p.max_blocks;
  const int32_t* lrow = p.tables + (int64_t)s0 * p.max_blocks + blk0;
  int bad = !fits;
  for (int i = threadIdx.x; fits && i < span; i += Cfg::kThreads) {
    const int e = ld_nc(lrow + i);
    bad |= (e < 0 || (int64_t)e >= p.num_blocks);
    stable[i] = e;
  }
  // The leader's entries are unusable: every member's row of this partition
  // is marked invalid below.
  bad = __syncthreads_or(bad);

  // ---- this thread's row (compute warps): lanes' B-fragment column gi -----
  const int gi = lane >> 2, ti = lane & 3;
  auto row_seq = [&](int col) {  // sequence of column col of this warp, or -1
    const int r = rb * Cfg::kRows + warp * 8 + col;
    const int m = r / G;
    if (warp >= NW || m >= gsize) return -1;
    const int s = s0 + m;
    return shared_owner(p, s) == g ? s : -1;
  };
  // Row status per column: 1 usable, 0 skip (invalid length: the plain
  // path zeroes it), -1 sharing contract broken (marked invalid).
  auto row_status = [&](int s) -> int {
    if (s < 0) return 0;
    const int L = ld_nc(p.seq_lens + s);
    if (L < 1 || L > p.max_len) return 0;
    if (bad || L < tok0 + PS) return -1;
    const int32_t* row = p.tables + (int64_t)s * p.max_blocks + blk0;
    for (int i = 0; i < span; ++i)
      if (ld_nc(row + i) != stable[i]) return -1;
    return 1;
  };

  if (warp == NW) {
    // ---- producer: chunk c = positions 16c .. 16c+15 of the partition ------
    const uint64_t policy = policy_evict_first();
    const int oob_block = p.num_blocks > 0x7FFFFFFF ? 0x7FFFFFFF : (int)p.num_blocks;
    bool ok = !bad;
    int issued = 0;
    for (int j = 0; j < nchunks && ok; ++j) {
      const int st = j % NST;
      if (j >= NST)
        ok = !__any_sync(kFullMask,
                         !mbar_wait(smem_addr(&empty[st]), (uint32_t)(((j / NST) - 1) & 1)));
      if (!ok) break;
      if (lane == 0) {
        const uint32_t bar = smem_addr(&full[st]);
        const uint32_t dst = smem_addr(smem) + st * Cfg::kStageBytes;
        constexpr int RB = Cfg::kBoxRows;
        mbar_arrive_expect_tx(bar, Cfg::kStageBytes);
        for (int hb = 0; hb < Cfg::kBoxesPerChunk; ++hb) {
          // A box past the partition's end (b = 8, odd number of blocks)
          // reads an out-of-range block: the copy fills it with zeros.
          const int pos = j * C + hb * RB;
          const int pb = pos < PS ? stable[pos / BS] : oob_block;
          const int row = pos < PS ? pos % BS : 0;
#pragma unroll
          for (int cb = 0; cb < Cfg::kCols; ++cb) {
            const uint32_t o = cb * Cfg::kBoxBytes + hb * RB * 128;
            tma_load_4d(dst + o, &tmk, cb * 64, row, kvh, pb, bar, policy);
            tma_load_4d(dst + Cfg::kTileBytes + o, &tmv, cb * 64, row, kvh, pb, bar, policy);
          }
        }
      }
      __syncwarp();
      issued = j + 1;
    }
    // Copies issued but possibly never consumed (a compute warp stopped).
    for (int j = issued - NST < 0 ? 0 : issued - NST; j < issued; ++j)
      mbar_wait(smem_addr(&full[j % NST]), (uint32_t)((j / NST) & 1), kWaitLimitNs / 8);
    if (!ok && !bad && lane == 0) set_error(p.err, PKV_DEV_TIMEOUT);
    return;
  }

  // ---- compute warps ---------------------------------------------------------
  // Column gi (B fragments): the query row this lane loads; columns 2ti and
  // 2ti+1 (accumulators): the rows this lane's results belong to.
  const int sq = row_seq(gi);
  const int hq = kvh * G + (rb * Cfg::kRows + warp * 8 + gi) % G;
  uint32_t qb[KSTEPS][2];
  {
    const uint32_t* qrow = reinterpret_cast<const uint32_t*>(
        static_cast<const T*>(p.q) + ((int64_t)(sq < 0 ? 0 : sq) * H + hq) * D);
#pragma unroll
    for (int kk = 0; kk < KSTEPS; ++kk) {
      qb[kk][0] = sq >= 0 ? qrow[(16 * kk + 2 * ti) / 2] : 0u;
      qb[kk][1] = sq >= 0 ? qrow[(16 * kk + 2 * ti + 8) / 2] : 0u;
    }
  }
  float acc[KSTEPS][4];
#pragma unroll
  for (int i = 0; i < KSTEPS; ++i)
#pragma unroll
    for (int c = 0; c < 4; ++c) acc[i][c] = 0.f;
  float m[2] = {-INFINITY, -INFINITY};
  float l[2] = {0.f, 0.f};
  bool timed_out = false;

  const int mm = lane >> 3, mr = lane & 7;
  const int k_tok = (mm & 1) * 8 + mr, k_col8 = mm >> 1;
  const int v_tok = (mm >> 1) * 8 + mr, v_col8 = mm & 1;
  uint16_t* pt = reinterpret_cast<uint16_t*>(smem + Cfg::kPtOff + warp * Cfg::kPtBytes);
  const uint32_t ring0 = smem_addr(smem);

  for (int j = 0; j < nchunks && !bad; ++j) {
    const int st = j % NST;
    timed_out = __any_sync(kFullMask, !mbar_wait(smem_addr(&full[st]), (uint32_t)((j / NST) & 1)));
    if (timed_out) break;
    const int nvalid = min(C, PS - j * C);
    const uint32_t ktile = ring0 + st * Cfg::kStageBytes;
    const uint32_t vtile = ktile + Cfg::kTileBytes;

    float sc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int kk = 0; kk < KSTEPS; ++kk) {
      const int col8 = 2 * (kk % 4) + k_col8;
      const uint32_t addr =
          ktile + (kk / 4) * Cfg::kBoxBytes + k_tok * 128 + ((col8 ^ (k_tok & 7)) << 4);
      uint32_t a[4];
      ldsm_x4(a, addr);
      Op::run(sc, a, qb[kk][0], qb[kk][1]);
    }
    const bool v0 = gi < nvalid, v1 = gi + 8 < nvalid;
    float x[4];
    x[0] = v0 ? sc[0] * p.qscale : -INFINITY;
    x[1] = v0 ? sc[1] * p.qscale : -INFINITY;
    x[2] = v1 ? sc[2] * p.qscale : -INFINITY;
    x[3] = v1 ? sc[3] * p.qscale : -INFINITY;
    float alpha[2], pr[4];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float cm = fmaxf(x[h], x[h + 2]);
      cm = fmaxf(cm, __shfl_xor_sync(kFullMask, cm, 4));
      cm = fmaxf(cm, __shfl_xor_sync(kFullMask, cm, 8));
      cm = fmaxf(cm, __shfl_xor_sync(kFullMask, cm, 16));
      const float mnew = fmaxf(m[h], cm);
      alpha[h] = exp2f(m[h] - mnew);
      pr[h] = exp2f(x[h] - mnew);
      pr[h + 2] = exp2f(x[h + 2] - mnew);
      float cs = pr[h] + pr[h + 2];
      cs += __shfl_xor_sync(kFullMask, cs, 4);
      cs += __shfl_xor_sync(kFullMask, cs, 8);
      cs += __shfl_xor_sync(kFullMask, cs, 16);
      l[h] = l[h] * alpha[h] + cs;
      m[h] = mnew;
    }
    if (__any_sync(kFullMask, alpha[0] != 1.f || alpha[1] != 1.f)) {
#pragma unroll
      for (int i = 0; i < KSTEPS; ++i) {
        acc[i][0] *= alpha[0];
        acc[i][1] *= alpha[1];
        acc[i][2] *= alpha[0];
        acc[i][3] *= alpha[1];
      }
    }
    {
      const int h0 = 2 * ti, h1 = 2 * ti + 1;
      const uint16_t q0 = Op::bits(pr[0]), q1 = Op::bits(pr[1]);
      const uint16_t q2 = Op::bits(pr[2]), q3 = Op::bits(pr[3]);
      pt[h0 * C + gi] = q0;
      pt[h1 * C + gi] = q1;
      pt[h0 * C + gi + 8] = q2;
      pt[h1 * C + gi + 8] = q3;
      if constexpr (kSplitP) {
        uint16_t* lo = pt + 8 * C;
        lo[h0 * C + gi] = Op::bits(pr[0] - Op::back(q0));
        lo[h1 * C + gi] = Op::bits(pr[1] - Op::back(q1));
        lo[h0 * C + gi + 8] = Op::bits(pr[2] - Op::back(q2));
        lo[h1 * C + gi + 8] = Op::bits(pr[3] - Op::back(q3));
      }
    }
    __syncwarp();
    const uint32_t* ptw = reinterpret_cast<const uint32_t*>(pt);
    const uint32_t bh0 = ptw[(gi * C + 2 * ti) / 2];
    const uint32_t bh1 = ptw[(gi * C + 2 * ti + 8) / 2];
    uint32_t bl0 = 0, bl1 = 0;
    if constexpr (kSplitP) {
      bl0 = ptw[(8 * C + gi * C + 2 * ti) / 2];
      bl1 = ptw[(8 * C + gi * C + 2 * ti + 8) / 2];
    }
#pragma unroll
    for (int i = 0; i < KSTEPS; ++i) {
      const int col8 = 2 * (i % 4) + v_col8;
      const uint32_t addr =
          vtile + (i / 4) * Cfg::kBoxBytes + v_tok * 128 + ((col8 ^ (v_tok & 7)) << 4);
      uint32_t a[4];
      ldsm_x4_trans(a, addr);
      Op::run(acc[i], a, bh0, bh1);
      if constexpr (kSplitP) Op::run(acc[i], a, bl0, bl1);
    }
    __syncwarp();  // this warp is done with the stage and with P^T
    if (lane == 0) mbar_arrive(smem_addr(&empty[st]));
  }
  if (timed_out && lane == 0) set_error(p.err, PKV_DEV_TIMEOUT);

  // ---- this warp's rows: (m, l) and o = acc / l, or the invalid marker ------
  // Lane (gi, ti) holds dims 16i + gi (+ 8) of columns 2ti and 2ti + 1.
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int col = 2 * ti + h;
    const int s = row_seq(col);
    const int st = row_status(s);
    if (st == 0) continue;
    const bool broken = st < 0 || bad || timed_out;
    if (st < 0 && gi == 0) set_error(p.err, PKV_DEV_SHARING);
    const int head = kvh * G + (rb * Cfg::kRows + warp * 8 + col) % G;
    const int L = ld_nc(p.seq_lens + s);
    const int nparts = (L + PS - 1) / PS;
    const float inv = 1.f / l[h];
    if (nparts == 1) {  // the whole sequence is this partition: final output
      T* orow = out + ((int64_t)s * H + head) * D;
#pragma unroll
      for (int i = 0; i < KSTEPS; ++i)
#pragma unroll
        for (int half = 0; half < 2; ++half)
          orow[16 * i + gi + 8 * half] = Elem<T>::from_f(broken ? 0.f : acc[i][2 * half + h] * inv);
    } else {
      const int64_t w = ((int64_t)s * H + head) * p.num_parts + part;
#pragma unroll
      for (int i = 0; i < KSTEPS; ++i)
#pragma unroll
        for (int half = 0; half < 2; ++half)
          p.ws_o[w * D + 16 * i + gi + 8 * half] = broken ? 0.f : acc[i][2 * half + h] * inv;
      if (gi == 0) p.ws_ml[w] = broken ? make_float2(-INFINITY, -1.f) : make_float2(m[h], l[h]);
    }
  }
}

}  // namespace pkv
