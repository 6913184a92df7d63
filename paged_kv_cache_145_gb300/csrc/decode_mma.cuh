// Grouped-query decode attention on tensor cores (fp16 / bf16 caches).
//
// Same method, partitioning, workspace and merge as decode_partition_kernel
// (decode.cuh); only the arithmetic of one chunk differs.  With G = H / Hk
// query heads sharing a KV head, a chunk of 16 positions is a small dense
// contraction on both sides of the softmax:
//
//   S^T[16 positions x 8 heads]  = K[16 x D] . Q^T[D x 8]      (D/16 MMAs)
//   O^T[D x 8 heads]            += V^T[D x 16] . P^T[16 x 8]   (D/16 MMAs)
//
// each an m16n8k16 tile (`mma.sync`, fp32 accumulation).  Heads G..7 of the
// 8-wide tile are zero padding.  S^T and O^T stay in registers; per lane,
// the S^T fragment holds positions lane/4 and lane/4 + 8 of heads 2(lane%4)
// and 2(lane%4)+1, which is where the online softmax (base 2, fp32) runs:
// column maxima and sums need three xor-shuffles.  P^T goes through a
// 512-byte shared buffer to become the B operand of the second product.
// For bf16, P is split into a bf16 high part and a bf16 remainder and both
// are multiplied (two MMAs), so P keeps about 16 significant bits.
//
// K and V chunks arrive by 4-D TMA tile loads (cp.async.bulk.tensor) from
// the [N][Hk][b][D] pools, in boxes of 16 rows x 64 elements with the
// 128-byte swizzle; `ldmatrix` (plain for K, transposing for V) then reads
// them without bank conflicts.  Rows of a final partial chunk beyond the
// sequence are masked in S and zeroed in the staged V tile, so stale slots
// of the last block cannot reach the output even if they hold NaNs.
//
// The tile and fragment layouts follow the PTX ISA description of
// mma.m16n8k16 and ldmatrix; the design (orientation, P^T staging, hi/lo
// split) is this library's.
#pragma once

#include <cuda.h>

#include <type_traits>

#include "decode.cuh"

namespace pkv {

template <typename T>
struct MmaOp;

template <>
struct MmaOp<__half> {
  static __device__ __forceinline__ void run(float (&d)[4], const uint32_t (&a)[4],
                                             uint32_t b0, uint32_t b1) {
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
  static __device__ __forceinline__ uint16_t bits(float x) {
    return __half_as_ushort(__float2half_rn(x));
  }
  static __device__ __forceinline__ float back(uint16_t h) { return __half2float(__ushort_as_half(h)); }
};

template <>
struct MmaOp<__nv_bfloat16> {
  static __device__ __forceinline__ void run(float (&d)[4], const uint32_t (&a)[4],
                                             uint32_t b0, uint32_t b1) {
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
  static __device__ __forceinline__ uint16_t bits(float x) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(x));
  }
  static __device__ __forceinline__ float back(uint16_t h) {
    return __uint_as_float((uint32_t)h << 16);
  }
};

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}

// 4-D tile load of one box (x = element column, y = row within the block,
// z = KV head, w = physical block) into shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            int z, int w, uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(bar),
      "l"(policy)
      : "memory");
}

template <typename T, int D, int BS, int G>
struct MmaCfg {
  static constexpr int kWarps = 4;
  static constexpr int kThreads = kWarps * 32;
  static constexpr int kChunk = 16;                     // positions per MMA tile
  static constexpr int kBoxRows = BS < 16 ? BS : 16;    // rows per TMA box
  static constexpr int kBoxesPerChunk = kChunk / kBoxRows;  // blocks a chunk spans
  static constexpr int kChunksPerBlock = BS < 16 ? 1 : BS / kChunk;
  static constexpr int kCols = D / 64;                  // 128-byte column boxes per row
  static constexpr int kBoxBytes = kChunk * 128;        // 16 rows x 128 B
  static constexpr int kTileBytes = kCols * kBoxBytes;  // one chunk of K (or V)
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kStages = 2;
  static constexpr int kRingBytes = kWarps * kStages * kStageBytes;
  static constexpr int kBarOff = kRingBytes;
  static constexpr int kPtOff = kBarOff + kWarps * kStages * 8;
  static constexpr int kPtBytes = 2 * 8 * kChunk * 2;   // P^T high and low parts
  static constexpr int kTableOff = kPtOff + kWarps * kPtBytes;
  static constexpr int kAlign = 1024;                   // 128-byte swizzle atom
  static constexpr int kMergeBytes = (kWarps * G * D + 3 * kWarps * G + 2 * G) * 4;
  static_assert(kMergeBytes <= kRingBytes, "merge scratch must fit in the ring");
  static_assert((BS % kChunk == 0 || kChunk % BS == 0) && D % 64 == 0 && G <= 8,
                "tensor-core geometry");
  static constexpr int smem_bytes(int part_size) {
    return kAlign + kTableOff + (part_size / BS) * 4;
  }
  static constexpr int kMaxSmem = kAlign + kTableOff + (kMaxPartSize / BS) * 4;
};

template <typename T, int D, int BS, int G>
__global__ void __launch_bounds__(MmaCfg<T, D, BS, G>::kThreads)
decode_partition_mma_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap tmk,
                            const __grid_constant__ CUtensorMap tmv) {
  using Cfg = MmaCfg<T, D, BS, G>;
  using Op = MmaOp<T>;
  constexpr int C = Cfg::kChunk;
  constexpr int NW = Cfg::kWarps;
  constexpr int NST = Cfg::kStages;
  constexpr int KSTEPS = D / 16;
  constexpr bool kSplitP = std::is_same<T, __nv_bfloat16>::value;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  // Swizzled boxes need 1024-byte alignment; round the dynamic base up.
  unsigned char* smem = smem_raw + ((Cfg::kAlign - (smem_addr(smem_raw) & (Cfg::kAlign - 1))) &
                                    (Cfg::kAlign - 1));

  const int kvh = blockIdx.x;
  const int s = blockIdx.y;
  const int z = blockIdx.z;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int gi = lane >> 2;  // fragment row group (position, or head for B)
  const int ti = lane & 3;   // fragment column pair
  const int H = p.num_heads;
  T* out = static_cast<T*>(p.out);
  const int64_t out0 = ((int64_t)s * H + (int64_t)kvh * G) * D;
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
  const uint32_t ring0 = smem_addr(smem) + warp * NST * Cfg::kStageBytes;
  const uint32_t bar0 = smem_addr(&bars[warp * NST]);
  const uint64_t policy = policy_evict_first();

  // Chunk c covers partition positions 16c .. 16c+15.  With b >= 16 that is
  // 16 rows of one block; with b = 8 it is two whole blocks,
  // loaded as two 8-row boxes stacked in shared memory (the same swizzled
  // layout as one 16-row box).  A second block past the partition's end is
  // not loaded; its rows are masked (K) and zeroed (V) like any tail.
  auto issue = [&](int j) {
    const int c = warp + j * NW;
    const int st = j % NST;
    const uint32_t bar = bar0 + st * 8;
    const uint32_t dst = ring0 + st * Cfg::kStageBytes;
    constexpr int RB = Cfg::kBoxRows;
    int nbox = 1;
    if constexpr (Cfg::kBoxesPerChunk > 1) nbox = (c * C + RB < ntok) ? 2 : 1;
    mbar_arrive_expect_tx(bar, nbox * (Cfg::kStageBytes / Cfg::kBoxesPerChunk));
    for (int hb = 0; hb < nbox; ++hb) {
      const int pos = c * C + hb * RB;  // first position of this box in the partition
      const int pb = stable[pos / BS];
      const int row = pos % BS;
#pragma unroll
      for (int cb = 0; cb < Cfg::kCols; ++cb) {
        const uint32_t o = cb * Cfg::kBoxBytes + hb * RB * 128;
        tma_load_4d(dst + o, &tmk, cb * 64, row, kvh, pb, bar, policy);
        tma_load_4d(dst + Cfg::kTileBytes + o, &tmv, cb * 64, row, kvh, pb, bar, policy);
      }
    }
  };
  if (lane == 0) {
    const int pre = count < NST ? count : NST;
    for (int j = 0; j < pre; ++j) issue(j);
  }

  // Q^T as B fragments: head gi (zero beyond G), rows 2*ti.. of each k-step.
  uint32_t qb[KSTEPS][2];
  {
    const uint32_t* qrow =
        reinterpret_cast<const uint32_t*>(static_cast<const T*>(p.q) + out0 + (int64_t)gi * D);
#pragma unroll
    for (int kk = 0; kk < KSTEPS; ++kk) {
      qb[kk][0] = gi < G ? qrow[(16 * kk + 2 * ti) / 2] : 0u;
      qb[kk][1] = gi < G ? qrow[(16 * kk + 2 * ti + 8) / 2] : 0u;
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

  // Per-lane ldmatrix row addresses (before the stage base is added).
  const int mm = lane >> 3, mr = lane & 7;
  // K (plain): matrix mm covers positions (mm & 1) * 8.. and columns (mm >> 1) * 8..
  const int k_tok = (mm & 1) * 8 + mr;
  const int k_col8 = mm >> 1;
  // V (transposed): matrix mm covers positions (mm >> 1) * 8.. and columns (mm & 1) * 8..
  const int v_tok = (mm >> 1) * 8 + mr;
  const int v_col8 = mm & 1;
  uint16_t* pt = reinterpret_cast<uint16_t*>(smem + Cfg::kPtOff + warp * Cfg::kPtBytes);

  int j = 0;
  for (; j < count; ++j) {
    const int st = j % NST;
    timed_out = __any_sync(kFullMask, !mbar_wait(bar0 + st * 8, (uint32_t)((j / NST) & 1)));
    if (timed_out) break;
    const int c = warp + j * NW;
    const int nvalid = min(C, ntok - c * C);
    const uint32_t ktile = ring0 + st * Cfg::kStageBytes;
    const uint32_t vtile = ktile + Cfg::kTileBytes;

    // ---- S^T = K . Q^T ----------------------------------------------------
    float sc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int kk = 0; kk < KSTEPS; ++kk) {
      const int col8 = 2 * (kk % 4) + k_col8;  // 16-byte column within the 128-byte box
      const uint32_t addr =
          ktile + (kk / 4) * Cfg::kBoxBytes + k_tok * 128 + ((col8 ^ (k_tok & 7)) << 4);
      uint32_t a[4];
      ldsm_x4(a, addr);
      Op::run(sc, a, qb[kk][0], qb[kk][1]);
    }

    // ---- online softmax over the chunk, per head column ------------------
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

    // ---- P^T to shared memory: [head][position], high (and low) parts ----
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
    // Positions past the sequence end in a final partial chunk: zero their
    // value rows so stale slot contents cannot reach the accumulator.
    if (nvalid < C) {
      unsigned char* vt = smem + (vtile - smem_addr(smem));
      for (int e = lane; e < (C - nvalid) * Cfg::kCols * 8; e += 32) {
        const int r = nvalid + e / (Cfg::kCols * 8);
        const int rest = e % (Cfg::kCols * 8);
        *reinterpret_cast<uint4*>(vt + (rest / 8) * Cfg::kBoxBytes + r * 128 + (rest % 8) * 16) =
            make_uint4(0u, 0u, 0u, 0u);
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

    // ---- O^T += V^T . P^T ------------------------------------------------
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

    __syncwarp();
    if (lane == 0 && j + NST < count) {
      fence_proxy_async();
      issue(j + NST);
    }
  }
  if (timed_out) {
    const int last = count < j + NST ? count : j + NST;
    for (int jj = j + 1; jj < last; ++jj)
      mbar_wait(bar0 + (jj % NST) * 8, (uint32_t)((jj / NST) & 1), kWaitLimitNs / 8);
    if (lane == 0) set_error(p.err, PKV_DEV_TIMEOUT);
  }

  // ---- merge the warps (same layout and arithmetic as the CUDA-core pass) --
  __syncthreads();
  float* red_acc = reinterpret_cast<float*>(smem);  // [NW][G][D]
  float* red_m = red_acc + NW * G * D;              // [NW][G]
  float* red_l = red_m + NW * G;                    // [NW][G]
  float* fac = red_l + NW * G;                      // [NW][G]
  float* fin = fac + NW * G;                        // [G] max, [G] sum
#pragma unroll
  for (int i = 0; i < KSTEPS; ++i)
#pragma unroll
    for (int cc = 0; cc < 4; ++cc) {
      const int head = 2 * ti + (cc & 1);
      const int dim = 16 * i + gi + 8 * (cc >> 1);
      if (head < G) red_acc[(warp * G + head) * D + dim] = acc[i][cc];
    }
  if (gi == 0) {
#pragma unroll
    for (int h = 0; h < 2; ++h)
      if (2 * ti + h < G) {
        red_m[warp * G + 2 * ti + h] = m[h];
        red_l[warp * G + 2 * ti + h] = l[h];
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
      const float f = exp2f(red_m[w * G + g] - big);
      fac[w * G + g] = f;
      tot += red_l[w * G + g] * f;
    }
    fin[g] = big;
    fin[G + g] = tot;
  }
  __syncthreads();
  for (int e = threadIdx.x; e < G * D; e += Cfg::kThreads) {
    const int g = e / D;
    const int d = e - g * D;
    float o = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) o = fmaf(red_acc[(w * G + g) * D + d], fac[w * G + g], o);
    o = o / fin[G + g];
    if (nparts == 1)
      out[out0 + e] = Elem<T>::from_f(o);
    else
      p.ws_o[(ws0 + (int64_t)g * p.num_parts) * D + d] = o;
  }
  if (nparts > 1 && threadIdx.x < G)
    p.ws_ml[ws0 + (int64_t)threadIdx.x * p.num_parts] =
        make_float2(fin[threadIdx.x], fin[G + threadIdx.x]);
}

}  // namespace pkv
