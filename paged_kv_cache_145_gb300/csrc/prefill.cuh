// Paged causal prefill attention on tensor cores (fp16 / bf16 pools).
//
// "vLLM and PagedAttention: Virtual Memory for LLM Serving" (opening
// paragraph): in prefill all prompt tokens are known, so their queries are
// processed together; "Inside vLLM and TGI: Paging, Versioned Schedulers
// and Operations" (launch notes: chunked prefill) splits long prompts into
// chunks that attend to the cached prefix.  Sequence s holds L positions
// after its chunk of Q new queries was written to the pool (paged_kv_write);
// query i sits at position L - Q + i and attends to positions 0 .. L - Q + i,
// read through the block table like decode.
//
// Work decomposition (this library's design): one CTA of 4 warps per
// (query tile, KV head, sequence).  A query tile is 64 rows, each row a
// (query, grouped head) pair -- 64 / G queries x G heads -- so the G query
// heads that share a KV head share every K/V tile.  Keys stream in tiles of
// 64 positions through a two-stage ring filled by 4-D TMA tile loads (boxes
// of min(b, 16) rows x 64 elements, 128-byte swizzle).  Each warp owns 16
// rows: S[16 x 64] = Q.K^T as m16n8k16 MMAs (Q fragments held in registers,
// K^T fragments by ldmatrix), an online softmax per row in base 2 (row
// statistics need two xor-shuffles), and O[16 x D] += P.V with P reused
// straight from the S accumulators as the A operand (bf16 P split into high
// and low parts) and V fragments by transposing ldmatrix.  Keys past a row's
// position are masked; value rows past the last needed key are zeroed in
// shared memory.  Tiles run heaviest first (the last query tiles see the
// most keys).
#pragma once

#include "decode_mma.cuh"

namespace pkv {

struct PrefillParams {
  const void* q;           // [total_queries][H][D]
  void* out;               // [total_queries][H][D]
  const int32_t* starts;   // [S + 1] first query of each sequence
  int64_t total_queries;
  const int32_t* tables;   // [S][max_blocks]
  int max_blocks;
  const int32_t* seq_lens; // [S] positions after the chunk was written
  int64_t num_blocks;
  int kv_heads;
  int num_heads;
  int max_queries;         // host bound on queries per sequence
  float qscale;            // scale * log2(e)
  unsigned* err;
  const float* k_scale;    // FP8 pools: [Hk] key / value scales (else unused)
  const float* v_scale;
  // tcgen05 kernel only (1-D grid of work items): query tiles per sequence,
  // sequences, (KV head, sequence) pairs per group (items run group by
  // group, heaviest query tiles first within a group), and the number of
  // items that run whole; each later item runs as two CTAs of one Q tile.
  int q_tiles;
  int num_seqs;
  int group_pairs;
  int n_full;
};

template <typename T, int D, int BS, int G>
struct PrefillCfg {
  static constexpr int kWarps = 4;
  static constexpr int kThreads = kWarps * 32;
  static constexpr int kRows = 64;               // (query, head) rows per CTA
  static constexpr int kQueries = kRows / G;     // queries per CTA
  static constexpr int kKeys = 64;               // keys per tile
  static constexpr int kCols = D / 64;           // 128-byte column boxes
  static constexpr int kBoxRows = BS < 16 ? BS : 16;
  static constexpr int kColBytes = kKeys * 128;  // 64 rows x 128 B
  static constexpr int kTileBytes = kCols * kColBytes;
  static constexpr int kStageBytes = 2 * kTileBytes;  // K + V
  static constexpr int kStages = 2;
  static constexpr int kAlign = 1024;
  static constexpr int kBarOff = kStages * kStageBytes;
  static constexpr int kTableOff = kBarOff + 64;
  static int smem_bytes(int table_entries) { return kAlign + kTableOff + table_entries * 4; }
};

template <typename T>
__device__ __forceinline__ uint32_t pack2(float a, float b) {
  const uint32_t lo = MmaOp<T>::bits(a), hi = MmaOp<T>::bits(b);
  return lo | (hi << 16);
}

template <typename T, int D, int BS, int G>
__global__ void __launch_bounds__(PrefillCfg<T, D, BS, G>::kThreads)
prefill_mma_kernel(const PrefillParams p, const __grid_constant__ CUtensorMap tmk,
                   const __grid_constant__ CUtensorMap tmv) {
  using Cfg = PrefillCfg<T, D, BS, G>;
  using Op = MmaOp<T>;
  constexpr int KSTEPS = D / 16;  // k-steps of Q.K^T
  constexpr int NT = D / 8;       // 8-wide output tiles
  constexpr int KT = Cfg::kKeys;
  constexpr bool kSplitP = std::is_same<T, __nv_bfloat16>::value;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((Cfg::kAlign - (smem_addr(smem_raw) & (Cfg::kAlign - 1))) &
                                    (Cfg::kAlign - 1));

  const int tile = gridDim.x - 1 - blockIdx.x;  // heaviest tiles first
  const int kvh = blockIdx.y;
  const int s = blockIdx.z;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int gi = lane >> 2;
  const int ti = lane & 3;
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
  // Rows of this CTA: (query qa + r / G, head kvh * G + r % G), r < 64.
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
  const int first = L - Q;          // position of query 0
  const int n_keys = first + qend;  // keys 0 .. n_keys-1 are visible to some row
  const int nblk = (n_keys + BS - 1) / BS;
  const int n_tiles = (n_keys + KT - 1) / KT;

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Cfg::kBarOff);
  int* stable = reinterpret_cast<int*>(smem + Cfg::kTableOff);
  if (threadIdx.x == 0) {
#pragma unroll
    for (int st = 0; st < Cfg::kStages; ++st) mbar_init(smem_addr(&bars[st]), 1);
    fence_mbar_init();
  }
  int bad = 0;
  const int32_t* trow = p.tables + (int64_t)s * p.max_blocks;
  for (int i = threadIdx.x; i < nblk; i += Cfg::kThreads) {
    const int e = trow[i];
    bad |= (e < 0 || (int64_t)e >= p.num_blocks);
    stable[i] = e;
  }
  bad = __syncthreads_or(bad);
  if (bad) {
    if (threadIdx.x == 0) set_error(p.err, PKV_DEV_TABLE_RANGE);
    zero_rows();
    return;
  }

  const uint32_t ring0 = smem_addr(smem);
  const uint32_t bar0 = smem_addr(&bars[0]);
  const uint64_t policy = policy_evict_first();
  constexpr int RB = Cfg::kBoxRows;
  auto issue = [&](int kt) {
    const int st = kt % Cfg::kStages;
    const uint32_t bar = bar0 + st * 8;
    const uint32_t dst = ring0 + st * Cfg::kStageBytes;
    int boxes = 0;
    for (int j = kt * KT; j < kt * KT + KT && j < n_keys; j += RB) ++boxes;
    mbar_arrive_expect_tx(bar, boxes * RB * 128 * Cfg::kCols * 2);
    for (int j = kt * KT; j < kt * KT + KT && j < n_keys; j += RB) {
      const int pb = stable[j / BS];
      const int row = j % BS;
#pragma unroll
      for (int cb = 0; cb < Cfg::kCols; ++cb) {
        const uint32_t o = cb * Cfg::kColBytes + (j - kt * KT) * 128;
        tma_load_4d(dst + o, &tmk, cb * 64, row, kvh, pb, bar, policy);
        tma_load_4d(dst + Cfg::kTileBytes + o, &tmv, cb * 64, row, kvh, pb, bar, policy);
      }
    }
  };
  if (threadIdx.x == 0) {
    for (int kt = 0; kt < Cfg::kStages && kt < n_tiles; ++kt) issue(kt);
  }

  // This lane's two rows (r and r + 8 of the warp's 16), their queries
  // (clamped to the last one, so padding rows compute harmless values) and
  // their positions.
  const int r_lo = warp * 16 + gi;
  const int r_hi = r_lo + 8;
  const int qi_lo = min(qa + r_lo / G, Q - 1);
  const int qi_hi = min(qa + r_hi / G, Q - 1);
  const int pos_lo = first + qi_lo;
  const int pos_hi = first + qi_hi;
  const int head_lo = kvh * G + r_lo % G;
  const int head_hi = kvh * G + r_hi % G;

  uint32_t qf[KSTEPS][4];
  {
    const uint32_t* ql = reinterpret_cast<const uint32_t*>(
        static_cast<const T*>(p.q) + ((int64_t)(q0 + qi_lo) * H + head_lo) * D);
    const uint32_t* qh = reinterpret_cast<const uint32_t*>(
        static_cast<const T*>(p.q) + ((int64_t)(q0 + qi_hi) * H + head_hi) * D);
#pragma unroll
    for (int kk = 0; kk < KSTEPS; ++kk) {
      qf[kk][0] = ql[(16 * kk + 2 * ti) / 2];
      qf[kk][1] = qh[(16 * kk + 2 * ti) / 2];
      qf[kk][2] = ql[(16 * kk + 2 * ti + 8) / 2];
      qf[kk][3] = qh[(16 * kk + 2 * ti + 8) / 2];
    }
  }

  float o[NT][4];
#pragma unroll
  for (int n = 0; n < NT; ++n)
#pragma unroll
    for (int c = 0; c < 4; ++c) o[n][c] = 0.f;
  float m_lo = -INFINITY, m_hi = -INFINITY, l_lo = 0.f, l_hi = 0.f;

  const int mm = lane >> 3, mr = lane & 7;
  bool timed_out = false;
  int kt = 0;
  for (; kt < n_tiles; ++kt) {
    const int st = kt % Cfg::kStages;
    timed_out = __syncthreads_or(!mbar_wait(bar0 + st * 8, (uint32_t)((kt / Cfg::kStages) & 1)));
    if (timed_out) break;
    const uint32_t ktile = ring0 + st * Cfg::kStageBytes;
    const uint32_t vtile = ktile + Cfg::kTileBytes;
    const int key0 = kt * KT;
    if (key0 + KT > n_keys) {
      // Value rows past the last needed key: stale or never loaded; zero them.
      unsigned char* vt = smem + (vtile - ring0);
      const int from = n_keys - key0;
      for (int e = threadIdx.x; e < (KT - from) * Cfg::kCols * 8; e += Cfg::kThreads) {
        const int r = from + e / (Cfg::kCols * 8);
        const int rest = e % (Cfg::kCols * 8);
        *reinterpret_cast<uint4*>(vt + (rest / 8) * Cfg::kColBytes + r * 128 + (rest % 8) * 16) =
            make_uint4(0u, 0u, 0u, 0u);
      }
      __syncthreads();
    }

    // ---- S = Q . K^T (16 rows x 64 keys per warp) ------------------------
    float sc[8][4];
#pragma unroll
    for (int n = 0; n < 8; ++n)
#pragma unroll
      for (int c = 0; c < 4; ++c) sc[n][c] = 0.f;
#pragma unroll
    for (int kk = 0; kk < KSTEPS; ++kk) {
      const int col8 = 2 * (kk % 4) + (mm & 1);
#pragma unroll
      for (int np = 0; np < 4; ++np) {
        const int key = 16 * np + (mm >> 1) * 8 + mr;
        const uint32_t addr =
            ktile + (kk / 4) * Cfg::kColBytes + key * 128 + ((col8 ^ (key & 7)) << 4);
        uint32_t b[4];
        ldsm_x4(b, addr);
        Op::run(sc[2 * np], qf[kk], b[0], b[1]);
        Op::run(sc[2 * np + 1], qf[kk], b[2], b[3]);
      }
    }

    // ---- causal mask, online softmax per row -----------------------------
    float mx_lo = -INFINITY, mx_hi = -INFINITY;
#pragma unroll
    for (int n = 0; n < 8; ++n) {
      const int k0 = key0 + 8 * n + 2 * ti;
      sc[n][0] = k0 <= pos_lo ? sc[n][0] * p.qscale : -INFINITY;
      sc[n][1] = k0 + 1 <= pos_lo ? sc[n][1] * p.qscale : -INFINITY;
      sc[n][2] = k0 <= pos_hi ? sc[n][2] * p.qscale : -INFINITY;
      sc[n][3] = k0 + 1 <= pos_hi ? sc[n][3] * p.qscale : -INFINITY;
      mx_lo = fmaxf(mx_lo, fmaxf(sc[n][0], sc[n][1]));
      mx_hi = fmaxf(mx_hi, fmaxf(sc[n][2], sc[n][3]));
    }
    mx_lo = fmaxf(mx_lo, __shfl_xor_sync(kFullMask, mx_lo, 1));
    mx_lo = fmaxf(mx_lo, __shfl_xor_sync(kFullMask, mx_lo, 2));
    mx_hi = fmaxf(mx_hi, __shfl_xor_sync(kFullMask, mx_hi, 1));
    mx_hi = fmaxf(mx_hi, __shfl_xor_sync(kFullMask, mx_hi, 2));
    // Every row sees key 0 in the first tile, so the running maximum is
    // finite from then on; a later tile fully masked for a row keeps it.
    const float mn_lo = fmaxf(m_lo, mx_lo), mn_hi = fmaxf(m_hi, mx_hi);
    const float al_lo = exp2f(m_lo - mn_lo), al_hi = exp2f(m_hi - mn_hi);
    float sum_lo = 0.f, sum_hi = 0.f;
#pragma unroll
    for (int n = 0; n < 8; ++n) {
      sc[n][0] = exp2f(sc[n][0] - mn_lo);
      sc[n][1] = exp2f(sc[n][1] - mn_lo);
      sc[n][2] = exp2f(sc[n][2] - mn_hi);
      sc[n][3] = exp2f(sc[n][3] - mn_hi);
      sum_lo += sc[n][0] + sc[n][1];
      sum_hi += sc[n][2] + sc[n][3];
    }
    sum_lo += __shfl_xor_sync(kFullMask, sum_lo, 1);
    sum_lo += __shfl_xor_sync(kFullMask, sum_lo, 2);
    sum_hi += __shfl_xor_sync(kFullMask, sum_hi, 1);
    sum_hi += __shfl_xor_sync(kFullMask, sum_hi, 2);
    l_lo = l_lo * al_lo + sum_lo;
    l_hi = l_hi * al_hi + sum_hi;
    m_lo = mn_lo;
    m_hi = mn_hi;
#pragma unroll
    for (int n = 0; n < NT; ++n) {
      o[n][0] *= al_lo;
      o[n][1] *= al_lo;
      o[n][2] *= al_hi;
      o[n][3] *= al_hi;
    }

    // ---- O += P . V ------------------------------------------------------
#pragma unroll
    for (int k2 = 0; k2 < 4; ++k2) {  // 16 keys per k-step
      uint32_t ph[4], pl[4];
      ph[0] = pack2<T>(sc[2 * k2][0], sc[2 * k2][1]);
      ph[1] = pack2<T>(sc[2 * k2][2], sc[2 * k2][3]);
      ph[2] = pack2<T>(sc[2 * k2 + 1][0], sc[2 * k2 + 1][1]);
      ph[3] = pack2<T>(sc[2 * k2 + 1][2], sc[2 * k2 + 1][3]);
      if constexpr (kSplitP) {
        auto rem = [](float x) { return x - MmaOp<T>::back(MmaOp<T>::bits(x)); };
        pl[0] = pack2<T>(rem(sc[2 * k2][0]), rem(sc[2 * k2][1]));
        pl[1] = pack2<T>(rem(sc[2 * k2][2]), rem(sc[2 * k2][3]));
        pl[2] = pack2<T>(rem(sc[2 * k2 + 1][0]), rem(sc[2 * k2 + 1][1]));
        pl[3] = pack2<T>(rem(sc[2 * k2 + 1][2]), rem(sc[2 * k2 + 1][3]));
      }
      const int key = 16 * k2 + (mm & 1) * 8 + mr;
#pragma unroll
      for (int np = 0; np < NT / 2; ++np) {
        const int dim0 = 16 * np + (mm >> 1) * 8;
        const int col8 = (dim0 % 64) / 8;
        const uint32_t addr =
            vtile + (dim0 / 64) * Cfg::kColBytes + key * 128 + ((col8 ^ (key & 7)) << 4);
        uint32_t b[4];
        ldsm_x4_trans(b, addr);
        Op::run(o[2 * np], ph, b[0], b[1]);
        Op::run(o[2 * np + 1], ph, b[2], b[3]);
        if constexpr (kSplitP) {
          Op::run(o[2 * np], pl, b[0], b[1]);
          Op::run(o[2 * np + 1], pl, b[2], b[3]);
        }
      }
    }

    __syncthreads();  // every warp is done with this stage
    if (threadIdx.x == 0 && kt + Cfg::kStages < n_tiles) {
      fence_proxy_async();
      issue(kt + Cfg::kStages);
    }
  }
  if (timed_out) {
    const int last = n_tiles < kt + Cfg::kStages ? n_tiles : kt + Cfg::kStages;
    for (int jj = kt + 1; jj < last; ++jj)
      mbar_wait(bar0 + (jj % Cfg::kStages) * 8, (uint32_t)((jj / Cfg::kStages) & 1),
                kWaitLimitNs / 8);
    if (threadIdx.x == 0) set_error(p.err, PKV_DEV_TIMEOUT);
  }

  // ---- epilogue: normalise and store the rows that are real queries ------
  const bool real_lo = qa + r_lo / G < qend;
  const bool real_hi = qa + r_hi / G < qend;
  const float inv_lo = 1.f / l_lo, inv_hi = 1.f / l_hi;
  T* out_lo = out + ((int64_t)(q0 + qi_lo) * H + head_lo) * D;
  T* out_hi = out + ((int64_t)(q0 + qi_hi) * H + head_hi) * D;
#pragma unroll
  for (int n = 0; n < NT; ++n) {
    const int d = 8 * n + 2 * ti;
    if (real_lo)
      *reinterpret_cast<uint32_t*>(out_lo + d) = pack2<T>(o[n][0] * inv_lo, o[n][1] * inv_lo);
    if (real_hi)
      *reinterpret_cast<uint32_t*>(out_hi + d) = pack2<T>(o[n][2] * inv_hi, o[n][3] * inv_hi);
  }
}

template <typename T, int D, int BS, int G>
int launch_prefill_cfg(const PrefillParams& p, int num_seqs, const CUtensorMap& mk,
                       const CUtensorMap& mv, cudaStream_t stream) {
  using Cfg = PrefillCfg<T, D, BS, G>;
  auto kern = prefill_mma_kernel<T, D, BS, G>;
  static std::atomic<uint64_t> ready{0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ERR_CUDA;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(ready.load() & bit)) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024) !=
        cudaSuccess)
      return PKV_ERR_CUDA;
    ready.fetch_or(bit);
  }
  const int smem = Cfg::smem_bytes(p.max_blocks);
  if (smem > 227 * 1024) return PKV_ERR_ARG;
  dim3 grid((unsigned)((p.max_queries + Cfg::kQueries - 1) / Cfg::kQueries), (unsigned)p.kv_heads,
            (unsigned)num_seqs);
  kern<<<grid, Cfg::kThreads, smem, stream>>>(p, mk, mv);
  return cudaPeekAtLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

template <typename T, int D, int BS>
int launch_prefill_g(const PrefillParams& p, int num_seqs, int group, const CUtensorMap& mk,
                     const CUtensorMap& mv, cudaStream_t stream) {
  switch (group) {
    case 1: return launch_prefill_cfg<T, D, BS, 1>(p, num_seqs, mk, mv, stream);
    case 2: return launch_prefill_cfg<T, D, BS, 2>(p, num_seqs, mk, mv, stream);
    case 4: return launch_prefill_cfg<T, D, BS, 4>(p, num_seqs, mk, mv, stream);
    case 8: return launch_prefill_cfg<T, D, BS, 8>(p, num_seqs, mk, mv, stream);
  }
  return PKV_ERR_GEOMETRY;
}

template <typename T>
int launch_prefill(const PrefillParams& p, int num_seqs, int head_dim, int block_size, int group,
                   const CUtensorMap& mk, const CUtensorMap& mv, cudaStream_t stream) {
  switch (head_dim * 1000 + block_size) {
    case 64008: return launch_prefill_g<T, 64, 8>(p, num_seqs, group, mk, mv, stream);
    case 64016: return launch_prefill_g<T, 64, 16>(p, num_seqs, group, mk, mv, stream);
    case 64032: return launch_prefill_g<T, 64, 32>(p, num_seqs, group, mk, mv, stream);
    case 64064: return launch_prefill_g<T, 64, 64>(p, num_seqs, group, mk, mv, stream);
    case 128008: return launch_prefill_g<T, 128, 8>(p, num_seqs, group, mk, mv, stream);
    case 128016: return launch_prefill_g<T, 128, 16>(p, num_seqs, group, mk, mv, stream);
    case 128032: return launch_prefill_g<T, 128, 32>(p, num_seqs, group, mk, mv, stream);
    case 128064: return launch_prefill_g<T, 128, 64>(p, num_seqs, group, mk, mv, stream);
  }
  return PKV_ERR_GEOMETRY;
}

}  // namespace pkv
