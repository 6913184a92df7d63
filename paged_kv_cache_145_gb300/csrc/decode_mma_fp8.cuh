// Decode attention over FP8 E4M3 pools on tensor cores.
//
// Same method, grid, partitioning, merge and workspace as the other decode
// kernels.  Two variants:
//
// decode_partition_mma_fp8_kernel (head_dim 128).  Per warp, 16-position
// chunks of codes (keys and values of one KV head) arrive by 4-D TMA tile
// loads with the 128-byte swizzle in a two-stage ring.  Keys go straight
// from shared memory into tensor-core fragments: `ldmatrix` on the codes
// viewed as 16-bit pairs hands each lane four consecutive codes of a row,
// which are widened in registers; the head dimension is permuted the same
// way in the query fragments, so the dot products are unchanged.  Values
// are widened into a swizzled 16-bit tile (they must be transposed for
// P . V, which `ldmatrix` does on 16-bit data).  Both products run in fp16
// (every E4M3 value is exact in fp16; P keeps 11 bits, or about 22 as two
// fp16 parts for heads whose value scale needs it, see fp8_split_p); bf16
// queries are converted to fp16, exact for magnitudes in [2^-14, 2^15) and
// kept in range by a power-of-two scale of the group.
//
// decode_partition_mma_fp8_widen_kernel (head_dim 64).  Widens both keys and
// values into 16-bit tiles and reuses the fp16/bf16 fragment code.
//
// Key rows past the sequence end are masked; value rows past it are written
// as zeros, so stale codes (NaN included) never reach the accumulator.  The
// per-head key scale is folded into the score scale, the value scale into
// the output.
#pragma once

#include "decode_mma.cuh"

namespace pkv {

template <typename T, int D, int BS, int G>
struct Fp8WidenCfg {
  static constexpr int kWarps = 4;
  static constexpr int kThreads = kWarps * 32;
  static constexpr int kChunk = 16;
  static constexpr int kRawBytes = kChunk * D;            // codes of one tensor's chunk
  static constexpr int kRawStage = 2 * kRawBytes;         // keys + values
  static constexpr int kStages = 2;
  static constexpr int kCols = D / 64;                    // 128-byte column boxes (16-bit)
  static constexpr int kBoxBytes = kChunk * 128;
  static constexpr int kTileBytes = kCols * kBoxBytes;    // one widened 16-bit tile
  static constexpr int kWideBytes = kWarps * 2 * kTileBytes;
  static constexpr int kRawOff = kWideBytes;
  static constexpr int kBarOff = kRawOff + kWarps * kStages * kRawStage;
  static constexpr int kPtOff = kBarOff + kWarps * kStages * 8;
  static constexpr int kPtBytes = 2 * 8 * kChunk * 2;     // P^T, fp16, and its low part
  static constexpr int kTableOff = kPtOff + kWarps * kPtBytes;
  static constexpr int kAlign = 1024;
  static constexpr int kMergeBytes = (kWarps * G * D + 3 * kWarps * G + 2 * G) * 4;
  static_assert(kMergeBytes <= kWideBytes, "merge scratch must fit in the widened tiles");
  static_assert(D % 64 == 0 && G <= 8 && (BS % 16 == 0 || 16 % BS == 0), "geometry");
  static constexpr int smem_bytes(int part_size) { return kAlign + kTableOff + (part_size / BS) * 4; }
  static constexpr int kMaxSmem = kAlign + kTableOff + (kMaxPartSize / BS) * 4;
};

// Widens 16 codes (one 16-byte chunk) into two 16-byte chunks of 16-bit
// values of type W.
template <typename W>
__device__ __forceinline__ void widen16(const uint4& c, uint4& lo, uint4& hi) {
  uint32_t in[4] = {c.x, c.y, c.z, c.w};
  uint32_t out[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint16_t pair = (uint16_t)(in[i] >> (16 * h));
      const __half2_raw r = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)pair, __NV_E4M3);
      uint32_t w = (uint32_t)r.x | ((uint32_t)r.y << 16);
      if constexpr (std::is_same<W, __nv_bfloat16>::value) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w));
        const __nv_bfloat162 b = __float22bfloat162_rn(f);  // exact: E4M3 values fit bf16
        w = *reinterpret_cast<const uint32_t*>(&b);
      }
      out[2 * i + h] = w;
    }
  }
  lo = make_uint4(out[0], out[1], out[2], out[3]);
  hi = make_uint4(out[4], out[5], out[6], out[7]);
}

// P enters P.V in fp16 (unit roundoff 2^-11) and the values are codes of
// magnitude up to 448 times the head's value scale, so rounding P moves an
// output by at most 2^-11 * 448 * |v_scale|.  When that bound could exceed
// half of the output type's error bar for attention (max abs 2e-3 for fp16
// outputs, 8e-3 for bf16), P is used as two fp16 parts, the rounded value
// and the rounded remainder (about 22 significant bits), with one P.V
// product per part.  The other half of the bar covers the output's own
// rounding.  T is the output type.
template <typename T>
__device__ __forceinline__ bool fp8_split_p(float v_scale) {
  const float half_bar = std::is_same<T, __half>::value ? 1e-3f : 4e-3f;
  return 448.f * 0x1p-11f * fabsf(v_scale) > half_bar;
}

// P^T of one chunk through shared memory: lane (gi, ti) holds P of
// positions gi and gi + 8 for heads 2ti, 2ti + 1; entry [head][position]
// (C positions per head) holds its fp16 bits, and, when split, the fp16
// bits of the remainder 8 * C entries further.
template <int C>
__device__ __forceinline__ void stage_pt(uint16_t* pt, int gi, int ti, const float (&pr)[4],
                                         bool split) {
  const int idx[4] = {(2 * ti) * C + gi, (2 * ti + 1) * C + gi, (2 * ti) * C + gi + 8,
                      (2 * ti + 1) * C + gi + 8};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __half h = __float2half_rn(pr[i]);
    pt[idx[i]] = __half_as_ushort(h);
    if (split) pt[8 * C + idx[i]] = __half_as_ushort(__float2half_rn(pr[i] - __half2float(h)));
  }
}

// Widens the four E4M3 codes of a 32-bit word into two fp16 pairs
// (codes 0-1 -> lo, codes 2-3 -> hi) with the hardware conversion.
__device__ __forceinline__ void e4m3x4_to_f16x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, l;\n\tcvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
}

template <typename T, int D, int BS, int G>
__global__ void __launch_bounds__(Fp8WidenCfg<T, D, BS, G>::kThreads)
decode_partition_mma_fp8_widen_kernel(const DecodeParams p) {
  using Cfg = Fp8WidenCfg<T, D, BS, G>;
  using OpK = MmaOp<T>;        // q . K in the query's type
  using OpV = MmaOp<__half>;   // P . V in fp16
  constexpr int C = Cfg::kChunk;
  constexpr int NW = Cfg::kWarps;
  constexpr int NST = Cfg::kStages;
  constexpr int KSTEPS = D / 16;
  constexpr int CPR = D / 16;     // 16-byte code chunks per row
  constexpr int RPP = 32 / CPR;   // rows widened per pass of the warp
  extern __shared__ __align__(128) unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((Cfg::kAlign - (smem_addr(smem_raw) & (Cfg::kAlign - 1))) &
                                    (Cfg::kAlign - 1));

  const int kvh = blockIdx.x;
  const int s = blockIdx.y;
  const int part = blockIdx.z;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int gi = lane >> 2;
  const int ti = lane & 3;
  const int H = p.num_heads;
  T* out = static_cast<T*>(p.out);
  const int64_t out0 = ((int64_t)s * H + (int64_t)kvh * G) * D;
  const int PS = p.part_size;
  const int tok0 = part * PS;
  const int blk0 = tok0 / BS;

  const int32_t* trow = p.tables + (int64_t)s * p.max_blocks + blk0;
  const int span = min(PS / BS, p.max_blocks - blk0);
  const int L = ld_nc(p.seq_lens + s);
  const int e_first = (int)threadIdx.x < span ? ld_nc(trow + threadIdx.x) : -1;

  if (L < 1 || L > p.max_len) {
    if (part == 0) {
      for (int e = threadIdx.x; e < G * D; e += Cfg::kThreads) out[out0 + e] = Elem<T>::from_f(0.f);
      if (threadIdx.x == 0) set_error(p.err, PKV_DEV_SEQ_LEN);
    }
    return;
  }
  if (tok0 >= L) return;
  const int ntok = min(L - tok0, PS);
  const int nparts = (L + PS - 1) / PS;
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
  const char* kbase = static_cast<const char*>(p.k_cache);
  const char* vbase = static_cast<const char*>(p.v_cache);
  const uint32_t raw0 = smem_addr(smem + Cfg::kRawOff) + warp * NST * Cfg::kRawStage;
  const uint32_t bar0 = smem_addr(&bars[warp * NST]);
  const uint64_t policy = policy_evict_first();
  constexpr int RB = BS < 16 ? BS : 16;

  // Chunk c covers partition positions 16c .. 16c+15: 16 rows of one block,
  // or (b = 8) two whole blocks; a second block past the partition's end is
  // not loaded.
  auto issue = [&](int j) {
    const int c = warp + j * NW;
    const int st = j % NST;
    const uint32_t bar = bar0 + st * 8;
    const uint32_t dst = raw0 + st * Cfg::kRawStage;
    const int nbox = (RB < 16 && c * C + RB < ntok) ? 2 : 1;
    mbar_arrive_expect_tx(bar, nbox * RB * D * 2);
    for (int hb = 0; hb < nbox; ++hb) {
      const int pos = c * C + hb * RB;
      const int pb = stable[pos / BS];
      const int64_t off = (((int64_t)pb * p.kv_heads + kvh) * BS + pos % BS) * D;
      bulk_g2s(dst + hb * RB * D, kbase + off, RB * D, bar, policy);
      bulk_g2s(dst + Cfg::kRawBytes + hb * RB * D, vbase + off, RB * D, bar, policy);
    }
  };
  if (lane == 0) {
    const int pre = count < NST ? count : NST;
    for (int j = 0; j < pre; ++j) issue(j);
  }

  // Q^T as B fragments (head gi, zero beyond G), in the query's type.
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
  const float qs = p.qscale * p.k_scale[kvh];

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
  unsigned char* ktw = smem + warp * 2 * Cfg::kTileBytes;  // widened keys
  unsigned char* vtw = ktw + Cfg::kTileBytes;              // widened values
  const uint32_t ktile = smem_addr(ktw), vtile = smem_addr(vtw);
  uint16_t* pt = reinterpret_cast<uint16_t*>(smem + Cfg::kPtOff + warp * Cfg::kPtBytes);
  // Each CTA uses P as one fp16 part or two (fp8_split_p, the same for the
  // whole CTA): the chunk loop is compiled once per form and chosen here,
  // so no per-chunk test of the form stays in it.
  const bool split_p = fp8_split_p<T>(p.v_scale[kvh]);
  auto chunks = [&](auto split_tag) {
    constexpr bool SPLIT = decltype(split_tag)::value;
    int j = 0;
    for (; j < count; ++j) {
      const int st = j % NST;
      timed_out = __any_sync(kFullMask, !mbar_wait(bar0 + st * 8, (uint32_t)((j / NST) & 1)));
      if (timed_out) break;
      const int c = warp + j * NW;
      const int nvalid = min(C, ntok - c * C);

      // ---- widen the chunk's codes into the swizzled 16-bit tiles ----------
      {
        const unsigned char* raw = smem + Cfg::kRawOff + (warp * NST + st) * Cfg::kRawStage;
        const int cc = lane % CPR;  // 16-byte code chunk = dims 16cc .. 16cc+15
  #pragma unroll
        for (int pass = 0; pass < C / RPP; ++pass) {
          const int r = pass * RPP + lane / CPR;
          const uint4 kc = *reinterpret_cast<const uint4*>(raw + r * D + cc * 16);
          const uint4 vc = *reinterpret_cast<const uint4*>(raw + Cfg::kRawBytes + r * D + cc * 16);
          uint4 k0, k1, v0, v1;
          widen16<T>(kc, k0, k1);
          widen16<__half>(vc, v0, v1);
          if (r >= nvalid) v0 = v1 = make_uint4(0u, 0u, 0u, 0u);
          const int box = (16 * cc) / 64;
          const int c8 = ((16 * cc) % 64) / 8;  // first of the two 16-byte chunks
          unsigned char* kr = ktw + box * Cfg::kBoxBytes + r * 128;
          unsigned char* vr = vtw + box * Cfg::kBoxBytes + r * 128;
          *reinterpret_cast<uint4*>(kr + ((c8 ^ (r & 7)) << 4)) = k0;
          *reinterpret_cast<uint4*>(kr + (((c8 + 1) ^ (r & 7)) << 4)) = k1;
          *reinterpret_cast<uint4*>(vr + ((c8 ^ (r & 7)) << 4)) = v0;
          *reinterpret_cast<uint4*>(vr + (((c8 + 1) ^ (r & 7)) << 4)) = v1;
        }
      }
      __syncwarp();
      if (lane == 0 && j + NST < count) {  // the raw stage is free again
        fence_proxy_async();
        issue(j + NST);
      }

      // ---- S^T = K . Q^T ----------------------------------------------------
      float sc[4] = {0.f, 0.f, 0.f, 0.f};
  #pragma unroll
      for (int kk = 0; kk < KSTEPS; ++kk) {
        const int col8 = 2 * (kk % 4) + k_col8;
        const uint32_t addr =
            ktile + (kk / 4) * Cfg::kBoxBytes + k_tok * 128 + ((col8 ^ (k_tok & 7)) << 4);
        uint32_t a[4];
        ldsm_x4(a, addr);
        OpK::run(sc, a, qb[kk][0], qb[kk][1]);
      }

      // ---- online softmax per head column ------------------------------------
      const bool v0 = gi < nvalid, v1 = gi + 8 < nvalid;
      float x[4];
      x[0] = v0 ? sc[0] * qs : -INFINITY;
      x[1] = v0 ? sc[1] * qs : -INFINITY;
      x[2] = v1 ? sc[2] * qs : -INFINITY;
      x[3] = v1 ? sc[3] * qs : -INFINITY;
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

      // ---- P^T (fp16) through shared memory ---------------------------------
      stage_pt<C>(pt, gi, ti, pr, SPLIT);
      __syncwarp();
      const uint32_t* ptw = reinterpret_cast<const uint32_t*>(pt);
      const uint32_t b0 = ptw[(gi * C + 2 * ti) / 2];
      const uint32_t b1 = ptw[(gi * C + 2 * ti + 8) / 2];
      const uint32_t b0l = SPLIT ? ptw[(8 * C + gi * C + 2 * ti) / 2] : 0u;
      const uint32_t b1l = SPLIT ? ptw[(8 * C + gi * C + 2 * ti + 8) / 2] : 0u;

      // ---- O^T += V^T . P^T (fp16; low part too when split) -------------------
  #pragma unroll
      for (int i = 0; i < KSTEPS; ++i) {
        const int col8 = 2 * (i % 4) + v_col8;
        const uint32_t addr =
            vtile + (i / 4) * Cfg::kBoxBytes + v_tok * 128 + ((col8 ^ (v_tok & 7)) << 4);
        uint32_t a[4];
        ldsm_x4_trans(a, addr);
        OpV::run(acc[i], a, b0, b1);
        if constexpr (SPLIT) OpV::run(acc[i], a, b0l, b1l);
      }
      __syncwarp();  // the widened tiles and P^T are rewritten next chunk
    }
    return j;
  };
  const int j = split_p ? chunks(std::true_type{}) : chunks(std::false_type{});
  if (timed_out) {
    const int last = count < j + NST ? count : j + NST;
    for (int jj = j + 1; jj < last; ++jj)
      mbar_wait(bar0 + (jj % NST) * 8, (uint32_t)((jj / NST) & 1), kWaitLimitNs / 8);
    if (lane == 0) set_error(p.err, PKV_DEV_TIMEOUT);
  }

  // ---- merge the warps ----------------------------------------------------
  __syncthreads();
  float* red_acc = reinterpret_cast<float*>(smem);
  float* red_m = red_acc + NW * G * D;
  float* red_l = red_m + NW * G;
  float* fac = red_l + NW * G;
  float* fin = fac + NW * G;
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
  const float vscale = p.v_scale[kvh];
  for (int e = threadIdx.x; e < G * D; e += Cfg::kThreads) {
    const int g = e / D;
    const int d = e - g * D;
    float o = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) o = fmaf(red_acc[(w * G + g) * D + d], fac[w * G + g], o);
    o = o / fin[G + g] * vscale;
    if (nparts == 1)
      out[out0 + e] = Elem<T>::from_f(o);
    else
      p.ws_o[(ws0 + (int64_t)g * p.num_parts) * D + d] = o;
  }
  if (nparts > 1 && threadIdx.x < G)
    p.ws_ml[ws0 + (int64_t)threadIdx.x * p.num_parts] =
        make_float2(fin[threadIdx.x], fin[G + threadIdx.x]);
}

template <typename T, int D, int BS, int G>
struct Fp8MmaCfg {
  static constexpr int kWarps = 4;
  static constexpr int kMinBlocks = 4;  // CTAs per SM the register budget targets
  static constexpr int kThreads = kWarps * 32;
  static constexpr int kChunk = 16;
  static constexpr int kBoxRows = BS < 16 ? BS : 16;
  static constexpr int kRawBytes = kChunk * D;            // 16 rows x 128 codes, swizzled
  static constexpr int kRawStage = 2 * kRawBytes;         // keys + values
  static constexpr int kStages = 2;  // raw stages per warp
  static constexpr int kRingBytes = kWarps * kStages * kRawStage;
  static constexpr int kBarOff = kRingBytes;
  static constexpr int kPtOff = kBarOff + kWarps * kStages * 8;
  static constexpr int kPtBytes = 2 * 8 * kChunk * 2;  // P^T, fp16, and its low part
  static constexpr int kTableOff = kPtOff + kWarps * kPtBytes;
  static constexpr int kAlign = 1024;
  static constexpr int kMergeBytes = (kWarps * G * D + 3 * kWarps * G + 2 * G) * 4;
  static_assert(D == 128, "direct key fragments need 128-byte code rows");
  static_assert(kMergeBytes <= kRingBytes, "merge scratch");
  static_assert(BS % 16 == 0 || 16 % BS == 0, "block size");
  static constexpr int smem_bytes(int part_size) { return kAlign + kTableOff + (part_size / BS) * 4; }
  static constexpr int kMaxSmem = kAlign + kTableOff + (kMaxPartSize / BS) * 4;
};

template <typename T, int D, int BS, int G>
__global__ void __launch_bounds__(Fp8MmaCfg<T, D, BS, G>::kThreads, Fp8MmaCfg<T, D, BS, G>::kMinBlocks)
decode_partition_mma_fp8_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap tmk,
                                const __grid_constant__ CUtensorMap tmv) {
  using Cfg = Fp8MmaCfg<T, D, BS, G>;
  using Op = MmaOp<__half>;  // q . K and P . V both in fp16
  constexpr int C = Cfg::kChunk;
  constexpr int NW = Cfg::kWarps;
  constexpr int NST = Cfg::kStages;
  constexpr int KSTEPS = D / 16;
  constexpr int RB = Cfg::kBoxRows;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((Cfg::kAlign - (smem_addr(smem_raw) & (Cfg::kAlign - 1))) &
                                    (Cfg::kAlign - 1));

  const int kvh = blockIdx.x;
  const int s = blockIdx.y;
  const int part = blockIdx.z;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int gi = lane >> 2;
  const int ti = lane & 3;
  const int H = p.num_heads;
  T* out = static_cast<T*>(p.out);
  const int64_t out0 = ((int64_t)s * H + (int64_t)kvh * G) * D;
  const int PS = p.part_size;
  const int tok0 = part * PS;
  const int blk0 = tok0 / BS;

  const int32_t* trow = p.tables + (int64_t)s * p.max_blocks + blk0;
  const int span = min(PS / BS, p.max_blocks - blk0);
  const int L = ld_nc(p.seq_lens + s);
  const int e_first = (int)threadIdx.x < span ? ld_nc(trow + threadIdx.x) : -1;

  if (L < 1 || L > p.max_len) {
    if (part == 0) {
      for (int e = threadIdx.x; e < G * D; e += Cfg::kThreads) out[out0 + e] = Elem<T>::from_f(0.f);
      if (threadIdx.x == 0) set_error(p.err, PKV_DEV_SEQ_LEN);
    }
    return;
  }
  if (tok0 >= L) return;
  const int ntok = min(L - tok0, PS);
  const int nparts = (L + PS - 1) / PS;
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
  const uint32_t raw0 = smem_addr(smem) + warp * NST * Cfg::kRawStage;
  const uint32_t bar0 = smem_addr(&bars[warp * NST]);
  const uint64_t policy = policy_evict_first();
  auto issue = [&](int j) {
    const int c = warp + j * NW;
    const int st = j % NST;
    const uint32_t bar = bar0 + st * 8;
    const uint32_t dst = raw0 + st * Cfg::kRawStage;
    const int nbox = (RB < 16 && c * C + RB < ntok) ? 2 : 1;
    mbar_arrive_expect_tx(bar, nbox * RB * D * 2);
    for (int hb = 0; hb < nbox; ++hb) {
      const int pos = c * C + hb * RB;
      const int pb = stable[pos / BS];
      tma_load_4d(dst + hb * RB * D, &tmk, 0, pos % BS, kvh, pb, bar, policy);
      tma_load_4d(dst + Cfg::kRawBytes + hb * RB * D, &tmv, 0, pos % BS, kvh, pb, bar, policy);
    }
  };
  if (lane == 0) {
    const int pre = count < NST ? count : NST;
    for (int j = 0; j < pre; ++j) issue(j);
  }

  // Q^T B fragments, in fp16, in the permuted head-dim order the key
  // fragments use: k-step kk covers dims 16kk .. 16kk+15; lane (gi, ti)
  // pairs logical rows 2ti, 2ti+1 with dims 16kk + 4ti, +1 and rows 2ti+8,
  // 2ti+9 with dims 16kk + 4ti + 2, +3.  bf16 queries whose largest
  // magnitude in the group reaches 2^15 are first scaled by a power of two
  // (undone in the score scale) so that they stay inside fp16's range.
  uint32_t qb[KSTEPS][2];
  float qs = p.qscale * p.k_scale[kvh];
  {
    const T* qrow = static_cast<const T*>(p.q) + out0 + (int64_t)gi * D;
    float f[KSTEPS][4];
    float amax = 0.f;
#pragma unroll
    for (int kk = 0; kk < KSTEPS; ++kk) {
#pragma unroll
      for (int c = 0; c < 4; ++c) f[kk][c] = 0.f;
      if (gi < G) RowLoad<T, 4>::load(qrow + 16 * kk + 4 * ti, f[kk]);
#pragma unroll
      for (int c = 0; c < 4; ++c) amax = fmaxf(amax, fabsf(f[kk][c]));
    }
    float shrink = 1.f;
    if (!std::is_same<T, __half>::value) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
      int e = 0;
      if (amax >= 32768.f && amax <= 3.0e38f) {
        frexpf(amax, &e);  // amax = m * 2^e, m in [0.5, 1)
        e -= 15;
        shrink = ldexpf(1.f, -e);
        qs = ldexpf(qs, e);
      }
    }
#pragma unroll
    for (int kk = 0; kk < KSTEPS; ++kk) {
      const __half2 a = __floats2half2_rn(f[kk][0] * shrink, f[kk][1] * shrink);
      const __half2 b = __floats2half2_rn(f[kk][2] * shrink, f[kk][3] * shrink);
      qb[kk][0] = *reinterpret_cast<const uint32_t*>(&a);
      qb[kk][1] = *reinterpret_cast<const uint32_t*>(&b);
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
  const int k_row = (mm & 1) * 8 + mr;  // ldmatrix row this lane addresses (keys)
  const int k_half = mm >> 1;           // which 16-code chunk of the pair
  uint16_t* pt = reinterpret_cast<uint16_t*>(smem + Cfg::kPtOff + warp * Cfg::kPtBytes);
  // Each CTA uses P as one fp16 part or two (fp8_split_p, the same for the
  // whole CTA): the chunk loop is compiled once per form and chosen here,
  // so no per-chunk test of the form stays in it.
  const bool split_p = fp8_split_p<T>(p.v_scale[kvh]);
  auto chunks = [&](auto split_tag) {
    constexpr bool SPLIT = decltype(split_tag)::value;
    int j = 0;
    for (; j < count; ++j) {
      const int st = j % NST;
      timed_out = __any_sync(kFullMask, !mbar_wait(bar0 + st * 8, (uint32_t)((j / NST) & 1)));
      if (timed_out) break;
      const int c = warp + j * NW;
      const int nvalid = min(C, ntok - c * C);
      const uint32_t kraw = raw0 + st * Cfg::kRawStage;
      const unsigned char* vraw = smem + (kraw - smem_addr(smem)) + Cfg::kRawBytes;

      // ---- S^T = K . Q^T, key fragments straight from the codes -------------
      float sc[4] = {0.f, 0.f, 0.f, 0.f};
  #pragma unroll
      for (int kp = 0; kp < KSTEPS / 2; ++kp) {  // two k-steps (32 codes) per ldmatrix
        const int chunk = 2 * kp + k_half;
        uint32_t r[4];
        ldsm_x4(r, kraw + k_row * 128 + ((chunk ^ (k_row & 7)) << 4));
        // r[0]: row gi, 4 codes of chunk 2kp; r[1]: row gi+8; r[2], r[3]: chunk 2kp+1.
  #pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t a[4];
          e4m3x4_to_f16x4(r[2 * h], a[0], a[2]);
          e4m3x4_to_f16x4(r[2 * h + 1], a[1], a[3]);
          Op::run(sc, a, qb[2 * kp + h][0], qb[2 * kp + h][1]);
        }
      }

      // ---- online softmax per head column ------------------------------------
      const bool v0 = gi < nvalid, v1 = gi + 8 < nvalid;
      float x[4];
      x[0] = v0 ? sc[0] * qs : -INFINITY;
      x[1] = v0 ? sc[1] * qs : -INFINITY;
      x[2] = v1 ? sc[2] * qs : -INFINITY;
      x[3] = v1 ? sc[3] * qs : -INFINITY;
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
      stage_pt<C>(pt, gi, ti, pr, SPLIT);
      __syncwarp();
      const uint32_t* ptw = reinterpret_cast<const uint32_t*>(pt);
      const uint32_t b0 = ptw[(gi * C + 2 * ti) / 2];
      const uint32_t b1 = ptw[(gi * C + 2 * ti + 8) / 2];
      const uint32_t b0l = SPLIT ? ptw[(8 * C + gi * C + 2 * ti) / 2] : 0u;
      const uint32_t b1l = SPLIT ? ptw[(8 * C + gi * C + 2 * ti + 8) / 2] : 0u;

      // ---- O^T += V^T . P^T, value fragments straight from the codes --------
      // The contraction runs over positions, which sit in different code rows,
      // so each lane gathers a 4 x 4 byte block: dims 4w .. 4w+3 (w = gi + 8q)
      // of rows 2ti, 2ti+1, 2ti+8, 2ti+9 (four 32-bit loads that hit 32
      // distinct banks under the 128-byte swizzle), pairs the bytes of two
      // rows per dim with byte permutes and widens them to fp16.  The M rows
      // of the two tiles of group q are dims 4w, 4w+1 (tile 2q) and 4w+2,
      // 4w+3 (tile 2q+1); the merge below undoes that order.
      {
        const int r0 = 2 * ti;
        const bool ok0 = r0 < nvalid, ok1 = r0 + 1 < nvalid, ok2 = r0 + 8 < nvalid,
                   ok3 = r0 + 9 < nvalid;
  #pragma unroll
        for (int q = 0; q < D / 32; ++q) {
          const int w = gi + 8 * q;
          const int ch = w >> 2, wo = (w & 3) * 4;
          auto word = [&](int r, bool ok) -> uint32_t {
            return ok ? *reinterpret_cast<const uint32_t*>(vraw + r * 128 + ((ch ^ (r & 7)) << 4) + wo)
                      : 0u;
          };
          const uint32_t x0 = word(r0, ok0), x1 = word(r0 + 1, ok1);
          const uint32_t x2 = word(r0 + 8, ok2), x3 = word(r0 + 9, ok3);
          uint32_t a[4], b[4];
          e4m3x4_to_f16x4(__byte_perm(x0, x1, 0x5140), a[0], a[1]);
          e4m3x4_to_f16x4(__byte_perm(x2, x3, 0x5140), a[2], a[3]);
          e4m3x4_to_f16x4(__byte_perm(x0, x1, 0x7362), b[0], b[1]);
          e4m3x4_to_f16x4(__byte_perm(x2, x3, 0x7362), b[2], b[3]);
          Op::run(acc[2 * q], a, b0, b1);
          Op::run(acc[2 * q + 1], b, b0, b1);
          if constexpr (SPLIT) {
            Op::run(acc[2 * q], a, b0l, b1l);
            Op::run(acc[2 * q + 1], b, b0l, b1l);
          }
        }
      }
      __syncwarp();  // the raw stage and P^T are rewritten next
      if (lane == 0 && j + NST < count) {  // raw stage consumed: refill it
        fence_proxy_async();
        issue(j + NST);
      }
    }
    return j;
  };
  const int j = split_p ? chunks(std::true_type{}) : chunks(std::false_type{});
  if (timed_out) {
    const int last = count < j + NST ? count : j + NST;
    for (int jj = j + 1; jj < last; ++jj)
      mbar_wait(bar0 + (jj % NST) * 8, (uint32_t)((jj / NST) & 1), kWaitLimitNs / 8);
    if (lane == 0) set_error(p.err, PKV_DEV_TIMEOUT);
  }

  // ---- merge the warps ----------------------------------------------------
  __syncthreads();
  float* red_acc = reinterpret_cast<float*>(smem);
  float* red_m = red_acc + NW * G * D;
  float* red_l = red_m + NW * G;
  float* fac = red_l + NW * G;
  float* fin = fac + NW * G;
  // Lane (gi, ti) holds dims 4w .. 4w+3 (w = gi + 8q) of heads 2ti, 2ti+1.
#pragma unroll
  for (int q = 0; q < D / 32; ++q)
#pragma unroll
    for (int h = 0; h < 2; ++h)
      if (2 * ti + h < G)
        *reinterpret_cast<float4*>(&red_acc[(warp * G + 2 * ti + h) * D + 4 * (gi + 8 * q)]) =
            make_float4(acc[2 * q][h], acc[2 * q][2 + h], acc[2 * q + 1][h], acc[2 * q + 1][2 + h]);
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
  const float vscale = p.v_scale[kvh];
  for (int e = threadIdx.x; e < G * D; e += Cfg::kThreads) {
    const int g = e / D;
    const int d = e - g * D;
    float o = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) o = fmaf(red_acc[(w * G + g) * D + d], fac[w * G + g], o);
    o = o / fin[G + g] * vscale;
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
