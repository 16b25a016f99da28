// Split-K paged GQA decode attention for GB300 (sm_103a).
//
// The computation (llama.cpp fork PR #2, split-K decode commit: "Split-K flash
// decoding for head size 256, GQA 6 and 1-4 query tokens (MTP verify widths)
// with ... packed in-register dequantization"; lucebox PR #555, Summary:
// "GQA-aware thread blocks, occupancy-aware context parallelism, adaptive
// long-context partitioning, and a stable split-softmax merge"):
//   for every (sequence, KV head) the 6 * n_qtok query rows of that KV head
//   attend to the sequence's rows, read page by page through the block table;
//   K/V are dequantised in registers, S = QK^T and O = PV run on the tensor
//   cores, the softmax is online, and the splits are merged by log-sum-exp.
//
// GB300 design:
//   * Work split.  Every (sequence, KV head) is a segment of 64-key tiles.  All
//     tiles of the batch are laid end to end and cut into equal contiguous
//     ranges, one per CTA, with as many CTAs as fit on the SMs at once
//     (occupancy x SM count).  A CTA's range may cover the tail of one segment
//     and the head of the next; each piece becomes one split partial.  The cut
//     depends only on the sequence lengths, so a paged and an identity-table
//     cache give the same splits, the same summation order and bit-identical
//     results (TensorFold #1156, Design/Kernels: "only the address changes;
//     the per-key summation order does not").
//   * Data movement.  One producer warp streams K and V tiles into a ring of
//     shared-memory stages with cp.async.bulk (the TMA engine's 1-D copy),
//     one copy per page run (or per row for F16, into a padded layout that
//     keeps the fragment loads bank-conflict free), completing on mbarriers.
//     The page table is read once per page run, never per key (TensorFold
//     #1156: "test once per block").  A table entry outside the pool is never
//     dereferenced: its rows are zero-filled and PA_ERR_BOUNDS is recorded.
//   * Compute.  Four consumer warps.  In the S phase warp w takes keys
//     16w..16w+15 of the tile and computes S^T = K Q^T with mma.sync
//     m16n8k16 (M = keys, N = query rows, K = head dims): K is dequantised
//     straight into A fragments, Q sits in shared memory pre-swizzled into B
//     fragments.  The dims are visited in whatever order makes each thread's
//     loads contiguous; Q is laid out in the same order, so the dot products
//     are unchanged.  Each warp publishes its tile max, row sums and fp16 P
//     (transposed into B-fragment order with movmatrix).  In the PV phase warp
//     w owns head dims 64w..64w+63 and computes O^T += V^T P^T over the whole
//     tile (M = dims, N = query rows, K = keys), V dequantised into A
//     fragments.  One named barrier per tile separates the phases.
//   * Merge.  Pieces that cover a whole segment write the final output; the
//     others write (m, l, O) partials to the caller's workspace, and a small
//     merge kernel combines them by log-sum-exp (llama.cpp fork PR #2, LSE
//     commit), with an all-masked row giving 0, not NaN (pd_combine fix).
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "pa.h"
#include "pa_device.cuh"

using namespace pa_dev;

namespace {

constexpr int kD = 256;          // head dim
constexpr int kGqa = 6;          // query heads per KV head
constexpr int kTile = 64;        // keys per tile
constexpr int kCWarps = 4;       // consumer warps
constexpr int kThreads = (kCWarps + 1) * 32;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// ------------------------------------------------------------------ formats

template <int T>
struct Fmt;
template <>
struct Fmt<PA_F16> {
  static constexpr int kRow = 512;     // bytes per stored row
  static constexpr int kStride = 528;  // shared-memory row stride (padded)
};
template <>
struct Fmt<PA_Q4_0> {
  static constexpr int kRow = 144;
  static constexpr int kStride = 144;
};
template <>
struct Fmt<PA_Q8_0> {
  static constexpr int kRow = 272;
  static constexpr int kStride = 272;
};

// Bytes of shared memory outside the stage ring for NT query-row tiles.
constexpr int extras_bytes(int NT) {
  return 2 * 16 * NT * 32 * 8 + 2 * kCWarps * NT * 32 * 8 + 2 * kCWarps * NT * 8 * 8 + 2 * 8 * 8 + 32;
}

// Ring depth: as many stages (2..6) as fit when two CTAs share an SM; if even
// three stages do not fit that way, one CTA per SM with up to 3 stages.
template <int KT, int VT, int NT>
struct Stages {
  static constexpr int kStageBytes = kTile * (Fmt<KT>::kStride + Fmt<VT>::kStride);
  static constexpr int kTwoPerSm = 115712;   // (228 KB - 2 x 1 KB reserved) / 2
  static constexpr int kOnePerSm = 232448;   // 227 KB per-CTA maximum
  static constexpr int kFit2 = (kTwoPerSm - extras_bytes(NT)) / kStageBytes;
  static constexpr int kFit1 = (kOnePerSm - extras_bytes(NT)) / kStageBytes;
  static constexpr int kN = kFit2 >= 3 ? (kFit2 > 6 ? 6 : kFit2) : (kFit1 > 3 ? 3 : kFit1);
  static_assert(kN >= 2, "stage ring does not fit");
};

// Head dim that k-step s, A/B k-index j of the S-MMA stands for, per K format.
// j = 2t + 8h + e (t = thread in quad, h = upper half, e = element in pair).
template <int KT>
__device__ __forceinline__ int kdim(int s, int j) {
  const int t = (j & 7) >> 1, e = j & 1, h = j >> 3;
  if (KT == PA_F16) {  // s = 4c + u: thread t loads dims 64c + 16t .. +15
    const int c = s >> 2, u = s & 3;
    return 64 * c + 16 * t + 4 * u + 2 * h + e;
  } else if (KT == PA_Q8_0) {  // s = 2b + u: thread t owns quants 8t..8t+7 of block b
    const int b = s >> 1, u = s & 1;
    return 32 * b + 8 * t + 4 * u + h + 2 * e;
  } else {  // Q4_0, s = 2b + u: thread t owns quant bytes 4t..4t+3 of block b
    const int b = s >> 1, u = s & 1;
    return 32 * b + 4 * t + 16 * u + h + 2 * e;
  }
}

// Head dim of O^T row (m-tile i, fragment row g + 8h) for warp w, per V format.
template <int VT>
__device__ __forceinline__ int vdim(int w, int g, int i, int h) {
  const int k = 2 * i + h;  // index into the thread's 8 dims
  if (VT == PA_F16) return 64 * w + 8 * g + k;
  const int blk = 2 * w + (g >> 2);
  if (VT == PA_Q8_0) return 32 * blk + 8 * (g & 3) + k;
  // Q4_0: [j0, j0+16, j0+1, j0+17, j0+2, j0+18, j0+3, j0+19]
  return 32 * blk + 4 * (g & 3) + (k >> 1) + 16 * (k & 1);
}

// ------------------------------------------------------------------ dequant helpers

constexpr uint32_t kHalf2_1032 = 0x64086408u;  // 1032.0
constexpr uint32_t kHalf2_1152 = 0x64806480u;  // 1152.0
constexpr uint32_t kHalf2_1_16 = 0x2c002c00u;  // 0.0625
constexpr uint32_t kHalf2_m72 = 0xd480d480u;   // -72.0

// 4 quant bytes 4t..4t+3 of Q4_0 block b of the row at `row` (shared address).
__device__ __forceinline__ uint32_t q4_word(uint32_t row, int b, int t) {
  const uint32_t o = row + 18 * b + 4 * t;
  if (b & 1) return lds32(o + 2);
  return prmt(lds32(o), lds32(o + 4), 0x5432);
}

// 8 int8 quants 8t..8t+7 of Q8_0 block b.
__device__ __forceinline__ void q8_words(uint32_t row, int b, int t, uint32_t& y0, uint32_t& y1) {
  const uint32_t o = row + 34 * b + 2 + 8 * t;
  if (b & 1) {
    y0 = lds32(o);
    y1 = lds32(o + 4);
  } else {
    const uint32_t w0 = lds32(o - 2), w1 = lds32(o + 2), w2 = lds32(o + 6);
    y0 = prmt(w0, w1, 0x5432);
    y1 = prmt(w1, w2, 0x5432);
  }
}

// fp16 scale of block b broadcast to both halves.
__device__ __forceinline__ uint32_t scale2(uint32_t row, int blk_bytes, int b) {
  const uint32_t d = lds16(row + blk_bytes * b);
  return d | (d << 16);
}

// Q4_0: nibbles of x = [c0 c1 c2 c3] -> (n - 8) * d as fp16 pairs.
//   lo0 = (c0.lo, c2.lo)  hi0 = (c0.hi, c2.hi)  lo1 = (c1.lo, c3.lo)  hi1 = (c1.hi, c3.hi)
__device__ __forceinline__ void q4_dequant(uint32_t x, uint32_t dd, uint32_t& lo0, uint32_t& hi0, uint32_t& lo1,
                                           uint32_t& hi1) {
  const uint32_t x8 = x >> 8;
  lo0 = hmul2(hadd2(and_or(x, 0x000f000fu, 0x64006400u), kHalf2_1032 ^ 0x80008000u), dd);
  hi0 = hmul2(hfma2(and_or(x, 0x00f000f0u, 0x64006400u), kHalf2_1_16, kHalf2_m72), dd);
  lo1 = hmul2(hadd2(and_or(x8, 0x000f000fu, 0x64006400u), kHalf2_1032 ^ 0x80008000u), dd);
  hi1 = hmul2(hfma2(and_or(x8, 0x00f000f0u, 0x64006400u), kHalf2_1_16, kHalf2_m72), dd);
}

// Q8_0: int8 quants y = [x0 x1 x2 x3] -> e0 = (x0, x2) * d, e1 = (x1, x3) * d.
__device__ __forceinline__ void q8_dequant(uint32_t y, uint32_t dd, uint32_t& e0, uint32_t& e1) {
  const uint32_t u = y ^ 0x80808080u;  // x + 128
  e0 = hmul2(hadd2(prmt(u, 0x64646464u, 0x4240), kHalf2_1152 ^ 0x80008000u), dd);
  e1 = hmul2(hadd2(prmt(u, 0x64646464u, 0x4341), kHalf2_1152 ^ 0x80008000u), dd);
}

// ------------------------------------------------------------------ S phase (K side)

// acc[nt] += K(16 keys: rows r0 = key g, r1 = key g+8) x Qfrag over all 16 k-steps.
// qf: shared address of this lane's Q fragments, [s][nt][lane] uint2.
template <int KT, int NT>
__device__ __forceinline__ void s_phase(float (&acc)[NT][4], uint32_t r0, uint32_t r1, uint32_t qf, int lane) {
  const int t = lane & 3;
  auto mma_ks = [&](int s, const uint32_t (&a)[4]) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const uint2 b = lds64(qf + ((s * NT + nt) * 32) * 8);
      mma_16816(acc[nt], a, b.x, b.y);
    }
  };
  if constexpr (KT == PA_F16) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const uint32_t off = 128 * c + 32 * t;
      const uint4 R0 = lds128(r0 + off), R1 = lds128(r0 + off + 16);
      const uint4 S0 = lds128(r1 + off), S1 = lds128(r1 + off + 16);
      { const uint32_t a[4] = {R0.x, S0.x, R0.y, S0.y}; mma_ks(4 * c + 0, a); }
      { const uint32_t a[4] = {R0.z, S0.z, R0.w, S0.w}; mma_ks(4 * c + 1, a); }
      { const uint32_t a[4] = {R1.x, S1.x, R1.y, S1.y}; mma_ks(4 * c + 2, a); }
      { const uint32_t a[4] = {R1.z, S1.z, R1.w, S1.w}; mma_ks(4 * c + 3, a); }
    }
  } else if constexpr (KT == PA_Q8_0) {
#pragma unroll
    for (int b = 0; b < 8; ++b) {
      uint32_t y00, y01, y10, y11;
      q8_words(r0, b, t, y00, y01);
      q8_words(r1, b, t, y10, y11);
      const uint32_t d0 = scale2(r0, 34, b), d1 = scale2(r1, 34, b);
      uint32_t e[2][2][2];  // [row][word][pair]
      q8_dequant(y00, d0, e[0][0][0], e[0][0][1]);
      q8_dequant(y01, d0, e[0][1][0], e[0][1][1]);
      q8_dequant(y10, d1, e[1][0][0], e[1][0][1]);
      q8_dequant(y11, d1, e[1][1][0], e[1][1][1]);
      { const uint32_t a[4] = {e[0][0][0], e[1][0][0], e[0][0][1], e[1][0][1]}; mma_ks(2 * b + 0, a); }
      { const uint32_t a[4] = {e[0][1][0], e[1][1][0], e[0][1][1], e[1][1][1]}; mma_ks(2 * b + 1, a); }
    }
  } else {  // Q4_0
#pragma unroll
    for (int b = 0; b < 8; ++b) {
      const uint32_t x0 = q4_word(r0, b, t), x1 = q4_word(r1, b, t);
      const uint32_t d0 = scale2(r0, 18, b), d1 = scale2(r1, 18, b);
      uint32_t l00, h00, l01, h01, l10, h10, l11, h11;
      q4_dequant(x0, d0, l00, h00, l01, h01);
      q4_dequant(x1, d1, l10, h10, l11, h11);
      { const uint32_t a[4] = {l00, l10, l01, l11}; mma_ks(2 * b + 0, a); }
      { const uint32_t a[4] = {h00, h10, h01, h11}; mma_ks(2 * b + 1, a); }
    }
  }
}

// ------------------------------------------------------------------ PV phase (V side)

// o[i][nt] += V^T(dims of warp w, m-tile i; keys of k-step kw) x P^T.
// vrow(k): shared address of tile row k of the V stage.  bp[nt] = B fragment.
template <int VT, int NT>
__device__ __forceinline__ void pv_kstep(float (&o)[4][NT][4], uint32_t vstage, int kw, int w, int lane,
                                         const uint32_t (&bp)[NT][2]) {
  constexpr int S = Fmt<VT>::kStride;
  const int g = lane >> 2, t = lane & 3;
  const uint32_t k0 = vstage + (16 * kw + 2 * t) * S;  // key 2t of this k-step
  const uint32_t rows[4] = {k0, k0 + S, k0 + 8 * S, k0 + 9 * S};
  uint32_t a[4][4];  // [m-tile][reg]
  if constexpr (VT == PA_F16) {
    const uint32_t off = 128 * w + 16 * g;
    uint4 R[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) R[k] = lds128(rows[k] + off);
#pragma unroll
    for (int p = 0; p < 2; ++p) {  // key pair p: keys (2p, 2p+1) of rows[]
      const uint4 A = R[2 * p], B = R[2 * p + 1];
      a[0][2 * p] = prmt(A.x, B.x, 0x5410); a[0][2 * p + 1] = prmt(A.x, B.x, 0x7632);
      a[1][2 * p] = prmt(A.y, B.y, 0x5410); a[1][2 * p + 1] = prmt(A.y, B.y, 0x7632);
      a[2][2 * p] = prmt(A.z, B.z, 0x5410); a[2][2 * p + 1] = prmt(A.z, B.z, 0x7632);
      a[3][2 * p] = prmt(A.w, B.w, 0x5410); a[3][2 * p + 1] = prmt(A.w, B.w, 0x7632);
    }
  } else if constexpr (VT == PA_Q8_0) {
    const int blk = 2 * w + (g >> 2), q = g & 3;
    uint32_t y[4][2], d[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      q8_words(rows[k], blk, q, y[k][0], y[k][1]);
      d[k] = lds16(rows[k] + 34 * blk);
    }
#pragma unroll
    for (int p = 0; p < 2; ++p) {
      const uint32_t dd = d[2 * p] | (d[2 * p + 1] << 16);
#pragma unroll
      for (int wd = 0; wd < 2; ++wd) {
        const uint32_t A = y[2 * p][wd] ^ 0x80808080u, B = y[2 * p + 1][wd] ^ 0x80808080u;
#pragma unroll
        for (int k = 0; k < 4; ++k) {  // quant 4*wd + k -> m-tile (4wd+k)/2, half (k&1)
          const uint32_t sel = k | (k << 4) | ((4 + k) << 8) | ((4 + k) << 12);
          const uint32_t e = and_xor(prmt(A, B, sel), 0x00ff00ffu, 0x64006400u);
          a[(4 * wd + k) >> 1][2 * p + (k & 1)] = hmul2(hadd2(e, kHalf2_1152 ^ 0x80008000u), dd);
        }
      }
    }
  } else {  // Q4_0
    const int blk = 2 * w + (g >> 2), q = g & 3;
    uint32_t x[4], d[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      x[k] = q4_word(rows[k], blk, q);
      d[k] = lds16(rows[k] + 18 * blk);
    }
#pragma unroll
    for (int p = 0; p < 2; ++p) {
      const uint32_t dd = d[2 * p] | (d[2 * p + 1] << 16);
      const uint32_t xa = prmt(x[2 * p], x[2 * p + 1], 0x5410);  // [k0.c0 k0.c1 k1.c0 k1.c1]
      const uint32_t xb = prmt(x[2 * p], x[2 * p + 1], 0x7632);  // [k0.c2 k0.c3 k1.c2 k1.c3]
      uint32_t l0, h0, l1, h1;
      q4_dequant(xa, dd, l0, h0, l1, h1);  // dims j0, j0+16, j0+1, j0+17
      a[0][2 * p] = l0; a[0][2 * p + 1] = h0;
      a[1][2 * p] = l1; a[1][2 * p + 1] = h1;
      q4_dequant(xb, dd, l0, h0, l1, h1);  // dims j0+2, j0+18, j0+3, j0+19
      a[2][2 * p] = l0; a[2][2 * p + 1] = h0;
      a[3][2 * p] = l1; a[3][2 * p + 1] = h1;
    }
  }
  // a[i] = {(dim g, keys 0-1), (dim g+8, keys 0-1), (dim g, keys 8-9), (dim g+8, keys 8-9)} -> reorder
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t A[4] = {a[i][0], a[i][1], a[i][2], a[i][3]};
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) mma_16816(o[i][nt], A, bp[nt][0], bp[nt][1]);
  }
}

// ------------------------------------------------------------------ kernel parameters

struct DecodeParams {
  const float* q;
  const uint8_t* k_pool;
  const uint8_t* v_pool;
  const int32_t* table;
  const int32_t* seq_lens;
  float* out;
  float* lse;
  int32_t* err;
  float2* part_ml;    // [slots][R] (m in log2 units, l)
  float* part_o;      // [slots][R][kD]
  long long total_tiles;
  int n_ctas;
  int n_seq;
  int n_qtok;
  int n_kv_heads;
  int n_q_heads;
  int page_size;
  int table_stride;
  int n_blocks;
  float scale_log2;   // scale * log2(e)
};

// Shared-memory layout (bytes from the dynamic base).
template <int KT, int VT, int NT>
struct Smem {
  static constexpr int kStages = Stages<KT, VT, NT>::kN;
  static constexpr int kKBytes = kTile * Fmt<KT>::kStride;
  static constexpr int kStageBytes = kTile * (Fmt<KT>::kStride + Fmt<VT>::kStride);
  static constexpr int kQ = kStages * kStageBytes;                 // [2][16][NT][32] uint2
  static constexpr int kP = kQ + 2 * 16 * NT * 32 * 8;             // [2][4][NT][32] uint2
  static constexpr int kStat = kP + 2 * kCWarps * NT * 32 * 8;     // [2][4][NT*8] float2
  static constexpr int kBar = kStat + 2 * kCWarps * NT * 8 * 8;    // full[kStages], empty[kStages]
  static constexpr int kMisc = kBar + 2 * kStages * 8;             // abort flag, start segment
  static constexpr int kTotal = kMisc + 32;
};

__device__ __forceinline__ int cta_of_tile(long long x, long long T, int G) {
  return (int)(((x + 1) * (long long)G - 1) / T);
}

// Find the segment holding global tile x: sequence s, KV head g, tile j within it.
__device__ void locate_tile(const DecodeParams& p, long long x, int& s_out, int& g_out, int& j_out) {
  long long base = 0;
  for (int s = 0; s < p.n_seq; ++s) {
    const long long nt = (p.seq_lens[s] + kTile - 1) / kTile;
    const long long span = nt * p.n_kv_heads;
    if (x < base + span) {
      const long long r = x - base;
      s_out = s;
      g_out = (int)(r / nt);
      j_out = (int)(r % nt);
      return;
    }
    base += span;
  }
  s_out = p.n_seq;  // past the end (only for an empty range)
  g_out = 0;
  j_out = 0;
}

// Producer warp: stream the CTA's tiles into the stage ring.
template <int KT, int VT, int NT>
__device__ void produce(const DecodeParams& p, uint8_t* smem, uint32_t bar_full, uint32_t bar_empty,
                        volatile int* abort, long long a, long long b, int s, int g, int j) {
  constexpr int kStages = Stages<KT, VT, NT>::kN;
  constexpr int RK = Fmt<KT>::kRow, RV = Fmt<VT>::kRow;
  constexpr int SK = Fmt<KT>::kStride, SV = Fmt<VT>::kStride;
  constexpr bool kPerRow = (SK != RK) || (SV != RV);
  constexpr int kStageBytes = kTile * (SK + SV);
  const int lane = threadIdx.x & 31;
  const uint32_t stage0 = smem_u32(smem);
  const int ps = p.page_size;
  const uint64_t policy = l2_evict_first_policy();
  int st = 0;
  uint32_t ph = 0;
  long long issued = 0;
  bool stop = false;
  for (long long x = a; x < b && !stop;) {
    const int L = p.seq_lens[s];
    const int nt = (L + kTile - 1) / kTile;
    for (; j < nt && x < b; ++j, ++x) {
      if (*abort) { stop = true; break; }
      const uint32_t fb = bar_full + 8 * st, eb = bar_empty + 8 * st;
      if (lane == 0) mbar_wait(eb, ph ^ 1, p.err, abort);
      __syncwarp();
      const int k0 = j * kTile;
      const int n = min(kTile, L - k0);
      const uint32_t sk = stage0 + st * kStageBytes, sv = sk + kTile * SK;
      const int32_t* trow = p.table + (long long)s * p.table_stride;
      // Pass 1: validate table entries, zero-fill rows with no valid source,
      // and count the bytes the copies will deliver.
      uint32_t bytes = 0;
      bool zeroed = false;
      if (kPerRow) {
        for (int r = lane; r < kTile; r += 32) {
          bool ok = false;
          if (r < n) {
            const int pos = k0 + r;
            const int blk = __ldg(trow + pos / ps);
            ok = blk >= 0 && blk < p.n_blocks;
            if (!ok) record_error(p.err, PA_ERR_BOUNDS);
          }
          if (ok) {
            bytes += RK + RV;
          } else {
            for (int c = 0; c < RK; c += 16) sts128_zero(sk + r * SK + c);
            for (int c = 0; c < RV; c += 16) sts128_zero(sv + r * SV + c);
            zeroed = true;
          }
        }
      } else {
        const int p0 = k0 / ps, p1 = (k0 + n - 1) / ps;
        for (int pg = p0 + lane; pg <= p1; pg += 32) {
          const int rs = max(k0, pg * ps), re = min(k0 + n, (pg + 1) * ps);
          const int blk = __ldg(trow + pg);
          if (blk >= 0 && blk < p.n_blocks) {
            bytes += (re - rs) * (RK + RV);
          } else {
            record_error(p.err, PA_ERR_BOUNDS);
            for (int r = rs - k0; r < re - k0; ++r) {
              for (int c = 0; c < RK; c += 16) sts128_zero(sk + r * SK + c);
              for (int c = 0; c < RV; c += 16) sts128_zero(sv + r * SV + c);
            }
            zeroed = true;
          }
        }
        // Rows past the sequence end: V must be finite (its weight is 0).
        for (int r = n + lane; r < kTile; r += 32) {
          for (int c = 0; c < RK; c += 16) sts128_zero(sk + r * SK + c);
          for (int c = 0; c < RV; c += 16) sts128_zero(sv + r * SV + c);
          zeroed = true;
        }
      }
      if (__any_sync(0xffffffffu, zeroed)) fence_proxy_async_smem();
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) bytes += __shfl_xor_sync(0xffffffffu, bytes, o);
      __syncwarp();
      if (lane == 0) mbar_arrive_expect_tx(fb, bytes);
      __syncwarp();
      // Pass 2: issue the copies.
      if (kPerRow) {
        for (int r = lane; r < n; r += 32) {
          const int pos = k0 + r;
          const int blk = __ldg(trow + pos / ps);
          if (blk >= 0 && blk < p.n_blocks) {
            const long long row = ((long long)blk * p.n_kv_heads + g) * ps + pos % ps;
            bulk_g2s_hint(sk + r * SK, p.k_pool + row * RK, RK, fb, policy);
            bulk_g2s_hint(sv + r * SV, p.v_pool + row * RV, RV, fb, policy);
          }
        }
      } else {
        const int p0 = k0 / ps, p1 = (k0 + n - 1) / ps;
        for (int pg = p0 + lane; pg <= p1; pg += 32) {
          const int rs = max(k0, pg * ps), re = min(k0 + n, (pg + 1) * ps);
          const int blk = __ldg(trow + pg);
          if (blk >= 0 && blk < p.n_blocks) {
            const long long row = ((long long)blk * p.n_kv_heads + g) * ps + (rs - pg * ps);
            bulk_g2s_hint(sk + (rs - k0) * SK, p.k_pool + row * RK, (re - rs) * RK, fb, policy);
            bulk_g2s_hint(sv + (rs - k0) * SV, p.v_pool + row * RV, (re - rs) * RV, fb, policy);
          }
        }
      }
      ++issued;
      if (++st == kStages) { st = 0; ph ^= 1; }
    }
    j = 0;
    if (++g == p.n_kv_heads) { g = 0; ++s; }
  }
  // Drain: make sure no copy is still in flight when the CTA retires.
  if (lane == 0) {
    const int n_last = (int)(issued < kStages ? issued : kStages);
    for (int k = 1; k <= n_last; ++k) {
      int sst = st - k;
      uint32_t sph = ph;
      if (sst < 0) { sst += kStages; sph ^= 1; }
      mbar_wait(bar_full + 8 * sst, sph, p.err, abort, /*honour_abort=*/false);
    }
  }
}

template <int KT, int VT, int NT>
__global__ void __launch_bounds__(kThreads, 2) pa_split_decode_kernel(const __grid_constant__ DecodeParams p) {
  using SM = Smem<KT, VT, NT>;
  constexpr int kStages = SM::kStages;
  constexpr int R8 = NT * 8;
  extern __shared__ __align__(128) uint8_t smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar_full = sbase + SM::kBar, bar_empty = bar_full + 8 * kStages;
  volatile int* abort = reinterpret_cast<volatile int*>(smem + SM::kMisc);
  int* start = reinterpret_cast<int*>(smem + SM::kMisc + 4);

  const long long T = p.total_tiles;
  const int G = p.n_ctas;
  const long long a = (long long)blockIdx.x * T / G, b = (long long)(blockIdx.x + 1) * T / G;

  if (tid == 0) {
    *abort = 0;
    for (int i = 0; i < kStages; ++i) {
      mbar_init(bar_full + 8 * i, 1);
      mbar_init(bar_empty + 8 * i, kCWarps);
    }
    fence_mbar_init();
    int s0, g0, j0;
    locate_tile(p, a, s0, g0, j0);
    start[0] = s0; start[1] = g0; start[2] = j0;
  }
  __syncthreads();
  int s = start[0], g = start[1], j = start[2];

  if (warp == kCWarps) {
    produce<KT, VT, NT>(p, smem, bar_full, bar_empty, abort, a, b, s, g, j);
    return;
  }

  // ------------------------------------------------------------ consumers
  const int gq = lane >> 2, tq = lane & 3;
  const int R = kGqa * p.n_qtok;
  const uint32_t qf_base = sbase + SM::kQ, pb_base = sbase + SM::kP;
  float2* stats = reinterpret_cast<float2*>(smem + SM::kStat);
  int st = 0;
  uint32_t ph = 0;
  int qbuf = 0, tbuf = 0;
  long long x = a;
  while (x < b) {
    const int L = p.seq_lens[s];
    const int ntl = (L + kTile - 1) / kTile;
    const int jb = j, je = (int)((long long)ntl < j + (b - x) ? (long long)ntl : j + (b - x));
    const int seg = s * p.n_kv_heads + g;
    const bool whole = (jb == 0 && je == ntl);

    // Stage Q for (s, g) as B fragments in the K format's dim order.
    {
      const uint32_t qf = qf_base + qbuf * (16 * NT * 32 * 8);
      for (int e = tid; e < 16 * NT * 32; e += kCWarps * 32) {
        const int ln = e & 31, nt = (e >> 5) % NT, ks = e / (32 * NT);
        const int row = nt * 8 + (ln >> 2), t4 = ln & 3;
        uint32_t b0 = 0, b1 = 0;
        if (row < R) {
          const int tqk = row / kGqa, hl = row % kGqa;
          const float* qr = p.q + (((long long)s * p.n_qtok + tqk) * p.n_q_heads + g * kGqa + hl) * kD;
          b0 = pack_half2(__ldg(qr + kdim<KT>(ks, 2 * t4)), __ldg(qr + kdim<KT>(ks, 2 * t4 + 1)));
          b1 = pack_half2(__ldg(qr + kdim<KT>(ks, 2 * t4 + 8)), __ldg(qr + kdim<KT>(ks, 2 * t4 + 9)));
        }
        asm volatile("st.shared.v2.b32 [%0], {%1, %2};" ::"r"(qf + ((ks * NT + nt) * 32 + ln) * 8), "r"(b0),
                     "r"(b1)
                     : "memory");
      }
      named_bar_sync(1, kCWarps * 32);
    }
    const uint32_t qf_lane = qf_base + qbuf * (16 * NT * 32 * 8) + lane * 8;

    float o[4][NT][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int c = 0; c < 4; ++c) o[i][nt][c] = 0.f;
    float m_run[NT], l_run[NT];  // for query row nt*8 + gq
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) { m_run[nt] = -INFINITY; l_run[nt] = 0.f; }

    const int vis0 = L - p.n_qtok;  // last key visible to query token 0
    for (int jt = jb; jt < je; ++jt) {
      const uint32_t fb = bar_full + 8 * st;
      if (!*abort) mbar_wait(fb, ph, p.err, abort);
      const uint32_t sk = sbase + st * SM::kStageBytes;
      const uint32_t sv = sk + SM::kKBytes;
      const int k0 = jt * kTile;

      // ---- S phase: keys 16*warp .. +15 of the tile
      float sacc[NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int c = 0; c < 4; ++c) sacc[nt][c] = 0.f;
      {
        const uint32_t r0 = sk + (16 * warp + gq) * Fmt<KT>::kStride;
        s_phase<KT, NT>(sacc, r0, r0 + 8 * Fmt<KT>::kStride, qf_lane, lane);
      }
      const bool need_mask = (k0 + kTile - 1) > vis0;
      const int key0 = k0 + 16 * warp + gq;
      float2* st_w = stats + (tbuf * kCWarps + warp) * R8;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        float xv[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          xv[c] = sacc[nt][c] * p.scale_log2;
          if (need_mask) {
            const int row = nt * 8 + 2 * tq + (c & 1);
            const int tk = min(row / kGqa, p.n_qtok - 1);
            const int key = key0 + ((c & 2) ? 8 : 0);
            if (key > vis0 + tk) xv[c] = -INFINITY;
          }
        }
        float mx0 = fmaxf(xv[0], xv[2]), mx1 = fmaxf(xv[1], xv[3]);
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
          mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
          mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
        }
        const float b0 = (mx0 == -INFINITY) ? 0.f : mx0, b1 = (mx1 == -INFINITY) ? 0.f : mx1;
        const float p0 = exp2f(xv[0] - b0), p1 = exp2f(xv[1] - b1);
        const float p2 = exp2f(xv[2] - b0), p3 = exp2f(xv[3] - b1);
        const uint32_t X0 = pack_half2(p0, p1), X1 = pack_half2(p2, p3);
        // Row sums of the fp16-rounded weights (what the PV product uses).
        const float2 f0 = __half22float2(*reinterpret_cast<const __half2*>(&X0));
        const float2 f1 = __half22float2(*reinterpret_cast<const __half2*>(&X1));
        float sm0 = f0.x + f1.x, sm1 = f0.y + f1.y;
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
          sm0 += __shfl_xor_sync(0xffffffffu, sm0, off);
          sm1 += __shfl_xor_sync(0xffffffffu, sm1, off);
        }
        if (gq == 0) {
          st_w[nt * 8 + 2 * tq] = make_float2(mx0, sm0);
          st_w[nt * 8 + 2 * tq + 1] = make_float2(mx1, sm1);
        }
        const uint32_t B0 = movmatrix_trans(X0), B1 = movmatrix_trans(X1);
        asm volatile("st.shared.v2.b32 [%0], {%1, %2};" ::"r"(
                         pb_base + (((tbuf * kCWarps + warp) * NT + nt) * 32 + lane) * 8),
                     "r"(B0), "r"(B1)
                     : "memory");
      }
      named_bar_sync(1, kCWarps * 32);

      // ---- PV phase: dims 64*warp .. +63 over all 64 keys
      const float2* st_t = stats + tbuf * kCWarps * R8;
      float fsc[kCWarps][NT];
      float alpha_c[NT][2];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const int row = nt * 8 + gq;
        float mt[kCWarps], mnew = m_run[nt];
#pragma unroll
        for (int w2 = 0; w2 < kCWarps; ++w2) {
          mt[w2] = st_t[w2 * R8 + row].x;
          mnew = fmaxf(mnew, mt[w2]);
        }
        const float base = (mnew == -INFINITY) ? 0.f : mnew;
        const float alpha = exp2f(m_run[nt] - base);
        float lsum = l_run[nt] * alpha;
#pragma unroll
        for (int w2 = 0; w2 < kCWarps; ++w2) {
          fsc[w2][nt] = exp2f(mt[w2] - base);
          lsum += st_t[w2 * R8 + row].y * fsc[w2][nt];
        }
        l_run[nt] = lsum;
        m_run[nt] = mnew;
        alpha_c[nt][0] = __shfl_sync(0xffffffffu, alpha, 8 * tq);       // row 2*tq lives at g = 2*tq
        alpha_c[nt][1] = __shfl_sync(0xffffffffu, alpha, 8 * tq + 4);   // row 2*tq+1
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int c = 0; c < 4; ++c) o[i][nt][c] *= alpha_c[nt][c & 1];
#pragma unroll
      for (int kw = 0; kw < kCWarps; ++kw) {
        uint32_t bp[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const uint2 v = lds64(pb_base + (((tbuf * kCWarps + kw) * NT + nt) * 32 + lane) * 8);
          const uint32_t f2 = pack_half2(fsc[kw][nt], fsc[kw][nt]);
          bp[nt][0] = hmul2(v.x, f2);
          bp[nt][1] = hmul2(v.y, f2);
        }
        pv_kstep<VT, NT>(o, sv, kw, warp, lane, bp);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_empty + 8 * st);
      if (++st == kStages) { st = 0; ph ^= 1; }
      tbuf ^= 1;
    }

    // ---- end of piece: final output or a split partial
    const int slot = (int)blockIdx.x + seg;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const float lc0 = __shfl_sync(0xffffffffu, l_run[nt], 8 * tq);
      const float lc1 = __shfl_sync(0xffffffffu, l_run[nt], 8 * tq + 4);
      const float mc0 = __shfl_sync(0xffffffffu, m_run[nt], 8 * tq);
      const float mc1 = __shfl_sync(0xffffffffu, m_run[nt], 8 * tq + 4);
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int row = nt * 8 + 2 * tq + c;
        if (row >= R) continue;
        const float lr = c ? lc1 : lc0;
        const int tk = row / kGqa, hl = row % kGqa;
        float* dst;
        float inv;
        if (whole) {
          dst = p.out + (((long long)s * p.n_qtok + tk) * p.n_q_heads + g * kGqa + hl) * kD;
          inv = lr > 0.f ? 1.f / lr : 0.f;
        } else {
          dst = p.part_o + ((long long)slot * R + row) * kD;
          inv = 1.f;
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          dst[vdim<VT>(warp, gq, i, 0)] = o[i][nt][c] * inv;
          dst[vdim<VT>(warp, gq, i, 1)] = o[i][nt][2 + c] * inv;
        }
        if (warp == 0 && gq == 0) {
          const float mr = c ? mc1 : mc0;
          if (whole) {
            if (p.lse) {
              p.lse[((long long)s * p.n_qtok + tk) * p.n_q_heads + g * kGqa + hl] =
                  lr > 0.f ? (mr + log2f(lr)) * kLn2 : -INFINITY;
            }
          } else {
            p.part_ml[(long long)slot * R + row] = make_float2(mr, lr);
          }
        }
      }
    }

    x += je - jb;
    qbuf ^= 1;
    j = 0;
    if (++g == p.n_kv_heads) { g = 0; ++s; }
  }
}

// Merge the split partials of every multi-piece segment by log-sum-exp.
// One CTA per segment, one thread per head dim.
__global__ void __launch_bounds__(kD) pa_merge_kernel(const __grid_constant__ DecodeParams p) {
  const int seg = blockIdx.x;
  const int s = seg / p.n_kv_heads, g = seg % p.n_kv_heads;
  const int L = p.seq_lens[s];
  const int ntl = (L + kTile - 1) / kTile;
  // The segment's tile range decides whether it was split, and over which CTAs.
  __shared__ long long seg_start;
  if (threadIdx.x == 0) {
    long long base = 0;
    for (int i = 0; i < s; ++i) base += (long long)((p.seq_lens[i] + kTile - 1) / kTile) * p.n_kv_heads;
    seg_start = base + (long long)g * ntl;
  }
  __syncthreads();
  const int c0 = cta_of_tile(seg_start, p.total_tiles, p.n_ctas);
  const int c1 = cta_of_tile(seg_start + ntl - 1, p.total_tiles, p.n_ctas);
  if (c0 == c1) return;  // written directly by its only CTA
  const int R = kGqa * p.n_qtok;
  const int d = threadIdx.x;
  for (int row = 0; row < R; ++row) {
    float M = -INFINITY;
    for (int c = c0; c <= c1; ++c) {
      const float2 ml = p.part_ml[(long long)(c + seg) * R + row];
      if (ml.y > 0.f) M = fmaxf(M, ml.x);
    }
    float W = 0.f, acc = 0.f;
    if (M != -INFINITY) {
      for (int c = c0; c <= c1; ++c) {
        const float2 ml = p.part_ml[(long long)(c + seg) * R + row];
        if (!(ml.y > 0.f)) continue;
        const float wgt = exp2f(ml.x - M);
        W += wgt * ml.y;
        acc += wgt * p.part_o[((long long)(c + seg) * R + row) * kD + d];
      }
    }
    const int tk = row / kGqa, hl = row % kGqa;
    const long long orow = ((long long)s * p.n_qtok + tk) * p.n_q_heads + g * kGqa + hl;
    p.out[orow * kD + d] = W > 0.f ? acc / W : 0.f;
    if (d == 0 && p.lse) p.lse[orow] = W > 0.f ? (M + log2f(W)) * kLn2 : -INFINITY;
  }
}

// ------------------------------------------------------------------ host side

using KernelFn = void (*)(DecodeParams);

struct KernelInfo {
  KernelFn fn;
  int smem;
};

template <int KT, int VT, int NT>
KernelInfo kernel_info() {
  return KernelInfo{pa_split_decode_kernel<KT, VT, NT>, Smem<KT, VT, NT>::kTotal};
}

int type_slot(int t) { return t == PA_F16 ? 0 : t == PA_Q4_0 ? 1 : t == PA_Q8_0 ? 2 : -1; }

bool lookup_kernel(int kt, int vt, int nt, KernelInfo* out) {
  const int ks = type_slot(kt), vs = type_slot(vt);
  if (ks < 0 || vs < 0 || nt < 1 || nt > 3) return false;
#define PA_K(KT, VT)                                                                              \
  if (kt == KT && vt == VT) {                                                                     \
    *out = nt == 1 ? kernel_info<KT, VT, 1>() : nt == 2 ? kernel_info<KT, VT, 2>() : kernel_info<KT, VT, 3>(); \
    return true;                                                                                  \
  }
  PA_K(PA_F16, PA_F16)
  PA_K(PA_Q4_0, PA_Q4_0)
  PA_K(PA_Q8_0, PA_Q8_0)
#undef PA_K
  return false;
}

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int g_sms[kMaxDevices];
int g_occ[kMaxDevices][3][3][3];  // [device][k][v][nt-1] CTAs per SM, 0 = not queried

pa_status device_caps(int device, int kt, int vt, int nt, const KernelInfo& ki, int* sms, int* occ) {
  if (device < 0 || device >= kMaxDevices) return PA_ERR_INVALID;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_sms[device] == 0) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) return PA_ERR_CUDA;
    g_sms[device] = v;
  }
  int& o = g_occ[device][type_slot(kt)][type_slot(vt)][nt - 1];
  if (o == 0) {
    int cur = 0;
    cudaGetDevice(&cur);
    if (cur != device) cudaSetDevice(device);
    cudaError_t e = cudaFuncSetAttribute(ki.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, ki.smem);
    int n = 0;
    if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, ki.fn, kThreads, ki.smem);
    if (cur != device) cudaSetDevice(cur);
    if (e != cudaSuccess || n <= 0) return PA_ERR_CUDA;
    o = n;
  }
  *sms = g_sms[device];
  *occ = o;
  return PA_OK;
}

pa_status check_shape(const pa_pool* pool, uint32_t n_qtok, uint32_t n_q_heads, pa_pool_desc* d) {
  if (!pool) return PA_ERR_INVALID;
  pa_pool_get_desc(pool, d);
  if (d->head_dim != kD) return PA_ERR_UNSUPPORTED;
  if (n_q_heads == 0 || n_q_heads != d->n_kv_heads * kGqa) return PA_ERR_UNSUPPORTED;
  if (n_qtok < 1 || n_qtok > 4) return PA_ERR_UNSUPPORTED;
  KernelInfo ki;
  if (!lookup_kernel(d->k_type, d->v_type, (kGqa * n_qtok + 7) / 8, &ki)) return PA_ERR_UNSUPPORTED;
  return PA_OK;
}

struct Plan {
  long long tiles;
  int ctas;
  int R;
  long long slots;
};

size_t workspace_bytes(long long max_ctas, long long n_seg, int R) {
  const long long slots = max_ctas + n_seg;
  size_t b = 0;
  b += ((size_t)slots * R * sizeof(float2) + 255) & ~size_t(255);
  b += (size_t)slots * R * kD * sizeof(float);
  return b;
}

}  // namespace

extern "C" size_t pa_decode_workspace_size(const pa_pool* pool, uint32_t n_seq, uint32_t n_qtok, int device) {
  pa_pool_desc d;
  if (pa_pool_get_desc(pool, &d) != PA_OK) return 0;
  if (d.head_dim != kD || n_qtok < 1 || n_qtok > 4) return 0;
  const int nt = (kGqa * (int)n_qtok + 7) / 8;
  KernelInfo ki;
  if (!lookup_kernel(d.k_type, d.v_type, nt, &ki)) return 0;
  int sms = 0, occ = 0;
  if (device_caps(device, d.k_type, d.v_type, nt, ki, &sms, &occ) != PA_OK) return 0;
  return workspace_bytes((long long)sms * occ, (long long)n_seq * d.n_kv_heads, kGqa * (int)n_qtok);
}

static pa_status make_plan(const pa_pool_desc& d, const int32_t* seq_lens_host, uint32_t n_seq, uint32_t n_qtok,
                           uint32_t table_stride, int device, KernelInfo* ki, Plan* plan) {
  const int nt = (kGqa * (int)n_qtok + 7) / 8;
  if (!lookup_kernel(d.k_type, d.v_type, nt, ki)) return PA_ERR_UNSUPPORTED;
  long long tiles = 0;
  for (uint32_t s = 0; s < n_seq; ++s) {
    const long long L = seq_lens_host[s];
    if (L < (long long)n_qtok) return PA_ERR_INVALID;
    if (table_stride && L > (long long)table_stride * d.page_size) return PA_ERR_INVALID;
    tiles += (L + kTile - 1) / kTile;
  }
  tiles *= d.n_kv_heads;
  int sms = 0, occ = 0;
  pa_status st = device_caps(device, d.k_type, d.v_type, nt, *ki, &sms, &occ);
  if (st != PA_OK) return st;
  plan->tiles = tiles;
  plan->ctas = (int)std::min<long long>(tiles, (long long)sms * occ);
  plan->R = kGqa * (int)n_qtok;
  plan->slots = (long long)plan->ctas + (long long)n_seq * d.n_kv_heads;
  return PA_OK;
}

extern "C" pa_status pa_decode_plan(const pa_pool* pool, const int32_t* seq_lens_host, uint32_t n_seq,
                                    uint32_t n_qtok, int device, uint32_t* n_ctas, uint32_t* n_tiles,
                                    uint32_t* tile_keys, uint32_t* n_partials) {
  pa_pool_desc d;
  if (!pool || (n_seq && !seq_lens_host)) return PA_ERR_INVALID;
  pa_pool_get_desc(pool, &d);
  if (d.head_dim != kD || n_qtok < 1 || n_qtok > 4) return PA_ERR_UNSUPPORTED;
  if (n_seq == 0) return PA_ERR_INVALID;
  KernelInfo ki;
  Plan plan{};
  const pa_status st = make_plan(d, seq_lens_host, n_seq, n_qtok, 0, device, &ki, &plan);
  if (st != PA_OK) return st;
  if (n_ctas) *n_ctas = (uint32_t)plan.ctas;
  if (n_tiles) *n_tiles = (uint32_t)plan.tiles;
  if (tile_keys) *tile_keys = kTile;
  if (n_partials) {
    // Pieces = CTA-range cuts plus segment cuts.
    uint32_t pieces = 0;
    long long base = 0;
    for (uint32_t s = 0; s < n_seq; ++s) {
      const long long ntl = (seq_lens_host[s] + kTile - 1) / kTile;
      for (uint32_t g = 0; g < d.n_kv_heads; ++g) {
        const long long a = base + g * ntl, e = a + ntl - 1;
        const int c0 = (int)(((a + 1) * plan.ctas - 1) / plan.tiles);
        const int c1 = (int)(((e + 1) * plan.ctas - 1) / plan.tiles);
        pieces += (uint32_t)(c1 - c0 + 1);
      }
      base += ntl * d.n_kv_heads;
    }
    *n_partials = pieces;
  }
  return PA_OK;
}

extern "C" pa_status pa_decode(const pa_pool* pool, const float* q, const void* k_pool, const void* v_pool,
                               const int32_t* block_table, uint32_t table_stride, const int32_t* seq_lens_dev,
                               const int32_t* seq_lens_host, uint32_t n_seq, uint32_t n_qtok, uint32_t n_q_heads,
                               float scale, float* out, float* lse, void* workspace, size_t ws_bytes, int32_t* err,
                               pa_stream_t stream) {
  pa_pool_desc d;
  pa_status st = check_shape(pool, n_qtok, n_q_heads, &d);
  if (st != PA_OK) return st;
  if (n_seq == 0) return PA_OK;
  if (!q || !k_pool || !v_pool || !block_table || !seq_lens_dev || !seq_lens_host || !out || !workspace || !err ||
      table_stride == 0)
    return PA_ERR_INVALID;
  if (((uintptr_t)q | (uintptr_t)out | (uintptr_t)k_pool | (uintptr_t)v_pool) & 15) return PA_ERR_INVALID;
  if ((uintptr_t)workspace & 255) return PA_ERR_INVALID;
  if (!(scale > 0.f) || !std::isfinite(scale)) return PA_ERR_INVALID;
  for (uint32_t i = 0; i < n_seq; ++i) {
    const long long L = seq_lens_host[i];
    if (L < (long long)n_qtok || L > (long long)table_stride * d.page_size) return PA_ERR_INVALID;
  }
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return PA_ERR_CUDA;
  KernelInfo ki;
  Plan plan{};
  st = make_plan(d, seq_lens_host, n_seq, n_qtok, table_stride, device, &ki, &plan);
  if (st != PA_OK) return st;
  int sms = 0, occ = 0;
  device_caps(device, d.k_type, d.v_type, (kGqa * (int)n_qtok + 7) / 8, ki, &sms, &occ);
  const long long n_seg = (long long)n_seq * d.n_kv_heads;
  if (ws_bytes < workspace_bytes((long long)sms * occ, n_seg, plan.R)) return PA_ERR_INVALID;

  DecodeParams p{};
  p.q = q;
  p.k_pool = static_cast<const uint8_t*>(k_pool);
  p.v_pool = static_cast<const uint8_t*>(v_pool);
  p.table = block_table;
  p.seq_lens = seq_lens_dev;
  p.out = out;
  p.lse = lse;
  p.err = err;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  p.part_ml = reinterpret_cast<float2*>(ws);
  ws += ((size_t)plan.slots * plan.R * sizeof(float2) + 255) & ~size_t(255);
  p.part_o = reinterpret_cast<float*>(ws);
  p.total_tiles = plan.tiles;
  p.n_ctas = plan.ctas;
  p.n_seq = (int)n_seq;
  p.n_qtok = (int)n_qtok;
  p.n_kv_heads = (int)d.n_kv_heads;
  p.n_q_heads = (int)n_q_heads;
  p.page_size = (int)d.page_size;
  p.table_stride = (int)table_stride;
  p.n_blocks = (int)d.n_blocks;
  p.scale_log2 = scale * kLog2e;

  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  ki.fn<<<plan.ctas, kThreads, ki.smem, cs>>>(p);
  if (cudaGetLastError() != cudaSuccess) return PA_ERR_CUDA;
  pa_merge_kernel<<<(unsigned)n_seg, kD, 0, cs>>>(p);
  if (cudaGetLastError() != cudaSuccess) return PA_ERR_CUDA;
  return PA_OK;
}
