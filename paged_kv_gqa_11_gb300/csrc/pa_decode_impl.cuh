// Device side of the split-K paged GQA decode (sm_103a).
//
// What is computed (llama.cpp fork PR #2, split-K decode commit: "Split-K
// flash decoding for head size 256, GQA 6 and 1-4 query tokens (MTP verify
// widths) with ... packed in-register dequantization"; lucebox PR #555,
// Summary: "GQA-aware thread blocks, occupancy-aware context parallelism,
// adaptive long-context partitioning, and a stable split-softmax merge"): for
// every (sequence, KV head) the 6 * n_qtok query rows of that KV head attend to
// the sequence's rows, read page by page through the block table; K/V are
// dequantised in registers, S = QK^T and O = PV run on the tensor cores
// (mma.sync m16n8k16, fp16 operands, fp32 accumulation), the softmax is
// online, and the splits are merged by log-sum-exp.
//
// Work split.  The batch is cut into segments (below), each a run of tiles.
// All tiles are laid end to end and cut into equal contiguous ranges, one per
// CTA, with as many CTAs as fit on the SMs at once.  A CTA's range may cover
// the tail of one segment and the head of the next; each piece becomes one
// split partial.  The cut depends only on the sequence lengths, so a paged and
// an identity-table cache give the same splits, the same summation order and
// bit-identical results (TensorFold #1156, Design/Kernels: "only the address
// changes; the per-key summation order does not").
//
// Data movement.  One producer warp streams K and V tiles into a ring of
// shared-memory stages with cp.async.bulk, completing on mbarriers.  The table
// is read one tile ahead, once per page (TensorFold #1156: "test once per
// block").  A table entry outside the pool is never dereferenced: its rows are
// zero-filled and PA_ERR_BOUNDS is recorded.
//
// One query token ("head-group" tiles).  A segment is (sequence, group of up
// to four KV heads); a tile is 16 keys of every head of the group, which for
// 16-row pages is one whole pool block (all heads), copied in one transfer per
// K and V.  Consumer warp w owns KV head w of the group end to end: it stages
// its six query rows, computes S^T = K Q^T (M = keys, N = query rows,
// K = dims), the softmax, and O^T += V^T P^T over all 256 dims (M = dims,
// N = rows, K = keys).  Warps never wait for each other.  The running max is
// raised only when a logit exceeds it by more than 2^8 (P <= 256 stays exact
// enough in fp16), so most tiles rescale nothing.
//
// Two to four query tokens ("per-head" tiles, 12-24 rows).  Holding O for all
// dims per warp would take 64 registers per 8 rows, so the warps split the
// tile instead: a segment is (sequence, KV head), a tile 64 keys of that head;
// in the S phase warp w computes keys 16w..16w+15, publishes its tile max, row
// sums and P (transposed with movmatrix) in shared memory, and after a named
// barrier computes O^T for dims 64w..64w+63 over all 64 keys.
//
// Dequantisation.  K goes into the MMA as raw magic-biased halves: a Q4_0
// nibble n becomes 1024+n (low) or 1024+16n (high nibble, against Q/16), a
// Q8_0 byte x becomes 1152+x.  Each 32-dim block gets its own accumulator;
// the bias (sum of the block's Q times 1032/1152, computed with the staged Q)
// is subtracted and the block scale d applied in fp32.  V for one query token
// is converted to the exact integers n-8 / x in fp16 and the block scale is
// folded into P (each MMA's 16 dims lie in one block).  The head dims are
// visited in whatever order makes each thread's loads contiguous; Q and the
// output use the same order, so the dot products are unchanged.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "pa.h"
#include "pa_device.cuh"

namespace pa_split {

using namespace pa_dev;

constexpr int kD = 256;       // head dim
constexpr int kGqa = 6;       // query heads per KV head
constexpr int kTile = 64;     // keys per per-head tile (two or more query tokens)
constexpr int kTileHG = 16;   // keys per head-group tile (one query token)
constexpr int kCWarps = 4;    // consumer warps = heads per head group (at most)
constexpr int kThreads = (kCWarps + 1) * 32;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kLazy = 8.0f;  // log2 headroom before the running max is raised

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

// Shared memory outside the stage ring.
constexpr int extras_bytes(int NT) {
  return (NT == 1 ? kCWarps * (16 * 32 * 8 + 8 * 8 * 4)  // per-warp Q fragments + block corrections
                  : (2 * 16 * NT * 32 * 8                  // Q fragments, double buffered
                     + 2 * 8 * NT * 8 * 4                  // block corrections
                     + 2 * kCWarps * NT * 32 * 8           // P fragments
                     + 2 * kCWarps * NT * 8 * 8))          // tile stats
         + 2 * 8 * 8 + 32;  // barriers (up to 8 stages), misc
}

// Keys and heads one stage holds: 16 keys x 4 heads (one token) or 64 keys x
// 1 head (more tokens).  Same bytes either way.
template <int NT>
struct TileShape {
  static constexpr int kKeys = NT == 1 ? kTileHG : kTile;
  static constexpr int kHeads = NT == 1 ? kCWarps : 1;
  static constexpr int kRows = kKeys * kHeads;  // stored rows per stage for K (and for V)
};

// CTAs per SM a configuration aims for: three for one-token Q4_0 (small
// stages, modest registers), otherwise two, or one when a stage is large.
template <int KT, int VT, int NT>
struct CtaTarget {
  static constexpr int kStageBytes = TileShape<NT>::kRows * (Fmt<KT>::kStride + Fmt<VT>::kStride);
  static constexpr int kN = (kStageBytes <= 20000 && NT == 1) ? 3 : (kStageBytes <= 40000 ? 2 : 1);
};

template <int KT, int VT, int NT>
struct Stages {
  static constexpr int kStageBytes = TileShape<NT>::kRows * (Fmt<KT>::kStride + Fmt<VT>::kStride);
  static constexpr int kCtas = CtaTarget<KT, VT, NT>::kN;
  static constexpr int kBudget = (233472 - kCtas * 1024) / kCtas;  // 228 KB per SM, 1 KB reserved per CTA
  static constexpr int kPerCtaMax = kBudget < 232448 ? kBudget : 232448;
  static constexpr int kFit = (kPerCtaMax - extras_bytes(NT)) / kStageBytes;
  static constexpr int kN = kFit > 8 ? 8 : kFit;
  static_assert(kN >= 2, "stage ring does not fit");
};

// Head dim that S-MMA k-step s, k-index j (= 2t + 8h + e) stands for.
template <int KT>
__device__ __forceinline__ int kdim(int s, int j) {
  const int t = (j & 7) >> 1, e = j & 1, h = j >> 3;
  if (KT == PA_F16) {  // s = 4c + u: thread t loads dims 64c + 16t .. +15
    const int c = s >> 2, u = s & 3;
    return 64 * c + 16 * t + 4 * u + 2 * h + e;
  } else if (KT == PA_Q8_0) {  // s = 2b + u: thread t owns quants 8t..8t+7 of block b
    const int b = s >> 1, u = s & 1;
    return 32 * b + 8 * t + 4 * u + h + 2 * e;
  } else {  // Q4_0, s = 2b + u: thread t owns quant bytes 4t..4t+3 of block b (u = 1: high nibbles)
    const int b = s >> 1, u = s & 1;
    return 32 * b + 4 * t + 16 * u + h + 2 * e;
  }
}

// Head dim of O^T row g + 8h of m-tile i (0..15), one-token path.
template <int VT>
__device__ __forceinline__ int vdim_solo(int g, int i, int h) {
  if (VT == PA_F16) return 64 * (i >> 2) + 8 * g + 2 * (i & 3) + h;
  if (VT == PA_Q8_0) return 32 * (i >> 1) + 4 * g + 2 * (i & 1) + h;
  return 32 * (i >> 1) + 2 * g + (i & 1) + 16 * h;  // Q4_0
}

// Head dim of O^T row g + 8h of m-tile i (0..3) for warp w, multi-token path.
template <int VT>
__device__ __forceinline__ int vdim_shared(int w, int g, int i, int h) {
  const int k = 2 * i + h;  // index into the thread's 8 dims
  if (VT == PA_F16) return 64 * w + 8 * g + k;
  const int blk = 2 * w + (g >> 2);
  if (VT == PA_Q8_0) return 32 * blk + 8 * (g & 3) + k;
  return 32 * blk + 4 * (g & 3) + (k >> 1) + 16 * (k & 1);  // Q4_0
}

// ------------------------------------------------------------------ dequant helpers

constexpr uint32_t kHalf2_m1032 = 0xe408e408u;  // -1032.0
constexpr uint32_t kHalf2_m1152 = 0xe480e480u;  // -1152.0
constexpr uint32_t kHalf2_1_16 = 0x2c002c00u;   // 0.0625
constexpr uint32_t kHalf2_m72 = 0xd480d480u;    // -72.0

__device__ __forceinline__ float half_bits_to_float(uint32_t h) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(h)));
}

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

// Q4_0 nibbles of x = [c0 c1 c2 c3] -> exact (n - 8) as fp16 pairs:
//   lo0 = (c0.lo, c2.lo)  hi0 = (c0.hi, c2.hi)  lo1 = (c1.lo, c3.lo)  hi1 = (c1.hi, c3.hi)
__device__ __forceinline__ void q4_exact(uint32_t x, uint32_t& lo0, uint32_t& hi0, uint32_t& lo1, uint32_t& hi1) {
  const uint32_t x8 = x >> 8;
  lo0 = hadd2(and_or(x, 0x000f000fu, 0x64006400u), kHalf2_m1032);
  hi0 = hfma2(and_or(x, 0x00f000f0u, 0x64006400u), kHalf2_1_16, kHalf2_m72);
  lo1 = hadd2(and_or(x8, 0x000f000fu, 0x64006400u), kHalf2_m1032);
  hi1 = hfma2(and_or(x8, 0x00f000f0u, 0x64006400u), kHalf2_1_16, kHalf2_m72);
}

// Same, times the per-half scales dd (fp16 pair).
__device__ __forceinline__ void q4_dequant(uint32_t x, uint32_t dd, uint32_t& lo0, uint32_t& hi0, uint32_t& lo1,
                                           uint32_t& hi1) {
  q4_exact(x, lo0, hi0, lo1, hi1);
  lo0 = hmul2(lo0, dd);
  hi0 = hmul2(hi0, dd);
  lo1 = hmul2(lo1, dd);
  hi1 = hmul2(hi1, dd);
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
  float2* part_ml;  // [slots][rows_per_seg] (m in log2 units, l)
  float* part_o;    // [slots][rows_per_seg][kD]
  float2* mid_ml;   // [slots][rows_per_seg] merge level-1 results, indexed by a chunk's first slot
  float* mid_o;     // [slots][rows_per_seg][kD]
  int* merge_count; // [n_seg][rows_per_seg] level-1 arrivals; zeroed by the split kernel
  int n_counters;   // n_seg * rows_per_seg
  long long total_tiles;
  int n_ctas;
  int n_seq;
  int n_qtok;
  int n_kv_heads;
  int n_q_heads;
  int page_size;
  int table_stride;
  int n_blocks;
  int tile_keys;     // keys per tile: 16 (head groups) or 64 (single heads)
  int seg_heads;     // KV heads per segment: the head-group size, or 1
  int segs_per_seq;  // n_kv_heads / seg_heads
  int rows_per_seg;  // query rows per segment: 6 * seg_heads * n_qtok
  float scale_log2;  // scale * log2(e)
};

// Shared-memory layout (byte offsets from the dynamic base).
template <int KT, int VT, int NT>
struct Smem {
  static constexpr int kStages = Stages<KT, VT, NT>::kN;
  static constexpr int kKBytes = TileShape<NT>::kRows * Fmt<KT>::kStride;
  static constexpr int kStageBytes = TileShape<NT>::kRows * (Fmt<KT>::kStride + Fmt<VT>::kStride);
  static constexpr int kRing = kStages * kStageBytes;
  // head-group path: per-warp Q fragments [4][16][32] uint2, corrections [4][8][8] float
  static constexpr int kWQ = kRing;
  static constexpr int kWQBytes = 16 * 32 * 8;
  static constexpr int kWCb = kWQ + kCWarps * kWQBytes;
  static constexpr int kWCbBytes = 8 * 8 * 4;
  // per-head path: Q fragments [2][16][NT][32] uint2, corrections [2][8][NT*8],
  // P fragments [2][4][NT][32] uint2, stats [2][4][NT*8] float2
  static constexpr int kQBuf = 16 * NT * 32 * 8;
  static constexpr int kQ = kRing;
  static constexpr int kCbBuf = 8 * NT * 8 * 4;
  static constexpr int kCb = kQ + 2 * kQBuf;
  static constexpr int kP = kCb + 2 * kCbBuf;
  static constexpr int kStat = kP + 2 * kCWarps * NT * 32 * 8;
  static constexpr int kWorkEnd = NT == 1 ? kWCb + kCWarps * kWCbBytes : kStat + 2 * kCWarps * NT * 8 * 8;
  static constexpr int kBar = kWorkEnd;                 // full[kStages], empty[kStages]
  static constexpr int kMisc = kBar + 2 * kStages * 8;  // abort flag, start position
  static constexpr int kTotal = kMisc + 32;
};

__device__ __forceinline__ int cta_of_tile(long long x, long long T, int G) {
  return (int)(((x + 1) * (long long)G - 1) / T);
}

__device__ __forceinline__ int tiles_of(const DecodeParams& p, int L) { return (L + p.tile_keys - 1) / p.tile_keys; }

// Find the segment holding global tile x: sequence s, segment-in-sequence g
// (KV head, or head group), tile j within it.
__device__ __forceinline__ void locate_tile(const DecodeParams& p, long long x, int& s_out, int& g_out, int& j_out) {
  long long base = 0;
  for (int s = 0; s < p.n_seq; ++s) {
    const long long nt = tiles_of(p, p.seq_lens[s]);
    const long long span = nt * p.segs_per_seq;
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

// Position of one tile in the CTA's walk: sequence s (length L, nt tiles),
// segment g of that sequence, tile j of the segment.
struct TilePos {
  int s, g, j, L, nt;
};

__device__ __forceinline__ void next_tile(const DecodeParams& p, TilePos& t) {
  if (++t.j < t.nt) return;
  t.j = 0;
  if (++t.g < p.segs_per_seq) return;
  t.g = 0;
  if (++t.s < p.n_seq) {
    t.L = p.seq_lens[t.s];
    t.nt = tiles_of(p, t.L);
  }
}

// Table entries one lane needs for a per-head tile: per-row copies use rows
// lane and lane+32, per-page copies pages p0+lane and p0+lane+32 (a 64-row
// tile spans at most 64 pages).  -1 where the lane has nothing.
template <bool kPerRow>
__device__ __forceinline__ void load_tile_table(const DecodeParams& p, const TilePos& t, int lane, int (&tb)[2]) {
  const int32_t* trow = p.table + (long long)t.s * p.table_stride;
  const int k0 = t.j * kTile, n = min(kTile, t.L - k0), ps = p.page_size;
  const int p0 = k0 / ps, p1 = (k0 + n - 1) / ps;
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    tb[u] = -1;
    if (kPerRow) {
      const int r = lane + 32 * u;
      if (r < n) tb[u] = __ldg(trow + (k0 + r) / ps);
    } else {
      const int pg = p0 + lane + 32 * u;
      if (pg <= p1) tb[u] = __ldg(trow + pg);
    }
  }
}

// Table entry for a head-group tile (16 keys, so at most 16 pages): lane l
// holds page p0 + l.
__device__ __forceinline__ int load_hg_table(const DecodeParams& p, const TilePos& t, int lane) {
  const int32_t* trow = p.table + (long long)t.s * p.table_stride;
  const int k0 = t.j * kTileHG, n = min(kTileHG, t.L - k0), ps = p.page_size;
  const int p0 = k0 / ps, p1 = (k0 + n - 1) / ps;
  return (p0 + lane <= p1) ? __ldg(trow + p0 + lane) : -1;
}

// Producer for head-group tiles: stage = K [4 heads][16 rows][SK] then V.
// A full 16-row page whose group covers every KV head is one contiguous pool
// block per K and V: one copy each.  Otherwise one copy per (page, head) run,
// or per row for the padded F16 layout.
template <int KT, int VT, int NT>
__device__ void produce_hg(const DecodeParams& p, uint8_t* smem, uint32_t bar_full, uint32_t bar_empty,
                           volatile int* abort, long long a, long long b, TilePos pos) {
  constexpr int kStages = Stages<KT, VT, NT>::kN;
  constexpr int RK = Fmt<KT>::kRow, RV = Fmt<VT>::kRow;
  constexpr int SK = Fmt<KT>::kStride, SV = Fmt<VT>::kStride;
  constexpr bool kPerRow = (SK != RK) || (SV != RV);
  constexpr int kStageBytes = TileShape<NT>::kRows * (SK + SV);
  constexpr int kHeadK = kTileHG * SK, kHeadV = kTileHG * SV;  // one head's rows in a stage
  const int lane = threadIdx.x & 31;
  const uint32_t stage0 = smem_u32(smem);
  const int ps = p.page_size, H = p.n_kv_heads, GH = p.seg_heads;
  const bool whole_blocks = (ps == kTileHG) && (GH == H);
  const uint64_t policy = l2_evict_first_policy();
  int st = 0;
  uint32_t ph = 0;
  long long issued = 0;
  int tb = load_hg_table(p, pos, lane), tbn = -1;
  for (long long x = a; x < b; ++x) {
    if (*abort) break;
    TilePos nxt = pos;
    if (x + 1 < b) {
      next_tile(p, nxt);
      tbn = load_hg_table(p, nxt, lane);
    }
    const uint32_t fb = bar_full + 8 * st, eb = bar_empty + 8 * st;
    const int k0 = pos.j * kTileHG;
    const int n = min(kTileHG, pos.L - k0);
    const int p0 = k0 / ps, p1 = (k0 + n - 1) / ps;
    const bool used = p0 + lane <= p1;
    const bool ok = !used || (tb >= 0 && tb < p.n_blocks);
    const bool all_ok = __all_sync(0xffffffffu, ok);
    const bool fast = all_ok && n == kTileHG && whole_blocks && !kPerRow;
    if (lane == 0) mbar_wait(eb, ph ^ 1, p.err, abort);
    __syncwarp();
    const uint32_t sk = stage0 + st * kStageBytes, sv = sk + kCWarps * kHeadK;
    const int h0 = pos.g * GH;  // first KV head of the group
    if (fast) {
      if (lane == 0) {
        mbar_arrive_expect_tx(fb, (uint32_t)H * kTileHG * (RK + RV));
        const long long row = (long long)tb * H * ps;  // block base, head 0, slot 0
        bulk_g2s_hint(sk, p.k_pool + row * RK, (uint32_t)H * kTileHG * RK, fb, policy);
        bulk_g2s_hint(sv, p.v_pool + row * RV, (uint32_t)H * kTileHG * RV, fb, policy);
      }
      __syncwarp();
    } else {
      if (!ok) record_error(p.err, PA_ERR_BOUNDS);
      // Lane covers row r = lane & 15 of heads (lane >> 4) and (lane >> 4) + 2.
      // Every lane takes part in the shuffle.
      const int r = lane & 15;
      const int pg_r = (k0 + r) / ps;
      const int blk_r = __shfl_sync(0xffffffffu, tb, min(pg_r - p0, 31));
      const bool row_ok = r < n && blk_r >= 0 && blk_r < p.n_blocks;
      uint32_t bytes = 0;
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int w = (lane >> 4) + 2 * k;
        if (w < GH && row_ok) {
          if (kPerRow) bytes += RK + RV;
        } else {
          for (int c = 0; c < RK; c += 16) sts128_zero(sk + w * kHeadK + r * SK + c);
          for (int c = 0; c < RV; c += 16) sts128_zero(sv + w * kHeadV + r * SV + c);
        }
      }
      // Page runs (packed layouts): the page's lane counts the run for all heads.
      int rs = 0, re = 0;
      if (!kPerRow && used && ok) {
        rs = max(k0, (p0 + lane) * ps);
        re = min(k0 + n, (p0 + lane + 1) * ps);
        bytes += (uint32_t)(re - rs) * GH * (RK + RV);
      }
      fence_proxy_async_smem();
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) bytes += __shfl_xor_sync(0xffffffffu, bytes, o);
      __syncwarp();
      if (lane == 0) mbar_arrive_expect_tx(fb, bytes);
      __syncwarp();
      if (kPerRow) {
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const int w = (lane >> 4) + 2 * k;
          if (w < GH && row_ok) {
            const long long row = ((long long)blk_r * H + h0 + w) * ps + (k0 + r) % ps;
            bulk_g2s_hint(sk + w * kHeadK + r * SK, p.k_pool + row * RK, RK, fb, policy);
            bulk_g2s_hint(sv + w * kHeadV + r * SV, p.v_pool + row * RV, RV, fb, policy);
          }
        }
      } else if (used && ok) {
        const int pg = p0 + lane;
        for (int w = 0; w < GH; ++w) {
          const long long row = ((long long)tb * H + h0 + w) * ps + (rs - pg * ps);
          bulk_g2s_hint(sk + w * kHeadK + (rs - k0) * SK, p.k_pool + row * RK, (re - rs) * RK, fb, policy);
          bulk_g2s_hint(sv + w * kHeadV + (rs - k0) * SV, p.v_pool + row * RV, (re - rs) * RV, fb, policy);
        }
      }
    }
    ++issued;
    if (++st == kStages) { st = 0; ph ^= 1; }
    pos = nxt;
    tb = tbn;
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

// ------------------------------------------------------------------ producer

// Producer for per-head tiles (64 keys of one KV head): stream the CTA's
// tiles into the stage ring.  The table
// entries of tile i+1 are loaded while tile i is waited for and issued, so the
// table's latency stays off the refill path.  A full tile whose entries are
// all valid takes the fast path (no zero fill, byte count known).
template <int KT, int VT, int NT>
__device__ void produce_head(const DecodeParams& p, uint8_t* smem, uint32_t bar_full, uint32_t bar_empty,
                        volatile int* abort, long long a, long long b, TilePos pos) {
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
  int tb[2], tbn[2] = {-1, -1};
  load_tile_table<kPerRow>(p, pos, lane, tb);
  for (long long x = a; x < b; ++x) {
    if (*abort) break;
    TilePos nxt = pos;
    if (x + 1 < b) {
      next_tile(p, nxt);
      load_tile_table<kPerRow>(p, nxt, lane, tbn);
    }
    const uint32_t fb = bar_full + 8 * st, eb = bar_empty + 8 * st;
    const int k0 = pos.j * kTile;
    const int n = min(kTile, pos.L - k0);
    const int p0 = k0 / ps, p1 = (k0 + n - 1) / ps;
    bool mine_ok = true;
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const bool used = kPerRow ? (lane + 32 * u < n) : (p0 + lane + 32 * u <= p1);
      if (used && !(tb[u] >= 0 && tb[u] < p.n_blocks)) mine_ok = false;
    }
    const bool fast = __all_sync(0xffffffffu, mine_ok) && n == kTile;
    if (lane == 0) mbar_wait(eb, ph ^ 1, p.err, abort);
    __syncwarp();
    const uint32_t sk = stage0 + st * kStageBytes, sv = sk + kTile * SK;
    uint32_t bytes = (uint32_t)kTile * (RK + RV);
    if (!fast) {
      // Zero-fill rows with no valid source (bad table entry, or past the end
      // of the sequence: their V must be finite, their weight is 0) and count
      // the bytes the copies will deliver.
      bytes = 0;
      if (kPerRow) {
        for (int r = lane; r < kTile; r += 32) {
          const int blk = r < n ? ((r >> 5) ? tb[1] : tb[0]) : -1;
          if (r < n && blk >= 0 && blk < p.n_blocks) {
            bytes += RK + RV;
          } else {
            if (r < n) record_error(p.err, PA_ERR_BOUNDS);
            for (int c = 0; c < RK; c += 16) sts128_zero(sk + r * SK + c);
            for (int c = 0; c < RV; c += 16) sts128_zero(sv + r * SV + c);
          }
        }
      } else {
        for (int pg = p0 + lane; pg <= p1; pg += 32) {
          const int rs = max(k0, pg * ps), re = min(k0 + n, (pg + 1) * ps);
          const int blk = (((pg - p0) >> 5) ? tb[1] : tb[0]);
          if (blk >= 0 && blk < p.n_blocks) {
            bytes += (re - rs) * (RK + RV);
          } else {
            record_error(p.err, PA_ERR_BOUNDS);
            for (int r = rs - k0; r < re - k0; ++r) {
              for (int c = 0; c < RK; c += 16) sts128_zero(sk + r * SK + c);
              for (int c = 0; c < RV; c += 16) sts128_zero(sv + r * SV + c);
            }
          }
        }
        for (int r = n + lane; r < kTile; r += 32) {
          for (int c = 0; c < RK; c += 16) sts128_zero(sk + r * SK + c);
          for (int c = 0; c < RV; c += 16) sts128_zero(sv + r * SV + c);
        }
      }
      fence_proxy_async_smem();
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) bytes += __shfl_xor_sync(0xffffffffu, bytes, o);
      __syncwarp();
    }
    if (lane == 0) mbar_arrive_expect_tx(fb, bytes);
    __syncwarp();
    if (kPerRow) {
      for (int r = lane; r < n; r += 32) {
        const int blk = ((r >> 5) ? tb[1] : tb[0]);
        if (blk >= 0 && blk < p.n_blocks) {
          const long long row = ((long long)blk * p.n_kv_heads + pos.g) * ps + (k0 + r) % ps;
          bulk_g2s_hint(sk + r * SK, p.k_pool + row * RK, RK, fb, policy);
          bulk_g2s_hint(sv + r * SV, p.v_pool + row * RV, RV, fb, policy);
        }
      }
    } else {
      for (int pg = p0 + lane; pg <= p1; pg += 32) {
        const int rs = max(k0, pg * ps), re = min(k0 + n, (pg + 1) * ps);
        const int blk = (((pg - p0) >> 5) ? tb[1] : tb[0]);
        if (blk >= 0 && blk < p.n_blocks) {
          const long long row = ((long long)blk * p.n_kv_heads + pos.g) * ps + (rs - pg * ps);
          bulk_g2s_hint(sk + (rs - k0) * SK, p.k_pool + row * RK, (re - rs) * RK, fb, policy);
          bulk_g2s_hint(sv + (rs - k0) * SV, p.v_pool + row * RV, (re - rs) * RV, fb, policy);
        }
      }
    }
    ++issued;
    if (++st == kStages) { st = 0; ph ^= 1; }
    pos = nxt;
    tb[0] = tbn[0];
    tb[1] = tbn[1];
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

// Head-group path: warp w stages its own KV head's six query rows (one
// query token) as S-MMA B fragments ([k-step][lane] uint2) and the per-block
// bias corrections cb[block][row], from coalesced float4 loads.  Rows 6 and 7
// of the fragment (padding) are zero.  Only this warp reads them.
template <int KT>
__device__ __forceinline__ int kdim_inverse(int d, int& ks, int& jj) {
  // returns nothing useful; fills the k-step and k-index that hold dim d
  int t, u, h, e;
  if (KT == PA_F16) {
    const int c = d >> 6, r = d & 63;
    t = r >> 4; u = (r & 15) >> 2; h = (r >> 1) & 1; e = r & 1;
    ks = 4 * c + u;
  } else if (KT == PA_Q8_0) {
    const int b = d >> 5, r = d & 31;
    t = r >> 3; u = (r >> 2) & 1; h = r & 1; e = (r >> 1) & 1;
    ks = 2 * b + u;
  } else {  // Q4_0
    const int b = d >> 5, r = d & 31;
    u = r >> 4; t = (r & 15) >> 2; h = r & 1; e = (r >> 1) & 1;
    ks = 2 * b + u;
  }
  jj = 2 * t + 8 * h + e;
  return t;
}

template <int KT>
__device__ void stage_q_warp(const DecodeParams& p, int s, int head, uint32_t qf, float* cb, int lane) {
  // zero the padding rows 6, 7 (lanes 24..31 of every k-step) and their
  // corrections, so the padding logits are exactly 0
  if (lane >= 24) {
#pragma unroll
    for (int ks = 0; ks < 16; ++ks)
      asm volatile("st.shared.v2.b32 [%0], {%1, %1};" ::"r"(qf + (ks * 32 + lane) * 8), "r"(0u) : "memory");
  }
  if (KT != PA_F16 && lane < 16) cb[(lane >> 1) * 8 + 6 + (lane & 1)] = 0.f;
  const float4* q4 = reinterpret_cast<const float4*>(p.q + ((long long)s * p.n_q_heads + head * kGqa) * kD);
#pragma unroll 4
  for (int i = 0; i < kGqa * kD / 4 / 32; ++i) {  // 12 float4 per lane
    const int f = lane + 32 * i;
    const int row = f >> 6, d0 = 4 * (f & 63);
    const float4 v = __ldg(q4 + f);
    const float vals[4] = {v.x, v.y, v.z, v.w};
    float lo = 0.f;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int d = d0 + k;
      int ks, jj;
      const int t = kdim_inverse<KT>(d, ks, jj);
      const float sc = (KT == PA_Q4_0 && (ks & 1)) ? 0.0625f : 1.f;
      const __half hv = __float2half_rn(sc * vals[k]);
      lo += __half2float(hv);
      const int ln = 4 * row + t;
      const uint32_t addr = qf + (ks * 32 + ln) * 8 + ((jj >> 3) << 2) + ((jj & 1) << 1);
      asm volatile("st.shared.b16 [%0], %1;" ::"r"(addr), "h"(__half_as_ushort(hv)) : "memory");
    }
    if (KT != PA_F16) {
      // lanes 8b'..8b'+7 hold the 8 float4 of block 4(i&1)+b' of row i/2:
      // k < 4 low 16 dims, k >= 4 high 16 dims.
      lo += __shfl_xor_sync(0xffffffffu, lo, 1);
      lo += __shfl_xor_sync(0xffffffffu, lo, 2);
      const float hi = __shfl_down_sync(0xffffffffu, lo, 4);
      if ((lane & 7) == 0) {
        const int blk = 4 * (i & 1) + (lane >> 3);
        cb[blk * 8 + (i >> 1)] = (KT == PA_Q4_0) ? 1032.f * lo + 1152.f * hi : 1152.f * (lo + hi);
      }
    }
  }
  __syncwarp();
}

// ------------------------------------------------------------------ Q staging

__device__ __forceinline__ const float* q_row(const DecodeParams& p, int s, int g, int row) {
  const int tq = row / kGqa, hl = row % kGqa;
  return p.q + (((long long)s * p.n_qtok + tq) * p.n_q_heads + g * kGqa + hl) * kD;
}

__device__ __forceinline__ float round_half(float v) { return __half2float(__float2half_rn(v)); }

// Stage Q of (sequence s, KV head g) as S-MMA B fragments in the K format's
// dim order ([k-step][nt][lane] uint2; high-nibble Q4_0 k-steps hold Q/16),
// and, for quantised K, the per-block bias corrections cb[block][row]: the
// exact sum of the block's fp16 Q values times the magic bias the A operand
// carries (1032 low / 1152 high nibbles for Q4_0, 1152 for Q8_0).
template <int KT, int NT>
__device__ void stage_q(const DecodeParams& p, int s, int g, uint32_t qf, float* cb, int tid) {
  const int R = kGqa * p.n_qtok;
  constexpr int kN = kCWarps * 32;
  for (int e = tid; e < 16 * NT * 32; e += kN) {
    const int ln = e & 31, nt = (e >> 5) % NT, ks = e / (32 * NT);
    const int row = nt * 8 + (ln >> 2), t4 = ln & 3;
    uint32_t b0 = 0, b1 = 0;
    if (row < R) {
      const float* qr = q_row(p, s, g, row);
      const float f = (KT == PA_Q4_0 && (ks & 1)) ? 0.0625f : 1.f;
      b0 = pack_half2(f * __ldg(qr + kdim<KT>(ks, 2 * t4)), f * __ldg(qr + kdim<KT>(ks, 2 * t4 + 1)));
      b1 = pack_half2(f * __ldg(qr + kdim<KT>(ks, 2 * t4 + 8)), f * __ldg(qr + kdim<KT>(ks, 2 * t4 + 9)));
    }
    asm volatile("st.shared.v2.b32 [%0], {%1, %2};" ::"r"(qf + ((ks * NT + nt) * 32 + ln) * 8), "r"(b0), "r"(b1)
                 : "memory");
  }
  if (KT != PA_F16) {
    for (int e = tid; e < 8 * NT * 8; e += kN) {
      const int blk = e / (NT * 8), row = e % (NT * 8);
      float c = 0.f;
      if (row < R) {
        const float* qr = q_row(p, s, g, row) + 32 * blk;
        float lo = 0.f, hi = 0.f;
#pragma unroll 8
        for (int i = 0; i < 16; ++i) lo += round_half(__ldg(qr + i));
        if (KT == PA_Q4_0) {
#pragma unroll 8
          for (int i = 16; i < 32; ++i) hi += round_half(0.0625f * __ldg(qr + i));
          c = 1032.f * lo + 1152.f * hi;
        } else {
#pragma unroll 8
          for (int i = 16; i < 32; ++i) lo += round_half(__ldg(qr + i));
          c = 1152.f * lo;
        }
      }
      cb[blk * NT * 8 + row] = c;
    }
  }
}

// ------------------------------------------------------------------ S phase (K side)

// acc[nt] += S^T for 16 keys (rows r0 = key g, r1 = key g+8 of the stage)
// against the staged Q fragments, over all 256 dims.  qf: this lane's Q
// fragments; cbl: shared address of cb[0][2t] for this lane.
template <int KT, int NT>
__device__ __forceinline__ void s_phase(float (&acc)[NT][4], uint32_t r0, uint32_t r1, uint32_t qf, uint32_t cbl,
                                        int lane) {
  const int t = lane & 3;
  if constexpr (KT == PA_F16) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const uint32_t off = 128 * c + 32 * t;
      const uint4 R0 = lds128(r0 + off), R1 = lds128(r0 + off + 16);
      const uint4 S0 = lds128(r1 + off), S1 = lds128(r1 + off + 16);
      const uint32_t a0[4] = {R0.x, S0.x, R0.y, S0.y}, a1[4] = {R0.z, S0.z, R0.w, S0.w};
      const uint32_t a2[4] = {R1.x, S1.x, R1.y, S1.y}, a3[4] = {R1.z, S1.z, R1.w, S1.w};
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const uint2 q0 = lds64(qf + ((4 * c + 0) * NT + nt) * 256), q1 = lds64(qf + ((4 * c + 1) * NT + nt) * 256);
        const uint2 q2 = lds64(qf + ((4 * c + 2) * NT + nt) * 256), q3 = lds64(qf + ((4 * c + 3) * NT + nt) * 256);
        mma_16816(acc[nt], a0, q0.x, q0.y);
        mma_16816(acc[nt], a1, q1.x, q1.y);
        mma_16816(acc[nt], a2, q2.x, q2.y);
        mma_16816(acc[nt], a3, q3.x, q3.y);
      }
    }
  } else {
#pragma unroll
    for (int b = 0; b < 8; ++b) {
      uint32_t a0[4], a1[4];  // k-steps 2b, 2b+1
      uint32_t d0h, d1h;
      if constexpr (KT == PA_Q4_0) {
        const uint32_t x0 = q4_word(r0, b, t), x1 = q4_word(r1, b, t);
        const uint32_t y0 = x0 >> 8, y1 = x1 >> 8;
        a0[0] = and_or(x0, 0x000f000fu, 0x64006400u);
        a0[1] = and_or(x1, 0x000f000fu, 0x64006400u);
        a0[2] = and_or(y0, 0x000f000fu, 0x64006400u);
        a0[3] = and_or(y1, 0x000f000fu, 0x64006400u);
        a1[0] = and_or(x0, 0x00f000f0u, 0x64006400u);
        a1[1] = and_or(x1, 0x00f000f0u, 0x64006400u);
        a1[2] = and_or(y0, 0x00f000f0u, 0x64006400u);
        a1[3] = and_or(y1, 0x00f000f0u, 0x64006400u);
        d0h = lds16(r0 + 18 * b);
        d1h = lds16(r1 + 18 * b);
      } else {  // Q8_0: byte x -> 1024 + (x + 128)
        uint32_t y00, y01, y10, y11;
        q8_words(r0, b, t, y00, y01);
        q8_words(r1, b, t, y10, y11);
        y00 ^= 0x80808080u; y01 ^= 0x80808080u; y10 ^= 0x80808080u; y11 ^= 0x80808080u;
        a0[0] = prmt(y00, 0x64646464u, 0x4240);
        a0[1] = prmt(y10, 0x64646464u, 0x4240);
        a0[2] = prmt(y00, 0x64646464u, 0x4341);
        a0[3] = prmt(y10, 0x64646464u, 0x4341);
        a1[0] = prmt(y01, 0x64646464u, 0x4240);
        a1[1] = prmt(y11, 0x64646464u, 0x4240);
        a1[2] = prmt(y01, 0x64646464u, 0x4341);
        a1[3] = prmt(y11, 0x64646464u, 0x4341);
        d0h = lds16(r0 + 34 * b);
        d1h = lds16(r1 + 34 * b);
      }
      const float d0 = half_bits_to_float(d0h), d1 = half_bits_to_float(d1h);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        float tmp[4] = {0.f, 0.f, 0.f, 0.f};
        const uint2 q0 = lds64(qf + ((2 * b) * NT + nt) * 256), q1 = lds64(qf + ((2 * b + 1) * NT + nt) * 256);
        mma_16816(tmp, a0, q0.x, q0.y);
        mma_16816(tmp, a1, q1.x, q1.y);
        const float2 c = lds64f(cbl + (b * NT * 8 + nt * 8) * 4);
        acc[nt][0] = fmaf(d0, tmp[0] - c.x, acc[nt][0]);
        acc[nt][1] = fmaf(d0, tmp[1] - c.y, acc[nt][1]);
        acc[nt][2] = fmaf(d1, tmp[2] - c.x, acc[nt][2]);
        acc[nt][3] = fmaf(d1, tmp[3] - c.y, acc[nt][3]);
      }
    }
  }
}

// ------------------------------------------------------------------ PV, one-token path

// o[i] (16 m-tiles, all 256 dims) += V^T (this warp's 16 keys) x P^T.
// rows[k]: shared addresses of V rows for keys 2t, 2t+1, 2t+8, 2t+9 of the
// warp's 16; bp0/bp1: P B fragments (keys 2t.., 2t+8..; row g).
template <int VT>
__device__ __forceinline__ void pv_solo(float (&o)[16][4], const uint32_t (&rows)[4], int lane, uint32_t bp0,
                                        uint32_t bp1) {
  const int g = lane >> 2;
  if constexpr (VT == PA_F16) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {  // dims 64k + 8g .. +7
      const uint32_t off = 128 * k + 16 * g;
      const uint4 A = lds128(rows[0] + off), B = lds128(rows[1] + off);
      const uint4 C = lds128(rows[2] + off), D = lds128(rows[3] + off);
      const uint32_t av[4] = {A.x, A.y, A.z, A.w}, bv[4] = {B.x, B.y, B.z, B.w};
      const uint32_t cv[4] = {C.x, C.y, C.z, C.w}, dv[4] = {D.x, D.y, D.z, D.w};
#pragma unroll
      for (int l = 0; l < 4; ++l) {  // m-tile 4k + l: rows g <-> dim 2l, g+8 <-> dim 2l+1
        const uint32_t a[4] = {prmt(av[l], bv[l], 0x5410), prmt(av[l], bv[l], 0x7632), prmt(cv[l], dv[l], 0x5410),
                               prmt(cv[l], dv[l], 0x7632)};
        mma_16816(o[4 * k + l], a, bp0, bp1);
      }
    }
  } else if constexpr (VT == PA_Q4_0) {
#pragma unroll
    for (int b = 0; b < 8; ++b) {  // m-tiles 2b, 2b+1 hold block b
      const uint32_t qo = 18 * b + 2 + 2 * g, so = 18 * b;
      const uint32_t x0 = lds16(rows[0] + qo), x1 = lds16(rows[1] + qo);
      const uint32_t x2 = lds16(rows[2] + qo), x3 = lds16(rows[3] + qo);
      const uint32_t d0 = lds16(rows[0] + so), d1 = lds16(rows[1] + so);
      const uint32_t d2 = lds16(rows[2] + so), d3 = lds16(rows[3] + so);
      uint32_t la0, ha0, la1, ha1, lc0, hc0, lc1, hc1;
      q4_exact(x0 | (x1 << 16), la0, ha0, la1, ha1);  // keys 2t, 2t+1: dims 2g, 2g+16, 2g+1, 2g+17
      q4_exact(x2 | (x3 << 16), lc0, hc0, lc1, hc1);  // keys 2t+8, 2t+9
      const uint32_t p0 = hmul2(bp0, d0 | (d1 << 16)), p1 = hmul2(bp1, d2 | (d3 << 16));
      const uint32_t A0[4] = {la0, ha0, lc0, hc0}, A1[4] = {la1, ha1, lc1, hc1};
      mma_16816(o[2 * b], A0, p0, p1);
      mma_16816(o[2 * b + 1], A1, p0, p1);
    }
  } else {  // Q8_0: thread g takes quants 4g..4g+3 of each block
#pragma unroll
    for (int b = 0; b < 8; ++b) {
      const uint32_t qo = 34 * b + 2 + 4 * g, so = 34 * b;
      uint32_t y[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        if (b & 1) y[k] = lds32(rows[k] + qo);
        else y[k] = prmt(lds32(rows[k] + qo - 2), lds32(rows[k] + qo + 2), 0x5432);
        y[k] ^= 0x80808080u;
      }
      const uint32_t d0 = lds16(rows[0] + so), d1 = lds16(rows[1] + so);
      const uint32_t d2 = lds16(rows[2] + so), d3 = lds16(rows[3] + so);
      uint32_t e[2][4];  // [key pair][quant]
#pragma unroll
      for (int pr = 0; pr < 2; ++pr)
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint32_t sel = k | (k << 4) | ((4 + k) << 8) | ((4 + k) << 12);
          e[pr][k] = hadd2(and_xor(prmt(y[2 * pr], y[2 * pr + 1], sel), 0x00ff00ffu, 0x64006400u), kHalf2_m1152);
        }
      const uint32_t p0 = hmul2(bp0, d0 | (d1 << 16)), p1 = hmul2(bp1, d2 | (d3 << 16));
      const uint32_t A0[4] = {e[0][0], e[0][1], e[1][0], e[1][1]}, A1[4] = {e[0][2], e[0][3], e[1][2], e[1][3]};
      mma_16816(o[2 * b], A0, p0, p1);
      mma_16816(o[2 * b + 1], A1, p0, p1);
    }
  }
}

// ------------------------------------------------------------------ PV, multi-token path

// o[i][nt] += V^T(dims of warp w, m-tile i; keys of k-step kw) x P^T.
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
    for (int pp = 0; pp < 2; ++pp) {  // key pair pp: keys (2pp, 2pp+1) of rows[]
      const uint4 A = R[2 * pp], B = R[2 * pp + 1];
      a[0][2 * pp] = prmt(A.x, B.x, 0x5410); a[0][2 * pp + 1] = prmt(A.x, B.x, 0x7632);
      a[1][2 * pp] = prmt(A.y, B.y, 0x5410); a[1][2 * pp + 1] = prmt(A.y, B.y, 0x7632);
      a[2][2 * pp] = prmt(A.z, B.z, 0x5410); a[2][2 * pp + 1] = prmt(A.z, B.z, 0x7632);
      a[3][2 * pp] = prmt(A.w, B.w, 0x5410); a[3][2 * pp + 1] = prmt(A.w, B.w, 0x7632);
    }
  } else if constexpr (VT == PA_Q8_0) {
    const int blk = 2 * w + (g >> 2), q = g & 3;
    const uint32_t off = 34 * blk + 2 + 8 * q, base = off & ~3u;
    const uint32_t sel = (off & 2) ? 0x5432u : 0x3210u;
    uint32_t y[4][2], d[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint32_t w0 = lds32(rows[k] + base), w1 = lds32(rows[k] + base + 4), w2 = lds32(rows[k] + base + 8);
      y[k][0] = prmt(w0, w1, sel);
      y[k][1] = prmt(w1, w2, sel);
      d[k] = lds16(rows[k] + 34 * blk);
    }
#pragma unroll
    for (int pp = 0; pp < 2; ++pp) {
      const uint32_t dd = d[2 * pp] | (d[2 * pp + 1] << 16);
#pragma unroll
      for (int wd = 0; wd < 2; ++wd) {
        const uint32_t A = y[2 * pp][wd] ^ 0x80808080u, B = y[2 * pp + 1][wd] ^ 0x80808080u;
#pragma unroll
        for (int k = 0; k < 4; ++k) {  // quant 4*wd + k -> m-tile (4wd+k)/2, half (k&1)
          const uint32_t s2 = k | (k << 4) | ((4 + k) << 8) | ((4 + k) << 12);
          const uint32_t e = and_xor(prmt(A, B, s2), 0x00ff00ffu, 0x64006400u);
          a[(4 * wd + k) >> 1][2 * pp + (k & 1)] = hmul2(hadd2(e, kHalf2_m1152), dd);
        }
      }
    }
  } else {  // Q4_0
    const int blk = 2 * w + (g >> 2), q = g & 3;
    // quant bytes 4q..4q+3 of block blk start 2 bytes past a word boundary
    // when blk is even: load the two words around them and shift by PRMT.
    const uint32_t off = 18 * blk + 2 + 4 * q, base = off & ~3u;
    const uint32_t sel = (off & 2) ? 0x5432u : 0x3210u;
    uint32_t x[4], d[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      x[k] = prmt(lds32(rows[k] + base), lds32(rows[k] + base + 4), sel);
      d[k] = lds16(rows[k] + 18 * blk);
    }
#pragma unroll
    for (int pp = 0; pp < 2; ++pp) {
      const uint32_t dd = d[2 * pp] | (d[2 * pp + 1] << 16);
      const uint32_t xa = prmt(x[2 * pp], x[2 * pp + 1], 0x5410);  // [k0.c0 k0.c1 k1.c0 k1.c1]
      const uint32_t xb = prmt(x[2 * pp], x[2 * pp + 1], 0x7632);  // [k0.c2 k0.c3 k1.c2 k1.c3]
      uint32_t l0, h0, l1, h1;
      q4_dequant(xa, dd, l0, h0, l1, h1);  // dims j0, j0+16, j0+1, j0+17
      a[0][2 * pp] = l0; a[0][2 * pp + 1] = h0;
      a[1][2 * pp] = l1; a[1][2 * pp + 1] = h1;
      q4_dequant(xb, dd, l0, h0, l1, h1);  // dims j0+2, j0+18, j0+3, j0+19
      a[2][2 * pp] = l0; a[2][2 * pp + 1] = h0;
      a[3][2 * pp] = l1; a[3][2 * pp + 1] = h1;
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t A[4] = {a[i][0], a[i][1], a[i][2], a[i][3]};
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) mma_16816(o[i][nt], A, bp[nt][0], bp[nt][1]);
  }
}

// ------------------------------------------------------------------ piece output

// Write one query row's result: the final output (out = O / l, lse) when the
// piece covers its whole segment, else the split partial (O, (m, l)).
__device__ __forceinline__ float* row_dst(const DecodeParams& p, bool whole, int slot, int s, int g, int row,
                                          int R) {
  if (whole) {
    const int tk = row / kGqa, hl = row % kGqa;
    return p.out + (((long long)s * p.n_qtok + tk) * p.n_q_heads + g * kGqa + hl) * kD;
  }
  return p.part_o + ((long long)slot * R + row) * kD;
}

__device__ __forceinline__ void write_row_stats(const DecodeParams& p, bool whole, int slot, int s, int g, int row,
                                                int R, float m, float l) {
  if (whole) {
    if (p.lse) {
      const int tk = row / kGqa, hl = row % kGqa;
      p.lse[((long long)s * p.n_qtok + tk) * p.n_q_heads + g * kGqa + hl] =
          l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
    }
  } else {
    p.part_ml[(long long)slot * R + row] = make_float2(m, l);
  }
}

// ------------------------------------------------------------------ head-group consumer

// One query token: warp w owns KV head (group * GH + w); see the file comment.
template <int KT, int VT>
__device__ void consume_hg(const DecodeParams& p, uint8_t* smem, uint32_t bar_full, uint32_t bar_empty,
                           volatile int* abort, long long a, long long b, int s, int g, int j) {
  using SM = Smem<KT, VT, 1>;
  constexpr int kStages = SM::kStages;
  constexpr int SK = Fmt<KT>::kStride, SV = Fmt<VT>::kStride;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gq = lane >> 2, tq = lane & 3;
  const uint32_t sbase = smem_u32(smem);
  const uint32_t qf = sbase + SM::kWQ + warp * SM::kWQBytes;
  float* cb = reinterpret_cast<float*>(smem + SM::kWCb + warp * SM::kWCbBytes);
  const uint32_t qf_lane = qf + lane * 8;
  const uint32_t cb_lane = smem_u32(cb) + 2 * tq * 4;
  const bool active = warp < p.seg_heads;
  int st = 0;
  uint32_t ph = 0;
  long long x = a;
  while (x < b) {
    const int L = p.seq_lens[s];
    const int ntl = tiles_of(p, L);
    const int jb = j, je = (int)((long long)ntl < j + (b - x) ? (long long)ntl : j + (b - x));
    const int seg = s * p.segs_per_seq + g;
    const bool whole = (jb == 0 && je == ntl);
    const int head = g * p.seg_heads + warp;
    if (active) stage_q_warp<KT>(p, s, head, qf, cb, lane);

    float o[16][4];
#pragma unroll
    for (int i = 0; i < 16; ++i)
#pragma unroll
      for (int c = 0; c < 4; ++c) o[i][c] = 0.f;
    float mref0 = -INFINITY, mref1 = -INFINITY;  // rows 2tq, 2tq+1
    float ls0 = 0.f, ls1 = 0.f;                  // this thread's share of the row sums

    const int vis = L - 1;  // last visible key (one query token)
    for (int jt = jb; jt < je; ++jt) {
      if (!*abort) mbar_wait(bar_full + 8 * st, ph, p.err, abort);
      if (active) {
        const uint32_t sk = sbase + st * SM::kStageBytes + warp * (kTileHG * SK);
        const uint32_t sv = sbase + st * SM::kStageBytes + SM::kKBytes + warp * (kTileHG * SV);
        const int k0 = jt * kTileHG;
        float sacc[1][4] = {{0.f, 0.f, 0.f, 0.f}};
        s_phase<KT, 1>(sacc, sk + gq * SK, sk + (gq + 8) * SK, qf_lane, cb_lane, lane);
        float xv[4];
        const bool need_mask = (k0 + kTileHG - 1) > vis;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          xv[c] = sacc[0][c] * p.scale_log2;
          if (need_mask && k0 + gq + ((c & 2) ? 8 : 0) > vis) xv[c] = -INFINITY;
        }
        // ---- lazy running max
        const bool up = (xv[0] > mref0 + kLazy) || (xv[2] > mref0 + kLazy) || (xv[1] > mref1 + kLazy) ||
                        (xv[3] > mref1 + kLazy);
        if (__any_sync(0xffffffffu, up)) {
          float mx0 = fmaxf(xv[0], xv[2]), mx1 = fmaxf(xv[1], xv[3]);
#pragma unroll
          for (int off = 4; off < 32; off <<= 1) {
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
          }
          const float mn0 = fmaxf(mref0, mx0), mn1 = fmaxf(mref1, mx1);
          const float al0 = (mn0 == -INFINITY) ? 1.f : exp2f(mref0 - mn0);
          const float al1 = (mn1 == -INFINITY) ? 1.f : exp2f(mref1 - mn1);
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            o[i][0] *= al0; o[i][2] *= al0;
            o[i][1] *= al1; o[i][3] *= al1;
          }
          ls0 *= al0;
          ls1 *= al1;
          mref0 = mn0;
          mref1 = mn1;
        }
        const float b0 = (mref0 == -INFINITY) ? 0.f : mref0, b1 = (mref1 == -INFINITY) ? 0.f : mref1;
        const uint32_t X0 = pack_half2(exp2f(xv[0] - b0), exp2f(xv[1] - b1));  // key gq: rows 2tq, 2tq+1
        const uint32_t X1 = pack_half2(exp2f(xv[2] - b0), exp2f(xv[3] - b1));  // key gq+8
        {
          const float2 f0 = __half22float2(*reinterpret_cast<const __half2*>(&X0));
          const float2 f1 = __half22float2(*reinterpret_cast<const __half2*>(&X1));
          ls0 += f0.x + f1.x;
          ls1 += f0.y + f1.y;
        }
        const uint32_t B0 = movmatrix_trans(X0), B1 = movmatrix_trans(X1);
        const uint32_t v0 = sv + 2 * tq * SV;
        const uint32_t rows[4] = {v0, v0 + SV, v0 + 8 * SV, v0 + 9 * SV};
        pv_solo<VT>(o, rows, lane, B0, B1);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_empty + 8 * st);
      if (++st == kStages) { st = 0; ph ^= 1; }
    }

    // ---- piece result for this warp's head: rows 2tq, 2tq+1 (< 6)
    if (active) {
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        ls0 += __shfl_xor_sync(0xffffffffu, ls0, off);
        ls1 += __shfl_xor_sync(0xffffffffu, ls1, off);
      }
      const int slot = (int)blockIdx.x + seg;
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int hl = 2 * tq + c;
        if (hl >= kGqa) continue;
        const float lr = c ? ls1 : ls0, mr = c ? mref1 : mref0;
        const int row = warp * kGqa + hl;  // row within the segment
        float* dst;
        float inv = 1.f;
        if (whole) {
          dst = p.out + ((long long)s * p.n_q_heads + head * kGqa + hl) * kD;
          inv = lr > 0.f ? 1.f / lr : 0.f;
        } else {
          dst = p.part_o + ((long long)slot * p.rows_per_seg + row) * kD;
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          dst[vdim_solo<VT>(gq, i, 0)] = o[i][c] * inv;
          dst[vdim_solo<VT>(gq, i, 1)] = o[i][2 + c] * inv;
        }
        if (gq == 0) {
          if (whole) {
            if (p.lse) p.lse[(long long)s * p.n_q_heads + head * kGqa + hl] = lr > 0.f ? (mr + log2f(lr)) * kLn2 : -INFINITY;
          } else {
            p.part_ml[(long long)slot * p.rows_per_seg + row] = make_float2(mr, lr);
          }
        }
      }
    }

    x += je - jb;
    j = 0;
    if (++g == p.segs_per_seq) { g = 0; ++s; }
  }
}

// ------------------------------------------------------------------ per-head consumer

// Multi-token path (NT = 2, 3): see the file comment.
template <int KT, int VT, int NT>
__device__ void consume_shared(const DecodeParams& p, uint8_t* smem, uint32_t bar_full, uint32_t bar_empty,
                               volatile int* abort, long long a, long long b, int s, int g, int j) {
  using SM = Smem<KT, VT, NT>;
  constexpr int kStages = SM::kStages;
  constexpr int R8 = NT * 8;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gq = lane >> 2, tq = lane & 3;
  const int R = kGqa * p.n_qtok;
  const uint32_t sbase = smem_u32(smem);
  const uint32_t pb_base = sbase + SM::kP;
  float2* stats = reinterpret_cast<float2*>(smem + SM::kStat);
  int st = 0;
  uint32_t ph = 0;
  int qbuf = 0, tbuf = 0;
  long long x = a;
  while (x < b) {
    const int L = p.seq_lens[s];
    const int ntl = tiles_of(p, L);
    const int jb = j, je = (int)((long long)ntl < j + (b - x) ? (long long)ntl : j + (b - x));
    const int seg = s * p.segs_per_seq + g;
    const bool whole = (jb == 0 && je == ntl);
    const uint32_t qf = sbase + SM::kQ + qbuf * SM::kQBuf;
    float* cb = reinterpret_cast<float*>(smem + SM::kCb + qbuf * SM::kCbBuf);
    stage_q<KT, NT>(p, s, g, qf, cb, tid);
    named_bar_sync(1, kCWarps * 32);
    const uint32_t qf_lane = qf + lane * 8;
    const uint32_t cb_lane = smem_u32(cb) + 2 * tq * 4;

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
        s_phase<KT, NT>(sacc, r0, r0 + 8 * Fmt<KT>::kStride, qf_lane, cb_lane, lane);
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
        const uint32_t X0 = pack_half2(exp2f(xv[0] - b0), exp2f(xv[1] - b1));
        const uint32_t X1 = pack_half2(exp2f(xv[2] - b0), exp2f(xv[3] - b1));
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
        alpha_c[nt][0] = __shfl_sync(0xffffffffu, alpha, 8 * tq);      // row 2*tq lives at g = 2*tq
        alpha_c[nt][1] = __shfl_sync(0xffffffffu, alpha, 8 * tq + 4);  // row 2*tq+1
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
        float* dst = row_dst(p, whole, slot, s, g, row, R);
        const float inv = whole ? (lr > 0.f ? 1.f / lr : 0.f) : 1.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          dst[vdim_shared<VT>(warp, gq, i, 0)] = o[i][nt][c] * inv;
          dst[vdim_shared<VT>(warp, gq, i, 1)] = o[i][nt][2 + c] * inv;
        }
        if (warp == 0 && gq == 0) write_row_stats(p, whole, slot, s, g, row, R, c ? mc1 : mc0, lr);
      }
    }

    x += je - jb;
    qbuf ^= 1;
    j = 0;
    if (++g == p.segs_per_seq) { g = 0; ++s; }
  }
}

// ------------------------------------------------------------------ the split kernel

template <int KT, int VT, int NT>
__global__ void __launch_bounds__(kThreads, CtaTarget<KT, VT, NT>::kN)
    pa_split_decode_kernel(const __grid_constant__ DecodeParams p) {
  using SM = Smem<KT, VT, NT>;
  constexpr int kStages = SM::kStages;
  extern __shared__ __align__(128) uint8_t smem[];
  const int tid = threadIdx.x, warp = tid >> 5;
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar_full = sbase + SM::kBar, bar_empty = bar_full + 8 * kStages;
  volatile int* abort = reinterpret_cast<volatile int*>(smem + SM::kMisc);
  int* start = reinterpret_cast<int*>(smem + SM::kMisc + 4);

  const long long T = p.total_tiles;
  const int G = p.n_ctas;
  const long long a = (long long)blockIdx.x * T / G, b = (long long)(blockIdx.x + 1) * T / G;

  // Zero the merge kernel's arrival counters (it reads them only after the
  // whole split grid has finished).
  for (int i = blockIdx.x * kThreads + tid; i < p.n_counters; i += gridDim.x * kThreads) p.merge_count[i] = 0;
  if (tid == 0) {
    // The merge kernel may launch now; it reads nothing of ours before its
    // griddepcontrol.wait.
    asm volatile("griddepcontrol.launch_dependents;");
    *abort = 0;
    for (int i = 0; i < kStages; ++i) {
      mbar_init(bar_full + 8 * i, 1);
      mbar_init(bar_empty + 8 * i, kCWarps);
    }
    fence_mbar_init();
    int s0, g0, j0;
    locate_tile(p, a, s0, g0, j0);
    start[0] = s0;
    start[1] = g0;
    start[2] = j0;
  }
  __syncthreads();
  const int s = start[0], g = start[1], j = start[2];

  if (warp == kCWarps) {
    TilePos pos;
    pos.s = s;
    pos.g = g;
    pos.j = j;
    pos.L = p.seq_lens[s];
    pos.nt = tiles_of(p, pos.L);
    if constexpr (NT == 1) {
      produce_hg<KT, VT, NT>(p, smem, bar_full, bar_empty, abort, a, b, pos);
    } else {
      produce_head<KT, VT, NT>(p, smem, bar_full, bar_empty, abort, a, b, pos);
    }
    return;
  }
  if constexpr (NT == 1) {
    consume_hg<KT, VT>(p, smem, bar_full, bar_empty, abort, a, b, s, g, j);
  } else {
    consume_shared<KT, VT, NT>(p, smem, bar_full, bar_empty, abort, a, b, s, g, j);
  }
}

// ------------------------------------------------------------------ host-side registry

using KernelFn = void (*)(DecodeParams);

struct KernelInfo {
  KernelFn fn;
  int smem;
  int ctas_per_sm_target;
};

template <int KT, int VT, int NT>
KernelInfo kernel_info() {
  return KernelInfo{pa_split_decode_kernel<KT, VT, NT>, Smem<KT, VT, NT>::kTotal, CtaTarget<KT, VT, NT>::kN};
}

// Defined once per K format (one translation unit each).
bool lookup_kernel_f16(int vt, int nt, KernelInfo* out);
bool lookup_kernel_q4_0(int vt, int nt, KernelInfo* out);
bool lookup_kernel_q8_0(int vt, int nt, KernelInfo* out);

}  // namespace pa_split
