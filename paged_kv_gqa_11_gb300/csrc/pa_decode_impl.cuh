// Device side of the split-K paged GQA decode (sm_103a).
//
// What is computed (llama.cpp fork PR #2, split-K decode commit; lucebox PR
// #555, Summary): for every (sequence, KV head) the 6 * n_qtok query rows of
// that KV head attend to the sequence's K/V rows, which are read page by page
// through the block table and dequantised in registers.  S = QK^T and O = PV
// run on the tensor cores (mma.sync m16n8k16, fp16 operands, fp32
// accumulation), the softmax is online, and the pieces of a split sequence are
// merged afterwards by log-sum-exp.
//
// Work split.  The batch is cut into segments (below), each a run of tiles.
// All tiles are laid end to end and cut into equal contiguous ranges, one per
// CTA, with as many CTAs as fit on the SMs at once.  A CTA's range may cover
// the tail of one segment and the head of the next; each piece becomes one
// split partial.  The cut depends only on the sequence lengths, so a paged and
// an identity-table cache give the same splits, the same summation order and
// bit-identical results (TensorFold #1156, Design / Kernels: paging changes
// where a row is read from, never the order in which keys are summed).
//
// Data movement.  The pool stores every page as row groups of 16 rows
// (pa_layout.cuh), so a group is one contiguous run and, for 16-row pages, a
// page of every KV head is one run per pool.  One producer warp streams the
// runs into a ring of shared-memory stages with cp.async.bulk, completing on
// mbarriers; the table is read one tile ahead, once per page (TensorFold
// #1156: the page lookup is done once per block, not per row).  A table entry
// outside the pool is never dereferenced: its rows are zero-filled and
// PA_ERR_BOUNDS is recorded.  Consumer warps read the stage with ldmatrix,
// whose row addresses follow the layout's chunk swizzle without bank
// conflicts.
//
// One query token ("head-group" tiles).  A segment is (sequence, group of up
// to four KV heads); a tile is one row group (16 keys) of every head of the
// group.  Consumer warp w owns KV head w of the group end to end: it stages
// its six query rows, computes S^T = K Q^T (M = keys, N = query rows,
// K = dims), the softmax, and O^T += V^T P^T over all 256 dims (M = dims,
// N = rows, K = keys).  Warps never wait for each other.  The running max is
// raised only when a logit exceeds it by more than 2^8 (P <= 256 stays exact
// enough in fp16), so most tiles rescale nothing.
//
// Two to eight query tokens ("per-head" tiles, 12-48 rows).  Holding O for all
// dims per warp would take 64 registers per 8 rows, so the warps split the
// tile instead: a segment is (sequence, KV head), a tile 64 keys (four row
// groups) of that head; in the S phase warp w computes the keys of group w
// against a reference maximum per row that the four warps share (raised, in
// a rare second step, only when a logit passes it by 2^8), publishes P
// (transposed with movmatrix) in shared memory, and after a named barrier
// computes O^T for dims 64w..64w+63 over all 64 keys.  Six to eight tokens run
// two such groups of four warps in one CTA, each taking half of the tokens,
// over the same stage ring.
//
// Dequantisation.  K goes into the MMA as raw magic-biased halves: a Q4_0
// nibble n becomes 1024+n (low) or 1024+16n (high nibble, against Q/16), a
// Q8_0 byte x becomes 1152+x.  Each 32-dim block gets its own accumulator,
// started at minus the bias (the sum of the block's fp16 Q times 1032/1152,
// computed when Q is staged), and the block scale d is applied in fp32.  V is
// converted to the exact integers n-8 / x in fp16 and the block scale is
// folded into P (each MMA's 16 dims lie in one block).  The head dims are
// visited in whatever order the fragment loads deliver them; Q and the output
// use the same order, so the dot products are unchanged.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <type_traits>

#include "pa.h"
#include "pa_device.cuh"
#include "pa_layout.cuh"

namespace pa_split {

using namespace pa_dev;
using pa_layout::Fmt;
using pa_layout::kGroup;

constexpr int kD = 256;       // head dim
constexpr int kGqa = 6;       // query heads per KV head
constexpr int kTile = 64;     // keys per per-head tile (two or more query tokens)
constexpr int kTileHG = 16;   // keys per head-group tile (one query token)
constexpr int kMaxQTok = 8;   // query tokens per sequence (speculative-verify widths)
constexpr int kMaxNT = (kGqa * kMaxQTok + 7) / 8;  // n-tiles of 8 query rows: 6
constexpr int kCWarps = 4;    // consumer warps per group (one-token path: = heads per head group, at most)
// Threads of a split-kernel CTA: kG groups of consumer warps and one producer
// warp.  Five to eight query tokens run two groups, each taking half of the
// tokens, over one shared stage ring.
__host__ __device__ constexpr int threads_of(int kG) { return (kCWarps * kG + 1) * 32; }
constexpr int kThreads = threads_of(1);
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kLazy = 8.0f;  // log2 headroom before the running max is raised
constexpr int kAlign = 512;    // stage-ring alignment the chunk addressing relies on
// Sequences one launch takes: their host lengths travel in the kernel
// parameters, and larger batches run as consecutive sub-batches.
constexpr int kInlineSeqs = 128;

// The CTA split.  A launch's T tiles, laid end to end in segment order
// (sequence, segment-in-sequence), are cut into G contiguous ranges of equal
// cost: a tile costs 1, and the first tile of each segment costs w more (the
// work of a new piece: staging its query rows, writing its partial).  Every
// segment of sequence s holds ceil(lens[s] / tile_keys) tiles.  The cost of
// tiles [0, x) is C(x) = x + w * (segments starting below x); CTA i starts at
// the smallest x with C(x) >= floor(i * C(T) / G).  w = 0 gives the equal cut
// i * T / G.  With w > 0 the caller ensures T >= G (1 + w), so that
// consecutive cuts differ by at least one tile.  The cut depends only on the
// lengths, never on page size or placement.

// Target cost c falls in sequence s (first tile st, first segment k0, segs
// segments of n tiles) when c <= C(end of s).
__host__ __device__ inline bool cut_falls_in(long long c, long long st, long long k0, long long n, int segs, int w) {
  return c <= st + segs * n + (long long)w * (k0 + segs);
}

// The cut for target c > C(st) inside sequence s: segment j of the sequence
// spans cuts (st + j n, st + (j + 1) n], where C(x) = x + w (k0 + j + 1).
__host__ __device__ inline long long cut_in_sequence(long long c, long long st, long long k0, long long n, int w) {
  const long long j = (c - st - w * k0 + n + w - 1) / (n + w) - 1;
  const long long x = c - w * (k0 + j + 1), lo = st + j * n + 1;
  return x > lo ? x : lo;
}

// First tile of CTA i (walked from the first sequence).
__host__ __device__ inline long long cta_first_tile(const int32_t* lens, int n_seq, int segs, int tile_keys,
                                                    long long T, int G, int w, int i) {
  if (w == 0) return (long long)i * T / G;
  const long long c = (long long)i * (T + (long long)w * n_seq * segs) / G;
  if (c <= 0) return 0;
  long long st = 0, k0 = 0;  // first tile and first segment of sequence s
  for (int s = 0; s < n_seq; ++s) {
    const long long n = (lens[s] + tile_keys - 1) / tile_keys;
    if (cut_falls_in(c, st, k0, n, segs, w)) return cut_in_sequence(c, st, k0, n, w);
    st += segs * n;
    k0 += segs;
  }
  return T;
}

// ------------------------------------------------------------------ stage geometry

// A stage holds four row groups of K then four of V: 16 keys x 4 heads (one
// token) or 64 keys x 1 head (more tokens).
template <int KT, int VT>
struct StageGeo {
  static constexpr int kKGroup = pa_layout::group_bytes<KT>();
  static constexpr int kVGroup = pa_layout::group_bytes<VT>();
  static constexpr int kKBytes = 4 * kKGroup;
  static constexpr int kBytes = 4 * (kKGroup + kVGroup);
  // Every chunk region must start on a multiple of its row's chunk bytes
  // (lane_chunk_offset); the ring base is kAlign-aligned.
  static_assert(kKBytes % kAlign == 0 && kBytes % kAlign == 0, "stage alignment");
  static_assert(kKGroup % Fmt<KT>::kRowQ == 0 && Fmt<KT>::kScales % Fmt<KT>::kRowQ == 0, "K group alignment");
  static_assert(kVGroup % Fmt<VT>::kRowQ == 0 && Fmt<VT>::kScales % Fmt<VT>::kRowQ == 0, "V group alignment");
};

// Shared memory outside the stage ring (kG consumer groups).
constexpr int extras_bytes(int NT, int kG = 1) {
  return (NT == 1 ? kCWarps * (16 * 32 * 8 + 8 * 4 * 16)        // per-warp Q fragments + block corrections
                  : kG * (2 * 16 * NT * 32 * 8                   // Q fragments, double buffered
                          + 2 * 8 * NT * 4 * 16                  // block corrections
                          + 2 * kCWarps * NT * 32 * 8            // P fragments
                          + 2 * kCWarps * NT * 8 * 8))           // tile stats
         + 2 * 8 * 8 + 32;  // barriers (up to 8 stages), misc
}

// CTAs per SM a configuration aims for: two, or one when a stage is large
// or the consumers hold many accumulators.  (Three CTAs of the one-token
// kernel with three stages each stream no faster than two with five, and cut
// a long sequence into half as many pieces again for the merge to read.)
template <int KT, int VT, int NT, int kG = 1>
struct CtaTarget {
  static constexpr int kStageBytes = StageGeo<KT, VT>::kBytes;
  static constexpr int kN = (NT > 3 || kG > 1) ? 1 : (kStageBytes <= 40000 ? 2 : 1);
};

template <int KT, int VT, int NT, int kG = 1>
struct Stages {
  static constexpr int kStageBytes = StageGeo<KT, VT>::kBytes;
  static constexpr int kCtas = CtaTarget<KT, VT, NT, kG>::kN;
  static constexpr int kBudget = (233472 - kCtas * 1024) / kCtas;  // 228 KB per SM, 1 KB reserved per CTA
  static constexpr int kPerCtaMax = kBudget < 232448 ? kBudget : 232448;
  static constexpr int kFit = (kPerCtaMax - extras_bytes(NT, kG) - kAlign) / kStageBytes;
  static constexpr int kN = kFit > 8 ? 8 : kFit;
  static_assert(kN >= 2, "stage ring does not fit");
};

// ------------------------------------------------------------------ dim orders

// Head dim that S-MMA k-step s, k-index j (= 2t + 8h + e) stands for: the
// order in which the K fragment loads deliver a row group's values.
template <int KT>
__device__ __forceinline__ int kdim(int s, int j) {
  const int t = (j & 7) >> 1, e = j & 1, h = j >> 3;
  if (KT == PA_F16) return 16 * s + j;  // chunks 2s, 2s+1 of the row, in order
  const int b = s >> 1, u = s & 1;
  if (KT == PA_Q8_0) return 32 * b + 16 * u + 4 * t + h + 2 * e;  // chunk 2b+u, bytes 4t..4t+3
  return 32 * b + 4 * t + 16 * u + h + 2 * e;  // Q4_0: block b bytes 4t..4t+3, u = 1: high nibbles
}

// Inverse of kdim: k-step and k-index holding dim d; returns t (= lane & 3).
template <int KT>
__device__ __forceinline__ int kdim_inverse(int d, int& ks, int& jj) {
  int t, u, h, e;
  if (KT == PA_F16) {
    ks = d >> 4;
    jj = d & 15;
    return (jj & 7) >> 1;
  } else if (KT == PA_Q8_0) {
    const int b = d >> 5, r = d & 31;
    u = r >> 4; t = (r & 15) >> 2; h = r & 1; e = (r >> 1) & 1;
    ks = 2 * b + u;
  } else {  // Q4_0
    const int b = d >> 5, r = d & 31;
    u = r >> 4; t = (r & 15) >> 2; h = r & 1; e = (r >> 1) & 1;
    ks = 2 * b + u;
  }
  jj = 2 * t + 8 * h + e;
  return t;
}

// Head dim of O^T row g + 8h of m-tile i (0..15): the order in which the V
// fragment loads deliver a row group's values.  The multi-token path gives
// warp w the m-tiles 4w..4w+3.
template <int VT>
__device__ __forceinline__ int vdim(int g, int i, int h) {
  if (VT == PA_F16) return 16 * i + 8 * h + g;
  if (VT == PA_Q8_0) return 32 * (i >> 1) + 16 * (i & 1) + 2 * g + h;
  return 32 * (i >> 1) + 2 * g + (i & 1) + 16 * h;  // Q4_0
}

// ------------------------------------------------------------------ dequant helpers

constexpr uint32_t kHalf2_m1032 = 0xe408e408u;  // -1032.0
constexpr uint32_t kHalf2_m1152 = 0xe480e480u;  // -1152.0
constexpr uint32_t kHalf2_1_16 = 0x2c002c00u;   // 0.0625
constexpr uint32_t kHalf2_m72 = 0xd480d480u;    // -72.0
constexpr uint32_t kMagic64 = 0x64646464u;

// Q4_0 nibbles of x = [c0 c1 c2 c3] -> exact (n - 8) as fp16 pairs:
//   lo0 = (c0.lo, c2.lo)  hi0 = (c0.hi, c2.hi)  lo1 = (c1.lo, c3.lo)  hi1 = (c1.hi, c3.hi)
__device__ __forceinline__ void q4_exact(uint32_t x, uint32_t& lo0, uint32_t& hi0, uint32_t& lo1, uint32_t& hi1) {
  const uint32_t x8 = x >> 8;
  lo0 = hadd2(and_or(x, 0x000f000fu, 0x64006400u), kHalf2_m1032);
  hi0 = hfma2(and_or(x, 0x00f000f0u, 0x64006400u), kHalf2_1_16, kHalf2_m72);
  lo1 = hadd2(and_or(x8, 0x000f000fu, 0x64006400u), kHalf2_m1032);
  hi1 = hfma2(and_or(x8, 0x00f000f0u, 0x64006400u), kHalf2_1_16, kHalf2_m72);
}

// Q8_0 bytes of x = [c0 c1 c2 c3] (already XOR 0x80) -> exact int8 values as
// fp16 pairs: even = (c0, c2), odd = (c1, c3).
__device__ __forceinline__ void q8_exact(uint32_t x, uint32_t& even, uint32_t& odd) {
  even = hadd2(prmt(x, kMagic64, 0x4240), kHalf2_m1152);
  odd = hadd2(prmt(x, kMagic64, 0x4341), kHalf2_m1152);
}

__device__ __forceinline__ float2 half2_bits_to_float2(uint32_t w) {
  return __half22float2(*reinterpret_cast<const __half2*>(&w));
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
  int rows_per_seg;  // query rows per segment: 6 * seg_heads * n_qtok, or a row tile
  int n_row_tiles;   // row tiles per KV head (9 to 96 query tokens), else 0
  float scale_log2;  // scale * log2(e)
  int piece_cost;    // w of cta_first_tile (0: equal tile ranges)
  // The host copy of the lengths (n_seq <= kInlineSeqs).  The tile walk, the
  // table reads and the masks use only these, so nothing the device copy
  // holds can move a read out of a sequence's table row; seq_lens (device) is
  // only compared with them, and a sequence whose two copies differ gives
  // zeros (lse -inf) and PA_ERR_BOUNDS.
  int lens[kInlineSeqs];
};

// Shared-memory layout (byte offsets from the kAlign-aligned base).
template <int KT, int VT, int NT, int kG = 1>
struct Smem {
  static constexpr int kStages = Stages<KT, VT, NT, kG>::kN;
  static constexpr int kKBytes = StageGeo<KT, VT>::kKBytes;
  static constexpr int kStageBytes = StageGeo<KT, VT>::kBytes;
  static constexpr int kRing = kStages * kStageBytes;
  // head-group path: per-warp Q fragments [16][32] uint2, corrections [8][4] float4
  static constexpr int kWQ = kRing;
  static constexpr int kWQBytes = 16 * 32 * 8;
  static constexpr int kWCb = kWQ + kCWarps * kWQBytes;
  static constexpr int kWCbBytes = 8 * 4 * 16;
  // per-head path, per consumer group (group g at + g * kGrpBytes): Q fragments
  // [2][16][NT][32] uint2, corrections [2][8][NT][4] float4, P fragments
  // [2][4][NT][32] uint2, stats [2][4][NT*8] float2
  static constexpr int kQBuf = 16 * NT * 32 * 8;
  static constexpr int kQ = kRing;
  static constexpr int kCbBuf = 8 * NT * 4 * 16;
  static constexpr int kCb = kQ + 2 * kQBuf;
  static constexpr int kP = kCb + 2 * kCbBuf;
  static constexpr int kStat = kP + 2 * kCWarps * NT * 32 * 8;
  static constexpr int kGrpBytes = kStat + 2 * kCWarps * NT * 8 * 8 - kQ;
  static constexpr int kWorkEnd = NT == 1 ? kWCb + kCWarps * kWCbBytes : kQ + kG * kGrpBytes;
  static constexpr int kBar = kWorkEnd;                 // full[kStages], empty[kStages]
  static constexpr int kMisc = kBar + 2 * kStages * 8;  // abort flag, start position, tile range
  static constexpr int kTotal = kMisc + 32;
  static constexpr int kLaunch = kTotal + kAlign;  // dynamic bytes requested (base aligned inside)
};

__device__ __forceinline__ int tiles_of(const DecodeParams& p, int L) { return (L + p.tile_keys - 1) / p.tile_keys; }

// Find the segment holding global tile x: sequence s, segment-in-sequence g
// (KV head, or head group), tile j within it.
__device__ __forceinline__ void locate_tile(const DecodeParams& p, long long x, int& s_out, int& g_out, int& j_out) {
  long long base = 0;
  for (int s = 0; s < p.n_seq; ++s) {
    const long long nt = tiles_of(p, p.lens[s]);
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
    t.L = p.lens[t.s];
    t.nt = tiles_of(p, t.L);
  }
}

// This lane's ldmatrix row address inside a row group's chunk region, for
// the matrix order used throughout: matrix 0 = keys 0-7, chunk c; 1 = keys
// 8-15, chunk c; 2 = keys 0-7, chunk c+1; 3 = keys 8-15, chunk c+1 (c even).
// The address of chunk pair (c, c+1) is then (region + lane_chunk_offset) ^
// (c << 4), because region starts on a multiple of the row's chunk bytes.
template <int T>
__device__ __forceinline__ uint32_t lane_chunk_offset(int lane) {
  const int l7 = lane & 7, key = l7 + 8 * ((lane >> 3) & 1), hi = lane >> 4;
  return (uint32_t)(key * Fmt<T>::kRowQ + ((l7 ^ hi) << 4));
}

// ------------------------------------------------------------------ producers

// Move a tile position k >= 0 tiles forward, across segments; past the last
// sequence it stops at s = n_seq.
__device__ __forceinline__ void advance_tiles(const DecodeParams& p, TilePos& t, long long k) {
  while (k > 0 && t.s < p.n_seq) {
    const long long left = t.nt - t.j;
    if (k < left) {
      t.j += (int)k;
      return;
    }
    k -= left;
    t.j = 0;
    if (++t.g == p.segs_per_seq) {
      t.g = 0;
      if (++t.s < p.n_seq) {
        t.L = p.lens[t.s];
        t.nt = tiles_of(p, t.L);
      }
    }
  }
}

// Pool row (K and V pools alike) of the first slot of head-group tile t for
// the group's first KV head, or -1 when its table entry is outside the pool.
__device__ __forceinline__ long long hg_tile_row(const DecodeParams& p, const TilePos& t) {
  const int k0 = t.j * kTileHG;
  const int tb = __ldg(p.table + (long long)t.s * p.table_stride + k0 / p.page_size);
  if (!(tb >= 0 && tb < p.n_blocks)) return -1;
  return ((long long)tb * p.n_kv_heads + (long long)t.g * p.seg_heads) * p.page_size + k0 % p.page_size;
}

// The producer warp resolves the pool rows of 32 consecutive tiles at once,
// lane l taking tile w0 + l (one table read per lane, issued together), and
// the next 32 a window ahead, so that no tile waits on its table read.
__device__ __forceinline__ long long hg_window(const DecodeParams& p, TilePos t, long long w0, long long b, int lane) {
  advance_tiles(p, t, lane);
  return (w0 + lane < b && t.s < p.n_seq) ? hg_tile_row(p, t) : -1;
}

// Table entry for row group `lane` (0..3) of a per-head tile, -1 past its keys.
__device__ __forceinline__ int head_table_entry(const DecodeParams& p, const TilePos& t, int lane) {
  const int k0 = t.j * kTile, n = min(kTile, t.L - k0);
  if (lane * kGroup >= n) return -1;
  return __ldg(p.table + (long long)t.s * p.table_stride + (k0 + lane * kGroup) / p.page_size);
}

// Wait for every copy still in flight (the last min(issued, stages) stages),
// so that none lands after the CTA retires.
template <int kStages>
__device__ __forceinline__ void drain_ring(const DecodeParams& p, uint32_t bar_full, volatile int* abort, int st,
                                           uint32_t ph, long long issued) {
  const int n_last = (int)(issued < kStages ? issued : kStages);
  for (int k = 1; k <= n_last; ++k) {
    int sst = st - k;
    uint32_t sph = ph;
    if (sst < 0) { sst += kStages; sph ^= 1; }
    mbar_wait(bar_full + 8 * sst, sph, p.err, abort, /*honour_abort=*/false);
  }
}

// Producer for head-group tiles: stage = K [4 heads][row group] then V.  A
// 16-row page whose group covers every KV head is one contiguous run per
// pool; otherwise each head's row group is one run.  Partial last tiles copy
// the whole group (it lies inside the page); the consumers mask the keys past
// the end.
template <int KT, int VT, int NT>
__device__ void produce_hg(const DecodeParams& p, uint32_t ring, uint32_t bar_full, uint32_t bar_empty,
                           volatile int* abort, long long a, long long b, TilePos pos) {
  using G = StageGeo<KT, VT>;
  constexpr int kStages = Stages<KT, VT, NT>::kN;
  constexpr int RK = Fmt<KT>::kRow, RV = Fmt<VT>::kRow;
  const int lane = threadIdx.x & 31;
  const int ps = p.page_size, H = p.n_kv_heads, GH = p.seg_heads;
  const bool whole_blocks = (ps == kGroup) && (GH == H);
  const uint64_t policy = l2_evict_first_policy();
  int st = 0;
  uint32_t ph = 0;
  long long issued = 0;
  // rows of tiles w0 .. w0+31 (this window) and w0+32 .. w0+63 (the next)
  long long w0 = a;
  TilePos wnext = pos;
  advance_tiles(p, wnext, 32);
  long long rows = hg_window(p, pos, w0, b, lane);
  long long rows_next = hg_window(p, wnext, w0 + 32, b, lane);
  for (long long x = a; x < b; ++x) {
    if (*abort) break;
    int k = (int)(x - w0);
    if (k == 32) {
      w0 += 32;
      k = 0;
      rows = rows_next;
      advance_tiles(p, wnext, 32);
      rows_next = hg_window(p, wnext, w0 + 32, b, lane);
    }
    const long long row0 = __shfl_sync(0xffffffffu, rows, k);  // this tile's first row, or -1
    const uint32_t fb = bar_full + 8 * st, eb = bar_empty + 8 * st;
    mbar_wait(eb, ph ^ 1, p.err, abort);  // every lane: no divergent branch
    const uint32_t sk = ring + st * G::kBytes, sv = sk + G::kKBytes;
    if (row0 < 0) {
      // Outside the pool: zero rows for every head of the group, no copy.
      if (lane == 0) record_error(p.err, PA_ERR_BOUNDS);
      for (int i = lane; i < GH * G::kKGroup / 16; i += 32) sts128_zero(sk + 16 * i);
      for (int i = lane; i < GH * G::kVGroup / 16; i += 32) sts128_zero(sv + 16 * i);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(fb);
    } else if (whole_blocks) {
      if (lane == 0) {
        mbar_arrive_expect_tx(fb, (uint32_t)H * (G::kKGroup + G::kVGroup));
        bulk_g2s_hint(sk, p.k_pool + row0 * RK, (uint32_t)H * G::kKGroup, fb, policy);
        bulk_g2s_hint(sv, p.v_pool + row0 * RV, (uint32_t)H * G::kVGroup, fb, policy);
      }
      __syncwarp();
    } else {
      if (lane == 0) mbar_arrive_expect_tx(fb, (uint32_t)GH * (G::kKGroup + G::kVGroup));
      __syncwarp();
      if (lane < GH) {
        const long long row = row0 + (long long)lane * ps;
        bulk_g2s_hint(sk + lane * G::kKGroup, p.k_pool + row * RK, G::kKGroup, fb, policy);
        bulk_g2s_hint(sv + lane * G::kVGroup, p.v_pool + row * RV, G::kVGroup, fb, policy);
      }
      __syncwarp();
    }
    ++issued;
    if (++st == kStages) { st = 0; ph ^= 1; }
  }
  if (lane == 0) drain_ring<kStages>(p, bar_full, abort, st, ph, issued);
}

// Producer for per-head tiles (64 keys = four row groups of one KV head).
// When the page size is a multiple of 64 the tile's groups are one run of one
// page; otherwise each group is its own run.  Groups past the last key are
// not copied (the consumers mask those keys); a group whose table entry is
// outside the pool is zero-filled and reported.
template <int KT, int VT, int NT, int kG>
__device__ void produce_head(const DecodeParams& p, uint32_t ring, uint32_t bar_full, uint32_t bar_empty,
                             volatile int* abort, long long a, long long b, TilePos pos) {
  using G = StageGeo<KT, VT>;
  constexpr int kStages = Stages<KT, VT, NT, kG>::kN;
  constexpr int RK = Fmt<KT>::kRow, RV = Fmt<VT>::kRow;
  const int lane = threadIdx.x & 31;
  const int ps = p.page_size, H = p.n_kv_heads;
  const uint64_t policy = l2_evict_first_policy();
  int st = 0;
  uint32_t ph = 0;
  long long issued = 0;
  int tb = head_table_entry(p, pos, lane), tbn = -1;
  for (long long x = a; x < b; ++x) {
    if (*abort) break;
    TilePos nxt = pos;
    if (x + 1 < b) {
      next_tile(p, nxt);
      tbn = head_table_entry(p, nxt, lane);
    }
    const uint32_t fb = bar_full + 8 * st, eb = bar_empty + 8 * st;
    const int k0 = pos.j * kTile, n = min(kTile, pos.L - k0), ng = (n + kGroup - 1) / kGroup;
    const bool mine = lane < ng;
    const bool ok = !mine || (tb >= 0 && tb < p.n_blocks);
    const unsigned bad = __ballot_sync(0xffffffffu, !ok);
    mbar_wait(eb, ph ^ 1, p.err, abort);  // every lane: no divergent branch
    const uint32_t sk = ring + st * G::kBytes, sv = sk + G::kKBytes;
    if (bad == 0 && ps % kTile == 0) {
      if (lane == 0) {
        const long long row = ((long long)tb * H + pos.g) * ps + k0 % ps;
        mbar_arrive_expect_tx(fb, (uint32_t)ng * (G::kKGroup + G::kVGroup));
        bulk_g2s_hint(sk, p.k_pool + row * RK, (uint32_t)ng * G::kKGroup, fb, policy);
        bulk_g2s_hint(sv, p.v_pool + row * RV, (uint32_t)ng * G::kVGroup, fb, policy);
      }
      __syncwarp();
    } else {
      if (bad) {
        if (lane == 0) record_error(p.err, PA_ERR_BOUNDS);
        for (int q = 0; q < 4; ++q) {
          if (!((bad >> q) & 1)) continue;
          for (int i = lane; i < G::kKGroup / 16; i += 32) sts128_zero(sk + q * G::kKGroup + 16 * i);
          for (int i = lane; i < G::kVGroup / 16; i += 32) sts128_zero(sv + q * G::kVGroup + 16 * i);
        }
        fence_proxy_async_smem();
      }
      const int n_good = __popc(__ballot_sync(0xffffffffu, mine && ok));
      if (lane == 0) mbar_arrive_expect_tx(fb, (uint32_t)n_good * (G::kKGroup + G::kVGroup));
      __syncwarp();
      if (mine && ok) {
        const long long row = ((long long)tb * H + pos.g) * ps + (k0 + lane * kGroup) % ps;
        bulk_g2s_hint(sk + lane * G::kKGroup, p.k_pool + row * RK, G::kKGroup, fb, policy);
        bulk_g2s_hint(sv + lane * G::kVGroup, p.v_pool + row * RV, G::kVGroup, fb, policy);
      }
      __syncwarp();
    }
    ++issued;
    if (++st == kStages) { st = 0; ph ^= 1; }
    pos = nxt;
    tb = tbn;
  }
  if (lane == 0) drain_ring<kStages>(p, bar_full, abort, st, ph, issued);
}

// ------------------------------------------------------------------ Q staging

// Block bias entry layout shared by both paths: for (block, n-tile, t) one
// float4 {-c[2t], -c[2t+1], -c[2t], -c[2t+1]} over the n-tile's rows, which is
// the MMA accumulator a block starts from (rows g and g+8 of S^T are keys).
// c = 1032 * (sum of the block's low-half fp16 Q) + 1152 * (sum of its
// high-half fp16 Q/16) for Q4_0, 1152 * (sum of its fp16 Q) for Q8_0: the
// magic bias the raw K halves carry, times Q.

// Q fragments are stored two k-steps at a time: entry (k-step pair kp, n-tile
// nt, lane) is a uint4 {b0, b1 of k-step 2kp, b0, b1 of k-step 2kp+1} at byte
// ((kp * NT + nt) * 32 + lane) * 16, so one 16-byte load feeds a block's two
// MMAs.

// One Q fragment entry: what lane (g, t) holds of k-steps 2kp and 2kp+1 as
// S-MMA B fragments (query row g), in the K format's dim order (kdim).  Quantised K:
// v0 = dims 32 kp + 4t .. +3 (the block's low half), v1 = the same + 16 (its
// high half, met as Q/16 by Q4_0's high nibbles); the entry is {(v0.x, v0.z),
// (v0.y, v0.w), (v1.x, v1.z), (v1.y, v1.w)} in binary16, and lo / hi return
// the fp32 sums, in dim order, of each half's binary16 values (the block bias
// terms).  F16 K: v0 = dims 32 kp + 2t, +1, +8, +9 and v1 the same + 16, in
// order.
template <int KT>
__device__ __forceinline__ uint4 q_entry(float4 v0, float4 v1, float& lo, float& hi) {
  if constexpr (KT == PA_F16) {
    lo = hi = 0.f;
    return make_uint4(pack_half2(v0.x, v0.y), pack_half2(v0.z, v0.w), pack_half2(v1.x, v1.y),
                      pack_half2(v1.z, v1.w));
  } else {
    constexpr float sc = KT == PA_Q4_0 ? 0.0625f : 1.f;
    const uint32_t b0 = pack_half2(v0.x, v0.z), b1 = pack_half2(v0.y, v0.w);
    const uint32_t b2 = pack_half2(sc * v1.x, sc * v1.z), b3 = pack_half2(sc * v1.y, sc * v1.w);
    const float2 f0 = half2_bits_to_float2(b0), f1 = half2_bits_to_float2(b1);
    const float2 f2 = half2_bits_to_float2(b2), f3 = half2_bits_to_float2(b3);
    lo = 0.f;
    lo += f0.x;
    lo += f1.x;
    lo += f0.y;
    lo += f1.y;
    hi = 0.f;
    hi += f2.x;
    hi += f3.x;
    hi += f2.y;
    hi += f3.y;
    return make_uint4(b0, b1, b2, b3);
  }
}

// The two loads of one entry (see q_entry) from query row qr (fp32, kD values).
template <int KT>
__device__ __forceinline__ void q_entry_load(const float* qr, int kp, int t, float4& v0, float4& v1) {
  if constexpr (KT == PA_F16) {
    const float* r = qr + 32 * kp + 2 * t;
    const float2 a = __ldg(reinterpret_cast<const float2*>(r)), b = __ldg(reinterpret_cast<const float2*>(r + 8));
    const float2 c = __ldg(reinterpret_cast<const float2*>(r + 16)), d = __ldg(reinterpret_cast<const float2*>(r + 24));
    v0 = make_float4(a.x, a.y, b.x, b.y);
    v1 = make_float4(c.x, c.y, d.x, d.y);
  } else {
    const float* r = qr + 32 * kp + 4 * t;
    v0 = __ldg(reinterpret_cast<const float4*>(r));
    v1 = __ldg(reinterpret_cast<const float4*>(r + 16));
  }
}

// Block bias of a quantised K format from the quad-reduced halves: the magic
// bias the raw K halves carry, times Q.
template <int KT>
__device__ __forceinline__ float q_block_bias(float lo, float hi) {
  return (KT == PA_Q4_0) ? 1032.f * lo + 1152.f * hi : 1152.f * (lo + hi);
}

// Head-group path: warp w stages its own KV head's six query rows (one query
// token) as S-MMA B fragments and the block biases ([block][t] float4), from
// coalesced float4 loads.  Rows 6 and 7 of the fragment (padding) are zero.
// Only this warp reads them.
template <int KT>
__device__ __noinline__ void stage_q_warp(const DecodeParams& p, int s, int head, uint32_t qf, float* cb4, int lane) {
  // zero the padding rows 6, 7 (lanes 24..31 of every k-step) and their biases
  if (lane >= 24) {
#pragma unroll
    for (int kp = 0; kp < 8; ++kp) sts128_zero(qf + (kp * 32 + lane) * 16);
  }
  if (KT != PA_F16 && lane < 8) sts128_zero(smem_u32(cb4 + (lane * 4 + 3) * 4));
  const float4* q4 = reinterpret_cast<const float4*>(p.q + ((long long)s * p.n_q_heads + head * kGqa) * kD);
  // All twelve loads first: they are in flight together (one round trip,
  // not one per batch), which matters while the bulk copies load HBM.
  constexpr int kLoads = kGqa * kD / 4 / 32;  // 12 float4 per lane
  float4 qv[kLoads];
#pragma unroll
  for (int i = 0; i < kLoads; ++i) qv[i] = __ldg(q4 + lane + 32 * i);
#pragma unroll
  for (int i = 0; i < kLoads; ++i) {
    const int f = lane + 32 * i;
    const int row = f >> 6, d0 = 4 * (f & 63);
    const float vals[4] = {qv[i].x, qv[i].y, qv[i].z, qv[i].w};
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
      const uint32_t addr = qf + ((ks >> 1) * 32 + ln) * 16 + (ks & 1) * 8 + ((jj >> 3) << 2) + ((jj & 1) << 1);
      asm volatile("st.shared.b16 [%0], %1;" ::"r"(addr), "h"(__half_as_ushort(hv)) : "memory");
    }
    if (KT != PA_F16) {
      // lanes 8b'..8b'+7 hold the 8 float4 of block 4(i&1)+b' of row i/2:
      // k < 4 low 16 dims, k >= 4 high 16 dims.
      lo += __shfl_xor_sync(0xffffffffu, lo, 1);
      lo += __shfl_xor_sync(0xffffffffu, lo, 2);
      const float hi = __shfl_down_sync(0xffffffffu, lo, 4);
      if ((lane & 7) == 0) {
        const int blk = 4 * (i & 1) + (lane >> 3), r = i >> 1;
        const float c = (KT == PA_Q4_0) ? 1032.f * lo + 1152.f * hi : 1152.f * (lo + hi);
        float* e = cb4 + (blk * 4 + (r >> 1)) * 4 + (r & 1);
        e[0] = -c;
        e[2] = -c;
      }
    }
  }
  __syncwarp();
}

__device__ __forceinline__ const float* q_row(const DecodeParams& p, int s, int g, int row) {
  const int tq = row / kGqa, hl = row % kGqa;
  return p.q + (((long long)s * p.n_qtok + tq) * p.n_q_heads + g * kGqa + hl) * kD;
}


// Per-head path: stage Q of (sequence s, KV head g) as S-MMA B fragments in
// the K format's dim order (high-nibble Q4_0 k-steps hold Q/16) and, for
// quantised K, the block biases ([block][nt][t] float4).  The 128 threads of
// one consumer group (tid 0..127) take part: thread tid builds fragment
// entries tid + 128 i, i.e. (k-step pair, n-tile) warp + 4 i, lane (g, t):
// query row nt * 8 + g of the R rows from segment row row0 on (rows R ..
// 8*NT-1 are zero), all of its loads in flight at once.
template <int KT, int NT>
__device__ __noinline__ void stage_q(const DecodeParams& p, int s, int g, uint32_t qf, float* cb4, int tid, int row0,
                                     int R) {
  constexpr int kE = 8 * NT * 32 / (kCWarps * 32);  // entries per thread
  const int lane = tid & 31, t = lane & 3, gq = lane >> 2, warp = tid >> 5;
  float4 v0[kE], v1[kE];
#pragma unroll
  for (int i = 0; i < kE; ++i) {
    const int q = warp + kCWarps * i, kp = q / NT, row = (q % NT) * 8 + gq;
    if (row < R) {
      q_entry_load<KT>(q_row(p, s, g, row0 + row), kp, t, v0[i], v1[i]);
    } else {
      v0[i] = make_float4(0.f, 0.f, 0.f, 0.f);
      v1[i] = v0[i];
    }
  }
#pragma unroll
  for (int i = 0; i < kE; ++i) {
    const int q = warp + kCWarps * i, kp = q / NT, nt = q % NT, row = nt * 8 + gq;
    float lo, hi;
    sts128(qf + (q * 32 + lane) * 16, q_entry<KT>(v0[i], v1[i], lo, hi));
    if constexpr (KT != PA_F16) {
      lo += __shfl_xor_sync(0xffffffffu, lo, 1);
      lo += __shfl_xor_sync(0xffffffffu, lo, 2);
      hi += __shfl_xor_sync(0xffffffffu, hi, 1);
      hi += __shfl_xor_sync(0xffffffffu, hi, 2);
      if (t == 0) {
        const float c = row < R ? -q_block_bias<KT>(lo, hi) : 0.f;
        float* e = cb4 + ((kp * NT + nt) * 4 + (gq >> 1)) * 4 + (gq & 1);
        e[0] = c;
        e[2] = c;
      }
    }
  }
}

// ------------------------------------------------------------------ S phase (K side)

// acc[nt] += S^T for the 16 keys of one K row group (rows = keys g, g+8)
// against the staged Q fragments, over all 256 dims.  kq: this lane's
// ldmatrix address in the group's chunk region (lane_chunk_offset); ksc: the
// group's scale region; qf: this lane's Q fragments (base + 16 * lane); cbl:
// this lane's block bias entries (t = lane & 3).
template <int KT, int NT>
__device__ __forceinline__ void s_phase(float (&acc)[NT][4], uint32_t kq, uint32_t ksc, uint32_t qf, uint32_t cbl,
                                        int lane) {
  if constexpr (KT == PA_F16) {
#pragma unroll
    for (int kp = 0; kp < 8; ++kp) {
      uint32_t a0[4], a1[4];
      ldsm_x4(kq ^ ((4 * kp) << 4), a0);
      ldsm_x4(kq ^ ((4 * kp + 2) << 4), a1);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const uint4 q = lds128(qf + (kp * NT + nt) * 512);
        mma_16816(acc[nt], a0, q.x, q.y);
        mma_16816(acc[nt], a1, q.z, q.w);
      }
    }
  } else {
    const int g = lane >> 2;
    const uint4 dg = lds128(ksc + 16 * g), dg8 = lds128(ksc + 16 * (g + 8));  // scales of keys g, g+8
    const uint32_t dgw[4] = {dg.x, dg.y, dg.z, dg.w}, dg8w[4] = {dg8.x, dg8.y, dg8.z, dg8.w};
#pragma unroll
    for (int bp = 0; bp < 4; ++bp) {  // block pair 2bp, 2bp+1
      const float2 dA = half2_bits_to_float2(dgw[bp]), dB = half2_bits_to_float2(dg8w[bp]);
      uint32_t x4[4];  // Q4_0: both blocks of the pair
      if constexpr (KT == PA_Q4_0) ldsm_x4(kq ^ ((2 * bp) << 4), x4);
#pragma unroll
      for (int hb = 0; hb < 2; ++hb) {
        const int b = 2 * bp + hb;
        uint32_t a0[4], a1[4];  // k-steps 2b, 2b+1
        if constexpr (KT == PA_Q4_0) {
          const uint32_t x0 = x4[2 * hb], x1 = x4[2 * hb + 1];  // keys g, g+8: bytes 4t..4t+3 of block b
          const uint32_t y0 = x0 >> 8, y1 = x1 >> 8;
          a0[0] = and_or(x0, 0x000f000fu, 0x64006400u);
          a0[1] = and_or(x1, 0x000f000fu, 0x64006400u);
          a0[2] = and_or(y0, 0x000f000fu, 0x64006400u);
          a0[3] = and_or(y1, 0x000f000fu, 0x64006400u);
          a1[0] = and_or(x0, 0x00f000f0u, 0x64006400u);
          a1[1] = and_or(x1, 0x00f000f0u, 0x64006400u);
          a1[2] = and_or(y0, 0x00f000f0u, 0x64006400u);
          a1[3] = and_or(y1, 0x00f000f0u, 0x64006400u);
        } else {  // Q8_0: chunks 2b (k-step 2b) and 2b+1; byte x -> 1024 + (x + 128)
          uint32_t y[4];
          ldsm_x4(kq ^ ((2 * b) << 4), y);  // key g / g+8 of chunk 2b, then of chunk 2b+1
#pragma unroll
          for (int k = 0; k < 4; ++k) y[k] ^= 0x80808080u;
          a0[0] = prmt(y[0], kMagic64, 0x4240);
          a0[1] = prmt(y[1], kMagic64, 0x4240);
          a0[2] = prmt(y[0], kMagic64, 0x4341);
          a0[3] = prmt(y[1], kMagic64, 0x4341);
          a1[0] = prmt(y[2], kMagic64, 0x4240);
          a1[1] = prmt(y[3], kMagic64, 0x4240);
          a1[2] = prmt(y[2], kMagic64, 0x4341);
          a1[3] = prmt(y[3], kMagic64, 0x4341);
        }
        const float d0 = hb ? dA.y : dA.x, d1 = hb ? dB.y : dB.x;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const float4 c = lds128f(cbl + (b * NT + nt) * 64);
          float tmp[4] = {c.x, c.y, c.z, c.w};
          const uint4 q = lds128(qf + (b * NT + nt) * 512);
          if constexpr (NT >= 4) {
            // One CTA per SM has the registers for two independent MMA
            // chains per block (measured faster there, neutral below).
            float tm2[4] = {0.f, 0.f, 0.f, 0.f};
            mma_16816(tmp, a0, q.x, q.y);
            mma_16816(tm2, a1, q.z, q.w);
#pragma unroll
            for (int e = 0; e < 4; ++e) tmp[e] += tm2[e];
          } else {
            mma_16816(tmp, a0, q.x, q.y);
            mma_16816(tmp, a1, q.z, q.w);
          }
          acc[nt][0] = fmaf(d0, tmp[0], acc[nt][0]);
          acc[nt][1] = fmaf(d0, tmp[1], acc[nt][1]);
          acc[nt][2] = fmaf(d1, tmp[2], acc[nt][2]);
          acc[nt][3] = fmaf(d1, tmp[3], acc[nt][3]);
        }
      }
    }
  }
}

// ------------------------------------------------------------------ PV, one-token path

// o[i] (16 m-tiles, all 256 dims) += V^T (the 16 keys of one V row group) x
// P^T.  vq: this lane's ldmatrix address in the group's chunk region; vsc:
// the group's scale region; bp0 / bp1: P B fragments (keys 2t, 2t+1 / 2t+8,
// 2t+9 of the group; query row g).  The V block scale is folded into P.
template <int VT>
__device__ __forceinline__ void pv_solo(float (&o)[16][4], uint32_t vq, uint32_t vsc, int lane, uint32_t bp0,
                                        uint32_t bp1) {
  const int t = lane & 3;
  if constexpr (VT == PA_F16) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {  // dims 16i .. 16i+15 = chunks 2i, 2i+1
      uint32_t r[4];
      ldsm_x4_trans(vq ^ ((2 * i) << 4), r);
      const uint32_t a[4] = {r[0], r[2], r[1], r[3]};
      mma_16816(o[i], a, bp0, bp1);
    }
  } else if constexpr (VT == PA_Q4_0) {
#pragma unroll
    for (int bp = 0; bp < 4; ++bp) {  // blocks 2bp, 2bp+1
      uint32_t x[4];  // keys (2t, 2t+1) / (2t+8, 2t+9), byte pair g, of block 2bp then 2bp+1
      ldsm_x4_trans(vq ^ ((2 * bp) << 4), x);
      const uint4 D = lds128(vsc + 64 * bp + 16 * t);  // the same key pairs' scales
#pragma unroll
      for (int hb = 0; hb < 2; ++hb) {
        const int b = 2 * bp + hb;
        uint32_t la0, ha0, la1, ha1, lc0, hc0, lc1, hc1;
        q4_exact(x[2 * hb], la0, ha0, la1, ha1);      // dims 2g, 2g+16, 2g+1, 2g+17
        q4_exact(x[2 * hb + 1], lc0, hc0, lc1, hc1);
        const uint32_t p0 = hmul2(bp0, hb ? D.z : D.x), p1 = hmul2(bp1, hb ? D.w : D.y);
        const uint32_t A0[4] = {la0, ha0, lc0, hc0}, A1[4] = {la1, ha1, lc1, hc1};
        mma_16816(o[2 * b], A0, p0, p1);
        mma_16816(o[2 * b + 1], A1, p0, p1);
      }
    }
  } else {  // Q8_0: m-tile i = chunk i (16 quants of block i/2)
#pragma unroll
    for (int bp = 0; bp < 4; ++bp) {
      const uint4 D = lds128(vsc + 64 * bp + 16 * t);
#pragma unroll
      for (int hb = 0; hb < 2; ++hb) {
        const int b = 2 * bp + hb;
        uint32_t x[4];
        ldsm_x4_trans(vq ^ ((2 * b) << 4), x);
        const uint32_t p0 = hmul2(bp0, hb ? D.z : D.x), p1 = hmul2(bp1, hb ? D.w : D.y);
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t ea, oa, ec, oc;
          q8_exact(x[2 * c] ^ 0x80808080u, ea, oa);
          q8_exact(x[2 * c + 1] ^ 0x80808080u, ec, oc);
          const uint32_t A[4] = {ea, oa, ec, oc};
          mma_16816(o[2 * b + c], A, p0, p1);
        }
      }
    }
  }
}

// ------------------------------------------------------------------ PV, multi-token path

// o[i][nt] += V^T(m-tile 4w + i; the 16 keys of one V row group) x P^T.
template <int VT, int NT>
__device__ __forceinline__ void pv_kstep(float (&o)[4][NT][4], uint32_t vq, uint32_t vsc, int w, int lane,
                                         const uint32_t (&bp)[NT][2]) {
  const int t = lane & 3;
  if constexpr (VT == PA_F16) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint32_t r[4];
      ldsm_x4_trans(vq ^ ((2 * (4 * w + i)) << 4), r);
      const uint32_t a[4] = {r[0], r[2], r[1], r[3]};
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) mma_16816(o[i][nt], a, bp[nt][0], bp[nt][1]);
    }
  } else {
    const uint4 D = lds128(vsc + 64 * w + 16 * t);  // blocks 2w, 2w+1
    if constexpr (VT == PA_Q4_0) {
      uint32_t x[4];
      ldsm_x4_trans(vq ^ ((2 * w) << 4), x);
#pragma unroll
      for (int hb = 0; hb < 2; ++hb) {
        uint32_t la0, ha0, la1, ha1, lc0, hc0, lc1, hc1;
        q4_exact(x[2 * hb], la0, ha0, la1, ha1);
        q4_exact(x[2 * hb + 1], lc0, hc0, lc1, hc1);
        const uint32_t A0[4] = {la0, ha0, lc0, hc0}, A1[4] = {la1, ha1, lc1, hc1};
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const uint32_t p0 = hmul2(bp[nt][0], hb ? D.z : D.x), p1 = hmul2(bp[nt][1], hb ? D.w : D.y);
          mma_16816(o[2 * hb][nt], A0, p0, p1);
          mma_16816(o[2 * hb + 1][nt], A1, p0, p1);
        }
      }
    } else {  // Q8_0: chunks 4w .. 4w+3
#pragma unroll
      for (int hb = 0; hb < 2; ++hb) {
        uint32_t x[4];
        ldsm_x4_trans(vq ^ ((2 * (2 * w + hb)) << 4), x);
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t ea, oa, ec, oc;
          q8_exact(x[2 * c] ^ 0x80808080u, ea, oa);
          q8_exact(x[2 * c + 1] ^ 0x80808080u, ec, oc);
          const uint32_t A[4] = {ea, oa, ec, oc};
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            const uint32_t p0 = hmul2(bp[nt][0], hb ? D.z : D.x), p1 = hmul2(bp[nt][1], hb ? D.w : D.y);
            mma_16816(o[2 * hb + c][nt], A, p0, p1);
          }
        }
      }
    }
  }
}

// ------------------------------------------------------------------ keys past the end

// The rows of a tile past the sequence's last key hold whatever the pool or
// the stage held before (a partly written page, an earlier tile, or nothing).
// Their P is exactly 0, so V only has to be finite: a consumer zeroes, before
// reading them, the V bytes of those keys that it is about to read -- the
// block scales of quantised V (the quants of any byte pattern are finite) or
// the F16 values.  The stage is later refilled by the async proxy, hence the
// proxy fence.

// One V row group, all dims, keys n..15 (head-group path).
template <int VT>
__device__ __forceinline__ void zero_tail_group(uint32_t vg, int n, int lane) {
  if constexpr (VT == PA_F16) {
    for (int i = lane; i < (kGroup - n) * (Fmt<PA_F16>::kRowQ / 16); i += 32)
      sts128_zero(vg + n * Fmt<PA_F16>::kRowQ + 16 * i);
  } else {
    for (int i = lane; i < (kGroup - n) * 8; i += 32)
      sts16_zero(vg + pa_layout::v_scale_offset(n + (i >> 3), i & 7));
  }
  fence_proxy_async_smem();
  __syncwarp();
}

// Four V row groups (64 keys), keys n..63, the dims of warp w's m-tiles
// (blocks 2w, 2w+1) (per-head path).
template <int VT>
__device__ __forceinline__ void zero_tail_tile(uint32_t vstage, int n, int w, int lane) {
  constexpr int VG = pa_layout::group_bytes<VT>();
  for (int i = lane; i < (kTile - n) * 2; i += 32) {
    const int key = n + (i >> 1), hb = i & 1;
    const uint32_t vg = vstage + (key / kGroup) * VG;
    const int r = key % kGroup;
    if constexpr (VT == PA_F16) {
#pragma unroll
      for (int c = 0; c < 4; ++c)  // chunks 8w + 4hb .. +3
        sts128_zero(vg + pa_layout::chunk_offset(0, Fmt<PA_F16>::kRowQ, r, 8 * w + 4 * hb + c));
    } else {
      sts16_zero(vg + pa_layout::v_scale_offset(r, 2 * w + hb));
    }
  }
  fence_proxy_async_smem();
  __syncwarp();
}

// ------------------------------------------------------------------ device lengths

// The device copy of sequence s's length, read past L1 (the caller may have
// written it just before the launch).  Issued when a piece starts and checked
// when it ends, so its latency hides behind the piece's tiles.
__device__ __forceinline__ int device_len(const DecodeParams& p, int s) { return __ldcg(p.seq_lens + s); }

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
// Only warps w < GH run this (the empty barriers count GH arrivals).
template <int KT, int VT>
__device__ void consume_hg(const DecodeParams& p, uint8_t* smem, uint32_t ring, uint32_t bar_full,
                           uint32_t bar_empty, volatile int* abort, long long a, long long b, int s, int g, int j) {
  using SM = Smem<KT, VT, 1>;
  using G = StageGeo<KT, VT>;
  constexpr int kStages = SM::kStages;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gq = lane >> 2, tq = lane & 3;
  const uint32_t qf = ring + SM::kWQ + warp * SM::kWQBytes;
  float* cb4 = reinterpret_cast<float*>(smem + SM::kWCb + warp * SM::kWCbBytes);
  const uint32_t qf_lane = qf + lane * 16;
  const uint32_t cb_lane = smem_u32(cb4) + 16 * tq;
  // This warp's K and V row groups in stage 0, and its lanes' fragment addresses.
  const uint32_t kg0 = ring + warp * G::kKGroup, vg0 = ring + G::kKBytes + warp * G::kVGroup;
  const uint32_t kq0 = kg0 + Fmt<KT>::kScales + lane_chunk_offset<KT>(lane);
  const uint32_t vq0 = vg0 + Fmt<VT>::kScales + lane_chunk_offset<VT>(lane);
  const float scale_log2 = p.scale_log2;
  int st = 0;
  uint32_t ph = 0;
  long long x = a;
  while (x < b) {
    const int L = p.lens[s];
    const int l_dev = device_len(p, s);
    const int ntl = tiles_of(p, L);
    const int jb = j, je = (int)((long long)ntl < j + (b - x) ? (long long)ntl : j + (b - x));
    const int seg = s * p.segs_per_seq + g;
    const bool whole = (jb == 0 && je == ntl);
    const int head = g * p.seg_heads + warp;
    stage_q_warp<KT>(p, s, head, qf, cb4, lane);

    float o[16][4];
#pragma unroll
    for (int i = 0; i < 16; ++i)
#pragma unroll
      for (int c = 0; c < 4; ++c) o[i][c] = 0.f;
    float mref0 = -INFINITY, mref1 = -INFINITY;  // rows 2tq, 2tq+1
    float ls0 = 0.f, ls1 = 0.f;                  // this thread's share of the row sums

    // One tile; kMask: the sequence's partial last tile (keys >= L masked).
    auto tile = [&](auto mask_tag, int jt) {
      constexpr bool kMask = decltype(mask_tag)::value;
      mbar_wait(bar_full + 8 * st, ph, p.err, abort);
      const uint32_t so = st * SM::kStageBytes;
      const int n = L - jt * kTileHG;  // keys of this tile that exist (< 16 only when masked)
      if (kMask) zero_tail_group<VT>(vg0 + so, n, lane);
      float sacc[1][4] = {{0.f, 0.f, 0.f, 0.f}};
      s_phase<KT, 1>(sacc, kq0 + so, kg0 + so, qf_lane, cb_lane, lane);
      float xv[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        xv[c] = sacc[0][c] * scale_log2;
        if (kMask && gq + ((c & 2) ? 8 : 0) >= n) xv[c] = -INFINITY;
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
        const float al0 = (mn0 == -INFINITY) ? 1.f : ex2(mref0 - mn0);
        const float al1 = (mn1 == -INFINITY) ? 1.f : ex2(mref1 - mn1);
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
      const uint32_t X0 = pack_half2(ex2(xv[0] - b0), ex2(xv[1] - b1));  // key gq: rows 2tq, 2tq+1
      const uint32_t X1 = pack_half2(ex2(xv[2] - b0), ex2(xv[3] - b1));  // key gq+8
      {
        const float2 f0 = half2_bits_to_float2(X0), f1 = half2_bits_to_float2(X1);
        ls0 += f0.x + f1.x;
        ls1 += f0.y + f1.y;
      }
      const uint32_t B0 = movmatrix_trans(X0), B1 = movmatrix_trans(X1);
      pv_solo<VT>(o, vq0 + so, vg0 + so, lane, B0, B1);
      __syncwarp();
      mbar_arrive_warp(bar_empty + 8 * st);
      if (++st == kStages) { st = 0; ph ^= 1; }
    };
    // Every tile but a partial last one runs unmasked.
    const int je_full = (je == ntl && (L % kTileHG) != 0) ? je - 1 : je;
    for (int jt = jb; jt < je_full; ++jt) tile(std::false_type{}, jt);
    if (je_full < je) tile(std::true_type{}, je_full);

    // ---- piece result for this warp's head: rows 2tq, 2tq+1 (< 6)
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      ls0 += __shfl_xor_sync(0xffffffffu, ls0, off);
      ls1 += __shfl_xor_sync(0xffffffffu, ls1, off);
    }
    // A device length that differs from the host's: the piece counts for
    // nothing (zeros, l = 0) and the mismatch is reported.
    const float keep = (l_dev == L) ? 1.f : 0.f;
    if (l_dev != L) {
      if (lane == 0) record_error(p.err, PA_ERR_BOUNDS);
      ls0 = 0.f;
      ls1 = 0.f;
    }
    const int slot = (int)blockIdx.x + seg;
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const int hl = 2 * tq + c;
      if (hl >= kGqa) continue;
      const float lr = c ? ls1 : ls0, mr = c ? mref1 : mref0;
      const int row = warp * kGqa + hl;  // row within the segment
      float* dst;
      float inv = keep;
      if (whole) {
        dst = p.out + ((long long)s * p.n_q_heads + head * kGqa + hl) * kD;
        inv = lr > 0.f ? 1.f / lr : 0.f;
      } else {
        dst = p.part_o + ((long long)slot * p.rows_per_seg + row) * kD;
      }
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        dst[vdim<VT>(gq, i, 0)] = o[i][c] * inv;
        dst[vdim<VT>(gq, i, 1)] = o[i][2 + c] * inv;
      }
      if (gq == 0) {
        if (whole) {
          if (p.lse)
            p.lse[(long long)s * p.n_q_heads + head * kGqa + hl] = lr > 0.f ? (mr + log2f(lr)) * kLn2 : -INFINITY;
        } else {
          p.part_ml[(long long)slot * p.rows_per_seg + row] = make_float2(mr, lr);
        }
      }
    }

    x += je - jb;
    j = 0;
    if (++g == p.segs_per_seq) { g = 0; ++s; }
  }
}

// ------------------------------------------------------------------ per-head consumer

// Multi-token path (NT = 2 to 4 n-tiles; with kG = 2 groups, each group of
// four warps runs this for its half of the query tokens): see the file
// comment.  The four warps of a group share one reference maximum per query
// row (m_ref), so in the common case a tile needs one barrier and no
// rescaling: each warp computes P for its 16 keys against m_ref and publishes
// it.  A warp whose logits exceed m_ref by more than 2^8 raises a flag and
// publishes its per-row base; then (rarely) a second barrier lets every warp
// form the new maximum, rescale O and its row sums, and scale each warp's P by
// 2^(base - new).  Row sums are kept per thread over its own keys and reduced
// once at the end of the piece.
template <int KT, int VT, int NT, int kG>
__device__ void consume_shared(const DecodeParams& p, uint8_t* smem, uint32_t ring, uint32_t bar_full,
                               uint32_t bar_empty, volatile int* abort, long long a, long long b, int s, int g,
                               int j, int grp) {
  using SM = Smem<KT, VT, NT, kG>;
  using G = StageGeo<KT, VT>;
  constexpr int kStages = SM::kStages;
  constexpr int R8 = NT * 8;
  // This group's warps, its query tokens [tok0, tok0 + ntok) and its rows
  // [row0, row0 + R) of the segment's Rg rows; its own shared memory and
  // named barrier.
  const int tid = threadIdx.x & (kCWarps * 32 - 1), warp = tid >> 5, lane = tid & 31;
  const int gq = lane >> 2, tq = lane & 3;
  const int ntok0 = (p.n_qtok + kG - 1) / kG;
  const int tok0 = grp * ntok0, ntok = grp == 0 ? ntok0 : p.n_qtok - ntok0;
  const int R = kGqa * ntok, row0 = kGqa * tok0, Rg = kGqa * p.n_qtok;
  const uint32_t bar_id = 1 + grp;
  const int goff = grp * SM::kGrpBytes;
  const uint32_t pb_base = ring + SM::kP + goff;
  float* mbase = reinterpret_cast<float*>(smem + SM::kStat + goff);             // [2][warp][R8] per-row P base
  int* flags = reinterpret_cast<int*>(smem + SM::kStat + goff + 2 * kCWarps * R8 * 4);  // [2][warp]
  // K row group `warp` and V row group 0 of stage 0, with this lane's offsets.
  const uint32_t kg0 = ring + warp * G::kKGroup, vs0 = ring + G::kKBytes;
  const uint32_t kq0 = kg0 + Fmt<KT>::kScales + lane_chunk_offset<KT>(lane);
  const uint32_t vq_off = Fmt<VT>::kScales + lane_chunk_offset<VT>(lane);
  const float scale_log2 = p.scale_log2;
  int st = 0;
  uint32_t ph = 0;
  int qbuf = 0, tbuf = 0;
  long long x = a;
  while (x < b) {
    const int L = p.lens[s];
    const int l_dev = device_len(p, s);
    const int ntl = tiles_of(p, L);
    const int jb = j, je = (int)((long long)ntl < j + (b - x) ? (long long)ntl : j + (b - x));
    const int seg = s * p.segs_per_seq + g;
    const bool whole = (jb == 0 && je == ntl);
    const uint32_t qf = ring + SM::kQ + goff + qbuf * SM::kQBuf;
    float* cb4 = reinterpret_cast<float*>(smem + SM::kCb + goff + qbuf * SM::kCbBuf);
    stage_q<KT, NT>(p, s, g, qf, cb4, tid, row0, R);
    named_bar_sync(bar_id, kCWarps * 32);
    const uint32_t qf_lane = qf + lane * 16;
    const uint32_t cb_lane = smem_u32(cb4) + 16 * tq;

    float o[4][NT][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int c = 0; c < 4; ++c) o[i][nt][c] = 0.f;
    float m_ref[NT][2], l_part[NT][2];  // rows nt*8 + 2tq + e; l over this thread's keys only
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) { m_ref[nt][e] = -INFINITY; l_part[nt][e] = 0.f; }

    const int vis0 = L - p.n_qtok + tok0;  // last key visible to this group's first token
    for (int jt = jb; jt < je; ++jt) {
      mbar_wait(bar_full + 8 * st, ph, p.err, abort);
      const uint32_t so = st * SM::kStageBytes;
      const int k0 = jt * kTile;
      if (k0 + kTile > L) zero_tail_tile<VT>(vs0 + so, L - k0, warp, lane);

      // ---- S phase: the keys of row group `warp`, all rows
      float xv[NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int c = 0; c < 4; ++c) xv[nt][c] = 0.f;
      s_phase<KT, NT>(xv, kq0 + so, kg0 + so, qf_lane, cb_lane, lane);
      const bool need_mask = (k0 + kTile - 1) > vis0;
      const int key0 = k0 + 16 * warp + gq;
      bool up = false;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          xv[nt][c] *= scale_log2;
          if (need_mask) {
            const int row = nt * 8 + 2 * tq + (c & 1);
            const int tk = min(row / kGqa, ntok - 1);
            if (key0 + ((c & 2) ? 8 : 0) > vis0 + tk) xv[nt][c] = -INFINITY;
          }
          up |= xv[nt][c] > m_ref[nt][c & 1] + kLazy;
        }
      const bool raised = __any_sync(0xffffffffu, up);
      float* mb_w = mbase + (tbuf * kCWarps + warp) * R8;
      float base[NT][2];  // this warp's P base per row
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) base[nt][e] = m_ref[nt][e];
      if (raised) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          float mx0 = fmaxf(xv[nt][0], xv[nt][2]), mx1 = fmaxf(xv[nt][1], xv[nt][3]);
#pragma unroll
          for (int off = 4; off < 32; off <<= 1) {
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
          }
          base[nt][0] = fmaxf(base[nt][0], mx0);
          base[nt][1] = fmaxf(base[nt][1], mx1);
        }
      }
      if (lane == 0) flags[tbuf * kCWarps + warp] = raised ? 1 : 0;
      float rs[NT][2];  // this thread's share of the tile's row sums, relative to base
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const float b0 = (base[nt][0] == -INFINITY) ? 0.f : base[nt][0];
        const float b1 = (base[nt][1] == -INFINITY) ? 0.f : base[nt][1];
        const uint32_t X0 = pack_half2(ex2(xv[nt][0] - b0), ex2(xv[nt][1] - b1));
        const uint32_t X1 = pack_half2(ex2(xv[nt][2] - b0), ex2(xv[nt][3] - b1));
        const float2 f0 = half2_bits_to_float2(X0), f1 = half2_bits_to_float2(X1);
        rs[nt][0] = f0.x + f1.x;
        rs[nt][1] = f0.y + f1.y;
        const uint32_t B0 = movmatrix_trans(X0), B1 = movmatrix_trans(X1);
        asm volatile("st.shared.v2.b32 [%0], {%1, %2};" ::"r"(
                         pb_base + (((tbuf * kCWarps + warp) * NT + nt) * 32 + lane) * 8),
                     "r"(B0), "r"(B1)
                     : "memory");
        if (gq == 0) {
          mb_w[nt * 8 + 2 * tq] = base[nt][0];
          mb_w[nt * 8 + 2 * tq + 1] = base[nt][1];
        }
      }
      named_bar_sync(bar_id, kCWarps * 32);
      const int4 fl = *reinterpret_cast<const int4*>(flags + tbuf * kCWarps);
      const bool any_raise = (fl.x | fl.y | fl.z | fl.w) != 0;  // the same in every warp

      // ---- rare: a new maximum for some rows; fold every warp's base
      float fsc[kCWarps][NT];  // P scale per producing warp, for query row nt*8 + gq
      if (any_raise) {
        const float* mb_t = mbase + tbuf * kCWarps * R8;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int row = nt * 8 + 2 * tq + e;
            float mn = m_ref[nt][e];
#pragma unroll
            for (int w2 = 0; w2 < kCWarps; ++w2) mn = fmaxf(mn, mb_t[w2 * R8 + row]);
            const float al = (mn == -INFINITY) ? 1.f : ex2(m_ref[nt][e] - mn);
            const float fo = (mn == -INFINITY) ? 1.f : ex2(base[nt][e] - mn);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              o[i][nt][e] *= al;
              o[i][nt][2 + e] *= al;
            }
            l_part[nt][e] = l_part[nt][e] * al + rs[nt][e] * fo;
            m_ref[nt][e] = mn;
          }
          const int rg = nt * 8 + gq;
          float mg = -INFINITY;
#pragma unroll
          for (int w2 = 0; w2 < kCWarps; ++w2) mg = fmaxf(mg, mb_t[w2 * R8 + rg]);
#pragma unroll
          for (int w2 = 0; w2 < kCWarps; ++w2) fsc[w2][nt] = (mg == -INFINITY) ? 1.f : ex2(mb_t[w2 * R8 + rg] - mg);
        }
      } else {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int e = 0; e < 2; ++e) l_part[nt][e] += rs[nt][e];
      }

      // ---- PV phase: dims of m-tiles 4*warp .. +3 over all 64 keys (from three
      // n-tiles on, unrolled by two only: the fully unrolled loop no longer
      // fits the instruction cache)
#pragma unroll(NT >= 3 ? 2 : kCWarps)
      for (int kw = 0; kw < kCWarps; ++kw) {
        uint32_t bp[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const uint2 v = lds64(pb_base + (((tbuf * kCWarps + kw) * NT + nt) * 32 + lane) * 8);
          bp[nt][0] = v.x;
          bp[nt][1] = v.y;
          if (any_raise) {
            const uint32_t f2 = pack_half2(fsc[kw][nt], fsc[kw][nt]);
            bp[nt][0] = hmul2(v.x, f2);
            bp[nt][1] = hmul2(v.y, f2);
          }
        }
        const uint32_t vg = vs0 + so + kw * G::kVGroup;
        pv_kstep<VT, NT>(o, vg + vq_off, vg, warp, lane, bp);
      }
      __syncwarp();
      mbar_arrive_warp(bar_empty + 8 * st);
      if (++st == kStages) { st = 0; ph ^= 1; }
      tbuf ^= 1;
    }

    // ---- end of piece: row sums over the warp's lanes, then over the warps
    float* lsum = mbase + tbuf * kCWarps * R8;  // the buffer the next tile would write first
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        float v = l_part[nt][e];
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
        if (gq == 0) lsum[warp * R8 + nt * 8 + 2 * tq + e] = v;
      }
    named_bar_sync(bar_id, kCWarps * 32);
    // A device length that differs from the host's: the piece counts for
    // nothing (zeros, l = 0) and the mismatch is reported.
    const bool len_ok = l_dev == L;
    if (!len_ok && tid == 0) record_error(p.err, PA_ERR_BOUNDS);
    const int slot = (int)blockIdx.x + seg;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int row = nt * 8 + 2 * tq + c;
        if (row >= R) continue;
        float lr = 0.f;
#pragma unroll
        for (int w2 = 0; w2 < kCWarps; ++w2) lr += lsum[w2 * R8 + row];
        if (!len_ok) lr = 0.f;
        float* dst = row_dst(p, whole, slot, s, g, row0 + row, Rg);
        const float inv = whole ? (lr > 0.f ? 1.f / lr : 0.f) : (len_ok ? 1.f : 0.f);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          dst[vdim<VT>(gq, 4 * warp + i, 0)] = o[i][nt][c] * inv;
          dst[vdim<VT>(gq, 4 * warp + i, 1)] = o[i][nt][2 + c] * inv;
        }
        if (warp == 0 && gq == 0) write_row_stats(p, whole, slot, s, g, row0 + row, Rg, m_ref[nt][c], lr);
      }
    }
    named_bar_sync(bar_id, kCWarps * 32);  // lsum is read before the next piece's tiles reuse it

    x += je - jb;
    qbuf ^= 1;
    j = 0;
    if (++g == p.segs_per_seq) { g = 0; ++s; }
  }
}

// ------------------------------------------------------------------ the split kernel

template <int KT, int VT, int NT, int kG>
__global__ void __launch_bounds__(threads_of(kG), CtaTarget<KT, VT, NT, kG>::kN)
    pa_split_decode_kernel(const __grid_constant__ DecodeParams p) {
  using SM = Smem<KT, VT, NT, kG>;
  constexpr int kStages = SM::kStages;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  // Align the ring (the chunk addressing needs kAlign); the launch asks for
  // kAlign spare bytes.
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((kAlign - (raw & (kAlign - 1))) & (kAlign - 1));
  const int tid = threadIdx.x, warp = tid >> 5;
  const uint32_t ring = smem_u32(smem);
  const uint32_t bar_full = ring + SM::kBar, bar_empty = bar_full + 8 * kStages;
  volatile int* abort = reinterpret_cast<volatile int*>(smem + SM::kMisc);
  int* start = reinterpret_cast<int*>(smem + SM::kMisc + 4);
  long long* range = reinterpret_cast<long long*>(smem + SM::kMisc + 16);
  // This CTA's tile range [a, b), the host plan's cuts: equal tile counts in
  // closed form, or (2-8 tokens, piece_cost > 0) the weighted cut, walked by
  // thread 0.
  const int cta = (int)blockIdx.x;
  long long a = (long long)cta * p.total_tiles / p.n_ctas, b = (long long)(cta + 1) * p.total_tiles / p.n_ctas;

  // Launched as a programmatic dependent of the previous kernel on the stream
  // (for example the append of this step's rows): every thread waits for it
  // to complete before it reads any input.
  asm volatile("griddepcontrol.wait;" ::: "memory");

  if (tid == 0) {
    // The merge kernel may launch now; it reads nothing of ours before its
    // griddepcontrol.wait.
    asm volatile("griddepcontrol.launch_dependents;");
    *abort = 0;
    for (int i = 0; i < kStages; ++i) {
      mbar_init(bar_full + 8 * i, 1);
      mbar_init(bar_empty + 8 * i, NT == 1 ? p.seg_heads : kCWarps * kG);  // one arrival per consuming warp
    }
    fence_mbar_init();
    if (NT > 1 && p.piece_cost) {
      a = cta_first_tile(p.lens, p.n_seq, p.segs_per_seq, p.tile_keys, p.total_tiles, p.n_ctas, p.piece_cost, cta);
      b = cta_first_tile(p.lens, p.n_seq, p.segs_per_seq, p.tile_keys, p.total_tiles, p.n_ctas, p.piece_cost,
                         cta + 1);
      range[0] = a;
      range[1] = b;
    }
    int s0, g0, j0;
    locate_tile(p, a, s0, g0, j0);
    start[0] = s0;
    start[1] = g0;
    start[2] = j0;
  }
  __syncthreads();
  if (NT > 1 && p.piece_cost) {
    a = range[0];
    b = range[1];
  }
  const int s = start[0], g = start[1], j = start[2];
  if (s >= p.n_seq) return;  // an empty range (the planner gives every CTA a tile)

  if (warp == kCWarps * kG) {
    TilePos pos;
    pos.s = s;
    pos.g = g;
    pos.j = j;
    pos.L = p.lens[s];
    pos.nt = tiles_of(p, pos.L);
    if constexpr (NT == 1) {
      produce_hg<KT, VT, NT>(p, ring, bar_full, bar_empty, abort, a, b, pos);
    } else {
      produce_head<KT, VT, NT, kG>(p, ring, bar_full, bar_empty, abort, a, b, pos);
    }
    return;
  }
  if constexpr (NT == 1) {
    if (warp >= p.seg_heads) return;  // a head group smaller than the warp count
    consume_hg<KT, VT>(p, smem, ring, bar_full, bar_empty, abort, a, b, s, g, j);
  } else {
    consume_shared<KT, VT, NT, kG>(p, smem, ring, bar_full, bar_empty, abort, a, b, s, g, j, warp / kCWarps);
  }
}

// ------------------------------------------------------------------ host-side registry

using KernelFn = void (*)(DecodeParams);

struct KernelInfo {
  KernelFn fn;
  int smem;
  int ctas_per_sm_target;
  int threads;
};

template <int KT, int VT, int NT, int kG = 1>
KernelInfo kernel_info() {
  return KernelInfo{pa_split_decode_kernel<KT, VT, NT, kG>, Smem<KT, VT, NT, kG>::kLaunch,
                    CtaTarget<KT, VT, NT, kG>::kN, threads_of(kG)};
}

// Defined once per (K, V) format pair, named by the pa_type numbers
// (pa_decode_kern.cu, one translation unit each).
#define PA_DECLARE_LOOKUP(k, v) bool lookup_kernel_##k##_##v(int nt, KernelInfo* out);
PA_DECLARE_LOOKUP(1, 1) PA_DECLARE_LOOKUP(1, 2) PA_DECLARE_LOOKUP(1, 8)
PA_DECLARE_LOOKUP(2, 1) PA_DECLARE_LOOKUP(2, 2) PA_DECLARE_LOOKUP(2, 8)
PA_DECLARE_LOOKUP(8, 1) PA_DECLARE_LOOKUP(8, 2) PA_DECLARE_LOOKUP(8, 8)
#undef PA_DECLARE_LOOKUP
static_assert(PA_F16 == 1 && PA_Q4_0 == 2 && PA_Q8_0 == 8, "lookup names use the pa_type numbers");

}  // namespace pa_split
