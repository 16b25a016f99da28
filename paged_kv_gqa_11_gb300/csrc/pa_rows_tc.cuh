// Row tiles on the fifth-generation tensor core: decode of 9 to 96 query
// tokens per sequence (sm_103a).
//
// What is computed is the causal verify decode of the narrower widths (query
// token t of n_qtok sits at position L - n_qtok + t and sees keys 0 .. L -
// n_qtok + t); batches of more than eight tokens take the decode kernel's row
// tiles, which the pages find faster than a chunked prefill up to 96 query
// tokens (llama.cpp fork PR #2, the commit on KV-streaming ubatches of more
// than 8 tokens).  With 6 * n_qtok query rows per KV head (54 to 576) this is a
// dense contraction, so it runs on tcgen05:
//
//   segment  = (sequence, KV head, row tile of 128 query rows); its tiles are
//              the 64-key tiles the row tile's last row sees;
//   S        = Q K^T    tcgen05.mma M = 128 rows, N = 64 keys, K = 256 dims:
//                       Q from tensor memory, K from shared memory, fp32 in
//                       tensor memory, double-buffered;
//   softmax  one thread per query row: the row's logits come from tensor
//            memory into registers (no shuffles), causal mask, lazy online
//            maximum (raised only past 2^8; then that row of O is rescaled in
//            tensor memory), P as binary16 into shared memory;
//   O       += P V     tcgen05.mma M = 128 rows, N = 256 dims, K = 64 keys,
//                       fp32 in tensor memory (256 columns).
//
// An MMA with N of 64 or less costs the tensor core about the same time
// whatever N is (the issue, not the arithmetic, sets it), so a key tile is as
// wide as shared memory allows: 64 keys, with K and S double-buffered and V^T
// and P single.  Tensor memory (512 columns x 128 lanes, lane = query row): O
// in columns 0-255, Q in 256-383 (two binary16 per column), S in 384-511.
//
// The CTA's warps specialise and run as a pipeline over its key tiles, each
// hand-off an mbarrier:
//   warps 0-3   softmax and output, one query row per thread (tensor-memory
//               lane quarters 0-3);
//   warps 4-7   K dequantisation, sixteen keys each per tile, into one of two
//               binary16 K buffers; Q into tensor memory at a segment start;
//   warps 8-11  V dequantisation into the V^T buffer, sixteen keys each;
//   warp 12     issues the MMAs (the whole warp runs the loop on warp-uniform
//               descriptors; one lane, chosen by elect.sync, issues): S of tile
//               j + 1 goes to the tensor core before O += P V of tile j, so S is
//               computed while the softmax of tile j runs;
//   warps 13-14 stream raw K (warp 13) and V (warp 14) row groups into two
//               rings of 32-key stages (bulk copies), two stages per key
//               tile; separate rings let K run ahead of V, which waits for
//               the previous tile's O += P V.
//
// The shared-memory operands sit in the MMA's canonical no-swizzle K-major
// layout (core matrices of 8 rows x 16 bytes): K [keys][dims], V^T
// [dims][keys] and P [rows][keys].  Dequantisation reads the raw quants
// with ldmatrix (thread 4g+t gets four bytes of key g), converts them in
// registers and writes core matrices with stmatrix (.trans for V), without
// bank conflicts.  That fixes a per-format order of the head dims inside each
// 32-dim window (dim_of below); Q is staged in K's order and O is written back
// through V's.
//
// Precision: Q, P and V (q * d rounded once) are binary16.  Quantised K is
// kept to about 2^-22: it is split as K = K_hi + K_lo, K_hi = q * d rounded to
// binary16 and K_lo = q * d - K_hi rounded once (a fused multiply-add), and S
// takes both products (32 MMAs per tile), so large logits carry no K
// rounding.  Every product is accumulated in fp32; the softmax denominator
// sums the fp32 weights before their rounding to binary16 (a relative
// difference of at most 2^-11 from the sum of the rounded P).
#pragma once

#include "pa_rows_impl.cuh"

namespace pa_split {

constexpr uint32_t kTcTmemCols = 512;
constexpr uint32_t kTcOCol = 0, kTcQCol = 256, kTcSCol = 384;  // O, Q, S[2] (64 columns each)
constexpr uint32_t kTcIdescS = idesc_f16_f32(kRowTile, kRowKeys);  // 128 x 64
constexpr uint32_t kTcIdescO = idesc_f16_f32(kRowTile, kD);        // 128 x 256
constexpr int kTcSmWarp0 = 0, kTcKWarp0 = 4, kTcVWarp0 = 8, kTcMmaWarp = 12, kTcCopyK = 13, kTcCopyV = 14;
constexpr int kRowThreads = 15 * 32;

template <int KT, int VT>
struct TcSmem {
  static constexpr bool kKSplit = KT != PA_F16;  // K_hi and K_lo
  static constexpr int kKStage = RowStageGeo<KT, VT>::kKBytes, kVStage = RowStageGeo<KT, VT>::kVBytes;
  static constexpr int kKBytes = kRowKeys * kD * 2;         // one K tile [64][256]: 32 KB
  static constexpr int kVBytes = kD * kRowKeys * 2;         // the V^T tile [256][64]: 32 KB
  static constexpr int kPBytes = kRowTile * kRowKeys * 2;   // the P tile [128][64]: 16 KB
  static constexpr int kKBuf = kKBytes * (kKSplit ? 2 : 1);  // K_hi [K_lo]
  static constexpr int kK0 = 0, kV0 = 2 * kKBuf, kP0 = kV0 + kVBytes;
  static constexpr int kRing = kP0 + kPBytes;
  // raw stages: three K stages first if they fit beside a V stage, then as many
  // V stages as fit (at most four), then K stages up to four
  static constexpr int kRoom = 232448 - 1024 - kRing - 512;
  static constexpr int kVFit = (kRoom - 3 * kKStage) / kVStage;
  static constexpr int kVStages = kVFit >= 1 ? (kVFit > 4 ? 4 : kVFit) : (kRoom - 2 * kKStage) / kVStage;
  static constexpr int kKFit = (kRoom - kVStages * kVStage) / kKStage;
  static constexpr int kKStages = kKFit > 4 ? 4 : kKFit;
  static_assert(kKStages >= 2 && kVStages >= 1, "row-tile stage rings do not fit");
  static_assert(kRing % 1024 == 0, "tile alignment");
  static constexpr int kVRing = kRing + kKStages * kKStage;
  // mbarriers: K raw full / empty [kKStages], V raw full / empty [kVStages],
  // k full / empty [2], v full [2], s full / empty [2], p full, pv done [2],
  // drain
  static constexpr int kBar = kVRing + kVStages * kVStage;
  static constexpr int kNBar = 2 * kKStages + 2 * kVStages + 4 + 2 + 4 + 1 + 2 + 1;
  static constexpr int kMisc = kBar + kNBar * 8;  // abort, start[3], tmem base
  static constexpr int kTotal = kMisc + 32;
  static constexpr int kLaunch = kTotal + 1024;  // the base is aligned to 1024 inside
  static_assert(kTotal - kBar <= 512, "barrier area");
};

// Canonical K-major offsets (bytes): operand with `kslots` 8-element slots
// along K; row r, slot s.
__device__ __forceinline__ uint32_t canon_off(int r, int s, int kslots) {
  return (uint32_t)((((r >> 3) * kslots + s) << 7) + ((r & 7) << 4));
}

// Head dim held at position p of a 32-dim window in the order the dequantised
// tiles of format T use (dim_of(T, p) - p stays inside the window): F16 keeps
// the natural order; Q8_0 and Q4_0 deliver dims in pairs 4j + {0,1} and
// 4j + {2,3} to separate 8-element slots.
template <int T>
__host__ __device__ constexpr int dim_of(int p) {
  if (T == PA_F16) return p;
  const int s = (p >> 3) & 3, k = p & 7;
  return (p & ~31) + 16 * (s >> 1) + 4 * (k >> 1) + 2 * (s & 1) + (k & 1);
}

// ------------------------------------------------------------------ dequantisation by ldmatrix / stmatrix

// Store four fragment matrices of slots s0 .. s0+3 (8 dims each) of eight
// keys: K as rows 8w .. 8w+7 of the [keys][dims] tile, V transposed into key
// slot w of the [dims][keys] tile.  Lane 8j + r gives the address of row r of
// matrix j.
template <bool kRoleV>
__device__ __forceinline__ void tc_store4(uint32_t dst, int w, int lane, int s0, uint32_t r0, uint32_t r1, uint32_t r2,
                                          uint32_t r3) {
  const int mj = lane >> 3, mr = lane & 7;
  if (kRoleV) stsm_x4_trans(dst + canon_off(8 * (s0 + mj) + mr, w, kRowKeys / 8), r0, r1, r2, r3);
  else stsm_x4(dst + canon_off(8 * w + mr, s0 + mj, kD / 8), r0, r1, r2, r3);
}

// K_hi (rounded product) and K_lo (its exact remainder, rounded once) of exact
// quants v with scale d2; V: v * d2.
__device__ __forceinline__ uint32_t tc_hi(uint32_t v, uint32_t d2) { return hmul2(v, d2); }
__device__ __forceinline__ uint32_t tc_lo(uint32_t v, uint32_t d2, uint32_t hi) {
  return hfma2(v, d2, hi ^ 0x80008000u);
}

// Eight keys (8w .. 8w+7) of a raw 32-key stage region of format T (two row
// groups), as binary16 core matrices: V values q * d into key slot `ds` of
// the V^T tile (kRoleV), K exact for F16 or as K_hi / K_lo rows 8w .. 8w+7 of
// the tiles at dst / dst_lo for Q8_0 and Q4_0.  Keys at or past n_keys are
// written as zeros.
template <int T, bool kRoleV>
__device__ __forceinline__ void tc_dequant_warp(uint32_t region, uint32_t dst, uint32_t dst_lo, int w, int ds, int lane,
                                                int n_keys) {
  const int dw = kRoleV ? ds : w;  // the store's row group (K) or key slot (V)
  constexpr int C = Fmt<T>::kRowQ / 16;  // 16-byte chunks per row: 32 / 16 / 8
  constexpr int GB = pa_layout::group_bytes<T>();
  // this lane's ldmatrix row: key 8w + (lane & 7) of matrix lane >> 3
  const int lk = 8 * w + (lane & 7), lr = lk & 15;
  const uint32_t lrow = region + (lk >> 4) * GB + Fmt<T>::kScales + lr * Fmt<T>::kRowQ;
  // this thread's fragment key (its scales): 8w + (lane >> 2)
  const int sk = 8 * w + (lane >> 2), sr = sk & 15;
  const uint32_t sgrp = region + (sk >> 4) * GB;
  const bool live = sk < n_keys;
  auto scale2 = [&](int blk) -> uint32_t {
    uint16_t dh;
    const uint32_t off = kRoleV ? pa_layout::v_scale_offset(sr, blk) : pa_layout::k_scale_offset(sr, blk);
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(dh) : "r"(sgrp + off));
    return live ? ((uint32_t)dh | ((uint32_t)dh << 16)) : 0u;  // a zero scale zeroes the key
  };
#pragma unroll 1  // rolled: fifteen warps run different code, and the instruction cache is the limit
  for (int i = 0; i < C / 4; ++i) {
    uint32_t x[4];  // chunk 4i + j of key g, bytes 4t .. 4t+3 (thread 4g + t)
    ldsm_x4(lrow + (((4 * i + (lane >> 3)) ^ (lr & 7)) << 4), x);
    if constexpr (T == PA_F16) {  // chunk = slot, natural order
      if (!live) x[0] = x[1] = x[2] = x[3] = 0u;
      tc_store4<kRoleV>(dst, dw, lane, 4 * i, x[0], x[1], x[2], x[3]);
    } else if constexpr (T == PA_Q8_0) {
      // chunk c = 4i + j: dims 16c + 4t, +1 -> slot 2c; 16c + 4t + 2, +3 -> slot 2c + 1
      uint32_t h[8], l[8];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t d2 = scale2(2 * i + (j >> 1));
        const uint32_t xx = x[j] ^ 0x80808080u;  // int8 -> 128 + q as an unsigned byte
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const uint32_t v = hadd2(prmt(xx, kMagic64, e ? 0x4342 : 0x4140), kHalf2_m1152);  // exact q pairs
          h[2 * j + e] = tc_hi(v, d2);
          if (!kRoleV) l[2 * j + e] = tc_lo(v, d2, h[2 * j + e]);
        }
      }
      tc_store4<kRoleV>(dst, dw, lane, 8 * i, h[0], h[1], h[2], h[3]);
      tc_store4<kRoleV>(dst, dw, lane, 8 * i + 4, h[4], h[5], h[6], h[7]);
      if (!kRoleV) {
        tc_store4<false>(dst_lo, dw, lane, 8 * i, l[0], l[1], l[2], l[3]);
        tc_store4<false>(dst_lo, dw, lane, 8 * i + 4, l[4], l[5], l[6], l[7]);
      }
    } else {  // Q4_0: block c = 4i + j; byte b holds dims b (low nibble) and b + 16 (high)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t d2 = scale2(4 * i + j);
        const uint32_t t0 = prmt(x[j], 0u, 0x4140), t1 = prmt(x[j], 0u, 0x4342);  // bytes (4t, 4t+1), (4t+2, 4t+3)
        const uint32_t v[4] = {hadd2(and_or(t0, 0x000f000fu, 0x64006400u), kHalf2_m1032),  // dims 4t, 4t+1
                               hadd2(and_or(t1, 0x000f000fu, 0x64006400u), kHalf2_m1032),  // 4t+2, 4t+3
                               hfma2(and_or(t0, 0x00f000f0u, 0x64006400u), kHalf2_1_16, kHalf2_m72),  // 16+4t, +1
                               hfma2(and_or(t1, 0x00f000f0u, 0x64006400u), kHalf2_1_16, kHalf2_m72)};  // 16+4t+2, +3
        uint32_t h[4], l[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          h[e] = tc_hi(v[e], d2);
          if (!kRoleV) l[e] = tc_lo(v[e], d2, h[e]);
        }
        const int c = 4 * i + j;
        tc_store4<kRoleV>(dst, dw, lane, 4 * c, h[0], h[1], h[2], h[3]);
        if (!kRoleV) tc_store4<false>(dst_lo, dw, lane, 4 * c, l[0], l[1], l[2], l[3]);
      }
    }
  }
}

// ------------------------------------------------------------------ Q staging

// Row 32 * quarter + lane of the row tile (zero past the 6 * n_qtok real rows)
// as binary16 into its tensor-memory lane: column c of the 128 holds positions
// 2c and 2c + 1 of K's dim order (dim_of), the pair of adjacent dims
// dim_of<KT>(2c), + 1.  taddr: Q's first column, lane field of the quarter.
// The whole warp calls this.
template <int KT>
__device__ __forceinline__ void tc_stage_q(const DecodeParams& p, int s, int head, int rt, uint32_t taddr, int quarter,
                                           int lane) {
  const int row = 32 * quarter + lane, rg = kRowTile * rt + row;
  const bool real = rg < kGqa * p.n_qtok;
  const float4* src = reinterpret_cast<const float4*>(
      p.q + (((long long)s * p.n_qtok + (real ? rg / kGqa : 0)) * p.n_q_heads + head * kGqa + (real ? rg % kGqa : 0)) *
                kD);
#pragma unroll 1
  for (int wp = 0; wp < kD / 64; ++wp) {
    uint32_t h[32];
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      float v[32];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float4 f = real ? __ldg(src + 8 * (2 * wp + half) + i) : make_float4(0.f, 0.f, 0.f, 0.f);
        v[4 * i] = f.x; v[4 * i + 1] = f.y; v[4 * i + 2] = f.z; v[4 * i + 3] = f.w;
      }
#pragma unroll
      for (int c = 0; c < 16; ++c) h[16 * half + c] = pack_half2(v[dim_of<KT>(2 * c)], v[dim_of<KT>(2 * c) + 1]);
    }
    __syncwarp();
    tmem_st32(taddr + 32 * wp, h);
  }
  tmem_st_wait();
}

// ------------------------------------------------------------------ the kernel

// A tile's place in the CTA's walk, as every role sees it.
struct TcTile {
  bool first;  // the first tile of a piece (a new segment, or the CTA's first)
  bool last;   // the last tile of a piece
};

__device__ __forceinline__ TcTile tc_tile(const RowPos& pos, long long x, long long a, long long b) {
  return TcTile{x == a || pos.j == 0, x + 1 == b || pos.j + 1 == pos.nt};
}

template <int KT, int VT>
__global__ void __launch_bounds__(kRowThreads, 1) pa_rows_tc_kernel(const __grid_constant__ DecodeParams p) {
  using SM = TcSmem<KT, VT>;
  constexpr int kKS = SM::kKStages, kVS = SM::kVStages;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024 - (raw & 1023)) & 1023);
  const uint32_t base = smem_u32(smem);
  const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
  // Hand-offs.  Tile j (the j-th of the CTA) uses K and S buffer kb = j & 1 for
  // the ku = j >> 1-th time; its stages are 2j and 2j + 1.  Every wait is on a
  // phase that cannot be two ahead of its waiter.
  //   kraw_*, vraw_*        copy warps <-> dequantisation, per ring stage
  //   k_full                K dequantisation -> MMA (also "Q is staged")
  //   k_empty               MMA commit after S(j): K buffer kb free, S(j) done
  //   v_full[h]             V dequantisation -> MMA: keys 32h .. 32h+31 of V^T
  //                         (tile half h) of tile j
  //   s_full / s_empty      S(j) in tensor memory / in the softmax registers
  //   p_full                softmax -> MMA: P(j) in shared memory
  //   pv_done[h]            MMA commit after O += P V of tile j's half h: that
  //                         half of V^T free; pv_done[1] also: P free,
  //                         O holds tiles .. j
  const uint32_t bars = base + SM::kBar;
  const uint32_t kraw_full = bars, kraw_empty = kraw_full + 8 * kKS, vraw_full = kraw_empty + 8 * kKS,
                 vraw_empty = vraw_full + 8 * kVS;
  const uint32_t k_full = vraw_empty + 8 * kVS, k_empty = k_full + 16, v_full = k_empty + 16, s_full = v_full + 16,
                 s_empty = s_full + 16, p_full = s_empty + 16, pv_done = p_full + 8, drain = pv_done + 16;
  volatile int* abort = reinterpret_cast<volatile int*>(smem + SM::kMisc);
  int* start = reinterpret_cast<int*>(smem + SM::kMisc + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + SM::kMisc + 16);
  const uint32_t kring = base + SM::kRing, vring = base + SM::kVRing;

  const long long T = p.total_tiles;
  const int Gn = p.n_ctas;
  const long long a = (long long)blockIdx.x * T / Gn, b = (long long)(blockIdx.x + 1) * T / Gn;
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (tid == 0) {
    asm volatile("griddepcontrol.launch_dependents;");
    *abort = 0;
    for (int i = 0; i < kKS; ++i) {
      mbar_init(kraw_full + 8 * i, 1);
      mbar_init(kraw_empty + 8 * i, 4);
    }
    for (int i = 0; i < kVS; ++i) {
      mbar_init(vraw_full + 8 * i, 1);
      mbar_init(vraw_empty + 8 * i, 4);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(k_full + 8 * i, 4);
      mbar_init(k_empty + 8 * i, 1);
      mbar_init(s_full + 8 * i, 1);
      mbar_init(s_empty + 8 * i, 4);
    }
    mbar_init(v_full, 4);
    mbar_init(v_full + 8, 4);
    mbar_init(p_full, 4);
    mbar_init(pv_done, 1);
    mbar_init(pv_done + 8, 1);
    mbar_init(drain, 1);
    fence_mbar_init();
    const RowPos r = row_locate(p, a);
    start[0] = r.s;
    start[1] = r.gi;
    start[2] = r.j;
  }
  if (w == 0) {
    tmem_alloc(smem_u32(tmem_slot), kTcTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const bool any = start[0] < p.n_seq;  // the planner gives every CTA a tile
  RowPos pos0;
  pos0.s = start[0];
  pos0.gi = start[1];
  pos0.j = start[2];
  pos0.L = any ? p.lens[pos0.s] : 0;
  pos0.nt = any ? row_seg_tiles(p, pos0.L, pos0.gi) : 0;
  const int R = kGqa * p.n_qtok;
  const int n = (int)(b - a);

  if (any && (w == kTcCopyK || w == kTcCopyV)) {
    // ---- raw K (or V) stages, two per key tile
    const bool isv = w == kTcCopyV;
    const int ns = isv ? kVS : kKS, sb = isv ? SM::kVStage : SM::kKStage;
    const uint32_t full = isv ? vraw_full : kraw_full, empty = isv ? vraw_empty : kraw_empty, rg0 = isv ? vring : kring;
    const uint64_t policy = l2_evict_first_policy();
    RowPos pos = pos0;
    for (int q = 0; q < 2 * n; ++q) {
      if (__any_sync(0xffffffffu, *abort != 0)) break;
      const int slot = q % ns, use = q / ns, half = q & 1;
      if (use > 0) mbar_wait(empty + 8 * slot, (use - 1) & 1, p.err, abort);
      const int tb = row_entry(p, pos, half, lane);
      if (isv) issue_half<VT, true>(p, pos, half, tb, rg0 + slot * sb, full + 8 * slot, policy, lane);
      else issue_half<KT, false>(p, pos, half, tb, rg0 + slot * sb, full + 8 * slot, policy, lane);
      if (half) row_next(p, pos);
    }
  } else if (any && w >= kTcKWarp0 && w < kTcKWarp0 + 4) {
    // ---- K dequantisation, and Q into tensor memory at every piece start
    const int dw = w - kTcKWarp0;
    RowPos pos = pos0;
    for (int j = 0; j < n; ++j) {
      const TcTile tt = tc_tile(pos, a + j, a, b);
      const int kb = j & 1, ku = j >> 1;
      if (tt.first) {
        if (j > 0) {  // S(j - 1), the previous piece's last, is done with Q
          mbar_wait(k_empty + 8 * ((j - 1) & 1), ((j - 1) >> 1) & 1, p.err, abort);
          __syncwarp();
          tc_fence_after();
        }
        tc_stage_q<KT>(p, pos.s, pos.gi / p.n_row_tiles, pos.gi % p.n_row_tiles,
                       tmem + kTcQCol + ((uint32_t)(32 * dw) << 16), dw, lane);
      }
      if (ku > 0) mbar_wait(k_empty + 8 * kb, (ku - 1) & 1, p.err, abort);  // S(j - 2) is done with the buffer
      const uint32_t kh = base + SM::kK0 + kb * SM::kKBuf;
#pragma unroll 1
      for (int half = 0; half < 2; ++half) {
        const int q = 2 * j + half, slot = q % kKS;
        mbar_wait(kraw_full + 8 * slot, (q / kKS) & 1, p.err, abort);
        __syncwarp();
        const int n_keys = min(kStageKeys, pos.L - pos.j * kRowKeys - half * kStageKeys);
        const uint32_t off = (uint32_t)(half * kStageKeys * kD * 2);
        tc_dequant_warp<KT, false>(kring + slot * SM::kKStage, kh + off, kh + SM::kKBytes + off, dw, 0, lane, n_keys);
        __syncwarp();
        if (lane == 0) mbar_arrive(kraw_empty + 8 * slot);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(k_full + 8 * kb);
      row_next(p, pos);
    }
  } else if (any && w >= kTcVWarp0 && w < kTcVWarp0 + 4) {
    // ---- V dequantisation into the single V^T buffer, half a tile at a time:
    // half h of tile j is written once O += P V of tile j - 1 has read that
    // half, so the conversion of one half overlaps the product of the other
    const int dw = w - kTcVWarp0;
    RowPos pos = pos0;
    for (int j = 0; j < n; ++j) {
#pragma unroll 1
      for (int half = 0; half < 2; ++half) {
        const int q = 2 * j + half, slot = q % kVS;
        if (j > 0) mbar_wait(pv_done + 8 * half, (j - 1) & 1, p.err, abort);
        mbar_wait(vraw_full + 8 * slot, (q / kVS) & 1, p.err, abort);
        __syncwarp();
        const int n_keys = min(kStageKeys, pos.L - pos.j * kRowKeys - half * kStageKeys);
        tc_dequant_warp<VT, true>(vring + slot * SM::kVStage, base + SM::kV0, 0u, dw, half * (kStageKeys / 8) + dw, lane,
                                  n_keys);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(vraw_empty + 8 * slot);
          mbar_arrive(v_full + 8 * half);
        }
      }
      row_next(p, pos);
    }
  } else if (any && w == kTcMmaWarp) {
    // ---- MMA issue (the whole warp, one elected lane issuing): S(j), then
    // O += P V of tile j - 1
    const uint32_t tq = __shfl_sync(0xffffffffu, tmem, 0), ub = __shfl_sync(0xffffffffu, base, 0);
    // descriptor start addresses count 16-byte units
    const uint64_t kdesc0 = smem_desc(ub + SM::kK0, 128, 4096), vdesc = smem_desc(ub + SM::kV0, 128, 1024),
                   pdesc = smem_desc(ub + SM::kP0, 128, 1024);
    auto pv = [&](int jj, bool first) {  // by tile halves, each as soon as its V^T is there
      mbar_wait(p_full, jj & 1, p.err, abort);
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        mbar_wait(v_full + 8 * half, jj & 1, p.err, abort);
        __syncwarp();
        tc_fence_after();
#pragma unroll
        for (int kk = 2 * half; kk < 2 * half + 2; ++kk)
          tc_mma_f16_warp(tq + kTcOCol, pdesc + 16 * kk, vdesc + 16 * kk, kTcIdescO, (first && kk == 0) ? 0u : 1u);
        tc_commit_warp(pv_done + 8 * half);
      }
    };
    RowPos pos = pos0;
    bool prev_first = false;
    for (int j = 0; j < n; ++j) {
      const int kb = j & 1, ku = j >> 1;
      const bool first = tc_tile(pos, a + j, a, b).first;
      mbar_wait(k_full + 8 * kb, ku & 1, p.err, abort);
      if (ku > 0) mbar_wait(s_empty + 8 * kb, (ku - 1) & 1, p.err, abort);
      __syncwarp();
      tc_fence_after();
      const uint32_t dS = tq + kTcSCol + kRowKeys * kb;
      const uint64_t kd = kdesc0 + (uint64_t)((kb * SM::kKBuf) >> 4);
#pragma unroll 4
      for (int ks = 0; ks < kD / 16; ++ks)
        tc_mma_f16_tmem_a_warp(dS, tq + kTcQCol + 8 * ks, kd + 16 * ks, kTcIdescS, ks > 0);
      if (SM::kKSplit) {
#pragma unroll 4
        for (int ks = 0; ks < kD / 16; ++ks)
          tc_mma_f16_tmem_a_warp(dS, tq + kTcQCol + 8 * ks, kd + (SM::kKBytes >> 4) + 16 * ks, kTcIdescS, 1);
      }
      tc_commit_warp(k_empty + 8 * kb);
      tc_commit_warp(s_full + 8 * kb);
      if (j > 0) pv(j - 1, prev_first);
      prev_first = first;
      row_next(p, pos);
    }
    if (n > 0) pv(n - 1, prev_first);
    // the last commits have arrived before the CTA's barriers go away
    for (int jj = max(0, n - 2); jj < n; ++jj) mbar_wait(k_empty + 8 * (jj & 1), (jj >> 1) & 1, p.err, abort);
    if (n > 0) {
      mbar_wait(pv_done, (n - 1) & 1, p.err, abort);
      mbar_wait(pv_done + 8, (n - 1) & 1, p.err, abort);
    }
    __syncwarp();
  } else if (any && w < kTcSmWarp0 + 4) {
    // ---- softmax and output: one query row per thread
    const int row = 32 * w + lane;
    const uint32_t t_lane = (uint32_t)(32 * w) << 16;
    const uint32_t tO = tmem + kTcOCol + t_lane;
    const float scale_log2 = p.scale_log2;
    const uint32_t pk = base + SM::kP0;
    RowPos pos = pos0;
    float m = -INFINITY, l = 0.f;
    int vis = -1, piece_j0 = 0;
    bool piece_whole = false;
    for (int j = 0; j < n; ++j) {
      const TcTile tt = tc_tile(pos, a + j, a, b);
      const int kb = j & 1, ku = j >> 1;
      const int rt = pos.gi % p.n_row_tiles, rg = kRowTile * rt + row;
      const bool smx = kRowTile * rt + 32 * w < R;  // the warp holds a real row
      if (tt.first) {
        m = -INFINITY;
        l = 0.f;
        vis = rg < R ? pos.L - p.n_qtok + rg / kGqa : -1;
        piece_j0 = j;
        piece_whole = pos.j == 0;
      }
      const int k0 = pos.j * kRowKeys;
      // S(j) into registers; the buffer is then free for S(j + 2)
      mbar_wait(s_full + 8 * kb, ku & 1, p.err, abort);
      __syncwarp();
      tc_fence_after();
      uint32_t sv[64];
      tmem_ld32(tmem + t_lane + kTcSCol + kRowKeys * kb, *reinterpret_cast<uint32_t(*)[32]>(sv));
      tmem_ld32(tmem + t_lane + kTcSCol + kRowKeys * kb + 32, *reinterpret_cast<uint32_t(*)[32]>(sv + 32));
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(s_empty + 8 * kb);
      if (k0 + kRowKeys - 1 > vis) {  // the causal edge (or padding rows): mask
        const int nv = vis - k0 + 1;  // keys of this tile the row sees (may be <= 0)
#pragma unroll
        for (int c = 0; c < kRowKeys; ++c) sv[c] = c < nv ? sv[c] : 0xff800000u;  // -inf
      }
      float mx[8];
#pragma unroll
      for (int c = 0; c < 8; ++c)
        mx[c] = fmaxf(fmaxf(fmaxf(__uint_as_float(sv[c]), __uint_as_float(sv[c + 8])),
                            fmaxf(__uint_as_float(sv[c + 16]), __uint_as_float(sv[c + 24]))),
                      fmaxf(fmaxf(__uint_as_float(sv[c + 32]), __uint_as_float(sv[c + 40])),
                            fmaxf(__uint_as_float(sv[c + 48]), __uint_as_float(sv[c + 56]))));
      const float tmax =
          fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])), fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7]))) *
          scale_log2;
      // Lazy maximum: raised (rarely, after a row's first tile) past 2^8.  The
      // row of O is rescaled in tensor memory once O += P V of tile j - 1 is
      // done; tensor-memory loads and stores are warp-wide, so the whole warp
      // runs them when any of its rows rises.
      const bool raise = tmax > m + kLazy;
      const float al = raise ? ((m == -INFINITY) ? 1.f : ex2(m - tmax)) : 1.f;
      // O += P V of tile j - 1 has read the P buffer (and, within a piece, O
      // holds it) before P(j) is written or O rescaled
      if (j > 0) mbar_wait(pv_done + 8, (j - 1) & 1, p.err, abort);
      if (smx && __any_sync(0xffffffffu, raise) && j > piece_j0) {
        __syncwarp();
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < kD; c += 32) {
          uint32_t ov[32];
          tmem_ld32(tO + c, ov);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * al);
          tmem_st32(tO + c, ov);
        }
        tmem_st_wait();
        tc_fence_before();
      }
      if (raise) {
        l *= al;
        m = tmax;
      }
      const float nbm = (m == -INFINITY) ? 0.f : -m;
      float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int kc = 0; kc < kRowKeys / 8; ++kc) {
        uint32_t ph[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int c = 8 * kc + 2 * e;
          const float e0 = ex2(fmaf(__uint_as_float(sv[c]), scale_log2, nbm)),
                      e1 = ex2(fmaf(__uint_as_float(sv[c + 1]), scale_log2, nbm));
          ls[e] += e0 + e1;
          ph[e] = pack_half2(e0, e1);
        }
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(pk + canon_off(row, kc, kRowKeys / 8)),
                     "r"(ph[0]), "r"(ph[1]), "r"(ph[2]), "r"(ph[3]) : "memory");
      }
      l += (ls[0] + ls[1]) + (ls[2] + ls[3]);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full);

      if (tt.last && smx) {
        // ---- piece result: this thread's row, once the piece's last O += P V is done
        const int s = pos.s, seg = s * p.segs_per_seq + pos.gi, head = pos.gi / p.n_row_tiles;
        const bool whole = piece_whole && pos.j + 1 == pos.nt;
        const bool len_ok = device_len(p, s) == pos.L;
        if (!len_ok && lane == 0) record_error(p.err, PA_ERR_BOUNDS);
        mbar_wait(pv_done + 8, j & 1, p.err, abort);
        __syncwarp();
        tc_fence_after();
        const bool real = rg < R;
        const float lr = (len_ok && real) ? l : 0.f;
        const int t = real ? rg / kGqa : 0, hl = real ? rg % kGqa : 0;
        const long long orow = ((long long)s * p.n_qtok + t) * p.n_q_heads + head * kGqa + hl;
        const int slot = (int)blockIdx.x + seg;
        float* dst;
        float inv;
        if (whole) {
          dst = p.out + orow * kD;
          inv = lr > 0.f ? 1.f / lr : 0.f;
          if (real && p.lse) p.lse[orow] = lr > 0.f ? (m + log2f(lr)) * kLn2 : -INFINITY;
        } else {
          dst = p.part_o + ((long long)slot * p.rows_per_seg + row) * kD;
          inv = len_ok ? 1.f : 0.f;
          p.part_ml[(long long)slot * p.rows_per_seg + row] = real ? make_float2(m, lr) : make_float2(-INFINITY, 0.f);
        }
        const bool store = real || !whole;
#pragma unroll 1
        for (int c = 0; c < kD; c += 32) {
          uint32_t ov[32];
          tmem_ld32(tO + c, ov);
          tmem_ld_wait();
          if (store) {
#pragma unroll
            for (int i = 0; i < 32; i += 2)
              *reinterpret_cast<float2*>(dst + c + dim_of<VT>(i)) =
                  make_float2(__uint_as_float(ov[i]) * inv, __uint_as_float(ov[i + 1]) * inv);
          }
        }
        tc_fence_before();
      }
      row_next(p, pos);
    }
  }
  // Every copy and MMA was waited for above, unless a wait expired (the abort
  // flag): then wait, with a bound, for what is still in flight before the
  // stages and tensor memory are released.
  if (w == kTcMmaWarp && __any_sync(0xffffffffu, *abort != 0)) {  // the lane that issued the MMAs commits
    tc_commit_warp(drain);
    mbar_wait(drain, 0, p.err, abort, /*honour_abort=*/false);
  }
  if (*abort && (w == kTcCopyK || w == kTcCopyV) && lane == 0) {
    const int ns = w == kTcCopyV ? kVS : kKS;
    const uint32_t full = w == kTcCopyV ? vraw_full : kraw_full;
    for (int k = 2 * n > ns ? 2 * n - ns : 0; k < 2 * n; ++k)
      mbar_wait(full + 8 * (k % ns), (uint32_t)((k / ns) & 1), p.err, abort, false, kWaitTimeoutNs / 8);
  }
  tc_fence_before();
  __syncthreads();
  if (w == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTcTmemCols);
  }
}

template <int KT, int VT>
KernelInfo rows_tc_kernel_info() {
  return KernelInfo{pa_rows_tc_kernel<KT, VT>, TcSmem<KT, VT>::kLaunch, 1, kRowThreads};
}

#define PA_DECLARE_ROWS_TC_LOOKUP(k, v) bool lookup_rows_tc_kernel_##k##_##v(KernelInfo* out);
PA_DECLARE_ROWS_TC_LOOKUP(1, 1) PA_DECLARE_ROWS_TC_LOOKUP(1, 2) PA_DECLARE_ROWS_TC_LOOKUP(1, 8)
PA_DECLARE_ROWS_TC_LOOKUP(2, 1) PA_DECLARE_ROWS_TC_LOOKUP(2, 2) PA_DECLARE_ROWS_TC_LOOKUP(2, 8)
PA_DECLARE_ROWS_TC_LOOKUP(8, 1) PA_DECLARE_ROWS_TC_LOOKUP(8, 2) PA_DECLARE_ROWS_TC_LOOKUP(8, 8)
#undef PA_DECLARE_ROWS_TC_LOOKUP

}  // namespace pa_split
