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
//   S        = Q K^T    tcgen05.mma M = 128 rows, N = 64 keys, K = 256 dims,
//                       fp32 in tensor memory (64 columns);
//   softmax  four warps, one thread per query row: the row's 64 logits come
//            from tensor memory into registers (no shuffles), causal mask,
//            lazy online maximum (raised only past 2^8; then that row of O is
//            rescaled in tensor memory), P as binary16 into shared memory;
//   O       += P V     tcgen05.mma M = 128 rows, N = 256 dims, K = 64 keys,
//                       fp32 in tensor memory (256 columns).
//
// Operands sit in shared memory in the MMA's canonical no-swizzle K-major
// layout (core matrices of 8 rows x 16 bytes): Q [rows][dims], K [keys][dims],
// V^T [dims][keys] and P [rows][keys].  Raw K/V row groups stream into a ring
// of stages with bulk copies (one lane of warp 0 refills a stage once every
// warp has dequantised it); each warp dequantises eight keys per tile: ldmatrix
// reads the raw quants (thread 4g+t gets four bytes of key g), the values are
// converted in registers and stmatrix writes them as core matrices (.trans
// for V), without bank conflicts.  That fixes a per-format order of the head
// dims inside each 32-dim window (dim_of below); Q is staged in K's order and O
// is written back through V's.
//
// Precision: Q, P and V (q * d rounded once) are binary16.  Quantised K is
// kept to about 2^-22: it is split as K = K_hi + K_lo, K_hi = q * d rounded to
// binary16 and K_lo = q * d - K_hi rounded once (a fused multiply-add), and S
// takes both products (16 more MMAs per tile, cheap on this tensor core), so
// large logits carry no K rounding.  Every product is accumulated in fp32.
#pragma once

#include "pa_rows_impl.cuh"

namespace pa_split {

constexpr uint32_t kTcTmemCols = 512;     // S at column 0 (64), O at column 256 (256)
constexpr uint32_t kTcOCol = 256;
constexpr uint32_t kTcIdescS = idesc_f16_f32(kRowTile, kTile);  // 128 x 64
constexpr uint32_t kTcIdescO = idesc_f16_f32(kRowTile, kD);     // 128 x 256

template <int KT, int VT>
struct TcSmem {
  static constexpr bool kKSplit = KT != PA_F16;                  // K_hi and K_lo
  static constexpr int kStageBytes = StageGeo<KT, VT>::kBytes;   // 64 keys raw: 4 K groups then 4 V groups
  static constexpr int kQ = 0;                                   // Q   [128][256] binary16: 64 KB
  static constexpr int kKh = kQ + kRowTile * kD * 2;             // K   [64][256]  (K_hi): 32 KB
  static constexpr int kKl = kKh + kTile * kD * 2;               // K_lo, then P (once S is done): 32 KB
  static constexpr int kP = kKSplit ? kKl : kKl;                 // P   [128][64]: 16 KB
  static constexpr int kVt = kKl + (kKSplit ? kTile * kD * 2 : kRowTile * kTile * 2);  // V^T [256][64]: 32 KB
  static constexpr int kRing = kVt + kD * kTile * 2;
  static constexpr int kFit = (232448 - 1024 - kAlign - kRing - 256) / kStageBytes;
  static constexpr int kStages = kFit > 3 ? 3 : kFit;
  static_assert(kStages >= 1, "tcgen05 row-tile stage does not fit");
  static constexpr int kBar = kRing + kStages * kStageBytes;    // full[kStages], s_done, pv_done, drain
  static constexpr int kMisc = kBar + (kStages + 3) * 8;        // abort, start[3], tmem base
  static constexpr int kTotal = kMisc + 32;
  static constexpr int kLaunch = kTotal + kAlign;
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

// Store four fragment matrices of slots s0 .. s0+3 (8 dims each) of the warp's
// eight keys: K as rows of the [keys][dims] tile, V transposed into the
// [dims][keys] tile.  Lane 8j + r gives the address of row r of matrix j.
template <bool kRoleV>
__device__ __forceinline__ void tc_store4(uint32_t dst, int w, int lane, int s0, uint32_t r0, uint32_t r1, uint32_t r2,
                                          uint32_t r3) {
  const int mj = lane >> 3, mr = lane & 7;
  if (kRoleV) stsm_x4_trans(dst + canon_off(8 * (s0 + mj) + mr, w, kTile / 8), r0, r1, r2, r3);
  else stsm_x4(dst + canon_off(8 * w + mr, s0 + mj, kD / 8), r0, r1, r2, r3);
}

// K_hi (rounded product) and K_lo (its exact remainder, rounded once) of exact
// quants v with scale d2; V: v * d2.
__device__ __forceinline__ uint32_t tc_hi(uint32_t v, uint32_t d2) { return hmul2(v, d2); }
__device__ __forceinline__ uint32_t tc_lo(uint32_t v, uint32_t d2, uint32_t hi) {
  return hfma2(v, d2, hi ^ 0x80008000u);
}

// Warp w's eight keys (8w .. 8w+7) of a raw 64-key stage region of format T
// (four row groups), as binary16 core matrices: V values q * d into the V^T
// tile (kRoleV), K exact for F16 or as K_hi / K_lo tiles for Q8_0 and Q4_0.
// Keys at or past n_keys are written as zeros.
template <int T, bool kRoleV>
__device__ __forceinline__ void tc_dequant_warp(uint32_t region, uint32_t dst, uint32_t dst_lo, int w, int lane,
                                                int n_keys) {
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
#pragma unroll
  for (int i = 0; i < C / 4; ++i) {
    uint32_t x[4];  // chunk 4i + j of key g, bytes 4t .. 4t+3 (thread 4g + t)
    ldsm_x4(lrow + (((4 * i + (lane >> 3)) ^ (lr & 7)) << 4), x);
    if constexpr (T == PA_F16) {  // chunk = slot, natural order
      if (!live) x[0] = x[1] = x[2] = x[3] = 0u;
      tc_store4<kRoleV>(dst, w, lane, 4 * i, x[0], x[1], x[2], x[3]);
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
      tc_store4<kRoleV>(dst, w, lane, 8 * i, h[0], h[1], h[2], h[3]);
      tc_store4<kRoleV>(dst, w, lane, 8 * i + 4, h[4], h[5], h[6], h[7]);
      if (!kRoleV) {
        tc_store4<false>(dst_lo, w, lane, 8 * i, l[0], l[1], l[2], l[3]);
        tc_store4<false>(dst_lo, w, lane, 8 * i + 4, l[4], l[5], l[6], l[7]);
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
        tc_store4<kRoleV>(dst, w, lane, 4 * c, h[0], h[1], h[2], h[3]);
        if (!kRoleV) tc_store4<false>(dst_lo, w, lane, 4 * c, l[0], l[1], l[2], l[3]);
      }
    }
  }
}

// ------------------------------------------------------------------ Q staging

// The row tile's 128 query rows (rows past the 6 * n_qtok real ones are zero)
// as binary16 in the [rows][dims] tile, each 32-dim window in K's dim order.
// Task = (row, window): eight float4 loads of the row's 32 dims, four slots out.
template <int KT>
__device__ __forceinline__ void tc_stage_q(const DecodeParams& p, int s, int head, int rt, uint32_t qsm, int tid) {
  const int R = kGqa * p.n_qtok;
#pragma unroll 1
  for (int task = tid; task < kRowTile * (kD / 32); task += kRowTile * 2) {
    const int row = task & (kRowTile - 1), win = task >> 7, rg = kRowTile * rt + row;
    float v[32];
    if (rg < R) {
      const float4* src = reinterpret_cast<const float4*>(
          p.q + (((long long)s * p.n_qtok + rg / kGqa) * p.n_q_heads + head * kGqa + rg % kGqa) * kD + 32 * win);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float4 f = __ldg(src + i);
        v[4 * i] = f.x; v[4 * i + 1] = f.y; v[4 * i + 2] = f.z; v[4 * i + 3] = f.w;
      }
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] = 0.f;
    }
#pragma unroll
    for (int sl = 0; sl < 4; ++sl) {
      uint32_t h[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int p0 = 8 * sl + 2 * k;
        h[k] = pack_half2(v[dim_of<KT>(p0)], v[dim_of<KT>(p0 + 1)]);
      }
      asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(qsm + canon_off(row, 4 * win + sl, kD / 8)),
                   "r"(h[0]), "r"(h[1]), "r"(h[2]), "r"(h[3]) : "memory");
    }
  }
}

// ------------------------------------------------------------------ the kernel

template <int KT, int VT>
__global__ void __launch_bounds__(kRowThreads, 1) pa_rows_tc_kernel(const __grid_constant__ DecodeParams p) {
  using SM = TcSmem<KT, VT>;
  using G = StageGeo<KT, VT>;
  constexpr int kStages = SM::kStages;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((kAlign - (raw & (kAlign - 1))) & (kAlign - 1));
  const uint32_t base = smem_u32(smem);
  const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
  const uint32_t bar_full = base + SM::kBar, bar_s = bar_full + 8 * kStages, bar_pv = bar_s + 8,
                 bar_drain = bar_pv + 8;
  volatile int* abort = reinterpret_cast<volatile int*>(smem + SM::kMisc);
  int* start = reinterpret_cast<int*>(smem + SM::kMisc + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + SM::kMisc + 16);
  const uint32_t ring = base + SM::kRing;

  const long long T = p.total_tiles;
  const int Gn = p.n_ctas;
  const long long a = (long long)blockIdx.x * T / Gn, b = (long long)(blockIdx.x + 1) * T / Gn;
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (tid == 0) {
    asm volatile("griddepcontrol.launch_dependents;");
    *abort = 0;
    for (int i = 0; i < kStages; ++i) mbar_init(bar_full + 8 * i, 1);
    mbar_init(bar_s, 1);
    mbar_init(bar_pv, 1);
    mbar_init(bar_drain, 1);
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
  RowPos pos;
  pos.s = start[0];
  pos.gi = start[1];
  pos.j = start[2];
  pos.L = any ? p.lens[pos.s] : 0;
  pos.nt = any ? row_seg_tiles(p, pos.L, pos.gi) : 0;

  // Raw stage copies (warp 0): tiles a .. a + kStages - 1 now, then tile
  // x + kStages once every warp has dequantised tile x from its slot.
  const uint64_t policy = l2_evict_first_policy();
  RowPos ipos = pos;
  long long issued = a;
  int ientry = -1;
  if (w == 0 && any) {
    ientry = row_entry(p, ipos, lane);
    for (; issued < b && issued < a + kStages; ++issued) {
      const int slot = (int)(issued - a);
      issue_stage<KT, VT>(p, ipos, ientry, ring + slot * G::kBytes, bar_full + 8 * slot, policy, lane);
      row_next(p, ipos);
      ientry = row_entry(p, ipos, lane);
    }
  }

  const int R = kGqa * p.n_qtok;
  const float scale_log2 = p.scale_log2;
  const uint32_t t_lane = (uint32_t)(32 * (w & 3)) << 16;  // this warp's tensor-memory lanes
  const uint32_t tS = tmem + t_lane, tO = tmem + kTcOCol + t_lane;
  int st = 0;
  uint32_t ph = 0, nt_done = 0;  // full-barrier ring position; tiles done (S / PV barrier parity)
  long long x = a;
  while (any && x < b) {
    const int s = pos.s, gi = pos.gi, L = pos.L, ntl = pos.nt;
    const int head = gi / p.n_row_tiles, rt = gi % p.n_row_tiles;
    const int l_dev = device_len(p, s);
    const int jb = pos.j, je = (int)((long long)ntl < jb + (b - x) ? (long long)ntl : jb + (b - x));
    const int seg = s * p.segs_per_seq + gi;
    const bool whole = (jb == 0 && je == ntl);
    tc_stage_q<KT>(p, s, head, rt, base + SM::kQ, tid);
    fence_proxy_async_smem();
    // softmax threads: warps 0..3, one query row each
    const int row = 32 * w + lane, rg = kRowTile * rt + row;
    const bool smx = w < 4 && kRowTile * rt + 32 * w < R;  // the warp holds a real row
    const int vis = rg < R ? L - p.n_qtok + rg / kGqa : -1;
    float m = -INFINITY, l = 0.f;

    for (int jt = jb; jt < je; ++jt) {
      const int k0 = jt * kTile, n_keys = min(kTile, L - k0);
      const uint32_t sk = ring + st * G::kBytes, sv = sk + G::kKBytes;
      mbar_wait(bar_full + 8 * st, ph, p.err, abort);
      tc_dequant_warp<KT, false>(sk, base + SM::kKh, base + SM::kKl, w, lane, n_keys);
      tc_dequant_warp<VT, true>(sv, base + SM::kVt, 0u, w, lane, n_keys);
      fence_proxy_async_smem();
      tc_fence_before();
      named_bar_sync(kRowBar, kRowThreads);  // Q, K and V^T tiles ready; the stage is free
      if (w == 0 && issued < b) {
        issue_stage<KT, VT>(p, ipos, ientry, ring + st * G::kBytes, bar_full + 8 * st, policy, lane);
        ++issued;
        row_next(p, ipos);
        ientry = row_entry(p, ipos, lane);
      }
      if (tid == 4 * 32) {  // S = Q K^T (+ Q K_lo^T)
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < kD / 16; ++ks)
          tc_mma_f16(tmem, smem_desc(base + SM::kQ + 256 * ks, 128, 4096),
                     smem_desc(base + SM::kKh + 256 * ks, 128, 4096), kTcIdescS, ks > 0);
        if (SM::kKSplit) {
#pragma unroll
          for (int ks = 0; ks < kD / 16; ++ks)
            tc_mma_f16(tmem, smem_desc(base + SM::kQ + 256 * ks, 128, 4096),
                       smem_desc(base + SM::kKl + 256 * ks, 128, 4096), kTcIdescS, 1);
        }
        tc_commit(bar_s);
      }
      if (smx) {
        mbar_wait(bar_s, nt_done & 1, p.err, abort);
        __syncwarp();  // tensor-memory loads are warp-wide
        tc_fence_after();
        uint32_t sv32[2][32];
        tmem_ld32(tS, sv32[0]);
        tmem_ld32(tS + 32, sv32[1]);
        tmem_ld_wait();
        float tmax = -INFINITY;
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const float v = (k0 + 32 * h + c <= vis) ? __uint_as_float(sv32[h][c]) * scale_log2 : -INFINITY;
            sv32[h][c] = __float_as_uint(v);
            tmax = fmaxf(tmax, v);
          }
        // Lazy maximum: raised (rarely, after a row's first tile) past 2^8.
        // The rows of O that hold weight are rescaled in tensor memory; the
        // tensor-memory loads and stores are warp-wide (.sync.aligned), so the
        // whole warp runs them when any of its rows rises.
        const bool raise = tmax > m + kLazy;
        const float al = raise ? ((m == -INFINITY) ? 1.f : ex2(m - tmax)) : 1.f;
        if (__any_sync(0xffffffffu, raise) && jt > jb) {
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
        }
        if (raise) {
          l *= al;
          m = tmax;
        }
        const float bm = (m == -INFINITY) ? 0.f : m;
#pragma unroll
        for (int kc = 0; kc < kTile / 8; ++kc) {  // P row, keys 8kc .. 8kc+7
          uint32_t ph4[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int c = 8 * kc + 2 * e;
            ph4[e] = pack_half2(ex2(__uint_as_float(sv32[c >> 5][c & 31]) - bm),
                                ex2(__uint_as_float(sv32[(c + 1) >> 5][(c + 1) & 31]) - bm));
            const float2 f = half2_bits_to_float2(ph4[e]);
            l += f.x + f.y;
          }
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(base + SM::kP + canon_off(row, kc, kTile / 8)),
                       "r"(ph4[0]), "r"(ph4[1]), "r"(ph4[2]), "r"(ph4[3]) : "memory");
        }
        fence_proxy_async_smem();
        tc_fence_before();
      }
      named_bar_sync(kRowBar, kRowThreads);  // P ready (and O rescaled)
      if (tid == 4 * 32) {  // O += P V
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk)
          tc_mma_f16(tmem + kTcOCol, smem_desc(base + SM::kP + 256 * kk, 128, 1024),
                     smem_desc(base + SM::kVt + 256 * kk, 128, 1024), kTcIdescO, (jt > jb || kk > 0) ? 1u : 0u);
        tc_commit(bar_pv);
      }
      mbar_wait(bar_pv, nt_done & 1, p.err, abort);  // every tile buffer is free again
      tc_fence_after();
      ++nt_done;
      if (++st == kStages) { st = 0; ph ^= 1; }
    }

    // ---- piece result: this thread's row
    const bool len_ok = l_dev == L;
    if (!len_ok && tid == 0) record_error(p.err, PA_ERR_BOUNDS);
    if (smx) {  // the whole warp reads O (warp-wide loads); real rows store it
      __syncwarp();
      const bool real = rg < R;
      const float lr = (len_ok && real) ? l : 0.f;
      const int t = real ? rg / kGqa : 0, hl = real ? rg % kGqa : 0;
      const long long orow = ((long long)s * p.n_qtok + t) * p.n_q_heads + head * kGqa + hl;
      float* dst;
      float inv;
      const int slot = (int)blockIdx.x + seg;
      if (whole) {
        dst = p.out + orow * kD;
        inv = lr > 0.f ? 1.f / lr : 0.f;
        if (real && p.lse) p.lse[orow] = lr > 0.f ? (m + log2f(lr)) * kLn2 : -INFINITY;
      } else {
        dst = p.part_o + ((long long)slot * p.rows_per_seg + row) * kD;
        inv = len_ok ? 1.f : 0.f;
        p.part_ml[(long long)slot * p.rows_per_seg + row] = real ? make_float2(m, lr) : make_float2(-INFINITY, 0.f);
      }
      const bool store = real || !whole;  // padding rows of a split piece store zeros-weighted partials
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
    }
    tc_fence_before();
    x += je - jb;
    pos.j = je - 1;
    row_next(p, pos);
  }
  // Every issued tile was waited for above, unless a wait expired (the abort
  // flag): then wait, with a bound, for the copies and MMAs still in flight
  // before the stages and tensor memory are released.
  if (*abort && tid == 0) {
    drain_ring<kStages>(p, bar_full, abort, (int)((issued - a) % kStages), (uint32_t)(((issued - a) / kStages) & 1),
                        issued - a);
  }
  if (*abort && tid == 4 * 32) {
    tc_commit(bar_drain);
    mbar_wait(bar_drain, 0, p.err, abort, /*honour_abort=*/false);
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
