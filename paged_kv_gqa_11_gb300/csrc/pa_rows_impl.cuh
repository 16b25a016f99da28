// Row tiles: decode of 9 to 96 query tokens per sequence (sm_103a).
//
// Batches of more than eight query tokens -- n-gram drafts verify up to 65
// tokens -- do not fit the decode kernels' 48-row tiles, and the pages route
// them to the decode kernel's row tiles, faster than a chunked prefill up to 96
// query tokens (llama.cpp fork PR #2, the commit on KV-streaming ubatches of
// more than 8 tokens).  The computation is the same causal decode: query token
// t of n_qtok sits at position L - n_qtok + t and sees keys 0 .. L - n_qtok + t.
//
// With 6 * n_qtok query rows per KV head (54 to 576) the rows are the MMA's M
// dimension.  A segment is (sequence, KV head, row tile of 128 rows); its tiles
// are the 64-key tiles its last row can see, so early row tiles of a long
// verify batch stop short of the newest keys.  Segments are cut into pieces by
// the same stream-K planner as the decode kernels and merged by the same LSE
// merge.
//
// A CTA is eight warps of 16 query rows each (eight warps, two per
// sub-partition, leave each thread the registers for its 16 x 256 O tile; a
// ninth, producer warp would cut that to 168).  Raw 64-key K/V tiles of one KV
// head stream into a ring of stages with bulk copies, issued by one lane of warp
// 0 when a tile's first barrier shows that every warp is done with the stage the
// previous tile used; the table entries are looked up a tile ahead.  Per tile
// the warps first dequantise K and V once, together, into binary16 tiles in
// shared memory (F16 pools are read where they land), then each warp
// computes S = Q K^T for its rows (mma.sync m16n8k16, fp32 accumulation), masks
// causally, runs a lazy online softmax (the reference maximum of a row is
// raised only past 2^8) and accumulates O += P V with the probabilities kept in
// registers as the A operand.  O (16 rows x 256 dims) stays in registers.
//
// Precision: Q, P and the dequantised V values (q * d rounded once) are
// binary16.  Quantised K stays exact: the tile holds its integer quants, each
// 32-dim block's two k-steps accumulate into a fresh fp32 tile and the block
// scale multiplies it in fp32 (as the decode kernels keep K exact), so that
// large logits carry no K rounding.  Every product is accumulated in fp32.
#pragma once

#include "pa_decode_impl.cuh"

namespace pa_split {

constexpr int kRowTile = 128;                  // query rows per row tile
constexpr int kRowWarps = kRowTile / 16;       // consumer warps, 16 rows each
constexpr int kRowThreads = kRowWarps * 32;
constexpr int kMaxRowsQTok = 96;               // query tokens the row tiles take
constexpr uint32_t kRowBar = 1;                // named barrier of the consumer warps

template <int KT, int VT>
struct RowSmem {
  static constexpr bool kKDirect = KT == PA_F16;  // K read where it lands
  static constexpr bool kVDirect = VT == PA_F16;
  static constexpr int kStageBytes = StageGeo<KT, VT>::kBytes;  // 64 keys: 4 K groups then 4 V groups
  static constexpr int kQ = 0;                                   // Q [128 rows][256] binary16, swizzled
  static constexpr int kKf = kQ + kRowTile * kD * 2;             // K [64 keys][256] binary16
  static constexpr int kVf = kKf + (kKDirect ? 0 : kTile * kD * 2);
  static constexpr int kKs = kVf + (kVDirect ? 0 : kTile * kD * 2);  // K scales [8 blocks][64 keys] fp32
  static constexpr int kRing = kKs + (kKDirect ? 0 : 8 * kTile * 4);
  static constexpr int kFit = (232448 - 1024 - kAlign - kRing - 128) / kStageBytes;
  static constexpr int kStages = kFit > 4 ? 4 : kFit;
  static_assert(kStages >= 2, "row-tile stage ring does not fit");
  static_assert(kRing % kAlign == 0, "ring alignment");
  static constexpr int kBar = kRing + kStages * kStageBytes;
  static constexpr int kMisc = kBar + 2 * kStages * 8;
  static constexpr int kTotal = kMisc + 32;
  static constexpr int kLaunch = kTotal + kAlign;
};

// Byte offset of 16-byte chunk c (8 dims) of row r in a [rows][256] binary16
// tile: chunks of a row are XOR-swizzled by r % 8 so that the eight rows an
// ldmatrix phase reads fall in eight different bank groups.  The pool's F16
// row groups use the same arrangement, so a stage of F16 rows is such a tile.
__device__ __forceinline__ uint32_t tile16_off(int r, int c) { return (uint32_t)(r * 512 + ((c ^ (r & 7)) << 4)); }

// ------------------------------------------------------------------ the walk

// Tiles of segment gi (KV head gi / n_row_tiles, row tile gi % n_row_tiles) of
// a sequence of length L: the 64-key tiles that the tile's last row sees.
__device__ __forceinline__ int row_seg_tiles(const DecodeParams& p, int L, int gi) {
  const int rt = gi % p.n_row_tiles;
  const int t_last = min(p.n_qtok - 1, (kRowTile * (rt + 1) - 1) / kGqa);
  return (L - p.n_qtok + t_last + 1 + kTile - 1) / kTile;
}

struct RowPos {
  int s, gi, j, L, nt;
};

// Position of global tile x: whole sequences are skipped by their tile
// count (every KV head has the same row tiles).
__device__ __forceinline__ RowPos row_locate(const DecodeParams& p, long long x) {
  long long base = 0;
  for (int s = 0; s < p.n_seq; ++s) {
    const int L = p.lens[s];
    long long per_head = 0;
    for (int rt = 0; rt < p.n_row_tiles; ++rt) per_head += row_seg_tiles(p, L, rt);
    if (x >= base + per_head * p.n_kv_heads) {
      base += per_head * p.n_kv_heads;
      continue;
    }
    for (int gi = 0; gi < p.segs_per_seq; ++gi) {
      const int nt = row_seg_tiles(p, L, gi);
      if (x < base + nt) return RowPos{s, gi, (int)(x - base), L, nt};
      base += nt;
    }
  }
  return RowPos{p.n_seq, 0, 0, 0, 0};
}

__device__ __forceinline__ void row_next(const DecodeParams& p, RowPos& t) {
  if (++t.j < t.nt) return;
  t.j = 0;
  if (++t.gi == p.segs_per_seq) {
    t.gi = 0;
    if (++t.s >= p.n_seq) return;
    t.L = p.lens[t.s];
  }
  t.nt = row_seg_tiles(p, t.L, t.gi);
}

// ------------------------------------------------------------------ stage copies

// Table entry of row group `lane` (0..3) of tile t, or -1 for lanes past the
// tile's row groups.
__device__ __forceinline__ int row_entry(const DecodeParams& p, const RowPos& t, int lane) {
  const int k0 = t.j * kTile, n = min(kTile, t.L - k0);
  if (lane >= 4 || lane * kGroup >= n || t.s >= p.n_seq) return -1;
  return __ldg(p.table + (long long)t.s * p.table_stride + (k0 + lane * kGroup) / p.page_size);
}

// Warp 0 fills one stage with tile t (four row groups of one KV head, K then
// V); tb: this lane's table entry (row_entry).  Groups past the sequence's
// last key are not copied; a group whose entry is outside the pool is
// zero-filled and reported.  The whole warp calls this.
template <int KT, int VT>
__device__ __forceinline__ void issue_stage(const DecodeParams& p, const RowPos& t, int tb, uint32_t sk, uint32_t fb,
                                            uint64_t policy, int lane) {
  using G = StageGeo<KT, VT>;
  constexpr int RK = Fmt<KT>::kRow, RV = Fmt<VT>::kRow;
  const int head = t.gi / p.n_row_tiles;
  const int k0 = t.j * kTile, n = min(kTile, t.L - k0), ng = (n + kGroup - 1) / kGroup;
  const uint32_t sv = sk + G::kKBytes;
  const bool mine = lane < ng;
  const bool ok = !mine || (tb >= 0 && tb < p.n_blocks);
  const unsigned bad = __ballot_sync(0xffffffffu, !ok);
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
  __syncwarp();
  if (lane == 0) mbar_arrive_expect_tx(fb, (uint32_t)n_good * (G::kKGroup + G::kVGroup));
  __syncwarp();
  if (mine && ok) {
    const long long row = ((long long)tb * p.n_kv_heads + head) * p.page_size + (k0 + lane * kGroup) % p.page_size;
    bulk_g2s_hint(sk + lane * G::kKGroup, p.k_pool + row * RK, G::kKGroup, fb, policy);
    bulk_g2s_hint(sv + lane * G::kVGroup, p.v_pool + row * RV, G::kVGroup, fb, policy);
  }
  __syncwarp();
}

// ------------------------------------------------------------------ dequantisation into binary16 tiles

// One 16-byte chunk of a stored row (format T, chunk c) -> its values times
// the block scale d, as 8 or 16 binary16 values in natural dim order, written
// to the [64][256] tile at key `key`.  Q8_0: chunk c holds dims 16c..16c+15
// (int8, block c/2).  Q4_0: chunk c is block c: byte j holds dim j (low
// nibble) and dim j + 16 (high nibble).
// kScaled = false keeps the exact integer quants (K; the scale is applied
// after the products).
template <int T, bool kScaled>
__device__ __forceinline__ void dequant_chunk(uint4 in, uint32_t d2, uint32_t tile, int key, int c) {
  const uint32_t w[4] = {in.x, in.y, in.z, in.w};
  auto sc = [&](uint32_t h) { return kScaled ? hmul2(h, d2) : h; };
  if constexpr (T == PA_Q8_0) {
    uint32_t h[8];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint32_t x = w[k] ^ 0x80808080u;  // int8 -> 128 + x as an unsigned byte
      h[2 * k] = sc(hadd2(prmt(x, kMagic64, 0x4140), kHalf2_m1152));      // dims 4k, 4k+1
      h[2 * k + 1] = sc(hadd2(prmt(x, kMagic64, 0x4342), kHalf2_m1152));  // dims 4k+2, 4k+3
    }
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(tile + tile16_off(key, 2 * c)), "r"(h[0]),
                 "r"(h[1]), "r"(h[2]), "r"(h[3]) : "memory");
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(tile + tile16_off(key, 2 * c + 1)), "r"(h[4]),
                 "r"(h[5]), "r"(h[6]), "r"(h[7]) : "memory");
  } else {  // Q4_0
    uint32_t lo[8], hi[8];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint32_t t0 = prmt(w[k], 0u, 0x4140), t1 = prmt(w[k], 0u, 0x4342);  // bytes (4k, 4k+1), (4k+2, 4k+3)
      lo[2 * k] = sc(hadd2(and_or(t0, 0x000f000fu, 0x64006400u), kHalf2_m1032));
      lo[2 * k + 1] = sc(hadd2(and_or(t1, 0x000f000fu, 0x64006400u), kHalf2_m1032));
      hi[2 * k] = sc(hfma2(and_or(t0, 0x00f000f0u, 0x64006400u), kHalf2_1_16, kHalf2_m72));
      hi[2 * k + 1] = sc(hfma2(and_or(t1, 0x00f000f0u, 0x64006400u), kHalf2_1_16, kHalf2_m72));
    }
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(tile + tile16_off(key, 4 * c + q)),
                   "r"(lo[4 * q]), "r"(lo[4 * q + 1]), "r"(lo[4 * q + 2]), "r"(lo[4 * q + 3]) : "memory");
      asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(tile + tile16_off(key, 4 * c + 2 + q)),
                   "r"(hi[4 * q]), "r"(hi[4 * q + 1]), "r"(hi[4 * q + 2]), "r"(hi[4 * q + 3]) : "memory");
    }
  }
}

// Dequantise keys 8w .. 8w+7 of a raw 64-key stage (four row groups of format
// T) into the binary16 tile; keys at or past n_keys become zeros (their
// probability is 0, and V must be finite).  V (kRoleV): values q * d.  K:
// the integer quants, with the scales as fp32 in ks[block][key].
template <int T, bool kRoleV>
__device__ __forceinline__ void dequant_warp(uint32_t stage, uint32_t tile, uint32_t ks, int w, int lane,
                                             int n_keys) {
  constexpr int C = Fmt<T>::kRowQ / 16;  // chunks per row: 16 (Q8_0) or 8 (Q4_0)
  constexpr int GB = pa_layout::group_bytes<T>();
#pragma unroll
  for (int i = 0; i < 8 * C / 32; ++i) {
    const int idx = lane + 32 * i, kl = idx / C, c = idx % C;
    const int key = 8 * w + kl, grp = key / kGroup, r = key % kGroup;
    const uint32_t g0 = stage + grp * GB;
    const int b = T == PA_Q8_0 ? c >> 1 : c;
    if (key >= n_keys) {
      const int outs = T == PA_Q8_0 ? 2 : 4, oc0 = T == PA_Q8_0 ? 2 * c : 4 * c;
      for (int q = 0; q < outs; ++q) sts128_zero(tile + tile16_off(key, oc0 + q));
      if (!kRoleV && (T == PA_Q4_0 || (c & 1) == 0))
        asm volatile("st.shared.f32 [%0], %1;" ::"r"(ks + (b * kTile + key) * 4), "f"(0.f) : "memory");
      continue;
    }
    const uint4 in = lds128(g0 + pa_layout::chunk_offset(Fmt<T>::kScales, Fmt<T>::kRowQ, r, c));
    uint16_t dh;
    const uint32_t so = kRoleV ? pa_layout::v_scale_offset(r, b) : pa_layout::k_scale_offset(r, b);
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(dh) : "r"(g0 + so));
    const uint32_t d2 = (uint32_t)dh | ((uint32_t)dh << 16);
    dequant_chunk<T, kRoleV>(in, d2, tile, key, c);
    if (!kRoleV && (T == PA_Q4_0 || (c & 1) == 0))
      asm volatile("st.shared.f32 [%0], %1;" ::"r"(ks + (b * kTile + key) * 4),
                   "f"(__half2float(__ushort_as_half(dh))) : "memory");
  }
}

// F16 V read where it lands: zero the rows of keys n_keys .. 63 that warp w
// owns (8w .. 8w+7), so that masked keys carry finite values.
__device__ __forceinline__ void zero_f16_rows(uint32_t stage_v, int w, int lane, int n_keys) {
  if (8 * w + 7 < n_keys) return;
  for (int i = lane; i < 8 * 32; i += 32) {
    const int key = 8 * w + i / 32, c = i % 32;
    if (key >= n_keys) sts128_zero(stage_v + tile16_off(key, c));
  }
  fence_proxy_async_smem();  // the stage is refilled by bulk copies later
}

// ------------------------------------------------------------------ Q staging

// Warp w's 16 query rows (row tile rt of KV head `head` of sequence s; rows
// past the 6 * n_qtok real ones are zero) as binary16 in its [16][256] slice.
static __device__ __noinline__ void stage_q_rows(const DecodeParams& p, int s, int head, int rt, int w, uint32_t qsm,
                                          int lane) {
  const int R = kGqa * p.n_qtok;
#pragma unroll 1
  for (int bt = 0; bt < 4; ++bt) {  // four batches of eight float4 loads in flight per lane
    float4 v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int f = lane + 32 * (8 * bt + i), r = f >> 6, c4 = f & 63;
      const int rg = kRowTile * rt + 16 * w + r;
      v[i] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (rg < R) {
        const int t = rg / kGqa, hl = rg % kGqa;
        v[i] = __ldg(reinterpret_cast<const float4*>(
                         p.q + (((long long)s * p.n_qtok + t) * p.n_q_heads + head * kGqa + hl) * kD) + c4);
      }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int f = lane + 32 * (8 * bt + i), r = f >> 6, c4 = f & 63;
      const uint32_t addr = qsm + tile16_off(r, c4 >> 1) + (c4 & 1) * 8;
      asm volatile("st.shared.v2.b32 [%0], {%1, %2};" ::"r"(addr), "r"(pack_half2(v[i].x, v[i].y)),
                   "r"(pack_half2(v[i].z, v[i].w)) : "memory");
    }
  }
  __syncwarp();
}

// ------------------------------------------------------------------ consumer

template <int KT, int VT>
__device__ void consume_rows(const DecodeParams& p, uint32_t base, uint32_t bar_full, volatile int* abort,
                             long long a, long long b, RowPos pos) {
  using SM = RowSmem<KT, VT>;
  using G = StageGeo<KT, VT>;
  constexpr int kStages = SM::kStages;
  const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
  const int g4 = lane >> 2, t4 = lane & 3;
  const uint32_t qsm = base + SM::kQ + w * 16 * 512;
  const uint32_t ring = base + SM::kRing;
  const int R = kGqa * p.n_qtok;
  // this lane's ldmatrix row / chunk within a matrix quad (see the fragment maps below)
  const int lq = lane >> 3, l7 = lane & 7;
  const float scale_log2 = p.scale_log2;
  // Stage copies (warp 0): tiles a .. a + kStages - 2 now, then tile
  // x + kStages - 1 at tile x's first barrier, into the slot tile x - 1 used.
  const uint64_t policy = l2_evict_first_policy();
  RowPos ipos = pos;      // the next tile to issue
  long long issued = a;   // its index
  int ientry = -1;        // its row groups' table entries (warp 0, lanes 0..3)
  if (w == 0) {
    ientry = row_entry(p, ipos, lane);
    for (; issued < b && issued < a + kStages - 1; ++issued) {
      const int slot = (int)((issued - a) % kStages);
      issue_stage<KT, VT>(p, ipos, ientry, ring + slot * G::kBytes, bar_full + 8 * slot, policy, lane);
      row_next(p, ipos);
      ientry = row_entry(p, ipos, lane);
    }
  }
  int st = 0;
  uint32_t ph = 0;
  long long x = a;
  while (x < b) {
    const int s = pos.s, gi = pos.gi, L = pos.L, ntl = pos.nt;
    const int head = gi / p.n_row_tiles, rt = gi % p.n_row_tiles;
    const int l_dev = device_len(p, s);
    const int jb = pos.j, je = (int)((long long)ntl < jb + (b - x) ? (long long)ntl : jb + (b - x));
    const int seg = s * p.segs_per_seq + gi;
    const bool whole = (jb == 0 && je == ntl);
    stage_q_rows(p, s, head, rt, w, qsm, lane);
    // rows g4 and g4 + 8 of this warp: global row, token, last visible key
    int vis[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int rg = kRowTile * rt + 16 * w + g4 + 8 * h;
      vis[h] = rg < R ? L - p.n_qtok + rg / kGqa : -1;
    }
    float o[32][4];
#pragma unroll
    for (int i = 0; i < 32; ++i)
#pragma unroll
      for (int c = 0; c < 4; ++c) o[i][c] = 0.f;
    float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};

    for (int jt = jb; jt < je; ++jt) {
      const int k0 = jt * kTile, n_keys = min(kTile, L - k0);
      const uint32_t sk = ring + st * G::kBytes, sv = sk + G::kKBytes;
      // Every warp is done with the previous tile: its binary16 tiles and the
      // stage it used are free; refill that stage a ring ahead.
      named_bar_sync(kRowBar, kRowWarps * 32);
      if (w == 0 && issued < b) {
        const int slot = (int)((issued - a) % kStages);
        issue_stage<KT, VT>(p, ipos, ientry, ring + slot * G::kBytes, bar_full + 8 * slot, policy, lane);
        ++issued;
        row_next(p, ipos);
        ientry = row_entry(p, ipos, lane);
      }
      mbar_wait(bar_full + 8 * st, ph, p.err, abort);
      if constexpr (!SM::kKDirect) dequant_warp<KT, false>(sk, base + SM::kKf, base + SM::kKs, w, lane, n_keys);
      if constexpr (!SM::kVDirect) dequant_warp<VT, true>(sv, base + SM::kVf, 0u, w, lane, n_keys);
      else zero_f16_rows(sv, w, lane, n_keys);
      named_bar_sync(kRowBar, kRowWarps * 32);  // the tile's K and V are ready
      const uint32_t kt = SM::kKDirect ? sk : base + SM::kKf;
      const uint32_t vt = SM::kVDirect ? sv : base + SM::kVf;

      // ---- S = Q K^T: 16 rows x 64 keys (8 n-tiles of 8 keys)
      float sc[8][4];
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int c = 0; c < 4; ++c) sc[i][c] = 0.f;
      // one k-step of 16 dims into acc (A: rows 0-7 / 8-15 by lq & 1, dims by
      // lq >> 1; B: keys 16np + 0-7 / 8-15 by lq >> 1, dims by lq & 1)
      auto kstep = [&](float (&acc)[8][4], int ks) {
        uint32_t A[4];
        ldsm_x4(qsm + tile16_off(8 * (lq & 1) + l7, 2 * ks + (lq >> 1)), A);
#pragma unroll
        for (int np = 0; np < 4; ++np) {
          uint32_t B[4];
          ldsm_x4(kt + tile16_off(16 * np + 8 * (lq >> 1) + l7, 2 * ks + (lq & 1)), B);
          mma_16816(acc[2 * np], A, B[0], B[1]);
          mma_16816(acc[2 * np + 1], A, B[2], B[3]);
        }
      };
      if constexpr (SM::kKDirect) {
#pragma unroll
        for (int ks = 0; ks < 16; ++ks) kstep(sc, ks);
      } else {
        const uint32_t ksc = base + SM::kKs + (2 * t4) * 4;
#pragma unroll 1
        for (int bk = 0; bk < 8; ++bk) {  // 32-dim blocks: exact integer products, then d in fp32
          float tb[8][4];
#pragma unroll
          for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int c = 0; c < 4; ++c) tb[i][c] = 0.f;
          kstep(tb, 2 * bk);
          kstep(tb, 2 * bk + 1);
#pragma unroll
          for (int nt = 0; nt < 8; ++nt) {
            const uint2 dk = lds64(ksc + (bk * kTile + 8 * nt) * 4);  // keys 8nt + 2t4, +1
            const float d0 = __uint_as_float(dk.x), d1 = __uint_as_float(dk.y);
            sc[nt][0] = fmaf(d0, tb[nt][0], sc[nt][0]);
            sc[nt][1] = fmaf(d1, tb[nt][1], sc[nt][1]);
            sc[nt][2] = fmaf(d0, tb[nt][2], sc[nt][2]);
            sc[nt][3] = fmaf(d1, tb[nt][3], sc[nt][3]);
          }
        }
      }
      // ---- mask, lazy online softmax, P
      float tmax[2] = {-INFINITY, -INFINITY};
#pragma unroll
      for (int nt = 0; nt < 8; ++nt)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int h = c >> 1, key = k0 + 8 * nt + 2 * t4 + (c & 1);
          const float v = key <= vis[h] ? sc[nt][c] * scale_log2 : -INFINITY;
          sc[nt][c] = v;
          tmax[h] = fmaxf(tmax[h], v);
        }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        tmax[h] = fmaxf(tmax[h], __shfl_xor_sync(0xffffffffu, tmax[h], 1));
        tmax[h] = fmaxf(tmax[h], __shfl_xor_sync(0xffffffffu, tmax[h], 2));
        if (tmax[h] > m[h] + kLazy) {  // rare after the first tile: raise and rescale this row
          const float al = (m[h] == -INFINITY) ? 1.f : ex2(m[h] - tmax[h]);
          m[h] = tmax[h];
          l[h] *= al;
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            o[i][2 * h] *= al;
            o[i][2 * h + 1] *= al;
          }
        }
      }
      const float b0 = m[0] == -INFINITY ? 0.f : m[0], b1 = m[1] == -INFINITY ? 0.f : m[1];
      uint32_t pa[8][2];  // P of n-tile nt: rows g4 (0) and g4+8 (1), keys 2t4, 2t4+1
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        pa[nt][0] = pack_half2(ex2(sc[nt][0] - b0), ex2(sc[nt][1] - b0));
        pa[nt][1] = pack_half2(ex2(sc[nt][2] - b1), ex2(sc[nt][3] - b1));
        const float2 f0 = half2_bits_to_float2(pa[nt][0]), f1 = half2_bits_to_float2(pa[nt][1]);
        l[0] += f0.x + f0.y;
        l[1] += f1.x + f1.y;
      }
      // ---- O += P V: k-steps of 16 keys, 32 n-tiles of 8 dims
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const uint32_t A[4] = {pa[2 * kk][0], pa[2 * kk][1], pa[2 * kk + 1][0], pa[2 * kk + 1][1]};
#pragma unroll
        for (int dp = 0; dp < 16; ++dp) {
          uint32_t B[4];  // keys 16kk + 0-7 / 8-15 (lq & 1) x dims 16dp + 0-7 / 8-15 (lq >> 1), transposed
          ldsm_x4_trans(vt + tile16_off(16 * kk + 8 * (lq & 1) + l7, 2 * dp + (lq >> 1)), B);
          mma_16816(o[2 * dp], A, B[0], B[1]);
          mma_16816(o[2 * dp + 1], A, B[2], B[3]);
        }
      }
      if (++st == kStages) { st = 0; ph ^= 1; }
    }

    // ---- piece result: rows g4, g4 + 8 of this warp
    const bool len_ok = l_dev == L;
    if (!len_ok && lane == 0) record_error(p.err, PA_ERR_BOUNDS);
    const int slot = (int)blockIdx.x + seg;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float lr = l[h];
      lr += __shfl_xor_sync(0xffffffffu, lr, 1);
      lr += __shfl_xor_sync(0xffffffffu, lr, 2);
      if (!len_ok) lr = 0.f;
      const int row = 16 * w + g4 + 8 * h, rg = kRowTile * rt + row;
      float* dst;
      float inv;
      if (whole) {
        if (rg >= R) continue;
        const int t = rg / kGqa, hl = rg % kGqa;
        const long long orow = ((long long)s * p.n_qtok + t) * p.n_q_heads + head * kGqa + hl;
        dst = p.out + orow * kD;
        inv = lr > 0.f ? 1.f / lr : 0.f;
        if (t4 == 0 && p.lse) p.lse[orow] = lr > 0.f ? (m[h] + log2f(lr)) * kLn2 : -INFINITY;
      } else {
        dst = p.part_o + ((long long)slot * p.rows_per_seg + row) * kD;
        inv = len_ok ? 1.f : 0.f;
        if (t4 == 0) p.part_ml[(long long)slot * p.rows_per_seg + row] = make_float2(m[h], lr);
      }
#pragma unroll
      for (int nt = 0; nt < 32; ++nt)
        *reinterpret_cast<float2*>(dst + 8 * nt + 2 * t4) = make_float2(o[nt][2 * h] * inv, o[nt][2 * h + 1] * inv);
    }
    x += je - jb;
    pos.j = je - 1;
    row_next(p, pos);
  }
  // Every issued tile was waited for above, unless a wait expired (the abort
  // flag): then wait, with a bound, for the copies still in flight so that
  // none lands after the CTA retires.
  if (w == 0 && lane == 0 && *abort)
    drain_ring<kStages>(p, bar_full, abort, (int)((issued - a) % kStages), (uint32_t)(((issued - a) / kStages) & 1),
                        issued - a);
}

// ------------------------------------------------------------------ the row-tile kernel

template <int KT, int VT>
__global__ void __launch_bounds__(kRowThreads, 1) pa_rows_decode_kernel(const __grid_constant__ DecodeParams p) {
  using SM = RowSmem<KT, VT>;
  constexpr int kStages = SM::kStages;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((kAlign - (raw & (kAlign - 1))) & (kAlign - 1));
  const int tid = threadIdx.x;
  const uint32_t base = smem_u32(smem);
  const uint32_t bar_full = base + SM::kBar;
  volatile int* abort = reinterpret_cast<volatile int*>(smem + SM::kMisc);
  int* start = reinterpret_cast<int*>(smem + SM::kMisc + 4);

  const long long T = p.total_tiles;
  const int Gn = p.n_ctas;
  const long long a = (long long)blockIdx.x * T / Gn, b = (long long)(blockIdx.x + 1) * T / Gn;
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (tid == 0) {
    asm volatile("griddepcontrol.launch_dependents;");
    *abort = 0;
    for (int i = 0; i < kStages; ++i) mbar_init(bar_full + 8 * i, 1);
    fence_mbar_init();
    const RowPos r = row_locate(p, a);
    start[0] = r.s;
    start[1] = r.gi;
    start[2] = r.j;
  }
  __syncthreads();
  if (start[0] >= p.n_seq) return;  // an empty range (the planner gives every CTA a tile)
  RowPos pos;
  pos.s = start[0];
  pos.gi = start[1];
  pos.j = start[2];
  pos.L = p.lens[pos.s];
  pos.nt = row_seg_tiles(p, pos.L, pos.gi);
  consume_rows<KT, VT>(p, base, bar_full, abort, a, b, pos);
}

template <int KT, int VT>
KernelInfo rows_kernel_info() {
  return KernelInfo{pa_rows_decode_kernel<KT, VT>, RowSmem<KT, VT>::kLaunch, 1, kRowThreads};
}

#define PA_DECLARE_ROWS_LOOKUP(k, v) bool lookup_rows_kernel_##k##_##v(KernelInfo* out);
PA_DECLARE_ROWS_LOOKUP(1, 1) PA_DECLARE_ROWS_LOOKUP(1, 2) PA_DECLARE_ROWS_LOOKUP(1, 8)
PA_DECLARE_ROWS_LOOKUP(2, 1) PA_DECLARE_ROWS_LOOKUP(2, 2) PA_DECLARE_ROWS_LOOKUP(2, 8)
PA_DECLARE_ROWS_LOOKUP(8, 1) PA_DECLARE_ROWS_LOOKUP(8, 2) PA_DECLARE_ROWS_LOOKUP(8, 8)
#undef PA_DECLARE_ROWS_LOOKUP

}  // namespace pa_split
