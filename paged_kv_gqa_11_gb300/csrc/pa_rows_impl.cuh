// Row tiles: the tile walk and stage copies shared by the row-tile kernel
// (pa_rows_tc.cuh), which decodes 9 to 96 query tokens per sequence.
//
// Batches of more than eight query tokens -- n-gram drafts verify up to 65
// tokens -- take the decode kernel's row tiles, which the pages find faster
// than a chunked prefill up to 96 query tokens (llama.cpp fork PR #2, the
// commit on KV-streaming ubatches of more than 8 tokens).  With 6 * n_qtok
// query rows per KV head the rows are the MMA's M dimension: a segment is
// (sequence, KV head, row tile of 128 rows), and its tiles are the 64-key tiles
// its last row can see, so early row tiles of a long verify batch stop short of
// the newest keys.  Segments are cut into pieces by the same stream-K planner as
// the decode kernels and merged by the same LSE merge.
#pragma once

#include "pa_decode_impl.cuh"

namespace pa_split {

constexpr int kRowTile = 128;                  // query rows per row tile
constexpr int kRowKeys = 64;                   // keys per row-tile key tile
constexpr int kStageKeys = 32;                 // keys per copy stage (two row groups); two stages per tile
constexpr int kMaxRowsQTok = 96;               // query tokens the row tiles take

// A K stage holds two K row groups (half a key tile); a V stage the same two
// V row groups.  K and V stages are separate rings.
template <int KT, int VT>
struct RowStageGeo {
  static constexpr int kKBytes = 2 * pa_layout::group_bytes<KT>();
  static constexpr int kVBytes = 2 * pa_layout::group_bytes<VT>();
};

// ------------------------------------------------------------------ the walk

// Tiles of segment gi (KV head gi / n_row_tiles, row tile gi % n_row_tiles) of
// a sequence of length L: the 64-key tiles that the tile's last row sees.
__device__ __forceinline__ int row_seg_tiles(const DecodeParams& p, int L, int gi) {
  const int rt = gi % p.n_row_tiles;
  const int t_last = min(p.n_qtok - 1, (kRowTile * (rt + 1) - 1) / kGqa);
  return (L - p.n_qtok + t_last + 1 + kRowKeys - 1) / kRowKeys;
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

// Table entry of row group `lane` (0..1) of stage `half` (0..1) of key tile
// t, or -1 for lanes past the stage's row groups.
__device__ __forceinline__ int row_entry(const DecodeParams& p, const RowPos& t, int half, int lane) {
  const int k0 = t.j * kRowKeys + half * kStageKeys, n = min(kStageKeys, t.L - k0);
  if (lane >= 2 || lane * kGroup >= n || t.s >= p.n_seq) return -1;
  return __ldg(p.table + (long long)t.s * p.table_stride + (k0 + lane * kGroup) / p.page_size);
}

// Fill one stage with half `half` of key tile t: its two row groups of one KV
// head from the K pool (kIsV false, format T = the K format) or the V pool;
// tb: this lane's table entry (row_entry).  Groups past the sequence's last
// key are not copied (a stage wholly past it completes with no bytes); a group
// whose entry is outside the pool is zero-filled and reported.  The whole warp
// calls this.
template <int T, bool kIsV>
__device__ __forceinline__ void issue_half(const DecodeParams& p, const RowPos& t, int half, int tb, uint32_t dst,
                                           uint32_t fb, uint64_t policy, int lane) {
  constexpr int GB = pa_layout::group_bytes<T>(), RB = Fmt<T>::kRow;
  const int head = t.gi / p.n_row_tiles;
  const int k0 = t.j * kRowKeys + half * kStageKeys, n = min(kStageKeys, t.L - k0);
  const int ng = n > 0 ? (n + kGroup - 1) / kGroup : 0;
  const bool mine = lane < ng;
  const bool ok = !mine || (tb >= 0 && tb < p.n_blocks);
  const unsigned bad = __ballot_sync(0xffffffffu, !ok);
  if (bad) {
    if (lane == 0) record_error(p.err, PA_ERR_BOUNDS);
    for (int q = 0; q < 2; ++q) {
      if (!((bad >> q) & 1)) continue;
      for (int i = lane; i < GB / 16; i += 32) sts128_zero(dst + q * GB + 16 * i);
    }
    fence_proxy_async_smem();
  }
  const int n_good = __popc(__ballot_sync(0xffffffffu, mine && ok));
  __syncwarp();
  if (lane == 0) mbar_arrive_expect_tx(fb, (uint32_t)n_good * GB);
  __syncwarp();
  if (mine && ok) {
    const long long row = ((long long)tb * p.n_kv_heads + head) * p.page_size + (k0 + lane * kGroup) % p.page_size;
    bulk_g2s_hint(dst + lane * GB, (kIsV ? p.v_pool : p.k_pool) + row * RB, GB, fb, policy);
  }
  __syncwarp();
}

}  // namespace pa_split
