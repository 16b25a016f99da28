// Split-K paged GQA decode: the merge kernel and the host side of pa_decode
// (validation, planning, launches).  The split kernel itself lives in
// pa_decode_impl.cuh and is instantiated in pa_decode_kern.cu, compiled once
// per (K format, V format) pair.
//
// Planning (lucebox PR #555, Summary: context parallelism sized by
// occupancy): the batch's tiles, counted from the host copy of the sequence
// lengths, are cut into as many equal contiguous ranges as CTAs of the chosen
// kernel fit on the device at once (occupancy x SM count, at most one range
// per tile).  The host also lists the merge tasks; the merge kernel follows
// as a programmatic dependent launch.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <vector>

#include "pa.h"
#include "pa_rows_tc.cuh"

using namespace pa_dev;
using namespace pa_split;

namespace {

// Merge the split partials of every multi-piece segment by log-sum-exp
// (llama.cpp fork PR #2, LSE commit): with M = max m_i and w_i = 2^(m_i - M),
// out = sum w_i O_i / sum w_i l_i and lse = (M + log2 sum w_i l_i) ln 2.  Pieces
// with l_i = 0 (every key masked) carry no weight; if all are empty the row is
// 0 with lse -inf (the pd_combine fix in the same fork).
//
// One level.  The host lists the multi-piece segments (task = segment, its
// first CTA c0, its piece count np, how many ways its 256 dims are split, and
// the task's first work item) in the launch parameters; the grid holds one
// CTA per work item (task, row, dim split), found by a binary search over the
// tasks' first items.  The CTA merges every piece of one row over
// 256 / splits dims: its 256 threads form `cols` float4 columns x `groups`
// piece groups (group q takes pieces q, q + groups, ...), so a long sequence
// cut into hundreds of pieces is read with every load of a thread in flight at
// once, and folded with two barriers: the row maximum, then the sums over the
// groups (within each warp by shuffles, then over the warps).  The fold order
// is fixed, so the result does not depend on timing.
// Launched as a programmatic dependent of the split kernel.
constexpr int kMergeThreads = 256;
constexpr int kMergeWarps = kMergeThreads / 32;
constexpr int kMaxSplits = 32;     // dims split up to 32 ways (8 dims, 2 float4 per CTA)
constexpr int kMaxPerThread = 6;   // pieces a thread holds in one round
constexpr int kMaxTasks = 1024;    // multi-piece segments: fewer than the split grid's CTAs

struct MergeTask {
  int seg, c0, np, splits, first_item;
};

// What the merge reads of a decode call.
struct MergeCore {
  const float2* part_ml;
  const float* part_o;
  float* out;
  float* lse;
  int n_qtok, n_q_heads, seg_heads, segs_per_seq, rows_per_seg;
  int n_row_tiles;  // row tiles per KV head (9 to 96 tokens), else 0
};

// The task list travels in the launch parameters; the kernel is compiled for
// a few list capacities and the launch takes the smallest that holds the
// call's tasks, so a batch with a handful of split segments does not ship a
// 20 KB parameter block.
template <int kCap>
struct MergeParams {
  MergeCore p;
  int n_tasks;
  MergeTask task[kCap];
};
constexpr int kMergeCaps[3] = {16, 128, kMaxTasks};

// Dim splits for a segment of np pieces: the fewest for which a thread holds
// at most kMaxPerThread pieces (4 * splits piece groups).
__host__ __device__ constexpr int merge_splits(int np) {
  int sp = 1;
  while (sp < kMaxSplits && np > 4 * sp * kMaxPerThread) sp *= 2;
  return sp;
}

template <int kCap>
__global__ void __launch_bounds__(kMergeThreads) pa_merge_kernel(const __grid_constant__ MergeParams<kCap> mp) {
  const MergeCore& p = mp.p;
  __shared__ float red_m[kMergeWarps];
  __shared__ float4 part[kMergeThreads];
  __shared__ float red_w[kMergeThreads];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // task of this work item: the last whose first item is <= blockIdx.x
  int lo = 0, hi = mp.n_tasks - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (mp.task[mid].first_item <= (int)blockIdx.x) lo = mid; else hi = mid - 1;
  }
  const MergeTask tk = mp.task[lo];
  const int seg = tk.seg, c0 = tk.c0, np = tk.np, splits = tk.splits;
  const int local = (int)blockIdx.x - tk.first_item;
  const int row = local / splits, split = local % splits, R = p.rows_per_seg;
  // Every CTA waits for the split grid before it reads a partial (and before
  // it exits, so the merge grid completing implies the split grid completed).
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int cols = (kD / 4) / splits;  // float4 columns of this CTA: 64, 16 or 8
  const int groups = kMergeThreads / cols;
  const int col = tid % cols, grp = tid / cols;
  const int col4 = split * cols + col;  // float4 index within the 256 dims
  const int s = seg / p.segs_per_seq, g = seg % p.segs_per_seq;

  float M = -INFINITY, W = 0.f;  // this thread's running state over its pieces
  float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int base = 0; base < np; base += groups * kMaxPerThread) {
    float2 ml[kMaxPerThread];
    float4 x[kMaxPerThread];
#pragma unroll
    for (int i = 0; i < kMaxPerThread; ++i) {
      const int c = base + grp + groups * i;
      ml[i] = make_float2(-INFINITY, 0.f);
      x[i] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (c < np) {
        const long long slot = (long long)(c0 + c + seg) * R + row;
        ml[i] = __ldcg(p.part_ml + slot);
        x[i] = __ldcg(reinterpret_cast<const float4*>(p.part_o + slot * kD) + col4);
      }
    }
    float mr = M;
#pragma unroll
    for (int i = 0; i < kMaxPerThread; ++i)
      if (ml[i].y > 0.f) mr = fmaxf(mr, ml[i].x);
    const float sa = (W > 0.f) ? exp2f(M - mr) : 0.f;  // earlier rounds, relative to the new maximum
    W *= sa;
    O = make_float4(O.x * sa, O.y * sa, O.z * sa, O.w * sa);
#pragma unroll
    for (int i = 0; i < kMaxPerThread; ++i) {
      const float f = (ml[i].y > 0.f) ? exp2f(ml[i].x - mr) : 0.f;
      W = fmaf(f, ml[i].y, W);
      O = make_float4(fmaf(f, x[i].x, O.x), fmaf(f, x[i].y, O.y), fmaf(f, x[i].z, O.z), fmaf(f, x[i].w, O.w));
    }
    M = mr;
  }
  // ---- the row maximum over every piece
  float mx = M;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if (lane == 0) red_m[warp] = mx;
  __syncthreads();
  float Mrow = -INFINITY;
#pragma unroll
  for (int i = 0; i < kMergeWarps; ++i) Mrow = fmaxf(Mrow, red_m[i]);
  const float f = (W > 0.f) ? exp2f(M - Mrow) : 0.f;
  float Wt = W * f;
  float4 Ot = make_float4(O.x * f, O.y * f, O.z * f, O.w * f);
  // ---- sums over the piece groups, in a fixed order: first the groups
  // within a warp (xor partners over the lane bits above the column bits),
  // then the warps' sums in warp order.
  const int wcols = cols < 32 ? cols : 32;  // columns a warp covers
  for (int off = wcols; off < 32; off <<= 1) {
    Wt += __shfl_xor_sync(0xffffffffu, Wt, off);
    Ot.x += __shfl_xor_sync(0xffffffffu, Ot.x, off);
    Ot.y += __shfl_xor_sync(0xffffffffu, Ot.y, off);
    Ot.z += __shfl_xor_sync(0xffffffffu, Ot.z, off);
    Ot.w += __shfl_xor_sync(0xffffffffu, Ot.w, off);
  }
  if (lane < wcols) {
    part[warp * wcols + lane] = Ot;
    red_w[warp * wcols + lane] = Wt;
  }
  __syncthreads();
  if (tid >= cols) return;
  // Warps holding column col: with cols >= 32, every (cols / 32)-th warp.
  const int wstep = cols > 32 ? cols / 32 : 1, w0 = cols > 32 ? col / 32 : 0;
  Wt = 0.f;
  Ot = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int w = w0; w < kMergeWarps; w += wstep) {
    const float4 v = part[w * wcols + col % wcols];
    Ot = make_float4(Ot.x + v.x, Ot.y + v.y, Ot.z + v.z, Ot.w + v.w);
    Wt += red_w[w * wcols + col % wcols];
  }
  // Segment row -> output row: a head group's rows are (head, query head) of
  // one token; a single head's rows are (token, query head), and a row tile's
  // rows continue them from 128 * (row tile).
  long long orow;
  if (p.n_row_tiles > 0) {
    const int head = g / p.n_row_tiles, rg = kRowTile * (g % p.n_row_tiles) + row;
    if (rg >= kGqa * p.n_qtok) return;  // a padding row of the last row tile
    orow = ((long long)s * p.n_qtok + rg / kGqa) * p.n_q_heads + head * kGqa + rg % kGqa;
  } else if (p.seg_heads > 1 || p.n_qtok == 1) {
    orow = (long long)s * p.n_q_heads + (long long)g * p.seg_heads * kGqa + row;
  } else {
    const int t = row / kGqa, hl = row % kGqa;
    orow = ((long long)s * p.n_qtok + t) * p.n_q_heads + g * kGqa + hl;
  }
  const float inv = Wt > 0.f ? 1.f / Wt : 0.f;
  reinterpret_cast<float4*>(p.out + orow * kD)[col4] = make_float4(Ot.x * inv, Ot.y * inv, Ot.z * inv, Ot.w * inv);
  if (split == 0 && col == 0 && p.lse) p.lse[orow] = Wt > 0.f ? (Mrow + log2f(Wt)) * kLn2 : -INFINITY;
}

// ------------------------------------------------------------------ host side

bool lookup_kernel(int kt, int vt, int nt, KernelInfo* out) {
#define PA_PAIR(k, v) \
  if (kt == k && vt == v) return lookup_kernel_##k##_##v(nt, out);
  PA_PAIR(1, 1) PA_PAIR(1, 2) PA_PAIR(1, 8)
  PA_PAIR(2, 1) PA_PAIR(2, 2) PA_PAIR(2, 8)
  PA_PAIR(8, 1) PA_PAIR(8, 2) PA_PAIR(8, 8)
#undef PA_PAIR
  return false;
}

bool lookup_rows_tc_kernel(int kt, int vt, KernelInfo* out) {
#define PA_PAIR(k, v) \
  if (kt == k && vt == v) return lookup_rows_tc_kernel_##k##_##v(out);
  PA_PAIR(1, 1) PA_PAIR(1, 2) PA_PAIR(1, 8)
  PA_PAIR(2, 1) PA_PAIR(2, 2) PA_PAIR(2, 8)
  PA_PAIR(8, 1) PA_PAIR(8, 2) PA_PAIR(8, 8)
#undef PA_PAIR
  return false;
}

// Query tokens from which the row-tile kernel takes over from the decode
// kernels (measured: the decode kernels are faster up to eight tokens).
constexpr uint32_t kRowsFromQTok = 9;

// Extra cost, in tiles, of a piece's first tile in the 2-8-token CTA split
// (cta_first_tile).
constexpr int kPieceCost = 2;

// The split kernel for n_qtok query tokens: the decode kernels below
// kRowsFromQTok tokens (by n-tiles of 8 query rows), the row-tile kernel from
// there to 96.  *slot: its index in the occupancy cache.
bool pick_kernel(int kt, int vt, uint32_t n_qtok, KernelInfo* ki, int* slot) {
  if (n_qtok >= 1 && n_qtok < kRowsFromQTok && n_qtok <= (uint32_t)kMaxQTok) {
    const int nt = (kGqa * (int)n_qtok + 7) / 8;
    *slot = nt - 1;
    return lookup_kernel(kt, vt, nt, ki);
  }
  if (n_qtok >= kRowsFromQTok && n_qtok <= (uint32_t)kMaxRowsQTok) {
    *slot = kMaxNT;
    return lookup_rows_tc_kernel(kt, vt, ki);
  }
  return false;
}

int type_slot(int t) { return t == PA_F16 ? 0 : t == PA_Q4_0 ? 1 : t == PA_Q8_0 ? 2 : -1; }

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int g_sms[kMaxDevices];
int g_occ[kMaxDevices][3][3][kMaxNT + 1];  // [device][k][v][kernel slot] CTAs per SM, 0 = not queried

pa_status device_caps(int device, int kt, int vt, int slot, const KernelInfo& ki, int* sms, int* occ) {
  if (device < 0 || device >= kMaxDevices) return PA_ERR_INVALID;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_sms[device] == 0) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) return PA_ERR_CUDA;
    g_sms[device] = v;
  }
  int& o = g_occ[device][type_slot(kt)][type_slot(vt)][slot];
  if (o == 0) {
    int cur = 0;
    cudaGetDevice(&cur);
    if (cur != device) cudaSetDevice(device);
    cudaError_t e = cudaFuncSetAttribute(ki.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, ki.smem);
    int n = 0;
    if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, ki.fn, ki.threads, ki.smem);
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
  KernelInfo ki;
  int slot = 0;
  if (!pick_kernel(d->k_type, d->v_type, n_qtok, &ki, &slot)) return PA_ERR_UNSUPPORTED;
  return PA_OK;
}

// Segment geometry for n_qtok query tokens: one token uses head-group tiles
// (16 keys of up to four KV heads; the group is the largest of 4, 3, 2, 1 that
// divides the KV head count), two to eight tokens per-head tiles of 64 keys,
// and nine to 96 tokens row tiles (segments of 128 query rows of one KV head,
// 64-key tiles).
struct Geometry {
  int tile_keys, seg_heads, segs_per_seq, rows_per_seg;
  int n_row_tiles;  // row tiles per KV head, or 0
};

Geometry geometry(const pa_pool_desc& d, uint32_t n_qtok) {
  Geometry g;
  g.n_row_tiles = 0;
  if (n_qtok >= kRowsFromQTok) {
    g.tile_keys = kRowKeys;
    g.seg_heads = 1;
    g.n_row_tiles = (kGqa * (int)n_qtok + kRowTile - 1) / kRowTile;
    g.segs_per_seq = (int)d.n_kv_heads * g.n_row_tiles;
    g.rows_per_seg = kRowTile;
    return g;
  }
  if (n_qtok == 1) {
    int gh = 1;
    for (int c = kCWarps; c >= 1; --c)
      if (d.n_kv_heads % c == 0) { gh = c; break; }
    g.tile_keys = kTileHG;
    g.seg_heads = gh;
  } else {
    g.tile_keys = kTile;
    g.seg_heads = 1;
  }
  g.segs_per_seq = (int)d.n_kv_heads / g.seg_heads;
  g.rows_per_seg = kGqa * g.seg_heads * (int)n_qtok;
  return g;
}

// Tiles of segment gi of a sequence of length L (the device side's
// tiles_of / row_seg_tiles): a row tile takes the key tiles its last row
// sees.
long long seg_tiles(const Geometry& geo, long long L, uint32_t n_qtok, int gi) {
  if (geo.n_row_tiles == 0) return (L + geo.tile_keys - 1) / geo.tile_keys;
  const int rt = gi % geo.n_row_tiles;
  const long long t_last = std::min<long long>(n_qtok - 1, (kRowTile * (rt + 1) - 1) / kGqa);
  return (L - n_qtok + t_last + 1 + geo.tile_keys - 1) / geo.tile_keys;
}

struct Plan {
  Geometry geo;
  long long tiles;
  int ctas;
  int piece_cost;  // w of cta_first_tile
  long long n_seg;
  long long slots;
  int merge_tasks;
  long long merge_items;  // CTAs of the merge grid
};

// The CTAs' first tiles (the split kernel's own cuts, cta_first_tile), ctas + 1
// entries, in one walk over the sequences: the targets only grow.
std::vector<long long> cta_cuts(const int32_t* seq_lens_host, uint32_t n_seq, const Geometry& geo, long long tiles,
                                int ctas, int piece_cost) {
  std::vector<long long> cut(ctas + 1);
  const int w = piece_cost, segs = geo.segs_per_seq;
  if (w == 0) {
    for (int i = 0; i <= ctas; ++i) cut[i] = (long long)i * tiles / ctas;
    return cut;
  }
  const long long total = tiles + (long long)w * n_seq * segs;
  uint32_t s = 0;
  long long st = 0, k0 = 0;
  for (int i = 0; i <= ctas; ++i) {
    const long long c = (long long)i * total / ctas;
    if (c <= 0) {
      cut[i] = 0;
      continue;
    }
    long long n = 0;
    for (; s < n_seq; ++s) {
      n = (seq_lens_host[s] + geo.tile_keys - 1) / geo.tile_keys;
      if (cut_falls_in(c, st, k0, n, segs, w)) break;
      st += segs * n;
      k0 += segs;
    }
    cut[i] = s < n_seq ? cut_in_sequence(c, st, k0, n, w) : tiles;
  }
  return cut;
}

// The CTA whose range holds tile x.
int cta_of(const std::vector<long long>& cut, long long x) {
  return (int)(std::upper_bound(cut.begin(), cut.end(), x) - cut.begin()) - 1;
}

// List the merge tasks (every segment with more than one piece) into task[];
// returns their number, or -1 past kMaxTasks.  *n_items gets the number of
// work items (CTAs of the merge grid).
int list_merge_tasks(const int32_t* seq_lens_host, uint32_t n_seq, uint32_t n_qtok, const Geometry& geo,
                     long long tiles, int ctas, int piece_cost, MergeTask* task, long long* n_items) {
  const std::vector<long long> cut = cta_cuts(seq_lens_host, n_seq, geo, tiles, ctas, piece_cost);
  int n = 0;
  long long items = 0;
  long long base = 0;
  for (uint32_t s = 0; s < n_seq; ++s) {
    for (int g = 0; g < geo.segs_per_seq; ++g) {
      const long long ntl = seg_tiles(geo, seq_lens_host[s], n_qtok, g);
      const long long a = base, e = a + ntl - 1;
      base += ntl;
      const int c0 = cta_of(cut, a), c1 = cta_of(cut, e);
      const int np = c1 - c0 + 1;
      if (np < 2) continue;
      if (n == kMaxTasks) return -1;
      const int sp = merge_splits(np);
      if (task) task[n] = MergeTask{(int)(s * geo.segs_per_seq + g), c0, np, sp, (int)items};
      items += (long long)sp * geo.rows_per_seg;
      ++n;
    }
  }
  if (n_items) *n_items = items;
  return n;
}

// Workspace: the piece partials, (m, l) and O per (slot, row).
struct WsLayout {
  size_t ml, o, total;
};

WsLayout workspace_layout(long long max_ctas, long long n_seg, int R) {
  const long long slots = max_ctas + n_seg;
  auto up = [](size_t b) { return (b + 255) & ~size_t(255); };
  WsLayout w;
  w.ml = 0;
  w.o = up((size_t)slots * R * sizeof(float2));
  w.total = w.o + up((size_t)slots * R * kD * sizeof(float));
  return w;
}

size_t workspace_bytes(long long max_ctas, long long n_seg, int R) { return workspace_layout(max_ctas, n_seg, R).total; }

}  // namespace

extern "C" size_t pa_decode_workspace_size(const pa_pool* pool, uint32_t n_seq, uint32_t n_qtok, int device) {
  pa_pool_desc d;
  if (pa_pool_get_desc(pool, &d) != PA_OK) return 0;
  if (d.head_dim != kD) return 0;
  KernelInfo ki;
  int slot = 0;
  if (!pick_kernel(d.k_type, d.v_type, n_qtok, &ki, &slot)) return 0;
  int sms = 0, occ = 0;
  if (device_caps(device, d.k_type, d.v_type, slot, ki, &sms, &occ) != PA_OK) return 0;
  const Geometry geo = geometry(d, n_qtok);
  // One launch takes at most kInlineSeqs sequences; larger batches reuse the
  // workspace sub-batch after sub-batch.
  const long long seqs = std::min<long long>(n_seq, kInlineSeqs);
  return workspace_bytes((long long)sms * occ, seqs * geo.segs_per_seq, geo.rows_per_seg);
}

static pa_status make_plan(const pa_pool_desc& d, const int32_t* seq_lens_host, uint32_t n_seq, uint32_t n_qtok,
                           uint32_t table_stride, int device, KernelInfo* ki, Plan* plan) {
  int slot = 0;
  if (!pick_kernel(d.k_type, d.v_type, n_qtok, ki, &slot)) return PA_ERR_UNSUPPORTED;
  const Geometry geo = geometry(d, n_qtok);
  long long tiles = 0;
  for (uint32_t s = 0; s < n_seq; ++s) {
    const long long L = seq_lens_host[s];
    if (L < (long long)n_qtok) return PA_ERR_INVALID;
    if (table_stride && L > (long long)table_stride * d.page_size) return PA_ERR_INVALID;
    for (int g = 0; g < geo.segs_per_seq; ++g) tiles += seg_tiles(geo, L, n_qtok, g);
  }
  int sms = 0, occ = 0;
  pa_status st = device_caps(device, d.k_type, d.v_type, slot, *ki, &sms, &occ);
  if (st != PA_OK) return st;
  plan->geo = geo;
  plan->tiles = tiles;
  plan->ctas = (int)std::min<long long>(tiles, (long long)sms * occ);
  // Two to eight query tokens: a new piece costs about two tiles of work
  // (staging its query rows, writing its partial), so ranges that hold
  // segment starts get fewer tiles -- when every range keeps at least one.
  plan->piece_cost =
      (geo.n_row_tiles == 0 && n_qtok >= 2 && tiles >= (long long)plan->ctas * (1 + kPieceCost)) ? kPieceCost : 0;
  plan->n_seg = (long long)n_seq * geo.segs_per_seq;
  plan->slots = (long long)plan->ctas + plan->n_seg;
  // Each multi-piece segment holds a CTA boundary, so there are fewer merge
  // tasks than CTAs: kMaxTasks covers any grid of up to 1024 CTAs.
  plan->merge_tasks =
      list_merge_tasks(seq_lens_host, n_seq, n_qtok, geo, tiles, plan->ctas, plan->piece_cost, nullptr,
                       &plan->merge_items);
  if (plan->merge_tasks < 0 || plan->merge_items >= (1ll << 31)) return PA_ERR_UNSUPPORTED;
  return PA_OK;
}

extern "C" pa_status pa_decode_plan(const pa_pool* pool, const int32_t* seq_lens_host, uint32_t n_seq,
                                    uint32_t n_qtok, int device, uint32_t* n_ctas, uint32_t* n_tiles,
                                    uint32_t* tile_keys, uint32_t* n_partials) {
  pa_pool_desc d;
  if (!pool || (n_seq && !seq_lens_host)) return PA_ERR_INVALID;
  pa_pool_get_desc(pool, &d);
  if (d.head_dim != kD || n_qtok < 1 || n_qtok > (uint32_t)kMaxRowsQTok) return PA_ERR_UNSUPPORTED;
  if (n_seq == 0) return PA_ERR_INVALID;
  // Sub-batches of up to kInlineSeqs sequences: the largest grid, and the
  // tiles and partials summed over the sub-batches.
  uint32_t ctas = 0, tiles = 0, keys = 0, pieces = 0;
  for (uint32_t c0 = 0; c0 < n_seq; c0 += kInlineSeqs) {
    const uint32_t cn = std::min<uint32_t>(kInlineSeqs, n_seq - c0);
    const int32_t* lens = seq_lens_host + c0;
    KernelInfo ki;
    Plan plan{};
    const pa_status st = make_plan(d, lens, cn, n_qtok, 0, device, &ki, &plan);
    if (st != PA_OK) return st;
    const Geometry& geo = plan.geo;
    ctas = std::max<uint32_t>(ctas, (uint32_t)plan.ctas);
    tiles += (uint32_t)plan.tiles;
    keys = (uint32_t)geo.tile_keys;
    // Pieces = CTA-range cuts plus segment cuts.
    const std::vector<long long> cut = cta_cuts(lens, cn, geo, plan.tiles, plan.ctas, plan.piece_cost);
    long long base = 0;
    for (uint32_t s = 0; s < cn; ++s) {
      for (int g = 0; g < geo.segs_per_seq; ++g) {
        const long long ntl = seg_tiles(geo, lens[s], n_qtok, g);
        const long long a = base, e = a + ntl - 1;
        base += ntl;
        pieces += (uint32_t)(cta_of(cut, e) - cta_of(cut, a) + 1);
      }
    }
  }
  if (n_ctas) *n_ctas = ctas;
  if (n_tiles) *n_tiles = tiles;
  if (tile_keys) *tile_keys = keys;
  if (n_partials) *n_partials = pieces;
  return PA_OK;
}

// Validate a decode call of at most kInlineSeqs sequences and fill its kernel
// parameters and launch shape.
static pa_status prepare_decode(const pa_pool* pool, const float* q, const void* k_pool, const void* v_pool,
                                const int32_t* block_table, uint32_t table_stride, const int32_t* seq_lens_dev,
                                const int32_t* seq_lens_host, uint32_t n_seq, uint32_t n_qtok, uint32_t n_q_heads,
                                float scale, float* out, float* lse, void* workspace, size_t ws_bytes, int32_t* err,
                                DecodeParams* pp, KernelInfo* ki, Plan* plan) {
  pa_pool_desc d;
  pa_status st = check_shape(pool, n_qtok, n_q_heads, &d);
  if (st != PA_OK) return st;
  if (n_seq > (uint32_t)kInlineSeqs) return PA_ERR_INVALID;
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
  st = make_plan(d, seq_lens_host, n_seq, n_qtok, table_stride, device, ki, plan);
  if (st != PA_OK) return st;
  int sms = 0, occ = 0, slot = 0;
  KernelInfo ki2;
  pick_kernel(d.k_type, d.v_type, n_qtok, &ki2, &slot);
  device_caps(device, d.k_type, d.v_type, slot, *ki, &sms, &occ);
  if (ws_bytes < workspace_bytes((long long)sms * occ, plan->n_seg, plan->geo.rows_per_seg)) return PA_ERR_INVALID;

  DecodeParams& p = *pp;
  p = DecodeParams{};
  p.q = q;
  p.k_pool = static_cast<const uint8_t*>(k_pool);
  p.v_pool = static_cast<const uint8_t*>(v_pool);
  p.table = block_table;
  p.seq_lens = seq_lens_dev;
  p.out = out;
  p.lse = lse;
  p.err = err;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const WsLayout lay = workspace_layout((long long)sms * occ, plan->n_seg, plan->geo.rows_per_seg);
  p.part_ml = reinterpret_cast<float2*>(ws + lay.ml);
  p.part_o = reinterpret_cast<float*>(ws + lay.o);
  p.total_tiles = plan->tiles;
  p.n_ctas = plan->ctas;
  p.piece_cost = plan->piece_cost;
  p.n_seq = (int)n_seq;
  p.n_qtok = (int)n_qtok;
  p.n_kv_heads = (int)d.n_kv_heads;
  p.n_q_heads = (int)n_q_heads;
  p.page_size = (int)d.page_size;
  p.table_stride = (int)table_stride;
  p.n_blocks = (int)d.n_blocks;
  p.tile_keys = plan->geo.tile_keys;
  p.seg_heads = plan->geo.seg_heads;
  p.segs_per_seq = plan->geo.segs_per_seq;
  p.rows_per_seg = plan->geo.rows_per_seg;
  p.n_row_tiles = plan->geo.n_row_tiles;
  p.scale_log2 = scale * kLog2e;
  for (uint32_t i = 0; i < n_seq; ++i) p.lens[i] = seq_lens_host[i];
  return PA_OK;
}

#define PA_DECODE_ARGS                                                                                       \
  const pa_pool *pool, const float *q, const void *k_pool, const void *v_pool, const int32_t *block_table,  \
      uint32_t table_stride, const int32_t *seq_lens_dev, const int32_t *seq_lens_host, uint32_t n_seq,     \
      uint32_t n_qtok, uint32_t n_q_heads, float scale, float *out, float *lse, void *workspace,             \
      size_t ws_bytes, int32_t *err, pa_stream_t stream
#define PA_DECODE_FWD                                                                                   \
  pool, q, k_pool, v_pool, block_table, table_stride, seq_lens_dev, seq_lens_host, n_seq, n_qtok, n_q_heads, \
      scale, out, lse, workspace, ws_bytes, err

// Launch the merge with the smallest task-list capacity that holds the call's
// tasks.
template <int kCap>
static pa_status launch_merge(const DecodeParams& p, const Plan& plan, const int32_t* seq_lens_host, uint32_t n_seq,
                              cudaStream_t cs) {
  static thread_local MergeParams<kCap> mp;  // up to 20 KB: kept off the stack
  mp.p = MergeCore{p.part_ml, p.part_o, p.out, p.lse, p.n_qtok, p.n_q_heads, p.seg_heads, p.segs_per_seq,
                   p.rows_per_seg, p.n_row_tiles};
  mp.n_tasks = list_merge_tasks(seq_lens_host, n_seq, (uint32_t)p.n_qtok, plan.geo, plan.tiles, plan.ctas,
                                plan.piece_cost, mp.task,
                                nullptr);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)plan.merge_items);
  cfg.blockDim = dim3(kMergeThreads);
  cfg.stream = cs;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, pa_merge_kernel<kCap>, mp) == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

// One launch pair over at most kInlineSeqs sequences.
static pa_status run_chunk(int passes, PA_DECODE_ARGS) {
  DecodeParams p;
  KernelInfo ki;
  Plan plan{};
  pa_status st = prepare_decode(PA_DECODE_FWD, &p, &ki, &plan);
  if (st != PA_OK) return st;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  if (passes & 1) {
    // A programmatic dependent of the previous kernel on the stream: its
    // launch and set-up overlap that kernel's tail (the split kernel waits for
    // it before reading any input).
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)plan.ctas);
    cfg.blockDim = dim3((unsigned)ki.threads);
    cfg.dynamicSmemBytes = (size_t)ki.smem;
    cfg.stream = cs;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, ki.fn, p) != cudaSuccess) return PA_ERR_CUDA;
  }
  if ((passes & 2) && plan.merge_tasks > 0) {
    if (plan.merge_tasks <= kMergeCaps[0]) return launch_merge<kMergeCaps[0]>(p, plan, seq_lens_host, n_seq, cs);
    if (plan.merge_tasks <= kMergeCaps[1]) return launch_merge<kMergeCaps[1]>(p, plan, seq_lens_host, n_seq, cs);
    return launch_merge<kMergeCaps[2]>(p, plan, seq_lens_host, n_seq, cs);
  }
  return PA_OK;
}

// Batches of more than kInlineSeqs sequences run as consecutive sub-batches
// that share the workspace; each sub-batch's split kernel waits for the
// previous sub-batch's kernels (programmatic dependent launch), so stream
// order is kept.  The separate split / merge passes take one sub-batch only.
static pa_status run_decode(int passes, PA_DECODE_ARGS) {
  if (n_seq == 0) {
    pa_pool_desc d;
    return check_shape(pool, n_qtok, n_q_heads, &d);
  }
  if (n_seq <= (uint32_t)kInlineSeqs) return run_chunk(passes, PA_DECODE_FWD, stream);
  if (passes != 3) return PA_ERR_UNSUPPORTED;
  if (!q || !block_table || !seq_lens_dev || !seq_lens_host || !out) return PA_ERR_INVALID;
  // Check every sub-batch before the first launch, so that a bad length in a
  // late sub-batch launches nothing.
  pa_pool_desc d;
  pa_status st = check_shape(pool, n_qtok, n_q_heads, &d);
  if (st != PA_OK) return st;
  for (uint32_t i = 0; i < n_seq; ++i) {
    const long long L = seq_lens_host[i];
    if (L < (long long)n_qtok || L > (long long)table_stride * d.page_size) return PA_ERR_INVALID;
  }
  const size_t row = (size_t)n_qtok * n_q_heads;  // query rows per sequence
  for (uint32_t c0 = 0; c0 < n_seq; c0 += kInlineSeqs) {
    const uint32_t cn = std::min<uint32_t>(kInlineSeqs, n_seq - c0);
    st = run_chunk(passes, pool, q + c0 * row * kD, k_pool, v_pool, block_table + (size_t)c0 * table_stride,
                   table_stride, seq_lens_dev + c0, seq_lens_host + c0, cn, n_qtok, n_q_heads, scale,
                   out + c0 * row * kD, lse ? lse + c0 * row : nullptr, workspace, ws_bytes, err, stream);
    if (st != PA_OK) return st;
  }
  return PA_OK;
}

extern "C" pa_status pa_decode(PA_DECODE_ARGS) { return run_decode(3, PA_DECODE_FWD, stream); }

extern "C" pa_status pa_decode_split(PA_DECODE_ARGS) { return run_decode(1, PA_DECODE_FWD, stream); }

extern "C" pa_status pa_decode_merge(PA_DECODE_ARGS) { return run_decode(2, PA_DECODE_FWD, stream); }

// ------------------------------------------------------------------ decode without allocation
//
// pa_decode_noalloc is pa_decode for callers that cannot hand over a device
// workspace: code that runs under a device-memory budget fixed at start-up
// (any later cudaMalloc is refused or is a policy violation), hot loops that
// must not pay cudaMalloc's implicit device synchronisation, and plain C
// callers with no allocator of their own.  Its scratch is this file-scope
// array, reserved on every GPU that loads the library until the process ends.
//
// `pa_noalloc_scratch` names a host-side stand-in in host code, not a device
// address, so the kernels are given the address cudaGetSymbolAddress returns.
// That lookup runs once per device, with the device current, on the first
// call there; the first call on a device should therefore come before any
// stream capture.  Every call shares the array and it keeps the last call's
// contents; partials are written before they are read, so nothing has to be
// cleared between calls.  Each GPU has its own copy of the array; calls whose work overlaps on
// one GPU (for example on two streams) race on it and must be serialised.
static __device__ __align__(256) uint8_t pa_noalloc_scratch[PA_NOALLOC_SCRATCH_BYTES];

namespace {
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices];
}  // namespace

extern "C" pa_status pa_decode_noalloc(const pa_pool* pool, const float* q, const void* k_pool, const void* v_pool,
                                       const int32_t* block_table, uint32_t table_stride,
                                       const int32_t* seq_lens_dev, const int32_t* seq_lens_host, uint32_t n_seq,
                                       uint32_t n_qtok, uint32_t n_q_heads, float scale, float* out, float* lse,
                                       int32_t* err, pa_stream_t stream) {
  if (!pool) return PA_ERR_INVALID;
  if (n_seq == 0) {
    pa_pool_desc d;
    return check_shape(pool, n_qtok, n_q_heads, &d);
  }
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return PA_ERR_CUDA;
  if (device < 0 || device >= kMaxDevices) return PA_ERR_UNSUPPORTED;
  // The scratch must hold this batch's workspace (an upper bound that does
  // not depend on the sequence lengths); larger batches are refused.
  const size_t need = pa_decode_workspace_size(pool, n_seq, n_qtok, device);
  if (need == 0) {
    pa_pool_desc d;
    const pa_status st = check_shape(pool, n_qtok, n_q_heads, &d);
    return st != PA_OK ? st : PA_ERR_UNSUPPORTED;
  }
  if (need > (size_t)PA_NOALLOC_SCRATCH_BYTES) return PA_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_ptr[device]) {
      void* ptr = nullptr;
      if (cudaGetSymbolAddress(&ptr, pa_noalloc_scratch) != cudaSuccess || !ptr) return PA_ERR_CUDA;
      g_scratch_ptr[device] = ptr;
    }
    scratch = g_scratch_ptr[device];
  }
  return run_decode(3, pool, q, k_pool, v_pool, block_table, table_stride, seq_lens_dev, seq_lens_host, n_seq,
                    n_qtok, n_q_heads, scale, out, lse, scratch, (size_t)PA_NOALLOC_SCRATCH_BYTES, err, stream);
}
