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

#include "pa.h"
#include "pa_decode_impl.cuh"

using namespace pa_dev;
using namespace pa_split;

namespace {

// Merge the split partials of every multi-piece segment by log-sum-exp
// (llama.cpp fork PR #2, LSE commit): with M = max m_i and w_i = 2^(m_i - M),
// out = sum w_i O_i / sum w_i l_i and lse = (M + log2 sum w_i l_i) ln 2.  Pieces
// with l_i = 0 (every key masked) carry no weight; if all are empty the row is
// 0 with lse -inf (the pd_combine fix in the same fork).
//
// Two levels in one launch, so a segment cut into hundreds of pieces (a long
// sequence spread over the whole GPU) still merges with every SM pulling data.
// A task is a chunk of up to 32 consecutive pieces of one multi-piece segment;
// the host lists the tasks in the launch parameters and the grid holds one CTA
// per (task, row).  Level 1: warp w loads its four pieces (partial and (m, l))
// in one go and folds them against its own maximum; one barrier later 64
// threads fold the eight warps, a float4 of dims each.  A segment with one
// chunk writes its result directly; otherwise each chunk stores (M, W, O) at
// its first piece's slot and the last chunk to arrive (a counter the split
// kernel zeroed) folds the chunk results in chunk order, so the result does
// not depend on timing.  Launched as a programmatic dependent of the split
// kernel: the task decode runs before griddepcontrol.wait.
constexpr int kMergeThreads = 256;
constexpr int kMergeWarps = kMergeThreads / 32;
constexpr int kChunk = 32;                      // pieces per task
constexpr int kPerWarp = kChunk / kMergeWarps;  // pieces per warp
constexpr int kMaxTasks = 1024;                 // bounded by about 1.04 x the split grid

// Task word: c0 (first CTA holding a piece of the segment) << 17 | chunk << 11 | pieces.
struct MergeParams {
  DecodeParams p;
  int2 task[kMaxTasks];  // {segment, packed word}
};

__device__ __forceinline__ float4 f4_fma(float f, float4 x, float4 acc) {
  return make_float4(fmaf(f, x.x, acc.x), fmaf(f, x.y, acc.y), fmaf(f, x.z, acc.z), fmaf(f, x.w, acc.w));
}

__global__ void __launch_bounds__(kMergeThreads) pa_merge_kernel(const __grid_constant__ MergeParams mp) {
  const DecodeParams& p = mp.p;
  __shared__ float wm[kMergeWarps], ww[kMergeWarps];
  __shared__ float4 part[kMergeWarps][kD / 4];
  __shared__ int is_last;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int row = blockIdx.y, R = p.rows_per_seg;
  const int2 tk = mp.task[blockIdx.x];
  const int seg = tk.x, c0 = tk.y >> 17, chunk = (tk.y >> 11) & 63, np = tk.y & 2047;
  const int n_chunks = (np + kChunk - 1) / kChunk;
  const int cbeg = c0 + kChunk * chunk, cend = min(c0 + np, cbeg + kChunk);  // pieces [cbeg, cend)
  const int s = seg / p.segs_per_seq, g = seg % p.segs_per_seq;
  // Segment row -> output row: a head group's rows are (head, query head) of
  // one token; a single head's rows are (token, query head).
  long long orow;
  if (p.seg_heads > 1 || p.n_qtok == 1) {
    orow = (long long)s * p.n_q_heads + (long long)g * p.seg_heads * kGqa + row;
  } else {
    const int t = row / kGqa, hl = row % kGqa;
    orow = ((long long)s * p.n_qtok + t) * p.n_q_heads + g * kGqa + hl;
  }
  // Every CTA waits for the split grid before it reads a partial (and before
  // it exits, so the merge grid completing implies the split grid completed).
  asm volatile("griddepcontrol.wait;" ::: "memory");

  // ---- level 1: warp w folds pieces cbeg + 4w + k against its own maximum
  float2 ml[kPerWarp];
  float4 x0[kPerWarp], x1[kPerWarp];
#pragma unroll
  for (int k = 0; k < kPerWarp; ++k) {
    const int c = cbeg + kPerWarp * warp + k;
    ml[k] = make_float2(-INFINITY, 0.f);
    x0[k] = x1[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (c < cend) {
      const long long slot = (long long)(c + seg) * R + row;
      ml[k] = __ldcg(p.part_ml + slot);
      const float4* src = reinterpret_cast<const float4*>(p.part_o + slot * kD);
      x0[k] = __ldcg(src + 2 * lane);
      x1[k] = __ldcg(src + 2 * lane + 1);
    }
  }
  float mw = -INFINITY;
#pragma unroll
  for (int k = 0; k < kPerWarp; ++k)
    if (ml[k].y > 0.f) mw = fmaxf(mw, ml[k].x);
  float wsum = 0.f;
  float4 a0 = make_float4(0.f, 0.f, 0.f, 0.f), a1 = a0;
#pragma unroll
  for (int k = 0; k < kPerWarp; ++k) {
    const float f = (ml[k].y > 0.f) ? exp2f(ml[k].x - mw) : 0.f;
    wsum = fmaf(f, ml[k].y, wsum);
    a0 = f4_fma(f, x0[k], a0);
    a1 = f4_fma(f, x1[k], a1);
  }
  part[warp][2 * lane] = a0;
  part[warp][2 * lane + 1] = a1;
  if (lane == 0) { wm[warp] = mw; ww[warp] = wsum; }
  __syncthreads();
  // Fold the warps (64 threads, one float4 of dims each).
  float M = -INFINITY, W = 0.f;
  float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
  if (tid < kD / 4) {
#pragma unroll
    for (int i = 0; i < kMergeWarps; ++i)
      if (ww[i] > 0.f) M = fmaxf(M, wm[i]);
#pragma unroll
    for (int i = 0; i < kMergeWarps; ++i) {
      const float f = (ww[i] > 0.f) ? exp2f(wm[i] - M) : 0.f;
      W = fmaf(f, ww[i], W);
      O = f4_fma(f, part[i][tid], O);
    }
  }

  if (n_chunks > 1) {
    const long long mslot = (long long)(cbeg + seg) * R + row;
    if (tid < kD / 4) reinterpret_cast<float4*>(p.mid_o + mslot * kD)[tid] = O;
    if (tid == 0) p.mid_ml[mslot] = make_float2(M, W);
    __syncthreads();
    if (tid == 0) {
      __threadfence();  // cumulative: publishes the CTA's stores ordered before it by the barrier
      is_last = atomicAdd(p.merge_count + (long long)seg * R + row, 1) == n_chunks - 1;
    }
    __syncthreads();
    if (!is_last) return;
    __threadfence();
    // ---- level 2: the chunk results, in chunk order.  Quarter q (64 threads,
    // a float4 of dims each) folds chunks q, q + 4, ... with every load in
    // flight at once, then 64 threads fold the quarters.
    const int q = tid >> 6, d4 = tid & 63;
    constexpr int kPerQ = 4;  // chunks per quarter per round (16 per round)
    float mq = -INFINITY, wq = 0.f;
    float4 oq = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int base = 0; base < n_chunks; base += 4 * kPerQ) {
      float2 cm[kPerQ];
      float4 cy[kPerQ];
#pragma unroll
      for (int i = 0; i < kPerQ; ++i) {
        const int k = base + q + 4 * i;
        cm[i] = make_float2(-INFINITY, 0.f);
        cy[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (k < n_chunks) {
          const long long ms = (long long)(c0 + kChunk * k + seg) * R + row;
          cm[i] = __ldcg(p.mid_ml + ms);
          cy[i] = __ldcg(reinterpret_cast<const float4*>(p.mid_o + ms * kD) + d4);
        }
      }
      float mr = mq;
#pragma unroll
      for (int i = 0; i < kPerQ; ++i)
        if (cm[i].y > 0.f) mr = fmaxf(mr, cm[i].x);
      const float sa = (wq > 0.f) ? exp2f(mq - mr) : 0.f;  // rescale the earlier rounds
      wq *= sa;
      oq = make_float4(oq.x * sa, oq.y * sa, oq.z * sa, oq.w * sa);
#pragma unroll
      for (int i = 0; i < kPerQ; ++i) {
        const float f = (cm[i].y > 0.f) ? exp2f(cm[i].x - mr) : 0.f;
        wq = fmaf(f, cm[i].y, wq);
        oq = f4_fma(f, cy[i], oq);
      }
      mq = mr;
    }
    part[q][d4] = oq;
    if (d4 == 0) { wm[q] = mq; ww[q] = wq; }
    __syncthreads();
    if (tid >= kD / 4) return;
    M = -INFINITY;
#pragma unroll
    for (int i = 0; i < 4; ++i)
      if (ww[i] > 0.f) M = fmaxf(M, wm[i]);
    W = 0.f;
    O = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float f = (ww[i] > 0.f) ? exp2f(wm[i] - M) : 0.f;
      W = fmaf(f, ww[i], W);
      O = f4_fma(f, part[i][tid], O);
    }
    if (tid == 0) p.merge_count[(long long)seg * R + row] = 0;
  } else if (tid >= kD / 4) {
    return;
  }

  const float inv = W > 0.f ? 1.f / W : 0.f;
  reinterpret_cast<float4*>(p.out + orow * kD)[tid] = make_float4(O.x * inv, O.y * inv, O.z * inv, O.w * inv);
  if (tid == 0 && p.lse) p.lse[orow] = W > 0.f ? (M + log2f(W)) * kLn2 : -INFINITY;
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

int type_slot(int t) { return t == PA_F16 ? 0 : t == PA_Q4_0 ? 1 : t == PA_Q8_0 ? 2 : -1; }

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int g_sms[kMaxDevices];
int g_occ[kMaxDevices][3][3][kMaxNT];  // [device][k][v][nt-1] CTAs per SM, 0 = not queried

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
  if (n_qtok < 1 || n_qtok > kMaxQTok) return PA_ERR_UNSUPPORTED;
  KernelInfo ki;
  if (!lookup_kernel(d->k_type, d->v_type, (kGqa * n_qtok + 7) / 8, &ki)) return PA_ERR_UNSUPPORTED;
  return PA_OK;
}

// Segment geometry for n_qtok query tokens: one token uses head-group tiles
// (16 keys of up to four KV heads; the group is the largest of 4, 3, 2, 1 that
// divides the KV head count), more tokens use per-head tiles of 64 keys.
struct Geometry {
  int tile_keys, seg_heads, segs_per_seq, rows_per_seg;
};

Geometry geometry(const pa_pool_desc& d, uint32_t n_qtok) {
  Geometry g;
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

struct Plan {
  Geometry geo;
  long long tiles;
  int ctas;
  long long n_seg;
  long long slots;
  int merge_tasks;
};

// List the merge tasks (chunks of up to 32 pieces of every segment with more
// than one piece) into task[]; returns their number, or -1 past kMaxTasks.
int list_merge_tasks(const int32_t* seq_lens_host, uint32_t n_seq, const Geometry& geo, long long tiles, int ctas,
                     int2* task) {
  int n = 0;
  long long base = 0;
  for (uint32_t s = 0; s < n_seq; ++s) {
    const long long ntl = (seq_lens_host[s] + geo.tile_keys - 1) / geo.tile_keys;
    for (int g = 0; g < geo.segs_per_seq; ++g) {
      const long long a = base + g * ntl, e = a + ntl - 1;
      const int c0 = (int)(((a + 1) * ctas - 1) / tiles), c1 = (int)(((e + 1) * ctas - 1) / tiles);
      const int np = c1 - c0 + 1;
      if (np < 2) continue;
      for (int k = 0; k * kChunk < np; ++k) {
        if (n == kMaxTasks) return -1;
        if (task) task[n] = make_int2((int)(s * geo.segs_per_seq + g), (c0 << 17) | (k << 11) | np);
        ++n;
      }
    }
    base += ntl * geo.segs_per_seq;
  }
  return n;
}

// Workspace: piece partials (m, l) and O, the merge's level-1 results of the
// same shape, and one arrival counter per (segment, row).
struct WsLayout {
  size_t ml, o, mid_ml, mid_o, count, total;
};

WsLayout workspace_layout(long long max_ctas, long long n_seg, int R) {
  const long long slots = max_ctas + n_seg;
  auto up = [](size_t b) { return (b + 255) & ~size_t(255); };
  WsLayout w;
  const size_t ml = up((size_t)slots * R * sizeof(float2)), o = up((size_t)slots * R * kD * sizeof(float));
  w.ml = 0;
  w.o = ml;
  w.mid_ml = ml + o;
  w.mid_o = 2 * ml + o;
  w.count = 2 * ml + 2 * o;
  w.total = w.count + up((size_t)n_seg * R * sizeof(int));
  return w;
}

size_t workspace_bytes(long long max_ctas, long long n_seg, int R) { return workspace_layout(max_ctas, n_seg, R).total; }

}  // namespace

extern "C" size_t pa_decode_workspace_size(const pa_pool* pool, uint32_t n_seq, uint32_t n_qtok, int device) {
  pa_pool_desc d;
  if (pa_pool_get_desc(pool, &d) != PA_OK) return 0;
  if (d.head_dim != kD || n_qtok < 1 || n_qtok > kMaxQTok) return 0;
  const int nt = (kGqa * (int)n_qtok + 7) / 8;
  KernelInfo ki;
  if (!lookup_kernel(d.k_type, d.v_type, nt, &ki)) return 0;
  int sms = 0, occ = 0;
  if (device_caps(device, d.k_type, d.v_type, nt, ki, &sms, &occ) != PA_OK) return 0;
  const Geometry geo = geometry(d, n_qtok);
  return workspace_bytes((long long)sms * occ, (long long)n_seq * geo.segs_per_seq, geo.rows_per_seg);
}

static pa_status make_plan(const pa_pool_desc& d, const int32_t* seq_lens_host, uint32_t n_seq, uint32_t n_qtok,
                           uint32_t table_stride, int device, KernelInfo* ki, Plan* plan) {
  const int nt = (kGqa * (int)n_qtok + 7) / 8;
  if (!lookup_kernel(d.k_type, d.v_type, nt, ki)) return PA_ERR_UNSUPPORTED;
  const Geometry geo = geometry(d, n_qtok);
  long long tiles = 0;
  for (uint32_t s = 0; s < n_seq; ++s) {
    const long long L = seq_lens_host[s];
    if (L < (long long)n_qtok) return PA_ERR_INVALID;
    if (table_stride && L > (long long)table_stride * d.page_size) return PA_ERR_INVALID;
    tiles += (L + geo.tile_keys - 1) / geo.tile_keys;
  }
  tiles *= geo.segs_per_seq;
  int sms = 0, occ = 0;
  pa_status st = device_caps(device, d.k_type, d.v_type, nt, *ki, &sms, &occ);
  if (st != PA_OK) return st;
  plan->geo = geo;
  plan->tiles = tiles;
  plan->ctas = (int)std::min<long long>(tiles, (long long)sms * occ);
  plan->n_seg = (long long)n_seq * geo.segs_per_seq;
  plan->slots = (long long)plan->ctas + plan->n_seg;
  // The task word packs c0 < 2^14, chunk < 2^6 and np < 2^11; the task count
  // is at most about 1.04 x the CTA count (each multi-piece segment holds a
  // CTA boundary), below kMaxTasks for any grid of fewer than 2000 CTAs.
  if (plan->ctas >= 2000) return PA_ERR_UNSUPPORTED;
  plan->merge_tasks = list_merge_tasks(seq_lens_host, n_seq, geo, tiles, plan->ctas, nullptr);
  if (plan->merge_tasks < 0) return PA_ERR_UNSUPPORTED;
  return PA_OK;
}

extern "C" pa_status pa_decode_plan(const pa_pool* pool, const int32_t* seq_lens_host, uint32_t n_seq,
                                    uint32_t n_qtok, int device, uint32_t* n_ctas, uint32_t* n_tiles,
                                    uint32_t* tile_keys, uint32_t* n_partials) {
  pa_pool_desc d;
  if (!pool || (n_seq && !seq_lens_host)) return PA_ERR_INVALID;
  pa_pool_get_desc(pool, &d);
  if (d.head_dim != kD || n_qtok < 1 || n_qtok > kMaxQTok) return PA_ERR_UNSUPPORTED;
  if (n_seq == 0) return PA_ERR_INVALID;
  KernelInfo ki;
  Plan plan{};
  const pa_status st = make_plan(d, seq_lens_host, n_seq, n_qtok, 0, device, &ki, &plan);
  if (st != PA_OK) return st;
  const Geometry& geo = plan.geo;
  if (n_ctas) *n_ctas = (uint32_t)plan.ctas;
  if (n_tiles) *n_tiles = (uint32_t)plan.tiles;
  if (tile_keys) *tile_keys = (uint32_t)geo.tile_keys;
  if (n_partials) {
    // Pieces = CTA-range cuts plus segment cuts.
    uint32_t pieces = 0;
    long long base = 0;
    for (uint32_t s = 0; s < n_seq; ++s) {
      const long long ntl = (seq_lens_host[s] + geo.tile_keys - 1) / geo.tile_keys;
      for (int g = 0; g < geo.segs_per_seq; ++g) {
        const long long a = base + g * ntl, e = a + ntl - 1;
        const int c0 = (int)(((a + 1) * plan.ctas - 1) / plan.tiles);
        const int c1 = (int)(((e + 1) * plan.ctas - 1) / plan.tiles);
        pieces += (uint32_t)(c1 - c0 + 1);
      }
      base += ntl * geo.segs_per_seq;
    }
    *n_partials = pieces;
  }
  return PA_OK;
}

// Validate a decode call and fill its kernel parameters and launch shape.
static pa_status prepare_decode(const pa_pool* pool, const float* q, const void* k_pool, const void* v_pool,
                                const int32_t* block_table, uint32_t table_stride, const int32_t* seq_lens_dev,
                                const int32_t* seq_lens_host, uint32_t n_seq, uint32_t n_qtok, uint32_t n_q_heads,
                                float scale, float* out, float* lse, void* workspace, size_t ws_bytes, int32_t* err,
                                DecodeParams* pp, KernelInfo* ki, Plan* plan) {
  pa_pool_desc d;
  pa_status st = check_shape(pool, n_qtok, n_q_heads, &d);
  if (st != PA_OK) return st;
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
  int sms = 0, occ = 0;
  device_caps(device, d.k_type, d.v_type, (kGqa * (int)n_qtok + 7) / 8, *ki, &sms, &occ);
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
  p.mid_ml = reinterpret_cast<float2*>(ws + lay.mid_ml);
  p.mid_o = reinterpret_cast<float*>(ws + lay.mid_o);
  p.merge_count = reinterpret_cast<int*>(ws + lay.count);
  p.n_counters = (int)(plan->n_seg * plan->geo.rows_per_seg);
  p.total_tiles = plan->tiles;
  p.n_ctas = plan->ctas;
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
  p.scale_log2 = scale * kLog2e;
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

static pa_status run_decode(int passes, PA_DECODE_ARGS) {
  if (n_seq == 0) {
    pa_pool_desc d;
    return check_shape(pool, n_qtok, n_q_heads, &d);
  }
  DecodeParams p;
  KernelInfo ki;
  Plan plan{};
  pa_status st = prepare_decode(PA_DECODE_FWD, &p, &ki, &plan);
  if (st != PA_OK) return st;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  if (passes & 1) {
    ki.fn<<<plan.ctas, kThreads, ki.smem, cs>>>(p);
    if (cudaGetLastError() != cudaSuccess) return PA_ERR_CUDA;
  }
  if ((passes & 2) && plan.merge_tasks > 0) {
    static thread_local MergeParams mp;  // 8 KB: kept off the stack
    mp.p = p;
    list_merge_tasks(seq_lens_host, n_seq, plan.geo, plan.tiles, plan.ctas, mp.task);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)plan.merge_tasks, (unsigned)plan.geo.rows_per_seg);
    cfg.blockDim = dim3(kMergeThreads);
    cfg.stream = cs;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, pa_merge_kernel, mp) != cudaSuccess) return PA_ERR_CUDA;
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
// contents; the split kernel zeroes the merge counters itself, and partials
// are written before they are read, so nothing has to be cleared between
// calls.  Each GPU has its own copy of the array; calls whose work overlaps on
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
