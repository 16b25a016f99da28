// Split-K paged GQA decode: the merge kernel and the host side of pa_decode
// (validation, planning, launches).  The split kernel itself lives in
// pa_decode_impl.cuh and is instantiated once per K format in
// pa_decode_kern_*.cu.
//
// Planning ("occupancy-aware context parallelism", lucebox PR #555, Summary):
// the batch's 64-key tiles, counted from the host copy of the sequence
// lengths, are cut into as many equal contiguous ranges as CTAs of the chosen
// kernel fit on the device at once (occupancy x SM count, at most one range
// per tile).  The merge kernel follows as a programmatic dependent launch.
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
// The grid holds exactly one CTA per (task, row), a task being a chunk of up
// to 32 pieces of a segment that has more than one piece; each CTA finds its
// task with a block scan over the sequence lengths.  Level 1: each of the 8
// warps loads its 4 pieces at once and folds them with the chunk maximum.  A
// segment with one chunk writes its result directly; otherwise each chunk
// stores (M, W, O) at its first piece's slot and the last chunk to arrive (a
// counter the split kernel zeroed) merges the chunk results in chunk order,
// so the result does not depend on timing.  Launched as a programmatic
// dependent of the split kernel.
constexpr int kMergeThreads = 256;
constexpr int kMergeWarps = kMergeThreads / 32;
constexpr int kChunk = 32;                          // pieces per task
constexpr int kPerWarp = kChunk / kMergeWarps;      // pieces per warp

// Exclusive block-wide prefix sum of one int per thread; *total gets the sum.
__device__ __forceinline__ int block_exclusive_scan(int v, int* sh, int* total) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  __syncthreads();
  if (lane == 31) sh[warp] = x;
  __syncthreads();
  int before = 0, all = 0;
  for (int i = 0; i < kMergeWarps; ++i) {
    if (i < warp) before += sh[i];
    all += sh[i];
  }
  *total = all;
  return before + x - v;
}

__device__ __forceinline__ int pieces_of(long long seg_start, int ntl, const DecodeParams& p, int* c0) {
  *c0 = cta_of_tile(seg_start, p.total_tiles, p.n_ctas);
  return cta_of_tile(seg_start + ntl - 1, p.total_tiles, p.n_ctas) - *c0 + 1;
}

// Fold per-warp states (m, W, O relative to m) into one: warp 0 finds the
// maximum and the scale of every warp; 64 threads add the float4 columns.
// Result: O (relative to M) in part[0], returns (M, W).
__device__ __forceinline__ float2 fold_warps(float m, float w, float4 a0, float4 a1, float* wm, float* ww,
                                             float* wf, float4 (*part)[kD / 4]) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  part[warp][2 * lane] = a0;
  part[warp][2 * lane + 1] = a1;
  if (lane == 0) { wm[warp] = m; ww[warp] = w; }
  __syncthreads();
  if (warp == 0) {
    const float mi = lane < kMergeWarps ? wm[lane] : -INFINITY;
    const float wi = lane < kMergeWarps ? ww[lane] : 0.f;
    float M = (wi > 0.f) ? mi : -INFINITY;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    const float f = (M == -INFINITY || !(wi > 0.f)) ? 0.f : exp2f(mi - M);
    float W = f * wi;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) W += __shfl_xor_sync(0xffffffffu, W, o);
    if (lane < kMergeWarps) wf[lane] = f;
    if (lane == 0) { wm[kMergeWarps] = M; ww[kMergeWarps] = W; }
  }
  __syncthreads();
  if (tid < kD / 4) {
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int i = 0; i < kMergeWarps; ++i) {
      const float f = wf[i];
      const float4 u = part[i][tid];
      o.x += f * u.x; o.y += f * u.y; o.z += f * u.z; o.w += f * u.w;
    }
    part[0][tid] = o;  // thread tid is the only reader and writer of entry tid here
  }
  __syncthreads();
  return make_float2(wm[kMergeWarps], ww[kMergeWarps]);
}

__global__ void __launch_bounds__(kMergeThreads) pa_merge_kernel(const __grid_constant__ DecodeParams p) {
  __shared__ int sh[kMergeWarps];
  __shared__ int found[4];
  __shared__ float wm[kMergeWarps + 1], ww[kMergeWarps + 1], wf[kMergeWarps];
  __shared__ float4 part[kMergeWarps][kD / 4];
  __shared__ int is_last;
  const int task = blockIdx.x, row = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  // ---- find this CTA's (segment, chunk): scan sequences in batches
  if (tid == 0) found[0] = -1;
  long long tiles_carry = 0;
  int task_carry = 0;
  for (int base = 0; base < p.n_seq; base += kMergeThreads) {
    const int s = base + tid;
    const int ntl = s < p.n_seq ? tiles_of(p, p.seq_lens[s]) : 0;
    int tile_total;
    const long long tb = tiles_carry + block_exclusive_scan(ntl, sh, &tile_total);
    int my_tasks = 0;
    for (int g = 0; s < p.n_seq && g < p.segs_per_seq; ++g) {
      int c0;
      const int np = pieces_of(tb * p.segs_per_seq + (long long)g * ntl, ntl, p, &c0);
      if (np > 1) my_tasks += (np + kChunk - 1) / kChunk;
    }
    int task_total;
    const int t0 = task_carry + block_exclusive_scan(my_tasks, sh, &task_total);
    if (task >= t0 && task < t0 + my_tasks) {  // exactly one thread
      int t = t0;
      for (int g = 0; g < p.segs_per_seq; ++g) {
        int c0;
        const int np = pieces_of(tb * p.segs_per_seq + (long long)g * ntl, ntl, p, &c0);
        const int nc = np > 1 ? (np + kChunk - 1) / kChunk : 0;
        if (task < t + nc) {
          found[0] = s * p.segs_per_seq + g;
          found[1] = task - t;
          found[2] = c0;
          found[3] = np;
          break;
        }
        t += nc;
      }
    }
    __syncthreads();
    if (found[0] >= 0) break;
    tiles_carry += tile_total;
    task_carry += task_total;
  }
  // Every CTA waits for the split grid before it exits, so the merge grid
  // completing implies the split grid completed (stream order for later work).
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int seg = found[0];
  if (seg < 0) return;
  const int chunk = found[1], c0 = found[2], np = found[3];
  const int n_chunks = (np + kChunk - 1) / kChunk;
  const int s = seg / p.segs_per_seq, g = seg % p.segs_per_seq;
  const int R = p.rows_per_seg;

  // ---- level 1: pieces c0 + 32 chunk + 4 warp + k
  const int cbeg = c0 + kChunk * chunk, cend = min(c0 + np, cbeg + kChunk);  // [cbeg, cend)
  float cm = -INFINITY;  // chunk maximum (over pieces with weight)
  if (warp == 0) {
    float v = -INFINITY;
    if (cbeg + lane < cend) {
      const float2 ml = __ldcg(p.part_ml + (long long)(cbeg + lane + seg) * R + row);
      if (ml.y > 0.f) v = ml.x;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    if (lane == 0) wm[kMergeWarps] = v;
  }
  __syncthreads();
  cm = wm[kMergeWarps];
  float2 mlv[kPerWarp];
  float4 x0[kPerWarp], x1[kPerWarp];
#pragma unroll
  for (int k = 0; k < kPerWarp; ++k) {
    const int c = cbeg + kPerWarp * warp + k;
    mlv[k] = make_float2(-INFINITY, 0.f);
    x0[k] = x1[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (c < cend) {
      const long long slot = (long long)(c + seg) * R + row;
      mlv[k] = __ldcg(p.part_ml + slot);
      const float4* src = reinterpret_cast<const float4*>(p.part_o + slot * kD);
      x0[k] = __ldcg(src + 2 * lane);
      x1[k] = __ldcg(src + 2 * lane + 1);
    }
  }
  float wsum = 0.f;
  float4 a0 = make_float4(0.f, 0.f, 0.f, 0.f), a1 = a0;
#pragma unroll
  for (int k = 0; k < kPerWarp; ++k) {
    const float wt = (mlv[k].y > 0.f && cm != -INFINITY) ? exp2f(mlv[k].x - cm) : 0.f;
    wsum += wt * mlv[k].y;
    a0.x += wt * x0[k].x; a0.y += wt * x0[k].y; a0.z += wt * x0[k].z; a0.w += wt * x0[k].w;
    a1.x += wt * x1[k].x; a1.y += wt * x1[k].y; a1.z += wt * x1[k].z; a1.w += wt * x1[k].w;
  }
  float2 MW = fold_warps(cm, wsum, a0, a1, wm, ww, wf, part);

  if (n_chunks > 1) {
    const long long mslot = (long long)(cbeg + seg) * R + row;
    if (tid < kD / 4) reinterpret_cast<float4*>(p.mid_o + mslot * kD)[tid] = part[0][tid];
    if (tid == 0) p.mid_ml[mslot] = MW;
    __threadfence();
    __syncthreads();
    if (tid == 0) is_last = atomicAdd(p.merge_count + (long long)seg * R + row, 1) == n_chunks - 1;
    __syncthreads();
    if (!is_last) return;
    __threadfence();
    // ---- level 2: chunk results; warp w folds chunks w, w+8, ... in order
    float m = -INFINITY, w = 0.f;
    a0 = make_float4(0.f, 0.f, 0.f, 0.f);
    a1 = a0;
    for (int k = warp; k < n_chunks; k += kMergeWarps) {
      const long long ms = (long long)(c0 + kChunk * k + seg) * R + row;
      const float2 v = __ldcg(p.mid_ml + ms);
      const float4* src = reinterpret_cast<const float4*>(p.mid_o + ms * kD);
      const float4 y0 = __ldcg(src + 2 * lane), y1 = __ldcg(src + 2 * lane + 1);
      if (!(v.y > 0.f)) continue;
      const float mn = fmaxf(m, v.x);
      const float sa = (m == -INFINITY) ? 0.f : exp2f(m - mn), sb = exp2f(v.x - mn);
      a0.x = a0.x * sa + y0.x * sb; a0.y = a0.y * sa + y0.y * sb;
      a0.z = a0.z * sa + y0.z * sb; a0.w = a0.w * sa + y0.w * sb;
      a1.x = a1.x * sa + y1.x * sb; a1.y = a1.y * sa + y1.y * sb;
      a1.z = a1.z * sa + y1.z * sb; a1.w = a1.w * sa + y1.w * sb;
      w = w * sa + v.y * sb;
      m = mn;
    }
    MW = fold_warps(m, w, a0, a1, wm, ww, wf, part);
    if (tid == 0) p.merge_count[(long long)seg * R + row] = 0;
  }

  // Segment row -> output row: a head group's rows are (head, query head) of
  // one token; a single head's rows are (token, query head).
  long long orow;
  if (p.seg_heads > 1 || p.n_qtok == 1) {
    orow = (long long)s * p.n_q_heads + (long long)g * p.seg_heads * kGqa + row;
  } else {
    const int tk = row / kGqa, hl = row % kGqa;
    orow = ((long long)s * p.n_qtok + tk) * p.n_q_heads + g * kGqa + hl;
  }
  const float inv = MW.y > 0.f ? 1.f / MW.y : 0.f;
  if (tid < kD / 4) {
    float4 o = part[0][tid];
    o.x *= inv; o.y *= inv; o.z *= inv; o.w *= inv;
    reinterpret_cast<float4*>(p.out + orow * kD)[tid] = o;
  }
  if (tid == 0 && p.lse) p.lse[orow] = MW.y > 0.f ? (MW.x + log2f(MW.y)) * kLn2 : -INFINITY;
}

// ------------------------------------------------------------------ host side

bool lookup_kernel(int kt, int vt, int nt, KernelInfo* out) {
  switch (kt) {
    case PA_F16: return lookup_kernel_f16(vt, nt, out);
    case PA_Q4_0: return lookup_kernel_q4_0(vt, nt, out);
    case PA_Q8_0: return lookup_kernel_q8_0(vt, nt, out);
    default: return false;
  }
}

int type_slot(int t) { return t == PA_F16 ? 0 : t == PA_Q4_0 ? 1 : t == PA_Q8_0 ? 2 : -1; }

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

// Merge tasks: chunks of up to 32 pieces of every segment with more than one piece.
int merge_tasks(const int32_t* seq_lens_host, uint32_t n_seq, const Geometry& geo, long long tiles, int ctas) {
  int most = 0;
  long long base = 0;
  for (uint32_t s = 0; s < n_seq; ++s) {
    const long long ntl = (seq_lens_host[s] + geo.tile_keys - 1) / geo.tile_keys;
    for (int g = 0; g < geo.segs_per_seq; ++g) {
      const long long a = base + g * ntl, e = a + ntl - 1;
      const int c0 = (int)(((a + 1) * ctas - 1) / tiles), c1 = (int)(((e + 1) * ctas - 1) / tiles);
      if (c1 > c0) most += (c1 - c0 + 32) / 32;
    }
    base += ntl * geo.segs_per_seq;
  }
  return most;
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
  plan->merge_tasks = merge_tasks(seq_lens_host, n_seq, geo, tiles, plan->ctas);
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
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)plan.merge_tasks, (unsigned)plan.geo.rows_per_seg);
    cfg.blockDim = dim3(kMergeThreads);
    cfg.stream = cs;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, pa_merge_kernel, p) != cudaSuccess) return PA_ERR_CUDA;
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
