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
// One CTA per (segment, query row), 16 warps.  The maximum over the pieces is
// found first (every thread loads a few (m, l) in parallel); then every piece's
// weight is known up front, so each warp's loads of its pieces' partial rows
// are independent and overlap.  Launched as a programmatic dependent of the
// split kernel: everything before griddepcontrol.wait overlaps its tail.
constexpr int kMergeThreads = 512;
constexpr int kMergeWarps = kMergeThreads / 32;

__global__ void __launch_bounds__(kMergeThreads) pa_merge_kernel(const __grid_constant__ DecodeParams p) {
  __shared__ float red[kMergeWarps];
  __shared__ float4 part[kMergeWarps][kD / 4];
  const int seg = blockIdx.x, row = blockIdx.y;
  const int s = seg / p.n_kv_heads, g = seg % p.n_kv_heads;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int ntl = (p.seq_lens[s] + kTile - 1) / kTile;
  // First tile of the segment: tiles of all earlier sequences, then earlier heads.
  int before = 0;
  for (int i = tid; i < s; i += kMergeThreads) before += (p.seq_lens[i] + kTile - 1) / kTile;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) before += __shfl_xor_sync(0xffffffffu, before, o);
  if (lane == 0) red[warp] = __int_as_float(before);
  __syncthreads();
  long long tiles_before = 0;
  for (int i = 0; i < kMergeWarps; ++i) tiles_before += __float_as_int(red[i]);
  const long long seg_start = tiles_before * p.n_kv_heads + (long long)g * ntl;
  const int c0 = cta_of_tile(seg_start, p.total_tiles, p.n_ctas);
  const int c1 = cta_of_tile(seg_start + ntl - 1, p.total_tiles, p.n_ctas);
  // Every CTA waits for the split grid before it exits, so the merge grid
  // completing implies the split grid completed (stream order for later work).
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (c0 == c1) return;  // written directly by its only CTA
  const int R = kGqa * p.n_qtok;
  const float2* ml = p.part_ml + row;  // piece c at ml[(c + seg) * R]
  float mloc = -INFINITY;
  for (int c = c0 + tid; c <= c1; c += kMergeThreads) {
    const float2 v = ml[(long long)(c + seg) * R];
    if (v.y > 0.f) mloc = fmaxf(mloc, v.x);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mloc = fmaxf(mloc, __shfl_xor_sync(0xffffffffu, mloc, o));
  __syncthreads();
  if (lane == 0) red[warp] = mloc;
  __syncthreads();
  float M = -INFINITY;
  for (int i = 0; i < kMergeWarps; ++i) M = fmaxf(M, red[i]);
  float wl = 0.f;
  float4 a0 = make_float4(0.f, 0.f, 0.f, 0.f), a1 = a0;
  if (M != -INFINITY) {
#pragma unroll 4
    for (int c = c0 + warp; c <= c1; c += kMergeWarps) {
      const long long slot = (long long)(c + seg) * R + row;
      const float2 v = p.part_ml[slot];
      const float4* src = reinterpret_cast<const float4*>(p.part_o + slot * kD);
      const float4 x0 = src[2 * lane], x1 = src[2 * lane + 1];
      const float wt = v.y > 0.f ? exp2f(v.x - M) : 0.f;
      wl += wt * v.y;
      a0.x += wt * x0.x; a0.y += wt * x0.y; a0.z += wt * x0.z; a0.w += wt * x0.w;
      a1.x += wt * x1.x; a1.y += wt * x1.y; a1.z += wt * x1.z; a1.w += wt * x1.w;
    }
  }
  part[warp][2 * lane] = a0;
  part[warp][2 * lane + 1] = a1;
  __syncthreads();
  if (lane == 0) red[warp] = wl;
  __syncthreads();
  float W = 0.f;
  for (int i = 0; i < kMergeWarps; ++i) W += red[i];
  const int tk = row / kGqa, hl = row % kGqa;
  const long long orow = ((long long)s * p.n_qtok + tk) * p.n_q_heads + g * kGqa + hl;
  if (tid < kD / 4) {
    float4 o = part[0][tid];
    for (int i = 1; i < kMergeWarps; ++i) {
      const float4 u = part[i][tid];
      o.x += u.x; o.y += u.y; o.z += u.z; o.w += u.w;
    }
    const float inv = W > 0.f ? 1.f / W : 0.f;
    o.x *= inv; o.y *= inv; o.z *= inv; o.w *= inv;
    reinterpret_cast<float4*>(p.out + orow * kD)[tid] = o;
  }
  if (tid == 0 && p.lse) p.lse[orow] = W > 0.f ? (M + log2f(W)) * kLn2 : -INFINITY;
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
  const long long n_seg = (long long)n_seq * d.n_kv_heads;
  if (ws_bytes < workspace_bytes((long long)sms * occ, n_seg, plan->R)) return PA_ERR_INVALID;

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
  p.part_ml = reinterpret_cast<float2*>(ws);
  ws += ((size_t)plan->slots * plan->R * sizeof(float2) + 255) & ~size_t(255);
  p.part_o = reinterpret_cast<float*>(ws);
  p.total_tiles = plan->tiles;
  p.n_ctas = plan->ctas;
  p.n_seq = (int)n_seq;
  p.n_qtok = (int)n_qtok;
  p.n_kv_heads = (int)d.n_kv_heads;
  p.n_q_heads = (int)n_q_heads;
  p.page_size = (int)d.page_size;
  p.table_stride = (int)table_stride;
  p.n_blocks = (int)d.n_blocks;
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
  if (passes & 2) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(n_seq * (uint32_t)p.n_kv_heads, (unsigned)plan.R);
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
