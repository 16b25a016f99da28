// Append: scatter newly written K/V rows into their page slots.
//
// colibri PR #372 (Summary): only the rows a step appends cross to the
// device, in one packed transfer, and a kernel scatters them.  The caller
// uploads the new rows once,
// packed as [n_rows][n_kv_heads][row_bytes] in their ggml format; this kernel
// places each (row, head) in block table[seq][pos / page_size], slot
// pos % page_size, arranging its bytes in the pool's row-group layout
// (pa_layout.cuh): quant bytes as 16-byte chunks at their swizzled chunk
// positions, block scales in the group's scale region.  One thread moves one
// 32-value block of a quantised row (one 16- or two 32-byte chunk stores and a
// 2-byte scale) or one 16-byte chunk of an F16 row; a warp covers consecutive
// units of consecutive rows.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "pa.h"
#include "pa_device.cuh"
#include "pa_layout.cuh"

using namespace pa_dev;
using namespace pa_layout;

namespace {

constexpr int kD_append = 256;  // values per row (the pool requires head_dim 256)

struct AppendParams {
  uint8_t* k_pool;
  uint8_t* v_pool;
  const uint8_t* k_rows;
  const uint8_t* v_rows;
  const int32_t* row_seq;
  const int32_t* row_pos;
  const int32_t* table;
  int32_t* err;
  long long n_rows;
  int n_kv_heads;
  int page_size;
  int table_stride;
  int n_seq;
  int n_blocks;
  int k_type, v_type;
  int k_units, v_units;  // units per row: 32 chunks (F16) or 8 blocks
  int k_row, v_row;      // row bytes
};

__device__ __forceinline__ uint32_t ld_u16(const uint8_t* p) { return *reinterpret_cast<const uint16_t*>(p); }

// Move unit u of a row (src, ggml format) into its group (dst = group base,
// r = row in the group).  role_v selects the V scale arrangement.
__device__ __forceinline__ void place_unit(int type, bool role_v, const uint8_t* src, uint8_t* grp, int r, int u) {
  if (type == PA_F16) {
    const uint4 v = *reinterpret_cast<const uint4*>(src + 16 * u);
    *reinterpret_cast<uint4*>(grp + chunk_offset(0, Fmt<PA_F16>::kRowQ, r, u)) = v;
    return;
  }
  const bool q4 = type == PA_Q4_0;
  const uint8_t* blk = src + (q4 ? 18 : 34) * u;  // 2-byte aligned
  const uint32_t d = ld_u16(blk);
  const int n_chunks = q4 ? 1 : 2;
  for (int c = 0; c < n_chunks; ++c) {
    const uint8_t* q = blk + 2 + 16 * c;
    uint4 v;
    v.x = ld_u16(q + 0) | (ld_u16(q + 2) << 16);
    v.y = ld_u16(q + 4) | (ld_u16(q + 6) << 16);
    v.z = ld_u16(q + 8) | (ld_u16(q + 10) << 16);
    v.w = ld_u16(q + 12) | (ld_u16(q + 14) << 16);
    const int chunk = q4 ? u : 2 * u + c;
    *reinterpret_cast<uint4*>(grp + chunk_offset(256, q4 ? Fmt<PA_Q4_0>::kRowQ : Fmt<PA_Q8_0>::kRowQ, r, chunk)) = v;
  }
  *reinterpret_cast<uint16_t*>(grp + (role_v ? v_scale_offset(r, u) : k_scale_offset(r, u))) = (uint16_t)d;
}

// Quantise-on-append: block u (32 values) of a binary16 row, converted to
// the pool's format and placed.  The rule is ggml's reference quantiser in
// float32, every operation rounded on its own (no fused multiply-add):
//   Q8_0: d = max|x| / 127, id = d ? 1/d : 0, q = round-half-away(x * id);
//   Q4_0: m = the x of largest |x| (first on ties), d = m / -8,
//         id = d ? 1/d : 0, q = min(15, trunc(x * id + 8.5)), byte j =
//         q_j | q_(j+16) << 4;
//   the scale is stored as fp16(d), rounded to nearest even.
__device__ __forceinline__ void place_block_f16(int type, bool role_v, const uint8_t* src_row, uint8_t* grp, int r,
                                                int u) {
  const uint4* s4 = reinterpret_cast<const uint4*>(src_row + 64 * u);
  uint4 c[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) c[k] = __ldg(s4 + k);
  if (type == PA_F16) {
#pragma unroll
    for (int k = 0; k < 4; ++k)
      *reinterpret_cast<uint4*>(grp + chunk_offset(0, Fmt<PA_F16>::kRowQ, r, 4 * u + k)) = c[k];
    return;
  }
  float x[32];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint32_t w[4] = {c[k].x, c[k].y, c[k].z, c[k].w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      x[8 * k + 2 * i] = __half2float(__ushort_as_half((unsigned short)(w[i] & 0xffffu)));
      x[8 * k + 2 * i + 1] = __half2float(__ushort_as_half((unsigned short)(w[i] >> 16)));
    }
  }
  float d;
  if (type == PA_Q8_0) {
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(x[i]));
    d = __fdiv_rn(amax, 127.f);
    const float id = d != 0.f ? __fdiv_rn(1.f, d) : 0.f;
    uint32_t wq[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      uint32_t v = 0;
#pragma unroll
      for (int b = 0; b < 4; ++b) v |= ((uint32_t)(uint8_t)(int8_t)(int)roundf(__fmul_rn(x[4 * j + b], id))) << (8 * b);
      wq[j] = v;
    }
    *reinterpret_cast<uint4*>(grp + chunk_offset(256, Fmt<PA_Q8_0>::kRowQ, r, 2 * u)) =
        make_uint4(wq[0], wq[1], wq[2], wq[3]);
    *reinterpret_cast<uint4*>(grp + chunk_offset(256, Fmt<PA_Q8_0>::kRowQ, r, 2 * u + 1)) =
        make_uint4(wq[4], wq[5], wq[6], wq[7]);
  } else {  // Q4_0
    float amax = 0.f, m = 0.f;
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (fabsf(x[i]) > amax) { amax = fabsf(x[i]); m = x[i]; }
    d = __fdiv_rn(m, -8.f);
    const float id = d != 0.f ? __fdiv_rn(1.f, d) : 0.f;
    int q[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) q[i] = min((int)truncf(__fadd_rn(__fmul_rn(x[i], id), 8.5f)), 15);
    uint32_t wq[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint32_t v = 0;
#pragma unroll
      for (int b = 0; b < 4; ++b) v |= (uint32_t)(q[4 * j + b] | (q[4 * j + b + 16] << 4)) << (8 * b);
      wq[j] = v;
    }
    *reinterpret_cast<uint4*>(grp + chunk_offset(256, Fmt<PA_Q4_0>::kRowQ, r, u)) = make_uint4(wq[0], wq[1], wq[2], wq[3]);
  }
  *reinterpret_cast<uint16_t*>(grp + (role_v ? v_scale_offset(r, u) : k_scale_offset(r, u))) =
      __half_as_ushort(__float2half_rn(d));
}

// One thread per unit of the packed input; K units first, then V.  kF16In:
// the input rows are binary16 [n_rows][n_kv_heads][head_dim] and every unit
// is a 32-value block, quantised to the pool's format.
template <bool kF16In>
__global__ void __launch_bounds__(256) pa_append_kernel(const __grid_constant__ AppendParams p) {
  // A decode launched next may start its set-up now: it reads nothing before
  // its griddepcontrol.wait, which waits for this grid to complete.
  if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;");
  const long long k_total = p.n_rows * p.n_kv_heads * p.k_units;
  const long long v_total = p.n_rows * p.n_kv_heads * p.v_units;
  const long long stride = (long long)gridDim.x * blockDim.x;
  // Index arithmetic in 32 bits when the launch's units fit (the common case:
  // a 64-bit division costs several times a 32-bit one, per unit).
  const bool narrow = k_total + v_total <= 0xffffffffll;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < k_total + v_total; i += stride) {
    const bool is_k = i < k_total;
    const long long li = is_k ? i : i - k_total;
    const int units = is_k ? p.k_units : p.v_units;
    long long rh, r;  // (row, head), row
    int u, h;
    if (narrow) {
      const uint32_t l = (uint32_t)li, rh32 = l / (uint32_t)units, r32 = rh32 / (uint32_t)p.n_kv_heads;
      u = (int)(l - rh32 * (uint32_t)units);
      h = (int)(rh32 - r32 * (uint32_t)p.n_kv_heads);
      rh = rh32;
      r = r32;
    } else {
      rh = li / units;
      u = (int)(li - rh * units);
      r = rh / p.n_kv_heads;
      h = (int)(rh - r * p.n_kv_heads);
    }
    const int s = __ldg(p.row_seq + r);
    const int pos = __ldg(p.row_pos + r);
    if (s < 0 || s >= p.n_seq || pos < 0 || (uint32_t)pos / (uint32_t)p.page_size >= (uint32_t)p.table_stride) {
      if (u == 0 && h == 0 && is_k) record_error(p.err, PA_ERR_BOUNDS);
      continue;
    }
    const uint32_t page = (uint32_t)pos / (uint32_t)p.page_size;
    const int blk = __ldg(p.table + (long long)s * p.table_stride + page);
    if (blk < 0 || blk >= p.n_blocks) {
      if (u == 0 && h == 0 && is_k) record_error(p.err, PA_ERR_BOUNDS);
      continue;
    }
    const int rb = is_k ? p.k_row : p.v_row;
    const int slot = (int)((uint32_t)pos - page * (uint32_t)p.page_size);
    const long long grp_row = ((long long)blk * p.n_kv_heads + h) * p.page_size + (slot & ~(kGroup - 1));
    uint8_t* grp = (is_k ? p.k_pool : p.v_pool) + grp_row * rb;
    if constexpr (kF16In) {
      const uint8_t* src = (is_k ? p.k_rows : p.v_rows) + rh * (2 * kD_append);
      place_block_f16(is_k ? p.k_type : p.v_type, !is_k, src, grp, slot & (kGroup - 1), u);
    } else {
      const uint8_t* src = (is_k ? p.k_rows : p.v_rows) + rh * rb;
      place_unit(is_k ? p.k_type : p.v_type, !is_k, src, grp, slot & (kGroup - 1), u);
    }
  }
}

// Copy-on-write, device half: whole blocks (every KV head's page, K and V)
// from src[i] to dst[i], 16 bytes per thread.  A pair with an index outside
// the pool is skipped and reported.
struct CopyParams {
  uint8_t* k_pool;
  uint8_t* v_pool;
  const int32_t* src;
  const int32_t* dst;
  int32_t* err;
  long long n;
  long long k_chunks, v_chunks;  // 16-byte chunks per block
  int n_blocks;
};

__global__ void __launch_bounds__(256) pa_copy_blocks_kernel(const __grid_constant__ CopyParams p) {
  const long long per = p.k_chunks + p.v_chunks;
  const long long total = p.n * per;
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += stride) {
    const long long pair = i / per, c = i - pair * per;
    const int s = __ldg(p.src + pair), d = __ldg(p.dst + pair);
    if (s < 0 || s >= p.n_blocks || d < 0 || d >= p.n_blocks) {
      if (c == 0) record_error(p.err, PA_ERR_BOUNDS);
      continue;
    }
    if (c < p.k_chunks) {
      const uint4* from = reinterpret_cast<const uint4*>(p.k_pool) + s * p.k_chunks + c;
      reinterpret_cast<uint4*>(p.k_pool)[d * p.k_chunks + c] = *from;
    } else {
      const long long cv = c - p.k_chunks;
      const uint4* from = reinterpret_cast<const uint4*>(p.v_pool) + s * p.v_chunks + cv;
      reinterpret_cast<uint4*>(p.v_pool)[d * p.v_chunks + cv] = *from;
    }
  }
}

__global__ void pa_wait_selftest_kernel(uint64_t limit_ns, int32_t* err) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  const uint32_t b = smem_u32(&bar);
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(b, 1);  // one arrival expected; nothing ever arrives
    fence_mbar_init();
  }
  __syncthreads();
  mbar_wait(b, 0, err, &abort_flag, false, limit_ns);  // the whole (single) warp waits
  __syncthreads();
}

}  // namespace

// Host validation and launch shared by both append entry points.
static pa_status launch_append(bool f16_in, const pa_pool* pool, void* k_pool, void* v_pool, const void* k_rows,
                               const void* v_rows, const int32_t* row_seq, const int32_t* row_pos, uint32_t n_rows,
                               const int32_t* block_table, uint32_t table_stride, uint32_t n_seq, int32_t* err,
                               pa_stream_t stream) {
  pa_pool_desc d;
  if (pa_pool_get_desc(pool, &d) != PA_OK) return PA_ERR_INVALID;
  if (n_rows == 0) return PA_OK;
  if (!k_pool || !v_pool || !k_rows || !v_rows || !row_seq || !row_pos || !block_table || !err ||
      table_stride == 0 || n_seq == 0)
    return PA_ERR_INVALID;
  const size_t rbk = pa_row_bytes(d.k_type, d.head_dim), rbv = pa_row_bytes(d.v_type, d.head_dim);
  if (rbk == 0 || rbv == 0) return PA_ERR_UNSUPPORTED;
  if ((rbk | rbv) & 15) return PA_ERR_UNSUPPORTED;  // every supported format is a multiple of 16
  if (d.head_dim != (uint32_t)kD_append) return PA_ERR_UNSUPPORTED;
  if (((uintptr_t)k_pool | (uintptr_t)v_pool | (uintptr_t)k_rows | (uintptr_t)v_rows) & 15) return PA_ERR_INVALID;
  AppendParams p{};
  p.k_pool = static_cast<uint8_t*>(k_pool);
  p.v_pool = static_cast<uint8_t*>(v_pool);
  p.k_rows = static_cast<const uint8_t*>(k_rows);
  p.v_rows = static_cast<const uint8_t*>(v_rows);
  p.row_seq = row_seq;
  p.row_pos = row_pos;
  p.table = block_table;
  p.err = err;
  p.n_rows = n_rows;
  p.n_kv_heads = (int)d.n_kv_heads;
  p.page_size = (int)d.page_size;
  p.table_stride = (int)table_stride;
  p.n_seq = (int)n_seq;
  p.n_blocks = (int)d.n_blocks;
  p.k_type = (int)d.k_type;
  p.v_type = (int)d.v_type;
  const int blocks = (int)(d.head_dim / 32);
  p.k_units = (!f16_in && d.k_type == PA_F16) ? (int)(rbk / 16) : blocks;
  p.v_units = (!f16_in && d.v_type == PA_F16) ? (int)(rbv / 16) : blocks;
  p.k_row = (int)rbk;
  p.v_row = (int)rbv;
  const long long total = (long long)n_rows * d.n_kv_heads * (p.k_units + p.v_units);
  int device = 0, sms = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return PA_ERR_CUDA;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) return PA_ERR_CUDA;
  const long long want = (total + 255) / 256;
  const int grid = (int)(want < (long long)sms * 16 ? want : (long long)sms * 16);
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  if (f16_in) {
    pa_append_kernel<true><<<grid, 256, 0, cs>>>(p);
  } else {
    pa_append_kernel<false><<<grid, 256, 0, cs>>>(p);
  }
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

extern "C" pa_status pa_append_rows(const pa_pool* pool, void* k_pool, void* v_pool, const void* k_rows,
                                    const void* v_rows, const int32_t* row_seq, const int32_t* row_pos,
                                    uint32_t n_rows, const int32_t* block_table, uint32_t table_stride,
                                    uint32_t n_seq, int32_t* err, pa_stream_t stream) {
  return launch_append(false, pool, k_pool, v_pool, k_rows, v_rows, row_seq, row_pos, n_rows, block_table,
                       table_stride, n_seq, err, stream);
}

extern "C" pa_status pa_append_rows_f16(const pa_pool* pool, void* k_pool, void* v_pool, const uint16_t* k_rows,
                                        const uint16_t* v_rows, const int32_t* row_seq, const int32_t* row_pos,
                                        uint32_t n_rows, const int32_t* block_table, uint32_t table_stride,
                                        uint32_t n_seq, int32_t* err, pa_stream_t stream) {
  return launch_append(true, pool, k_pool, v_pool, k_rows, v_rows, row_seq, row_pos, n_rows, block_table,
                       table_stride, n_seq, err, stream);
}

extern "C" pa_status pa_copy_blocks(const pa_pool* pool, void* k_pool, void* v_pool, const int32_t* src,
                                    const int32_t* dst, uint32_t n, int32_t* err, pa_stream_t stream) {
  pa_pool_desc d;
  if (pa_pool_get_desc(pool, &d) != PA_OK) return PA_ERR_INVALID;
  if (n == 0) return PA_OK;
  if (!k_pool || !v_pool || !src || !dst || !err) return PA_ERR_INVALID;
  if (((uintptr_t)k_pool | (uintptr_t)v_pool) & 15) return PA_ERR_INVALID;
  const size_t bk = (size_t)d.n_kv_heads * d.page_size * pa_row_bytes(d.k_type, d.head_dim);
  const size_t bv = (size_t)d.n_kv_heads * d.page_size * pa_row_bytes(d.v_type, d.head_dim);
  if (bk == 0 || bv == 0 || ((bk | bv) & 15)) return PA_ERR_UNSUPPORTED;
  CopyParams p{};
  p.k_pool = static_cast<uint8_t*>(k_pool);
  p.v_pool = static_cast<uint8_t*>(v_pool);
  p.src = src;
  p.dst = dst;
  p.err = err;
  p.n = n;
  p.k_chunks = (long long)(bk / 16);
  p.v_chunks = (long long)(bv / 16);
  p.n_blocks = (int)d.n_blocks;
  int device = 0, sms = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return PA_ERR_CUDA;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) return PA_ERR_CUDA;
  const long long want = ((long long)n * (p.k_chunks + p.v_chunks) + 255) / 256;
  const int grid = (int)(want < (long long)sms * 16 ? want : (long long)sms * 16);
  pa_copy_blocks_kernel<<<grid, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(p);
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

extern "C" pa_status pa_get_error(int32_t* err, pa_stream_t stream) {
  if (!err) return PA_ERR_INVALID;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  int32_t host = 0;
  if (cudaMemcpyAsync(&host, err, sizeof(host), cudaMemcpyDeviceToHost, cs) != cudaSuccess) return PA_ERR_CUDA;
  if (cudaStreamSynchronize(cs) != cudaSuccess) return PA_ERR_CUDA;
  if (host != 0) {
    if (cudaMemsetAsync(err, 0, sizeof(int32_t), cs) != cudaSuccess) return PA_ERR_CUDA;
    if (cudaStreamSynchronize(cs) != cudaSuccess) return PA_ERR_CUDA;
  }
  if (host < 0 || host > PA_ERR_CUDA) return PA_ERR_CUDA;
  return static_cast<pa_status>(host);
}

extern "C" pa_status pa_selftest_wait_timeout(uint32_t timeout_us, int32_t* err, pa_stream_t stream) {
  if (!err || timeout_us == 0 || timeout_us > 10u * 1000u * 1000u) return PA_ERR_INVALID;
  pa_wait_selftest_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>((uint64_t)timeout_us * 1000ull,
                                                                                   err);
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}
