// Append: scatter newly written K/V rows into their page slots.
//
// colibri PR #372 (Summary): "upload only newly appended KV rows through one
// packed transfer and scatter kernel".  The caller uploads the new rows once,
// packed as [n_rows][n_kv_heads][row_bytes]; this kernel copies each (row,
// head) to pool[block][head][slot] with block = table[seq][pos / page_size]
// and slot = pos % page_size.  The copy is byte-exact (rows are already in
// storage format) and moves 16-byte vectors: every row size of the supported
// formats (F16 512, Q4_0 144, Q8_0 272 bytes per 256 values) is a multiple of
// 16, so each thread moves one aligned uint4 and a warp covers consecutive
// chunks of consecutive rows.
#include <cuda_runtime.h>

#include <cstdint>

#include "pa.h"
#include "pa_device.cuh"

using namespace pa_dev;

namespace {

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
  int k_chunks;  // 16-byte chunks per K row
  int v_chunks;
};

// One thread per 16-byte chunk of the packed input; K chunks first, then V.
__global__ void __launch_bounds__(256) pa_append_kernel(const __grid_constant__ AppendParams p) {
  const long long k_total = p.n_rows * p.n_kv_heads * p.k_chunks;
  const long long v_total = p.n_rows * p.n_kv_heads * p.v_chunks;
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < k_total + v_total; i += stride) {
    const bool is_k = i < k_total;
    const long long li = is_k ? i : i - k_total;
    const int chunks = is_k ? p.k_chunks : p.v_chunks;
    const long long rh = li / chunks;  // (row, head)
    const int c = (int)(li - rh * chunks);
    const long long r = rh / p.n_kv_heads;
    const int h = (int)(rh - r * p.n_kv_heads);
    const int s = __ldg(p.row_seq + r);
    const int pos = __ldg(p.row_pos + r);
    if (s < 0 || s >= p.n_seq || pos < 0 || pos / p.page_size >= p.table_stride) {
      if (c == 0 && h == 0 && is_k) record_error(p.err, PA_ERR_BOUNDS);
      continue;
    }
    const int blk = __ldg(p.table + (long long)s * p.table_stride + pos / p.page_size);
    if (blk < 0 || blk >= p.n_blocks) {
      if (c == 0 && h == 0 && is_k) record_error(p.err, PA_ERR_BOUNDS);
      continue;
    }
    const long long dst_row = ((long long)blk * p.n_kv_heads + h) * p.page_size + pos % p.page_size;
    const uint4* src = reinterpret_cast<const uint4*>(is_k ? p.k_rows : p.v_rows) + li;
    uint4* dst = reinterpret_cast<uint4*>(is_k ? p.k_pool : p.v_pool) + dst_row * chunks + c;
    *dst = __ldg(src);
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
  if (threadIdx.x == 0) mbar_wait(b, 0, err, &abort_flag, false, limit_ns);
  __syncthreads();
}

}  // namespace

extern "C" pa_status pa_append_rows(const pa_pool* pool, void* k_pool, void* v_pool, const void* k_rows,
                                    const void* v_rows, const int32_t* row_seq, const int32_t* row_pos,
                                    uint32_t n_rows, const int32_t* block_table, uint32_t table_stride,
                                    uint32_t n_seq, int32_t* err, pa_stream_t stream) {
  pa_pool_desc d;
  if (pa_pool_get_desc(pool, &d) != PA_OK) return PA_ERR_INVALID;
  if (n_rows == 0) return PA_OK;
  if (!k_pool || !v_pool || !k_rows || !v_rows || !row_seq || !row_pos || !block_table || !err ||
      table_stride == 0 || n_seq == 0)
    return PA_ERR_INVALID;
  const size_t rbk = pa_row_bytes(d.k_type, d.head_dim), rbv = pa_row_bytes(d.v_type, d.head_dim);
  if (rbk == 0 || rbv == 0) return PA_ERR_UNSUPPORTED;
  if ((rbk | rbv) & 15) return PA_ERR_UNSUPPORTED;  // every supported format is a multiple of 16
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
  p.k_chunks = (int)(rbk / 16);
  p.v_chunks = (int)(rbv / 16);
  const long long total = (long long)n_rows * d.n_kv_heads * (p.k_chunks + p.v_chunks);
  int device = 0, sms = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return PA_ERR_CUDA;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) return PA_ERR_CUDA;
  const long long want = (total + 255) / 256;
  const int grid = (int)(want < (long long)sms * 16 ? want : (long long)sms * 16);
  pa_append_kernel<<<grid, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(p);
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
