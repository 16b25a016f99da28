// Pool byte layout, shared by the append kernel (which writes it) and the
// decode kernels (which read it).
//
// A pool is [block][kv_head][page_size rows] with page_size a multiple of 16.
// Each page is cut into row groups of 16 consecutive slots, and a group keeps
// its 16 rows in 16 * row_bytes bytes arranged for the decode kernel's
// fragment loads (ldmatrix) rather than row after row:
//
//   scale region (Q4_0, Q8_0 only; 256 bytes for 8 blocks per row):
//     K pool: scale of (row r, block b) at 16 r + 2 b, so one 16-byte load
//             gives a key's eight scales;
//     V pool: at 64 (b/2) + 16 ((r%8)/2) + 8 (b%2) + 4 (r/8) + 2 (r%2), so one
//             16-byte load gives the (2t, 2t+1) and (2t+8, 2t+9) key pairs'
//             scales of two neighbouring blocks -- the pairs an MMA B
//             fragment column holds;
//   chunk region: the rest of each row (an F16 row; a quantised row's quant
//     bytes, block after block) as 16-byte chunks, row after row; chunk c of
//     row r is stored at chunk position c ^ (r % 8), so the eight rows an
//     ldmatrix phase reads fall in eight different bank groups.
//
// The row's own format (ggml F16 / Q4_0 / Q8_0) is unchanged; only where each
// byte sits differs.  Bytes per group are 16 * row_bytes, so pool sizes are
// those of a row-major pool.
#pragma once

#include <cstdint>

#include "pa.h"

namespace pa_layout {

constexpr int kGroup = 16;  // slots per row group

// Per-format constants for head_dim 256.
template <int T>
struct Fmt;
template <>
struct Fmt<PA_F16> {
  static constexpr int kRow = 512;     // bytes per row (ggml format)
  static constexpr int kScales = 0;    // scale-region bytes per group
  static constexpr int kRowQ = 512;    // chunk-region bytes per row
  static constexpr int kBlockQ = 64;   // chunk bytes per 32-value block
};
template <>
struct Fmt<PA_Q4_0> {
  static constexpr int kRow = 144;
  static constexpr int kScales = 256;
  static constexpr int kRowQ = 128;
  static constexpr int kBlockQ = 16;
};
template <>
struct Fmt<PA_Q8_0> {
  static constexpr int kRow = 272;
  static constexpr int kScales = 256;
  static constexpr int kRowQ = 256;
  static constexpr int kBlockQ = 32;
};

template <int T>
__host__ __device__ constexpr int group_bytes() {
  return kGroup * Fmt<T>::kRow;
}

// Byte offset in the group of 16-byte chunk c of row r (chunk region).
__host__ __device__ constexpr int chunk_offset(int scales, int row_q, int r, int c) {
  return scales + r * row_q + ((c ^ (r & 7)) << 4);
}

// Byte offset in the group of the scale of (row r, block b).
__host__ __device__ constexpr int k_scale_offset(int r, int b) { return 16 * r + 2 * b; }
__host__ __device__ constexpr int v_scale_offset(int r, int b) {
  return 64 * (b >> 1) + 16 * ((r & 7) >> 1) + 8 * (b & 1) + 4 * (r >> 3) + 2 * (r & 1);
}

static_assert(group_bytes<PA_Q4_0>() == Fmt<PA_Q4_0>::kScales + kGroup * Fmt<PA_Q4_0>::kRowQ, "Q4_0 group");
static_assert(group_bytes<PA_Q8_0>() == Fmt<PA_Q8_0>::kScales + kGroup * Fmt<PA_Q8_0>::kRowQ, "Q8_0 group");
static_assert(group_bytes<PA_F16>() == kGroup * Fmt<PA_F16>::kRowQ, "F16 group");
static_assert(v_scale_offset(15, 7) == 254 && k_scale_offset(15, 7) == 254, "scale regions hold 256 bytes");

}  // namespace pa_layout
