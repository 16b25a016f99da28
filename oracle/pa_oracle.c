/*
 * Float64 CPU oracle for paged GQA decode attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library calls this code; only the
 * test suite, the smoke check and the CPU-baseline leg of the benchmark load
 * it.  It shares no source, header or table with the CUDA library.
 *
 * What it computes (each step cites the passage it follows):
 *
 *  - Row formats.  K and V rows are stored as ggml F16, Q4_0 or Q8_0 blocks
 *    (lucebox PR #555, Summary: the decode op covers head size 256 with GQA
 *    and K/V in those three formats).  Q4_0: fp16 scale d then 16
 *    bytes, byte j holding element j (low nibble) and element j+16 (high
 *    nibble), value (nibble-8)*d; 18 bytes per 32 values, which is what the
 *    capacity table of lucebox PR #555 (K/V capacity: 207 MiB paged vs 1152
 *    MiB padded) implies.  Q8_0: fp16 d then 32 int8 q, value q*d.  The
 *    nibble order is a reading (ggml's layout); the pages do not print it.
 *
 *  - Gather through the page table.  K and V live in a pool of pages and a
 *    table maps each logical page to one of them (llama.cpp fork PR #2,
 *    ggml_flash_attn_ext_set_pages commit); every row address comes from the
 *    table, the page stride and the positions per page (TensorFold #1156,
 *    Design / Kernels, kv_row()).  Which bytes of the pool hold a row is this
 *    library's own choice (the pages print no byte layout); it is written out
 *    in orc_group_offset below.
 *
 *  - Attention.  Query head h uses KV head h / (Hq/Hkv) (GQA with six query
 *    heads per KV head, llama.cpp fork PR #2, split-K decode commit;
 *    contiguous grouping is a reading).  Query token t of n_qtok sees keys
 *    0..L-n_qtok+t (causal among the speculative-verify tokens of the same
 *    commit, one to four of them, later up to eight).  Logits
 *    z_j = scale * q.k_j; two-pass softmax in float64: m = max z, w = exp(z-m),
 *    out = sum w v / sum w, and the log-sum-exp m + ln(sum w) in the natural-log
 *    units of the scaled, masked logits (llama.cpp fork PR #2, LSE commit).
 *    A row with no visible key gives out = 0 and lse = -inf (the pd_combine
 *    fix in llama.cpp fork PR #2: a fully masked row is 0, not 0/0).
 *
 *  - Split merge (used by the self-tests only): partials over disjoint key
 *    ranges, each (m_i, l_i, o_i) with o_i normalised, combine by
 *    M = max m_i, w_i = l_i exp(m_i - M), out = sum w_i o_i / sum w_i,
 *    lse = M + ln(sum w_i)  (llama.cpp fork PR #2, LSE commit: partial
 *    attentions over parts of K/V combine exactly once each carries its
 *    log-sum-exp).
 *
 *  - Scatter (append): row (seq, pos) goes to block table[seq][pos/ps], slot
 *    pos%ps (colibri PR #372, Summary: upload new rows, scatter them into
 *    their page slots), its bytes placed as orc_group_offset says.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_F16 1
#define ORC_Q4_0 2
#define ORC_Q8_0 8

#define ORC_OK 0
#define ORC_ERR_ARG (-1)
#define ORC_ERR_BOUNDS (-2)
#define ORC_ERR_NOMEM (-3)

#define ORC_ROLE_K 0
#define ORC_ROLE_V 1
#define ORC_GROUP 16

/* IEEE 754 binary16 -> double, from the format definition:
 * 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double orc_half_to_double(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 0x1f;
  int f = h & 0x3ff;
  double v;
  if (e == 0) {
    v = ldexp((double)f, -24); /* subnormal: f * 2^-14 * 2^-10 */
  } else if (e == 31) {
    v = f ? NAN : INFINITY;
  } else {
    v = ldexp((double)(1024 + f), e - 25); /* (1 + f/1024) * 2^(e-15) */
  }
  return sign ? -v : v;
}

static uint16_t rd_u16(const uint8_t* p) { return (uint16_t)(p[0] | (p[1] << 8)); }

long orc_row_bytes(int type, int d) {
  if (d <= 0 || d % 32) return -1;
  switch (type) {
    case ORC_F16: return 2L * d;
    case ORC_Q4_0: return (long)(d / 32) * 18;
    case ORC_Q8_0: return (long)(d / 32) * 34;
    default: return -1;
  }
}

/* Dequantise one stored row of d values into out[0..d). */
int orc_dequant_row(int type, const uint8_t* row, int d, double* out) {
  if (orc_row_bytes(type, d) < 0) return ORC_ERR_ARG;
  if (type == ORC_F16) {
    for (int i = 0; i < d; ++i) out[i] = orc_half_to_double(rd_u16(row + 2 * i));
    return ORC_OK;
  }
  for (int b = 0; b < d / 32; ++b) {
    if (type == ORC_Q8_0) {
      const uint8_t* blk = row + 34 * b;
      double s = orc_half_to_double(rd_u16(blk));
      for (int i = 0; i < 32; ++i) out[32 * b + i] = (double)(int8_t)blk[2 + i] * s;
    } else {
      const uint8_t* blk = row + 18 * b;
      double s = orc_half_to_double(rd_u16(blk));
      for (int j = 0; j < 16; ++j) {
        int lo = blk[2 + j] & 0x0f;
        int hi = blk[2 + j] >> 4;
        out[32 * b + j] = (double)(lo - 8) * s;
        out[32 * b + j + 16] = (double)(hi - 8) * s;
      }
    }
  }
  return ORC_OK;
}

/* float -> IEEE binary16 bits, rounding to nearest, ties to even; overflow
 * gives infinity, NaN stays NaN.  Written from the binary16 format
 * definition (1 sign, 5 exponent bits biased by 15, 10 fraction bits). */
uint16_t orc_float_to_half(float f) {
  uint32_t x;
  memcpy(&x, &f, 4);
  const uint16_t sign = (uint16_t)((x >> 16) & 0x8000u);
  const int e = (int)((x >> 23) & 0xff);
  const uint32_t frac = x & 0x7fffffu;
  if (e == 255) return (uint16_t)(sign | 0x7c00u | (frac ? 0x200u : 0u));
  /* value = 1.frac * 2^(e-127); binary16 keeps exponents -14 .. 15 normal */
  const int he = e - 127 + 15;
  if (he >= 31) return (uint16_t)(sign | 0x7c00u);
  uint32_t mant, shift;
  if (he >= 1) {           /* normal: keep 10 of the 23 fraction bits */
    mant = (1u << 23) | frac;
    shift = 13;
  } else {                 /* subnormal or zero: units of 2^-24 */
    if (e == 0 || he < -10) return sign;  /* below half of the smallest subnormal */
    mant = (1u << 23) | frac;
    shift = (uint32_t)(14 - he);          /* 13 + (1 - he) */
  }
  uint32_t q = mant >> shift;
  const uint32_t rem = mant & ((1u << shift) - 1u), half = 1u << (shift - 1);
  if (rem > half || (rem == half && (q & 1u))) ++q;
  if (he >= 1) {
    /* q holds 1.f in 11 bits; a carry to 2^11 moves to the next exponent */
    uint32_t exp = (uint32_t)he;
    if (q >> 11) { q >>= 1; ++exp; }
    if (exp >= 31) return (uint16_t)(sign | 0x7c00u);
    return (uint16_t)(sign | (exp << 10) | (q & 0x3ffu));
  }
  return (uint16_t)(sign | q); /* q == 0x400 becomes the smallest normal, correctly */
}

/* Quantise one 32-value block given as binary16 bits, as ggml's reference
 * quantisers do (a reading: the pages write new cells into quantised cache
 * pages without printing the rule), in float32 with no fused operations:
 *   Q8_0: amax = max |x|; d = amax / 127; id = d ? 1/d : 0;
 *         q = round-half-away(x * id); bytes: fp16(d), then 32 int8 q.
 *   Q4_0: m = the x of largest |x| (the first on ties); d = m / -8;
 *         id = d ? 1/d : 0; q = min(15, trunc(x * id + 8.5));
 *         bytes: fp16(d), then byte j = q_j | q_(j+16) << 4.
 * F16 blocks are copied.  Returns the block's byte count, or -1. */
int orc_quantize_block(int type, const uint16_t* h, uint8_t* out) {
  float x[32];
  for (int i = 0; i < 32; ++i) x[i] = (float)orc_half_to_double(h[i]);
  if (type == ORC_F16) {
    memcpy(out, h, 64);
    return 64;
  }
  if (type == ORC_Q8_0) {
    float amax = 0.0f;
    for (int i = 0; i < 32; ++i) amax = fabsf(x[i]) > amax ? fabsf(x[i]) : amax;
    const float d = amax / 127.0f;
    const float id = d != 0.0f ? 1.0f / d : 0.0f;
    const uint16_t dh = orc_float_to_half(d);
    out[0] = (uint8_t)(dh & 0xff);
    out[1] = (uint8_t)(dh >> 8);
    for (int i = 0; i < 32; ++i) {
      const float v = x[i] * id;
      out[2 + i] = (uint8_t)(int8_t)roundf(v);
    }
    return 34;
  }
  if (type == ORC_Q4_0) {
    float amax = 0.0f, m = 0.0f;
    for (int i = 0; i < 32; ++i)
      if (fabsf(x[i]) > amax) { amax = fabsf(x[i]); m = x[i]; }
    const float d = m / -8.0f;
    const float id = d != 0.0f ? 1.0f / d : 0.0f;
    const uint16_t dh = orc_float_to_half(d);
    out[0] = (uint8_t)(dh & 0xff);
    out[1] = (uint8_t)(dh >> 8);
    int q[32];
    for (int i = 0; i < 32; ++i) {
      const float v = x[i] * id + 8.5f;
      const int t = (int)truncf(v);
      q[i] = t < 15 ? t : 15;
    }
    for (int j = 0; j < 16; ++j) out[2 + j] = (uint8_t)(q[j] | (q[j + 16] << 4));
    return 18;
  }
  return -1;
}

/* Pool layout.  A pool is [block][kv_head][page_size rows] with page_size a
 * multiple of ORC_GROUP (16); each page is cut into groups of 16 consecutive
 * slots, and a group stores its 16 rows in 16 * row_bytes bytes, arranged for
 * the decode kernel's tensor-core fragment loads instead of row after row:
 *
 *   1. Quantised formats (Q4_0, Q8_0) first keep the block scales of the 16
 *      rows, 2 bytes each, in a region of 32 * nb bytes (nb = d / 32 blocks
 *      per row).  In a K pool the scale of (row r, block b) sits at byte
 *      2 * (r * nb + b).  In a V pool it sits at
 *        64 * (b / 2) + 16 * ((r % 8) / 2) + 8 * (b % 2) + 4 * (r / 8) + 2 * (r % 2).
 *   2. The rest of every row (all of an F16 row; the quant bytes of a Q4_0 or
 *      Q8_0 row, block after block) follows as 16-byte chunks, row 0 first.
 *      With C chunks per row, chunk c of row r is stored at chunk position
 *      r * C + (c XOR (r % 8)).
 *
 * Returns the byte offset within the group of byte i (0 <= i < row_bytes) of
 * the row stored in group row r, or -1 for an argument outside the layout. */
long orc_group_offset(int type, int role, int d, int r, long i) {
  const long rb = orc_row_bytes(type, d);
  if (rb < 0 || r < 0 || r >= ORC_GROUP || i < 0 || i >= rb) return -1;
  if (role != ORC_ROLE_K && role != ORC_ROLE_V) return -1;
  const int nb = d / 32;
  if (type == ORC_F16) {
    const long chunks = rb / 16;
    if (chunks % 8) return -1;
    const long c = i / 16;
    return (r * chunks + (c ^ (r % 8))) * 16 + i % 16;
  }
  const long bb = (type == ORC_Q4_0) ? 18 : 34; /* bytes per 32-value block */
  const long b = i / bb, o = i % bb;
  if (o < 2) { /* scale byte o of block b */
    if (role == ORC_ROLE_K) return 2L * (r * nb + b) + o;
    if (nb % 2) return -1;
    return 64 * (b / 2) + 16 * ((r % 8) / 2) + 8 * (b % 2) + 4 * (r / 8) + 2 * (r % 2) + o;
  }
  const long per_row = nb * (bb - 2); /* quant bytes per row */
  const long chunks = per_row / 16;
  if (chunks % 8) return -1;
  const long qi = b * (bb - 2) + (o - 2); /* index among the row's quant bytes */
  const long c = qi / 16;
  return 32L * nb + (r * chunks + (c ^ (r % 8))) * 16 + qi % 16;
}

/* Geometry of one paged cache. */
typedef struct {
  int n_seq, n_qtok, hq, hkv, d, page_size;
  long n_blocks;
  int k_type, v_type;
  const int32_t* table; /* [n_seq][table_stride] */
  long table_stride;
  const int32_t* seq_lens; /* [n_seq] */
  const uint8_t* k_pool;   /* [n_blocks][hkv][page_size][rowbytes_k] */
  const uint8_t* v_pool;
} orc_cache;

/* Copy row `pos` of sequence s, KV head g out of a pool (role K or V) into
 * out[0..row_bytes) in the row's own format.  ORC_ERR_BOUNDS when the position
 * is past the table or the table entry is outside the pool. */
static int fetch_row(const orc_cache* c, int role, int s, int g, long pos, uint8_t* out) {
  const int type = role == ORC_ROLE_K ? c->k_type : c->v_type;
  const uint8_t* pool = role == ORC_ROLE_K ? c->k_pool : c->v_pool;
  const long rb = orc_row_bytes(type, c->d);
  long page = pos / c->page_size;
  long slot = pos % c->page_size;
  if (page >= c->table_stride) return ORC_ERR_BOUNDS;
  long blk = c->table[(long)s * c->table_stride + page];
  if (blk < 0 || blk >= c->n_blocks) return ORC_ERR_BOUNDS;
  const uint8_t* grp = pool + ((blk * c->hkv + g) * (long)c->page_size + slot / ORC_GROUP * ORC_GROUP) * rb;
  for (long i = 0; i < rb; ++i) out[i] = grp[orc_group_offset(type, role, c->d, (int)(slot % ORC_GROUP), i)];
  return ORC_OK;
}

/* Plain attention over keys [j0, j1) of sequence s for query (t, h):
 * z_j = scale*q.k_j for visible keys (j <= L - n_qtok + t), two-pass softmax.
 * Writes o[d] (normalised), *m_out (max logit, -inf if no visible key) and
 * *l_out (sum of exp(z - m)).  Returns ORC_OK / ORC_ERR_BOUNDS. */
int orc_attend_range(const orc_cache* c, const float* q, double scale, int s, int t, int h,
                     long j0, long j1, double* o, double* m_out, double* l_out) {
  const int d = c->d;
  const int g = h / (c->hq / c->hkv);
  const long L = c->seq_lens[s];
  const long last = L - c->n_qtok + t; /* last visible key */
  const long rbk = orc_row_bytes(c->k_type, d), rbv = orc_row_bytes(c->v_type, d);
  const float* qv = q + (((long)s * c->n_qtok + t) * c->hq + h) * d;
  if (j1 > last + 1) j1 = last + 1;
  if (j0 < 0) j0 = 0;
  for (int i = 0; i < d; ++i) o[i] = 0.0;
  *m_out = -INFINITY;
  *l_out = 0.0;
  if (j1 <= j0) return ORC_OK;
  long n = j1 - j0;
  double* z = (double*)malloc(sizeof(double) * n);
  double* row = (double*)malloc(sizeof(double) * d);
  uint8_t* bytes = (uint8_t*)malloc((size_t)(rbk > rbv ? rbk : rbv));
  if (!z || !row || !bytes) { free(z); free(row); free(bytes); return ORC_ERR_NOMEM; }
  int rc = ORC_OK;
  double m = -INFINITY;
  for (long j = j0; j < j1 && rc == ORC_OK; ++j) {
    rc = fetch_row(c, ORC_ROLE_K, s, g, j, bytes);
    if (rc != ORC_OK) break;
    orc_dequant_row(c->k_type, bytes, d, row);
    double acc = 0.0;
    for (int i = 0; i < d; ++i) acc += (double)qv[i] * row[i];
    z[j - j0] = scale * acc;
    if (z[j - j0] > m) m = z[j - j0];
  }
  double l = 0.0;
  for (long j = j0; j < j1 && rc == ORC_OK; ++j) {
    rc = fetch_row(c, ORC_ROLE_V, s, g, j, bytes);
    if (rc != ORC_OK) break;
    orc_dequant_row(c->v_type, bytes, d, row);
    double w = exp(z[j - j0] - m);
    l += w;
    for (int i = 0; i < d; ++i) o[i] += w * row[i];
  }
  if (rc == ORC_OK) {
    for (int i = 0; i < d; ++i) o[i] /= l;
    *m_out = m;
    *l_out = l;
  } else {
    for (int i = 0; i < d; ++i) o[i] = 0.0;
  }
  free(z);
  free(row);
  free(bytes);
  return rc;
}

/* Merge partials (m_i, l_i, o_i normalised) over disjoint key ranges. */
void orc_merge(int n_parts, const double* m, const double* l, const double* o, int d,
               double* out, double* lse) {
  double M = -INFINITY;
  for (int i = 0; i < n_parts; ++i)
    if (l[i] > 0.0 && m[i] > M) M = m[i];
  for (int k = 0; k < d; ++k) out[k] = 0.0;
  if (M == -INFINITY) { *lse = -INFINITY; return; }
  double W = 0.0;
  for (int i = 0; i < n_parts; ++i) {
    if (!(l[i] > 0.0)) continue;
    double w = l[i] * exp(m[i] - M);
    W += w;
    for (int k = 0; k < d; ++k) out[k] += w * o[(long)i * d + k];
  }
  for (int k = 0; k < d; ++k) out[k] /= W;
  *lse = M + log(W);
}

/* Full decode: out[n_seq][n_qtok][hq][d], lse[n_seq][n_qtok][hq] (natural
 * log).  Only (seq, q-head) pairs with sel == NULL or sel[s*hq+h] != 0 are
 * computed; the rest are left untouched.  n_threads > 1 uses OpenMP over
 * (seq, q-head) when compiled with it. */
int orc_decode(const orc_cache* c, const float* q, double scale, const uint8_t* sel,
               double* out, double* lse, int n_threads) {
  if (!c || c->hkv <= 0 || c->hq % c->hkv || c->page_size <= 0 || c->page_size % ORC_GROUP || c->n_qtok <= 0)
    return ORC_ERR_ARG;
  if (orc_row_bytes(c->k_type, c->d) < 0 || orc_row_bytes(c->v_type, c->d) < 0) return ORC_ERR_ARG;
  const long npairs = (long)c->n_seq * c->hq;
  int rc_all = ORC_OK;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1) num_threads(n_threads > 0 ? n_threads : 1)
#endif
  for (long p = 0; p < npairs; ++p) {
    int s = (int)(p / c->hq), h = (int)(p % c->hq);
    if (sel && !sel[p]) continue;
    for (int t = 0; t < c->n_qtok; ++t) {
      long base = ((long)s * c->n_qtok + t) * c->hq + h;
      double m, l;
      int rc = orc_attend_range(c, q, scale, s, t, h, 0, c->seq_lens[s], out + base * c->d, &m, &l);
      if (rc != ORC_OK) {
#ifdef _OPENMP
#pragma omp critical
#endif
        rc_all = rc;
      }
      lse[base] = (l > 0.0) ? m + log(l) : -INFINITY;
    }
  }
  (void)n_threads;
  return rc_all;
}

/* Scatter n_rows packed rows ([n][hkv][rb], row format `type`) into a pool
 * (role K or V) through the table, placing each row's bytes as
 * orc_group_offset says.  Returns ORC_ERR_BOUNDS (and skips the row) for a
 * position past the table or an entry outside the pool. */
int orc_scatter(uint8_t* pool, long n_blocks, int hkv, int page_size, int type, int role, int d,
                const uint8_t* rows, const int32_t* row_seq, const int32_t* row_pos, long n_rows,
                const int32_t* table, long table_stride, int n_seq) {
  const long rb = orc_row_bytes(type, d);
  if (rb < 0 || page_size <= 0 || page_size % ORC_GROUP) return ORC_ERR_ARG;
  if (orc_group_offset(type, role, d, 0, 0) < 0) return ORC_ERR_ARG;
  int rc = ORC_OK;
  for (long i = 0; i < n_rows; ++i) {
    int s = row_seq[i];
    long pos = row_pos[i];
    if (s < 0 || s >= n_seq || pos < 0 || pos / page_size >= table_stride) { rc = ORC_ERR_BOUNDS; continue; }
    long blk = table[(long)s * table_stride + pos / page_size];
    if (blk < 0 || blk >= n_blocks) { rc = ORC_ERR_BOUNDS; continue; }
    long slot = pos % page_size;
    for (int g = 0; g < hkv; ++g) {
      uint8_t* grp = pool + ((blk * hkv + g) * (long)page_size + slot / ORC_GROUP * ORC_GROUP) * rb;
      const uint8_t* src = rows + (i * hkv + g) * rb;
      for (long b = 0; b < rb; ++b) grp[orc_group_offset(type, role, d, (int)(slot % ORC_GROUP), b)] = src[b];
    }
  }
  return rc;
}
