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
 *    ("a CUDA/HIP GGML_OP_PAGED_ATTN decode op for D=256 GQA with F16, Q4_0,
 *    and Q8_0 K/V", lucebox PR #555, Summary).  Q4_0: fp16 scale d then 16
 *    bytes, byte j holding element j (low nibble) and element j+16 (high
 *    nibble), value (nibble-8)*d; 18 bytes per 32 values, which is what the
 *    capacity table of lucebox PR #555 (K/V capacity: 207 MiB paged vs 1152
 *    MiB padded) implies.  Q8_0: fp16 d then 32 int8 q, value q*d.  The
 *    nibble order is a reading (ggml's layout); the pages do not print it.
 *
 *  - Gather through the page table.  "k/v are a pool of pages, and each
 *    logical page is either a pool page ..." (llama.cpp fork PR #2,
 *    ggml_flash_attn_ext_set_pages commit); every row address comes from the
 *    table, the page stride and the positions per page (TensorFold #1156,
 *    Design / Kernels, kv_row()).  Pool layout (a reading):
 *    pool[block][kv_head][slot][row_bytes].
 *
 *  - Attention.  Query head h uses KV head h / (Hq/Hkv) ("GQA 6", llama.cpp
 *    fork PR #2, split-K decode commit; contiguous grouping is a reading).
 *    Query token t of n_qtok sees keys 0..L-n_qtok+t (causal among the verify
 *    tokens, same commit: "1-4 query tokens (MTP verify widths)").  Logits
 *    z_j = scale * q.k_j; two-pass softmax in float64: m = max z, w = exp(z-m),
 *    out = sum w v / sum w, and the log-sum-exp m + ln(sum w) in the natural-log
 *    units of the scaled, masked logits (llama.cpp fork PR #2, LSE commit).
 *    A row with no visible key gives out = 0 and lse = -inf (the pd_combine
 *    fix in llama.cpp fork PR #2: a fully masked row is 0, not 0/0).
 *
 *  - Split merge (used by the self-tests only): partials over disjoint key
 *    ranges, each (m_i, l_i, o_i) with o_i normalised, combine by
 *    M = max m_i, w_i = l_i exp(m_i - M), out = sum w_i o_i / sum w_i,
 *    lse = M + ln(sum w_i)  (llama.cpp fork PR #2, LSE commit: "attend to parts
 *    of K/V separately and merge the normalized results exactly").
 *
 *  - Scatter (append): row (seq, pos) goes to block table[seq][pos/ps], slot
 *    pos%ps (colibri PR #372, Summary: upload new rows, scatter them into
 *    their page slots).
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

/* Address of row `pos` of sequence s, KV head g, or NULL when the table entry
 * is outside the pool. */
static const uint8_t* row_addr(const orc_cache* c, const uint8_t* pool, long rb, int s, int g,
                               long pos) {
  long page = pos / c->page_size;
  long slot = pos % c->page_size;
  if (page >= c->table_stride) return NULL;
  long blk = c->table[(long)s * c->table_stride + page];
  if (blk < 0 || blk >= c->n_blocks) return NULL;
  return pool + (((blk * c->hkv + g) * (long)c->page_size + slot) * rb);
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
  if (!z || !row) { free(z); free(row); return ORC_ERR_NOMEM; }
  int rc = ORC_OK;
  double m = -INFINITY;
  for (long j = j0; j < j1 && rc == ORC_OK; ++j) {
    const uint8_t* kr = row_addr(c, c->k_pool, rbk, s, g, j);
    if (!kr) { rc = ORC_ERR_BOUNDS; break; }
    orc_dequant_row(c->k_type, kr, d, row);
    double acc = 0.0;
    for (int i = 0; i < d; ++i) acc += (double)qv[i] * row[i];
    z[j - j0] = scale * acc;
    if (z[j - j0] > m) m = z[j - j0];
  }
  double l = 0.0;
  for (long j = j0; j < j1 && rc == ORC_OK; ++j) {
    const uint8_t* vr = row_addr(c, c->v_pool, rbv, s, g, j);
    if (!vr) { rc = ORC_ERR_BOUNDS; break; }
    orc_dequant_row(c->v_type, vr, d, row);
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
  if (!c || c->hkv <= 0 || c->hq % c->hkv || c->page_size <= 0 || c->n_qtok <= 0) return ORC_ERR_ARG;
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

/* Scatter n_rows packed rows ([n][hkv][rb]) into a pool through the table.
 * Returns ORC_ERR_BOUNDS (and skips the row) for an entry outside the pool. */
int orc_scatter(uint8_t* pool, long n_blocks, int hkv, int page_size, long rb, const uint8_t* rows,
                const int32_t* row_seq, const int32_t* row_pos, long n_rows, const int32_t* table,
                long table_stride, int n_seq) {
  int rc = ORC_OK;
  for (long i = 0; i < n_rows; ++i) {
    int s = row_seq[i];
    long pos = row_pos[i];
    if (s < 0 || s >= n_seq || pos < 0 || pos / page_size >= table_stride) { rc = ORC_ERR_BOUNDS; continue; }
    long blk = table[(long)s * table_stride + pos / page_size];
    if (blk < 0 || blk >= n_blocks) { rc = ORC_ERR_BOUNDS; continue; }
    for (int g = 0; g < hkv; ++g)
      memcpy(pool + ((blk * hkv + g) * (long)page_size + pos % page_size) * rb,
             rows + (i * hkv + g) * rb, (size_t)rb);
  }
  return rc;
}
