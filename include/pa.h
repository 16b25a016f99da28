/*
 * pa.h -- C ABI of libpa: paged GQA decode attention for GB300 (sm_103a).
 *
 * The library holds three things:
 *   1. a fixed-block K/V page allocator (host metadata only),
 *   2. an append kernel that scatters newly written K/V rows into their pages,
 *   3. a split-K decode kernel that reads K/V through a block table, plus the
 *      log-sum-exp merge of its splits.
 *
 * Conventions for every entry point:
 *   - Pointers marked "device" are CUDA device pointers owned by the caller
 *     (for example torch tensors); the library never frees them.  Pointers
 *     marked "host" are ordinary host memory.
 *   - Calls that take a stream are asynchronous and stream-ordered.  Errors
 *     found on the host (bad sizes, unsupported shapes, null pointers) are
 *     returned before anything is launched.  Errors found on the device (a
 *     table entry outside the pool, a bounded wait that expired) are written
 *     to the caller's device error word `err` (first error wins) and read back
 *     with pa_get_error().
 *   - No call allocates device memory.  Scratch space for pa_decode is passed
 *     in by the caller, sized by pa_decode_workspace_size().
 *
 * Data layout.  The pages describe a pool of pages plus a page table but
 * print no byte layout; this one is the library's own:
 *   K pool and V pool are separate device buffers, each
 *       pool[block][kv_head][page_size rows]
 *   with page_size a multiple of 16.  Row (seq s, position p) of kv head g
 *   lives in block block_table[s * table_stride + p / page_size] at slot
 *   p % page_size.  Each (block, kv_head) page is cut into row groups of 16
 *   consecutive slots; a group holds its 16 rows in 16 * row_bytes bytes,
 *   arranged for the decode kernel's tensor-core fragment loads:
 *     1. Q4_0/Q8_0 only: the rows' block scales (2 bytes each) in a 256-byte
 *        scale region.  K pool: scale of (row r, block b) at 16 r + 2 b.
 *        V pool: at 64 (b/2) + 16 ((r%8)/2) + 8 (b%2) + 4 (r/8) + 2 (r%2).
 *     2. The rest of each row -- an F16 row, or a quantised row's quant bytes
 *        block after block -- as 16-byte chunks, row after row; with C chunks
 *        per row, chunk c of row r sits at chunk position r C + (c XOR r%8).
 *   A row group is therefore one contiguous run that one bulk copy moves, and
 *   a whole 16-row page of every head is one run per pool.  Write pools with
 *   pa_append_rows, which takes rows in their ordinary format.
 *   Row formats are ggml's: F16 (IEEE binary16, 2*head_dim bytes), Q8_0
 *   (32-value blocks: fp16 scale d, 32 int8 q, value q*d; 34 bytes) and Q4_0
 *   (32-value blocks: fp16 d, 16 bytes whose byte j holds element j in the low
 *   nibble and element j+16 in the high nibble, value (nibble-8)*d; 18 bytes).
 */
#ifndef PA_H
#define PA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; 0 is the legacy default stream. */
typedef struct CUstream_st* pa_stream_t;

typedef enum {
  PA_OK = 0,
  PA_ERR_INVALID = 1,     /* bad argument: null pointer, size, alignment, length */
  PA_ERR_UNSUPPORTED = 2, /* shape or format this library does not implement */
  PA_ERR_OOM = 3,         /* not enough free blocks; nothing was allocated */
  PA_ERR_STALE = 4,       /* a handle is released, unknown or repeated; nothing was released */
  PA_ERR_BOUNDS = 5,      /* device: a table entry or position outside the pool or table */
  PA_ERR_TIMEOUT = 6,     /* device: a bounded wait inside a kernel expired */
  PA_ERR_CUDA = 7         /* a CUDA runtime call failed */
} pa_status;

/* Row formats, numbered as ggml numbers them. */
typedef enum { PA_F16 = 1, PA_Q4_0 = 2, PA_Q8_0 = 8 } pa_type;

typedef struct {
  uint32_t n_blocks;   /* blocks in the pool, 1 .. 2^31-1 */
  uint32_t page_size;  /* positions (rows) per block, a multiple of 16 */
  uint32_t n_kv_heads; /* KV heads per row */
  uint32_t head_dim;   /* values per row; 256 */
  int32_t k_type;      /* pa_type of K rows */
  int32_t v_type;      /* pa_type of V rows */
} pa_pool_desc;

/* A block handle: (generation << 32) | block index. */
typedef uint64_t pa_block;

typedef struct pa_pool pa_pool;

/* ------------------------------------------------------------------ allocator
 * lucebox PR #555, Summary: an exact allocator of fixed-size K/V blocks whose
 * allocations are transactional, whose stale handles are detected and whose
 * releases take effect at once.  Host metadata only; the K and V pools themselves are device buffers of
 * pa_pool_bytes() bytes that the caller allocates.  Thread-safe (one mutex
 * per pool). */

/* Create a pool's allocator state.  PA_ERR_INVALID for a zero or oversize
 * field, PA_ERR_UNSUPPORTED for an unknown type, a head_dim other than 256 or
 * a page_size that is not a multiple of 16.  *out is owned by the caller and
 * freed with pa_pool_destroy. */
pa_status pa_pool_create(const pa_pool_desc* desc, pa_pool** out);

/* Free the allocator state (not the device pools).  NULL is ignored. */
void pa_pool_destroy(pa_pool* pool);

/* Copy of the descriptor the pool was created with. */
pa_status pa_pool_get_desc(const pa_pool* pool, pa_pool_desc* out);

/* Bytes of one stored row of `head_dim` values of `type`; 0 if unsupported. */
size_t pa_row_bytes(int32_t type, uint32_t head_dim);

/* Bytes of the device K pool (which = 0) or V pool (which = 1):
 * n_blocks * n_kv_heads * page_size * row_bytes.  0 for a bad argument. */
size_t pa_pool_bytes(const pa_pool* pool, int which);

/* Allocate n blocks, all or nothing.  Writes n handles to out (host).
 * Blocks come from a LIFO free list that starts as 0, 1, 2, ...; a block
 * released earlier is handed out again first.  PA_ERR_OOM (pool unchanged)
 * when fewer than n blocks are free. */
pa_status pa_alloc_blocks(pa_pool* pool, uint32_t n, pa_block* out);

/* Release n handles (host array), all or nothing, immediately: the blocks
 * are free on return and the handles become stale (the block's generation
 * is bumped).  PA_ERR_STALE, with nothing released, if any handle is out of
 * range, not allocated, of an old generation, or repeated in the call.  The
 * caller must make sure no queued kernel still reads or writes the blocks. */
pa_status pa_release(pa_pool* pool, const pa_block* handles, uint32_t n);

/* Block index of a live handle, for building block tables.  PA_ERR_STALE
 * for a handle that is not live. */
pa_status pa_block_index(const pa_pool* pool, pa_block handle, int32_t* idx);

/* Number of free blocks. */
uint32_t pa_pool_free_count(const pa_pool* pool);

/* ------------------------------------------------------------------ prefix sharing
 * Prefix blocks shared between sequences by reference count, with
 * copy-on-write (lucebox PR #555, roadmap item 6).  A block holds one
 * reference after pa_alloc_blocks; pa_release drops one reference per
 * occurrence of a handle and frees the block (bumping its generation) when
 * the count reaches 0, so a handle may occur in one pa_release call as many
 * times as it has references (more is PA_ERR_STALE, nothing released).
 * Thread-safe; every call checks everything before it commits. */

/* Take one more reference per occurrence of each handle (a sequence that
 * forks another puts the same blocks in its own table).  PA_ERR_STALE for a
 * handle that is not live: nothing changes. */
pa_status pa_share_blocks(pa_pool* pool, const pa_block* handles, uint32_t n);

/* Reference count of a live block (PA_ERR_STALE otherwise). */
pa_status pa_block_refcount(const pa_pool* pool, pa_block handle, uint32_t* count);

/* Prepare blocks for writing.  Taking the handles in order, a block held by
 * one reference comes back unchanged in out[i]; a shared block loses the
 * caller's reference and out[i] is a freshly allocated block, with the pair
 * (old index, new index) appended to copy_src / copy_dst (host arrays of
 * capacity n; *n_copies pairs written).  The caller then copies the listed
 * blocks on the device (pa_copy_blocks) before writing to them, and puts
 * out[i] in its table.  PA_ERR_STALE (a handle not live) or PA_ERR_OOM (too
 * few free blocks for the copies): nothing changes. */
pa_status pa_cow_blocks(pa_pool* pool, const pa_block* handles, uint32_t n, pa_block* out,
                        int32_t* copy_src, int32_t* copy_dst, uint32_t* n_copies);

/* Device half of copy-on-write: copy whole blocks (every KV head's page of K
 * and of V) from block src[i] to block dst[i], i < n.  src, dst: device int32
 * arrays.  A pair with an index outside the pool is skipped and sets
 * *err = PA_ERR_BOUNDS.  Pairs that write one block twice race. */
pa_status pa_copy_blocks(const pa_pool* pool, void* k_pool, void* v_pool, const int32_t* src,
                         const int32_t* dst, uint32_t n, int32_t* err, pa_stream_t stream);

/* ------------------------------------------------------------------ append
 * New rows are uploaded once, packed, and a kernel scatters them into their
 * page slots (colibri PR #372, Summary: one packed transfer of the newly
 * appended rows plus a scatter kernel; llama.cpp fork PR #2, KV-pool commit:
 * cache writes reach pool rows through index tensors).
 *
 * k_rows, v_rows: device, packed [n_rows][n_kv_heads][row_bytes], already in
 *                 storage format; 16-byte aligned.
 * row_seq, row_pos: device int32 [n_rows]: sequence and position of each row.
 *                 Positions are appended in order with no gap (a row is
 *                 written at the sequence's current length, lucebox PR #555,
 *                 first-token bookkeeping fix); the kernel does not check it.
 * block_table:    device int32 [n_seq][table_stride].
 * k_pool, v_pool: device pools (pa_pool_bytes each), 16-byte aligned.
 * err:            device int32 error word.
 * A row whose sequence, page or table entry is out of range is skipped and
 * sets *err = PA_ERR_BOUNDS; no out-of-range address is written.  The copy
 * is byte-exact.  Rows with the same (seq, pos) in one call race. */
pa_status pa_append_rows(const pa_pool* pool, void* k_pool, void* v_pool, const void* k_rows,
                         const void* v_rows, const int32_t* row_seq, const int32_t* row_pos,
                         uint32_t n_rows, const int32_t* block_table, uint32_t table_stride,
                         uint32_t n_seq, int32_t* err, pa_stream_t stream);

/* Quantise on append: the same scatter, from rows given as IEEE binary16
 * values, converted to the pool's K and V formats on the way in (a cache
 * write into quantised pages, as the llama.cpp fork's pool writes do; the
 * pages print no rule, so the rule is ggml's reference quantiser, a
 * reading).  Per 32-value block, in float32 with every operation rounded on
 * its own (no fused multiply-add):
 *   Q8_0: d = max|x| / 127, id = d ? 1/d : 0, q = round-half-away(x * id);
 *   Q4_0: m = the x of largest |x| (the first on ties), d = m / -8,
 *         id = d ? 1/d : 0, q = min(15, trunc(x * id + 8.5));
 *   both store fp16(d), rounded to nearest even; F16 pools take the values
 *   as they are.
 * k_rows, v_rows: device binary16 [n_rows][n_kv_heads][head_dim], 16-byte
 * aligned, finite values.  Everything else as pa_append_rows; the bytes
 * written equal those of quantising each block with the rule above and
 * appending the result with pa_append_rows. */
pa_status pa_append_rows_f16(const pa_pool* pool, void* k_pool, void* v_pool, const uint16_t* k_rows,
                             const uint16_t* v_rows, const int32_t* row_seq, const int32_t* row_pos,
                             uint32_t n_rows, const int32_t* block_table, uint32_t table_stride,
                             uint32_t n_seq, int32_t* err, pa_stream_t stream);

/* ------------------------------------------------------------------ decode
 * Single-step GQA decode attention over a paged cache: split-K flash decoding
 * through a block table, with a log-sum-exp merge of the splits (llama.cpp
 * fork PR #2, split-K decode commit: head size 256, GQA 6, one to four query
 * tokens for speculative verification, a later commit taking batches of up
 * to eight tokens, and the commit on ubatches of more than eight tokens, which
 * gives paged K/V of up to 96 query tokens the decode kernel's row tiles;
 * lucebox PR #555, Summary: a numerically stable merge of split softmaxes).
 * One to eight query tokens run the decode kernels; nine to 96 run row tiles
 * (128 query rows of one KV head, K and V dequantised once per tile into
 * binary16).
 *
 * For sequence s with L = seq_lens[s] cached rows (the n_qtok new rows
 * included), query token t in [0, n_qtok) sits at position L - n_qtok + t and
 * attends to keys 0 .. L - n_qtok + t.  Query head h reads KV head
 * h / (n_q_heads / n_kv_heads).  Logits are scale * q.k; the output is the
 * softmax-weighted sum of V rows, and lse the natural-log log-sum-exp of the
 * scaled, masked logits (llama.cpp fork PR #2, LSE commit: the row maximum
 * plus the log of the row sum).  A row with no visible key would give
 * out = 0 and lse = -inf.
 *
 * Supported: head_dim 256, n_q_heads / n_kv_heads = 6, n_qtok 1..96, K and V
 * each F16, Q4_0 or Q8_0 (PA_ERR_UNSUPPORTED otherwise).
 *
 * q:            device fp32 [n_seq][n_qtok][n_q_heads][head_dim], 16-byte aligned.
 * k_pool/v_pool: device pools laid out as described at the top.
 * block_table:  device int32 [n_seq][table_stride]; only entries for pages
 *               holding positions < seq_lens[s] are read.
 * seq_lens_dev / seq_lens_host: the same int32 [n_seq] lengths on the device
 *               and on the host.  Each host length must be >= n_qtok and
 *               <= table_stride * page_size (PA_ERR_INVALID otherwise).  The
 *               host copy alone sizes the launch and drives every read: the
 *               kernels walk tiles, read table entries and mask keys from it
 *               (it travels in the launch parameters).  The device copy is
 *               only compared with it: a sequence whose device length differs
 *               (whatever its value) gives out = 0 and lse = -inf for all its
 *               rows and sets *err = PA_ERR_BOUNDS (lucebox PR #555,
 *               Validation: corrupt bounds must be caught, not followed).
 * out:          device fp32 [n_seq][n_qtok][n_q_heads][head_dim], 16-byte aligned.
 * lse:          device fp32 [n_seq][n_qtok][n_q_heads], or NULL.
 * workspace:    device scratch of ws_bytes >= pa_decode_workspace_size(),
 *               256-byte aligned; its contents need no initialisation and
 *               are garbage afterwards.  Concurrent calls need separate
 *               workspaces.
 * err:          device int32 error word.  A table entry outside [0, n_blocks)
 *               sets *err = PA_ERR_BOUNDS; the rows it would have supplied are
 *               read as zeros (no out-of-range read).
 * The result depends only on the inputs and on seq_lens (not on page size or
 * page placement): a paged cache and an identity-table cache holding the same
 * rows give bit-identical outputs.
 *
 * Launches: the split kernel, then (when a sequence is split) the merge
 * kernel, on `stream`.  Both are programmatic dependent launches: each may
 * start while the previous kernel on the stream finishes, but waits for it to
 * complete before reading anything, so stream order is kept.  One launch pair
 * takes at most 128 sequences; a larger batch runs as consecutive sub-batches
 * of 128 (in order, sharing the workspace), each planned on its own lengths. */
pa_status pa_decode(const pa_pool* pool, const float* q, const void* k_pool, const void* v_pool,
                    const int32_t* block_table, uint32_t table_stride, const int32_t* seq_lens_dev,
                    const int32_t* seq_lens_host, uint32_t n_seq, uint32_t n_qtok,
                    uint32_t n_q_heads, float scale, float* out, float* lse, void* workspace,
                    size_t ws_bytes, int32_t* err, pa_stream_t stream);

/* The two passes of pa_decode as separate calls, with pa_decode's arguments.
 * pa_decode_split runs the split-K pass: sequences handled by one CTA get
 * their final out/lse, the others leave split partials in `workspace`.
 * pa_decode_merge then merges those partials into out/lse.  Calling split then
 * merge on one stream, with the same arguments and workspace and nothing in
 * between that touches the workspace, is exactly pa_decode; the split lets a
 * caller time or schedule the passes separately.  Both take at most 128
 * sequences (PA_ERR_UNSUPPORTED above that, nothing launched). */
pa_status pa_decode_split(const pa_pool* pool, const float* q, const void* k_pool, const void* v_pool,
                          const int32_t* block_table, uint32_t table_stride, const int32_t* seq_lens_dev,
                          const int32_t* seq_lens_host, uint32_t n_seq, uint32_t n_qtok, uint32_t n_q_heads,
                          float scale, float* out, float* lse, void* workspace, size_t ws_bytes, int32_t* err,
                          pa_stream_t stream);
pa_status pa_decode_merge(const pa_pool* pool, const float* q, const void* k_pool, const void* v_pool,
                          const int32_t* block_table, uint32_t table_stride, const int32_t* seq_lens_dev,
                          const int32_t* seq_lens_host, uint32_t n_seq, uint32_t n_qtok, uint32_t n_q_heads,
                          float scale, float* out, float* lse, void* workspace, size_t ws_bytes, int32_t* err,
                          pa_stream_t stream);

/* Scratch bytes pa_decode needs for up to n_seq sequences of n_qtok query
 * tokens on CUDA device `device`, whatever their lengths.  Reported up front
 * so that a caller with a fixed memory budget can reserve it before the first
 * step instead of failing in the middle of one (llama.cpp fork PR #2, scratch
 * commit).  0 for an unsupported shape. */
size_t pa_decode_workspace_size(const pa_pool* pool, uint32_t n_seq, uint32_t n_qtok, int device);

/* How pa_decode would split this batch (lucebox PR #555, Summary: the
 * context is split across the GPU by occupancy, adaptively for long
 * contexts): *n_ctas decode CTAs (the largest grid over the sub-batches),
 * *n_tiles key tiles of `*tile_keys` keys each in total, and *n_partials
 * split partials (pieces).  The tiles, laid end to end by (sequence, KV
 * head), are cut into contiguous per-CTA ranges: of equal tile counts for one
 * query token and for row tiles; for 2-8 tokens of equal cost, where the first
 * tile of each (sequence, KV head) counts two tiles more, whenever every range
 * still gets a tile.  Host only, nothing launched; for tests and tools.
 * PA_ERR_INVALID for a null pool or lengths, n_seq = 0 or a length below
 * n_qtok; PA_ERR_UNSUPPORTED for a shape pa_decode does not take. */
pa_status pa_decode_plan(const pa_pool* pool, const int32_t* seq_lens_host, uint32_t n_seq,
                         uint32_t n_qtok, int device, uint32_t* n_ctas, uint32_t* n_tiles,
                         uint32_t* tile_keys, uint32_t* n_partials);

/* ------------------------------------------------------------------ decode without allocation
 * The pages describe no counterpart of this call; it exists for users of this
 * library.  pa_decode_noalloc is pa_decode without the workspace arguments:
 * its scratch is a fixed array of PA_NOALLOC_SCRATCH_BYTES bytes that the
 * library reserves (as a static device variable) on every GPU that loads it,
 * until the process exits.  It is meant for callers that cannot allocate
 * device memory: code running under a memory budget fixed at start-up, hot
 * loops that must avoid cudaMalloc's implicit synchronisation, plain C callers
 * without an allocator.  It allocates nothing and calls no allocating routine.
 *
 * Arguments, results and device errors are those of pa_decode.  A batch whose
 * workspace (pa_decode_workspace_size) exceeds PA_NOALLOC_SCRATCH_BYTES is
 * refused with PA_ERR_UNSUPPORTED before anything is launched.  The first call
 * on a device looks up the array's device address (once per device); make
 * that first call before any stream capture.  All calls share the one array:
 * calls whose work overlaps on the GPU race and must be serialised by the
 * caller.  The array keeps the previous call's contents; the call needs no
 * clearing. */
#define PA_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)

pa_status pa_decode_noalloc(const pa_pool* pool, const float* q, const void* k_pool, const void* v_pool,
                            const int32_t* block_table, uint32_t table_stride, const int32_t* seq_lens_dev,
                            const int32_t* seq_lens_host, uint32_t n_seq, uint32_t n_qtok, uint32_t n_q_heads,
                            float scale, float* out, float* lse, int32_t* err, pa_stream_t stream);

/* ------------------------------------------------------------------ errors */

/* Device-detected failures are reported, not trapped (lucebox PR #555,
 * Validation: bad block-table bounds are guarded against; llama.cpp fork
 * PR #2, SDMA copy commit: a stalled wait fails instead of hanging).  The
 * kernels record the first failure in the caller's int32 word.
 *
 * pa_get_error: synchronise `stream`, read the device error word, reset it
 * to 0 and return it as a pa_status.  PA_ERR_INVALID for a null word,
 * PA_ERR_CUDA if the read itself fails or the word holds no status. */
pa_status pa_get_error(int32_t* err, pa_stream_t stream);

/* Static, human-readable name of a status (the same failure classes; a
 * value outside pa_status gives "PA_ERR_UNKNOWN").  Never NULL. */
const char* pa_status_string(pa_status s);

/* Runs one kernel that waits, with the same bounded wait the decode kernel
 * uses, on a shared-memory barrier that nothing ever completes; after about
 * timeout_us microseconds the wait gives up and sets *err = PA_ERR_TIMEOUT.
 * Exists so tests can check the expiry path without hanging a GPU. */
pa_status pa_selftest_wait_timeout(uint32_t timeout_us, int32_t* err, pa_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* PA_H */
