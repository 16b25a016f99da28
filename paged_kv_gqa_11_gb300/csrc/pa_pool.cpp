// Fixed-block K/V page allocator: host metadata only.
//
// lucebox PR #555: the Summary asks for an exact fixed-block allocator with
// transactional allocation, stale-handle detection and immediate release;
// roadmap item 6 adds prefix caching, prefix blocks shared by reference
// count with copy-on-write.  Design:
//   * free blocks sit on a LIFO stack that starts as 0, 1, 2, ... from the
//     top, so a fresh pool hands out blocks in order and a freed block is
//     reused first;
//   * every block carries a 32-bit generation, starting at 1 and bumped when
//     the block returns to the free stack (skipping 0), and a handle is
//     (generation << 32) | index, so a handle kept after that no longer
//     validates;
//   * an allocated block has a reference count (1 after alloc); share adds
//     references, release drops them and frees the block at 0, and cow
//     swaps a shared block for a fresh one the caller copies into;
//   * every call checks everything first and then commits, so a failed call
//     leaves the pool exactly as it was.
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "pa.h"

struct pa_pool {
  pa_pool_desc desc;
  std::vector<uint32_t> gen;
  std::vector<uint32_t> ref;    // 0 = free
  std::vector<uint32_t> stack;  // back() is the next block handed out
  std::vector<uint32_t> mark;   // per-block stamp: cnt[] is valid for this call
  std::vector<uint32_t> cnt;    // per-block occurrences (or references left) in this call
  uint32_t stamp = 0;
  mutable std::mutex mu;
};

// Start a call that counts per-block occurrences.
static void new_stamp(pa_pool* p) {
  if (++p->stamp == 0) {  // wrapped: clear the marks once
    std::fill(p->mark.begin(), p->mark.end(), 0u);
    p->stamp = 1;
  }
}

static uint32_t& counter(pa_pool* p, uint32_t idx, uint32_t start) {
  if (p->mark[idx] != p->stamp) {
    p->mark[idx] = p->stamp;
    p->cnt[idx] = start;
  }
  return p->cnt[idx];
}

extern "C" size_t pa_row_bytes(int32_t type, uint32_t head_dim) {
  if (head_dim == 0 || head_dim % 32) return 0;
  switch (type) {
    case PA_F16: return 2ull * head_dim;
    case PA_Q4_0: return (size_t)(head_dim / 32) * 18;
    case PA_Q8_0: return (size_t)(head_dim / 32) * 34;
    default: return 0;
  }
}

extern "C" pa_status pa_pool_create(const pa_pool_desc* desc, pa_pool** out) {
  if (!desc || !out) return PA_ERR_INVALID;
  *out = nullptr;
  if (desc->n_blocks == 0 || desc->n_blocks > 0x7fffffffu || desc->page_size == 0 ||
      desc->n_kv_heads == 0 || desc->head_dim == 0)
    return PA_ERR_INVALID;
  if (pa_row_bytes(desc->k_type, desc->head_dim) == 0 || pa_row_bytes(desc->v_type, desc->head_dim) == 0)
    return PA_ERR_UNSUPPORTED;
  // The pool's row-group layout is defined for 256-value rows and pages of
  // whole 16-row groups.
  if (desc->head_dim != 256 || desc->page_size % 16 != 0) return PA_ERR_UNSUPPORTED;
  pa_pool* p = new (std::nothrow) pa_pool();
  if (!p) return PA_ERR_OOM;
  try {
    p->desc = *desc;
    p->gen.assign(desc->n_blocks, 1u);
    p->ref.assign(desc->n_blocks, 0u);
    p->mark.assign(desc->n_blocks, 0u);
    p->cnt.assign(desc->n_blocks, 0u);
    p->stack.resize(desc->n_blocks);
    for (uint32_t i = 0; i < desc->n_blocks; ++i) p->stack[i] = desc->n_blocks - 1 - i;
  } catch (...) {
    delete p;
    return PA_ERR_OOM;
  }
  *out = p;
  return PA_OK;
}

extern "C" void pa_pool_destroy(pa_pool* pool) { delete pool; }

extern "C" pa_status pa_pool_get_desc(const pa_pool* pool, pa_pool_desc* out) {
  if (!pool || !out) return PA_ERR_INVALID;
  *out = pool->desc;
  return PA_OK;
}

extern "C" size_t pa_pool_bytes(const pa_pool* pool, int which) {
  if (!pool || (which != 0 && which != 1)) return 0;
  const pa_pool_desc& d = pool->desc;
  size_t rb = pa_row_bytes(which == 0 ? d.k_type : d.v_type, d.head_dim);
  return (size_t)d.n_blocks * d.n_kv_heads * d.page_size * rb;
}

extern "C" pa_status pa_alloc_blocks(pa_pool* pool, uint32_t n, pa_block* out) {
  if (!pool || (n && !out)) return PA_ERR_INVALID;
  std::lock_guard<std::mutex> lk(pool->mu);
  if (n > pool->stack.size()) return PA_ERR_OOM;
  for (uint32_t i = 0; i < n; ++i) {
    uint32_t idx = pool->stack.back();
    pool->stack.pop_back();
    pool->ref[idx] = 1;
    out[i] = ((uint64_t)pool->gen[idx] << 32) | idx;
  }
  return PA_OK;
}

static bool handle_live(const pa_pool* p, pa_block h) {
  uint32_t idx = (uint32_t)(h & 0xffffffffu), gen = (uint32_t)(h >> 32);
  return idx < p->desc.n_blocks && p->ref[idx] > 0 && p->gen[idx] == gen;
}

static void free_block(pa_pool* p, uint32_t idx) {
  p->ref[idx] = 0;
  uint32_t g = p->gen[idx] + 1;
  p->gen[idx] = g ? g : 1;
  p->stack.push_back(idx);
}

extern "C" pa_status pa_release(pa_pool* pool, const pa_block* handles, uint32_t n) {
  if (!pool || (n && !handles)) return PA_ERR_INVALID;
  std::lock_guard<std::mutex> lk(pool->mu);
  // Validate everything first: live, right generation, no more occurrences
  // than references.
  new_stamp(pool);
  for (uint32_t i = 0; i < n; ++i) {
    if (!handle_live(pool, handles[i])) return PA_ERR_STALE;
    uint32_t idx = (uint32_t)(handles[i] & 0xffffffffu);
    if (++counter(pool, idx, 0) > pool->ref[idx]) return PA_ERR_STALE;
  }
  for (uint32_t i = 0; i < n; ++i) {
    uint32_t idx = (uint32_t)(handles[i] & 0xffffffffu);
    if (--pool->ref[idx] == 0) free_block(pool, idx);
  }
  return PA_OK;
}

extern "C" pa_status pa_share_blocks(pa_pool* pool, const pa_block* handles, uint32_t n) {
  if (!pool || (n && !handles)) return PA_ERR_INVALID;
  std::lock_guard<std::mutex> lk(pool->mu);
  new_stamp(pool);
  for (uint32_t i = 0; i < n; ++i) {
    if (!handle_live(pool, handles[i])) return PA_ERR_STALE;
    uint32_t idx = (uint32_t)(handles[i] & 0xffffffffu);
    if ((uint64_t)pool->ref[idx] + ++counter(pool, idx, 0) > 0x7fffffffu) return PA_ERR_INVALID;
  }
  for (uint32_t i = 0; i < n; ++i) ++pool->ref[(uint32_t)(handles[i] & 0xffffffffu)];
  return PA_OK;
}

extern "C" pa_status pa_block_refcount(const pa_pool* pool, pa_block handle, uint32_t* count) {
  if (!pool || !count) return PA_ERR_INVALID;
  std::lock_guard<std::mutex> lk(pool->mu);
  if (!handle_live(pool, handle)) return PA_ERR_STALE;
  *count = pool->ref[(uint32_t)(handle & 0xffffffffu)];
  return PA_OK;
}

extern "C" pa_status pa_cow_blocks(pa_pool* pool, const pa_block* handles, uint32_t n, pa_block* out,
                                   int32_t* copy_src, int32_t* copy_dst, uint32_t* n_copies) {
  if (!pool || (n && (!handles || !out || !copy_src || !copy_dst)) || !n_copies) return PA_ERR_INVALID;
  std::lock_guard<std::mutex> lk(pool->mu);
  // Count the copies the handles need, taken in order (a block shared r
  // times gives at most r - 1 copies in one call).
  new_stamp(pool);
  size_t copies = 0;
  for (uint32_t i = 0; i < n; ++i) {
    if (!handle_live(pool, handles[i])) return PA_ERR_STALE;
    uint32_t idx = (uint32_t)(handles[i] & 0xffffffffu);
    uint32_t& left = counter(pool, idx, pool->ref[idx]);
    if (left > 1) {
      ++copies;
      --left;
    }
  }
  if (copies > pool->stack.size()) return PA_ERR_OOM;
  uint32_t k = 0;
  for (uint32_t i = 0; i < n; ++i) {
    uint32_t idx = (uint32_t)(handles[i] & 0xffffffffu);
    if (pool->ref[idx] > 1) {
      --pool->ref[idx];
      uint32_t fresh = pool->stack.back();
      pool->stack.pop_back();
      pool->ref[fresh] = 1;
      out[i] = ((uint64_t)pool->gen[fresh] << 32) | fresh;
      copy_src[k] = (int32_t)idx;
      copy_dst[k] = (int32_t)fresh;
      ++k;
    } else {
      out[i] = handles[i];
    }
  }
  *n_copies = k;
  return PA_OK;
}

extern "C" pa_status pa_block_index(const pa_pool* pool, pa_block handle, int32_t* idx) {
  if (!pool || !idx) return PA_ERR_INVALID;
  std::lock_guard<std::mutex> lk(pool->mu);
  if (!handle_live(pool, handle)) return PA_ERR_STALE;
  *idx = (int32_t)(handle & 0xffffffffu);
  return PA_OK;
}

extern "C" uint32_t pa_pool_free_count(const pa_pool* pool) {
  if (!pool) return 0;
  std::lock_guard<std::mutex> lk(pool->mu);
  return (uint32_t)pool->stack.size();
}

extern "C" const char* pa_status_string(pa_status s) {
  switch (s) {
    case PA_OK: return "PA_OK";
    case PA_ERR_INVALID: return "PA_ERR_INVALID";
    case PA_ERR_UNSUPPORTED: return "PA_ERR_UNSUPPORTED";
    case PA_ERR_OOM: return "PA_ERR_OOM";
    case PA_ERR_STALE: return "PA_ERR_STALE";
    case PA_ERR_BOUNDS: return "PA_ERR_BOUNDS";
    case PA_ERR_TIMEOUT: return "PA_ERR_TIMEOUT";
    case PA_ERR_CUDA: return "PA_ERR_CUDA";
  }
  return "PA_ERR_UNKNOWN";
}
