// residency.cu -- pressure-driven page residency over one block pool.
//
// [P2] "vLLM's Hybrid HiSparse ...", "Three residency states, one block
// pool": KV starts on the GPU and gives up residency page by page as the pool
// runs short.  Full residency keeps every page in the pool while completed
// prefix pages are copied to host memory ahead of need; a request under
// pressure releases its coldest pages to host memory and keeps its tail on the
// GPU (mixed residency; the block table holds real blocks and null
// placeholders side by side); a request that reuses a prefix held only in host
// memory starts with placeholders (no residency).  The LRU hot-buffer resolver
// (skv_resolve_rows_lru) serves the placeholders' tokens.
//
// The policy is host code: a residency manager that owns the pool's free list
// and every request's page table, decides which pages to release, and lists
// the completed pages that still need their host copy (and the tail pages
// whose first rows must come back from host memory).  The device work is the
// page copy between the pool and the host tier (skv_materialize_pages,
// skv_fill_pages: one CTA per page, 16-byte loads and stores, the host side
// through its alias).  A page is released only after its host copy was
// issued on the stream that later decode work follows, so a reader never sees
// a placeholder whose host rows are not written.
#include <algorithm>
#include <new>
#include <vector>

#include "common.cuh"

namespace skv {
namespace {

constexpr int kCopyThreads = 256;

// Copies whole pages between the pool and the host tier: to_host = 1 writes a
// resident page's rows to the host (a completed page's copy ahead of need),
// 0 brings a page's host rows into its block (a tail page that becomes
// resident while earlier tokens of it live only in host memory).
__global__ __launch_bounds__(kCopyThreads) void page_copy_kernel(const int32_t* __restrict__ pages, int B, int page,
                                                                 const int32_t* __restrict__ block_table,
                                                                 int64_t n_pages, uint8_t* pool, int64_t row_bytes,
                                                                 int64_t n_pool_rows, uint8_t* host, int64_t t_cap,
                                                                 int to_host, int32_t* status) {
  const int j = blockIdx.x;
  const int b = pages[2 * j], p = pages[2 * j + 1];
  if (b < 0 || b >= B || p < 0 || p >= n_pages || static_cast<int64_t>(p + 1) * page > t_cap) {
    if (threadIdx.x == 0) set_status(status, SKV_DEV_RANGE);
    return;
  }
  const int64_t blk = block_table[static_cast<int64_t>(b) * n_pages + p];
  if (blk < 0 || (blk + 1) * page > n_pool_rows) {  // not resident: nothing to copy from
    if (threadIdx.x == 0) set_status(status, SKV_DEV_RANGE);
    return;
  }
  uint4* pp = reinterpret_cast<uint4*>(pool + blk * page * row_bytes);
  uint4* hp = reinterpret_cast<uint4*>(host + (static_cast<int64_t>(b) * t_cap + static_cast<int64_t>(p) * page) *
                                               row_bytes);
  const uint4* src = to_host ? pp : hp;
  uint4* dst = to_host ? hp : pp;
  const int64_t n16 = page * row_bytes / 16;
  constexpr int kU = 4;
  for (int64_t i0 = threadIdx.x; i0 < n16; i0 += kCopyThreads * kU) {
    uint4 v[kU];
#pragma unroll
    for (int u = 0; u < kU; u++)
      if (i0 + u * kCopyThreads < n16) v[u] = ld_nc16(src + i0 + u * kCopyThreads);
#pragma unroll
    for (int u = 0; u < kU; u++)
      if (i0 + u * kCopyThreads < n16) dst[i0 + u * kCopyThreads] = v[u];
  }
}

}  // namespace
}  // namespace skv

// ---------------------------------------------------------------------------
// The residency manager (host).
// ---------------------------------------------------------------------------
struct skv_residency {
  struct Req {
    bool live = false;
    int64_t n_tokens = 0;
    std::vector<int32_t> block;      // per page: pool block, or -1 (placeholder: host only)
    std::vector<uint8_t> host_copy;  // per page: its host rows are written (the copy was issued)
    std::vector<uint8_t> need_fill;  // per page: resident, earlier rows still only in host memory
    int64_t resident = 0;            // resident pages
    int64_t first_pending = 0;       // pages below: copied, placeholders or awaiting a fill
    int64_t first_release = 0;       // pages below: placeholders
    std::vector<int32_t> hot;        // blocks leased as the request's hot buffer
  };
  int n_blocks = 0, page = 0, tail_pages = 0;
  int64_t max_pages = 0;
  std::vector<int32_t> free_list;  // free blocks, a stack: the last one freed is taken first
  std::vector<Req> req;

  int64_t pages_of(int64_t n) const { return (n + page - 1) / page; }

  // Releases one page: among the releasable pages (resident, host copy
  // issued, neither the newest page nor among the last tail_pages pages), the
  // oldest page of the request holding the most resident pages (ties: the
  // lowest request number).
  // Oldest releasable page of a request, or -1.  Placeholders at the front
  // are skipped for good (a released page never comes back), so with pages
  // copied in order the search stops at its first step.
  int64_t oldest_releasable(Req& r) const {
    const int64_t keep = tail_pages > 1 ? tail_pages : 1;
    const int64_t used = pages_of(r.n_tokens);
    while (r.first_release < used && r.block[r.first_release] < 0) r.first_release++;
    for (int64_t p = r.first_release; p < used - keep; p++)
      if (r.block[p] >= 0 && r.host_copy[p] && !r.need_fill[p]) return p;
    return -1;
  }

  bool release_one(int32_t* out_b, int32_t* out_p) {
    int best = -1;
    int64_t best_res = 0, best_page = -1;
    for (size_t b = 0; b < req.size(); b++) {
      Req& r = req[b];
      if (!r.live || r.resident <= best_res) continue;
      const int64_t first = oldest_releasable(r);
      if (first >= 0) {
        best = static_cast<int>(b);
        best_res = r.resident;
        best_page = first;
      }
    }
    if (best < 0) return false;
    Req& r = req[best];
    free_list.push_back(r.block[best_page]);
    r.block[best_page] = -1;
    r.resident--;
    if (out_b) *out_b = best;
    if (out_p) *out_p = static_cast<int32_t>(best_page);
    return true;
  }

  // A free block, releasing a page under pressure when none is free; -1 if
  // nothing can be released.
  int32_t take_block() {
    if (free_list.empty() && !release_one(nullptr, nullptr)) return -1;
    const int32_t blk = free_list.back();
    free_list.pop_back();
    return blk;
  }

  bool valid(int b) const { return b >= 0 && b < static_cast<int>(req.size()) && req[b].live; }
};

using namespace skv;

SKV_EXPORT int skv_residency_create(int n_blocks, int page, int max_requests, int64_t max_pages, int tail_pages,
                                    skv_residency** out) {
  if (!out || n_blocks < 0 || page < 1 || max_requests < 1 || max_pages < 1 || tail_pages < 0) return SKV_EINVAL;
  skv_residency* r = new (std::nothrow) skv_residency;
  if (!r) return SKV_ENOMEM;
  r->n_blocks = n_blocks;
  r->page = page;
  r->tail_pages = tail_pages;
  r->max_pages = max_pages;
  r->req.resize(max_requests);
  r->free_list.reserve(n_blocks);
  for (int i = n_blocks - 1; i >= 0; i--) r->free_list.push_back(i);  // block 0 is taken first
  *out = r;
  return SKV_OK;
}

SKV_EXPORT void skv_residency_destroy(skv_residency* r) { delete r; }

SKV_EXPORT int skv_residency_add(skv_residency* r, int b, int64_t n_tokens, int host_prefix) {
  if (!r || b < 0 || b >= static_cast<int>(r->req.size()) || n_tokens < 0 || r->req[b].live) return SKV_EINVAL;
  if (r->pages_of(n_tokens) > r->max_pages) return SKV_EINVAL;
  skv_residency::Req q;
  q.live = true;
  q.n_tokens = n_tokens;
  q.block.assign(r->max_pages, -1);
  q.host_copy.assign(r->max_pages, 0);
  q.need_fill.assign(r->max_pages, 0);
  const int64_t used = r->pages_of(n_tokens);
  std::vector<int32_t> taken;
  for (int64_t p = 0; p < used; p++) {
    const bool partial = (p + 1) * r->page > n_tokens;
    if (host_prefix && !partial) {  // no residency: complete prefix pages live in host memory only
      q.host_copy[p] = 1;
      continue;
    }
    const int32_t blk = r->take_block();  // may release pages of the other requests
    if (blk < 0) {  // the pool cannot hold it: undo
      for (int32_t t : taken) r->free_list.push_back(t);
      r->req[b] = skv_residency::Req();
      return SKV_ENOMEM;
    }
    taken.push_back(blk);
    q.block[p] = blk;
    q.resident++;
    if (host_prefix) q.need_fill[p] = 1;  // the partial tail page: its first rows come from host memory
  }
  r->req[b] = q;
  return SKV_OK;
}

SKV_EXPORT int skv_residency_remove(skv_residency* r, int b) {
  if (!r || !r->valid(b)) return SKV_EINVAL;
  for (int32_t blk : r->req[b].block)
    if (blk >= 0) r->free_list.push_back(blk);
  for (int32_t blk : r->req[b].hot) r->free_list.push_back(blk);
  r->req[b] = skv_residency::Req();
  return SKV_OK;
}

SKV_EXPORT int skv_residency_append(skv_residency* r, int b, int64_t n) {
  if (!r || !r->valid(b) || n < 0) return SKV_EINVAL;
  if (r->pages_of(r->req[b].n_tokens + n) > r->max_pages) return SKV_EINVAL;
  const int64_t end = r->req[b].n_tokens + n;
  for (int64_t t = r->req[b].n_tokens; t < end; t++) {
    const int64_t p = t / r->page;
    if (r->req[b].block[p] >= 0) continue;  // the resident tail page
    const int32_t blk = r->take_block();    // may release pages of any request (never this tail)
    skv_residency::Req& q = r->req[b];
    if (blk < 0) {
      q.n_tokens = t;
      return SKV_ENOMEM;
    }
    q.block[p] = blk;
    q.resident++;
    q.host_copy[p] = 0;
    q.need_fill[p] = t % r->page != 0;  // earlier rows of the page are in host memory only
    q.n_tokens = t + 1;
  }
  r->req[b].n_tokens = end;
  return SKV_OK;
}

SKV_EXPORT int skv_residency_pending(const skv_residency* r, int b, int32_t* pages, int max_out, int* n_out) {
  if (!r || !n_out || !r->valid(b) || max_out < 0) return SKV_EINVAL;
  skv_residency::Req& q = const_cast<skv_residency*>(r)->req[b];  // the scan start is a cache
  const int64_t complete = q.n_tokens / r->page;
  while (q.first_pending < complete &&
         (q.block[q.first_pending] < 0 || q.host_copy[q.first_pending]) && !q.need_fill[q.first_pending])
    q.first_pending++;
  int n = 0;
  for (int64_t p = q.first_pending; p < complete; p++)
    if (q.block[p] >= 0 && !q.host_copy[p] && !q.need_fill[p]) {
      if (n >= max_out) return SKV_ENOMEM;
      if (pages) pages[n] = static_cast<int32_t>(p);
      n++;
    }
  *n_out = n;
  return SKV_OK;
}

SKV_EXPORT int skv_residency_mark_copied(skv_residency* r, int b, const int32_t* pages, int n) {
  if (!r || !r->valid(b) || n < 0 || (n > 0 && !pages)) return SKV_EINVAL;
  skv_residency::Req& q = r->req[b];
  const int64_t complete = q.n_tokens / r->page;
  for (int i = 0; i < n; i++)
    if (pages[i] < 0 || pages[i] >= complete || q.block[pages[i]] < 0 || q.need_fill[pages[i]]) return SKV_EINVAL;
  for (int i = 0; i < n; i++) q.host_copy[pages[i]] = 1;
  return SKV_OK;
}

SKV_EXPORT int skv_residency_fills(const skv_residency* r, int b, int32_t* pages, int max_out, int* n_out) {
  if (!r || !n_out || !r->valid(b) || max_out < 0) return SKV_EINVAL;
  const skv_residency::Req& q = r->req[b];
  int n = 0;
  for (int64_t p = 0; p < r->max_pages; p++)
    if (q.block[p] >= 0 && q.need_fill[p]) {
      if (n >= max_out) return SKV_ENOMEM;
      if (pages) pages[n] = static_cast<int32_t>(p);
      n++;
    }
  *n_out = n;
  return SKV_OK;
}

SKV_EXPORT int skv_residency_mark_filled(skv_residency* r, int b, const int32_t* pages, int n) {
  if (!r || !r->valid(b) || n < 0 || (n > 0 && !pages)) return SKV_EINVAL;
  skv_residency::Req& q = r->req[b];
  for (int i = 0; i < n; i++)
    if (pages[i] < 0 || pages[i] >= r->max_pages || q.block[pages[i]] < 0 || !q.need_fill[pages[i]])
      return SKV_EINVAL;
  for (int i = 0; i < n; i++) {  // the page's later rows are pool-only: it is copied out once complete
    q.need_fill[pages[i]] = 0;
    q.host_copy[pages[i]] = 0;
  }
  return SKV_OK;
}

SKV_EXPORT int skv_residency_lease_hot(skv_residency* r, int b, int n_pages, int32_t* blocks) {
  if (!r || !r->valid(b) || n_pages < 1 || !blocks || !r->req[b].hot.empty()) return SKV_EINVAL;
  std::vector<int32_t> got;
  for (int i = 0; i < n_pages; i++) {
    const int32_t blk = r->take_block();  // may release pages of any request, this one's included
    if (blk < 0) {
      for (int32_t t : got) r->free_list.push_back(t);
      return SKV_ENOMEM;
    }
    got.push_back(blk);
  }
  r->req[b].hot = got;
  for (int i = 0; i < n_pages; i++) blocks[i] = got[i];
  return SKV_OK;
}

SKV_EXPORT int skv_residency_reclaim(skv_residency* r, int n_wanted, int32_t* released, int* n_out) {
  if (!r || !n_out || n_wanted < 0 || (n_wanted > 0 && !released)) return SKV_EINVAL;
  int n = 0;
  while (n < n_wanted && r->release_one(released + 2 * n, released + 2 * n + 1)) n++;
  *n_out = n;
  return SKV_OK;
}

SKV_EXPORT int skv_residency_block_table(const skv_residency* r, int32_t* table) {
  if (!r || !table) return SKV_EINVAL;
  for (size_t b = 0; b < r->req.size(); b++)
    for (int64_t p = 0; p < r->max_pages; p++)
      table[b * r->max_pages + p] = r->req[b].live ? r->req[b].block[p] : -1;
  return SKV_OK;
}

SKV_EXPORT int skv_residency_state(const skv_residency* r, int b) {
  if (!r || !r->valid(b)) return -1;
  const skv_residency::Req& q = r->req[b];
  const int64_t used = r->pages_of(q.n_tokens);
  int64_t res = 0;
  for (int64_t p = 0; p < used; p++) res += q.block[p] >= 0;
  return res == used ? SKV_RESIDENCY_FULL : (res == 0 ? SKV_RESIDENCY_NONE : SKV_RESIDENCY_MIXED);
}

SKV_EXPORT int skv_residency_free_blocks(const skv_residency* r) {
  return r ? static_cast<int>(r->free_list.size()) : -1;
}

namespace {
int page_copy(int n, const int32_t* pages, int B, int page, const int32_t* block_table, int64_t n_pages,
              uint8_t* pool, int64_t row_bytes, int64_t n_pool_rows, uint8_t* host, int64_t t_cap, int to_host,
              int32_t* dev_status, void* stream) {
  if (n < 0 || B < 1 || page < 1 || n_pages < 1 || row_bytes < 16 || row_bytes % 16 || n_pool_rows < 0 || t_cap < 0)
    return SKV_EINVAL;
  if (n == 0) return SKV_OK;
  if (!pages || !block_table || !pool || !host || !aligned16(pool) || !aligned16(host)) return SKV_EINVAL;
  page_copy_kernel<<<n, kCopyThreads, 0, as_stream(stream)>>>(pages, B, page, block_table, n_pages, pool, row_bytes,
                                                               n_pool_rows, host, t_cap, to_host, dev_status);
  return launch_status();
}
}  // namespace

SKV_EXPORT int skv_materialize_pages(int n, const int32_t* pages, int B, int page, const int32_t* block_table,
                                     int64_t n_pages, const uint8_t* pool, int64_t row_bytes, int64_t n_pool_rows,
                                     uint8_t* host, int64_t t_cap, int32_t* dev_status, void* stream) {
  return page_copy(n, pages, B, page, block_table, n_pages, const_cast<uint8_t*>(pool), row_bytes, n_pool_rows, host,
                   t_cap, 1, dev_status, stream);
}

SKV_EXPORT int skv_fill_pages(int n, const int32_t* pages, int B, int page, const int32_t* block_table,
                              int64_t n_pages, uint8_t* pool, int64_t row_bytes, int64_t n_pool_rows,
                              const uint8_t* host, int64_t t_cap, int32_t* dev_status, void* stream) {
  return page_copy(n, pages, B, page, block_table, n_pages, pool, row_bytes, n_pool_rows, const_cast<uint8_t*>(host),
                   t_cap, 0, dev_status, stream);
}
