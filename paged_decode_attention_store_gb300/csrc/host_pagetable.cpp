// Host-side page-table bookkeeping of libpagedkv (pure C++, no CUDA).
//
// Chapter 15 of silicon_compiler_from_scratch, "A Paged KV Cache and
// Sliding-Window Attention", section "The model", defines the semantics:
// a LIFO free list, one reference count per physical page, a block table per
// request, a fresh page when the length reaches a page boundary, a whole-page
// copy before writing into a shared tail page (lazy copy-on-write), fork by
// sharing every page, release of front pages that the window no longer
// reaches, release of a finished request. With attention sinks (the
// chapter's exercise "Attention sinks": the first S rows stay in every
// context) the first ceil(S / P) pages are kept and the pages after them are
// released the same way.
//
// Layout here is built for the device: each request keeps its pages in a
// vector indexed by ABSOLUTE logical page, with -1 for pages the window has
// released, so that a row of the device block table is exactly that vector
// (chapter 15, Figure 15.1: the released pages leave holes at the front).
// Every change that lands in device memory is emitted as a table write
// (row, logical page, value) or a copy-on-write page pair.
#include <cstdint>
#include <cstring>
#include <new>
#include <vector>

#include "pagedkv.h"

namespace {

struct Request {
  bool live = false;
  int length = 0;            // rows stored
  int dropped = 0;           // pages released by trim (after the sink pages)
  int sink_pages = 0;        // front pages kept for attention sinks
  std::vector<int32_t> pages;  // absolute logical page -> physical page (-1 = hole)
};

}  // namespace

struct kvp_host {
  int num_pages = 0;
  int page_size = 0;
  std::vector<int32_t> free_stack;  // back() is handed out next
  std::vector<int32_t> ref;
  std::vector<Request> req;
};

namespace {

bool valid_rid(const kvp_host* h, int rid) {
  return h && rid >= 0 && rid < static_cast<int>(h->req.size());
}

// One reversible step of a batched append.
struct Undo {
  enum Kind { kAlloc, kPush, kCow, kLength } kind;
  int rid;
  int32_t a, b;
};

int32_t alloc_page(kvp_host* h, std::vector<Undo>& log) {
  int32_t p = h->free_stack.back();
  h->free_stack.pop_back();
  h->ref[p] = 1;
  log.push_back({Undo::kAlloc, -1, p, 0});
  return p;
}

void unref_page(kvp_host* h, int32_t p) {
  if (--h->ref[p] == 0) h->free_stack.push_back(p);
}

void rollback(kvp_host* h, std::vector<Undo>& log) {
  for (auto it = log.rbegin(); it != log.rend(); ++it) {
    Request& r = it->rid >= 0 ? h->req[it->rid] : h->req[0];
    switch (it->kind) {
      case Undo::kAlloc:  // page a went out with ref 1
        h->ref[it->a] = 0;
        h->free_stack.push_back(it->a);
        break;
      case Undo::kPush:
        r.pages.pop_back();
        break;
      case Undo::kCow:  // tail was a (shared), became b; a lost one reference
        r.pages.back() = it->a;
        h->ref[it->a] += 1;
        break;
      case Undo::kLength:
        r.length -= 1;
        break;
    }
  }
  log.clear();
}

}  // namespace

extern "C" {

int kvp_host_create(int num_pages, int page_size, int max_requests,
                    const int32_t* free_stack, kvp_host** out) {
  if (!out || num_pages <= 0 || page_size <= 0 || max_requests <= 0) return KVP_ERR_INVALID_ARG;
  kvp_host* h = new (std::nothrow) kvp_host;
  if (!h) return KVP_ERR_INVALID_ARG;
  h->num_pages = num_pages;
  h->page_size = page_size;
  h->ref.assign(num_pages, 0);
  h->req.resize(max_requests);
  h->free_stack.resize(num_pages);
  if (free_stack) {
    std::vector<char> seen(num_pages, 0);
    for (int i = 0; i < num_pages; ++i) {
      int32_t p = free_stack[i];
      if (p < 0 || p >= num_pages || seen[p]) {
        delete h;
        return KVP_ERR_INVALID_ARG;
      }
      seen[p] = 1;
      h->free_stack[i] = p;
    }
  } else {
    for (int i = 0; i < num_pages; ++i) h->free_stack[i] = num_pages - 1 - i;
  }
  *out = h;
  return KVP_OK;
}

int kvp_host_destroy(kvp_host* h) {
  delete h;
  return KVP_OK;
}

int kvp_host_new(kvp_host* h, int rid) {
  if (!valid_rid(h, rid) || h->req[rid].live) return KVP_ERR_INVALID_ARG;
  Request& r = h->req[rid];
  r.live = true;
  r.length = 0;
  r.dropped = 0;
  r.sink_pages = 0;
  r.pages.clear();
  return KVP_OK;
}

int kvp_host_fork(kvp_host* h, int src, int dst, int32_t* tw_rows, int32_t* tw_cols, int32_t* tw_vals,
                  int tw_cap, int* n_tw) {
  if (!valid_rid(h, src) || !valid_rid(h, dst) || src == dst || !n_tw) return KVP_ERR_INVALID_ARG;
  if (!h->req[src].live || h->req[dst].live) return KVP_ERR_INVALID_ARG;
  const int cnt = static_cast<int>(h->req[src].pages.size());
  if (cnt > tw_cap || (cnt > 0 && (!tw_rows || !tw_cols || !tw_vals))) return KVP_ERR_INVALID_ARG;
  Request& d = h->req[dst];
  d = h->req[src];
  for (int i = 0; i < cnt; ++i) {
    const int32_t p = d.pages[i];
    if (p >= 0) h->ref[p] += 1;
    tw_rows[i] = dst;
    tw_cols[i] = i;
    tw_vals[i] = p;
  }
  *n_tw = cnt;
  return KVP_OK;
}

int kvp_host_release(kvp_host* h, int rid) {
  if (!valid_rid(h, rid) || !h->req[rid].live) return KVP_ERR_INVALID_ARG;
  Request& r = h->req[rid];
  for (int32_t p : r.pages)
    if (p >= 0) unref_page(h, p);
  r.live = false;
  r.pages.clear();
  r.length = r.dropped = r.sink_pages = 0;
  return KVP_OK;
}

int kvp_host_append(kvp_host* h, const int32_t* rids, int n, int32_t* slots,
                    int32_t* tw_rows, int32_t* tw_cols, int32_t* tw_vals,
                    int tw_cap, int* n_tw, int32_t* cow_src, int32_t* cow_dst,
                    int* n_cow) {
  if (!h || n < 0 || (n > 0 && (!rids || !slots))) return KVP_ERR_INVALID_ARG;
  if (!n_tw || !n_cow || (n > 0 && (!tw_rows || !tw_cols || !tw_vals || !cow_src || !cow_dst)))
    return KVP_ERR_INVALID_ARG;
  for (int i = 0; i < n; ++i)
    if (!valid_rid(h, rids[i]) || !h->req[rids[i]].live) return KVP_ERR_INVALID_ARG;

  const int P = h->page_size;
  std::vector<Undo> log;
  log.reserve(4 * static_cast<size_t>(n));
  int ntw = 0, ncow = 0;
  for (int i = 0; i < n; ++i) {
    const int rid = rids[i];
    Request& r = h->req[rid];
    const int off = r.length % P;
    if (off == 0) {
      if (h->free_stack.empty() || ntw >= tw_cap) {
        int code = h->free_stack.empty() ? KVP_ERR_OUT_OF_PAGES : KVP_ERR_INVALID_ARG;
        rollback(h, log);
        return code;
      }
      int32_t p = alloc_page(h, log);
      r.pages.push_back(p);
      log.push_back({Undo::kPush, rid, 0, 0});
      tw_rows[ntw] = rid;
      tw_cols[ntw] = static_cast<int32_t>(r.pages.size()) - 1;
      tw_vals[ntw] = p;
      ++ntw;
    } else {
      const int32_t shared = r.pages.back();
      if (h->ref[shared] > 1) {
        if (h->free_stack.empty() || ntw >= tw_cap) {
          int code = h->free_stack.empty() ? KVP_ERR_OUT_OF_PAGES : KVP_ERR_INVALID_ARG;
          rollback(h, log);
          return code;
        }
        int32_t q = alloc_page(h, log);
        h->ref[shared] -= 1;  // stays >= 1: another owner still holds it
        r.pages.back() = q;
        log.push_back({Undo::kCow, rid, shared, q});
        cow_src[ncow] = shared;
        cow_dst[ncow] = q;
        ++ncow;
        tw_rows[ntw] = rid;
        tw_cols[ntw] = static_cast<int32_t>(r.pages.size()) - 1;
        tw_vals[ntw] = q;
        ++ntw;
      }
    }
    slots[i] = r.pages.back() * P + off;
    r.length += 1;
    log.push_back({Undo::kLength, rid, 0, 0});
  }
  *n_tw = ntw;
  *n_cow = ncow;
  return KVP_OK;
}

int kvp_host_trim_sinks(kvp_host* h, int rid, int keep_from, int sink_rows, int32_t* tw_rows,
                        int32_t* tw_cols, int32_t* tw_vals, int tw_cap, int* n_tw) {
  if (!valid_rid(h, rid) || !h->req[rid].live || !n_tw || sink_rows < 0) return KVP_ERR_INVALID_ARG;
  Request& r = h->req[rid];
  const int P = h->page_size;
  const int sp = static_cast<int>((static_cast<long long>(sink_rows) + P - 1) / P);
  if (r.dropped > 0 && sp != r.sink_pages) return KVP_ERR_INVALID_ARG;  // sinks fixed once pages went
  // Count first so that a short output buffer changes nothing.
  int count = 0;
  for (int d = sp + r.dropped; d < static_cast<int>(r.pages.size()) && static_cast<long long>(d + 1) * P <= keep_from;
       ++d)
    ++count;
  if (count > 0 && (!tw_rows || !tw_cols || !tw_vals || count > tw_cap)) return KVP_ERR_INVALID_ARG;
  r.sink_pages = sp;
  for (int k = 0; k < count; ++k) {
    const int d = sp + r.dropped;
    unref_page(h, r.pages[d]);
    r.pages[d] = -1;
    tw_rows[k] = rid;
    tw_cols[k] = d;
    tw_vals[k] = -1;
    r.dropped += 1;
  }
  *n_tw = count;
  return KVP_OK;
}

int kvp_host_trim(kvp_host* h, int rid, int keep_from, int32_t* tw_rows,
                  int32_t* tw_cols, int32_t* tw_vals, int tw_cap, int* n_tw) {
  return kvp_host_trim_sinks(h, rid, keep_from, 0, tw_rows, tw_cols, tw_vals, tw_cap, n_tw);
}

int kvp_host_rewind(kvp_host* h, int rid, int n, int32_t* tw_rows, int32_t* tw_cols, int32_t* tw_vals,
                    int tw_cap, int* n_tw) {
  if (!valid_rid(h, rid) || !h->req[rid].live || !n_tw) return KVP_ERR_INVALID_ARG;
  Request& r = h->req[rid];
  const int P = h->page_size;
  if (n < 0 || n > r.length) return KVP_ERR_INVALID_ARG;
  const int keep_len = r.length - n;
  // Rows a later step may read must stay: no rewind into released pages.
  if (r.dropped > 0 && static_cast<long long>(keep_len) < static_cast<long long>(r.sink_pages + r.dropped) * P)
    return KVP_ERR_INVALID_ARG;
  const int keep_pages = static_cast<int>((static_cast<long long>(keep_len) + P - 1) / P);
  const int count = static_cast<int>(r.pages.size()) - keep_pages;
  if (count > 0 && (!tw_rows || !tw_cols || !tw_vals || count > tw_cap)) return KVP_ERR_INVALID_ARG;
  // Tail first, so that the stack hands the pages back in logical order.
  for (int k = 0; k < count; ++k) {
    const int d = static_cast<int>(r.pages.size()) - 1;
    unref_page(h, r.pages[d]);
    r.pages.pop_back();
    tw_rows[k] = rid;
    tw_cols[k] = d;
    tw_vals[k] = -1;
  }
  r.length = keep_len;
  *n_tw = count > 0 ? count : 0;
  return KVP_OK;
}

int kvp_host_used(const kvp_host* h, int* used) {
  if (!h || !used) return KVP_ERR_INVALID_ARG;
  *used = h->num_pages - static_cast<int>(h->free_stack.size());
  return KVP_OK;
}

int kvp_host_length(const kvp_host* h, int rid, int* length, int* dropped) {
  if (!valid_rid(h, rid) || !h->req[rid].live) return KVP_ERR_INVALID_ARG;
  if (length) *length = h->req[rid].length;
  if (dropped) *dropped = h->req[rid].dropped;
  return KVP_OK;
}

int kvp_host_block_row(const kvp_host* h, int rid, int32_t* out, int cap, int* n) {
  if (!valid_rid(h, rid) || !h->req[rid].live || !n) return KVP_ERR_INVALID_ARG;
  const auto& pages = h->req[rid].pages;
  const int cnt = static_cast<int>(pages.size());
  if (cnt > cap || (cnt > 0 && !out)) return KVP_ERR_INVALID_ARG;
  if (cnt > 0) std::memcpy(out, pages.data(), sizeof(int32_t) * cnt);
  *n = cnt;
  return KVP_OK;
}

int kvp_host_refcounts(const kvp_host* h, int32_t* out, int cap) {
  if (!h || !out || cap < h->num_pages) return KVP_ERR_INVALID_ARG;
  std::memcpy(out, h->ref.data(), sizeof(int32_t) * h->num_pages);
  return KVP_OK;
}

int kvp_host_free_list(const kvp_host* h, int32_t* out, int cap, int* n) {
  if (!h || !n) return KVP_ERR_INVALID_ARG;
  const int cnt = static_cast<int>(h->free_stack.size());
  if (cnt > cap || (cnt > 0 && !out)) return KVP_ERR_INVALID_ARG;
  if (cnt > 0) std::memcpy(out, h->free_stack.data(), sizeof(int32_t) * cnt);
  *n = cnt;
  return KVP_OK;
}

}  // extern "C"
