// Device-side page allocation of libpagedkv: the block-table bookkeeping of
// chapter 15 of silicon_compiler_from_scratch ("A Paged KV Cache and
// Sliding-Window Attention", section "The model": a LIFO free list, one
// reference count per page, a fresh page on a page boundary, a whole-page
// copy before writing into a shared tail page, release of the pages a
// window no longer reaches) kept in device memory, so that a decode step
// needs no host decision and no host->device copy of table writes (the
// mini-sglang code series, part 4, section "할당은 페이지로, 기록은 토큰으로":
// allocate by page, record by token; here both happen on the device).
//
// The state lives in one caller-owned device buffer:
//   [top, error word, pad][stack: num_pages][ref: num_pages]
//   [len | dropped | sink pages: max_requests each]
// stack[0 .. top) is the free list, stack[top - 1] handed out next.
//
// Each call runs as ONE thread block (n <= 1024 requests), which gathers the
// requests' state in parallel, orders every decision exactly as the host
// bookkeeping would take them one request after the other (block scans for
// the pop and push positions, ranks among requests that share a page), and
// scatters the results. The whole call is all-or-nothing: a bad argument,
// a full pool or a short output buffer records an error and changes nothing.
#include <new>

#include "attention.cuh"

struct kvp_dev_pages {
  int num_pages, page_size, max_requests;
  int32_t* top;  // [0] top, [1] error word
  int32_t* stack;
  int32_t* ref;
  int32_t* len;
  int32_t* dropped;
  int32_t* sinkp;
  int32_t* table;
  int rows, cols, raw;
  // copy streams (host to device, device to host) and events of the
  // host-buffer steps, created on their first call
  void* io_stream;
  void* io_stream2;
  void** io_events;
  int io_nevents;
};

namespace kvp {

namespace {

constexpr int kDevThreads = 1024;
constexpr int kMaxReleases = 4096;  // pages one trim or release call may let go

size_t align16(size_t x) { return (x + 15) & ~size_t(15); }

struct DevState {
  int num_pages, P, max_requests;
  int32_t* top;
  int32_t* err;
  int32_t* stack;
  int32_t* ref;
  int32_t* len;
  int32_t* dropped;
  int32_t* sinkp;
  int32_t* table;
  int rows, cols, raw;
};

DevState state_of(const kvp_dev_pages* d) {
  DevState s;
  s.num_pages = d->num_pages;
  s.P = d->page_size;
  s.max_requests = d->max_requests;
  s.top = d->top;
  s.err = d->top + 1;
  s.stack = d->stack;
  s.ref = d->ref;
  s.len = d->len;
  s.dropped = d->dropped;
  s.sinkp = d->sinkp;
  s.table = d->table;
  s.rows = d->rows;
  s.cols = d->cols;
  s.raw = d->raw;
  return s;
}

// Physical page behind absolute logical page lp of table row r (-1: none).
__device__ __forceinline__ int page_at(const DevState& s, int r, int lp) {
  const long long c = s.raw ? (long long)lp * s.P : lp;
  if (lp < 0 || c >= s.cols) return -1;
  const int e = s.table[(size_t)r * s.cols + c];
  if (e < 0) return -1;
  return s.raw ? e / s.P : e;
}

// Table entry (or the P token entries) of logical page lp := page (-1: released).
__device__ __forceinline__ void set_page(const DevState& s, int r, int lp, int page) {
  int32_t* row = s.table + (size_t)r * s.cols;
  if (s.raw) {
    for (int j = 0; j < s.P; ++j) row[(size_t)lp * s.P + j] = page < 0 ? -1 : page * s.P + j;
  } else {
    row[lp] = page;
  }
}

__device__ __forceinline__ int ceil_div_d(int a, int b) { return (a + b - 1) / b; }

__global__ void dev_init_kernel(DevState s, const int32_t* free_stack) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < s.num_pages; i += gridDim.x * blockDim.x) {
    s.stack[i] = free_stack ? free_stack[i] : s.num_pages - 1 - i;
    s.ref[i] = 0;
  }
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < s.max_requests; i += gridDim.x * blockDim.x)
    s.len[i] = s.dropped[i] = s.sinkp[i] = 0;
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    *s.top = s.num_pages;
    *s.err = 0;
  }
}

__global__ void dev_new_kernel(DevState s, const int32_t* rids, int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const int r = rids[i];
  if ((unsigned)r >= (unsigned)s.max_requests) {
    set_error(s.err, KVP_ERR_INVALID_ARG);
    return;
  }
  s.len[r] = s.dropped[r] = s.sinkp[r] = 0;
}

// ``uniform`` token rows per request when counts is NULL; counts[i] rows for
// request i otherwise (a verify step's drafts). Request-major slots in out_loc.
__global__ void __launch_bounds__(kDevThreads) dev_append_kernel(DevState s, const int32_t* rids,
                                                                  const int32_t* counts, int uniform, int n,
                                                                  int32_t* out_loc, int max_tokens, int32_t* cow_src,
                                                                  int32_t* cow_dst, int32_t* n_cow,
                                                                  int32_t* lens_out) {
  __shared__ int s_tail[kDevThreads];
  __shared__ int s_rid[kDevThreads];
  const int i = threadIdx.x;
  const int P = s.P;
  bool ok = true;
  int r = -1, L = 0, c = 0, off = 0, tl = -1, tail = -1, ref0 = 0, first_new = 0, b = 0;
  griddep_wait();  // a programmatic dependent launch: the previous kernels' state is visible from here on
  griddep_launch_dependents();
  if (i < n) {
    r = rids[i];
    c = counts ? counts[i] : uniform;
    if ((unsigned)r >= (unsigned)s.max_requests || r >= s.rows || c < 0) {
      ok = false;
    } else {
      L = s.len[r];
      off = L % P;
      first_new = ceil_div_d(L, P);           // first logical page this call may add
      const int last = ceil_div_d(L + c, P);  // logical pages after the call
      b = last - first_new;
      if ((long long)last * (s.raw ? P : 1) > s.cols) ok = false;  // the row cannot hold them
      if (c > 0 && off != 0) {
        tl = L / P;
        tail = page_at(s, r, tl);
        if ((unsigned)tail >= (unsigned)s.num_pages) ok = false;
        else ref0 = s.ref[tail];
      }
    }
  }
  s_rid[i] = i < n ? r : -1;
  s_tail[i] = (i < n && ok && c > 0 && off != 0) ? tail : -1;
  __syncthreads();
  if (i < n && ok) {
    for (int j = 0; j < i; ++j)
      if (s_rid[j] == r) ok = false;  // one entry per request and call
  }
  if (__syncthreads_or(i < n && !ok)) {
    if (i == 0) set_error(s.err, KVP_ERR_INVALID_ARG);
    return;
  }
  // Lazy copy-on-write in call order: the k-th request (0-based) of this
  // call writing into shared tail page t sees ref[t] - k.
  int rank = 0;
  if (tail >= 0 && c > 0 && off != 0)
    for (int j = 0; j < i; ++j) rank += s_tail[j] == tail;
  const int cow = (i < n && c > 0 && off != 0 && ref0 - rank > 1) ? 1 : 0;
  const int need = i < n ? cow + b : 0;
  long long tot_need, tot_tok, tot_cow;
  const int o_pop = (int)block_exclusive_scan(need, &tot_need);
  const int o_tok = (int)block_exclusive_scan(i < n ? c : 0, &tot_tok);
  const int o_cow = (int)block_exclusive_scan(cow, &tot_cow);
  const int top = *s.top;
  if (tot_need > top || tot_tok > max_tokens) {
    if (i == 0) set_error(s.err, tot_need > top ? KVP_ERR_OUT_OF_PAGES : KVP_ERR_INVALID_ARG);
    return;
  }
  if (i < n) {
    // pops of this request, in order: the copy (if any), then the new pages
    int q = -1;
    if (cow) {
      q = s.stack[top - 1 - o_pop];
      s.ref[q] = 1;
      atomicSub(&s.ref[tail], 1);  // stays >= 1: another owner keeps it
      set_page(s, r, tl, q);
      cow_src[o_cow] = tail;
      cow_dst[o_cow] = q;
    }
    for (int k = 0; k < b; ++k) {
      const int p = s.stack[top - 1 - (o_pop + cow + k)];
      s.ref[p] = 1;
      set_page(s, r, first_new + k, p);
    }
    for (int k = 0; k < c; ++k) {
      const int t = L + k, lp = t / P;
      const int page = (off != 0 && lp == tl) ? (cow ? q : tail) : s.stack[top - 1 - (o_pop + cow + lp - first_new)];
      out_loc[o_tok + k] = page * P + t % P;
    }
    s.len[r] = L + c;
    if (lens_out) lens_out[i] = L + c;
  }
  __syncthreads();
  if (i == 0) {
    *s.top = top - (int)tot_need;
    if (n_cow) *n_cow = (int)tot_cow;
  }
}

// Trim (mode 0): release the pages after the sink pages that lie wholly
// below keep_from[i]; release (mode 1): let go of every live page and end
// the request; rewind (mode 2): drop the newest keep_from[i] rows and let go
// of the pages past the new length, tail first (the host's rewind, so that
// the stack hands them back in logical order). Pages go back in call order,
// each pushed by the release that drops its count to zero (that is the
// host's order).
__global__ void __launch_bounds__(kDevThreads) dev_release_kernel(DevState s, const int32_t* rids,
                                                                   const int32_t* keep_from, int window, int sinks,
                                                                   int n, int mode) {
  __shared__ int s_page[kMaxReleases];
  __shared__ int s_ref0[kMaxReleases];
  __shared__ int s_rid[kDevThreads];
  const int i = threadIdx.x;
  const int P = s.P;
  bool ok = true;
  int r = -1, cnt = 0, lo = 0, sp = 0, d = 0, pages = 0, keep_len = 0;
  griddep_wait();
  griddep_launch_dependents();
  if (i < n) {
    r = rids[i];
    if ((unsigned)r >= (unsigned)s.max_requests || r >= s.rows) {
      ok = false;
    } else {
      const int L = s.len[r];
      d = s.dropped[r];
      pages = ceil_div_d(L, P);
      if (mode == 0) {
        sp = ceil_div_d(sinks, P);
        if (sinks < 0 || (d > 0 && sp != s.sinkp[r])) ok = false;  // sinks fixed once pages went
        // without keep_from: what the next decode step reads, L + 1 - (W - S)
        const int kf = keep_from ? keep_from[i] : L + 1 - (window - sinks);
        const int hi = min(kf > 0 ? kf / P : 0, pages);
        lo = sp + d;
        cnt = max(0, hi - lo);
      } else if (mode == 1) {
        sp = s.sinkp[r];
        cnt = pages - d;  // every live page: the sink pages, then the ones after the holes
      } else {
        const int back = keep_from[i];
        keep_len = L - back;
        sp = s.sinkp[r];
        // no rewind into the rows a window or its sinks released
        if (back < 0 || back > L || (d > 0 && (long long)keep_len < (long long)(sp + d) * P)) ok = false;
        lo = ceil_div_d(keep_len, P);  // first logical page let go
        cnt = ok ? pages - lo : 0;
      }
    }
  }
  s_rid[i] = i < n ? r : -1;
  __syncthreads();
  if (i < n && ok)
    for (int j = 0; j < i; ++j)
      if (s_rid[j] == r) ok = false;
  if (__syncthreads_or(i < n && !ok)) {
    if (i == 0) set_error(s.err, KVP_ERR_INVALID_ARG);
    return;
  }
  long long total;
  const int o = (int)block_exclusive_scan(cnt, &total);
  if (total > kMaxReleases) {
    if (i == 0) set_error(s.err, KVP_ERR_INVALID_ARG);
    return;
  }
  for (int k = 0; k < cnt; ++k) {
    // logical page of the k-th release: trim [lo, lo + cnt); release skips the
    // holes [sp, sp + d); rewind goes from the tail down to lo
    const int lp = mode == 0 ? lo + k : mode == 1 ? (d > 0 && k >= sp ? k + d : k) : pages - 1 - k;
    const int p = page_at(s, r, lp);
    s_page[o + k] = p;
    s_ref0[o + k] = (unsigned)p < (unsigned)s.num_pages ? s.ref[p] : 0;
  }
  __syncthreads();
  // Entries e = 4 * tid .. 4 * tid + 3 (call order): which ones push their page.
  const int E = (int)total;
  int pushed[4];
  int mine = 0;
  for (int u = 0; u < 4; ++u) {
    const int e = 4 * i + u;
    pushed[u] = 0;
    if (e < E && (unsigned)s_page[e] < (unsigned)s.num_pages) {
      int rank = 0;
      for (int e2 = 0; e2 < e; ++e2) rank += s_page[e2] == s_page[e];
      pushed[u] = s_ref0[e] - rank == 1;
    }
    mine += pushed[u];
  }
  long long n_push;
  int pos = (int)block_exclusive_scan(mine, &n_push);
  const int top = *s.top;
  __syncthreads();
  for (int u = 0; u < 4; ++u) {
    const int e = 4 * i + u;
    if (e >= E) break;
    const int p = s_page[e];
    if ((unsigned)p >= (unsigned)s.num_pages) {
      set_error(s.err, KVP_ERR_BAD_INDEX);
      continue;
    }
    atomicSub(&s.ref[p], 1);
    if (pushed[u]) s.stack[top + pos++] = p;
  }
  if (i < n) {
    if (mode == 0) {
      for (int k = 0; k < cnt; ++k) set_page(s, r, lo + k, -1);
      s.dropped[r] = d + cnt;
      s.sinkp[r] = sp;
    } else if (mode == 1) {
      s.len[r] = s.dropped[r] = s.sinkp[r] = 0;
    } else {
      for (int k = 0; k < cnt; ++k) set_page(s, r, lo + k, -1);
      s.len[r] = keep_len;
    }
  }
  __syncthreads();
  if (i == 0) *s.top = top + (int)n_push;
}

// Fork (chapter 15, "The model"): request dst[i] gets src[i]'s table row,
// length, released pages and sink pages; every live page gains a reference.
// One block per pair.
__global__ void dev_fork_kernel(DevState s, const int32_t* src, const int32_t* dst, int n) {
  const int i = blockIdx.x;
  const int a = src[i], b = dst[i];
  if ((unsigned)a >= (unsigned)s.max_requests || (unsigned)b >= (unsigned)s.max_requests || a >= s.rows ||
      b >= s.rows || a == b) {
    if (threadIdx.x == 0) set_error(s.err, KVP_ERR_INVALID_ARG);
    return;
  }
  const int pages = ceil_div_d(s.len[a], s.P);
  for (int lp = threadIdx.x; lp < pages; lp += blockDim.x) {
    const int p = page_at(s, a, lp);
    set_page(s, b, lp, p);
    if (p >= 0) atomicAdd(&s.ref[p], 1);
  }
  if (threadIdx.x == 0) {
    s.len[b] = s.len[a];
    s.dropped[b] = s.dropped[a];
    s.sinkp[b] = s.sinkp[a];
  }
}

// One block of kDevThreads as a programmatic dependent launch: it may start
// while the previous kernel of the stream finishes, and waits for it
// (griddep_wait) before touching anything.
template <typename... Args>
cudaError_t launch_one_block(void (*kernel)(Args...), cudaStream_t stream, Args... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1);
  cfg.blockDim = dim3(kDevThreads);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

}  // namespace

}  // namespace kvp

using namespace kvp;

extern "C" int kvp_dev_pages_bytes(int num_pages, int max_requests, size_t* bytes) {
  if (num_pages <= 0 || max_requests <= 0 || !bytes) return KVP_ERR_INVALID_ARG;
  *bytes = 16 + 2 * align16(sizeof(int32_t) * num_pages) + 3 * align16(sizeof(int32_t) * max_requests);
  return KVP_OK;
}

extern "C" int kvp_dev_pages_create(int num_pages, int page_size, int max_requests, void* state, size_t state_bytes,
                                    int32_t* table, int table_rows, int table_cols, int table_mode,
                                    kvp_dev_pages** out) {
  size_t need = 0;
  if (!out || !state || !table || page_size <= 0 || table_rows < max_requests || table_cols <= 0)
    return KVP_ERR_INVALID_ARG;
  if (kvp_dev_pages_bytes(num_pages, max_requests, &need) != KVP_OK || state_bytes < need) return KVP_ERR_INVALID_ARG;
  if (table_mode != KVP_BLOCK_TABLE && table_mode != KVP_RAW_LOCATIONS) return KVP_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(state) & 15) return KVP_ERR_INVALID_ARG;
  if ((long long)num_pages * page_size > 0x7fffffffLL) return KVP_ERR_INVALID_ARG;
  kvp_dev_pages* d = new (std::nothrow) kvp_dev_pages;
  if (!d) return KVP_ERR_INVALID_ARG;
  char* p = static_cast<char*>(state);
  d->num_pages = num_pages;
  d->page_size = page_size;
  d->max_requests = max_requests;
  d->top = reinterpret_cast<int32_t*>(p);
  p += 16;
  d->stack = reinterpret_cast<int32_t*>(p);
  p += align16(sizeof(int32_t) * num_pages);
  d->ref = reinterpret_cast<int32_t*>(p);
  p += align16(sizeof(int32_t) * num_pages);
  d->len = reinterpret_cast<int32_t*>(p);
  p += align16(sizeof(int32_t) * max_requests);
  d->dropped = reinterpret_cast<int32_t*>(p);
  p += align16(sizeof(int32_t) * max_requests);
  d->sinkp = reinterpret_cast<int32_t*>(p);
  d->table = table;
  d->rows = table_rows;
  d->cols = table_cols;
  d->raw = table_mode == KVP_RAW_LOCATIONS;
  d->io_stream = nullptr;
  d->io_stream2 = nullptr;
  d->io_events = nullptr;
  d->io_nevents = 0;
  *out = d;
  return KVP_OK;
}

extern "C" int kvp_dev_pages_destroy(kvp_dev_pages* d) {
  if (!d) return KVP_OK;
  for (int i = 0; i < d->io_nevents; ++i)
    if (d->io_events[i]) cudaEventDestroy(static_cast<cudaEvent_t>(d->io_events[i]));
  delete[] d->io_events;
  if (d->io_stream) cudaStreamDestroy(static_cast<cudaStream_t>(d->io_stream));
  if (d->io_stream2) cudaStreamDestroy(static_cast<cudaStream_t>(d->io_stream2));
  delete d;
  return KVP_OK;
}

// The two copy streams and ``nevents`` events of the host-buffer steps
// (created once, kept until kvp_dev_pages_destroy).
int kvp_dev_io_resources(kvp_dev_pages* d, int nevents, void** stream, void** stream2, void*** events) {
  if (!d->io_stream) {
    cudaStream_t s;
    if (cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking) != cudaSuccess) return KVP_ERR_CUDA;
    d->io_stream = s;
  }
  if (!d->io_stream2) {
    cudaStream_t s;
    if (cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking) != cudaSuccess) return KVP_ERR_CUDA;
    d->io_stream2 = s;
  }
  if (d->io_nevents < nevents) {
    void** ev = new (std::nothrow) void*[nevents];
    if (!ev) return KVP_ERR_INVALID_ARG;
    for (int i = 0; i < d->io_nevents; ++i) ev[i] = d->io_events[i];
    delete[] d->io_events;
    d->io_events = ev;
    for (int i = d->io_nevents; i < nevents; ++i) {
      cudaEvent_t e;
      if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) return KVP_ERR_CUDA;
      d->io_events[i] = e;
      d->io_nevents = i + 1;
    }
  }
  *stream = d->io_stream;
  *stream2 = d->io_stream2;
  *events = d->io_events;
  return KVP_OK;
}

extern "C" int kvp_dev_pages_init(kvp_dev_pages* d, const int32_t* free_stack, void* stream) {
  if (!d) return KVP_ERR_INVALID_ARG;
  const int work = d->num_pages > d->max_requests ? d->num_pages : d->max_requests;
  const int blocks = (work + 255) / 256 < 1024 ? (work + 255) / 256 : 1024;
  dev_init_kernel<<<blocks, 256, 0, static_cast<cudaStream_t>(stream)>>>(state_of(d), free_stack);
  return cudaGetLastError() == cudaSuccess ? KVP_OK : KVP_ERR_CUDA;
}

extern "C" int kvp_dev_new(kvp_dev_pages* d, const int32_t* rids, int n, void* stream) {
  if (!d || n < 0 || (n > 0 && !rids)) return KVP_ERR_INVALID_ARG;
  if (n == 0) return KVP_OK;
  dev_new_kernel<<<(n + 255) / 256, 256, 0, static_cast<cudaStream_t>(stream)>>>(state_of(d), rids, n);
  return cudaGetLastError() == cudaSuccess ? KVP_OK : KVP_ERR_CUDA;
}

extern "C" int kvp_dev_append(kvp_dev_pages* d, const int32_t* rids, const int32_t* counts, int n, int32_t* out_loc,
                              int max_tokens, int32_t* cow_src, int32_t* cow_dst, int32_t* n_cow, int32_t* lens_out,
                              void* stream) {
  if (!d || n < 0 || n > kDevThreads || max_tokens < 0) return KVP_ERR_INVALID_ARG;
  if (n == 0) return KVP_OK;
  if (!rids || !out_loc || !cow_src || !cow_dst) return KVP_ERR_INVALID_ARG;
  const cudaError_t e = launch_one_block(dev_append_kernel, static_cast<cudaStream_t>(stream), state_of(d), rids,
                                         counts, 1, n, out_loc, max_tokens, cow_src, cow_dst, n_cow, lens_out);
  return e == cudaSuccess ? KVP_OK : KVP_ERR_CUDA;
}

// kvp_dev_append with the same number of rows (``count``) for every request,
// without a device array of counts (the verify step's drafts).
int kvp_dev_append_uniform(kvp_dev_pages* d, const int32_t* rids, int count, int n, int32_t* out_loc, int max_tokens,
                           int32_t* cow_src, int32_t* cow_dst, int32_t* n_cow, int32_t* lens_out, void* stream) {
  if (!d || n < 0 || n > kDevThreads || max_tokens < 0 || count < 0) return KVP_ERR_INVALID_ARG;
  if (n == 0) return KVP_OK;
  if (!rids || !out_loc || !cow_src || !cow_dst) return KVP_ERR_INVALID_ARG;
  const cudaError_t e = launch_one_block(dev_append_kernel, static_cast<cudaStream_t>(stream), state_of(d), rids,
                                         static_cast<const int32_t*>(nullptr), count, n, out_loc, max_tokens, cow_src,
                                         cow_dst, n_cow, lens_out);
  return e == cudaSuccess ? KVP_OK : KVP_ERR_CUDA;
}

extern "C" int kvp_dev_rewind(kvp_dev_pages* d, const int32_t* rids, const int32_t* n_back, int n, void* stream) {
  if (!d || n < 0 || n > kDevThreads) return KVP_ERR_INVALID_ARG;
  if (n == 0) return KVP_OK;
  if (!rids || !n_back) return KVP_ERR_INVALID_ARG;
  const cudaError_t e = launch_one_block(dev_release_kernel, static_cast<cudaStream_t>(stream), state_of(d), rids,
                                         n_back, 0, 0, n, 2);
  return e == cudaSuccess ? KVP_OK : KVP_ERR_CUDA;
}

extern "C" int kvp_dev_trim(kvp_dev_pages* d, const int32_t* rids, const int32_t* keep_from, int n, int window,
                            int sinks, void* stream) {
  if (!d || n < 0 || n > kDevThreads || sinks < 0) return KVP_ERR_INVALID_ARG;
  if (!keep_from && (window <= 0 || sinks >= window)) return KVP_ERR_INVALID_ARG;
  if (n == 0) return KVP_OK;
  if (!rids) return KVP_ERR_INVALID_ARG;
  const cudaError_t e = launch_one_block(dev_release_kernel, static_cast<cudaStream_t>(stream), state_of(d), rids,
                                         keep_from, window, sinks, n, 0);
  return e == cudaSuccess ? KVP_OK : KVP_ERR_CUDA;
}

extern "C" int kvp_dev_release(kvp_dev_pages* d, const int32_t* rids, int n, void* stream) {
  if (!d || n < 0 || n > kDevThreads) return KVP_ERR_INVALID_ARG;
  if (n == 0) return KVP_OK;
  if (!rids) return KVP_ERR_INVALID_ARG;
  const cudaError_t e = launch_one_block(dev_release_kernel, static_cast<cudaStream_t>(stream), state_of(d), rids,
                                         static_cast<const int32_t*>(nullptr), 0, 0, n, 1);
  return e == cudaSuccess ? KVP_OK : KVP_ERR_CUDA;
}

extern "C" int kvp_dev_fork(kvp_dev_pages* d, const int32_t* src, const int32_t* dst, int n, void* stream) {
  if (!d || n < 0 || (n > 0 && (!src || !dst))) return KVP_ERR_INVALID_ARG;
  if (n == 0) return KVP_OK;
  dev_fork_kernel<<<n, 256, 0, static_cast<cudaStream_t>(stream)>>>(state_of(d), src, dst, n);
  return cudaGetLastError() == cudaSuccess ? KVP_OK : KVP_ERR_CUDA;
}

extern "C" int kvp_dev_sync_error(kvp_dev_pages* d, void* stream, int* err) {
  if (!d || !err) return KVP_ERR_INVALID_ARG;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  int32_t h = 0;
  if (cudaMemcpyAsync(&h, d->top + 1, sizeof(int32_t), cudaMemcpyDeviceToHost, st) != cudaSuccess) return KVP_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return KVP_ERR_CUDA;
  if (h != 0) {
    if (cudaMemsetAsync(d->top + 1, 0, sizeof(int32_t), st) != cudaSuccess) return KVP_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return KVP_ERR_CUDA;
  }
  *err = h;
  return KVP_OK;
}
