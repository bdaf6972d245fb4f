// kvp_decode_step: one decode step of the whole path in one native call.
//
// The order of chapter 15's host loop ("A Paged KV Cache and Sliding-Window
// Attention", section "The model"), with the attention after a separate
// store: host bookkeeping appends one token per request (a fresh page on a
// page boundary, a copy of a shared tail page), the step's slots, table
// writes, copy pairs, lengths and rows go to the device in one copy (the
// mini-sglang code series, part 4: host-built lists, one scatter), then the
// page copies, the table writes, store_cache and attention of every layer,
// and last the window's trim writes (the pages a step attends are released
// only after it). Each layer is one store_cache_and_attention launch; the
// first carries the step's new-page table writes. A step that copies pages
// writes its table entries first, on their own: a copied tail page's entry
// is one that the attention reads.
#include <cstring>
#include <vector>

#include "common.cuh"

namespace {

int ceil_div(int a, int b) { return (a + b - 1) / b; }

}  // namespace

extern "C" int kvp_decode_step(kvp_host* h, const kvp_pool* pool, int32_t* table, int table_rows_total,
                               int table_cols, int table_mode, const int32_t* rids, int n, int window,
                               int sinks, int num_q_heads, float scale, const void* const* q, const void* const* k,
                               const void* const* v, void* const* out, void* const* layer_ready,
                               void* const* layer_done, int32_t* host_meta, int32_t* dev_meta, int meta_cap,
                               void* workspace, size_t workspace_bytes, void* stream, kvp_step_info* info) {
  if (!h || !pool || !table || !rids || n <= 0 || !q || !k || !v || !out || !host_meta || !dev_meta || !info)
    return KVP_ERR_INVALID_ARG;
  if (table_mode != KVP_BLOCK_TABLE && table_mode != KVP_RAW_LOCATIONS) return KVP_ERR_INVALID_ARG;
  if (sinks < 0 || (window > 0 && sinks >= window)) return KVP_ERR_INVALID_ARG;
  if (window <= 0) sinks = 0;
  const int P = pool->page_size;
  const int sp = ceil_div(sinks, P);  // sink pages, kept by the trim
  const cudaStream_t st = static_cast<cudaStream_t>(stream);

  // Lengths and dropped pages before the step, and the trim writes the step
  // will need, so that every capacity is checked before anything changes.
  std::vector<int> len0(n), drop0(n);
  for (int i = 0; i < n; ++i) {
    if (kvp_host_length(h, rids[i], &len0[i], &drop0[i]) != KVP_OK) return KVP_ERR_INVALID_ARG;
    for (int j = 0; j < i; ++j)
      if (rids[j] == rids[i]) return KVP_ERR_INVALID_ARG;  // one token per request per step
  }
  int trims = 0;
  if (window > 0) {
    for (int i = 0; i < n; ++i) {
      const int L = len0[i] + 1, keep = L + 1 - (window - sinks);
      const int pages = ceil_div(L, P);
      const int to = keep > 0 ? (keep / P < pages ? keep / P : pages) : 0;  // pages wholly below keep
      if (to > sp + drop0[i]) trims += to - sp - drop0[i];
    }
  }
  const long long need = 3LL * n + 3LL * n + 2LL * n + 3LL * trims;  // slots, tw, cow, lens, rows, trim
  if (need > meta_cap) return KVP_ERR_INVALID_ARG;

  int32_t* slots = host_meta;
  std::vector<int32_t> tw(3 * n), cow(2 * n);
  int ntw = 0, ncow = 0;
  int rc = kvp_host_append(h, rids, n, slots, tw.data(), tw.data() + n, tw.data() + 2 * n, n, &ntw, cow.data(),
                           cow.data() + n, &ncow);
  if (rc != KVP_OK) return rc;  // nothing changed (out of pages is all-or-nothing)
  int32_t* p = host_meta + n;
  const int o_tw = n;
  std::memcpy(p, tw.data(), sizeof(int32_t) * ntw);
  std::memcpy(p + ntw, tw.data() + n, sizeof(int32_t) * ntw);
  std::memcpy(p + 2 * ntw, tw.data() + 2 * n, sizeof(int32_t) * ntw);
  p += 3 * ntw;
  const int o_cow = o_tw + 3 * ntw;
  std::memcpy(p, cow.data(), sizeof(int32_t) * ncow);
  std::memcpy(p + ncow, cow.data() + n, sizeof(int32_t) * ncow);
  p += 2 * ncow;
  const int o_len = o_cow + 2 * ncow;
  for (int i = 0; i < n; ++i) p[i] = len0[i] + 1;
  p += n;
  const int o_rows = o_len + n;
  std::memcpy(p, rids, sizeof(int32_t) * n);
  p += n;
  const int o_trim = o_rows + n;
  int ntrim = 0;
  if (trims > 0) {
    std::vector<int32_t> tr(3 * trims);
    for (int i = 0; i < n; ++i) {
      const int keep = len0[i] + 2 - (window - sinks);
      int got = 0;
      rc = kvp_host_trim_sinks(h, rids[i], keep, sinks, tr.data() + ntrim, tr.data() + trims + ntrim,
                               tr.data() + 2 * trims + ntrim, trims - ntrim, &got);
      if (rc != KVP_OK) return rc;
      ntrim += got;
    }
    std::memcpy(p, tr.data(), sizeof(int32_t) * ntrim);
    std::memcpy(p + ntrim, tr.data() + trims, sizeof(int32_t) * ntrim);
    std::memcpy(p + 2 * ntrim, tr.data() + 2 * trims, sizeof(int32_t) * ntrim);
  }
  const int total = o_trim + 3 * ntrim;
  info->n_table_writes = ntw;
  info->n_copies = ncow;
  info->n_trim_writes = ntrim;
  info->meta_ints = total;

  if (cudaMemcpyAsync(dev_meta, host_meta, sizeof(int32_t) * total, cudaMemcpyHostToDevice, st) != cudaSuccess)
    return KVP_ERR_CUDA;
  const int expand = table_mode == KVP_RAW_LOCATIONS ? P : 1;
  if (ncow && (rc = copy_pages(pool, dev_meta + o_cow, dev_meta + o_cow + ncow, ncow, stream)) != KVP_OK) return rc;
  int fused_tw = ntw;
  if (ncow && ntw) {
    if ((rc = page_table_write(table, table_rows_total, table_cols, dev_meta + o_tw, dev_meta + o_tw + ntw,
                               dev_meta + o_tw + 2 * ntw, ntw, expand, pool->err, stream)) != KVP_OK)
      return rc;
    fused_tw = 0;
  }
  for (int l = 0; l < pool->num_layers; ++l) {
    if (layer_ready && layer_ready[l] &&
        cudaStreamWaitEvent(st, static_cast<cudaEvent_t>(layer_ready[l]), 0) != cudaSuccess)
      return KVP_ERR_CUDA;
    const int ltw = l == 0 ? fused_tw : 0;
    if ((rc = store_cache_and_attention(pool, l, q[l], k[l], v[l], dev_meta, n, num_q_heads, table, table_rows_total,
                                        table_cols, table_mode, dev_meta + o_rows, dev_meta + o_len,
                                        ltw ? dev_meta + o_tw : nullptr, ltw ? dev_meta + o_tw + ntw : nullptr,
                                        ltw ? dev_meta + o_tw + 2 * ntw : nullptr, ltw, window, sinks, scale, out[l],
                                        workspace, workspace_bytes, stream)) != KVP_OK)
      return rc;
    if (layer_done && layer_done[l] && cudaEventRecord(static_cast<cudaEvent_t>(layer_done[l]), st) != cudaSuccess)
      return KVP_ERR_CUDA;
  }
  if (ntrim && (rc = page_table_write(table, table_rows_total, table_cols, dev_meta + o_trim,
                                      dev_meta + o_trim + ntrim, dev_meta + o_trim + 2 * ntrim, ntrim, expand,
                                      pool->err, stream)) != KVP_OK)
    return rc;
  return KVP_OK;
}

// kvp_decode_step_device: the same step with the page bookkeeping on the
// device (kvp_dev_*): nothing is decided on the host and nothing but the
// caller's q/k/v crosses to the device. The append kernel pops the new
// pages, writes the table entries and hands the slots and the new lengths
// to the fused store + attention launches of every layer; the window's
// trim runs last, on the device too.
extern "C" int kvp_decode_step_device(kvp_dev_pages* d, const kvp_pool* pool, int32_t* table, int table_rows_total,
                                      int table_cols, int table_mode, const int32_t* rids, int n, int window,
                                      int sinks, int num_q_heads, float scale, const void* const* q,
                                      const void* const* k, const void* const* v, void* const* out,
                                      void* const* layer_ready, void* const* layer_done, int32_t* scratch,
                                      int may_share, void* workspace, size_t workspace_bytes, void* stream) {
  if (!d || !pool || !table || !rids || n <= 0 || !q || !k || !v || !out || !scratch) return KVP_ERR_INVALID_ARG;
  if (sinks < 0 || (window > 0 && sinks >= window)) return KVP_ERR_INVALID_ARG;
  if (window <= 0) sinks = 0;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  int32_t* out_loc = scratch;
  int32_t* lens = scratch + n;
  int32_t* cow_src = scratch + 2 * n;
  int32_t* cow_dst = scratch + 3 * n;
  int32_t* n_cow = scratch + 4 * n;
  int rc = kvp_dev_append(d, rids, nullptr, n, out_loc, n, cow_src, cow_dst, n_cow, lens, stream);
  if (rc != KVP_OK) return rc;
  if (may_share && (rc = copy_pages_device_count(pool, cow_src, cow_dst, n_cow, n, stream)) != KVP_OK) return rc;
  for (int l = 0; l < pool->num_layers; ++l) {
    if (layer_ready && layer_ready[l] &&
        cudaStreamWaitEvent(st, static_cast<cudaEvent_t>(layer_ready[l]), 0) != cudaSuccess)
      return KVP_ERR_CUDA;
    if ((rc = store_cache_and_attention(pool, l, q[l], k[l], v[l], out_loc, n, num_q_heads, table, table_rows_total,
                                        table_cols, table_mode, rids, lens, nullptr, nullptr, nullptr, 0, window,
                                        sinks, scale, out[l], workspace, workspace_bytes, stream)) != KVP_OK)
      return rc;
    if (layer_done && layer_done[l] && cudaEventRecord(static_cast<cudaEvent_t>(layer_done[l]), st) != cudaSuccess)
      return KVP_ERR_CUDA;
  }
  if (window > 0 && (rc = kvp_dev_trim(d, rids, nullptr, n, window, sinks, stream)) != KVP_OK) return rc;
  return KVP_OK;
}

// The page state's two copy streams and its events (device_pages.cu).
int kvp_dev_io_resources(kvp_dev_pages* d, int nevents, void** stream, void** stream2, void*** events);

// kvp_decode_step_device_io: kvp_decode_step_device with host buffers in and
// out. Each layer's q, k, v are copied from host memory into the caller's
// device staging on the state's first copy stream, while the page append
// runs on ``stream``; layer l's attention waits for layer l's copies only.
// Each layer's output goes back on the second copy stream as soon as that
// layer is done, while the next layers run. The call returns once the
// outputs are on the host. One native call per step.
// Events: [0] the step's start, [1 + l] layer l's inputs in, [1 + L + l]
// layer l done.
extern "C" int kvp_decode_step_device_io(kvp_dev_pages* d, const kvp_pool* pool, int32_t* table,
                                         int table_rows_total, int table_cols, int table_mode, const int32_t* rids,
                                         int n, int window, int sinks, int num_q_heads, float scale,
                                         const void* const* q_host, const void* const* k_host,
                                         const void* const* v_host, void* const* out_host, void* const* q_dev,
                                         void* const* k_dev, void* const* v_dev, void* const* out_dev,
                                         int32_t* scratch, int may_share, void* workspace, size_t workspace_bytes,
                                         void* stream) {
  if (!d || !pool || !q_host || !k_host || !v_host || !out_host || !q_dev || !k_dev || !v_dev || !out_dev ||
      n <= 0 || num_q_heads <= 0)
    return KVP_ERR_INVALID_ARG;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int layers = pool->num_layers;
  void* io = nullptr;
  void* io2 = nullptr;
  void** ev = nullptr;
  int rc = kvp_dev_io_resources(d, 2 * layers + 1, &io, &io2, &ev);
  if (rc != KVP_OK) return rc;
  const cudaStream_t cs = static_cast<cudaStream_t>(io), ds = static_cast<cudaStream_t>(io2);
  const size_t qbytes = (size_t)n * num_q_heads * pool->head_dim * pool->elem;
  const size_t kvbytes = (size_t)n * pool->row_bytes;
  // the copies start after the work already on ``stream`` (the staging may still be read there)
  if (cudaEventRecord(static_cast<cudaEvent_t>(ev[0]), st) != cudaSuccess ||
      cudaStreamWaitEvent(cs, static_cast<cudaEvent_t>(ev[0]), 0) != cudaSuccess)
    return KVP_ERR_CUDA;
  for (int l = 0; l < layers; ++l) {
    if (cudaMemcpyAsync(q_dev[l], q_host[l], qbytes, cudaMemcpyHostToDevice, cs) != cudaSuccess ||
        cudaMemcpyAsync(k_dev[l], k_host[l], kvbytes, cudaMemcpyHostToDevice, cs) != cudaSuccess ||
        cudaMemcpyAsync(v_dev[l], v_host[l], kvbytes, cudaMemcpyHostToDevice, cs) != cudaSuccess ||
        cudaEventRecord(static_cast<cudaEvent_t>(ev[1 + l]), cs) != cudaSuccess)
      return KVP_ERR_CUDA;
  }
  rc = kvp_decode_step_device(d, pool, table, table_rows_total, table_cols, table_mode, rids, n, window, sinks,
                              num_q_heads, scale, q_dev, k_dev, v_dev, out_dev, ev + 1, ev + 1 + layers, scratch,
                              may_share, workspace, workspace_bytes, stream);
  if (rc != KVP_OK) {
    cudaStreamSynchronize(cs);  // the host buffers stay in use until the copies are done
    return rc;
  }
  for (int l = 0; l < layers; ++l)
    if (cudaStreamWaitEvent(ds, static_cast<cudaEvent_t>(ev[1 + layers + l]), 0) != cudaSuccess ||
        cudaMemcpyAsync(out_host[l], out_dev[l], qbytes, cudaMemcpyDeviceToHost, ds) != cudaSuccess)
      return KVP_ERR_CUDA;
  return cudaStreamSynchronize(ds) == cudaSuccess && cudaStreamSynchronize(st) == cudaSuccess ? KVP_OK
                                                                                               : KVP_ERR_CUDA;
}

// kvp_dev_append for ``count`` rows of every request (device_pages.cu).
int kvp_dev_append_uniform(kvp_dev_pages* d, const int32_t* rids, int count, int n, int32_t* out_loc, int max_tokens,
                           int32_t* cow_src, int32_t* cow_dst, int32_t* n_cow, int32_t* lens_out, void* stream);

// kvp_verify_step_device_io: one speculative-decoding verify step with the
// page bookkeeping on the device and host buffers in and out ("Week 3 Day 3:
// Paged KV Cache" of tiny-llm: rewind(n) drops the rejected drafts). The M
// drafts of every request are appended on the device (new pages popped, a
// shared tail page copied first), stored and verified at once, layer by
// layer; then each request's rejected drafts are rewound on the device, and
// with a window the pages it no longer reaches are released. The inputs
// travel on the page state's first copy stream while the append runs; layer
// l's store and verify wait for layer l's copies only, and its output goes
// back on the second copy stream as soon as it is done. One native call per
// step.
extern "C" int kvp_verify_step_device_io(kvp_dev_pages* d, const kvp_pool* pool, int32_t* table,
                                         int table_rows_total, int table_cols, int table_mode, const int32_t* rids,
                                         int n, int num_q_tokens, int window, int sinks, int num_q_heads, float scale,
                                         const void* const* q_host, const void* const* k_host,
                                         const void* const* v_host, const int32_t* n_back_host,
                                         void* const* out_host, void* const* q_dev, void* const* k_dev,
                                         void* const* v_dev, void* const* out_dev, int32_t* scratch, int may_share,
                                         void* workspace, size_t workspace_bytes, void* stream) {
  const int M = num_q_tokens;
  if (!d || !pool || !table || !rids || n <= 0 || M < 1 || num_q_heads <= 0 || !q_host || !k_host || !v_host ||
      !n_back_host || !out_host || !q_dev || !k_dev || !v_dev || !out_dev || !scratch)
    return KVP_ERR_INVALID_ARG;
  if (sinks < 0 || (window > 0 && sinks >= window)) return KVP_ERR_INVALID_ARG;
  if (window <= 0) sinks = 0;
  for (int i = 0; i < n; ++i)
    if (n_back_host[i] < 0 || n_back_host[i] > M) return KVP_ERR_INVALID_ARG;  // only this step's drafts go back
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int layers = pool->num_layers;
  void* io = nullptr;
  void* io2 = nullptr;
  void** ev = nullptr;
  int rc = kvp_dev_io_resources(d, 2 * layers + 1, &io, &io2, &ev);
  if (rc != KVP_OK) return rc;
  const cudaStream_t cs = static_cast<cudaStream_t>(io), ds = static_cast<cudaStream_t>(io2);
  int32_t* out_loc = scratch;             // n * M slots, request-major
  int32_t* lens = scratch + n * M;        // n
  int32_t* cow_src = lens + n;            // n
  int32_t* cow_dst = cow_src + n;         // n
  int32_t* n_cow = cow_dst + n;           // 1
  int32_t* n_back = n_cow + 1;            // n
  const size_t qbytes = (size_t)n * M * num_q_heads * pool->head_dim * pool->elem;
  const size_t kvbytes = (size_t)n * M * pool->row_bytes;
  if (cudaEventRecord(static_cast<cudaEvent_t>(ev[0]), st) != cudaSuccess ||
      cudaStreamWaitEvent(cs, static_cast<cudaEvent_t>(ev[0]), 0) != cudaSuccess)
    return KVP_ERR_CUDA;
  for (int l = 0; l < layers; ++l) {
    if (cudaMemcpyAsync(q_dev[l], q_host[l], qbytes, cudaMemcpyHostToDevice, cs) != cudaSuccess ||
        cudaMemcpyAsync(k_dev[l], k_host[l], kvbytes, cudaMemcpyHostToDevice, cs) != cudaSuccess ||
        cudaMemcpyAsync(v_dev[l], v_host[l], kvbytes, cudaMemcpyHostToDevice, cs) != cudaSuccess ||
        (l == 0 && cudaMemcpyAsync(n_back, n_back_host, sizeof(int32_t) * n, cudaMemcpyHostToDevice, cs) !=
                       cudaSuccess) ||
        cudaEventRecord(static_cast<cudaEvent_t>(ev[1 + l]), cs) != cudaSuccess)
      return KVP_ERR_CUDA;
  }
  rc = kvp_dev_append_uniform(d, rids, M, n, out_loc, n * M, cow_src, cow_dst, n_cow, lens, stream);
  if (rc == KVP_OK && may_share) rc = copy_pages_device_count(pool, cow_src, cow_dst, n_cow, n, stream);
  for (int l = 0; rc == KVP_OK && l < layers; ++l) {
    if (cudaStreamWaitEvent(st, static_cast<cudaEvent_t>(ev[1 + l]), 0) != cudaSuccess) {
      rc = KVP_ERR_CUDA;
      break;
    }
    rc = store_cache(pool, l, k_dev[l], v_dev[l], out_loc, n * M, stream);
    if (rc == KVP_OK)
      rc = paged_verify_attention(pool, l, q_dev[l], n, M, num_q_heads, table, table_rows_total, table_cols,
                                  table_mode, rids, lens, window, sinks, scale, out_dev[l], workspace,
                                  workspace_bytes, stream);
    // layer l's output goes back while the next layers run
    if (rc == KVP_OK &&
        (cudaEventRecord(static_cast<cudaEvent_t>(ev[1 + layers + l]), st) != cudaSuccess ||
         cudaStreamWaitEvent(ds, static_cast<cudaEvent_t>(ev[1 + layers + l]), 0) != cudaSuccess ||
         cudaMemcpyAsync(out_host[l], out_dev[l], qbytes, cudaMemcpyDeviceToHost, ds) != cudaSuccess))
      rc = KVP_ERR_CUDA;
  }
  // the rejected drafts go back (n_back was copied with layer 0's inputs), then the window's releases
  if (rc == KVP_OK) rc = kvp_dev_rewind(d, rids, n_back, n, stream);
  if (rc == KVP_OK && window > 0) rc = kvp_dev_trim(d, rids, nullptr, n, window, sinks, stream);
  if (rc != KVP_OK) {
    cudaStreamSynchronize(cs);  // the host buffers stay in use until the copies are done
    cudaStreamSynchronize(ds);
    return rc;
  }
  return cudaStreamSynchronize(ds) == cudaSuccess && cudaStreamSynchronize(st) == cudaSuccess ? KVP_OK
                                                                                               : KVP_ERR_CUDA;
}
