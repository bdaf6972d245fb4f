// Device writes of the paged KV cache: store_cache (new K/V rows to their
// slots), page_table_write (new / released / copied-on-write table entries,
// with the page->token expansion of raw-location tables) and copy_pages
// (copy-on-write of whole pages). All three are bandwidth- or latency-bound
// byte moves: 16-byte vector accesses, consecutive threads on consecutive
// bytes of one row, a grid sized in multiples of the SM count.
#include "common.cuh"

namespace kvp {

// One thread moves one 16-byte chunk. Work unit u covers (row i, K or V,
// chunk c): u = (i * 2 + kv) * chunks + c, so a warp streams contiguous
// bytes of one row.
__global__ void store_cache_kernel(char* __restrict__ kbase, size_t kv_bytes, const uint4* __restrict__ k,
                                   const uint4* __restrict__ v, const int32_t* __restrict__ out_loc, int n,
                                   int chunks, int num_slots, int32_t* err) {
  const long long total = (long long)n * 2 * chunks;
  for (long long u = blockIdx.x * (long long)blockDim.x + threadIdx.x; u < total;
       u += (long long)gridDim.x * blockDim.x) {
    const int c = (int)(u % chunks);
    const long long ik = u / chunks;
    const int kv = (int)(ik & 1);
    const int i = (int)(ik >> 1);
    const int slot = __ldg(out_loc + i);
    if ((unsigned)slot >= (unsigned)num_slots) {
      if (kv == 0 && c == 0) set_error(err, KVP_ERR_BAD_INDEX);
      continue;
    }
    const uint4* src = kv ? v : k;
    uint4 val = __ldg(src + (size_t)i * chunks + c);
    uint4* dst = reinterpret_cast<uint4*>(kbase + kv * kv_bytes) + (size_t)slot * chunks + c;
    *dst = val;
  }
}

// Pair p, layer l, K or V: page dst[p] <- page src[p]; one page of one layer
// is page_size contiguous rows.
// With n_dev, the number of pairs is read on the device (at most n).
__global__ void copy_pages_kernel(char* __restrict__ buf, size_t layer_bytes, int num_layers,
                                  const int32_t* __restrict__ src, const int32_t* __restrict__ dst, int n,
                                  const int32_t* __restrict__ n_dev, int page_chunks, int num_pages, int32_t* err) {
  if (n_dev) n = min(n, max(0, __ldg(n_dev)));
  const long long total = (long long)n * num_layers * 2 * page_chunks;
  for (long long u = blockIdx.x * (long long)blockDim.x + threadIdx.x; u < total;
       u += (long long)gridDim.x * blockDim.x) {
    const int c = (int)(u % page_chunks);
    long long rest = u / page_chunks;
    const int kvl = (int)(rest % (2LL * num_layers));  // kv * num_layers + layer
    const int p = (int)(rest / (2LL * num_layers));
    const int s = __ldg(src + p), d = __ldg(dst + p);
    if ((unsigned)s >= (unsigned)num_pages || (unsigned)d >= (unsigned)num_pages) {
      if (c == 0 && kvl == 0) set_error(err, KVP_ERR_BAD_INDEX);
      continue;
    }
    const uint4* from = reinterpret_cast<const uint4*>(buf + kvl * layer_bytes) + (size_t)s * page_chunks + c;
    uint4* to = reinterpret_cast<uint4*>(buf + kvl * layer_bytes) + (size_t)d * page_chunks + c;
    *to = *from;
  }
}

__global__ void page_table_write_kernel(int32_t* __restrict__ table, int rows_total, int cols,
                                        const int32_t* __restrict__ rows, const int32_t* __restrict__ colv,
                                        const int32_t* __restrict__ vals, int n, int expand, int32_t* err) {
  const long long total = (long long)n * expand;
  for (long long u = blockIdx.x * (long long)blockDim.x + threadIdx.x; u < total;
       u += (long long)gridDim.x * blockDim.x) {
    const int i = (int)(u / expand);
    const int j = (int)(u % expand);
    const int r = __ldg(rows + i);
    const long long c = (long long)__ldg(colv + i) * expand + j;
    const int v = __ldg(vals + i);
    if ((unsigned)r >= (unsigned)rows_total || c < 0 || c >= cols) {
      set_error(err, KVP_ERR_BAD_INDEX);
      continue;
    }
    table[(size_t)r * cols + c] = v < 0 ? -1 : v * expand + j;
  }
}

static int grid_for(long long work, int threads, int num_sms) {
  long long blocks = (work + threads - 1) / threads;
  long long cap = (long long)num_sms * 8;  // 8 resident 256-thread blocks per SM
  if (blocks > cap) blocks = cap;
  return (int)(blocks < 1 ? 1 : blocks);
}

static int sm_count_current() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return sms;
}

}  // namespace kvp

extern "C" int store_cache(const kvp_pool* pool, int layer, const void* k, const void* v, const int32_t* out_loc,
                           int n, void* stream) {
  if (!pool || n < 0 || layer < 0 || layer >= pool->num_layers) return KVP_ERR_INVALID_ARG;
  if (n == 0) return KVP_OK;
  if (!k || !v || !out_loc) return KVP_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v)) & 15) return KVP_ERR_INVALID_ARG;
  const int chunks = (int)(pool->row_bytes / 16);
  const long long work = (long long)n * 2 * chunks;
  const int threads = 256;
  kvp::store_cache_kernel<<<kvp::grid_for(work, threads, pool->num_sms), threads, 0, (cudaStream_t)stream>>>(
      pool->buf + (size_t)layer * pool->layer_bytes, pool->kv_bytes, static_cast<const uint4*>(k),
      static_cast<const uint4*>(v), out_loc, n, chunks, pool->num_slots, pool->err);
  return cudaGetLastError() == cudaSuccess ? KVP_OK : KVP_ERR_CUDA;
}

extern "C" int copy_pages(const kvp_pool* pool, const int32_t* src, const int32_t* dst, int n, void* stream) {
  if (!pool || n < 0) return KVP_ERR_INVALID_ARG;
  if (n == 0) return KVP_OK;
  if (!src || !dst) return KVP_ERR_INVALID_ARG;
  const int page_chunks = (int)(pool->row_bytes * pool->page_size / 16);
  const long long work = (long long)n * pool->num_layers * 2 * page_chunks;
  const int threads = 256;
  kvp::copy_pages_kernel<<<kvp::grid_for(work, threads, pool->num_sms), threads, 0, (cudaStream_t)stream>>>(
      pool->buf, pool->layer_bytes, pool->num_layers, src, dst, n, nullptr, page_chunks, pool->num_pages, pool->err);
  return cudaGetLastError() == cudaSuccess ? KVP_OK : KVP_ERR_CUDA;
}

extern "C" int copy_pages_device_count(const kvp_pool* pool, const int32_t* src, const int32_t* dst,
                                       const int32_t* n_dev, int max_n, void* stream) {
  if (!pool || max_n < 0 || (max_n > 0 && (!src || !dst || !n_dev))) return KVP_ERR_INVALID_ARG;
  if (max_n == 0) return KVP_OK;
  const int page_chunks = (int)(pool->row_bytes * pool->page_size / 16);
  const long long work = (long long)max_n * pool->num_layers * 2 * page_chunks;
  const int threads = 256;
  kvp::copy_pages_kernel<<<kvp::grid_for(work, threads, pool->num_sms), threads, 0, (cudaStream_t)stream>>>(
      pool->buf, pool->layer_bytes, pool->num_layers, src, dst, max_n, n_dev, page_chunks, pool->num_pages,
      pool->err);
  return cudaGetLastError() == cudaSuccess ? KVP_OK : KVP_ERR_CUDA;
}

extern "C" int page_table_write(int32_t* table, int table_rows_total, int table_cols, const int32_t* rows,
                                const int32_t* cols, const int32_t* vals, int n, int expand, int32_t* error_word,
                                void* stream) {
  if (!table || table_rows_total <= 0 || table_cols <= 0 || n < 0 || expand <= 0) return KVP_ERR_INVALID_ARG;
  if (n == 0) return KVP_OK;
  if (!rows || !cols || !vals) return KVP_ERR_INVALID_ARG;
  const int sms = kvp::sm_count_current();
  if (sms <= 0) return KVP_ERR_CUDA;
  const long long work = (long long)n * expand;
  const int threads = 256;
  kvp::page_table_write_kernel<<<kvp::grid_for(work, threads, sms), threads, 0, (cudaStream_t)stream>>>(
      table, table_rows_total, table_cols, rows, cols, vals, n, expand, error_word);
  return cudaGetLastError() == cudaSuccess ? KVP_OK : KVP_ERR_CUDA;
}
