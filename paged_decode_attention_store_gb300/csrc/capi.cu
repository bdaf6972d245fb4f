// Pool descriptor and device error word of libpagedkv.
#include <new>

#include "common.cuh"

extern "C" int kv_pool_create(int num_pages, int page_size, int kv_heads, int head_dim, int dtype, int num_layers,
                              void* kv_buffer, int32_t* error_word, kvp_pool** out) {
  if (!out || !kv_buffer || !error_word) return KVP_ERR_INVALID_ARG;
  if (num_pages <= 0 || page_size <= 0 || kv_heads <= 0 || head_dim <= 0 || num_layers <= 0) return KVP_ERR_INVALID_ARG;
  if (dtype != KVP_F32 && dtype != KVP_BF16) return KVP_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(kv_buffer) & 15) return KVP_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(error_word) & 3) return KVP_ERR_INVALID_ARG;
  const long long slots = (long long)num_pages * page_size;
  if (slots > 0x7fffffffLL) return KVP_ERR_INVALID_ARG;
  const int elem = dtype == KVP_F32 ? 4 : 2;
  const size_t row_bytes = (size_t)kv_heads * head_dim * elem;
  if (row_bytes % 16) return KVP_ERR_INVALID_ARG;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KVP_ERR_CUDA;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
    return KVP_ERR_CUDA;
  kvp_pool* p = new (std::nothrow) kvp_pool;
  if (!p) return KVP_ERR_INVALID_ARG;
  p->num_pages = num_pages;
  p->page_size = page_size;
  p->kv_heads = kv_heads;
  p->head_dim = head_dim;
  p->dtype = dtype;
  p->num_layers = num_layers;
  p->elem = elem;
  p->num_slots = (int)slots;
  p->row_bytes = row_bytes;
  p->layer_bytes = (size_t)slots * row_bytes;
  p->kv_bytes = p->layer_bytes * num_layers;
  p->buf = static_cast<char*>(kv_buffer);
  p->err = error_word;
  p->num_sms = sms;
  p->device = dev;
  p->ev_before = nullptr;
  p->ev_after = nullptr;
  p->tmap_hg = 0;
  p->tmap1_state = 0;
  *out = p;
  return KVP_OK;
}

extern "C" int kv_pool_destroy(kvp_pool* pool) {
  delete pool;
  return KVP_OK;
}

extern "C" int kvp_sync_error(const kvp_pool* pool, void* stream, int* err) {
  if (!pool || !err) return KVP_ERR_INVALID_ARG;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  int32_t h = 0;
  if (cudaMemcpyAsync(&h, pool->err, sizeof(int32_t), cudaMemcpyDeviceToHost, st) != cudaSuccess) return KVP_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return KVP_ERR_CUDA;
  if (h != 0) {
    if (cudaMemsetAsync(pool->err, 0, sizeof(int32_t), st) != cudaSuccess) return KVP_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return KVP_ERR_CUDA;
  }
  *err = h;
  return KVP_OK;
}

extern "C" int kvp_pool_set_timing_events(kvp_pool* pool, void* before, void* after) {
  if (!pool || (before == nullptr) != (after == nullptr)) return KVP_ERR_INVALID_ARG;
  pool->ev_before = before;
  pool->ev_after = after;
  return KVP_OK;
}
