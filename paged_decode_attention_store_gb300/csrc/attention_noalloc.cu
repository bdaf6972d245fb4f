// paged_decode_attention_noalloc: decode attention without any allocation.
//
// Some callers cannot allocate device memory at the point where they run
// attention: code that runs inside another framework's memory pool or under
// a strict memory budget that forbids new reservations, callers that must
// not call into the allocator from their own thread or callback, and
// embedded or plug-in hosts that receive only their input and output
// buffers. paged_decode_attention needs a caller-provided workspace for its
// split-K partials; this entry point takes that scratch from a fixed array in
// the library's own device memory instead, so the caller passes only inputs
// and outputs.
//
// The array is a file-scope __device__ variable of kNoAllocScratchBytes
// (12 MiB). Every GPU that loads this part of the library holds it until the
// process exits. Host code cannot use the array's name as a device address:
// the first call on a device, with that device current, looks the address up
// with cudaGetSymbolAddress and keeps it, together with the CUDA context it
// belongs to, for later calls. A call that finds a different context current
// on that device (the primary context was reset and created again) looks the
// address up again instead of using a stale one.
#include <mutex>

#include "attention.cuh"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(12) << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_setup_mu;
void* g_scratch_ptr[kMaxDevices];  // device address of g_noalloc_scratch, per device
void* g_scratch_ctx[kMaxDevices];  // the context that address was looked up in

typedef CUresult (*ctx_get_current_fn)(CUcontext*);

// The current driver context (no allocation; the driver entry point is
// fetched once). Returns false when it cannot be read.
bool current_context(void** ctx) {
  static ctx_get_current_fn get = nullptr;
  static bool looked = false;
  if (!looked) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get = reinterpret_cast<ctx_get_current_fn>(fn);
    looked = true;
  }
  CUcontext c = nullptr;
  if (!get || get(&c) != CUDA_SUCCESS || !c) return false;
  *ctx = c;
  return true;
}

}  // namespace

extern "C" int paged_decode_attention_noalloc(const kvp_pool* pool, int layer, const void* q, int batch,
                                              int num_q_heads, const int32_t* table, int table_rows_total,
                                              int table_cols, int table_mode, const int32_t* table_rows,
                                              const int32_t* context_lens, int window, int sinks, float scale,
                                              void* out, void* stream) {
  if (!pool) return KVP_ERR_INVALID_ARG;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return KVP_ERR_CUDA;
  if (dev != pool->device || dev < 0 || dev >= kMaxDevices) return KVP_ERR_INVALID_ARG;
  size_t need = 0;
  const int rc = paged_decode_attention_workspace_size(pool, batch, num_q_heads, &need);
  if (rc != KVP_OK) return rc;
  if (need > kNoAllocScratchBytes) return KVP_ERR_INVALID_ARG;  // the shape needs more scratch than the fixed array
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_setup_mu);
    // A context that is not current yet (no runtime call has needed it) is
    // created by the symbol lookup, which then runs before the query.
    void* ctx = nullptr;
    const bool have_ctx = current_context(&ctx);
    if (!have_ctx || !g_scratch_ptr[dev] || g_scratch_ctx[dev] != ctx) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return KVP_ERR_CUDA;
      if (!current_context(&ctx)) return KVP_ERR_CUDA;
      g_scratch_ptr[dev] = p;
      g_scratch_ctx[dev] = ctx;
    }
    scratch = g_scratch_ptr[dev];
  }
  // Nothing in the scratch has to start at zero: every call writes the merge
  // records and partials it reads.
  return paged_decode_attention(pool, layer, q, batch, num_q_heads, table, table_rows_total, table_cols, table_mode,
                                table_rows, context_lens, window, sinks, scale, out, scratch, kNoAllocScratchBytes,
                                stream);
}
