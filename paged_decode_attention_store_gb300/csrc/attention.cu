// Decode attention: the general CUDA-core kernel, the index dump, and the C
// ABI that picks between it and the tensor-core kernel (attention_tc.cu).
#include <cstring>

#include "attention.cuh"

namespace kvp {

namespace {

// ---------------------------------------------------------------------------
// General kernel (any dtype, head_dim <= 256, any group size): one warp per
// (request, query head). Lane j scores token t0+j of a 32-token chunk against
// q held in shared memory; the warp then streams the chunk's V rows with
// lanes on the head dimension (coalesced) and a running (max, sum) rescale.
// Used for fp32 caches and shapes the tensor-core kernel does not take.
// ---------------------------------------------------------------------------
template <typename T>
__device__ __forceinline__ float to_f(T x);
template <>
__device__ __forceinline__ float to_f<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T>
__device__ __forceinline__ T from_f(float x);
template <>
__device__ __forceinline__ float from_f<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

struct GenArgs {
  TableRef T;
  const char* kv_layer;
  size_t kv_bytes;
  const void* q;
  void* out;
  const int32_t* context_lens;
  const int32_t* table_rows;
  int B, Hq, Hkv, D, window, sinks;
  int M;  // query tokens per request (query j at position L - M + j)
  const int32_t* q_lens;  // per request, <= M (NULL: M); rows j >= q_lens[b] are not written
  float scale_log2;
  int32_t* err;
};

constexpr int kGenWarps = 4;
constexpr int kGenMaxD = 256;

template <typename T>
__global__ void __launch_bounds__(32 * kGenWarps) generic_decode_kernel(const GenArgs a) {
  __shared__ float qs[kGenWarps][kGenMaxD];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long wid = (long long)blockIdx.x * kGenWarps + warp;
  if (wid >= (long long)a.B * a.M * a.Hq) return;
  const int bj = (int)(wid / a.Hq), h = (int)(wid % a.Hq);  // (request, query token), query head
  const int b = bj / a.M, j = bj % a.M;
  const int G = a.Hq / a.Hkv, kvh = h / G;
  const int D = a.D;
  T* out = static_cast<T*>(a.out) + ((size_t)bj * a.Hq + h) * D;
  const T* q = static_cast<const T*>(a.q) + ((size_t)bj * a.Hq + h) * D;
  const int Lr = a.context_lens[b];
  const int row = a.table_rows ? a.table_rows[b] : b;
  const int Mb = a.q_lens ? a.q_lens[b] : a.M;
  if (Mb < 1 || Mb > a.M || Lr < Mb || Lr > table_capacity(a.T) || row < 0 || row >= a.T.rows_total) {
    if (h == 0 && j == 0 && lane == 0) set_error(a.err, KVP_ERR_BAD_INDEX);
    for (int d = lane; d < D; d += 32) out[d] = from_f<T>(0.f);
    return;
  }
  if (j >= Mb) return;
  const int L = Lr - Mb + j + 1;  // the query token's own context (causal)
  for (int d = lane; d < D; d += 32) qs[warp][d] = to_f<T>(q[d]);
  __syncwarp();
  const Span sp = attend_span(L, a.window, a.sinks);
  const int n = sp.se + L - sp.lo;  // attended rows: [0, se) and [lo, L)
  const size_t row_elems = (size_t)a.Hkv * D;
  const T* K = reinterpret_cast<const T*>(a.kv_layer);
  const T* Vp = reinterpret_cast<const T*>(a.kv_layer + a.kv_bytes);
  constexpr int kPerLane = kGenMaxD / 32;
  float acc[kPerLane];
#pragma unroll
  for (int i = 0; i < kPerLane; ++i) acc[i] = 0.f;
  float m = -INFINITY, l = 0.f;
  for (int o0 = 0; o0 < n; o0 += 32) {
    const int o = o0 + lane;
    int slot = -1;
    float s = -INFINITY;
    if (o < n) {
      slot = resolve_slot(a.T, row, span_pos(sp, o), a.err);
      if (slot >= 0) {
        const T* kr = K + (size_t)slot * row_elems + (size_t)kvh * D;
        float dot = 0.f;
        for (int d = 0; d < D; ++d) dot = fmaf(qs[warp][d], to_f<T>(kr[d]), dot);
        s = dot * a.scale_log2;
      }
    }
    float mx = s;
#pragma unroll
    for (int sh = 16; sh > 0; sh >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, sh));
    const float mn = fmaxf(m, mx);
    if (mn == -INFINITY) continue;
    const float alpha = exp2f(m - mn);
    const float p = exp2f(s - mn);
    float ps = p;
#pragma unroll
    for (int sh = 16; sh > 0; sh >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, sh);
    l = l * alpha + ps;
    m = mn;
#pragma unroll
    for (int i = 0; i < kPerLane; ++i) acc[i] *= alpha;
    const int nt = min(32, n - o0);
    for (int jj = 0; jj < nt; ++jj) {
      const float pj = __shfl_sync(0xffffffffu, p, jj);
      const int sj = __shfl_sync(0xffffffffu, slot, jj);
      if (sj < 0) continue;
      const T* vr = Vp + (size_t)sj * row_elems + (size_t)kvh * D;
#pragma unroll
      for (int i = 0; i < kPerLane; ++i) {
        const int d = lane + 32 * i;
        if (d < D) acc[i] = fmaf(pj, to_f<T>(vr[d]), acc[i]);
      }
    }
  }
  const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
  for (int i = 0; i < kPerLane; ++i) {
    const int d = lane + 32 * i;
    if (d < D) out[d] = from_f<T>(acc[i] * inv);
  }
}

__global__ void gather_indices_kernel(TableRef T, const int32_t* context_lens, const int32_t* table_rows, int window,
                                      int sinks, int32_t* out, int max_tokens, int32_t* err) {
  const int b = blockIdx.x;
  const int L = context_lens[b];
  const int row = table_rows ? table_rows[b] : b;
  const bool valid = L >= 1 && L <= table_capacity(T) && row >= 0 && row < T.rows_total;
  const Span sp = attend_span(valid ? L : 0, window, sinks);
  const int n = valid ? sp.se + L - sp.lo : 0;
  if ((!valid || n > max_tokens) && threadIdx.x == 0) set_error(err, KVP_ERR_BAD_INDEX);
  for (int i = threadIdx.x; i < max_tokens; i += blockDim.x) {
    int s = -1;
    if (i < n) s = resolve_slot(T, row, span_pos(sp, i), err);
    out[(size_t)b * max_tokens + i] = s;
  }
}

// The tensor-core kernel's shape for Hq query heads and M query tokens per
// request: the M * G (token, head) columns of a KV head go to T consumer
// warps of NT 8-column tiles, HG KV heads per CTA, HG * T <= 8 warps.
struct TcShape {
  int HG, NT, T, S;
};

bool tc_eligible(const kvp_pool* pool, int Hq, int B, int M, TcShape* out) {
  if (pool->dtype != KVP_BF16 || pool->head_dim != 128) return false;
  const int Hkv = pool->kv_heads;
  if (Hq % Hkv || M < 1 || M > 32) return false;
  // One 8-column tile per warp keeps a consumer warp's stage work (and its
  // registers) at the decode kernel's; two tiles only when eight warps of
  // one tile cannot hold the columns.
  const int C = (Hq / Hkv) * M;
  int NT = 1, T = (C + 7) / 8;
  if (T > 8) {
    NT = 2;
    T = (C + 15) / 16;
  }
  if (T > 8) return false;
  for (int HG = 8 / T; HG >= 1; --HG) {
    if (Hkv % HG) continue;
    const int S = tc_num_stages(HG, C);
    if (tc_num_qbuf(HG, C, S) == 0) continue;
    if (B > tc_max_batch(HG, S)) return false;
    out->HG = HG;
    out->NT = NT;
    out->T = T;
    out->S = S;
    return true;
  }
  return false;
}

size_t workspace_bytes_for(const kvp_pool* pool, int batch, int M, int num_q_heads) {
  TcShape sh;
  if (!tc_eligible(pool, num_q_heads, batch, M, &sh)) return 256;  // the general kernel needs no scratch
  const int QH = sh.HG * (num_q_heads / pool->kv_heads);
  return ws_layout(pool->num_sms, M * QH, 128).total;
}

TableRef make_table(const kvp_pool* pool, const int32_t* table, int rows_total, int cols, int mode) {
  TableRef T;
  T.table = table;
  T.rows_total = rows_total;
  T.cols = cols;
  T.raw = mode == KVP_RAW_LOCATIONS ? 1 : 0;
  T.page_size = pool->page_size;
  T.num_pages = pool->num_pages;
  T.num_slots = pool->num_slots;
  return T;
}

}  // namespace

}  // namespace kvp

using namespace kvp;

extern "C" int paged_decode_attention_workspace_size(const kvp_pool* pool, int batch, int num_q_heads,
                                                     size_t* bytes) {
  if (!pool || !bytes || batch <= 0 || num_q_heads <= 0) return KVP_ERR_INVALID_ARG;
  *bytes = workspace_bytes_for(pool, batch, 1, num_q_heads);
  return KVP_OK;
}

extern "C" int paged_verify_attention_workspace_size(const kvp_pool* pool, int batch, int num_q_tokens,
                                                     int num_q_heads, size_t* bytes) {
  if (!pool || !bytes || batch <= 0 || num_q_heads <= 0 || num_q_tokens < 1) return KVP_ERR_INVALID_ARG;
  *bytes = workspace_bytes_for(pool, batch, num_q_tokens, num_q_heads);
  return KVP_OK;
}

namespace {

// The extra inputs of a fused step (store_cache_and_attention).
struct FuseIn {
  const void* k;
  const void* v;
  const int32_t* out_loc;
  int32_t* table;
  const int32_t* tw_rows;
  const int32_t* tw_cols;
  const int32_t* tw_vals;
  int n_tw;
};

int attention_impl(const kvp_pool* pool, int layer, const void* q, int batch, int M, int num_q_heads,
                   const int32_t* table, int table_rows_total, int table_cols, int table_mode,
                   const int32_t* table_rows, const int32_t* context_lens, int window, int sinks, float scale,
                   void* out, void* workspace, size_t workspace_bytes, void* stream, const FuseIn* fz) {
  if (!pool || !q || !table || !context_lens || !out) return KVP_ERR_INVALID_ARG;
  if (M < 1 || M > 32 || (fz && M != 1)) return KVP_ERR_INVALID_ARG;
  if (layer < 0 || layer >= pool->num_layers || batch <= 0 || num_q_heads <= 0) return KVP_ERR_INVALID_ARG;
  if (num_q_heads % pool->kv_heads) return KVP_ERR_INVALID_ARG;
  if (table_rows_total <= 0 || table_cols <= 0) return KVP_ERR_INVALID_ARG;
  if (table_mode != KVP_BLOCK_TABLE && table_mode != KVP_RAW_LOCATIONS) return KVP_ERR_INVALID_ARG;
  if (!(scale == scale)) return KVP_ERR_INVALID_ARG;
  if (sinks < 0 || (window > 0 && sinks >= window)) return KVP_ERR_INVALID_ARG;
  if (window <= 0) sinks = 0;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  const TableRef T = make_table(pool, table, table_rows_total, table_cols, table_mode);
  const char* kv_layer = pool->buf + (size_t)layer * pool->layer_bytes;
  const float scale_log2 = scale * 1.4426950408889634f;

  TcShape sh;
  kvp_pool* mp = const_cast<kvp_pool*>(pool);
  const int expand = table_mode == KVP_RAW_LOCATIONS ? pool->page_size : 1;
  if (fz && !tc_eligible(pool, num_q_heads, batch, M, &sh)) {
    // no fused kernel for this pool: the same three operations in sequence
    int rc;
    if (fz->n_tw && (rc = page_table_write(fz->table, table_rows_total, table_cols, fz->tw_rows, fz->tw_cols,
                                           fz->tw_vals, fz->n_tw, expand, pool->err, stream)) != KVP_OK)
      return rc;
    if ((rc = store_cache(pool, layer, fz->k, fz->v, fz->out_loc, batch, stream)) != KVP_OK) return rc;
    fz = nullptr;
  }
  if (tc_eligible(pool, num_q_heads, batch, M, &sh)) {
    if (reinterpret_cast<uintptr_t>(q) & 15) return KVP_ERR_INVALID_ARG;
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255)) return KVP_ERR_INVALID_ARG;
    const int HG = sh.HG;
    const int G = num_q_heads / pool->kv_heads;
    const int QH = HG * G;
    const WsLayout L = ws_layout(pool->num_sms, M * QH, 128);
    if (workspace_bytes < L.total) return KVP_ERR_INVALID_ARG;
    char* ws = static_cast<char*>(workspace);

    TcArgs ta;
    // The map is encoded once per pool and head group. Whether a stage can
    // use it (16 contiguous, 16-aligned slots) is decided per stage in the
    // kernel; without a map every row is loaded with its own copy.
    if (mp->tmap_hg != HG && mp->tmap_hg != -HG) mp->tmap_hg = tc_encode_tmap(pool, HG, &mp->tmap) ? HG : -HG;
    ta.use_tmap = mp->tmap_hg == HG;
    if (ta.use_tmap) ta.tmap = mp->tmap;
    else memset(&ta.tmap, 0, sizeof(ta.tmap));
    ta.kvl_k = layer;
    ta.kvl_v = pool->num_layers + layer;
    ta.nq = tc_num_qbuf(HG, G * M, sh.S);
    ta.stages = sh.S;
    ta.T = T;
    ta.kv_layer = kv_layer;
    ta.kv_bytes = pool->kv_bytes;
    ta.row_bytes = pool->row_bytes;
    ta.q = static_cast<const __nv_bfloat16*>(q);
    ta.out = static_cast<__nv_bfloat16*>(out);
    ta.context_lens = context_lens;
    ta.table_rows = table_rows;
    ta.B = batch;
    ta.Hq = num_q_heads;
    ta.G = G;
    ta.HG = HG;
    ta.n_groups = pool->kv_heads / HG;
    ta.window = window;
    ta.sinks = sinks;
    ta.M = M;
    ta.NT = sh.NT;
    ta.tiles = sh.T;
    ta.CW = HG * sh.T;
    ta.num_ctas = pool->num_sms;
    ta.scale_log2 = scale_log2;
    ta.merge = reinterpret_cast<int4*>(ws + L.merge);
    ta.part_ml = reinterpret_cast<float*>(ws + L.part_ml);
    ta.part_o = reinterpret_cast<float*>(ws + L.part_o);
    ta.err = pool->err;
    ta.fused = fz != nullptr;
    ta.knew = static_cast<const uint4*>(fz ? fz->k : nullptr);
    ta.vnew = static_cast<const uint4*>(fz ? fz->v : nullptr);
    ta.out_loc = fz ? fz->out_loc : nullptr;
    ta.tw_table = fz ? fz->table : nullptr;
    ta.tw_rows = fz ? fz->tw_rows : nullptr;
    ta.tw_cols = fz ? fz->tw_cols : nullptr;
    ta.tw_vals = fz ? fz->tw_vals : nullptr;
    ta.n_tw = fz ? fz->n_tw : 0;
    ta.tw_expand = expand;

    CombineArgs ca;
    ca.merge = ta.merge;
    ca.part_ml = ta.part_ml;
    ca.part_o = ta.part_o;
    ca.out = out;
    ca.dtype = pool->dtype;
    ca.n_groups = ta.n_groups;
    ca.QH = QH;
    ca.Hq = num_q_heads;
    ca.D = 128;
    ca.M = M;
    const cudaError_t e = launch_tc(ta, ca, st, mp->ev_before, mp->ev_after);
    mp->ev_before = mp->ev_after = nullptr;
    return e == cudaSuccess ? KVP_OK : KVP_ERR_CUDA;
  }

  if (pool->head_dim > kGenMaxD) return KVP_ERR_INVALID_ARG;
  GenArgs ga;
  ga.T = T;
  ga.kv_layer = kv_layer;
  ga.kv_bytes = pool->kv_bytes;
  ga.q = q;
  ga.out = out;
  ga.context_lens = context_lens;
  ga.table_rows = table_rows;
  ga.B = batch;
  ga.Hq = num_q_heads;
  ga.Hkv = pool->kv_heads;
  ga.D = pool->head_dim;
  ga.window = window;
  ga.sinks = sinks;
  ga.M = M;
  ga.q_lens = nullptr;
  ga.scale_log2 = scale_log2;
  ga.err = pool->err;
  const long long warps = (long long)batch * M * num_q_heads;
  const unsigned blocks = (unsigned)((warps + kGenWarps - 1) / kGenWarps);
  const bool timed = mp->ev_before != nullptr;
  if (timed && cudaEventRecord(static_cast<cudaEvent_t>(mp->ev_before), st) != cudaSuccess) return KVP_ERR_CUDA;
  if (pool->dtype == KVP_F32)
    generic_decode_kernel<float><<<blocks, 32 * kGenWarps, 0, st>>>(ga);
  else
    generic_decode_kernel<__nv_bfloat16><<<blocks, 32 * kGenWarps, 0, st>>>(ga);
  if (timed) {
    if (cudaEventRecord(static_cast<cudaEvent_t>(mp->ev_after), st) != cudaSuccess) return KVP_ERR_CUDA;
    mp->ev_before = mp->ev_after = nullptr;
  }
  return cudaGetLastError() == cudaSuccess ? KVP_OK : KVP_ERR_CUDA;
}

}  // namespace

extern "C" int paged_decode_attention(const kvp_pool* pool, int layer, const void* q, int batch, int num_q_heads,
                                      const int32_t* table, int table_rows_total, int table_cols, int table_mode,
                                      const int32_t* table_rows, const int32_t* context_lens, int window,
                                      int sinks, float scale, void* out, void* workspace, size_t workspace_bytes,
                                      void* stream) {
  return attention_impl(pool, layer, q, batch, 1, num_q_heads, table, table_rows_total, table_cols, table_mode,
                        table_rows, context_lens, window, sinks, scale, out, workspace, workspace_bytes, stream,
                        nullptr);
}

extern "C" int paged_verify_attention(const kvp_pool* pool, int layer, const void* q, int batch, int num_q_tokens,
                                      int num_q_heads, const int32_t* table, int table_rows_total, int table_cols,
                                      int table_mode, const int32_t* table_rows, const int32_t* context_lens,
                                      int window, int sinks, float scale, void* out, void* workspace,
                                      size_t workspace_bytes, void* stream) {
  return attention_impl(pool, layer, q, batch, num_q_tokens, num_q_heads, table, table_rows_total, table_cols,
                        table_mode, table_rows, context_lens, window, sinks, scale, out, workspace, workspace_bytes,
                        stream, nullptr);
}

extern "C" int store_cache_and_attention(const kvp_pool* pool, int layer, const void* q, const void* k,
                                         const void* v, const int32_t* out_loc, int batch, int num_q_heads,
                                         int32_t* table, int table_rows_total, int table_cols, int table_mode,
                                         const int32_t* table_rows, const int32_t* context_lens,
                                         const int32_t* tw_rows, const int32_t* tw_cols, const int32_t* tw_vals,
                                         int n_tw, int window, int sinks, float scale, void* out, void* workspace,
                                         size_t workspace_bytes, void* stream) {
  if (!k || !v || !out_loc || n_tw < 0 || (n_tw > 0 && (!tw_rows || !tw_cols || !tw_vals)))
    return KVP_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v)) & 15) return KVP_ERR_INVALID_ARG;
  const FuseIn fz = {k, v, out_loc, table, tw_rows, tw_cols, tw_vals, n_tw};
  return attention_impl(pool, layer, q, batch, 1, num_q_heads, table, table_rows_total, table_cols, table_mode,
                        table_rows, context_lens, window, sinks, scale, out, workspace, workspace_bytes, stream,
                        &fz);
}

extern "C" int paged_prefill_attention(const kvp_pool* pool, int layer, const void* q, int batch, int chunk,
                                       int num_q_heads, const int32_t* q_lens, const int32_t* table,
                                       int table_rows_total, int table_cols, int table_mode,
                                       const int32_t* table_rows, const int32_t* context_lens, int window, int sinks,
                                       float scale, void* out, void* stream) {
  if (!pool || !q || !table || !context_lens || !out) return KVP_ERR_INVALID_ARG;
  if (layer < 0 || layer >= pool->num_layers || batch <= 0 || chunk <= 0 || num_q_heads <= 0) return KVP_ERR_INVALID_ARG;
  if (num_q_heads % pool->kv_heads) return KVP_ERR_INVALID_ARG;
  if (table_rows_total <= 0 || table_cols <= 0) return KVP_ERR_INVALID_ARG;
  if (table_mode != KVP_BLOCK_TABLE && table_mode != KVP_RAW_LOCATIONS) return KVP_ERR_INVALID_ARG;
  if (!(scale == scale)) return KVP_ERR_INVALID_ARG;
  if (sinks < 0 || (window > 0 && sinks >= window)) return KVP_ERR_INVALID_ARG;
  if (window <= 0) sinks = 0;
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(out)) & 15) return KVP_ERR_INVALID_ARG;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  const TableRef T = make_table(pool, table, table_rows_total, table_cols, table_mode);
  kvp_pool* mp = const_cast<kvp_pool*>(pool);
  if (prefill_tc_eligible(pool, num_q_heads, chunk, scale)) {
    if (mp->ev_before && cudaEventRecord(static_cast<cudaEvent_t>(mp->ev_before), st) != cudaSuccess)
      return KVP_ERR_CUDA;
    const int rc = launch_prefill_tc(pool, layer, q, batch, chunk, num_q_heads, q_lens, T, table_rows, context_lens,
                                     window, sinks, scale, out, st);
    if (rc == KVP_OK && mp->ev_after && cudaEventRecord(static_cast<cudaEvent_t>(mp->ev_after), st) != cudaSuccess)
      return KVP_ERR_CUDA;
    mp->ev_before = mp->ev_after = nullptr;
    return rc;
  }
  if (pool->head_dim > kGenMaxD) return KVP_ERR_INVALID_ARG;
  GenArgs ga;
  ga.T = T;
  ga.kv_layer = pool->buf + (size_t)layer * pool->layer_bytes;
  ga.kv_bytes = pool->kv_bytes;
  ga.q = q;
  ga.out = out;
  ga.context_lens = context_lens;
  ga.table_rows = table_rows;
  ga.B = batch;
  ga.Hq = num_q_heads;
  ga.Hkv = pool->kv_heads;
  ga.D = pool->head_dim;
  ga.window = window;
  ga.sinks = sinks;
  ga.M = chunk;
  ga.q_lens = q_lens;
  ga.scale_log2 = scale * 1.4426950408889634f;
  ga.err = pool->err;
  const long long warps = (long long)batch * chunk * num_q_heads;
  const unsigned blocks = (unsigned)((warps + kGenWarps - 1) / kGenWarps);
  if (pool->dtype == KVP_F32)
    generic_decode_kernel<float><<<blocks, 32 * kGenWarps, 0, st>>>(ga);
  else
    generic_decode_kernel<__nv_bfloat16><<<blocks, 32 * kGenWarps, 0, st>>>(ga);
  return cudaGetLastError() == cudaSuccess ? KVP_OK : KVP_ERR_CUDA;
}

extern "C" int gather_indices(const kvp_pool* pool, const int32_t* table, int table_rows_total, int table_cols,
                              int table_mode, const int32_t* table_rows, const int32_t* context_lens, int batch,
                              int window, int sinks, int32_t* slots_out, int max_tokens, void* stream) {
  if (!pool || !table || !context_lens || !slots_out || batch <= 0 || max_tokens <= 0) return KVP_ERR_INVALID_ARG;
  if (sinks < 0 || (window > 0 && sinks >= window)) return KVP_ERR_INVALID_ARG;
  if (window <= 0) sinks = 0;
  if (table_rows_total <= 0 || table_cols <= 0) return KVP_ERR_INVALID_ARG;
  if (table_mode != KVP_BLOCK_TABLE && table_mode != KVP_RAW_LOCATIONS) return KVP_ERR_INVALID_ARG;
  const TableRef T = make_table(pool, table, table_rows_total, table_cols, table_mode);
  gather_indices_kernel<<<batch, 256, 0, static_cast<cudaStream_t>(stream)>>>(T, context_lens, table_rows, window,
                                                                               sinks, slots_out, max_tokens, pool->err);
  return cudaGetLastError() == cudaSuccess ? KVP_OK : KVP_ERR_CUDA;
}
