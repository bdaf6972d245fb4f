// Decode attention: work plan, split-K combine, the general CUDA-core kernel,
// the index dump, and the C ABI that picks between the kernels.
//
// Split-K plan (the flash-decoding idea, sized for a persistent grid): the
// attended positions of all requests are laid end to end in one token stream
// and the stream is cut into one equal range per CTA, so every CTA streams
// the same number of K/V bytes whatever the length mix. A request that falls
// inside one range is finished by that CTA; a request cut by range
// boundaries leaves one fp32 partial per piece, merged by the combine kernel
// with the usual rescaling: M = max m_i, out = sum 2^(m_i-M) o_i / sum
// 2^(m_i-M) l_i (pieces with no token have m_i = -inf and weight 0).
#include "attention.cuh"

namespace kvp {

namespace {

constexpr int kPlanThreads = 1024;
constexpr int kMinTokensPerCta = 64;

// Exclusive scan of one value per thread over a 1024-thread block.
__device__ long long block_exclusive_scan(long long x, long long* total) {
  __shared__ long long warp_sums[32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  long long incl = x;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    long long y = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= d) incl += y;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int nw = blockDim.x >> 5;
    long long v = lane < nw ? warp_sums[lane] : 0;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      long long y = __shfl_up_sync(0xffffffffu, v, d);
      if (lane >= d) v += y;
    }
    if (lane < nw) warp_sums[lane] = v;  // inclusive over warps
  }
  __syncthreads();
  const long long before = (warp > 0 ? warp_sums[warp - 1] : 0) + incl - x;
  *total = warp_sums[(blockDim.x >> 5) - 1];
  __syncthreads();
  return before;
}

__device__ __forceinline__ long long ceil_div_ll(long long a, long long b) { return (a + b - 1) / b; }

__global__ void __launch_bounds__(kPlanThreads) plan_kernel(const PlanArgs p) {
  int* cta_first = reinterpret_cast<int*>(p.ws + p.L.cta_first);
  ReqInfo* req = reinterpret_cast<ReqInfo*>(p.ws + p.L.req);
  int* nv = reinterpret_cast<int*>(p.ws + p.L.nv);
  long long* sv = reinterpret_cast<long long*>(p.ws + p.L.sv);
  WorkItem* items = reinterpret_cast<WorkItem*>(p.ws + p.L.items);

  const int V = p.B * p.n_groups;
  const int per = (V + kPlanThreads - 1) / kPlanThreads;
  const int v0 = min(V, (int)threadIdx.x * per), v1 = min(V, v0 + per);
  const long long cap = table_capacity(p.T);

  // Phase 1: attended positions per virtual request, stream offsets.
  long long local = 0;
  for (int v = v0; v < v1; ++v) {
    const int b = v / p.n_groups;
    const int L = p.context_lens[b];
    const int row = p.table_rows ? p.table_rows[b] : b;
    const bool valid = L >= 1 && L <= cap && row >= 0 && row < p.T.rows_total;
    if (!valid && (v % p.n_groups) == 0) set_error(p.err, KVP_ERR_BAD_INDEX);
    const int n = valid ? L - window_lo(L, p.window) : 0;
    nv[v] = n;
    local += n;
  }
  long long T;
  long long base = block_exclusive_scan(local, &T);
  for (int v = v0; v < v1; ++v) {
    sv[v] = base;
    base += nv[v];
  }
  const long long Ne = T > 0 ? min((long long)p.num_ctas, ceil_div_ll(T, kMinTokensPerCta)) : 0;

  // Phase 2: items per virtual request (1 + CTA boundaries strictly inside it).
  local = 0;
  for (int v = v0; v < v1; ++v) {
    const long long n = nv[v], S = sv[v];
    if (n == 0) continue;
    const long long k_lo = ceil_div_ll((S + 1) * Ne, T);
    const long long k_hi = ceil_div_ll((S + n) * Ne, T) - 1;
    local += 1 + max(0LL, k_hi - k_lo + 1);
  }
  long long n_items;
  long long first = block_exclusive_scan(local, &n_items);
  for (int v = v0; v < v1; ++v) {
    const long long n = nv[v], S = sv[v];
    const int b = v / p.n_groups, grp = v % p.n_groups;
    if (n == 0) {
      req[v] = ReqInfo{(int)first, 0};
      continue;
    }
    const int L = p.context_lens[b];
    const int lo = window_lo(L, p.window);
    const int row = p.table_rows ? p.table_rows[b] : b;
    const long long k_lo = ceil_div_ll((S + 1) * Ne, T);
    const long long k_hi = ceil_div_ll((S + n) * Ne, T) - 1;
    const long long kz = ceil_div_ll(S * Ne, T);
    const int cnt = 1 + (int)max(0LL, k_hi - k_lo + 1);
    req[v] = ReqInfo{(int)first, cnt};
    for (long long k = kz; k < k_lo; ++k) cta_first[k] = (int)first;  // ranges that start at S
    long long seg_start = S;
    for (int j = 0; j < cnt; ++j) {
      const long long k = k_lo + j;  // boundary ending segment j
      const long long seg_end = (j == cnt - 1) ? S + n : (k * T) / Ne;
      WorkItem w;
      w.v = v;
      w.b = b;
      w.row = row;
      w.group = grp;
      w.t_begin = lo + (int)(seg_start - S);
      w.t_end = lo + (int)(seg_end - S);
      w.part = cnt > 1 ? (int)(first + j) : -1;
      w.pad = 0;
      items[first + j] = w;
      if (j > 0) cta_first[k_lo + j - 1] = (int)(first + j);
      seg_start = seg_end;
    }
    first += cnt;
  }
  for (long long k = Ne + threadIdx.x; k <= p.num_ctas; k += blockDim.x) cta_first[k] = (int)n_items;
}

// One warp per (virtual request, query head of its group).
__global__ void combine_kernel(const CombineArgs a) {
  const long long wid = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (wid >= (long long)a.V * a.QH) return;
  const int v = (int)(wid / a.QH), qhl = (int)(wid % a.QH);
  const ReqInfo r = a.req[v];
  if (r.count == 1) return;  // finished by the attention kernel
  const int b = v / a.n_groups, grp = v % a.n_groups;
  const size_t orow = ((size_t)b * a.Hq + (size_t)grp * a.QH + qhl) * a.D;
  float M = -INFINITY;
  for (int i = 0; i < r.count; ++i) M = fmaxf(M, a.part_ml[((size_t)(r.first + i) * a.QH + qhl) * 2]);
  for (int d0 = lane * 4; d0 < a.D; d0 += 128) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float Ls = 0.f;
    for (int i = 0; i < r.count; ++i) {
      const size_t pi = (size_t)(r.first + i) * a.QH + qhl;
      const float mi = a.part_ml[pi * 2], li = a.part_ml[pi * 2 + 1];
      const float wgt = (mi == -INFINITY) ? 0.f : exp2f(mi - M);
      Ls += wgt * li;
      const float4 o = *reinterpret_cast<const float4*>(a.part_o + pi * a.D + d0);
      acc.x += wgt * o.x;
      acc.y += wgt * o.y;
      acc.z += wgt * o.z;
      acc.w += wgt * o.w;
    }
    const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
    if (a.dtype == KVP_BF16) {
      __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out) + orow + d0;
      __nv_bfloat162 lo2 = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
      __nv_bfloat162 hi2 = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
      uint2 packed;
      packed.x = *reinterpret_cast<uint32_t*>(&lo2);
      packed.y = *reinterpret_cast<uint32_t*>(&hi2);
      *reinterpret_cast<uint2*>(out) = packed;
    } else {
      float* out = static_cast<float*>(a.out) + orow + d0;
      *reinterpret_cast<float4*>(out) = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
    }
  }
}

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
  int B, Hq, Hkv, D, window;
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
  if (wid >= (long long)a.B * a.Hq) return;
  const int b = (int)(wid / a.Hq), h = (int)(wid % a.Hq);
  const int G = a.Hq / a.Hkv, kvh = h / G;
  const int D = a.D;
  T* out = static_cast<T*>(a.out) + ((size_t)b * a.Hq + h) * D;
  const T* q = static_cast<const T*>(a.q) + ((size_t)b * a.Hq + h) * D;
  const int L = a.context_lens[b];
  const int row = a.table_rows ? a.table_rows[b] : b;
  if (L < 1 || L > table_capacity(a.T) || row < 0 || row >= a.T.rows_total) {
    if (h == 0 && lane == 0) set_error(a.err, KVP_ERR_BAD_INDEX);
    for (int d = lane; d < D; d += 32) out[d] = from_f<T>(0.f);
    return;
  }
  for (int d = lane; d < D; d += 32) qs[warp][d] = to_f<T>(q[d]);
  __syncwarp();
  const int lo = window_lo(L, a.window);
  const size_t row_elems = (size_t)a.Hkv * D;
  const T* K = reinterpret_cast<const T*>(a.kv_layer);
  const T* Vp = reinterpret_cast<const T*>(a.kv_layer + a.kv_bytes);
  constexpr int kPerLane = kGenMaxD / 32;
  float acc[kPerLane];
#pragma unroll
  for (int i = 0; i < kPerLane; ++i) acc[i] = 0.f;
  float m = -INFINITY, l = 0.f;
  for (int t0 = lo; t0 < L; t0 += 32) {
    const int t = t0 + lane;
    int slot = -1;
    float s = -INFINITY;
    if (t < L) {
      slot = resolve_slot(a.T, row, t, a.err);
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
    const int nt = min(32, L - t0);
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
                                      int32_t* out, int max_tokens, int32_t* err) {
  const int b = blockIdx.x;
  const int L = context_lens[b];
  const int row = table_rows ? table_rows[b] : b;
  const bool valid = L >= 1 && L <= table_capacity(T) && row >= 0 && row < T.rows_total;
  const int lo = valid ? window_lo(L, window) : 0;
  const int n = valid ? L - lo : 0;
  if ((!valid || n > max_tokens) && threadIdx.x == 0) set_error(err, KVP_ERR_BAD_INDEX);
  for (int i = threadIdx.x; i < max_tokens; i += blockDim.x) {
    int s = -1;
    if (i < n) s = resolve_slot(T, row, lo + i, err);
    out[(size_t)b * max_tokens + i] = s;
  }
}

bool tc_eligible(const kvp_pool* pool, int Hq, int* HG_out) {
  if (pool->dtype != KVP_BF16 || pool->head_dim != 128) return false;
  const int Hkv = pool->kv_heads;
  if (Hq % Hkv) return false;
  const int G = Hq / Hkv;
  if (G > 16) return false;
  for (int HG = 8; HG >= 1; --HG) {
    if (Hkv % HG) continue;
    if (tc_smem_bytes(HG, G) == 0) continue;
    *HG_out = HG;
    return true;
  }
  return false;
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
  int HG = 0;
  if (!tc_eligible(pool, num_q_heads, &HG)) {
    *bytes = 256;  // the general kernel needs no scratch
    return KVP_OK;
  }
  const int n_groups = pool->kv_heads / HG;
  const int QH = HG * (num_q_heads / pool->kv_heads);
  *bytes = ws_layout(batch * n_groups, pool->num_sms, QH, 128).total;
  return KVP_OK;
}

extern "C" int paged_decode_attention(const kvp_pool* pool, int layer, const void* q, int batch, int num_q_heads,
                                      const int32_t* table, int table_rows_total, int table_cols, int table_mode,
                                      const int32_t* table_rows, const int32_t* context_lens, int window,
                                      float scale, void* out, void* workspace, size_t workspace_bytes,
                                      void* stream) {
  if (!pool || !q || !table || !context_lens || !out) return KVP_ERR_INVALID_ARG;
  if (layer < 0 || layer >= pool->num_layers || batch <= 0 || num_q_heads <= 0) return KVP_ERR_INVALID_ARG;
  if (num_q_heads % pool->kv_heads) return KVP_ERR_INVALID_ARG;
  if (table_rows_total <= 0 || table_cols <= 0) return KVP_ERR_INVALID_ARG;
  if (table_mode != KVP_BLOCK_TABLE && table_mode != KVP_RAW_LOCATIONS) return KVP_ERR_INVALID_ARG;
  if (!(scale == scale)) return KVP_ERR_INVALID_ARG;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  const TableRef T = make_table(pool, table, table_rows_total, table_cols, table_mode);
  const char* kv_layer = pool->buf + (size_t)layer * pool->layer_bytes;
  const float scale_log2 = scale * 1.4426950408889634f;

  int HG = 0;
  if (tc_eligible(pool, num_q_heads, &HG)) {
    if (reinterpret_cast<uintptr_t>(q) & 15) return KVP_ERR_INVALID_ARG;
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255)) return KVP_ERR_INVALID_ARG;
    const int G = num_q_heads / pool->kv_heads;
    const int n_groups = pool->kv_heads / HG;
    const int QH = HG * G;
    const WsLayout L = ws_layout(batch * n_groups, pool->num_sms, QH, 128);
    if (workspace_bytes < L.total) return KVP_ERR_INVALID_ARG;
    char* ws = static_cast<char*>(workspace);

    PlanArgs pa;
    pa.T = T;
    pa.context_lens = context_lens;
    pa.table_rows = table_rows;
    pa.B = batch;
    pa.n_groups = n_groups;
    pa.window = window;
    pa.num_ctas = pool->num_sms;
    pa.ws = ws;
    pa.L = L;
    pa.err = pool->err;
    plan_kernel<<<1, kPlanThreads, 0, st>>>(pa);

    TcArgs ta;
    ta.T = T;
    ta.kv_layer = kv_layer;
    ta.kv_bytes = pool->kv_bytes;
    ta.row_bytes = pool->row_bytes;
    ta.q = static_cast<const __nv_bfloat16*>(q);
    ta.out = static_cast<__nv_bfloat16*>(out);
    ta.Hq = num_q_heads;
    ta.G = G;
    ta.HG = HG;
    ta.scale_log2 = scale_log2;
    ta.cta_first = reinterpret_cast<const int*>(ws + L.cta_first);
    ta.items = reinterpret_cast<const WorkItem*>(ws + L.items);
    ta.part_ml = reinterpret_cast<float*>(ws + L.part_ml);
    ta.part_o = reinterpret_cast<float*>(ws + L.part_o);
    ta.err = pool->err;
    kvp_pool* mp = const_cast<kvp_pool*>(pool);
    const bool timed = mp->ev_before != nullptr;
    if (timed && cudaEventRecord(static_cast<cudaEvent_t>(mp->ev_before), st) != cudaSuccess) return KVP_ERR_CUDA;
    if (launch_tc(ta, pool->num_sms, st) != cudaSuccess) return KVP_ERR_CUDA;
    if (timed) {
      if (cudaEventRecord(static_cast<cudaEvent_t>(mp->ev_after), st) != cudaSuccess) return KVP_ERR_CUDA;
      mp->ev_before = mp->ev_after = nullptr;
    }

    CombineArgs ca;
    ca.req = reinterpret_cast<const ReqInfo*>(ws + L.req);
    ca.part_ml = ta.part_ml;
    ca.part_o = ta.part_o;
    ca.out = out;
    ca.dtype = pool->dtype;
    ca.V = batch * n_groups;
    ca.n_groups = n_groups;
    ca.QH = QH;
    ca.Hq = num_q_heads;
    ca.D = 128;
    const long long warps = (long long)ca.V * QH;
    combine_kernel<<<(unsigned)((warps * 32 + 255) / 256), 256, 0, st>>>(ca);
    return cudaGetLastError() == cudaSuccess ? KVP_OK : KVP_ERR_CUDA;
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
  ga.scale_log2 = scale_log2;
  ga.err = pool->err;
  const long long warps = (long long)batch * num_q_heads;
  const unsigned blocks = (unsigned)((warps + kGenWarps - 1) / kGenWarps);
  kvp_pool* mp = const_cast<kvp_pool*>(pool);
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

extern "C" int gather_indices(const kvp_pool* pool, const int32_t* table, int table_rows_total, int table_cols,
                              int table_mode, const int32_t* table_rows, const int32_t* context_lens, int batch,
                              int window, int32_t* slots_out, int max_tokens, void* stream) {
  if (!pool || !table || !context_lens || !slots_out || batch <= 0 || max_tokens <= 0) return KVP_ERR_INVALID_ARG;
  if (table_rows_total <= 0 || table_cols <= 0) return KVP_ERR_INVALID_ARG;
  if (table_mode != KVP_BLOCK_TABLE && table_mode != KVP_RAW_LOCATIONS) return KVP_ERR_INVALID_ARG;
  const TableRef T = make_table(pool, table, table_rows_total, table_cols, table_mode);
  gather_indices_kernel<<<batch, 256, 0, static_cast<cudaStream_t>(stream)>>>(T, context_lens, table_rows, window,
                                                                               slots_out, max_tokens, pool->err);
  return cudaGetLastError() == cudaSuccess ? KVP_OK : KVP_ERR_CUDA;
}
