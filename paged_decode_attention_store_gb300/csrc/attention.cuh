// Internal declarations of the decode-attention kernels of libpagedkv.
#pragma once

#include <cuda.h>

#include "common.cuh"

namespace kvp {

// Work split. A virtual request is one (request b, KV-head group g) pair,
// v = b * n_groups + g. The attended positions [lo, L) of all virtual
// requests are laid end to end in one token stream of T positions; CTA k of
// Ne takes the range [k*T/Ne, (k+1)*T/Ne), so every CTA streams the same
// number of K/V bytes whatever the length mix. A request cut by a range
// boundary leaves one fp32 partial per piece in a fixed slot: the first piece
// of CTA k (it starts at the range start) uses slot 2k, its last piece slot
// 2k+1. The CTA that holds a split request's final piece records the request
// in merge[k] = {v, k_first, slot_first, k}; the combine kernel merges the
// pieces: slot_first, then 2j for k_first < j <= k.

// Workspace layout (offsets in bytes from the 256-byte aligned base).
struct WsLayout {
  size_t merge;    // int4[num_ctas]
  size_t part_ml;  // float[2 * num_ctas * QH * 2]  (running max in log2 units, sum)
  size_t part_o;   // float[2 * num_ctas * QH * D]  (unnormalised output)
  size_t total;
};

__host__ inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

__host__ inline WsLayout ws_layout(int num_ctas, int QH, int D) {
  WsLayout w;
  size_t o = 0;
  w.merge = o;
  o = align256(o + sizeof(int4) * num_ctas);
  w.part_ml = o;
  o = align256(o + sizeof(float) * 2 * 2 * (size_t)num_ctas * QH);
  w.part_o = o;
  o = align256(o + sizeof(float) * 2 * (size_t)num_ctas * QH * D);
  w.total = o;
  return w;
}

struct TcArgs {
  // Tensor map over the whole KV buffer viewed as (d, slot, kv head, K/V x
  // layer) with strides (2 B, row bytes, 256 B, layer bytes): the slot and
  // head axes are deliberately not in stride order, so that a box of 16
  // slots x HG heads lands in shared memory head-major (rows head*16+slot).
  CUtensorMap tmap;
  int use_tmap;            // load full, contiguous 16-slot groups with tensor copies
  int kvl_k, kvl_v;        // the map's last coordinate for this layer's K and V
  int nq;                  // Q buffers in shared memory (1 or 2)
  TableRef T;
  const char* kv_layer;    // K of this layer
  size_t kv_bytes;         // K -> V distance
  size_t row_bytes;        // one token, all KV heads
  const __nv_bfloat16* q;  // [B, M, Hq, D]
  __nv_bfloat16* out;      // [B, M, Hq, D]
  const int32_t* context_lens;
  const int32_t* table_rows;
  int B, Hq, G, HG, n_groups, window, sinks, num_ctas;
  // Query tokens per request (1: decode; M > 1: the M newest tokens verified
  // at once, query j at position L - M + j, causal). The M * G (token, head)
  // columns of a KV head are split over ``tiles`` consumer warps of NT
  // 8-column MMA tiles each; CW = HG * tiles consumer warps in all.
  int M, NT, tiles, CW;
  int stages;  // ring depth (3 for 8 KV heads per CTA, deeper for fewer)
  float scale_log2;
  int4* merge;
  float* part_ml;
  float* part_o;
  int32_t* err;
  // Fused step (store_cache_and_attention): this launch also applies the
  // step's table writes and stores the new K/V rows; each request's newest
  // position is read from the new rows rather than from the cache.
  int fused;
  const uint4* knew;       // [B, kv_heads, D] new K rows
  const uint4* vnew;       // [B, kv_heads, D] new V rows
  const int32_t* out_loc;  // [B] slots of the new rows
  int32_t* tw_table;       // the table, writable
  const int32_t* tw_rows;
  const int32_t* tw_cols;
  const int32_t* tw_vals;
  int n_tw, tw_expand;
};

struct CombineArgs {
  const int4* merge;
  const float* part_ml;
  const float* part_o;
  void* out;
  int dtype;
  int n_groups, QH, Hq, D;
  int M;  // query tokens per request: the partials hold M * QH columns, token-major
};

// Programmatic dependent launch: a kernel launched with the programmatic
// stream-serialization attribute may start while its predecessor in the
// stream is still running; griddep_wait() blocks until that predecessor has
// completed and its memory is visible. Every kernel here waits before its
// first global access, so the overlap only hides launch latency.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Exclusive scan of one value per thread over the whole block (at most 32
// warps); *total receives the sum. Contains __syncthreads.
__device__ __forceinline__ long long block_exclusive_scan(long long x, long long* total) {
  __shared__ long long warp_sums[32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
  long long incl = x;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const long long y = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= d) incl += y;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    long long v = lane < nw ? warp_sums[lane] : 0;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const long long y = __shfl_up_sync(0xffffffffu, v, d);
      if (lane >= d) v += y;
    }
    if (lane < nw) warp_sums[lane] = v;  // inclusive over warps
  }
  __syncthreads();
  const long long before = (warp > 0 ? warp_sums[warp - 1] : 0) + incl - x;
  *total = warp_sums[nw - 1];
  __syncthreads();
  return before;
}

// Shared-memory bytes of the tensor-core kernel for HG KV heads per CTA and
// C query columns per KV head (G heads x M tokens) with nq Q buffers (0 if it
// does not fit), and the number of Q buffers it will use (2 when they fit,
// else 1; 0 if neither).
size_t tc_smem_bytes(int HG, int C, int nq, int S);
int tc_num_qbuf(int HG, int C, int S);
// Ring depth for HG KV heads per CTA and C query columns per head.
int tc_num_stages(int HG, int C);
// Encode the tensor map of a bf16 pool for HG heads per box; false if the
// driver refuses it.
bool tc_encode_tmap(const kvp_pool* pool, int HG, CUtensorMap* out);
// Largest batch the in-kernel work split can take for HG and ring depth S.
int tc_max_batch(int HG, int S);
// Chunked prefill on tcgen05 (prefill_tc.cu): whether a pool and query-head
// count take it, and its launch over batch requests of up to C new tokens.
bool prefill_tc_eligible(const kvp_pool* pool, int Hq, int C, float scale);
int launch_prefill_tc(const kvp_pool* pool, int layer, const void* q, int batch, int C, int Hq, const int32_t* q_lens,
                      const TableRef& T, const int32_t* table_rows, const int32_t* context_lens, int window, int sinks,
                      float scale, void* out, cudaStream_t stream);
// Launch the bf16, head_dim-128 kernel (one CTA per SM) and the combine
// kernel after it, both as programmatic dependents.
cudaError_t launch_tc(const TcArgs& a, const CombineArgs& c, cudaStream_t stream, void* ev_before, void* ev_after);

}  // namespace kvp
