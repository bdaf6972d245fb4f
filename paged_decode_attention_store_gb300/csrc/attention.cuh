// Internal declarations of the decode-attention kernels of libpagedkv.
#pragma once

#include "common.cuh"

namespace kvp {

// A virtual request is one (request b, KV-head group g) pair: v = b * n_groups + g.
// Its attended positions [lo, L) form one segment of a token stream that
// concatenates all virtual requests; the stream is cut into one equal range
// per CTA, and a work item is the intersection of a range with a request.
struct __align__(16) WorkItem {
  int v;        // virtual request
  int b;        // request
  int row;      // table row of the request
  int group;    // KV-head group
  int t_begin;  // first position of this item
  int t_end;    // one past its last position
  int part;     // partial slot (the item index) when the request is split, else -1
  int pad;
};

struct ReqInfo {
  int first;  // first item of the virtual request
  int count;  // its number of items: 0 invalid (zero output), 1 direct, >1 combined
};

// Workspace layout (offsets in bytes from the 256-byte aligned base).
struct WsLayout {
  size_t cta_first;  // int[num_ctas + 1]
  size_t req;        // ReqInfo[V]
  size_t nv;         // int[V]    attended positions per virtual request
  size_t sv;         // long long[V] stream offset per virtual request
  size_t items;      // WorkItem[cap]
  size_t part_ml;    // float[cap * QH * 2]  (running max in log2 units, sum)
  size_t part_o;     // float[cap * QH * D]  (unnormalised output)
  size_t total;
  int cap;           // maximum number of items
};

__host__ inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

__host__ inline WsLayout ws_layout(int V, int num_ctas, int QH, int D) {
  WsLayout w;
  w.cap = V + num_ctas + 1;
  size_t o = 0;
  w.cta_first = o; o = align256(o + sizeof(int) * (num_ctas + 1));
  w.req = o;       o = align256(o + sizeof(ReqInfo) * V);
  w.nv = o;        o = align256(o + sizeof(int) * V);
  w.sv = o;        o = align256(o + sizeof(long long) * V);
  w.items = o;     o = align256(o + sizeof(WorkItem) * w.cap);
  w.part_ml = o;   o = align256(o + sizeof(float) * 2 * (size_t)w.cap * QH);
  w.part_o = o;    o = align256(o + sizeof(float) * (size_t)w.cap * QH * D);
  w.total = o;
  return w;
}

struct PlanArgs {
  TableRef T;
  const int32_t* context_lens;
  const int32_t* table_rows;
  int B;
  int n_groups;
  int window;
  int num_ctas;
  char* ws;
  WsLayout L;
  int32_t* err;
};

struct TcArgs {
  TableRef T;
  const char* kv_layer;     // K of this layer
  size_t kv_bytes;          // K -> V distance
  size_t row_bytes;         // one token, all KV heads
  const __nv_bfloat16* q;   // [B, Hq, D]
  __nv_bfloat16* out;       // [B, Hq, D]
  int Hq, G, HG;            // q heads, group size, KV heads per CTA
  float scale_log2;
  const int* cta_first;
  const WorkItem* items;
  float* part_ml;
  float* part_o;
  int32_t* err;
};

struct CombineArgs {
  const ReqInfo* req;
  const float* part_ml;
  const float* part_o;
  void* out;
  int dtype;
  int V, n_groups, QH, Hq, D;
};

// Shared-memory bytes of the tensor-core kernel for HG KV heads per CTA and
// G query heads per KV head (0 if it does not fit).
size_t tc_smem_bytes(int HG, int G);
// Launch the bf16, head_dim-128 kernel (NT = 1 for G <= 8, 2 for G <= 16).
cudaError_t launch_tc(const TcArgs& a, int num_ctas, cudaStream_t stream);

}  // namespace kvp
