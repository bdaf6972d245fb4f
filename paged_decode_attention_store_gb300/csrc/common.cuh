// Shared device helpers of libpagedkv (CUDA path only).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pagedkv.h"

struct kvp_pool {
  int num_pages;    // pages in the buffer (dummy page included)
  int page_size;
  int kv_heads;
  int head_dim;
  int dtype;        // kvp_dtype
  int num_layers;
  int elem;         // bytes per element
  int num_slots;    // num_pages * page_size
  size_t row_bytes;    // one token, all KV heads, K or V: kv_heads*head_dim*elem
  size_t layer_bytes;  // one layer's K (or V): num_slots * row_bytes
  size_t kv_bytes;     // K -> V distance: num_layers * layer_bytes
  char* buf;
  int32_t* err;
  int num_sms;
  int device;
  void* ev_before;  // optional timing events around the next attention kernel
  void* ev_after;
  CUtensorMap tmap;  // tensor map of the whole buffer for the tensor-core kernel,
  int tmap_hg;       // heads per box it was encoded for (0: none yet, -HG: refused for HG)
  CUtensorMap tmap1; // the buffer as (d % 64, slot, d / 64, head, K/V x layer), for the prefill kernel:
  CUtensorMap tmap2; //   box (64, 16, 2, 1, 1) (tmap1, V) and box (64, 16, 1, 1, 1) (tmap2, K halves)
  int tmap1_state;   // 0: not encoded yet, 1: both encoded, -1: refused
};

namespace kvp {

__device__ __forceinline__ void set_error(int32_t* err, int code) {
  if (err) atomicCAS(reinterpret_cast<int*>(err), 0, code);
}

// Table addressing shared by every kernel that reads a request's rows.
struct TableRef {
  const int32_t* table;
  int rows_total;
  int cols;
  int raw;          // 1: raw token locations, 0: block table
  int page_size;
  int num_pages;
  int num_slots;
};

// Capacity in token positions of one table row.
__host__ __device__ __forceinline__ long long table_capacity(const TableRef& T) {
  return T.raw ? (long long)T.cols : (long long)T.cols * T.page_size;
}

// Flat slot of position t of the request in table row ``row``:
//   block mode  table[row][t / P] * P + t % P   ("PagedAttention block
//               allocator", section "Sequence block table")
//   raw mode    table[row][t]                   (mini-sglang code series,
//               part 4: the table holds raw token locations)
// Returns -1 (and records KVP_ERR_BAD_INDEX) for a hole or an entry outside
// the pool. The caller has checked 0 <= t < table_capacity(T).
__device__ __forceinline__ int resolve_slot(const TableRef& T, int row, int t, int32_t* err) {
  const int32_t* r = T.table + (size_t)row * T.cols;
  if (T.raw) {
    int s = __ldg(r + t);
    if ((unsigned)s >= (unsigned)T.num_slots) {
      set_error(err, KVP_ERR_BAD_INDEX);
      return -1;
    }
    return s;
  }
  int page = __ldg(r + t / T.page_size);
  if ((unsigned)page >= (unsigned)T.num_pages) {
    set_error(err, KVP_ERR_BAD_INDEX);
    return -1;
  }
  return page * T.page_size + t % T.page_size;
}

__device__ __forceinline__ int window_lo(int L, int window) {
  return window > 0 ? max(0, L - window) : 0;
}

// The positions a step with context L attends: [0, se) and [lo, L).
// Chapter 15 ("The model"): the window W is the new token and at most W-1
// earlier ones; its exercise "Attention sinks" keeps the first S rows too
// and takes the last W - S for the rest, so
//   lo = max(0, L - (W - S)),  se = min(S, lo).
// No window (W <= 0): everything. When the two ranges touch (lo <= S) the
// span is the whole context and is returned as se = lo = 0.
struct Span {
  int se, lo;
};

__host__ __device__ __forceinline__ Span attend_span(int L, int window, int sinks) {
  Span s = {0, 0};
  if (window > 0) {
    const int lo = L - (window - sinks);
    s.lo = lo > 0 ? lo : 0;
    s.se = sinks < s.lo ? sinks : s.lo;
    if (s.se == s.lo) s.se = s.lo = 0;
  }
  return s;
}

// Position of the o-th attended row (0 <= o < se + L - lo).
__host__ __device__ __forceinline__ int span_pos(const Span& s, int o) { return o < s.se ? o : s.lo + (o - s.se); }

// ---------------------------------------------------------------------------
// PTX wrappers (sm_90+ async proxy, sm_80+ tensor-core fragments).
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t tx) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(tx)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Wait for the phase with the given parity to complete, for at most
// ``limit_ns``; on timeout records KVP_ERR_TIMEOUT, raises the CTA's abort
// flag and returns false. Also returns false as soon as another warp of the
// CTA has raised the abort flag.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                                  int32_t* err, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63) == 0) {
      if (*abort_flag) return false;
      if (global_timer_ns() - t0 > limit_ns) {
        set_error(err, KVP_ERR_TIMEOUT);
        *abort_flag = 1;
        return false;
      }
    }
  }
}

// Bulk (non-tensor) async copy global -> this CTA's shared memory, completing
// ``bytes`` of transaction count on ``bar``. Addresses 16-byte aligned, size
// a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void bulk_g2s_hint(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                              uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// TMA tensor load of one box of a 4-D tensor map into this CTA's shared
// memory, completing its bytes on ``bar``. The map lives in kernel-parameter
// (grid constant) memory; c0 is the innermost coordinate.
__device__ __forceinline__ void tma_load_4d(void* dst, const void* tmap, int c0, int c1, int c2, int c3, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5}], "
      "[%6];" ::"r"(smem_u32(dst)),
      "l"(tmap), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_u32(bar))
      : "memory");
}

// 4-byte asynchronous copy global -> shared (sm_80 cp.async), grouped per commit.
__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Order this thread's generic-proxy shared-memory writes before later
// async-proxy (bulk copy) writes to the same addresses.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}

// D(16x8, f32) += A(16x16, bf16, row) * B(16x8, bf16, col)
__device__ __forceinline__ void mma_bf16_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Transpose an 8x8 matrix of 16-bit elements held one row pair per lane.
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float bf16_lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t x) { return __uint_as_float(x & 0xFFFF0000u); }

}  // namespace kvp
