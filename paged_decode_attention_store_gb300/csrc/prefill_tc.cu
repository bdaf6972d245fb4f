// Paged chunked-prefill attention on the fifth-generation tensor cores
// (tcgen05 MMAs with TMEM accumulators), bf16, head_dim 128.
//
// What it computes (the multi-query form of the decode step; "Week 3 Day 3:
// Paged KV Cache" of tiny-llm prefills in chunks and appends each chunk's
// K/V to the pages before attending): request b's q_lens[b] newest tokens,
// already stored, are queries at once; query j at position
// p = L - q_lens[b] + j attends what a one-token step with context p + 1
// attends (causal, the same window and sinks; chapter 15, "The model", and
// its exercise "Attention sinks"), reading K/V in place through the table.
//
// How (one CTA of four warps per 128-row query tile):
// * A tile is 128 / G consecutive query tokens of one request times the G
//   query heads of one KV head: 128 rows of Q, loaded once by TMA (128-byte
//   swizzle, two 64-element halves of head_dim).
// * The keys the tile needs (the union of its queries' spans) stream in
//   blocks of 128: a 16-slot group whose slots are contiguous and 16-aligned
//   comes by TMA (K and V, two halves each), any other key row is copied by
//   its thread into the same swizzled layout.
// * S = Q K^T (M 128, N 128, K 128: eight kind::f16 MMAs, both operands
//   K-major) accumulates in TMEM columns 0-127. Each thread owns one query
//   row: it reads its 128 scores from TMEM, masks them (causal, window,
//   sinks, block end), and keeps an online softmax in log2 units. O is
//   rescaled (read, scaled, written back in TMEM) only when the row maximum
//   grows by more than 8, so P = 2^(x - m) <= 256 always fits bf16 and the
//   normalisation stays exact (numerator and denominator use the same m).
// * P (bf16, K-major, 128-byte swizzle) goes to shared memory, in K's
//   place, and O += P V (V as the MN-major operand) accumulates in TMEM
//   columns 128-255. The epilogue divides by the row sum and stores bf16.
// * 97 KB of shared memory and 256 TMEM columns per CTA: two CTAs share an
//   SM, so one's loads and softmax overlap the other's MMAs.
// * Every wait is bounded (2 s): on timeout the CTA records KVP_ERR_TIMEOUT,
//   issues nothing more, waits (bounded) for what it issued and frees TMEM.
#include <cudaTypedefs.h>

#include "attention.cuh"

namespace kvp {

namespace {

constexpr int kPM = 128;  // query rows per tile
constexpr int kPN = 128;  // keys per block
constexpr int kPD = 128;  // head_dim
constexpr int kPThreads = 128;
constexpr uint32_t kHalf = 16384;  // one 64-element half of a 128-row operand: 128 rows x 128 B
constexpr uint64_t kPWaitNs = 2000000000ull;

struct PrefillArgs {
  CUtensorMap qmap;   // q as (d, head, token, request), box (64, G, 128 / G, 1)
  CUtensorMap kvmap;  // the KV buffer as (d, slot, kv head, K/V x layer), box (64, 16, 1, 1)
  int use_kvmap;
  int kvl_k, kvl_v;
  TableRef T;
  const char* kv_layer;
  size_t kv_bytes, row_bytes;
  __nv_bfloat16* out;  // [B, C, Hq, D]
  const int32_t* q_lens;
  const int32_t* context_lens;
  const int32_t* table_rows;
  int B, C, Hq, Hkv, G, tiles;
  int window, sinks;
  float scale_log2;
  int32_t* err;
};

__device__ __forceinline__ uint64_t umma_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  // tcgen05 shared-memory matrix descriptor: start >> 4, leading and stride
  // byte offsets >> 4, version 1, 128-byte swizzle
  return (uint64_t)((addr & 0x3FFFF) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// kind::f16 instruction descriptor: fp32 accumulate, bf16 A and B, M 128, N 128.
__host__ __device__ constexpr uint32_t umma_idesc(int b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)b_mn_major << 16) | ((uint32_t)(kPN >> 3) << 17) |
         ((uint32_t)(kPM >> 4) << 24);
}

__device__ __forceinline__ void umma_f16(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}

__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])),
      "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])),
      "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])),
      "r"(__float_as_uint(v[11])), "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])),
      "r"(__float_as_uint(v[14])), "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])),
      "r"(__float_as_uint(v[17])), "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])),
      "r"(__float_as_uint(v[20])), "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])),
      "r"(__float_as_uint(v[23])), "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])),
      "r"(__float_as_uint(v[26])), "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])),
      "r"(__float_as_uint(v[29])), "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
      : "memory");
}

// Byte offset of 16-byte chunk c (0..7) of row r in a 128-byte-swizzled operand half.
__device__ __forceinline__ uint32_t sw128(int r, int c) { return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4)); }

__global__ void __launch_bounds__(kPThreads, 2) prefill_tc_kernel(const __grid_constant__ PrefillArgs a) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  __shared__ uint64_t bar_q, bar_kv, bar_mma;
  __shared__ uint32_t s_taddr;
  __shared__ int s_abort;
  unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  unsigned char* sQ = smem;              // [2 halves][128 rows][128 B]
  unsigned char* sK = smem + 2 * kHalf;  // [2 halves][128 keys][128 B]
  unsigned char* sV = smem + 4 * kHalf;
  // P [2 key halves][128 rows][128 B] takes K's place once S = Q K^T is done
  // with it, so that a CTA needs 97 KB and two fit on an SM
  unsigned char* sP = sK;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  volatile int* abort_flag = &s_abort;

  // Tile order: the last tiles of the requests (the most keys) first.
  const int per_tile = a.B * a.Hkv;
  const int tile = a.tiles - 1 - (int)(blockIdx.x / per_tile);
  const int b = (int)(blockIdx.x % per_tile) / a.Hkv, g = (int)(blockIdx.x % per_tile) % a.Hkv;
  const int TT = kPM / a.G;  // query tokens per tile
  const int j0 = tile * TT;
  const int L = a.context_lens[b];
  const int ql = a.q_lens ? a.q_lens[b] : a.C;
  const int row = a.table_rows ? a.table_rows[b] : b;
  const bool valid = ql >= 1 && ql <= a.C && ql <= L && L <= table_capacity(a.T) && row >= 0 && row < a.T.rows_total;
  const int rt = tid / a.G, hh = tid % a.G;  // this thread's query row: token j0 + rt, head hh of the group
  __nv_bfloat16* orow = a.out + (((size_t)b * a.C + j0 + rt) * a.Hq + (size_t)g * a.G + hh) * kPD;
  if (!valid) {
    if (tid == 0 && g == 0 && tile == 0) set_error(a.err, KVP_ERR_BAD_INDEX);
    if (j0 + rt < a.C)
      for (int d = 0; d < kPD; d += 8) *reinterpret_cast<uint4*>(orow + d) = make_uint4(0u, 0u, 0u, 0u);
    return;
  }
  if (j0 >= ql) return;  // no query of this request falls in the tile
  const int jn = min(TT, ql - j0);
  const int p_first = L - ql + j0, p_last = p_first + jn - 1;
  // the union of the tile's spans: the first query reaches furthest back
  const Span u = attend_span(p_last + 1, a.window > 0 ? a.window + (p_last - p_first) : 0, a.sinks);
  const int n_keys = u.se + (p_last + 1 - u.lo);
  const int nblk = (n_keys + kPN - 1) / kPN;
  const bool rv = rt < jn;
  const int pr = p_first + rt;
  const Span sr = attend_span(pr + 1, a.window, a.sinks);

  if (tid == 0) {
    mbar_init(&bar_q, 1);
    mbar_init(&bar_kv, 1);
    mbar_init(&bar_mma, 1);
    s_abort = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 256;" ::"r"(smem_u32(&s_taddr))
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tS = s_taddr, tO = s_taddr + 128;
  const uint32_t lane_base = (uint32_t)(warp * 32) << 16;  // this warp's 32 TMEM lanes = its 32 query rows

  if (tid == 0) {
    mbar_arrive_expect_tx(&bar_q, 2 * kHalf);
    tma_load_4d(sQ, &a.qmap, 0, g * a.G, j0, b, &bar_q);
    tma_load_4d(sQ + kHalf, &a.qmap, 64, g * a.G, j0, b, &bar_q);
  }

  const uint32_t qa = smem_u32(sQ), ka = smem_u32(sK), va = smem_u32(sV), pa = smem_u32(sP);
  const uint32_t id_s = umma_idesc(0), id_o = umma_idesc(1);
  float m_used = -INFINITY, lsum = 0.f;
  uint32_t ph_mma = 0;
  bool issued_unwaited = false;

  for (int blk = 0; blk < nblk; ++blk) {
    // ---- keys o0 .. o0 + 127: one per thread -------------------------------
    const int o0 = blk * kPN, o = o0 + tid;
    const int slot = o < n_keys ? resolve_slot(a.T, row, span_pos(u, o), a.err) : -1;
    const int slot0 = __shfl_sync(0xffffffffu, slot, lane & 16);
    const unsigned okm = __ballot_sync(0xffffffffu, slot >= 0 && slot == slot0 + (lane & 15));
    const unsigned halfm = (lane & 16) ? 0xffff0000u : 0x0000ffffu;
    const bool grp_tma = a.use_kvmap && slot0 >= 0 && (slot0 & 15) == 0 && (okm & halfm) == halfm;
    const int n_tma = __syncthreads_count(grp_tma && (lane & 15) == 0);
    if (tid == 0) mbar_arrive_expect_tx(&bar_kv, (uint32_t)n_tma * 4u * 2048u);
    __syncthreads();
    if (grp_tma && (lane & 15) == 0) {
      const uint32_t off = (uint32_t)(tid >> 4) * 16u * 128u;  // the group's 16 key rows
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        tma_load_4d(sK + h * kHalf + off, &a.kvmap, h * 64, slot0, g, a.kvl_k, &bar_kv);
        tma_load_4d(sV + h * kHalf + off, &a.kvmap, h * 64, slot0, g, a.kvl_v, &bar_kv);
      }
    }
    if (!grp_tma) {  // this key's rows by plain loads, into the same swizzled places (zeros past the end)
      const uint4* ks = slot >= 0 ? reinterpret_cast<const uint4*>(a.kv_layer + (size_t)slot * a.row_bytes +
                                                                   (size_t)g * kPD * 2)
                                  : nullptr;
      const uint4* vs = slot >= 0 ? reinterpret_cast<const uint4*>(reinterpret_cast<const char*>(ks) + a.kv_bytes)
                                  : nullptr;
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        const uint4 kx = ks ? __ldg(ks + c) : make_uint4(0u, 0u, 0u, 0u);
        const uint4 vx = vs ? __ldg(vs + c) : make_uint4(0u, 0u, 0u, 0u);
        *reinterpret_cast<uint4*>(sK + (c >> 3) * kHalf + sw128(tid, c & 7)) = kx;
        *reinterpret_cast<uint4*>(sV + (c >> 3) * kHalf + sw128(tid, c & 7)) = vx;
      }
      fence_proxy_async_smem();
    }
    __syncthreads();
    bool okw = mbar_wait_bounded(&bar_kv, (uint32_t)(blk & 1), abort_flag, a.err, kPWaitNs);
    if (blk == 0) okw = okw && mbar_wait_bounded(&bar_q, 0u, abort_flag, a.err, kPWaitNs);
    if (!okw) *abort_flag = 1;
    __syncthreads();
    if (*abort_flag) break;

    // ---- S = Q K^T ---------------------------------------------------------
    tc_fence_after();
    if (tid == 0) {
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const uint32_t koff = (uint32_t)(ks >> 2) * kHalf + (uint32_t)(ks & 3) * 32u;
        umma_f16(tS, umma_desc(qa + koff, 16, 1024), umma_desc(ka + koff, 16, 1024), id_s, ks > 0);
      }
      umma_commit(&bar_mma);
    }
    issued_unwaited = true;
    if (!mbar_wait_bounded(&bar_mma, ph_mma & 1, abort_flag, a.err, kPWaitNs)) *abort_flag = 1;
    __syncthreads();
    if (*abort_flag) break;
    ++ph_mma;
    issued_unwaited = false;
    tc_fence_after();

    // ---- online softmax of this thread's row ------------------------------
    float s[kPN];
#pragma unroll
    for (int c4 = 0; c4 < 4; ++c4) tmem_ld32(tS + lane_base + c4 * 32, s + c4 * 32);
    float rmax = -INFINITY;
#pragma unroll
    for (int c = 0; c < kPN; ++c) {
      const int oc = o0 + c;
      bool keep = rv && oc < n_keys;
      if (keep) {
        const int t = span_pos(u, oc);
        keep = t <= pr && (t >= sr.lo || t < sr.se);
      }
      s[c] = keep ? s[c] * a.scale_log2 : -INFINITY;
      rmax = fmaxf(rmax, s[c]);
    }
    const bool grow = rmax > m_used + 8.f;  // also when nothing was kept before
    if (__any_sync(0xffffffffu, grow && lsum > 0.f)) {  // rescale O (a warp-wide TMEM read and write)
      const float f = (grow && lsum > 0.f) ? exp2f(m_used - rmax) : 1.f;
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) {
        float ov[32];
        tmem_ld32(tO + lane_base + c4 * 32, ov);
#pragma unroll
        for (int i = 0; i < 32; ++i) ov[i] *= f;
        tmem_st32(tO + lane_base + c4 * 32, ov);
      }
      asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      lsum *= f;
    }
    if (grow) m_used = rmax;
    float psum = 0.f;
#pragma unroll
    for (int c8 = 0; c8 < kPN / 8; ++c8) {
      uint32_t w[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float x0 = s[c8 * 8 + 2 * i], x1 = s[c8 * 8 + 2 * i + 1];
        const float p0 = m_used == -INFINITY ? 0.f : exp2f(x0 - m_used);
        const float p1 = m_used == -INFINITY ? 0.f : exp2f(x1 - m_used);
        w[i] = pack_bf16(p0, p1);
        psum += bf16_lo(w[i]) + bf16_hi(w[i]);
      }
      *reinterpret_cast<uint4*>(sP + (c8 >> 3) * kHalf + sw128(tid, c8 & 7)) = make_uint4(w[0], w[1], w[2], w[3]);
    }
    lsum += psum;
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    // ---- O += P V ----------------------------------------------------------
    if (tid == 0) {
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const uint32_t poff = (uint32_t)(ks >> 2) * kHalf + (uint32_t)(ks & 3) * 32u;
        umma_f16(tO, umma_desc(pa + poff, 16, 1024), umma_desc(va + (uint32_t)ks * 2048u, kHalf, 1024), id_o,
                 (blk > 0 || ks > 0) ? 1u : 0u);
      }
      umma_commit(&bar_mma);
    }
    issued_unwaited = true;
    if (!mbar_wait_bounded(&bar_mma, ph_mma & 1, abort_flag, a.err, kPWaitNs)) *abort_flag = 1;
    __syncthreads();
    if (*abort_flag) break;
    ++ph_mma;
    issued_unwaited = false;
    tc_fence_after();
  }

  if (!*abort_flag) {
    // ---- epilogue: O / l -> bf16 -------------------------------------------
    const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
#pragma unroll
    for (int c4 = 0; c4 < 4; ++c4) {
      float ov[32];
      tmem_ld32(tO + lane_base + c4 * 32, ov);
      if (rv) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint4 w;
          w.x = pack_bf16(ov[8 * q + 0] * inv, ov[8 * q + 1] * inv);
          w.y = pack_bf16(ov[8 * q + 2] * inv, ov[8 * q + 3] * inv);
          w.z = pack_bf16(ov[8 * q + 4] * inv, ov[8 * q + 5] * inv);
          w.w = pack_bf16(ov[8 * q + 6] * inv, ov[8 * q + 7] * inv);
          *reinterpret_cast<uint4*>(orow + c4 * 32 + q * 8) = w;
        }
      }
    }
  } else if (issued_unwaited) {
    // let the MMAs in flight finish (bounded) before their TMEM goes back
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(&bar_mma, ph_mma & 1))
      if (global_timer_ns() - t0 > 100000000ull) break;
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 256;" ::"r"(tS) : "memory");
}

bool encode_qmap(const void* q, int B, int C, int Hq, int G, CUtensorMap* out) {
  static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  static bool looked_up = false;
  if (!looked_up) {
    cudaDriverEntryPointQueryResult qr;
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &qr) ==
            cudaSuccess &&
        qr == cudaDriverEntryPointSuccess)
      encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    looked_up = true;
  }
  if (!encode) return false;
  cuuint64_t dims[4] = {(cuuint64_t)kPD, (cuuint64_t)Hq, (cuuint64_t)C, (cuuint64_t)B};
  cuuint64_t strides[3] = {(cuuint64_t)kPD * 2, (cuuint64_t)Hq * kPD * 2, (cuuint64_t)C * Hq * kPD * 2};
  cuuint32_t box[4] = {64, (cuuint32_t)G, (cuuint32_t)(kPM / G), 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return encode(out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(q), dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

constexpr size_t kPrefillSmem = 6 * kHalf + 1024;

bool prefill_tc_eligible(const kvp_pool* pool, int Hq, int C) {
  if (pool->dtype != KVP_BF16 || pool->head_dim != kPD || Hq % pool->kv_heads) return false;
  const int G = Hq / pool->kv_heads;
  return G >= 1 && G <= kPM && kPM % G == 0 && C >= 1;
}

int launch_prefill_tc(const kvp_pool* pool, int layer, const void* q, int batch, int C, int Hq, const int32_t* q_lens,
                      const TableRef& T, const int32_t* table_rows, const int32_t* context_lens, int window, int sinks,
                      float scale, void* out, cudaStream_t stream) {
  kvp_pool* mp = const_cast<kvp_pool*>(pool);
  PrefillArgs a;
  const int G = Hq / pool->kv_heads;
  if (!encode_qmap(q, batch, C, Hq, G, &a.qmap)) return KVP_ERR_CUDA;
  if (mp->tmap1_state == 0) mp->tmap1_state = tc_encode_tmap(pool, 1, &mp->tmap1) ? 1 : -1;
  a.use_kvmap = mp->tmap1_state == 1;
  if (a.use_kvmap) a.kvmap = mp->tmap1;
  else memset(&a.kvmap, 0, sizeof(a.kvmap));
  a.kvl_k = layer;
  a.kvl_v = pool->num_layers + layer;
  a.T = T;
  a.kv_layer = pool->buf + (size_t)layer * pool->layer_bytes;
  a.kv_bytes = pool->kv_bytes;
  a.row_bytes = pool->row_bytes;
  a.out = static_cast<__nv_bfloat16*>(out);
  a.q_lens = q_lens;
  a.context_lens = context_lens;
  a.table_rows = table_rows;
  a.B = batch;
  a.C = C;
  a.Hq = Hq;
  a.Hkv = pool->kv_heads;
  a.G = G;
  a.tiles = (C + kPM / G - 1) / (kPM / G);
  a.window = window;
  a.sinks = sinks;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.err = pool->err;
  static bool attr = false;
  if (!attr) {
    if (cudaFuncSetAttribute(prefill_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kPrefillSmem) !=
        cudaSuccess)
      return KVP_ERR_CUDA;
    attr = true;
  }
  const long long grid = (long long)a.tiles * batch * pool->kv_heads;
  if (grid <= 0 || grid > 0x7fffffffLL) return KVP_ERR_INVALID_ARG;
  prefill_tc_kernel<<<(unsigned)grid, kPThreads, kPrefillSmem, stream>>>(a);
  return cudaGetLastError() == cudaSuccess ? KVP_OK : KVP_ERR_CUDA;
}

}  // namespace kvp
