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
// How (one CTA of 22 warps per 128-row query tile):
// * A tile is 128 / G consecutive query tokens of one request times the G
//   query heads of one KV head: 128 rows of Q, loaded once by TMA (128-byte
//   swizzle, two 64-element halves of head_dim). The tiles of one request
//   and KV head are adjacent in the grid, so L2 serves their shared K/V.
// * The keys the tile needs (the union of its queries' spans) stream in
//   blocks of 128. A 16-slot group whose slots are contiguous and 16-aligned
//   comes by TMA copies (4 KB of K or V), any other key row is copied by a
//   loader warp into the same layout. With a block table whose page size is
//   a multiple of 16, a 16-aligned group needs one table read. K lies
//   half-major (each half of d is 128 key rows of 128 B, 8-row atoms 1 KB
//   apart: two copies per group), so that S = Q K^T of a block is eight MMAs
//   of N 128; V lies group-major (one copy per group), the B operand of
//   O += P V.
// * A chain of MMAs into one accumulator runs at 60-100 ns per MMA
//   (measured), well below the tensor cores' rate, so the kernel keeps two
//   chains in flight: S(i + 1) = Q K(i + 1)^T (M 128, N 128, K 128, both
//   operands K-major) goes into one of two 128-column TMEM S buffers while
//   O += P(i) V(i) accumulates in the 128-column O, each from its own
//   issuing warp, and the softmax works on S(i) meanwhile. P (bf16, two per
//   32-bit column, keys in order) goes to one of two 64-column TMEM P
//   buffers and is the A operand, read from TMEM, of O += P V (V the
//   MN-major operand in shared memory, one 16-key group per K step).
// * Four softmax threads per query row, each on 32 keys of the block: they
//   read their scores from TMEM (then the S buffer is free for S(i + 2)),
//   agree on the row maximum through shared memory, and keep an online
//   softmax in log2 units. A part that no row of the warp masks (causal,
//   window, sinks, block end) skips the mask; the maximum is taken on
//   unscaled scores and P = 2^(s * scale - m) is one packed fma.rn.f32x2 per
//   pair of scores and one ex2 per score; each part's row sum adds the fp32
//   exponentials (packed add.rn.f32x2), P V their bf16 roundings. O is
//   rescaled (read, scaled, written back in TMEM) only when the row maximum
//   grows by more than 8, so P <= 256 always fits bf16. The epilogue adds
//   the parts' row sums, divides and stores bf16.
// * Warp-specialised pipeline: two K loader warps (even and odd blocks) fill
//   a three-stage K ring and two V loader warps a two-stage V ring, each
//   resolving its own slots; the S issuer, the P V issuer and the softmax
//   hand off through mbarriers.
// * Every wait is bounded (2 s): on timeout the CTA records KVP_ERR_TIMEOUT,
//   issues nothing more, waits (bounded) for what it issued and frees TMEM.
#include <cudaTypedefs.h>

#include "attention.cuh"

namespace kvp {

namespace {

constexpr int kPM = 128;  // query rows per tile
constexpr int kPN = 128;  // keys per block
constexpr int kPD = 128;  // head_dim
// warps: 0 and 1 K loaders (even and odd blocks; 0 also loads Q), 2 and 3 V
// loaders, 4 S issuer, 5 P V issuer, 6..21 softmax (four warps per TMEM lane
// quadrant, each on 32 of a block's 128 keys)
constexpr int kPThreads = 704;
constexpr int kVWarp = 2;
constexpr int kSWarp = 4;
constexpr int kPVWarp = 5;
constexpr int kSoftWarp0 = 6;
constexpr int kParts = 4;  // softmax threads per query row
constexpr int kKS = 3;  // K ring stages
constexpr int kVS = 2;  // V ring stages
constexpr uint32_t kHalf = 16384;  // one 64-element half of a 128-row operand: 128 rows x 128 B
constexpr uint32_t kGroupBytes = 4096;  // K or V of one 16-key group: 2 halves x 16 rows x 128 B
constexpr uint64_t kPWaitNs = 2000000000ull;

struct PrefillArgs {
  CUtensorMap qmap;   // q as (d, head, token, request), box (64, G, 128 / G, 1)
  CUtensorMap kvmap;  // the KV buffer as (d % 64, slot, d / 64, kv head, K/V x layer), box (64, 16, 2, 1, 1)
  CUtensorMap kmap;   // the same view, box (64, 16, 1, 1, 1): one half of d of a 16-slot group
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

// kind::f16 instruction descriptor: fp32 accumulate, bf16 A and B, M 128, N n.
__host__ __device__ constexpr uint32_t umma_idesc(int b_mn_major, int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)b_mn_major << 16) | ((uint32_t)(n >> 3) << 17) |
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

// 16 consecutive fp32 columns of this thread's TMEM lane (no wait).
__device__ __forceinline__ void tmem_ld16_nowait(uint32_t taddr, float* v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// 16 consecutive 32-bit columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}

// D (TMEM) (+)= A (TMEM, K-major, two bf16 per column) * B (shared-memory descriptor).
__device__ __forceinline__ void umma_f16_ts(uint32_t tmem_d, uint32_t tmem_a, uint64_t b, uint32_t idesc,
                                            uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(tmem_d),
      "r"(tmem_a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}

// (d0, d1) = (a0, a1) * (b, b) + (c, c) and (d0, d1) += (a0, a1): Blackwell's
// packed fp32 instructions, one issue for two lanes of work.
__device__ __forceinline__ void fma2_bc(float& d0, float& d1, float a0, float a1, float b, float c) {
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %4};\n\t"
      "mov.b64 rc, {%5, %5};\n\tfma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b), "f"(c));
}
__device__ __forceinline__ void add2(float& d0, float& d1, float a0, float a1) {
  asm("{\n\t.reg .b64 ra, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rd, {%0, %1};\n\t"
      "add.rn.f32x2 rd, rd, ra;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "+f"(d0), "+f"(d1)
      : "f"(a0), "f"(a1));
}

// max(a, b, c) in one instruction (sm_100 and later).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// 2^x by the PTX approximate base-2 exponential (flush-to-zero; 2^-inf = +0).
__device__ __forceinline__ float ex2_ftz(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}


// Byte offset of 16-byte chunk c (0..7) of row r in a 128-byte-swizzled operand half.
__device__ __forceinline__ uint32_t sw128(int r, int c) { return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4)); }

// Barriers and flags of one CTA (static shared memory). Block i uses S and
// P buffer i % 2; the barriers of a buffer complete once per block using it.
struct PrefillBars {
  uint64_t q_full;
  uint64_t k_full[kKS];   // K loaders -> S issuer: K block in K stage s (TMA bytes and thread copies)
  uint64_t k_empty[kKS];  // S issuer (commit) -> K loader: S has read K stage s
  uint64_t v_full[kVS];   // V loaders -> P V issuer: V block in V stage s
  uint64_t v_empty[kVS];  // P V issuer (commit) -> V loader: P V has read V stage s
  uint64_t s_full[2];     // S issuer (commit) -> softmax: S = Q K^T of the block in S buffer b
  uint64_t s_free[2];     // softmax (16 warps) -> S issuer: S buffer b read into registers
  uint64_t p_full[2];     // softmax (16 warps) -> P V issuer: P of the block in P buffer b
  uint64_t pv_done[2];    // P V issuer (commit) -> softmax: O += P V of the block done, P buffer b free
  uint64_t drain;         // both issuers (commit) -> all: everything issued is done
  uint64_t vtail;         // TMA -> V loader: the last block's partial group landed (used once)
  uint64_t xbar[4];       // the four softmax warps of a row quadrant: their partials are in xch
  uint32_t taddr;
  int abort;
  int slots[4][kPN];      // each loader's slots of the block it is loading
  float xch[2][kParts][kPM];  // [block % 2][part][row]: the part's row maximum (the row sum at the end)
};

// Wait for phase ``k`` of ``bar`` (parity k & 1), bounded.
__device__ __forceinline__ bool pwait(uint64_t* bar, int k, volatile int* abort_flag, int32_t* err) {
  return mbar_wait_bounded(bar, (uint32_t)(k & 1), abort_flag, err, kPWaitNs);
}

// 5-D tiled TMA load (coordinates innermost first) completing on ``bar``.
__device__ __forceinline__ void tma_load_5d(void* dst, const void* tmap, int c0, int c1, int c2, int c3, int c4,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5, "
      "%6}], [%7];" ::"r"(smem_u32(dst)),
      "l"(tmap), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4), "r"(smem_u32(bar))
      : "memory");
}

// tx bytes for ``bar``'s current phase, without an arrival.
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t tx) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(tx) : "memory");
}

// Tracing build (-DKVP_PREFILL_TRACE; paged_decode_attention_store_gb300.
// trace_prefill builds it beside the library): every CTA records its entry
// and exit times, SM and key blocks, and one armed CTA the global-timer time
// of each pipeline event of its first kTraceBlocks blocks. The product build
// compiles none of it.
enum PrefillTraceEvent {
  kTrKResolved,  // K loader: the block's slots resolved (before its stage wait)
  kTrKIssued,    // K loader: the block's copies issued
  kTrVResolved,
  kTrVIssued,
  kTrSFull,      // S issuer: K(i) landed
  kTrSIssued,    // S issuer: S(i) issued and committed
  kTrPvV,        // P V issuer: V(i) landed
  kTrPvP,        // P V issuer: P(i) written
  kTrPvIssued,   // P V issuer: P V(i) issued and committed
  kTrSmS,        // softmax (first warp, lane 0): S(i) in TMEM
  kTrSmMax,      // softmax: the row maximum agreed
  kTrSmP,        // softmax: P(i) computed (before waiting for its P buffer)
  kTrSmArrive,   // softmax: P(i) written and handed to the P V issuer
  kTrEvents
};
#ifdef KVP_PREFILL_TRACE
constexpr int kTraceBlocks = 128;
constexpr int kTraceCtas = 4096;
__device__ unsigned long long g_ptrace_ev[kTrEvents][kTraceBlocks];
__device__ unsigned long long g_ptrace_cta[kTraceCtas][4];  // entry, SM, exit, blocks
__device__ int g_ptrace_target = -1;
#define PTRACE(e, i)                                                                \
  do {                                                                              \
    if (traced && (i) < kTraceBlocks) g_ptrace_ev[e][i] = global_timer_ns();        \
  } while (0)
#else
#define PTRACE(e, i) \
  do {               \
  } while (0)
#endif

// The paths of load_rows for a block with a partial or empty groups (the
// last block of a CTA) or groups that are not 16-aligned in one page.
__device__ __forceinline__ bool load_rows_slow(const PrefillArgs& a, unsigned char* dst, const int* slots, unsigned tm,
                                            unsigned tp, int kp, unsigned te, int g, bool is_v, uint64_t* bar,
                                            uint64_t* vtail, int lane, volatile int* abort_flag) {
  const int kvl = is_v ? a.kvl_v : a.kvl_k;
  const uint4 z = make_uint4(0u, 0u, 0u, 0u);
  if ((tm | tp | te) == 0xFFu && !is_v) {  // K with a partial or empty groups: TMA alone
    if (lane == 0) {
      const unsigned tt = tm | tp;
      mbar_arrive_expect_tx(bar, (uint32_t)__popc(tt) * kGroupBytes);
      for (int gi = 0; gi < 8; ++gi) {
        if (!((tt >> gi) & 1)) continue;
        const int s0 = slots[16 * gi];
        tma_load_5d(dst + gi * (kGroupBytes / 2), &a.kmap, 0, s0, 0, g, kvl, bar);
        tma_load_5d(dst + kHalf + gi * (kGroupBytes / 2), &a.kmap, 0, s0, 1, g, kvl, bar);
      }
    }
    __syncwarp();
    return true;
  }
  if ((tm | tp | te) == 0xFFu) {  // V with a partial or empty groups
    const int gp = tp ? __ffs(tp) - 1 : -1;
    if (lane == 0) {
      if (gp >= 0) {
        mbar_arrive_expect_tx(vtail, kGroupBytes);
        tma_load_5d(dst + gp * kGroupBytes, &a.kvmap, 0, slots[16 * gp], 0, g, kvl, vtail);
      }
      mbar_expect_tx(bar, (uint32_t)__popc(tm) * kGroupBytes);
#pragma unroll
      for (int gi = 0; gi < 8; ++gi)
        if ((tm >> gi) & 1) tma_load_5d(dst + gi * kGroupBytes, &a.kvmap, 0, slots[16 * gi], 0, g, kvl, bar);
    }
    for (int gi = 0; gi < 8; ++gi)
      if ((te >> gi) & 1)
        for (int x = lane; x < kGroupBytes / 16; x += 32) reinterpret_cast<uint4*>(dst + gi * kGroupBytes)[x] = z;
    if (gp >= 0) {
      if (!__all_sync(0xffffffffu, pwait(vtail, 0, abort_flag, a.err))) return false;
      // rows kp .. 15 of both halves: 16 B chunk c of row r at h * 2 KB + r * 128 B
      for (int x = kp * 16 + lane; x < 16 * 16; x += 32) {
        const int r = x >> 4, c = x & 15;
        *reinterpret_cast<uint4*>(dst + gp * kGroupBytes + (c >> 3) * (kGroupBytes / 2) + r * 128 + (c & 7) * 16) = z;
      }
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(bar);
    __syncwarp();
    return true;
  }
  const size_t base = is_v ? a.kv_bytes : 0;
  for (int gi = 0; gi < 8; ++gi) {
    if ((tm >> gi) & 1) continue;
    for (int x = lane; x < 16 * 16; x += 32) {
      const int key = 16 * gi + x / 16, c = x % 16;
      const int sl = slots[key];
      uint4 val = z;
      if (sl >= 0)
        val = __ldg(reinterpret_cast<const uint4*>(a.kv_layer + base + (size_t)sl * a.row_bytes +
                                                   (size_t)g * kPD * 2) + c);
      const uint32_t off = is_v ? gi * kGroupBytes + (c >> 3) * (kGroupBytes / 2) + sw128(key & 15, c & 7)
                                : (c >> 3) * kHalf + sw128(key, c & 7);
      *reinterpret_cast<uint4*>(dst + off) = val;
    }
  }
  // the thread copies' writes are visible to the tensor cores' (async proxy) reads
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) mbar_arrive_expect_tx(bar, (uint32_t)__popc(tm) * kGroupBytes);
  __syncwarp();
  if (is_v) {
    if (lane < 8 && ((tm >> lane) & 1))
      tma_load_5d(dst + lane * kGroupBytes, &a.kvmap, 0, slots[16 * lane], 0, g, kvl, bar);
  } else if (lane < 16 && ((tm >> (lane & 7)) & 1)) {  // lane = group + 8 * half
    const int gi = lane & 7, h = lane >> 3;
    tma_load_5d(dst + h * kHalf + gi * (kGroupBytes / 2), &a.kmap, 0, slots[16 * gi], h, g, kvl, bar);
  }
  __syncwarp();
  return true;
}

// The loader warp fills one 128-key operand; ``bar`` (count 1) gets the
// arrival and the TMA byte count. Both layouts use the 128-byte swizzle with
// 8-row atoms of 1 KB.
//  - K (``is_v`` false), half-major: half h of d at h * 16 KB, key row k at
//    + k * 128 B, so the 128 keys of a half are 16 evenly spaced atoms (the
//    N 128 B operand of S = Q K^T). A group is two copies (one per half).
//  - V, group-major: group gi (keys 16 gi .. 16 gi + 15) at gi * 4 KB, its
//    half h at + h * 2 KB, key row r at + r * 128 B (the MN-major B operand
//    of O += P V, one group per 16-key K step). A group is one copy.
// Groups in ``tm`` go by TMA from the 16 slots starting at slots[16 gi]. When
// the other groups are all in ``tp`` (the block's last group with keys, whose
// first ``kp`` keys are in the span and whose 16 slots lie in one page) or
// ``te`` (no key in the span), they are handled without thread copies: K's
// partial group goes by TMA whole and its empty groups stay as they are (the
// scores of keys past the span are masked); V's empty groups are zeroed, and
// its partial group goes by TMA on ``vtail`` and has its rows from kp on
// zeroed once it has landed (P is 0 there, and 0 times what the page holds
// past the span must stay 0). Otherwise the groups outside ``tm`` are copied
// by the threads from ``slots`` (zeros for slots < 0). Returns false when a
// wait gave up.
__device__ __forceinline__ bool load_rows(const PrefillArgs& a, unsigned char* dst, const int* slots, unsigned tm,
                                          unsigned tp, int kp, unsigned te, int g, bool is_v, uint64_t* bar,
                                          uint64_t* vtail, int lane, volatile int* abort_flag) {
  const int kvl = is_v ? a.kvl_v : a.kvl_k;
  if (tm == 0xFFu) {  // every group full, by TMA (the common case): one lane issues all copies
    if (lane == 0) {
      mbar_arrive_expect_tx(bar, 8u * kGroupBytes);
      if (is_v) {
#pragma unroll
        for (int gi = 0; gi < 8; ++gi) tma_load_5d(dst + gi * kGroupBytes, &a.kvmap, 0, slots[16 * gi], 0, g, kvl, bar);
      } else {
#pragma unroll
        for (int gi = 0; gi < 8; ++gi) {
          const int s0 = slots[16 * gi];
          tma_load_5d(dst + gi * (kGroupBytes / 2), &a.kmap, 0, s0, 0, g, kvl, bar);
          tma_load_5d(dst + kHalf + gi * (kGroupBytes / 2), &a.kmap, 0, s0, 1, g, kvl, bar);
        }
      }
    }
    __syncwarp();
    return true;
  }
  return load_rows_slow(a, dst, slots, tm, tp, kp, te, g, is_v, bar, vtail, lane, abort_flag);
}


// Warp roles: 0 and 1 load K blocks (even, odd) into a three-stage ring, 0
// loads Q first; 2 and 3 load V blocks into a two-stage ring; 4 issues the
// S MMAs and 5 the P V MMAs (lane 0 each); 6..21 run the softmax and the
// epilogue, four threads per query row (TMEM lane quadrant = warp % 4, part
// = (warp - 6) / 4: keys 32 part .. 32 part + 31 of each block).
__global__ void __launch_bounds__(kPThreads, 1) prefill_tc_kernel(const __grid_constant__ PrefillArgs a) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  __shared__ PrefillBars sb;
  unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  unsigned char* sQ = smem;                  // Q: [2 halves][128 rows][128 B]
  unsigned char* sK = smem + 2 * kHalf;      // K stage s at s * 2 kHalf
  unsigned char* sV = sK + kKS * 2 * kHalf;  // V stage s at s * 2 kHalf
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  volatile int* abort_flag = &sb.abort;
#ifdef KVP_PREFILL_TRACE
  const unsigned long long t_entry = global_timer_ns();
  const bool traced = (int)blockIdx.x == g_ptrace_target;
#endif

  // CTA order: request and KV head major, the tile with the most keys first,
  // so that the tiles reading the same K/V run side by side (L2 serves all
  // but the first of them).
  const int tile = a.tiles - 1 - (int)(blockIdx.x % a.tiles);
  const int bg = (int)(blockIdx.x / a.tiles);
  const int b = bg / a.Hkv, g = bg % a.Hkv;
  const int TT = kPM / a.G;  // query tokens per tile
  const int j0 = tile * TT;  // first query token of the tile
  const int L = a.context_lens[b];
  const int ql = a.q_lens ? a.q_lens[b] : a.C;
  const int row = a.table_rows ? a.table_rows[b] : b;
  const bool valid = ql >= 1 && ql <= a.C && ql <= L && L <= table_capacity(a.T) && row >= 0 && row < a.T.rows_total;
  // softmax threads: query row r = 32 * (warp % 4) + lane (token j0 + r / G,
  // head r % G of the group), keys 32 part .. 32 part + 31 of each block
  const bool soft = warp >= kSoftWarp0;
  const int part = soft ? (warp - kSoftWarp0) >> 2 : 0;
  const int r = 32 * (warp & 3) + lane;
  const int rt = r / a.G, hh = r % a.G;
  __nv_bfloat16* orow = a.out + (((size_t)b * a.C + j0 + rt) * a.Hq + (size_t)g * a.G + hh) * kPD + 32 * part;
  if (!valid) {
    if (tid == 0 && g == 0 && tile == 0) set_error(a.err, KVP_ERR_BAD_INDEX);
    if (soft && j0 + rt < a.C)
      for (int d = 0; d < 32; d += 8) *reinterpret_cast<uint4*>(orow + d) = make_uint4(0u, 0u, 0u, 0u);
    return;
  }
  if (j0 >= ql) return;  // no query of this request falls in the tile
  const int jn = min(TT, ql - j0);  // query tokens of the tile
  const int p_first = L - ql + j0, p_last = p_first + jn - 1;
  // the union of the tile's spans: the first query reaches furthest back
  const Span u = attend_span(p_last + 1, a.window > 0 ? a.window + (p_last - p_first) : 0, a.sinks);
  const int n_keys = u.se + (p_last + 1 - u.lo);
  const int nblk = (n_keys + kPN - 1) / kPN;
#ifdef KVP_PREFILL_TRACE
  if (tid == 0 && blockIdx.x < kTraceCtas) {
    unsigned smid;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
    g_ptrace_cta[blockIdx.x][0] = t_entry;
    g_ptrace_cta[blockIdx.x][1] = smid;
    g_ptrace_cta[blockIdx.x][3] = (unsigned long long)nblk;
  }
#endif

  if (tid == 0) {
    mbar_init(&sb.q_full, 1);
    for (int s2 = 0; s2 < kKS; ++s2) {
      mbar_init(&sb.k_full[s2], 1);
      mbar_init(&sb.k_empty[s2], 1);
    }
    for (int s2 = 0; s2 < kVS; ++s2) {
      mbar_init(&sb.v_full[s2], 1);
      mbar_init(&sb.v_empty[s2], 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(&sb.s_full[x], 1);
      mbar_init(&sb.s_free[x], 4 * kParts);
      mbar_init(&sb.p_full[x], 4 * kParts);
      mbar_init(&sb.pv_done[x], 1);
    }
    for (int qd = 0; qd < 4; ++qd) mbar_init(&sb.xbar[qd], kParts);
    mbar_init(&sb.drain, 2);
    mbar_init(&sb.vtail, 1);
    sb.abort = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(smem_u32(&sb.taddr))
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // TMEM: S buffers at columns 0 and 128, O at 256, P buffers (bf16, two
  // keys per column) at 384 and 448
  const uint32_t tbase = sb.taddr;
  const uint32_t tO = tbase + 256u;

  if (warp < kSWarp) {
    // ======================= loaders ==========================================
    // Warps 0 and 1 load K(i) (i even, odd) once S(i - kKS) has read its
    // stage, warp 0 Q first; warps 2 and 3 load V(i) once P V(i - kVS) has.
    // Each resolves its own slots; one loader's table reads overlap the
    // other's copies.
    const bool is_v = warp >= kVWarp;
    const int NS = is_v ? kVS : kKS;
    const int par = warp & 1;
    if (warp == 0 && lane == 0) {
      mbar_arrive_expect_tx(&sb.q_full, 2u * kHalf);
      tma_load_4d(sQ, &a.qmap, 0, g * a.G, j0, b, &sb.q_full);
      tma_load_4d(sQ + kHalf, &a.qmap, 64, g * a.G, j0, b, &sb.q_full);
    }
    int* slots = sb.slots[warp];
    // A block table whose page size is a multiple of 16 keeps every
    // 16-aligned run of 16 positions in one page: such a group needs one
    // table read (lane gi reads group gi's) and goes by TMA.
    const bool group_reads = a.use_kvmap && !a.T.raw && (a.T.page_size & 15) == 0;
    for (int i = par; i < nblk; i += 2) {
      const int st = i % NS;
      const int o0 = i * kPN;
      unsigned tm = 0, tp = 0, te = 0;
      int kp = 0;
      bool whole = false;  // every group of the block full, partial or empty by its one read
      if (group_reads) {
        // lane gi < 8: group gi is full (its 16 keys in the span, in one
        // segment, 16-aligned positions), partial (the span ends inside it,
        // in the window segment, aligned) or empty (past the span)
        const int og = o0 + 16 * lane;
        int s0 = -1;
        bool empty = false;
        if (lane < 8) {
          if (og >= n_keys) {
            empty = true;
          } else if (og >= u.se || og + 15 < u.se) {
            const int p = span_pos(u, og);
            if ((p & 15) == 0) s0 = resolve_slot(a.T, row, p, a.err);
          }
        }
        const unsigned full = __ballot_sync(0xffffffffu, s0 >= 0 && og + 15 < n_keys) & 0xFFu;
        tp = __ballot_sync(0xffffffffu, s0 >= 0 && og + 15 >= n_keys) & 0xFFu;
        te = __ballot_sync(0xffffffffu, empty) & 0xFFu;
        whole = (full | tp | te) == 0xFFu;
        __syncwarp();  // this warp's previous copies have read the slot list
        if (whole && lane < 8 && s0 >= 0) slots[16 * lane] = s0;
        if (whole) {
          tm = full;
          kp = tp ? n_keys - (o0 + 16 * (__ffs(tp) - 1)) : 0;
        } else {
          tp = te = 0;
        }
      }
      if (!whole) {
        // lane l resolves keys 4l .. 4l+3 (four independent table reads);
        // group gi (lanes 4gi .. 4gi+3) goes by TMA when its 16 slots are
        // contiguous and 16-aligned
        int sl[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int o = o0 + 4 * lane + k;
          sl[k] = o < n_keys ? resolve_slot(a.T, row, span_pos(u, o), a.err) : -1;
        }
        __syncwarp();  // this warp's previous copies have read the slot list
#pragma unroll
        for (int k = 0; k < 4; ++k) slots[4 * lane + k] = sl[k];
        const int g0 = __shfl_sync(0xffffffffu, sl[0], lane & ~3);
        const bool mine = a.use_kvmap && sl[0] >= 0 && sl[1] == sl[0] + 1 && sl[2] == sl[0] + 2 &&
                          sl[3] == sl[0] + 3 && sl[0] == g0 + 4 * (lane & 3) && (g0 & 15) == 0;
        const unsigned okb = __ballot_sync(0xffffffffu, mine);
#pragma unroll
        for (int gi = 0; gi < 8; ++gi)
          if (((okb >> (4 * gi)) & 0xFu) == 0xFu) tm |= 1u << gi;
      }
      __syncwarp();
      if (lane == 0) PTRACE(is_v ? kTrVResolved : kTrKResolved, i);
      if (i >= NS && !__all_sync(0xffffffffu, pwait(is_v ? &sb.v_empty[st] : &sb.k_empty[st], (i - NS) / NS,
                                                    abort_flag, a.err)))
        break;
      if (!load_rows(a, (is_v ? sV : sK) + st * 2 * kHalf, slots, tm, tp, kp, te, g, is_v,
                     is_v ? &sb.v_full[st] : &sb.k_full[st], &sb.vtail, lane, abort_flag))
        break;
      if (lane == 0) PTRACE(is_v ? kTrVIssued : kTrKIssued, i);
    }
  } else if (warp == kSWarp) {
    // ======================= S issuer ==========================================
    // S(i) = Q K(i)^T into S buffer i % 2: eight N 128 MMAs (one per 16-wide
    // K step of d), column c holding key c of the block. It needs K(i) and the
    // softmax's read of S(i - 2), so it runs while the softmax works on
    // S(i - 1). The whole warp walks the schedule; lane 0 issues.
    const bool issuer = lane == 0;
    const uint32_t id_n128 = umma_idesc(0, kPN);
    const uint64_t dq = umma_desc(smem_u32(sQ), 16, 1024);
    const uint64_t dk0 = umma_desc(smem_u32(sK), 16, 1024);
    bool ok = __all_sync(0xffffffffu, pwait(&sb.q_full, 0, abort_flag, a.err));
    for (int i = 0; ok && i < nblk; ++i) {
      const int ks = i % kKS, sbuf = i & 1;
      ok = __all_sync(0xffffffffu, pwait(&sb.k_full[ks], i / kKS, abort_flag, a.err));
      if (lane == 0) PTRACE(kTrSFull, i);
      if (ok && i >= 2) ok = __all_sync(0xffffffffu, pwait(&sb.s_free[sbuf], (i - 2) >> 1, abort_flag, a.err));
      if (!ok) break;
      tc_fence_after();
      const uint64_t dk = dk0 + (uint64_t)((ks * 2 * kHalf) >> 4);
      if (issuer) {
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint64_t off = (uint64_t)((((kk >> 2) * kHalf) + (kk & 3) * 32) >> 4);
          umma_f16(tbase + 128u * (uint32_t)sbuf, dq + off, dk + off, id_n128, kk > 0);
        }
        umma_commit(&sb.s_full[sbuf]);
        umma_commit(&sb.k_empty[ks]);
        PTRACE(kTrSIssued, i);
      }
      __syncwarp();
    }
    if (issuer) umma_commit(&sb.drain);  // arrives once everything this warp issued is done
    __syncwarp();
  } else if (warp == kPVWarp) {
    // ======================= P V issuer ========================================
    // O += P(i) V(i): P from TMEM (8 columns per 16 keys), V group m the
    // MN-major B operand of K step m (halves of d 2 KB apart, 8-key atoms 1 KB).
    const bool issuer = lane == 0;
    const uint32_t id_o = umma_idesc(1, kPN);
    const uint64_t dv0 = umma_desc(smem_u32(sV), kGroupBytes / 2, 1024);
    bool ok = true;
    for (int i = 0; ok && i < nblk; ++i) {
      const int vs = i % kVS, pbuf = i & 1;
      ok = __all_sync(0xffffffffu, pwait(&sb.v_full[vs], i / kVS, abort_flag, a.err));
      if (lane == 0) PTRACE(kTrPvV, i);
      if (ok) ok = __all_sync(0xffffffffu, pwait(&sb.p_full[pbuf], i >> 1, abort_flag, a.err));
      if (lane == 0) PTRACE(kTrPvP, i);
      if (!ok) break;
      tc_fence_after();
      const uint64_t dv = dv0 + (uint64_t)((vs * 2 * kHalf) >> 4);
      const uint32_t tP = tbase + 384u + 64u * (uint32_t)pbuf;
      if (issuer) {
#pragma unroll
        for (int m = 0; m < 8; ++m)
          umma_f16_ts(tO, tP + (uint32_t)m * 8u, dv + (uint64_t)((m * kGroupBytes) >> 4), id_o,
                      (i > 0 || m > 0) ? 1u : 0u);
        umma_commit(&sb.pv_done[pbuf]);
        umma_commit(&sb.v_empty[vs]);
        PTRACE(kTrPvIssued, i);
      }
      __syncwarp();
    }
    if (issuer) umma_commit(&sb.drain);
    __syncwarp();
  } else {
    // ======================= softmax warps =====================================
    // Four threads per query row, each on 32 of a block's keys. They read
    // their scores (then free the S buffer for S(i + 2)), agree on the row
    // maximum through xch (an mbarrier per quadrant, bounded wait), write P
    // of their keys into P buffer i % 2 once P V(i - 2) has read it, and keep
    // their part of the row sum, added at the end. O is rescaled (each
    // thread its 32 columns) only when the row maximum grows by more than 8.
    const bool rv = rt < jn;
    const int pr = p_first + rt;
    const Span sr0 = attend_span(pr + 1, a.window, a.sinks);
    // In key offsets of the tile's span u: the row's sink rows are offsets
    // [0, sr.se) (when u keeps a sink segment its width is the row's; when it
    // does not, u starts at position 0 and offsets are positions), and its
    // window [sr.lo, pr] starts at or after u.lo. Rows past the chunk keep nothing.
    const Span sr = rv ? sr0 : Span{0, 0};
    const int wb0 = rv ? u.se + (sr.lo - u.lo) : 1 << 30, we0 = rv ? u.se + (pr - u.lo) : -1;
    const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
    const uint32_t tOp = tO + lane_base + 32u * (uint32_t)part;
    uint64_t* xbar = &sb.xbar[warp & 3];
    // hand this thread's partial to the row's other parts (phase k) and
    // combine the four with ``op``
    auto exchange = [&](float v, int k, bool use_max, float& res) -> bool {
      volatile float* xc = &sb.xch[k & 1][0][0];
      xc[part * kPM + r] = v;
      __threadfence_block();
      __syncwarp();
      if (lane == 0) mbar_arrive(xbar);
      if (!__all_sync(0xffffffffu, pwait(xbar, k, abort_flag, a.err))) return false;
      const float v0 = xc[r], v1 = xc[kPM + r], v2 = xc[2 * kPM + r], v3 = xc[3 * kPM + r];
      res = use_max ? fmaxf(fmaxf(v0, v1), fmaxf(v2, v3)) : (v0 + v1) + (v2 + v3);
      return true;
    };
    const float sl2 = a.scale_log2;
    float m_used = -INFINITY, lsum = 0.f;  // m in scaled log2 units; lsum over this part's keys
    bool ok = true;
    for (int i = 0; i < nblk; ++i) {
      const int sbuf = i & 1;
      ok = __all_sync(0xffffffffu, pwait(&sb.s_full[sbuf], i >> 1, abort_flag, a.err));
      if (!ok) break;
      if (lane == 0 && warp == kSoftWarp0) PTRACE(kTrSmS, i);
      tc_fence_after();
      // the part's 32 scores, read from TMEM once; then S buffer sbuf is free
      float sv[32];
      const uint32_t tS = tbase + 128u * (uint32_t)sbuf + lane_base + 32u * (uint32_t)part;
      tmem_ld16_nowait(tS, sv);
      tmem_ld16_nowait(tS + 16, sv + 16);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sb.s_free[sbuf]);
      // The row attends key offsets [0, ea) (its sink rows) and [wb, we] (its
      // window), relative to this part's first key; column c of the part is key c.
      const int o0 = i * kPN + 32 * part;
      const int ea = sr.se - o0, wb = wb0 - o0, we = we0 - o0;
      if (!__all_sync(0xffffffffu, wb <= 0 && we >= 31)) {  // some row of the warp masks
#pragma unroll
        for (int c = 0; c < 32; ++c)
          if (!(c < ea || (c >= wb && c <= we))) sv[c] = -INFINITY;
      }
      // the part's maximum on unscaled scores (scale > 0)
      float mx[4];
#pragma unroll
      for (int t = 0; t < 4; ++t)
        mx[t] = fmax3(fmax3(sv[8 * t], sv[8 * t + 1], sv[8 * t + 2]), fmax3(sv[8 * t + 3], sv[8 * t + 4], sv[8 * t + 5]),
                      fmaxf(sv[8 * t + 6], sv[8 * t + 7]));
      float rmax;
      if (!(ok = exchange(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * sl2, i, true, rmax))) break;
      if (lane == 0 && warp == kSoftWarp0) PTRACE(kTrSmMax, i);
      const bool grow = rmax > m_used + 8.f;  // also when nothing was kept before
      const bool scale_o = grow && m_used > -INFINITY;  // O and lsum hold kept keys
      const float f = scale_o ? exp2f(m_used - rmax) : 1.f;
      if (grow) m_used = rmax;
      const float msub = m_used == -INFINITY ? 0.f : m_used;  // masked scores give 2^-inf = 0 either way
      // P of the part's keys, in order, two per 32-bit column, into P buffer
      // sbuf (columns 16 part .. 16 part + 15) once P V(i - 2) has read it
      uint32_t w[16];
      float ps0 = 0.f, ps1 = 0.f;  // the part's row sum, two lanes of a packed add
#pragma unroll
      for (int x = 0; x < 16; ++x) {
        float x0, x1;
        fma2_bc(x0, x1, sv[2 * x], sv[2 * x + 1], sl2, -msub);
        const float p0 = ex2_ftz(x0), p1 = ex2_ftz(x1);
        w[x] = pack_bf16(p0, p1);
        add2(ps0, ps1, p0, p1);
      }
      if (lane == 0 && warp == kSoftWarp0) PTRACE(kTrSmP, i);
      if (i >= 2) {
        ok = __all_sync(0xffffffffu, pwait(&sb.pv_done[sbuf], (i - 2) >> 1, abort_flag, a.err));
        if (!ok) break;
        tc_fence_after();
      }
      tmem_st16(tbase + 384u + 64u * (uint32_t)sbuf + lane_base + 16u * (uint32_t)part, w);
      lsum = lsum * f + (ps0 + ps1);
      if (__any_sync(0xffffffffu, scale_o)) {
        // O holds blocks < i in the old maximum: rescale this part's columns
        // once P V(i - 1) is in (P V(i) waits for this block's P)
        ok = __all_sync(0xffffffffu, pwait(&sb.pv_done[(i - 1) & 1], (i - 1) >> 1, abort_flag, a.err));
        if (!ok) break;
        tc_fence_after();
        float ov[32];
        tmem_ld32(tOp, ov);
#pragma unroll
        for (int x = 0; x < 32; ++x) ov[x] *= f;
        tmem_st32(tOp, ov);
      }
      asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sb.p_full[sbuf]);
      if (lane == 0 && warp == kSoftWarp0) PTRACE(kTrSmArrive, i);
    }
    // ---- epilogue: O / l -> bf16 (this part's 32 columns), once the last P V is in O
    float tot = 0.f;
    if (ok) ok = __all_sync(0xffffffffu, pwait(&sb.pv_done[(nblk - 1) & 1], (nblk - 1) >> 1, abort_flag, a.err));
    if (ok) ok = exchange(lsum, nblk, false, tot);
    if (ok) {
      tc_fence_after();
      const float inv = tot > 0.f ? 1.f / tot : 0.f;
      float ov[32];
      tmem_ld32(tOp, ov);
      if (rv) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint4 w;
          w.x = pack_bf16(ov[8 * q + 0] * inv, ov[8 * q + 1] * inv);
          w.y = pack_bf16(ov[8 * q + 2] * inv, ov[8 * q + 3] * inv);
          w.z = pack_bf16(ov[8 * q + 4] * inv, ov[8 * q + 5] * inv);
          w.w = pack_bf16(ov[8 * q + 6] * inv, ov[8 * q + 7] * inv);
          *reinterpret_cast<uint4*>(orow + q * 8) = w;
        }
      }
    }
  }
  // Everything the issuers issued is done (bounded) before TMEM goes back.
  {
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(&sb.drain, 0u))
      if (global_timer_ns() - t0 > 2 * kPWaitNs) {
        set_error(a.err, KVP_ERR_TIMEOUT);
        break;
      }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tbase) : "memory");
#ifdef KVP_PREFILL_TRACE
  if (tid == 0 && blockIdx.x < kTraceCtas) g_ptrace_cta[blockIdx.x][2] = global_timer_ns();
#endif
}

PFN_cuTensorMapEncodeTiled_v12000 tmap_encoder() {
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
  return encode;
}

// The K/V buffer as (d % 64, slot, d / 64, kv head, K/V x layer): one box
// (64, 16, halves, 1, 1) is a 16-slot group of one head with ``halves`` (2:
// both, 1: one) halves of d.
bool encode_kvmap(const kvp_pool* pool, int halves, CUtensorMap* out) {
  const auto encode = tmap_encoder();
  if (!encode || pool->dtype != KVP_BF16 || pool->head_dim != kPD) return false;
  cuuint64_t dims[5] = {64, (cuuint64_t)pool->num_slots, 2, (cuuint64_t)pool->kv_heads,
                        (cuuint64_t)(2 * pool->num_layers)};
  cuuint64_t strides[4] = {(cuuint64_t)pool->row_bytes, 128, (cuuint64_t)kPD * 2, (cuuint64_t)pool->layer_bytes};
  cuuint32_t box[5] = {64, 16, (cuuint32_t)halves, 1, 1};
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  return encode(out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, pool->buf, dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_qmap(const void* q, int B, int C, int Hq, int G, CUtensorMap* out) {
  const auto encode = tmap_encoder();
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

#ifdef KVP_PREFILL_TRACE
// Tracing build only: arm CTA ``cta`` for the per-block events (-1: none).
extern "C" int kvp_prefill_trace_arm(int cta) {
  return cudaMemcpyToSymbol(g_ptrace_target, &cta, sizeof(int)) == cudaSuccess ? KVP_OK : KVP_ERR_CUDA;
}

// Tracing build only: copy the records out. ``events`` gets kTrEvents x
// kTraceBlocks global-timer times (ns) of the armed CTA, ``ctas`` kTraceCtas x 4
// (entry ns, SM, exit ns, key blocks) of every CTA; ``dims`` gets kTrEvents,
// kTraceBlocks and kTraceCtas. Synchronous.
extern "C" int kvp_prefill_trace_read(unsigned long long* events, unsigned long long* ctas, int32_t* dims) {
  if (!events || !ctas || !dims) return KVP_ERR_INVALID_ARG;
  dims[0] = kTrEvents;
  dims[1] = kTraceBlocks;
  dims[2] = kTraceCtas;
  if (cudaMemcpyFromSymbol(events, g_ptrace_ev, sizeof(g_ptrace_ev)) != cudaSuccess) return KVP_ERR_CUDA;
  if (cudaMemcpyFromSymbol(ctas, g_ptrace_cta, sizeof(g_ptrace_cta)) != cudaSuccess) return KVP_ERR_CUDA;
  return KVP_OK;
}
#endif

constexpr size_t kPrefillSmem = (2 + 2 * kKS + 2 * kVS) * kHalf + 1024;  // Q, the K and V rings

bool prefill_tc_eligible(const kvp_pool* pool, int Hq, int C, float scale) {
  // the row maximum is taken on unscaled scores, which needs scale > 0
  if (!(scale > 0.f) || pool->dtype != KVP_BF16 || pool->head_dim != kPD || Hq % pool->kv_heads) return false;
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
  if (mp->tmap1_state == 0)
    mp->tmap1_state = encode_kvmap(pool, 2, &mp->tmap1) && encode_kvmap(pool, 1, &mp->tmap2) ? 1 : -1;
  a.use_kvmap = mp->tmap1_state == 1;
  if (a.use_kvmap) {
    a.kvmap = mp->tmap1;
    a.kmap = mp->tmap2;
  } else {
    memset(&a.kvmap, 0, sizeof(a.kvmap));
    memset(&a.kmap, 0, sizeof(a.kmap));
  }
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
