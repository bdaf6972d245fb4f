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
// How (one CTA of eleven warps per pair of 128-row query tiles):
// * A tile is 128 / G consecutive query tokens of one request times the G
//   query heads of one KV head: 128 rows of Q, loaded once by TMA (128-byte
//   swizzle, two 64-element halves of head_dim). A CTA takes two adjacent
//   tiles (A and B) of the same request and KV head, so every K/V block it
//   loads serves 256 query rows.
// * The keys the pair needs (the union of its queries' spans) stream in
//   blocks of 128. A 16-slot group whose slots are contiguous and 16-aligned
//   comes by TMA copies (4 KB of K or V), any other key row is copied by the
//   loader warp into the same layout. K lies half-major (each half of d is
//   128 key rows of 128 B, 8-row atoms 1 KB apart: two copies per group), so
//   that S = Q K^T of a block is eight MMAs of N 128; V lies group-major
//   (one copy per group), the B operand of O += P V.
// * The tensor cores take the same time per MMA instruction for any N up to
//   256 (measured), so the kernel keeps N large: S_X = Q_X K^T (M 128, N 128,
//   K 128, both operands K-major) accumulates in the tile's 128-column TMEM
//   S buffer, column c holding key c of the block. Each softmax thread owns
//   one query row: it reads its 128 scores from TMEM (one wait for all) and
//   keeps an online softmax in log2 units. A block that no row of the warp
//   masks (causal, window, sinks, block end) skips the mask;
//   the row maximum is taken on unscaled scores and P = 2^(s * scale - m) is
//   one FMA and one ex2 per score. O is rescaled (read, scaled, written back
//   in TMEM) only when the row maximum grows by more than 8, so P <= 256
//   always fits bf16 (numerator and denominator use the same m; the row sum
//   adds the fp32 exponentials, P V their bf16 roundings).
// * P (bf16, two per 32-bit column, keys in order) is written back into the
//   first 64 columns of S_X and is the A operand, read from TMEM, of O += P V
//   (V the MN-major operand in shared memory, one 16-key group per K step).
//   The epilogue divides by the row sum and stores bf16.
// * Warp-specialised pipeline: two loader warps fill a three-stage K ring
//   and a two-stage V ring (a K stage is free once both tiles' S have read
//   it, a V stage once both P V have), each resolving its own slots; an MMA
//   warp per tile issues S_X(0), then per block i: P_X(i) V and S_X(i + 1)
//   (one issuing thread cannot keep the tensor core busy: measured); two
//   groups of four softmax warps turn each tile's scores into P. S_X(i + 1)
//   overwrites P_X(i), so it is issued once P_X(i) V is done. mbarriers carry
//   every hand-off.
// * The softmax is bound by instruction issue: the scale-and-shift of a pair
//   of scores is one packed fma.rn.f32x2, their row sum one packed
//   add.rn.f32x2 (of the fp32 exponentials, before the bf16 rounding of P).
// * Every wait is bounded (2 s): on timeout the CTA records KVP_ERR_TIMEOUT,
//   issues nothing more, waits (bounded) for what it issued and frees TMEM.
#include <cudaTypedefs.h>

#include "attention.cuh"

namespace kvp {

namespace {

constexpr int kPM = 128;  // query rows per tile
constexpr int kPN = 128;  // keys per block
constexpr int kPD = 128;  // head_dim
constexpr int kPThreads = 384;  // warps: K loader, MMA (tile A), 4 softmax (tile A), 4 softmax (tile B), V loader, MMA (tile B)
constexpr int kVWarp = 10;
constexpr int kMmaWarpB = 11;
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

// 2^x by the PTX approximate base-2 exponential (flush-to-zero; 2^-inf = +0).
__device__ __forceinline__ float ex2_ftz(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}


// Byte offset of 16-byte chunk c (0..7) of row r in a 128-byte-swizzled operand half.
__device__ __forceinline__ uint32_t sw128(int r, int c) { return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4)); }

// Barriers and flags of one CTA (static shared memory). Per-tile barriers
// are indexed by the tile (0: A, 1: B) and complete once per key block.
struct PrefillBars {
  uint64_t q_full;
  uint64_t k_full[kKS];   // loader -> MMA: K block in K stage s (TMA bytes and thread copies)
  uint64_t k_empty[kKS];  // MMA (one commit per tile) -> loader: both tiles' S have read K stage s
  uint64_t v_full[kVS];   // loader -> MMA: V block in V stage s
  uint64_t v_empty[kVS];  // MMA (one commit per tile) -> loader: both tiles' P V have read V stage s
  uint64_t s_full[2];     // MMA -> softmax of tile X: S_X = Q_X K^T of the block in TMEM
  uint64_t p_full[2];     // softmax of tile X (4 warps) -> MMA: P_X of the block in TMEM
  uint64_t pv_done[2];    // MMA -> all: O_X += P_X V of the block done (S_X's columns free again)
  uint64_t drain;         // MMA (one commit per tile) -> all: everything issued is done
  uint32_t taddr;
  int abort;
  int slots[2][kPN];      // the K and the V loader's slots of the block being loaded
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

// The loader warp fills one 128-key operand from ``slots``: 16-slot groups
// flagged in ``tm`` by TMA copies, the others by plain 16-byte copies (zeros
// for slots < 0); ``bar`` (count 1) gets the arrival and the TMA byte count.
// Both layouts use the 128-byte swizzle with 8-row atoms of 1 KB.
//  - K (``is_v`` false), half-major: half h of d at h * 16 KB, key row k at
//    + k * 128 B, so the 128 keys of a half are 16 evenly spaced atoms (the
//    N 128 B operand of S = Q K^T). A group is two copies (one per half).
//  - V, group-major: group gi (keys 16 gi .. 16 gi + 15) at gi * 4 KB, its
//    half h at + h * 2 KB, key row r at + r * 128 B (the MN-major B operand
//    of O += P V, one group per 16-key K step). A group is one copy.
__device__ __forceinline__ void load_rows(const PrefillArgs& a, unsigned char* dst, const int* slots, unsigned tm,
                                          int g, bool is_v, uint64_t* bar, int lane) {
  const size_t base = is_v ? a.kv_bytes : 0;
  const int kvl = is_v ? a.kvl_v : a.kvl_k;
  for (int gi = 0; gi < 8; ++gi) {
    if ((tm >> gi) & 1) continue;
    for (int x = lane; x < 16 * 16; x += 32) {
      const int key = 16 * gi + x / 16, c = x % 16;
      const int sl = slots[key];
      uint4 val = make_uint4(0u, 0u, 0u, 0u);
      if (sl >= 0)
        val = __ldg(reinterpret_cast<const uint4*>(a.kv_layer + base + (size_t)sl * a.row_bytes +
                                                   (size_t)g * kPD * 2) + c);
      const uint32_t off = is_v ? gi * kGroupBytes + (c >> 3) * (kGroupBytes / 2) + sw128(key & 15, c & 7)
                                : (c >> 3) * kHalf + sw128(key, c & 7);
      *reinterpret_cast<uint4*>(dst + off) = val;
    }
  }
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
}

// Warp roles: 0 loads Q once, then K blocks into a three-stage ring; 10
// loads V blocks into a two-stage ring; 1 issues tile A's MMAs and 11 tile
// B's (lane 0 each: one issuing thread cannot keep the tensor core busy);
// 2..5 run the softmax of tile A and 6..9 that of tile B, one query row per
// thread (TMEM lane quadrant = warp % 4), and their epilogues.
__global__ void __launch_bounds__(kPThreads, 1) prefill_tc_kernel(const __grid_constant__ PrefillArgs a) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  __shared__ PrefillBars sb;
  unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  unsigned char* sQ = smem;                   // tile X's Q at X * 2 kHalf: [2 halves][128 rows][128 B]
  unsigned char* sK = smem + 4 * kHalf;       // K stage s at s * 2 kHalf
  unsigned char* sV = sK + kKS * 2 * kHalf;   // V stage s at s * 2 kHalf
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  volatile int* abort_flag = &sb.abort;

  // CTA order: request and KV head major, the pair with the most keys first,
  // so that the pairs reading the same K/V run side by side (L2 serves all
  // but the first of them).
  const int pairs = (a.tiles + 1) >> 1;
  const int pair = pairs - 1 - (int)(blockIdx.x % pairs);
  const int bg = (int)(blockIdx.x / pairs);
  const int b = bg / a.Hkv, g = bg % a.Hkv;
  const int TT = kPM / a.G;  // query tokens per tile
  const int j0 = 2 * pair * TT;  // first token of tile A; tile B starts at j0 + TT
  const int L = a.context_lens[b];
  const int ql = a.q_lens ? a.q_lens[b] : a.C;
  const int row = a.table_rows ? a.table_rows[b] : b;
  const bool valid = ql >= 1 && ql <= a.C && ql <= L && L <= table_capacity(a.T) && row >= 0 && row < a.T.rows_total;
  // softmax threads: tile X = (warp - 2) / 4, query row r = 32 * (warp % 4) + lane: token j0 + X TT + r / G,
  // head r % G of the group (the MMA warps: tile X = warp == kMmaWarpB)
  const int X = warp >= 6 ? (warp == kVWarp ? 0 : 1) : 0;
  const int r = 32 * (warp & 3) + lane;
  const int rt = X * TT + r / a.G, hh = r % a.G;  // token offset from j0, head in the group
  __nv_bfloat16* orow = a.out + (((size_t)b * a.C + j0 + rt) * a.Hq + (size_t)g * a.G + hh) * kPD;
  if (!valid) {
    if (tid == 0 && g == 0 && pair == 0) set_error(a.err, KVP_ERR_BAD_INDEX);
    if (warp >= 2 && warp < kVWarp && j0 + rt < a.C)
      for (int d = 0; d < kPD; d += 8) *reinterpret_cast<uint4*>(orow + d) = make_uint4(0u, 0u, 0u, 0u);
    return;
  }
  if (j0 >= ql) return;  // no query of this request falls in the pair
  const int jn = min(2 * TT, ql - j0);  // query tokens of the pair
  const bool has_b = jn > TT;
  const int p_first = L - ql + j0, p_last = p_first + jn - 1;
  // the union of the pair's spans: the first query reaches furthest back
  const Span u = attend_span(p_last + 1, a.window > 0 ? a.window + (p_last - p_first) : 0, a.sinks);
  const int n_keys = u.se + (p_last + 1 - u.lo);
  const int nblk = (n_keys + kPN - 1) / kPN;

  if (tid == 0) {
    mbar_init(&sb.q_full, 1);
    const uint32_t ntile = has_b ? 2 : 1;
    for (int s2 = 0; s2 < kKS; ++s2) {
      mbar_init(&sb.k_full[s2], 1);
      mbar_init(&sb.k_empty[s2], ntile);
    }
    for (int s2 = 0; s2 < kVS; ++s2) {
      mbar_init(&sb.v_full[s2], 1);
      mbar_init(&sb.v_empty[s2], ntile);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(&sb.s_full[x], 1);
      mbar_init(&sb.p_full[x], 4);
      mbar_init(&sb.pv_done[x], 1);
    }
    mbar_init(&sb.drain, ntile);
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
  // TMEM: S_A at columns 0, S_B at 128, O_A at 256, O_B at 384; P_X in the
  // first 64 columns of S_X
  const uint32_t tbase = sb.taddr;

  if (warp == 0 || warp == kVWarp) {
    // ======================= loaders ==========================================
    // Warp 0 loads Q, then K(i) once both S of block i - kKS have read its
    // stage; warp kVWarp loads V(i) once both P V of block i - kVS have. Each
    // resolves its own slots, so neither waits on the other's ring.
    const bool is_v = warp == kVWarp;
    const int NS = is_v ? kVS : kKS;
    if (!is_v && lane == 0) {
      mbar_arrive_expect_tx(&sb.q_full, (has_b ? 4u : 2u) * kHalf);
      tma_load_4d(sQ, &a.qmap, 0, g * a.G, j0, b, &sb.q_full);
      tma_load_4d(sQ + kHalf, &a.qmap, 64, g * a.G, j0, b, &sb.q_full);
      if (has_b) {
        tma_load_4d(sQ + 2 * kHalf, &a.qmap, 0, g * a.G, j0 + TT, b, &sb.q_full);
        tma_load_4d(sQ + 3 * kHalf, &a.qmap, 64, g * a.G, j0 + TT, b, &sb.q_full);
      }
    }
    int* slots = sb.slots[is_v ? 1 : 0];
    for (int i = 0; i < nblk; ++i) {
      const int st = i % NS;
      const int o0 = i * kPN;
      // lane l resolves keys 4l .. 4l+3 (four independent table reads); group
      // gi (lanes 4gi .. 4gi+3) goes by one TMA copy when its 16 slots are
      // contiguous and 16-aligned
      int sl[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int o = o0 + 4 * lane + k;
        sl[k] = o < n_keys ? resolve_slot(a.T, row, span_pos(u, o), a.err) : -1;
      }
      __syncwarp();  // the previous block's copies have read the slot list
#pragma unroll
      for (int k = 0; k < 4; ++k) slots[4 * lane + k] = sl[k];
      const int g0 = __shfl_sync(0xffffffffu, sl[0], lane & ~3);
      const bool mine = a.use_kvmap && sl[0] >= 0 && sl[1] == sl[0] + 1 && sl[2] == sl[0] + 2 &&
                        sl[3] == sl[0] + 3 && sl[0] == g0 + 4 * (lane & 3) && (g0 & 15) == 0;
      const unsigned okb = __ballot_sync(0xffffffffu, mine);
      unsigned tm = 0;
#pragma unroll
      for (int gi = 0; gi < 8; ++gi)
        if (((okb >> (4 * gi)) & 0xFu) == 0xFu) tm |= 1u << gi;
      __syncwarp();
      if (i >= NS && !__all_sync(0xffffffffu, pwait(is_v ? &sb.v_empty[st] : &sb.k_empty[st], (i - NS) / NS,
                                                    abort_flag, a.err)))
        break;
      load_rows(a, (is_v ? sV : sK) + st * 2 * kHalf, slots, tm, g, is_v, is_v ? &sb.v_full[st] : &sb.k_full[st],
                lane);
    }
  } else if (warp == 1 || warp == kMmaWarpB) {
    // ======================= MMA issuers (one per tile) ========================
    // S_X(i) = Q_X K(i)^T is eight N 128 MMAs (one per 16-wide K step of d),
    // so S column c is key c of the block. S_X(i + 1) overwrites P_X(i), so
    // it waits for P_X(i) V. Per block i: P_X(i) V, then S_X(i + 1); the two
    // tiles' issuers run side by side, so while one tile's softmax runs the
    // tensor core works on the other tile. The whole warp walks the schedule
    // and waits (no divergent spin beside the issuing lane); lane 0 alone
    // issues the MMAs and the commits. A K (V) stage is free once both
    // tiles' issuers have committed their S (P V) of it.
    if (X == 0 || has_b) {
      const bool issuer = lane == 0;
      const uint32_t id_n128 = umma_idesc(0, kPN), id_o = umma_idesc(1, kPN);
      const uint32_t tS = tbase + (uint32_t)X * 128u, tO = tbase + 256u + (uint32_t)X * 128u;
      // descriptors of the operands' starts; a K step adds its byte offset >> 4
      const uint64_t dq = umma_desc(smem_u32(sQ + X * 2 * kHalf), 16, 1024);
      const uint64_t dk0 = umma_desc(smem_u32(sK), 16, 1024);
      const uint64_t dv0 = umma_desc(smem_u32(sV), kGroupBytes / 2, 1024);
      auto issue_s = [&](int blk) {
        const uint64_t dk = dk0 + (uint64_t)(((blk % kKS) * 2 * kHalf) >> 4);
        if (issuer) {
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            const uint64_t off = (uint64_t)((((ks >> 2) * kHalf) + (ks & 3) * 32) >> 4);
            umma_f16(tS, dq + off, dk + off, id_n128, ks > 0);
          }
          umma_commit(&sb.s_full[X]);
          umma_commit(&sb.k_empty[blk % kKS]);
        }
        __syncwarp();
      };
      bool ok = __all_sync(0xffffffffu, pwait(&sb.q_full, 0, abort_flag, a.err));
      if (ok) ok = __all_sync(0xffffffffu, pwait(&sb.k_full[0], 0, abort_flag, a.err));
      if (ok) {
        tc_fence_after();
        issue_s(0);
      }
      for (int i = 0; ok && i < nblk; ++i) {
        const int sv = i % kVS;
        ok = __all_sync(0xffffffffu, pwait(&sb.v_full[sv], i / kVS, abort_flag, a.err));
        if (ok) ok = __all_sync(0xffffffffu, pwait(&sb.p_full[X], i, abort_flag, a.err));
        if (!ok) break;
        tc_fence_after();
        // O_X += P_X(i) V(i): P_X from TMEM (8 columns per 16 keys), V group m
        // the MN-major B operand of K step m (halves of d 2 KB apart, 8-key atoms 1 KB)
        const uint64_t dv = dv0 + (uint64_t)((sv * 2 * kHalf) >> 4);
        if (issuer) {
#pragma unroll
          for (int m = 0; m < 8; ++m)
            umma_f16_ts(tO, tS + (uint32_t)m * 8u, dv + (uint64_t)((m * kGroupBytes) >> 4), id_o,
                        (i > 0 || m > 0) ? 1u : 0u);
          umma_commit(&sb.pv_done[X]);
          umma_commit(&sb.v_empty[sv]);
        }
        __syncwarp();
        if (i + 1 < nblk) {
          ok = __all_sync(0xffffffffu, pwait(&sb.k_full[(i + 1) % kKS], (i + 1) / kKS, abort_flag, a.err));
          if (ok) ok = __all_sync(0xffffffffu, pwait(&sb.pv_done[X], i, abort_flag, a.err));
          if (!ok) break;
          tc_fence_after();
          issue_s(i + 1);
        }
      }
      if (issuer) umma_commit(&sb.drain);  // arrives once everything this warp issued is done
      __syncwarp();
    }
  } else if (warp < kVWarp && (X == 0 || has_b)) {
    // ======================= softmax warps (tile X) ============================
    const bool rv = rt < jn;
    const int pr = p_first + rt;
    const Span sr0 = attend_span(pr + 1, a.window, a.sinks);
    // In key offsets of the pair's span u: the row's sink rows are offsets
    // [0, sr.se) (when u keeps a sink segment its width is the row's; when it
    // does not, u starts at position 0 and offsets are positions), and its
    // window [sr.lo, pr] starts at or after u.lo. Rows past the chunk keep nothing.
    const Span sr = rv ? sr0 : Span{0, 0};
    const int wb0 = rv ? u.se + (sr.lo - u.lo) : 1 << 30, we0 = rv ? u.se + (pr - u.lo) : -1;
    const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
    const uint32_t tS = tbase + (uint32_t)X * 128u + lane_base, tO = tbase + 256u + (uint32_t)X * 128u + lane_base;
    const float sl2 = a.scale_log2;
    float m_used = -INFINITY, lsum = 0.f;  // m in scaled log2 units
    bool ok = true;
    for (int i = 0; i < nblk; ++i) {
      ok = __all_sync(0xffffffffu, pwait(&sb.s_full[X], i, abort_flag, a.err));
      if (!ok) break;
      tc_fence_after();
      // The row attends key offsets [0, ea) (its sink rows) and [wb, we] (its
      // window), relative to this block's first offset; S column c is key c.
      const int o0 = i * kPN;
      const int ea = sr.se - o0, wb = wb0 - o0, we = we0 - o0;
      const bool unmasked = __all_sync(0xffffffffu, wb <= 0 && we >= kPN - 1);  // no row of the warp masks
      // The row's 128 scores, read from TMEM once (one wait for four loads).
      float sv[128];
#pragma unroll
      for (int c8 = 0; c8 < 8; ++c8) tmem_ld16_nowait(tS + 16 * c8, sv + 16 * c8);
      tmem_wait_ld();
      if (!unmasked) {
#pragma unroll
        for (int c = 0; c < 128; ++c)
          if (!(c < ea || (c >= wb && c <= we))) sv[c] = -INFINITY;
      }
      // the row maximum, taken on unscaled scores (scale > 0) and scaled once
      float rmax = -INFINITY;
#pragma unroll
      for (int c = 0; c < 128; ++c) rmax = fmaxf(rmax, sv[c]);
      rmax *= sl2;
      const bool grow = rmax > m_used + 8.f;  // also when nothing was kept before
      const bool scale_o = grow && lsum > 0.f;
      const float f = scale_o ? exp2f(m_used - rmax) : 1.f;
      if (grow) m_used = rmax;
      const float msub = m_used == -INFINITY ? 0.f : m_used;  // masked scores give 2^-inf = 0 either way
      // P_X(i), keys in order, two per 32-bit column, over the first 64
      // columns of S_X (S_X(i + 1) is issued only after P_X(i) V(i) is done)
      float ps0 = 0.f, ps1 = 0.f;  // the row sum, two lanes of a packed add
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint32_t w[16];
#pragma unroll
        for (int x = 0; x < 16; ++x) {
          float x0, x1;
          fma2_bc(x0, x1, sv[32 * q + 2 * x], sv[32 * q + 2 * x + 1], sl2, -msub);
          const float p0 = ex2_ftz(x0), p1 = ex2_ftz(x1);
          w[x] = pack_bf16(p0, p1);
          add2(ps0, ps1, p0, p1);
        }
        tmem_st16(tS + 16 * q, w);
      }
      lsum = lsum * f + (ps0 + ps1);
      if (__any_sync(0xffffffffu, scale_o)) {
        // O_X holds blocks < i in the old maximum: rescale it once P V(i - 1) is
        // in, before P V(i) may start (a warp-wide TMEM read and write)
        ok = __all_sync(0xffffffffu, pwait(&sb.pv_done[X], i - 1, abort_flag, a.err));
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4) {
          float ov[32];
          tmem_ld32(tO + c4 * 32, ov);
#pragma unroll
          for (int x = 0; x < 32; ++x) ov[x] *= f;
          tmem_st32(tO + c4 * 32, ov);
        }
      }
      asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sb.p_full[X]);
    }
    // ---- epilogue: O / l -> bf16, once the last P V is in O ------------------
    if (ok) ok = __all_sync(0xffffffffu, pwait(&sb.pv_done[X], nblk - 1, abort_flag, a.err));
    if (ok) {
      tc_fence_after();
      const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) {
        float ov[32];
        tmem_ld32(tO + c4 * 32, ov);
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
    }
  }
  // Everything the MMA lane issued is done (bounded) before TMEM goes back.
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

constexpr size_t kPrefillSmem = (4 + 2 * kKS + 2 * kVS) * kHalf + 1024;  // two Q tiles, the K and V rings

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
  const long long grid = (long long)((a.tiles + 1) / 2) * batch * pool->kv_heads;
  if (grid <= 0 || grid > 0x7fffffffLL) return KVP_ERR_INVALID_ARG;
  prefill_tc_kernel<<<(unsigned)grid, kPThreads, kPrefillSmem, stream>>>(a);
  return cudaGetLastError() == cudaSuccess ? KVP_OK : KVP_ERR_CUDA;
}

}  // namespace kvp
