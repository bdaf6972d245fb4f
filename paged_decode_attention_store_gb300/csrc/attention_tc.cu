// bf16 paged decode attention, head_dim 128, on sm_103a.
//
// What it computes: for each request, each query head h (KV head h / G) and
// the positions lo <= t < L read through the block table or raw-location
// table, s_t = scale * <q_h, k_t>, softmax over t, sum of p_t * v_t
// (chapter 15 of silicon_compiler_from_scratch, section "The model": the new
// token and at most W-1 earlier ones; tiny-llm week 3 day 3, "Correctness
// Checkpoint": dense attention over the rows gathered in logical order,
// here read in place from the pages).
//
// How (GB300 design):
// * The path is HBM-bound (G flop per byte of K/V), so the kernel is built to
//   keep bytes in flight: one CTA per SM, persistent over an equal share of
//   the batch's attended tokens, two PRODUCER warps that issue one
//   cp.async.bulk per token row (all KV heads of the group, HG*256 contiguous
//   bytes, K and V) into a 3-stage ring of 16-token stages completed by
//   mbarrier transaction counts, and HG CONSUMER warps, one per KV head.
//   The producers take alternate stages: the copy engine drains one
//   producer's 32 row copies while the other does its bookkeeping, so it
//   never waits for work (one producer alone left it idle part of every
//   stage, which capped the stream below the DRAM rate).
// * Stages are 16-position groups aligned to multiples of 16. A full group
//   whose 16 slots are contiguous and 16-aligned (always true for a block
//   table whose page size is a multiple of 16; checked per stage for a raw
//   location table) is loaded with four TMA tensor copies (K and V, two
//   64-element halves of head_dim, 16 slots x HG heads each) through a map
//   whose slot and head axes are swapped, so the rows land head-major with
//   the 128-byte swizzle and ldmatrix stays conflict-free. Other stages
//   (partial groups, scattered slots) take one bulk copy per token row at a
//   pitch of HG*256+16 bytes, which spreads an ldmatrix's 8 rows over 8 bank
//   groups as well.
// * Each consumer warp runs the GQA group of its KV head on the legacy
//   tensor-core path (mma.sync m16n8k16, bf16 in, fp32 accumulate) with the
//   16 TOKENS of a stage on the M dimension and the G <= 8 query heads on N:
//     S^T[16 x 8]  = K[16 x 128] . Q^T[128 x 8]       (8 MMAs)
//     O^T[128 x 8] += V^T[128 x 16] . P^T[16 x 8]     (8 MMAs)
//   K feeds A through ldmatrix, V^T through ldmatrix.trans, Q^T stays in
//   registers for the whole item, and P^T comes from the S^T accumulator
//   with two movmatrix.trans (no shared-memory round trip).
//   A 128-row tcgen05 tile would be 8x larger than a stage and buys nothing
//   on a bandwidth-bound path at 1-4 flop/byte.
// * Online softmax in log2 units with warp-shuffle reductions over the
//   token rows; P is rounded to bf16 for the MMA and the row sum is taken of
//   the rounded values so numerator and denominator agree.
// * Work split without a separate planning kernel: every CTA reads the
//   batch's context lengths, scans them in shared memory and takes an equal
//   share of the attended tokens (see attention.cuh); the producer then walks
//   the requests of its share. A request that ends inside the share writes
//   the final bf16 output; a request cut by a share boundary writes fp32
//   partials (max, sum, unnormalised output) that the combine kernel merges
//   (split-K, flash-decoding style). Both kernels are programmatic dependent
//   launches, so their launch latency hides behind the preceding kernel.
// * Every wait is bounded (2 s); on timeout the CTA records KVP_ERR_TIMEOUT,
//   raises its abort flag, waits (bounded) for its own copies and returns.
#include <cudaTypedefs.h>

#include "attention.cuh"

namespace kvp {

namespace {

constexpr int kTok = 16;      // tokens per stage (the MMA M dimension)
constexpr int kMaxStages = 8; // ring depth limit (the depth a.stages is chosen per head group)
constexpr int kQBars = 8;     // Q-buffer barriers, by piece mod 8 (>= kMaxStages)
constexpr int kProducers = 2; // producer warps, alternate stages
constexpr int kAhead = 2;     // own stages whose table entries are fetched ahead of issue
constexpr int kQueue = 4;     // entry-queue slots per producer (> kAhead)
constexpr int kD = 128;       // head_dim
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr int kMinTokensPerCta = 64;
constexpr int kStaticSmemBound = 512;                      // PlanState + the scan's warp sums
constexpr int kAlignSlack = 1024;                          // the stage buffers start on 1024 bytes
constexpr int kMaxDynamicSmem = 232448 - kStaticSmemBound;  // per-block opt-in limit minus static

// Stage header, written by the producer, read by the consumers.
struct __align__(16) StageHdr {
  int live;    // 1: a stage of a piece, 0: no more work
  int t0;      // first position of the stage
  int vmask;   // bit j: token t0+j has K/V rows in the stage
  int flags;   // 1 first stage of the piece, 2 last stage, (qbuf << 2), 8 tensor-copy layout,
               // (piece % kQBars) << 4 (selects the qempty barrier)
  int b;       // request
  int group;   // KV-head group
  int part;    // partial slot of a split piece, -1 when the piece is the whole request
  int L;       // context length of the request (positions of multi-token queries)
};

// What the producer's lookahead cursor records for a stage it has queued.
struct __align__(16) StageMeta {
  int live;    // 0: no more work; t0 then holds the number of stages of the CTA
  int t0;
  int t_end;   // end of the piece
  int flags;   // 1 first stage of the piece, 2 last stage, 16 the stage holds a fused step's newest position
  int b;
  int group;
  int part;
  int piece;   // index of the piece within the CTA (selects the Q buffer)
  int L;       // context length of the request
  int pad0, pad1, pad2;
};

struct SmemMap {
  int pitch, stage_bytes, qbytes, nq;
  unsigned char* stages;
  unsigned char* qbuf;
  StageMeta* meta;     // [kProducers][kQueue]
  int* entries;        // [kProducers][kQueue][kTok] table entries of queued stages
  StageHdr* hdr;
  uint64_t* full;
  uint64_t* empty;
  uint64_t* qempty;
  volatile int* abort_flag;
};

__host__ __device__ __forceinline__ int stage_stride(int HG) {
  return (2 * kTok * (HG * 256 + 16) + 1023) & ~1023;
}

__device__ __forceinline__ SmemMap map_smem(unsigned char* smem, int HG, int C, int nq, int S) {
  SmemMap s;
  s.pitch = HG * 256 + 16;
  s.stage_bytes = stage_stride(HG);
  s.qbytes = HG * C * kD * 2;  // C = G * M query columns per KV head
  s.nq = nq;
  s.stages = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem) + 1023) & ~uintptr_t(1023));
  s.qbuf = s.stages + S * s.stage_bytes;
  s.meta = reinterpret_cast<StageMeta*>(s.qbuf + nq * s.qbytes);
  s.entries = reinterpret_cast<int*>(s.meta + kProducers * kQueue);
  s.hdr = reinterpret_cast<StageHdr*>(s.entries + kProducers * kQueue * kTok);
  s.full = reinterpret_cast<uint64_t*>(s.hdr + S);
  s.empty = s.full + S;
  s.qempty = s.empty + S;
  s.abort_flag = reinterpret_cast<volatile int*>(s.qempty + kQBars);
  return s;
}

__device__ __forceinline__ int entry_to_slot(const TableRef& T, int e, int t, int32_t* err) {
  if (T.raw) {
    if ((unsigned)e >= (unsigned)T.num_slots) {
      set_error(err, KVP_ERR_BAD_INDEX);
      return -1;
    }
    return e;
  }
  if ((unsigned)e >= (unsigned)T.num_pages) {
    set_error(err, KVP_ERR_BAD_INDEX);
    return -1;
  }
  return e * T.page_size + t % T.page_size;
}

// Attended positions of a request (0 when its length or table row is
// invalid): the se sink rows [0, se), then [lo, L) (see attend_span).
// With M query tokens the span is the union of theirs: query 0 (context
// L - M + 1) reaches furthest back, so the window is widened by M - 1.
__device__ __forceinline__ int attended(const TcArgs& a, int L, int row, long long cap, int* lo, int* se) {
  const bool valid = L >= a.M && L >= 1 && L <= cap && row >= 0 && row < a.T.rows_total;
  const Span sp = attend_span(valid ? L : 0, a.window > 0 ? a.window + a.M - 1 : a.window, a.sinks);
  *lo = sp.lo;
  *se = sp.se;
  return valid ? sp.se + L - sp.lo : 0;
}

// ---------------------------------------------------------------------------
// Work split of this CTA (see attention.cuh), computed by the whole CTA with
// the stage buffers as scratch: n_b in shared ints, their exclusive prefix
// sums in shared 64-bit ints.
// ---------------------------------------------------------------------------
struct PlanState {
  long long R0, R1;  // this CTA's share of the token stream
  long long Sv0;     // stream start of the first virtual request in the share
  int active;        // the share is not empty
  int b0, g0;        // first request and group of the share
  int L0, row0;      // its context length and table row
  int merge_v, merge_ka, merge_sa;  // split request whose final piece is here
};

// Scratch of the plan, in the stage buffers: per request n, L, row (ints)
// and the exclusive prefix of n (64-bit).
constexpr int kPlanScratchPerRequest = 20;

__device__ void plan_cta(const TcArgs& a, const SmemMap& s, PlanState* ps) {
  long long* sS = reinterpret_cast<long long*>(s.stages);
  int* sN = reinterpret_cast<int*>(sS + a.B);
  int* sL = sN + a.B;
  int* sR = sL + a.B;
  const long long cap = table_capacity(a.T);
  for (int b = threadIdx.x; b < a.B; b += blockDim.x) {
    const int L = __ldg(a.context_lens + b);
    const int row = a.table_rows ? __ldg(a.table_rows + b) : b;
    int lo, se;
    const int n = attended(a, L, row, cap, &lo, &se);
    sN[b] = n;
    sL[b] = L;
    sR[b] = row;
    if (n == 0 && blockIdx.x == 0) set_error(a.err, KVP_ERR_BAD_INDEX);
  }
  __syncthreads();
  const int per = (a.B + blockDim.x - 1) / blockDim.x;
  const int b0 = min(a.B, (int)threadIdx.x * per), b1 = min(a.B, b0 + per);
  long long local = 0;
  for (int b = b0; b < b1; ++b) local += sN[b];
  long long total;
  long long base = block_exclusive_scan(local, &total);
  for (int b = b0; b < b1; ++b) {
    sS[b] = base;
    base += sN[b];
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const long long T = total * a.n_groups;
    const long long Ne = T > 0 ? min((long long)a.num_ctas, (T + kMinTokensPerCta - 1) / kMinTokensPerCta) : 0;
    const long long k = blockIdx.x;
    ps->active = k < Ne;
    ps->merge_v = -1;
    ps->merge_ka = ps->merge_sa = 0;
    if (k < Ne) {
      const long long R0 = k * T / Ne, R1 = (k + 1) * T / Ne;
      int lo = 0, hi = a.B - 1;  // first request whose stream range ends after R0
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if ((long long)a.n_groups * (sS[mid] + sN[mid]) > R0)
          hi = mid;
        else
          lo = mid + 1;
      }
      const int b = lo;
      const long long nb = sN[b];
      const long long base_b = (long long)a.n_groups * sS[b];
      const int g = (int)((R0 - base_b) / nb);
      const long long Sv = base_b + g * nb;
      ps->R0 = R0;
      ps->R1 = R1;
      ps->Sv0 = Sv;
      ps->b0 = b;
      ps->g0 = g;
      ps->L0 = sL[b];
      ps->row0 = sR[b];
      if ((Sv < R0 || Sv + nb > R1) && Sv + nb <= R1) {  // split, and its final piece is here
        const long long ka = ((Sv + 1) * Ne + T - 1) / T - 1;  // CTA holding the request's first piece
        ps->merge_v = b * a.n_groups + g;
        ps->merge_ka = (int)ka;
        ps->merge_sa = (int)((ka * T / Ne == Sv) ? 2 * ka : 2 * ka + 1);
      }
    }
  }
  __syncthreads();
}

// The producer's walk over the pieces of its share.
// A piece covers the stream offsets [x - Sv, e - Sv) of its request, which
// map to positions through the span: offsets below se are the sink rows
// themselves, the rest start at lo. So a piece is one or two position
// segments; the walk takes the stages of the first, then of the second.
struct Cursor {
  long long R0, R1, x, Sv, cap;
  int k, B;
  int b, g, row, lo, se, L, n;       // current virtual request
  int t_begin, t_end, part, t0;      // current piece: first position, end of the current segment, next stage start
  int nxt_begin, nxt_end;            // the piece's second segment, or nxt_begin = -1
  int piece;                         // index of the current piece
  bool done;
  int nb, nL, nrow;                  // next request, prefetched
};

__device__ __forceinline__ void cur_set_piece(Cursor& c) {
  const long long e = min(c.R1, c.Sv + c.n);
  const int ob = (int)(c.x - c.Sv), oe = (int)(e - c.Sv);
  c.nxt_begin = -1;
  if (ob < c.se) {  // starts among the sink rows
    c.t_begin = ob;
    c.t_end = min(oe, c.se);
    if (oe > c.se) {
      c.nxt_begin = c.lo;
      c.nxt_end = c.lo + (oe - c.se);
    }
  } else {
    c.t_begin = c.lo + (ob - c.se);
    c.t_end = c.lo + (oe - c.se);
  }
  const bool split = c.Sv < c.R0 || c.Sv + c.n > c.R1;
  c.part = split ? (c.x == c.R0 ? 2 * c.k : 2 * c.k + 1) : -1;
  c.t0 = c.t_begin;
}

__device__ __forceinline__ void cur_prefetch(const TcArgs& a, Cursor& c) {
  c.nb = c.b + 1;
  if (c.nb < c.B) {
    c.nL = __ldg(a.context_lens + c.nb);
    c.nrow = a.table_rows ? __ldg(a.table_rows + c.nb) : c.nb;
  }
}

__device__ void cur_init(const TcArgs& a, const PlanState& ps, Cursor& c) {
  c.k = blockIdx.x;
  c.B = a.B;
  c.cap = table_capacity(a.T);
  c.done = !ps.active;
  if (c.done) return;
  c.R0 = ps.R0;
  c.R1 = ps.R1;
  c.x = ps.R0;
  c.Sv = ps.Sv0;
  c.b = ps.b0;
  c.g = ps.g0;
  c.row = ps.row0;
  c.n = attended(a, ps.L0, c.row, c.cap, &c.lo, &c.se);
  c.L = ps.L0;
  c.piece = 0;
  cur_prefetch(a, c);
  cur_set_piece(c);
}


__device__ void cur_next_piece(const TcArgs& a, Cursor& c) {
  c.x = min(c.R1, c.Sv + c.n);
  if (c.x >= c.R1) {
    c.done = true;
    return;
  }
  if (c.g + 1 < a.n_groups) {
    ++c.g;
    c.Sv += c.n;
    cur_set_piece(c);
    return;
  }
  for (;;) {
    if (c.nb >= c.B) {  // cannot happen while x < R1; stop rather than read past the batch
      c.done = true;
      return;
    }
    c.b = c.nb;
    c.row = c.nrow;
    const int L = c.nL;
    cur_prefetch(a, c);
    c.n = attended(a, L, c.row, c.cap, &c.lo, &c.se);
    c.L = L;
    if (c.n > 0) break;
  }
  c.g = 0;
  c.Sv = c.x;
  cur_set_piece(c);
}

// End of the stage that starts at t0: the next multiple of 16, or the piece end.
__device__ __forceinline__ int stage_end(int t0, int t_end) { return min((t0 & ~(kTok - 1)) + kTok, t_end); }

// Move the cursor past one stage.
__device__ __forceinline__ void cur_advance(const TcArgs& a, Cursor& c) {
  c.t0 = (c.t0 & ~(kTok - 1)) + kTok;
  if (c.t0 >= c.t_end) {
    if (c.nxt_begin >= 0) {  // from the sink rows to the window
      c.t0 = c.nxt_begin;
      c.t_end = c.nxt_end;
      c.nxt_begin = -1;
    } else {
      cur_next_piece(a, c);
      ++c.piece;
    }
  }
}

// ---------------------------------------------------------------------------
// Producer warp.
// ---------------------------------------------------------------------------
__device__ void tc_producer(const TcArgs& a, const SmemMap& s, const PlanState& ps, int pid, int lane) {
  const int HG = a.HG;
  const uint32_t row_copy = (uint32_t)HG * 256u;
  const int j = lane & 15;          // token within the stage
  const bool is_v = lane >= 16;     // lanes 16..31 copy V rows
  StageMeta* meta = s.meta + pid * kQueue;
  int* entries = s.entries + pid * kQueue * kTok;

  // Lookahead cursor over all of the CTA's stages; for this producer's own
  // stages (global index = pid mod 2) it records the metadata and starts the
  // asynchronous fetch of the table entries kAhead own stages before issue,
  // so that issuing never waits on a global load.
  Cursor c;
  cur_init(a, ps, c);
  long long next_gs = 0;  // global index of the stage the cursor describes
  long long queued = 0;   // own stages queued
  auto queue_next = [&]() {
    while (!c.done && (next_gs & 1) != pid) {
      cur_advance(a, c);
      ++next_gs;
    }
    const int qs = (int)(queued % kQueue);
    if (!c.done) {
      const int se = stage_end(c.t0, c.t_end);
      const bool last = se == c.t_end && c.nxt_begin < 0;  // the piece's last stage
      // In a fused step the request's newest position (the piece ends at
      // the request's end) is read from the new rows, at the slot out_loc
      // gives: its table entry may be written by this very launch.
      const int t_new = (a.fused && last && c.t_end == c.L) ? c.t_end - 1 : -1;
      if (lane == 0) {
        StageMeta m;
        m.live = 1;
        m.t0 = c.t0;
        m.t_end = c.t_end;
        m.flags = (c.t0 == c.t_begin ? 1 : 0) | (last ? 2 : 0) | (t_new >= 0 ? 16 : 0);
        m.b = c.b;
        m.group = c.g;
        m.part = c.part;
        m.piece = c.piece;
        m.L = c.L;
        meta[qs] = m;
      }
      if (lane < kTok && c.t0 + lane < se) {
        const int t = c.t0 + lane;
        cp_async4(&entries[qs * kTok + lane], t == t_new ? a.out_loc + c.b
                                                         : a.T.table + (size_t)c.row * a.T.cols +
                                                               (a.T.raw ? t : t / a.T.page_size));
      }
      cur_advance(a, c);
      ++next_gs;
    } else if (lane == 0) {
      meta[qs].live = 0;
      meta[qs].t0 = (int)next_gs;  // stages of the CTA
    }
    cp_async_commit();
    ++queued;
  };
  for (int k = 0; k < kAhead; ++k) queue_next();

  long long gs = pid;     // global index of the stage to issue
  long long n_stages = -1;
  bool ok = true;
  for (long long k = 0;; ++k, gs += kProducers) {
    queue_next();
    cp_async_wait<kAhead>();  // the entries of own stage k have landed
    __syncwarp();
    const int qs = (int)(k % kQueue);
    const StageMeta m = meta[qs];
    if (!m.live) {
      n_stages = m.t0;
      break;
    }
    const bool first_stage = m.flags & 1;
    const bool last_stage = m.flags & 2;
    const int qi = m.piece % s.nq;
    const int S = a.stages;
    const int st = (int)(gs % S);
    if (gs >= S) {
      ok = __all_sync(0xffffffffu, mbar_wait_bounded(&s.empty[st], (uint32_t)((gs / S - 1) & 1),
                                                     s.abort_flag, a.err, kWaitLimitNs));
      if (!ok) break;
    }
    // Q buffer reuse: piece p overwrites the buffer of piece p - nq, so it
    // waits until the consumers have loaded that piece's Q. Consumers
    // arrive on qempty[piece % kQBars]; piece p - nq is phase
    // (p - nq) / kQBars of barrier (p - nq) % kQBars. The parity test is
    // exact because every stage up to gs - S is consumed (the wait above)
    // and the barrier's previous piece, p - nq - kQBars, has its first stage
    // at most at gs - kQBars <= gs - S: it has been loaded, so the barrier
    // is at most one phase behind.
    if (first_stage && m.piece >= s.nq) {
      const int pw = m.piece - s.nq;
      ok = __all_sync(0xffffffffu, mbar_wait_bounded(&s.qempty[pw % kQBars], (uint32_t)((pw / kQBars) & 1),
                                                     s.abort_flag, a.err, kWaitLimitNs));
      if (!ok) break;
    }
    const int t = m.t0 + j;
    const int send = stage_end(m.t0, m.t_end);
    const bool fresh = (m.flags & 16) && t == m.t_end - 1;  // the newest position of a fused step
    int slot = -1;
    if (fresh) {
      slot = entries[qs * kTok + j];  // out_loc of the request
      if ((unsigned)slot >= (unsigned)a.T.num_slots) {
        set_error(a.err, KVP_ERR_BAD_INDEX);
        slot = -1;
      }
    } else if (t < send) {
      slot = entry_to_slot(a.T, entries[qs * kTok + j], t, a.err);
    }
    // A full, 16-aligned group of contiguous, 16-aligned slots goes by tensor
    // copies (never the group of a fused step's newest position).
    const int slot0 = __shfl_sync(0xffffffffu, slot, 0);
    const bool page = a.use_tmap && !(m.flags & 16) && (m.t0 & (kTok - 1)) == 0 && send - m.t0 == kTok &&
                      slot0 >= 0 && (slot0 & (kTok - 1)) == 0 && __all_sync(0xffffffffu, slot == slot0 + j);
    unsigned char* sbuf = s.stages + (size_t)st * s.stage_bytes;
    if (page) {
      if (lane == 0) {
        StageHdr h;
        h.live = 1;
        h.t0 = m.t0;
        h.vmask = 0xffff;
        h.flags = (first_stage ? 1 : 0) | (last_stage ? 2 : 0) | (qi << 2) | 8 | ((m.piece % kQBars) << 4);
        h.b = m.b;
        h.group = m.group;
        h.part = m.part;
        h.L = m.L;
        s.hdr[st] = h;
        const uint32_t box = (uint32_t)HG * kTok * 128u;  // 16 slots x HG heads x 64 elements
        mbar_arrive_expect_tx(&s.full[st], 4 * box + (first_stage ? (uint32_t)s.qbytes : 0u));
        const int hd0 = m.group * HG;
        tma_load_4d(sbuf, &a.tmap, 0, slot0, hd0, a.kvl_k, &s.full[st]);
        tma_load_4d(sbuf + box, &a.tmap, 64, slot0, hd0, a.kvl_k, &s.full[st]);
        tma_load_4d(sbuf + 2 * box, &a.tmap, 0, slot0, hd0, a.kvl_v, &s.full[st]);
        tma_load_4d(sbuf + 3 * box, &a.tmap, 64, slot0, hd0, a.kvl_v, &s.full[st]);
      }
      __syncwarp();
    } else {
      const unsigned copies = __ballot_sync(0xffffffffu, slot >= 0);
      if (lane == 0) {
        StageHdr h;
        h.live = 1;
        h.t0 = m.t0;
        h.vmask = (int)(copies & copies >> 16 & 0xffffu);
        h.flags = (first_stage ? 1 : 0) | (last_stage ? 2 : 0) | (qi << 2) | ((m.piece % kQBars) << 4);
        h.b = m.b;
        h.group = m.group;
        h.part = m.part;
        h.L = m.L;
        s.hdr[st] = h;
        const uint32_t tx = (uint32_t)__popc(copies) * row_copy + (first_stage ? (uint32_t)s.qbytes : 0u);
        mbar_arrive_expect_tx(&s.full[st], tx);
      }
      __syncwarp();
      if (slot >= 0) {
        const char* src =
            fresh ? reinterpret_cast<const char*>(is_v ? a.vnew : a.knew) + (size_t)m.b * a.row_bytes +
                        (size_t)m.group * row_copy
                  : a.kv_layer + (is_v ? a.kv_bytes : 0) + (size_t)slot * a.row_bytes + (size_t)m.group * row_copy;
        unsigned char* dst = sbuf + (is_v ? kTok * s.pitch : 0) + j * s.pitch;
        bulk_g2s(dst, src, row_copy, &s.full[st]);
      }
    }
    if (first_stage && lane < a.M) {  // the group's heads of each query token
      const uint32_t tok_bytes = (uint32_t)HG * a.G * kD * 2;
      const __nv_bfloat16* qsrc = a.q + (((size_t)m.b * a.M + lane) * a.Hq + (size_t)m.group * HG * a.G) * kD;
      bulk_g2s(s.qbuf + qi * s.qbytes + lane * tok_bytes, qsrc, tok_bytes, &s.full[st]);
    }
  }
  cp_async_wait<0>();

  // The producer that owns the first stage without work tells the consumers.
  if (ok && n_stages >= 0 && (n_stages % kProducers) == pid) {
    const int st = (int)(n_stages % a.stages);
    if (n_stages >= a.stages)
      ok = __all_sync(0xffffffffu, mbar_wait_bounded(&s.empty[st], (uint32_t)((n_stages / a.stages - 1) & 1),
                                                     s.abort_flag, a.err, kWaitLimitNs));
    if (ok && lane == 0) {
      s.hdr[st].live = 0;
      mbar_arrive(&s.full[st]);
    }
  }
  if (!ok) {
    // Abort: let the copies this warp issued land before the CTA exits.
    *s.abort_flag = 1;
    for (long long g2 = gs - kProducers; g2 >= 0 && g2 >= gs - kProducers * a.stages; g2 -= kProducers) {
      const int st = (int)(g2 % a.stages);
      const uint64_t t_start = global_timer_ns();
      while (!mbar_try_wait(&s.full[st], (uint32_t)((g2 / a.stages) & 1))) {
        if (global_timer_ns() - t_start > 100000000ull) break;
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Consumer warps: one KV head each.
// ---------------------------------------------------------------------------
template <int NT>
__device__ void tc_consumer(const TcArgs& a, const SmemMap& s, int w, int lane) {
  const int G = a.G, HG = a.HG, M = a.M;
  const int h = w / a.tiles;                   // KV head within the group
  const int col0 = (w % a.tiles) * 8 * NT;     // first (token, head) column of this warp
  const int C = M * G;                     // columns of the KV head
  const int g = lane >> 2, c = lane & 3;
  const uint32_t stages_u32 = smem_u32(s.stages);
  const uint32_t qbuf_u32 = smem_u32(s.qbuf);
  // ldmatrix row addresses of this lane (see the fragment layouts of
  // mma.m16n8k16: K as A[token][d], V^T as A[d][token] via .trans).
  const int ktok = (lane & 7) + ((lane >> 3) & 1) * 8, vtok = (lane & 7) + (lane >> 4) * 8;
  const uint32_t k_off = (uint32_t)(ktok * s.pitch + h * 256 + (lane >> 4) * 16);
  const uint32_t v_off = (uint32_t)(kTok * s.pitch + vtok * s.pitch + h * 256 + ((lane >> 3) & 1) * 16);
  // Tensor-copy layout: four boxes [K d0-63 | K d64-127 | V d0-63 | V d64-127],
  // each rows (head*16 + slot) of 128 bytes, 16-byte chunk c stored at
  // c ^ (row % 8); row % 8 is lane % 8 for both fragment row maps.
  const uint32_t box = (uint32_t)HG * kTok * 128u;
  const uint32_t kp_row = (uint32_t)(h * kTok + ktok) * 128u, vp_row = (uint32_t)(h * kTok + vtok) * 128u;
  const uint32_t sw = (uint32_t)(lane & 7);

  if (a.fused) {
    // The step's table writes and new K/V rows, spread over every consumer
    // thread of the grid while the first stages are in flight. Nothing this
    // launch reads depends on them (the newest positions come from the new
    // rows; the table writes only add pages for those positions).
    const long long tid = (long long)blockIdx.x * (a.CW * 32) + w * 32 + lane;
    const long long nthreads = (long long)a.num_ctas * a.CW * 32;
    const long long tw_total = (long long)a.n_tw * a.tw_expand;
    for (long long u = tid; u < tw_total; u += nthreads) {
      const int i = (int)(u / a.tw_expand), jj = (int)(u % a.tw_expand);
      const int r = __ldg(a.tw_rows + i);
      const long long col = (long long)__ldg(a.tw_cols + i) * a.tw_expand + jj;
      const int v = __ldg(a.tw_vals + i);
      if ((unsigned)r >= (unsigned)a.T.rows_total || col < 0 || col >= a.T.cols) {
        set_error(a.err, KVP_ERR_BAD_INDEX);
        continue;
      }
      a.tw_table[(size_t)r * a.T.cols + col] = v < 0 ? -1 : v * a.tw_expand + jj;
    }
    const int chunks = (int)(a.row_bytes / 16);
    const long long st_total = (long long)a.B * 2 * chunks;
    for (long long u = tid; u < st_total; u += nthreads) {
      const int cch = (int)(u % chunks);
      const long long ik = u / chunks;
      const int kv = (int)(ik & 1), i = (int)(ik >> 1);
      const int slot = __ldg(a.out_loc + i);
      if ((unsigned)slot >= (unsigned)a.T.num_slots) {
        if (kv == 0 && cch == 0) set_error(a.err, KVP_ERR_BAD_INDEX);
        continue;
      }
      const uint4 val = __ldg((kv ? a.vnew : a.knew) + (size_t)i * chunks + cch);
      reinterpret_cast<uint4*>(const_cast<char*>(a.kv_layer) + (kv ? a.kv_bytes : 0))[(size_t)slot * chunks + cch] = val;
    }
  }

  uint32_t qf[8][NT][2];
  float o[8][NT][4];
  float m[NT][2], l[NT][2];
  // Multi-token queries: position p, and the window [lo, p] plus sinks
  // [0, se), of the query token of each of this lane's columns.
  int qp[NT][2], qlo[NT][2], qse[NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    m[nt][0] = m[nt][1] = -INFINITY;
    l[nt][0] = l[nt][1] = 0.f;
    qp[nt][0] = qp[nt][1] = qlo[nt][0] = qlo[nt][1] = qse[nt][0] = qse[nt][1] = 0;
  }

  for (long long it = 0;; ++it) {
    const int st = (int)(it % a.stages);
    if (!__all_sync(0xffffffffu, mbar_wait_bounded(&s.full[st], (uint32_t)((it / a.stages) & 1), s.abort_flag,
                                                   a.err, kWaitLimitNs)))
      return;
    const volatile StageHdr* vh = &s.hdr[st];
    const int live = vh->live;
    if (!live) return;
    const int vm = vh->vmask;
    const int flags = vh->flags;
    const uint32_t sbase = stages_u32 + (uint32_t)st * (uint32_t)s.stage_bytes;

    if (flags & 1) {  // first stage of a piece: Q^T fragments, reset state
      const int qi = (flags >> 2) & 1;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        // column (token j, head hh) of the KV head; Q is [M][HG * G][D] in shared memory
        const int col = col0 + nt * 8 + (lane & 7);
        const int qrow = col < C ? (col / G) * HG * G + h * G + col % G : 0;
        const uint32_t row = qbuf_u32 + (uint32_t)qi * (uint32_t)s.qbytes + (uint32_t)(qrow * kD * 2) +
                             (uint32_t)(lane >> 3) * 16u;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          uint32_t r[4];
          ldmatrix_x4(r, row + kk * 64);
          qf[2 * kk][nt][0] = r[0];
          qf[2 * kk][nt][1] = r[1];
          qf[2 * kk + 1][nt][0] = r[2];
          qf[2 * kk + 1][nt][1] = r[3];
        }
        if (col0 + nt * 8 + g >= C) {
#pragma unroll
          for (int k = 0; k < 8; ++k) qf[k][nt][0] = qf[k][nt][1] = 0u;
        }
        if (M > 1) {
          const int Lh = vh->L;
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int cj = min(col0 + nt * 8 + 2 * c + e, C - 1) / G;
            const int p = Lh - M + cj;
            const Span sq = attend_span(p + 1, a.window, a.sinks);
            qp[nt][e] = p;
            qlo[nt][e] = sq.lo;
            qse[nt][e] = sq.se;
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&s.qempty[(flags >> 4) & (kQBars - 1)]);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        m[nt][0] = m[nt][1] = -INFINITY;
        l[nt][0] = l[nt][1] = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) o[i][nt][0] = o[i][nt][1] = o[i][nt][2] = o[i][nt][3] = 0.f;
      }
    }

    if (vm != 0xffff) {  // rows without data: zero this head's V so that 0 * garbage cannot be NaN
      for (int r = lane >> 4; r < kTok; r += 2) {
        if (!((vm >> r) & 1)) {
          uint4* p = reinterpret_cast<uint4*>(s.stages + (size_t)st * s.stage_bytes + (kTok + r) * s.pitch + h * 256) +
                     (lane & 15);
          *p = make_uint4(0u, 0u, 0u, 0u);
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
    }

    // S^T = K . Q^T, two accumulator chains.
    float sa[NT][4], sb[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) sa[nt][e] = sb[nt][e] = 0.f;
    const bool pg = flags & 8;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      uint32_t af[4];
      const uint32_t chunk = (uint32_t)(((k & 3) << 1) | (lane >> 4));
      ldmatrix_x4(af, pg ? sbase + (uint32_t)(k >> 2) * box + kp_row + ((chunk ^ sw) << 4) : sbase + k_off + k * 32);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        if (k & 1)
          mma_bf16_16816(sb[nt], af, qf[k][nt][0], qf[k][nt][1]);
        else
          mma_bf16_16816(sa[nt], af, qf[k][nt][0], qf[k][nt][1]);
      }
    }

    // Online softmax over the stage's 16 tokens (rows g and g+8 of S^T).
    const bool va = (vm >> g) & 1, vb = (vm >> (g + 8)) & 1;
    const int ta = vh->t0 + g, tb = ta + 8;  // positions of rows g and g+8
    uint32_t pb[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      bool va0 = va, va1 = va, vb0 = vb, vb1 = vb;
      if (M > 1) {  // causal window of each column's query token
        va0 = va0 && ta <= qp[nt][0] && (ta >= qlo[nt][0] || ta < qse[nt][0]);
        va1 = va1 && ta <= qp[nt][1] && (ta >= qlo[nt][1] || ta < qse[nt][1]);
        vb0 = vb0 && tb <= qp[nt][0] && (tb >= qlo[nt][0] || tb < qse[nt][0]);
        vb1 = vb1 && tb <= qp[nt][1] && (tb >= qlo[nt][1] || tb < qse[nt][1]);
      }
      const float x0 = va0 ? (sa[nt][0] + sb[nt][0]) * a.scale_log2 : -INFINITY;
      const float x1 = va1 ? (sa[nt][1] + sb[nt][1]) * a.scale_log2 : -INFINITY;
      const float x2 = vb0 ? (sa[nt][2] + sb[nt][2]) * a.scale_log2 : -INFINITY;
      const float x3 = vb1 ? (sa[nt][3] + sb[nt][3]) * a.scale_log2 : -INFINITY;
      float mx0 = fmaxf(x0, x2), mx1 = fmaxf(x1, x3);
#pragma unroll
      for (int sh = 4; sh < 32; sh <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, sh));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, sh));
      }
      const float mn0 = fmaxf(m[nt][0], mx0), mn1 = fmaxf(m[nt][1], mx1);
      const float b0 = mn0 == -INFINITY ? 0.f : mn0, b1 = mn1 == -INFINITY ? 0.f : mn1;
      const float al0 = exp2f(m[nt][0] - b0), al1 = exp2f(m[nt][1] - b1);
      m[nt][0] = mn0;
      m[nt][1] = mn1;
      const uint32_t X0 = pack_bf16(exp2f(x0 - b0), exp2f(x1 - b1));
      const uint32_t X1 = pack_bf16(exp2f(x2 - b0), exp2f(x3 - b1));
      l[nt][0] = l[nt][0] * al0 + (bf16_lo(X0) + bf16_lo(X1));
      l[nt][1] = l[nt][1] * al1 + (bf16_hi(X0) + bf16_hi(X1));
      pb[nt][0] = movmatrix_trans(X0);
      pb[nt][1] = movmatrix_trans(X1);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        o[i][nt][0] *= al0;
        o[i][nt][1] *= al1;
        o[i][nt][2] *= al0;
        o[i][nt][3] *= al1;
      }
    }

    // O^T += V^T . P^T
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      uint32_t af[4];
      const uint32_t chunk = (uint32_t)(((i & 3) << 1) | ((lane >> 3) & 1));
      ldmatrix_x4_trans(af, pg ? sbase + (uint32_t)(2 + (i >> 2)) * box + vp_row + ((chunk ^ sw) << 4)
                               : sbase + v_off + i * 32);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) mma_bf16_16816(o[i][nt], af, pb[nt][0], pb[nt][1]);
    }
    // Read the rest of the header before the stage can be refilled.
    const int hb = vh->b, hgroup = vh->group, hpart = vh->part;
    __syncwarp();
    if (lane == 0) mbar_arrive(&s.empty[st]);

    if (flags & 2) {  // last stage of the piece: write the result
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          float ls = l[nt][e];
#pragma unroll
          for (int sh = 4; sh < 32; sh <<= 1) ls += __shfl_xor_sync(0xffffffffu, ls, sh);
          const int col = col0 + nt * 8 + 2 * c + e;
          if (col >= C) continue;
          const int cj = col / G;              // query token
          const int qh = h * G + col % G;      // query head within the group
          if (hpart < 0) {
            const float inv = ls > 0.f ? 1.f / ls : 0.f;
            __nv_bfloat16* dst = a.out + (((size_t)hb * M + cj) * a.Hq + (size_t)hgroup * HG * G + qh) * kD;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              dst[16 * i + g] = __float2bfloat16_rn(o[i][nt][e] * inv);
              dst[16 * i + g + 8] = __float2bfloat16_rn(o[i][nt][2 + e] * inv);
            }
          } else {
            const size_t base = ((size_t)hpart * M + cj) * HG * G + qh;
            float* po = a.part_o + base * kD;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              po[16 * i + g] = o[i][nt][e];
              po[16 * i + g + 8] = o[i][nt][2 + e];
            }
            if (g == 0) {
              a.part_ml[base * 2 + 0] = m[nt][e];
              a.part_ml[base * 2 + 1] = ls;
            }
          }
        }
      }
    }
  }
}

template <int NT>
__global__ void __launch_bounds__(32 * (8 + kProducers), 1) tc_decode_kernel(const __grid_constant__ TcArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ PlanState ps;
  const SmemMap s = map_smem(smem, a.HG, a.G * a.M, a.nq, a.stages);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < a.stages; ++i) {
      mbar_init(&s.full[i], 1);
      mbar_init(&s.empty[i], a.CW);
    }
    for (int i = 0; i < kQBars; ++i) mbar_init(&s.qempty[i], a.CW);
    *s.abort_flag = 0;
    fence_mbar_init();
  }
  griddep_wait();  // the previous kernel's writes (new K/V rows, tables) are visible from here on
  griddep_launch_dependents();
  plan_cta(a, s, &ps);
  if (threadIdx.x == 0) a.merge[blockIdx.x] = make_int4(ps.merge_v, ps.merge_ka, ps.merge_sa, (int)blockIdx.x);
  {  // requests whose length or table row is invalid get a zero output
    const int* sN = reinterpret_cast<const int*>(reinterpret_cast<const long long*>(s.stages) + a.B);
    for (int b = blockIdx.x; b < a.B; b += a.num_ctas) {
      if (sN[b] != 0) continue;
      __nv_bfloat16* o = a.out + (size_t)b * a.M * a.Hq * kD;
      for (int i = threadIdx.x; i < a.M * a.Hq * kD; i += blockDim.x) o[i] = __float2bfloat16_rn(0.f);
    }
  }
  __syncthreads();  // the scratch in the stage buffers is free from here on
  if (warp >= a.CW)
    tc_producer(a, s, ps, warp - a.CW, lane);
  else
    tc_consumer<NT>(a, s, warp, lane);
}

// Merge the pieces of the split request recorded by CTA blockIdx.x: one warp
// per query head, M = max m_i, out = sum 2^(m_i-M) o_i / sum 2^(m_i-M) l_i.
__global__ void __launch_bounds__(256) combine_kernel(const CombineArgs a) {
  griddep_wait();
  const int4 mg = a.merge[blockIdx.x];
  if (mg.x < 0) return;
  const int v = mg.x, ka = mg.y, sa = mg.z, kb = mg.w;
  const int b = v / a.n_groups, grp = v % a.n_groups;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  const int pieces = 1 + kb - ka;
  const int MQ = a.M * a.QH;  // columns: query token j, head hl at j * QH + hl
  for (int qhl = blockIdx.y * nw + warp; qhl < MQ; qhl += nw * gridDim.y) {
    float M = -INFINITY;
    for (int i = 0; i < pieces; ++i) {
      const int slot = i == 0 ? sa : 2 * (ka + i);
      M = fmaxf(M, __ldcg(a.part_ml + ((size_t)slot * MQ + qhl) * 2));
    }
    const int cj = qhl / a.QH, hl = qhl % a.QH;
    const size_t orow = (((size_t)b * a.M + cj) * a.Hq + (size_t)grp * a.QH + hl) * a.D;
    for (int d0 = lane * 4; d0 < a.D; d0 += 128) {
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      float Ls = 0.f;
      for (int i = 0; i < pieces; ++i) {
        const size_t pi = (size_t)(i == 0 ? sa : 2 * (ka + i)) * MQ + qhl;
        const float mi = __ldcg(a.part_ml + pi * 2), li = __ldcg(a.part_ml + pi * 2 + 1);
        const float wgt = (mi == -INFINITY) ? 0.f : exp2f(mi - M);
        Ls += wgt * li;
        const float4 o = __ldcg(reinterpret_cast<const float4*>(a.part_o + pi * a.D + d0));
        acc.x += wgt * o.x;
        acc.y += wgt * o.y;
        acc.z += wgt * o.z;
        acc.w += wgt * o.w;
      }
      const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
      __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out) + orow + d0;
      out[0] = __float2bfloat16_rn(acc.x * inv);
      out[1] = __float2bfloat16_rn(acc.y * inv);
      out[2] = __float2bfloat16_rn(acc.z * inv);
      out[3] = __float2bfloat16_rn(acc.w * inv);
    }
  }
}

}  // namespace

size_t tc_smem_bytes(int HG, int C, int nq, int S) {
  if (S < 3 || S > kMaxStages) return 0;
  const size_t bytes = kAlignSlack + (size_t)S * stage_stride(HG) + (size_t)nq * HG * C * kD * 2 +
                       kProducers * kQueue * (sizeof(StageMeta) + kTok * sizeof(int)) + S * sizeof(StageHdr) +
                       (2 * S + kQBars) * sizeof(uint64_t) + 16;
  // the dynamic allocation plus the kernel's static shared memory (under
  // kStaticSmemBound) must fit one block
  return bytes <= kMaxDynamicSmem ? bytes : 0;
}

int tc_num_qbuf(int HG, int C, int S) {
  if (tc_smem_bytes(HG, C, 2, S)) return 2;
  return tc_smem_bytes(HG, C, 1, S) ? 1 : 0;
}

int tc_num_stages(int HG, int C) {
  // about 192 KB of K/V in flight per SM, whatever the group's row size
  int S = 24 / HG;
  S = S < 3 ? 3 : (S > kMaxStages ? kMaxStages : S);
  while (S > 3 && !tc_smem_bytes(HG, C, 1, S)) --S;
  return S;
}

bool tc_encode_tmap(const kvp_pool* pool, int HG, CUtensorMap* out) {
  static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  static bool looked_up = false;
  if (!looked_up) {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    looked_up = true;
  }
  if (!encode || pool->dtype != KVP_BF16 || pool->head_dim != kD) return false;
  cuuint64_t dims[4] = {(cuuint64_t)kD, (cuuint64_t)pool->num_slots, (cuuint64_t)pool->kv_heads,
                        (cuuint64_t)(2 * pool->num_layers)};
  cuuint64_t strides[3] = {(cuuint64_t)pool->row_bytes, (cuuint64_t)kD * 2, (cuuint64_t)pool->layer_bytes};
  cuuint32_t box[4] = {64, (cuuint32_t)kTok, (cuuint32_t)HG, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return encode(out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, pool->buf, dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int tc_max_batch(int HG, int S) {
  const size_t scratch = (size_t)S * stage_stride(HG);
  return (int)(scratch / kPlanScratchPerRequest);
}

cudaError_t launch_tc(const TcArgs& a, const CombineArgs& cb, cudaStream_t stream, void* ev_before, void* ev_after) {
  const size_t smem = tc_smem_bytes(a.HG, a.G * a.M, a.nq, a.stages);
  if (smem == 0 || a.NT < 1 || a.NT > 2 || a.CW != a.HG * a.tiles || a.CW > 8 || a.tiles * 8 * a.NT < a.G * a.M ||
      a.M > 32 || a.B > tc_max_batch(a.HG, a.stages))
    return cudaErrorInvalidValue;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.num_ctas);
  cfg.blockDim = dim3(32 * (a.CW + kProducers));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e;
  if (ev_before && (e = cudaEventRecord(static_cast<cudaEvent_t>(ev_before), stream)) != cudaSuccess) return e;
  if (a.NT == 1) {
    static bool attr1 = false;
    if (!attr1) {
      e = cudaFuncSetAttribute(tc_decode_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxDynamicSmem);
      if (e != cudaSuccess) return e;
      attr1 = true;
    }
    e = cudaLaunchKernelEx(&cfg, tc_decode_kernel<1>, a);
  } else {
    static bool attr2 = false;
    if (!attr2) {
      e = cudaFuncSetAttribute(tc_decode_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxDynamicSmem);
      if (e != cudaSuccess) return e;
      attr2 = true;
    }
    e = cudaLaunchKernelEx(&cfg, tc_decode_kernel<2>, a);
  }
  if (e != cudaSuccess) return e;
  if (ev_after && (e = cudaEventRecord(static_cast<cudaEvent_t>(ev_after), stream)) != cudaSuccess) return e;
  cudaLaunchConfig_t cc = {};
  cc.gridDim = dim3(a.num_ctas, (cb.M * cb.QH + 7) / 8);
  cc.blockDim = dim3(256);
  cc.dynamicSmemBytes = 0;
  cc.stream = stream;
  cc.attrs = attr;
  cc.numAttrs = 1;
  return cudaLaunchKernelEx(&cc, combine_kernel, cb);
}

}  // namespace kvp
