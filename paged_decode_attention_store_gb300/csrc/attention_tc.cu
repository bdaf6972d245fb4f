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
//   the batch's attended tokens (see the plan kernel), one PRODUCER warp that
//   issues one cp.async.bulk per token row (all KV heads of the group,
//   HG*256 contiguous bytes, K and V) into a 3-stage ring of 16-token stages
//   completed by mbarrier transaction counts, and HG CONSUMER warps, one per
//   KV head.
// * Rows land at a pitch of HG*256+16 bytes, so the 8 rows an ldmatrix reads
//   fall in 8 different 16-byte bank groups.
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
// * An item that covers a whole request writes the final bf16 output; a
//   request split across CTAs writes fp32 partials (max, sum, unnormalised
//   output) for the combine kernel (split-K, flash-decoding style).
// * Every wait is bounded (2 s); on timeout the CTA records KVP_ERR_TIMEOUT,
//   raises its abort flag, waits (bounded) for its own copies and returns.
#include "attention.cuh"

namespace kvp {

namespace {

constexpr int kTok = 16;      // tokens per stage (the MMA M dimension)
constexpr int kStages = 3;    // ring depth
constexpr int kD = 128;       // head_dim
constexpr uint64_t kWaitLimitNs = 2000000000ull;

struct __align__(16) StageHdr {
  int item;    // work item index, -1 = end of work
  int t0;      // first position of the stage
  int vmask;   // bit j: token t0+j has K/V rows in the stage
  int flags;   // 1 first stage of the item, 2 last stage, (qbuf << 2)
};

struct SmemMap {
  int pitch, stage_bytes, qbytes;
  unsigned char* stages;
  unsigned char* qbuf;
  StageHdr* hdr;
  uint64_t* full;
  uint64_t* empty;
  uint64_t* qempty;
  volatile int* abort_flag;
};

__device__ __forceinline__ SmemMap map_smem(unsigned char* smem, int HG, int G) {
  SmemMap s;
  s.pitch = HG * 256 + 16;
  s.stage_bytes = 2 * kTok * s.pitch;
  s.qbytes = HG * G * kD * 2;
  s.stages = smem;
  s.qbuf = smem + kStages * s.stage_bytes;
  s.hdr = reinterpret_cast<StageHdr*>(s.qbuf + 2 * s.qbytes);
  s.full = reinterpret_cast<uint64_t*>(s.hdr + kStages);
  s.empty = s.full + kStages;
  s.qempty = s.empty + kStages;
  s.abort_flag = reinterpret_cast<volatile int*>(s.qempty + 2);
  return s;
}

__device__ __forceinline__ int load_entry(const TableRef& T, int row, int t) {
  const int32_t* r = T.table + (size_t)row * T.cols;
  return __ldg(r + (T.raw ? t : t / T.page_size));
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

// ---------------------------------------------------------------------------
// Producer warp.
// ---------------------------------------------------------------------------
__device__ void tc_producer(const TcArgs& a, const SmemMap& s, int lane) {
  const int HG = a.HG;
  const uint32_t row_copy = (uint32_t)HG * 256u;
  const int j = lane & 15;          // token within the stage
  const bool is_v = lane >= 16;     // lanes 16..31 copy V rows
  const int first = a.cta_first[blockIdx.x];
  const int end = a.cta_first[blockIdx.x + 1];

  long long issued = 0;  // stages issued
  int started = 0;       // items started
  bool ok = true;

  int idx = first;
  WorkItem w{};
  if (idx < end) w = a.items[idx];
  WorkItem wn = (idx + 1 < end) ? a.items[idx + 1] : w;
  int t0 = w.t_begin;
  int entry = (idx < end && t0 + j < w.t_end) ? load_entry(a.T, w.row, t0 + j) : -1;

  while (idx < end) {
    // Look one stage ahead: which stage comes next, and its table entry.
    int idx2 = idx, t02 = t0 + kTok;
    WorkItem w2 = w;
    if (t02 >= w.t_end) {
      idx2 = idx + 1;
      w2 = wn;
      t02 = wn.t_begin;
      if (idx2 < end) wn = (idx2 + 1 < end) ? a.items[idx2 + 1] : wn;
    }
    const int entry2 = (idx2 < end && t02 + j < w2.t_end) ? load_entry(a.T, w2.row, t02 + j) : -1;

    const bool first_stage = (t0 == w.t_begin);
    const bool last_stage = (t0 + kTok >= w.t_end);
    const int qi = started & 1;
    if (first_stage && started >= 2) {
      ok = __all_sync(0xffffffffu,
                      mbar_wait_bounded(&s.qempty[qi], ((started - 2) >> 1) & 1, s.abort_flag, a.err, kWaitLimitNs));
      if (!ok) break;
    }
    const int st = (int)(issued % kStages);
    if (issued >= kStages) {
      ok = __all_sync(0xffffffffu, mbar_wait_bounded(&s.empty[st], (uint32_t)((issued / kStages - 1) & 1),
                                                     s.abort_flag, a.err, kWaitLimitNs));
      if (!ok) break;
    }
    const bool has_row = (t0 + j < w.t_end);
    const int slot = has_row ? entry_to_slot(a.T, entry, t0 + j, a.err) : -1;
    const unsigned copies = __ballot_sync(0xffffffffu, slot >= 0);
    if (lane == 0) {
      StageHdr h;
      h.item = idx;
      h.t0 = t0;
      h.vmask = (int)(copies & copies >> 16 & 0xffffu);
      h.flags = (first_stage ? 1 : 0) | (last_stage ? 2 : 0) | (qi << 2);
      s.hdr[st] = h;
      const uint32_t tx = (uint32_t)__popc(copies) * row_copy + (first_stage ? (uint32_t)s.qbytes : 0u);
      mbar_arrive_expect_tx(&s.full[st], tx);
    }
    __syncwarp();
    if (slot >= 0) {
      const char* src = a.kv_layer + (is_v ? a.kv_bytes : 0) + (size_t)slot * a.row_bytes + (size_t)w.group * row_copy;
      unsigned char* dst = s.stages + (size_t)st * s.stage_bytes + (is_v ? kTok * s.pitch : 0) + j * s.pitch;
      bulk_g2s(dst, src, row_copy, &s.full[st]);
    }
    if (first_stage && lane == 0) {
      const __nv_bfloat16* qsrc = a.q + ((size_t)w.b * a.Hq + (size_t)w.group * HG * a.G) * kD;
      bulk_g2s(s.qbuf + qi * s.qbytes, qsrc, (uint32_t)s.qbytes, &s.full[st]);
    }
    ++issued;
    if (last_stage) ++started;
    idx = idx2;
    w = w2;
    t0 = t02;
    entry = entry2;
  }

  if (ok) {
    const int st = (int)(issued % kStages);
    if (issued >= kStages)
      ok = __all_sync(0xffffffffu, mbar_wait_bounded(&s.empty[st], (uint32_t)((issued / kStages - 1) & 1),
                                                     s.abort_flag, a.err, kWaitLimitNs));
    if (ok && lane == 0) {
      s.hdr[st].item = -1;
      mbar_arrive(&s.full[st]);
    }
  }
  if (!ok) {
    // Abort: let the copies this warp issued land before the CTA exits.
    *s.abort_flag = 1;
    const long long from = issued > kStages ? issued - kStages : 0;
    for (long long k = from; k < issued; ++k) {
      const int st = (int)(k % kStages);
      const uint64_t t_start = global_timer_ns();
      while (!mbar_try_wait(&s.full[st], (uint32_t)((k / kStages) & 1))) {
        if (global_timer_ns() - t_start > 100000000ull) break;
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Consumer warps: one KV head each.
// ---------------------------------------------------------------------------
template <int NT>
__device__ void tc_consumer(const TcArgs& a, const SmemMap& s, int h, int lane) {
  const int G = a.G, HG = a.HG;
  const int g = lane >> 2, c = lane & 3;
  const uint32_t stages_u32 = smem_u32(s.stages);
  const uint32_t qbuf_u32 = smem_u32(s.qbuf);
  // ldmatrix row addresses of this lane (see the fragment layouts of
  // mma.m16n8k16: K as A[token][d], V^T as A[d][token] via .trans).
  const uint32_t k_off = (uint32_t)(((lane & 7) + ((lane >> 3) & 1) * 8) * s.pitch + h * 256 + (lane >> 4) * 16);
  const uint32_t v_off =
      (uint32_t)(kTok * s.pitch + ((lane & 7) + (lane >> 4) * 8) * s.pitch + h * 256 + ((lane >> 3) & 1) * 16);

  uint32_t qf[8][NT][2];
  float o[8][NT][4];
  float m[NT][2], l[NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    m[nt][0] = m[nt][1] = -INFINITY;
    l[nt][0] = l[nt][1] = 0.f;
  }

  for (long long it = 0;; ++it) {
    const int st = (int)(it % kStages);
    if (!__all_sync(0xffffffffu, mbar_wait_bounded(&s.full[st], (uint32_t)((it / kStages) & 1), s.abort_flag,
                                                   a.err, kWaitLimitNs)))
      return;
    const volatile StageHdr* vh = &s.hdr[st];
    StageHdr hd;
    hd.item = vh->item;
    hd.t0 = vh->t0;
    hd.vmask = vh->vmask;
    hd.flags = vh->flags;
    if (hd.item < 0) return;
    const uint32_t sbase = stages_u32 + (uint32_t)st * (uint32_t)s.stage_bytes;

    if (hd.flags & 1) {  // first stage of an item: Q^T fragments, reset state
      const int qi = (hd.flags >> 2) & 1;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const int head = nt * 8 + (lane & 7);
        const uint32_t row = qbuf_u32 + (uint32_t)qi * (uint32_t)s.qbytes +
                             (uint32_t)((head < G ? h * G + head : 0) * kD * 2) + (uint32_t)(lane >> 3) * 16u;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          uint32_t r[4];
          ldmatrix_x4(r, row + kk * 64);
          qf[2 * kk][nt][0] = r[0];
          qf[2 * kk][nt][1] = r[1];
          qf[2 * kk + 1][nt][0] = r[2];
          qf[2 * kk + 1][nt][1] = r[3];
        }
        if (nt * 8 + g >= G) {
#pragma unroll
          for (int k = 0; k < 8; ++k) qf[k][nt][0] = qf[k][nt][1] = 0u;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&s.qempty[qi]);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        m[nt][0] = m[nt][1] = -INFINITY;
        l[nt][0] = l[nt][1] = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) o[i][nt][0] = o[i][nt][1] = o[i][nt][2] = o[i][nt][3] = 0.f;
      }
    }

    const int vm = hd.vmask;
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
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      uint32_t af[4];
      ldmatrix_x4(af, sbase + k_off + k * 32);
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
    uint32_t pb[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const float x0 = va ? (sa[nt][0] + sb[nt][0]) * a.scale_log2 : -INFINITY;
      const float x1 = va ? (sa[nt][1] + sb[nt][1]) * a.scale_log2 : -INFINITY;
      const float x2 = vb ? (sa[nt][2] + sb[nt][2]) * a.scale_log2 : -INFINITY;
      const float x3 = vb ? (sa[nt][3] + sb[nt][3]) * a.scale_log2 : -INFINITY;
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
      ldmatrix_x4_trans(af, sbase + v_off + i * 32);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) mma_bf16_16816(o[i][nt], af, pb[nt][0], pb[nt][1]);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&s.empty[st]);

    if (hd.flags & 2) {  // last stage of the item: write the result
      const WorkItem w = a.items[hd.item];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          float ls = l[nt][e];
#pragma unroll
          for (int sh = 4; sh < 32; sh <<= 1) ls += __shfl_xor_sync(0xffffffffu, ls, sh);
          const int hh = nt * 8 + 2 * c + e;
          if (hh >= G) continue;
          const int qh = h * G + hh;  // query head within the group
          if (w.part < 0) {
            const float inv = ls > 0.f ? 1.f / ls : 0.f;
            __nv_bfloat16* dst = a.out + ((size_t)w.b * a.Hq + (size_t)w.group * HG * G + qh) * kD;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              dst[16 * i + g] = __float2bfloat16_rn(o[i][nt][e] * inv);
              dst[16 * i + g + 8] = __float2bfloat16_rn(o[i][nt][2 + e] * inv);
            }
          } else {
            const size_t base = (size_t)w.part * HG * G + qh;
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
__global__ void __launch_bounds__(32 * 9, 1) tc_decode_kernel(const TcArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  const SmemMap s = map_smem(smem, a.HG, a.G);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&s.full[i], 1);
      mbar_init(&s.empty[i], a.HG);
    }
    mbar_init(&s.qempty[0], a.HG);
    mbar_init(&s.qempty[1], a.HG);
    *s.abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (warp == a.HG)
    tc_producer(a, s, lane);
  else
    tc_consumer<NT>(a, s, warp, lane);
}

}  // namespace

size_t tc_smem_bytes(int HG, int G) {
  const size_t pitch = (size_t)HG * 256 + 16;
  const size_t bytes = kStages * 2 * kTok * pitch + 2 * (size_t)HG * G * kD * 2 + kStages * sizeof(StageHdr) +
                       (2 * kStages + 2) * sizeof(uint64_t) + 16;
  return bytes <= 232448 ? bytes : 0;
}

cudaError_t launch_tc(const TcArgs& a, int num_ctas, cudaStream_t stream) {
  const size_t smem = tc_smem_bytes(a.HG, a.G);
  if (smem == 0 || a.G > 16 || a.HG > 8) return cudaErrorInvalidValue;
  const dim3 block(32 * (a.HG + 1));
  cudaError_t e;
  if (a.G <= 8) {
    static bool attr1 = false;
    if (!attr1) {
      e = cudaFuncSetAttribute(tc_decode_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, 232448);
      if (e != cudaSuccess) return e;
      attr1 = true;
    }
    tc_decode_kernel<1><<<num_ctas, block, smem, stream>>>(a);
  } else {
    static bool attr2 = false;
    if (!attr2) {
      e = cudaFuncSetAttribute(tc_decode_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, 232448);
      if (e != cudaSuccess) return e;
      attr2 = true;
    }
    tc_decode_kernel<2><<<num_ctas, block, smem, stream>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace kvp
