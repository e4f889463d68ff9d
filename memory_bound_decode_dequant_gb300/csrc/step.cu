// step.cu -- the whole decode step as one persistent kernel.
//
// The step ("infer" page, data-flow figure) is a chain of phases -- per layer: QKV
// GEMV with RMSNorm prologue and RoPE + paged K/V write; attention; O-proj + residual;
// gate/up + SwiGLU with RMSNorm prologue; down + residual; then the LM head with
// argmax.  Launched as separate kernels every phase pays launch, ramp-up and tail
// (about 7 us measured on GB300).  Here one cooperative grid of one CTA per SM runs
// them all:
//  * The weights of every GEMV phase are known before the step starts, so the
//    producer warp of each CTA streams its share of all of them, phase after phase,
//    through a ring of shared-memory stages (TMA bulk copies, mbarrier handoff) and
//    never waits for activations -- only for a free slot.  HBM stays busy across phase
//    boundaries; the ring absorbs the synchronisation latency.
//  * Consumer warps run the phases in order.  There is no grid barrier: every phase
//    writes its output vector as tagged 64-bit words (value | launch tag), each in its
//    own buffer, and the next phase polls the words it needs until they carry this
//    launch's tag.  A phase boundary so costs one round trip to L2 instead of a barrier
//    (atomic, then polling a counter) followed by the loads of the vector.  The last CTA
//    to finish advances the tag for the next launch.
//  * A wait that gives up sets a global abort flag (every CTA then leaves), latches an
//    error the host reads back, and drains this CTA's copies still in flight.
#include "attn_core.cuh"

namespace mie {

// Eight consumer warps + one producer warp.  Measured and not kept: seven consumer
// warps (a 256-thread CTA may use 255 registers a thread instead of 168) left the down
// projection with four active warps per stage and slowed the step by 6 %.
constexpr int kPW = 8;                     // consumer warps
constexpr int kPThreads = 32 * (kPW + 1);  // + one producer warp
constexpr int kPCT = kPW * 32;             // consumer threads
constexpr int kPRingMax = 32;              // ring slots (static mbarriers)

struct ConsSync {
  __device__ static void sync() { asm volatile("bar.sync 1, %0;" ::"n"(kPCT) : "memory"); }
  // barrier that also returns whether v holds on every consumer thread
  __device__ static bool all(bool v) {
    int r;
    asm volatile(
        "{\n .reg .pred p, q;\n setp.ne.s32 p, %1, 0;\n bar.red.and.pred q, 1, %2, p;\n selp.s32 %0, 1, 0, q;\n}"
        : "=r"(r)
        : "r"((int)v), "n"(kPCT)
        : "memory");
    return r != 0;
  }
};

__device__ __forceinline__ int ld_volatile(const int *p) { return *reinterpret_cast<const volatile int *>(p); }

__device__ __forceinline__ unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// Optional timeline: thread 0 of each CTA stamps kTracePoints moments of each phase.
__device__ __forceinline__ void stamp(unsigned long long *trace, int phase, int point) {
  if (trace && threadIdx.x == 0) trace[((size_t)phase * gridDim.x + blockIdx.x) * kTracePoints + point] = globaltimer();
}

// Optional per-stage stamps (the producer lane, or consumer thread 0), compiled only into
// an instrumented build (MIE_STAGE_TRACE defined): in the stage loops they would cost
// registers that the Q4_0 kernels do not have.
#ifdef MIE_STAGE_TRACE
__shared__ unsigned long long *s_stage_trace;
__device__ __forceinline__ void stage_stamp(int s, int point) {
  unsigned long long *tr = *reinterpret_cast<unsigned long long *volatile *>(&s_stage_trace);
  if (tr && s < kStageTrace) tr[((size_t)blockIdx.x * kStageTrace + s) * kStagePoints + point] = globaltimer();
}
#define STAGE_STAMP(cond, s, point) \
  do {                              \
    if (cond) stage_stamp(s, point); \
  } while (0)
// Points inside a phase, after the stage stamps: [n_phases][grid][8] (thread 0).
__shared__ int s_cur_phase;
__device__ __forceinline__ void sub_stamp(int point) {
  unsigned long long *tr = *reinterpret_cast<unsigned long long *volatile *>(&s_stage_trace);
  if (tr && threadIdx.x == 0) {
    tr += (size_t)gridDim.x * kStageTrace * kStagePoints;
    tr[((size_t)*reinterpret_cast<volatile int *>(&s_cur_phase) * gridDim.x + blockIdx.x) * 8 + point] = globaltimer();
  }
}
#define SUB_STAMP(point) sub_stamp(point)
#else
#define SUB_STAMP(point) \
  do {                   \
  } while (0)
#define STAGE_STAMP(cond, s, point) \
  do {                              \
  } while (0)
#endif

// Values fixed for the whole step, read once per launch: the launch's tag, the token
// and position, the block ids of the context (when it has at most kStepMaxBlocks
// blocks) and the RoPE angles of the position.  Later phases read them from shared
// memory instead of chasing pointers in global memory.
constexpr int kStepMaxBlocks = 512;
struct StepConst {
  uint32_t tag;
  int tok, pos;
  int ctx;           // attention context: pos + 1, clamped to the block table
  int n_table;       // block-table entries of the slot
  const int32_t *bt; // the slot's block table
  int nblk_staged;
  int blk[kStepMaxBlocks];
  float rc[64], rs[64];
};

// The attention context of the step: positions 0..pos, clamped to the n_table blocks
// the table holds (the clamp is reported as a position error).
__device__ __forceinline__ int attn_ctx(int pos, int n_table, int bs) {
  int ctx = pos + 1;
  if (ctx > n_table * bs) ctx = n_table * bs;
  return ctx < 0 ? 0 : ctx;
}

struct PersistShared {
  float red[kPW];
  float bv[kPW];
  int bi[kPW];
  unsigned last;
  int ok;
};

// Row range of this CTA for a GEMV phase (units of RU rows, balanced over the grid).
struct RowRange {
  int u0, u1, row0, row1, KS, WR, RPS, n_stages;  // WR: warps per slice column; RPS = WR * rows per warp
};

__device__ __forceinline__ RowRange row_range(const DevMat &m, int epi) {
  RowRange r;
  const int RU = (epi == EPI_SWIGLU || epi == EPI_QKV) ? 2 : 1;
  const int n_units = (m.rows + RU - 1) / RU;
  r.u0 = (int)((int64_t)blockIdx.x * n_units / gridDim.x);
  r.u1 = (int)((int64_t)(blockIdx.x + 1) * n_units / gridDim.x);
  r.row0 = r.u0 * RU;
  r.row1 = min(r.u1 * RU, m.rows);
  r.KS = (m.kp + kSlice - 1) / kSlice;
  r.WR = r.KS >= kPW ? 1 : kPW / r.KS;
  r.RPS = r.WR * fmt_rows_per_warp(m.fmt);
  r.n_stages = r.row1 > r.row0 ? (r.row1 - r.row0 + r.RPS - 1) / r.RPS : 0;
  return r;
}

struct Ring {
  uint8_t *w, *sc;
  uint32_t slot_bytes, slot_sc_bytes;
  int nst;
  uint64_t *full, *empty;
};

// ---------------------------------------------------------------------- GEMV phase

// The QKV epilogue for pair unit u, tagged variant: RoPE on q and k rows; k and v
// rounded to bf16 go into the paged cache; q | k | v go out as tagged words for the
// attention phase.  x0, x1 are the GEMV results of rows i and i + hd/2 of head h.
__device__ __forceinline__ void qkv_store_tagged(const GemvArgs &a, const QkvPrefetch &q, int u, float x0, float x1,
                                                 uint32_t tag) {
  const int h2 = a.hd / 2;
  const int h = u / h2, i = u % h2;
  if (h < a.Hq + a.Hkv && q.pos_ok) {
    const float c = q.crow[i], sn = q.srow[i];
    const float r0 = x0 * c - x1 * sn, r1 = x1 * c + x0 * sn;
    x0 = r0;
    x1 = r1;
  }
  if (h >= a.Hq) {
    x0 = round_bf16(x0);
    x1 = round_bf16(x1);
    if (q.blk_ok) {
      const int isv = h >= a.Hq + a.Hkv;
      const int g = h - a.Hq - (isv ? a.Hkv : 0);
      uint16_t *dst = a.kv_layer + (int64_t)q.blk * a.block_stride + (int64_t)isv * a.Hkv * a.bs * a.hd +
                      ((int64_t)g * a.bs + q.pos % a.bs) * a.hd;
      dst[i] = (uint16_t)(__float_as_uint(x0) >> 16);
      dst[i + h2] = (uint16_t)(__float_as_uint(x1) >> 16);
    }
  }
  st_tagged(a.y_t + (int64_t)h * a.hd + i, x0, tag);
  st_tagged(a.y_t + (int64_t)h * a.hd + i + h2, x1, tag);
}

__device__ __forceinline__ void give_up(const PersistArgs &pa) {
  if (threadIdx.x == 0) {
    atomicExch(pa.abort, 1);
    latch_error(pa.err, ERR_TIMEOUT);
  }
}

template <int F>
__device__ bool gemv_phase(const Phase &ph, const Ring &ring, int &s_global, float *scratch, PersistShared &ps,
                           const StepConst &sc, const PersistArgs &pa, int pidx) {
  using T = FmtT<F>;
  constexpr int EPC = T::EPC, CPL = T::CPL;
  constexpr int kBitsPerElem = (F == MIE_FMT_BF16) ? 16 : (F == MIE_FMT_I8 ? 8 : 4);
  constexpr int kSliceBytes = kSlice * kBitsPerElem / 8;
  const GemvArgs &a = ph.g;
  const DevMat &m = a.m;
  const int Kp = m.kp, K = m.cols, M = m.rows;
  const RowRange rr = row_range(m, ph.epi);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t tag = sc.tag;
  const bool has_rows = rr.row1 > rr.row0;
  float *xs = scratch;                            // [xs_floats(Kp)], element k at xs_at(k)
  float *part = xs + xs_floats(Kp);               // [rows of this CTA][KS]
  float *resv = part + (rr.row1 - rr.row0) * rr.KS;  // EPI_RESID: residual of this CTA's rows

  QkvPrefetch qp;
  if (ph.epi == EPI_QKV) {
    qp.pos = sc.pos;
    qp.pos_ok = sc.pos >= 0 && sc.pos < a.max_pos && sc.pos / a.bs < sc.n_table;
    const int b = qp.pos_ok ? sc.pos / a.bs : 0;
    qp.blk = (b < sc.nblk_staged) ? sc.blk[b] : sc.bt[b];
    qp.blk_ok = qp.pos_ok && qp.blk >= 0 && qp.blk < a.n_kv_blocks;
    qp.crow = sc.rc;
    qp.srow = sc.rs;
  }

  // input: the gains and the embedding are constants, loaded before the tagged words
  // of the previous phases are polled; the residual rows are polled with the input
  if (has_rows) {
    constexpr int B = 8;
    const bool one_batch = ph.pro != PRO_PLAIN && K <= kPCT * B;
    float g0[B], sq = 0.f;
    if (one_batch) {
#pragma unroll
      for (int j = 0; j < B; ++j) g0[j] = __ldg(a.gain + min(tid + j * kPCT, K - 1));
    }
    if (ph.epi == EPI_RESID && !a.res_t)
      for (int r = rr.row0 + tid; r < rr.row1; r += kPCT) resv[r - rr.row0] = embed_at(a.embed, sc.tok, r);
    if (ph.pro == PRO_EMBED_NORM) {
      for (int k0 = tid; k0 < Kp; k0 += kPCT * B) {
        float v[B];
#pragma unroll
        for (int j = 0; j < B; ++j) v[j] = embed_at(a.embed, sc.tok, min(k0 + j * kPCT, K - 1));
#pragma unroll
        for (int j = 0; j < B; ++j) {
          const int k = k0 + j * kPCT;
          if (k < Kp) xs[xs_at(k)] = (k < K) ? v[j] : 0.f;
          if (k < K) sq = fmaf(v[j], v[j], sq);
        }
      }
    }
    const int n_in = (ph.pro == PRO_EMBED_NORM) ? 0 : (K + 1) / 2;
    const int n_res = (ph.epi == EPI_RESID && a.res_t) ? rr.row1 - rr.row0 : 0;
    bool ok = poll_pairs<kPCT, B>(n_in + n_res, tag, pa.abort, pa.wait_polls,
                                  [&](int j, const uint64_t *&src, float *&dst, int &c) {
      if (j < n_in) {
        src = a.x_t + 2 * j;
        dst = xs + xs_at(2 * j);  // a pair never straddles a padding gap
        c = (2 * j + 1 < K) ? 2 : 1;
      } else {
        src = a.res_t + rr.row0 + (j - n_in);
        dst = resv + (j - n_in);
        c = 1;
      }
    }, ph.pro == PRO_NORM ? n_in : 0, &sq);
    if (ph.pro != PRO_EMBED_NORM)
      for (int k = K + tid; k < Kp; k += kPCT) xs[xs_at(k)] = 0.f;
    SUB_STAMP(0);
    if (ph.pro != PRO_PLAIN) {  // the warps' sums of squares ride on the poll's barrier
      sq = warp_sum(sq);
      if (lane == 0) ps.red[warp] = sq;
    }
    if (!ConsSync::all(ok)) {
      give_up(pa);
      return false;
    }
    stamp(pa.trace, pidx, 1);
    normalize_staged<kPCT, ConsSync>(a, ph.pro, xs, K, ps.red, one_batch ? g0 : nullptr, 0.f, true);
    SUB_STAMP(1);
    ConsSync::sync();
  }
  stamp(pa.trace, pidx, 2);

  constexpr int RPW = FmtT<F>::RPW;
  const int ri = warp / rr.KS, ks = warp % rr.KS;
  const bool has_slice = warp < rr.WR * rr.KS;
  const int e0 = ks * kSlice + lane * EPC;
  float2 xr[CPL * EPC / 2];
  float nb[CPL], cs[CPL];
  load_lane_xr<F>(xs, e0, Kp, has_slice, xr, nb, cs);
  SUB_STAMP(2);

  // stream this CTA's stages of the phase; a wait that gives up stops the math, and a
  // warp hands a slot back only after it saw the slot's copy land, so after a failure
  // the producer can never refill a slot whose copy is still in flight
  bool ok = true;
  for (int st = 0; st < rr.n_stages; ++st, ++s_global) {
    const int slot = s_global % ring.nst, k = s_global / ring.nst;
    STAGE_STAMP(tid == 0, s_global, 1);
    if (ok && !mbar_wait_or_abort(&ring.full[slot], k & 1, pa.wait_polls, pa.abort)) {
      ok = false;
      atomicExch(pa.abort, 1);
      latch_error(pa.err, ERR_TIMEOUT);
    }
    STAGE_STAMP(tid == 0, s_global, 2);
    const int r = rr.row0 + st * rr.RPS + ri * RPW;  // this warp's first row of the stage
    if (ok && has_slice && r < rr.row1) {
      const int nr = min(RPW, rr.row1 - r);
      const uint32_t rowa = smem_u32(ring.w) + (uint32_t)slot * ring.slot_bytes + (uint32_t)(ri * RPW * m.row_bytes) +
                            (uint32_t)ks * kSliceBytes;
      const uint32_t sca = smem_u32(ring.sc) + (uint32_t)slot * ring.slot_sc_bytes +
                           (uint32_t)(ri * RPW * m.s_stride + ks * (kSlice >> (5 + m.gshift))) * 2;
      float sum[RPW];
      stage_rows_dot<F>(rowa, (uint32_t)m.row_bytes, sca, (uint32_t)m.s_stride * 2, nr, xr, nb, cs, e0, Kp, lane, sum,
                        m.gshift);
#pragma unroll
      for (int i = 0; i < RPW; ++i) {
        const float v = warp_sum(sum[i]);
        if (lane == 0 && i < nr) part[(r + i - rr.row0) * rr.KS + ks] = v;
      }
    }
    __syncwarp();
    if (lane == 0 && ok) mbar_arrive(&ring.empty[slot]);
    STAGE_STAMP(tid == 0, s_global, 3);
  }
  if (!ConsSync::all(ok)) return false;
  stamp(pa.trace, pidx, 3);

  // epilogue
  auto row_value = [&](int r) {
    float v = 0.f;
    for (int q = 0; q < rr.KS; ++q) v += part[(r - rr.row0) * rr.KS + q];
    if constexpr (F == MIE_FMT_I8) v *= reinterpret_cast<const float *>(m.s)[r];
    return v;
  };
  if (ph.epi == EPI_STORE || ph.epi == EPI_RESID) {
    for (int r = rr.row0 + tid; r < rr.row1; r += kPCT) {
      const float v = row_value(r);
      st_tagged(a.y_t + r, (ph.epi == EPI_RESID) ? resv[r - rr.row0] + v : v, tag);
    }
  } else if (ph.epi == EPI_SWIGLU) {
    for (int u = rr.u0 + tid; u < rr.u1; u += kPCT) {
      const float g = row_value(2 * u), up = row_value(2 * u + 1);
      st_tagged(a.y_t + u, g / (1.0f + expf(-g)) * up, tag);
    }
  } else if (ph.epi == EPI_QKV) {
    if (tid == 0 && blockIdx.x == 0 && !qp.blk_ok) latch_error(pa.err, qp.pos_ok ? ERR_BLOCK_ID : ERR_POS);
    for (int u = rr.u0 + tid; u < rr.u1; u += kPCT)
      qkv_store_tagged(a, qp, u, row_value(2 * u), row_value(2 * u + 1), tag);
  } else if (ph.epi == EPI_ARGMAX) {
    float *logits = a.sp ? a.sp->logits_out : nullptr;
    if (logits) logits += (int64_t)a.slot * M;
    float bv = -INFINITY;
    int bi = 0x7fffffff;
    for (int r = rr.row0 + tid; r < rr.row1; r += kPCT) {
      const float v = row_value(r);
      if (logits) logits[r] = v;
      if (better(v, r, bv, bi)) { bv = v; bi = r; }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (better(ov, oi, bv, bi)) { bv = ov; bi = oi; }
    }
    if (lane == 0) { ps.bv[warp] = bv; ps.bi[warp] = bi; }
    ConsSync::sync();
    if (tid == 0) {
      for (int w = 1; w < kPW; ++w)
        if (better(ps.bv[w], ps.bi[w], bv, bi)) { bv = ps.bv[w]; bi = ps.bi[w]; }
      a.am_part[blockIdx.x] = make_float2(bv, __int_as_float(bi));
      __threadfence();
      ps.last = (atomicAdd(a.am_count, 1u) == gridDim.x - 1);
    }
    ConsSync::sync();
    if (ps.last) {
      __threadfence();
      float fv = -INFINITY;
      int fi = 0x7fffffff;
      for (int b = tid; b < (int)gridDim.x; b += kPCT) {
        const float2 p = __ldcg(a.am_part + b);
        if (better(p.x, __float_as_int(p.y), fv, fi)) { fv = p.x; fi = __float_as_int(p.y); }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, fv, o);
        const int oi = __shfl_xor_sync(0xffffffffu, fi, o);
        if (better(ov, oi, fv, fi)) { fv = ov; fi = oi; }
      }
      ConsSync::sync();
      if (lane == 0) { ps.bv[warp] = fv; ps.bi[warp] = fi; }
      ConsSync::sync();
      if (tid == 0) {
        for (int w = 1; w < kPW; ++w)
          if (better(ps.bv[w], ps.bi[w], fv, fi)) { fv = ps.bv[w]; fi = ps.bi[w]; }
        if (fi == 0x7fffffff) fi = 0;
        if (a.sp) {
          if (a.sp->argmax_out) a.sp->argmax_out[a.slot] = fi;
          if (a.sp->advance) {
            a.sp->token[a.slot] = fi;
            a.sp->pos[a.slot] += 1;
          }
        }
        *a.am_count = 0u;
      }
    }
  }
  return true;
}

// ---------------------------------------------------------------------- attention phase
//
// One attention item = (KV head g, split sp of nsplit).  Its K/V arrive as ring
// stages of up to `cap` whole blocks, K of the stage's token t at byte t*hd*2 and V at
// cap*kb + t*hd*2 (kb = bs*hd*2 bytes per block).  With a whole chunk in shared
// memory the item runs three CTA-wide passes per stage instead of the per-warp online
// softmax of the standalone kernel, whose shuffle chains cost about 5000 cycles per
// 16 tokens at one CTA per SM (measured): (1) a score for every (head, token) pair,
// lanes starting at different 16-byte chunks of their key rows so that the reads
// avoid bank conflicts; (2) one warp per head takes max, exp and sum and rescales
// the running (m, l); (3) every thread accumulates its (head, dim) outputs over the
// chunk.  The softmax is the same two-pass definition, evaluated per stage with the
// running maximum carried across stages.

// Blocks per attention split of the persistent step: 256 tokens (two 128-token ring
// stages at hd 64), so up to that context one CTA per KV head finishes attention
// without a merge (a merge costs a fence, an atomic and a round trip, ~2.5 us); longer
// contexts spread over more CTAs and the last split of each head merges.
__host__ __device__ inline int ring_attn_blocks_per_split(int bs) { return bs >= 256 ? 1 : 256 / bs; }

// Blocks per attention stage: as many as a ring slot holds, at most kChunkTok tokens.
__host__ __device__ inline int attn_stage_blocks(uint32_t slot_bytes, int bs, int hd) {
  const int cap = (int)(slot_bytes / (2u * (uint32_t)bs * hd * 2));
  const int lim = kChunkTok / bs;
  return cap < lim ? cap : lim;
}

// Attention items.  While the context needs few splits, one item per (query head,
// split) spreads the work over Hq * nsplit CTAs (each reads its KV head's K/V for
// itself; the group's other query heads read the same bytes, mostly from L2); longer
// contexts take one item per (KV head, split), whose CTA serves the group's G query
// heads from one read.  The producer walks the items in the same order.
__host__ __device__ inline bool attn_items_per_query_head(int Hq, int Hkv, int nsplit, int grid) {
  return Hq > Hkv && Hq * nsplit <= grid;
}

// One item: unit u of GI query heads from query head h0 on, KV head g, split sp.
template <int GI, int HD>
__device__ bool attn_ring_item(const AttnArgs &at, int u, int g, int h0, int sp, int nsplit, int ctx,
                               const Ring &ring, int &s_global, ChunkSmem<GI, HD> &sm, const StepConst &sc,
                               const PersistArgs &pa) {
  constexpr int G = GI;
  constexpr int NO = (G * HD + kPCT - 1) / kPCT;  // outputs per thread
  static_assert(2 * HD <= kPCT, "one thread per element of the current token's k and v");
  const int tid = threadIdx.x, lane = tid & 31;
  const int nblk = (ctx + at.bs - 1) / at.bs;
  const int b0 = (int)((int64_t)sp * nblk / nsplit), b1 = (int)((int64_t)(sp + 1) * nblk / nsplit);
  const int t_end = min(b1 * at.bs, ctx);
  const int pos = ctx - 1;
  const bool has_pos = t_end == ctx && ctx > 0;
  const int kb = at.bs * HD * 2, cap = attn_stage_blocks(ring.slot_bytes, at.bs, HD);
  if (tid < G) {
    sm.m[tid] = -INFINITY;
    sm.l[tid] = 0.f;
  }
  if (!tagged_inputs<G, HD, kPCT, ConsSync>(at, h0, g, has_pos, sm, sc.tag, pa.abort, pa.wait_polls)) return false;
  SUB_STAMP(3);
  float o[NO];
#pragma unroll
  for (int j = 0; j < NO; ++j) o[j] = 0.f;
  bool ok = true;
  for (int cb = b0; cb < b1; cb += cap, ++s_global) {
    const int slot = s_global % ring.nst, k = s_global / ring.nst;
    STAGE_STAMP(tid == 0, s_global, 1);
    if (ok && !mbar_wait_or_abort(&ring.full[slot], k & 1, pa.wait_polls, pa.abort)) {
      ok = false;
      atomicExch(pa.abort, 1);
      latch_error(pa.err, ERR_TIMEOUT);
    }
    STAGE_STAMP(tid == 0, s_global, 2);
    if (cb == b0) SUB_STAMP(4);
    const uint32_t kbase = smem_u32(ring.w) + (uint32_t)slot * ring.slot_bytes;
    const uint32_t vbase = kbase + (uint32_t)(cap * kb);
    const int t0 = cb * at.bs, ntok = min(min(cb + cap, b1) * at.bs, t_end) - t0;
    if (ok) {
      // the current token's k and v replace what the stage holds at its slot
      if (has_pos && pos >= t0 && pos < t0 + ntok) {
        const uint32_t off = (uint32_t)(pos - t0) * (HD * 2);
        if (tid < HD) sts16(kbase + off + tid * 2, (uint16_t)(__float_as_uint(sm.kn[tid]) >> 16));
        else if (tid < 2 * HD) sts16(vbase + off + (tid - HD) * 2, (uint16_t)(__float_as_uint(sm.vn[tid - HD]) >> 16));
        ConsSync::sync();
      }
      chunk_passes<G, HD, kPCT, ConsSync>(kbase, vbase, ntok, at.scale, sm, o);
      if (cb == b0) SUB_STAMP(5);
    }
    fence_proxy_async_smem();  // the patch above was a generic write into a bulk-copy slot
    __syncwarp();
    if (lane == 0 && ok) mbar_arrive(&ring.empty[slot]);  // only a slot whose copy landed
    STAGE_STAMP(tid == 0, s_global, 3);
    ConsSync::sync();  // the next stage rewrites sm.s
  }
  if (!ConsSync::all(ok)) return false;
  if (nsplit == 1) {
#pragma unroll
    for (int j = 0; j < NO; ++j) {
      const int i = tid + j * kPCT;
      if (i < G * HD) {
        const float L = sm.l[i / HD];
        st_tagged(at.out_t + (int64_t)h0 * HD + i, (L > 0.f) ? o[j] / L : 0.f, sc.tag);
      }
    }
    SUB_STAMP(6);
    ConsSync::sync();  // the scratch is reused by the next item
    return true;
  }
  float *part = at.ws_part + ((int64_t)u * at.n_splits + sp) * (G * (2 + HD));
#pragma unroll
  for (int j = 0; j < NO; ++j) {
    const int i = tid + j * kPCT;
    if (i < G * HD) {
      const int h = i / HD;
      part[2 * G + i] = o[j];
      if (i % HD == 0) {
        part[h] = sm.m[h];
        part[G + h] = sm.l[h];
      }
    }
  }
  attn_merge_splits<G, HD, kPCT, ConsSync, true>(at, u, nsplit, sm.last, sc.tag);
  return true;
}

template <int G, int HD>
__device__ bool attn_phase(const AttnArgs &at, const Ring &ring, int &s_global, float *scratch, const StepConst &sc,
                           const PersistArgs &pa) {
  const int ctx = sc.ctx;
  const int nblk = (ctx + at.bs - 1) / at.bs;
  const int nsplit = attn_nsplit(nblk, at.n_splits, ring_attn_blocks_per_split(at.bs));
  const bool per_q = attn_items_per_query_head(at.Hq, at.Hkv, nsplit, gridDim.x);
  const int items = (per_q ? at.Hq : at.Hkv) * nsplit;
  for (int it = blockIdx.x; it < items; it += gridDim.x) {
    const int u = it / nsplit, sp = it % nsplit;
    const bool ok = per_q ? attn_ring_item<1, HD>(at, u, u / G, u, sp, nsplit, ctx, ring, s_global,
                                                  *reinterpret_cast<ChunkSmem<1, HD> *>(scratch), sc, pa)
                          : attn_ring_item<G, HD>(at, u, u, u * G, sp, nsplit, ctx, ring, s_global,
                                                  *reinterpret_cast<ChunkSmem<G, HD> *>(scratch), sc, pa);
    if (!ok) {
      give_up(pa);
      return false;
    }
  }
  return true;
}

// ---------------------------------------------------------------------- producer
//
// Walks the stages of every phase in order and copies each into the next free ring
// slot: a GEMV stage is RPS whole weight rows (plus their Q4_0 scales); an attention
// stage is the K and V of up to `cap` consecutive context blocks of one KV head, for
// the attention items this CTA runs.  Neither depends on the step's activations, so
// the K/V of old positions are in shared memory before the attention phase starts;
// only the current token's k/v (and q) arrive as tagged words.  Measured on GB300 and
// not kept: prefetching weights into L2 ahead of the ring halved the streaming rate,
// and capping the bytes in flight per CTA slowed streaming without shortening the
// consumers' load latencies.

template <int HD>
struct StageCursor {
  const PersistArgs *a;
  const StepConst *sc;
  int ctx = 0;  // the step's attention context, clamped like the consumers clamp it
  int p = -1, kind = PH_GEMV;
  bool done = false;
  // GEMV phase, held in registers: the issue loop touches no memory
  RowRange rr;
  int st = 0;
  const uint8_t *w = nullptr, *s = nullptr;
  int64_t row_bytes = 0;
  int s_stride = 0;
  bool q4 = false;
  // attention phase
  const uint8_t *kbase = nullptr, *vbase = nullptr;
  int64_t blk_bytes = 0;  // bytes between consecutive pool blocks
  const int32_t *bt = nullptr;
  int n_pool = 0, bs = 0, kb = 0, cap = 0, nblk = 0, nsplit = 1, items = 0, it = 0, cb = 0, b1 = 0;
  int group = 1;  // query heads per item unit's KV head: G for per-query-head items, else 1
  int64_t hoff = 0;

  __device__ bool next_item() {  // this CTA's next attention item with blocks (consumers' order)
    for (it += gridDim.x; it < items; it += gridDim.x) {
      const int g = (it / nsplit) / group, sp = it % nsplit;
      const int b0 = (int)((int64_t)sp * nblk / nsplit);
      b1 = (int)((int64_t)(sp + 1) * nblk / nsplit);
      if (b0 < b1) {
        cb = b0;
        hoff = (int64_t)g * bs * HD * 2;
        return true;
      }
    }
    return false;
  }
  __device__ bool enter(int q) {  // phase q has stages for this CTA
    const Phase &ph = a->ph[q];
    kind = ph.kind;
    if (ph.kind == PH_GEMV) {
      const DevMat m = ph.g.m;
      rr = row_range(m, ph.epi);
      st = 0;
      w = m.w;
      s = reinterpret_cast<const uint8_t *>(m.s);
      row_bytes = m.row_bytes;
      s_stride = m.s_stride;
      q4 = m.fmt == MIE_FMT_Q4_0;
      return rr.n_stages > 0;
    }
    const AttnArgs &at = ph.at;
    kbase = reinterpret_cast<const uint8_t *>(at.k);
    vbase = reinterpret_cast<const uint8_t *>(at.v);
    blk_bytes = at.block_stride * 2;
    n_pool = at.n_pool_blocks;
    bs = at.bs;
    kb = bs * HD * 2;
    cap = attn_stage_blocks(a->slot_bytes, bs, HD);
    nblk = (ctx + bs - 1) / bs;
    nsplit = attn_nsplit(nblk, at.n_splits, ring_attn_blocks_per_split(bs));
    const bool per_q = attn_items_per_query_head(at.Hq, at.Hkv, nsplit, gridDim.x);
    group = per_q ? at.Hq / at.Hkv : 1;
    items = (per_q ? at.Hq : at.Hkv) * nsplit;
    it = (int)blockIdx.x - (int)gridDim.x;
    return next_item();
  }
  __device__ void advance() {
    while (++p < a->n_phases)
      if (enter(p)) return;
    done = true;
  }
  __device__ void next() {
    if (kind == PH_GEMV) {
      if (++st >= rr.n_stages) advance();
    } else {
      cb += cap;
      if (cb >= b1 && !next_item()) advance();
    }
  }
  __device__ int first_row() const { return rr.row0 + st * rr.RPS; }
  __device__ int rows() const { return min(rr.RPS, rr.row1 - first_row()); }
};

template <int HD>
__device__ void produce(const PersistArgs &a, const Ring &ring, const StepConst &sc, volatile int &s_sc_ready,
                        volatile int &s_issued, volatile int &s_prod_done) {
  const uint64_t pol = evict_first_policy();
  StageCursor<HD> ld;
  ld.a = &a;
  ld.sc = &sc;
  {
    const GemvArgs &g0 = a.ph[0].g;
    const StepParams *sp = g0.sp;
    ld.ctx = attn_ctx(sp->pos[g0.slot], sp->max_blocks, g0.bs);
    ld.bt = sp->block_table + (int64_t)g0.slot * sp->max_blocks;
  }
  ld.advance();
  int s_global = 0;
  bool sc_ready = false;
  while (!ld.done) {
    const int slot = s_global % a.n_slots, k = s_global / a.n_slots;
    if (k > 0 && !mbar_wait_or_abort(&ring.empty[slot], (k - 1) & 1, a.wait_polls, a.abort)) {
      atomicExch(a.abort, 1);
      latch_error(a.err, ERR_TIMEOUT);
      break;
    }
    if (ld_volatile(a.abort)) break;
    uint8_t *dst = ring.w + (size_t)slot * a.slot_bytes;
    if (ld.kind == PH_GEMV) {
      const int r = ld.first_row();
      const uint32_t wb = (uint32_t)(ld.rows() * ld.row_bytes);
      const uint32_t sb = ld.q4 ? (uint32_t)(ld.rows() * ld.s_stride * 2) : 0u;
      mbar_expect_tx(&ring.full[slot], wb + sb);
      bulk_load(dst, ld.w + (int64_t)r * ld.row_bytes, wb, &ring.full[slot], pol);
      if (sb)
        bulk_load(ring.sc + (size_t)slot * a.slot_sc_bytes, ld.s + (int64_t)r * ld.s_stride * 2, sb, &ring.full[slot],
                  pol);
    } else {
      if (!sc_ready) {  // the block ids are staged in shared memory by the consumers
        for (long it = 0; it < a.wait_polls && !s_sc_ready; ++it) __nanosleep(64);
        __threadfence_block();
        sc_ready = true;
      }
      const int nb = min(ld.cap, ld.b1 - ld.cb);
      mbar_expect_tx(&ring.full[slot], 2u * nb * ld.kb);
      for (int j = 0; j < nb; ++j) {
        const int b = ld.cb + j;
        int blk = (b < sc.nblk_staged && s_sc_ready) ? sc.blk[b] : ld.bt[b];
        if (blk < 0 || blk >= ld.n_pool) {
          latch_error(a.err, ERR_BLOCK_ID);
          blk = 0;
        }
        const int64_t off = (int64_t)blk * ld.blk_bytes + ld.hoff;
        bulk_load(dst + (size_t)j * ld.kb, ld.kbase + off, ld.kb, &ring.full[slot], pol);
        bulk_load(dst + (size_t)(ld.cap + j) * ld.kb, ld.vbase + off, ld.kb, &ring.full[slot], pol);
      }
    }
    STAGE_STAMP(true, s_global, 0);
    ++s_global;
    s_issued = s_global;
    ld.next();
  }
  s_prod_done = 1;
}

// ---------------------------------------------------------------------- the kernel

template <int FL, int FH, int G, int HD>
__global__ void __launch_bounds__(kPThreads, 1) persistent_step(const PersistArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t full_bar[kPRingMax], empty_bar[kPRingMax];
  __shared__ PersistShared ps;
  __shared__ StepConst sc;
  // descriptors of the current and the next phase, in shared memory; the one after
  // is loaded into registers while the current phase runs
  __shared__ __align__(16) Phase s_ph[2];
  __shared__ volatile int s_issued, s_prod_done, s_sc_ready;
  constexpr int kPhWords = sizeof(Phase) / 4;
  static_assert(sizeof(Phase) % 4 == 0 && kPhWords <= kPCT, "one descriptor word per consumer thread");

  Ring ring;
  ring.nst = a.n_slots;
  ring.slot_bytes = a.slot_bytes;
  ring.slot_sc_bytes = a.slot_sc_bytes;
  ring.w = smem;
  ring.sc = smem + (size_t)a.n_slots * a.slot_bytes;
  ring.full = full_bar;
  ring.empty = empty_bar;
  float *scratch = reinterpret_cast<float *>(ring.sc + (size_t)a.n_slots * a.slot_sc_bytes);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int i = 0; i < a.n_slots; ++i) {
      mbar_init(&full_bar[i], 1);
      mbar_init(&empty_bar[i], kPW);
    }
    s_issued = 0;
    s_prod_done = 0;
    s_sc_ready = 0;
#ifdef MIE_STAGE_TRACE
    s_stage_trace = a.stage_trace;
#endif
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  if (warp == kPW) {
    if (lane == 0) produce<HD>(a, ring, sc, s_sc_ready, s_issued, s_prod_done);
    return;
  }

  // consumers: the step's constants first
  {
    const GemvArgs &g0 = a.ph[0].g;  // layer 0's QKV phase carries the step's tables
    const StepParams *sp = g0.sp;
    const int pos = sp->pos[g0.slot];
    int tok = sp->token[g0.slot];
    const int n_table = sp->max_blocks;
    const int ctx = attn_ctx(pos, n_table, g0.bs);
    const int nblk = (ctx + g0.bs - 1) / g0.bs;
    const int staged = nblk <= kStepMaxBlocks ? nblk : 0;
    const int32_t *bt = sp->block_table + (int64_t)g0.slot * n_table;
    constexpr int kIds = (kStepMaxBlocks + kPCT - 1) / kPCT;
    int ids[kIds];
#pragma unroll
    for (int j = 0; j < kIds; ++j) ids[j] = bt[min(tid + j * kPCT, max(staged - 1, 0))];
#pragma unroll
    for (int j = 0; j < kIds; ++j) {
      const int i = tid + j * kPCT;
      if (i < staged) {
        int b = ids[j];
        if (b < 0 || b >= g0.n_kv_blocks) {
          latch_error(a.err, ERR_BLOCK_ID);
          b = -1;
        }
        sc.blk[i] = b;
      }
    }
    const int h2 = g0.hd / 2;
    const int pos_c = (pos >= 0 && pos < g0.max_pos) ? pos : 0;
    if (tid < h2) {
      sc.rc[tid] = g0.rope_cos[(int64_t)pos_c * h2 + tid];
      sc.rs[tid] = g0.rope_sin[(int64_t)pos_c * h2 + tid];
    }
    if (tid == 0) {
      if (tok < 0 || tok >= g0.vocab) {
        latch_error(a.err, ERR_TOKEN);
        tok = 0;
      }
      if (ctx != pos + 1) latch_error(a.err, ERR_POS);
      sc.tag = __ldcg(a.epoch);
      sc.tok = tok;
      sc.pos = pos;
      sc.ctx = ctx;
      sc.n_table = n_table;
      sc.bt = bt;
      sc.nblk_staged = staged;
    }
  }
  const uint32_t *ph_words = reinterpret_cast<const uint32_t *>(a.ph);
  for (int p = 0; p < 2 && p < a.n_phases; ++p)
    if (tid < kPhWords) reinterpret_cast<uint32_t *>(&s_ph[p])[tid] = __ldcg(ph_words + (size_t)p * kPhWords + tid);
  ConsSync::sync();
  if (tid == 0) {  // the step constants are complete: the producer may read the block ids
    __threadfence_block();
    s_sc_ready = 1;
  }
  int s_global = 0;
  bool ok = true;
  for (int p = 0; p < a.n_phases; ++p) {
    const uint32_t next_word =
        (p + 2 < a.n_phases && tid < kPhWords) ? __ldcg(ph_words + (size_t)(p + 2) * kPhWords + tid) : 0u;
    const Phase &ph = s_ph[p & 1];
#ifdef MIE_STAGE_TRACE
    if (tid == 0) s_cur_phase = p;
#endif
    stamp(a.trace, p, 0);
    if (ph.kind == PH_GEMV) {
      // one inlined copy per distinct format: the kernel's code is kept small so that the
      // phases run once per layer (attention, epilogues) hit the instruction cache
      if constexpr (FL == FH) ok = gemv_phase<FL>(ph, ring, s_global, scratch, ps, sc, a, p);
      else if (ph.g.m.fmt == FL) ok = gemv_phase<FL>(ph, ring, s_global, scratch, ps, sc, a, p);
      else ok = gemv_phase<FH>(ph, ring, s_global, scratch, ps, sc, a, p);
    } else {
      stamp(a.trace, p, 1);
      stamp(a.trace, p, 2);
      ok = attn_phase<G, HD>(ph.at, ring, s_global, scratch, sc, a);
      stamp(a.trace, p, 3);
    }
    ConsSync::sync();
    stamp(a.trace, p, 4);
    if (!ok) break;
    if (p + 2 < a.n_phases && tid < kPhWords) reinterpret_cast<uint32_t *>(&s_ph[p & 1])[tid] = next_word;
  }
  if (ok) {
    // the last CTA to finish advances the tag for the next launch (never 0, the tag of
    // words no launch has written)
    if (tid == 0) {
      __threadfence();
      if (atomicAdd(a.fin, 1u) == gridDim.x - 1) {
        const unsigned next = sc.tag + 1u;
        *a.epoch = next ? next : 1u;
        *a.fin = 0u;
        __threadfence();
      }
    }
    return;
  }
  // a wait gave up: no copy may still be writing into shared memory when we leave
  if (tid == 0) {
    for (long it = 0; it < kWaitPolls && !s_prod_done; ++it) __nanosleep(64);
    const int issued = s_issued;
    for (int s = max(0, issued - a.n_slots); s < issued; ++s) mbar_wait(&full_bar[s % a.n_slots], (s / a.n_slots) & 1);
  }
}

// ---------------------------------------------------------------------- host side

template <int FL, int FH, int G, int HD>
static const void *kernel_ptr() {
  return reinterpret_cast<const void *>(&persistent_step<FL, FH, G, HD>);
}

static const void *pick_kernel(int fl, int fh, int G, int HD) {
#define MIE_K(A, B, C, D) \
  if (fl == A && fh == B && G == C && HD == D) return kernel_ptr<A, B, C, D>();
#define MIE_K_SHAPES(A, B) MIE_K(A, B, 4, 32) MIE_K(A, B, 8, 64) MIE_K(A, B, 4, 64)
  MIE_K_SHAPES(MIE_FMT_BF16, MIE_FMT_BF16)
  MIE_K_SHAPES(MIE_FMT_I8, MIE_FMT_I8)
  MIE_K_SHAPES(MIE_FMT_Q4_0, MIE_FMT_Q4_0)
  MIE_K_SHAPES(MIE_FMT_Q4_0, MIE_FMT_I8)
#undef MIE_K_SHAPES
#undef MIE_K
  return nullptr;
}

size_t persist_attn_smem(int G, int HD) {
  switch (G * 1000 + HD) {
    case 4032: return sizeof(ChunkSmem<4, 32>);
    case 8064: return sizeof(ChunkSmem<8, 64>);
    case 4064: return sizeof(ChunkSmem<4, 64>);
  }
  return 0;
}

mie_status persist_plan(const Phase *host_phases, int n, int G, int HD, PersistPlan *plan) {
  const int grid = sm_count();
  uint32_t slot = 0, slot_sc = 0;
  size_t scratch = persist_attn_smem(G, HD);
  int fl = -1, fh = -1;
  for (int p = 0; p < n; ++p) {
    const Phase &ph = host_phases[p];
    if (ph.kind != PH_GEMV) {  // an attention stage holds the K and V of at least one block
      const uint32_t kv = (uint32_t)(2 * ph.at.bs * HD * 2 + 127) / 128 * 128;
      if (kv > slot) slot = kv;
      continue;
    }
    const DevMat &m = ph.g.m;
    if (fl < 0) fl = m.fmt;
    else if (m.fmt != fl && fh < 0) fh = m.fmt;
    const int RU = (ph.epi == EPI_SWIGLU || ph.epi == EPI_QKV) ? 2 : 1;
    const int n_units = (m.rows + RU - 1) / RU;
    const int KS = (m.kp + kSlice - 1) / kSlice;
    const int RPS = (KS >= kPW ? 1 : kPW / KS) * fmt_rows_per_warp(m.fmt);
    const int rows_max = ((n_units + grid - 1) / grid) * RU;
    const uint32_t sb = (uint32_t)((RPS * m.row_bytes + 127) / 128 * 128);
    const uint32_t scb = m.fmt == MIE_FMT_Q4_0 ? (uint32_t)((RPS * m.s_stride * 2 + 127) / 128 * 128) : 0u;
    if (sb > slot) slot = sb;
    if (scb > slot_sc) slot_sc = scb;
    const size_t need = sizeof(float) * ((size_t)xs_floats(m.kp) + (size_t)rows_max * (KS + 1));
    if (need > scratch) scratch = need;
    if (((uintptr_t)m.w & 15) || (m.row_bytes & 15)) return fail(MIE_E_SHAPE, "persistent step: unaligned rows");
  }
  if (fh < 0) fh = fl;
  if (!pick_kernel(fl, fh, G, HD)) return fail(MIE_E_SHAPE, "persistent step: no kernel for this shape");
  scratch = (scratch + 127) / 128 * 128;
  const void *kern = pick_kernel(fl, fh, G, HD);
  int dev = 0, max_smem = 0;
  cudaFuncAttributes fa;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, kern);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return cuda_fail(e, "persistent step: kernel attributes");
  }
  // dynamic + static shared memory must fit the per-block opt-in limit
  const long avail = (long)max_smem - (long)fa.sharedSizeBytes - (long)scratch - 256;
  int nst = (int)(avail / (long)(slot + slot_sc));
  if (nst > kPRingMax) nst = kPRingMax;
  if (nst < 2) return fail(MIE_E_SHAPE, "persistent step: shared memory too small for the ring");
  plan->kernel = kern;
  plan->grid = grid;
  plan->threads = kPThreads;
  plan->n_slots = nst;
  plan->slot_bytes = slot;
  plan->slot_sc_bytes = slot_sc;
  plan->smem = (size_t)nst * (slot + slot_sc) + scratch;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)plan->smem);
  int blocks = 0;
  if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, kern, kPThreads, plan->smem);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return cuda_fail(e, "persistent step: shared-memory plan");
  }
  if (blocks < 1) return fail(MIE_E_SHAPE, "persistent step: one CTA per SM does not fit");
  return MIE_OK;
}

mie_status persist_launch(const PersistPlan &plan, const PersistArgs &args, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(plan.grid);
  cfg.blockDim = dim3(plan.threads);
  cfg.dynamicSmemBytes = plan.smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  void *params[] = {const_cast<PersistArgs *>(&args)};
  MIE_CUDA(cudaLaunchKernelExC(&cfg, plan.kernel, params));
  return MIE_OK;
}

}  // namespace mie
