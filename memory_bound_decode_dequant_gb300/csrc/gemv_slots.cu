// gemv_slots.cu -- the weight GEMVs of the few-slot step ("Mini Inference Engine",
// "Continuous batching": several sequences advance one token per step and share one
// pass over the weights).
//
// Every weight row is read from HBM once per step and multiplied with the input
// vectors of all n_slots (<= 8) slots on the tensor cores, with mma.sync m16n8k16
// (bf16 operands, fp32 accumulators) in transposed form:
//   Y^T[slot][row] = X^T[slot][k] * W^T[k][row]
//   A = X^T: 16 x 16, rows 0..7 = the slots' x_hi, rows 8..15 = their x_lo (below),
//       held in registers;
//   B = W^T: 16 k x 8 weight rows -- the staged rows read as they lie in memory;
//   C = Y^T: thread (g = lane/4, t = lane%4) holds the x_hi and x_lo parts of
//       Y[row 2t, 2t+1][slot g], added at the end.
// x is fp32 in the method, so each x value is split into x_hi = bf16(x) and
// x_lo = bf16(x - x_hi), which fill the sixteen rows of one MMA: the products are
// exact in fp32 and x keeps about 16 significant bits (int8 weights become bf16
// exactly).
// Within each 16-column k-step the fragment positions 2t, 2t+1, 2t+8, 2t+9 of lane
// (g, t) are mapped to columns 4t .. 4t+3 for both A and B (a sum over k does not depend
// on its order), so a lane's x is one float4 and its weights one 8-byte (bf16) or
// 4-byte (int8, Q4_0: both nibbles of four bytes) shared load per k-step.
// Q4_0: the B values are the codes minus 8 (exact in bf16); each warp owns whole
// 32-column blocks, accumulates a block's MMAs apart and adds them times the f16 block
// scale of each output row.
//
// A producer warp streams stages of 8 weight rows x one 2048-column slice through a
// ring in shared memory (one bulk copy per row into rows padded so that the B-fragment
// loads hit distinct banks); the 8 consumer warps each own 16 of the
// slice's 128 k-steps and keep their x fragments in registers for the whole slice.
// Warp partials are summed in a fixed order, so results do not depend on timing.
#include "device.cuh"

namespace mie {

constexpr int kSW = 8;               // consumer warps
constexpr int kSCT = 32 * kSW;       // consumer threads
constexpr int kST = kSCT + 32;       // + one producer warp
constexpr int kSRows = 8;            // weight rows per stage (the MMA's N)
constexpr int kSSlice = 2048;        // columns per stage
constexpr int kSKSteps = kSSlice / 16 / kSW;  // k-steps per warp per slice (16)
constexpr int kSMaxNst = 8;
constexpr int kSMaxAccTiles = 16;    // tiles per CTA whose partial sums persist across slices
constexpr int kSBurst = 2;           // stages issued before the consumers have their first input

struct SSync {
  __device__ static void sync() { asm volatile("bar.sync 1, %0;" ::"n"(kSCT) : "memory"); }
  // barrier that also returns whether v holds on any consumer thread
  __device__ static bool any(bool v) {
    int r;
    asm volatile(
        "{\n .reg .pred p, q;\n setp.ne.s32 p, %1, 0;\n bar.red.or.pred q, 1, %2, p;\n selp.s32 %0, 1, 0, q;\n}"
        : "=r"(r)
        : "r"((int)v), "n"(kSCT)
        : "memory");
    return r != 0;
  }
};

__device__ __forceinline__ uint32_t bf16x2_bits(float lo, float hi) {
  return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(lo)) |
         ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(hi)) << 16);
}

// hi / lo bf16 pairs of two fp32 values
__device__ __forceinline__ void split2(float v0, float v1, uint32_t &hi, uint32_t &lo) {
  const float h0 = __bfloat162float(__float2bfloat16_rn(v0)), h1 = __bfloat162float(__float2bfloat16_rn(v1));
  hi = bf16x2_bits(h0, h1);
  lo = bf16x2_bits(v0 - h0, v1 - h1);
}

// One m16n8k16 bf16 MMA with all four A registers (not volatile: a pure function of its
// registers, so the compiler may schedule it): a0 / a2 rows g (x_hi of slot g),
// a1 / a3 rows g + 8 (x_lo of slot g); c[0], c[1] and c[2], c[3] come back as the hi and
// lo products of rows 2t, 2t + 1.
__device__ __forceinline__ void mma_hl(float (&c)[4], uint32_t ah0, uint32_t al0, uint32_t ah2, uint32_t al2,
                                       uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(ah0), "r"(al0), "r"(ah2), "r"(al2), "r"(b0), "r"(b1));
}

// B fragment words of one k-step: the lane's four consecutive weights of a staged row
// (columns 4t .. 4t+3) as bf16 pairs b0 = (4t, 4t+1), b1 = (4t+2, 4t+3).
template <int F>
__device__ __forceinline__ void b_words(uint32_t addr, uint32_t &b0, uint32_t &b1);
template <>
__device__ __forceinline__ void b_words<MIE_FMT_Q4_0>(uint32_t, uint32_t &b0, uint32_t &b1) {  // own loop
  b0 = b1 = 0u;
}
template <>
__device__ __forceinline__ void b_words<MIE_FMT_BF16>(uint32_t addr, uint32_t &b0, uint32_t &b1) {
  asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(b0), "=r"(b1) : "r"(addr));
}
template <>
__device__ __forceinline__ void b_words<MIE_FMT_I8>(uint32_t addr, uint32_t &b0, uint32_t &b1) {
  const uint32_t v = lds32(addr);
  b0 = bf16x2_bits((float)(int8_t)(v & 0xffu), (float)(int8_t)((v >> 8) & 0xffu));  // exact: |q| <= 127
  b1 = bf16x2_bits((float)(int8_t)((v >> 16) & 0xffu), (float)(int8_t)(v >> 24));
}

// The k-step of a slice that warp `warp` handles as its j-th (0..kSKSteps-1): the slice's
// 128 k-steps are dealt round robin, or, for Q4_0, as whole blocks (two k-steps each).
template <int F>
__device__ __forceinline__ int kstep_of(int warp, int j) {
  if constexpr (F == MIE_FMT_Q4_0) return 2 * (warp + kSW * (j >> 1)) + (j & 1);
  return warp + kSW * j;
}

// bf16 bits of a Q4_0 code minus 8 (exact), two codes packed
__device__ __forceinline__ uint32_t q4_pair(uint32_t n0, uint32_t n1) {
  return bf16x2_bits((float)(int)n0 - 8.f, (float)(int)n1 - 8.f);
}

// Shared state of one CTA.
struct SlotShared {
  float ss[kSW][kMaxSlots];                    // per-warp sums of squares (RMSNorm)
  float rs[kMaxSlots];                         // RMSNorm scale per slot
  unsigned cnt[2][kSMaxNst];                   // warps done with the stage, per ring cycle parity and slot
  float acc[kSMaxAccTiles][kMaxSlots][kSRows];  // partial sums across slices
  unsigned long long best[kMaxSlots];          // argmax per slot: orderable value << 32 | ~row
  int pos[kMaxSlots], blk[kMaxSlots], tok[kMaxSlots];
  bool pos_ok[kMaxSlots], blk_ok[kMaxSlots];
  float rc[kMaxSlots][64], rsn[kMaxSlots][64];  // RoPE cos / sin of each slot's position (hd <= 128)
  float gain[kSSlice];                           // RMSNorm gains (the normalising prologues have K <= kSSlice)
  unsigned last;
};

// Orderable key of (value, row): larger value first, then lower row; 0 = no row yet.
__device__ __forceinline__ unsigned long long argmax_key(float v, int row) {
  const uint32_t b = __float_as_uint(v);
  const uint32_t o = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
  return ((unsigned long long)o << 32) | (unsigned long long)(0xffffffffu - (uint32_t)row);
}
__device__ __forceinline__ void argmax_unkey(unsigned long long k, float &v, int &row) {
  if (k == 0ull) {
    v = -INFINITY;
    row = 0x7fffffff;
    return;
  }
  const uint32_t o = (uint32_t)(k >> 32);
  v = __uint_as_float((o & 0x80000000u) ? (o & 0x7fffffffu) : ~o);
  row = (int)(0xffffffffu - (uint32_t)k);
}

struct SlotPlan {
  int nst = 0;
  uint32_t x_off = 0, x_pitch = 0;      // the slots' input slice after the ring: [kMaxSlots][x_pitch]
  uint32_t pitch = 0, stage_bytes = 0;  // padded row bytes in shared memory, bytes per slot
  uint32_t sc_off = 0;                  // Q4_0: offset of the stage's scale rows (128 bytes each)
  uint32_t red_off = 0;                 // warp partials [2 cycle parities][nst][kSW][kMaxSlots][kSRows] floats
  int n_tiles = 0, KS = 1;
  size_t smem = 0;
};

template <int F, int PRO, int EPI>
__global__ void __launch_bounds__(kST, 1) gemv_slots_kernel(const GemvArgs a, const SlotPlan pl) {
  constexpr int ES = (F == MIE_FMT_BF16) ? 2 : 1;  // bytes per weight (bf16, int8)
  constexpr bool Q4 = F == MIE_FMT_Q4_0;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t full_bar[kSMaxNst], empty_bar[kSMaxNst], x_bar;
  __shared__ SlotShared sh;
  __shared__ volatile int s_issued, s_prod_done, s_abort, s_x_ready, s_x_last;

  const DevMat &m = a.m;
  const int M = m.rows, K = m.cols, Kp = m.kp;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int tt0 = (int)((int64_t)blockIdx.x * pl.n_tiles / gridDim.x);
  const int tt1 = (int)((int64_t)(blockIdx.x + 1) * pl.n_tiles / gridDim.x);
  const int n_my = tt1 - tt0;
  const int n_stages = n_my * pl.KS;
  const int S = a.sp->n_slots;

  if (tid == 0) {
    for (int i = 0; i < pl.nst; ++i) {
      mbar_init(&full_bar[i], 1);
      mbar_init(&empty_bar[i], kSW);
    }
    mbar_init(&x_bar, 1);
    s_issued = 0;
    s_prod_done = 0;
    s_abort = 0;
    s_x_ready = 0;
    s_x_last = -1;
    for (int i = 0; i < kSMaxNst; ++i) sh.cnt[0][i] = sh.cnt[1][i] = 0u;
    for (int i = 0; i < kMaxSlots; ++i) sh.best[i] = 0ull;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  pdl_trigger();

  if (warp == kSW) {  // producer: weights do not depend on earlier kernels
    if (lane == 0) {
      const uint64_t pol = evict_first_policy();
      for (int s = 0; s < n_stages; ++s) {
        const int slot = s % pl.nst, k = s / pl.nst;
        if (s == kSBurst) {
          // the consumers' input loads go out before the rest of the ring's copies: L2 and
          // HBM requests queue behind bulk copies in flight (measured 5-10 us otherwise)
          for (long it = 0; it < kWaitPolls && !s_x_ready && !s_abort; ++it) __nanosleep(128);
        }
        if (k > 0 && !mbar_wait(&empty_bar[slot], (k - 1) & 1)) {
          s_abort = 1;
          latch_error(a.err, ERR_TIMEOUT);
          break;
        }
        if (s_abort) break;
        const int q = s / n_my, r0 = (tt0 + s % n_my) * kSRows;
        const int rows = min(kSRows, M - r0);
        uint8_t *dst = smem + (size_t)slot * pl.stage_bytes;
        if constexpr (Q4) {
          const int nb = min(kSSlice, Kp - q * kSSlice) / 32;  // blocks of this slice
          const int ns = (nb + (1 << m.gshift) - 1) >> m.gshift;  // its scales (one per group)
          const uint32_t cb = (uint32_t)nb * 16, sb = (uint32_t)((ns + 7) / 8 * 8) * 2;  // scales: whole 16 B
          mbar_expect_tx(&full_bar[slot], rows * (cb + sb));
          for (int j = 0; j < rows; ++j) {
            bulk_load(dst + (size_t)j * pl.pitch, m.w + (int64_t)(r0 + j) * m.row_bytes + (int64_t)q * (kSSlice / 32) * 16,
                      cb, &full_bar[slot], pol);
            bulk_load(dst + pl.sc_off + (size_t)j * 128,
                      reinterpret_cast<const uint8_t *>(m.s) +
                          ((int64_t)(r0 + j) * m.s_stride + q * (kSSlice >> (5 + m.gshift))) * 2,
                      sb, &full_bar[slot], pol);
          }
        } else {
          const uint32_t cb = (uint32_t)(min(kSSlice, Kp - q * kSSlice) * ES);
          mbar_expect_tx(&full_bar[slot], rows * cb);
          for (int j = 0; j < rows; ++j)
            bulk_load(dst + (size_t)j * pl.pitch, m.w + (int64_t)(r0 + j) * m.row_bytes + (int64_t)q * kSSlice * ES, cb,
                      &full_bar[slot], pol);
        }
        s_issued = s + 1;
      }
      s_prod_done = 1;
    }
    return;
  }

  if (PRO != PRO_PLAIN)  // gains are weights: loaded before waiting for the previous kernel
    for (int i = tid; i < K && i < kSSlice; i += kSCT) sh.gain[i] = __ldg(a.gain + i);
  pdl_wait();
  const int g = lane >> 2, t = lane & 3;

  // per-slot constants of the epilogue
  if (tid < kMaxSlots) {
    const int s = tid;
    int tok = 0, pos = 0, blk = -1;
    bool pos_ok = false, blk_ok = false;
    if (s < S) {
      tok = a.sp->token[s];
      if (tok < 0 || tok >= a.vocab) {
        if (PRO == PRO_EMBED_NORM) latch_error(a.err, ERR_TOKEN);
        tok = 0;
      }
      if constexpr (EPI == EPI_QKV) {
        pos = a.sp->pos[s];
        pos_ok = pos >= 0 && pos < a.max_pos && pos / a.bs < a.sp->max_blocks;
        blk = a.sp->block_table[(int64_t)s * a.sp->max_blocks + (pos_ok ? pos / a.bs : 0)];
        blk_ok = pos_ok && blk >= 0 && blk < a.n_kv_blocks;
        if (!blk_ok) latch_error(a.err, pos_ok ? ERR_BLOCK_ID : ERR_POS);
      }
    }
    sh.tok[s] = tok;
    sh.pos[s] = pos;
    sh.blk[s] = blk;
    sh.pos_ok[s] = pos_ok;
    sh.blk_ok[s] = blk_ok;
  }
  if constexpr (EPI == EPI_QKV) {  // each slot's RoPE row, so the epilogue issues no dependent loads
    const int h2 = a.hd / 2;
    for (int i = tid; i < kMaxSlots * h2; i += kSCT) {
      const int s = i / h2, j = i % h2;
      int pos = (s < S) ? a.sp->pos[s] : 0;
      if (pos < 0 || pos >= a.max_pos) pos = 0;
      sh.rc[s][j] = a.rope_cos[(int64_t)pos * h2 + j];
      sh.rsn[s][j] = a.rope_sin[(int64_t)pos * h2 + j];
    }
  }
  SSync::sync();

  // A fragments of slice q: x of slot g at columns kk + 4t .. kk + 4t + 3 of this warp's
  // k-steps, as hi / lo bf16 pairs.  Every load of the slice (x and gains, 16 bytes each)
  // is issued before the first use, so staging costs one round trip; the values stay in
  // registers through the RMSNorm.
  uint32_t ah0[kSKSteps], ah2[kSKSteps], al0[kSKSteps], al2[kSKSteps];
  const uint32_t xsm = smem_u32(smem) + pl.x_off;
  auto load_quad = [&](int e) -> float4 {  // x of slot g at columns e .. e + 3 (e % 4 == 0)
    if (g >= S || e >= K) return make_float4(0.f, 0.f, 0.f, 0.f);
    if (PRO == PRO_EMBED_NORM) {
      if (a.embed.fmt == MIE_FMT_BF16 && e + 3 < K) {
        const uint2 w = __ldg(reinterpret_cast<const uint2 *>(a.embed.w + (int64_t)sh.tok[g] * a.embed.row_bytes) + e / 4);
        return make_float4(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xffff0000u), __uint_as_float(w.y << 16),
                           __uint_as_float(w.y & 0xffff0000u));
      }
      float v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) v[u] = e + u < K ? embed_at(a.embed, sh.tok[g], e + u) : 0.f;
      return make_float4(v[0], v[1], v[2], v[3]);
    }
    // the slice staged in shared memory (K % 4 == 0: a quad is all in or all out)
    return lds128f(xsm + (uint32_t)g * pl.x_pitch + (uint32_t)(e % kSSlice) * 4);
  };
  // the slots' x of slice q into shared memory by bulk copies (one per slot row): one
  // request per row instead of a load per lane.  Thread 0 issues slice 0 here and slice
  // q + 1 once every warp holds its fragments of slice q, so the copy overlaps slice q's
  // stages.
  auto issue_x = [&](int q) {
    const int cols = min(kSSlice, K - q * kSSlice);
    if (PRO == PRO_EMBED_NORM || cols <= 0) return;
    fence_proxy_async_smem();  // generic reads of the previous slice before the async writes
    mbar_expect_tx(&x_bar, (uint32_t)(S * cols * 4));
    for (int sl = 0; sl < S; ++sl)
      bulk_load(smem + pl.x_off + (size_t)sl * pl.x_pitch, a.x + (int64_t)sl * K + (int64_t)q * kSSlice,
                (uint32_t)cols * 4, &x_bar, 0ull);
    s_x_last = q;
  };
  auto stage_x = [&](int q) {
    if (PRO == PRO_EMBED_NORM || min(kSSlice, K - q * kSSlice) <= 0) return;
    if (q == 0 && tid == 0) issue_x(0);
    if (!mbar_wait(&x_bar, q & 1)) {
      s_abort = 1;
      latch_error(a.err, ERR_TIMEOUT);
    }
  };
  auto gain_quad = [&](int e) -> float4 {  // staged in shared memory before the kernel waited
    float v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) v[u] = e + u < K ? sh.gain[e + u] : 0.f;
    return make_float4(v[0], v[1], v[2], v[3]);
  };
  auto load_slice = [&](int q) {
    stage_x(q);
    float4 xv[kSKSteps];
#pragma unroll
    for (int j = 0; j < kSKSteps; ++j) xv[j] = load_quad(q * kSSlice + kstep_of<F>(warp, j) * 16 + 4 * t);
    if (PRO == PRO_EMBED_NORM && blockIdx.x == 0 && g < S) {  // the residual stream starts as x
#pragma unroll
      for (int j = 0; j < kSKSteps; ++j) {
        const int e = q * kSSlice + kstep_of<F>(warp, j) * 16 + 4 * t;
        const float v[4] = {xv[j].x, xv[j].y, xv[j].z, xv[j].w};
#pragma unroll
        for (int u = 0; u < 4; ++u)
          if (e + u < K) a.x_store[(int64_t)g * K + e + u] = v[u];
      }
    }
    if (PRO != PRO_PLAIN) {
      // RMSNorm over the whole vector: the prologues that normalise have K <= kSSlice
      float ss = 0.f;
#pragma unroll
      for (int j = 0; j < kSKSteps; ++j) ss += xv[j].x * xv[j].x + xv[j].y * xv[j].y + xv[j].z * xv[j].z + xv[j].w * xv[j].w;
      ss += __shfl_xor_sync(0xffffffffu, ss, 1);
      ss += __shfl_xor_sync(0xffffffffu, ss, 2);
      if (t == 0) sh.ss[warp][g] = ss;
      SSync::sync();
      if (tid < kMaxSlots) {
        float tot = 0.f;
        for (int w = 0; w < kSW; ++w) tot += sh.ss[w][tid];
        sh.rs[tid] = 1.0f / sqrtf(tot / (float)K + a.eps);
      }
      SSync::sync();
      const float rn = sh.rs[g];
#pragma unroll
      for (int j = 0; j < kSKSteps; ++j) {
        const float4 gg = gain_quad(q * kSSlice + kstep_of<F>(warp, j) * 16 + 4 * t);
        xv[j].x = xv[j].x * rn * gg.x;
        xv[j].y = xv[j].y * rn * gg.y;
        xv[j].z = xv[j].z * rn * gg.z;
        xv[j].w = xv[j].w * rn * gg.w;
      }
    }
#pragma unroll
    for (int j = 0; j < kSKSteps; ++j) {
      float v[4] = {xv[j].x, xv[j].y, xv[j].z, xv[j].w};
      if (a.act_bf16) {
#pragma unroll
        for (int u = 0; u < 4; ++u) v[u] = round_bf16(v[u]);
      }
      split2(v[0], v[1], ah0[j], al0[j]);
      split2(v[2], v[3], ah2[j], al2[j]);
    }
  };

  // epilogue of one tile: the warp that completes it calls this twice, lane l holding
  // output i = l + 32h = (slot i / 8, row r0 + i % 8); all 32 lanes call it together
  auto epilogue = [&](int r0, int es, int er, float v) {
    const int r = r0 + er;
    if (F == MIE_FMT_I8 && r < M) v *= reinterpret_cast<const float *>(m.s)[r];
    if constexpr (EPI == EPI_STORE) {
      if (es < S && r < M) a.y[(int64_t)es * M + r] = v;
    } else if constexpr (EPI == EPI_RESID) {
      if (es < S && r < M) a.y[(int64_t)es * M + r] += v;
    } else if constexpr (EPI == EPI_SWIGLU) {
      const float up = __shfl_down_sync(0xffffffffu, v, 1);  // row r + 1 of the same slot
      if (es < S && (er & 1) == 0 && r + 1 < M) a.y[(int64_t)es * (M / 2) + r / 2] = v / (1.0f + expf(-v)) * up;
    } else if constexpr (EPI == EPI_QKV) {
      const float x1 = __shfl_down_sync(0xffffffffu, v, 1);
      if (es < S && (er & 1) == 0 && r + 1 < M) {
        const int h2 = a.hd / 2, u = r / 2;
        const int h = u / h2, i = u % h2;
        float x0 = v, y1 = x1;
        if (h < a.Hq + a.Hkv && sh.pos_ok[es]) {
          const float c = sh.rc[es][i], sn = sh.rsn[es][i];
          const float r0v = x0 * c - y1 * sn, r1v = y1 * c + x0 * sn;
          x0 = r0v;
          y1 = r1v;
        }
        if (h < a.Hq) {
          float *qo = a.q_out + (int64_t)es * a.Hq * a.hd + h * a.hd;
          qo[i] = x0;
          qo[i + h2] = y1;
        } else if (sh.blk_ok[es]) {
          const int isv = h >= a.Hq + a.Hkv;
          const int gh = h - a.Hq - (isv ? a.Hkv : 0);
          uint16_t *dst = a.kv_layer + (int64_t)sh.blk[es] * a.block_stride + (int64_t)isv * a.Hkv * a.bs * a.hd +
                          ((int64_t)gh * a.bs + sh.pos[es] % a.bs) * a.hd;
          dst[i] = __bfloat16_as_ushort(__float2bfloat16_rn(x0));
          dst[i + h2] = __bfloat16_as_ushort(__float2bfloat16_rn(y1));
        }
      }
    } else if constexpr (EPI == EPI_ARGMAX) {
      unsigned long long key = 0ull;
      if (es < S && r < M) {
        if (a.sp->logits_out) a.sp->logits_out[(int64_t)es * M + r] = v;
        key = argmax_key(v, r);
      }
#pragma unroll
      for (int o = 1; o < kSRows; o <<= 1) {  // the 8 lanes of one slot
        const unsigned long long ok2 = __shfl_xor_sync(0xffffffffu, key, o);
        key = ok2 > key ? ok2 : key;
      }
      if (er == 0 && es < S && key) atomicMax(&sh.best[es], key);
    }
  };

  // Stage loop without CTA barriers: each warp posts its partial of the stage's tile and
  // counts itself done in shared memory; the last warp of the stage sums the eight
  // partials in a fixed order and finishes the tile.  Every warp releases the ring slot
  // after that, so a slot's partials are read before its next stage can be written.
  bool ok = true;
  int s = 0;
  const uint32_t ring = smem_u32(smem);
  for (int q = 0; q < pl.KS; ++q) {
    load_slice(q);
    SSync::sync();  // every warp holds its fragments of slice q: the input buffer is free
    if (tid == 0) {
      if (q == 0) s_x_ready = 1;  // the producer may fill the rest of the ring
      if (q + 1 < pl.KS) issue_x(q + 1);
    }
    const int nk = min(kSSlice, Kp - q * kSSlice) / 16;  // k-steps of this slice
    for (int tl = 0; tl < n_my; ++tl, ++s) {
      const int slot = s % pl.nst, k = s / pl.nst;
      if (ok && !mbar_wait(&full_bar[slot], k & 1)) {
        ok = false;
        s_abort = 1;
        latch_error(a.err, ERR_TIMEOUT);
      }
      // four independent accumulator chains over the warp's k-steps
      float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
      float c2[4] = {0.f, 0.f, 0.f, 0.f}, c3[4] = {0.f, 0.f, 0.f, 0.f};
      if (ok && Q4) {
        // whole blocks: b = warp + kSW * i, k-steps 2b (low nibbles) and 2b + 1 (high)
        const uint32_t sbase = ring + (uint32_t)slot * pl.stage_bytes;
        const uint32_t nrow = sbase + (uint32_t)g * pl.pitch + 4 * t;  // row g's bytes 4t .. 4t + 3 of a block
        const uint32_t srow = sbase + pl.sc_off + (uint32_t)(2 * t) * 128;  // scales of output rows 2t, 2t + 1
#pragma unroll
        for (int i = 0; i < kSKSteps / 2; ++i) {
          const int b = warp + kSW * i;
          if (2 * b < nk) {
            const uint32_t w = lds32(nrow + b * 16);  // codes 4t.. (low nibbles) and 4t+16.. (high)
            const float d0 = __half2float(__ushort_as_half((unsigned short)lds16(srow + (b >> m.gshift) * 2)));
            const float d1 = __half2float(__ushort_as_half((unsigned short)lds16(srow + 128 + (b >> m.gshift) * 2)));
            float ct[4] = {0.f, 0.f, 0.f, 0.f};
            const uint32_t lb0 = q4_pair(w & 0xFu, (w >> 8) & 0xFu), lb1 = q4_pair((w >> 16) & 0xFu, (w >> 24) & 0xFu);
            const uint32_t hb0 = q4_pair((w >> 4) & 0xFu, (w >> 12) & 0xFu);
            const uint32_t hb1 = q4_pair((w >> 20) & 0xFu, (w >> 28) & 0xFu);
            mma_hl(ct, ah0[2 * i], al0[2 * i], ah2[2 * i], al2[2 * i], lb0, lb1);
            mma_hl(ct, ah0[2 * i + 1], al0[2 * i + 1], ah2[2 * i + 1], al2[2 * i + 1], hb0, hb1);
            c0[0] = fmaf(d0, ct[0] + ct[2], c0[0]);
            c0[1] = fmaf(d1, ct[1] + ct[3], c0[1]);
          }
        }
      } else if (ok) {
        const uint32_t base = ring + (uint32_t)slot * pl.stage_bytes + (uint32_t)g * pl.pitch + (uint32_t)(4 * t) * ES;
        // B words of eight k-steps are loaded in one batch (k-steps past the slice read
        // its first k-step: their A fragments are zero), then the MMAs run
        constexpr int H = kSKSteps / 2;
#pragma unroll
        for (int h0 = 0; h0 < kSKSteps; h0 += H) {
          uint32_t b0[H], b1[H];
#pragma unroll
          for (int j = 0; j < H; ++j) {
            const int ks = warp + kSW * (h0 + j);
            b_words<F>(base + (uint32_t)((ks < nk ? ks : 0) * 16) * ES, b0[j], b1[j]);
          }
#pragma unroll
          for (int j = 0; j < H; j += 4) {  // four independent accumulator chains
            mma_hl(c0, ah0[h0 + j], al0[h0 + j], ah2[h0 + j], al2[h0 + j], b0[j], b1[j]);
            mma_hl(c1, ah0[h0 + j + 1], al0[h0 + j + 1], ah2[h0 + j + 1], al2[h0 + j + 1], b0[j + 1], b1[j + 1]);
            mma_hl(c2, ah0[h0 + j + 2], al0[h0 + j + 2], ah2[h0 + j + 2], al2[h0 + j + 2], b0[j + 2], b1[j + 2]);
            mma_hl(c3, ah0[h0 + j + 3], al0[h0 + j + 3], ah2[h0 + j + 3], al2[h0 + j + 3], b0[j + 3], b1[j + 3]);
          }
        }
      }
      // c[0], c[1] = Y[row 2t, 2t+1][slot g] of this warp's k-steps
      // hi + lo parts (Q4_0 carries them summed in c0[0], c0[1])
      const int par = k & 1;  // the stage's ring cycle parity picks its partial buffers
      float *rs = reinterpret_cast<float *>(smem + pl.red_off) + (size_t)(par * pl.nst + slot) * (kSW * kMaxSlots * kSRows);
      rs[(warp * kMaxSlots + g) * kSRows + 2 * t] = ((c0[0] + c0[2]) + (c1[0] + c1[2])) + ((c2[0] + c2[2]) + (c3[0] + c3[2]));
      rs[(warp * kMaxSlots + g) * kSRows + 2 * t + 1] =
          ((c0[1] + c0[3]) + (c1[1] + c1[3])) + ((c2[1] + c2[3]) + (c3[1] + c3[3]));
      __threadfence_block();
      __syncwarp();
      unsigned prev = 0u;
      if (lane == 0) prev = atomicAdd(&sh.cnt[par][slot], 1u);
      prev = __shfl_sync(0xffffffffu, prev, 0);
      // the stage's weights are in registers and consumed: the slot goes back to the
      // producer now, and the last warp's sums and epilogue below overlap the next stages
      // (their partials live in buffers of their own, two per slot by ring cycle, reused
      // only after every warp has passed the next cycle of the slot)
      if (lane == 0) mbar_arrive(&empty_bar[slot]);
      if (prev == kSW - 1) {  // the last warp of this stage
        __threadfence_block();
        const int r0 = (tt0 + tl) * kSRows;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int i = lane + 32 * h, es = i >> 3, er = i & 7;
          float v = 0.f;
#pragma unroll
          for (int w = 0; w < kSW; ++w) v += rs[(w * kMaxSlots + es) * kSRows + er];
          if (q > 0) v += sh.acc[tl][es][er];
          if (q + 1 < pl.KS) sh.acc[tl][es][er] = v;
          else epilogue(r0, es, er, v);
        }
        if (lane == 0) sh.cnt[par][slot] = 0u;
        __threadfence_block();
        __syncwarp();
      }
    }
  }
  if (SSync::any(!ok || s_abort)) {
    if (tid == 0) {
      if (s_x_last >= 0) mbar_wait(&x_bar, s_x_last & 1);  // the last input copy (bounded)
      for (long it = 0; it < kWaitPolls && !s_prod_done; ++it) __nanosleep(64);
      const int issued = s_issued;
      for (int x = max(s, issued - pl.nst); x < issued; ++x) mbar_wait(&full_bar[x % pl.nst], (x / pl.nst) & 1);
    }
    return;
  }
  if constexpr (EPI == EPI_ARGMAX) {
    // per slot: this CTA's best (shared-memory key), then the last CTA over all CTAs
    if (tid < kMaxSlots) {
      float bv;
      int bi;
      argmax_unkey(sh.best[tid], bv, bi);
      a.am_part[(int64_t)tid * gridDim.x + blockIdx.x] = make_float2(bv, __int_as_float(bi));
    }
    __threadfence();
    SSync::sync();
    if (tid == 0) sh.last = (atomicAdd(a.am_count, 1u) == gridDim.x - 1);
    SSync::sync();
    if (sh.last) {
      __threadfence();
      // warp w reduces slot w
      const int sl = warp;
      if (sl < S) {
        float fv = -INFINITY;
        int fi = 0x7fffffff;
        for (int b = lane; b < (int)gridDim.x; b += 32) {
          const float2 p = __ldcg(a.am_part + (int64_t)sl * gridDim.x + b);
          if (better(p.x, __float_as_int(p.y), fv, fi)) { fv = p.x; fi = __float_as_int(p.y); }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const float ov = __shfl_xor_sync(0xffffffffu, fv, o);
          const int oi = __shfl_xor_sync(0xffffffffu, fi, o);
          if (better(ov, oi, fv, fi)) { fv = ov; fi = oi; }
        }
        if (lane == 0) {
          if (fi == 0x7fffffff) fi = 0;
          if (a.sp->argmax_out) a.sp->argmax_out[sl] = fi;
          if (a.sp->advance) {
            a.sp->token[sl] = fi;
            a.sp->pos[sl] += 1;
          }
        }
      }
      SSync::sync();
      if (tid == 0) *a.am_count = 0u;
    }
  }
}

// ------------------------------------------------------------------------- host side

static SlotPlan slot_plan(const DevMat &m, int grid) {
  SlotPlan p;
  p.KS = (m.kp + kSSlice - 1) / kSSlice;
  const int slice = min(kSSlice, m.kp);
  if (m.fmt == MIE_FMT_Q4_0) {
    p.pitch = (uint32_t)(slice / 32 * 16 + 16);
    p.sc_off = (uint32_t)((kSRows * p.pitch + 15) / 16 * 16);
    p.stage_bytes = (uint32_t)((p.sc_off + kSRows * 128 + 127) / 128 * 128);
  } else {
    // rows padded so the 8 rows of a B fragment start 8 (bf16: 8-byte loads, served per
    // half warp) or 4 (int8: 4-byte loads) banks apart: no bank conflicts
    const int ES = (m.fmt == MIE_FMT_BF16) ? 2 : 1;
    p.pitch = (uint32_t)(slice * ES + (ES == 2 ? 32 : 16));
    p.stage_bytes = (uint32_t)((kSRows * p.pitch + 127) / 128 * 128);
  }
  p.n_tiles = (m.rows + kSRows - 1) / kSRows;
  int dev = 0, max_smem = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  p.x_pitch = (uint32_t)(slice * 4 + 64);  // slot rows 16 banks apart: a quarter warp's 16-byte reads cover 2 rows
  const long x_bytes = (long)kMaxSlots * p.x_pitch;
  const long avail = (long)max_smem - (long)sizeof(SlotShared) - 1024 - x_bytes;
  const long red_stage = 2L * kSW * kMaxSlots * kSRows * 4;  // partial buffers of one ring slot
  int nst = (int)(avail / ((long)p.stage_bytes + red_stage));
  p.nst = nst > kSMaxNst ? kSMaxNst : nst;
  p.x_off = (uint32_t)p.nst * p.stage_bytes;
  p.red_off = (uint32_t)((p.x_off + x_bytes + 15) / 16 * 16);
  p.smem = (size_t)p.red_off + (size_t)p.nst * red_stage;
  (void)grid;
  return p;
}

template <int F, int PRO, int EPI>
static mie_status launch_slots_t(const GemvArgs &a, const SlotPlan &p, int grid, cudaStream_t st, bool pdl) {
  auto kern = gemv_slots_kernel<F, PRO, EPI>;
  MIE_CUDA(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p.smem));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kST);
  cfg.dynamicSmemBytes = p.smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  MIE_CUDA(cudaLaunchKernelEx(&cfg, kern, a, p));
  return MIE_OK;
}

template <int F>
static mie_status launch_slots_f(int pro, int epi, const GemvArgs &a, const SlotPlan &p, int grid, cudaStream_t st,
                                 bool pdl) {
#define MIE_S(P, E) \
  if (pro == P && epi == E) return launch_slots_t<F, P, E>(a, p, grid, st, pdl);
  MIE_S(PRO_EMBED_NORM, EPI_QKV)
  MIE_S(PRO_NORM, EPI_QKV)
  MIE_S(PRO_PLAIN, EPI_RESID)
  MIE_S(PRO_NORM, EPI_SWIGLU)
  MIE_S(PRO_NORM, EPI_ARGMAX)
  MIE_S(PRO_PLAIN, EPI_STORE)
#undef MIE_S
  return fail(MIE_E_SHAPE, "slot GEMV: prologue %d / epilogue %d not built", pro, epi);
}

// Checks that the batched GEMV covers matrix m with prologue pro.
mie_status slots_gemv_supported(const DevMat &m, int pro) {
  if (m.fmt != MIE_FMT_BF16 && m.fmt != MIE_FMT_I8 && m.fmt != MIE_FMT_Q4_0)
    return fail(MIE_E_SHAPE, "few-slot step: weight format %d", m.fmt);
  if (m.kp % 16) return fail(MIE_E_SHAPE, "few-slot step: padded width %d is not a multiple of 16", m.kp);
  if (m.cols % 4)
    return fail(MIE_E_SHAPE, "few-slot step: input length %d is not a multiple of 4 (inputs are read in fours)", m.cols);
  if (pro != PRO_PLAIN && m.cols > kSSlice)
    return fail(MIE_E_SHAPE, "few-slot step: RMSNorm over %d > %d columns", m.cols, kSSlice);
  if (((uintptr_t)m.w & 15) || (m.row_bytes & 15)) return fail(MIE_E_SHAPE, "few-slot step: unaligned rows");
  const SlotPlan p = slot_plan(m, 1);
  if (p.nst < 2) return fail(MIE_E_SHAPE, "few-slot step: shared memory too small for the ring");
  const int grid = sm_count();
  if (p.KS > 1 && (p.n_tiles + grid - 1) / grid > kSMaxAccTiles)
    return fail(MIE_E_SHAPE, "few-slot step: %d rows are too many for a %d-column input", m.rows, m.cols);
  return MIE_OK;
}

mie_status launch_gemv_slots(int pro, int epi, const GemvArgs &a, cudaStream_t st, bool pdl) {
  if (!a.sp) return fail(MIE_E_ARG, "slot GEMV: no step parameters");  // the kernel reads the slot count there
  const int grid = sm_count();
  const SlotPlan p = slot_plan(a.m, grid);
  if (a.m.fmt == MIE_FMT_BF16) return launch_slots_f<MIE_FMT_BF16>(pro, epi, a, p, grid, st, pdl);
  if (a.m.fmt == MIE_FMT_I8) return launch_slots_f<MIE_FMT_I8>(pro, epi, a, p, grid, st, pdl);
  if (a.m.fmt == MIE_FMT_Q4_0) return launch_slots_f<MIE_FMT_Q4_0>(pro, epi, a, p, grid, st, pdl);
  return fail(MIE_E_SHAPE, "few-slot step: weight format %d", a.m.fmt);
}

}  // namespace mie
