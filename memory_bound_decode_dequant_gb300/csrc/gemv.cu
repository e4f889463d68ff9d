// gemv.cu -- fused-dequant GEMV kernels for batch-1 decode on sm_103a.
//
// y = W x with W in bf16, int8 (one fp32 scale per row) or Q4_0 (32-weight blocks of
// 4-bit codes with one f16 scale), fp32 activations and accumulation ("infer" page:
// decode GEMV with fused norm, residual and SwiGLU; weight-only quantization with
// dequant in registers; "Writing an LLM inference engine from scratch in Rust",
// Lesson 1: decode speed is set by how fast the weights stream from memory).
//
// Design (GB300): the weights are read exactly once, so the kernel is a stream.
//  * One CTA per SM owns a contiguous range of rows.  A producer warp streams that
//    range through a ring of shared-memory stages with TMA bulk copies
//    (cp.async.bulk, completion on mbarriers, L2 evict-first), so tens of KB per SM
//    are in flight without holding registers.  The producer never waits on the
//    previous kernel (weights do not depend on it); only the consumers execute
//    griddepcontrol.wait before they read the input vector, so under programmatic
//    dependent launch the weights of kernel N+1 stream in while kernel N finishes.
//  * Each consumer warp owns one 2048-column slice of K; its slice of the normalised
//    input vector sits in 64 registers per lane for the whole kernel, so per 16-byte
//    chunk the inner loop is one shared-memory load, an in-register unpack and packed
//    fp32x2 FMAs.
//  * Unpack without int->float conversions: a code is moved into the mantissa of
//    2^23 by one LOP3 (Q4_0) or PRMT (int8), and one packed fp32x2 add removes both
//    the 2^23 and the stored bias (+8 for Q4_0, +128 after flipping the int8 sign
//    bit) exactly.  Q4_0 codes are masked in place at bit offset p and the matching
//    input element is pre-scaled by 2^-p, which is exact.
//  * Rows of a CTA are reduced across lanes with shuffles and across K slices through
//    shared memory in a fixed order, then an epilogue applies the row scale and the
//    fused operation (residual add, SwiGLU, RoPE + paged K/V write, argmax).
//  * Every mbarrier wait is bounded; a wait that gives up latches an error, drains
//    the copies still in flight and leaves the kernel.
#include <cstdarg>
#include <cstdio>

#include "device.cuh"

namespace mie {

constexpr int kCWarps = 8;                    // consumer warps (12 for large int8 GEMVs, below)
constexpr int kCWarpsWide = 12;
constexpr int kWideRows = 32768;
constexpr int kMaxStages = 16;
constexpr size_t kSmemMax = 200 * 1024;
// bf16 rows need little arithmetic per byte: two CTAs per SM (a kernel and its
// successor prefetching under programmatic dependent launch), each under 110 KB of
// shared memory.  int8 and Q4_0 rows are unpacked in registers and the arithmetic per
// byte sets the pace: one CTA per SM with the whole register file and ring (measured
// on the 128256 x 2048 int8 GEMV: 69 -> 80 % of HBM).
template <int F> constexpr int kMinBlocks = F == MIE_FMT_BF16 ? 2 : 1;
constexpr size_t smem_budget(int fmt) { return fmt == MIE_FMT_BF16 ? 110 * 1024 : kSmemMax; }

int gemv_chunk_elems(int fmt) {
  return fmt == MIE_FMT_BF16 ? 8 : fmt == MIE_FMT_I8 ? 16 : fmt == MIE_FMT_Q4_0 ? 32 : 0;
}

int sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return 148;
  if (!cached[dev]) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cached[dev] = n > 0 ? n : 148;
  }
  return cached[dev];
}

// Barrier over the consumer warps only (the producer warp never joins it).
template <int NW>
__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 1, %0;" ::"n"(NW * 32) : "memory"); }
template <int NW>
struct CSync {
  __device__ static void sync() { consumer_sync<NW>(); }
};


// --------------------------------------------------------------- the kernel
//
// One CTA per SM: warp NW is the producer, warps 0..NW-1 consume.  A stage
// is RPS whole rows of the CTA's (contiguous) row range, RPS = NW / KS, so each
// consumer warp reduces one 2048-column slice of one row per stage.  The producer
// issues the first ring-full of stages before any dependency wait.

template <int F, int PRO, int EPI, int NW>
__global__ void __launch_bounds__(32 * (NW + 1), kMinBlocks<F>) gemv_kernel(const GemvArgs a) {
  using T = FmtT<F>;
  constexpr int EPC = T::EPC, CPL = T::CPL;
  constexpr int RU = (EPI == EPI_SWIGLU || EPI == EPI_QKV) ? 2 : 1;
  constexpr int kBitsPerElem = (F == MIE_FMT_BF16) ? 16 : (F == MIE_FMT_I8 ? 8 : 4);
  constexpr int kSliceBytes = kSlice * kBitsPerElem / 8;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[kMaxStages], empty_bar[kMaxStages];
  __shared__ float red[NW];
  __shared__ float s_bv[NW];
  __shared__ int s_bi[NW];
  __shared__ unsigned s_last;
  __shared__ volatile int s_abort, s_issued, s_prod_done;
  __shared__ int s_abort_final;

  pdl_trigger();

  const DevMat &m = a.m;
  const int Kp = m.kp, K = m.cols, M = m.rows;
  const int KS = (Kp + kSlice - 1) / kSlice;
  constexpr int RPW = T::RPW;
  const int WR = KS >= NW ? 1 : NW / KS;  // warps per slice column
  const int RPS = WR * RPW;                          // rows per stage
  const int NST = a.n_stages;
  const uint32_t stage_bytes = a.stage_bytes, sc_bytes = a.sc_stage_bytes;
  uint8_t *ring = smem_raw;
  uint8_t *sring = ring + (size_t)NST * stage_bytes;
  float *xs = reinterpret_cast<float *>(sring + (size_t)NST * sc_bytes);  // element k at xs_at(k)
  float *part = xs + xs_floats(Kp);                                        // [rows][KS]

  const int n_units = (M + RU - 1) / RU;
  const int u0 = (int)((int64_t)blockIdx.x * n_units / gridDim.x);
  const int u1 = (int)((int64_t)(blockIdx.x + 1) * n_units / gridDim.x);
  const int row0 = u0 * RU, row1 = min(u1 * RU, M);
  const int n_stages = (row1 - row0 + RPS - 1) / RPS;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tid = threadIdx.x;

  if (tid == 0) {
    for (int i = 0; i < NST; ++i) {
      mbar_init(&full_bar[i], 1);
      mbar_init(&empty_bar[i], NW);
    }
    s_abort = 0;
    s_issued = 0;
    s_prod_done = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  // ---------------------------------------------------------------- producer
  if (warp == NW) {
    if (lane == 0) {
      const uint64_t pol = evict_first_policy();
      for (int s = 0; s < n_stages; ++s) {
        const int slot = s % NST, k = s / NST;
        if (k > 0 && !mbar_wait(&empty_bar[slot], (k - 1) & 1)) {
          s_abort = 1;
          latch_error(a.err, ERR_TIMEOUT);
          break;
        }
        if (s_abort) break;
        const int r = row0 + s * RPS;
        const int nr = min(RPS, row1 - r);
        const uint32_t wb = (uint32_t)(nr * m.row_bytes);
        const uint32_t sb = (F == MIE_FMT_Q4_0) ? (uint32_t)(nr * m.s_stride * 2) : 0u;
        mbar_expect_tx(&full_bar[slot], wb + sb);
        bulk_load(ring + (size_t)slot * stage_bytes, m.w + (int64_t)r * m.row_bytes, wb, &full_bar[slot], pol);
        if constexpr (F == MIE_FMT_Q4_0)
          bulk_load(sring + (size_t)slot * sc_bytes,
                    reinterpret_cast<const uint8_t *>(m.s) + (int64_t)r * m.s_stride * 2, sb, &full_bar[slot], pol);
        s_issued = s + 1;
      }
      s_prod_done = 1;
    }
    return;
  }

  // ---------------------------------------------------------------- consumers
  pdl_wait();
  stage_input<NW * 32, CSync<NW>>(a, PRO, xs, K, Kp, red, a.err);
  QkvPrefetch qp;
  if constexpr (EPI == EPI_QKV) qp = qkv_prefetch(a);

  const int ri = warp / KS, ks = warp % KS;
  const bool has_slice = warp < WR * KS;
  const int e0 = ks * kSlice + lane * EPC;
  float2 xr[CPL * EPC / 2];
  float nb[CPL], cs[CPL];
  load_lane_xr<F>(xs, e0, Kp, has_slice, xr, nb, cs);

  int consumed = 0;
  for (int s = 0; s < n_stages; ++s) {
    const int slot = s % NST, k = s / NST;
    if (!mbar_wait(&full_bar[slot], k & 1)) {
      s_abort = 1;
      latch_error(a.err, ERR_TIMEOUT);
      break;
    }
    consumed = s + 1;
    const int r = row0 + s * RPS + ri * RPW;  // this warp's first row of the stage
    if (has_slice && r < row1) {
      const int nr = min(RPW, row1 - r);
      const uint32_t rowa = smem_u32(ring) + (uint32_t)slot * stage_bytes + (uint32_t)(ri * RPW * m.row_bytes) +
                            (uint32_t)ks * kSliceBytes;
      const uint32_t sca = smem_u32(sring) + (uint32_t)slot * sc_bytes +
                           (uint32_t)(ri * RPW * m.s_stride + ks * (kSlice >> (5 + m.gshift))) * 2;
      float sum[RPW];
      stage_rows_dot<F>(rowa, (uint32_t)m.row_bytes, sca, (uint32_t)m.s_stride * 2, nr, xr, nb, cs, e0, Kp, lane, sum,
                        m.gshift);
#pragma unroll
      for (int i = 0; i < RPW; ++i) {
        const float v = warp_sum(sum[i]);
        if (lane == 0 && i < nr) part[(r + i - row0) * KS + ks] = v;
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty_bar[slot]);
  }
  consumer_sync<NW>();
  if (tid == 0) s_abort_final = s_abort;
  consumer_sync<NW>();
  if (s_abort_final) {
    // a wait gave up: make sure no bulk copy is still writing into shared memory
    if (tid == 0) {
      for (long it = 0; it < kWaitPolls && !s_prod_done; ++it) __nanosleep(64);
      const int issued = s_issued;
      for (int s = max(consumed, issued - NST); s < issued; ++s) mbar_wait(&full_bar[s % NST], (s / NST) & 1);
    }
    return;
  }

  // ---------------------------------------------------------------- epilogue
  auto row_value = [&](int r) {
    float v = 0.f;
    for (int q = 0; q < KS; ++q) v += part[(r - row0) * KS + q];
    if constexpr (F == MIE_FMT_I8) v *= reinterpret_cast<const float *>(m.s)[r];
    return v;
  };
  constexpr int kCT = NW * 32;

  if constexpr (EPI == EPI_STORE || EPI == EPI_RESID) {
    for (int r = row0 + tid; r < row1; r += kCT) {
      const float v = row_value(r);
      if constexpr (EPI == EPI_STORE) a.y[r] = v;
      else a.y[r] = a.y[r] + v;
    }
  } else if constexpr (EPI == EPI_SWIGLU) {
    // packed rows 2i = gate_i, 2i+1 = up_i -> y_i = silu(gate_i) * up_i
    for (int u = u0 + tid; u < u1; u += kCT) {
      const float g = row_value(2 * u), up = row_value(2 * u + 1);
      a.y[u] = g / (1.0f + expf(-g)) * up;
    }
  } else if constexpr (EPI == EPI_QKV) {
    if (tid == 0 && blockIdx.x == 0 && !qp.blk_ok) latch_error(a.err, qp.pos_ok ? ERR_BLOCK_ID : ERR_POS);
    for (int u = u0 + tid; u < u1; u += kCT) qkv_store(a, qp, u, row_value(2 * u), row_value(2 * u + 1));
  } else if constexpr (EPI == EPI_ARGMAX) {
    float *logits = a.y ? a.y : (a.sp ? a.sp->logits_out : nullptr);
    if (logits && a.sp && !a.y) logits += (int64_t)a.slot * M;
    float bv = -INFINITY;
    int bi = 0x7fffffff;
    for (int r = row0 + tid; r < row1; r += kCT) {
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
    if (lane == 0) { s_bv[warp] = bv; s_bi[warp] = bi; }
    consumer_sync<NW>();
    if (tid == 0) {
      for (int w = 1; w < NW; ++w)
        if (better(s_bv[w], s_bi[w], bv, bi)) { bv = s_bv[w]; bi = s_bi[w]; }
      a.am_part[blockIdx.x] = make_float2(bv, __int_as_float(bi));
      __threadfence();
      s_last = (atomicAdd(a.am_count, 1u) == gridDim.x - 1);
    }
    consumer_sync<NW>();
    if (s_last) {
      __threadfence();
      float fv = -INFINITY;
      int fi = 0x7fffffff;
      for (int b = tid; b < (int)gridDim.x; b += kCT) {
        const float2 p = __ldcg(a.am_part + b);
        if (better(p.x, __float_as_int(p.y), fv, fi)) { fv = p.x; fi = __float_as_int(p.y); }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, fv, o);
        const int oi = __shfl_xor_sync(0xffffffffu, fi, o);
        if (better(ov, oi, fv, fi)) { fv = ov; fi = oi; }
      }
      consumer_sync<NW>();
      if (lane == 0) { s_bv[warp] = fv; s_bi[warp] = fi; }
      consumer_sync<NW>();
      if (tid == 0) {
        for (int w = 1; w < NW; ++w)
          if (better(s_bv[w], s_bi[w], fv, fi)) { fv = s_bv[w]; fi = s_bi[w]; }
        if (fi == 0x7fffffff) fi = 0;  // all values NaN: fall back to index 0
        if (a.am_out) a.am_out[a.slot] = fi;
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
}

// --------------------------------------------------------------- launching

// Shared-memory plan of one launch: ring of n_stages stages plus the staged input and
// the per-row partial sums, kept under smem_budget(fmt) when possible (for bf16, so
// that a kernel and its successor prefetching under programmatic dependent launch fit
// on one SM).
struct Plan {
  int grid, n_stages;
  uint32_t stage_bytes, sc_bytes;
  size_t smem;
};

static Plan make_plan(const DevMat &m, int epi, int grid, int nw) {
  const int RU = (epi == EPI_SWIGLU || epi == EPI_QKV) ? 2 : 1;
  const int n_units = (m.rows + RU - 1) / RU;
  const int KS = (m.kp + kSlice - 1) / kSlice;
  const int RPS = (KS >= nw ? 1 : nw / KS) * fmt_rows_per_warp(m.fmt);
  const int rows_max = ((n_units + grid - 1) / grid) * RU;
  Plan p;
  p.grid = grid;
  p.stage_bytes = (uint32_t)((RPS * m.row_bytes + 127) / 128 * 128);
  p.sc_bytes = m.fmt == MIE_FMT_Q4_0 ? (uint32_t)((RPS * m.s_stride * 2 + 127) / 128 * 128) : 0u;
  const size_t fixed = sizeof(float) * ((size_t)xs_floats(m.kp) + (size_t)rows_max * KS);
  const int need = (rows_max + RPS - 1) / RPS;  // stages one CTA streams
  long avail = (long)smem_budget(m.fmt) - (long)fixed;
  int ns = (int)(avail > 0 ? avail / (long)(p.stage_bytes + p.sc_bytes) : 0);
  if (ns > kMaxStages) ns = kMaxStages;
  if (ns > need) ns = need;
  if (ns < 2) ns = 2;
  p.n_stages = ns;
  p.smem = fixed + (size_t)ns * (p.stage_bytes + p.sc_bytes);
  return p;
}

template <int F, int PRO, int EPI, int NW = kCWarps>
static mie_status launch_t(const GemvArgs &a0, int grid, cudaStream_t st, bool pdl) {
  const Plan p = make_plan(a0.m, EPI, grid, NW);
  if (p.smem > kSmemMax) return fail(MIE_E_SHAPE, "gemv: %zu bytes of shared memory needed", p.smem);
  GemvArgs a = a0;
  a.n_stages = p.n_stages;
  a.stage_bytes = p.stage_bytes;
  a.sc_stage_bytes = p.sc_bytes;
  auto kern = gemv_kernel<F, PRO, EPI, NW>;
  static bool configured[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !configured[dev]) {
    MIE_CUDA(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemMax));
    configured[dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.grid);
  cfg.blockDim = dim3(32 * (NW + 1));
  cfg.dynamicSmemBytes = p.smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  MIE_CUDA(cudaLaunchKernelEx(&cfg, kern, a));
  return MIE_OK;
}

template <int F>
static mie_status launch_f(int pro, int epi, const GemvArgs &a, int grid, cudaStream_t st, bool pdl) {
  // a long int8 or Q4_0 stream hides its unpack latency better with 12 consumer warps
  // (128256 x 2048: int8 82 -> 91 %, Q4_0 46 -> 49 % of HBM); smaller matrices measured
  // slower with them
  if constexpr (F == MIE_FMT_I8 || F == MIE_FMT_Q4_0)
    if (pro == PRO_PLAIN && epi == EPI_STORE && a.m.rows >= kWideRows)
      return launch_t<F, PRO_PLAIN, EPI_STORE, kCWarpsWide>(a, grid, st, pdl);
#define MIE_CASE(P, E) \
  if (pro == P && epi == E) return launch_t<F, P, E>(a, grid, st, pdl);
  MIE_CASE(PRO_PLAIN, EPI_STORE)
  MIE_CASE(PRO_PLAIN, EPI_RESID)
  MIE_CASE(PRO_NORM, EPI_SWIGLU)
  MIE_CASE(PRO_NORM, EPI_QKV)
  MIE_CASE(PRO_EMBED_NORM, EPI_QKV)
  MIE_CASE(PRO_NORM, EPI_ARGMAX)
#undef MIE_CASE
  return fail(MIE_E_ARG, "gemv: unsupported prologue/epilogue %d/%d", pro, epi);
}

int gemv_default_grid(const DevMat &m, int epi) {
  const int RU = (epi == EPI_SWIGLU || epi == EPI_QKV) ? 2 : 1;
  const int n_units = (m.rows + RU - 1) / RU;
  const int target = sm_count();
  return n_units < target ? n_units : target;
}

mie_status launch_gemv(int pro, int epi, const GemvArgs &a, int grid, cudaStream_t st, bool pdl) {
  if (a.m.kp > kMaxK) return fail(MIE_E_SHAPE, "gemv: K = %d exceeds %d", a.m.kp, kMaxK);
  if (((uintptr_t)a.m.w & 15) || (a.m.row_bytes & 15))
    return fail(MIE_E_SHAPE, "gemv: weight rows must start on 16-byte boundaries");
  if (a.m.fmt == MIE_FMT_Q4_0 && (((uintptr_t)a.m.s & 15) || (a.m.s_stride & 7)))
    return fail(MIE_E_SHAPE, "gemv: Q4_0 scale rows must start on 16-byte boundaries");
  if (grid < 1) grid = 1;
  switch (a.m.fmt) {
    case MIE_FMT_BF16: return launch_f<MIE_FMT_BF16>(pro, epi, a, grid, st, pdl);
    case MIE_FMT_I8: return launch_f<MIE_FMT_I8>(pro, epi, a, grid, st, pdl);
    case MIE_FMT_Q4_0: return launch_f<MIE_FMT_Q4_0>(pro, epi, a, grid, st, pdl);
    default: return fail(MIE_E_ARG, "gemv: unknown weight format %d", a.m.fmt);
  }
}

}  // namespace mie

// --------------------------------------------------------------- C ABI: stateless GEMVs

using namespace mie;

static mie_status gemv_entry(DevMat m, const float *x, float *y, void *stream) {
  if (!m.w || !x || !y) return fail(MIE_E_ARG, "gemv: null pointer");
  if (m.rows < 1 || m.cols < 1 || m.cols > kMaxK) return fail(MIE_E_SHAPE, "gemv: bad shape %d x %d", m.rows, m.cols);
  if (((uintptr_t)m.w & 15) != 0) return fail(MIE_E_SHAPE, "gemv: weights not 16-byte aligned");
  if ((const void *)x == (const void *)y) return fail(MIE_E_ARG, "gemv: y aliases x");
  GemvArgs a;
  a.m = m;
  a.x = x;
  a.y = y;
  // programmatic dependent launch: the weight stream may start during the previous
  // kernel's tail; x and y are touched only after its completion (see mie.h)
  return launch_gemv(PRO_PLAIN, EPI_STORE, a, gemv_default_grid(m, EPI_STORE), (cudaStream_t)stream, true);
}

extern "C" mie_status mie_gemv_bf16(const uint16_t *W, const float *x, float *y, int M, int K, void *stream) {
  if (K % 8 != 0) return fail(MIE_E_SHAPE, "mie_gemv_bf16: K = %d is not a multiple of 8", K);
  DevMat m;
  m.fmt = MIE_FMT_BF16;
  m.rows = M;
  m.cols = K;
  m.kp = K;
  m.w = reinterpret_cast<const uint8_t *>(W);
  m.row_bytes = (int64_t)K * 2;
  return gemv_entry(m, x, y, stream);
}

extern "C" mie_status mie_gemv_i8(const int8_t *W, const float *row_scale, const float *x, float *y, int M, int K,
                                  void *stream) {
  if (K % 16 != 0) return fail(MIE_E_SHAPE, "mie_gemv_i8: K = %d is not a multiple of 16", K);
  if (!row_scale) return fail(MIE_E_ARG, "mie_gemv_i8: null row_scale");
  DevMat m;
  m.fmt = MIE_FMT_I8;
  m.rows = M;
  m.cols = K;
  m.kp = K;
  m.w = reinterpret_cast<const uint8_t *>(W);
  m.s = row_scale;
  m.row_bytes = K;
  return gemv_entry(m, x, y, stream);
}

// GPU layout of a 4-bit matrix with `group` weights per scale: rows padded to whole
// groups, a nibble plane [M][kp/32][16], then at the next 256-byte boundary a scale plane
// [M][s_stride] of f16.
static bool q4_group_ok(int group) { return group == 32 || group == 64 || group == 128; }

extern "C" size_t mie_q4_packed_bytes(int M, int K, int group) {
  if (M < 1 || K < 1 || !q4_group_ok(group)) return 0;
  const size_t ng = (size_t)(K + group - 1) / group, nb = ng * (group / 32);
  const size_t nib = ((size_t)M * nb * 16 + 255) & ~(size_t)255;
  return nib + (size_t)M * q4_scale_stride((int)ng) * 2;
}

extern "C" size_t mie_q4_0_packed_bytes(int M, int K) { return mie_q4_packed_bytes(M, K, 32); }

extern "C" mie_status mie_gemv_q4(const void *packed, int group, const float *x, float *y, int M, int K,
                                  void *stream) {
  if (M < 1 || K < 1) return fail(MIE_E_SHAPE, "mie_gemv_q4: bad shape %d x %d", M, K);
  if (!q4_group_ok(group)) return fail(MIE_E_ARG, "mie_gemv_q4: group %d not 32, 64 or 128", group);
  const int ng = (K + group - 1) / group, nb = ng * (group / 32);
  DevMat m;
  m.fmt = MIE_FMT_Q4_0;
  m.gshift = q4_gshift(group);
  m.rows = M;
  m.cols = K;
  m.kp = nb * 32;
  m.w = reinterpret_cast<const uint8_t *>(packed);
  m.row_bytes = (int64_t)nb * 16;
  const size_t nib = ((size_t)M * nb * 16 + 255) & ~(size_t)255;
  m.s = reinterpret_cast<const uint8_t *>(packed) + nib;
  m.s_stride = q4_scale_stride(ng);
  return gemv_entry(m, x, y, stream);
}

extern "C" mie_status mie_gemv_q4_0(const void *packed, const float *x, float *y, int M, int K, void *stream) {
  return mie_gemv_q4(packed, 32, x, y, M, K, stream);
}
