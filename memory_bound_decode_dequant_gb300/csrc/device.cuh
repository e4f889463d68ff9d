// device.cuh -- device code shared by the GEMV kernels and the persistent step kernel:
// weight-format traits, in-register dequantisation, mbarrier and bulk-copy helpers.
#pragma once

#include "internal.h"

namespace mie {

template <int F> struct FmtT;
// EPC: elements per 16-byte chunk; CPL: chunks per lane per 2048-column slice; RPW:
// rows a warp reduces per stage, so that every format moves 8 x 16 bytes per lane per
// stage (a stage of one row per warp would be 8 KB for Q4_0, and the per-stage handoff
// would then cost more than the bytes: measured 27 % of HBM on the Q4_0 LM head).
template <> struct FmtT<MIE_FMT_BF16> { static constexpr int EPC = 8, CPL = 8, RPW = 1; };
template <> struct FmtT<MIE_FMT_I8> { static constexpr int EPC = 16, CPL = 4, RPW = 2; };
template <> struct FmtT<MIE_FMT_Q4_0> { static constexpr int EPC = 32, CPL = 2, RPW = 4; };

__host__ __device__ inline int fmt_rows_per_warp(int fmt) { return fmt == MIE_FMT_Q4_0 ? 4 : (fmt == MIE_FMT_I8 ? 2 : 1); }
constexpr int kSlice = 2048;  // = 32 * EPC * CPL for every format
constexpr int kMaxK = 16384;  // eight 2048-column slices

// --------------------------------------------------------------- element decoding

__device__ __forceinline__ float embed_at(const DevMat &m, int row, int k) {
  if (m.fmt == MIE_FMT_BF16) {
    return bf16_bits_to_f32(reinterpret_cast<const uint16_t *>(m.w + (int64_t)row * m.row_bytes)[k]);
  } else if (m.fmt == MIE_FMT_I8) {
    const int8_t q = reinterpret_cast<const int8_t *>(m.w + (int64_t)row * m.row_bytes)[k];
    return reinterpret_cast<const float *>(m.s)[row] * (float)q;
  } else {
    const uint8_t byte = m.w[(int64_t)row * m.row_bytes + (k >> 5) * 16 + (k & 15)];
    const int code = ((k & 31) < 16) ? (byte & 0xF) : (byte >> 4);
    const float h =
        __half2float(reinterpret_cast<const __half *>(m.s)[(int64_t)row * m.s_stride + (k >> (5 + m.gshift))]);
    return h * (float)(code - 8);
  }
}

// Dot product of one 16-byte chunk with the lane's input registers.
template <int F>
__device__ __forceinline__ void chunk_fma(const uint4 &w, const float2 *xr, float2 *acc);

template <>
__device__ __forceinline__ void chunk_fma<MIE_FMT_BF16>(const uint4 &w, const float2 *xr, float2 *acc) {
  const uint32_t v[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const float2 wf = make_float2(__uint_as_float(v[t] << 16), __uint_as_float(v[t] & 0xffff0000u));
    acc[t] = __ffma2_rn(wf, xr[t], acc[t]);
  }
}

// The quantised formats read their codes as subnormal floats.  A code n of b bits left
// in place at bit offset p, every other bit cleared, is the float n 2^(p-149) as long as
// the word stays below 2^24 (exponent field 0 or 1, where the value of the bits is the
// integer times 2^-149).  The input registers hold x 2^(126-p-E), where E is the binary
// exponent of the largest |x| of the registers' group (a Q4_0 chunk, or all of an int8
// lane's chunks) clamped to [-1, 104]: every register stays below 2^127, and one packed
// FMA adds n x 2^-(E+23) with a single rounding, a normal float for every x down to
// 2^-103 of the group's largest.  The group's sum times 2^(E+23) plus its bias term (-8
// or -128 times the sum of its inputs, formed when the inputs are loaded) is then the
// dot product with the signed codes.  This leaves one packed FMA per two codes in the
// inner loop, where a biased-mantissa form also needs a packed add.  Inputs of 2^105 or
// more in magnitude overflow the registers.  Flush-to-zero would erase every code, so
// these kernels are never built with it.
#if defined(__USE_FAST_MATH__)
#error "the quantised dot products need subnormal floats: build without fast math"
#endif
template <uint32_t MASK>
__device__ __forceinline__ float code_bits(uint32_t a) {
  return __uint_as_float(a & MASK);
}

// int8 chunk: word t holds elements 4t..4t+3, byte j = element 4t+j; b ^ 0x80 = b + 128
// is the unsigned code.  Bytes 0..2 are read in place (p = 0, 8, 16); byte 3 is moved
// down to byte 2 (p = 16), since in place it would reach the exponent's upper bits.
template <>
__device__ __forceinline__ void chunk_fma<MIE_FMT_I8>(const uint4 &w, const float2 *xr, float2 *acc) {
  const uint32_t v[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const uint32_t u = v[t] ^ 0x80808080u;
    const float2 a = make_float2(code_bits<0xFFu>(u), code_bits<0xFF00u>(u));
    const float2 b = make_float2(code_bits<0xFF0000u>(u), __uint_as_float(__byte_perm(u, 0u, 0x4344)));
    acc[t] = __ffma2_rn(a, xr[2 * t], acc[t]);
    acc[t] = __ffma2_rn(b, xr[2 * t + 1], acc[t]);
  }
}

// Q4_0 chunk = one block: word t holds bytes 4t..4t+3; byte j carries element j (low
// nibble) and element j+16 (high nibble).  Unpack order per word, with the bit offset
// p the code sits at: 4t(p0) 4t+16(p4) 4t+1(p8) 4t+17(p12) 4t+2(p16), then from
// w >> 12: 4t+18(p8) 4t+3(p12) 4t+19(p16); load_lane_xr puts x 2^(126-p-E) in that order.
template <>
__device__ __forceinline__ void chunk_fma<MIE_FMT_Q4_0>(const uint4 &w, const float2 *xr, float2 *acc) {
  const uint32_t v[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const uint32_t a = v[t], s = v[t] >> 12;
    acc[t] = __ffma2_rn(make_float2(code_bits<0xFu>(a), code_bits<0xF0u>(a)), xr[4 * t + 0], acc[t]);
    acc[t] = __ffma2_rn(make_float2(code_bits<0xF00u>(a), code_bits<0xF000u>(a)), xr[4 * t + 1], acc[t]);
    acc[t] = __ffma2_rn(make_float2(code_bits<0xF0000u>(a), code_bits<0xF00u>(s)), xr[4 * t + 2], acc[t]);
    acc[t] = __ffma2_rn(make_float2(code_bits<0xF000u>(s), code_bits<0xF0000u>(s)), xr[4 * t + 3], acc[t]);
  }
}

// Staged input vectors keep four spare floats after every 32 elements: element k sits
// at xs_at(k).  A lane's chunk (8, 16 or 32 consecutive elements) then starts 36, 18
// or 9 float4 slots after its neighbour's, so the float4 reads of a warp fill the 32
// banks evenly (unpadded, the 32 lanes of a Q4_0 warp all start on the same bank).
__host__ __device__ constexpr int xs_at(int k) { return k + ((k >> 5) << 2); }
__host__ __device__ constexpr int xs_floats(int Kp) { return Kp + ((Kp + 31) >> 5) * 4; }

// 2^k for -126 <= k <= 127
__device__ __forceinline__ float pow2i(int k) { return __uint_as_float((uint32_t)(k + 127) << 23); }

// Largest |value| and sum of the N float pairs v, both by pairwise trees (short
// dependency chains: this runs at the start of every GEMV phase).
template <int N>
__device__ __forceinline__ void group_max_sum(const float2 *v, float &m, float &sum) {
  float mx[N], sm[N];
#pragma unroll
  for (int i = 0; i < N; ++i) {
    mx[i] = fmaxf(fabsf(v[i].x), fabsf(v[i].y));
    sm[i] = v[i].x + v[i].y;
  }
#pragma unroll
  for (int w = N / 2; w >= 1; w /= 2) {
#pragma unroll
    for (int i = 0; i < w; ++i) {
      mx[i] = fmaxf(mx[i], mx[i + w]);
      sm[i] += sm[i + w];
    }
  }
  m = mx[0];
  sum = sm[0];
}

// The exponent E of the subnormal-code scaling for a group whose largest |x| is m.
__device__ __forceinline__ int code_exp(float m) {
  const int e = (int)((__float_as_uint(m) >> 23) & 0xFFu) - 127;
  return min(max(e, -1), 104);
}

// A lane's input registers for a phase, from the staged vector xs: chunk c covers
// elements e0 + c*32*EPC .. +EPC-1 (zeros where the lane has no slice or the chunk is
// at or past Kp), in chunk_fma's order and scaling.  nb and cs get the bias terms and
// the scales 2^(E+23) that stage_rows_dot applies: per chunk for Q4_0, nb[0] and cs[0]
// for the whole lane for int8, none for bf16.
template <int F>
__device__ __forceinline__ void load_lane_xr(const float *xs, int e0, int Kp, bool has_slice, float2 *xr, float *nb,
                                             float *cs) {
  using T = FmtT<F>;
  constexpr int EPC = T::EPC, CPL = T::CPL, R = EPC / 2;  // R registers per chunk
#pragma unroll
  for (int c = 0; c < CPL; ++c) {
    const int e = e0 + c * 32 * EPC;
    float2 *r = xr + c * R;
    if (has_slice && e < Kp) {
      const float4 *q4 = reinterpret_cast<const float4 *>(xs + xs_at(e));
      if constexpr (F == MIE_FMT_Q4_0) {
#pragma unroll
        for (int t = 0; t < 4; ++t) {  // register 4t+j pairs elements 4t+j and 4t+16+j
          const float4 a = q4[t], b = q4[t + 4];
          r[4 * t + 0] = make_float2(a.x, b.x);
          r[4 * t + 1] = make_float2(a.y, b.y);
          r[4 * t + 2] = make_float2(a.z, b.z);
          r[4 * t + 3] = make_float2(a.w, b.w);
        }
      } else {
#pragma unroll
        for (int i = 0; i < EPC / 4; ++i) {
          const float4 q = q4[i];
          r[2 * i] = make_float2(q.x, q.y);
          r[2 * i + 1] = make_float2(q.z, q.w);
        }
      }
    } else {
#pragma unroll
      for (int i = 0; i < R; ++i) r[i] = make_float2(0.f, 0.f);
    }
  }
  if constexpr (F == MIE_FMT_Q4_0) {
#pragma unroll
    for (int c = 0; c < CPL; ++c) {
      float2 *r = xr + c * R;
      float m, sx;
      group_max_sum<R>(r, m, sx);
      const int E = code_exp(m);
      // bit offsets of the pairs: (0, 4), (8, 12), (16, 8), (12, 16)
      const float s0 = pow2i(126 - E), s4 = pow2i(122 - E), s8 = pow2i(118 - E), s12 = pow2i(114 - E),
                  s16 = pow2i(110 - E);
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        r[4 * t + 0] = make_float2(r[4 * t + 0].x * s0, r[4 * t + 0].y * s4);
        r[4 * t + 1] = make_float2(r[4 * t + 1].x * s8, r[4 * t + 1].y * s12);
        r[4 * t + 2] = make_float2(r[4 * t + 2].x * s16, r[4 * t + 2].y * s8);
        r[4 * t + 3] = make_float2(r[4 * t + 3].x * s12, r[4 * t + 3].y * s16);
      }
      nb[c] = -8.f * sx;
      cs[c] = pow2i(E + 23);
    }
  } else if constexpr (F == MIE_FMT_I8) {
    float m, sx;
    group_max_sum<CPL * R>(xr, m, sx);
    const int E = code_exp(m);
    const float s0 = pow2i(126 - E), s8 = pow2i(118 - E), s16 = pow2i(110 - E);  // bytes 0, 1, 2 and 3
#pragma unroll
    for (int i = 0; i < CPL * R / 2; ++i) {
      xr[2 * i] = make_float2(xr[2 * i].x * s0, xr[2 * i].y * s8);
      xr[2 * i + 1] = make_float2(xr[2 * i + 1].x * s16, xr[2 * i + 1].y * s16);
    }
    nb[0] = -128.f * sx;
    cs[0] = pow2i(E + 23);
  }
}

// --------------------------------------------------------------- mbarrier / bulk copy

__device__ __forceinline__ uint32_t smem_u32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

// Explicit shared-memory loads by 32-bit shared address (pointers into the dynamic
// shared memory of the persistent kernel reach the math through structs, where the
// compiler could not prove their address space and would emit generic loads).
__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
  return v;
}
__device__ __forceinline__ float4 lds128f(uint32_t a) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(a));
  return v;
}
__device__ __forceinline__ uint32_t lds32(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ uint32_t lds16(uint32_t a) {
  unsigned short v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(a));
  return v;
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Waits for the phase of the given parity to complete; gives up after a bounded number
// of polls (each poll may suspend the thread for a hardware-defined time) and returns
// false, so a lost transfer can never hang the GPU.
__device__ __forceinline__ bool mbar_try(uint32_t addr, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(addr), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, long limit = kWaitPolls) {
  const uint32_t addr = smem_u32(bar);
  for (long it = 0; it < limit; ++it)
    if (mbar_try(addr, parity)) return true;
  return false;
}
// The same wait that also gives up once *abort is set (checked every 64 polls): a CTA
// whose partner warps or other CTAs have left stops waiting for them at once.
__device__ __forceinline__ bool mbar_wait_or_abort(uint64_t *bar, uint32_t parity, long limit, const int *abort) {
  const uint32_t addr = smem_u32(bar);
  for (long it = 0; it < limit; ++it) {
    if (mbar_try(addr, parity)) return true;
    if ((it & 63) == 63 && *reinterpret_cast<const volatile int *>(abort)) return false;
  }
  return false;
}

// One bulk (TMA 1-D) copy global -> shared, completing on an mbarrier; weights are
// streamed once, so they are marked evict-first in L2.
__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes, uint64_t *bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(pol)
      : "memory");
}

// Orders this thread's generic-proxy accesses to shared memory before later async-proxy
// (bulk copy) accesses, e.g. before a ring slot written by threads goes back to TMA.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void sts16(uint32_t a, uint16_t v) {
  asm volatile("st.shared.u16 [%0], %1;" ::"r"(a), "h"(v) : "memory");
}

__device__ __forceinline__ uint64_t evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// Dot products of this lane's part of the RPW consecutive weight rows of this warp,
// staged in shared memory, with its input registers xr: row = shared address of the
// first row's 2048-column slice (the others at row + i*row_bytes), sc = shared address
// of its 4-bit scales (the others at sc + i*s_bytes; chunk j of the slice uses scale
// j >> gshift).  Every chunk and scale of all rows is loaded before any math, so the
// loads cost one shared-memory latency.  Chunks at or
// past Kp are read from the slice start instead (always staged) and meet zero input
// registers, so they add exact zeros.  nrows (<= RPW) rows are valid; the others read
// the first row.  nb and cs hold load_lane_xr's bias terms and scales.
template <int F>
__device__ __forceinline__ void stage_rows_dot(uint32_t row, uint32_t row_bytes, uint32_t sc, uint32_t s_bytes,
                                               int nrows, const float2 *xr, const float *nb, const float *cs,
                                               int e0, int Kp, int lane, float (&sum)[FmtT<F>::RPW],
                                               int gshift = 0) {
  using T = FmtT<F>;
  constexpr int EPC = T::EPC, CPL = T::CPL, R = T::RPW, kChunkStride = 32 * EPC;
  uint4 w[R][CPL];
#pragma unroll
  for (int i = 0; i < R; ++i) {
    const uint32_t ra = row + (uint32_t)(i < nrows ? i : 0) * row_bytes;
#pragma unroll
    for (int c = 0; c < CPL; ++c) w[i][c] = lds128(e0 + c * kChunkStride < Kp ? ra + (uint32_t)(c * 32 + lane) * 16 : ra);
  }
  if constexpr (F == MIE_FMT_Q4_0) {
    uint32_t hb[R][CPL];
#pragma unroll
    for (int i = 0; i < R; ++i) {
      const uint32_t sa = sc + (uint32_t)(i < nrows ? i : 0) * s_bytes;
#pragma unroll
      for (int c = 0; c < CPL; ++c)
        hb[i][c] = lds16(e0 + c * kChunkStride < Kp ? sa + (uint32_t)((c * 32 + lane) >> gshift) * 2 : sa);
    }
#pragma unroll
    for (int i = 0; i < R; ++i) {
      float acc_s = 0.f;
#pragma unroll
      for (int c = 0; c < CPL; ++c) {
        float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
        chunk_fma<F>(w[i][c], xr + c * (EPC / 2), acc);
        const float t = (acc[0].x + acc[0].y) + (acc[1].x + acc[1].y) + (acc[2].x + acc[2].y) + (acc[3].x + acc[3].y);
        acc_s = fmaf(__half2float(__ushort_as_half((unsigned short)hb[i][c])), fmaf(t, cs[c], nb[c]), acc_s);
      }
      sum[i] = acc_s;
    }
  } else {
#pragma unroll
    for (int i = 0; i < R; ++i) {
      float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
      for (int c = 0; c < CPL; ++c) chunk_fma<F>(w[i][c], xr + c * (EPC / 2), acc);
      const float t = (acc[0].x + acc[0].y) + (acc[1].x + acc[1].y) + (acc[2].x + acc[2].y) + (acc[3].x + acc[3].y);
      if constexpr (F == MIE_FMT_I8) {
        sum[i] = fmaf(t, cs[0], nb[0]);
      } else {
        sum[i] = t;
      }
    }
  }
}

__device__ __forceinline__ bool better(float v, int i, float bv, int bi) {
  return v > bv || (v == bv && i < bi);
}

// RMSNorm of the staged vector xs (element k at xs_at(k), k < K) in place (PRO_NORM,
// PRO_EMBED_NORM), or only the bf16 rounding of PRO_PLAIN inputs when act_bf16 is set.
// sq is this thread's share of the sum of squares of the staged values, taken while
// they were staged; with `published` the warps' sums already sit in red[] behind a
// barrier, otherwise they are reduced here.  Every thread then forms the same scale
// from red[] (same order), so no thread waits on another for it.  g0, when not null,
// holds the gains of elements tid + j*NT (j < 8), loaded by the caller ahead of time
// (K <= 8*NT).  NT threads take part; Sync is a barrier over them.  The caller
// synchronises before xs is read.
template <int NT, class Sync>
__device__ void normalize_staged(const GemvArgs &a, int pro, float *xs, int K, float *red, const float *g0, float sq,
                                 bool published) {
  constexpr int B = 8;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (pro != PRO_PLAIN) {
    if (!published) {
      sq = warp_sum(sq);
      if (lane == 0) red[warp] = sq;
      Sync::sync();
    }
    float t = 0.f;
#pragma unroll
    for (int w = 0; w < NT / 32; ++w) t += red[w];
    const float r = 1.0f / sqrtf(t / (float)K + a.eps);
    for (int k0 = tid; k0 < K; k0 += NT * B) {
      float g[B];
#pragma unroll
      for (int j = 0; j < B; ++j) g[j] = g0 ? g0[j] : __ldg(a.gain + min(k0 + j * NT, K - 1));
#pragma unroll
      for (int j = 0; j < B; ++j) {
        const int k = k0 + j * NT;
        if (k < K) {
          float v = xs[xs_at(k)] * r * g[j];
          if (a.act_bf16) v = round_bf16(v);
          xs[xs_at(k)] = v;
        }
      }
    }
  } else if (a.act_bf16) {
    for (int k = tid; k < K; k += NT) xs[xs_at(k)] = round_bf16(xs[xs_at(k)]);
  }
}

// Stages a GEMV input vector into shared memory xs (element k at xs_at(k), zeros from K
// to Kp), applying the
// prologue: PRO_PLAIN copies x; PRO_NORM applies RMSNorm with the gain; PRO_EMBED_NORM
// gathers row sp->token of the embedding first (CTA 0 also stores it as the residual).
// With act_bf16 the staged values are rounded to bf16.  Each thread issues a batch of
// independent loads (addresses clamped into range, values masked afterwards) before
// its first shared-memory store, so the staging costs one round trip per batch instead
// of one per element.  NT threads take part; Sync is a barrier over them.
template <int NT, class Sync>
__device__ void stage_input(const GemvArgs &a, int pro, float *xs, int K, int Kp, float *red, int *err) {
  constexpr int B = 8;
  const int tid = threadIdx.x;
  // a vector that one batch covers gets its gains loaded together with its values
  const bool one_batch = pro != PRO_PLAIN && K <= NT * B;
  float g0[B], sq = 0.f;
  if (one_batch) {
#pragma unroll
    for (int j = 0; j < B; ++j) g0[j] = __ldg(a.gain + min(tid + j * NT, K - 1));
  }
  if (pro == PRO_EMBED_NORM) {
    int tok = a.sp ? a.sp->token[a.slot] : 0;
    if (tok < 0 || tok >= a.vocab) {
      if (tid == 0 && blockIdx.x == 0) latch_error(err, ERR_TOKEN);
      tok = 0;
    }
    for (int k0 = tid; k0 < Kp; k0 += NT * B) {
      float v[B];
#pragma unroll
      for (int j = 0; j < B; ++j) v[j] = embed_at(a.embed, tok, min(k0 + j * NT, K - 1));
#pragma unroll
      for (int j = 0; j < B; ++j) {
        const int k = k0 + j * NT;
        if (k < Kp) xs[xs_at(k)] = (k < K) ? v[j] : 0.f;
        if (k < K) sq = fmaf(v[j], v[j], sq);
        if (blockIdx.x == 0 && k < K) a.x_store[k] = v[j];
      }
    }
  } else {
    for (int k0 = tid; k0 < Kp; k0 += NT * B) {
      float v[B];
#pragma unroll
      for (int j = 0; j < B; ++j) v[j] = __ldcg(a.x + min(k0 + j * NT, K - 1));
#pragma unroll
      for (int j = 0; j < B; ++j) {
        const int k = k0 + j * NT;
        if (k < Kp) xs[xs_at(k)] = (k < K) ? v[j] : 0.f;
        if (k < K) sq = fmaf(v[j], v[j], sq);
      }
    }
  }
  normalize_staged<NT, Sync>(a, pro, xs, K, red, one_batch ? g0 : nullptr, sq, false);
  Sync::sync();
}

// --------------------------------------------------------------- tagged words
//
// Between the phases of the persistent step every value travels as one 64-bit word:
// the fp32 bits in the low half and the launch's tag in the high half.  A 64-bit
// aligned access is single-copy atomic, so a reader that sees the current tag also
// sees the value written with it; it polls the words themselves instead of meeting the
// writers at a barrier first.  Words left by an earlier launch carry an older tag.

__device__ __forceinline__ void st_tagged(uint64_t *p, float v, uint32_t tag) {
  const uint64_t w = ((uint64_t)tag << 32) | (uint64_t)__float_as_uint(v);
  asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(w) : "memory");
}

__device__ __forceinline__ void ld_tagged2(const uint64_t *p, uint64_t &w0, uint64_t &w1) {
  asm volatile("ld.relaxed.gpu.global.v2.b64 {%0, %1}, [%2];" : "=l"(w0), "=l"(w1) : "l"(p) : "memory");
}

__device__ __forceinline__ uint64_t ld_tagged(const uint64_t *p) {
  uint64_t w;
  asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(w) : "l"(p) : "memory");
  return w;
}

__device__ __forceinline__ bool tag_ok(uint64_t w, uint32_t tag) { return (uint32_t)(w >> 32) == tag; }
__device__ __forceinline__ float tag_val(uint64_t w) { return __uint_as_float((uint32_t)w); }

constexpr long kTagPolls = 1L << 22;  // bounded polling of tagged words (seconds)

// Polls n pairs of tagged words until all carry `tag`.  map(j, src, dst, n) names pair
// j: its source (16-byte aligned when both words are wanted), its destination in
// shared memory, and how many words it has (1 or 2).  The squares of the values of
// pairs j < n_sq are added to *sq.  Each thread polls its own pairs, B per round trip,
// and gives up after `limit` rounds or once *abort is set; returns false then.
template <int NT, int B, class Map>
__device__ bool poll_pairs(int n, uint32_t tag, const int *abort, long limit, Map map, int n_sq = 0,
                           float *sq = nullptr) {
  const int tid = threadIdx.x;
  for (int j0 = tid; j0 < n; j0 += NT * B) {
    uint32_t pending = 0;
#pragma unroll
    for (int i = 0; i < B; ++i)
      if (j0 + i * NT < n) pending |= 1u << i;
    for (long it = 0; pending; ++it) {
      uint64_t w0[B], w1[B];
#pragma unroll
      for (int i = 0; i < B; ++i) {
        w0[i] = w1[i] = 0;
        if ((pending >> i) & 1u) {
          const uint64_t *src;
          float *dst;
          int cnt;
          map(j0 + i * NT, src, dst, cnt);
          if (cnt == 2) ld_tagged2(src, w0[i], w1[i]);
          else w0[i] = ld_tagged(src);
        }
      }
#pragma unroll
      for (int i = 0; i < B; ++i) {
        if (!((pending >> i) & 1u)) continue;
        const uint64_t *src;
        float *dst;
        int cnt;
        map(j0 + i * NT, src, dst, cnt);
        if (tag_ok(w0[i], tag) && (cnt < 2 || tag_ok(w1[i], tag))) {
          const float v0 = tag_val(w0[i]), v1 = cnt == 2 ? tag_val(w1[i]) : 0.f;
          dst[0] = v0;
          if (cnt == 2) dst[1] = v1;
          if (j0 + i * NT < n_sq) *sq = fmaf(v1, v1, fmaf(v0, v0, *sq));
          pending &= ~(1u << i);
        }
      }
      if (pending) {
        if (it >= limit) return false;
        if ((it & 63) == 63 && *reinterpret_cast<const volatile int *>(abort)) return false;
        __nanosleep(32);
      }
    }
  }
  return true;
}

// What the QKV epilogue needs besides the GEMV results, read before the weights are
// streamed so that the epilogue issues no dependent loads: the position, its KV
// block, and the rows of RoPE angles for that position.
struct QkvPrefetch {
  int pos = 0, blk = -1;
  bool pos_ok = false, blk_ok = false;
  const float *crow = nullptr, *srow = nullptr;
};

__device__ __forceinline__ QkvPrefetch qkv_prefetch(const GemvArgs &a) {
  QkvPrefetch q;
  q.pos = a.sp->pos[a.slot];
  const int h2 = a.hd / 2;
  q.pos_ok = q.pos >= 0 && q.pos < a.max_pos && q.pos / a.bs < a.sp->max_blocks;
  const int pos_c = q.pos_ok ? q.pos : 0;
  q.blk = a.sp->block_table[(int64_t)a.slot * a.sp->max_blocks + pos_c / a.bs];
  q.blk_ok = q.pos_ok && q.blk >= 0 && q.blk < a.n_kv_blocks;
  q.crow = a.rope_cos + (int64_t)pos_c * h2;
  q.srow = a.rope_sin + (int64_t)pos_c * h2;
  return q;
}

// The QKV epilogue for pair unit u: RoPE on q and k rows, q to q_out, bf16 k/v into
// the paged cache.  x0, x1 are the GEMV results of rows i and i + hd/2 of head h.
__device__ __forceinline__ void qkv_store(const GemvArgs &a, const QkvPrefetch &q, int u, float x0, float x1) {
  const int h2 = a.hd / 2;
  const int h = u / h2, i = u % h2;
  if (h < a.Hq + a.Hkv && q.pos_ok) {
    const float c = q.crow[i], sn = q.srow[i];
    const float r0 = x0 * c - x1 * sn, r1 = x1 * c + x0 * sn;
    x0 = r0;
    x1 = r1;
  }
  if (h < a.Hq) {
    a.q_out[h * a.hd + i] = x0;
    a.q_out[h * a.hd + i + h2] = x1;
  } else if (q.blk_ok) {
    const int isv = h >= a.Hq + a.Hkv;
    const int g = h - a.Hq - (isv ? a.Hkv : 0);
    uint16_t *dst = a.kv_layer + (int64_t)q.blk * a.block_stride + (int64_t)isv * a.Hkv * a.bs * a.hd +
                    ((int64_t)g * a.bs + q.pos % a.bs) * a.hd;
    dst[i] = __bfloat16_as_ushort(__float2bfloat16_rn(x0));
    dst[i + h2] = __bfloat16_as_ushort(__float2bfloat16_rn(x1));
  }
}

}  // namespace mie
