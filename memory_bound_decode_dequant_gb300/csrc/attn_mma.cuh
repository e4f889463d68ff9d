// attn_mma.cuh -- decode attention over a chunk of K/V on the tensor cores (mma.sync
// m16n8k16, bf16 operands, fp32 accumulation), one warp per 32 tokens with its own
// online softmax ("Writing an LLM inference engine from scratch in Rust", Lesson 4:
// running maximum and sum; "infer" page, design notes, the split-KV attention item: the
// query heads of one KV head share every K/V load, partial softmaxes are merged).
//
// Layout.  K and V of a chunk sit in shared memory as the tiles a 2-D tensor copy with
// 128-byte swizzle writes: per 64-dimension half of a row, `rows` token rows of 128 bytes,
// the 16-byte chunk c of row r stored at chunk position c ^ (r & 7) (buffers start on a
// 1024-byte boundary).  Operand fragments are read with ldmatrix (K as is, V transposed),
// whose eight row addresses then fall in eight different bank groups.  (Copies of 16-byte
// boxes into an unswizzled chunk-major layout were measured on GB300 to take longer than
// the tensor-core math saved.)
//
// Rows of the MMA.  fp32 queries are split into three bf16 planes q = q0 + q1 + q2 (24
// significant bits, so q * k is the fp32 product); row 4h + p of a 16-row tile holds plane
// p of head h (four heads per tile, row 4h + 3 zero), so S = Q K^T comes out per plane and
// two shuffles add the planes.  The probabilities P (in [0, 1]) are split the same way
// for O = P V.  Scores are taken in log2 units: q is scaled by scale * log2(e) first and
// exp2 replaces exp.
#pragma once

#include "device.cuh"

namespace mie {

constexpr int kMmaTokPerWarp = 32;  // tokens of a chunk per warp (four 8-token score tiles)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Shared address of 16-byte chunk c (0 .. HD/8-1) of token row r in a swizzled K or V
// buffer of `rows` rows per 64-dimension half.
__device__ __forceinline__ uint32_t swz_addr(uint32_t base, int rows, int r, int c) {
  return base + (uint32_t)(c >> 3) * (uint32_t)rows * 128u + (uint32_t)r * 128u + ((uint32_t)((c & 7) ^ (r & 7)) << 4);
}

// One 2-D tensor copy (box of the map at element column x, row y) into shared memory,
// completing on the mbarrier at shared address bar.
__device__ __forceinline__ void tma_load_tile(uint32_t dst, const CUtensorMap *map, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void sts128_zero(uint32_t addr) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(addr), "r"(0u) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

// D += A B for one m16n8k16 tile, bf16 operands, fp32 accumulators.
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Plane p (0, 1, 2) of an exact three-plane bf16 split of v, as a float (plane 3: zero):
// t0 = v with its low 16 bits cleared, t1 = v - t0 likewise, t2 = v - t0 - t1.  Both
// differences are exact and each plane holds at most 8 significant bits, so the planes
// are bf16 values that add up to v.  Bit masks instead of rounding conversions: those
// run on a narrow pipe and were measured on GB300 to cost more than the MMAs they feed.
__device__ __forceinline__ float bf16_plane(float v, int p) {
  const float t0 = __uint_as_float(__float_as_uint(v) & 0xffff0000u);
  const float r = v - t0;
  const float t1 = __uint_as_float(__float_as_uint(r) & 0xffff0000u);
  const float t2 = r - t1;
  return p == 0 ? t0 : (p == 1 ? t1 : (p == 2 ? t2 : 0.f));
}
// Two bf16-exact floats as a bf16 pair (lo in the low half).
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  return __byte_perm(__float_as_uint(lo), __float_as_uint(hi), 0x7632);
}

// Running state of one warp for the two head rows of one 16-row tile that its lanes
// hold (h1 = 4 mt + (lane >> 4), h2 = h1 + 2): statistics in log2 units, the lane's
// part of the row sums, and the output fragments (dims 8n + 2t, 8n + 2t + 1 of plane p).
template <int HD>
struct WarpAttn {
  float m[2], l[2];
  float o[HD / 8][4];
  __device__ __forceinline__ void reset() {
    m[0] = m[1] = -INFINITY;
    l[0] = l[1] = 0.f;
#pragma unroll
    for (int n = 0; n < HD / 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  }
};

// The A fragments of the queries, built once per CTA into shared memory: q holds the
// G x HD queries of the group, c = scale * log2(e).  Lane (gq, t) holds rows gq and
// gq + 8 of tile mt, i.e. plane p = gq & 3 of heads h1 = 4 mt + gq / 4 and h2 = h1 + 2
// (zero past G); item (mt, s) of k-step s sits at qf[(mt * HD / 16 + s) * 32 + lane],
// computed by warp (item mod NW).  The caller synchronises before the fragments are read.
template <int G, int HD, int NW>
__device__ __forceinline__ void q_fragments_shared(const float *q, float c, uint4 *qf) {
  constexpr int MT = (G + 3) / 4, KS = HD / 16;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, gq = lane >> 2, t = lane & 3, p = gq & 3;
  for (int item = warp; item < MT * KS; item += NW) {
    const int mt = item / KS, s = item % KS;
    const int h1 = 4 * mt + (gq >> 2), h2 = h1 + 2;
    float v[2][4];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int h = r ? h2 : h1;
      if (h < G && p < 3) {
        const float *qr = q + h * HD + 16 * s + 2 * t;
        v[r][0] = bf16_plane(qr[0] * c, p);
        v[r][1] = bf16_plane(qr[1] * c, p);
        v[r][2] = bf16_plane(qr[8] * c, p);
        v[r][3] = bf16_plane(qr[9] * c, p);
      } else {
        v[r][0] = v[r][1] = v[r][2] = v[r][3] = 0.f;
      }
    }
    qf[item * 32 + lane] = make_uint4(pack_bf16(v[0][0], v[0][1]), pack_bf16(v[1][0], v[1][1]),
                                      pack_bf16(v[0][2], v[0][3]), pack_bf16(v[1][2], v[1][3]));
  }
}

// One warp over tokens tok0 .. tok0 + 31 (those below ntok) of a swizzled K/V chunk of
// `rows` rows: scores, the online-softmax update of st, and O += P V.  V rows from ntok up
// to the next multiple of 16 must hold finite values (their P is zero).
template <int HD>
__device__ __forceinline__ void warp_chunk_mma(uint32_t kb, uint32_t vb, int rows, int tok0, int ntok,
                                               const uint32_t (&qa)[HD / 16][4], WarpAttn<HD> &st) {
  const int lane = threadIdx.x & 31, gq = lane >> 2, t = lane & 3, p = gq & 3;
  if (tok0 >= ntok) return;
  // S = Q K^T over four 8-token tiles; ldmatrix x4 brings two k-steps of one tile
  float s[4][4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
    const int row = tok0 + 8 * j + (lane & 7);
#pragma unroll
    for (int q2 = 0; q2 < HD / 32; ++q2) {
      uint32_t b[4];
      ldsm_x4(swz_addr(kb, rows, row, 4 * q2 + (lane >> 3)), b);
      mma16816(s[j], qa[2 * q2], b[0], b[1]);
      mma16816(s[j], qa[2 * q2 + 1], b[2], b[3]);
    }
  }
  // add the three planes (lanes gq, gq ^ 1, gq ^ 2, gq ^ 3 of the same head rows), mask
  float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      float v = s[j][e];
      v += __shfl_xor_sync(0xffffffffu, v, 4);
      v += __shfl_xor_sync(0xffffffffu, v, 8);
      const int tok = tok0 + 8 * j + 2 * t + (e & 1);
      v = tok < ntok ? v : -INFINITY;
      s[j][e] = v;
      mx[e >> 1] = fmaxf(mx[e >> 1], v);
    }
  }
  float corr[2];
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
    mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
    const float m_new = fmaxf(st.m[r], mx[r]);
    corr[r] = (st.m[r] == -INFINITY) ? 0.f : exp2f(st.m[r] - m_new);
    st.m[r] = m_new;
  }
  // probabilities; the lane keeps plane p of them for the A fragments of P V
  float pl[4][4];
#pragma unroll
  for (int r = 0; r < 2; ++r) st.l[r] *= corr[r];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float m = st.m[e >> 1];
      const float pr = (s[j][e] == -INFINITY) ? 0.f : exp2f(s[j][e] - m);
      st.l[e >> 1] += pr;
      pl[j][e] = bf16_plane(pr, p);
    }
  }
#pragma unroll
  for (int n = 0; n < HD / 8; ++n) {
    st.o[n][0] *= corr[0];
    st.o[n][1] *= corr[0];
    st.o[n][2] *= corr[1];
    st.o[n][3] *= corr[1];
  }
  // O += P V: two 16-token k-steps; ldmatrix x4 (transposed) brings two 8-dim tiles
#pragma unroll
  for (int kk = 0; kk < 2; ++kk) {
    if (tok0 + 16 * kk >= ntok) break;
    uint32_t a[4];
    a[0] = pack_bf16(pl[2 * kk][0], pl[2 * kk][1]);
    a[1] = pack_bf16(pl[2 * kk][2], pl[2 * kk][3]);
    a[2] = pack_bf16(pl[2 * kk + 1][0], pl[2 * kk + 1][1]);
    a[3] = pack_bf16(pl[2 * kk + 1][2], pl[2 * kk + 1][3]);
    const int row = tok0 + 16 * kk + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
    for (int c2 = 0; c2 < HD / 16; ++c2) {
      uint32_t b[4];
      ldsm_x4_t(swz_addr(vb, rows, row, 2 * c2 + (lane >> 4)), b);
      mma16816(st.o[2 * c2], a, b[0], b[1]);
      mma16816(st.o[2 * c2 + 1], a, b[2], b[3]);
    }
  }
}

// End of a warp's tokens for tile mt: row sums over the quad, planes added, and the
// warp's (m, l, O) for its heads written to shared memory: wm / wl [warp][G], wo
// [warp][G][HD].  Warps that saw no token write m = -inf.
template <int G, int HD>
__device__ __forceinline__ void warp_attn_store(WarpAttn<HD> &st, int mt, float *wm, float *wl, float *wo) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, gq = lane >> 2, t = lane & 3, p = gq & 3;
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    st.l[r] += __shfl_xor_sync(0xffffffffu, st.l[r], 1);
    st.l[r] += __shfl_xor_sync(0xffffffffu, st.l[r], 2);
  }
#pragma unroll
  for (int n = 0; n < HD / 8; ++n) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      float v = st.o[n][e];
      v += __shfl_xor_sync(0xffffffffu, v, 4);
      v += __shfl_xor_sync(0xffffffffu, v, 8);
      st.o[n][e] = v;
    }
  }
  if (p != 0) return;
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int h = 4 * mt + (gq >> 2) + 2 * r;
    if (h >= G) continue;
    if (t == 0) {
      wm[warp * G + h] = st.m[r];
      wl[warp * G + h] = st.l[r];
    }
    float *dst = wo + ((size_t)warp * G + h) * HD;
#pragma unroll
    for (int n = 0; n < HD / 8; ++n) {
      dst[8 * n + 2 * t] = st.o[n][2 * r];
      dst[8 * n + 2 * t + 1] = st.o[n][2 * r + 1];
    }
  }
}

// Output i (head i / HD, dim i % HD) of the CTA from the NW warps' parts: the log2-unit
// maximum M, the sum L and the unnormalised output O.
template <int G, int HD, int NW>
__device__ __forceinline__ void cta_attn_combine(int i, const float *wm, const float *wl, const float *wo, float &M,
                                                 float &L, float &O) {
  const int h = i / HD;
  M = -INFINITY;
#pragma unroll
  for (int w = 0; w < NW; ++w) M = fmaxf(M, wm[w * G + h]);
  L = 0.f;
  O = 0.f;
  if (M == -INFINITY) return;
#pragma unroll
  for (int w = 0; w < NW; ++w) {
    const float mw = wm[w * G + h];
    if (mw == -INFINITY) continue;
    const float f = exp2f(mw - M);
    L = fmaf(wl[w * G + h], f, L);
    O = fmaf(wo[(size_t)w * G * HD + i], f, O);
  }
}

}  // namespace mie
