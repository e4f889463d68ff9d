// prefill.cu -- the prompt's token-parallel kernels around the tensor-core GEMM.
//
// "infer" page, summary table and "Limitations": a prompt of T tokens goes through the
// same layer as a decode step, for all T positions at once: RMSNorm, the QKV product,
// RoPE and the K/V write into the paged cache, causal attention of every position over
// the cache up to itself, the O product with the residual, RMSNorm, gate/up, SwiGLU, the
// down product with the residual ("Writing an LLM inference engine from scratch in
// Rust", "How a Llama model generates text"; "Mini Inference Engine", the paged cache).
// The products run in gemm.cu; here are the row-wise steps between them, which also cut
// every GEMM input into bf16 planes, and the flash-style prefill attention.
//
// Attention (one CTA = one query head x 64 query positions, 4 warps x 16 rows): the K/V
// of 64 keys at a time come from the paged cache through the block table into shared
// memory; S = Q K^T and O += P V run on mma.sync m16n8k16 with Q and P as three bf16
// planes each (K and V are bf16 already), with a running maximum and sum per row; keys
// after a query's own position are masked (causal).
#include <mutex>

#include "internal.h"
#include "device.cuh"

namespace mie {

namespace {

__device__ __forceinline__ uint16_t bf16_bits_rn(float v) { return __bfloat16_as_ushort(__float2bfloat16_rn(v)); }

// hi = bf16(v), mid = bf16(v - hi), lo = bf16(v - hi - mid): both differences are exact in
// fp32, and hi + mid + lo is v to 2^-25 of v
__device__ __forceinline__ void split3(float v, uint16_t &hi, uint16_t &mid, uint16_t &lo) {
  hi = bf16_bits_rn(v);
  const float r = v - bf16_bits_to_f32(hi);
  mid = bf16_bits_rn(r);
  lo = bf16_bits_rn(r - bf16_bits_to_f32(mid));
}
// hi = bf16(v), lo = bf16(v - hi): a 4-bit weight (at most 14 significant bits) exactly
__device__ __forceinline__ void split2(float v, uint16_t &hi, uint16_t &lo) {
  hi = bf16_bits_rn(v);
  lo = bf16_bits_rn(v - bf16_bits_to_f32(hi));
}

__device__ __forceinline__ uint32_t pack2(uint16_t a, uint16_t b) { return (uint32_t)a | ((uint32_t)b << 16); }

template <int NT>
__device__ __forceinline__ float block_sum(float v, float *red) {
  v = warp_sum(v);
  const int w = threadIdx.x >> 5;
  if ((threadIdx.x & 31) == 0) red[w] = v;
  __syncthreads();
  float t = 0.f;
#pragma unroll
  for (int i = 0; i < NT / 32; ++i) t += red[i];
  __syncthreads();
  return t;
}

constexpr int kRowThreads = 256;

// Token rows of the embedding: R[t] = E[tok[t]] (dequantised).
__global__ void __launch_bounds__(kRowThreads) embed_rows_kernel(DevMat e, const int32_t *tok, int vocab, int d,
                                                                 float *R, int *err) {
  const int t = blockIdx.x;
  int id = tok[t];
  if (id < 0 || id >= vocab) {
    if (threadIdx.x == 0) latch_error(err, ERR_TOKEN);
    id = 0;
  }
  for (int k = threadIdx.x; k < d; k += kRowThreads) R[(int64_t)t * d + k] = embed_at(e, id, k);
}

// One row of x (RMSNorm with gain g first when g is set) as planes hi / mid / lo;
// act_bf16: the value is rounded to bf16 (hi alone), as the decode step rounds its GEMV
// inputs of such models.
__global__ void __launch_bounds__(kRowThreads) norm_split_kernel(const float *x, int64_t ldx, int K, const float *g,
                                                                 float eps, int act_bf16, uint16_t *hi, uint16_t *mid,
                                                                 uint16_t *lo, int64_t ldp) {
  __shared__ float red[kRowThreads / 32];
  const int t = blockIdx.x;
  const float *row = x + (int64_t)t * ldx;
  float r = 1.f;
  if (g) {
    float sq = 0.f;
    for (int k = threadIdx.x; k < K; k += kRowThreads) sq = fmaf(row[k], row[k], sq);
    const float tot = block_sum<kRowThreads>(sq, red);
    r = 1.0f / sqrtf(tot / (float)K + eps);
  }
  for (int k = threadIdx.x; k < K; k += kRowThreads) {
    float v = g ? row[k] * r * g[k] : row[k];
    if (act_bf16) v = round_bf16(v);
    uint16_t h, m, l;
    split3(v, h, m, l);
    hi[(int64_t)t * ldp + k] = h;
    if (mid) mid[(int64_t)t * ldp + k] = m;
    if (lo) lo[(int64_t)t * ldp + k] = l;
  }
}

// QKV epilogue of every position: Y[t] holds the product's rows in the step's pair order
// (row 2u = row i of head h, row 2u + 1 = row i + hd/2, u = h * hd/2 + i); RoPE at
// position pos0 + t on q and k, q to Q[t][h*hd + ...] in fp32, k and v rounded to bf16
// into the paged cache through the block table.
__global__ void __launch_bounds__(kRowThreads) rope_kv_kernel(RopeKvArgs a) {
  const int t = blockIdx.x, pos = a.pos0 + t, h2 = a.hd / 2;
  const int n_pairs = (a.Hq + 2 * a.Hkv) * h2;
  const int b = pos / a.bs;
  int blk = (b < a.n_table) ? a.bt[b] : -1;
  if (blk < 0 || blk >= a.n_pool) {
    if (threadIdx.x == 0) latch_error(a.err, b < a.n_table ? ERR_BLOCK_ID : ERR_POS);
    blk = -1;
  }
  const float *crow = a.cos_t + (int64_t)pos * h2, *srow = a.sin_t + (int64_t)pos * h2;
  for (int u = threadIdx.x; u < n_pairs; u += kRowThreads) {
    const int h = u / h2, i = u % h2;
    float x0 = a.Y[(int64_t)t * a.ldy + 2 * u], x1 = a.Y[(int64_t)t * a.ldy + 2 * u + 1];
    if (h < a.Hq + a.Hkv) {
      const float c = crow[i], sn = srow[i];
      const float r0 = x0 * c - x1 * sn, r1 = x1 * c + x0 * sn;
      x0 = r0;
      x1 = r1;
    }
    if (h < a.Hq) {
      a.Q[(int64_t)t * a.Hq * a.hd + h * a.hd + i] = x0;
      a.Q[(int64_t)t * a.Hq * a.hd + h * a.hd + i + h2] = x1;
    } else if (blk >= 0) {
      const int isv = h >= a.Hq + a.Hkv;
      const int g = h - a.Hq - (isv ? a.Hkv : 0);
      uint16_t *dst = a.kv_layer + (int64_t)blk * a.block_stride + (int64_t)isv * a.Hkv * a.bs * a.hd +
                      ((int64_t)g * a.bs + pos % a.bs) * a.hd;
      dst[i] = bf16_bits_rn(x0);
      dst[i + h2] = bf16_bits_rn(x1);
    }
  }
}

// SwiGLU of every position (Y[t][2u] gate, Y[t][2u + 1] up) as planes hi / mid / lo.
__global__ void __launch_bounds__(kRowThreads) swiglu_split_kernel(const float *Y, int64_t ldy, int F, int act_bf16,
                                                                   uint16_t *hi, uint16_t *mid, uint16_t *lo,
                                                                   int64_t ldp) {
  const int t = blockIdx.x;
  for (int u = threadIdx.x; u < F; u += kRowThreads) {
    const float g = Y[(int64_t)t * ldy + 2 * u], up = Y[(int64_t)t * ldy + 2 * u + 1];
    float v = g / (1.0f + expf(-g)) * up;
    if (act_bf16) v = round_bf16(v);
    uint16_t h, m, l;
    split3(v, h, m, l);
    hi[(int64_t)t * ldp + u] = h;
    if (mid) mid[(int64_t)t * ldp + u] = m;
    if (lo) lo[(int64_t)t * ldp + u] = l;
  }
}

// A quantised matrix as bf16 planes for the GEMM: int8 rows as their codes (exact; the
// row scale is applied by the GEMM), 4-bit rows as hi / lo of scale * (code - 8).
__global__ void __launch_bounds__(kRowThreads) dequant_planes_kernel(DevMat m, uint16_t *hi, uint16_t *lo,
                                                                     int64_t ldp) {
  const int r = blockIdx.x;
  for (int k = threadIdx.x; k < m.cols; k += kRowThreads) {
    if (m.fmt == MIE_FMT_I8) {
      hi[(int64_t)r * ldp + k] = bf16_bits_rn((float)reinterpret_cast<const int8_t *>(m.w + (int64_t)r * m.row_bytes)[k]);
    } else {
      uint16_t h, l;
      split2(embed_at(m, r, k), h, l);
      hi[(int64_t)r * ldp + k] = h;
      lo[(int64_t)r * ldp + k] = l;
    }
  }
}

// ------------------------------------------------------------------ attention

__device__ __forceinline__ void mma_bf16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

constexpr int kAttnRows = 64;  // query positions per CTA
constexpr int kAttnKeys = 64;  // keys per shared-memory tile
constexpr int kAttnThreads = 128;

// Dynamic shared memory of the kernel: two buffers (the next 64 keys are copied while the
// current 64 are reduced), each K then V, rows padded to HD*2 + 16 bytes.
__host__ __device__ constexpr int attn_pitch(int hd) { return hd * 2 + 16; }
__host__ __device__ constexpr size_t attn_smem_bytes(int hd) { return 2u * 2u * kAttnKeys * attn_pitch(hd); }

template <int HD>
__global__ void __launch_bounds__(kAttnThreads) prefill_attn_kernel(PrefillAttnArgs a) {
  constexpr int PITCH = attn_pitch(HD);  // bytes per staged key row: conflict-free fragment loads
  constexpr int NKS = HD / 16, NOT = HD / 8, CPR = HD / 8;  // Q k-steps, O n-tiles, 16-byte chunks per row
  constexpr uint32_t kBuf = 2u * kAttnKeys * PITCH;         // one buffer: K then V
  extern __shared__ __align__(16) uint8_t att_smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, quad = lane >> 2, tq4 = lane & 3;
  const int h = blockIdx.y, g = h / (a.Hq / a.Hkv);
  const int qt0 = blockIdx.x * kAttnRows;
  const int qlast = min(qt0 + kAttnRows, a.T) - 1;  // last query row of this CTA
  const int kend = a.pos0 + qlast + 1;               // keys 0 .. kend - 1 are needed

  // Q fragments of this warp's 16 rows (rows quad and quad + 8), pre-scaled by
  // scale * log2(e) so that the softmax runs on exp2
  int tr[2];
  tr[0] = qt0 + warp * 16 + quad;
  tr[1] = tr[0] + 8;
  const float qs = a.scale * 1.4426950408889634f;
  uint32_t qp[3][NKS][4];  // planes hi / mid / lo
#pragma unroll
  for (int ks = 0; ks < NKS; ++ks) {
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int row = tr[r & 1], d = ks * 16 + tq4 * 2 + (r >> 1) * 8;
      float2 v = make_float2(0.f, 0.f);
      if (row < a.T) v = *reinterpret_cast<const float2 *>(a.q + (int64_t)row * a.ldq + h * HD + d);
      uint16_t p0[3], p1[3];
      split3(v.x * qs, p0[0], p0[1], p0[2]);
      split3(v.y * qs, p1[0], p1[1], p1[2]);
#pragma unroll
      for (int j = 0; j < 3; ++j) qp[j][ks][r] = pack2(p0[j], p1[j]);
    }
  }
  float o[NOT][4];
#pragma unroll
  for (int n = 0; n < NOT; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
  const int qpos[2] = {a.pos0 + tr[0], a.pos0 + tr[1]};
  const int qpos_min = a.pos0 + qt0;  // keys up to it are visible to every row of the CTA
  const uint16_t *kbase = a.k + (int64_t)g * a.bs * HD, *vbase = a.v + (int64_t)g * a.bs * HD;
  const uint32_t sm0 = smem_u32(att_smem);

  // keys k0 .. k0 + 63 into buffer b (zeros past kend), as one cp.async group
  auto stage = [&](int b, int k0) {
    const uint32_t kb = sm0 + (uint32_t)b * kBuf, vb = kb + (uint32_t)(kAttnKeys * PITCH);
    for (int c = threadIdx.x; c < kAttnKeys * CPR; c += kAttnThreads) {
      const int key = c / CPR, ch = c % CPR, p = k0 + key;
      const uint32_t off = (uint32_t)(key * PITCH + ch * 16);
      if (p < kend) {
        int blk = a.bt[p / a.bs];
        if (blk < 0 || blk >= a.n_pool) {
          latch_error(a.err, ERR_BLOCK_ID);
          blk = 0;
        }
        const int64_t e = (int64_t)blk * a.block_stride + (int64_t)(p % a.bs) * HD + ch * 8;
        cp_async16(kb + off, kbase + e);
        cp_async16(vb + off, vbase + e);
      } else {
        asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(kb + off), "r"(0u) : "memory");
        asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(vb + off), "r"(0u) : "memory");
      }
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  };

  stage(0, 0);
  int t = 0;
  for (int k0 = 0; k0 < kend; k0 += kAttnKeys, ++t) {
    const bool more = k0 + kAttnKeys < kend;
    if (more) stage((t + 1) & 1, k0 + kAttnKeys);  // its buffer was released by the last barrier
    if (more) asm volatile("cp.async.wait_group 1;" ::: "memory");
    else asm volatile("cp.async.wait_group 0;" ::: "memory");
    __syncthreads();
    const uint32_t ks0 = sm0 + (uint32_t)(t & 1) * kBuf, vs0 = ks0 + (uint32_t)(kAttnKeys * PITCH);

    // S = Q K^T for 8 tiles of 8 keys (log2 units)
    float s[8][4];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
      const uint32_t krow = ks0 + (uint32_t)((j * 8 + quad) * PITCH + tq4 * 4);
#pragma unroll
      for (int ks = 0; ks < NKS; ++ks) {
        const uint32_t b0 = lds32(krow + ks * 32), b1 = lds32(krow + ks * 32 + 16);
#pragma unroll
        for (int pl = 2; pl >= 0; --pl)  // smallest plane first
          mma_bf16(s[j], qp[pl][ks][0], qp[pl][ks][1], qp[pl][ks][2], qp[pl][ks][3], b0, b1);
      }
    }
    // causal mask (only a tile reaching past the CTA's first position needs it), running
    // maximum and sum per row
    const bool masked = k0 + kAttnKeys - 1 > qpos_min;
    float corr[2];
#pragma unroll
    for (int rh = 0; rh < 2; ++rh) {
      float mx = -INFINITY;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          float v = s[j][rh * 2 + e];
          if (masked && k0 + j * 8 + tq4 * 2 + e > qpos[rh]) v = -INFINITY;
          s[j][rh * 2 + e] = v;
          mx = fmaxf(mx, v);
        }
      }
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      const float m_new = fmaxf(m[rh], mx);
      float sum = 0.f;
      if (m_new == -INFINITY) {
        corr[rh] = 1.f;
#pragma unroll
        for (int j = 0; j < 8; ++j) s[j][rh * 2] = s[j][rh * 2 + 1] = 0.f;
      } else {
        corr[rh] = exp2f(m[rh] - m_new);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const float p = exp2f(s[j][rh * 2 + e] - m_new);
            s[j][rh * 2 + e] = p;
            sum += p;
          }
        }
      }
      l[rh] = l[rh] * corr[rh] + sum;
      m[rh] = m_new;
    }
#pragma unroll
    for (int n = 0; n < NOT; ++n) {
      o[n][0] *= corr[0];
      o[n][1] *= corr[0];
      o[n][2] *= corr[1];
      o[n][3] *= corr[1];
    }
    // O += P V, 16 keys per step
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      // A fragments of P (keys 16 kk ..): registers 0 / 1 rows quad / quad + 8 of the
      // first 8 keys, 2 / 3 the same rows of the next 8; three planes each
      uint32_t pp[3][4];
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const float *src = s[2 * kk + (r >> 1)] + (r & 1) * 2;
        uint16_t p0[3], p1[3];
        split3(src[0], p0[0], p0[1], p0[2]);
        split3(src[1], p1[0], p1[1], p1[2]);
#pragma unroll
        for (int j = 0; j < 3; ++j) pp[j][r] = pack2(p0[j], p1[j]);
      }
      const int mi = lane >> 3, ri = lane & 7;
#pragma unroll
      for (int np = 0; np < NOT / 2; ++np) {
        const uint32_t addr =
            vs0 + (uint32_t)((kk * 16 + (mi & 1) * 8 + ri) * PITCH + (np * 16 + (mi >> 1) * 8) * 2);
        uint32_t r0, r1, r2, r3;
        ldsm_x4_trans(addr, r0, r1, r2, r3);
#pragma unroll
        for (int pl = 2; pl >= 0; --pl) {
          mma_bf16(o[2 * np], pp[pl][0], pp[pl][1], pp[pl][2], pp[pl][3], r0, r1);
          mma_bf16(o[2 * np + 1], pp[pl][0], pp[pl][1], pp[pl][2], pp[pl][3], r2, r3);
        }
      }
    }
    __syncthreads();  // the buffer is free for the copy two tiles on
  }
  // normalise and store
#pragma unroll
  for (int rh = 0; rh < 2; ++rh) {
    float L = l[rh];
    L += __shfl_xor_sync(0xffffffffu, L, 1);
    L += __shfl_xor_sync(0xffffffffu, L, 2);
    const float inv = L > 0.f ? 1.f / L : 0.f;
    if (tr[rh] < a.T) {
      float *dst = a.out + (int64_t)tr[rh] * a.ldo + h * HD;
#pragma unroll
      for (int n = 0; n < NOT; ++n) {
        dst[n * 8 + tq4 * 2] = o[n][rh * 2] * inv;
        dst[n * 8 + tq4 * 2 + 1] = o[n][rh * 2 + 1] * inv;
      }
    }
  }
}

int blocks_of(int64_t n, int per) { return (int)((n + per - 1) / per); }

}  // namespace

mie_status launch_embed_rows(const DevMat &e, const int32_t *tok, int T, int vocab, int d, float *R, int *err,
                             cudaStream_t st) {
  embed_rows_kernel<<<T, kRowThreads, 0, st>>>(e, tok, vocab, d, R, err);
  MIE_CUDA(cudaGetLastError());
  return MIE_OK;
}

mie_status launch_norm_split(const float *x, int64_t ldx, int K, const float *g, float eps, int act_bf16, int T,
                             uint16_t *hi, uint16_t *mid, uint16_t *lo, int64_t ldp, cudaStream_t st) {
  norm_split_kernel<<<T, kRowThreads, 0, st>>>(x, ldx, K, g, eps, act_bf16, hi, mid, lo, ldp);
  MIE_CUDA(cudaGetLastError());
  return MIE_OK;
}

mie_status launch_rope_kv(const RopeKvArgs &a, cudaStream_t st) {
  rope_kv_kernel<<<a.T, kRowThreads, 0, st>>>(a);
  MIE_CUDA(cudaGetLastError());
  return MIE_OK;
}

mie_status launch_swiglu_split(const float *Y, int64_t ldy, int F, int act_bf16, int T, uint16_t *hi, uint16_t *mid,
                               uint16_t *lo, int64_t ldp, cudaStream_t st) {
  swiglu_split_kernel<<<T, kRowThreads, 0, st>>>(Y, ldy, F, act_bf16, hi, mid, lo, ldp);
  MIE_CUDA(cudaGetLastError());
  return MIE_OK;
}

mie_status launch_dequant_planes(const DevMat &m, uint16_t *hi, uint16_t *lo, int64_t ldp, cudaStream_t st) {
  if (m.fmt != MIE_FMT_I8 && m.fmt != MIE_FMT_Q4_0) return fail(MIE_E_ARG, "dequant planes: format %d", m.fmt);
  if (m.fmt == MIE_FMT_Q4_0 && !lo) return fail(MIE_E_ARG, "dequant planes: 4-bit weights need a lo plane");
  dequant_planes_kernel<<<m.rows, kRowThreads, 0, st>>>(m, hi, lo, ldp);
  MIE_CUDA(cudaGetLastError());
  return MIE_OK;
}

mie_status launch_prefill_attn(const PrefillAttnArgs &a, cudaStream_t st) {
  if (a.T < 1) return MIE_OK;
  if (a.Hq % a.Hkv) return fail(MIE_E_SHAPE, "prefill attention: Hq %% Hkv != 0");
  if (kAttnKeys % a.bs) return fail(MIE_E_SHAPE, "prefill attention: block size %d", a.bs);
  const dim3 grid((unsigned)blocks_of(a.T, kAttnRows), (unsigned)a.Hq);
  auto go = [&](auto kern, int hd) -> mie_status {
    const size_t smem = attn_smem_bytes(hd);
    if (smem > 48 * 1024) {
      static std::once_flag once;
      static cudaError_t set = cudaSuccess;
      std::call_once(once, [&] { set = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem); });
      if (set != cudaSuccess) return cuda_fail(set, "prefill attention: cudaFuncSetAttribute");
    }
    kern<<<grid, kAttnThreads, smem, st>>>(a);
    return MIE_OK;
  };
  mie_status s;
  switch (a.hd) {
    case 32: s = go(prefill_attn_kernel<32>, 32); break;
    case 64: s = go(prefill_attn_kernel<64>, 64); break;
    case 128: s = go(prefill_attn_kernel<128>, 128); break;
    default: return fail(MIE_E_SHAPE, "prefill attention: head_dim %d", a.hd);
  }
  if (s != MIE_OK) return s;
  MIE_CUDA(cudaGetLastError());
  return MIE_OK;
}

}  // namespace mie

using namespace mie;

extern "C" mie_status mie_split_bf16(const float *x, int64_t n, uint16_t *hi, uint16_t *mid, uint16_t *lo,
                                     void *stream) {
  if (!x || !hi) return fail(MIE_E_ARG, "mie_split_bf16: null pointer");
  if (n < 1 || n >= (int64_t)1 << 31) return fail(MIE_E_SHAPE, "mie_split_bf16: n = %lld", (long long)n);
  // one row of n values
  return launch_norm_split(x, n, (int)n, nullptr, 0.f, 0, 1, hi, mid, lo, n, (cudaStream_t)stream);
}

extern "C" mie_status mie_paged_attn_prefill(const float *q, const uint16_t *k_pool, const uint16_t *v_pool,
                                             int64_t block_stride, int n_pool_blocks, const int32_t *block_table,
                                             int n_table, int pos0, int T, int n_q_heads, int n_kv_heads,
                                             int head_dim, int block_size, float scale, float *out, void *stream) {
  if (!q || !k_pool || !v_pool || !block_table || !out) return fail(MIE_E_ARG, "mie_paged_attn_prefill: null pointer");
  if (T < 0 || pos0 < 0 || n_kv_heads < 1 || n_q_heads < n_kv_heads || n_pool_blocks < 1 || block_size < 1)
    return fail(MIE_E_ARG, "mie_paged_attn_prefill: bad sizes");
  if ((int64_t)pos0 + T > (int64_t)n_table * block_size)
    return fail(MIE_E_ARG, "mie_paged_attn_prefill: positions up to %d need more than %d table entries", pos0 + T - 1,
                n_table);
  PrefillAttnArgs a;
  a.q = q;
  a.ldq = (int64_t)n_q_heads * head_dim;
  a.k = k_pool;
  a.v = v_pool;
  a.block_stride = block_stride;
  a.n_pool = n_pool_blocks;
  a.bt = block_table;
  a.pos0 = pos0;
  a.T = T;
  a.Hq = n_q_heads;
  a.Hkv = n_kv_heads;
  a.hd = head_dim;
  a.bs = block_size;
  a.scale = scale;
  a.out = out;
  a.ldo = (int64_t)n_q_heads * head_dim;
  a.err = device_error_flag();
  return launch_prefill_attn(a, (cudaStream_t)stream);
}
