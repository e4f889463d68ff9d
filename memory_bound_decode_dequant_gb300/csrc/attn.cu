// attn.cu -- paged GQA decode attention and argmax on sm_103a.
//
// Attention ("Mini Inference Engine", "The KV cache, paged like virtual memory": the
// kernel reads K/V through a block table; "infer" page, "GQA-aware split-KV attention":
// one CTA per KV head serves the query heads of its group, the context is split and
// the partial softmaxes are merged; "Writing an LLM inference engine from scratch in
// Rust", Lesson 4: an online softmax with a running maximum and sum).
//
// Grid (splits, KV heads), 128 threads; the number of splits in use follows the
// context (at least 4 blocks each).  A CTA stages the block ids of its split in shared
// memory, then each warp takes groups of 32/LPT tokens (LPT = head_dim/32 lanes per
// token) and issues all of a group's loads before any math: 64 bytes of one key per
// lane, plus the lane's head_dim/32 value dims of every token in the group.  Each
// key is dotted with every query head of the group (one K/V read serves them all),
// the LPT lanes of a token combine with a shuffle, and each warp keeps an online
// softmax per head.  Warps merge in shared memory; with one split the CTA writes the
// result, otherwise CTAs write (m, l, o) partials and the last CTA of each KV head to
// finish (an atomic counter, no waiting) merges them and resets the counter.
#include "internal.h"

namespace mie {

constexpr int kAttnThreads = 128;
constexpr int kAttnWarps = kAttnThreads / 32;
constexpr int kAttnMaxBlocks = 256;     // block ids staged in shared memory at a time
constexpr int kAttnBlocksPerSplit = 4;  // one block per warp per split, at least

__device__ int g_device_error;  // latched by the stateless kernels of this device

template <int G, int HD>
__global__ void __launch_bounds__(kAttnThreads) attn_kernel(const AttnArgs a) {
  constexpr int LPT = HD / 32;          // lanes per token (each lane dots 32 dims)
  constexpr int TPI = 32 / LPT;         // tokens per warp iteration
  constexpr int DPL = HD / 32;          // value dims per lane
  constexpr int PART = G * (2 + HD);    // floats of one (head group, split) partial
  __shared__ __align__(16) float q_s[G * HD];
  __shared__ int s_blk[kAttnMaxBlocks];
  __shared__ float w_m[kAttnWarps][G], w_l[kAttnWarps][G];
  __shared__ float w_o[kAttnWarps][G][HD];
  __shared__ unsigned s_last;
  __shared__ int s_nsplit;

  pdl_trigger();
  pdl_wait();

  const int g = blockIdx.y, s = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int ctx;
  const int32_t *bt;
  int n_table;
  if (a.sp) {
    ctx = a.sp->pos[a.slot] + 1;
    bt = a.sp->block_table + (int64_t)a.slot * a.sp->max_blocks;
    n_table = a.sp->max_blocks;
  } else {
    ctx = a.ctx;
    bt = a.block_table;
    n_table = a.n_table;
  }
  if (ctx > n_table * a.bs) {
    if (threadIdx.x == 0 && s == 0 && g == 0) latch_error(a.err, ERR_POS);
    ctx = n_table * a.bs;
  }
  if (ctx < 0) ctx = 0;
  const int nblk = (ctx + a.bs - 1) / a.bs;
  // at least kAttnBlocksPerSplit blocks per split, so every warp has a block to read
  const int nsplit = max(1, min(a.n_splits, (nblk + kAttnBlocksPerSplit - 1) / kAttnBlocksPerSplit));
  if (s >= nsplit) return;
  const int b0 = (int)((int64_t)s * nblk / nsplit), b1 = (int)((int64_t)(s + 1) * nblk / nsplit);
  const int t_end = min(b1 * a.bs, ctx);

  for (int i = threadIdx.x; i < G * HD; i += kAttnThreads) q_s[i] = a.q[(g * G) * HD + i];

  float m[G], l[G], o[G][DPL];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    m[h] = -INFINITY;
    l[h] = 0.f;
#pragma unroll
    for (int d = 0; d < DPL; ++d) o[h][d] = 0.f;
  }
  const int tok_in = lane / LPT, part_in = lane % LPT;
  const int64_t head_off = (int64_t)g * a.bs * HD;

  // the split's blocks, staged kAttnMaxBlocks at a time (one coalesced load each)
  for (int cb = b0; cb < b1; cb += kAttnMaxBlocks) {
    const int ce = min(b1, cb + kAttnMaxBlocks);
    __syncthreads();
    for (int i = threadIdx.x; i < ce - cb; i += kAttnThreads) {
      int blk = bt[cb + i];
      if (blk < 0 || blk >= a.n_pool_blocks) {
        latch_error(a.err, ERR_BLOCK_ID);
        blk = -1;
      }
      s_blk[i] = blk;
    }
    __syncthreads();
    const int t0 = cb * a.bs, t1 = min(ce * a.bs, t_end);
    for (int tb = t0 + warp * TPI; tb < t1; tb += kAttnWarps * TPI) {
      const int nt = min(TPI, t1 - tb);
      // issue every load of this token group first: my key slice, then my value dims
      const int t = tb + tok_in;
      const int kblk = (t < t1) ? s_blk[t / a.bs - cb] : -1;
      uint4 kv[4];
      if (kblk >= 0) {
        const uint16_t *kp = a.k + (int64_t)kblk * a.block_stride + head_off + (int64_t)(t % a.bs) * HD + part_in * 32;
#pragma unroll
        for (int i = 0; i < 4; ++i) kv[i] = *reinterpret_cast<const uint4 *>(kp + 8 * i);
      }
      float vf[TPI][DPL];
#pragma unroll
      for (int i = 0; i < TPI; ++i) {
        const int t2 = tb + i;
        const int vblk = (i < nt) ? s_blk[t2 / a.bs - cb] : -1;
        if (vblk >= 0) {
          const uint16_t *vp = a.v + (int64_t)vblk * a.block_stride + head_off + (int64_t)(t2 % a.bs) * HD + lane * DPL;
          if constexpr (DPL == 1) {
            vf[i][0] = bf16_bits_to_f32(*vp);
          } else if constexpr (DPL == 2) {
            const uint32_t w = *reinterpret_cast<const uint32_t *>(vp);
            vf[i][0] = __uint_as_float(w << 16);
            vf[i][1] = __uint_as_float(w & 0xffff0000u);
          } else {
            const uint2 w = *reinterpret_cast<const uint2 *>(vp);
            vf[i][0] = __uint_as_float(w.x << 16);
            vf[i][1] = __uint_as_float(w.x & 0xffff0000u);
            vf[i][2] = __uint_as_float(w.y << 16);
            vf[i][3] = __uint_as_float(w.y & 0xffff0000u);
          }
        } else {
#pragma unroll
          for (int d = 0; d < DPL; ++d) vf[i][d] = 0.f;
        }
      }
      // scores of my token for every query head of the group
      float sc[G];
      if (kblk >= 0) {
        float kf[32];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint32_t w[4] = {kv[i].x, kv[i].y, kv[i].z, kv[i].w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            kf[8 * i + 2 * j] = __uint_as_float(w[j] << 16);
            kf[8 * i + 2 * j + 1] = __uint_as_float(w[j] & 0xffff0000u);
          }
        }
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float *qh = q_s + h * HD + part_in * 32;
          float d0 = 0.f, d1 = 0.f;
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            d0 = fmaf(qh[i], kf[i], d0);
            d1 = fmaf(qh[i + 1], kf[i + 1], d1);
          }
          sc[h] = d0 + d1;
        }
      } else {
#pragma unroll
        for (int h = 0; h < G; ++h) sc[h] = 0.f;
      }
#pragma unroll
      for (int h = 0; h < G; ++h) {
#pragma unroll
        for (int off = 1; off < LPT; off <<= 1) sc[h] += __shfl_xor_sync(0xffffffffu, sc[h], off);
        sc[h] = (kblk >= 0) ? sc[h] * a.scale : -INFINITY;
      }
      // online softmax: rescale the running sums to the new maximum
      float p[G];
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float mn = fmaxf(m[h], warp_max(sc[h]));
        if (mn == -INFINITY) {
          p[h] = 0.f;
          continue;
        }
        const float corr = expf(m[h] - mn);  // 0 while m was -inf
        p[h] = (sc[h] == -INFINITY) ? 0.f : expf(sc[h] - mn);
        const float ps = warp_sum(part_in == 0 ? p[h] : 0.f);  // each token counted once
        l[h] = l[h] * corr + ps;
#pragma unroll
        for (int d = 0; d < DPL; ++d) o[h][d] *= corr;
        m[h] = mn;
      }
#pragma unroll
      for (int i = 0; i < TPI; ++i) {
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float ph = __shfl_sync(0xffffffffu, p[h], i * LPT);
#pragma unroll
          for (int d = 0; d < DPL; ++d) o[h][d] = fmaf(ph, vf[i][d], o[h][d]);
        }
      }
    }
  }

  // merge the warps of this CTA
  if (lane == 0) {
#pragma unroll
    for (int h = 0; h < G; ++h) { w_m[warp][h] = m[h]; w_l[warp][h] = l[h]; }
  }
#pragma unroll
  for (int h = 0; h < G; ++h)
#pragma unroll
    for (int d = 0; d < DPL; ++d) w_o[warp][h][lane * DPL + d] = o[h][d];
  __syncthreads();
  if (nsplit == 1) {  // the only split: write the result directly
    for (int i = threadIdx.x; i < G * HD; i += kAttnThreads) {
      const int h = i / HD, d = i % HD;
      float M = -INFINITY;
      for (int w = 0; w < kAttnWarps; ++w) M = fmaxf(M, w_m[w][h]);
      float O = 0.f, L = 0.f;
      for (int w = 0; w < kAttnWarps; ++w) {
        const float f = (w_m[w][h] == -INFINITY) ? 0.f : expf(w_m[w][h] - M);
        O = fmaf(w_o[w][h][d], f, O);
        L = fmaf(w_l[w][h], f, L);
      }
      a.out[(g * G) * HD + i] = (L > 0.f) ? O / L : 0.f;
    }
    return;
  }
  float *part = a.ws_part + ((int64_t)g * a.n_splits + s) * PART;
  for (int i = threadIdx.x; i < G * HD; i += kAttnThreads) {
    const int h = i / HD, d = i % HD;
    float M = -INFINITY;
    for (int w = 0; w < kAttnWarps; ++w) M = fmaxf(M, w_m[w][h]);
    float O = 0.f, L = 0.f;
    for (int w = 0; w < kAttnWarps; ++w) {
      const float f = (w_m[w][h] == -INFINITY) ? 0.f : expf(w_m[w][h] - M);
      O = fmaf(w_o[w][h][d], f, O);
      L = fmaf(w_l[w][h], f, L);
    }
    part[2 * G + i] = O;
    if (d == 0) { part[h] = M; part[G + h] = L; }
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    s_last = (atomicAdd(a.ws_count + g, 1u) == (unsigned)nsplit - 1);
    s_nsplit = nsplit;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  // last CTA of this KV head: merge the splits
  const float *base = a.ws_part + (int64_t)g * a.n_splits * PART;
  for (int i = threadIdx.x; i < G * HD; i += kAttnThreads) {
    const int h = i / HD;
    float M = -INFINITY;
    for (int sp = 0; sp < s_nsplit; ++sp) M = fmaxf(M, __ldcg(base + (int64_t)sp * PART + h));
    float O = 0.f, L = 0.f;
    if (M != -INFINITY) {
      for (int sp = 0; sp < s_nsplit; ++sp) {
        const float *p = base + (int64_t)sp * PART;
        const float ms = __ldcg(p + h);
        const float f = (ms == -INFINITY) ? 0.f : expf(ms - M);
        O = fmaf(__ldcg(p + 2 * G + i), f, O);
        L = fmaf(__ldcg(p + G + h), f, L);
      }
    }
    a.out[(g * G) * HD + i] = (L > 0.f) ? O / L : 0.f;
  }
  if (threadIdx.x == 0) a.ws_count[g] = 0u;
}

// Empty context: the output is zero (no split has a position).
__global__ void zero_kernel(float *out, int n) {
  pdl_trigger();
  pdl_wait();
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) out[i] = 0.f;
}

size_t attn_workspace_bytes(int Hq, int Hkv, int hd, int n_splits) {
  const int G = Hq / Hkv;
  const size_t counters = 256 + ((size_t)Hkv * 4 + 255) / 256 * 256;
  return counters + (size_t)Hkv * n_splits * G * (2 + hd) * sizeof(float);
}

int attn_splits_for(int Hkv, int max_ctx, int bs) {
  const int nblk = (max_ctx + bs - 1) / bs;
  int s = (2 * sm_count() + Hkv - 1) / Hkv;
  if (s > nblk) s = nblk;
  return s < 1 ? 1 : s;
}

template <int G, int HD>
static mie_status launch_attn_t(const AttnArgs &a, cudaStream_t st, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.n_splits, a.Hkv);
  cfg.blockDim = dim3(kAttnThreads);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  MIE_CUDA(cudaLaunchKernelEx(&cfg, attn_kernel<G, HD>, a));
  return MIE_OK;
}

template <int HD>
static mie_status launch_attn_hd(const AttnArgs &a, cudaStream_t st, bool pdl) {
  switch (a.Hq / a.Hkv) {
    case 1: return launch_attn_t<1, HD>(a, st, pdl);
    case 2: return launch_attn_t<2, HD>(a, st, pdl);
    case 4: return launch_attn_t<4, HD>(a, st, pdl);
    case 8: return launch_attn_t<8, HD>(a, st, pdl);
    default: return fail(MIE_E_SHAPE, "attention: group size %d not in {1,2,4,8}", a.Hq / a.Hkv);
  }
}

mie_status launch_attn(const AttnArgs &a, cudaStream_t st, bool pdl) {
  switch (a.hd) {
    case 32: return launch_attn_hd<32>(a, st, pdl);
    case 64: return launch_attn_hd<64>(a, st, pdl);
    case 128: return launch_attn_hd<128>(a, st, pdl);
    default: return fail(MIE_E_SHAPE, "attention: head_dim %d not in {32,64,128}", a.hd);
  }
}

// --------------------------------------------------------------- argmax (stateless)

constexpr int kArgmaxThreads = 512;

__device__ __forceinline__ bool am_better(float v, int i, float bv, int bi) {
  return v > bv || (v == bv && i < bi);
}

__device__ __forceinline__ void block_best(float &bv, int &bi, float *sv, int *si) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
    if (am_better(ov, oi, bv, bi)) { bv = ov; bi = oi; }
  }
  if (lane == 0) { sv[warp] = bv; si[warp] = bi; }
  __syncthreads();
  if (threadIdx.x == 0)
    for (int w = 1; w < (int)(blockDim.x >> 5); ++w)
      if (am_better(sv[w], si[w], bv, bi)) { bv = sv[w]; bi = si[w]; }
}

// Each CTA reduces a contiguous range; the last CTA to finish reduces the partials.
__global__ void __launch_bounds__(kArgmaxThreads) argmax_kernel(const float *v, int n, int32_t *out,
                                                                float2 *part, unsigned *count) {
  __shared__ float sv[kArgmaxThreads / 32];
  __shared__ int si[kArgmaxThreads / 32];
  __shared__ unsigned s_last;
  pdl_trigger();
  pdl_wait();
  const int i0 = (int)((int64_t)blockIdx.x * n / gridDim.x), i1 = (int)((int64_t)(blockIdx.x + 1) * n / gridDim.x);
  float bv = -INFINITY;
  int bi = 0x7fffffff;
  for (int i = i0 + threadIdx.x; i < i1; i += blockDim.x) {
    const float x = __ldcs(v + i);
    if (am_better(x, i, bv, bi)) { bv = x; bi = i; }
  }
  block_best(bv, bi, sv, si);
  if (threadIdx.x == 0) {
    part[blockIdx.x] = make_float2(bv, __int_as_float(bi));
    __threadfence();
    s_last = (atomicAdd(count, 1u) == gridDim.x - 1);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  bv = -INFINITY;
  bi = 0x7fffffff;
  for (int b = threadIdx.x; b < (int)gridDim.x; b += blockDim.x) {
    const float2 p = __ldcg(part + b);
    if (am_better(p.x, __float_as_int(p.y), bv, bi)) { bv = p.x; bi = __float_as_int(p.y); }
  }
  __syncthreads();
  block_best(bv, bi, sv, si);
  if (threadIdx.x == 0) {
    *out = (bi == 0x7fffffff) ? 0 : bi;
    *count = 0u;
  }
}

int argmax_grid(int n) {
  int g = (n + 4095) / 4096;
  const int cap = sm_count();
  return g < 1 ? 1 : (g > cap ? cap : g);
}

mie_status launch_argmax(const float *v, int n, int32_t *out, float2 *part, unsigned *count, int grid,
                         cudaStream_t st) {
  argmax_kernel<<<grid, kArgmaxThreads, 0, st>>>(v, n, out, part, count);
  MIE_CUDA(cudaGetLastError());
  return MIE_OK;
}

int *device_error_flag() {
  static int *cached[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  if (!cached[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return nullptr;
    cached[dev] = static_cast<int *>(p);
  }
  return cached[dev];
}

}  // namespace mie

// --------------------------------------------------------------- C ABI

using namespace mie;

extern "C" size_t mie_paged_attn_workspace_bytes(int n_q_heads, int n_kv_heads, int head_dim, int ctx_len,
                                                 int block_size) {
  if (n_kv_heads < 1 || n_q_heads < n_kv_heads || head_dim < 1 || block_size < 1 || ctx_len < 0) return 0;
  const int splits = attn_splits_for(n_kv_heads, ctx_len < 1 ? 1 : ctx_len, block_size);
  return attn_workspace_bytes(n_q_heads, n_kv_heads, head_dim, splits);
}

extern "C" mie_status mie_paged_attn_decode(const float *q, const uint16_t *k_pool, const uint16_t *v_pool,
                                            int64_t block_stride, int n_pool_blocks, const int32_t *block_table,
                                            int n_table, int ctx_len, int n_q_heads, int n_kv_heads, int head_dim,
                                            int block_size, float scale, float *out, void *workspace,
                                            size_t workspace_bytes, void *stream) {
  if (!q || !k_pool || !v_pool || !block_table || !out || !workspace)
    return fail(MIE_E_ARG, "mie_paged_attn_decode: null pointer");
  if (n_kv_heads < 1 || n_q_heads < 1 || n_q_heads % n_kv_heads != 0)
    return fail(MIE_E_SHAPE, "mie_paged_attn_decode: %d query heads over %d KV heads", n_q_heads, n_kv_heads);
  const int G = n_q_heads / n_kv_heads;
  if (G != 1 && G != 2 && G != 4 && G != 8)
    return fail(MIE_E_SHAPE, "mie_paged_attn_decode: group size %d not in {1,2,4,8}", G);
  if (head_dim != 32 && head_dim != 64 && head_dim != 128)
    return fail(MIE_E_SHAPE, "mie_paged_attn_decode: head_dim %d not in {32,64,128}", head_dim);
  if (block_size != 8 && block_size != 16 && block_size != 32)
    return fail(MIE_E_SHAPE, "mie_paged_attn_decode: block_size %d not in {8,16,32}", block_size);
  if (ctx_len < 0 || n_table < 0 || (int64_t)ctx_len > (int64_t)n_table * block_size)
    return fail(MIE_E_SHAPE, "mie_paged_attn_decode: ctx_len %d does not fit %d blocks", ctx_len, n_table);
  if (n_pool_blocks < 1 || block_stride < (int64_t)n_kv_heads * block_size * head_dim)
    return fail(MIE_E_SHAPE, "mie_paged_attn_decode: bad pool geometry");
  if (((uintptr_t)k_pool & 15) || ((uintptr_t)v_pool & 15) || (block_stride % 8) || ((uintptr_t)workspace & 255))
    return fail(MIE_E_SHAPE, "mie_paged_attn_decode: misaligned pool, stride or workspace");
  cudaStream_t st = (cudaStream_t)stream;
  if (ctx_len == 0) {
    zero_kernel<<<1, 256, 0, st>>>(out, n_q_heads * head_dim);
    MIE_CUDA(cudaGetLastError());
    return MIE_OK;
  }
  AttnArgs a;
  a.n_splits = attn_splits_for(n_kv_heads, ctx_len, block_size);
  const size_t need = attn_workspace_bytes(n_q_heads, n_kv_heads, head_dim, a.n_splits);
  if (workspace_bytes < need)
    return fail(MIE_E_ARG, "mie_paged_attn_decode: workspace %zu bytes < %zu", workspace_bytes, need);
  const size_t counters = 256 + ((size_t)n_kv_heads * 4 + 255) / 256 * 256;
  a.ws_count = reinterpret_cast<unsigned *>(workspace);
  a.ws_part = reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(workspace) + counters);
  MIE_CUDA(cudaMemsetAsync(workspace, 0, (size_t)n_kv_heads * 4, st));
  a.q = q;
  a.k = k_pool;
  a.v = v_pool;
  a.block_stride = block_stride;
  a.n_pool_blocks = n_pool_blocks;
  a.block_table = block_table;
  a.n_table = n_table;
  a.ctx = ctx_len;
  a.Hq = n_q_heads;
  a.Hkv = n_kv_heads;
  a.hd = head_dim;
  a.bs = block_size;
  a.scale = scale;
  a.out = out;
  a.err = device_error_flag();
  return launch_attn(a, st, false);
}

extern "C" size_t mie_argmax_workspace_bytes(int n) {
  if (n < 1) return 0;
  return 256 + (size_t)argmax_grid(n) * sizeof(float2);
}

extern "C" mie_status mie_argmax(const float *v, int n, int32_t *out, void *workspace, size_t workspace_bytes,
                                 void *stream) {
  if (!v || !out || !workspace) return fail(MIE_E_ARG, "mie_argmax: null pointer");
  if (n < 1) return fail(MIE_E_SHAPE, "mie_argmax: n = %d", n);
  if (((uintptr_t)workspace & 255)) return fail(MIE_E_SHAPE, "mie_argmax: workspace not 256-byte aligned");
  if (workspace_bytes < mie_argmax_workspace_bytes(n))
    return fail(MIE_E_ARG, "mie_argmax: workspace too small");
  cudaStream_t st = (cudaStream_t)stream;
  MIE_CUDA(cudaMemsetAsync(workspace, 0, 4, st));
  const int grid = argmax_grid(n);
  return launch_argmax(v, n, out, reinterpret_cast<float2 *>(reinterpret_cast<uint8_t *>(workspace) + 256),
                       reinterpret_cast<unsigned *>(workspace), grid, st);
}

extern "C" mie_status mie_check(void *stream) {
  MIE_CUDA(cudaStreamSynchronize((cudaStream_t)stream));
  int *flag = device_error_flag();
  if (!flag) return fail(MIE_E_CUDA, "mie_check: no device error flag");
  int v = 0;
  MIE_CUDA(cudaMemcpy(&v, flag, sizeof(int), cudaMemcpyDeviceToHost));
  if (v) {
    const int zero = 0;
    MIE_CUDA(cudaMemcpy(flag, &zero, sizeof(int), cudaMemcpyHostToDevice));
    return fail(MIE_E_DEVICE, "device bounds check fired (code %d)", v);
  }
  return MIE_OK;
}
