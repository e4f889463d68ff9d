// attn.cu -- paged GQA decode attention and argmax on sm_103a.
//
// Attention ("Mini Inference Engine", "The KV cache, paged like virtual memory": the
// kernel reads K/V through a block table; "infer" page, design notes, the split-KV attention item:
// one CTA per KV head serves the query heads of its group, the context is split and
// the partial softmaxes are merged; "Writing an LLM inference engine from scratch in
// Rust", Lesson 4: an online softmax with a running maximum and sum).
//
// Grid (splits, KV heads[, slots]), 256 threads; splits of 256 tokens; each split's
// K/V blocks come into shared memory by bulk copies and are reduced by the chunk
// passes of attn_core.cuh.
#include <mutex>

#include "attn_core.cuh"
#include "attn_mma.cuh"

namespace mie {

__device__ int g_device_error;  // latched by the stateless kernels of this device

// The kernel: 8 warps per (split, KV head[, slot]); the split's K/V blocks are
// brought into shared memory by bulk copies (one per block for K and one for V) and
// reduced by the three CTA-wide passes of chunk_passes.  Splits of 256 tokens, merged by
// the last split.  A split is one chunk: the passes cost ~1 us whatever the chunk's
// length, and the second CTA on the SM overlaps one CTA's copies with the other's math
// (two 128-token chunks in flight per CTA measured slower).
constexpr int kCThreads = 256;
constexpr int kCTok = 256;       // tokens per chunk
constexpr int kCSplitTok = 256;  // tokens per split
constexpr int kCBufs = kCSplitTok / kCTok >= 2 ? 2 : 1;  // chunks in flight per CTA
constexpr int kCSlotGrid = 16;   // few-slot step: CTAs per (KV head, slot)

struct CSync {
  __device__ static void sync() { __syncthreads(); }
  __device__ static bool all(bool v) { return __syncthreads_and(v) != 0; }
};

template <int G, int HD>
__global__ void __launch_bounds__(kCThreads, 2) attn_chunk_kernel(const AttnArgs a_in) {
  constexpr int NO = (G * HD + kCThreads - 1) / kCThreads;
  extern __shared__ __align__(128) uint8_t cbuf[];  // 2 x [K: kCTok*HD*2 bytes][V: same]
  __shared__ ChunkSmem<G, HD> sm;
  __shared__ __align__(8) uint64_t bar[2];
  __shared__ int ids[kCSplitTok / 8];
  pdl_trigger();
  AttnArgs a = a_in;
  if (a_in.slot_z) {  // one grid layer per slot of the few-slot step
    const int z = blockIdx.z;
    if (z >= a_in.sp->n_slots) return;
    a.slot = z;
    a.q += (int64_t)z * a.Hq * a.hd;
    a.out += (int64_t)z * a.Hq * a.hd;
    a.ws_count = reinterpret_cast<unsigned *>(reinterpret_cast<uint8_t *>(a.ws_count) + z * a.ws_slot_bytes);
    a.ws_part = reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(a.ws_part) + z * a.ws_slot_bytes);
  }
  pdl_wait();
  const int tid = threadIdx.x, g = blockIdx.y;
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
    if (tid == 0 && blockIdx.x == 0 && g == 0) latch_error(a.err, ERR_POS);
    ctx = n_table * a.bs;
  }
  if (ctx < 0) ctx = 0;
  const int nblk = (ctx + a.bs - 1) / a.bs;
  const int nsplit = attn_nsplit(nblk, a.n_splits, kCSplitTok / a.bs);
  if ((int)blockIdx.x >= nsplit) return;
  const int kb = a.bs * HD * 2;           // bytes of one block of one head
  const int cb = kCTok / a.bs;            // blocks per chunk
  const uint32_t buf_bytes = 2u * kCTok * HD * 2;
  const int64_t head_off = (int64_t)g * a.bs * HD;  // elements

  for (int i = tid; i < G * HD; i += kCThreads) sm.q[i] = __ldcg(a.q + (int64_t)(g * G) * HD + i);
  if (tid == 0) {
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  // splits blockIdx.x, + gridDim.x, ... (the few-slot grid has fewer CTAs than splits a
  // long context needs); chunk c of this CTA uses buffer c % kCBufs, phase c / kCBufs
  int done = 0, issued = 0;
  for (int sp = blockIdx.x; sp < nsplit; sp += gridDim.x) {
    const int b0 = (int)((int64_t)sp * nblk / nsplit), b1 = (int)((int64_t)(sp + 1) * nblk / nsplit);
    const int t_end = min(b1 * a.bs, ctx);
    const int nch = (b1 - b0 + cb - 1) / cb;
    if (tid < b1 - b0) {
      int blk = bt[b0 + tid];
      if (blk < 0 || blk >= a.n_pool_blocks) {
        latch_error(a.err, ERR_BLOCK_ID);
        blk = 0;  // a valid block: the result is wrong but the error is reported
      }
      ids[tid] = blk;
    }
    if (tid < G) {
      sm.m[tid] = -INFINITY;
      sm.l[tid] = 0.f;
    }
    __syncthreads();  // block ids, statistics; the previous split is done with everything
    auto issue = [&](int ci) {  // thread 0: the bulk copies of chunk ci of this split
      const int first = ci * cb, nb = min(cb, b1 - b0 - first), c = done + ci, bi = c % kCBufs;
      uint8_t *kd = cbuf + (size_t)bi * buf_bytes, *vd = kd + (size_t)kCTok * HD * 2;
      fence_proxy_async_smem();  // earlier generic reads of the buffer before the async writes
      mbar_expect_tx(&bar[bi], 2u * nb * kb);
      for (int j = 0; j < nb; ++j) {
        const int64_t off = (int64_t)ids[first + j] * a.block_stride + head_off;
        bulk_load(kd + (size_t)j * kb, a.k + off, kb, &bar[bi], 0ull);
        bulk_load(vd + (size_t)j * kb, a.v + off, kb, &bar[bi], 0ull);
      }
      issued = c + 1;
    };
    if (tid == 0)
      for (int ci = 0; ci < kCBufs && ci < nch; ++ci) issue(ci);
    float o[NO];
#pragma unroll
    for (int j = 0; j < NO; ++j) o[j] = 0.f;
    bool ok = true;
    int ci = 0;
    for (; ci < nch; ++ci) {
      const int c = done + ci;
      ok = CSync::all(ok && mbar_wait(&bar[c % kCBufs], (c / kCBufs) & 1));
      if (!ok) break;
      const uint32_t kbase = smem_u32(cbuf) + (uint32_t)(c % kCBufs) * buf_bytes,
                     vbase = kbase + (uint32_t)kCTok * HD * 2;
      const int t0 = (b0 + ci * cb) * a.bs;
      const int ntok = min((b0 + min((ci + 1) * cb, b1 - b0)) * a.bs, t_end) - t0;
      chunk_passes<G, HD, kCThreads, CSync>(kbase, vbase, ntok, a.scale, sm, o);
      __syncthreads();  // every thread is done with the buffer
      if (tid == 0 && ci + kCBufs < nch) issue(ci + kCBufs);
    }
    if (!ok) {  // a copy never completed: report, and leave no copy writing into shared memory
      if (tid == 0) {
        latch_error(a.err, ERR_TIMEOUT);
        for (int c = done + ci; c < issued; ++c) mbar_wait(&bar[c % kCBufs], (c / kCBufs) & 1);
      }
      return;
    }
    done += nch;
    if (nsplit == 1) {
#pragma unroll
      for (int j = 0; j < NO; ++j) {
        const int i = tid + j * kCThreads;
        if (i < G * HD) {
          const float L = sm.l[i / HD];
          a.out[(int64_t)(g * G) * HD + i] = (L > 0.f) ? o[j] / L : 0.f;
        }
      }
      return;
    }
    float *part = a.ws_part + ((int64_t)g * a.n_splits + sp) * (G * (2 + HD));
#pragma unroll
    for (int j = 0; j < NO; ++j) {
      const int i = tid + j * kCThreads;
      if (i < G * HD) {
        const int h = i / HD;
        part[2 * G + i] = o[j];
        if (i % HD == 0) {
          part[h] = sm.m[h];
          part[G + h] = sm.l[h];
        }
      }
    }
    attn_merge_splits<G, HD, kCThreads, CSync, false, 16>(a, g, nsplit, sm.last, 0u);
  }
}

// Tensor-core variant (head_dim 64 or 128, block stride a multiple of head_dim): the
// split's K and V arrive by 2-D tensor copies (one per block and 64-dimension half) as
// 128-byte swizzled tiles, and each warp reduces 32 of its tokens on the tensor cores
// with its own online softmax (attn_mma.cuh); the CTA then combines its 8 warps and the
// splits merge as above.  Measured on GB300 for one 256-token split of a KV head with
// four query heads: the three CUDA-core passes of chunk_passes took 3.1-4.6 us.
constexpr uint32_t kMmaHalf = (uint32_t)kCTok * 128u;  // bytes of one 64-dim half of a K or V buffer

template <int G, int HD>
constexpr size_t attn_mma_smem() {
  return 1024 + 2 * (HD / 64) * (size_t)kMmaHalf + (size_t)(kCThreads / 32) * G * HD * 4;
}

template <int G, int HD>
__global__ void __launch_bounds__(kCThreads, HD == 64 ? 2 : 1)
    attn_mma_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                    const AttnArgs a_in) {
  constexpr int MT = (G + 3) / 4, NH = HD / 64, NW = kCThreads / 32;
  extern __shared__ uint8_t dbuf[];
  __shared__ __align__(8) uint64_t bar;
  __shared__ int ids[kCSplitTok / 8];
  __shared__ float wm[NW * G], wl[NW * G];
  __shared__ float qs[G * HD];
  __shared__ uint4 qf[MT * (HD / 16) * 32];  // query A fragments per (tile, k-step, lane)
  __shared__ unsigned last;
  pdl_trigger();
  // the few-slot step runs one grid layer per slot: slot z's queries, outputs and
  // workspace follow those of slot z - 1 (every pointer formed from the launch's own
  // arguments; measured on GB300, the queries read through a shifted copy of the
  // argument struct came from slot 0)
  const int z = a_in.slot_z ? (int)blockIdx.z : a_in.slot;
  if (a_in.slot_z && z >= a_in.sp->n_slots) return;
  const int64_t zq = a_in.slot_z ? (int64_t)z * a_in.Hq * HD : 0;
  const size_t zw = a_in.slot_z ? (size_t)z * a_in.ws_slot_bytes : 0;
  AttnArgs a = a_in;
  a.slot = z;
  a.q = a_in.q + zq;
  a.out = a_in.out + zq;
  a.ws_count = reinterpret_cast<unsigned *>(reinterpret_cast<uint8_t *>(a_in.ws_count) + zw);
  a.ws_part = reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(a_in.ws_part) + zw);
  pdl_wait();
  const int tid = threadIdx.x, warp = tid >> 5, g = blockIdx.y;
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
    if (tid == 0 && blockIdx.x == 0 && g == 0) latch_error(a.err, ERR_POS);
    ctx = n_table * a.bs;
  }
  if (ctx < 0) ctx = 0;
  const int nblk = (ctx + a.bs - 1) / a.bs;
  const int nsplit = attn_nsplit(nblk, a.n_splits, kCSplitTok / a.bs);
  if ((int)blockIdx.x >= nsplit) return;
  // the queries come from the previous kernel: read at L2 (a line this SM's L1 kept from
  // an earlier kernel could be stale under programmatic dependent launch)
  for (int i = tid; i < G * HD; i += kCThreads) qs[i] = __ldcg(a_in.q + zq + (int64_t)(g * G) * HD + i);
  const uint32_t kbuf = (smem_u32(dbuf) + 1023u) & ~1023u, vbuf = kbuf + NH * kMmaHalf;
  float *wo = reinterpret_cast<float *>(dbuf + (vbuf + NH * kMmaHalf - smem_u32(dbuf)));  // [NW][G][HD]
  const int64_t rows_per_blk = a.block_stride / HD;
  if (tid == 0) {
    mbar_init(&bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  int it = 0;
  for (int sp = blockIdx.x; sp < nsplit; sp += gridDim.x, ++it) {
    const int b0 = (int)((int64_t)sp * nblk / nsplit), b1 = (int)((int64_t)(sp + 1) * nblk / nsplit);
    const int nb = b1 - b0, ntok = min(b1 * a.bs, ctx) - b0 * a.bs;
    if (nb > kCSplitTok / a.bs) {  // a context longer than the workspace's splits were sized for
      if (tid == 0) latch_error(a.err, ERR_POS);
      return;
    }
    fence_proxy_async_smem();  // this thread's generic accesses of the previous split before the copies
    if (tid < nb) {
      int blk = bt[b0 + tid];
      if (blk < 0 || blk >= a.n_pool_blocks) {
        latch_error(a.err, ERR_BLOCK_ID);
        blk = 0;  // a valid block: the result is wrong but the error is reported
      }
      ids[tid] = blk;
    }
    __syncthreads();  // block ids; every warp is done with the buffers
    if (tid == 0) {
      mbar_expect_tx(&bar, (uint32_t)nb * a.bs * HD * 2 * 2);
      for (int j = 0; j < nb; ++j) {
        const int y = (int)((int64_t)ids[j] * rows_per_blk + (int64_t)g * a.bs);
#pragma unroll
        for (int hh = 0; hh < NH; ++hh) {
          const uint32_t off = hh * kMmaHalf + (uint32_t)(j * a.bs) * 128u;
          tma_load_tile(kbuf + off, &tmk, hh * 64, y, smem_u32(&bar));
          tma_load_tile(vbuf + off, &tmv, hh * 64, y, smem_u32(&bar));
        }
      }
    }
    // the query fragments, once, while the first split's copies fly (the queries were
    // stored before the barrier above; the fragments are read after the one below)
    if (it == 0) q_fragments_shared<G, HD, NW>(qs, a.scale * kLog2e, qf);
    if (!CSync::all(mbar_wait(&bar, it & 1))) {  // a copy never completed
      if (tid == 0) {
        latch_error(a.err, ERR_TIMEOUT);
        mbar_wait(&bar, it & 1);  // leave no copy writing into shared memory
      }
      return;
    }
    // V rows from ntok to the next multiple of 16 meet zero probabilities: make them finite
    const int rz = min((ntok + 15) & ~15, kCTok);
    for (int i = tid; i < (rz - ntok) * (HD / 8); i += kCThreads)
      sts128_zero(swz_addr(vbuf, kCTok, ntok + i / (HD / 8), i % (HD / 8)));
    __syncthreads();
#pragma unroll 1
    for (int mt = 0; mt < MT; ++mt) {
      uint32_t qa[HD / 16][4];
#pragma unroll
      for (int k = 0; k < HD / 16; ++k) {
        const uint4 f = qf[(mt * (HD / 16) + k) * 32 + (tid & 31)];
        qa[k][0] = f.x;
        qa[k][1] = f.y;
        qa[k][2] = f.z;
        qa[k][3] = f.w;
      }
      WarpAttn<HD> st;
      st.reset();
      warp_chunk_mma<HD>(kbuf, vbuf, kCTok, kMmaTokPerWarp * warp, ntok, qa, st);
      warp_attn_store<G, HD>(st, mt, wm, wl, wo);
    }
    __syncthreads();
    float *part = a.ws_part + ((int64_t)g * a.n_splits + sp) * (G * (2 + HD));
    for (int i = tid; i < G * HD; i += kCThreads) {
      float M, L, O;
      cta_attn_combine<G, HD, NW>(i, wm, wl, wo, M, L, O);
      if (nsplit == 1) {
        a.out[(int64_t)(g * G) * HD + i] = (L > 0.f) ? O / L : 0.f;
      } else {
        const int h = i / HD;
        part[2 * G + i] = O;
        if (i % HD == 0) {
          part[h] = (M == -INFINITY) ? -INFINITY : M * kLn2;  // the merge works in natural-log units
          part[G + h] = L;
        }
      }
    }
    if (nsplit == 1) return;
    attn_merge_splits<G, HD, kCThreads, CSync, false, 16>(a, g, nsplit, last, 0u);
  }
}

// Empty context: the output is zero (no split has a position).
__global__ void zero_kernel(float *out, int n) {
  pdl_trigger();
  pdl_wait();
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) out[i] = 0.f;
}

size_t attn_counter_bytes(int Hkv) { return 256 + ((size_t)Hkv * 4 + 255) / 256 * 256; }

size_t attn_workspace_bytes(int Hq, int Hkv, int hd, int n_splits) {
  const int G = Hq / Hkv;
  return attn_counter_bytes(Hkv) + (size_t)Hkv * n_splits * G * (2 + hd) * sizeof(float);
}

// Splits a workspace is sized for: two CTAs per SM over the KV heads, and at least
// enough that no split of the chunked kernel exceeds kCSplitTok tokens (the block ids
// of a split are cached in shared memory).
int attn_splits_for(int Hkv, int max_ctx, int bs) {
  const int nblk = (max_ctx + bs - 1) / bs;
  int s = (2 * sm_count() + Hkv - 1) / Hkv;
  if (s > nblk) s = nblk;
  const int per = kCSplitTok / bs;
  const int need = (nblk + per - 1) / per;
  if (s < need) s = need;
  return s < 1 ? 1 : s;
}

template <int G, int HD>
static mie_status launch_attn_t(const AttnArgs &a, cudaStream_t st, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  // few-slot step: the grid is captured once for any context, so it holds at most
  // kCSlotGrid CTAs per (KV head, slot) and each loops over its splits; CTAs past a slot's
  // splits only read its position and leave (a grid of n_splits left ~3/4 of them idle)
  cfg.gridDim = dim3(a.slot_z ? min(a.n_splits, kCSlotGrid) : a.n_splits, a.Hkv, a.slot_z ? a.max_slots : 1);
  cfg.blockDim = dim3(kCThreads);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  if constexpr (HD == 64 || HD == 128) {
    if (a.block_stride % HD == 0) {  // K/V rows addressable as a 2-D tensor of head_dim columns
      const int64_t rows = ((int64_t)(a.n_pool_blocks - 1) * a.block_stride + (int64_t)a.Hkv * a.bs * HD) / HD;
      CUtensorMap mk, mv;
      mie_status s = make_bf16_map(&mk, a.k, rows, HD, HD * 2, a.bs);
      if (s == MIE_OK) s = make_bf16_map(&mv, a.v, rows, HD, HD * 2, a.bs);
      if (s != MIE_OK) return s;
      auto kern = attn_mma_kernel<G, HD>;
      constexpr size_t smem = attn_mma_smem<G, HD>();
      MIE_CUDA(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
      cfg.dynamicSmemBytes = smem;
      MIE_CUDA(cudaLaunchKernelEx(&cfg, kern, mk, mv, a));
      return MIE_OK;
    }
  }
  const size_t smem = (size_t)kCBufs * 2u * kCTok * HD * 2;
  auto kern = attn_chunk_kernel<G, HD>;
  MIE_CUDA(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
  cfg.dynamicSmemBytes = smem;
  MIE_CUDA(cudaLaunchKernelEx(&cfg, kern, a));
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

// Device address of the error flag on the current device, looked up once per device;
// the lookup table is shared by every host thread, so it is filled under a lock.
int *device_error_flag() {
  static std::mutex mu;
  static int *cached[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> g(mu);
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

// --------------------------------------------------------------- C ABI: allocation-free attention
//
// Some callers cannot allocate device memory at the moment they need attention: code
// running where cudaMalloc is not allowed or not wanted (inside a real-time loop that
// must never hit the allocator, or while a custom allocator owns all device memory).
// mie_paged_attn_decode_noalloc serves them: it needs no caller workspace and allocates
// nothing, because its partial results live in one fixed array that is part of the
// library's device image.  Every GPU that loads the library holds that array until the
// process exits.

namespace {

constexpr size_t kNoAllocScratchBytes = 1u << 20;  // 1 MiB: the largest workspace served
__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_noalloc_mu;
unsigned char *g_noalloc_ptr[64] = {nullptr};

// Device address of the scratch array on the current device, looked up once per device.
mie_status noalloc_scratch(unsigned char **out) {
  int dev = 0;
  MIE_CUDA(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64) return fail(MIE_E_ARG, "mie_paged_attn_decode_noalloc: device %d", dev);
  std::lock_guard<std::mutex> g(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "mie_paged_attn_decode_noalloc: cudaGetSymbolAddress");
    g_noalloc_ptr[dev] = static_cast<unsigned char *>(p);
  }
  *out = g_noalloc_ptr[dev];
  return MIE_OK;
}

}  // namespace

extern "C" mie_status mie_paged_attn_decode_noalloc(const float *q, const uint16_t *k_pool, const uint16_t *v_pool,
                                                    int64_t block_stride, int n_pool_blocks, const int32_t *block_table,
                                                    int n_table, int ctx_len, int n_q_heads, int n_kv_heads,
                                                    int head_dim, int block_size, float scale, float *out,
                                                    void *stream) {
  if (!q || !k_pool || !v_pool || !block_table || !out)
    return fail(MIE_E_ARG, "mie_paged_attn_decode_noalloc: null pointer");
  if (n_kv_heads < 1 || n_q_heads < n_kv_heads || head_dim < 1 || block_size < 1 || ctx_len < 0)
    return fail(MIE_E_SHAPE, "mie_paged_attn_decode_noalloc: bad sizes");
  const size_t need = mie_paged_attn_workspace_bytes(n_q_heads, n_kv_heads, head_dim, ctx_len, block_size);
  if (need > kNoAllocScratchBytes)
    return fail(MIE_E_SHAPE,
                "mie_paged_attn_decode_noalloc: these sizes need %zu bytes of scratch, more than the %zu-byte "
                "built-in array; use mie_paged_attn_decode with a workspace",
                need, kNoAllocScratchBytes);
  unsigned char *scratch = nullptr;
  const mie_status s = noalloc_scratch(&scratch);
  if (s != MIE_OK) return s;
  // the same checks, counter clearing and launch as the workspace entry point
  return mie_paged_attn_decode(q, k_pool, v_pool, block_stride, n_pool_blocks, block_table, n_table, ctx_len,
                               n_q_heads, n_kv_heads, head_dim, block_size, scale, out, scratch,
                               kNoAllocScratchBytes, stream);
}
