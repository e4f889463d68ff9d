// attn_core.cuh -- one (KV head, context split) of paged GQA decode attention, shared
// by the standalone attention kernel and the persistent step kernel.
//
// "Mini Inference Engine", "The KV cache, paged like virtual memory": K/V are read
// through a block table; "infer" page, "GQA-aware split-KV attention": the query heads
// of one KV head share every K/V load, the context is split and partial softmaxes are
// merged; "Writing an LLM inference engine from scratch in Rust", Lesson 4: an online
// softmax with a running maximum and sum.
//
// NW warps take groups of 32/LPT tokens (LPT = head_dim/32 lanes per token) and issue
// all loads of a group before any math: 64 bytes of one key per lane, then the lane's
// head_dim/32 value dims of every token of the group.  K/V are loaded with ld.global.cg
// so that values written earlier in the same launch (by another SM) are read from L2.
#pragma once

#include "device.cuh"

namespace mie {

constexpr int kAttnMaxBlocks = 256;  // block ids staged in shared memory at a time

// Splits in use for a context of nblk blocks: every split gets at least per_split
// blocks (so its warps have work), at most max_splits splits.
__host__ __device__ inline int attn_nsplit(int nblk, int max_splits, int per_split) {
  int s = (nblk + per_split - 1) / per_split;
  if (s > max_splits) s = max_splits;
  return s < 1 ? 1 : s;
}

// Blocks per split: two token groups per warp, so each warp overlaps the loads of its
// second group with the math of its first.
template <int HD, int NW>
__host__ __device__ inline int attn_blocks_per_split(int bs) {
  const int tokens = 2 * NW * (32 / (HD / 32));
  const int b = tokens / bs;
  return b < 1 ? 1 : b;
}

// Shared-memory scratch of one attention CTA.
template <int G, int HD, int NW>
struct AttnSmem {
  float q[G * HD];
  float kn[HD], vn[HD];  // tagged variant: the current token's k and v
  int blk[kAttnMaxBlocks];
  float m[NW][G], l[NW][G];
  float o[NW][G][HD];
  unsigned last;
};

// The loads of one group of tokens for one lane: 64 bytes of its key, and its value
// dims of every token of the group.  Masked tokens read a valid address and are
// zeroed later, so the loads carry no branches and issue back to back.
template <int HD>
struct KvGroup {
  static constexpr int LPT = HD / 32, TPI = 32 / LPT, DPL = HD / 32, VW = DPL == 4 ? 2 : 1;
  uint4 kv[4];
  uint32_t vraw[TPI][VW];
  unsigned vmask;  // bit i: token i of the group is valid
  int kblk;        // >= 0: this lane's key token is valid

  // From the paged pool in global memory, through the block ids ids[.. - id0].
  __device__ __forceinline__ void load(const AttnArgs &a, const int *ids, int id0, int tb, int t1, int64_t head_off,
                                       int lane) {
    const int tok_in = lane / LPT, part_in = lane % LPT;
    const int t = tb + tok_in;
    kblk = (t < t1) ? ids[t / a.bs - id0] : -1;
    const uint16_t *kp =
        (kblk >= 0) ? a.k + (int64_t)kblk * a.block_stride + head_off + (int64_t)(t % a.bs) * HD + part_in * 32 : a.k;
#pragma unroll
    for (int i = 0; i < 4; ++i) kv[i] = __ldcg(reinterpret_cast<const uint4 *>(kp + 8 * i));
    vmask = 0u;
#pragma unroll
    for (int i = 0; i < TPI; ++i) {
      const int t2 = tb + i;
      const int vblk = (t2 < t1) ? ids[t2 / a.bs - id0] : -1;
      if (vblk >= 0) vmask |= 1u << i;
      const uint16_t *vp =
          vblk >= 0 ? a.v + (int64_t)vblk * a.block_stride + head_off + (int64_t)(t2 % a.bs) * HD + lane * DPL : a.v;
      if constexpr (DPL == 1) {
        vraw[i][0] = __ldcg(reinterpret_cast<const unsigned short *>(vp));
      } else if constexpr (DPL == 2) {
        vraw[i][0] = __ldcg(reinterpret_cast<const unsigned int *>(vp));
      } else {
        const uint2 w = __ldcg(reinterpret_cast<const uint2 *>(vp));
        vraw[i][0] = w.x;
        vraw[i][1] = w.y;
      }
    }
  }
};

// bf16 bits of two values that are already bf16-exact, packed as the cache holds them.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  return (__float_as_uint(lo) >> 16) | (__float_as_uint(hi) & 0xffff0000u);
}

// Puts the current token's k and v (bf16-exact floats kn[HD], vn[HD]) in place of
// what the group loaded for it; pi = its index in the group (warp-uniform).
template <int HD>
__device__ __forceinline__ void patch_current(KvGroup<HD> &cur, int pi, const float *kn, const float *vn, int lane) {
  using KG = KvGroup<HD>;
  constexpr int LPT = KG::LPT, TPI = KG::TPI, DPL = KG::DPL, VW = KG::VW;
  if (pi < 0 || pi >= TPI) return;
  if (lane / LPT == pi) {
    const float *k = kn + (lane % LPT) * 32;
#pragma unroll
    for (int i = 0; i < 4; ++i)
      cur.kv[i] = make_uint4(pack_bf16x2(k[8 * i], k[8 * i + 1]), pack_bf16x2(k[8 * i + 2], k[8 * i + 3]),
                             pack_bf16x2(k[8 * i + 4], k[8 * i + 5]), pack_bf16x2(k[8 * i + 6], k[8 * i + 7]));
  }
#pragma unroll
  for (int i = 0; i < TPI; ++i) {
    if (i != pi) continue;
    if constexpr (DPL == 1) {
      cur.vraw[i][0] = __float_as_uint(vn[lane]) >> 16;
    } else {
#pragma unroll
      for (int w = 0; w < VW; ++w) cur.vraw[i][w] = pack_bf16x2(vn[lane * DPL + 2 * w], vn[lane * DPL + 2 * w + 1]);
    }
  }
}

// The group's values as fp32 (zero for masked tokens).
template <int HD>
__device__ __forceinline__ void group_values(const KvGroup<HD> &cur, float (&vf)[KvGroup<HD>::TPI][KvGroup<HD>::DPL]) {
  using KG = KvGroup<HD>;
  constexpr int TPI = KG::TPI, DPL = KG::DPL, VW = KG::VW;
#pragma unroll
  for (int i = 0; i < TPI; ++i) {
    const bool ok = (cur.vmask >> i) & 1u;
    if constexpr (DPL == 1) {
      vf[i][0] = ok ? __uint_as_float(cur.vraw[i][0] << 16) : 0.f;
    } else {
#pragma unroll
      for (int w = 0; w < VW; ++w) {
        vf[i][2 * w] = ok ? __uint_as_float(cur.vraw[i][w] << 16) : 0.f;
        vf[i][2 * w + 1] = ok ? __uint_as_float(cur.vraw[i][w] & 0xffff0000u) : 0.f;
      }
    }
  }
}

// Partial dot products of this lane's 32 key dims with the G queries at shared
// address q (fp32, 16-byte aligned), read as float4 into four accumulators.
template <int G, int HD>
__device__ __forceinline__ void group_scores(const KvGroup<HD> &cur, uint32_t q, int part_in, float (&sc)[G]) {
  float kf[32];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t w[4] = {cur.kv[i].x, cur.kv[i].y, cur.kv[i].z, cur.kv[i].w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      kf[8 * i + 2 * j] = __uint_as_float(w[j] << 16);
      kf[8 * i + 2 * j + 1] = __uint_as_float(w[j] & 0xffff0000u);
    }
  }
#pragma unroll
  for (int h = 0; h < G; ++h) {
    const uint32_t qh = q + (uint32_t)(h * HD + part_in * 32) * 4;
    float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float4 qq = lds128f(qh + 16 * i);
      d[0] = fmaf(qq.x, kf[4 * i], d[0]);
      d[1] = fmaf(qq.y, kf[4 * i + 1], d[1]);
      d[2] = fmaf(qq.z, kf[4 * i + 2], d[2]);
      d[3] = fmaf(qq.w, kf[4 * i + 3], d[3]);
    }
    sc[h] = (d[0] + d[1]) + (d[2] + d[3]);
  }
}

// Online-softmax update of (m, l, o) with one group: scores summed over the lanes of a
// token, masked, scaled; then the values weighted by the new probabilities.
template <int G, int HD>
__device__ __forceinline__ void group_update(float (&sc)[G], const float (&vf)[KvGroup<HD>::TPI][KvGroup<HD>::DPL],
                                             int kblk, float scale, int part_in, float (&m)[G], float (&l)[G],
                                             float (&o)[G][KvGroup<HD>::DPL]) {
  using KG = KvGroup<HD>;
  constexpr int LPT = KG::LPT, TPI = KG::TPI, DPL = KG::DPL;
#pragma unroll
  for (int h = 0; h < G; ++h) {
#pragma unroll
    for (int off = 1; off < LPT; off <<= 1) sc[h] += __shfl_xor_sync(0xffffffffu, sc[h], off);
    sc[h] = (kblk >= 0) ? sc[h] * scale : -INFINITY;
  }
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

// Tagged variant: polls the group's queries into sm.q and, when has_pos, the current
// token's k and v of KV head g into sm.kn / sm.vn, all in one batch of round trips.
template <int G, int HD, int NT, class Sync, class SM>
__device__ bool tagged_inputs(const AttnArgs &a, int g, bool has_pos, SM &sm, uint32_t tag, const int *abort) {
  constexpr int NQ = G * HD / 2, NK = HD / 2;
  const uint64_t *qs = a.qkv_t + (int64_t)(g * G) * HD;
  const uint64_t *ks = a.qkv_t + (int64_t)(a.Hq + g) * HD;
  const uint64_t *vs = a.qkv_t + (int64_t)(a.Hq + a.Hkv + g) * HD;
  const int n = NQ + (has_pos ? 2 * NK : 0);
  bool ok = poll_pairs<NT, 4>(n, tag, abort, [&](int j, const uint64_t *&src, float *&dst, int &c) {
    c = 2;
    if (j < NQ) {
      src = qs + 2 * j;
      dst = sm.q + 2 * j;
    } else if (j < NQ + NK) {
      src = ks + 2 * (j - NQ);
      dst = sm.kn + 2 * (j - NQ);
    } else {
      src = vs + 2 * (j - NQ - NK);
      dst = sm.vn + 2 * (j - NQ - NK);
    }
  });
  return Sync::all(ok);
}

// After a split of KV head g wrote its partial (m, l, o) to the workspace: the last
// split of the head to arrive (atomic counter, no waiting) merges all nsplit partials
// into the output and resets the counter.  `last` is a shared-memory flag.
template <int G, int HD, int NT, class Sync, bool Tagged>
__device__ void attn_merge_splits(const AttnArgs &a, int g, int nsplit, unsigned &last, uint32_t tag) {
  constexpr int PART = G * (2 + HD);
  const int tid = threadIdx.x;
  __threadfence();
  Sync::sync();
  if (tid == 0) last = (atomicAdd(a.ws_count + g, 1u) == (unsigned)nsplit - 1);
  Sync::sync();
  if (!last) return;
  __threadfence();
  const float *base = a.ws_part + (int64_t)g * a.n_splits * PART;
  for (int i = tid; i < G * HD; i += NT) {
    const int h = i / HD;
    // one pass with online rescaling, eight splits' partials loaded per round trip
    float M = -INFINITY, O = 0.f, L = 0.f;
    for (int s0 = 0; s0 < nsplit; s0 += 8) {
      float ms[8], os[8], ls[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float *p = base + (int64_t)min(s0 + j, nsplit - 1) * PART;
        ms[j] = __ldcg(p + h);
        ls[j] = __ldcg(p + G + h);
        os[j] = __ldcg(p + 2 * G + i);
      }
      float mb = M;
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (s0 + j < nsplit) mb = fmaxf(mb, ms[j]);
      if (mb == -INFINITY) continue;
      const float c = (M == -INFINITY) ? 0.f : expf(M - mb);
      O *= c;
      L *= c;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (s0 + j < nsplit && ms[j] != -INFINITY) {
          const float f = expf(ms[j] - mb);
          O = fmaf(os[j], f, O);
          L = fmaf(ls[j], f, L);
        }
      }
      M = mb;
    }
    const float r = (L > 0.f) ? O / L : 0.f;
    if constexpr (Tagged) st_tagged(a.out_t + (g * G) * HD + i, r, tag);
    else a.out[(g * G) * HD + i] = r;
  }
  if (tid == 0) a.ws_count[g] = 0u;
  Sync::sync();
}

// Finishes split s of nsplit for KV head g from every warp's (m, l, o): with one split
// the result goes straight to the output; otherwise the split's partial goes to the
// workspace and the last split of the head to finish (atomic counter, no waiting)
// merges all partials and resets the counter.  Tagged: the output is written as
// tagged words to a.out_t, else as floats to a.out.
template <int G, int HD, int NW, class Sync, bool Tagged>
__device__ void attn_store(const AttnArgs &a, int g, int s, int nsplit, const float (&m)[G], const float (&l)[G],
                           const float (&o)[G][KvGroup<HD>::DPL], AttnSmem<G, HD, NW> &sm, uint32_t tag) {
  constexpr int DPL = KvGroup<HD>::DPL;
  constexpr int PART = G * (2 + HD);
  constexpr int NT = NW * 32;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  auto put = [&](int i, float r) {
    if constexpr (Tagged) st_tagged(a.out_t + (g * G) * HD + i, r, tag);
    else a.out[(g * G) * HD + i] = r;
  };
  // merge the warps
  if (lane == 0) {
#pragma unroll
    for (int h = 0; h < G; ++h) { sm.m[warp][h] = m[h]; sm.l[warp][h] = l[h]; }
  }
#pragma unroll
  for (int h = 0; h < G; ++h)
#pragma unroll
    for (int d = 0; d < DPL; ++d) sm.o[warp][h][lane * DPL + d] = o[h][d];
  Sync::sync();
  float *part = a.ws_part + ((int64_t)g * a.n_splits + s) * PART;
  for (int i = tid; i < G * HD; i += NT) {
    const int h = i / HD, d = i % HD;
    float M = -INFINITY;
    for (int w = 0; w < NW; ++w) M = fmaxf(M, sm.m[w][h]);
    float O = 0.f, L = 0.f;
    for (int w = 0; w < NW; ++w) {
      const float f = (sm.m[w][h] == -INFINITY) ? 0.f : expf(sm.m[w][h] - M);
      O = fmaf(sm.o[w][h][d], f, O);
      L = fmaf(sm.l[w][h], f, L);
    }
    if (nsplit == 1) {
      put(i, (L > 0.f) ? O / L : 0.f);
    } else {
      part[2 * G + i] = O;
      if (d == 0) { part[h] = M; part[G + h] = L; }
    }
  }
  if (nsplit == 1) {
    Sync::sync();  // the scratch is reused by the caller's next item
    return;
  }
  attn_merge_splits<G, HD, NT, Sync, Tagged>(a, g, nsplit, sm.last, tag);
}

// ------------------------------------------------------------------ chunk passes
//
// Attention over a chunk of K/V held in shared memory -- token t's key at byte t*hd*2
// from kbase, its value likewise from vbase (a run of whole blocks: kb = bs*hd*2 bytes
// per block makes the block arithmetic vanish) -- in three passes over the whole CTA
// instead of the per-warp online softmax above, whose shuffle chains cost ~5000 cycles
// per 16 tokens when few warps share an SM (measured on GB300): (1) a score for every
// (head, token) pair, lanes starting at different 16-byte chunks of their key rows so
// that the reads avoid bank conflicts; (2) one warp per head takes max, exp and sum and
// rescales the running (m, l); (3) every thread accumulates its (head, dim) outputs
// over the chunk.  The softmax is the two-pass definition evaluated per chunk with the
// running maximum carried across chunks.

constexpr int kChunkTok = 256;  // tokens of one chunk at most

// Shared scratch of the chunk passes.  buf holds the per-part scores in pass 1 and the
// per-token-group partial outputs in pass 3 (sized for up to 256 threads).
template <int G, int HD>
struct ChunkSmem {
  static constexpr int kParts = HD / 32;                       // 32-dim parts of a key row
  static constexpr int kGroupsMax = 512 / HD;                  // token groups of pass 3 at 256 threads
  static constexpr int kBuf = (kParts * kChunkTok > kGroupsMax * HD ? kParts * kChunkTok : kGroupsMax * HD) * G;
  float q[G * HD];
  float kn[HD], vn[HD];          // persistent step: the current token's k and v (bf16-exact)
  float pt[kChunkTok][G];        // probabilities, [token][head]
  float buf[kBuf];
  float m[G], l[G], corr[G];
  unsigned last;
};

// One chunk of ntok (1..kChunkTok) tokens.  sm.q holds the queries, sm.m / sm.l the
// running statistics (-inf / 0 before the first chunk); o[j] is this thread's output
// i = tid + j*NT of the G*HD outputs, rescaled and accumulated.  NT threads take part;
// Sync is a barrier over them.  The caller synchronises before the next chunk.
template <int G, int HD, int NT, class Sync>
__device__ __forceinline__ void chunk_passes(uint32_t kbase, uint32_t vbase, int ntok, float scale,
                                             ChunkSmem<G, HD> &sm, float (&o)[(G * HD + NT - 1) / NT]) {
  constexpr int NO = (G * HD + NT - 1) / NT;
  constexpr int P = ChunkSmem<G, HD>::kParts;
  constexpr int DP = HD / 2;        // dim pairs
  constexpr int TG = NT / DP;       // token groups of pass 3
  constexpr int NW = NT / 32;
  static_assert(TG <= ChunkSmem<G, HD>::kGroupsMax && TG >= 1, "pass-3 groups fit the buffer");
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t qa = smem_u32(sm.q);
  // (1) scores: one (token, 32-dim part) per item, all heads at once
  for (int it = tid; it < ntok * P; it += NT) {
    const int t = it / P, part = it % P;
    const uint32_t krow = kbase + (uint32_t)t * (HD * 2) + part * 64;
    uint4 kw[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) kw[c] = lds128(krow + ((c + lane) & 3) * 16);
    float acc[G][2];
#pragma unroll
    for (int h = 0; h < G; ++h) {
      acc[h][0] = acc[h][1] = 0.f;
      const uint32_t qrow = qa + (uint32_t)(h * HD + part * 32) * 4;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const uint32_t qo = qrow + ((c + lane) & 3) * 32;
        const float4 q0 = lds128f(qo), q1 = lds128f(qo + 16);
        acc[h][0] = fmaf(q0.x, __uint_as_float(kw[c].x << 16), acc[h][0]);
        acc[h][1] = fmaf(q0.y, __uint_as_float(kw[c].x & 0xffff0000u), acc[h][1]);
        acc[h][0] = fmaf(q0.z, __uint_as_float(kw[c].y << 16), acc[h][0]);
        acc[h][1] = fmaf(q0.w, __uint_as_float(kw[c].y & 0xffff0000u), acc[h][1]);
        acc[h][0] = fmaf(q1.x, __uint_as_float(kw[c].z << 16), acc[h][0]);
        acc[h][1] = fmaf(q1.y, __uint_as_float(kw[c].z & 0xffff0000u), acc[h][1]);
        acc[h][0] = fmaf(q1.z, __uint_as_float(kw[c].w << 16), acc[h][0]);
        acc[h][1] = fmaf(q1.w, __uint_as_float(kw[c].w & 0xffff0000u), acc[h][1]);
      }
    }
#pragma unroll
    for (int h = 0; h < G; ++h) sm.buf[(part * G + h) * kChunkTok + t] = acc[h][0] + acc[h][1];
  }
  Sync::sync();
  // (2) softmax statistics, one warp per head; probabilities to pt[token][head]
  for (int h = warp; h < G; h += NW) {
    auto score = [&](int t) {
      float v = 0.f;
#pragma unroll
      for (int part = 0; part < P; ++part) v += sm.buf[(part * G + h) * kChunkTok + t];
      return v * scale;
    };
    float mx = -INFINITY;
    for (int t = lane; t < ntok; t += 32) mx = fmaxf(mx, score(t));
    mx = warp_max(mx);
    const float m_old = sm.m[h], m_new = fmaxf(m_old, mx);
    float sum = 0.f;
    for (int t = lane; t < ntok; t += 32) {
      const float pr = expf(score(t) - m_new);
      sm.pt[t][h] = pr;
      sum += pr;
    }
    sum = warp_sum(sum);
    if (lane == 0) {
      const float c = (m_old == -INFINITY) ? 0.f : expf(m_old - m_new);
      sm.corr[h] = c;
      sm.l[h] = sm.l[h] * c + sum;
      sm.m[h] = m_new;
    }
  }
  Sync::sync();
  // (3) outputs: thread (dim pair dp, token group tg) over tokens tg, tg + TG, ...
  if (tid < TG * DP) {
    const int dp = tid % DP, tg = tid / DP;
    float a[G][2];
#pragma unroll
    for (int h = 0; h < G; ++h) a[h][0] = a[h][1] = 0.f;
    const uint32_t vcol = vbase + dp * 4, pa = smem_u32(&sm.pt[0][0]);
    for (int t = tg; t < ntok; t += TG) {
      const uint32_t vw = lds32(vcol + (uint32_t)t * (HD * 2));
      const float v0 = __uint_as_float(vw << 16), v1 = __uint_as_float(vw & 0xffff0000u);
      float pv[G];
      if constexpr (G % 4 == 0) {
#pragma unroll
        for (int h = 0; h < G; h += 4) {
          const float4 p4 = lds128f(pa + (uint32_t)(t * G + h) * 4);
          pv[h] = p4.x;
          pv[h + 1] = p4.y;
          pv[h + 2] = p4.z;
          pv[h + 3] = p4.w;
        }
      } else {
#pragma unroll
        for (int h = 0; h < G; ++h) pv[h] = sm.pt[t][h];
      }
#pragma unroll
      for (int h = 0; h < G; ++h) {
        a[h][0] = fmaf(pv[h], v0, a[h][0]);
        a[h][1] = fmaf(pv[h], v1, a[h][1]);
      }
    }
#pragma unroll
    for (int h = 0; h < G; ++h) {
      sm.buf[(tg * G + h) * HD + 2 * dp] = a[h][0];
      sm.buf[(tg * G + h) * HD + 2 * dp + 1] = a[h][1];
    }
  }
  Sync::sync();
#pragma unroll
  for (int j = 0; j < NO; ++j) {
    const int i = tid + j * NT;
    if (i < G * HD) {
      const int h = i / HD, d = i % HD;
      float acc = o[j] * sm.corr[h];
#pragma unroll 4
      for (int tg = 0; tg < TG; ++tg) acc += sm.buf[(tg * G + h) * HD + d];
      o[j] = acc;
    }
  }
}

// Computes split s of nsplit for KV head g, reading K/V from the paged pool.
// blk_pre, when not null, holds the block ids of blocks [0, nblk) already staged in
// shared memory; otherwise they are read from bt in chunks.  Sync::sync() is a barrier
// over the NW participating warps, whose threads are numbered 0 .. NW*32-1.
//
// Tagged (the persistent step): q and the current token's k and v (position ctx-1)
// are polled as tagged words from a.qkv_t, whose k and v values are already rounded
// to bf16; the token's K/V then replace whatever the cache held at its slot (its
// write into the cache by another SM may not be visible yet), and the output is
// written as tagged words to a.out_t.  Returns false if a poll gave up.
template <int G, int HD, int NW, class Sync, bool Tagged = false>
__device__ bool attn_split(const AttnArgs &a, int g, int s, int nsplit, int ctx, const int32_t *bt, const int *blk_pre,
                           AttnSmem<G, HD, NW> &sm, uint32_t tag = 0, const int *abort = nullptr) {
  using KG = KvGroup<HD>;
  constexpr int TPI = KG::TPI, DPL = KG::DPL, LPT = KG::LPT;
  constexpr int NT = NW * 32;
  constexpr int QB = (G * HD + NT - 1) / NT;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nblk = (ctx + a.bs - 1) / a.bs;
  const int b0 = (int)((int64_t)s * nblk / nsplit), b1 = (int)((int64_t)(s + 1) * nblk / nsplit);
  const int t_end = min(b1 * a.bs, ctx);
  const int part_in = lane % LPT;
  const int64_t head_off = (int64_t)g * a.bs * HD;

  // the queries of the group: loads issued now, stored once the first K/V loads are out
  float qv[QB];
  if constexpr (!Tagged) {
#pragma unroll
    for (int j = 0; j < QB; ++j) qv[j] = __ldcg(a.q + (g * G) * HD + min(tid + j * NT, G * HD - 1));
  }
  bool q_stored = false;
  const int pos = ctx - 1;
  const bool has_pos = Tagged && t_end == ctx && ctx > 0;  // this split holds the current token

  float m[G], l[G], o[G][DPL];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    m[h] = -INFINITY;
    l[h] = 0.f;
#pragma unroll
    for (int d = 0; d < DPL; ++d) o[h][d] = 0.f;
  }

  for (int cb = b0; cb < b1; cb += kAttnMaxBlocks) {
    const int ce = blk_pre ? b1 : min(b1, cb + kAttnMaxBlocks);
    const int *ids = blk_pre;
    int id0 = 0;
    if (!blk_pre) {
      Sync::sync();
      for (int i = tid; i < ce - cb; i += NT) {
        int blk = bt[cb + i];
        if (blk < 0 || blk >= a.n_pool_blocks) {
          latch_error(a.err, ERR_BLOCK_ID);
          blk = -1;
        }
        sm.blk[i] = blk;
      }
      Sync::sync();
      ids = sm.blk;
      id0 = cb;
    }
    const int t0 = cb * a.bs, t1 = min(ce * a.bs, t_end);
    int tb = t0 + warp * TPI;
    KG cur;
    cur.load(a, ids, id0, tb, t1, head_off, lane);
    if (!q_stored) {
      if constexpr (Tagged) {
        if (!tagged_inputs<G, HD, NT, Sync>(a, g, has_pos, sm, tag, abort)) return false;
      } else {
#pragma unroll
        for (int j = 0; j < QB; ++j)
          if (tid + j * NT < G * HD) sm.q[tid + j * NT] = qv[j];
        Sync::sync();
      }
      q_stored = true;
    }
    for (; tb < t1; tb += NW * TPI) {
      if (has_pos) patch_current<HD>(cur, pos - tb, sm.kn, sm.vn, lane);
      const int kblk = cur.kblk;
      float vf[TPI][DPL];
      group_values<HD>(cur, vf);
      float sc[G];
      group_scores<G, HD>(cur, smem_u32(sm.q), part_in, sc);
      // the next group's loads go out before this group's softmax
      if (tb + NW * TPI < t1) cur.load(a, ids, id0, tb + NW * TPI, t1, head_off, lane);
      group_update<G, HD>(sc, vf, kblk, a.scale, part_in, m, l, o);
    }
  }
  if (!q_stored) {  // empty split: keep the barrier count of the other paths
    if constexpr (Tagged) {
      if (!tagged_inputs<G, HD, NT, Sync>(a, g, false, sm, tag, abort)) return false;
    } else {
      Sync::sync();
    }
  }
  attn_store<G, HD, NW, Sync, Tagged>(a, g, s, nsplit, m, l, o, sm, tag);
  return true;
}

}  // namespace mie
