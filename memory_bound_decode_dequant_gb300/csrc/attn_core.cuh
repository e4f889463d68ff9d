// attn_core.cuh -- one (KV head, context split) of paged GQA decode attention, shared
// by the standalone attention kernel and the persistent step kernel.
//
// "Mini Inference Engine", "The KV cache, paged like virtual memory": K/V are read
// through a block table; "infer" page, design notes, the split-KV attention item: the query heads
// of one KV head share every K/V load, the context is split and partial softmaxes are
// merged; "Writing an LLM inference engine from scratch in Rust", Lesson 4: an online
// softmax with a running maximum and sum.
//
// A split's K/V reach shared memory as runs of whole blocks (bulk copies through the
// block table, issued by the caller) and each run is reduced by chunk_passes below.
#pragma once

#include "device.cuh"

namespace mie {

// Splits in use for a context of nblk blocks: every split gets at least per_split
// blocks (so its warps have work), at most max_splits splits.
__host__ __device__ inline int attn_nsplit(int nblk, int max_splits, int per_split) {
  int s = (nblk + per_split - 1) / per_split;
  if (s > max_splits) s = max_splits;
  return s < 1 ? 1 : s;
}

// Tagged variant: polls the G queries from query head h0 on into sm.q and, when
// has_pos, the current token's k and v of KV head g into sm.kn / sm.vn, all in one
// batch of round trips.
template <int G, int HD, int NT, class Sync, class SM>
__device__ bool tagged_inputs(const AttnArgs &a, int h0, int g, bool has_pos, SM &sm, uint32_t tag,
                              const int *abort, long limit) {
  constexpr int NQ = G * HD / 2, NK = HD / 2;
  const uint64_t *qs = a.qkv_t + (int64_t)h0 * HD;
  const uint64_t *ks = a.qkv_t + (int64_t)(a.Hq + g) * HD;
  const uint64_t *vs = a.qkv_t + (int64_t)(a.Hq + a.Hkv + g) * HD;
  const int n = NQ + (has_pos ? 2 * NK : 0);
  bool ok = poll_pairs<NT, 4>(n, tag, abort, limit, [&](int j, const uint64_t *&src, float *&dst, int &c) {
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

// After a split of unit g (a KV head with its G query heads, or with G = 1 a single
// query head) wrote its partial (m, l, o) to the workspace: the last split of the unit
// to arrive (atomic counter, no waiting) merges all nsplit partials into the outputs of
// query heads g*G .. g*G+G-1 and resets the counter.  `last` is a shared-memory flag.
// B splits' partials are loaded per round trip (the standalone kernels take 16; the
// persistent step, short of registers, 8).
template <int G, int HD, int NT, class Sync, bool Tagged, int B = 8>
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
    // one pass with online rescaling, B splits' partials loaded per round trip
    float M = -INFINITY, O = 0.f, L = 0.f;
    for (int s0 = 0; s0 < nsplit; s0 += B) {
      float ms[B], os[B], ls[B];
#pragma unroll
      for (int j = 0; j < B; ++j) {
        const float *p = base + (int64_t)min(s0 + j, nsplit - 1) * PART;
        ms[j] = __ldcg(p + h);
        ls[j] = __ldcg(p + G + h);
        os[j] = __ldcg(p + 2 * G + i);
      }
      float mb = M;
#pragma unroll
      for (int j = 0; j < B; ++j)
        if (s0 + j < nsplit) mb = fmaxf(mb, ms[j]);
      if (mb == -INFINITY) continue;
      const float c = (M == -INFINITY) ? 0.f : expf(M - mb);
      O *= c;
      L *= c;
#pragma unroll
      for (int j = 0; j < B; ++j) {
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

// ------------------------------------------------------------------ chunk passes
//
// Attention over a chunk of K/V held in shared memory -- token t's key at byte t*hd*2
// from kbase, its value likewise from vbase (a run of whole blocks: kb = bs*hd*2 bytes
// per block makes the block arithmetic vanish) -- in three passes over the whole CTA
// instead of a per-warp online softmax, whose shuffle chains cost ~5000 cycles per 16
// tokens when few warps share an SM (measured on GB300): (1) a score for every
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

}  // namespace mie
