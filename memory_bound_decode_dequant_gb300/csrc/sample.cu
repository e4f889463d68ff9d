// sample.cu -- temperature / top-k / top-p sampling of the next token on the GPU.
//
// "infer" page, design notes: sampling runs on the GPU, with radix select for the top-k
// and top-p cut-offs and per-position random numbers drawn from a seed, so that a sampled
// step is still one CUDA graph and runs reproduce.  The sampler takes the plain
// definition: with q_i = exp((l_i - max) / T), top-k keeps the tokens whose logit is at
// least the k-th largest (ties kept), top-p then keeps those whose logit is at least the
// largest t with mass(l >= t) >= p * (kept mass) (ties kept), and the token is the
// Gumbel-max draw argmax_i (l_i / T - log(-log u_i)) over the kept set, u_i from
// splitmix64 of (seed, pos << 32 | i); T <= 0 is greedy.
//
// A launch of several short passes over the logits, each a grid of a few CTAs:
//   pass 0       the maximum logit (and, greedy, the token);
//   passes 1..4  top-k: radix select of the k-th largest logit, eight key bits a pass;
//   passes 5..8  top-p: radix select of the mass cut-off over the top-k survivors;
//   pass 9       the Gumbel-max draw over the kept tokens.
// Each pass adds its CTAs' histograms into global bins with integer atomics (counts,
// and masses in 2^40 fixed point), so the sums -- and therefore the cut-offs -- do not
// depend on the order the CTAs run in; the last CTA of a pass (atomic counter) picks the
// radix digit and leaves the bins zeroed for the next pass.  The maximum and the draw are
// 64-bit atomicMax over (monotone key of the value, inverted index): the lowest index
// wins a tie.
#include "internal.h"

namespace mie {

constexpr int kSampleThreads = 256;
constexpr int kSampleMaxGrid = 64;
constexpr int kSampleElemsPerThread = 8;
constexpr double kMassScale = 1099511627776.0;  // 2^40: q in (0, 1] -> fixed point

struct SampleWs {
  unsigned long long best;        // packed (key << 32 | ~index) maximum
  unsigned long long mass[256];   // digit histogram: fixed-point softmax mass
  unsigned count[256];            // digit histogram: element count
  unsigned done;                  // CTAs finished with the current pass
  float mx;                       // the maximum logit
  uint32_t kprefix, pprefix;      // key bits fixed so far (top-k, top-p)
  unsigned need_k;                // elements still to take at and below the top-k prefix
  unsigned long long need_mass;   // mass still to take at and below the top-p prefix
  uint32_t tk_key, tp_key;        // cut-off keys (0: keep all)
};

size_t sample_workspace_bytes() { return (sizeof(SampleWs) + 255) / 256 * 256; }

struct SampleArgs {
  const float *logits = nullptr;  // used when sp == null (else sp->logits_out + slot * n)
  int n = 0;
  float temperature = 0.f;
  int top_k = 0;
  float top_p = 1.f;
  uint64_t seed = 0;
  int pos = 0;                    // used when sp == null
  StepParams *sp = nullptr;       // in-step: logits, position, output, advance from here
  int slot = 0;
  int32_t *out = nullptr;         // used when sp == null
  SampleWs *ws = nullptr;
  int pass = 0;
};

__device__ __forceinline__ uint32_t fkey(float v) {
  const uint32_t b = __float_as_uint(v);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float fkey_inv(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

__device__ __forceinline__ uint64_t splitmix64(uint64_t seed, uint64_t i) {
  uint64_t z = seed + (i + 1) * 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

// warp-wide maximum of a packed 64-bit key
__device__ __forceinline__ unsigned long long warp_max_u64(unsigned long long v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long w = __shfl_xor_sync(0xffffffffu, v, o);
    v = w > v ? w : v;
  }
  return v;
}

// Ends a pass: the last CTA to arrive runs `last(ws)` (every CTA's global atomics of the
// pass are visible to it) and re-arms the counter.
template <class Last>
__device__ void end_pass(SampleWs *ws, Last last) {
  __shared__ unsigned s_last;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = (atomicAdd(&ws->done, 1u) == gridDim.x - 1);
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  last(ws);
  __syncthreads();
  if (threadIdx.x == 0) ws->done = 0u;
}

__global__ void __launch_bounds__(kSampleThreads) sample_pass_kernel(const SampleArgs a) {
  __shared__ unsigned long long s_mass[256];
  __shared__ unsigned s_count[256];
  __shared__ unsigned long long s_best[kSampleThreads / 32];
  pdl_trigger();
  pdl_wait();
  SampleWs *ws = a.ws;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n = a.n;
  const float *logits = a.sp ? a.sp->logits_out + (int64_t)a.slot * n : a.logits;
  const int pos = a.sp ? a.sp->pos[a.slot] : a.pos;
  const int stride = gridDim.x * kSampleThreads;
  const int pass = a.pass;

  if (pass == 0 || pass == 9) {  // maximum, or the Gumbel-max draw over the kept tokens
    const uint32_t cut = max(ws->tk_key, ws->tp_key);
    unsigned long long best = 0ull;
    for (int i = blockIdx.x * kSampleThreads + tid; i < n; i += stride) {
      const float l = logits[i];
      float v = l;
      if (pass == 9) {
        if (fkey(l) < cut) continue;
        const uint64_t z = splitmix64(a.seed, ((uint64_t)(uint32_t)pos << 32) | (uint32_t)i);
        const float u = ((float)(uint32_t)(z >> 40) + 0.5f) * 5.9604644775390625e-08f;  // / 2^24
        v = __fdiv_rn(l, a.temperature) - logf(-logf(u));
      }
      const unsigned long long p = ((unsigned long long)fkey(v) << 32) | (uint32_t)(0xffffffffu - (uint32_t)i);
      best = p > best ? p : best;
    }
    best = warp_max_u64(best);
    if (lane == 0) s_best[warp] = best;
    __syncthreads();
    if (tid == 0) {
      for (int w = 1; w < kSampleThreads / 32; ++w) best = s_best[w] > best ? s_best[w] : best;
      atomicMax(&ws->best, best);
    }
    end_pass(ws, [&](SampleWs *w) {
      if (threadIdx.x != 0) return;
      const unsigned long long b = w->best;
      const int idx = (int)(0xffffffffu - (uint32_t)b);
      w->best = 0ull;
      const bool finish = pass == 9 || !(a.temperature > 0.f);
      if (pass == 0) {
        w->mx = fkey_inv((uint32_t)(b >> 32));
        w->kprefix = w->pprefix = 0u;
        w->need_k = (unsigned)a.top_k;
        w->need_mass = 0ull;
        w->tk_key = w->tp_key = 0u;
      }
      if (finish) {
        const int tok = (idx >= 0 && idx < n) ? idx : 0;
        if (a.sp) {
          if (a.sp->argmax_out) a.sp->argmax_out[a.slot] = tok;
          if (a.sp->sample_advance) {  // the step's token advance, deferred to the sampler
            a.sp->token[a.slot] = tok;
            a.sp->pos[a.slot] += 1;
          }
        } else {
          *a.out = tok;
        }
        w->tk_key = w->tp_key = 0u;
      }
    });
    return;
  }

  // radix passes: digit d of the key (bits shift .. shift+7), among the keys whose higher
  // bits equal the prefix fixed so far
  const bool topk = pass <= 4;
  const int d = topk ? pass - 1 : pass - 5;
  const int shift = 24 - 8 * d;
  const uint32_t hi_mask = shift == 24 ? 0u : (0xffffffffu << (shift + 8));
  const uint32_t prefix = topk ? ws->kprefix : ws->pprefix;
  const uint32_t tk = ws->tk_key;
  const float mx = ws->mx, inv_t = 1.0f / a.temperature;
  for (int b = tid; b < 256; b += kSampleThreads) {
    s_mass[b] = 0ull;
    s_count[b] = 0u;
  }
  __syncthreads();
  for (int i = blockIdx.x * kSampleThreads + tid; i < n; i += stride) {
    const float l = logits[i];
    const uint32_t k = fkey(l);
    if ((k & hi_mask) != (prefix & hi_mask)) continue;
    const int bin = (int)((k >> shift) & 255u);
    if (topk) {
      atomicAdd(&s_count[bin], 1u);
    } else if (k >= tk) {
      const float q = expf((l - mx) * inv_t);
      const unsigned long long m = (unsigned long long)((double)q * kMassScale + 0.5);
      if (m) atomicAdd(&s_mass[bin], m);
    }
  }
  __syncthreads();
  for (int b = tid; b < 256; b += kSampleThreads) {
    if (topk) {
      if (s_count[b]) atomicAdd(&ws->count[b], s_count[b]);
    } else if (s_mass[b]) {
      atomicAdd(&ws->mass[b], s_mass[b]);
    }
  }
  end_pass(ws, [&](SampleWs *w) {
    if (threadIdx.x != 0) return;
    if (topk) {
      unsigned cum = 0u;
      int pick = 0;
      for (int b = 255; b >= 0; --b) {
        const unsigned c = w->count[b];
        if (c && cum + c >= w->need_k) {
          pick = b;
          w->need_k -= cum;
          break;
        }
        cum += c;
      }
      w->kprefix |= (uint32_t)pick << shift;
      if (d == 3) w->tk_key = w->kprefix;
      for (int b = 0; b < 256; ++b) w->count[b] = 0u;
    } else {
      if (d == 0) {  // the kept mass and the top-p target
        unsigned long long z = 0ull;
        for (int b = 0; b < 256; ++b) z += w->mass[b];
        w->need_mass = (unsigned long long)((double)a.top_p * (double)z);
      }
      unsigned long long cum = 0ull;
      int pick = 0;
      for (int b = 255; b >= 0; --b) {
        const unsigned long long m = w->mass[b];
        if (m && cum + m >= w->need_mass) {
          pick = b;
          w->need_mass -= cum;
          break;
        }
        cum += m;
      }
      w->pprefix |= (uint32_t)pick << shift;
      if (d == 3) w->tp_key = w->pprefix;
      for (int b = 0; b < 256; ++b) w->mass[b] = 0ull;
    }
  });
}

static int sample_grid(int n) {
  const int g = (n + kSampleThreads * kSampleElemsPerThread - 1) / (kSampleThreads * kSampleElemsPerThread);
  return g < 1 ? 1 : (g > kSampleMaxGrid ? kSampleMaxGrid : g);
}

// Enqueues the passes the parameters need; ws must be zero before the first launch on it
// (every launch leaves it zeroed again).
mie_status launch_sample(const SampleArgs &base, cudaStream_t st, bool pdl) {
  int passes[10], np = 0;
  passes[np++] = 0;
  if (base.temperature > 0.f) {
    if (base.top_k > 0 && base.top_k < base.n)
      for (int p = 1; p <= 4; ++p) passes[np++] = p;
    if (base.top_p < 1.f)
      for (int p = 5; p <= 8; ++p) passes[np++] = p;
    passes[np++] = 9;
  }
  for (int i = 0; i < np; ++i) {
    SampleArgs a = base;
    a.pass = passes[i];
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(sample_grid(a.n));
    cfg.blockDim = dim3(kSampleThreads);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    MIE_CUDA(cudaLaunchKernelEx(&cfg, sample_pass_kernel, a));
  }
  return MIE_OK;
}

mie_status launch_step_sample(StepParams *sp, int vocab, float temperature, int top_k, float top_p, uint64_t seed,
                              void *ws, cudaStream_t st) {
  SampleArgs a;
  a.n = vocab;
  a.temperature = temperature;
  a.top_k = top_k;
  a.top_p = top_p;
  a.seed = seed;
  a.sp = sp;
  a.ws = reinterpret_cast<SampleWs *>(ws);
  return launch_sample(a, st, true);
}

int sample_launches(float temperature, int top_k, float top_p, int n) {
  if (!(temperature > 0.f)) return 1;
  return 2 + ((top_k > 0 && top_k < n) ? 4 : 0) + (top_p < 1.f ? 4 : 0);
}

}  // namespace mie

using namespace mie;

extern "C" size_t mie_sample_workspace_bytes(void) { return sample_workspace_bytes(); }

extern "C" mie_status mie_sample(const float *logits, int n, float temperature, int top_k, float top_p,
                                 uint64_t seed, int32_t pos, int32_t *out, void *workspace, size_t workspace_bytes,
                                 void *stream) {
  if (!logits || !out || !workspace) return fail(MIE_E_ARG, "mie_sample: null pointer");
  if (n < 1) return fail(MIE_E_SHAPE, "mie_sample: n = %d", n);
  if (top_k < 0 || !(top_p > 0.f) || top_p > 1.f || temperature != temperature)
    return fail(MIE_E_ARG, "mie_sample: top_k %d, top_p %g, temperature %g", top_k, top_p, temperature);
  if (((uintptr_t)workspace & 255) || workspace_bytes < sample_workspace_bytes())
    return fail(MIE_E_ARG, "mie_sample: workspace of %zu bytes, 256-byte aligned, needed", sample_workspace_bytes());
  cudaStream_t st = (cudaStream_t)stream;
  MIE_CUDA(cudaMemsetAsync(workspace, 0, sample_workspace_bytes(), st));
  SampleArgs a;
  a.logits = logits;
  a.n = n;
  a.temperature = temperature;
  a.top_k = top_k;
  a.top_p = top_p;
  a.seed = seed;
  a.pos = pos;
  a.out = out;
  a.ws = reinterpret_cast<SampleWs *>(workspace);
  return launch_sample(a, st, false);
}
