/*
 * mie_oracle.c -- the oracle for the batch-1 / few-slot decode step.
 *
 * TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT.  Only the tests, the smoke check and
 * the bench's CPU-baseline leg load this library.  It shares no code, header, table
 * or helper with the CUDA library; both sides draw their inputs from the separate
 * `synth` generator module.
 *
 * What it is: a plain, slow CPU implementation of what the decode step computes,
 * written for a reader to check against the pages by eye (single-threaded unless
 * or_set_threads asks for more; the result is the same).  Tensors are stored at the
 * precision the pages fix -- fp32 activations and residual stream, bf16 K/V cache,
 * quantised weights (the "infer" page, design notes: weights in bf16, activations and
 * sums in fp32, the cache in bf16; its reference rounds K and V to bf16 when they
 * enter the cache).  Inside one operation every sum is taken in fp64 and the result
 * rounded once to fp32, so each function returns its plain definition rounded to the
 * storage type.
 * Compile with -ffp-contract=off so that no multiply-add is fused behind the reader's
 * back (the quantisers' rounding decisions depend on it).
 *
 * Pages cited (titles):
 *  [RUST]  "Writing an LLM inference engine from scratch in Rust"
 *  [MIE]   "Mini Inference Engine"
 *  [INFER] "infer" -- an LLM inference engine in C++ and CUDA for Llama-3.2-1B
 *
 * Readings of points the pages leave open are marked READING below, each with the
 * reason it was taken.
 *
 * Parity pins: every function here is pinned by a `-m "not gpu"` test against
 * something other than itself (closed forms, invariants, brute force, numpy's IEEE
 * conversions).  The composed full-model logits are "parity unpinned" beyond the
 * composition of pinned parts; the incremental-vs-no-cache invariant pins the cache
 * plumbing.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------ threads */

/* Host threads used by the loops marked "parallel over independent ..." below (GEMV
 * output rows, attention heads, quantiser rows, element conversions).  Each output
 * keeps its own serial arithmetic, so the results are bit-identical for every thread
 * count; 1 (the default) runs everything on the calling thread.  Built without
 * OpenMP the pragmas are ignored and the count stays 1. */
static int g_threads = 1;

int or_set_threads(int n) {
#ifdef _OPENMP
  g_threads = n < 1 ? 1 : n;
#else
  (void)n;
  g_threads = 1;
#endif
  return g_threads;
}

int or_max_threads(void) {
#ifdef _OPENMP
  return omp_get_num_procs();
#else
  return 1;
#endif
}

/* ------------------------------------------------------------------ conversions */

/* Round v to the nearest value with p fraction bits at its binade (binades below
 * 2^emin use the spacing of 2^emin), ties to even.  Exact in double for the
 * formats used here; nearbyint() rounds in the default nearest-even mode. */
static double round_to_grid(double v, int p, int emin) {
  if (v == 0.0 || !isfinite(v)) return v;
  int E;
  frexp(v, &E); /* |v| = m * 2^E, m in [0.5, 1) */
  int e = E - 1;
  if (e < emin) e = emin;
  const double sp = ldexp(1.0, e - p);
  return nearbyint(v / sp) * sp;
}

static uint32_t f32_bits(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }
static float bits_f32(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }

/* fp32 -> bf16, round to nearest even (bf16: 7 fraction bits, fp32's exponent range). */
uint16_t or_f32_to_bf16(float f) {
  if (isnan(f)) return (uint16_t)((f32_bits(f) >> 16) | 0x0040);
  const float r = (float)round_to_grid((double)f, 7, -126); /* overflow -> inf */
  return (uint16_t)(f32_bits(r) >> 16);
}

float or_bf16_to_f32(uint16_t h) { return bits_f32((uint32_t)h << 16); }

/* fp32 -> IEEE binary16, round to nearest even, subnormals kept, overflow -> inf. */
uint16_t or_f32_to_f16(float f) {
  const uint16_t sign = (uint16_t)((f32_bits(f) >> 16) & 0x8000);
  if (isnan(f)) return (uint16_t)(sign | 0x7E00);
  double a = fabs((double)f);
  if (isinf(f)) return (uint16_t)(sign | 0x7C00);
  a = round_to_grid(a, 10, -14);
  if (a >= 65536.0) return (uint16_t)(sign | 0x7C00);
  if (a < ldexp(1.0, -14)) return (uint16_t)(sign | (uint16_t)(a * ldexp(1.0, 24)));
  int E;
  frexp(a, &E);
  const int e = E - 1;
  const uint16_t mant = (uint16_t)(a / ldexp(1.0, e - 10) - 1024.0);
  return (uint16_t)(sign | ((e + 15) << 10) | mant);
}

float or_f16_to_f32(uint16_t h) {
  const int e = (h >> 10) & 0x1F, m = h & 0x3FF;
  double v;
  if (e == 0) v = ldexp((double)m, -24);
  else if (e == 31) v = m ? NAN : INFINITY;
  else v = ldexp((double)(1024 + m), e - 25);
  return (float)((h & 0x8000) ? -v : v);
}

void or_f32_to_bf16_n(const float *x, int64_t n, uint16_t *out) {
#pragma omp parallel for schedule(static) num_threads(g_threads) if (g_threads > 1) /* independent elements */
  for (int64_t i = 0; i < n; ++i) out[i] = or_f32_to_bf16(x[i]);
}
void or_bf16_to_f32_n(const uint16_t *x, int64_t n, float *out) {
  for (int64_t i = 0; i < n; ++i) out[i] = or_bf16_to_f32(x[i]);
}
void or_f32_to_f16_n(const float *x, int64_t n, uint16_t *out) {
  for (int64_t i = 0; i < n; ++i) out[i] = or_f32_to_f16(x[i]);
}
void or_f16_to_f32_n(const uint16_t *x, int64_t n, float *out) {
  for (int64_t i = 0; i < n; ++i) out[i] = or_f16_to_f32(x[i]);
}

/* ------------------------------------------------------------------ quantisers */

enum { OR_BF16 = 0, OR_I8 = 1, OR_Q4_0 = 2, OR_F32 = 3, OR_Q4_G64 = 4, OR_Q4_G128 = 5 };

/* Weights per scale of the 4-bit formats (0 for the others). */
int or_q4_group(int fmt) {
  return fmt == OR_Q4_0 ? 32 : fmt == OR_Q4_G64 ? 64 : fmt == OR_Q4_G128 ? 128 : 0;
}

/* 4-bit groups ([RUST] "Lesson 1" and "Is the 4-bit model still good?"; [INFER] design
 * notes, weight-only quantization: int4 with one 2-byte scale per group of weights,
 * 4-bit values stored as w + 8 in 0..15; the scale is the group's signed extreme (the
 * element whose magnitude is largest) over -8, so that element's code is exactly -8, the
 * end of the 4-bit range that has no positive twin; the [INFER] page's int4 uses groups
 * of 32 like Q4_0, started from groups of 128 and also measured groups of 64).
 * READING: first such element on ties; d = m / -8 in fp32 (exact); stored h = f16(d)
 * rounded to nearest even; codes use the stored scale: id = 1/h (0 when h == 0),
 * q = clamp(floor(w*id + 8.5), 0, 15) with the product and the sum each rounded in
 * fp32.  Every 32 consecutive codes of a group form one 16-byte sub-block whose byte j
 * holds code j in its low nibble and code j+16 in its high nibble (the low/high pairing
 * of [RUST] "Lesson 6"); a group is stored as its f16 scale (little-endian) followed by
 * its GS/32 sub-blocks: 2 + GS/2 bytes, 18 for GS = 32 (Q4_0).  A row whose length is
 * not a multiple of GS is zero-padded to the next group; zeros code to 8 = exactly 0.
 * Output: rows of ceil(K/GS) groups, [M][ng][2 + GS/2]. */
void or_q4_quantize(const float *w, int M, int K, int GS, uint8_t *out) {
  const int ng = (K + GS - 1) / GS, gbytes = 2 + GS / 2;
#pragma omp parallel for schedule(static) num_threads(g_threads) if (g_threads > 1) /* independent rows */
  for (int r = 0; r < M; ++r) {
    for (int b = 0; b < ng; ++b) {
      float v[128];
      for (int j = 0; j < GS; ++j) {
        const int k = b * GS + j;
        v[j] = (k < K) ? w[(int64_t)r * K + k] : 0.0f;
      }
      float amax = 0.0f, m = 0.0f;
      for (int j = 0; j < GS; ++j)
        if (fabsf(v[j]) > amax) { amax = fabsf(v[j]); m = v[j]; }
      const float d = m / -8.0f;
      const uint16_t h = or_f32_to_f16(d);
      const float hd = or_f16_to_f32(h);
      const float id = (hd != 0.0f) ? 1.0f / hd : 0.0f;
      int q[128];
      for (int j = 0; j < GS; ++j) {
        float t = v[j] * id;
        t = t + 8.5f;
        int c = (int)floorf(t);
        q[j] = c < 0 ? 0 : (c > 15 ? 15 : c);
      }
      uint8_t *grp = out + ((int64_t)r * ng + b) * gbytes;
      grp[0] = (uint8_t)(h & 0xFF);
      grp[1] = (uint8_t)(h >> 8);
      for (int sb = 0; sb < GS / 32; ++sb)
        for (int j = 0; j < 16; ++j)
          grp[2 + sb * 16 + j] = (uint8_t)(q[sb * 32 + j] | (q[sb * 32 + j + 16] << 4));
    }
  }
}

/* Q4_0: the 4-bit format with groups of 32. */
void or_q4_0_quantize(const float *w, int M, int K, uint8_t *out) { or_q4_quantize(w, M, K, 32, out); }

/* Element k of row r of a canonical 4-bit matrix with groups of GS (ng per row):
 * h * (q - 8). */
static float q4_at(const uint8_t *wq, int GS, int ng, int r, int k) {
  const uint8_t *grp = wq + ((int64_t)r * ng + k / GS) * (2 + GS / 2);
  const float h = or_f16_to_f32((uint16_t)(grp[0] | (grp[1] << 8)));
  const int j = k % GS, sb = j / 32, i = j % 32;
  const uint8_t byte = grp[2 + sb * 16 + (i % 16)];
  const int q = (i < 16) ? (byte & 0x0F) : (byte >> 4);
  return h * (float)(q - 8); /* exact: |q-8| <= 8 */
}

void or_q4_dequantize(const uint8_t *wq, int M, int K, int GS, float *w) {
  const int ng = (K + GS - 1) / GS;
  for (int r = 0; r < M; ++r)
    for (int k = 0; k < K; ++k) w[(int64_t)r * K + k] = q4_at(wq, GS, ng, r, k);
}

void or_q4_0_dequantize(const uint8_t *wq, int M, int K, float *w) { or_q4_dequantize(wq, M, K, 32, w); }

/* int8 with one scale per row ([INFER] design notes, weight-only quantization: each
 * output row carries its own scale).
 * READING: s = max|w| / 127 in fp32; q = round-half-away(w / s) clamped to
 * [-127, 127]; a zero row has s = 0 and all q = 0. */
void or_i8_quantize(const float *w, int M, int K, int8_t *q, float *s) {
#pragma omp parallel for schedule(static) num_threads(g_threads) if (g_threads > 1) /* independent rows */
  for (int r = 0; r < M; ++r) {
    const float *row = w + (int64_t)r * K;
    float amax = 0.0f;
    for (int k = 0; k < K; ++k) amax = fmaxf(amax, fabsf(row[k]));
    const float sc = amax / 127.0f;
    s[r] = sc;
    for (int k = 0; k < K; ++k) {
      int c = 0;
      if (sc != 0.0f) {
        const float t = row[k] / sc;
        c = (int)roundf(t);
      }
      q[(int64_t)r * K + k] = (int8_t)(c < -127 ? -127 : (c > 127 ? 127 : c));
    }
  }
}

void or_i8_dequantize(const int8_t *q, const float *s, int M, int K, float *w) {
  for (int r = 0; r < M; ++r)
    for (int k = 0; k < K; ++k)
      w[(int64_t)r * K + k] = (float)((double)s[r] * (double)q[(int64_t)r * K + k]);
}

/* ------------------------------------------------------------------ GEMV */

/* y = W x for one storage format ([INFER] per-kernel table, "gemv"; [RUST] "Lesson 1").
 * Each output is the fp64 sum of (dequantised weight) * x over the row, rounded once
 * to fp32.  The int8 scale multiplies the row sum (y_i = s_i * sum_k q_ik x_k), which
 * equals sum_k (s_i q_ik) x_k exactly in real arithmetic.
 * Layouts: bf16 [M][K] uint16; i8 [M][K] int8 + s[M]; 4-bit canonical groups
 * [M][ng][2 + GS/2] (Q4_0: [M][nb][18]); f32 [M][K]. */
void or_gemv(int fmt, const void *W, const float *s, const float *x, int M, int K, float *y) {
  const int GS = or_q4_group(fmt), ng = GS ? (K + GS - 1) / GS : 0;
#pragma omp parallel for schedule(static) num_threads(g_threads) if (g_threads > 1 && M >= 64) /* independent rows */
  for (int r = 0; r < M; ++r) {
    double acc = 0.0;
    if (fmt == OR_BF16) {
      const uint16_t *row = (const uint16_t *)W + (int64_t)r * K;
      for (int k = 0; k < K; ++k) acc += (double)or_bf16_to_f32(row[k]) * (double)x[k];
    } else if (fmt == OR_I8) {
      const int8_t *row = (const int8_t *)W + (int64_t)r * K;
      for (int k = 0; k < K; ++k) acc += (double)row[k] * (double)x[k];
      acc *= (double)s[r];
    } else if (GS) {
      for (int k = 0; k < K; ++k) acc += (double)q4_at((const uint8_t *)W, GS, ng, r, k) * (double)x[k];
    } else {
      const float *row = (const float *)W + (int64_t)r * K;
      for (int k = 0; k < K; ++k) acc += (double)row[k] * (double)x[k];
    }
    y[r] = (float)acc;
  }
}

/* One row of the embedding table as fp32 (the gather at the start of the step,
 * [INFER] data-flow figure: the token's embedding row starts the fp32 residual). */
void or_embed_row(int fmt, const void *E, const float *s, int V, int d, int token, float *x) {
  (void)V;
  const int GS = or_q4_group(fmt), ng = GS ? (d + GS - 1) / GS : 0;
  for (int k = 0; k < d; ++k) {
    float v;
    if (fmt == OR_BF16) v = or_bf16_to_f32(((const uint16_t *)E)[(int64_t)token * d + k]);
    else if (fmt == OR_I8) v = (float)((double)s[token] * (double)((const int8_t *)E)[(int64_t)token * d + k]);
    else if (GS) v = q4_at((const uint8_t *)E, GS, ng, token, k);
    else v = ((const float *)E)[(int64_t)token * d + k];
    x[k] = v;
  }
}

/* ------------------------------------------------------------------ elementwise ops */

/* RMSNorm ([RUST] "How a Llama model generates text"; [INFER] design notes, fusion:
 * the norm is folded into the input staging of the next GEMV): out_i = x_i / sqrt(mean(x^2) + eps) * g_i. */
void or_rmsnorm(const float *x, const float *g, int n, float eps, float *out) {
  double ss = 0.0;
  for (int i = 0; i < n; ++i) ss += (double)x[i] * (double)x[i];
  const double r = 1.0 / sqrt(ss / (double)n + (double)eps);
  for (int i = 0; i < n; ++i) out[i] = (float)((double)x[i] * r * (double)g[i]);
}

/* RoPE angle tables ([RUST] "Lesson 4": angles depend only on the position and are
 * computed once per position).  READING: rotate-half pairing (i, i + hd/2),
 * theta_i = base^(-2i/hd), angle = pos * theta_i in fp64, cos and sin stored as fp32.
 * Output layout [n_pos][hd/2]. */
void or_rope_table(int n_pos, int hd, double base, float *cos_t, float *sin_t) {
  const int h2 = hd / 2;
  for (int p = 0; p < n_pos; ++p)
    for (int i = 0; i < h2; ++i) {
      const double inv = pow(base, -2.0 * (double)i / (double)hd);
      const double a = (double)p * inv;
      cos_t[(int64_t)p * h2 + i] = (float)cos(a);
      sin_t[(int64_t)p * h2 + i] = (float)sin(a);
    }
}

/* Rotate every head of v ([n_heads][hd]) by the angles of one position:
 * (a, b) = (v_i, v_{i+hd/2}) -> (a c - b s, b c + a s). */
void or_rope_apply(float *v, int n_heads, int hd, const float *c, const float *s) {
  const int h2 = hd / 2;
  for (int h = 0; h < n_heads; ++h)
    for (int i = 0; i < h2; ++i) {
      const double a = v[h * hd + i], b = v[h * hd + i + h2];
      v[h * hd + i] = (float)(a * c[i] - b * s[i]);
      v[h * hd + i + h2] = (float)(b * c[i] + a * s[i]);
    }
}

/* SwiGLU ([RUST] "How a Llama model generates text"; [INFER] design notes, fusion: the
 * gate and up rows are read as pairs): a_i = silu(g_i) * u_i, silu(z) = z / (1 + e^-z). */
void or_swiglu(const float *g, const float *u, int n, float *a) {
  for (int i = 0; i < n; ++i) {
    const double z = g[i];
    a[i] = (float)(z / (1.0 + exp(-z)) * (double)u[i]);
  }
}

/* Index of the largest value; the lowest index wins a tie (first maximum). */
int or_argmax(const float *v, int n) {
  int best = 0;
  for (int i = 1; i < n; ++i)
    if (v[i] > v[best]) best = i;
  return n > 0 ? best : -1;
}

/* ------------------------------------------------------------------ sampling */

/* splitmix64 (Steele, Lea & Flood, "Fast splittable pseudorandom number generators",
 * 2014): output i (0-based) of the stream started from `seed` -- the state advances by
 * the golden gamma 0x9E3779B97F4A7C15 before each output, then the finaliser mixes it. */
uint64_t or_splitmix64(uint64_t seed, uint64_t i) {
  uint64_t z = seed + (i + 1) * 0x9E3779B97F4A7C15ULL;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

/* READING: the random number of token i at position pos is (top 24 bits of splitmix64
 * output (pos << 32 | i) + 1/2) / 2^24, strictly inside (0, 1): one number per token of
 * each position, drawn from the seed alone, so a step's draw does not depend on any
 * other step. */
double or_sample_uniform(uint64_t seed, int pos, int i) {
  const uint64_t z = or_splitmix64(seed, ((uint64_t)(uint32_t)pos << 32) | (uint32_t)i);
  return ((double)(z >> 40) + 0.5) / 16777216.0;
}

typedef struct {
  float v;
  int i;
} or_ranked;

static int ranked_desc(const void *a, const void *b) {
  const or_ranked *x = (const or_ranked *)a, *y = (const or_ranked *)b;
  if (x->v != y->v) return x->v > y->v ? -1 : 1;
  return x->i - y->i;
}

/* Temperature / top-k / top-p sampling ([INFER] design notes: sampling on the GPU with
 * radix select for the top-k and top-p cut-offs and per-position random numbers from a
 * seed, so runs reproduce).
 * READING: temperature T <= 0 is greedy (argmax).  Otherwise, with q_i = exp((l_i - max)
 * / T): top-k keeps the tokens whose logit is at least the k-th largest logit (every
 * token tied with it too; k <= 0 or k >= n keeps all); top-p then keeps, of those, the
 * tokens whose logit is at least the largest value t for which the kept tokens with
 * logit >= t hold at least p of the kept mass sum q (ties at t kept; p >= 1 keeps all);
 * the token is drawn from the kept tokens' renormalised distribution by the Gumbel-max
 * rule -- argmax over kept i of l_i / T - log(-log(u_i)), u_i = or_sample_uniform(seed,
 * pos, i), lowest index on ties -- which picks token i with probability q_i / sum q over
 * the kept set.  Plain definition: a full sort, fp64 masses in descending order. */
int or_sample(const float *logits, int n, float T, int top_k, float top_p, uint64_t seed, int pos) {
  if (n <= 0) return -1;
  if (!(T > 0.0f)) return or_argmax(logits, n);
  or_ranked *r = (or_ranked *)malloc(sizeof(or_ranked) * (size_t)n);
  for (int i = 0; i < n; ++i) { r[i].v = logits[i]; r[i].i = i; }
  qsort(r, (size_t)n, sizeof(or_ranked), ranked_desc);
  const double mx = r[0].v;
  int kept = n;
  if (top_k > 0 && top_k < n) {
    const float tk = r[top_k - 1].v;
    kept = top_k;
    while (kept < n && r[kept].v == tk) ++kept;
  }
  if (top_p < 1.0f) {
    double z = 0.0;
    for (int j = 0; j < kept; ++j) z += exp(((double)r[j].v - mx) / (double)T);
    const double target = (double)top_p * z;
    double cum = 0.0;
    int j = 0;
    for (; j < kept; ++j) {
      cum += exp(((double)r[j].v - mx) / (double)T);
      if (cum >= target) break;
    }
    if (j >= kept) j = kept - 1;
    const float tp = r[j].v;
    int k2 = j + 1;
    while (k2 < kept && r[k2].v == tp) ++k2;
    kept = k2;
  }
  int best = -1;
  double bs = -INFINITY;
  for (int j = 0; j < kept; ++j) {
    const int i = r[j].i;
    const double sc = (double)logits[i] / (double)T - log(-log(or_sample_uniform(seed, pos, i)));
    if (sc > bs || (sc == bs && i < best)) { bs = sc; best = i; }
  }
  free(r);
  return best;
}

/* ------------------------------------------------------------------ attention */

/* Softmax attention of one query head over t = 0..ctx-1 with keys/values supplied by
 * a lookup; plain two-pass softmax in fp64. */
typedef const uint16_t *(*kv_lookup)(const void *ctx, int which, int g, int t);

static void attend_head(const float *qh, int hd, int ctx, int g, double scale, kv_lookup look,
                        const void *lc, float *out, double *score) {
  if (ctx <= 0) { /* READING: an empty context yields a zero output */
    for (int d = 0; d < hd; ++d) out[d] = 0.0f;
    return;
  }
  double mx = -INFINITY;
  for (int t = 0; t < ctx; ++t) {
    const uint16_t *k = look(lc, 0, g, t);
    double dot = 0.0;
    for (int d = 0; d < hd; ++d) dot += (double)qh[d] * (double)or_bf16_to_f32(k[d]);
    score[t] = dot * scale;
    if (score[t] > mx) mx = score[t];
  }
  double l = 0.0;
  for (int t = 0; t < ctx; ++t) { score[t] = exp(score[t] - mx); l += score[t]; }
  for (int d = 0; d < hd; ++d) {
    double o = 0.0;
    for (int t = 0; t < ctx; ++t) o += score[t] * (double)or_bf16_to_f32(look(lc, 1, g, t)[d]);
    out[d] = (float)(o / l);
  }
}

typedef struct {
  const uint16_t *k, *v;
  int64_t block_stride;
  const int32_t *bt;
  int bs, hd;
} paged_view;

static const uint16_t *paged_look(const void *c, int which, int g, int t) {
  const paged_view *p = (const paged_view *)c;
  const int64_t blk = p->bt[t / p->bs];
  const uint16_t *base = which ? p->v : p->k;
  return base + blk * p->block_stride + ((int64_t)g * p->bs + (t % p->bs)) * p->hd;
}

/* Paged GQA decode attention ([MIE] "The KV cache, paged like virtual memory": a block
 * table maps logical positions to physical 16-token blocks; [INFER] design notes, the
 * split-KV attention item; [RUST] "Lesson 4": query heads sharing a KV head).  Query head h reads KV
 * head h / (Hq/Hkv).  Key t of KV head g lives in physical block bt[t / bs], slot t % bs:
 * element d at k_pool[blk * block_stride + (g * bs + t % bs) * hd + d] (bf16); the same
 * for v_pool.  out[h][d] = sum_t softmax_t(scale * q_h . k_t) v_t[d]. */
void or_attention_paged(const float *q, const uint16_t *k_pool, const uint16_t *v_pool,
                        int64_t block_stride, const int32_t *block_table, int ctx, int Hq,
                        int Hkv, int hd, int bs, float scale, float *out) {
  paged_view pv = {k_pool, v_pool, block_stride, block_table, bs, hd};
  const int64_t per_head = ctx > 0 ? ctx : 1;
  double *score = (double *)malloc(sizeof(double) * (size_t)(per_head * Hq));
  const int group = Hq / Hkv;
#pragma omp parallel for schedule(static) num_threads(g_threads) if (g_threads > 1) /* independent heads */
  for (int h = 0; h < Hq; ++h)
    attend_head(q + h * hd, hd, ctx, h / group, (double)scale, paged_look, &pv, out + h * hd,
                score + h * per_head);
  free(score);
}

typedef struct {
  const uint16_t *k, *v;
  int Hkv, hd;
} contig_view;

static const uint16_t *contig_look(const void *c, int which, int g, int t) {
  const contig_view *p = (const contig_view *)c;
  return (which ? p->v : p->k) + ((int64_t)t * p->Hkv + g) * p->hd;
}

/* The same attention over a contiguous cache k[t][g][d], v[t][g][d] (bf16). */
void or_attention_contig(const float *q, const uint16_t *k, const uint16_t *v, int ctx, int Hq,
                         int Hkv, int hd, float scale, float *out) {
  contig_view cv = {k, v, Hkv, hd};
  double *score = (double *)malloc(sizeof(double) * (ctx > 0 ? ctx : 1));
  const int group = Hq / Hkv;
  for (int h = 0; h < Hq; ++h)
    attend_head(q + h * hd, hd, ctx, h / group, (double)scale, contig_look, &cv, out + h * hd, score);
  free(score);
}

/* ------------------------------------------------------------------ block pool */

/* Paged KV block pool with reference counts and copy-on-write ([MIE] "The KV cache,
 * paged like virtual memory" and "Prefix sharing and copy-on-write"): one arena
 * allocated up front, a refcount per block id, a LIFO free list; an exhausted pool
 * returns the sentinel -1 instead of failing.  READING: the free list starts as
 * n-1 .. 0 so that a fresh pool hands out 0, 1, 2, ... */
typedef struct {
  int n_blocks;
  int64_t bytes_per_block;
  uint8_t *arena;
  int *refcount;
  int *free_list;
  int n_free;
} or_pool;

or_pool *or_pool_create(int n_blocks, int64_t bytes_per_block) {
  or_pool *p = (or_pool *)calloc(1, sizeof(or_pool));
  p->n_blocks = n_blocks;
  p->bytes_per_block = bytes_per_block;
  p->arena = (uint8_t *)calloc((size_t)n_blocks * (size_t)bytes_per_block + 1, 1);
  p->refcount = (int *)calloc((size_t)n_blocks + 1, sizeof(int));
  p->free_list = (int *)calloc((size_t)n_blocks + 1, sizeof(int));
  for (int i = 0; i < n_blocks; ++i) p->free_list[i] = n_blocks - 1 - i;
  p->n_free = n_blocks;
  return p;
}

void or_pool_destroy(or_pool *p) {
  if (!p) return;
  free(p->arena); free(p->refcount); free(p->free_list); free(p);
}

int or_pool_alloc(or_pool *p) {
  if (p->n_free == 0) return -1;
  const int id = p->free_list[--p->n_free];
  p->refcount[id] = 1;
  return id;
}

static int pool_valid(const or_pool *p, int id) { return id >= 0 && id < p->n_blocks && p->refcount[id] > 0; }

int or_pool_incref(or_pool *p, int id) {
  if (!pool_valid(p, id)) return -1;
  return ++p->refcount[id];
}

/* Drops one reference; a block whose count reaches 0 goes back on the free list.
 * Returns the new count, or -1 for an id that is not live. */
int or_pool_decref(or_pool *p, int id) {
  if (!pool_valid(p, id)) return -1;
  if (--p->refcount[id] == 0) p->free_list[p->n_free++] = id;
  return p->refcount[id];
}

int or_pool_refcount(const or_pool *p, int id) { return (id >= 0 && id < p->n_blocks) ? p->refcount[id] : -1; }
int or_pool_free_count(const or_pool *p) { return p->n_free; }
uint8_t *or_pool_data(or_pool *p, int id) { return p->arena + (int64_t)id * p->bytes_per_block; }

/* The block that a write at logical position `pos` may go to.  A private block
 * (refcount 1) is returned as is; a shared one is split: allocate, copy the contents,
 * drop one reference to the old block, then point the table at the copy -- in that
 * order, so the source stays alive during the copy.  -1 when the pool is exhausted. */
int or_table_writable(or_pool *p, int32_t *table, int pos, int block_size) {
  const int old = table[pos / block_size];
  if (!pool_valid(p, old)) return -1;
  if (p->refcount[old] == 1) return old;
  const int nw = or_pool_alloc(p);
  if (nw < 0) return -1;
  memcpy(or_pool_data(p, nw), or_pool_data(p, old), (size_t)p->bytes_per_block);
  or_pool_decref(p, old);
  table[pos / block_size] = nw;
  return nw;
}

/* ------------------------------------------------------------------ the model */

/* Decode step of a Llama-style GQA decoder ([RUST] "How a Llama model generates text";
 * [INFER] data-flow figure):
 *   x = E[token]
 *   per layer: q|k|v = Wqkv rmsnorm(x); rope(q, k); cache <- bf16(k), bf16(v) at pos;
 *              o = attention(q, cache[0..pos]); x += Wo o;
 *              a = silu(Wg rmsnorm(x)) * (Wu rmsnorm(x)); x += Wd a
 *   logits = Whead rmsnorm(x); token' = argmax(logits)
 * READING: the token at 0-based position pos writes its K/V at slot pos and attends to
 * positions 0..pos (ctx = pos + 1); scale = fp32(1/sqrt(hd)).  With act_bf16 every GEMV
 * input vector (the normed x, the attention output, a) is rounded to bf16 before the
 * product; the residual stream stays fp32.
 * KV pool layout: [n_blocks][n_layers][2 (k, v)][Hkv][block_size][hd] bf16. */
typedef struct {
  int n_layers, d_model, n_heads, n_kv_heads, head_dim, ffn, vocab, block_size, act_bf16;
  float rms_eps;
  double rope_theta;
} or_config;

typedef struct {
  int fmt;
  const void *w;
  const float *s;
  int rows, cols;
} or_mat;

enum { T_QKV = 0, T_O, T_GATE, T_UP, T_DOWN, T_NORM_ATTN, T_NORM_MLP, T_PER_LAYER };

typedef struct {
  or_config c;
  or_mat *layer; /* [n_layers][T_PER_LAYER] */
  or_mat head, embed, norm_final;
  uint16_t *kv;
  int n_kv_blocks, max_pos;
  float *cos_t, *sin_t;
} or_model;

or_model *or_model_create(const or_config *c, int n_kv_blocks, int max_pos) {
  or_model *m = (or_model *)calloc(1, sizeof(or_model));
  m->c = *c;
  m->layer = (or_mat *)calloc((size_t)c->n_layers * T_PER_LAYER, sizeof(or_mat));
  m->n_kv_blocks = n_kv_blocks;
  m->max_pos = max_pos;
  const int64_t per_block = (int64_t)c->n_layers * 2 * c->n_kv_heads * c->block_size * c->head_dim;
  m->kv = (uint16_t *)calloc((size_t)(n_kv_blocks * per_block + 1), sizeof(uint16_t));
  m->cos_t = (float *)malloc(sizeof(float) * (size_t)max_pos * (c->head_dim / 2));
  m->sin_t = (float *)malloc(sizeof(float) * (size_t)max_pos * (c->head_dim / 2));
  or_rope_table(max_pos, c->head_dim, c->rope_theta, m->cos_t, m->sin_t);
  return m;
}

void or_model_destroy(or_model *m) {
  if (!m) return;
  free(m->layer); free(m->kv); free(m->cos_t); free(m->sin_t); free(m);
}

int64_t or_model_block_elems(const or_model *m) {
  return (int64_t)m->c.n_layers * 2 * m->c.n_kv_heads * m->c.block_size * m->c.head_dim;
}

uint16_t *or_model_kv(or_model *m) { return m->kv; }

/* Attach a caller-owned weight (the oracle keeps the pointer, not a copy).
 * which: 0 qkv, 1 o, 2 gate, 3 up, 4 down, 5 attention-norm gain, 6 MLP-norm gain
 * (per layer); 100 LM head, 101 embedding, 102 final-norm gain. */
int or_model_set(or_model *m, int which, int layer, int fmt, const void *w, const float *s,
                 int rows, int cols) {
  or_mat t = {fmt, w, s, rows, cols};
  if (which >= 0 && which < T_PER_LAYER) {
    if (layer < 0 || layer >= m->c.n_layers) return -1;
    m->layer[layer * T_PER_LAYER + which] = t;
  } else if (which == 100) m->head = t;
  else if (which == 101) m->embed = t;
  else if (which == 102) m->norm_final = t;
  else return -1;
  return 0;
}

static void gemv_mat(const or_mat *t, const float *x, float *y) { or_gemv(t->fmt, t->w, t->s, x, t->rows, t->cols, y); }

static void maybe_bf16(const or_model *m, float *v, int n) {
  if (!m->c.act_bf16) return;
  for (int i = 0; i < n; ++i) v[i] = or_bf16_to_f32(or_f32_to_bf16(v[i]));
}

static void add_into(float *x, const float *y, int n) {
  for (int i = 0; i < n; ++i) x[i] = x[i] + y[i];
}

/* The MLP half of a layer: x += Wd (silu(Wg n(x)) * Wu n(x)). */
static void mlp_block(const or_model *m, int l, float *x, float *xn, float *g, float *u, float *tmp) {
  const or_config *c = &m->c;
  const or_mat *L = m->layer + l * T_PER_LAYER;
  or_rmsnorm(x, (const float *)L[T_NORM_MLP].w, c->d_model, c->rms_eps, xn);
  maybe_bf16(m, xn, c->d_model);
  gemv_mat(&L[T_GATE], xn, g);
  gemv_mat(&L[T_UP], xn, u);
  or_swiglu(g, u, c->ffn, g);
  maybe_bf16(m, g, c->ffn);
  gemv_mat(&L[T_DOWN], g, tmp);
  add_into(x, tmp, c->d_model);
}

static void head_block(const or_model *m, const float *x, float *xn, float *logits) {
  const or_config *c = &m->c;
  or_rmsnorm(x, (const float *)m->norm_final.w, c->d_model, c->rms_eps, xn);
  maybe_bf16(m, xn, c->d_model);
  gemv_mat(&m->head, xn, logits);
}

typedef struct { float *x, *xn, *qkv, *att, *g, *u, *tmp; } scratch;

static scratch scratch_new(const or_config *c) {
  scratch s;
  const int qkv = (c->n_heads + 2 * c->n_kv_heads) * c->head_dim;
  s.x = malloc(sizeof(float) * c->d_model);
  s.xn = malloc(sizeof(float) * (c->d_model > c->ffn ? c->d_model : c->ffn));
  s.qkv = malloc(sizeof(float) * qkv);
  s.att = malloc(sizeof(float) * c->n_heads * c->head_dim);
  s.g = malloc(sizeof(float) * c->ffn);
  s.u = malloc(sizeof(float) * c->ffn);
  s.tmp = malloc(sizeof(float) * c->d_model);
  return s;
}

static void scratch_free(scratch *s) {
  free(s->x); free(s->xn); free(s->qkv); free(s->att); free(s->g); free(s->u); free(s->tmp);
}

/* One decode step with the paged cache.  Returns argmax(logits), or -1 on a bad
 * argument (position out of range, block id outside the pool). */
int or_decode_step(or_model *m, int token, int pos, const int32_t *block_table, int n_table,
                   float *logits) {
  const or_config *c = &m->c;
  if (pos < 0 || pos >= m->max_pos || pos / c->block_size >= n_table) return -1;
  for (int i = 0; i <= pos / c->block_size; ++i)
    if (block_table[i] < 0 || block_table[i] >= m->n_kv_blocks) return -1;
  if (token < 0 || token >= c->vocab) return -1;
  const int d = c->d_model, hd = c->head_dim, Hq = c->n_heads, Hkv = c->n_kv_heads;
  const int h2 = hd / 2;
  const int64_t blk_elems = or_model_block_elems(m);
  const int64_t kv_half = (int64_t)Hkv * c->block_size * hd; /* one of k or v, one layer */
  const float scale = (float)(1.0 / sqrt((double)hd));
  scratch s = scratch_new(c);
  or_embed_row(m->embed.fmt, m->embed.w, m->embed.s, c->vocab, d, token, s.x);
  for (int l = 0; l < c->n_layers; ++l) {
    const or_mat *L = m->layer + l * T_PER_LAYER;
    or_rmsnorm(s.x, (const float *)L[T_NORM_ATTN].w, d, c->rms_eps, s.xn);
    maybe_bf16(m, s.xn, d);
    gemv_mat(&L[T_QKV], s.xn, s.qkv);
    float *q = s.qkv, *k = s.qkv + Hq * hd, *v = k + Hkv * hd;
    or_rope_apply(q, Hq, hd, m->cos_t + (int64_t)pos * h2, m->sin_t + (int64_t)pos * h2);
    or_rope_apply(k, Hkv, hd, m->cos_t + (int64_t)pos * h2, m->sin_t + (int64_t)pos * h2);
    const int64_t blk = block_table[pos / c->block_size];
    uint16_t *kl = m->kv + blk * blk_elems + (int64_t)l * 2 * kv_half;
    uint16_t *vl = kl + kv_half;
    for (int g = 0; g < Hkv; ++g)
      for (int e = 0; e < hd; ++e) {
        const int64_t off = ((int64_t)g * c->block_size + pos % c->block_size) * hd + e;
        kl[off] = or_f32_to_bf16(k[g * hd + e]);
        vl[off] = or_f32_to_bf16(v[g * hd + e]);
      }
    or_attention_paged(q, m->kv + (int64_t)l * 2 * kv_half, m->kv + (int64_t)l * 2 * kv_half + kv_half,
                       blk_elems, block_table, pos + 1, Hq, Hkv, hd, c->block_size, scale, s.att);
    maybe_bf16(m, s.att, Hq * hd);
    gemv_mat(&L[T_O], s.att, s.tmp);
    add_into(s.x, s.tmp, d);
    mlp_block(m, l, s.x, s.xn, s.g, s.u, s.tmp);
  }
  head_block(m, s.x, s.xn, logits);
  scratch_free(&s);
  return or_argmax(logits, c->vocab);
}

/* The same model run without a cache: all n tokens are pushed through every layer
 * with causal attention over contiguous K/V (rounded to bf16 as the cache rounds
 * them), and the logits of the last position are returned.  Used to pin the cache
 * plumbing: incremental decode must give the same bits. */
int or_forward_nocache(const or_model *m, const int32_t *tokens, int n, float *logits) {
  const or_config *c = &m->c;
  if (n <= 0 || n > m->max_pos) return -1;
  const int d = c->d_model, hd = c->head_dim, Hq = c->n_heads, Hkv = c->n_kv_heads, h2 = hd / 2;
  const int nq = (Hq + 2 * Hkv) * hd;
  const float scale = (float)(1.0 / sqrt((double)hd));
  float *X = malloc(sizeof(float) * (size_t)n * d);
  float *QKV = malloc(sizeof(float) * (size_t)n * nq);
  uint16_t *K = malloc(sizeof(uint16_t) * (size_t)n * Hkv * hd);
  uint16_t *V = malloc(sizeof(uint16_t) * (size_t)n * Hkv * hd);
  scratch s = scratch_new(c);
  for (int t = 0; t < n; ++t) {
    if (tokens[t] < 0 || tokens[t] >= c->vocab) { n = -1; break; }
    or_embed_row(m->embed.fmt, m->embed.w, m->embed.s, c->vocab, d, tokens[t], X + (int64_t)t * d);
  }
  if (n < 0) { free(X); free(QKV); free(K); free(V); scratch_free(&s); return -1; }
  for (int l = 0; l < c->n_layers; ++l) {
    const or_mat *L = m->layer + l * T_PER_LAYER;
    for (int t = 0; t < n; ++t) {
      float *qkv = QKV + (int64_t)t * nq;
      or_rmsnorm(X + (int64_t)t * d, (const float *)L[T_NORM_ATTN].w, d, c->rms_eps, s.xn);
      maybe_bf16(m, s.xn, d);
      gemv_mat(&L[T_QKV], s.xn, qkv);
      or_rope_apply(qkv, Hq, hd, m->cos_t + (int64_t)t * h2, m->sin_t + (int64_t)t * h2);
      or_rope_apply(qkv + Hq * hd, Hkv, hd, m->cos_t + (int64_t)t * h2, m->sin_t + (int64_t)t * h2);
      for (int e = 0; e < Hkv * hd; ++e) {
        K[(int64_t)t * Hkv * hd + e] = or_f32_to_bf16(qkv[Hq * hd + e]);
        V[(int64_t)t * Hkv * hd + e] = or_f32_to_bf16(qkv[Hq * hd + Hkv * hd + e]);
      }
    }
    for (int t = 0; t < n; ++t) {
      float *x = X + (int64_t)t * d;
      or_attention_contig(QKV + (int64_t)t * nq, K, V, t + 1, Hq, Hkv, hd, scale, s.att);
      maybe_bf16(m, s.att, Hq * hd);
      gemv_mat(&L[T_O], s.att, s.tmp);
      add_into(x, s.tmp, d);
      mlp_block(m, l, x, s.xn, s.g, s.u, s.tmp);
    }
  }
  head_block(m, X + (int64_t)(n - 1) * d, s.xn, logits);
  const int best = or_argmax(logits, c->vocab);
  free(X); free(QKV); free(K); free(V); scratch_free(&s);
  return best;
}

/* Few-slot step ([MIE] "Continuous batching"): every slot advances one token; the
 * result of the batched step is defined as that of independent single-slot steps,
 * each through its own block table (row s of block_tables, max_blocks wide). */
int or_decode_step_slots(or_model *m, int n_slots, const int32_t *tokens, const int32_t *pos,
                         const int32_t *block_tables, int max_blocks, float *logits, int32_t *argmax_out) {
  for (int sl = 0; sl < n_slots; ++sl) {
    const int r = or_decode_step(m, tokens[sl], pos[sl], block_tables + (int64_t)sl * max_blocks, max_blocks,
                                 logits + (int64_t)sl * m->c.vocab);
    if (r < 0) return -1;
    argmax_out[sl] = r;
  }
  return 0;
}
