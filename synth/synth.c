/*
 * synth.c -- seeded synthetic inputs shared by the oracle, the tests and the bench.
 *
 * This file holds random-number generation only: none of the decode step's
 * arithmetic (no quantisation, no rounding to bf16/f16, no GEMV) lives here, so
 * the oracle and the CUDA path can both draw their inputs from it without sharing
 * any part of the method.
 *
 * Generator: splitmix64 (Steele, Lea & Flood, "Fast splittable pseudorandom number
 * generators", OOPSLA 2014).  Output i of a stream with seed s is
 * mix(s + (i + 1) * 0x9E3779B97F4A7C15), so every element can be drawn on its own
 * (counter-based): the result does not depend on how the work is split between
 * threads, and one row of a large tensor can be regenerated without the others.
 *
 * Normal variates: Box-Muller (Box & Muller 1958) in double precision.  Element e
 * of a normal stream uses outputs 2*(e/2) and 2*(e/2)+1 of the integer stream:
 * u1 = (h1 >> 11 + 1) * 2^-53 in (0, 1], u2 = (h2 >> 11) * 2^-53 in [0, 1),
 * r = sqrt(-2 ln u1); even e takes r cos(2 pi u2), odd e takes r sin(2 pi u2).
 * The stored value is (float)(mean + std * z).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define GOLDEN 0x9E3779B97F4A7C15ULL

static inline uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

/* Output number i (0-based) of the splitmix64 stream started from seed. */
uint64_t synth_u64(uint64_t seed, uint64_t i) { return mix64(seed + (i + 1) * GOLDEN); }

static inline double normal_at(uint64_t seed, uint64_t e) {
  const uint64_t p = e >> 1;
  const uint64_t h1 = synth_u64(seed, 2 * p);
  const uint64_t h2 = synth_u64(seed, 2 * p + 1);
  const double u1 = ((double)(h1 >> 11) + 1.0) * (1.0 / 9007199254740992.0);
  const double u2 = (double)(h2 >> 11) * (1.0 / 9007199254740992.0);
  const double r = sqrt(-2.0 * log(u1));
  const double a = 6.283185307179586476925286766559 * u2;
  return (e & 1) ? r * sin(a) : r * cos(a);
}

typedef struct {
  uint64_t seed, offset, begin, end;
  double mean, std;
  float *out;
} normal_job;

static void *normal_worker(void *arg) {
  normal_job *j = (normal_job *)arg;
  for (uint64_t k = j->begin; k < j->end; ++k)
    j->out[k] = (float)(j->mean + j->std * normal_at(j->seed, j->offset + k));
  return NULL;
}

/* out[k] = N(mean, std) element (offset + k) of stream `seed`, k < n. */
void synth_normal_f32(uint64_t seed, uint64_t offset, uint64_t n, double mean, double std,
                      float *out, int threads) {
  if (threads < 1) threads = 1;
  if (threads > 256) threads = 256;
  if (n < (1u << 16)) threads = 1;
  normal_job jobs[256];
  pthread_t tid[256];
  int joined[256] = {0};
  for (int t = 0; t < threads; ++t) {
    jobs[t].seed = seed;
    jobs[t].offset = offset;
    jobs[t].begin = n * (uint64_t)t / (uint64_t)threads;
    jobs[t].end = n * (uint64_t)(t + 1) / (uint64_t)threads;
    jobs[t].mean = mean;
    jobs[t].std = std;
    jobs[t].out = out;
  }
  for (int t = 1; t < threads; ++t) {
    if (pthread_create(&tid[t], NULL, normal_worker, &jobs[t]) == 0)
      joined[t] = 1;
    else
      normal_worker(&jobs[t]); /* no thread available: do the share here */
  }
  normal_worker(&jobs[0]);
  for (int t = 1; t < threads; ++t)
    if (joined[t]) pthread_join(tid[t], NULL);
}

/* out[k] = lo + floor(((h >> 32) * (hi - lo)) / 2^32) for output (offset + k) of
 * stream `seed`: integers in [lo, hi) (hi > lo, hi - lo < 2^32). */
void synth_uniform_i32(uint64_t seed, uint64_t offset, uint64_t n, int32_t lo, int32_t hi,
                       int32_t *out) {
  const uint64_t range = (uint64_t)((int64_t)hi - (int64_t)lo);
  for (uint64_t k = 0; k < n; ++k) {
    const uint64_t h = synth_u64(seed, offset + k) >> 32;
    out[k] = (int32_t)((int64_t)lo + (int64_t)((h * range) >> 32));
  }
}

/* A permutation of 0..n-1: Fisher-Yates (Durstenfeld) driven by stream `seed`. */
void synth_permutation(uint64_t seed, int32_t n, int32_t *out) {
  for (int32_t i = 0; i < n; ++i) out[i] = i;
  for (int32_t i = n - 1; i > 0; --i) {
    const uint64_t h = synth_u64(seed, (uint64_t)(n - 1 - i)) >> 32;
    const int32_t j = (int32_t)((h * (uint64_t)(i + 1)) >> 32);
    const int32_t t = out[i];
    out[i] = out[j];
    out[j] = t;
  }
}
