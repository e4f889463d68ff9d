// common.cuh -- helpers shared by the CUDA translation units of libmie.so.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "../../include/mie.h"

namespace mie {

// ----------------------------------------------------------------- host error state

void set_error(const char *fmt, ...);
mie_status fail(mie_status s, const char *fmt, ...);
mie_status cuda_fail(cudaError_t e, const char *what);

#define MIE_CUDA(call)                                           \
  do {                                                           \
    cudaError_t e_ = (call);                                     \
    if (e_ != cudaSuccess) return ::mie::cuda_fail(e_, #call);   \
  } while (0)

// Device error flag of the current device for the stateless kernels.
int *device_error_flag();

// ----------------------------------------------------------------- device helpers

// Kernels are launched with programmatic dependent launch inside the step graph:
// everything before pdl_wait() may only read data no earlier kernel writes (weights,
// tables); pdl_trigger() lets the next kernel start its own weight prefetch.  Both
// are no-ops for a kernel launched without the attribute.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ uint16_t ldg_u16(const void *p) {
  uint16_t v;
  asm volatile("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float bf16_bits_to_f32(uint16_t h) { return __uint_as_float((uint32_t)h << 16); }

__device__ __forceinline__ float round_bf16(float v) { return __bfloat162float(__float2bfloat16_rn(v)); }

__device__ __forceinline__ void latch_error(int *flag, int code) {
  if (flag) atomicOr(flag, code);
}

// Device error codes latched by bounds checks.
enum : int { ERR_BLOCK_ID = 1, ERR_POS = 2, ERR_TOKEN = 4, ERR_TIMEOUT = 8 };

// ----------------------------------------------------------------- step parameters

// Per-step values the captured graph reads from device memory, so one graph serves
// every step; the host rewrites them before a replay, or the LM-head kernel advances
// them (token = argmax, pos + 1) for a device-side greedy continuation.
constexpr int kMaxSlots = 8;
struct StepParams {
  int32_t token[kMaxSlots];
  int32_t pos[kMaxSlots];
  const int32_t *block_table;  // [n_slots][max_blocks]
  int32_t max_blocks;
  int32_t n_slots;
  float *logits_out;           // [n_slots][vocab] or null
  int32_t *argmax_out;         // [n_slots] or null
  int32_t advance;             // 1: the head kernel sets token = argmax, pos += 1
  int32_t sample_advance;      // 1: the sampler sets token = its draw, pos += 1 (advance is 0 then)
  int32_t pad[2];
};

}  // namespace mie
