// probe.cu -- the read-only streaming-bandwidth probe.
//
// The "infer" page states every kernel's speed as a fraction of a bandwidth it
// measured itself with a read probe, not of the datasheet figure.  This kernel is that
// probe for this GPU: it reads every byte of a device buffer exactly once and writes
// almost nothing, so the bytes moved are the buffer's size.  Each word is folded into
// an XOR (one atomicXor per CTA at the end), which keeps the loads from being removed
// and gives a result that can be checked exactly against the host.
//
// Loads bypass L1 (no_allocate) and are marked evict-first in L2; the caller passes a
// buffer many times larger than L2, so the figure is HBM's.  The grid is a multiple of
// the SM count with a grid-stride loop; each thread keeps W independent loads in flight.
#include "common.cuh"

namespace mie {

__device__ __forceinline__ uint32_t ld16_xor(const uint8_t *p, uint64_t pol) {
  uint32_t a, b, c, d;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
               : "=r"(a), "=r"(b), "=r"(c), "=r"(d)
               : "l"(p), "l"(pol));
  return a ^ b ^ c ^ d;
}

__device__ __forceinline__ uint32_t ld32_xor(const uint8_t *p, uint64_t pol) {
  uint32_t r[8];
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8], %9;"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "l"(p), "l"(pol));
  return r[0] ^ r[1] ^ r[2] ^ r[3] ^ r[4] ^ r[5] ^ r[6] ^ r[7];
}

constexpr int kProbeThreads = 512;

// WB: bytes per load (16 or 32).  n: number of WB-byte words.
template <int WB>
__global__ void __launch_bounds__(kProbeThreads) read_probe_kernel(const uint8_t *__restrict__ src, uint64_t n,
                                                                  uint32_t *out) {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  constexpr int W = 4;  // loads in flight per thread
  uint32_t acc = 0;
  const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
  for (; i + (W - 1) * stride < n; i += W * stride) {
    uint32_t v[W];
#pragma unroll
    for (int j = 0; j < W; ++j)
      v[j] = (WB == 32) ? ld32_xor(src + 32 * (i + j * stride), pol) : ld16_xor(src + 16 * (i + j * stride), pol);
#pragma unroll
    for (int j = 0; j < W; ++j) acc ^= v[j];
  }
  for (; i < n; i += stride) acc ^= (WB == 32) ? ld32_xor(src + 32 * i, pol) : ld16_xor(src + 16 * i, pol);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc ^= __shfl_xor_sync(0xffffffffu, acc, o);
  __shared__ uint32_t red[kProbeThreads / 32];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t t = 0;
    for (int w = 0; w < kProbeThreads / 32; ++w) t ^= red[w];
    atomicXor(out, t);
  }
}

int sm_count();

}  // namespace mie

using namespace mie;

extern "C" mie_status mie_hbm_read_probe(const void *buf, size_t bytes, uint32_t *xor_out, int load_bytes,
                                         int blocks_per_sm, void *stream) {
  if (!buf || !xor_out) return fail(MIE_E_ARG, "mie_hbm_read_probe: null pointer");
  if (load_bytes != 16 && load_bytes != 32) return fail(MIE_E_ARG, "mie_hbm_read_probe: load_bytes %d", load_bytes);
  if (blocks_per_sm < 1 || blocks_per_sm > 4)
    return fail(MIE_E_ARG, "mie_hbm_read_probe: blocks_per_sm %d outside [1, 4]", blocks_per_sm);
  if (bytes == 0 || bytes % (size_t)load_bytes || (uintptr_t)buf % (uintptr_t)load_bytes || (uintptr_t)xor_out % 4)
    return fail(MIE_E_SHAPE, "mie_hbm_read_probe: %zu bytes at %p are not whole aligned %d-byte words", bytes, buf,
                load_bytes);
  cudaStream_t st = (cudaStream_t)stream;
  MIE_CUDA(cudaMemsetAsync(xor_out, 0, sizeof(uint32_t), st));
  const int grid = sm_count() * blocks_per_sm;
  const uint8_t *src = static_cast<const uint8_t *>(buf);
  if (load_bytes == 32) read_probe_kernel<32><<<grid, kProbeThreads, 0, st>>>(src, bytes / 32, xor_out);
  else read_probe_kernel<16><<<grid, kProbeThreads, 0, st>>>(src, bytes / 16, xor_out);
  MIE_CUDA(cudaGetLastError());
  return MIE_OK;
}
