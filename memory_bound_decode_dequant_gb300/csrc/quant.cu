// quant.cu -- load-time quantisation and packing kernels, RoPE tables.
//
// Q4_0 ("Writing an LLM inference engine from scratch in Rust", Lesson 1 and "Is the
// 4-bit model still good?"; "infer" page, weight-only quantization): blocks of 32,
// scale from the element of largest magnitude with its sign kept, divided by -8 so
// that element lands exactly on code 0 (-8), stored as f16.  int8: one scale per row.
// Every rounding step is an explicit single-rounding intrinsic so the bytes are the
// same on any compiler setting.
#include "internal.h"

namespace mie {

__global__ void convert_bf16_kernel(const float *w, int64_t n, uint16_t *out) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
    out[i] = __bfloat16_as_ushort(__float2bfloat16_rn(w[i]));
}

// One warp per row: max |w| (order-independent, so exact), s = max / 127, then codes.
__global__ void quantize_i8_kernel(const float *w, int M, int K, int8_t *q, float *s) {
  const int warp = (int)(((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5), lane = threadIdx.x & 31;
  if (warp >= M) return;
  const float *row = w + (int64_t)warp * K;
  float amax = 0.f;
  for (int k = lane; k < K; k += 32) amax = fmaxf(amax, fabsf(row[k]));
  amax = warp_max(amax);
  const float sc = __fdiv_rn(amax, 127.0f);
  if (lane == 0) s[warp] = sc;
  for (int k = lane; k < K; k += 32) {
    int c = 0;
    if (sc != 0.f) c = (int)roundf(__fdiv_rn(row[k], sc));
    q[(int64_t)warp * K + k] = (int8_t)(c < -127 ? -127 : (c > 127 ? 127 : c));
  }
}

// One thread per 32-weight block; canonical output [M][nb][18].
__global__ void quantize_q4_0_kernel(const float *w, int M, int K, uint8_t *out) {
  const int nb = (K + 31) / 32;
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (int64_t)M * nb) return;
  const int r = (int)(idx / nb), b = (int)(idx % nb);
  float v[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    const int k = b * 32 + j;
    v[j] = (k < K) ? w[(int64_t)r * K + k] : 0.f;
  }
  float amax = 0.f, m = 0.f;
#pragma unroll
  for (int j = 0; j < 32; ++j)
    if (fabsf(v[j]) > amax) { amax = fabsf(v[j]); m = v[j]; }
  const float d = __fdiv_rn(m, -8.0f);
  const __half h = __float2half_rn(d);
  const float hd = __half2float(h);
  const float id = (hd != 0.f) ? __fdiv_rn(1.0f, hd) : 0.f;
  uint8_t *blk = out + idx * 18;
  const uint16_t hb = __half_as_ushort(h);
  blk[0] = (uint8_t)(hb & 0xFF);
  blk[1] = (uint8_t)(hb >> 8);
  int q[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    const float t = __fadd_rn(__fmul_rn(v[j], id), 8.5f);
    const int c = (int)floorf(t);
    q[j] = c < 0 ? 0 : (c > 15 ? 15 : c);
  }
#pragma unroll
  for (int j = 0; j < 16; ++j) blk[2 + j] = (uint8_t)(q[j] | (q[j + 16] << 4));
}

// Canonical blocks -> nibble plane + scale plane; source row r goes to row map[r].
__global__ void q4_0_pack_kernel(const uint8_t *blocks, int M, int nb, uint8_t *nib, __half *scales,
                                 int s_stride, const int *map) {
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (int64_t)M * nb) return;
  const int r = (int)(idx / nb), b = (int)(idx % nb);
  const int dr = map ? map[r] : r;
  const uint8_t *src = blocks + idx * 18;
  uint8_t *dst = nib + ((int64_t)dr * nb + b) * 16;
#pragma unroll
  for (int j = 0; j < 16; ++j) dst[j] = src[2 + j];
  scales[(int64_t)dr * s_stride + b] = __ushort_as_half((uint16_t)(src[0] | (src[1] << 8)));
}

// Row copy with optional scatter (source row r -> destination row map[r]) and zero
// padding of wider destination rows.
__global__ void copy_rows_kernel(const uint8_t *src, int64_t srb, uint8_t *dst, int64_t drb, int M, const int *map) {
  const int r = blockIdx.y * gridDim.z + blockIdx.z;
  if (r >= M) return;
  const int dr = map ? map[r] : r;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < drb; i += (int64_t)gridDim.x * blockDim.x)
    dst[(int64_t)dr * drb + i] = (i < srb) ? src[(int64_t)r * srb + i] : 0;
}

__global__ void rope_table_kernel(float *cos_t, float *sin_t, int n_pos, int hd, double base) {
  const int h2 = hd / 2;
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (int64_t)n_pos * h2) return;
  const int p = (int)(idx / h2), i = (int)(idx % h2);
  const double inv = pow(base, -2.0 * (double)i / (double)hd);
  const double ang = (double)p * inv;
  cos_t[idx] = (float)cos(ang);
  sin_t[idx] = (float)sin(ang);
}

static int blocks_for(int64_t n, int t) { return (int)((n + t - 1) / t); }

mie_status launch_convert_bf16(const float *w, int64_t n, uint16_t *out, cudaStream_t st) {
  if (n <= 0) return MIE_OK;
  int grid = blocks_for(n, 256);
  if (grid > 65535 * 4) grid = 65535 * 4;
  convert_bf16_kernel<<<grid, 256, 0, st>>>(w, n, out);
  MIE_CUDA(cudaGetLastError());
  return MIE_OK;
}

mie_status launch_quantize_i8(const float *w, int M, int K, int8_t *q, float *s, cudaStream_t st) {
  quantize_i8_kernel<<<blocks_for((int64_t)M * 32, 256), 256, 0, st>>>(w, M, K, q, s);
  MIE_CUDA(cudaGetLastError());
  return MIE_OK;
}

mie_status launch_quantize_q4_0(const float *w, int M, int K, uint8_t *blocks, cudaStream_t st) {
  const int64_t n = (int64_t)M * ((K + 31) / 32);
  quantize_q4_0_kernel<<<blocks_for(n, 128), 128, 0, st>>>(w, M, K, blocks);
  MIE_CUDA(cudaGetLastError());
  return MIE_OK;
}

mie_status launch_q4_0_pack(const uint8_t *blocks, int M, int K, uint8_t *nib, __half *scales, int s_stride,
                            const int *row_map, cudaStream_t st) {
  const int nb = (K + 31) / 32;
  q4_0_pack_kernel<<<blocks_for((int64_t)M * nb, 256), 256, 0, st>>>(blocks, M, nb, nib, scales, s_stride, row_map);
  MIE_CUDA(cudaGetLastError());
  return MIE_OK;
}

mie_status launch_pad_rows(const uint8_t *src, int64_t srb, uint8_t *dst, int64_t drb, int M, const int *map,
                           cudaStream_t st) {
  if (M <= 0) return MIE_OK;
  const int z = M < 65535 ? M : 65535;
  const int y = (M + z - 1) / z;
  const int x = blocks_for(drb, 256) < 8 ? blocks_for(drb, 256) : 8;
  copy_rows_kernel<<<dim3(x, y, z), 256, 0, st>>>(src, srb, dst, drb, M, map);
  MIE_CUDA(cudaGetLastError());
  return MIE_OK;
}

mie_status launch_row_permute(const uint8_t *src, uint8_t *dst, int64_t row_bytes, int M, const int *map,
                              cudaStream_t st) {
  return launch_pad_rows(src, row_bytes, dst, row_bytes, M, map, st);
}

mie_status launch_rope_table(float *cos_t, float *sin_t, int n_pos, int hd, double base, cudaStream_t st) {
  rope_table_kernel<<<blocks_for((int64_t)n_pos * (hd / 2), 256), 256, 0, st>>>(cos_t, sin_t, n_pos, hd, base);
  MIE_CUDA(cudaGetLastError());
  return MIE_OK;
}

}  // namespace mie

using namespace mie;

extern "C" mie_status mie_convert_bf16(const float *w, int64_t n, uint16_t *out, void *stream) {
  if (!w || !out) return fail(MIE_E_ARG, "mie_convert_bf16: null pointer");
  if (n < 0) return fail(MIE_E_SHAPE, "mie_convert_bf16: n = %lld", (long long)n);
  return launch_convert_bf16(w, n, out, (cudaStream_t)stream);
}

extern "C" mie_status mie_quantize_i8(const float *w, int M, int K, int8_t *q, float *scale, void *stream) {
  if (!w || !q || !scale) return fail(MIE_E_ARG, "mie_quantize_i8: null pointer");
  if (M < 1 || K < 1) return fail(MIE_E_SHAPE, "mie_quantize_i8: bad shape %d x %d", M, K);
  return launch_quantize_i8(w, M, K, q, scale, (cudaStream_t)stream);
}

extern "C" mie_status mie_quantize_q4_0(const float *w, int M, int K, uint8_t *blocks, void *stream) {
  if (!w || !blocks) return fail(MIE_E_ARG, "mie_quantize_q4_0: null pointer");
  if (M < 1 || K < 1) return fail(MIE_E_SHAPE, "mie_quantize_q4_0: bad shape %d x %d", M, K);
  return launch_quantize_q4_0(w, M, K, blocks, (cudaStream_t)stream);
}

extern "C" mie_status mie_q4_0_pack(const uint8_t *blocks, int M, int K, void *packed, void *stream) {
  if (!blocks || !packed) return fail(MIE_E_ARG, "mie_q4_0_pack: null pointer");
  if (M < 1 || K < 1) return fail(MIE_E_SHAPE, "mie_q4_0_pack: bad shape %d x %d", M, K);
  if ((uintptr_t)packed & 255) return fail(MIE_E_SHAPE, "mie_q4_0_pack: output not 256-byte aligned");
  const int nb = (K + 31) / 32;
  const size_t nib = ((size_t)M * nb * 16 + 255) & ~(size_t)255;
  uint8_t *sc = reinterpret_cast<uint8_t *>(packed) + nib;
  MIE_CUDA(cudaMemsetAsync(sc, 0, (size_t)M * q4_scale_stride(nb) * 2, (cudaStream_t)stream));
  return launch_q4_0_pack(blocks, M, K, reinterpret_cast<uint8_t *>(packed), reinterpret_cast<__half *>(sc),
                          q4_scale_stride(nb), nullptr, (cudaStream_t)stream);
}
