// quant.cu -- load-time quantisation and packing kernels, RoPE tables.
//
// 4-bit ("Writing an LLM inference engine from scratch in Rust", Lesson 1 and "Is the
// 4-bit model still good?"; "infer" page, weight-only quantization): groups of 32 (Q4_0),
// 64 or 128, scale from the element of largest magnitude with its sign kept, divided by
// -8 so that element lands exactly on code 0 (-8), stored as f16.  int8: one scale per
// row.
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

// One thread per group of GS weights; canonical output [M][ng][2 + GS/2]: the f16 scale
// (little-endian), then GS/32 sub-blocks of 16 bytes, byte j of sub-block b holding code
// 32b + j in its low nibble and code 32b + j + 16 in its high nibble (GS = 32: Q4_0).
template <int GS>
__global__ void quantize_q4_kernel(const float *w, int M, int K, uint8_t *out) {
  const int ng = (K + GS - 1) / GS;
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (int64_t)M * ng) return;
  const int r = (int)(idx / ng), b = (int)(idx % ng);
  const float *row = w + (int64_t)r * K;
  float amax = 0.f, m = 0.f;
  for (int j = 0; j < GS; ++j) {
    const int k = b * GS + j;
    const float v = (k < K) ? row[k] : 0.f;
    if (fabsf(v) > amax) { amax = fabsf(v); m = v; }
  }
  const float d = __fdiv_rn(m, -8.0f);
  const __half h = __float2half_rn(d);
  const float hd = __half2float(h);
  const float id = (hd != 0.f) ? __fdiv_rn(1.0f, hd) : 0.f;
  uint8_t *grp = out + idx * (2 + GS / 2);
  const uint16_t hb = __half_as_ushort(h);
  grp[0] = (uint8_t)(hb & 0xFF);
  grp[1] = (uint8_t)(hb >> 8);
  auto code = [&](int j) {
    const int k = b * GS + j;
    const float v = (k < K) ? row[k] : 0.f;
    const float t = __fadd_rn(__fmul_rn(v, id), 8.5f);
    const int c = (int)floorf(t);
    return c < 0 ? 0 : (c > 15 ? 15 : c);
  };
  for (int sb = 0; sb < GS / 32; ++sb)
#pragma unroll 4
    for (int j = 0; j < 16; ++j) grp[2 + sb * 16 + j] = (uint8_t)(code(sb * 32 + j) | (code(sb * 32 + j + 16) << 4));
}

// Canonical groups -> nibble plane + scale plane; source row r goes to row map[r].  One
// thread per 32-weight sub-block.
__global__ void q4_pack_kernel(const uint8_t *groups, int M, int ng, int GS, uint8_t *nib, __half *scales,
                               int s_stride, const int *map) {
  const int per = GS / 32, nb = ng * per;
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (int64_t)M * nb) return;
  const int r = (int)(idx / nb), c = (int)(idx % nb), g = c / per, sb = c % per;
  const int dr = map ? map[r] : r;
  const uint8_t *src = groups + ((int64_t)r * ng + g) * (2 + GS / 2);
  uint8_t *dst = nib + ((int64_t)dr * nb + c) * 16;
#pragma unroll
  for (int j = 0; j < 16; ++j) dst[j] = src[2 + sb * 16 + j];
  if (sb == 0) scales[(int64_t)dr * s_stride + g] = __ushort_as_half((uint16_t)(src[0] | (src[1] << 8)));
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

mie_status launch_quantize_q4(const float *w, int M, int K, int group, uint8_t *groups, cudaStream_t st) {
  const int64_t n = (int64_t)M * ((K + group - 1) / group);
  if (group == 32) quantize_q4_kernel<32><<<blocks_for(n, 128), 128, 0, st>>>(w, M, K, groups);
  else if (group == 64) quantize_q4_kernel<64><<<blocks_for(n, 128), 128, 0, st>>>(w, M, K, groups);
  else if (group == 128) quantize_q4_kernel<128><<<blocks_for(n, 128), 128, 0, st>>>(w, M, K, groups);
  else return fail(MIE_E_ARG, "4-bit group %d not 32, 64 or 128", group);
  MIE_CUDA(cudaGetLastError());
  return MIE_OK;
}

mie_status launch_q4_pack(const uint8_t *groups, int M, int K, int group, uint8_t *nib, __half *scales, int s_stride,
                          const int *row_map, cudaStream_t st) {
  const int ng = (K + group - 1) / group;
  const int64_t n = (int64_t)M * ng * (group / 32);
  q4_pack_kernel<<<blocks_for(n, 256), 256, 0, st>>>(groups, M, ng, group, nib, scales, s_stride, row_map);
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

extern "C" mie_status mie_quantize_q4(const float *w, int M, int K, int group, uint8_t *groups, void *stream) {
  if (!w || !groups) return fail(MIE_E_ARG, "mie_quantize_q4: null pointer");
  if (M < 1 || K < 1) return fail(MIE_E_SHAPE, "mie_quantize_q4: bad shape %d x %d", M, K);
  if (group != 32 && group != 64 && group != 128) return fail(MIE_E_ARG, "mie_quantize_q4: group %d", group);
  return launch_quantize_q4(w, M, K, group, groups, (cudaStream_t)stream);
}

extern "C" mie_status mie_quantize_q4_0(const float *w, int M, int K, uint8_t *blocks, void *stream) {
  return mie_quantize_q4(w, M, K, 32, blocks, stream);
}

extern "C" mie_status mie_q4_pack(const uint8_t *groups, int M, int K, int group, void *packed, void *stream) {
  if (!groups || !packed) return fail(MIE_E_ARG, "mie_q4_pack: null pointer");
  if (M < 1 || K < 1) return fail(MIE_E_SHAPE, "mie_q4_pack: bad shape %d x %d", M, K);
  if (group != 32 && group != 64 && group != 128) return fail(MIE_E_ARG, "mie_q4_pack: group %d", group);
  if ((uintptr_t)packed & 255) return fail(MIE_E_SHAPE, "mie_q4_pack: output not 256-byte aligned");
  const int ng = (K + group - 1) / group, nb = ng * (group / 32);
  const size_t nib = ((size_t)M * nb * 16 + 255) & ~(size_t)255;
  uint8_t *sc = reinterpret_cast<uint8_t *>(packed) + nib;
  MIE_CUDA(cudaMemsetAsync(sc, 0, (size_t)M * q4_scale_stride(ng) * 2, (cudaStream_t)stream));
  return launch_q4_pack(groups, M, K, group, reinterpret_cast<uint8_t *>(packed), reinterpret_cast<__half *>(sc),
                        q4_scale_stride(ng), nullptr, (cudaStream_t)stream);
}

extern "C" mie_status mie_q4_0_pack(const uint8_t *blocks, int M, int K, void *packed, void *stream) {
  return mie_q4_pack(blocks, M, K, 32, packed, stream);
}
