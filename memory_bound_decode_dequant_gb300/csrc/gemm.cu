// gemm.cu -- the prompt's dense contractions on the fifth-generation tensor cores.
//
// "infer" page, summary table and "Limitations": prefill runs every prompt token through
// the same matrices, so it is a matrix-matrix product (a real dense contraction), and
// tensor cores are what would make it several times faster than the CUDA-core path.
//
//   Y[t][n] (+)= s[n] * sum_k (A0 + A1)[n][k] * (B0 + B1 + B2)[t][k]
//
// A = weight rows (bf16, K contiguous), B = activation rows (bf16, K contiguous).  Each
// operand comes as bf16 planes whose sum is the value, plane j of magnitude 2^-8j of the
// value: an fp32 activation as hi = bf16(x), mid = bf16(x - hi), lo = bf16(x - hi - mid)
// (to 2^-25 of x; two planes leave 2^-18, which measured 1e-5 of the output's RMS and
// flipped the bf16 rounding of 0.8 % of the K/V values written from it), a bf16 or int8
// weight as one plane, a dequantised 4-bit weight as two (an f16 scale times a 4-bit
// code has up to 14 significant bits).  Every product of planes is exact in fp32; the
// products whose levels add up to more than 2 (below 2^-24 of the terms) are skipped.
// s is an optional per-row scale (int8 rows: the codes are exact in bf16).
//
// Persistent: one CTA per SM takes 128 (weight rows) x 128 (tokens) tiles in turn, each
// over the whole K, its stage ring and accumulators running on from one tile to the next:
//   warp 0, one lane : TMA producer, 64-column stages of every plane (128-byte swizzle)
//   warp 1, one lane : issues tcgen05.mma (M = 128, N = 128, K = 16) into one of four TMEM
//                      accumulators of 128 lanes x 128 fp32 columns, a segment of
//                      kSegBlocks stages each, and tcgen05.commit to hand stages back
//                      and to announce a finished segment; four buffers let the MMAs run
//                      three segments ahead of the drain
//   warps 2-9        : drain: tcgen05.ld of their 32 TMEM lanes and half of the columns
//                      after every segment, summed in fp32 registers, then scaled and
//                      stored
// The tensor cores' own sums lose about 2^-24 of the accumulator per MMA (measured on
// GB300: 8e-7 of sum |w x| at K = 2048 when one accumulator takes the whole K, against
// 1.5e-8 for the fp32-FMA GEMV); draining every 128 columns of K keeps each tensor-core
// sum short and leaves the long sum to fp32 adds.
// Every mbarrier wait is bounded and gives up early once another role has failed; a
// failure latches ERR_TIMEOUT, the CTA still waits (bounded) for its own copies and
// MMAs, and frees its TMEM before it exits.
#include <cuda.h>

#include <algorithm>
#include <mutex>

#include "internal.h"
#include "device.cuh"

namespace mie {

namespace {

constexpr int kTM = 128;        // weight rows per tile (UMMA M)
constexpr int kTN = 128;        // tokens per tile (UMMA N)
constexpr int kTK = 64;         // K per stage: one 128-byte swizzle atom of bf16
constexpr int kPlaneBytes = kTM * kTK * 2;  // 16 KB per plane per stage (kTN == kTM)
constexpr int kDrainWarps = 8;                       // two per TMEM lane quarter
constexpr int kDrainCols = kTN * 4 / kDrainWarps;  // accumulator columns a drain warp reads
constexpr int kGemmThreads = 64 + 32 * kDrainWarps;  // producer warp, MMA warp, drain warps
constexpr int kAccBufs = 4;                // fp32 accumulator buffers of kTN columns in TMEM
constexpr int kTmemCols = kAccBufs * kTN;  // all 512 columns: one CTA per SM
constexpr int kSegBlocks = 2;       // stages summed by the tensor cores before a drain
constexpr int kSmemBudget = 200 * 1024;

static_assert(kTN == kTM, "A and B stage planes have the same size");

struct GemmDev {
  int T, N, K;
  float *y;
  int64_t ldy;
  const float *row_scale;
  int accumulate;
  int *err;
  long wait_polls;
};

__host__ __device__ constexpr int gemm_stages(int na, int nb) {
  return kSmemBudget / ((na + nb) * kPlaneBytes) > 8 ? 8 : kSmemBudget / ((na + nb) * kPlaneBytes);
}
__host__ __device__ constexpr size_t gemm_smem_bytes(int na, int nb) {
  // stages, then the barriers, the TMEM address and the failure flag; +1024 to align the stages
  return (size_t)gemm_stages(na, nb) * (na + nb) * kPlaneBytes + 256 + 1024;
}

// Shared-memory matrix descriptor of a K-major operand tile laid out by a TMA copy with
// 128-byte swizzle: rows of 128 bytes, 8-row groups 1024 bytes apart (stride byte
// offset), leading byte offset unused for this layout (1), descriptor version 1 (bits
// 46-47), swizzle mode 2 = 128 bytes (bits 61-63).  `addr` advances by 32 bytes per
// 16-column step inside the 1024-byte-aligned atom.
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t addr) {
  uint64_t d = 0;
  d |= (uint64_t)((addr >> 4) & 0x3FFF);
  d |= (uint64_t)1 << 16;                  // leading byte offset (16 B, unused)
  d |= (uint64_t)(1024 >> 4) << 32;        // stride byte offset
  d |= (uint64_t)1 << 46;                  // version
  d |= (uint64_t)2 << 61;                  // 128-byte swizzle
  return d;
}

// Instruction descriptor of tcgen05.mma kind::f16: fp32 accumulator (bits 4-5 = 1), bf16
// A and B (bits 7-9, 10-12 = 1), both K-major (bits 15, 16 = 0), N >> 3 at bits 17-22,
// M >> 4 at bits 24-28.
__host__ __device__ constexpr uint32_t umma_idesc_bf16(int m, int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void umma_bf16(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t idesc, int acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}

// The mbarrier arrives once every tcgen05 operation this thread issued before has
// completed.
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 32 consecutive fp32 columns of this warp's 32 TMEM lanes, one lane per thread; the
// caller waits (tmem_wait_ld) before it reads r.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

template <int NA, int NB>
__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA0, const __grid_constant__ CUtensorMap tmA1,
                   const __grid_constant__ CUtensorMap tmB0, const __grid_constant__ CUtensorMap tmB1,
                   const __grid_constant__ CUtensorMap tmB2, GemmDev g) {
  constexpr int S = gemm_stages(NA, NB);
  constexpr int kStageBytes = (NA + NB) * kPlaneBytes;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;  // 128-byte swizzle atoms need 1024-byte alignment
  uint8_t *gen = smem_raw + (base - raw);
  uint64_t *full = reinterpret_cast<uint64_t *>(gen + (size_t)S * kStageBytes);
  uint64_t *empty = full + S;
  uint64_t *tfull = empty + S;          // [kAccBufs] a segment's sums are in buffer b
  uint64_t *tempty = tfull + kAccBufs;  // [kAccBufs] the drain warps have read buffer b
  uint64_t *done = tempty + kAccBufs;   // every MMA has completed
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(done + 1);
  int *fail_flag = reinterpret_cast<int *>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nk = (g.K + kTK - 1) / kTK;
  const int nseg = (nk + kSegBlocks - 1) / kSegBlocks;  // segments per tile
  const int tiles_n = (g.N + kTM - 1) / kTM, n_tiles = tiles_n * ((g.T + kTN - 1) / kTN);
  // persistent: this CTA's tiles are blockIdx.x, + gridDim.x, ... (weight tiles fastest,
  // so the CTAs running at one time share their activation tile through L2)
  const int my_tiles = blockIdx.x < n_tiles ? (n_tiles - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < kAccBufs; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], kDrainWarps);
    }
    mbar_init(done, 1);
    *fail_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // producer: stage c (counted over all of this CTA's tiles) into slot c % S
      int issued = 0, c = 0;
      bool ok = true;
      for (int i = 0; i < my_tiles && ok; ++i) {
        const int tile = (int)blockIdx.x + i * (int)gridDim.x;
        const int n0 = (tile % tiles_n) * kTM, t0 = (tile / tiles_n) * kTN;
        for (int kb = 0; kb < nk; ++kb, ++c) {
          const int s = c % S, r = c / S;
          if (r > 0 && !mbar_wait_or_abort(&empty[s], (r - 1) & 1, g.wait_polls, fail_flag)) {
            *fail_flag = 1;
            ok = false;
            break;
          }
          const uint32_t st = base + (uint32_t)s * kStageBytes, bar = smem_u32(&full[s]);
          mbar_expect_tx(&full[s], (uint32_t)kStageBytes);
          tma_load_2d(st, &tmA0, kb * kTK, n0, bar);
          if (NA == 2) tma_load_2d(st + kPlaneBytes, &tmA1, kb * kTK, n0, bar);
          tma_load_2d(st + NA * kPlaneBytes, &tmB0, kb * kTK, t0, bar);
          if (NB >= 2) tma_load_2d(st + (NA + 1) * kPlaneBytes, &tmB1, kb * kTK, t0, bar);
          if (NB >= 3) tma_load_2d(st + (NA + 2) * kPlaneBytes, &tmB2, kb * kTK, t0, bar);
          issued = c + 1;
        }
      }
      // before the CTA may exit, every issued copy must have landed: wait for the last
      // round of each slot that was filled
      for (int q = issued - S < 0 ? 0 : issued - S; q < issued; ++q)
        if (!mbar_wait(&full[q % S], (q / S) & 1, g.wait_polls)) *fail_flag = 1;
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // MMA issuer: segment q (counted over all tiles) of kSegBlocks stages into
      // accumulator buffer q % kAccBufs
      constexpr uint32_t idesc = umma_idesc_bf16(kTM, kTN);
      bool ok = true;
      int c = 0, q = 0;
      for (int i = 0; i < my_tiles && ok; ++i) {
        for (int sg = 0; sg < nseg && ok; ++sg, ++q) {
          const int b = q % kAccBufs;
          if (q >= kAccBufs && !mbar_wait_or_abort(&tempty[b], (q / kAccBufs - 1) & 1, g.wait_polls, fail_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t acc = tmem + (uint32_t)(b * kTN);
          const int kb1 = min(nk, (sg + 1) * kSegBlocks);
          for (int kb = sg * kSegBlocks; kb < kb1; ++kb, ++c) {
            const int s = c % S, r = c / S;
            if (!mbar_wait_or_abort(&full[s], r & 1, g.wait_polls, fail_flag)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t st = base + (uint32_t)s * kStageBytes;
            const bool first = kb == sg * kSegBlocks;
#pragma unroll
            for (int ks = 0; ks < kTK / 16; ++ks) {
#pragma unroll
              for (int a = 0; a < NA; ++a) {
#pragma unroll
                for (int pb = 0; pb < NB; ++pb) {
                  if (a + pb > 2) continue;  // plane products below 2^-24 of the sum's terms
                  const uint64_t ad = umma_desc_sw128(st + a * kPlaneBytes + ks * 32);
                  const uint64_t bd = umma_desc_sw128(st + (NA + pb) * kPlaneBytes + ks * 32);
                  umma_bf16(acc, ad, bd, idesc, !(first && ks == 0 && a == 0 && pb == 0));
                }
              }
            }
            umma_commit(smem_u32(&empty[s]));  // the slot is free once these MMAs have read it
          }
          if (ok) umma_commit(smem_u32(&tfull[b]));  // the segment's sums are complete
        }
      }
      if (!ok) *fail_flag = 1;
      umma_commit(smem_u32(done));  // arrives when every MMA above has completed
    }
  } else {
    // drain warps: warp w reads accumulator lanes 32 (w % 4) .. + 31 = weight rows
    // n0 + 32 (w % 4) + lane, columns (positions) c1 .. c1 + kDrainCols - 1, and sums a
    // tile's segments in fp32 registers, so the tensor cores accumulate only kSegBlocks
    // stages before each sum is rounded to fp32; both loads of a segment are in flight
    // before the one wait; the stores of one tile overlap the MMAs of the next
    const int quarter = warp & 3, c1 = ((warp - 2) / 4) * kDrainCols;
    bool ok = true;
    int q = 0;
    for (int i = 0; i < my_tiles && ok; ++i) {
      const int tile = (int)blockIdx.x + i * (int)gridDim.x;
      const int n0 = (tile % tiles_n) * kTM, t0 = (tile / tiles_n) * kTN;
      float sum[kDrainCols];
#pragma unroll
      for (int cc = 0; cc < kDrainCols; ++cc) sum[cc] = 0.f;
      for (int sg = 0; sg < nseg; ++sg, ++q) {
        const int b = q % kAccBufs;
        ok = __all_sync(0xffffffffu, mbar_wait_or_abort(&tfull[b], (q / kAccBufs) & 1, g.wait_polls, fail_flag));
        if (!ok) {
          if (lane == 0) *fail_flag = 1;
          break;
        }
        tc_fence_after();
        const uint32_t taddr = tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(b * kTN + c1);
        uint32_t r[kDrainCols / 32][32];
#pragma unroll
        for (int h = 0; h < kDrainCols / 32; ++h) tmem_ld32(taddr + (uint32_t)(h * 32), r[h]);
        tmem_wait_ld();
#pragma unroll
        for (int h = 0; h < kDrainCols / 32; ++h)
#pragma unroll
          for (int j = 0; j < 32; ++j) sum[h * 32 + j] += __uint_as_float(r[h][j]);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[b]);
      }
      const int n = n0 + quarter * 32 + lane;
      if (ok && !*reinterpret_cast<volatile int *>(fail_flag) && n < g.N) {
        const float sc = g.row_scale ? g.row_scale[n] : 1.0f;
#pragma unroll
        for (int cc = 0; cc < kDrainCols; ++cc) {
          const int t = t0 + c1 + cc;
          if (t < g.T) {
            float *dst = g.y + (int64_t)t * g.ldy + n;
            *dst = g.accumulate ? *dst + sum[cc] * sc : sum[cc] * sc;
          }
        }
      }
    }
  }
  __syncwarp();
  if (warp == 1) {  // no MMA may still be writing the accumulators when they are freed
    if (!__all_sync(0xffffffffu, mbar_wait(done, 0, g.wait_polls)) && lane == 0) *fail_flag = 1;
  }
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0 && *reinterpret_cast<volatile int *>(fail_flag)) latch_error(g.err, ERR_TIMEOUT);
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
  }
}

// ------------------------------------------------------------------ host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

}  // namespace

// A 2-D bf16 tensor map over rows of `cols` elements, `pitch` bytes apart, boxes of 64
// columns x box_rows rows with 128-byte swizzle; reads outside the tensor return zeros.
mie_status make_bf16_map(CUtensorMap *map, const void *base, int64_t rows, int64_t cols, int64_t pitch,
                         int box_rows) {
  EncodeTiledFn enc = encode_tiled();
  if (!enc) return fail(MIE_E_CUDA, "tensor map: cuTensorMapEncodeTiled is not available");
  if (((uintptr_t)base & 15) || (pitch & 15)) return fail(MIE_E_SHAPE, "tensor map: base or pitch not 16-byte aligned");
  if (box_rows < 1 || box_rows > 256) return fail(MIE_E_SHAPE, "tensor map: box of %d rows", box_rows);
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)pitch};
  const cuuint32_t box[2] = {(cuuint32_t)kTK, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(MIE_E_CUDA, "tensor map: encode failed (%d)", (int)r);
  return MIE_OK;
}

template <int NA, int NB>
static mie_status launch_gemm_t(const GemmPlan &p, cudaStream_t st) {
  auto kern = gemm_tc_kernel<NA, NB>;
  const size_t smem = gemm_smem_bytes(NA, NB);
  static std::once_flag once;
  static cudaError_t attr = cudaSuccess;
  std::call_once(once, [&] { attr = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem); });
  if (attr != cudaSuccess) return cuda_fail(attr, "gemm: cudaFuncSetAttribute");
  GemmDev g;
  g.T = p.T;
  g.N = p.N;
  g.K = p.K;
  g.y = p.y;
  g.ldy = p.ldy;
  g.row_scale = p.row_scale;
  g.accumulate = p.accumulate;
  g.err = p.err;
  g.wait_polls = kWaitPolls;
  const int n_tiles = ((p.N + kTM - 1) / kTM) * ((p.T + kTN - 1) / kTN);
  const dim3 grid((unsigned)std::min(n_tiles, sm_count()));  // persistent: one CTA per SM
  kern<<<grid, kGemmThreads, smem, st>>>(p.a[0], p.a[NA - 1], p.b[0], p.b[NB > 1 ? 1 : 0], p.b[NB - 1], g);
  MIE_CUDA(cudaGetLastError());
  return MIE_OK;
}

mie_status launch_gemm(const GemmPlan &p, cudaStream_t st) {
  if (p.T < 1 || p.N < 1 || p.K < 1 || !p.y) return fail(MIE_E_ARG, "gemm: empty problem");
  if (p.T > 65535 * kTN) return fail(MIE_E_SHAPE, "gemm: %d rows of activations", p.T);
  if (p.na == 1 && p.nb == 1) return launch_gemm_t<1, 1>(p, st);
  if (p.na == 1 && p.nb == 2) return launch_gemm_t<1, 2>(p, st);
  if (p.na == 1 && p.nb == 3) return launch_gemm_t<1, 3>(p, st);
  if (p.na == 2 && p.nb == 1) return launch_gemm_t<2, 1>(p, st);
  if (p.na == 2 && p.nb == 3) return launch_gemm_t<2, 3>(p, st);
  return fail(MIE_E_ARG, "gemm: %d weight planes, %d activation planes", p.na, p.nb);
}

}  // namespace mie

using namespace mie;

extern "C" mie_status mie_gemm_bf16(const uint16_t *W, int N, int K, const uint16_t *x_hi, const uint16_t *x_mid,
                                    const uint16_t *x_lo, int T, float *y, int64_t ldy, int accumulate,
                                    void *stream) {
  if (!W || !x_hi || !y) return fail(MIE_E_ARG, "mie_gemm_bf16: null pointer");
  if (x_lo && !x_mid) return fail(MIE_E_ARG, "mie_gemm_bf16: x_lo without x_mid");
  if (N < 1 || K < 1 || T < 1) return fail(MIE_E_SHAPE, "mie_gemm_bf16: N = %d, K = %d, T = %d", N, K, T);
  if (K % 8) return fail(MIE_E_SHAPE, "mie_gemm_bf16: K = %d is not a multiple of 8", K);
  if (ldy < N) return fail(MIE_E_ARG, "mie_gemm_bf16: ldy %lld < N %d", (long long)ldy, N);
  GemmPlan p;
  p.T = T;
  p.N = N;
  p.K = K;
  p.y = y;
  p.ldy = ldy;
  p.accumulate = accumulate != 0;
  p.err = device_error_flag();
  p.na = 1;
  p.nb = x_lo ? 3 : x_mid ? 2 : 1;
  const uint16_t *planes[3] = {x_hi, x_mid, x_lo};
  mie_status s = make_bf16_map(&p.a[0], W, N, K, (int64_t)K * 2);
  for (int j = 0; j < p.nb && s == MIE_OK; ++j) s = make_bf16_map(&p.b[j], planes[j], T, K, (int64_t)K * 2);
  if (s != MIE_OK) return s;
  return launch_gemm(p, (cudaStream_t)stream);
}
