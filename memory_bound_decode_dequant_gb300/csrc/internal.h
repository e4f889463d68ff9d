// internal.h -- host-side interfaces shared by the translation units of libmie.so.
#pragma once

#include <cuda.h>

#include "common.cuh"

namespace mie {

enum Prologue { PRO_PLAIN = 0, PRO_NORM = 1, PRO_EMBED_NORM = 2 };
enum Epilogue { EPI_STORE = 0, EPI_RESID = 1, EPI_SWIGLU = 2, EPI_QKV = 3, EPI_ARGMAX = 4 };

// One weight matrix in its GPU layout.
struct DevMat {
  int fmt = -1;            // mie_format
  int rows = 0, cols = 0;  // logical shape
  int kp = 0;              // padded columns (multiple of the format's chunk)
  const uint8_t *w = nullptr;  // bf16/i8 row-major [rows][kp]; Q4_0 nibble plane [rows][kp/32][16]
  const void *s = nullptr;     // i8: float[rows]; 4-bit: half[rows][s_stride]
  int64_t row_bytes = 0;
  int s_stride = 0;            // 4-bit: scales per row, kp/group rounded up to a multiple of 8
  int gshift = 0;              // 4-bit: log2(weights per scale / 32): 0, 1, 2 for groups of 32, 64, 128
  int pub_fmt = -1;            // the public format (mie_format) the matrix was created with
};

// Weights per f16 scale of a public 4-bit format (0 for the others); the kernels run all
// of them as MIE_FMT_Q4_0 with DevMat::gshift selecting the group.
inline int q4_group(int fmt) {
  return fmt == MIE_FMT_Q4_0 ? 32 : fmt == MIE_FMT_Q4_G64 ? 64 : fmt == MIE_FMT_Q4_G128 ? 128 : 0;
}
inline int q4_gshift(int group) { return group == 128 ? 2 : group == 64 ? 1 : 0; }

// Q4_0 scale-plane row stride: whole 16-byte groups, so a bulk copy of whole rows of
// scales starts and ends on 16-byte boundaries.
inline int q4_scale_stride(int nb) { return (nb + 7) / 8 * 8; }

// Arguments of one GEMV launch (plain or fused).
struct GemvArgs {
  DevMat m;
  const float *x = nullptr;     // input vector [cols] (PRO_PLAIN, PRO_NORM)
  const float *gain = nullptr;  // RMSNorm gain [cols]
  float eps = 0.f;
  int act_bf16 = 0;
  DevMat embed;                 // PRO_EMBED_NORM: table to gather token sp->token[slot] from
  float *x_store = nullptr;     // PRO_EMBED_NORM: residual stream written by CTA 0
  int vocab = 0;
  float *y = nullptr;           // STORE/RESID/SWIGLU output; ARGMAX logits (nullable)
  // EPI_QKV
  float *q_out = nullptr;
  uint16_t *kv_layer = nullptr; // this layer's K half of block 0; V follows after Hkv*bs*hd
  int64_t block_stride = 0;     // elements between consecutive KV blocks
  int n_kv_blocks = 0;
  const float *rope_cos = nullptr, *rope_sin = nullptr;  // [max_pos][hd/2]
  int max_pos = 0;
  int Hq = 0, Hkv = 0, hd = 0, bs = 0;
  // EPI_ARGMAX
  float2 *am_part = nullptr;    // [grid] (value, index bits)
  unsigned *am_count = nullptr; // zero before the first launch; the kernel resets it
  int32_t *am_out = nullptr;    // argmax written here (besides sp->argmax_out)
  StepParams *sp = nullptr;
  int slot = 0;
  int *err = nullptr;
  // persistent step: vectors as tagged words (fp32 bits | tag << 32) instead of x / y
  const uint64_t *x_t = nullptr;  // input (PRO_PLAIN, PRO_NORM)
  const uint64_t *res_t = nullptr;  // EPI_RESID residual; null: the token's embedding row
  uint64_t *y_t = nullptr;        // RESID / SWIGLU output; QKV: q | k | v after RoPE
  // filled in by launch_gemv: the shared-memory ring of weight stages
  int n_stages = 0;
  uint32_t stage_bytes = 0, sc_stage_bytes = 0;
};

int gemv_chunk_elems(int fmt);  // elements per 16-byte chunk: 8 / 16 / 32
int sm_count();

// Launches one GEMV; `pdl` adds the programmatic-dependent-launch attribute.
mie_status launch_gemv(int pro, int epi, const GemvArgs &a, int grid, cudaStream_t st, bool pdl);
int gemv_default_grid(const DevMat &m, int epi);

// Attention (split context, merge by the last CTA of each KV head).
struct AttnArgs {
  const float *q = nullptr;
  const uint16_t *k = nullptr, *v = nullptr;  // this layer's K and V bases
  int64_t block_stride = 0;
  int n_pool_blocks = 0;
  const int32_t *block_table = nullptr;  // used when sp == nullptr
  int n_table = 0;
  int ctx = 0;                           // used when sp == nullptr
  StepParams *sp = nullptr;
  int slot = 0;
  int Hq = 0, Hkv = 0, hd = 0, bs = 0;
  float scale = 0.f;
  float *out = nullptr;
  float *ws_part = nullptr;
  unsigned *ws_count = nullptr;
  int n_splits = 1;
  int *err = nullptr;
  // persistent step: the current token's q | k | v and the output as tagged words
  const uint64_t *qkv_t = nullptr;
  uint64_t *out_t = nullptr;
  // few-slot step: grid layer z is slot z (z >= sp->n_slots exits); q, out and the
  // workspace of slot z are offset by z * (Hq * hd) floats and z * ws_slot_bytes
  int slot_z = 0;
  int max_slots = 1;
  size_t ws_slot_bytes = 0;
};
size_t attn_workspace_bytes(int Hq, int Hkv, int hd, int n_splits);
size_t attn_counter_bytes(int Hkv);  // the counters at the start of a workspace
int attn_splits_for(int Hkv, int max_ctx, int bs);
mie_status launch_attn(const AttnArgs &a, cudaStream_t st, bool pdl);

// Prompt GEMM on tcgen05 (gemm.cu): Y[t][n] (+)= s[n] * sum_k (A0 + A1)[n][k] (B0 + B1 + B2)[t][k]
// with bf16 planes A (weight rows) and B (activation rows) behind 2-D tensor maps
// (make_bf16_map: 64-column boxes of 128 rows by default, 128-byte swizzle, zeros outside).
struct GemmPlan {
  CUtensorMap a[2], b[3];
  int na = 1, nb = 1;  // planes in use: na 1 or 2, nb 1 to 3
  int T = 0, N = 0, K = 0;
  float *y = nullptr;
  int64_t ldy = 0;
  const float *row_scale = nullptr;
  bool accumulate = false;
  int *err = nullptr;
};
mie_status make_bf16_map(CUtensorMap *map, const void *base, int64_t rows, int64_t cols, int64_t pitch,
                         int box_rows = 128);
mie_status launch_gemm(const GemmPlan &p, cudaStream_t st);

// The prompt's row-wise kernels and attention (prefill.cu).
struct RopeKvArgs {
  const float *Y = nullptr;  // [T][ldy] QKV product rows in the step's pair order
  int64_t ldy = 0;
  int T = 0, pos0 = 0;
  const float *cos_t = nullptr, *sin_t = nullptr;
  int Hq = 0, Hkv = 0, hd = 0, bs = 0;
  uint16_t *kv_layer = nullptr;  // this layer's K half of block 0; V follows after Hkv*bs*hd
  int64_t block_stride = 0;
  const int32_t *bt = nullptr;
  int n_table = 0, n_pool = 0;
  float *Q = nullptr;  // [T][Hq*hd]
  int *err = nullptr;
};
struct PrefillAttnArgs {
  const float *q = nullptr;  // [T][ldq]
  int64_t ldq = 0;
  const uint16_t *k = nullptr, *v = nullptr;  // this layer's K and V bases
  int64_t block_stride = 0;
  int n_pool = 0;
  const int32_t *bt = nullptr;
  int pos0 = 0, T = 0, Hq = 0, Hkv = 0, hd = 0, bs = 0;
  float scale = 0.f;
  float *out = nullptr;  // [T][ldo]
  int64_t ldo = 0;
  int *err = nullptr;
};
mie_status launch_embed_rows(const DevMat &e, const int32_t *tok, int T, int vocab, int d, float *R, int *err,
                             cudaStream_t st);
// The row-wise kernels write their output as bf16 planes hi / mid / lo (mid, lo nullable).
mie_status launch_norm_split(const float *x, int64_t ldx, int K, const float *g, float eps, int act_bf16, int T,
                             uint16_t *hi, uint16_t *mid, uint16_t *lo, int64_t ldp, cudaStream_t st);
mie_status launch_rope_kv(const RopeKvArgs &a, cudaStream_t st);
mie_status launch_swiglu_split(const float *Y, int64_t ldy, int F, int act_bf16, int T, uint16_t *hi, uint16_t *mid,
                               uint16_t *lo, int64_t ldp, cudaStream_t st);
mie_status launch_dequant_planes(const DevMat &m, uint16_t *hi, uint16_t *lo, int64_t ldp, cudaStream_t st);
mie_status launch_prefill_attn(const PrefillAttnArgs &a, cudaStream_t st);

// Rounds after which a bounded device-side wait gives up (a few seconds).
constexpr long kWaitPolls = 1L << 22;

// The whole step as one persistent cooperative kernel (step.cu).
enum { PH_GEMV = 0, PH_ATTN = 1 };
struct Phase {
  int kind = PH_GEMV, pro = PRO_PLAIN, epi = EPI_STORE;
  GemvArgs g;
  AttnArgs at;
};
struct PersistArgs {
  const Phase *ph = nullptr;  // device array of n_phases descriptors
  int n_phases = 0;
  unsigned *epoch = nullptr;  // tag of this launch's words (never 0); advanced by the last CTA
  unsigned *fin = nullptr;    // CTAs done with the launch, zero between launches
  int *abort = nullptr;       // nonzero once a bounded wait gave up
  int n_slots = 0;
  uint32_t slot_bytes = 0, slot_sc_bytes = 0;
  int *err = nullptr;
  unsigned long long *trace = nullptr;  // [n_phases][grid][kTracePoints] globaltimer ns, or null
  unsigned long long *stage_trace = nullptr;  // [grid][kStageTrace][kStagePoints], or null
  long wait_polls = kWaitPolls;         // rounds after which a bounded wait of the step gives up
};
constexpr int kTracePoints = 5;  // phase entry, inputs arrived, input staged, stages consumed, outputs written
// Optional per-stage stamps after the phase stamps: [grid][kStageTrace][kStagePoints] =
// copy issued (producer), consumer warp 0 starts waiting for it, the wait returns, warp
// 0 done with the stage; the first kStageTrace ring stages of each CTA.
constexpr int kStageTrace = 1024, kStagePoints = 4;
struct PersistPlan {
  const void *kernel = nullptr;
  int grid = 0, threads = 0, n_slots = 0;
  uint32_t slot_bytes = 0, slot_sc_bytes = 0;
  size_t smem = 0;
};
mie_status persist_plan(const Phase *host_phases, int n, int G, int HD, PersistPlan *plan);
mie_status persist_launch(const PersistPlan &plan, const PersistArgs &args, cudaStream_t st);

// The few-slot step's GEMVs (gemv_slots.cu): every vector argument is slot 0's of
// [n_slots][length] arrays; sp->n_slots slots are computed.
mie_status slots_gemv_supported(const DevMat &m, int pro);
mie_status launch_gemv_slots(int pro, int epi, const GemvArgs &a, cudaStream_t st, bool pdl);

// Sampling (sample.cu).
struct SampleArgs;
size_t sample_workspace_bytes();
int sample_launches(float temperature, int top_k, float top_p, int n);
// Enqueues the sampler for slot 0 of the step parameters sp: logits sp->logits_out, the
// RNG position sp->pos[0]; the draw goes to sp->argmax_out and, with sp->sample_advance,
// into token / pos.  ws: sample_workspace_bytes() of zeroed device memory.
mie_status launch_step_sample(StepParams *sp, int vocab, float temperature, int top_k, float top_p, uint64_t seed,
                              void *ws, cudaStream_t st);

// Load-time kernels.
mie_status launch_convert_bf16(const float *w, int64_t n, uint16_t *out, cudaStream_t st);
mie_status launch_quantize_i8(const float *w, int M, int K, int8_t *q, float *s, cudaStream_t st);
mie_status launch_quantize_q4(const float *w, int M, int K, int group, uint8_t *groups, cudaStream_t st);
mie_status launch_q4_pack(const uint8_t *groups, int M, int K, int group, uint8_t *nib, __half *scales, int s_stride,
                          const int *row_map, cudaStream_t st);
mie_status launch_row_permute(const uint8_t *src, uint8_t *dst, int64_t row_bytes, int M,
                              const int *row_map, cudaStream_t st);
mie_status launch_pad_rows(const uint8_t *src, int64_t src_row_bytes, uint8_t *dst,
                           int64_t dst_row_bytes, int M, const int *row_map, cudaStream_t st);
mie_status launch_rope_table(float *cos_t, float *sin_t, int n_pos, int hd, double base,
                             cudaStream_t st);
mie_status launch_argmax(const float *v, int n, int32_t *out, float2 *part, unsigned *count,
                         int grid, cudaStream_t st);
int argmax_grid(int n);

}  // namespace mie
