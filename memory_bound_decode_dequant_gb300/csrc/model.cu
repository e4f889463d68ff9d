// model.cu -- the decode-step context: weights in GPU layouts, the paged KV pool, the
// step as a chain of fused kernels captured once into a CUDA graph.
//
// Step ("infer" page, data-flow figure; "Writing an LLM inference engine from scratch
// in Rust", "How a Llama model generates text"), per layer:
//   qkv   : RMSNorm(x) staged in the GEMV prologue (layer 0 gathers x = E[token]
//           first), Wqkv rows paired (i, i + hd/2) so the epilogue applies RoPE and
//           writes bf16 K/V into the paged pool through the block table
//   attn  : split-context paged GQA attention, merged by the last CTA of each KV head
//   o     : x += Wo o (residual epilogue)
//   gu    : RMSNorm(x), gate/up rows interleaved, epilogue silu(gate) * up
//   down  : x += Wd a
// then the LM head with RMSNorm prologue and an argmax epilogue.  Every kernel is
// launched with programmatic dependent launch, so inside the graph each one issues
// its first weight loads while its predecessor drains.  Token, position and block
// table are read from device memory (StepParams), so one graph serves every step.
#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cmath>
#include <cstring>
#include <new>
#include <string>
#include <vector>

#include "internal.h"

namespace mie {

static thread_local std::string g_last_error;

void set_error(const char *fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
}

mie_status fail(mie_status s, const char *fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return s;
}

mie_status cuda_fail(cudaError_t e, const char *what) {
  return fail(MIE_E_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

}  // namespace mie

using namespace mie;

extern "C" const char *mie_last_error(void) { return g_last_error.c_str(); }

extern "C" const char *mie_status_string(mie_status s) {
  switch (s) {
    case MIE_OK: return "ok";
    case MIE_E_ARG: return "invalid argument";
    case MIE_E_SHAPE: return "unsupported shape";
    case MIE_E_OOM: return "out of memory";
    case MIE_E_CUDA: return "CUDA error";
    case MIE_E_TIMEOUT: return "timeout";
    case MIE_E_STATE: return "invalid state";
    case MIE_E_DEVICE: return "device bounds check";
  }
  return "unknown status";
}

namespace {

enum { T_QKV = 0, T_O, T_GATE, T_UP, T_DOWN, T_ANORM, T_MNORM, T_COUNT };

struct Layer {
  DevMat qkv, o, gu, down;
  float *attn_norm = nullptr, *mlp_norm = nullptr;
  bool loaded[T_COUNT] = {false, false, false, false, false, true, true};
};

int pad_to(int v, int m) { return (v + m - 1) / m * m; }

}  // namespace

struct mie_ctx {
  mie_config cfg{};
  cudaStream_t stream = nullptr;
  bool own_stream = false;
  std::vector<void *> allocs;
  std::vector<Layer> layers;
  DevMat head, embed;
  bool head_loaded = false, embed_loaded = false;
  float *final_norm = nullptr;
  uint16_t *kv = nullptr;
  int64_t block_elems = 0;
  float *x = nullptr, *q = nullptr, *att = nullptr, *act = nullptr;
  float *rope_cos = nullptr, *rope_sin = nullptr;
  uint8_t *attn_ws = nullptr;  // per layer: split counters, then split partials
  size_t attn_ws_bytes = 0;    // one layer's share
  int attn_splits = 1;
  float2 *am_part = nullptr;
  unsigned *am_count = nullptr;
  StepParams *sp = nullptr;
  // Host side of the step parameters: a ring of pinned buffers, so each upload is a DMA
  // that runs in stream order; a buffer is rewritten only after the event recorded
  // behind its previous upload has fired.
  static constexpr int kParamRing = 8;
  StepParams *sp_pinned = nullptr;
  cudaEvent_t sp_uploaded[kParamRing] = {};
  int sp_next = 0;
  int *err = nullptr;
  cudaGraphExec_t graph = nullptr;
  bool graph_ok = true;  // false: the step is launched directly (capture unsupported)
  int launches = 0;
  bool primed = false;
  mie_pool *pool = nullptr;
  // persistent step
  int mode = MIE_STEP_PERSISTENT;  // prepare_step falls back to the chain for other shapes
  std::vector<Phase> phases;
  Phase *d_phases = nullptr;
  size_t d_phases_cap = 0;
  uint64_t *tagged = nullptr;  // per layer: q|k|v, attention out, x after o, act, x after down
  size_t tagged_words = 0;
  unsigned *epoch = nullptr;   // [0]: the next launch's tag; [1]: CTAs finished
  int *abort = nullptr;
  PersistPlan plan;
  unsigned long long *trace = nullptr;
  size_t trace_bytes = 0;
  // testing aid for the bounded waits (mie_debug_stall): phase whose input is read from
  // never-written words, and the rounds after which a wait gives up
  int stall_phase = -1;
  long wait_polls = kWaitPolls;
  uint64_t *stall_words = nullptr;
  // sampling of the next token (mie_set_sampling); temperature <= 0: greedy
  float temperature = 0.f, top_p = 1.f;
  int top_k = 0;
  uint64_t seed = 0;
  float *logits_buf = nullptr;  // the step's logits when the caller passes none
  void *sample_ws = nullptr;
  // verify passes and generation (mie_verify_step, mie_generate)
  int32_t *verify_table = nullptr;  // [kMaxSlots][verify_cap] copies of one sequence's table
  int verify_cap = 0;
  int32_t *gen_argmax = nullptr;    // [kMaxSlots]
  int32_t *next_pinned = nullptr;   // mie_decode_step_sync: the step's token, read back
  // prompt prefill on the tensor cores (mie_prefill): buffers for chunks of up to
  // prefill_chunk positions, allocated on the first call
  int prefill_chunk = 0;
  int64_t prefill_ldp = 0;      // elements per row of the bf16 activation planes
  float *pf_R = nullptr, *pf_Y = nullptr, *pf_Q = nullptr, *pf_O = nullptr;
  uint16_t *pf_xh = nullptr, *pf_xm = nullptr, *pf_xl = nullptr, *pf_wh = nullptr, *pf_wl = nullptr;
  int32_t *pf_tok = nullptr;
  // few-slot step: its own phase list and graph (always the kernel chain)
  std::vector<Phase> slot_phases;
  cudaGraphExec_t slot_graph = nullptr;
  bool slot_graph_ok = true, slot_primed = false;
  int slot_launches = 0;

  void *dalloc(size_t bytes) {
    void *p = nullptr;
    if (cudaMalloc(&p, bytes ? bytes : 16) != cudaSuccess) return nullptr;
    allocs.push_back(p);
    return p;
  }
};

// Tagged words of one layer's phase outputs (each vector rounded up to whole 16-byte
// pairs): q|k|v, attention output, x after O-proj, SwiGLU activation, x after down.
static int64_t even_words(int64_t n) { return (n + 1) / 2 * 2; }
static int64_t tagged_layer_words(const mie_config &c) {
  return even_words((int64_t)(c.n_heads + 2 * c.n_kv_heads) * c.head_dim) +
         even_words((int64_t)c.n_heads * c.head_dim) + 2 * even_words(c.d_model) + even_words(c.ffn);
}

// Every tagged word back to tag 0 (no launch writes it) and the next tag to 1.
static cudaError_t reset_tags(mie_ctx *ctx) {
  static const unsigned init[2] = {1u, 0u};
  cudaError_t e = cudaMemsetAsync(ctx->tagged, 0, sizeof(uint64_t) * ctx->tagged_words, ctx->stream);
  if (e == cudaSuccess) e = cudaMemcpyAsync(ctx->epoch, init, sizeof init, cudaMemcpyHostToDevice, ctx->stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(ctx->stream);
  return e;
}

static mie_status check_config(const mie_config &c) {
  if (c.n_layers < 1 || c.d_model < 1 || c.n_heads < 1 || c.n_kv_heads < 1 || c.head_dim < 1 || c.ffn < 1 ||
      c.vocab < 1)
    return fail(MIE_E_ARG, "mie_create: non-positive model dimension");
  if (c.n_heads % c.n_kv_heads) return fail(MIE_E_SHAPE, "mie_create: n_heads %% n_kv_heads != 0");
  const int G = c.n_heads / c.n_kv_heads;
  if (G != 1 && G != 2 && G != 4 && G != 8) return fail(MIE_E_SHAPE, "mie_create: group size %d", G);
  if (c.head_dim != 32 && c.head_dim != 64 && c.head_dim != 128)
    return fail(MIE_E_SHAPE, "mie_create: head_dim %d", c.head_dim);
  if (c.block_size != 8 && c.block_size != 16 && c.block_size != 32)
    return fail(MIE_E_SHAPE, "mie_create: block_size %d", c.block_size);
  const int kmax = 16384;
  if (c.d_model > kmax || c.ffn > kmax || c.n_heads * c.head_dim > kmax)
    return fail(MIE_E_SHAPE, "mie_create: a GEMV input is longer than %d", kmax);
  if (c.max_slots < 1 || c.max_slots > kMaxSlots) return fail(MIE_E_SHAPE, "mie_create: max_slots %d", c.max_slots);
  if (c.n_kv_blocks < 1 || c.max_pos < 1) return fail(MIE_E_ARG, "mie_create: n_kv_blocks / max_pos");
  auto stored = [](int f) { return f == MIE_FMT_BF16 || f == MIE_FMT_I8 || q4_group(f) != 0; };
  for (int f : {c.wfmt, c.head_fmt})
    if (!stored(f)) return fail(MIE_E_ARG, "mie_create: format %d", f);
  if (!c.tied && !stored(c.embed_fmt))
    return fail(MIE_E_ARG, "mie_create: embed format %d", c.embed_fmt);
  return MIE_OK;
}

extern "C" void mie_destroy(mie_ctx *ctx) {
  if (!ctx) return;
  if (ctx->stream) cudaStreamSynchronize(ctx->stream);
  if (ctx->graph) cudaGraphExecDestroy(ctx->graph);
  if (ctx->slot_graph) cudaGraphExecDestroy(ctx->slot_graph);
  for (void *p : ctx->allocs) cudaFree(p);
  for (cudaEvent_t ev : ctx->sp_uploaded)
    if (ev) cudaEventDestroy(ev);
  if (ctx->sp_pinned) cudaFreeHost(ctx->sp_pinned);
  if (ctx->next_pinned) cudaFreeHost(ctx->next_pinned);
  if (ctx->own_stream && ctx->stream) cudaStreamDestroy(ctx->stream);
  mie_pool_destroy(ctx->pool);
  delete ctx;
}

extern "C" mie_status mie_create(const mie_config *cfg, void *stream, mie_ctx **out) {
  if (!cfg || !out) return fail(MIE_E_ARG, "mie_create: null pointer");
  *out = nullptr;
  mie_status s = check_config(*cfg);
  if (s != MIE_OK) return s;
  mie_ctx *ctx = new (std::nothrow) mie_ctx;
  if (!ctx) return fail(MIE_E_OOM, "mie_create: host allocation");
  ctx->cfg = *cfg;
  const mie_config &c = ctx->cfg;
  if (stream) {
    ctx->stream = (cudaStream_t)stream;
  } else {
    if (cudaStreamCreateWithFlags(&ctx->stream, cudaStreamNonBlocking) != cudaSuccess) {
      delete ctx;
      return fail(MIE_E_CUDA, "mie_create: cudaStreamCreate");
    }
    ctx->own_stream = true;
  }
  ctx->layers.resize((size_t)c.n_layers);
  ctx->block_elems = (int64_t)c.n_layers * 2 * c.n_kv_heads * c.block_size * c.head_dim;
  const size_t kv_bytes = (size_t)c.n_kv_blocks * ctx->block_elems * 2;
  const int S = c.max_slots;
  ctx->kv = (uint16_t *)ctx->dalloc(kv_bytes);
  ctx->x = (float *)ctx->dalloc(sizeof(float) * S * c.d_model);
  ctx->q = (float *)ctx->dalloc(sizeof(float) * S * c.n_heads * c.head_dim);
  ctx->att = (float *)ctx->dalloc(sizeof(float) * S * c.n_heads * c.head_dim);
  ctx->act = (float *)ctx->dalloc(sizeof(float) * S * c.ffn);
  ctx->rope_cos = (float *)ctx->dalloc(sizeof(float) * (size_t)c.max_pos * (c.head_dim / 2));
  ctx->rope_sin = (float *)ctx->dalloc(sizeof(float) * (size_t)c.max_pos * (c.head_dim / 2));
  ctx->attn_splits = attn_splits_for(c.n_kv_heads, c.max_pos, c.block_size);
  // per layer: split counters of the attention units (query heads or KV heads), then the
  // split partials (m, l, o) of every query head
  ctx->attn_ws_bytes = attn_counter_bytes(c.n_heads) +
                       (size_t)c.n_heads * ctx->attn_splits * (2 + c.head_dim) * sizeof(float);
  const size_t aws_total = ctx->attn_ws_bytes * c.n_layers * S;
  uint8_t *ws = (uint8_t *)ctx->dalloc(aws_total);
  ctx->tagged_words = tagged_layer_words(c) * c.n_layers;
  ctx->tagged = (uint64_t *)ctx->dalloc(sizeof(uint64_t) * ctx->tagged_words);
  ctx->am_part = (float2 *)ctx->dalloc(sizeof(float2) * 4 * sm_count() * S);
  ctx->am_count = (unsigned *)ctx->dalloc(sizeof(unsigned) * 64);
  ctx->sp = (StepParams *)ctx->dalloc(sizeof(StepParams));
  ctx->err = (int *)ctx->dalloc(sizeof(int) * 4);
  ctx->epoch = (unsigned *)ctx->dalloc(sizeof(unsigned) * 2);
  ctx->abort = (int *)ctx->dalloc(sizeof(int));
  std::vector<float> ones((size_t)c.d_model, 1.0f);
  for (auto &L : ctx->layers) {
    L.attn_norm = (float *)ctx->dalloc(sizeof(float) * c.d_model);
    L.mlp_norm = (float *)ctx->dalloc(sizeof(float) * c.d_model);
  }
  ctx->final_norm = (float *)ctx->dalloc(sizeof(float) * c.d_model);
  bool ok = ctx->kv && ctx->x && ctx->q && ctx->att && ctx->act && ctx->rope_cos && ctx->rope_sin && ws &&
            ctx->am_part && ctx->am_count && ctx->sp && ctx->err && ctx->final_norm && ctx->tagged && ctx->epoch &&
            ctx->abort;
  for (auto &L : ctx->layers) ok = ok && L.attn_norm && L.mlp_norm;
  if (!ok) {
    mie_destroy(ctx);
    return fail(MIE_E_OOM, "mie_create: device allocation of %zu KV bytes failed", kv_bytes);
  }
  if (cudaMallocHost((void **)&ctx->sp_pinned, sizeof(StepParams) * mie_ctx::kParamRing) != cudaSuccess) {
    ctx->sp_pinned = nullptr;
    mie_destroy(ctx);
    return fail(MIE_E_OOM, "mie_create: pinned host allocation of the step parameters");
  }
  for (cudaEvent_t &ev : ctx->sp_uploaded) {
    const cudaError_t r = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
    if (r != cudaSuccess) {
      ev = nullptr;
      mie_destroy(ctx);
      return cuda_fail(r, "mie_create: cudaEventCreate");
    }
  }
  ctx->attn_ws = ws;
  cudaError_t e = cudaSuccess;
  auto chk = [&](cudaError_t r) { if (e == cudaSuccess) e = r; };
  chk(cudaMemsetAsync(ctx->kv, 0, kv_bytes, ctx->stream));
  chk(cudaMemsetAsync(ws, 0, aws_total, ctx->stream));
  chk(reset_tags(ctx));
  chk(cudaMemsetAsync(ctx->am_count, 0, sizeof(unsigned) * 64, ctx->stream));
  chk(cudaMemsetAsync(ctx->err, 0, sizeof(int) * 4, ctx->stream));
  chk(cudaMemsetAsync(ctx->sp, 0, sizeof(StepParams), ctx->stream));
  chk(cudaMemsetAsync(ctx->abort, 0, sizeof(int), ctx->stream));
  for (auto &L : ctx->layers) {
    chk(cudaMemcpyAsync(L.attn_norm, ones.data(), sizeof(float) * c.d_model, cudaMemcpyHostToDevice, ctx->stream));
    chk(cudaMemcpyAsync(L.mlp_norm, ones.data(), sizeof(float) * c.d_model, cudaMemcpyHostToDevice, ctx->stream));
  }
  chk(cudaMemcpyAsync(ctx->final_norm, ones.data(), sizeof(float) * c.d_model, cudaMemcpyHostToDevice, ctx->stream));
  if (e != cudaSuccess) {
    mie_destroy(ctx);
    return cuda_fail(e, "mie_create: initialisation");
  }
  s = launch_rope_table(ctx->rope_cos, ctx->rope_sin, c.max_pos, c.head_dim, (double)c.rope_theta, ctx->stream);
  if (s == MIE_OK && cudaStreamSynchronize(ctx->stream) != cudaSuccess) s = fail(MIE_E_CUDA, "mie_create: sync");
  if (s == MIE_OK) s = mie_pool_create(c.n_kv_blocks, &ctx->pool);
  if (s != MIE_OK) {
    mie_destroy(ctx);
    return s;
  }
  *out = ctx;
  return MIE_OK;
}

// ------------------------------------------------------------------ weight loading

namespace {

// Allocates a matrix in its GPU layout (zero-filled so padding reads as zeros).
mie_status alloc_mat(mie_ctx *ctx, DevMat &m, int fmt, int rows, int cols) {
  m.pub_fmt = fmt;
  m.fmt = q4_group(fmt) ? MIE_FMT_Q4_0 : fmt;  // every 4-bit group size runs as Q4_0 with a group shift
  m.rows = rows;
  m.cols = cols;
  size_t wbytes = 0, sbytes = 0;
  if (fmt == MIE_FMT_BF16) {
    m.kp = pad_to(cols, 8);
    m.row_bytes = (int64_t)m.kp * 2;
  } else if (fmt == MIE_FMT_I8) {
    m.kp = pad_to(cols, 16);
    m.row_bytes = m.kp;
    sbytes = sizeof(float) * rows;
  } else {
    const int group = q4_group(fmt);
    m.gshift = q4_gshift(group);
    m.kp = pad_to(cols, group);  // whole groups
    m.row_bytes = (int64_t)(m.kp / 32) * 16;
    m.s_stride = q4_scale_stride(m.kp / group);
    sbytes = sizeof(__half) * (size_t)rows * m.s_stride;
  }
  wbytes = (size_t)rows * m.row_bytes;
  uint8_t *w = (uint8_t *)ctx->dalloc(wbytes);
  void *s = sbytes ? ctx->dalloc(sbytes) : nullptr;
  if (!w || (sbytes && !s)) return fail(MIE_E_OOM, "weights: device allocation of %zu bytes", wbytes + sbytes);
  if (cudaMemsetAsync(w, 0, wbytes, ctx->stream) != cudaSuccess) return fail(MIE_E_CUDA, "weights: memset");
  if (s && cudaMemsetAsync(s, 0, sbytes, ctx->stream) != cudaSuccess) return fail(MIE_E_CUDA, "weights: memset");
  m.w = w;
  m.s = s;
  return MIE_OK;
}

struct Temp {
  std::vector<void *> p;
  ~Temp() {
    for (void *q : p) cudaFree(q);
  }
  void *get(size_t n) {
    void *q = nullptr;
    if (cudaMalloc(&q, n ? n : 16) != cudaSuccess) return nullptr;
    p.push_back(q);
    return q;
  }
};

// Writes source rows [rows][cols] given as host data in `fmt` (F32 or the matrix's own
// canonical format) into matrix m, source row r landing on row map[r].
mie_status fill_mat_body(mie_ctx *ctx, Temp &tmp, DevMat &m, int fmt, const void *host, size_t bytes,
                         const float *host_scale, int rows, int cols, const std::vector<int> &map) {
  cudaStream_t st = ctx->stream;
  const int group = q4_group(m.pub_fmt), ng = group ? (cols + group - 1) / group : 0;
  size_t expect = 0;
  if (fmt == MIE_FMT_F32) expect = (size_t)rows * cols * 4;
  else if (fmt == MIE_FMT_BF16) expect = (size_t)rows * cols * 2;
  else if (fmt == MIE_FMT_I8) expect = (size_t)rows * cols;
  else if (q4_group(fmt)) expect = (size_t)rows * ng * (2 + group / 2);
  if (fmt != MIE_FMT_F32 && fmt != m.pub_fmt)
    return fail(MIE_E_ARG, "weights: host format %d is neither F32 nor the tensor's format %d", fmt, m.pub_fmt);
  if (bytes != expect) return fail(MIE_E_ARG, "weights: %zu bytes given, %zu expected", bytes, expect);
  if (fmt == MIE_FMT_I8 && !host_scale) return fail(MIE_E_ARG, "weights: int8 data without row scales");
  void *src = tmp.get(bytes);
  int *dmap = nullptr;
  if (!map.empty()) dmap = (int *)tmp.get(sizeof(int) * map.size());
  if (!src || (!map.empty() && !dmap)) return fail(MIE_E_OOM, "weights: staging allocation");
  MIE_CUDA(cudaMemcpyAsync(src, host, bytes, cudaMemcpyHostToDevice, st));
  if (dmap) MIE_CUDA(cudaMemcpyAsync(dmap, map.data(), sizeof(int) * map.size(), cudaMemcpyHostToDevice, st));
  // bring the data into the canonical layout of the matrix's format
  const void *canon = src;
  const float *canon_scale = nullptr;
  mie_status s = MIE_OK;
  if (m.fmt == MIE_FMT_BF16) {
    if (fmt == MIE_FMT_F32) {
      uint16_t *b = (uint16_t *)tmp.get((size_t)rows * cols * 2);
      if (!b) return fail(MIE_E_OOM, "weights: staging allocation");
      if ((s = launch_convert_bf16((const float *)src, (int64_t)rows * cols, b, st)) != MIE_OK) return s;
      canon = b;
    }
    return launch_pad_rows((const uint8_t *)canon, (int64_t)cols * 2, const_cast<uint8_t *>(m.w), m.row_bytes, rows,
                           dmap, st);
  }
  if (m.fmt == MIE_FMT_I8) {
    float *sc = (float *)tmp.get(sizeof(float) * rows);
    if (!sc) return fail(MIE_E_OOM, "weights: staging allocation");
    if (fmt == MIE_FMT_F32) {
      int8_t *q = (int8_t *)tmp.get((size_t)rows * cols);
      if (!q) return fail(MIE_E_OOM, "weights: staging allocation");
      if ((s = launch_quantize_i8((const float *)src, rows, cols, q, sc, st)) != MIE_OK) return s;
      canon = q;
    } else {
      MIE_CUDA(cudaMemcpyAsync(sc, host_scale, sizeof(float) * rows, cudaMemcpyHostToDevice, st));
    }
    canon_scale = sc;
    if ((s = launch_pad_rows((const uint8_t *)canon, cols, const_cast<uint8_t *>(m.w), m.row_bytes, rows, dmap, st)) !=
        MIE_OK)
      return s;
    return launch_pad_rows((const uint8_t *)canon_scale, 4, (uint8_t *)const_cast<void *>(m.s), 4, rows, dmap, st);
  }
  // 4-bit groups
  if (fmt == MIE_FMT_F32) {
    uint8_t *b = (uint8_t *)tmp.get((size_t)rows * ng * (2 + group / 2));
    if (!b) return fail(MIE_E_OOM, "weights: staging allocation");
    if ((s = launch_quantize_q4((const float *)src, rows, cols, group, b, st)) != MIE_OK) return s;
    canon = b;
  }
  if (m.kp / group != ng) return fail(MIE_E_SHAPE, "weights: 4-bit group count mismatch");
  return launch_q4_pack((const uint8_t *)canon, rows, cols, group, const_cast<uint8_t *>(m.w),
                        (__half *)const_cast<void *>(m.s), m.s_stride, dmap, st);
}

mie_status fill_mat(mie_ctx *ctx, DevMat &m, int fmt, const void *host, size_t bytes, const float *host_scale, int rows,
                    int cols, const std::vector<int> &map) {
  Temp tmp;
  const mie_status s = fill_mat_body(ctx, tmp, m, fmt, host, bytes, host_scale, rows, cols, map);
  // the staging buffers are freed on return: let the work that reads them finish
  const cudaError_t e = cudaStreamSynchronize(ctx->stream);
  if (s != MIE_OK) return s;
  if (e != cudaSuccess) return cuda_fail(e, "weights: cudaStreamSynchronize");
  return MIE_OK;
}

}  // namespace

extern "C" mie_status mie_load_weights(mie_ctx *ctx, const char *name, int fmt, const void *host_data, size_t bytes,
                                       const int64_t *shape, int ndim, const float *host_scale) {
  if (!ctx || !name || !host_data || !shape) return fail(MIE_E_ARG, "mie_load_weights: null pointer");
  const mie_config &c = ctx->cfg;
  std::string n(name);
  // norm gains
  auto load_gain = [&](float *dst) -> mie_status {
    if (fmt != MIE_FMT_F32 || ndim != 1 || shape[0] != c.d_model || bytes != sizeof(float) * c.d_model)
      return fail(MIE_E_ARG, "mie_load_weights(%s): gains are fp32 [d_model]", name);
    MIE_CUDA(cudaMemcpyAsync(dst, host_data, bytes, cudaMemcpyHostToDevice, ctx->stream));
    MIE_CUDA(cudaStreamSynchronize(ctx->stream));
    return MIE_OK;
  };
  if (n == "final_norm") return load_gain(ctx->final_norm);
  if (ndim != 2) return fail(MIE_E_ARG, "mie_load_weights(%s): ndim %d", name, ndim);
  const int rows = (int)shape[0], cols = (int)shape[1];
  const int hd = c.head_dim, Hq = c.n_heads, Hkv = c.n_kv_heads, d = c.d_model;
  auto want = [&](int r, int k) -> mie_status {
    if (rows != r || cols != k) return fail(MIE_E_SHAPE, "mie_load_weights(%s): shape %d x %d, expected %d x %d", name, rows, cols, r, k);
    return MIE_OK;
  };
  mie_status s;
  std::vector<int> none;
  ctx->primed = false;  // weights changed: the next step re-captures
  ctx->slot_primed = false;
  if (n == "head" || n == "embed") {
    const bool is_head = n == "head";
    if (!is_head && c.tied) return fail(MIE_E_ARG, "mie_load_weights: tied model has no separate embedding");
    if ((s = want(c.vocab, d)) != MIE_OK) return s;
    DevMat &m = is_head ? ctx->head : ctx->embed;
    if (!m.w && (s = alloc_mat(ctx, m, is_head ? c.head_fmt : c.embed_fmt, rows, cols)) != MIE_OK) return s;
    if ((s = fill_mat(ctx, m, fmt, host_data, bytes, host_scale, rows, cols, none)) != MIE_OK) return s;
    if (is_head) ctx->head_loaded = true;
    else ctx->embed_loaded = true;
    if (is_head && c.tied) {
      ctx->embed = ctx->head;
      ctx->embed_loaded = true;
    }
    MIE_CUDA(cudaStreamSynchronize(ctx->stream));
    return MIE_OK;
  }
  int layer = -1;
  char part[32] = {0};
  if (sscanf(name, "l%d.%31s", &layer, part) != 2 || layer < 0 || layer >= c.n_layers)
    return fail(MIE_E_ARG, "mie_load_weights: unknown tensor name '%s'", name);
  Layer &L = ctx->layers[(size_t)layer];
  std::string p(part);
  if (p == "attn_norm") return load_gain(L.attn_norm);
  if (p == "mlp_norm") return load_gain(L.mlp_norm);
  if (p == "qkv") {
    const int R = (Hq + 2 * Hkv) * hd;
    if ((s = want(R, d)) != MIE_OK) return s;
    // row R' of head h, index i' -> pair slot p = h*hd/2 + i' % (hd/2), half i' / (hd/2)
    std::vector<int> map((size_t)R);
    for (int r = 0; r < R; ++r) {
      const int h = r / hd, i = r % hd, half = hd / 2;
      map[(size_t)r] = 2 * (h * half + (i % half)) + (i >= half ? 1 : 0);
    }
    if (!L.qkv.w && (s = alloc_mat(ctx, L.qkv, c.wfmt, R, d)) != MIE_OK) return s;
    if ((s = fill_mat(ctx, L.qkv, fmt, host_data, bytes, host_scale, rows, cols, map)) != MIE_OK) return s;
    L.loaded[T_QKV] = true;
  } else if (p == "o") {
    if ((s = want(d, Hq * hd)) != MIE_OK) return s;
    if (!L.o.w && (s = alloc_mat(ctx, L.o, c.wfmt, d, Hq * hd)) != MIE_OK) return s;
    if ((s = fill_mat(ctx, L.o, fmt, host_data, bytes, host_scale, rows, cols, none)) != MIE_OK) return s;
    L.loaded[T_O] = true;
  } else if (p == "gate" || p == "up") {
    if ((s = want(c.ffn, d)) != MIE_OK) return s;
    std::vector<int> map((size_t)c.ffn);
    const int which = p == "up" ? 1 : 0;
    for (int r = 0; r < c.ffn; ++r) map[(size_t)r] = 2 * r + which;
    if (!L.gu.w && (s = alloc_mat(ctx, L.gu, c.wfmt, 2 * c.ffn, d)) != MIE_OK) return s;
    if ((s = fill_mat(ctx, L.gu, fmt, host_data, bytes, host_scale, rows, cols, map)) != MIE_OK) return s;
    L.loaded[which ? T_UP : T_GATE] = true;
  } else if (p == "down") {
    if ((s = want(d, c.ffn)) != MIE_OK) return s;
    if (!L.down.w && (s = alloc_mat(ctx, L.down, c.wfmt, d, c.ffn)) != MIE_OK) return s;
    if ((s = fill_mat(ctx, L.down, fmt, host_data, bytes, host_scale, rows, cols, none)) != MIE_OK) return s;
    L.loaded[T_DOWN] = true;
  } else {
    return fail(MIE_E_ARG, "mie_load_weights: unknown tensor name '%s'", name);
  }
  MIE_CUDA(cudaStreamSynchronize(ctx->stream));
  return MIE_OK;
}

extern "C" mie_pool *mie_ctx_pool(mie_ctx *ctx) { return ctx ? ctx->pool : nullptr; }
extern "C" uint16_t *mie_kv_pool(mie_ctx *ctx) { return ctx ? ctx->kv : nullptr; }
extern "C" int64_t mie_kv_block_elems(const mie_ctx *ctx) { return ctx ? ctx->block_elems : 0; }

extern "C" mie_status mie_kv_copy_block(mie_ctx *ctx, int32_t src, int32_t dst) {
  if (!ctx) return fail(MIE_E_ARG, "mie_kv_copy_block: null context");
  if (src < 0 || dst < 0 || src >= ctx->cfg.n_kv_blocks || dst >= ctx->cfg.n_kv_blocks)
    return fail(MIE_E_ARG, "mie_kv_copy_block: block %d -> %d out of range", src, dst);
  const size_t bytes = (size_t)ctx->block_elems * 2;
  MIE_CUDA(cudaMemcpyAsync(ctx->kv + (int64_t)dst * ctx->block_elems, ctx->kv + (int64_t)src * ctx->block_elems, bytes,
                           cudaMemcpyDeviceToDevice, ctx->stream));
  return MIE_OK;
}

// Copy-on-write in the order that keeps the shared block alive until its copy is
// queued: split (the sequence still holds the shared block), queue the copy, release.
extern "C" mie_status mie_kv_writable(mie_ctx *ctx, int32_t *table, int pos, int32_t *block) {
  if (!ctx || !table || !block) return fail(MIE_E_ARG, "mie_kv_writable: null pointer");
  int32_t src = -1, dst = -1;
  mie_status s = mie_pool_writable(ctx->pool, table, pos, ctx->cfg.block_size, block, &src, &dst);
  if (s != MIE_OK || src < 0) return s;
  if ((s = mie_kv_copy_block(ctx, src, dst)) != MIE_OK) return s;
  return mie_pool_decref(ctx->pool, src);
}

// ------------------------------------------------------------------ the step

static bool all_loaded(const mie_ctx *ctx) {
  if (!ctx->head_loaded || !ctx->embed_loaded) return false;
  for (const auto &L : ctx->layers)
    for (bool b : L.loaded)
      if (!b) return false;
  return true;
}

// The step's phases for slot 0, in execution order.
static void build_phases(mie_ctx *ctx, std::vector<Phase> &out) {
  const mie_config &c = ctx->cfg;
  out.clear();
  const int64_t half = (int64_t)c.n_kv_heads * c.block_size * c.head_dim;
  // the persistent step's tagged vectors of each layer, and the previous layer's x
  const int64_t w_qkv = even_words((int64_t)(c.n_heads + 2 * c.n_kv_heads) * c.head_dim);
  const int64_t w_att = even_words((int64_t)c.n_heads * c.head_dim), w_d = even_words(c.d_model);
  const uint64_t *x_prev = nullptr;  // layer 0 reads the embedding instead
  for (int l = 0; l < c.n_layers; ++l) {
    Layer &L = ctx->layers[(size_t)l];
    uint16_t *kv_layer = ctx->kv + (int64_t)l * 2 * half;
    uint64_t *t_qkv = ctx->tagged + (int64_t)l * tagged_layer_words(c);
    uint64_t *t_att = t_qkv + w_qkv, *t_x1 = t_att + w_att, *t_act = t_x1 + w_d, *t_x2 = t_act + even_words(c.ffn);
    uint8_t *ws = ctx->attn_ws + (size_t)l * ctx->attn_ws_bytes;
    Phase qkv;  // qkv + RoPE + K/V write (layer 0 gathers the embedding first)
    qkv.kind = PH_GEMV;
    qkv.pro = l == 0 ? PRO_EMBED_NORM : PRO_NORM;
    qkv.epi = EPI_QKV;
    GemvArgs &a = qkv.g;
    a.m = L.qkv;
    a.x = ctx->x;
    a.gain = L.attn_norm;
    a.eps = c.rms_eps;
    a.act_bf16 = c.act_bf16;
    a.embed = ctx->embed;
    a.x_store = ctx->x;
    a.vocab = c.vocab;
    a.q_out = ctx->q;
    a.kv_layer = kv_layer;
    a.block_stride = ctx->block_elems;
    a.n_kv_blocks = c.n_kv_blocks;
    a.rope_cos = ctx->rope_cos;
    a.rope_sin = ctx->rope_sin;
    a.max_pos = c.max_pos;
    a.Hq = c.n_heads;
    a.Hkv = c.n_kv_heads;
    a.hd = c.head_dim;
    a.bs = c.block_size;
    a.sp = ctx->sp;
    a.err = ctx->err;
    a.x_t = x_prev;
    a.y_t = t_qkv;
    out.push_back(qkv);

    Phase at;
    at.kind = PH_ATTN;
    AttnArgs &t = at.at;
    t.q = ctx->q;
    t.k = kv_layer;
    t.v = kv_layer + half;
    t.block_stride = ctx->block_elems;
    t.n_pool_blocks = c.n_kv_blocks;
    t.sp = ctx->sp;
    t.Hq = c.n_heads;
    t.Hkv = c.n_kv_heads;
    t.hd = c.head_dim;
    t.bs = c.block_size;
    t.scale = (float)(1.0 / std::sqrt((double)c.head_dim));
    t.out = ctx->att;
    t.ws_count = reinterpret_cast<unsigned *>(ws);
    t.ws_part = reinterpret_cast<float *>(ws + attn_counter_bytes(c.n_heads));
    t.n_splits = ctx->attn_splits;
    t.err = ctx->err;
    t.qkv_t = t_qkv;
    t.out_t = t_att;
    out.push_back(at);

    Phase o;  // x += Wo att
    o.kind = PH_GEMV;
    o.pro = PRO_PLAIN;
    o.epi = EPI_RESID;
    o.g.m = L.o;
    o.g.x = ctx->att;
    o.g.act_bf16 = c.act_bf16;
    o.g.y = ctx->x;
    o.g.err = ctx->err;
    o.g.x_t = t_att;
    o.g.res_t = x_prev;
    o.g.embed = ctx->embed;
    o.g.y_t = t_x1;
    out.push_back(o);

    Phase gu;  // act = silu(Wg n(x)) * (Wu n(x))
    gu.kind = PH_GEMV;
    gu.pro = PRO_NORM;
    gu.epi = EPI_SWIGLU;
    gu.g.m = L.gu;
    gu.g.x = ctx->x;
    gu.g.gain = L.mlp_norm;
    gu.g.eps = c.rms_eps;
    gu.g.act_bf16 = c.act_bf16;
    gu.g.y = ctx->act;
    gu.g.err = ctx->err;
    gu.g.x_t = t_x1;
    gu.g.y_t = t_act;
    out.push_back(gu);

    Phase dn;  // x += Wd act
    dn.kind = PH_GEMV;
    dn.pro = PRO_PLAIN;
    dn.epi = EPI_RESID;
    dn.g.m = L.down;
    dn.g.x = ctx->act;
    dn.g.act_bf16 = c.act_bf16;
    dn.g.y = ctx->x;
    dn.g.err = ctx->err;
    dn.g.x_t = t_act;
    dn.g.res_t = t_x1;
    dn.g.y_t = t_x2;
    out.push_back(dn);
    x_prev = t_x2;
  }
  Phase hd;  // logits = Whead n(x); argmax
  hd.kind = PH_GEMV;
  hd.pro = PRO_NORM;
  hd.epi = EPI_ARGMAX;
  hd.g.m = ctx->head;
  hd.g.x = ctx->x;
  hd.g.gain = ctx->final_norm;
  hd.g.eps = c.rms_eps;
  hd.g.act_bf16 = c.act_bf16;
  hd.g.am_part = ctx->am_part;
  hd.g.am_count = ctx->am_count;
  hd.g.sp = ctx->sp;
  hd.g.err = ctx->err;
  hd.g.x_t = x_prev;
  out.push_back(hd);
}

// Enqueues one decode step (the graph body) and counts its kernel launches.
static mie_status enqueue_step(mie_ctx *ctx, int *launches) {
  cudaStream_t st = ctx->stream;
  mie_status s;
  if (ctx->mode == MIE_STEP_PERSISTENT) {
    PersistArgs pa;
    pa.ph = ctx->d_phases;
    pa.n_phases = (int)ctx->phases.size();
    pa.epoch = ctx->epoch;
    pa.fin = ctx->epoch + 1;
    pa.abort = ctx->abort;
    pa.n_slots = ctx->plan.n_slots;
    pa.slot_bytes = ctx->plan.slot_bytes;
    pa.slot_sc_bytes = ctx->plan.slot_sc_bytes;
    pa.err = ctx->err;
    const size_t need = sizeof(unsigned long long) * ctx->phases.size() * ctx->plan.grid * kTracePoints;
    // per-stage stamps, then (instrumented build) 8 points per phase and CTA
    const size_t need_st = sizeof(unsigned long long) * ctx->plan.grid *
                           ((size_t)kStageTrace * kStagePoints + ctx->phases.size() * 8);
    pa.trace = (ctx->trace && ctx->trace_bytes >= need) ? ctx->trace : nullptr;
    pa.stage_trace = (pa.trace && ctx->trace_bytes >= need + need_st) ? ctx->trace + need / 8 : nullptr;
    pa.wait_polls = ctx->wait_polls;
    if ((s = persist_launch(ctx->plan, pa, st)) != MIE_OK) return s;
    *launches = 1;
  } else {
    int n = 0;
    for (const Phase &ph : ctx->phases) {
      if (ph.kind == PH_GEMV) s = launch_gemv(ph.pro, ph.epi, ph.g, gemv_default_grid(ph.g.m, ph.epi), st, true);
      else s = launch_attn(ph.at, st, true);
      if (s != MIE_OK) return s;
      ++n;
    }
    *launches = n;
  }
  if (ctx->temperature > 0.f) {  // the draw replaces the head's argmax as the next token
    const mie_config &c = ctx->cfg;
    if ((s = launch_step_sample(ctx->sp, c.vocab, ctx->temperature, ctx->top_k, ctx->top_p, ctx->seed,
                                ctx->sample_ws, st)) != MIE_OK)
      return s;
    *launches += sample_launches(ctx->temperature, ctx->top_k, ctx->top_p, c.vocab);
  }
  return MIE_OK;
}

// Builds the phase list, uploads it and plans the persistent kernel; a shape the
// persistent kernel does not cover falls back to the kernel chain.
static mie_status prepare_step(mie_ctx *ctx) {
  build_phases(ctx, ctx->phases);
  if (ctx->stall_phase >= 0 && ctx->stall_phase < (int)ctx->phases.size()) {
    Phase &ph = ctx->phases[(size_t)ctx->stall_phase];
    if (ph.kind == PH_GEMV) ph.g.x_t = ctx->stall_words;
    else ph.at.qkv_t = ctx->stall_words;
  }
  const size_t bytes = sizeof(Phase) * ctx->phases.size();
  if (ctx->d_phases_cap < bytes) {
    Phase *p = (Phase *)ctx->dalloc(bytes);
    if (!p) return fail(MIE_E_OOM, "decode step: phase table");
    ctx->d_phases = p;
    ctx->d_phases_cap = bytes;
  }
  MIE_CUDA(cudaMemcpyAsync(ctx->d_phases, ctx->phases.data(), bytes, cudaMemcpyHostToDevice, ctx->stream));
  MIE_CUDA(cudaStreamSynchronize(ctx->stream));
  if (ctx->mode == MIE_STEP_PERSISTENT &&
      persist_plan(ctx->phases.data(), (int)ctx->phases.size(), ctx->cfg.n_heads / ctx->cfg.n_kv_heads,
                   ctx->cfg.head_dim, &ctx->plan) != MIE_OK) {
    cudaGetLastError();
    ctx->mode = MIE_STEP_CHAIN;  // a shape the persistent kernel does not cover
  }
  return MIE_OK;
}

static mie_status capture(mie_ctx *ctx) {
  if (ctx->graph) {
    cudaGraphExecDestroy(ctx->graph);
    ctx->graph = nullptr;
  }
  mie_status s = prepare_step(ctx);
  if (s != MIE_OK) return s;
  ctx->graph_ok = true;
  cudaGraph_t g = nullptr;
  MIE_CUDA(cudaStreamBeginCapture(ctx->stream, cudaStreamCaptureModeThreadLocal));
  int n = 0;
  s = enqueue_step(ctx, &n);
  cudaError_t e = cudaStreamEndCapture(ctx->stream, &g);
  if (s == MIE_OK && e == cudaSuccess) e = cudaGraphInstantiate(&ctx->graph, g, 0);
  if (g) cudaGraphDestroy(g);
  if (s != MIE_OK || e != cudaSuccess) {
    // the launch is not capturable here: run the step without a graph
    cudaGetLastError();
    ctx->graph = nullptr;
    ctx->graph_ok = false;
  }
  ctx->launches = n;
  ctx->primed = true;
  return MIE_OK;
}

static mie_status run_step(mie_ctx *ctx) {
  if (ctx->graph_ok && ctx->graph) {
    MIE_CUDA(cudaGraphLaunch(ctx->graph, ctx->stream));
    return MIE_OK;
  }
  int n = 0;
  return enqueue_step(ctx, &n);
}

// Copies the step parameters to the device from the next pinned buffer of the ring.
static mie_status upload_params(mie_ctx *ctx, const StepParams &p) {
  const int i = ctx->sp_next;
  ctx->sp_next = (i + 1) % mie_ctx::kParamRing;
  MIE_CUDA(cudaEventSynchronize(ctx->sp_uploaded[i]));  // the buffer's previous upload has run
  ctx->sp_pinned[i] = p;
  MIE_CUDA(cudaMemcpyAsync(ctx->sp, ctx->sp_pinned + i, sizeof p, cudaMemcpyHostToDevice, ctx->stream));
  MIE_CUDA(cudaEventRecord(ctx->sp_uploaded[i], ctx->stream));
  return MIE_OK;
}

extern "C" mie_status mie_decode_step(mie_ctx *ctx, int32_t token, int32_t pos, const int32_t *block_table,
                                      int n_blocks, float *logits_out, int32_t *argmax_out) {
  if (!ctx || !block_table) return fail(MIE_E_ARG, "mie_decode_step: null pointer");
  const mie_config &c = ctx->cfg;
  if (!all_loaded(ctx)) return fail(MIE_E_STATE, "mie_decode_step: not every weight is loaded");
  if (token < 0 || token >= c.vocab) return fail(MIE_E_ARG, "mie_decode_step: token %d outside [0, %d)", token, c.vocab);
  if (pos < 0 || pos >= c.max_pos) return fail(MIE_E_ARG, "mie_decode_step: pos %d outside [0, %d)", pos, c.max_pos);
  if (n_blocks < 1 || pos / c.block_size >= n_blocks)
    return fail(MIE_E_ARG, "mie_decode_step: pos %d needs more than %d blocks", pos, n_blocks);
  StepParams p;
  memset(&p, 0, sizeof p);
  p.token[0] = token;
  p.pos[0] = pos;
  p.block_table = block_table;
  p.max_blocks = n_blocks;
  p.n_slots = 1;
  p.logits_out = logits_out;
  p.argmax_out = argmax_out;
  p.advance = 1;
  if (ctx->temperature > 0.f) {  // the sampler reads the logits and advances instead
    if (!p.logits_out) p.logits_out = ctx->logits_buf;
    p.advance = 0;
    p.sample_advance = 1;
  }
  const mie_status su = upload_params(ctx, p);
  if (su != MIE_OK) return su;
  if (!ctx->primed) {
    mie_status s = capture(ctx);
    if (s != MIE_OK) return s;
  }
  return run_step(ctx);
}

extern "C" mie_status mie_decode_step_sync(mie_ctx *ctx, int32_t token, int32_t pos, const int32_t *block_table,
                                           int n_blocks, float *logits_out, int32_t *next_token) {
  if (!ctx || !next_token) return fail(MIE_E_ARG, "mie_decode_step_sync: null pointer");
  if (!ctx->gen_argmax && !(ctx->gen_argmax = (int32_t *)ctx->dalloc(sizeof(int32_t) * kMaxSlots)))
    return fail(MIE_E_OOM, "mie_decode_step_sync: device buffer");
  if (!ctx->next_pinned && cudaMallocHost((void **)&ctx->next_pinned, sizeof(int32_t)) != cudaSuccess) {
    ctx->next_pinned = nullptr;
    cudaGetLastError();
    return fail(MIE_E_OOM, "mie_decode_step_sync: pinned host buffer");
  }
  const mie_status s = mie_decode_step(ctx, token, pos, block_table, n_blocks, logits_out, ctx->gen_argmax);
  if (s != MIE_OK) return s;
  MIE_CUDA(cudaMemcpyAsync(ctx->next_pinned, ctx->gen_argmax, sizeof(int32_t), cudaMemcpyDeviceToHost, ctx->stream));
  MIE_CUDA(cudaStreamSynchronize(ctx->stream));
  *next_token = *ctx->next_pinned;
  return MIE_OK;
}

extern "C" mie_status mie_decode_continue(mie_ctx *ctx, int n_steps) {
  if (!ctx) return fail(MIE_E_ARG, "mie_decode_continue: null context");
  if (!ctx->primed) return fail(MIE_E_STATE, "mie_decode_continue: call mie_decode_step first");
  if (n_steps < 0) return fail(MIE_E_ARG, "mie_decode_continue: n_steps %d", n_steps);
  for (int i = 0; i < n_steps; ++i) {
    const mie_status s = run_step(ctx);
    if (s != MIE_OK) return s;
  }
  return MIE_OK;
}

// The few-slot step's phases: those of the single-slot step, with attention launched
// as one grid layer per slot (each slot's workspace follows the previous slot's).
static mie_status build_slot_phases(mie_ctx *ctx) {
  build_phases(ctx, ctx->slot_phases);
  for (Phase &ph : ctx->slot_phases) {
    if (ph.kind == PH_ATTN) {
      ph.at.slot_z = 1;
      ph.at.max_slots = ctx->cfg.max_slots;
      ph.at.ws_slot_bytes = ctx->attn_ws_bytes * ctx->cfg.n_layers;
    } else {
      ph.g.sp = ctx->sp;  // every batched GEMV reads the slot count from the step parameters
      const mie_status s = slots_gemv_supported(ph.g.m, ph.pro);
      if (s != MIE_OK) return s;
    }
  }
  return MIE_OK;
}

static mie_status enqueue_slots(mie_ctx *ctx, int *launches) {
  int n = 0;
  for (const Phase &ph : ctx->slot_phases) {
    const mie_status s =
        ph.kind == PH_GEMV ? launch_gemv_slots(ph.pro, ph.epi, ph.g, ctx->stream, true) : launch_attn(ph.at, ctx->stream, true);
    if (s != MIE_OK) return s;
    ++n;
  }
  *launches = n;
  return MIE_OK;
}

static mie_status capture_slots(mie_ctx *ctx) {
  if (ctx->slot_graph) {
    cudaGraphExecDestroy(ctx->slot_graph);
    ctx->slot_graph = nullptr;
  }
  mie_status s = build_slot_phases(ctx);
  if (s != MIE_OK) return s;
  ctx->slot_graph_ok = true;
  cudaGraph_t g = nullptr;
  MIE_CUDA(cudaStreamBeginCapture(ctx->stream, cudaStreamCaptureModeThreadLocal));
  int n = 0;
  s = enqueue_slots(ctx, &n);
  cudaError_t e = cudaStreamEndCapture(ctx->stream, &g);
  if (s == MIE_OK && e == cudaSuccess) e = cudaGraphInstantiate(&ctx->slot_graph, g, 0);
  if (g) cudaGraphDestroy(g);
  if (s != MIE_OK || e != cudaSuccess) {
    cudaGetLastError();
    ctx->slot_graph = nullptr;
    ctx->slot_graph_ok = false;
  }
  ctx->slot_launches = n;
  ctx->slot_primed = true;
  return MIE_OK;
}

extern "C" mie_status mie_decode_step_slots(mie_ctx *ctx, int n_slots, const int32_t *tokens, const int32_t *pos,
                                            const int32_t *block_tables, int max_blocks, float *logits_out,
                                            int32_t *argmax_out) {
  if (!ctx || !tokens || !pos || !block_tables) return fail(MIE_E_ARG, "mie_decode_step_slots: null pointer");
  const mie_config &c = ctx->cfg;
  if (n_slots < 1 || n_slots > c.max_slots)
    return fail(MIE_E_ARG, "mie_decode_step_slots: n_slots %d outside [1, %d]", n_slots, c.max_slots);
  if (max_blocks < 1) return fail(MIE_E_ARG, "mie_decode_step_slots: max_blocks %d", max_blocks);
  if (!all_loaded(ctx)) return fail(MIE_E_STATE, "mie_decode_step_slots: not every weight is loaded");
  for (int s = 0; s < n_slots; ++s) {
    if (tokens[s] < 0 || tokens[s] >= c.vocab)
      return fail(MIE_E_ARG, "mie_decode_step_slots: slot %d token %d outside [0, %d)", s, tokens[s], c.vocab);
    if (pos[s] < 0 || pos[s] >= c.max_pos)
      return fail(MIE_E_ARG, "mie_decode_step_slots: slot %d pos %d outside [0, %d)", s, pos[s], c.max_pos);
    if (pos[s] / c.block_size >= max_blocks)
      return fail(MIE_E_ARG, "mie_decode_step_slots: slot %d pos %d needs more than %d blocks", s, pos[s], max_blocks);
  }
  StepParams p;
  memset(&p, 0, sizeof p);
  for (int s = 0; s < n_slots; ++s) {
    p.token[s] = tokens[s];
    p.pos[s] = pos[s];
  }
  p.block_table = block_tables;
  p.max_blocks = max_blocks;
  p.n_slots = n_slots;
  p.logits_out = logits_out;
  p.argmax_out = argmax_out;
  p.advance = 0;
  const mie_status su = upload_params(ctx, p);
  if (su != MIE_OK) return su;
  if (!ctx->slot_primed) {
    const mie_status s = capture_slots(ctx);
    if (s != MIE_OK) return s;
  }
  if (ctx->slot_graph_ok && ctx->slot_graph) {
    MIE_CUDA(cudaGraphLaunch(ctx->slot_graph, ctx->stream));
    return MIE_OK;
  }
  int n = 0;
  return enqueue_slots(ctx, &n);
}

// k consecutive positions of one sequence as k slots of the few-slot step: slot j is
// token tokens[j] at position pos + j, every slot reading the same block table, so slot j
// attends to the K/V the pass itself wrote for positions pos .. pos + j - 1.
extern "C" mie_status mie_verify_step(mie_ctx *ctx, const int32_t *tokens, int n, int32_t pos,
                                      const int32_t *block_table, int max_blocks, float *logits_out,
                                      int32_t *argmax_out) {
  if (!ctx || !tokens || !block_table) return fail(MIE_E_ARG, "mie_verify_step: null pointer");
  if (n < 1 || n > ctx->cfg.max_slots)
    return fail(MIE_E_ARG, "mie_verify_step: %d positions outside [1, %d]", n, ctx->cfg.max_slots);
  if (max_blocks < 1) return fail(MIE_E_ARG, "mie_verify_step: max_blocks %d", max_blocks);
  if (max_blocks > ctx->verify_cap) {
    int32_t *t = (int32_t *)ctx->dalloc(sizeof(int32_t) * (size_t)kMaxSlots * max_blocks);
    if (!t) return fail(MIE_E_OOM, "mie_verify_step: table copies");
    ctx->verify_table = t;
    ctx->verify_cap = max_blocks;
  }
  for (int s = 0; s < n; ++s)
    MIE_CUDA(cudaMemcpyAsync(ctx->verify_table + (size_t)s * max_blocks, block_table, sizeof(int32_t) * max_blocks,
                             cudaMemcpyDeviceToDevice, ctx->stream));
  int32_t p[kMaxSlots];
  for (int s = 0; s < n; ++s) p[s] = pos + s;
  return mie_decode_step_slots(ctx, n, tokens, p, ctx->verify_table, max_blocks, logits_out, argmax_out);
}

// Greedy generation through the few-slot kernels, speculative when spec_max > 1.
// ------------------------------------------------------------------ prefill

static constexpr int kPrefillChunk = 2048;

static mie_status prefill_alloc(mie_ctx *ctx) {
  if (ctx->pf_R) return MIE_OK;
  const mie_config &c = ctx->cfg;
  const int T = std::min(kPrefillChunk, c.max_pos);
  const int64_t na = (int64_t)c.n_heads * c.head_dim, nqkv = (int64_t)(c.n_heads + 2 * c.n_kv_heads) * c.head_dim;
  const int64_t kmax = std::max<int64_t>(std::max<int64_t>(c.d_model, c.ffn), na);
  ctx->prefill_ldp = (kmax + 7) / 8 * 8;
  const int64_t ny = std::max<int64_t>(nqkv, 2 * (int64_t)c.ffn);
  ctx->pf_R = (float *)ctx->dalloc(sizeof(float) * T * c.d_model);
  ctx->pf_Y = (float *)ctx->dalloc(sizeof(float) * T * ny);
  ctx->pf_Q = (float *)ctx->dalloc(sizeof(float) * T * na);
  ctx->pf_O = (float *)ctx->dalloc(sizeof(float) * T * na);
  ctx->pf_xh = (uint16_t *)ctx->dalloc(2 * T * ctx->prefill_ldp);
  ctx->pf_xm = (uint16_t *)ctx->dalloc(2 * T * ctx->prefill_ldp);
  ctx->pf_xl = (uint16_t *)ctx->dalloc(2 * T * ctx->prefill_ldp);
  ctx->pf_tok = (int32_t *)ctx->dalloc(sizeof(int32_t) * T);
  bool ok = ctx->pf_R && ctx->pf_Y && ctx->pf_Q && ctx->pf_O && ctx->pf_xh && ctx->pf_xm && ctx->pf_xl && ctx->pf_tok;
  if (ok && c.wfmt != MIE_FMT_BF16) {  // the largest layer matrix as bf16 planes
    size_t most = 0;
    for (const Layer &L : ctx->layers)
      for (const DevMat *m : {&L.qkv, &L.o, &L.gu, &L.down})
        most = std::max(most, (size_t)m->rows * (size_t)((m->cols + 7) / 8 * 8));
    ctx->pf_wh = (uint16_t *)ctx->dalloc(2 * most);
    ctx->pf_wl = (uint16_t *)ctx->dalloc(2 * most);
    ok = ctx->pf_wh && ctx->pf_wl;
  }
  if (!ok) {
    ctx->pf_R = nullptr;  // the buffers stay with the context and are freed with it
    return fail(MIE_E_OOM, "mie_prefill: device buffers");
  }
  ctx->prefill_chunk = T;
  return MIE_OK;
}

// y[t][n] (+)= (W x_t)[n] for the T rows of the activation planes, on the tensor cores;
// quantised weights are first expanded to bf16 planes.
static mie_status prefill_gemm(mie_ctx *ctx, const DevMat &m, int T, float *y, int64_t ldy, bool accumulate) {
  cudaStream_t st = ctx->stream;
  GemmPlan p;
  p.T = T;
  p.N = m.rows;
  p.K = m.cols;
  p.y = y;
  p.ldy = ldy;
  p.accumulate = accumulate;
  p.err = ctx->err;
  p.nb = ctx->cfg.act_bf16 ? 1 : 3;
  mie_status s;
  if (m.fmt == MIE_FMT_BF16) {
    p.na = 1;
    s = make_bf16_map(&p.a[0], m.w, m.rows, m.cols, m.row_bytes);
  } else {
    const int64_t ld = (m.cols + 7) / 8 * 8;
    p.na = m.fmt == MIE_FMT_I8 ? 1 : 2;
    if (m.fmt == MIE_FMT_I8) p.row_scale = reinterpret_cast<const float *>(m.s);
    s = launch_dequant_planes(m, ctx->pf_wh, p.na == 2 ? ctx->pf_wl : nullptr, ld, st);
    if (s == MIE_OK) s = make_bf16_map(&p.a[0], ctx->pf_wh, m.rows, m.cols, ld * 2);
    if (s == MIE_OK && p.na == 2) s = make_bf16_map(&p.a[1], ctx->pf_wl, m.rows, m.cols, ld * 2);
  }
  if (s == MIE_OK) s = make_bf16_map(&p.b[0], ctx->pf_xh, T, m.cols, ctx->prefill_ldp * 2);
  if (s == MIE_OK && p.nb == 3) s = make_bf16_map(&p.b[1], ctx->pf_xm, T, m.cols, ctx->prefill_ldp * 2);
  if (s == MIE_OK && p.nb == 3) s = make_bf16_map(&p.b[2], ctx->pf_xl, T, m.cols, ctx->prefill_ldp * 2);
  if (s != MIE_OK) return s;
  return launch_gemm(p, st);
}

// One chunk of T prompt positions pos0 .. pos0 + T - 1 through every layer.  The last
// layer stops after its K/V write: nothing of a prompt position beyond its K/V is kept.
static mie_status prefill_chunk(mie_ctx *ctx, const int32_t *tokens, int T, int pos0, const int32_t *bt,
                                int n_table) {
  const mie_config &c = ctx->cfg;
  cudaStream_t st = ctx->stream;
  const int64_t half = (int64_t)c.n_kv_heads * c.block_size * c.head_dim;
  const int64_t na = (int64_t)c.n_heads * c.head_dim, nqkv = (int64_t)(c.n_heads + 2 * c.n_kv_heads) * c.head_dim;
  const int64_t ldp = ctx->prefill_ldp;
  uint16_t *xm = c.act_bf16 ? nullptr : ctx->pf_xm, *xl = c.act_bf16 ? nullptr : ctx->pf_xl;
  mie_status s;
  MIE_CUDA(cudaMemcpyAsync(ctx->pf_tok, tokens, sizeof(int32_t) * T, cudaMemcpyHostToDevice, st));
  if ((s = launch_embed_rows(ctx->embed, ctx->pf_tok, T, c.vocab, c.d_model, ctx->pf_R, ctx->err, st)) != MIE_OK)
    return s;
  for (int l = 0; l < c.n_layers; ++l) {
    const Layer &L = ctx->layers[(size_t)l];
    uint16_t *kv_layer = ctx->kv + (int64_t)l * 2 * half;
    if ((s = launch_norm_split(ctx->pf_R, c.d_model, c.d_model, L.attn_norm, c.rms_eps, c.act_bf16, T, ctx->pf_xh, xm,
                               xl, ldp, st)) != MIE_OK)
      return s;
    if ((s = prefill_gemm(ctx, L.qkv, T, ctx->pf_Y, nqkv, false)) != MIE_OK) return s;
    RopeKvArgs r;
    r.Y = ctx->pf_Y;
    r.ldy = nqkv;
    r.T = T;
    r.pos0 = pos0;
    r.cos_t = ctx->rope_cos;
    r.sin_t = ctx->rope_sin;
    r.Hq = c.n_heads;
    r.Hkv = c.n_kv_heads;
    r.hd = c.head_dim;
    r.bs = c.block_size;
    r.kv_layer = kv_layer;
    r.block_stride = ctx->block_elems;
    r.bt = bt;
    r.n_table = n_table;
    r.n_pool = c.n_kv_blocks;
    r.Q = ctx->pf_Q;
    r.err = ctx->err;
    if ((s = launch_rope_kv(r, st)) != MIE_OK) return s;
    if (l == c.n_layers - 1) break;
    PrefillAttnArgs a;
    a.q = ctx->pf_Q;
    a.ldq = na;
    a.k = kv_layer;
    a.v = kv_layer + half;
    a.block_stride = ctx->block_elems;
    a.n_pool = c.n_kv_blocks;
    a.bt = bt;
    a.pos0 = pos0;
    a.T = T;
    a.Hq = c.n_heads;
    a.Hkv = c.n_kv_heads;
    a.hd = c.head_dim;
    a.bs = c.block_size;
    a.scale = (float)(1.0 / std::sqrt((double)c.head_dim));
    a.out = ctx->pf_O;
    a.ldo = na;
    a.err = ctx->err;
    if ((s = launch_prefill_attn(a, st)) != MIE_OK) return s;
    if ((s = launch_norm_split(ctx->pf_O, na, (int)na, nullptr, 0.f, c.act_bf16, T, ctx->pf_xh, xm, xl, ldp, st)) != MIE_OK)
      return s;
    if ((s = prefill_gemm(ctx, L.o, T, ctx->pf_R, c.d_model, true)) != MIE_OK) return s;
    if ((s = launch_norm_split(ctx->pf_R, c.d_model, c.d_model, L.mlp_norm, c.rms_eps, c.act_bf16, T, ctx->pf_xh, xm,
                               xl, ldp, st)) != MIE_OK)
      return s;
    if ((s = prefill_gemm(ctx, L.gu, T, ctx->pf_Y, 2 * (int64_t)c.ffn, false)) != MIE_OK) return s;
    if ((s = launch_swiglu_split(ctx->pf_Y, 2 * (int64_t)c.ffn, c.ffn, c.act_bf16, T, ctx->pf_xh, xm, xl, ldp, st)) !=
        MIE_OK)
      return s;
    if ((s = prefill_gemm(ctx, L.down, T, ctx->pf_R, c.d_model, true)) != MIE_OK) return s;
  }
  return MIE_OK;
}

extern "C" mie_status mie_prefill(mie_ctx *ctx, const int32_t *tokens, int n, int32_t pos0, const int32_t *block_table,
                                  int n_blocks) {
  if (!ctx || !tokens || !block_table) return fail(MIE_E_ARG, "mie_prefill: null pointer");
  const mie_config &c = ctx->cfg;
  if (!all_loaded(ctx)) return fail(MIE_E_STATE, "mie_prefill: not every weight is loaded");
  if (n < 0 || pos0 < 0 || (int64_t)pos0 + n > c.max_pos)
    return fail(MIE_E_ARG, "mie_prefill: positions %d .. %d outside [0, %d)", pos0, pos0 + n - 1, c.max_pos);
  if (n == 0) return MIE_OK;
  if (n_blocks < 1 || (int64_t)(pos0 + n - 1) / c.block_size >= n_blocks)
    return fail(MIE_E_ARG, "mie_prefill: position %d needs more than %d blocks", pos0 + n - 1, n_blocks);
  for (int i = 0; i < n; ++i)
    if (tokens[i] < 0 || tokens[i] >= c.vocab)
      return fail(MIE_E_ARG, "mie_prefill: token %d outside [0, %d)", tokens[i], c.vocab);
  mie_status s = prefill_alloc(ctx);
  if (s != MIE_OK) return s;
  for (int p = 0; p < n; p += ctx->prefill_chunk) {
    const int T = std::min(ctx->prefill_chunk, n - p);
    if ((s = prefill_chunk(ctx, tokens + p, T, pos0 + p, block_table, n_blocks)) != MIE_OK) return s;
  }
  return MIE_OK;
}

extern "C" mie_status mie_generate(mie_ctx *ctx, int32_t *ids, int n_prompt, int n_new, const int32_t *block_table,
                                   int max_blocks, int spec_max, int *stats) {
  if (!ctx || !ids || !block_table) return fail(MIE_E_ARG, "mie_generate: null pointer");
  const mie_config &c = ctx->cfg;
  if (n_prompt < 1 || n_new < 0 || n_prompt + n_new > c.max_pos || (n_prompt + n_new - 1) / c.block_size >= max_blocks)
    return fail(MIE_E_ARG, "mie_generate: %d + %d tokens do not fit (max_pos %d, %d blocks)", n_prompt, n_new,
                c.max_pos, max_blocks);
  if (spec_max < 1) spec_max = 1;
  if (spec_max > c.max_slots) spec_max = c.max_slots;
  if (!ctx->gen_argmax && !(ctx->gen_argmax = (int32_t *)ctx->dalloc(sizeof(int32_t) * kMaxSlots)))
    return fail(MIE_E_OOM, "mie_generate: argmax buffer");
  int passes = 0, proposed = 0, accepted = 0;
  mie_status s;
  // the prompt but its last token, on the tensor cores
  if (n_prompt > 1 && (s = mie_prefill(ctx, ids, n_prompt - 1, 0, block_table, max_blocks)) != MIE_OK) return s;
  std::vector<uint8_t> gate_mem(mie_spec_gate_bytes());
  mie_spec_gate *gate = reinterpret_cast<mie_spec_gate *>(gate_mem.data());
  mie_spec_gate_init(gate, 10, 0.3f, 5, 80);
  int len = n_prompt;
  const int end = n_prompt + n_new;
  int32_t toks[kMaxSlots], best[kMaxSlots];
  while (len < end) {
    // the anchor (the last token, whose K/V is not computed yet) and the guesses after it
    int m = 0;
    toks[0] = ids[len - 1];
    const int room = std::min(spec_max - 1, c.max_pos - len);
    if (room > 0 && mie_spec_gate_open(gate)) m = mie_lookup_propose(ids, len, 2, 4, room, toks + 1);
    if ((s = mie_verify_step(ctx, toks, m + 1, len - 1, block_table, max_blocks, nullptr, ctx->gen_argmax)) != MIE_OK)
      return s;
    if ((s = mie_sync(ctx)) != MIE_OK) return s;
    MIE_CUDA(cudaMemcpy(best, ctx->gen_argmax, sizeof(int32_t) * (m + 1), cudaMemcpyDeviceToHost));
    ++passes;
    // the model's token after the anchor is new; each guess it agrees with adds the
    // model's token after that guess
    int acc = 0;
    while (acc < m && toks[1 + acc] == best[acc]) ++acc;
    if (m > 0) mie_spec_gate_record(gate, m, acc);
    proposed += m;
    accepted += acc;
    for (int j = 0; j <= acc && len < end; ++j) ids[len++] = best[j];
  }
  if (stats) {
    stats[0] = passes;
    stats[1] = proposed;
    stats[2] = accepted;
  }
  return MIE_OK;
}

extern "C" mie_status mie_sync(mie_ctx *ctx) {
  if (!ctx) return fail(MIE_E_ARG, "mie_sync: null context");
  MIE_CUDA(cudaStreamSynchronize(ctx->stream));
  int v = 0, ab = 0;
  MIE_CUDA(cudaMemcpy(&v, ctx->err, sizeof(int), cudaMemcpyDeviceToHost));
  MIE_CUDA(cudaMemcpy(&ab, ctx->abort, sizeof(int), cudaMemcpyDeviceToHost));
  if (ab) {
    // a bounded wait gave up: the step's counters and tags are in an unknown state
    const mie_config &c = ctx->cfg;
    MIE_CUDA(cudaMemset(ctx->abort, 0, sizeof(int)));
    MIE_CUDA(cudaMemset(ctx->am_count, 0, sizeof(unsigned) * 64));
    MIE_CUDA(cudaMemset(ctx->attn_ws, 0, ctx->attn_ws_bytes * c.n_layers * c.max_slots));
    MIE_CUDA(reset_tags(ctx));
    MIE_CUDA(cudaMemset(ctx->err, 0, sizeof(int)));
    return fail(MIE_E_TIMEOUT, "decode step: a bounded device wait gave up (code %d)", v);
  }
  if (v) {
    MIE_CUDA(cudaMemset(ctx->err, 0, sizeof(int)));
    return fail(MIE_E_DEVICE, "decode step: device bounds check fired (code %d)", v);
  }
  return MIE_OK;
}

extern "C" mie_status mie_set_step_mode(mie_ctx *ctx, int mode) {
  if (!ctx) return fail(MIE_E_ARG, "mie_set_step_mode: null context");
  if (mode != MIE_STEP_PERSISTENT && mode != MIE_STEP_CHAIN) return fail(MIE_E_ARG, "mie_set_step_mode: mode %d", mode);
  MIE_CUDA(cudaStreamSynchronize(ctx->stream));
  const int old = ctx->mode;
  ctx->mode = mode;
  ctx->primed = false;
  if (mode == MIE_STEP_PERSISTENT && all_loaded(ctx)) {
    build_phases(ctx, ctx->phases);
    const mie_status s = persist_plan(ctx->phases.data(), (int)ctx->phases.size(),
                                      ctx->cfg.n_heads / ctx->cfg.n_kv_heads, ctx->cfg.head_dim, &ctx->plan);
    if (s != MIE_OK) {
      ctx->mode = old;
      return s;
    }
  }
  return MIE_OK;
}

extern "C" int mie_step_mode(const mie_ctx *ctx) { return ctx ? ctx->mode : -1; }

extern "C" mie_status mie_set_trace(mie_ctx *ctx, void *device_buffer, size_t bytes, int *n_phases, int *n_ctas) {
  if (!ctx) return fail(MIE_E_ARG, "mie_set_trace: null context");
  MIE_CUDA(cudaStreamSynchronize(ctx->stream));
  ctx->trace = static_cast<unsigned long long *>(device_buffer);
  ctx->trace_bytes = device_buffer ? bytes : 0;
  ctx->primed = false;  // the next step re-captures with (or without) the trace
  if (n_phases) *n_phases = 5 * ctx->cfg.n_layers + 1;
  if (n_ctas) *n_ctas = sm_count();
  return MIE_OK;
}

// Temperature / top-k / top-p sampling of the next token inside the step's graph.
extern "C" mie_status mie_set_sampling(mie_ctx *ctx, float temperature, int top_k, float top_p, uint64_t seed) {
  if (!ctx) return fail(MIE_E_ARG, "mie_set_sampling: null context");
  if (top_k < 0 || !(top_p > 0.f) || top_p > 1.f || temperature != temperature)
    return fail(MIE_E_ARG, "mie_set_sampling: top_k %d, top_p %g, temperature %g", top_k, top_p, temperature);
  MIE_CUDA(cudaStreamSynchronize(ctx->stream));
  if (temperature > 0.f && !ctx->sample_ws) {
    ctx->logits_buf = (float *)ctx->dalloc(sizeof(float) * (size_t)ctx->cfg.vocab);
    ctx->sample_ws = ctx->dalloc(sample_workspace_bytes());
    if (!ctx->logits_buf || !ctx->sample_ws) return fail(MIE_E_OOM, "mie_set_sampling: buffers");
    MIE_CUDA(cudaMemset(ctx->sample_ws, 0, sample_workspace_bytes()));
  }
  ctx->temperature = temperature > 0.f ? temperature : 0.f;
  ctx->top_k = top_k;
  ctx->top_p = top_p;
  ctx->seed = seed;
  ctx->primed = false;  // the next step re-captures with (or without) the sampler
  return MIE_OK;
}

// Testing aid: phase `phase` of the persistent step reads its input from words that no
// phase writes (tag 0, which no launch uses), so its wait can only run out.
extern "C" mie_status mie_debug_stall(mie_ctx *ctx, int phase, long wait_polls) {
  if (!ctx) return fail(MIE_E_ARG, "mie_debug_stall: null context");
  const mie_config &c = ctx->cfg;
  const int n_phases = 5 * c.n_layers + 1;
  if (phase == 0 || phase >= n_phases || (phase > 0 && wait_polls < 1))
    return fail(MIE_E_ARG, "mie_debug_stall: phase %d (1..%d), wait_polls %ld", phase, n_phases - 1, wait_polls);
  MIE_CUDA(cudaStreamSynchronize(ctx->stream));
  if (phase > 0 && !ctx->stall_words) {
    // the longest input vector of any phase, as tagged words
    int64_t n = std::max<int64_t>({(int64_t)(c.n_heads + 2 * c.n_kv_heads) * c.head_dim, c.d_model, c.ffn});
    ctx->stall_words = (uint64_t *)ctx->dalloc(sizeof(uint64_t) * (size_t)n);
    if (!ctx->stall_words) return fail(MIE_E_OOM, "mie_debug_stall: word buffer");
    MIE_CUDA(cudaMemset(ctx->stall_words, 0, sizeof(uint64_t) * (size_t)n));
  }
  ctx->stall_phase = phase < 0 ? -1 : phase;
  ctx->wait_polls = phase < 0 ? kWaitPolls : wait_polls;
  ctx->primed = false;  // the next step re-captures with the changed phase table and limit
  return MIE_OK;
}

extern "C" int mie_step_launches(const mie_ctx *ctx) { return ctx ? ctx->launches : 0; }

extern "C" int mie_slot_step_launches(const mie_ctx *ctx) { return ctx ? ctx->slot_launches : 0; }
