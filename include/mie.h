/*
 * mie.h -- C ABI of the GB300 decode-step library (libmie.so).
 *
 * The library runs the batch-1 and few-slot decode step of a Llama-style GQA decoder
 * on one GPU: fused-dequant GEMVs over bf16, int8 per-row and Q4_0 weights, RoPE and
 * a K/V write into a paged cache, split-context paged decode attention, RMSNorm,
 * SwiGLU, the LM head and argmax, the whole step captured in a CUDA graph.
 *
 * Pages cited (titles):
 *  [RUST]  "Writing an LLM inference engine from scratch in Rust"
 *  [MIE]   "Mini Inference Engine"
 *  [INFER] "infer" -- an LLM inference engine in C++ and CUDA for Llama-3.2-1B
 *
 * Conventions (every entry point):
 *  - Status codes, never exceptions or aborts ([MIE]: an exhausted pool returns a
 *    sentinel instead of throwing).  After a failure mie_last_error() returns a
 *    message for the calling thread.
 *  - Pointers documented "device" are CUDA device pointers (for example a torch
 *    tensor's data_ptr()); "host" pointers are ordinary process memory.  The caller
 *    owns every pointer it passes; the library keeps none of them after the call
 *    returns, except where stated (mie_decode_step's block table and outputs are read
 *    or written by work that is still queued on the stream).
 *  - `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream).
 *    Kernel entry points only enqueue work: results are ready once the stream is
 *    synchronised.  Arguments are validated on the host before anything is enqueued.
 *  - A model context (mie_ctx) may be used by one host thread at a time; distinct
 *    contexts are independent.  A block pool serialises its calls internally (one
 *    lock per pool).  Stateless entry points may be called from several threads; the
 *    scratch of mie_paged_attn_decode_noalloc is the one shared resource (see there).
 *  - Storage formats: MIE_FMT_BF16 (uint16 bit patterns), MIE_FMT_I8 (int8 plus one
 *    fp32 scale per row), MIE_FMT_Q4_0 (blocks of 32 four-bit codes plus one f16
 *    scale), MIE_FMT_F32.
 */
#ifndef MIE_H_
#define MIE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum mie_status {
  MIE_OK = 0,
  MIE_E_ARG = 1,     /* null pointer, unknown name/format, id or value out of range */
  MIE_E_SHAPE = 2,   /* a size or alignment the entry point does not support */
  MIE_E_OOM = 3,     /* a device allocation failed, or the KV block pool is exhausted */
  MIE_E_CUDA = 4,    /* a CUDA runtime call failed (the message names it) */
  MIE_E_TIMEOUT = 5, /* a bounded device-side wait gave up */
  MIE_E_STATE = 6,   /* call out of order, e.g. a step before all weights are loaded */
  MIE_E_DEVICE = 7   /* a kernel's own bounds check rejected an index (see mie_check) */
} mie_status;

typedef enum mie_format {
  MIE_FMT_BF16 = 0,
  MIE_FMT_I8 = 1,
  MIE_FMT_Q4_0 = 2,    /* 4-bit, one f16 scale per 32 weights */
  MIE_FMT_F32 = 3,
  MIE_FMT_Q4_G64 = 4,  /* 4-bit, one f16 scale per 64 weights */
  MIE_FMT_Q4_G128 = 5  /* 4-bit, one f16 scale per 128 weights */
} mie_format;

/* Message for the last failure on the calling thread ("" if none). */
const char *mie_last_error(void);
const char *mie_status_string(mie_status s);

/* ======================================================================== load time */

/* fp32 -> bf16, round to nearest even.  w, out: device, n elements. */
mie_status mie_convert_bf16(const float *w, int64_t n, uint16_t *out, void *stream);

/* int8 with one scale per row ([INFER] design notes, weight-only quantization: each
 * row has its own scale).  Per row: s = max|w| / 127 (fp32), q = round-half-away(w / s) clamped to
 * [-127, 127]; a zero row gives s = 0, q = 0.  w: device [M][K] fp32 row-major;
 * q: device [M][K]; scale: device [M]. */
mie_status mie_quantize_i8(const float *w, int M, int K, int8_t *q, float *scale, void *stream);

/* Q4_0 ([RUST] "Lesson 1" and "Is the 4-bit model still good?"; [INFER] design notes):
 * blocks of 32 weights; the element of largest magnitude (first on ties), sign kept,
 * divided by -8 gives d; h = f16(d) rounded to nearest even is stored; codes are
 * q = clamp(floor(w * (1/h) + 8.5), 0, 15) (0 for h == 0), each step rounded in fp32.
 * A row is zero-padded to a whole number of blocks.  Output is the canonical block
 * layout [M][ceil(K/32)][18]: f16 scale little-endian, then 16 bytes whose byte j holds
 * element j in the low nibble and element j+16 in the high nibble.
 * w: device [M][K] fp32; blocks: device. */
mie_status mie_quantize_q4_0(const float *w, int M, int K, uint8_t *blocks, void *stream);

/* Size of the GPU layout of an M x K Q4_0 matrix: a nibble plane [M][nb][16] followed,
 * at the next 256-byte boundary, by a scale plane [M][nbp] of f16, nb = ceil(K/32),
 * nbp = nb rounded up to a multiple of 8 (the extra scales are zero). */
size_t mie_q4_0_packed_bytes(int M, int K);

/* Canonical blocks (device) -> GPU layout (device, mie_q4_0_packed_bytes(M, K) bytes). */
mie_status mie_q4_0_pack(const uint8_t *blocks, int M, int K, void *packed, void *stream);

/* 4-bit weights with one f16 scale per `group` (32, 64 or 128) weights ([INFER] design
 * notes, weight-only quantization: int4 per 32 weights as in Q4_0, groups of 128 as its
 * starting point; its perplexity table also measures groups of 64).  The Q4_0 rule
 * applied to groups of `group` weights: the group's signed extreme over -8 is the scale,
 * codes q = clamp(floor(w * (1/h) + 8.5), 0, 15).  A row is zero-padded to whole groups.
 * Canonical layout [M][ceil(K/group)][2 + group/2]: the f16 scale (little-endian), then
 * group/32 sub-blocks of 16 bytes, byte j of sub-block b holding code 32b+j in its low
 * nibble and code 32b+j+16 in its high nibble; group 32 is Q4_0.  MIE_E_ARG for another
 * group size.  w: device [M][K] fp32; groups: device. */
mie_status mie_quantize_q4(const float *w, int M, int K, int group, uint8_t *groups, void *stream);

/* Size of the GPU layout: a nibble plane [M][ng*group/32][16], ng = ceil(K/group),
 * followed at the next 256-byte boundary by a scale plane [M][ngp] of f16, ngp = ng
 * rounded up to a multiple of 8.  0 for an unsupported group. */
size_t mie_q4_packed_bytes(int M, int K, int group);

/* Canonical groups (device) -> GPU layout (device, mie_q4_packed_bytes bytes, 256-byte
 * aligned). */
mie_status mie_q4_pack(const uint8_t *groups, int M, int K, int group, void *packed, void *stream);

/* ============================================================================ GEMV */

/* y = W x with fp32 accumulation ([INFER] per-kernel table, "gemv"; [RUST] "Lesson 1":
 * each weight is read once, so the kernel streams W at memory bandwidth).
 *   mie_gemv_bf16: W device [M][K] bf16 row-major, K % 8 == 0, W 16-byte aligned.
 *   mie_gemv_i8:   W device [M][K] int8 row-major, K % 16 == 0; row_scale device [M];
 *                  y_i = s_i * sum_k q_ik x_k.
 *   mie_gemv_q4_0: packed: device GPU layout from mie_q4_0_pack; any K >= 1.
 * x: device [K] fp32; y: device [M] fp32 (must not alias x).  1 <= K <= 16384,
 * M >= 1.  MIE_E_SHAPE for other sizes or misaligned pointers.  x is fp32 only: the
 * activations are fp32 ([INFER] design notes), and a bf16 activation vector widens to
 * fp32 exactly, so an fp32 x carries it without loss.
 * Launched with programmatic dependent launch: when the previous kernel on the stream is
 * one of this library's GEMV, attention or argmax kernels, W starts streaming while that
 * kernel finishes; x is read and y written only after it has completed.  (None of those
 * kernels writes weights; the quantise / convert / pack kernels do not release their
 * successor early.) */
mie_status mie_gemv_bf16(const uint16_t *W, const float *x, float *y, int M, int K, void *stream);
mie_status mie_gemv_i8(const int8_t *W, const float *row_scale, const float *x, float *y, int M,
                       int K, void *stream);
mie_status mie_gemv_q4_0(const void *packed, const float *x, float *y, int M, int K, void *stream);
/* The same GEMV over a 4-bit matrix with `group` weights per scale (GPU layout from
 * mie_q4_pack); group 32 is mie_gemv_q4_0. */
mie_status mie_gemv_q4(const void *packed, int group, const float *x, float *y, int M, int K,
                       void *stream);

/* ============================================================ prompt GEMM (tcgen05) */

/* Cuts x[0..n) (device fp32) into bf16 planes hi = bf16(x), mid = bf16(x - hi),
 * lo = bf16(x - hi - mid) (round to nearest even; both differences are exact in fp32),
 * the activation operand of mie_gemm_bf16: hi + mid + lo is x to 2^-25 of x, and every
 * product of a plane with a bf16 weight is exact in fp32.  mid and lo may be NULL.
 * 1 <= n < 2^31. */
mie_status mie_split_bf16(const float *x, int64_t n, uint16_t *hi, uint16_t *mid, uint16_t *lo, void *stream);

/* The prompt's matrix-matrix product on the tensor cores ([INFER] summary table and
 * "Limitations": prefill multiplies every weight matrix by all prompt positions at once,
 * a dense contraction that tensor cores make several times faster than the CUDA-core
 * path):
 *   y[t * ldy + n] (+)= sum_k W[n][k] * (x_hi + x_mid + x_lo)[t][k],  t < T, n < N,
 * on tcgen05 (one CTA per SM taking 128 weight rows x 128 positions tiles in turn,
 * operands staged by TMA with 128-byte swizzle, accumulators in tensor memory, drained
 * every 128 columns of K into fp32 registers).  W: device bf16 [N][K] row-major; x_hi, x_mid, x_lo: device bf16
 * [T][K] planes (mie_split_bf16; x_mid and x_lo NULL: x_hi alone; x_lo NULL: hi + mid);
 * y: device fp32, rows ldy >= N floats apart; accumulate != 0 adds to y.  Pointers
 * 16-byte aligned, K % 8 == 0 (MIE_E_SHAPE otherwise).  A device-side wait that gives
 * up is latched as a device error (mie_check). */
mie_status mie_gemm_bf16(const uint16_t *W, int N, int K, const uint16_t *x_hi, const uint16_t *x_mid,
                         const uint16_t *x_lo, int T, float *y, int64_t ldy, int accumulate, void *stream);

/* ======================================================================= attention */

/* Workspace bytes that mie_paged_attn_decode needs for these sizes. */
size_t mie_paged_attn_workspace_bytes(int n_q_heads, int n_kv_heads, int head_dim, int ctx_len,
                                      int block_size);

/* Paged GQA decode attention, split over the context with an online softmax and a
 * merge ([MIE] "The KV cache, paged like virtual memory"; [INFER] design notes, the
 * split-KV attention item; [RUST] "Lesson 4": running maximum and sum, query heads sharing a KV
 * head read it together).
 *   out[h][d] = sum_{t < ctx_len} softmax_t(scale * q_h . k_{g,t}) v_{g,t}[d],
 *   g = h / (n_q_heads / n_kv_heads).
 * Key t of KV head g is at k_pool[block_table[t / block_size] * block_stride
 *   + (g * block_size + t % block_size) * head_dim + d] (bf16); v_pool likewise.
 * q: device [n_q_heads][head_dim] fp32; out: device, same shape; block_table: device
 * int32 [n_table], entries in [0, n_pool_blocks).  head_dim in {32, 64, 128},
 * n_q_heads % n_kv_heads == 0, group size <= 8, ctx_len <= n_table * block_size,
 * block_size in {8, 16, 32}.  ctx_len == 0 gives a zero output.  workspace: device,
 * at least mie_paged_attn_workspace_bytes(...) bytes, 256-byte aligned; its contents
 * need not be initialised and are overwritten.  Calls sharing one workspace must not
 * overlap on the GPU.  A block-table entry outside [0, n_pool_blocks) is skipped and
 * latched as a device error, reported by mie_check as MIE_E_DEVICE. */
mie_status mie_paged_attn_decode(const float *q, const uint16_t *k_pool, const uint16_t *v_pool,
                                 int64_t block_stride, int n_pool_blocks,
                                 const int32_t *block_table, int n_table, int ctx_len,
                                 int n_q_heads, int n_kv_heads, int head_dim, int block_size,
                                 float scale, float *out, void *workspace,
                                 size_t workspace_bytes, void *stream);

/* Allocation-free variant of mie_paged_attn_decode.  The pages have no counterpart:
 * they never consider callers that cannot allocate.  Some callers cannot call
 * cudaMalloc at the moment they run attention -- a loop that must never enter the
 * device allocator, or code whose device memory is owned entirely by another
 * allocator -- so they cannot provide a workspace.  This entry point takes none and
 * allocates nothing: its partial results live in a 1 MiB array compiled into the
 * library, which every GPU that loads the library holds until the process exits.
 * Arguments, results and errors are those of mie_paged_attn_decode, except that sizes
 * needing more scratch than the array holds (mie_paged_attn_workspace_bytes(...) >
 * 1048576) are rejected with MIE_E_SHAPE.  The first call on each device looks up the
 * array's device address (cudaGetSymbolAddress); make that first call before any stream
 * capture.  Each call clears the counters it needs before its kernel runs.  All calls
 * on one device share the array and it keeps the last call's partial results, so
 * calls that overlap on the GPU (other streams, other host threads) race: the caller
 * must serialise them. */
mie_status mie_paged_attn_decode_noalloc(const float *q, const uint16_t *k_pool,
                                         const uint16_t *v_pool, int64_t block_stride,
                                         int n_pool_blocks, const int32_t *block_table,
                                         int n_table, int ctx_len, int n_q_heads, int n_kv_heads,
                                         int head_dim, int block_size, float scale, float *out,
                                         void *stream);

/* Causal paged GQA attention of T consecutive positions pos0 .. pos0 + T - 1 of one
 * sequence, whose K/V (and those of every earlier position) are already in the cache
 * ([INFER] "Limitations": the prompt's flash-style attention; [MIE] "The KV cache, paged
 * like virtual memory"):
 *   out[t][h][d] = sum_{p <= pos0 + t} softmax_p(scale * q[t][h] . k_{g,p}) v_{g,p}[d],
 * the cache addressed as in mie_paged_attn_decode.  q, out: device fp32 [T][n_q_heads]
 * [head_dim]; block_table: device int32 [n_table] with pos0 + T <= n_table * block_size.
 * head_dim in {32, 64, 128}, block_size dividing 64.  Runs on mma.sync with q and the
 * probabilities as three bf16 planes each.  A block-table entry outside [0, n_pool_blocks)
 * is read as block 0 and latched as a device error (mie_check). */
mie_status mie_paged_attn_prefill(const float *q, const uint16_t *k_pool, const uint16_t *v_pool,
                                  int64_t block_stride, int n_pool_blocks, const int32_t *block_table,
                                  int n_table, int pos0, int T, int n_q_heads, int n_kv_heads,
                                  int head_dim, int block_size, float scale, float *out, void *stream);

/* ========================================================================== argmax */

size_t mie_argmax_workspace_bytes(int n);

/* Index of the largest of v[0..n) (device fp32); the lowest index wins a tie.
 * out: device int32.  workspace: device, mie_argmax_workspace_bytes(n) bytes, need
 * not be initialised.  n >= 1. */
mie_status mie_argmax(const float *v, int n, int32_t *out, void *workspace, size_t workspace_bytes,
                      void *stream);

/* ================================================================ bandwidth probe */

/* Read-only streaming probe ([INFER]: every kernel's bandwidth is quoted as a fraction
 * of a peak the page measured with its own read probe, not of the datasheet figure).
 * Reads each of the `bytes` bytes of buf (device) exactly once, with load_bytes-wide
 * loads (16 or 32) that bypass L1 and are marked evict-first in L2, from a grid of
 * blocks_per_sm (1..4) CTAs of 512 threads per SM; *xor_out (device uint32, zeroed by
 * the call) receives the XOR of all of the buffer's 32-bit words, so the result is
 * exact and checkable.  To measure HBM rather than L2, pass a buffer many times the
 * 129 MB L2.  bytes must be a nonzero multiple of load_bytes and buf load_bytes-aligned
 * (MIE_E_SHAPE otherwise).  Asynchronous on `stream`. */
mie_status mie_hbm_read_probe(const void *buf, size_t bytes, uint32_t *xor_out, int load_bytes,
                              int blocks_per_sm, void *stream);

/* ======================================================================== sampling */

/* Workspace bytes of mie_sample (independent of the vocabulary size). */
size_t mie_sample_workspace_bytes(void);

/* Draws the next token from logits v[0..n) (device fp32) ([INFER] design notes:
 * temperature / top-k / top-p sampling on the GPU, radix select for the top-k and top-p
 * cut-offs, per-position random numbers from a seed so that runs reproduce).
 * temperature <= 0: the argmax (lowest index on ties).  Otherwise, with
 * q_i = exp((v_i - max v) / temperature): top-k keeps the tokens whose value is at least
 * the top_k-th largest (ties at it kept; top_k 0 or >= n keeps all); top-p then keeps, of
 * those, the tokens whose value is at least the largest t for which the kept tokens with
 * value >= t hold at least top_p of the kept mass (ties kept; top_p 1 keeps all); the
 * token is the Gumbel-max draw argmax over kept i of v_i / temperature - log(-log u_i),
 * u_i = (top 24 bits of splitmix64(seed, output (pos << 32 | i)) + 1/2) / 2^24, which
 * picks i with probability q_i / (kept mass).  The masses are summed in 2^-40 fixed
 * point, so the cut-offs, and the token, are the same on every run.  out: device int32.
 * workspace: device, mie_sample_workspace_bytes() bytes, 256-byte aligned (zeroed by the
 * call).  MIE_E_ARG for top_k < 0, top_p outside (0, 1] or a NaN temperature. */
mie_status mie_sample(const float *logits, int n, float temperature, int top_k, float top_p,
                      uint64_t seed, int32_t pos, int32_t *out, void *workspace,
                      size_t workspace_bytes, void *stream);

/* Reads and clears the device error flag that kernels latch when a bounds check
 * fails (stateless kernels share one flag per device).  Synchronises `stream`.
 * MIE_E_DEVICE if a check fired since the last call. */
mie_status mie_check(void *stream);

/* ============================================================ KV block pool (host) */

/* Reference-counted pool of KV blocks ([MIE] "The KV cache, paged like virtual
 * memory" and "Prefix sharing and copy-on-write"): a refcount per block id, a LIFO
 * free list; a fresh pool hands out 0, 1, 2, ...  Host bookkeeping only: the block
 * contents live in the model context's device KV pool. */
typedef struct mie_pool mie_pool;

mie_status mie_pool_create(int n_blocks, mie_pool **out);
void mie_pool_destroy(mie_pool *p);
/* *id = a block with refcount 1, or -1 and MIE_E_OOM when the pool is exhausted. */
mie_status mie_pool_alloc(mie_pool *p, int32_t *id);
/* Adds a reference to a live block (a sequence borrowing it); MIE_E_ARG for an id out
 * of range or not live. */
mie_status mie_pool_incref(mie_pool *p, int32_t id);
/* Drops one reference; a block reaching 0 returns to the free list.  MIE_E_ARG for an
 * id out of range or not live. */
mie_status mie_pool_decref(mie_pool *p, int32_t id);
int mie_pool_refcount(const mie_pool *p, int32_t id); /* -1 for an id out of range */
int mie_pool_free_count(const mie_pool *p);
/* Copy-on-write ([MIE] "Prefix sharing and copy-on-write": a sequence writing into a
 * block that others share first moves to a private copy, and the shared block must
 * stay alive until the copy is made) for a write at logical position pos of a sequence
 * whose block table (host int32, updated in place) is `table`.  A block this sequence
 * holds alone is returned as is (*copy_src = *copy_dst = -1).  For a shared block a
 * fresh block is allocated and the table entry points at it (*block = *copy_dst = the
 * new id, *copy_src = the shared id), but the sequence KEEPS its reference on the
 * shared block: the caller enqueues the contents copy src -> dst (mie_kv_copy_block for
 * a model context's pool) and only then calls mie_pool_decref(p, *copy_src).  Until that
 * decref no other thread can free the shared block and have it reused, so the copy
 * never reads overwritten contents.  MIE_E_OOM (table and counts untouched, outputs -1)
 * when no block is free; MIE_E_ARG when the table's block is not live.  A model
 * context's mie_kv_writable does all three steps in order. */
mie_status mie_pool_writable(mie_pool *p, int32_t *table, int pos, int block_size, int32_t *block,
                             int32_t *copy_src, int32_t *copy_dst);

/* ============================================================== model and step */

typedef struct mie_ctx mie_ctx;

typedef struct mie_config {
  int n_layers, d_model, n_heads, n_kv_heads, head_dim, ffn, vocab;
  int tied;        /* 1: the LM head matrix doubles as the embedding table */
  int block_size;  /* tokens per KV block (16) */
  int act_bf16;    /* 1: round each GEMV input vector to bf16 (residual stays fp32) */
  float rms_eps;
  float rope_theta;
  int wfmt;        /* format of the layer matrices (mie_format: bf16, i8 or a 4-bit format) */
  int head_fmt;    /* format of the LM head (and of the embedding when tied) */
  int embed_fmt;   /* format of an untied embedding table */
  int n_kv_blocks; /* device KV pool size in blocks */
  int max_slots;   /* largest n_slots of mie_decode_step_slots (>= 1, <= 8) */
  int max_pos;     /* positions 0 .. max_pos-1 are valid */
} mie_config;

/* Creates a context on the current CUDA device ([RUST] "Try it": the engine is loaded
 * once and hands out a session that owns its KV cache; [INFER] the table of where each
 * piece lives: one engine object holds the KV cache, the decode step and its CUDA graph):
 * device KV pool
 * [n_kv_blocks][n_layers][2][n_kv_heads][block_size][head_dim] bf16 (zeroed), RoPE
 * tables, activations, a host block pool of n_kv_blocks blocks.  stream: the stream
 * every step of this context runs on. */
mie_status mie_create(const mie_config *cfg, void *stream, mie_ctx **out);
void mie_destroy(mie_ctx *ctx);

/* Copies one weight from host memory into the context and repacks it for the
 * kernels ([RUST] "Keeping the benchmark fair": the engine quantises the weights itself
 * when it loads them; [INFER] the table of pieces: weights are converted at load time
 * and packed by the weight-only quantization kernels).  name: "l<i>.qkv" [(Hq+2Hkv)*hd][d] (rows q heads, then k, then v),
 * "l<i>.o" [d][Hq*hd], "l<i>.gate" [ffn][d], "l<i>.up" [ffn][d], "l<i>.down" [d][ffn],
 * "head" [vocab][d], "embed" [vocab][d] (untied only), "l<i>.attn_norm",
 * "l<i>.mlp_norm", "final_norm" [d] (fp32 gains; all default to 1).
 * fmt: MIE_FMT_F32 (fp32 [rows][cols]; quantised on the device into the context's
 * format for that tensor) or that format itself in canonical layout (bf16 [rows][cols];
 * i8 [rows][cols] with host_scale [rows]; 4-bit canonical groups, e.g. Q4_0 blocks
 * [rows][ceil(cols/32)][18]).
 * bytes must equal the canonical size.  shape: {rows, cols} (gains: {d}). */
mie_status mie_load_weights(mie_ctx *ctx, const char *name, int fmt, const void *host_data,
                            size_t bytes, const int64_t *shape, int ndim,
                            const float *host_scale);

/* The context's host block pool (n_kv_blocks blocks), owned by the context: valid until
 * mie_destroy, never passed to mie_pool_destroy. */
mie_pool *mie_ctx_pool(mie_ctx *ctx);
/* Device pointer of the KV pool (owned by the context) and the elements of one block
 * (all layers, k and v). */
uint16_t *mie_kv_pool(mie_ctx *ctx);
int64_t mie_kv_block_elems(const mie_ctx *ctx);
/* Enqueues a device copy of block src into block dst (copy-on-write) on the context's
 * stream; MIE_E_ARG for a block id outside 0..n_kv_blocks-1. */
mie_status mie_kv_copy_block(mie_ctx *ctx, int32_t src, int32_t dst);
/* Copy-on-write on the context's pool, in the safe order: mie_pool_writable (allocate,
 * repoint the table entry), then the contents copy enqueued on the context's stream,
 * then the sequence's reference on the shared block dropped.  Every later step of this
 * context, and any reuse of the shared block by work on the same stream, is ordered
 * after the copy.  table: host int32 block table of the sequence, updated in place;
 * *block receives the block to write.  Errors as mie_pool_writable; a failed copy
 * enqueue (MIE_E_CUDA) leaves the table pointing at the fresh block and keeps the
 * reference on the shared one, for the caller to retry or release. */
mie_status mie_kv_writable(mie_ctx *ctx, int32_t *table, int pos, int32_t *block);

/* One decode step ([INFER] data-flow figure; [RUST] "How a Llama model generates
 * text"): the token at 0-based position pos writes its K/V into block
 * block_table[pos / block_size] and attends to positions 0..pos.  block_table: device
 * int32 [n_blocks] (entries < n_kv_blocks).  logits_out: device fp32 [vocab] or NULL;
 * argmax_out: device int32 or NULL (lowest index on ties).  The first call captures
 * the step into a CUDA graph (call it outside any stream capture); later calls replay
 * it.  The step reads token/pos/table from device memory, so one graph serves every
 * step.  Asynchronous on the context's stream. */
mie_status mie_decode_step(mie_ctx *ctx, int32_t token, int32_t pos, const int32_t *block_table,
                           int n_blocks, float *logits_out, int32_t *argmax_out);

/* One decode step with host input and output ([RUST] "How a Llama model generates text":
 * the argmax of a step's logits is the next token): mie_decode_step for the token at
 * position pos, then the step's next token (its argmax, or the sampler's draw under
 * mie_set_sampling) copied back to the host int32 *next_token, waiting for the step.
 * block_table: device int32 [n_blocks]; logits_out: device fp32 [vocab] or NULL.
 * Errors as mie_decode_step; MIE_E_ARG for a null next_token, MIE_E_OOM if its small
 * device and pinned host buffers (allocated on the first call) cannot be had. */
mie_status mie_decode_step_sync(mie_ctx *ctx, int32_t token, int32_t pos, const int32_t *block_table,
                                int n_blocks, float *logits_out, int32_t *next_token);

/* Greedy continuation: replays the step n_steps times with token = previous argmax
 * and pos = previous pos + 1, all on the device.  Requires one mie_decode_step first
 * (which fixes block table and outputs); the outputs hold the last step's results. */
mie_status mie_decode_continue(mie_ctx *ctx, int n_steps);

/* Few-slot step ([MIE] "Continuous batching"): every slot s advances one token,
 * tokens[s] at pos[s] (host arrays), through row s of block_tables (device int32
 * [n_slots][max_blocks]).  The weights are read once for all slots (tensor-core MMAs
 * over the slots' input vectors, split into bf16 hi + lo).  logits_out: device
 * [n_slots][vocab] or NULL; argmax_out: device [n_slots] or NULL.  Layers and head in
 * bf16, int8 or Q4_0 with input lengths a multiple of 4; otherwise MIE_E_SHAPE.  The first call
 * captures the few-slot step into its own CUDA graph.  Slots never write into a block
 * another slot's table shares (block-aligned prefixes; see mie_pool_writable). */
mie_status mie_decode_step_slots(mie_ctx *ctx, int n_slots, const int32_t *tokens,
                                 const int32_t *pos, const int32_t *block_tables, int max_blocks,
                                 float *logits_out, int32_t *argmax_out);

/* Verify pass ([RUST] "Speculative decoding without a draft model": several tokens of one
 * sequence are checked in one batched pass, the weights read once): positions pos .. pos+n-1
 * of one sequence (tokens[j] host int32 at pos + j) as n slots of the few-slot step,
 * every slot reading the same block table (device int32 [max_blocks]), slot j attending
 * to positions 0 .. pos + j including the K/V this pass writes.  1 <= n <= max_slots.
 * logits_out: device [n][vocab] or NULL; argmax_out: device [n] or NULL.  The few-slot
 * kernels compute each (row, slot) output on its own, in an order that does not depend
 * on the number of slots, so a pass of n positions gives the bits of n passes of one
 * position through the same kernels. */
mie_status mie_verify_step(mie_ctx *ctx, const int32_t *tokens, int n, int32_t pos,
                           const int32_t *block_table, int max_blocks, float *logits_out,
                           int32_t *argmax_out);

/* Prompt lookup ([RUST] "Speculative decoding without a draft model"): the tokens that
 * followed the most recent earlier occurrence of the last g tokens of ids[0..n), for the
 * longest g in [min_ngram, max_ngram] that occurs earlier (ending before the last g
 * tokens begin); at most k of them, never past the end.  Writes them to out (host) and
 * returns their number (0: no match).  Host only. */
int mie_lookup_propose(const int32_t *ids, int n, int min_ngram, int max_ngram, int k, int32_t *out);

/* Acceptance gate of speculative decoding ([RUST], same section: acceptance is tracked
 * over the last 10 attempts; below 30 % speculation pauses for 5 steps, each consecutive
 * pause doubling up to 80).  A full window of `window` attempts whose accepted / proposed
 * guesses fall below `threshold` starts a pause of the current length, which then
 * doubles up to pause_max; a full window at or above the threshold resets the length to
 * `pause`.  The window keeps its attempts across a pause.  Caller-owned memory of
 * mie_spec_gate_bytes() bytes.  Host only. */
typedef struct mie_spec_gate mie_spec_gate;
size_t mie_spec_gate_bytes(void);
void mie_spec_gate_init(mie_spec_gate *g, int window, float threshold, int pause, int pause_max);
int mie_spec_gate_open(mie_spec_gate *g);  /* 1: this pass may guess (a paused gate counts it off) */
void mie_spec_gate_record(mie_spec_gate *g, int proposed, int accepted);

/* Prompt prefill on the tensor cores ([INFER] summary table and "Limitations": the
 * prompt as matrix-matrix products instead of one decode step per token).  Runs the n
 * tokens tokens[0..n) (host int32) at positions pos0 .. pos0 + n - 1 of one sequence
 * through every layer, in chunks of up to 2048 positions -- RMSNorm, the QKV product
 * (mie_gemm_bf16's kernel; int8 and 4-bit matrices are first expanded to bf16 planes),
 * RoPE, the K/V write into the paged cache through block_table (device int32
 * [n_blocks]), causal attention (mie_paged_attn_prefill's kernel), the O product, the
 * MLP -- and leaves their K/V in every layer's cache; the last layer stops after its K/V
 * write.  It produces no logits: the decode step of the next position (the prompt's last
 * token) does.  Activations enter the products as three bf16 planes (bf16 alone for
 * act_bf16 models), so the cache matches the decode step's to within rounding of the
 * summation order.  Asynchronous on the context's stream; the buffers (about 280 MB at
 * the Llama-3.2-1B shape, plus the largest weight matrix as bf16 planes for quantised
 * models) are allocated on the first call.  MIE_E_ARG for a token outside [0, vocab) or
 * positions outside [0, max_pos) or the table; device bounds checks are reported by the
 * next mie_sync. */
mie_status mie_prefill(mie_ctx *ctx, const int32_t *tokens, int n, int32_t pos0, const int32_t *block_table,
                       int n_blocks);

/* Greedy generation.  ids: host int32 [n_prompt + n_new]; ids[0..n_prompt) is the
 * prompt, ids[n_prompt..) receives the n_new generated tokens.  The prompt but its last
 * token goes through mie_prefill; each later pass, through the few-slot kernels, takes
 * the last token and, with spec_max > 1, up to
 * spec_max - 1 prompt-lookup guesses (2- to 4-token matches, behind the acceptance gate
 * of 10 attempts / 30 % / pauses of 5 .. 80 passes), verifies them in one mie_verify_step
 * and keeps the guesses up to the first the model disagrees with, plus the model's own
 * next token.  Because a pass of several positions equals single-position passes bit for
 * bit, the tokens do not depend on spec_max.  block_table: device int32 [max_blocks].
 * stats (host int [3], nullable): passes, guesses proposed, guesses accepted. */
mie_status mie_generate(mie_ctx *ctx, int32_t *ids, int n_prompt, int n_new, const int32_t *block_table,
                        int max_blocks, int spec_max, int *stats);

/* How mie_decode_step runs the step.  MIE_STEP_PERSISTENT (the default where the shape
 * is covered): one cooperative kernel of one CTA per SM runs every phase; its producer
 * warps stream all weights and the K/V of old positions through shared-memory rings,
 * and consumer warps pass each phase's output vector to the next as tagged words
 * (value + launch tag), polled with bounded waits instead of grid barriers.
 * MIE_STEP_CHAIN: one kernel per phase with programmatic dependent launch.  Either is
 * captured in a CUDA graph.  The persistent kernel covers group/head-dim shapes
 * (4, 32), (8, 64), (4, 64) and the format pairs (layers, head) bf16/bf16, i8/i8,
 * q4_0/q4_0, q4_0/i8; selecting it for another shape returns MIE_E_SHAPE and keeps the
 * chain, and a context created for such a shape runs the chain from its first step. */
enum { MIE_STEP_PERSISTENT = 0, MIE_STEP_CHAIN = 1 };
mie_status mie_set_step_mode(mie_ctx *ctx, int mode);
int mie_step_mode(const mie_ctx *ctx);

/* Timeline of the persistent step (tracing).  device_buffer: device memory of at least
 * n_phases * n_ctas * 5 * 8 bytes (NULL switches tracing off); every later step
 * overwrites it.  Entry [phase][cta][point] is the GPU's global timer in ns when CTA
 * `cta` reached point 0 = phase entry, 1 = input words arrived, 2 = input vector
 * staged (normalised), 3 = ring stages consumed, 4 = outputs written.  In a library built
 * with MIE_STAGE_TRACE defined, and when the buffer is at least
 * n_ctas * (1024 * 4 + n_phases * 8) * 8 bytes larger, those bytes receive per-stage stamps
 * [cta][stage][point] for the first 1024 ring stages of each CTA: 0 = the stage's copy
 * issued, 1 = consumer warp 0 starts waiting for it, 2 = that wait returns (the copy
 * had landed), 3 = warp 0 done with the stage; then 8 points per [phase][cta] inside
 * the phase (GEMV: input polled, normalised, in registers; attention: inputs polled,
 * first K/V stage landed, first chunk reduced, outputs written).  *n_phases and *n_ctas
 * (nullable) receive the dimensions.  Takes effect at the next mie_decode_step. */
mie_status mie_set_trace(mie_ctx *ctx, void *device_buffer, size_t bytes, int *n_phases, int *n_ctas);

/* Synchronises the context's stream, then reads and clears its device error flags:
 * MIE_E_DEVICE when a bounds check fired, MIE_E_TIMEOUT when a bounded device wait of
 * the persistent step gave up (its counters and tagged words are reset for the next
 * step). */
mie_status mie_sync(mie_ctx *ctx);

/* Testing aid for the bounded waits of the persistent step.  From the next
 * mie_decode_step on, phase `phase` (0-based, five per layer -- QKV, attention, O-proj,
 * gate/up, down -- then the LM head; 1 <= phase <= 5 * n_layers) reads its input vector
 * from words that no phase ever writes, and every bounded wait of the step gives up
 * after `wait_polls` rounds (one round: one L2 round trip or one mbarrier probe).  The
 * step therefore ends early with its waits timed out; mie_sync then returns
 * MIE_E_TIMEOUT and resets the step's counters and tagged words.  phase < 0 restores
 * the normal phase table and the default limit (a few seconds), after which steps are
 * correct again.  The chain mode has no tagged inputs and is not affected.  MIE_E_ARG
 * for phase 0 (it has no input to withhold), a phase past the LM head, or
 * wait_polls < 1. */
mie_status mie_debug_stall(mie_ctx *ctx, int phase, long wait_polls);

/* Sampling of the next token inside the step's graph (mie_sample's rule, with seed
 * `seed` and the step's position pos: the step that writes position pos draws with
 * u_i(seed, pos, i)).  From the next mie_decode_step on, the draw replaces the argmax:
 * it goes to argmax_out and, in mie_decode_continue, becomes the next token.  The logits
 * pass through a buffer of the context when the caller passes none.  temperature <= 0
 * switches back to greedy decoding.  The few-slot step stays greedy.  MIE_E_ARG as for
 * mie_sample. */
mie_status mie_set_sampling(mie_ctx *ctx, float temperature, int top_k, float top_p,
                            uint64_t seed);

/* Kernel launches one mie_decode_step replay performs (for launch accounting). */
int mie_step_launches(const mie_ctx *ctx);

/* Kernel launches one mie_decode_step_slots replay performs (0 before its first call). */
int mie_slot_step_launches(const mie_ctx *ctx);

#ifdef __cplusplus
}
#endif

#endif /* MIE_H_ */
