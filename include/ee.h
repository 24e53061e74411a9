/*
 * ee.h -- C ABI of the GB300 early-exit decoding library (libee.so).
 *
 * What the library computes.  Greedy autoregressive decoding of B
 * independent sequences through a Llama-style decoder (RMSNorm, rotary GQA
 * attention over a paged KV cache, SwiGLU FFN, tied embedding / LM head),
 * with early exit:
 *  - every sequence runs the bf16 backbone layers until a checkpoint layer l
 *    whose exit head is confident, conf = max softmax(RMSNorm_f(h_l) T_l E^T)
 *    > gamma_l (the low-rank exit head softmax(h T E^T) with T in R^{d x d}
 *    and the test p > gamma of "大语言模型解码加速：自适应层并行机制解析" §2.1-2.2;
 *    a sharp softmax is a confident one and thresholds are per layer, CALM
 *    article §2.1-2.2 and the decode loop of §3.1);
 *  - after the exit the remaining layers l+1..L-1 run as W4A16 copies of the
 *    same layers (group-128 symmetric int4 with bf16 scales) which write their
 *    K/V into the same cache slots as the backbone would ("River-LLM 深度解析"
 *    §4.1-4.3, ExitLayer and SharedKVCache of §8.1-8.2), so no layer ever
 *    misses K/V for later tokens;
 *  - the emitted token is the final LM head's argmax (lowest index on ties).
 * Each decode step compacts the batch per layer into a "full" (bf16) and an
 * "exit" (int4) sub-batch instead of masking exited rows (the dynamic batch
 * regrouping of the CALM article §3.3).
 *
 * Precision.  Backbone weights, E and T are bf16; exit-layer weights int4
 * with bf16 scales; activations fed to the projections and the K/V cache are
 * fp16 (16-bit activations, the A16 of W4A16); accumulation, the residual
 * stream, softmax and RoPE are fp32.
 *
 * Conventions.
 *  - Everything on the device lives in one arena that the CALLER allocates
 *    (ee_arena_bytes tells how much); the library never calls cudaMalloc.
 *    It allocates only a few KB of pinned host staging (cudaHostAlloc) per
 *    context for its per-step host<->device copies.
 *  - All calls run on the stream given to ee_create and return after that
 *    stream has finished the call's work (synchronous), unless stated.
 *  - Weight pointers may be host or device memory (copied with
 *    cudaMemcpyDefault); the caller keeps ownership.  bf16 tensors are passed
 *    as uint16_t bit patterns, row-major [out, in] as in nn.Linear.
 *  - Errors return a status, set ee_last_error(ctx) and leave the context
 *    usable unless the status is EE_ERR_CUDA.  Arguments are validated on the
 *    host before any launch.
 *  - A context is not thread-safe; use one per host thread.
 */
#ifndef EE_H_
#define EE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  EE_OK = 0,
  EE_ERR_INVALID_ARG = 1,     /* bad pointer, size, shape, token id, ... */
  EE_ERR_STATE = 2,           /* call out of order (e.g. decode before prefill) */
  EE_ERR_CAPACITY = 3,        /* batch or sequence length beyond the context's limits */
  EE_ERR_OOM_ARENA = 4,       /* arena smaller than ee_arena_bytes() */
  EE_ERR_CUDA = 5,            /* a CUDA runtime call failed; context unusable */
  EE_ERR_DEVICE_TIMEOUT = 6,  /* a bounded device-side wait gave up (see ee_last_error) */
  EE_ERR_UNSUPPORTED = 7      /* shape the kernels do not handle (see ee_last_error) */
} ee_status;

/* Limits of this build. */
#define EE_MAX_BATCH 64
#define EE_MAX_CHECKPOINTS 32
#define EE_QUANT_GROUP 128
#define EE_KV_BLOCK 16

/* Model shape and runtime limits.
 * Requirements: d_model, n_heads*head_dim and ffn_dim multiples of 32;
 * head_dim 64 or 128; n_heads / n_kv_heads in {1, 2, 4, 8}; vocab even;
 * max_seq_len <= 16384;
 * quant_group == 128; kv_block == 16; 1 <= max_batch <= EE_MAX_BATCH;
 * checkpoint_layers strictly ascending, each in [0, n_layers-2]. */
typedef struct {
  int32_t n_layers, d_model, n_heads, n_kv_heads, head_dim, ffn_dim, vocab;
  float rms_eps;     /* RMSNorm epsilon, e.g. 1e-5 */
  float rope_theta;  /* RoPE base, e.g. 10000 */
  int32_t quant_group;
  int32_t kv_block;
  int32_t max_batch;
  int32_t max_seq_len;        /* prompt + generated tokens per sequence */
  int32_t n_checkpoints;
  const int32_t *checkpoint_layers; /* [n_checkpoints], copied by ee_create */
} ee_config;

typedef struct ee_ctx ee_ctx;

/* Matrix order used by the int4 arrays below and by ee_debug_int4. */
enum { EE_WQ = 0, EE_WK, EE_WV, EE_WO, EE_WG, EE_WU, EE_WD, EE_N_MATS };

/* One decoder layer.  bf16 bit patterns, [out, in] row-major:
 *   wq [n_heads*head_dim, d], wk/wv [n_kv_heads*head_dim, d],
 *   wo [d, n_heads*head_dim], wg/wu [ffn_dim, d], wd [d, ffn_dim],
 *   g_attn/g_ffn [d] RMSNorm gains.
 * q4[m]/s4[m] optionally give the int4 exit copy of matrix m (EE_WQ..EE_WD):
 *   q4 [out, in/2] bytes, byte j of a row = column 2j (low nibble) and 2j+1
 *   (high nibble), two's complement; s4 [out, ceil(in/128)] bf16 scales,
 *   value = q * s.  If q4[m] is NULL the library quantises the bf16 matrix
 *   itself: per row and group of 128 columns, s = bf16(amax/7) and
 *   q = clamp(round_half_even(w/s), -8, 7) in float32 ("River-LLM 深度解析"
 *   §8.1 _quantize_int4, applied per group). */
typedef struct {
  const uint16_t *g_attn, *wq, *wk, *wv, *wo, *g_ffn, *wg, *wu, *wd;
  const uint8_t *q4[EE_N_MATS];
  const uint16_t *s4[EE_N_MATS];
} ee_layer_weights;

/* Tensors shared by all layers: embed = E [vocab, d] (input embedding and,
 * tied, the LM head), g_final [d], exit_T[c] = T_c [d, d] for checkpoint c in
 * the row-vector convention u = n T (so u[j] = sum_i n[i] T[i][j]). */
typedef struct {
  const uint16_t *embed;
  const uint16_t *g_final;
  const uint16_t *const *exit_T;
} ee_shared_weights;

typedef struct {
  const ee_layer_weights *layers; /* [n_layers] */
  ee_shared_weights shared;
} ee_weights;

/* ---------------------------------------------------------------- lifecycle */

/* Device bytes the context needs for cfg (weights, int4 copies, KV cache,
 * activations, scratch).  0 if cfg is invalid.  No CUDA call. */
size_t ee_arena_bytes(const ee_config *cfg);

/* Validates cfg (before any CUDA call), carves the caller's arena
 * (dev_arena, 256-byte aligned, >= ee_arena_bytes(cfg)) and binds the
 * context to the current device.  All work is queued on `stream` (a
 * cudaStream_t, not the legacy default stream, which cannot be captured into
 * a graph); with stream = NULL the context creates its own non-blocking
 * stream and orders it after the legacy default stream at every call.  The
 * arena and the stream must outlive the context. */
ee_status ee_create(const ee_config *cfg, void *dev_arena, size_t arena_bytes, void *stream,
                    ee_ctx **out);
void ee_destroy(ee_ctx *ctx);
const char *ee_last_error(const ee_ctx *ctx);

/* Loads all weights (ee_load_layer for every layer, then ee_load_shared):
 * the bf16 backbone, its int4 exit copies (each exit layer is a parameter
 * copy of the original layer quantised to 4 bits, "River-LLM 深度解析" §4.1-4.2
 * and ExitLayer in §8.1), E and the exit transforms T_l (the low-rank head
 * softmax(h T E^T) of "大语言模型解码加速：自适应层并行机制解析" §2.1).
 * Host or device pointers; copied, the caller keeps ownership.  Fails with
 * EE_ERR_INVALID_ARG on a NULL tensor; layers loaded before the failing one
 * stay loaded, and decoding is refused (EE_ERR_STATE) until every layer and
 * the shared tensors are in (a CUDA error makes the context unusable). */
ee_status ee_load_weights(ee_ctx *ctx, const ee_weights *w);
/* Loads one layer: re-lays its matrices out for the kernels and builds (or
 * copies) its int4 exit copy.  Layers may be loaded in any order. */
ee_status ee_load_layer(ee_ctx *ctx, int32_t layer, const ee_layer_weights *lw);
/* Loads E, g_final and every T_c. */
ee_status ee_load_shared(ee_ctx *ctx, const ee_shared_weights *sw);

/* gamma[c] is the threshold of checkpoint c: a sequence exits there when
 * conf > gamma[c] (strict).  One fixed threshold per exit layer (CALM article
 * §2.2); the test p(t | h^(l)) > gamma of "大语言模型解码加速：自适应层并行机制解析"
 * §2.2.  +INF never exits, -INF always exits.  Default: all +INF.  gamma is
 * a host array of n_checkpoints floats, copied; NaN is refused
 * (EE_ERR_INVALID_ARG). */
ee_status ee_set_thresholds(ee_ctx *ctx, const float *gamma);

/* enabled = 0: forced no-exit baseline -- no exit head is evaluated and every
 * layer runs in bf16 (the same kernels, minus the heads).  Default 1. */
ee_status ee_set_exit_enabled(ee_ctx *ctx, int32_t enabled);

/* Exit criteria at the checkpoint layers (ee_set_exit_criterion):
 *  EE_EXIT_MAXPROB (default): conf = max softmax(RMSNorm_f(h_l) T_l E^T)
 *    (the low-rank exit head and test p > gamma of "大语言模型解码加速：自适应层并行机制解析"
 *    §2.1-2.2);
 *  EE_EXIT_STS: the state transition similarity of the checkpoint layer,
 *    cos(layer input, layer output) with both states scaled to unit L2 norm
 *    ("River-LLM 深度解析" §5.1-5.2): a sequence's token exits when its score
 *    is above the layer's threshold tau (each token decides, §6.1).  O(d) per
 *    token, no vocabulary read (§5.3);
 *  EE_EXIT_STS_BATCH: the same score with the batch rule of §5.2: the
 *    sequences still on the full-precision path exit together when the
 *    minimum of their scores is above tau (and each records that minimum).
 * Either way the thresholds are those of ee_set_thresholds (strict >) and
 * ee_debug_conf returns the scores. */
enum { EE_EXIT_MAXPROB = 0, EE_EXIT_STS = 1, EE_EXIT_STS_BATCH = 2 };
ee_status ee_set_exit_criterion(ee_ctx *ctx, int32_t criterion);

/* Token source of an exited sequence (ee_set_token_source):
 *  EE_TOKEN_FINAL_HEAD (default): the final LM head's argmax after the
 *    sequence's remaining layers ran on the int4 copies;
 *  EE_TOKEN_EXIT_HEAD: the argmax of the exit head that let it leave (the
 *    CALM article §3.1 loop returns the exit head's prediction; page 3 of
 *    "大语言模型解码加速：自适应层并行机制解析" §2.2).  Its remaining layers still
 *    run on the int4 copies to write their K/V, except that in the last layer
 *    only the QKV projection (the K/V write) runs for it; the final head
 *    serves the sequences that never exited.  Needs EE_EXIT_MAXPROB
 *    (ee_decode_step returns EE_ERR_STATE otherwise). */
enum { EE_TOKEN_FINAL_HEAD = 0, EE_TOKEN_EXIT_HEAD = 1 };
ee_status ee_set_token_source(ee_ctx *ctx, int32_t source);

/* use_graph = 1 (default): a decode step is replayed from a CUDA graph
 * captured on first use for the batch size and exit mode (all per-step
 * state lives on the device).  0: launch kernels one by one. */
ee_status ee_set_use_graph(ee_ctx *ctx, int32_t use_graph);

/* ---------------------------------------------------------------- decoding */

/* Prefill phase ("River-LLM 深度解析" §6.1, the first of its two phases; it
 * is run here without an exit, in full precision).
 * Starts `batch` new sequences (any previous ones are dropped as by
 * ee_reset) and runs the bf16 stack over every prompt position with no exit,
 * writing every layer's K/V at positions 0..len-1.  tokens_concat holds the
 * prompts back to back (sum(prompt_lens) ids in [0, vocab)); each
 * prompt_lens[s] >= 1 and < max_seq_len.  first_tokens_out[s] (host, [batch])
 * receives the argmax of the final head at the prompt's last position. */
ee_status ee_prefill(ee_ctx *ctx, int32_t batch, const int32_t *prompt_lens,
                     const int32_t *tokens_concat, int32_t *first_tokens_out);

/* Sequence-level exit in prefill ("River-LLM 深度解析" §6.1, the prefill half
 * of its two-phase strategy): with tau set (n_checkpoints floats, host,
 * copied), ee_prefill scores every prompt token with the state transition
 * similarity at each checkpoint layer (§5.1) and a prompt leaves the
 * full-precision path at the first checkpoint where the minimum over its
 * tokens is above tau[c] (strict; the batch rule of §5.2 over the prompt's
 * tokens): its later layers run on the int4 copies for all of its tokens
 * and write their K/V.  The prefill then takes two passes over the prompts
 * (scoring, then the run with those exits).  tau = NULL (default) turns it
 * off: plain bf16 prefill.  ee_prefill_exit_layers writes, per sequence of
 * the last prefill, the layer its prompt left at (n_layers - 1: none). */
ee_status ee_set_prefill_exit(ee_ctx *ctx, const float *tau);
ee_status ee_prefill_exit_layers(const ee_ctx *ctx, int32_t *out);

/* One early-exit greedy decode step for every sequence (the per-token loop
 * of the CALM article §3.1: run a layer, write its K/V, score the exit head at
 * a checkpoint and leave the full-precision path once it clears gamma; the
 * head and test of "大语言模型解码加速：自适应层并行机制解析" §2.1-2.2; after the
 * exit the int4 copies of "River-LLM 深度解析" §4.1-4.3 run the remaining
 * layers and write their K/V into the shared cache).  in_tokens[s] (host,
 * [batch]) is the token at the sequence's next position; ids outside
 * [0, vocab) give EE_ERR_INVALID_ARG before any launch.  Writes
 * next_tokens_out[s] and exit_layers_out[s] (host, [batch]): the checkpoint
 * layer at which s exited, or n_layers-1 if it ran the whole bf16 stack.
 * Fails with EE_ERR_CAPACITY if a sequence would pass max_seq_len. */
ee_status ee_decode_step(ee_ctx *ctx, const int32_t *in_tokens, int32_t *next_tokens_out,
                         int32_t *exit_layers_out);

/* Drops all sequences and frees every KV block; weights and thresholds stay.
 * The pages' shared cache (SharedKVCache of "River-LLM 深度解析" §8.2) grows
 * per layer by concatenation; here it is a paged pool, and reset returns
 * every block to the pool (the slots are refilled with a sentinel). */
ee_status ee_reset(ee_ctx *ctx);

/* Number of active sequences and the position (tokens in the cache) of
 * sequence seq. */
ee_status ee_seq_info(const ee_ctx *ctx, int32_t *batch, int32_t seq, int32_t *pos);

/* Device time of the last prefill/decode step: CUDA events recorded on the
 * context's stream right before and after the step's work (the graph replay,
 * with its two small copies).  In profile mode, the sum of the launches. */
ee_status ee_last_step_ms(const ee_ctx *ctx, float *ms);

/* Bytes one decode step copies host -> device and device -> host for a batch
 * of `batch` sequences, and the number of kernels it launches with exit heads
 * enabled (heads = 1) or not.  No CUDA call. */
ee_status ee_step_io(const ee_ctx *ctx, int32_t batch, int32_t heads, size_t *h2d_bytes,
                     size_t *d2h_bytes, int32_t *launches);

/* Kinds of kernel launch in a decode step (ee_launch_record.kind). */
enum {
  EE_K_BEGIN = 0,      /* embedding gather, positions, lists            */
  EE_K_NORM = 1,       /* attention / FFN RMSNorm                       */
  EE_K_QKV = 2,        /* QKV GEMV + RoPE + K/V write                   */
  EE_K_ATTN = 3,       /* decode attention                              */
  EE_K_O = 4,          /* O GEMV + residual                             */
  EE_K_GATEUP = 5,     /* gate/up GEMV + SwiGLU                         */
  EE_K_DOWN = 6,       /* down GEMV + residual                          */
  EE_K_HEAD_NORM = 7,  /* checkpoint: final-norm of the full sub-batch  */
  EE_K_HEAD_T = 8,     /* checkpoint: u = n T GEMV                      */
  EE_K_HEAD_E = 9,     /* checkpoint: vocabulary head + exit decision   */
  EE_K_FINAL_NORM = 10,
  EE_K_FINAL_HEAD = 11, /* final LM head, argmax                         */
  EE_K_EXIT_STS = 12    /* checkpoint: similarity score + exit decision   */
};
/* Sub-batch lists a projection or head launch serves (ee_launch_record.lists). */
enum {
  EE_LISTS_BOTH = 0,  /* the full list on bf16 weights and the exit list on int4 in one launch: the
                         GEMV, and the tensor-core GEMM after the first checkpoint (also every
                         launch that is not a projection or head) */
  EE_LISTS_FULL = 1   /* the full list only: tensor-core GEMM launches up to the first checkpoint,
                         and the heads */
};
typedef struct {
  int32_t kind;     /* EE_K_* */
  int32_t layer;    /* decoder layer, or -1 */
  float ms;         /* device time between events around the launch */
  float kernel_ms;  /* GEMV and tensor-core GEMM launches: the kernel's own
                       time, first CTA start to last CTA end (%globaltimer),
                       no launch gaps; 0 for the other kernels */
  int32_t lists;    /* EE_LISTS_* */
} ee_launch_record;

/* profile = 1: the following decode steps run without the CUDA graph and
 * with a CUDA event pair around every kernel launch (this serialises the
 * launches, so step times are longer than without profiling);
 * ee_profile_read returns the last step's launches in order. */
ee_status ee_set_profile(ee_ctx *ctx, int32_t profile);
ee_status ee_profile_read(ee_ctx *ctx, ee_launch_record *out, int32_t cap, int32_t *n);

/* ------------------------------------------------- inspection (tests, tools) */

/* debug = 1 makes each step also keep the residual stream after every layer
 * (for ee_debug_hidden).  It adds one small write per layer. */
ee_status ee_set_debug(ee_ctx *ctx, int32_t debug);
/* Residual stream h after `layer` in the last step (debug mode): [batch, d] fp32. */
ee_status ee_debug_hidden(ee_ctx *ctx, int32_t layer, float *out);
/* Exit-head confidences of the last step, [batch, n_checkpoints] fp32, NaN
 * where the head was not evaluated. */
ee_status ee_debug_conf(ee_ctx *ctx, float *out);
/* K and V (fp16 bits, [n_kv_heads*head_dim] each, host) stored for sequence
 * seq at layer `layer`, position pos (pos < the sequence's position). */
ee_status ee_debug_kv(ee_ctx *ctx, int32_t seq, int32_t layer, int32_t pos, uint16_t *k,
                      uint16_t *v);
/* Block ids of sequence seq's block table: out[i] for i < *n_blocks. */
ee_status ee_debug_block_table(ee_ctx *ctx, int32_t seq, int32_t *out, int32_t cap,
                               int32_t *n_blocks);
/* The int4 exit copy of matrix `mat` of `layer` in the input layout above:
 * packed [out, in/2] bytes and scales [out, ceil(in/128)] bf16 bits (host),
 * whatever layout the kernels keep internally (the read-back undoes it), so
 * that the codes and scales can be compared bit for bit with the host
 * quantiser of "River-LLM 深度解析" §8.1 (dequantised value = q * s). */
ee_status ee_debug_int4(ee_ctx *ctx, int32_t layer, int32_t mat, uint8_t *packed,
                        uint16_t *scales);

/* ------------------------------------------- single kernels (device pointers)
 * The building blocks of a decode step, each on the given stream, with
 * device pointers.  They return after enqueueing (asynchronous) and report
 * only argument errors; `err_flag` (device int32, may be NULL) receives a
 * non-zero code if a bounded device wait gave up. */

/* Group-128 int4 quantiser (see ee_layer_weights): w [rows, cols] bf16 ->
 * packed [rows, cols/2] and scales [rows, scale_stride] (scale_stride >=
 * ceil(cols/128)).  cols % 32 == 0. */
ee_status ee_op_quantize_int4(const uint16_t *w, int32_t rows, int32_t cols, uint8_t *packed,
                              uint16_t *scales, int32_t scale_stride, void *stream);

/* Activations.  The kernels carry activations in fp16 (the A16 of W4A16)
 * and accumulate in fp32.  An activation row of K values is stored in "pair
 * order": within each run of 8 columns c..c+7 the stored order is
 * c, c+4, c+1, c+5, c+2, c+6, c+3, c+7, so that one 16-byte load gives the
 * (c+j, c+j+4) pairs that match the nibble pairs of a packed int4 word. */

/* y[m, n] = sum_k x[m, k] W[n, k] for m < M (M <= EE_MAX_BATCH): bf16 W
 * [N, K], x fp16 [M, K] in pair order, y fp32 [M, N].  K % 32 == 0, N even. */
ee_status ee_op_linear_bf16(int32_t M, int32_t N, int32_t K, const uint16_t *x_f16,
                            const uint16_t *w, float *y, int32_t *err_flag, void *stream);
/* Same with the int4 copy: packed [N, K/2], scales [N, scale_stride] bf16
 * with scale_stride >= ceil(K/128) (scale_stride = K/128 with K % 512 == 0
 * lets the scales stream with the weights); x fp16 [M, K] in pair order. */
ee_status ee_op_linear_int4(int32_t M, int32_t N, int32_t K, const uint16_t *x_f16,
                            const uint8_t *packed, const uint16_t *scales, int32_t scale_stride,
                            float *y, int32_t *err_flag, void *stream);

/* Paged GQA decode attention (one query position per sequence, causal over
 * positions 0..pos[s], pos[s] + 1 <= max_ctx <= 16384):  o[s, h*hd + i] = sum_t softmax_t(q_h . k_t / sqrt(hd)) v_t[i]
 * with kv head g = floor(h * Hkv / Hq).
 *   q [B, Hq*hd] fp32; kcache/vcache [n_blocks, Hkv, 16, hd] fp16 (one
 *   layer, the layout of the context's shared cache); block_table [B, bt_stride] int32; pos [B] int32 (the query's
 *   position, so ctx = pos + 1); o [B, Hq*hd] fp32.
 * scratch: device buffer of ee_attention_scratch_bytes(B, Hq, Hkv, hd, max_ctx) bytes;
 * its counters must be zero on the first call (ee_create does this for the
 * context's own scratch; for this entry point, zero it once with cudaMemset)
 * and are left at zero by every call. */
size_t ee_attention_scratch_bytes(int32_t B, int32_t n_heads, int32_t n_kv_heads,
                                  int32_t head_dim, int32_t max_ctx);
ee_status ee_op_attention(int32_t B, int32_t n_heads, int32_t n_kv_heads, int32_t head_dim,
                          int32_t max_ctx, const float *q, const uint16_t *kcache,
                          const uint16_t *vcache,
                          const int32_t *block_table, int32_t bt_stride, const int32_t *pos,
                          float *o, void *scratch, int32_t *err_flag, void *stream);

/* Vocabulary head over M rows: z[m, v] = u[m, :] . E[v, :] (u fp16 [M, d]
 * in pair order, E bf16 [V, d]); writes conf[m] = max_v softmax(z[m])_v = 1/sum_v exp(z_v - z_max)
 * and argmax[m] (lowest index on ties).  scratch: ee_head_scratch_bytes(M)
 * bytes, counters zero on the first call and left zero. */
size_t ee_head_scratch_bytes(int32_t M);
ee_status ee_op_vocab_head(int32_t M, int32_t V, int32_t d, const uint16_t *u_f16, const uint16_t *E,
                           float *conf, int32_t *argmax, void *scratch, int32_t *err_flag,
                           void *stream);

/* ---- attention without a caller-provided scratch buffer ------------------
 * Not part of the early-exit method: the pages have no counterpart.  It is
 * for callers that cannot allocate device memory, or hand the library a
 * buffer, at the time they call: a host whose caching allocator has already
 * reserved the device's free memory (a cudaMalloc from outside it may fail or
 * synchronise the device), or one that allows no allocation after start-up.
 *
 * Same operation, arguments, layouts and results as ee_op_attention, minus
 * `scratch`.  The scratch is a fixed array of EE_ATTN_STATIC_SCRATCH_BYTES
 * inside the library; the call allocates nothing (no cudaMalloc, cudaFree or
 * allocating library call).  A shape whose ee_attention_scratch_bytes(...)
 * exceeds that size returns EE_ERR_CAPACITY without touching the device (for
 * Llama-3.1-8B heads, Hq 32, Hkv 8, hd 128, it fits B = 1 at every max_ctx up
 * to 16384, and B <= 9 at max_ctx 2048).  Invalid shapes return
 * EE_ERR_INVALID_ARG.
 *
 *  - The first call on each device looks up the array's device address
 *    (cudaGetSymbolAddress, with that device current); make that first call
 *    before capturing any stream into a graph.
 *  - Each call zeroes the array's merge counters on `stream` (cudaMemsetAsync)
 *    and then launches the kernel; it returns without waiting for either.
 *  - The array is shared by every call on a device and keeps the last call's
 *    partial results.  Calls that overlap in time on one device (from two
 *    streams or host threads) race on it: order them, e.g. on one stream. */
#define EE_ATTN_STATIC_SCRATCH_BYTES (4u << 20)
ee_status ee_op_attention_noalloc(int32_t B, int32_t n_heads, int32_t n_kv_heads,
                                  int32_t head_dim, int32_t max_ctx, const float *q,
                                  const uint16_t *kcache, const uint16_t *vcache,
                                  const int32_t *block_table, int32_t bt_stride,
                                  const int32_t *pos, float *o, int32_t *err_flag, void *stream);

#ifdef __cplusplus
}
#endif
#endif /* EE_H_ */
