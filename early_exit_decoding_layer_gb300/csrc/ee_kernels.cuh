// Launch parameters and host-side launchers of the decode-step kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/ee.h"

namespace ee {

// ------------------------------------------------------------------ lists
// A sequence list in device memory: [0] = count, [1 + i] = sequence id.
constexpr int kListLen = 1 + EE_MAX_BATCH;

// Per-step device state that the kernels read and update.
struct StepLists {
  int32_t part[kListLen];   // sequences taking part in this step
  int32_t full[kListLen];   // still on the bf16 backbone (ascending ids)
  int32_t exitl[kListLen];  // exited, running the int4 copies (ascending ids)
  int32_t fin[kListLen];    // rows of the final LM head
  int32_t forced[EE_MAX_BATCH];  // by sequence id: checkpoint layer where it must exit, or -1
};

// Host -> device step descriptor (copied each step from pinned staging).
struct StepDesc {
  int32_t n_part;
  int32_t part[EE_MAX_BATCH];
  int32_t n_fin;
  int32_t fin[EE_MAX_BATCH];
  int32_t tokens[EE_MAX_BATCH];     // by sequence id
  int32_t pos[EE_MAX_BATCH];        // position of this step's token, by sequence id
  int32_t new_block[EE_MAX_BATCH];  // block to map at pos/16, or -1, by sequence id
  int32_t forced_exit[EE_MAX_BATCH];  // checkpoint layer where the sequence must exit, or -1
  int32_t debug;                    // keep per-layer hidden states
};

// Device -> host step outputs.  One copy per step of the head of the struct
// up to the confidences of the batch's sequences.
struct StepOut {
  int32_t err;                      // first device error code, 0 if none
  int32_t pad[3];
  int32_t next_token[EE_MAX_BATCH];
  int32_t exit_layer[EE_MAX_BATCH];
  float conf[EE_MAX_BATCH * EE_MAX_CHECKPOINTS];  // [seq][checkpoint], NaN = not evaluated
};

// ------------------------------------------------------------------ GEMV
enum Epi : int32_t {
  EPI_F32 = 0,     // out_f32[seq * out_stride + n] = y
  EPI_QKV = 1,     // RoPE on q/k row pairs, q -> q_out, k/v (fp16) -> paged cache
  EPI_RESID = 2,   // h[seq, n] += y (+ debug copy)
  EPI_SWIGLU = 3,  // rows (2i, 2i+1) = (gate_i, up_i) -> x_out[seq, i] = silu(g) u (fp16)
  EPI_X = 4,       // x_out[seq, n] = y (fp16, pair order)
  EPI_HEAD = 5,    // vocabulary head: per-row softmax statistics and argmax
};

enum HeadMode : int32_t { HEAD_CONF_ARGMAX = 0, HEAD_CHECKPOINT = 1, HEAD_FINAL = 2 };

struct LinearParams {
  // profile mode: globaltimer (ns) of the first CTA's start (atomic min) and
  // the last CTA's end (atomic max) of this launch; null: not recorded
  unsigned long long* stamp_start;
  unsigned long long* stamp_end;
  int32_t N, K;
  int32_t max_rows;          // upper bound of the list counts (sequences of the step)
  // filled by launch_linear: staged activation rows (0: read from global),
  // sequences per pass, per-row sum capacity
  int32_t xs_rows, mcap, rows_cap;
  // weights: bf16 [N, K]; int4 packed [N, K/2] with bf16 scales [N, sstride]
  const uint16_t* w;
  const uint8_t* wq;
  const uint16_t* ws;
  int32_t sstride;           // scale row stride (elements); ceil(K/128) keeps rows unpadded
  const uint8_t* wq4t;       // the same int4 copy in the tensor-core GEMM's blocks (or null)
  // rows: either lists (count + ids) or a direct count with ids 0..m_direct-1
  const int32_t* list_full;  // rows on the bf16 weights (may be null)
  const int32_t* list_exit;  // rows on the int4 weights (may be null)
  // nonzero: the previous launch wrote the lists, so they are read only after
  // the grid dependency wait (and no weights are requested before it)
  int32_t lists_after_wait;
  int32_t m_direct_full;     // used when list_full == null
  int32_t m_direct_exit;     // used when list_exit == null
  // activations by sequence id, fp16 in pair order (runs of 8: 0,4,1,5,2,6,3,7)
  const uint16_t* xh;
  int32_t x_stride;
  // RMSNorm applied while staging (only when linear_stages_x() holds): the
  // staged row is fp16(h * rsqrt(mean(h^2) + eps) * g) from the fp32 residual
  // stream instead of xh (null: stage xh as is)
  const float* norm_h;
  int32_t norm_stride;
  const uint16_t* norm_g;
  float norm_eps;
  int32_t epi;
  // EPI_F32
  float* out_f32;
  int32_t out_stride;
  // EPI_QKV
  float* q_out;              // [seq][Hq*hd]
  uint16_t* kc;              // this layer's K cache [blocks][Hkv][16][hd] fp16
  uint16_t* vc;
  const int32_t* block_table;
  int32_t bt_stride;
  const int32_t* pos;        // by sequence id
  const float2* rope;        // [max_seq_len][hd/2] (cos, sin)
  int32_t n_heads, n_kv_heads, head_dim;
  // EPI_RESID
  float* h;
  int32_t h_stride;
  float* hdbg;               // [seq][h_stride] copy when *dbg_flag != 0
  const int32_t* dbg_flag;
  float* hsave;              // non-null: [seq][h_stride] copy of the new h (the next layer's input state)
  // EPI_SWIGLU / EPI_X (fp16, pair order)
  uint16_t* xh_out;
  int32_t xo_stride;
  // EPI_HEAD
  int32_t head_mode;
  float* head_part;          // [grid][EE_MAX_BATCH][4] partial (max, sum, argmax, -)
  int32_t* head_counter;     // zero between launches
  float* conf_out;           // HEAD_CONF_ARGMAX: [m]; HEAD_CHECKPOINT: StepOut.conf
  int32_t* argmax_out;       // HEAD_CONF_ARGMAX: [m]; HEAD_FINAL: StepOut.next_token;
                             // HEAD_CHECKPOINT (non-null: exit-head tokens): StepOut.next_token of the exiting
  StepLists* lists;          // HEAD_CHECKPOINT: lists to compact
  int32_t* exit_layer;       // HEAD_CHECKPOINT: StepOut.exit_layer
  const float* gamma;        // thresholds [n_checkpoints]
  int32_t ckpt_index, ckpt_layer;
  int32_t* err;
};

// ------------------------------------------------------------------ tensor-core GEMM
// For steps whose batch is above the GEMV's staging limit: one launch serves
// one sub-batch list (MODE 0: the full list on the bf16 weights through
// `amap`; MODE 1: the exit list on the int4 copy), 128 weight rows per tile,
// the K range split `ksplit` ways.
struct TcParams {
  CUtensorMap amap;     // bf16 weights [N, K]: box 64 (K) x 128 (rows), 128-byte swizzle
  LinearParams lp;      // shapes, lists, activations, epilogue (as for the GEMV)
  const uint8_t* q4t;   // MODE 1: the int4 copy in blocks (int4_tc_layout_bytes)
  int32_t ntiles, ksplit, nks, nk;  // tiles, K splits, 64-wide K steps per split, K steps
  int32_t modes;        // 1: the full list's units (bf16) only; 2: then the exit list's (int4)
  float* part;          // [mode][tile][split][64 columns][128 rows] fp32 partial sums
  int32_t* tile_cnt;    // [mode][ntiles] split counters, zero between launches
};
struct TcPlan {
  int ntiles, ksplit, nks, nk;
};
// K splits: the fewest that fill the waves, within max_units work units.
TcPlan gemm_tc_plan(int N, int K, int num_sms, int max_units);
bool gemm_tc_shape_ok(int K);
size_t gemm_tc_part_floats(int units);
cudaError_t gemm_tc_prepare();
cudaError_t launch_gemm_tc(const TcParams& tp, bool pdl, cudaStream_t st);
// The int4 copy for MODE 1: per 128-row tile and 64-column K step, one
// block of 128 rows x 32 bytes of nibbles and 128 bf16 scales.
size_t int4_tc_layout_bytes(int rows, int cols);
cudaError_t launch_int4_tc_layout(const uint8_t* packed, const uint16_t* scales, int rows, int cols, int sstride,
                                  uint8_t* out, cudaStream_t st);
// Tensor map of a bf16 weight matrix [N, K] (row stride K) for MODE 0.
bool encode_weight_map(CUtensorMap* map, const uint16_t* w, int N, int K);

// Bytes of dynamic shared memory the GEMV kernel uses.
size_t linear_smem_bytes();
// Sets the kernels' shared-memory attributes on the current device (call once
// per device before the first launch, outside stream capture).
cudaError_t linear_prepare();
// Launches the GEMV on `grid` CTAs (grid <= number of SMs).  pdl: launch
// with programmatic stream serialisation.
cudaError_t launch_linear(const LinearParams& p, int grid, bool pdl, cudaStream_t st);
int linear_grid(int N, int num_sms);
// True if rows of K bf16 or int4 weights can be streamed in row-aligned stages.
bool linear_shape_ok(int K);
// True when a launch over at most max_rows sequences stages its activations
// in shared memory (and so can apply RMSNorm itself).
bool linear_stages_x(int max_rows, int K);

// ------------------------------------------------------------------ attention
struct AttnParams {
  const int32_t* list;       // sequences (count + ids) or null -> ids 0..m_direct-1
  int32_t m_direct;
  int32_t n_heads, n_kv_heads, head_dim;
  const float* q;            // [seq][Hq*hd]
  int32_t q_stride;
  const uint16_t* kc;
  const uint16_t* vc;
  const int32_t* block_table;
  int32_t bt_stride;
  const int32_t* pos;        // query position by sequence id (ctx = pos + 1)
  int32_t nsplit;            // CTAs per (sequence, kv head): attention_nsplit(max context)
  int32_t bpc;               // 16-slot blocks per CTA: attention_blocks_per_cta(head_dim)
  float* part;               // scratch partials
  int32_t* counters;         // [batch_slots][Hkv], zero between launches
  float* o_f32;              // [seq][Hq*hd] (op) or null
  uint16_t* oh;              // fp16 in pair order, or null
  int32_t o_stride;
  int32_t* err;
};
size_t attention_part_floats(int batch_slots, int n_heads, int n_kv_heads, int head_dim, int nsplit);
cudaError_t launch_attention(const AttnParams& p, int batch_slots, bool pdl, cudaStream_t st);
int attention_blocks_per_cta(int head_dim);
int attention_nsplit(int max_ctx, int head_dim);
int attention_max_split();
cudaError_t attention_prepare();

// ------------------------------------------------------------------ small kernels
struct NormParams {
  const int32_t* list;
  const float* h;
  int32_t h_stride;
  const uint16_t* g;
  int32_t d;
  float eps;
  uint16_t* xh;               // fp16, pair order
  int32_t x_stride;
};
cudaError_t launch_rmsnorm(const NormParams& p, int batch_slots, bool pdl, cudaStream_t st);

struct BeginParams {
  const StepDesc* desc;
  StepLists* lists;
  StepOut* out;
  const uint16_t* embed;
  int32_t d;
  float* h;
  int32_t h_stride;
  int32_t* pos;
  int32_t* block_table;
  int32_t bt_stride;
  int32_t n_layers;
  int32_t n_ckpt;
  int32_t* dbg_flag;
  float* hsave;              // non-null: also store the embedding there (input state of layer 0)
};
cudaError_t launch_step_begin(const BeginParams& p, int batch_slots, cudaStream_t st);

// State-transition-similarity exit decision at a checkpoint layer: for each
// sequence of the full list, cos(h_in, h) of the layer's input and output
// states; exit when it is above the threshold (strict); the lists are rebuilt
// as after an exit head.  One CTA per list entry, the last CTA decides.
struct StsParams {
  StepLists* lists;
  const float* h;            // residual stream after the checkpoint layer [seq][h_stride]
  const float* h_in;         // its input state [seq][h_stride]
  int32_t d, h_stride;
  const float* gamma;        // thresholds [n_checkpoints]
  int32_t ckpt_index, ckpt_layer;
  float* conf_out;           // StepOut.conf ([seq][EE_MAX_CHECKPOINTS])
  int32_t* exit_layer;       // StepOut.exit_layer
  float* score;              // scratch [EE_MAX_BATCH]
  int32_t* counter;          // zero between launches
  int32_t batch_min;         // nonzero: the list's minimum score decides for all of it
};
cudaError_t launch_sts(const StsParams& p, int batch_slots, bool pdl, cudaStream_t st);

cudaError_t launch_quantize_int4(const uint16_t* w, int rows, int cols, uint8_t* packed,
                                 uint16_t* scales, int sstride, cudaStream_t st);

// Row copy with an optional row permutation (load-time re-layout).
enum RowMap : int32_t {
  MAP_IDENTITY = 0,     // dst row = r
  MAP_ROPE_PAIRS = 1,   // within heads of `param` rows: i < hd/2 -> 2i, else 2(i-hd/2)+1
  MAP_INTERLEAVE = 2,   // dst row = 2r + param
};
cudaError_t launch_copy_rows(void* dst, int64_t dst_stride_bytes, int64_t dst_row0,
                             const void* src, int64_t src_stride_bytes, int64_t row_bytes,
                             int64_t nrows, int map, int param, cudaStream_t st);
cudaError_t launch_transpose_bf16(uint16_t* dst, const uint16_t* src, int n, cudaStream_t st);
cudaError_t launch_fill_u16(uint16_t* p, uint16_t v, int64_t n, cudaStream_t st);


}  // namespace ee
