// Runtime of the early-exit decode library: context, arena layout, weight
// loading and re-layout, host-side paged-KV allocator, the decode-step
// orchestrator (kernels chained with programmatic dependent launch and
// replayed from CUDA graphs), and the C ABI declared in include/ee.h.
#include <cuda_runtime.h>
#include <math.h>
#include <stdarg.h>
#include <stddef.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <map>
#include <string>
#include <vector>

#include "../../include/ee.h"
#include "ee_kernels.cuh"

using namespace ee;

namespace {

constexpr size_t kAlign = 256;

size_t step_d2h_bytes(int B) { return offsetof(StepOut, conf) + (size_t)B * EE_MAX_CHECKPOINTS * sizeof(float); }
constexpr int kHeadGridMax = 1024;      // partials of a vocabulary-head launch (GEMV CTAs or GEMM tiles)
constexpr int kTcMinBatch = 9;          // steps with more sequences use the tensor-core GEMM
constexpr int kTcMaxUnits = 1024;       // (tile, K split) work units of one tensor-core launch
constexpr int kTcMaxTiles = 1024;

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
int sstride_of(int K) { return (int)ceil_div(K, EE_QUANT_GROUP); }

constexpr int kProfMax = 4096;  // launches per profiled step with stamps

struct Carver {
  uint8_t* base;
  size_t off = 0;
  explicit Carver(uint8_t* b) : base(b) {}
  template <class T>
  T* take(size_t count) {
    off = align_up(off, kAlign);
    T* p = base ? reinterpret_cast<T*>(base + off) : nullptr;
    off += count * sizeof(T);
    return p;
  }
};

struct Mat4 {  // int4 copy of one fused matrix
  uint8_t* q;     // row layout (GEMV)
  uint16_t* s;
  uint8_t* qt;    // tensor-core GEMM blocks (contexts that may run a step on it), else null
};

struct LayerBufs {
  uint16_t *wqkv, *wo, *wgu, *wd, *g_attn, *g_ffn;
  Mat4 qkv, o, gu, d;
};

struct Dims {
  int L, d, hq, hkv, hd, F, V, nck, maxb, maxs;
  int dq, dk, nqkv, bps, nblocks;
  size_t kv_layer_elems;
};

Dims dims_of(const ee_config& c) {
  Dims m;
  m.L = c.n_layers;
  m.d = c.d_model;
  m.hq = c.n_heads;
  m.hkv = c.n_kv_heads;
  m.hd = c.head_dim;
  m.F = c.ffn_dim;
  m.V = c.vocab;
  m.nck = c.n_checkpoints;
  m.maxb = c.max_batch;
  m.maxs = c.max_seq_len;
  m.dq = m.hq * m.hd;
  m.dk = m.hkv * m.hd;
  m.nqkv = m.dq + 2 * m.dk;
  m.bps = (int)ceil_div(m.maxs, EE_KV_BLOCK);
  m.nblocks = m.maxb * m.bps;
  m.kv_layer_elems = (size_t)m.nblocks * m.hkv * EE_KV_BLOCK * m.hd;
  return m;
}

// The GEMV stages a step's activations in shared memory only for a few short
// rows; a step whose activations it cannot stage for every projection (more
// than kTcMinBatch - 1 sequences, or rows of the widest input too long for
// the staging area) runs its projections and heads on the tensor-core GEMM.
int widest_input(const Dims& m) { return std::max({m.d, m.dq, m.F}); }
bool batch_uses_tc(const Dims& m, int B) { return B >= kTcMinBatch || !linear_stages_x(B, widest_input(m)); }
// contexts that may run such a step carry the tensor-core GEMM's buffers
bool ctx_needs_tc(const Dims& m) { return batch_uses_tc(m, m.maxb); }

}  // namespace

struct ee_ctx {
  ee_config cfg;
  std::vector<int32_t> ckpts;
  Dims m;
  int dev = 0, num_sms = 0;
  bool pdl = true;  // programmatic dependent launch between the step's kernels
  cudaStream_t user_stream = nullptr;
  cudaStream_t st = nullptr;   // the caller's stream, or our own if the caller gave NULL
  bool own_stream = false;
  cudaEvent_t ev = nullptr;
  cudaEvent_t step_ev[2] = {nullptr, nullptr};
  float last_step_ms = 0.0f;
  uint8_t* arena = nullptr;
  size_t arena_bytes = 0;

  std::vector<LayerBufs> layers;
  uint16_t *E = nullptr, *g_final = nullptr;
  std::vector<uint16_t*> Tt;
  uint16_t *kcache = nullptr, *vcache = nullptr;
  int32_t* block_table = nullptr;
  int32_t* pos = nullptr;
  float2* rope = nullptr;
  float* h = nullptr;
  // fp16 activations in the GEMV kernels' pair order, by sequence id
  uint16_t *xh = nullptr, *ah = nullptr, *acth = nullptr, *uh = nullptr;
  float* q = nullptr;
  float* attn_part = nullptr;
  int32_t* attn_cnt = nullptr;
  float* head_part = nullptr;
  int32_t* head_cnt = nullptr;
  // tensor-core GEMM (contexts whose max_batch exceeds the GEMV's staging
  // limit): weight tensor maps, split-K partials, per-tile counters
  bool tc = false;
  std::vector<CUtensorMap> tm_layer;  // [layer][qkv, o, gate/up, down]
  std::vector<CUtensorMap> tm_T;
  CUtensorMap tm_E;
  float* tc_part = nullptr;
  int32_t* tc_cnt = nullptr;
  float* hdbg = nullptr;
  StepLists* lists = nullptr;
  StepDesc* desc_dev = nullptr;
  StepOut* out_dev = nullptr;
  int32_t* dbg_flag = nullptr;
  float* gamma_dev = nullptr;
  uint8_t* staging = nullptr;
  size_t staging_bytes = 0;
  size_t zero_begin = 0, zero_end = 0;  // arena range cleared at create (counters)

  StepDesc* desc_host = nullptr;
  StepOut* out_host = nullptr;

  // host bookkeeping
  std::vector<int32_t> free_blocks;  // descending; back() is the lowest free id
  std::vector<std::vector<int32_t>> seq_blocks;
  std::vector<int32_t> seq_pos;
  int batch = 0;
  std::vector<char> layer_loaded;
  bool shared_loaded = false;
  std::vector<float> gamma;
  int exit_enabled = 1, use_graph = 1, debug = 0;
  int criterion = EE_EXIT_MAXPROB;
  std::vector<float> prefill_tau;        // sequence-level prefill exit thresholds (empty: off)
  std::vector<int32_t> prefill_exit;     // per sequence: layer its prompt left at (n_layers - 1: none)
  int token_source = EE_TOKEN_FINAL_HEAD;
  // input states of the checkpoint layers (similarity criterion): checkpoint c
  // uses buffer c % 2, so that the save for checkpoint c + 1 (by the down
  // projection of checkpoint layer c when the two are adjacent) does not
  // overwrite it before its decision
  float* hin = nullptr;
  float* sts_score = nullptr;
  int32_t* sts_cnt = nullptr;
  bool cuda_broken = false;
  std::map<std::pair<int, int>, cudaGraphExec_t> graphs;
  // profiling: events around each launch of a step, and the GEMV launches'
  // own start/end stamps ([0, kProfMax) starts, [kProfMax, 2 kProfMax) ends)
  int profile = 0;
  std::vector<cudaEvent_t> prof_ev;
  struct ProfTag {
    int kind, layer, lists;
  };
  std::vector<ProfTag> prof_tag;  // per launch of the last step
  std::vector<float> prof_ms, prof_kernel_ms;
  unsigned long long* prof_stamp = nullptr;
  int launches[2] = {0, 0};                   // kernels per step without / with heads
  std::string err;
};

namespace {

ee_status fail(ee_ctx* c, ee_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  if (c) {
    c->err = buf;
    if (s == EE_ERR_CUDA) c->cuda_broken = true;
  }
  return s;
}

#define EE_CUDA(ctx, call)                                                                       \
  do {                                                                                           \
    cudaError_t e_ = (call);                                                                     \
    if (e_ != cudaSuccess)                                                                       \
      return fail((ctx), EE_ERR_CUDA, "%s failed: %s (%s:%d)", #call, cudaGetErrorString(e_),   \
                  __FILE__, __LINE__);                                                           \
  } while (0)

const char* validate_config(const ee_config* c) {
  if (!c) return "config is NULL";
  if (c->n_layers < 1 || c->d_model < 32 || c->n_heads < 1 || c->n_kv_heads < 1 ||
      c->head_dim < 2 || c->ffn_dim < 32 || c->vocab < 2)
    return "shape fields must be positive (d_model, ffn_dim >= 32, vocab >= 2)";
  if (c->d_model % 32 || c->ffn_dim % 32 || (c->n_heads * c->head_dim) % 32)
    return "d_model, ffn_dim and n_heads*head_dim must be multiples of 32";
  if (c->n_heads % c->n_kv_heads) return "n_heads must be a multiple of n_kv_heads";
  if (c->head_dim != 64 && c->head_dim != 128) return "head_dim must be 64 or 128";
  const int G = c->n_heads / c->n_kv_heads;
  if (G != 1 && G != 2 && G != 4 && G != 8) return "n_heads / n_kv_heads must be 1, 2, 4 or 8";
  if (c->vocab % 2) return "vocab must be even";
  if (c->quant_group != EE_QUANT_GROUP) return "quant_group must be 128";
  if (c->kv_block != EE_KV_BLOCK) return "kv_block must be 16";
  if (c->max_batch < 1 || c->max_batch > EE_MAX_BATCH) return "max_batch must be in [1, 64]";
  if (c->max_seq_len < 2) return "max_seq_len must be >= 2";
  if (!linear_shape_ok(c->d_model) || !linear_shape_ok(c->n_heads * c->head_dim) ||
      !linear_shape_ok(c->ffn_dim))
    return "a projection width is not supported by the GEMV stage geometry";
  if (attention_nsplit(c->max_seq_len, c->head_dim) > attention_max_split())
    return "max_seq_len too large for the attention kernel";
  if (!(c->rms_eps > 0.0f) || !(c->rope_theta > 0.0f)) return "rms_eps and rope_theta must be > 0";
  if (c->n_checkpoints < 0 || c->n_checkpoints > EE_MAX_CHECKPOINTS) return "n_checkpoints out of range";
  if (c->n_checkpoints > 0 && !c->checkpoint_layers) return "checkpoint_layers is NULL";
  for (int i = 0; i < c->n_checkpoints; ++i) {
    const int l = c->checkpoint_layers[i];
    if (l < 0 || l > c->n_layers - 2) return "checkpoint layer out of [0, n_layers-2]";
    if (i > 0 && l <= c->checkpoint_layers[i - 1]) return "checkpoint layers must be strictly ascending";
  }
  return nullptr;
}

// Lays the arena out (base == null: sizing only).
size_t carve(ee_ctx* c, const ee_config& cfg, uint8_t* base) {
  const Dims m = dims_of(cfg);
  Carver cv(base);
  std::vector<LayerBufs> layers(m.L);
  for (int j = 0; j < m.L; ++j) {
    LayerBufs& b = layers[j];
    b.wqkv = cv.take<uint16_t>((size_t)m.nqkv * m.d);
    b.wo = cv.take<uint16_t>((size_t)m.d * m.dq);
    b.wgu = cv.take<uint16_t>((size_t)2 * m.F * m.d);
    b.wd = cv.take<uint16_t>((size_t)m.d * m.F);
    b.g_attn = cv.take<uint16_t>(m.d);
    b.g_ffn = cv.take<uint16_t>(m.d);
    b.qkv.q = cv.take<uint8_t>((size_t)m.nqkv * m.d / 2);
    b.qkv.s = cv.take<uint16_t>((size_t)m.nqkv * sstride_of(m.d));
    b.o.q = cv.take<uint8_t>((size_t)m.d * m.dq / 2);
    b.o.s = cv.take<uint16_t>((size_t)m.d * sstride_of(m.dq));
    b.gu.q = cv.take<uint8_t>((size_t)2 * m.F * m.d / 2);
    b.gu.s = cv.take<uint16_t>((size_t)2 * m.F * sstride_of(m.d));
    b.d.q = cv.take<uint8_t>((size_t)m.d * m.F / 2);
    b.d.s = cv.take<uint16_t>((size_t)m.d * sstride_of(m.F));
    const bool tcl = ctx_needs_tc(m);
    b.qkv.qt = tcl ? cv.take<uint8_t>(int4_tc_layout_bytes(m.nqkv, m.d)) : nullptr;
    b.o.qt = tcl ? cv.take<uint8_t>(int4_tc_layout_bytes(m.d, m.dq)) : nullptr;
    b.gu.qt = tcl ? cv.take<uint8_t>(int4_tc_layout_bytes(2 * m.F, m.d)) : nullptr;
    b.d.qt = tcl ? cv.take<uint8_t>(int4_tc_layout_bytes(m.d, m.F)) : nullptr;
  }
  uint16_t* E = cv.take<uint16_t>((size_t)m.V * m.d);
  uint16_t* gf = cv.take<uint16_t>(m.d);
  std::vector<uint16_t*> Tt(m.nck);
  for (int i = 0; i < m.nck; ++i) Tt[i] = cv.take<uint16_t>((size_t)m.d * m.d);
  uint16_t* kc = cv.take<uint16_t>(m.kv_layer_elems * m.L);
  uint16_t* vc = cv.take<uint16_t>(m.kv_layer_elems * m.L);
  int32_t* bt = cv.take<int32_t>((size_t)m.maxb * m.bps);
  int32_t* pos = cv.take<int32_t>(EE_MAX_BATCH);
  float2* rope = cv.take<float2>((size_t)m.maxs * (m.hd / 2));
  float* h = cv.take<float>((size_t)EE_MAX_BATCH * m.d);
  uint16_t* xh = cv.take<uint16_t>((size_t)EE_MAX_BATCH * m.d);
  uint16_t* ah = cv.take<uint16_t>((size_t)EE_MAX_BATCH * m.dq);
  uint16_t* acth = cv.take<uint16_t>((size_t)EE_MAX_BATCH * m.F);
  uint16_t* uh = cv.take<uint16_t>((size_t)EE_MAX_BATCH * m.d);
  float* q = cv.take<float>((size_t)EE_MAX_BATCH * m.dq);
  float* apart = cv.take<float>(
      attention_part_floats(m.maxb, m.hq, m.hkv, m.hd, attention_nsplit(m.maxs, m.hd)));
  float* hpart = cv.take<float>((size_t)kHeadGridMax * EE_MAX_BATCH * 4);
  float* hdbg = cv.take<float>((size_t)m.L * EE_MAX_BATCH * m.d);
  float* hin = cv.take<float>((size_t)2 * EE_MAX_BATCH * m.d);
  float* stss = cv.take<float>(EE_MAX_BATCH);
  const bool tc = ctx_needs_tc(m);
  float* tcpart = tc ? cv.take<float>(gemm_tc_part_floats(2 * kTcMaxUnits)) : nullptr;  // per list
  StepDesc* desc = cv.take<StepDesc>(1);
  StepOut* out = cv.take<StepOut>(1);
  float* gam = cv.take<float>(EE_MAX_CHECKPOINTS);
  unsigned long long* pstamp = cv.take<unsigned long long>(2 * (size_t)kProfMax);  // reset per profiled step
  const size_t zb = align_up(cv.off, kAlign);
  StepLists* lists = cv.take<StepLists>(1);
  int32_t* acnt = cv.take<int32_t>((size_t)EE_MAX_BATCH * m.hkv);
  int32_t* hcnt = cv.take<int32_t>(64);
  int32_t* dflag = cv.take<int32_t>(1);
  int32_t* stsc = cv.take<int32_t>(1);
  int32_t* tccnt = tc ? cv.take<int32_t>(2 * kTcMaxTiles) : nullptr;  // per list
  const size_t ze = align_up(cv.off, kAlign);
  const size_t stg = 2 * (size_t)std::max({(size_t)m.F * m.d, (size_t)m.dq * m.d, (size_t)m.d * m.d,
                                          (size_t)m.dk * m.d});
  uint8_t* staging = cv.take<uint8_t>(stg);
  const size_t total = align_up(cv.off, kAlign);
  if (c) {
    c->layers = layers;
    c->E = E;
    c->g_final = gf;
    c->Tt = Tt;
    c->kcache = kc;
    c->vcache = vc;
    c->block_table = bt;
    c->pos = pos;
    c->rope = rope;
    c->h = h;
    c->xh = xh;
    c->ah = ah;
    c->acth = acth;
    c->uh = uh;
    c->q = q;
    c->attn_part = apart;
    c->head_part = hpart;
    c->hdbg = hdbg;
    c->hin = hin;
    c->sts_score = stss;
    c->sts_cnt = stsc;
    c->desc_dev = desc;
    c->out_dev = out;
    c->gamma_dev = gam;
    c->prof_stamp = pstamp;
    c->lists = lists;
    c->attn_cnt = acnt;
    c->head_cnt = hcnt;
    c->tc = tc;
    c->tc_part = tcpart;
    c->tc_cnt = tccnt;
    c->dbg_flag = dflag;
    c->staging = staging;
    c->staging_bytes = stg;
    c->zero_begin = zb;
    c->zero_end = ze;
  }
  return total;
}

struct DeviceGuard {
  int prev = -1;
  explicit DeviceGuard(int dev) {
    cudaGetDevice(&prev);
    if (prev != dev) cudaSetDevice(dev);
  }
  ~DeviceGuard() {
    int cur;
    if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
  }
};

// Orders our stream after everything already queued on the caller's stream.
ee_status join_user_stream(ee_ctx* c) {
  if (!c->own_stream) return EE_OK;
  EE_CUDA(c, cudaEventRecord(c->ev, c->user_stream));
  EE_CUDA(c, cudaStreamWaitEvent(c->st, c->ev, 0));
  return EE_OK;
}

// Launch bookkeeping of one step: counts launches and, in profile mode,
// records an event before the first and after every launch.
struct LaunchLog {
  ee_ctx* c;
  bool prof;
  int n = 0;
  LaunchLog(ee_ctx* cc, bool p) : c(cc), prof(p) {
    if (prof) c->prof_tag.clear();
  }
  ee_status before() {
    if (!prof) return EE_OK;
    if (n == 0) {
      if ((int)c->prof_ev.size() < 1 && add_event() != EE_OK) return EE_ERR_CUDA;
      EE_CUDA(c, cudaEventRecord(c->prof_ev[0], c->st));
    }
    return EE_OK;
  }
  ee_status after(int kind, int layer, int lists = EE_LISTS_BOTH) {
    ++n;
    if (!prof) return EE_OK;
    while ((int)c->prof_ev.size() < n + 1)
      if (add_event() != EE_OK) return EE_ERR_CUDA;
    EE_CUDA(c, cudaEventRecord(c->prof_ev[n], c->st));
    c->prof_tag.push_back(ee_ctx::ProfTag{kind, layer, lists});
    return EE_OK;
  }
  ee_status add_event() {
    cudaEvent_t e;
    EE_CUDA(c, cudaEventCreate(&e));
    c->prof_ev.push_back(e);
    return EE_OK;
  }
};

#define EE_LAUNCH_L(log, kind, layer, lists, call) \
  do {                                             \
    ee_status s_ = (log).before();                 \
    if (s_ != EE_OK) return s_;                    \
    EE_CUDA(c, (call));                            \
    s_ = (log).after((kind), (layer), (lists));    \
    if (s_ != EE_OK) return s_;                    \
  } while (0)
#define EE_LAUNCH(log, kind, layer, call) EE_LAUNCH_L(log, kind, layer, EE_LISTS_BOTH, call)

// ---------------------------------------------------------------- step enqueue
ee_status enqueue_step(ee_ctx* c, int B, bool heads, bool prof) {
  const Dims& m = c->m;
  cudaStream_t st = c->st;
  LaunchLog log(c, prof);
  if (prof) {
    EE_CUDA(c, cudaMemsetAsync(c->prof_stamp, 0xFF, kProfMax * sizeof(unsigned long long), st));
    EE_CUDA(c, cudaMemsetAsync(c->prof_stamp + kProfMax, 0, kProfMax * sizeof(unsigned long long), st));
  }
  EE_CUDA(c, cudaMemcpyAsync(c->desc_dev, c->desc_host, sizeof(StepDesc), cudaMemcpyHostToDevice, st));

  BeginParams bp = {};
  bp.desc = c->desc_dev;
  bp.lists = c->lists;
  bp.out = c->out_dev;
  bp.embed = c->E;
  bp.d = m.d;
  bp.h = c->h;
  bp.h_stride = m.d;
  bp.pos = c->pos;
  bp.block_table = c->block_table;
  bp.bt_stride = m.bps;
  bp.n_layers = m.L;
  bp.n_ckpt = m.nck;
  bp.dbg_flag = c->dbg_flag;
  // similarity criterion: each checkpoint layer's input state is kept (for
  // layer 0 by the step start, otherwise by the previous layer's down projection)
  const bool sts = heads && (c->criterion == EE_EXIT_STS || c->criterion == EE_EXIT_STS_BATCH);
  // exit-head tokens: an exited sequence's token comes from its exit head; in
  // the last layer only its QKV (the K/V write) runs, and the final head
  // serves the sequences that never exited
  const bool head_tok = heads && !sts && c->token_source == EE_TOKEN_EXIT_HEAD;
  auto ckpt_index = [&](int j) {
    const auto it = std::find(c->ckpts.begin(), c->ckpts.end(), j);
    return it == c->ckpts.end() ? -1 : (int)(it - c->ckpts.begin());
  };
  auto hin_of = [&](int ci) { return c->hin + (size_t)(ci % 2) * EE_MAX_BATCH * m.d; };
  bp.hsave = sts && ckpt_index(0) >= 0 ? hin_of(0) : nullptr;
  EE_LAUNCH(log, EE_K_BEGIN, -1, launch_step_begin(bp, B, st));

  int32_t* err = &c->out_dev->err;
  const int nsplit = attention_nsplit(m.maxs, m.hd);

  NormParams np = {};
  np.h = c->h;
  np.h_stride = m.d;
  np.d = m.d;
  np.eps = c->cfg.rms_eps;
  np.x_stride = m.d;

  LinearParams base = {};
  base.err = err;
  base.block_table = c->block_table;
  base.bt_stride = m.bps;
  base.pos = c->pos;
  base.rope = c->rope;
  base.n_heads = m.hq;
  base.n_kv_heads = m.hkv;
  base.head_dim = m.hd;
  base.h = c->h;
  base.h_stride = m.d;
  base.dbg_flag = c->dbg_flag;
  base.head_part = c->head_part;
  base.gamma = c->gamma_dev;

  // With at most a few sequences the GEMV stages its activations in shared
  // memory and applies each RMSNorm itself; otherwise a norm kernel runs first.
  const bool use_tc = c->tc && batch_uses_tc(m, B);
  const bool fuse_norm = !use_tc && linear_stages_x(B, m.d);
  auto norm_on_stage = [&](LinearParams& lp, const uint16_t* g) {
    lp.norm_h = c->h;
    lp.norm_stride = m.d;
    lp.norm_g = g;
    lp.norm_eps = c->cfg.rms_eps;
  };
  bool lists_just_written = true;  // by the step-begin kernel
  // A projection or head: the GEMV, or for larger batches the tensor-core
  // GEMM (one launch per non-empty-capable sub-batch list).
  auto project = [&](int kind, int layer, const LinearParams& lp, const CUtensorMap* map, int grid) -> ee_status {
    if (use_tc && map && gemm_tc_shape_ok(lp.K)) {
      const TcPlan pl = gemm_tc_plan(lp.N, lp.K, c->num_sms, kTcMaxUnits);
      if (pl.ntiles * pl.ksplit <= kTcMaxUnits && pl.ntiles <= kTcMaxTiles) {
        TcParams tp;
        memset(&tp, 0, sizeof(tp));
        tp.amap = *map;
        tp.lp = lp;
        tp.ntiles = pl.ntiles;
        tp.ksplit = pl.ksplit;
        tp.nks = pl.nks;
        tp.nk = pl.nk;
        tp.part = c->tc_part;
        tp.q4t = lp.wq4t;
        tp.tile_cnt = c->tc_cnt;
        // the exit list is empty until a head has run (no units for it then)
        const bool exit_rows = heads && m.nck > 0 && layer > c->ckpts[0];
        tp.modes = lp.wq && lp.wq4t && exit_rows ? 2 : 1;
        const bool on = prof && log.n < kProfMax;  // this launch's own start/end stamps (profiled steps)
        tp.lp.stamp_start = on ? c->prof_stamp + log.n : nullptr;
        tp.lp.stamp_end = on ? c->prof_stamp + kProfMax + log.n : nullptr;
        if (lp.w)
          EE_LAUNCH_L(log, kind, layer, tp.modes == 2 ? EE_LISTS_BOTH : EE_LISTS_FULL, launch_gemm_tc(tp, c->pdl, st));
        return EE_OK;
      }
    }
    LinearParams lq = lp;
    if (prof && log.n < kProfMax) {  // this launch's stamps
      lq.stamp_start = c->prof_stamp + log.n;
      lq.stamp_end = c->prof_stamp + kProfMax + log.n;
    }
    EE_LAUNCH(log, kind, layer, launch_linear(lq, grid, c->pdl, st));
    return EE_OK;
  };
#define EE_PROJECT(kind, layer, lp, map, grid)                  \
  do {                                                          \
    const ee_status ps_ = project((kind), (layer), (lp), (map), (grid)); \
    if (ps_ != EE_OK) return ps_;                               \
  } while (0)

  for (int j = 0; j < m.L; ++j) {
    const LayerBufs& w = c->layers[j];
    // attention RMSNorm of every participating sequence
    if (!fuse_norm) {
      np.list = c->lists->part;
      np.g = w.g_attn;
      np.xh = c->xh;
      EE_LAUNCH(log, EE_K_NORM, j, launch_rmsnorm(np, B, c->pdl, st));
    }
    // QKV projection + RoPE + K/V write into the shared paged cache
    LinearParams pq = base;
    pq.N = m.nqkv;
    pq.K = m.d;
    pq.w = w.wqkv;
    pq.wq = w.qkv.q;
    pq.ws = w.qkv.s;
    pq.wq4t = w.qkv.qt;
    pq.sstride = sstride_of(m.d);
    pq.list_full = c->lists->full;
    pq.list_exit = c->lists->exitl;
    pq.xh = c->xh;
    pq.x_stride = m.d;
    if (fuse_norm) {
      norm_on_stage(pq, w.g_attn);
      pq.lists_after_wait = lists_just_written ? 1 : 0;
    }
    pq.epi = EPI_QKV;
    pq.q_out = c->q;
    pq.kc = c->kcache + (size_t)j * m.kv_layer_elems;
    pq.vc = c->vcache + (size_t)j * m.kv_layer_elems;
    pq.max_rows = B;
    // decode attention
    AttnParams ap = {};
    const bool dead_exit = head_tok && j == m.L - 1;  // exited rows' attention, O and FFN are not needed
    ap.list = dead_exit ? c->lists->full : c->lists->part;
    ap.n_heads = m.hq;
    ap.n_kv_heads = m.hkv;
    ap.head_dim = m.hd;
    ap.q = c->q;
    ap.q_stride = m.dq;
    ap.kc = pq.kc;
    ap.vc = pq.vc;
    ap.block_table = c->block_table;
    ap.bt_stride = m.bps;
    ap.pos = c->pos;
    ap.nsplit = nsplit;
    ap.bpc = attention_blocks_per_cta(m.hd);
    ap.part = c->attn_part;
    ap.counters = c->attn_cnt;
    ap.oh = c->ah;
    ap.o_stride = m.dq;
    ap.err = err;
    // O projection + residual
    LinearParams po = base;
    po.N = m.d;
    po.K = m.dq;
    po.w = w.wo;
    po.wq = dead_exit ? nullptr : w.o.q;
    po.ws = dead_exit ? nullptr : w.o.s;
    po.wq4t = w.o.qt;
    po.sstride = sstride_of(m.dq);
    po.list_full = c->lists->full;
    po.list_exit = c->lists->exitl;
    po.xh = c->ah;
    po.x_stride = m.dq;
    po.epi = EPI_RESID;
    po.max_rows = B;
    // gate/up + SwiGLU
    LinearParams pg = base;
    pg.N = 2 * m.F;
    pg.K = m.d;
    pg.w = w.wgu;
    pg.wq = dead_exit ? nullptr : w.gu.q;
    pg.ws = dead_exit ? nullptr : w.gu.s;
    pg.wq4t = w.gu.qt;
    pg.sstride = sstride_of(m.d);
    pg.list_full = c->lists->full;
    pg.list_exit = c->lists->exitl;
    pg.xh = c->xh;
    pg.x_stride = m.d;
    if (fuse_norm) norm_on_stage(pg, w.g_ffn);
    pg.epi = EPI_SWIGLU;
    pg.xh_out = c->acth;
    pg.xo_stride = m.F;
    pg.max_rows = B;
    // down projection + residual (+ per-layer copy in debug mode)
    LinearParams pd = base;
    pd.N = m.d;
    pd.K = m.F;
    pd.w = w.wd;
    pd.wq = dead_exit ? nullptr : w.d.q;
    pd.ws = dead_exit ? nullptr : w.d.s;
    pd.wq4t = w.d.qt;
    pd.sstride = sstride_of(m.F);
    pd.list_full = c->lists->full;
    pd.list_exit = c->lists->exitl;
    pd.xh = c->acth;
    pd.x_stride = m.F;
    pd.epi = EPI_RESID;
    pd.hdbg = c->hdbg + (size_t)j * EE_MAX_BATCH * m.d;
    pd.hsave = sts && ckpt_index(j + 1) >= 0 ? hin_of(ckpt_index(j + 1)) : nullptr;
    pd.max_rows = B;

    EE_PROJECT(EE_K_QKV, j, pq, c->tc ? &c->tm_layer[4 * j + 0] : nullptr, linear_grid(pq.N, c->num_sms));
    lists_just_written = false;
    EE_LAUNCH(log, EE_K_ATTN, j, launch_attention(ap, B, c->pdl, st));
    EE_PROJECT(EE_K_O, j, po, c->tc ? &c->tm_layer[4 * j + 1] : nullptr, linear_grid(po.N, c->num_sms));
    // FFN RMSNorm
    if (!fuse_norm) {
      np.g = w.g_ffn;
      EE_LAUNCH(log, EE_K_NORM, j, launch_rmsnorm(np, B, c->pdl, st));
    }
    EE_PROJECT(EE_K_GATEUP, j, pg, c->tc ? &c->tm_layer[4 * j + 2] : nullptr, linear_grid(pg.N, c->num_sms));
    EE_PROJECT(EE_K_DOWN, j, pd, c->tc ? &c->tm_layer[4 * j + 3] : nullptr, linear_grid(pd.N, c->num_sms));
    LinearParams p;

    const auto ck = std::find(c->ckpts.begin(), c->ckpts.end(), j);
    if (sts && ck != c->ckpts.end()) {
      // cos(layer input, layer output) against the threshold, lists compacted
      StsParams sp = {};
      sp.lists = c->lists;
      sp.h = c->h;
      sp.h_in = hin_of((int)(ck - c->ckpts.begin()));
      sp.d = m.d;
      sp.h_stride = m.d;
      sp.gamma = c->gamma_dev;
      sp.ckpt_index = (int)(ck - c->ckpts.begin());
      sp.ckpt_layer = j;
      sp.conf_out = c->out_dev->conf;
      sp.exit_layer = c->out_dev->exit_layer;
      sp.score = c->sts_score;
      sp.counter = c->sts_cnt;
      sp.batch_min = c->criterion == EE_EXIT_STS_BATCH;
      EE_LAUNCH(log, EE_K_EXIT_STS, j, launch_sts(sp, B, c->pdl, st));
      lists_just_written = true;
    } else if (heads && ck != c->ckpts.end()) {
      const int ci = (int)(ck - c->ckpts.begin());
      // u = RMSNorm_final(h) T_c for the sequences still on the backbone
      if (!fuse_norm) {
        NormParams fp = np;
        fp.list = c->lists->full;
        fp.g = c->g_final;
        EE_LAUNCH(log, EE_K_HEAD_NORM, j, launch_rmsnorm(fp, B, c->pdl, st));
      }
      p = base;
      p.N = m.d;
      p.K = m.d;
      p.w = c->Tt[ci];
      p.list_full = c->lists->full;
      p.list_exit = nullptr;
      p.xh = c->xh;
      p.x_stride = m.d;
      if (fuse_norm) norm_on_stage(p, c->g_final);
      p.epi = EPI_X;
      p.xh_out = c->uh;
      p.xo_stride = m.d;
      p.max_rows = B;
      EE_PROJECT(EE_K_HEAD_T, j, p, c->tc ? &c->tm_T[ci] : nullptr, linear_grid(p.N, c->num_sms));
      // z = u E^T, conf = max softmax, exit if conf > gamma_c, compact the lists
      p = base;
      p.N = m.V;
      p.K = m.d;
      p.w = c->E;
      p.list_full = c->lists->full;
      p.list_exit = c->lists->exitl;  // merged into the new exit list; no int4 work (wq is null)
      p.xh = c->uh;
      p.x_stride = m.d;
      p.epi = EPI_HEAD;
      p.head_mode = HEAD_CHECKPOINT;
      p.head_counter = c->head_cnt + 1 + ci;
      p.conf_out = c->out_dev->conf;
      p.lists = c->lists;
      p.exit_layer = c->out_dev->exit_layer;
      p.argmax_out = head_tok ? c->out_dev->next_token : nullptr;
      p.ckpt_index = ci;
      p.ckpt_layer = j;
      p.max_rows = B;
      EE_PROJECT(EE_K_HEAD_E, j, p, c->tc ? &c->tm_E : nullptr,
                 std::min(linear_grid(p.N, c->num_sms), kHeadGridMax));
      lists_just_written = true;  // compacted by the exit head
    }
  }
  // final LM head: argmax of RMSNorm_final(h) E^T
  int32_t* fin_list = head_tok ? c->lists->full : c->lists->fin;
  if (!fuse_norm) {
    NormParams fp = np;
    fp.list = fin_list;
    fp.g = c->g_final;
    EE_LAUNCH(log, EE_K_FINAL_NORM, -1, launch_rmsnorm(fp, B, c->pdl, st));
  }
  LinearParams p = base;
  p.N = m.V;
  p.K = m.d;
  p.w = c->E;
  p.list_full = fin_list;
  p.list_exit = nullptr;
  p.xh = c->xh;
  p.x_stride = m.d;
  if (fuse_norm) norm_on_stage(p, c->g_final);
  p.epi = EPI_HEAD;
  p.head_mode = HEAD_FINAL;
  p.head_counter = c->head_cnt;
  p.argmax_out = c->out_dev->next_token;
  p.max_rows = B;
  EE_PROJECT(EE_K_FINAL_HEAD, -1, p, c->tc ? &c->tm_E : nullptr,
             std::min(linear_grid(p.N, c->num_sms), kHeadGridMax));
#undef EE_PROJECT
  EE_CUDA(c, cudaMemcpyAsync(c->out_host, c->out_dev, step_d2h_bytes(B), cudaMemcpyDeviceToHost, st));
  c->launches[heads ? 1 : 0] = log.n;
  return EE_OK;
}

// One step in profile mode: eager launches with an event pair around each.
ee_status run_step_profiled(ee_ctx* c, int B, bool heads) {
  const ee_status s = enqueue_step(c, B, heads, true);
  if (s != EE_OK) return s;
  EE_CUDA(c, cudaStreamSynchronize(c->st));
  c->prof_ms.assign(c->prof_tag.size(), 0.0f);
  for (size_t i = 0; i < c->prof_tag.size(); ++i)
    EE_CUDA(c, cudaEventElapsedTime(&c->prof_ms[i], c->prof_ev[i], c->prof_ev[i + 1]));
  // the GEMV launches' own durations: first CTA start to last CTA end
  const size_t nst = std::min(c->prof_tag.size(), (size_t)kProfMax);
  std::vector<unsigned long long> t0(nst), t1(nst);
  if (nst > 0) {
    EE_CUDA(c, cudaMemcpy(t0.data(), c->prof_stamp, nst * 8, cudaMemcpyDeviceToHost));
    EE_CUDA(c, cudaMemcpy(t1.data(), c->prof_stamp + kProfMax, nst * 8, cudaMemcpyDeviceToHost));
  }
  c->prof_kernel_ms.assign(c->prof_tag.size(), 0.0f);
  for (size_t i = 0; i < nst; ++i)
    if (t1[i] > t0[i]) c->prof_kernel_ms[i] = (float)((double)(t1[i] - t0[i]) * 1e-6);
  c->last_step_ms = 0.0f;
  for (float v : c->prof_ms) c->last_step_ms += v;
  return EE_OK;
}

// One step replayed from the graph of (B, heads) -- captured on first use --
// or launched eagerly, timed by an event pair on the context's stream.
ee_status run_step_timed(ee_ctx* c, int B, bool heads) {
  EE_CUDA(c, cudaEventRecord(c->step_ev[0], c->st));
  if (c->use_graph) {
    const auto key = std::make_pair(B, heads ? 1 + c->criterion + 3 * c->token_source : 0);
    auto it = c->graphs.find(key);
    if (it == c->graphs.end()) {
      cudaGraph_t g = nullptr;
      EE_CUDA(c, cudaStreamBeginCapture(c->st, cudaStreamCaptureModeThreadLocal));
      const ee_status s = enqueue_step(c, B, heads, false);
      const cudaError_t e = cudaStreamEndCapture(c->st, &g);
      if (s != EE_OK) {
        if (g) cudaGraphDestroy(g);
        return s;
      }
      if (e != cudaSuccess) return fail(c, EE_ERR_CUDA, "graph capture failed: %s", cudaGetErrorString(e));
      cudaGraphExec_t ex = nullptr;
      const cudaError_t ei = cudaGraphInstantiate(&ex, g, 0);
      cudaGraphDestroy(g);
      if (ei != cudaSuccess)
        return fail(c, EE_ERR_CUDA, "graph instantiate failed: %s", cudaGetErrorString(ei));
      it = c->graphs.emplace(key, ex).first;
    }
    EE_CUDA(c, cudaGraphLaunch(it->second, c->st));
  } else {
    const ee_status s = enqueue_step(c, B, heads, false);
    if (s != EE_OK) return s;
  }
  EE_CUDA(c, cudaEventRecord(c->step_ev[1], c->st));
  EE_CUDA(c, cudaStreamSynchronize(c->st));
  EE_CUDA(c, cudaEventElapsedTime(&c->last_step_ms, c->step_ev[0], c->step_ev[1]));
  return EE_OK;
}

ee_status run_step(ee_ctx* c, int B, bool heads) {
  const ee_status s = c->profile ? run_step_profiled(c, B, heads) : run_step_timed(c, B, heads);
  if (s != EE_OK) return s;
  if (c->out_host->err != 0)
    return fail(c, EE_ERR_DEVICE_TIMEOUT,
                "device error code %d (1 = stage fill, 2 = stage drain, 3 = exit drain; >= 10: a checked "
                "access was refused) info %d %d",
                c->out_host->err, c->out_host->pad[0], c->out_host->pad[1]);
  return EE_OK;
}

void reset_blocks(ee_ctx* c) {
  c->free_blocks.resize(c->m.nblocks);
  for (int i = 0; i < c->m.nblocks; ++i) c->free_blocks[i] = c->m.nblocks - 1 - i;
  c->seq_blocks.assign(c->m.maxb, {});
  c->seq_pos.assign(c->m.maxb, 0);
  c->batch = 0;
}

int32_t alloc_block(ee_ctx* c) {
  if (c->free_blocks.empty()) return -1;
  const int32_t b = c->free_blocks.back();
  c->free_blocks.pop_back();
  return b;
}

ee_status fill_sentinel(ee_ctx* c) {
  const size_t n = c->m.kv_layer_elems * c->m.L;
  EE_CUDA(c, launch_fill_u16(c->kcache, 0xFFFF, (int64_t)n, c->st));
  EE_CUDA(c, launch_fill_u16(c->vcache, 0xFFFF, (int64_t)n, c->st));
  return EE_OK;
}

ee_status check_ready(ee_ctx* c) {
  if (c->cuda_broken) return fail(c, EE_ERR_CUDA, "context unusable after an earlier CUDA error");
  for (int j = 0; j < c->m.L; ++j)
    if (!c->layer_loaded[j]) return fail(c, EE_ERR_STATE, "layer %d weights not loaded", j);
  if (!c->shared_loaded) return fail(c, EE_ERR_STATE, "shared weights (E, g_final, T) not loaded");
  return EE_OK;
}

// copy a host/device matrix [rows, cols] bf16 into its place in a fused block
ee_status place_bf16(ee_ctx* c, const uint16_t* src, int rows, int cols, uint16_t* dst, int row0,
                     int map, int param) {
  const size_t bytes = (size_t)rows * cols * 2;
  if (bytes > c->staging_bytes) return fail(c, EE_ERR_INVALID_ARG, "matrix larger than staging");
  EE_CUDA(c, cudaMemcpyAsync(c->staging, src, bytes, cudaMemcpyDefault, c->st));
  EE_CUDA(c, launch_copy_rows(dst, (int64_t)cols * 2, row0, c->staging, (int64_t)cols * 2,
                              (int64_t)cols * 2, rows, map, param, c->st));
  return EE_OK;
}

ee_status place_int4(ee_ctx* c, const uint8_t* q, const uint16_t* s, int rows, int cols, Mat4 dst,
                     int row0, int map, int param) {
  const int ng = (int)ceil_div(cols, EE_QUANT_GROUP), ss = sstride_of(cols);
  size_t bytes = (size_t)rows * cols / 2;
  EE_CUDA(c, cudaMemcpyAsync(c->staging, q, bytes, cudaMemcpyDefault, c->st));
  EE_CUDA(c, launch_copy_rows(dst.q, cols / 2, row0, c->staging, cols / 2, cols / 2, rows, map, param, c->st));
  bytes = (size_t)rows * ng * 2;
  EE_CUDA(c, cudaMemcpyAsync(c->staging, s, bytes, cudaMemcpyDefault, c->st));
  EE_CUDA(c, launch_copy_rows(dst.s, (int64_t)ss * 2, row0, c->staging, (int64_t)ng * 2, (int64_t)ng * 2,
                              rows, map, param, c->st));
  return EE_OK;
}

struct MatPlace {
  int block;  // 0 qkv, 1 o, 2 gu, 3 d
  int row0, rows, cols, map, param;
};

MatPlace placement(const Dims& m, int mat) {
  switch (mat) {
    case EE_WQ: return {0, 0, m.dq, m.d, MAP_ROPE_PAIRS, m.hd};
    case EE_WK: return {0, m.dq, m.dk, m.d, MAP_ROPE_PAIRS, m.hd};
    case EE_WV: return {0, m.dq + m.dk, m.dk, m.d, MAP_IDENTITY, 0};
    case EE_WO: return {1, 0, m.d, m.dq, MAP_IDENTITY, 0};
    case EE_WG: return {2, 0, m.F, m.d, MAP_INTERLEAVE, 0};
    case EE_WU: return {2, 0, m.F, m.d, MAP_INTERLEAVE, 1};
    default: return {3, 0, m.d, m.F, MAP_IDENTITY, 0};
  }
}

int64_t device_row(const MatPlace& pl, int64_t r) {
  if (pl.map == MAP_ROPE_PAIRS) {
    const int64_t head = r / pl.param, i = r % pl.param, half = pl.param / 2;
    return pl.row0 + head * pl.param + (i < half ? 2 * i : 2 * (i - half) + 1);
  }
  if (pl.map == MAP_INTERLEAVE) return pl.row0 + 2 * r + pl.param;
  return pl.row0 + r;
}

}  // namespace

// ======================================================================= C ABI
extern "C" {

size_t ee_arena_bytes(const ee_config* cfg) {
  if (validate_config(cfg)) return 0;
  return carve(nullptr, *cfg, nullptr);
}

ee_status ee_create(const ee_config* cfg, void* dev_arena, size_t arena_bytes, void* stream,
                    ee_ctx** out) {
  if (!out) return EE_ERR_INVALID_ARG;
  *out = nullptr;
  if (const char* why = validate_config(cfg)) {
    (void)why;
    return EE_ERR_INVALID_ARG;
  }
  if (!dev_arena || (uintptr_t)dev_arena % kAlign) return EE_ERR_INVALID_ARG;
  const size_t need = carve(nullptr, *cfg, nullptr);
  if (arena_bytes < need) return EE_ERR_OOM_ARENA;

  ee_ctx* c = new ee_ctx();
  c->cfg = *cfg;
  c->ckpts.assign(cfg->checkpoint_layers, cfg->checkpoint_layers + cfg->n_checkpoints);
  c->cfg.checkpoint_layers = c->ckpts.data();
  c->m = dims_of(*cfg);
  c->arena = (uint8_t*)dev_arena;
  c->arena_bytes = arena_bytes;
  c->user_stream = (cudaStream_t)stream;
  c->layer_loaded.assign(c->m.L, 0);
  c->gamma.assign(c->m.nck, INFINITY);
  carve(c, *cfg, c->arena);
  auto bail = [&](ee_status s) {
    ee_destroy(c);
    return s;
  };
  if (cudaGetDevice(&c->dev) != cudaSuccess) return bail(EE_ERR_CUDA);
  if (cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, c->dev) != cudaSuccess)
    return bail(EE_ERR_CUDA);
  if (2 * c->num_sms > kHeadGridMax) c->num_sms = kHeadGridMax / 2;
  {
    // EE_PDL=0 launches the step's kernels without programmatic dependent
    // launch (each waits for the previous one to finish), for comparison.
    const char* e = getenv("EE_PDL");
    c->pdl = !(e && e[0] == '0');
  }
  if (linear_prepare() != cudaSuccess || attention_prepare() != cudaSuccess) return bail(EE_ERR_CUDA);
  if (c->tc) {
    // tensor maps of every bf16 matrix the tensor-core GEMM streams (the
    // arena addresses are fixed; the contents are loaded later)
    if (gemm_tc_prepare() != cudaSuccess) return bail(EE_ERR_CUDA);
    const Dims& m = c->m;
    c->tm_layer.resize((size_t)m.L * 4);
    c->tm_T.resize(m.nck);
    bool ok = encode_weight_map(&c->tm_E, c->E, m.V, m.d);
    for (int j = 0; j < m.L && ok; ++j) {
      const LayerBufs& b = c->layers[j];
      ok = encode_weight_map(&c->tm_layer[4 * j + 0], b.wqkv, m.nqkv, m.d) &&
           encode_weight_map(&c->tm_layer[4 * j + 1], b.wo, m.d, m.dq) &&
           encode_weight_map(&c->tm_layer[4 * j + 2], b.wgu, 2 * m.F, m.d) &&
           encode_weight_map(&c->tm_layer[4 * j + 3], b.wd, m.d, m.F);
    }
    for (int i = 0; i < m.nck && ok; ++i) ok = encode_weight_map(&c->tm_T[i], c->Tt[i], m.d, m.d);
    if (!ok) {
      c->err = "encoding the weight tensor maps failed";
      return bail(EE_ERR_CUDA);
    }
  }
  if (c->user_stream) {
    c->st = c->user_stream;
  } else {
    if (cudaStreamCreateWithFlags(&c->st, cudaStreamNonBlocking) != cudaSuccess) return bail(EE_ERR_CUDA);
    c->own_stream = true;
  }
  if (cudaEventCreateWithFlags(&c->ev, cudaEventDisableTiming) != cudaSuccess) return bail(EE_ERR_CUDA);
  if (cudaEventCreate(&c->step_ev[0]) != cudaSuccess || cudaEventCreate(&c->step_ev[1]) != cudaSuccess)
    return bail(EE_ERR_CUDA);
  if (cudaHostAlloc((void**)&c->desc_host, sizeof(StepDesc), cudaHostAllocDefault) != cudaSuccess ||
      cudaHostAlloc((void**)&c->out_host, sizeof(StepOut), cudaHostAllocDefault) != cudaSuccess)
    return bail(EE_ERR_CUDA);
  memset(c->desc_host, 0, sizeof(StepDesc));
  for (int q = 0; q < EE_MAX_BATCH; ++q) c->desc_host->forced_exit[q] = -1;
  memset(c->out_host, 0, sizeof(StepOut));
  if (join_user_stream(c) != EE_OK) return bail(EE_ERR_CUDA);
  // counters and lists start at zero
  if (cudaMemsetAsync(c->arena + c->zero_begin, 0, c->zero_end - c->zero_begin, c->st) != cudaSuccess)
    return bail(EE_ERR_CUDA);
  // RoPE table: angle = pos * theta^(-2i/hd), in double, stored as float (cos, sin)
  {
    const int half = c->m.hd / 2;
    std::vector<float2> tab((size_t)c->m.maxs * half);
    for (int p = 0; p < c->m.maxs; ++p)
      for (int i = 0; i < half; ++i) {
        const double inv = pow((double)cfg->rope_theta, -2.0 * i / (double)c->m.hd);
        const double a = (double)p * inv;
        tab[(size_t)p * half + i] = make_float2((float)cos(a), (float)sin(a));
      }
    if (cudaMemcpyAsync(c->rope, tab.data(), tab.size() * sizeof(float2), cudaMemcpyHostToDevice, c->st) !=
        cudaSuccess)
      return bail(EE_ERR_CUDA);
    std::vector<float> g(EE_MAX_CHECKPOINTS, INFINITY);
    if (cudaMemcpyAsync(c->gamma_dev, g.data(), g.size() * sizeof(float), cudaMemcpyHostToDevice, c->st) !=
        cudaSuccess)
      return bail(EE_ERR_CUDA);
    if (fill_sentinel(c) != EE_OK) return bail(EE_ERR_CUDA);
    if (cudaStreamSynchronize(c->st) != cudaSuccess) return bail(EE_ERR_CUDA);
  }
  reset_blocks(c);
  *out = c;
  return EE_OK;
}

void ee_destroy(ee_ctx* c) {
  if (!c) return;
  for (auto& kv : c->graphs) cudaGraphExecDestroy(kv.second);
  for (auto e : c->prof_ev) cudaEventDestroy(e);
  if (c->st) cudaStreamSynchronize(c->st);
  if (c->desc_host) cudaFreeHost(c->desc_host);
  if (c->out_host) cudaFreeHost(c->out_host);
  if (c->ev) cudaEventDestroy(c->ev);
  for (auto e : c->step_ev)
    if (e) cudaEventDestroy(e);
  if (c->st && c->own_stream) cudaStreamDestroy(c->st);
  delete c;
}

const char* ee_last_error(const ee_ctx* c) { return c ? c->err.c_str() : "null context"; }

ee_status ee_load_layer(ee_ctx* c, int32_t layer, const ee_layer_weights* lw) {
  if (!c) return EE_ERR_INVALID_ARG;
  if (layer < 0 || layer >= c->m.L) return fail(c, EE_ERR_INVALID_ARG, "layer %d out of range", layer);
  if (!lw || !lw->g_attn || !lw->g_ffn || !lw->wq || !lw->wk || !lw->wv || !lw->wo || !lw->wg ||
      !lw->wu || !lw->wd)
    return fail(c, EE_ERR_INVALID_ARG, "layer %d: a bf16 weight pointer is NULL", layer);
  int given = 0;
  for (int k = 0; k < EE_N_MATS; ++k) {
    if ((lw->q4[k] == nullptr) != (lw->s4[k] == nullptr))
      return fail(c, EE_ERR_INVALID_ARG, "layer %d: q4[%d] and s4[%d] must both be set or both NULL", layer, k, k);
    given += lw->q4[k] != nullptr;
  }
  if (given != 0 && given != EE_N_MATS)
    return fail(c, EE_ERR_INVALID_ARG, "layer %d: give all seven int4 copies or none", layer);
  if (c->cuda_broken) return fail(c, EE_ERR_CUDA, "context unusable after an earlier CUDA error");
  DeviceGuard dg(c->dev);
  if (join_user_stream(c) != EE_OK) return EE_ERR_CUDA;
  const Dims& m = c->m;
  LayerBufs& b = c->layers[layer];
  uint16_t* blocks_bf[4] = {b.wqkv, b.wo, b.wgu, b.wd};
  Mat4 blocks_q[4] = {b.qkv, b.o, b.gu, b.d};
  const uint16_t* srcs[EE_N_MATS] = {lw->wq, lw->wk, lw->wv, lw->wo, lw->wg, lw->wu, lw->wd};
  for (int k = 0; k < EE_N_MATS; ++k) {
    const MatPlace pl = placement(m, k);
    ee_status s = place_bf16(c, srcs[k], pl.rows, pl.cols, blocks_bf[pl.block], pl.row0, pl.map, pl.param);
    if (s != EE_OK) return s;
    if (given) {
      s = place_int4(c, lw->q4[k], lw->s4[k], pl.rows, pl.cols, blocks_q[pl.block], pl.row0, pl.map, pl.param);
      if (s != EE_OK) return s;
    }
  }
  if (!given) {
    // the exit copy: quantise each fused block in its kernel row order
    const int rows[4] = {m.nqkv, m.d, 2 * m.F, m.d};
    const int cols[4] = {m.d, m.dq, m.d, m.F};
    for (int k = 0; k < 4; ++k)
      EE_CUDA(c, launch_quantize_int4(blocks_bf[k], rows[k], cols[k], blocks_q[k].q, blocks_q[k].s,
                                      sstride_of(cols[k]), c->st));
  }
  if (c->tc) {  // the tensor-core GEMM's blocks of the exit copy
    const int rows[4] = {m.nqkv, m.d, 2 * m.F, m.d};
    const int cols[4] = {m.d, m.dq, m.d, m.F};
    for (int k = 0; k < 4; ++k)
      EE_CUDA(c, launch_int4_tc_layout(blocks_q[k].q, blocks_q[k].s, rows[k], cols[k], sstride_of(cols[k]),
                                       blocks_q[k].qt, c->st));
  }
  EE_CUDA(c, cudaMemcpyAsync(b.g_attn, lw->g_attn, (size_t)m.d * 2, cudaMemcpyDefault, c->st));
  EE_CUDA(c, cudaMemcpyAsync(b.g_ffn, lw->g_ffn, (size_t)m.d * 2, cudaMemcpyDefault, c->st));
  EE_CUDA(c, cudaStreamSynchronize(c->st));
  c->layer_loaded[layer] = 1;
  return EE_OK;
}

ee_status ee_load_shared(ee_ctx* c, const ee_shared_weights* sw) {
  if (!c) return EE_ERR_INVALID_ARG;
  if (!sw || !sw->embed || !sw->g_final || (c->m.nck > 0 && !sw->exit_T))
    return fail(c, EE_ERR_INVALID_ARG, "shared weights: NULL pointer");
  for (int i = 0; i < c->m.nck; ++i)
    if (!sw->exit_T[i]) return fail(c, EE_ERR_INVALID_ARG, "exit_T[%d] is NULL", i);
  if (c->cuda_broken) return fail(c, EE_ERR_CUDA, "context unusable after an earlier CUDA error");
  DeviceGuard dg(c->dev);
  if (join_user_stream(c) != EE_OK) return EE_ERR_CUDA;
  const Dims& m = c->m;
  EE_CUDA(c, cudaMemcpyAsync(c->E, sw->embed, (size_t)m.V * m.d * 2, cudaMemcpyDefault, c->st));
  EE_CUDA(c, cudaMemcpyAsync(c->g_final, sw->g_final, (size_t)m.d * 2, cudaMemcpyDefault, c->st));
  for (int i = 0; i < m.nck; ++i) {
    EE_CUDA(c, cudaMemcpyAsync(c->staging, sw->exit_T[i], (size_t)m.d * m.d * 2, cudaMemcpyDefault, c->st));
    EE_CUDA(c, launch_transpose_bf16(c->Tt[i], (const uint16_t*)c->staging, m.d, c->st));
  }
  EE_CUDA(c, cudaStreamSynchronize(c->st));
  c->shared_loaded = true;
  return EE_OK;
}

ee_status ee_load_weights(ee_ctx* c, const ee_weights* w) {
  if (!c) return EE_ERR_INVALID_ARG;
  if (!w || !w->layers) return fail(c, EE_ERR_INVALID_ARG, "weights: NULL pointer");
  for (int j = 0; j < c->m.L; ++j) {
    const ee_status s = ee_load_layer(c, j, &w->layers[j]);
    if (s != EE_OK) return s;
  }
  return ee_load_shared(c, &w->shared);
}

ee_status ee_set_thresholds(ee_ctx* c, const float* gamma) {
  if (!c) return EE_ERR_INVALID_ARG;
  if (c->m.nck > 0 && !gamma) return fail(c, EE_ERR_INVALID_ARG, "gamma is NULL");
  for (int i = 0; i < c->m.nck; ++i)
    if (isnan(gamma[i])) return fail(c, EE_ERR_INVALID_ARG, "gamma[%d] is NaN", i);
  if (c->cuda_broken) return fail(c, EE_ERR_CUDA, "context unusable after an earlier CUDA error");
  DeviceGuard dg(c->dev);
  std::vector<float> g(EE_MAX_CHECKPOINTS, INFINITY);
  for (int i = 0; i < c->m.nck; ++i) g[i] = gamma[i];
  c->gamma.assign(g.begin(), g.begin() + c->m.nck);
  if (join_user_stream(c) != EE_OK) return EE_ERR_CUDA;
  EE_CUDA(c, cudaMemcpyAsync(c->gamma_dev, g.data(), g.size() * sizeof(float), cudaMemcpyHostToDevice, c->st));
  EE_CUDA(c, cudaStreamSynchronize(c->st));
  return EE_OK;
}

ee_status ee_set_exit_enabled(ee_ctx* c, int32_t enabled) {
  if (!c) return EE_ERR_INVALID_ARG;
  c->exit_enabled = enabled ? 1 : 0;
  return EE_OK;
}

ee_status ee_set_exit_criterion(ee_ctx* c, int32_t criterion) {
  if (!c) return EE_ERR_INVALID_ARG;
  if (criterion != EE_EXIT_MAXPROB && criterion != EE_EXIT_STS && criterion != EE_EXIT_STS_BATCH)
    return fail(c, EE_ERR_INVALID_ARG, "unknown exit criterion %d", criterion);
  c->criterion = criterion;
  return EE_OK;
}

ee_status ee_set_token_source(ee_ctx* c, int32_t source) {
  if (!c) return EE_ERR_INVALID_ARG;
  if (source != EE_TOKEN_FINAL_HEAD && source != EE_TOKEN_EXIT_HEAD)
    return fail(c, EE_ERR_INVALID_ARG, "unknown token source %d", source);
  c->token_source = source;
  return EE_OK;
}

ee_status ee_set_use_graph(ee_ctx* c, int32_t use_graph) {
  if (!c) return EE_ERR_INVALID_ARG;
  c->use_graph = use_graph ? 1 : 0;
  return EE_OK;
}

ee_status ee_last_step_ms(const ee_ctx* c, float* ms) {
  if (!c || !ms) return EE_ERR_INVALID_ARG;
  *ms = c->last_step_ms;
  return EE_OK;
}

ee_status ee_set_profile(ee_ctx* c, int32_t profile) {
  if (!c) return EE_ERR_INVALID_ARG;
  c->profile = profile ? 1 : 0;
  return EE_OK;
}

ee_status ee_profile_read(ee_ctx* c, ee_launch_record* out, int32_t cap, int32_t* n) {
  if (!c || !n) return EE_ERR_INVALID_ARG;
  *n = (int32_t)c->prof_ms.size();
  if (out)
    for (int i = 0; i < *n && i < cap; ++i)
      out[i] = ee_launch_record{c->prof_tag[i].kind, c->prof_tag[i].layer, c->prof_ms[i],
                                i < (int)c->prof_kernel_ms.size() ? c->prof_kernel_ms[i] : 0.0f,
                                c->prof_tag[i].lists};
  return EE_OK;
}

ee_status ee_step_io(const ee_ctx* c, int32_t batch, int32_t heads, size_t* h2d, size_t* d2h,
                     int32_t* launches) {
  if (!c || batch < 1 || batch > EE_MAX_BATCH) return EE_ERR_INVALID_ARG;
  if (h2d) *h2d = sizeof(StepDesc);
  if (d2h) *d2h = step_d2h_bytes(batch);
  if (launches) {
    // begin + per layer (2 norms unless the GEMVs apply them, QKV, attention,
    // O, gate/up, down) + heads (norm, T, E) + final norm and head
    const int with_heads = heads && c->m.nck > 0;
    const bool tc = c->tc && batch_uses_tc(c->m, batch);
    const int norms = !tc && linear_stages_x(batch, c->m.d) ? 0 : 1;
    // the tensor-core GEMM serves both sub-batch lists in one launch
    const int per_layer = 5 + 2 * norms;
    // the similarity criterion replaces each head's launches by one decision launch
    const int per_ckpt = c->criterion == EE_EXIT_MAXPROB ? 2 + norms : 1;
    *launches = 1 + per_layer * c->m.L + (with_heads ? per_ckpt * c->m.nck : 0) + 1 + norms;
  }
  return EE_OK;
}

ee_status ee_set_debug(ee_ctx* c, int32_t debug) {
  if (!c) return EE_ERR_INVALID_ARG;
  c->debug = debug ? 1 : 0;
  return EE_OK;
}

ee_status ee_reset(ee_ctx* c) {
  if (!c) return EE_ERR_INVALID_ARG;
  if (c->cuda_broken) return fail(c, EE_ERR_CUDA, "context unusable after an earlier CUDA error");
  DeviceGuard dg(c->dev);
  if (join_user_stream(c) != EE_OK) return EE_ERR_CUDA;
  reset_blocks(c);
  if (fill_sentinel(c) != EE_OK) return EE_ERR_CUDA;
  EE_CUDA(c, cudaStreamSynchronize(c->st));
  return EE_OK;
}

ee_status ee_prefill(ee_ctx* c, int32_t batch, const int32_t* prompt_lens, const int32_t* tokens_concat,
                     int32_t* first_tokens_out) {
  if (!c) return EE_ERR_INVALID_ARG;
  const Dims& m = c->m;
  if (batch < 1 || batch > m.maxb)
    return fail(c, EE_ERR_CAPACITY, "batch %d outside [1, max_batch=%d]", batch, m.maxb);
  if (!prompt_lens || !tokens_concat || !first_tokens_out)
    return fail(c, EE_ERR_INVALID_ARG, "prefill: NULL pointer");
  int64_t total = 0;
  int Tmax = 0;
  for (int s = 0; s < batch; ++s) {
    if (prompt_lens[s] < 1) return fail(c, EE_ERR_INVALID_ARG, "prompt %d is empty", s);
    if (prompt_lens[s] >= m.maxs)
      return fail(c, EE_ERR_CAPACITY, "prompt %d length %d >= max_seq_len %d", s, prompt_lens[s], m.maxs);
    total += prompt_lens[s];
    Tmax = std::max(Tmax, prompt_lens[s]);
  }
  for (int64_t i = 0; i < total; ++i)
    if (tokens_concat[i] < 0 || tokens_concat[i] >= m.V)
      return fail(c, EE_ERR_INVALID_ARG, "prompt token %lld = %d outside [0, vocab)", (long long)i,
                  tokens_concat[i]);
  ee_status s = check_ready(c);
  if (s != EE_OK) return s;
  DeviceGuard dg(c->dev);
  if (join_user_stream(c) != EE_OK) return EE_ERR_CUDA;
  reset_blocks(c);
  c->batch = batch;
  // blocks for every prompt, sequence by sequence, lowest ids first
  std::vector<int32_t> bt((size_t)m.maxb * m.bps, 0);
  std::vector<int64_t> offs(batch);
  int64_t off = 0;
  for (int q = 0; q < batch; ++q) {
    offs[q] = off;
    off += prompt_lens[q];
    const int nb = (int)ceil_div(prompt_lens[q], EE_KV_BLOCK);
    for (int i = 0; i < nb; ++i) {
      const int32_t b = alloc_block(c);
      if (b < 0) return fail(c, EE_ERR_CAPACITY, "KV cache out of blocks");
      c->seq_blocks[q].push_back(b);
      bt[(size_t)q * m.bps + i] = b;
    }
  }
  EE_CUDA(c, cudaMemcpyAsync(c->block_table, bt.data(), bt.size() * sizeof(int32_t), cudaMemcpyHostToDevice,
                             c->st));
  EE_CUDA(c, cudaStreamSynchronize(c->st));
  c->prefill_exit.assign(batch, m.L - 1);
  const bool seq_exit = !c->prefill_tau.empty() && m.nck > 0;
  // One pass over the prompts, one position per step.  Sequence-level exit
  // ("River-LLM 深度解析" §6.1) takes two: the first scores every prompt
  // token with the state transition similarity at each checkpoint (no exit)
  // and keeps each prompt's minimum; a prompt leaves at the first checkpoint
  // whose minimum is above its threshold (strict); the second pass reruns the
  // prompts with those exits forced, so the layers after them run on the
  // int4 copies and rewrite their K/V (the layers before recompute the same
  // values).
  std::vector<float> low((size_t)batch * std::max(m.nck, 1), INFINITY);
  const int saved_criterion = c->criterion;
  if (seq_exit) {
    c->criterion = EE_EXIT_STS;
    std::vector<float> inf(EE_MAX_CHECKPOINTS, INFINITY);
    EE_CUDA(c, cudaMemcpyAsync(c->gamma_dev, inf.data(), inf.size() * sizeof(float), cudaMemcpyHostToDevice, c->st));
  }
  auto restore = [&]() -> ee_status {
    c->criterion = saved_criterion;
    if (!seq_exit) return EE_OK;
    std::vector<float> g(EE_MAX_CHECKPOINTS, INFINITY);
    for (int i = 0; i < m.nck; ++i) g[i] = c->gamma[i];
    EE_CUDA(c, cudaMemcpyAsync(c->gamma_dev, g.data(), g.size() * sizeof(float), cudaMemcpyHostToDevice, c->st));
    EE_CUDA(c, cudaStreamSynchronize(c->st));
    return EE_OK;
  };
  StepDesc* d = c->desc_host;
  const int passes = seq_exit ? 2 : 1;
  for (int pass = 0; pass < passes; ++pass) {
    if (pass == 1) {
      bool any = false;
      for (int q = 0; q < batch; ++q)
        for (int k = 0; k < m.nck; ++k)
          if (c->prefill_exit[q] == m.L - 1 && low[(size_t)q * m.nck + k] > c->prefill_tau[k]) {
            c->prefill_exit[q] = c->ckpts[k];
            any = true;
          }
      if (!any) break;  // no prompt leaves: the first pass was the plain prefill
    }
    for (int t = 0; t < Tmax; ++t) {
      d->n_part = 0;
      d->n_fin = 0;
      for (int q = 0; q < EE_MAX_BATCH; ++q) d->forced_exit[q] = -1;
      for (int q = 0; q < batch; ++q) {
        d->new_block[q] = -1;
        if (pass == 1 && c->prefill_exit[q] != m.L - 1) d->forced_exit[q] = c->prefill_exit[q];
        if (t < prompt_lens[q]) {
          d->part[d->n_part++] = q;
          d->tokens[q] = tokens_concat[offs[q] + t];
          d->pos[q] = t;
          if (t == prompt_lens[q] - 1) d->fin[d->n_fin++] = q;
        }
      }
      d->debug = c->debug;
      s = run_step(c, batch, seq_exit);
      if (s != EE_OK) {
        restore();
        return s;
      }
      if (seq_exit && pass == 0)
        for (int i = 0; i < d->n_part; ++i) {
          const int q = d->part[i];
          for (int k = 0; k < m.nck; ++k)
            low[(size_t)q * m.nck + k] =
                std::min(low[(size_t)q * m.nck + k], c->out_host->conf[q * EE_MAX_CHECKPOINTS + k]);
        }
      for (int i = 0; i < d->n_fin; ++i) first_tokens_out[d->fin[i]] = c->out_host->next_token[d->fin[i]];
    }
  }
  s = restore();
  if (s != EE_OK) return s;
  for (int q = 0; q < batch; ++q) c->seq_pos[q] = prompt_lens[q];
  return EE_OK;
}

ee_status ee_set_prefill_exit(ee_ctx* c, const float* tau) {
  if (!c) return EE_ERR_INVALID_ARG;
  if (!tau) {
    c->prefill_tau.clear();
    return EE_OK;
  }
  for (int i = 0; i < c->m.nck; ++i)
    if (isnan(tau[i])) return fail(c, EE_ERR_INVALID_ARG, "tau[%d] is NaN", i);
  c->prefill_tau.assign(tau, tau + c->m.nck);
  return EE_OK;
}

ee_status ee_prefill_exit_layers(const ee_ctx* c, int32_t* out) {
  if (!c || !out) return EE_ERR_INVALID_ARG;
  for (int q = 0; q < c->batch; ++q) out[q] = q < (int)c->prefill_exit.size() ? c->prefill_exit[q] : c->m.L - 1;
  return EE_OK;
}

ee_status ee_decode_step(ee_ctx* c, const int32_t* in_tokens, int32_t* next_tokens_out,
                         int32_t* exit_layers_out) {
  if (!c) return EE_ERR_INVALID_ARG;
  if (c->batch < 1) return fail(c, EE_ERR_STATE, "decode before prefill");
  if (!in_tokens || !next_tokens_out || !exit_layers_out)
    return fail(c, EE_ERR_INVALID_ARG, "decode: NULL pointer");
  const Dims& m = c->m;
  const int B = c->batch;
  for (int q = 0; q < B; ++q) {
    if (in_tokens[q] < 0 || in_tokens[q] >= m.V)
      return fail(c, EE_ERR_INVALID_ARG, "token %d of sequence %d outside [0, vocab)", in_tokens[q], q);
    if (c->seq_pos[q] >= m.maxs)
      return fail(c, EE_ERR_CAPACITY, "sequence %d reached max_seq_len %d", q, m.maxs);
  }
  if (c->token_source == EE_TOKEN_EXIT_HEAD && c->criterion != EE_EXIT_MAXPROB && c->exit_enabled)
    return fail(c, EE_ERR_STATE, "exit-head tokens need the exit-head criterion (EE_EXIT_MAXPROB)");
  ee_status s = check_ready(c);
  if (s != EE_OK) return s;
  DeviceGuard dg(c->dev);
  if (join_user_stream(c) != EE_OK) return EE_ERR_CUDA;
  StepDesc* d = c->desc_host;
  d->n_part = B;
  d->n_fin = B;
  for (int q = 0; q < EE_MAX_BATCH; ++q) d->forced_exit[q] = -1;
  for (int q = 0; q < B; ++q) {
    d->part[q] = q;
    d->fin[q] = q;
    d->tokens[q] = in_tokens[q];
    d->pos[q] = c->seq_pos[q];
    d->new_block[q] = -1;
    if (c->seq_pos[q] % EE_KV_BLOCK == 0) {
      const int32_t b = alloc_block(c);
      if (b < 0) return fail(c, EE_ERR_CAPACITY, "KV cache out of blocks");
      c->seq_blocks[q].push_back(b);
      d->new_block[q] = b;
    }
  }
  d->debug = c->debug;
  s = run_step(c, B, c->exit_enabled && m.nck > 0);
  if (s != EE_OK) return s;
  for (int q = 0; q < B; ++q) {
    next_tokens_out[q] = c->out_host->next_token[q];
    exit_layers_out[q] = c->out_host->exit_layer[q];
    c->seq_pos[q] += 1;
  }
  return EE_OK;
}

ee_status ee_seq_info(const ee_ctx* c, int32_t* batch, int32_t seq, int32_t* pos) {
  if (!c) return EE_ERR_INVALID_ARG;
  if (batch) *batch = c->batch;
  if (pos) {
    if (seq < 0 || seq >= c->batch) return EE_ERR_INVALID_ARG;
    *pos = c->seq_pos[seq];
  }
  return EE_OK;
}

ee_status ee_debug_hidden(ee_ctx* c, int32_t layer, float* out) {
  if (!c || !out) return EE_ERR_INVALID_ARG;
  if (layer < 0 || layer >= c->m.L) return fail(c, EE_ERR_INVALID_ARG, "layer out of range");
  DeviceGuard dg(c->dev);
  EE_CUDA(c, cudaMemcpy(out, c->hdbg + (size_t)layer * EE_MAX_BATCH * c->m.d,
                        (size_t)c->batch * c->m.d * sizeof(float), cudaMemcpyDeviceToHost));
  return EE_OK;
}

ee_status ee_debug_conf(ee_ctx* c, float* out) {
  if (!c || !out) return EE_ERR_INVALID_ARG;
  for (int q = 0; q < c->batch; ++q)
    for (int k = 0; k < c->m.nck; ++k) out[q * c->m.nck + k] = c->out_host->conf[q * EE_MAX_CHECKPOINTS + k];
  return EE_OK;
}

ee_status ee_debug_kv(ee_ctx* c, int32_t seq, int32_t layer, int32_t pos, uint16_t* k, uint16_t* v) {
  if (!c || !k || !v) return EE_ERR_INVALID_ARG;
  const Dims& m = c->m;
  if (seq < 0 || seq >= c->batch || layer < 0 || layer >= m.L || pos < 0 || pos >= c->seq_pos[seq])
    return fail(c, EE_ERR_INVALID_ARG, "debug_kv: index out of range");
  DeviceGuard dg(c->dev);
  const int32_t block = c->seq_blocks[seq][pos / EE_KV_BLOCK];
  const int off = pos % EE_KV_BLOCK;
  for (int g = 0; g < m.hkv; ++g) {
    const size_t e = (size_t)layer * m.kv_layer_elems + (((size_t)block * m.hkv + g) * EE_KV_BLOCK + off) * m.hd;
    EE_CUDA(c, cudaMemcpy(k + (size_t)g * m.hd, c->kcache + e, (size_t)m.hd * 2, cudaMemcpyDeviceToHost));
    EE_CUDA(c, cudaMemcpy(v + (size_t)g * m.hd, c->vcache + e, (size_t)m.hd * 2, cudaMemcpyDeviceToHost));
  }
  return EE_OK;
}

ee_status ee_debug_block_table(ee_ctx* c, int32_t seq, int32_t* out, int32_t cap, int32_t* n_blocks) {
  if (!c || !n_blocks) return EE_ERR_INVALID_ARG;
  if (seq < 0 || seq >= c->batch) return fail(c, EE_ERR_INVALID_ARG, "seq out of range");
  const auto& b = c->seq_blocks[seq];
  *n_blocks = (int32_t)b.size();
  if (out)
    for (int i = 0; i < (int)b.size() && i < cap; ++i) out[i] = b[i];
  // cross-check with the device copy
  DeviceGuard dg(c->dev);
  std::vector<int32_t> dev(c->m.bps);
  EE_CUDA(c, cudaMemcpy(dev.data(), c->block_table + (size_t)seq * c->m.bps, dev.size() * 4,
                        cudaMemcpyDeviceToHost));
  for (size_t i = 0; i < b.size(); ++i)
    if (dev[i] != b[i]) return fail(c, EE_ERR_STATE, "device block table differs at %zu", i);
  return EE_OK;
}

ee_status ee_debug_int4(ee_ctx* c, int32_t layer, int32_t mat, uint8_t* packed, uint16_t* scales) {
  if (!c || !packed || !scales) return EE_ERR_INVALID_ARG;
  if (layer < 0 || layer >= c->m.L || mat < 0 || mat >= EE_N_MATS)
    return fail(c, EE_ERR_INVALID_ARG, "debug_int4: index out of range");
  DeviceGuard dg(c->dev);
  const Dims& m = c->m;
  const MatPlace pl = placement(m, mat);
  const LayerBufs& b = c->layers[layer];
  const Mat4 blk[4] = {b.qkv, b.o, b.gu, b.d};
  const int K = pl.cols, ng = (int)ceil_div(K, EE_QUANT_GROUP), ss = sstride_of(K);
  for (int r = 0; r < pl.rows; ++r) {
    const int64_t dr = device_row(pl, r);
    EE_CUDA(c, cudaMemcpy(packed + (size_t)r * K / 2, blk[pl.block].q + dr * K / 2, K / 2,
                          cudaMemcpyDeviceToHost));
    EE_CUDA(c, cudaMemcpy(scales + (size_t)r * ng, blk[pl.block].s + dr * ss, (size_t)ng * 2,
                          cudaMemcpyDeviceToHost));
  }
  return EE_OK;
}

// ------------------------------------------------------------------ single kernels
// Kernel attributes set and SM count read once per device (the op entry
// points are called per launch, so they skip the per-call attribute calls).
constexpr int kMaxOpDevices = 64;
static std::atomic<int> g_op_sms[kMaxOpDevices];

static int device_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxOpDevices) return 0;
  const int cached = g_op_sms[dev].load(std::memory_order_acquire);
  if (cached > 0) return cached;
  if (linear_prepare() != cudaSuccess || attention_prepare() != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  n = 2 * n > kHeadGridMax ? kHeadGridMax / 2 : n;
  g_op_sms[dev].store(n, std::memory_order_release);
  return n;
}

ee_status ee_op_quantize_int4(const uint16_t* w, int32_t rows, int32_t cols, uint8_t* packed,
                              uint16_t* scales, int32_t scale_stride, void* stream) {
  if (!w || !packed || !scales || rows < 0 || cols <= 0 || cols % 32 ||
      scale_stride < ceil_div(cols, EE_QUANT_GROUP))
    return EE_ERR_INVALID_ARG;
  return launch_quantize_int4(w, rows, cols, packed, scales, scale_stride, (cudaStream_t)stream) ==
                 cudaSuccess
             ? EE_OK
             : EE_ERR_CUDA;
}

static ee_status op_linear(int32_t M, int32_t N, int32_t K, const uint16_t* xh, const uint16_t* w, const uint8_t* q, const uint16_t* s, int32_t sstride, float* y,
                           int32_t* err, void* stream) {
  if (M < 1 || M > EE_MAX_BATCH || N < 2 || N % 2 || !linear_shape_ok(K) || !y) return EE_ERR_INVALID_ARG;
  if (q && ((uintptr_t)q % 16 || (uintptr_t)s % 16)) return EE_ERR_INVALID_ARG;
  if (w && (uintptr_t)w % 16) return EE_ERR_INVALID_ARG;
  const int sms = device_sms();
  if (sms <= 0) return EE_ERR_CUDA;
  LinearParams p = {};
  p.N = N;
  p.K = K;
  p.w = w;
  p.wq = q;
  p.ws = s;
  p.sstride = sstride;
  p.m_direct_full = w ? M : 0;
  p.m_direct_exit = q ? M : 0;
  p.xh = xh;
  p.x_stride = K;
  p.epi = EPI_F32;
  p.out_f32 = y;
  p.out_stride = N;
  p.err = err;
  p.max_rows = M;
  return launch_linear(p, linear_grid(N, sms), false, (cudaStream_t)stream) == cudaSuccess ? EE_OK
                                                                                           : EE_ERR_CUDA;
}

ee_status ee_op_linear_bf16(int32_t M, int32_t N, int32_t K, const uint16_t* x_f16, const uint16_t* w,
                            float* y, int32_t* err_flag, void* stream) {
  if (!x_f16 || !w) return EE_ERR_INVALID_ARG;
  return op_linear(M, N, K, x_f16, w, nullptr, nullptr, 0, y, err_flag, stream);
}

ee_status ee_op_linear_int4(int32_t M, int32_t N, int32_t K, const uint16_t* x_f16, const uint8_t* packed,
                            const uint16_t* scales, int32_t scale_stride, float* y, int32_t* err_flag,
                            void* stream) {
  if (!x_f16 || !packed || !scales || scale_stride < ceil_div(K, EE_QUANT_GROUP)) return EE_ERR_INVALID_ARG;
  return op_linear(M, N, K, x_f16, nullptr, packed, scales, scale_stride, y, err_flag, stream);
}

size_t ee_attention_scratch_bytes(int32_t B, int32_t n_heads, int32_t n_kv_heads, int32_t head_dim,
                                  int32_t max_ctx) {
  if (B < 1 || B > EE_MAX_BATCH || n_kv_heads < 1 || n_heads % n_kv_heads || max_ctx < 1 ||
      (head_dim != 64 && head_dim != 128))
    return 0;
  const int nsplit = attention_nsplit(max_ctx, head_dim);
  if (nsplit > attention_max_split()) return 0;
  return align_up(attention_part_floats(B, n_heads, n_kv_heads, head_dim, nsplit) * 4, kAlign) +
         (size_t)EE_MAX_BATCH * n_kv_heads * 4;
}

}  // extern "C"

// Argument checks of the attention entry points (scratch checked by the caller).
ee_status ee_attention_args_check(int32_t B, int32_t n_heads, int32_t n_kv_heads, int32_t head_dim,
                                  int32_t max_ctx, const float* q, const uint16_t* kcache,
                                  const uint16_t* vcache, const int32_t* block_table, int32_t bt_stride,
                                  const int32_t* pos, const float* o) {
  if (B < 1 || B > EE_MAX_BATCH || n_kv_heads < 1 || n_heads % n_kv_heads || (head_dim != 64 && head_dim != 128))
    return EE_ERR_INVALID_ARG;
  if (max_ctx < 1 || attention_nsplit(max_ctx, head_dim) > attention_max_split()) return EE_ERR_INVALID_ARG;
  const int G = n_heads / n_kv_heads;
  if (G != 1 && G != 2 && G != 4 && G != 8) return EE_ERR_INVALID_ARG;
  if (!q || !kcache || !vcache || !block_table || !pos || !o || bt_stride < 1) return EE_ERR_INVALID_ARG;
  return EE_OK;
}

extern "C" {

ee_status ee_op_attention(int32_t B, int32_t n_heads, int32_t n_kv_heads, int32_t head_dim, int32_t max_ctx,
                          const float* q, const uint16_t* kcache, const uint16_t* vcache,
                          const int32_t* block_table, int32_t bt_stride, const int32_t* pos, float* o,
                          void* scratch, int32_t* err_flag, void* stream) {
  const ee_status chk = ee_attention_args_check(B, n_heads, n_kv_heads, head_dim, max_ctx, q, kcache, vcache,
                                                block_table, bt_stride, pos, o);
  if (chk != EE_OK) return chk;
  if (!scratch) return EE_ERR_INVALID_ARG;
  const int sms = device_sms();
  if (sms <= 0) return EE_ERR_CUDA;
  AttnParams p = {};
  p.m_direct = B;
  p.n_heads = n_heads;
  p.n_kv_heads = n_kv_heads;
  p.head_dim = head_dim;
  p.q = q;
  p.q_stride = n_heads * head_dim;
  p.kc = kcache;
  p.vc = vcache;
  p.block_table = block_table;
  p.bt_stride = bt_stride;
  p.pos = pos;
  p.nsplit = attention_nsplit(max_ctx, head_dim);
  p.bpc = attention_blocks_per_cta(head_dim);
  const size_t pbytes = align_up(attention_part_floats(B, n_heads, n_kv_heads, head_dim, p.nsplit) * 4, kAlign);
  p.part = (float*)scratch;
  p.counters = (int32_t*)((uint8_t*)scratch + pbytes);
  p.o_f32 = o;
  p.o_stride = n_heads * head_dim;
  p.err = err_flag;
  return launch_attention(p, B, false, (cudaStream_t)stream) == cudaSuccess ? EE_OK : EE_ERR_CUDA;
}

size_t ee_head_scratch_bytes(int32_t M) {
  if (M < 1 || M > EE_MAX_BATCH) return 0;
  return (size_t)kHeadGridMax * EE_MAX_BATCH * 4 * 4 + kAlign;
}

ee_status ee_op_vocab_head(int32_t M, int32_t V, int32_t d, const uint16_t* u_f16, const uint16_t* E, float* conf,
                           int32_t* argmax, void* scratch, int32_t* err_flag, void* stream) {
  if (M < 1 || M > EE_MAX_BATCH || V < 2 || V % 2 || !linear_shape_ok(d) || !u_f16 || !E || !conf || !argmax ||
      !scratch)
    return EE_ERR_INVALID_ARG;
  const int sms = device_sms();
  if (sms <= 0) return EE_ERR_CUDA;
  LinearParams p = {};
  p.N = V;
  p.K = d;
  p.w = E;
  p.m_direct_full = M;
  p.xh = u_f16;
  p.x_stride = d;
  p.epi = EPI_HEAD;
  p.head_mode = HEAD_CONF_ARGMAX;
  p.head_part = (float*)scratch;
  p.head_counter = (int32_t*)((uint8_t*)scratch + (size_t)kHeadGridMax * EE_MAX_BATCH * 4 * 4);
  p.conf_out = conf;
  p.argmax_out = argmax;
  p.err = err_flag;
  p.max_rows = M;
  return launch_linear(p, std::min(linear_grid(V, sms), kHeadGridMax), false, (cudaStream_t)stream) ==
                 cudaSuccess
             ? EE_OK
             : EE_ERR_CUDA;
}

}  // extern "C"
