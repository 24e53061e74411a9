// Split-K GQA decode attention over the paged KV cache.
//
// One query position per sequence attends over positions 0..pos (causal).
// The grid is (split, kv head, sequence slot).  A CTA owns up to BPC whole
// 16-slot blocks of one sequence's context for one kv head and serves all
// Hq/Hkv query heads of that group from one read of each K and V row.
//
// Data movement: the CTA's K and V tiles ([16][hd] fp16 each, contiguous in
// the cache) are bulk-copied into shared memory by one thread.  Blocks that
// hold only earlier positions were written by earlier steps, so their copies
// are issued before the grid dependency wait and overlap the QKV projection
// still running; the block holding the current position is copied after it.
//
// Compute, in three phases over the CTA's tokens (at most BPC * 16): (1)
// scores s = q_h . k_t / sqrt(hd) for every query head of the group into
// shared memory -- lanes own 8 head dims (one 16-byte shared load per row),
// hd/8 lanes form a token group and reduce with xor shuffles; (2) per head
// the CTA-wide max m and p_t = exp(s_t - m), l = sum p_t; (3) acc = sum p_t
// v_t with independent accumulators per lane, reduced over token groups and
// warps.  The CTA writes one partial (acc, m, l) per head, and the last CTA
// of each (sequence, kv head) -- found with an atomic counter, nothing waits
// -- merges the partials:
// o = sum_i acc_i exp(m_i - M) / sum_i l_i exp(m_i - M), M = max_i m_i.
// The grid covers the longest context; a CTA whose split lies beyond its own
// sequence's context returns at once, and the merge counts only the splits
// that context needs.
//
// Cache layout (one layer): [block][kv head][16 slots][head_dim] fp16.
#include <math.h>

#include "ee_attention.cuh"
#include "ee_common.cuh"
#include "ee_kernels.cuh"

namespace ee {

namespace {

template <int HD, int G>
__global__ void __launch_bounds__(kThreadsA) k_attention(const AttnParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ AttnShared<HD, G> sh;
  attention_item<HD, G>(p, blockIdx.x, blockIdx.y, blockIdx.z, smem, sh);
}

template <int HD, int G>
cudaError_t set_attr_t() {
  static_assert(kThreadsA * 16 + 3 * kMaxSplit * G * 4 + G * 4 <= kKvSmem, "merge scratch");
  static_assert(kAttnWarps * (G * HD + 8 * G) * 4 <= kKvSmem, "warp partials");
  return cudaFuncSetAttribute(k_attention<HD, G>, cudaFuncAttributeMaxDynamicSharedMemorySize, kKvSmem);
}

template <int HD, int G>
cudaError_t launch_t(const AttnParams& p, int batch_slots, bool pdl, cudaStream_t st) {
  constexpr size_t smem = kKvSmem;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.nsplit, p.n_kv_heads, batch_slots);
  cfg.blockDim = dim3(kThreadsA);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, k_attention<HD, G>, p);
}

}  // namespace

int attention_blocks_per_cta(int head_dim) { return head_dim == 64 ? blocks_per_cta<64>() : blocks_per_cta<128>(); }

size_t attention_part_floats(int batch_slots, int n_heads, int n_kv_heads, int head_dim, int nsplit) {
  const int G = n_heads / n_kv_heads;
  return (size_t)batch_slots * n_kv_heads * nsplit * (G * head_dim + ((2 * G + 3) / 4) * 4);
}

int attention_max_split() { return kMaxSplit; }

cudaError_t attention_prepare() {
  cudaError_t e;
#define EE_ATT_ATTR(HD_, G_) \
  if ((e = set_attr_t<HD_, G_>()) != cudaSuccess) return e;
  EE_ATT_ATTR(64, 1)
  EE_ATT_ATTR(64, 2)
  EE_ATT_ATTR(64, 4)
  EE_ATT_ATTR(64, 8)
  EE_ATT_ATTR(128, 1)
  EE_ATT_ATTR(128, 2)
  EE_ATT_ATTR(128, 4)
  EE_ATT_ATTR(128, 8)
#undef EE_ATT_ATTR
  return cudaSuccess;
}

int attention_nsplit(int max_ctx, int head_dim) {
  const int nb = (max_ctx + 15) / 16;
  const int bpc = attention_blocks_per_cta(head_dim);
  return (nb + bpc - 1) / bpc;
}

cudaError_t launch_attention(const AttnParams& p, int batch_slots, bool pdl, cudaStream_t st) {
  const int G = p.n_heads / p.n_kv_heads;
  if (p.nsplit < 1 || p.nsplit > kMaxSplit || p.bpc != attention_blocks_per_cta(p.head_dim))
    return cudaErrorInvalidValue;
#define EE_ATT_CASE(HD_, G_) \
  if (p.head_dim == HD_ && G == G_) return launch_t<HD_, G_>(p, batch_slots, pdl, st);
  EE_ATT_CASE(64, 1)
  EE_ATT_CASE(64, 2)
  EE_ATT_CASE(64, 4)
  EE_ATT_CASE(64, 8)
  EE_ATT_CASE(128, 1)
  EE_ATT_CASE(128, 2)
  EE_ATT_CASE(128, 4)
  EE_ATT_CASE(128, 8)
#undef EE_ATT_CASE
  return cudaErrorInvalidValue;
}

}  // namespace ee
