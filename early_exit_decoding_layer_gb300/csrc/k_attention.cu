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

#include "ee_common.cuh"
#include "ee_kernels.cuh"

namespace ee {

namespace {

constexpr int kWarps = 8;
constexpr int kThreadsA = kWarps * 32;
constexpr int kKvSmem = 64 * 1024;  // K + V tiles of one CTA
constexpr int kMaxSplit = 128;

EE_DEV void to_float8(const uint4& v, float* f) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 t = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}

template <int HD>
constexpr int blocks_per_cta() {
  return kKvSmem / (2 * 16 * HD * 2);
}
static_assert(blocks_per_cta<64>() <= 32 && blocks_per_cta<128>() <= 32, "one lane per block");

template <int HD, int G>
__global__ void __launch_bounds__(kThreadsA) k_attention(const AttnParams p) {
  constexpr int LPT = HD / 8;    // lanes per token
  constexpr int TPW = 32 / LPT;  // tokens per warp step
  constexpr int TILE = 16 * HD;  // elements of one (block, kv head) tile
  constexpr int BPC = blocks_per_cta<HD>();
  constexpr int PSZ = G * HD + ((2 * G + 3) / 4) * 4;  // partial: acc [G][HD], m [G], l [G] (16-B rows)
  extern __shared__ __align__(128) uint8_t smem[];
  uint16_t* Ks = reinterpret_cast<uint16_t*>(smem);
  uint16_t* Vs = Ks + BPC * TILE;
  __shared__ __align__(8) uint64_t bar;
  __shared__ int s_last;

  const int split = blockIdx.x, g = blockIdx.y, z = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int sub = lane / LPT, dl = lane % LPT;
  const int hkv = p.n_kv_heads;

  // The list, the positions and the block-table entries of earlier blocks
  // were written at least two launches back: safe before the dependency wait.
  const int count = p.list ? ld_volatile_i32(p.list) : p.m_direct;
  const bool active = z < count;
  int seq = 0, ctx = 0, b0 = 0, b1 = 0, last = -1, nact = 0;
  if (active) {
    seq = p.list ? ld_volatile_i32(p.list + 1 + z) : z;
    ctx = ld_volatile_i32(p.pos + seq) + 1;
    const int nb = (ctx + 15) >> 4;
    nact = (nb + p.bpc - 1) / p.bpc;  // splits this sequence's context needs
    b0 = split * p.bpc;
    b1 = min(nb, b0 + p.bpc);
    last = nb - 1;
  }
  // a split beyond the context has nothing to read, write or merge
  if (!active || split >= nact) return;
  const bool have = b0 < b1;
  const int32_t* bt = p.block_table + (size_t)seq * p.bt_stride;
  if (tid == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  const uint64_t pol = l2_evict_first_policy();
  if (warp == 0 && have) {
    // one lane per block: the block-table reads and the copies go out in parallel
    if (lane == 0) mbar_arrive_expect_tx(&bar, (uint32_t)(b1 - b0) * 2 * TILE * 2);
    __syncwarp();
    const int b = b0 + lane;
    if (b < b1 && b != last) {
      const size_t off = ((size_t)ld_volatile_i32(bt + b) * hkv + g) * TILE;
      bulk_g2s(Ks + lane * TILE, p.kc + off, TILE * 2, &bar, pol);
      bulk_g2s(Vs + lane * TILE, p.vc + off, TILE * 2, &bar, pol);
    }
  }
  grid_dep_wait();
  grid_dep_launch();
  if (tid == 0 && have && last >= b0 && last < b1) {
    const size_t off = ((size_t)ld_volatile_i32(bt + last) * hkv + g) * TILE;
    bulk_g2s(Ks + (last - b0) * TILE, p.kc + off, TILE * 2, &bar, pol);
    bulk_g2s(Vs + (last - b0) * TILE, p.vc + off, TILE * 2, &bar, pol);
  }
  constexpr int TOK = BPC * 16;  // tokens per CTA at most
  __shared__ float S[G][TOK];    // scores, then exp(s - m)
  __shared__ float hm[G], hl[G];
  float* wpart = reinterpret_cast<float*>(smem);  // [warp][PSZ], after the tiles are consumed

  bool ok = true;
  if (have) ok = mbar_wait_bounded(&bar, 0, p.err, DERR_FULL_WAIT);
  if (have && !ok) mbar_wait_bounded(&bar, 0, p.err, DERR_DRAIN_WAIT);  // copies land before reuse
  const bool run = have && ok;
  const int t0 = b0 * 16, n = run ? min(ctx, b1 * 16) - t0 : 0;  // tokens of this CTA

  // (1) scores
  if (n > 0) {
    const float scale = rsqrtf((float)HD);
    float q[G][8];
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const float4* qp =
          reinterpret_cast<const float4*>(p.q + (size_t)seq * p.q_stride + (g * G + h) * HD + dl * 8);
      const float4 a = qp[0], b = qp[1];
      q[h][0] = a.x * scale;
      q[h][1] = a.y * scale;
      q[h][2] = a.z * scale;
      q[h][3] = a.w * scale;
      q[h][4] = b.x * scale;
      q[h][5] = b.y * scale;
      q[h][6] = b.z * scale;
      q[h][7] = b.w * scale;
    }
    for (int base = warp * TPW; base < n; base += kWarps * TPW) {
      const int r = base + sub;
      float kf[8];
      to_float8(*reinterpret_cast<const uint4*>(Ks + min(r, n - 1) * HD + dl * 8), kf);
      float sc[G];
#pragma unroll
      for (int h = 0; h < G; ++h) {
        float d = 0.0f;
#pragma unroll
        for (int i = 0; i < 8; ++i) d = fmaf(q[h][i], kf[i], d);
        sc[h] = d;
      }
#pragma unroll
      for (int o = LPT / 2; o > 0; o >>= 1) {
#pragma unroll
        for (int h = 0; h < G; ++h) sc[h] += __shfl_xor_sync(0xffffffffu, sc[h], o);
      }
      if (dl == 0 && r < n) {
#pragma unroll
        for (int h = 0; h < G; ++h) S[h][r] = sc[h];
      }
    }
  }
  __syncthreads();
  // (2) per head: m = max s, p = exp(s - m), l = sum p
  if (warp < G) {
    const int h = warp;
    float m = -INFINITY;
    for (int r = lane; r < n; r += 32) m = fmaxf(m, S[h][r]);
    m = warp_max(m);
    float l = 0.0f;
    for (int r = lane; r < n; r += 32) {
      const float e = expf(S[h][r] - m);
      S[h][r] = e;
      l += e;
    }
    l = warp_sum(l);
    if (lane == 0) {
      hm[h] = n > 0 ? m : -INFINITY;
      hl[h] = l;
    }
  }
  __syncthreads();
  // (3) acc = sum_t p_t v_t
  float acc[G][8];
#pragma unroll
  for (int h = 0; h < G; ++h)
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[h][i] = 0.0f;
  for (int base = warp * TPW; base < n; base += kWarps * TPW) {
    const int r = base + sub;
    if (r < n) {
      float vf[8];
      to_float8(*reinterpret_cast<const uint4*>(Vs + r * HD + dl * 8), vf);
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float pr = S[h][r];
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[h][i] = fmaf(pr, vf[i], acc[h][i]);
      }
    }
  }
  // sum the token groups of this warp (lanes with the same dims)
#pragma unroll
  for (int o = LPT; o < 32; o <<= 1) {
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[h][i] += __shfl_xor_sync(0xffffffffu, acc[h][i], o);
  }
  __syncthreads();  // the K/V tiles are no longer read: reuse the space
  if (sub == 0) {
    float* dst = wpart + warp * PSZ;
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
      for (int i = 0; i < 8; ++i) dst[h * HD + dl * 8 + i] = acc[h][i];
  }
  __syncthreads();

  // CTA partial: sum the warps (one m per head for the whole CTA)
  float* part = p.part + (((size_t)z * hkv + g) * p.nsplit + split) * PSZ;
  for (int idx = tid; idx < G * HD; idx += kThreadsA) {
    float a = 0.0f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) a += wpart[w * PSZ + idx];
    part[idx] = a;
  }
  if (tid < G) {
    part[G * HD + tid] = hm[tid];
    part[G * HD + G + tid] = hl[tid];
  }
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    const int old = atomicAdd(p.counters + (size_t)z * hkv + g, 1);
    s_last = (old == nact - 1);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  // last CTA of this (sequence, kv head): merge the splits.  Warp w takes
  // heads w, w+4, ...: M = max m, weights exp(m - M), L = sum weight * l.
  const float* parts = p.part + ((size_t)z * hkv + g) * p.nsplit * PSZ;
  float* wts = reinterpret_cast<float*>(smem);  // [split][G]
  float* inv_l = wts + kMaxSplit * G;           // [G]
  for (int h = warp; h < G; h += kWarps) {
    float mloc = -INFINITY;
    for (int s = lane; s < nact; s += 32) {
      const float l = __ldcg(parts + (size_t)s * PSZ + G * HD + G + h);
      if (l > 0.0f) mloc = fmaxf(mloc, __ldcg(parts + (size_t)s * PSZ + G * HD + h));
    }
    const float M = warp_max(mloc);
    float lsum = 0.0f;
    for (int s = lane; s < nact; s += 32) {
      const float l = __ldcg(parts + (size_t)s * PSZ + G * HD + G + h);
      const float w = l > 0.0f ? expf(__ldcg(parts + (size_t)s * PSZ + G * HD + h) - M) : 0.0f;
      wts[s * G + h] = w;
      lsum += w * l;
    }
    lsum = warp_sum(lsum);
    if (lane == 0) inv_l[h] = 1.0f / lsum;
  }
  __syncthreads();
  for (int i4 = tid; i4 < G * HD / 4; i4 += kThreadsA) {
    const int h = (i4 * 4) / HD;
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
    int s = 0;
    for (; s + 8 <= nact; s += 8) {
      float4 v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) v[u] = __ldcg(reinterpret_cast<const float4*>(parts + (size_t)(s + u) * PSZ) + i4);
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const float w = wts[(s + u) * G + h];
        o.x = fmaf(w, v[u].x, o.x);
        o.y = fmaf(w, v[u].y, o.y);
        o.z = fmaf(w, v[u].z, o.z);
        o.w = fmaf(w, v[u].w, o.w);
      }
    }
    for (; s < nact; ++s) {
      const float4 v = __ldcg(reinterpret_cast<const float4*>(parts + (size_t)s * PSZ) + i4);
      const float w = wts[s * G + h];
      o.x = fmaf(w, v.x, o.x);
      o.y = fmaf(w, v.y, o.y);
      o.z = fmaf(w, v.z, o.z);
      o.w = fmaf(w, v.w, o.w);
    }
    const float il = inv_l[h];
    const float ov[4] = {o.x * il, o.y * il, o.z * il, o.w * il};
    const int col0 = g * G * HD + i4 * 4;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (p.o_f32) p.o_f32[(size_t)seq * p.o_stride + col0 + u] = ov[u];
      if (p.oh) p.oh[(size_t)seq * p.o_stride + xh_slot(col0 + u)] = float_to_half_bits(ov[u]);
    }
  }
  if (tid == 0) p.counters[(size_t)z * hkv + g] = 0;
}

template <int HD, int G>
cudaError_t set_attr_t() {
  static_assert(kMaxSplit * G * 4 + G * 4 <= kKvSmem, "merge scratch");
  static_assert(kWarps * (G * HD + 8 * G) * 4 <= kKvSmem, "warp partials");
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
