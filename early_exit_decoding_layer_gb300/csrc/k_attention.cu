// Split-K GQA decode attention over the paged KV cache.
//
// One query position per sequence attends over positions 0..pos (causal).
// The grid is (split, kv head, sequence slot).  A CTA takes one contiguous
// slice of the context for one kv head and serves all Hq/Hkv query heads of
// that group from one read of each K and V row.  Lanes own 8 head dims (one
// 16-byte load per row), hd/8 lanes form a token group, and each warp works
// on 32/(hd/8) tokens at a time, four tokens per group in flight.  Scores are
// reduced across the token group with xor shuffles; the softmax is online
// (running max m, sum l, weighted values acc).  Token groups, then warps, are
// merged in registers and shared memory; the CTA writes one partial
// (m, l, acc) and the last CTA of each (sequence, kv head) -- found with an
// atomic counter, no waiting -- merges the partials and writes the output:
// o = sum_i acc_i exp(m_i - M) / sum_i l_i exp(m_i - M).
//
// Cache layout (one layer): [block][kv head][16 slots][head_dim] fp16.
#include <math.h>

#include "ee_common.cuh"
#include "ee_kernels.cuh"

namespace ee {

namespace {

constexpr int kWarps = 4;
constexpr int kUnroll = 4;

EE_DEV void to_float8(const uint4& v, float* f) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 t = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}

// Merge (m2, l2, a2) into (m1, l1, a1).
template <int N>
EE_DEV void merge_state(float& m1, float& l1, float* a1, float m2, float l2, const float* a2) {
  if (l2 == 0.0f) return;
  if (l1 == 0.0f) {
    m1 = m2;
    l1 = l2;
#pragma unroll
    for (int i = 0; i < N; ++i) a1[i] = a2[i];
    return;
  }
  const float m = fmaxf(m1, m2);
  const float c1 = expf(m1 - m), c2 = expf(m2 - m);
  l1 = l1 * c1 + l2 * c2;
#pragma unroll
  for (int i = 0; i < N; ++i) a1[i] = a1[i] * c1 + a2[i] * c2;
  m1 = m;
}

template <int HD, int G>
__global__ void __launch_bounds__(kWarps * 32) k_attention(const AttnParams p) {
  constexpr int LPT = HD / 8;    // lanes per token
  constexpr int TPW = 32 / LPT;  // tokens per warp step
  constexpr int PSZ = G * (HD + 2);
  __shared__ float sm_part[kWarps][PSZ];
  __shared__ int s_last;

  const int split = blockIdx.x, g = blockIdx.y, z = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int sub = lane / LPT, dl = lane % LPT;
  const int hkv = p.n_kv_heads;

  grid_dep_wait();
  grid_dep_launch();
  const int count = p.list ? ld_volatile_i32(p.list) : p.m_direct;
  if (z >= count) return;
  const int seq = p.list ? p.list[1 + z] : z;
  const int ctx = p.pos[seq] + 1;
  const int per = (ctx + p.nsplit - 1) / p.nsplit;
  const int t0 = split * per;
  const int t1 = min(ctx, t0 + per);

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
  float mrun[G], lrun[G], acc[G][8];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    mrun[h] = -INFINITY;
    lrun[h] = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[h][i] = 0.0f;
  }

  const int32_t* bt = p.block_table + (size_t)seq * p.bt_stride;
  constexpr int kStep = kWarps * TPW;  // tokens per CTA step
  for (int base = t0 + warp * TPW; base < t1; base += kStep * kUnroll) {
    uint4 kr[kUnroll], vr[kUnroll];
    bool valid[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int t = base + u * kStep + sub;
      valid[u] = t < t1;
      if (valid[u]) {
        const int block = bt[t >> 4];
        const size_t off = ((((size_t)block * hkv + g) * 16) + (t & 15)) * HD + dl * 8;
        kr[u] = ldg_nc_v4(p.kc + off);
        vr[u] = ldg_nc_v4(p.vc + off);
      } else {
        kr[u] = make_uint4(0, 0, 0, 0);
        vr[u] = kr[u];
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      float kf[8], vf[8];
      to_float8(kr[u], kf);
      to_float8(vr[u], vf);
#pragma unroll
      for (int h = 0; h < G; ++h) {
        float s = 0.0f;
#pragma unroll
        for (int i = 0; i < 8; ++i) s = fmaf(q[h][i], kf[i], s);
#pragma unroll
        for (int o = LPT / 2; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        if (valid[u]) {
          const float mn = fmaxf(mrun[h], s);
          const float c = expf(mrun[h] - mn);
          const float e = expf(s - mn);
          lrun[h] = lrun[h] * c + e;
#pragma unroll
          for (int i = 0; i < 8; ++i) acc[h][i] = fmaf(acc[h][i], c, e * vf[i]);
          mrun[h] = mn;
        }
      }
    }
  }

  // merge the token groups of this warp (lanes with the same dims)
#pragma unroll
  for (int o = LPT; o < 32; o <<= 1) {
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const float m2 = __shfl_xor_sync(0xffffffffu, mrun[h], o);
      const float l2 = __shfl_xor_sync(0xffffffffu, lrun[h], o);
      float a2[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) a2[i] = __shfl_xor_sync(0xffffffffu, acc[h][i], o);
      merge_state<8>(mrun[h], lrun[h], acc[h], m2, l2, a2);
    }
  }
  if (sub == 0) {
#pragma unroll
    for (int h = 0; h < G; ++h) {
      float* dst = sm_part[warp] + h * (HD + 2);
#pragma unroll
      for (int i = 0; i < 8; ++i) dst[dl * 8 + i] = acc[h][i];
      if (dl == 0) {
        dst[HD] = mrun[h];
        dst[HD + 1] = lrun[h];
      }
    }
  }
  __syncthreads();

  // CTA partial: merge the warps (thread i handles head i / HD, dim i % HD)
  float* part = p.part + (((size_t)z * hkv + g) * p.nsplit + split) * PSZ;
  for (int idx = tid; idx < G * HD; idx += kWarps * 32) {
    const int h = idx / HD, dd = idx % HD;
    float m = -INFINITY, l = 0.0f, a = 0.0f;
    for (int w = 0; w < kWarps; ++w) {
      const float* src = sm_part[w] + h * (HD + 2);
      float a2 = src[dd];
      merge_state<1>(m, l, &a, src[HD], src[HD + 1], &a2);
    }
    part[h * (HD + 2) + dd] = a;
    if (dd == 0) {
      part[h * (HD + 2) + HD] = m;
      part[h * (HD + 2) + HD + 1] = l;
    }
  }
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    const int old = atomicAdd(p.counters + (size_t)z * hkv + g, 1);
    s_last = (old == p.nsplit - 1);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  // last CTA of this (sequence, kv head): merge all splits
  const float* parts = p.part + (((size_t)z * hkv + g) * p.nsplit) * PSZ;
  for (int idx = tid; idx < G * HD; idx += kWarps * 32) {
    const int h = idx / HD, dd = idx % HD;
    float m = -INFINITY, l = 0.0f, a = 0.0f;
    for (int s = 0; s < p.nsplit; ++s) {
      const float* src = parts + (size_t)s * PSZ + h * (HD + 2);
      float a2 = __ldcg(src + dd);
      merge_state<1>(m, l, &a, __ldcg(src + HD), __ldcg(src + HD + 1), &a2);
    }
    const float o = a / l;
    const int col = (g * G + h) * HD + dd;
    if (p.o_f32) p.o_f32[(size_t)seq * p.o_stride + col] = o;
    if (p.oh) p.oh[(size_t)seq * p.o_stride + xh_slot(col)] = float_to_half_bits(o);
  }
  if (tid == 0) p.counters[(size_t)z * hkv + g] = 0;
}

template <int HD, int G>
cudaError_t launch_t(const AttnParams& p, int batch_slots, bool pdl, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.nsplit, p.n_kv_heads, batch_slots);
  cfg.blockDim = dim3(kWarps * 32);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, k_attention<HD, G>, p);
}

}  // namespace

size_t attention_part_floats(int batch_slots, int n_heads, int n_kv_heads, int head_dim, int nsplit) {
  const int G = n_heads / n_kv_heads;
  return (size_t)batch_slots * n_kv_heads * nsplit * G * (head_dim + 2);
}

int attention_nsplit(int batch, int n_kv_heads, int num_sms) {
  int s = (4 * num_sms + n_kv_heads * batch - 1) / (n_kv_heads * batch);
  if (s < 1) s = 1;
  if (s > 128) s = 128;
  return s;
}

cudaError_t launch_attention(const AttnParams& p, int batch_slots, bool pdl, cudaStream_t st) {
  const int G = p.n_heads / p.n_kv_heads;
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
