// Device code of the split-K paged decode attention (see k_attention.cu for
// the design): one work item = one split of one kv head of one sequence, run
// by a whole CTA.
#pragma once

#include <math.h>

#include "ee_common.cuh"
#include "ee_kernels.cuh"

namespace ee {
namespace {


constexpr int kAttnWarps = 8;
constexpr int kThreadsA = kAttnWarps * 32;
constexpr int kKvSmem = 40 * 1024;  // K + V tiles of one CTA
constexpr int kMaxSplit = 256;

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

// Shared-memory state of one attention work item (besides the K/V tiles).
template <int HD, int G>
struct AttnShared {
  uint64_t bar;
  int s_last;
  float S[G][blocks_per_cta<HD>() * 16];  // scores, then exp(s - m)
  float hm[G], hl[G];
};

// One work item: split `split` of kv head `g` of sequence slot `z`, run by a
// whole CTA of kThreadsA threads.  smem: the K/V tile space (kKvSmem bytes).
template <int HD, int G>
EE_DEV void attention_item(const AttnParams& p, int split, int g, int z, uint8_t* smem, AttnShared<HD, G>& sh) {
  constexpr int LPT = HD / 8;    // lanes per token
  constexpr int TPW = 32 / LPT;  // tokens per warp step
  constexpr int TILE = 16 * HD;  // elements of one (block, kv head) tile
  constexpr int BPC = blocks_per_cta<HD>();
  constexpr int PSZ = G * HD + ((2 * G + 3) / 4) * 4;  // partial: acc [G][HD], m [G], l [G] (16-B rows)
  uint16_t* Ks = reinterpret_cast<uint16_t*>(smem);
  uint16_t* Vs = Ks + BPC * TILE;
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
    mbar_init(&sh.bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  const uint64_t pol = l2_evict_first_policy();
  if (warp == 0 && have) {
    // one lane per block: the block-table reads and the copies go out in parallel
    if (lane == 0) mbar_arrive_expect_tx(&sh.bar, (uint32_t)(b1 - b0) * 2 * TILE * 2);
    __syncwarp();
    const int b = b0 + lane;
    if (b < b1 && b != last) {
      const size_t off = ((size_t)ld_volatile_i32(bt + b) * hkv + g) * TILE;
      bulk_g2s(Ks + lane * TILE, p.kc + off, TILE * 2, &sh.bar, pol);
      bulk_g2s(Vs + lane * TILE, p.vc + off, TILE * 2, &sh.bar, pol);
    }
  }
  grid_dep_wait();
  grid_dep_launch();
  if (tid == 0 && have && last >= b0 && last < b1) {
    const size_t off = ((size_t)ld_volatile_i32(bt + last) * hkv + g) * TILE;
    bulk_g2s(Ks + (last - b0) * TILE, p.kc + off, TILE * 2, &sh.bar, pol);
    bulk_g2s(Vs + (last - b0) * TILE, p.vc + off, TILE * 2, &sh.bar, pol);
  }
  auto& S = sh.S;
  auto& hm = sh.hm;
  auto& hl = sh.hl;
  float* wpart = reinterpret_cast<float*>(smem);  // [warp][PSZ], after the tiles are consumed

  // the queries (written by the previous kernel) load while the K/V copies land
  const float scale = rsqrtf((float)HD);
  float q[G][8];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    const float4* qp = reinterpret_cast<const float4*>(p.q + (size_t)seq * p.q_stride + (g * G + h) * HD + dl * 8);
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
  bool ok = true;
  if (have) ok = mbar_wait_bounded(&sh.bar, 0, p.err, DERR_FULL_WAIT);
  if (have && !ok) mbar_wait_bounded(&sh.bar, 0, p.err, DERR_DRAIN_WAIT);  // copies land before reuse
  const bool run = have && ok;
  const int t0 = b0 * 16, n = run ? min(ctx, b1 * 16) - t0 : 0;  // tokens of this CTA

  // (1) scores
  if (n > 0) {
    for (int base = warp * TPW; base < n; base += kAttnWarps * TPW) {
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
  for (int base = warp * TPW; base < n; base += kAttnWarps * TPW) {
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
    for (int w = 0; w < kAttnWarps; ++w) a += wpart[w * PSZ + idx];
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
    sh.s_last = (old == nact - 1);
  }
  __syncthreads();
  if (!sh.s_last) return;
  __threadfence();

  // last CTA of this (sequence, kv head): merge the splits.  One pass reads
  // every split's (m, l) from L2 into shared memory (warp w takes heads w,
  // w+8, ...): M = max m, weights exp(m - M), L = sum weight * l.  Then all
  // threads accumulate the outputs: thread (item i4, part) sums the splits
  // s = part, part + parts, ... of its 4 output values, eight loads in
  // flight, and the parts are added in part order (fixed: results do not
  // depend on timing).
  const float* parts = p.part + ((size_t)z * hkv + g) * p.nsplit * PSZ;
  float4* comb = reinterpret_cast<float4*>(smem);                  // [kThreadsA] (16-byte aligned)
  float* wts = reinterpret_cast<float*>(smem + kThreadsA * 16);  // [split][G]
  float* inv_l = wts + kMaxSplit * G;                            // [G]
  float* msm = inv_l + G;                                        // [split][G]
  float* lsm = msm + kMaxSplit * G;                              // [split][G]
  for (int h = warp; h < G; h += kAttnWarps) {
    float mloc = -INFINITY;
    for (int s = lane; s < nact; s += 32) {
      const float m = __ldcg(parts + (size_t)s * PSZ + G * HD + h);
      const float l = __ldcg(parts + (size_t)s * PSZ + G * HD + G + h);
      msm[s * G + h] = m;
      lsm[s * G + h] = l;
      if (l > 0.0f) mloc = fmaxf(mloc, m);
    }
    const float M = warp_max(mloc);
    float lsum = 0.0f;
    for (int s = lane; s < nact; s += 32) {
      const float l = lsm[s * G + h];
      const float w = l > 0.0f ? expf(msm[s * G + h] - M) : 0.0f;
      wts[s * G + h] = w;
      lsum += w * l;
    }
    lsum = warp_sum(lsum);
    if (lane == 0) inv_l[h] = 1.0f / lsum;
  }
  __syncthreads();
  constexpr int NI = G * HD / 4;                                 // float4 output items
  constexpr int NPART = NI >= kThreadsA ? 1 : kThreadsA / NI;    // threads per item
  static_assert(NI % kThreadsA == 0 || kThreadsA % NI == 0, "item split");
  for (int base = 0; base < NI; base += kThreadsA / NPART) {
    const int i4 = base + tid % (kThreadsA / NPART), part = tid / (kThreadsA / NPART);
    const int h = (i4 * 4) / HD;
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
    if (i4 < NI) {
      int s = part;
      for (; s + 7 * NPART < nact; s += 8 * NPART) {
        float4 v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u)
          v[u] = __ldcg(reinterpret_cast<const float4*>(parts + (size_t)(s + u * NPART) * PSZ) + i4);
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const float w = wts[(s + u * NPART) * G + h];
          o.x = fmaf(w, v[u].x, o.x);
          o.y = fmaf(w, v[u].y, o.y);
          o.z = fmaf(w, v[u].z, o.z);
          o.w = fmaf(w, v[u].w, o.w);
        }
      }
      for (; s < nact; s += NPART) {
        const float4 v = __ldcg(reinterpret_cast<const float4*>(parts + (size_t)s * PSZ) + i4);
        const float w = wts[s * G + h];
        o.x = fmaf(w, v.x, o.x);
        o.y = fmaf(w, v.y, o.y);
        o.z = fmaf(w, v.z, o.z);
        o.w = fmaf(w, v.w, o.w);
      }
    }
    if (NPART > 1) {
      comb[tid] = o;
      __syncthreads();
      if (part == 0 && i4 < NI) {
        for (int q = 1; q < NPART; ++q) {
          const float4 t = comb[q * (kThreadsA / NPART) + tid];
          o.x += t.x;
          o.y += t.y;
          o.z += t.z;
          o.w += t.w;
        }
      }
      __syncthreads();
    }
    if (part == 0 && i4 < NI) {
      const float il = inv_l[h];
      const float ov[4] = {o.x * il, o.y * il, o.z * il, o.w * il};
      const int col0 = g * G * HD + i4 * 4;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (p.o_f32) p.o_f32[(size_t)seq * p.o_stride + col0 + u] = ov[u];
        if (p.oh) p.oh[(size_t)seq * p.o_stride + xh_slot(col0 + u)] = float_to_half_bits(ov[u]);
      }
    }
  }
  if (tid == 0) p.counters[(size_t)z * hkv + g] = 0;
}

}  // namespace
}  // namespace ee
