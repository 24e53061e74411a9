// Per-row-pair epilogues of the projections, shared by the GEMV and the
// tensor-core GEMM: RoPE and the paged K/V write after QKV, the residual add
// after O and down, SwiGLU after gate/up, fp16 output of the exit-head
// transform, and plain fp32 output.  Activations written for a following
// projection are fp16 in pair order (see xh_slot).
#pragma once

#include <math.h>

#include "ee_common.cuh"
#include "ee_kernels.cuh"

namespace ee {

EE_DEV uint16_t* kv_slot(uint16_t* cache, const LinearParams& p, int seq, int pos, int head) {
  const int block = p.block_table[(size_t)seq * p.bt_stride + (pos >> 4)];
  return cache + ((((size_t)block * p.n_kv_heads + head) * 16) + (pos & 15)) * p.head_dim;
}

// Epilogue of one row pair (ra, ra+1) for one sequence.
template <int EPI>
EE_DEV void epi_pair(const LinearParams& p, int seq, int ra, float ya, float yb) {
  if constexpr (EPI == EPI_F32) {
    float* o = p.out_f32 + (size_t)seq * p.out_stride + ra;
    o[0] = ya;
    o[1] = yb;
  } else if constexpr (EPI == EPI_QKV) {
    const int hd = p.head_dim;
    const int dq = p.n_heads * hd, dk = p.n_kv_heads * hd;
    const int pos = p.pos[seq];
    if (ra < dq + dk) {
      // rows (ra, ra+1) hold head dims (i, i + hd/2): rotate-half RoPE
      const bool isq = ra < dq;
      const int rr = isq ? ra : ra - dq;
      const int head = rr / hd, i = (rr % hd) >> 1;
      const float2 cs = p.rope[(size_t)pos * (hd >> 1) + i];
      const float o1 = ya * cs.x - yb * cs.y;
      const float o2 = yb * cs.x + ya * cs.y;
      if (isq) {
        float* q = p.q_out + (size_t)seq * dq + head * hd;
        q[i] = o1;
        q[i + (hd >> 1)] = o2;
      } else {
        uint16_t* k = kv_slot(p.kc, p, seq, pos, head);
        k[i] = float_to_half_bits(o1);
        k[i + (hd >> 1)] = float_to_half_bits(o2);
      }
    } else {
      const int rr = ra - dq - dk;
      const int head = rr / hd, i = rr % hd;
      uint16_t* v = kv_slot(p.vc, p, seq, pos, head);
      const uint32_t packed =
          uint32_t(float_to_half_bits(ya)) | (uint32_t(float_to_half_bits(yb)) << 16);
      *reinterpret_cast<uint32_t*>(v + i) = packed;
    }
  } else if constexpr (EPI == EPI_RESID) {
    float* hp = p.h + (size_t)seq * p.h_stride + ra;
    const float2 old = *reinterpret_cast<float2*>(hp);
    const float2 nw = make_float2(old.x + ya, old.y + yb);
    *reinterpret_cast<float2*>(hp) = nw;
    if (p.hdbg != nullptr && *p.dbg_flag)
      *reinterpret_cast<float2*>(p.hdbg + (size_t)seq * p.h_stride + ra) = nw;
  } else if constexpr (EPI == EPI_SWIGLU) {
    const int i = ra >> 1;
    const float a = ya / (1.0f + expf(-ya)) * yb;
    p.xh_out[(size_t)seq * p.xo_stride + xh_slot(i)] = float_to_half_bits(a);
  } else if constexpr (EPI == EPI_X) {
    uint16_t* ho = p.xh_out + (size_t)seq * p.xo_stride;
    ho[xh_slot(ra)] = float_to_half_bits(ya);
    ho[xh_slot(ra + 1)] = float_to_half_bits(yb);
  }
}

}  // namespace ee
