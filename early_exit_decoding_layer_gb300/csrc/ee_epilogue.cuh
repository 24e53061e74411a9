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

// Per-sequence values an epilogue needs: the position of the step's token,
// the cache block holding it (QKV), and whether per-layer debug copies of the
// residual stream are on (RESID).
struct EpiSeq {
  int seq, pos, block;
  bool dbg;
};

EE_DEV EpiSeq epi_seq(const LinearParams& p, int seq) {
  EpiSeq e;
  e.seq = seq;
  e.pos = e.block = 0;
  if (p.epi == EPI_QKV) {
    e.pos = p.pos[seq];
    e.block = p.block_table[(size_t)seq * p.bt_stride + (e.pos >> 4)];
  }
  e.dbg = p.epi == EPI_RESID && p.hdbg != nullptr && *p.dbg_flag;
  return e;
}

EE_DEV uint16_t* kv_slot_at(uint16_t* cache, const LinearParams& p, int block, int pos, int head) {
  return cache + ((((size_t)block * p.n_kv_heads + head) * 16) + (pos & 15)) * p.head_dim;
}

// Epilogue of one row pair (ra, ra+1) for one sequence.
template <int EPI>
EE_DEV void epi_pair_at(const LinearParams& p, const EpiSeq& e, int ra, float ya, float yb) {
  const int seq = e.seq;
  if constexpr (EPI == EPI_F32) {
    float* o = p.out_f32 + (size_t)seq * p.out_stride + ra;
    o[0] = ya;
    o[1] = yb;
  } else if constexpr (EPI == EPI_QKV) {
    const int hd = p.head_dim;
    const int dq = p.n_heads * hd, dk = p.n_kv_heads * hd;
    if (ra < dq + dk) {
      // rows (ra, ra+1) hold head dims (i, i + hd/2): rotate-half RoPE
      const bool isq = ra < dq;
      const int rr = isq ? ra : ra - dq;
      const int head = rr / hd, i = (rr % hd) >> 1;
      const float2 cs = p.rope[(size_t)e.pos * (hd >> 1) + i];
      const float o1 = ya * cs.x - yb * cs.y;
      const float o2 = yb * cs.x + ya * cs.y;
      if (isq) {
        float* q = p.q_out + (size_t)seq * dq + head * hd;
        q[i] = o1;
        q[i + (hd >> 1)] = o2;
      } else {
        uint16_t* k = kv_slot_at(p.kc, p, e.block, e.pos, head);
        k[i] = float_to_half_bits(o1);
        k[i + (hd >> 1)] = float_to_half_bits(o2);
      }
    } else {
      const int rr = ra - dq - dk;
      const int head = rr / hd, i = rr % hd;
      uint16_t* v = kv_slot_at(p.vc, p, e.block, e.pos, head);
      const uint32_t packed =
          uint32_t(float_to_half_bits(ya)) | (uint32_t(float_to_half_bits(yb)) << 16);
      *reinterpret_cast<uint32_t*>(v + i) = packed;
    }
  } else if constexpr (EPI == EPI_RESID) {
    float* hp = p.h + (size_t)seq * p.h_stride + ra;
    const float2 old = *reinterpret_cast<float2*>(hp);
    const float2 nw = make_float2(old.x + ya, old.y + yb);
    *reinterpret_cast<float2*>(hp) = nw;
    if (e.dbg) *reinterpret_cast<float2*>(p.hdbg + (size_t)seq * p.h_stride + ra) = nw;
    if (p.hsave) *reinterpret_cast<float2*>(p.hsave + (size_t)seq * p.h_stride + ra) = nw;
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

template <int EPI>
EE_DEV void epi_pair(const LinearParams& p, int seq, int ra, float ya, float yb) {
  epi_pair_at<EPI>(p, epi_seq(p, seq), ra, ya, yb);
}

}  // namespace ee
