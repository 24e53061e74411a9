// Skinny GEMV / GEMM for decode: Y[m, n] = sum_k X[m, k] W[n, k] for the few
// sequences of a step, with the weights streamed once from HBM.  Activations
// are fp16 (the A16 of W4A16), accumulation fp32.
//
// One launch serves both sub-batches of a layer: the rows still on the bf16
// backbone ("full" list) read the bf16 matrix, the rows that exited read the
// W4A16 copy ("exit" list: packed two's-complement nibbles, one bf16 scale per
// group of 128 input columns, dequantised in registers and never written
// back).  An empty list reads no byte of its matrix.
//
// Data flow per CTA (persistent, one per SM): warp 8 is a producer whose lane
// 0 streams the CTA's contiguous row range through a 6-stage shared-memory
// ring with bulk asynchronous copies (cp.async.bulk, completion counted on
// mbarriers, L2 evict-first); warps 0-7 consume.  A stage holds 16 rows x
// 1 KB (512 bf16 columns, or 2048 int4 columns plus their 16 scales).  Warp w
// owns rows (2w, 2w+1) of each 16-row tile, so the pairs that RoPE and SwiGLU
// combine are reduced by the same warp.  Activations come from L1/L2 (they are
// a few KB per sequence) in fp16, permuted within runs of 8 so that one
// 16-byte load yields the half2 pairs that match the nibble pairs of a packed
// int4 word (see xh_slot); the bf16 path reads the same layout.
//
// int4 dequantisation: a packed word holds columns c..c+7 in nibbles 0..7;
// (w ^ 0x88888888) turns two's complement into offset binary, then
// ((t >> 4j) & 0x000F000F) | 0x64006400 is the half2 (1024 + q_j + 8,
// 1024 + q_{j+4} + 8), and subtracting 1032 leaves (q_j, q_{j+4}) exactly.
// Products accumulate in fp16 over 32 columns, then in fp32 with the scale.
#include <math.h>

#include "ee_common.cuh"
#include "ee_kernels.cuh"

namespace ee {

namespace {

constexpr int kConsumerWarps = 8;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kTileRows = 2 * kConsumerWarps;
constexpr int kChunkBytes = 1024;
constexpr int kScaleBytes = 32;
constexpr int kStageBytes = kTileRows * (kChunkBytes + kScaleBytes);
constexpr int kMaxStages = 6;
constexpr int kMM = 8;  // sequences per pass over the weights
constexpr int kBfChunk = kChunkBytes / 2;  // bf16 columns per stage row
constexpr int kQChunk = kChunkBytes * 2;   // int4 columns per stage row

// Shared memory: a small header (barriers, lists, head statistics), then the
// activations of the step's rows when they are staged (XS mode), then the ring.
constexpr size_t kHeaderBytes = 1536;
constexpr size_t kXsMaxBytes = 48 * 1024;
constexpr size_t kSmemTarget = 112 * 1024;  // two CTAs per SM: the next kernel's CTA can prefetch
constexpr size_t kSmemMax = kHeaderBytes + kXsMaxBytes + size_t(kMaxStages) * kStageBytes;
static_assert((2 * kMaxStages + 1) * 8 + 2 * kListLen * 4 + kConsumerWarps * kMM * 3 * 4 <= kHeaderBytes,
              "header overflow");

EE_DEV __half2 u32_as_h2(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }

// 8 bf16 weights w0..w7 (natural order) times 8 fp16 activations given in
// pair order (x0,x4) (x1,x5) (x2,x6) (x3,x7), accumulated in fp32.
EE_DEV float dot8_bf16(const uint4& w, const uint4& x, float acc) {
  const float2 x04 = __half22float2(u32_as_h2(x.x)), x15 = __half22float2(u32_as_h2(x.y));
  const float2 x26 = __half22float2(u32_as_h2(x.z)), x37 = __half22float2(u32_as_h2(x.w));
  acc = fmaf(bf16_lo(w.x), x04.x, acc);
  acc = fmaf(bf16_hi(w.x), x15.x, acc);
  acc = fmaf(bf16_lo(w.y), x26.x, acc);
  acc = fmaf(bf16_hi(w.y), x37.x, acc);
  acc = fmaf(bf16_lo(w.z), x04.y, acc);
  acc = fmaf(bf16_hi(w.z), x15.y, acc);
  acc = fmaf(bf16_lo(w.w), x26.y, acc);
  acc = fmaf(bf16_hi(w.w), x37.y, acc);
  return acc;
}

// 8 int4 weights (one packed word) times 8 fp16 activations in pair order.
EE_DEV __half2 dot8_int4(uint32_t word, const uint4& x, __half2 acc) {
  const uint32_t t = word ^ 0x88888888u;
  const __half2 bias = __half2half2(__ushort_as_half((unsigned short)0x6408));  // 1032
  acc = __hfma2(__hsub2(u32_as_h2((t & 0x000F000Fu) | 0x64006400u), bias), u32_as_h2(x.x), acc);
  acc = __hfma2(__hsub2(u32_as_h2(((t >> 4) & 0x000F000Fu) | 0x64006400u), bias), u32_as_h2(x.y), acc);
  acc = __hfma2(__hsub2(u32_as_h2(((t >> 8) & 0x000F000Fu) | 0x64006400u), bias), u32_as_h2(x.z), acc);
  acc = __hfma2(__hsub2(u32_as_h2(((t >> 12) & 0x000F000Fu) | 0x64006400u), bias), u32_as_h2(x.w), acc);
  return acc;
}

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

// Online (max, sum of exp(z - max), argmax) statistics.
struct Stat {
  float mx, sum;
  int arg;
};
EE_DEV void stat_push(Stat& s, float z, int idx) {
  if (z > s.mx) {
    s.sum = s.sum * expf(s.mx - z) + 1.0f;
    s.mx = z;
    s.arg = idx;
  } else {
    s.sum += expf(z - s.mx);
    if (z == s.mx && idx < s.arg) s.arg = idx;
  }
}
EE_DEV Stat stat_merge(Stat a, Stat b) {
  if (b.sum == 0.0f) return a;
  if (a.sum == 0.0f) return b;
  Stat r;
  r.mx = fmaxf(a.mx, b.mx);
  r.sum = a.sum * expf(a.mx - r.mx) + b.sum * expf(b.mx - r.mx);
  r.arg = a.mx > b.mx ? a.arg : (b.mx > a.mx ? b.arg : min(a.arg, b.arg));
  return r;
}

EE_DEV void consumer_bar() { asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory"); }

// Iteration order shared by the producer and the consumers: phase (0 bf16
// rows, 1 int4 rows), pass over at most kMM sequences, 16-row tile of the
// CTA's rows, K chunk.  Each iteration fills one ring stage.
struct Plan {
  int r0, r1, ntiles, nc[2], passes[2];
  EE_DEV int rows(int t) const { return min(kTileRows, r1 - (r0 + t * kTileRows)); }
  EE_DEV uint32_t total() const {
    return (uint32_t)(passes[0] * ntiles * nc[0] + passes[1] * ntiles * nc[1]);
  }
};

// Issues the bulk copies of one ring stage (weights and, for int4, scales).
EE_DEV void issue_stage(const LinearParams& p, const Plan& pl, int phase, int t, int c, uint8_t* sbase,
                        uint64_t* bar, uint64_t pol) {
  const int tr0 = pl.r0 + t * kTileRows;
  const int rows = pl.rows(t);
  if (phase == 0) {
    const int ce = min(kBfChunk, p.K - c * kBfChunk);
    const uint32_t cb = ce * 2;
    mbar_arrive_expect_tx(bar, rows * cb);
    for (int r = 0; r < rows; ++r)
      bulk_g2s(sbase + r * kChunkBytes, p.w + (size_t)(tr0 + r) * p.K + c * kBfChunk, cb, bar, pol);
  } else {
    const int ce = min(kQChunk, p.K - c * kQChunk);
    const uint32_t cb = ce / 2;
    const int ng = (ce + EE_QUANT_GROUP - 1) / EE_QUANT_GROUP;
    const uint32_t sb = ((ng * 2 + 15) / 16) * 16;
    mbar_arrive_expect_tx(bar, rows * (cb + sb));
    for (int r = 0; r < rows; ++r) {
      bulk_g2s(sbase + r * kChunkBytes, p.wq + (size_t)(tr0 + r) * (p.K / 2) + (size_t)c * (kQChunk / 2),
               cb, bar, pol);
      bulk_g2s(sbase + kTileRows * kChunkBytes + r * kScaleBytes,
               p.ws + (size_t)(tr0 + r) * p.sstride + c * (kQChunk / EE_QUANT_GROUP), sb, bar, pol);
    }
  }
}

// XS = true: the activations of all the step's rows (at most p.xs_rows
// sequences) are bulk-copied into shared memory once, after the dependency
// wait, while the weight stream already runs; XS = false: activations are
// read from global memory (L1/L2) at every stage.
template <int EPI, bool XS>
__global__ void __launch_bounds__(kThreads, 1) k_linear(const LinearParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty = full + kMaxStages;
  uint64_t* xbar = empty + kMaxStages;
  int32_t* lf = reinterpret_cast<int32_t*>(smem + 128);
  int32_t* le = lf + kListLen;
  float* hst = reinterpret_cast<float*>(smem + 128 + 2 * kListLen * 4 + 8);
  uint8_t* xs = smem + kHeaderBytes;
  uint8_t* ring = xs + (XS ? (size_t)p.xs_rows * p.K * 2 : 0);
  const int nst = p.nstages;
  __shared__ int s_last;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < nst; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
    mbar_init(xbar, 1);
    fence_mbar_init();
  }
  // Lists were written at least two launches back (see grid_dep_wait), so
  // they may be read before this grid's dependency wait.
  if (tid < kListLen) {
    lf[tid] = p.list_full ? ld_volatile_i32(p.list_full + tid) : (tid == 0 ? p.m_direct_full : tid - 1);
    le[tid] = p.list_exit ? ld_volatile_i32(p.list_exit + tid) : (tid == 0 ? p.m_direct_exit : tid - 1);
  }
  __syncthreads();

  const int nf = p.w ? min(lf[0], EE_MAX_BATCH) : 0;
  const int ne = p.wq ? min(le[0], EE_MAX_BATCH) : 0;
  const int nx = nf + ne;  // XS mode: rows staged (full rows first, then exit rows)
  Plan pl;
  {
    const int npairs = p.N >> 1;
    pl.r0 = 2 * (int)(((long long)blockIdx.x * npairs) / gridDim.x);
    pl.r1 = 2 * (int)(((long long)(blockIdx.x + 1) * npairs) / gridDim.x);
    pl.ntiles = (pl.r1 - pl.r0 + kTileRows - 1) / kTileRows;
    pl.nc[0] = (p.K + kBfChunk - 1) / kBfChunk;
    pl.nc[1] = (p.K + kQChunk - 1) / kQChunk;
    pl.passes[0] = (nf + kMM - 1) / kMM;
    pl.passes[1] = (ne + kMM - 1) / kMM;
  }

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol = l2_evict_first_policy();
      const uint32_t total = pl.total();
      const uint32_t prefill = total < (uint32_t)nst ? total : (uint32_t)nst;
      bool xdone = !XS;
      auto stage_x = [&]() {
        // activations are written by the previous kernel: copy them after the wait
        grid_dep_wait();
        if (nx > 0) {
          const uint32_t rb = (uint32_t)p.K * 2;
          mbar_arrive_expect_tx(xbar, nx * rb);
          for (int m = 0; m < nx; ++m) {
            const int seq = m < nf ? lf[1 + m] : le[1 + m - nf];
            bulk_g2s(xs + (size_t)m * rb, p.xh + (size_t)seq * p.x_stride, rb, xbar, pol);
          }
        }
        xdone = true;
      };
      uint32_t it = 0;
      bool ok = true;
      for (int phase = 0; phase < 2 && ok; ++phase) {
        for (int pass = 0; pass < pl.passes[phase] && ok; ++pass) {
          for (int t = 0; t < pl.ntiles && ok; ++t) {
            for (int c = 0; c < pl.nc[phase]; ++c, ++it) {
              if (!xdone && it == prefill) stage_x();
              const int st = it % nst;
              const uint32_t n = it / nst;
              if (n > 0 && !mbar_wait_bounded(&empty[st], (n - 1) & 1, p.err, DERR_EMPTY_WAIT)) {
                ok = false;
                break;
              }
              issue_stage(p, pl, phase, t, c, ring + (size_t)st * kStageBytes, &full[st], pol);
            }
          }
        }
      }
      if (!xdone) stage_x();
      // every copy this thread issued lands before the CTA may exit
      const uint32_t j0 = it > (uint32_t)nst ? it - nst : 0;
      for (uint32_t j = j0; j < it; ++j)
        mbar_wait_bounded(&full[j % nst], (j / nst) & 1, p.err, DERR_DRAIN_WAIT);
      if (XS && nx > 0) mbar_wait_bounded(xbar, 0, p.err, DERR_DRAIN_WAIT);
    }
  } else {
    // ------------------------------------------------------------ consumers
    grid_dep_wait();
    grid_dep_launch();
    bool ok = true;
    if (XS && nx > 0) ok = mbar_wait_bounded(xbar, 0, p.err, DERR_FULL_WAIT);
    uint32_t it = 0;
    for (int phase = 0; phase < 2; ++phase) {
      const int nlist = phase == 0 ? nf : ne;
      const int32_t* lst = phase == 0 ? lf : le;
      const int nc = pl.nc[phase];
      const int xbase = phase == 0 ? 0 : nf;  // XS row of the phase's first sequence
      for (int pass = 0; pass < pl.passes[phase]; ++pass) {
        const int m0 = pass * kMM;
        const int mc = min(kMM, nlist - m0);
        int seqs[kMM];
        const uint16_t* xrow[kMM];
#pragma unroll
        for (int m = 0; m < kMM; ++m) {
          const int mm = min(m, mc - 1);
          seqs[m] = lst[1 + m0 + mm];
          xrow[m] = XS ? reinterpret_cast<const uint16_t*>(xs) + (size_t)(xbase + m0 + mm) * p.K
                       : p.xh + (size_t)seqs[m] * p.x_stride;
        }
        Stat stat = {-INFINITY, 0.0f, 0x7fffffff};
        for (int t = 0; t < pl.ntiles; ++t) {
          const int tr0 = pl.r0 + t * kTileRows;
          const bool have = 2 * warp < pl.rows(t);
          float acc0[kMM], acc1[kMM];
#pragma unroll
          for (int m = 0; m < kMM; ++m) acc0[m] = acc1[m] = 0.0f;
          for (int c = 0; c < nc; ++c, ++it) {
            const int st = it % nst;
            if (ok) ok = mbar_wait_bounded(&full[st], (it / nst) & 1, p.err, DERR_FULL_WAIT);
            if (ok && have) {
              const uint8_t* sa = ring + (size_t)st * kStageBytes + (2 * warp) * kChunkBytes;
              const uint8_t* sb = sa + kChunkBytes;
              if (phase == 0) {
                const int nvec = min(kBfChunk, p.K - c * kBfChunk) >> 3;
                for (int v = lane; v < nvec; v += 32) {
                  const uint4 wa = *reinterpret_cast<const uint4*>(sa + v * 16);
                  const uint4 wb = *reinterpret_cast<const uint4*>(sb + v * 16);
                  const int k0 = c * kBfChunk + v * 8;
#pragma unroll
                  for (int m = 0; m < kMM; ++m) {
                    if (m < mc) {
                      const uint4 xv = XS ? *reinterpret_cast<const uint4*>(xrow[m] + k0)
                                          : ldg_nc_v4(xrow[m] + k0);
                      acc0[m] = dot8_bf16(wa, xv, acc0[m]);
                      acc1[m] = dot8_bf16(wb, xv, acc1[m]);
                    }
                  }
                }
              } else {
                const int nvec = min(kQChunk, p.K - c * kQChunk) >> 5;
                const uint16_t* sca = reinterpret_cast<const uint16_t*>(
                    ring + (size_t)st * kStageBytes + kTileRows * kChunkBytes + (2 * warp) * kScaleBytes);
                const uint16_t* scb = sca + kScaleBytes / 2;
                for (int v = lane; v < nvec; v += 32) {
                  const uint4 qa = *reinterpret_cast<const uint4*>(sa + v * 16);
                  const uint4 qb = *reinterpret_cast<const uint4*>(sb + v * 16);
                  const float s_a = bf16_bits_to_float(sca[v >> 2]);
                  const float s_b = bf16_bits_to_float(scb[v >> 2]);
                  const int k0 = c * kQChunk + v * 32;
#pragma unroll
                  for (int m = 0; m < kMM; ++m) {
                    if (m < mc) {
                      const uint16_t* xp = xrow[m] + k0;
                      uint4 x0, x1, x2, x3;
                      if (XS) {
                        x0 = *reinterpret_cast<const uint4*>(xp);
                        x1 = *reinterpret_cast<const uint4*>(xp + 8);
                        x2 = *reinterpret_cast<const uint4*>(xp + 16);
                        x3 = *reinterpret_cast<const uint4*>(xp + 24);
                      } else {
                        x0 = ldg_nc_v4(xp);
                        x1 = ldg_nc_v4(xp + 8);
                        x2 = ldg_nc_v4(xp + 16);
                        x3 = ldg_nc_v4(xp + 24);
                      }
                      __half2 ha = __float2half2_rn(0.0f), hb = ha;
                      ha = dot8_int4(qa.x, x0, ha);
                      hb = dot8_int4(qb.x, x0, hb);
                      ha = dot8_int4(qa.y, x1, ha);
                      hb = dot8_int4(qb.y, x1, hb);
                      ha = dot8_int4(qa.z, x2, ha);
                      hb = dot8_int4(qb.z, x2, hb);
                      ha = dot8_int4(qa.w, x3, ha);
                      hb = dot8_int4(qb.w, x3, hb);
                      const float2 fa = __half22float2(ha), fb = __half22float2(hb);
                      acc0[m] = fmaf(s_a, fa.x + fa.y, acc0[m]);
                      acc1[m] = fmaf(s_b, fb.x + fb.y, acc1[m]);
                    }
                  }
                }
              }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[st]);
          }
          if (have) {
            const int ra = tr0 + 2 * warp;
#pragma unroll
            for (int m = 0; m < kMM; ++m) {
              if (m < mc) {
                const float ya = warp_sum(acc0[m]);
                const float yb = warp_sum(acc1[m]);
                if constexpr (EPI == EPI_HEAD) {
                  if (lane == m) {
                    stat_push(stat, ya, ra);
                    stat_push(stat, yb, ra + 1);
                  }
                } else {
                  if (lane == m) epi_pair<EPI>(p, seqs[m], ra, ya, yb);
                }
              }
            }
          }
        }
        if constexpr (EPI == EPI_HEAD) {
          // combine the 8 warps' statistics of this pass; one partial per CTA and row
          if (lane < kMM) {
            float* hs = hst + (warp * kMM + lane) * 3;
            hs[0] = stat.mx;
            hs[1] = stat.sum;
            hs[2] = __int_as_float(stat.arg);
          }
          consumer_bar();
          if (warp == 0 && lane < mc) {
            Stat s = {-INFINITY, 0.0f, 0x7fffffff};
            for (int w = 0; w < kConsumerWarps; ++w) {
              const float* hs = hst + (w * kMM + lane) * 3;
              s = stat_merge(s, Stat{hs[0], hs[1], __float_as_int(hs[2])});
            }
            float* dst = p.head_part + ((size_t)blockIdx.x * EE_MAX_BATCH + m0 + lane) * 4;
            dst[0] = s.mx;
            dst[1] = s.sum;
            dst[2] = __int_as_float(s.arg);
          }
          consumer_bar();
        }
      }
    }
  }

  if constexpr (EPI == EPI_HEAD) {
    // Last CTA to finish merges the per-CTA partials (no spin wait: a counter).
    __syncthreads();
    if (tid == 0) {
      __threadfence();
      const int old = atomicAdd(p.head_counter, 1);
      s_last = (old == (int)gridDim.x - 1);
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    float* res = hst;  // reuse: [m] (conf, argmax)
    const int nrows = nf;
    for (int m = warp; m < nrows; m += kConsumerWarps + 1) {
      Stat s = {-INFINITY, 0.0f, 0x7fffffff};
      for (int c = lane; c < (int)gridDim.x; c += 32) {
        const float* src = p.head_part + ((size_t)c * EE_MAX_BATCH + m) * 4;
        s = stat_merge(s, Stat{__ldcg(src), __ldcg(src + 1), __float_as_int(__ldcg(src + 2))});
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        Stat t;
        t.mx = __shfl_xor_sync(0xffffffffu, s.mx, o);
        t.sum = __shfl_xor_sync(0xffffffffu, s.sum, o);
        t.arg = __shfl_xor_sync(0xffffffffu, s.arg, o);
        s = stat_merge(s, t);
      }
      if (lane == 0) {
        res[2 * m] = 1.0f / s.sum;  // max softmax = exp(zmax - lse) = 1 / sum exp(z - zmax)
        res[2 * m + 1] = __int_as_float(s.arg);
      }
    }
    __syncthreads();
    if (tid == 0) {
      if (p.head_mode == HEAD_CONF_ARGMAX) {
        for (int m = 0; m < nrows; ++m) {
          p.conf_out[m] = res[2 * m];
          p.argmax_out[m] = __float_as_int(res[2 * m + 1]);
        }
      } else if (p.head_mode == HEAD_FINAL) {
        for (int m = 0; m < nrows; ++m) p.argmax_out[lf[1 + m]] = __float_as_int(res[2 * m + 1]);
      } else {  // HEAD_CHECKPOINT: decide, then rebuild the two sub-batch lists
        const float gamma = p.gamma[p.ckpt_index];
        int32_t nfull = 0, nexit = 0;
        int32_t newly[EE_MAX_BATCH];
        int nnew = 0;
        for (int m = 0; m < nrows; ++m) {
          const int seq = lf[1 + m];
          const float conf = res[2 * m];
          p.conf_out[seq * EE_MAX_CHECKPOINTS + p.ckpt_index] = conf;
          if (conf > gamma) {
            newly[nnew++] = seq;
            p.exit_layer[seq] = p.ckpt_layer;
          } else {
            p.lists->full[1 + nfull++] = seq;
          }
        }
        // exit list = merge of the previous exit list and the newly exited, by id
        const int nold = min(le[0], EE_MAX_BATCH);
        int a = 0, b = 0;
        while (a < nold || b < nnew) {
          const bool take_old = b >= nnew || (a < nold && le[1 + a] < newly[b]);
          p.lists->exitl[1 + nexit++] = take_old ? le[1 + a++] : newly[b++];
        }
        p.lists->full[0] = nfull;
        p.lists->exitl[0] = nexit;
      }
      __threadfence();
      *p.head_counter = 0;
    }
  }
}

template <int EPI>
cudaError_t set_smem_attr() {
  cudaError_t e = cudaFuncSetAttribute(k_linear<EPI, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)kSmemMax);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(k_linear<EPI, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemMax);
}

template <int EPI>
cudaError_t launch_one(const LinearParams& p, int grid, bool pdl, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kHeaderBytes + (p.xs_rows > 0 ? (size_t)p.xs_rows * p.K * 2 : 0) +
                         (size_t)p.nstages * kStageBytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  if (p.xs_rows > 0) return cudaLaunchKernelEx(&cfg, k_linear<EPI, true>, p);
  return cudaLaunchKernelEx(&cfg, k_linear<EPI, false>, p);
}

}  // namespace

size_t linear_smem_bytes() { return kSmemMax; }

void linear_plan_smem(LinearParams& p, int max_rows) {
  const size_t xb = (size_t)max_rows * p.K * 2;
  int nst = kMaxStages;
  bool xs = max_rows <= kMM && xb <= kXsMaxBytes;
  if (xs) {
    const size_t room = kSmemTarget - kHeaderBytes - xb;
    nst = (int)(room / kStageBytes);
    if (nst > kMaxStages) nst = kMaxStages;
    if (nst < 4) xs = false;
  }
  if (!xs) nst = kMaxStages;
  p.xs_rows = xs ? max_rows : 0;
  p.nstages = nst;
}

cudaError_t linear_prepare() {
  cudaError_t e;
  if ((e = set_smem_attr<EPI_F32>()) != cudaSuccess) return e;
  if ((e = set_smem_attr<EPI_QKV>()) != cudaSuccess) return e;
  if ((e = set_smem_attr<EPI_RESID>()) != cudaSuccess) return e;
  if ((e = set_smem_attr<EPI_SWIGLU>()) != cudaSuccess) return e;
  if ((e = set_smem_attr<EPI_X>()) != cudaSuccess) return e;
  return set_smem_attr<EPI_HEAD>();
}

int linear_grid(int N, int num_sms) {
  const int tiles = (N + kTileRows - 1) / kTileRows;
  return tiles < num_sms ? (tiles > 0 ? tiles : 1) : num_sms;
}

cudaError_t launch_linear(const LinearParams& p, int grid, bool pdl, cudaStream_t st) {
  switch (p.epi) {
    case EPI_F32: return launch_one<EPI_F32>(p, grid, pdl, st);
    case EPI_QKV: return launch_one<EPI_QKV>(p, grid, pdl, st);
    case EPI_RESID: return launch_one<EPI_RESID>(p, grid, pdl, st);
    case EPI_SWIGLU: return launch_one<EPI_SWIGLU>(p, grid, pdl, st);
    case EPI_X: return launch_one<EPI_X>(p, grid, pdl, st);
    case EPI_HEAD: return launch_one<EPI_HEAD>(p, grid, pdl, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace ee
