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
// Data flow: one CTA of 8 warps per SM owns a balanced, pair-aligned range of
// output rows; warp w owns the CTA's rows w, w+8, ... and streams each of them
// with coalesced 16-byte loads (a warp reads 512 contiguous bytes per load
// instruction) straight into registers, double-buffered in batches of 8
// vectors per lane so that 16 loads per lane (64 KB per SM) are in flight --
// what the HBM needs to run at peak.  The first batch is requested before the
// grid dependency wait (weights never change), so the stream starts while the
// previous kernel drains; the activations of the step's rows (fp16, a few KB
// per sequence), written by that kernel, are copied into shared memory after
// the wait.  A warp finishes each of its rows alone (one warp reduction), so
// results do not depend on timing.  The epilogue (RoPE + KV write, SwiGLU,
// residual add, head statistics) runs once over the CTA's rows.
//
// Activations are stored in "pair order" (within each run of 8 columns:
// 0,4,1,5,2,6,3,7, see xh_slot) so that one 16-byte load yields the half2
// pairs that match the nibble pairs of a packed int4 word.
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

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kBatch = 8;  // 16-byte vectors per lane per batch
constexpr int kMM = 8;     // sequences per pass over the weights

// Shared memory: header (lists, head statistics), the staged activations
// (XS mode), the per-row sums [rows][mcap], then per-warp copy rings of
// nslots batches (kBatch vectors of 16 bytes per lane, plus 16 bytes of int4
// scales per vector slot).
constexpr size_t kHeaderBytes = 1536;
constexpr size_t kXsMaxBytes = 64 * 1024;
constexpr size_t kSmemMax = 227 * 1024 - 1024;
constexpr size_t kSmemPair = 112 * 1024;  // two CTAs per SM
constexpr int kMaxSlots = 4;
constexpr size_t kSlotBytes = (size_t)kBatch * 512 + kBatch * 16;  // one warp, one batch
static_assert(2 * kListLen * 4 + 16 + kWarps * kMM * 3 * 4 <= kHeaderBytes, "header overflow");

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

EE_DEV uint16_t ldg_u16(const uint16_t* p) {
  uint16_t v;
  asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}

struct Plan {
  int r0, r1, mcap;
  int passes[2];
};

// Copies one batch of this warp's stream into its ring slot: positions
// base + 32 j + lane (j < kBatch) of the concatenation of the warp's rows, nv
// vectors each (nv % 32 == 0, so the 32 positions of one j lie in one row).
// For int4 with K % 1024 == 0, lane j also copies the 8 scales of slot j.
#ifdef EE_CHECKED
// Debug builds: every asynchronous access is checked; a bad one is recorded
// (site code in err[0], value in err[1..2]) and skipped.
EE_DEV uint32_t dyn_smem_size() {
  uint32_t v;
  asm volatile("mov.u32 %0, %dynamic_smem_size;" : "=r"(v));
  return v;
}
extern __shared__ __align__(1024) uint8_t smem_base_sym[];
EE_DEV bool check_ok(int32_t* err, bool ok, int site, long long v1, long long v2) {
  if (!ok && err && atomicCAS(err, 0, site) == 0) {
    err[1] = (int32_t)v1;
    err[2] = (int32_t)v2;
  }
  return ok;
}
#define EE_CHECK(err, cond, site, v1, v2) check_ok((err), (cond), (site), (long long)(v1), (long long)(v2))
#else
#define EE_CHECK(err, cond, site, v1, v2) true
#endif

template <int PH>
EE_DEV void issue_batch(const LinearParams& p, const Plan& pl, int warp, int lane, int nv, int total,
                        int base, uint8_t* slot, bool sc_async, uint64_t pol) {
  const size_t rstride = PH == 0 ? (size_t)p.K * 2 : (size_t)p.K / 2;
  const uint8_t* wbase = PH == 0 ? reinterpret_cast<const uint8_t*>(p.w) : p.wq;
  int ri = base / nv;
  int v0 = base - ri * nv;
#pragma unroll
  for (int j = 0; j < kBatch; ++j) {
    if (base + 32 * j < total) {
      const int row = pl.r0 + warp + kWarps * ri;
      uint8_t* dst = slot + j * 512 + lane * 16;
      const uint8_t* src = wbase + (size_t)row * rstride + (size_t)(v0 + lane) * 16;
#ifdef EE_CHECKED
      const uint32_t so = smem_addr(dst) - smem_addr(smem_base_sym);
      const bool okd = EE_CHECK(p.err, so % 16 == 0 && so + 16 <= dyn_smem_size(), 11, so, dyn_smem_size());
      const bool oks = EE_CHECK(p.err, ((uintptr_t)src & 15) == 0 && row >= pl.r0 && row < pl.r1 && v0 + lane < nv,
                                12, row, v0 + lane);
      if (okd && oks)
#endif
        cp_async16(dst, src);
      if (PH == 1 && sc_async && lane == j) {
        const uint16_t* ssrc = p.ws + (size_t)row * p.sstride + (v0 >> 2);
        if (EE_CHECK(p.err, ((uintptr_t)ssrc & 15) == 0, 13, row, v0))
          cp_async16(slot + kBatch * 512 + j * 16, ssrc);
      }
    }
    v0 += 32;
    if (v0 >= nv) {
      v0 -= nv;
      ++ri;
    }
  }
}

template <int PH, bool XS, int MMAX>
EE_DEV void dot_vec(const uint4& wv, uint16_t sbits, const uint16_t* const* xrow, int k, int mc, float* acc) {
  if (PH == 0) {
#pragma unroll
    for (int m = 0; m < MMAX; ++m) {
      if (m < mc) {
        const uint4 xv = XS ? *reinterpret_cast<const uint4*>(xrow[m] + k) : ldg_nc_v4(xrow[m] + k);
        acc[m] = dot8_bf16(wv, xv, acc[m]);
      }
    }
  } else {
    const float sc = bf16_bits_to_float(sbits);
#pragma unroll
    for (int m = 0; m < MMAX; ++m) {
      if (m < mc) {
        const uint16_t* xp = xrow[m] + k;
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
        __half2 h = __float2half2_rn(0.0f);
        h = dot8_int4(wv.x, x0, h);
        h = dot8_int4(wv.y, x1, h);
        h = dot8_int4(wv.z, x2, h);
        h = dot8_int4(wv.w, x3, h);
        const float2 f = __half22float2(h);
        acc[m] = fmaf(sc, f.x + f.y, acc[m]);
      }
    }
  }
}

template <int MMAX>
EE_DEV void flush_row(float* rowsum, int mcap, int row_local, int mc, float* acc, int lane) {
#pragma unroll
  for (int m = 0; m < MMAX; ++m) {
    if (m < mc) {
      const float t = warp_sum(acc[m]);
      if (lane == 0) rowsum[row_local * mcap + m] = t;
    }
    acc[m] = 0.0f;
  }
}

template <int PH, bool XS, int MMAX>
EE_DEV void compute_batch(const LinearParams& p, const Plan& pl, const uint8_t* slot, bool sc_async, int base,
                          int total, int nv, int& cur, const uint16_t* const* xrow, int mc, float* acc,
                          float* rowsum, int warp, int lane) {
  const int epv = PH == 0 ? 8 : 32;  // elements per vector
  int ri = base / nv;
  int v0 = base - ri * nv;  // warp-uniform vector index of lane 0
#pragma unroll
  for (int j = 0; j < kBatch; ++j) {
    if (base + 32 * j < total) {
      if (ri != cur) {
        flush_row<MMAX>(rowsum, pl.mcap, warp + kWarps * cur, mc, acc, lane);
        cur = ri;
      }
      const uint4 wv = *reinterpret_cast<const uint4*>(slot + j * 512 + lane * 16);
      uint16_t sbits = 0;
      if (PH == 1)
        sbits = sc_async ? reinterpret_cast<const uint16_t*>(slot + kBatch * 512 + j * 16)[lane >> 2]
                         : ldg_u16(p.ws + (size_t)(pl.r0 + warp + kWarps * ri) * p.sstride + ((v0 + lane) >> 2));
      dot_vec<PH, XS, MMAX>(wv, sbits, xrow, (v0 + lane) * epv, mc, acc);
    }
    v0 += 32;
    if (v0 >= nv) {
      v0 -= nv;
      ++ri;
    }
  }
}

EE_DEV void wait_slots(int nslots) {
  if (nslots >= 4)
    cp_async_wait<3>();
  else if (nslots == 3)
    cp_async_wait<2>();
  else
    cp_async_wait<1>();
}

// The first nslots - 1 batches of a warp's stream (weights only, so they may
// be requested before the grid dependency wait).
template <int PH>
EE_DEV void stream_prologue(const LinearParams& p, const Plan& pl, int warp, int lane, uint8_t* ring,
                            bool sc_async, uint64_t pol) {
  const int nrows = pl.r1 - pl.r0;
  const int nrw = nrows > warp ? (nrows - warp + kWarps - 1) / kWarps : 0;
  const int nv = PH == 0 ? p.K / 8 : p.K / 32;
  if (nv % 32 != 0) return;
  const int total = nrw * nv;
  for (int b = 0; b < p.nslots - 1; ++b) {
    if (b * 32 * kBatch < total)
      issue_batch<PH>(p, pl, warp, lane, nv, total, b * 32 * kBatch, ring + (size_t)b * kSlotBytes, sc_async, pol);
    cp_async_commit();
  }
}

// Streams this warp's rows of one phase (PH 0: bf16 weights, 1: int4) for
// the mc sequences of one pass and writes each row's sums into rowsum.
// `pre`: stream_prologue already ran for this pass.
template <int PH, bool XS, int MMAX>
EE_DEV void stream_rows(const LinearParams& p, const Plan& pl, int warp, int lane, int mc,
                        const uint16_t* const* xrow, float* rowsum, uint8_t* ring, bool sc_async, bool pre,
                        uint64_t pol) {
  const int nrows = pl.r1 - pl.r0;
  const int nrw = nrows > warp ? (nrows - warp + kWarps - 1) / kWarps : 0;  // rows of this warp
  const int nv = PH == 0 ? p.K / 8 : p.K / 32;                             // vectors per row
  float acc[MMAX];
#pragma unroll
  for (int m = 0; m < MMAX; ++m) acc[m] = 0.0f;
  if (nv % 32 == 0) {
    const int total = nrw * nv;
    const int bstep = 32 * kBatch;
    const int nb = (total + bstep - 1) / bstep;
    const int ns = p.nslots;
    if (!pre) stream_prologue<PH>(p, pl, warp, lane, ring, sc_async, pol);
    int cur = 0;
    for (int b = 0; b < nb; ++b) {
      const int bn = b + ns - 1;
      if (bn < nb)
        issue_batch<PH>(p, pl, warp, lane, nv, total, bn * bstep, ring + (size_t)(bn % ns) * kSlotBytes, sc_async,
                        pol);
      cp_async_commit();
      wait_slots(ns);  // batch b has landed
      __syncwarp();
      compute_batch<PH, XS, MMAX>(p, pl, ring + (size_t)(b % ns) * kSlotBytes, sc_async, b * bstep, total, nv, cur,
                                  xrow, mc, acc, rowsum, warp, lane);
      __syncwarp();  // the slot is refilled next iteration
    }
    if (nrw > 0) flush_row<MMAX>(rowsum, pl.mcap, warp + kWarps * cur, mc, acc, lane);
    cp_async_wait<0>();
  } else {
    // short or odd rows: one row at a time, lanes stride over its vectors
    const size_t rstride = PH == 0 ? (size_t)p.K * 2 : (size_t)p.K / 2;
    const uint8_t* wbase = PH == 0 ? reinterpret_cast<const uint8_t*>(p.w) : p.wq;
    for (int ri = 0; ri < nrw; ++ri) {
      const int row = pl.r0 + warp + kWarps * ri;
      for (int v = lane; v < nv; v += 32) {
        const uint4 wv = ldg_nc_v4(wbase + (size_t)row * rstride + (size_t)v * 16);
        const uint16_t sbits = PH == 1 ? ldg_u16(p.ws + (size_t)row * p.sstride + (v >> 2)) : 0;
        dot_vec<PH, XS, MMAX>(wv, sbits, xrow, v * (PH == 0 ? 8 : 32), mc, acc);
      }
      flush_row<MMAX>(rowsum, pl.mcap, warp + kWarps * ri, mc, acc, lane);
    }
  }
}

template <int EPI, bool XS, int MMAX>
__global__ void __launch_bounds__(kThreads, 1) k_linear(const LinearParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  int32_t* lf = reinterpret_cast<int32_t*>(smem);
  int32_t* le = lf + kListLen;
  float* hst = reinterpret_cast<float*>(smem + 2 * kListLen * 4 + 16);
  uint8_t* xs = smem + kHeaderBytes;
  float* rowsum = reinterpret_cast<float*>(xs + (XS ? (size_t)p.xs_rows * p.K * 2 : 0));
  uint8_t* rings = reinterpret_cast<uint8_t*>(rowsum) + (((size_t)p.rows_cap * p.mcap * 4 + 15) / 16 * 16);
  __shared__ int s_last;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
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
    pl.mcap = p.mcap;
    pl.passes[0] = (nf + pl.mcap - 1) / pl.mcap;
    pl.passes[1] = (ne + pl.mcap - 1) / pl.mcap;
  }
  const int nrows = pl.r1 - pl.r0;

  uint8_t* ring = rings + (size_t)warp * p.nslots * kSlotBytes;
  const uint64_t pol = l2_evict_first_policy();
  const bool sc_async = p.K % 1024 == 0 && p.sstride * EE_QUANT_GROUP == p.K;
  // Weights do not depend on the previous kernel: start this warp's stream now.
  const int first_phase = pl.passes[0] > 0 ? 0 : (pl.passes[1] > 0 ? 1 : -1);
  if (first_phase == 0) stream_prologue<0>(p, pl, warp, lane, ring, sc_async, pol);
  if (first_phase == 1) stream_prologue<1>(p, pl, warp, lane, ring, sc_async, pol);
  grid_dep_wait();
  grid_dep_launch();
  if (XS && nx > 0) {
    // the activations of the step's rows, written by the previous kernel
    const int v16 = p.K / 8;  // 16-byte vectors per row
    for (int i = tid; i < nx * v16; i += kThreads) {
      const int m = i / v16, c = i - m * v16;
      const int seq = m < nf ? lf[1 + m] : le[1 + m - nf];
#ifdef EE_CHECKED
      if (!EE_CHECK(p.err, (size_t)(i + 1) * 16 <= (size_t)p.xs_rows * p.K * 2 && seq >= 0 && seq < EE_MAX_BATCH, 15,
                    i, seq))
        continue;
#endif
      reinterpret_cast<uint4*>(xs)[i] = *reinterpret_cast<const uint4*>(p.xh + (size_t)seq * p.x_stride + c * 8);
    }
  }
  __syncthreads();

  for (int phase = 0; phase < 2; ++phase) {
    const int nlist = phase == 0 ? nf : ne;
    const int32_t* lst = phase == 0 ? lf : le;
    const int xbase = phase == 0 ? 0 : nf;  // XS row of the phase's first sequence
    for (int pass = 0; pass < pl.passes[phase]; ++pass) {
      const int m0 = pass * pl.mcap;
      const int mc = min(pl.mcap, nlist - m0);
      const uint16_t* xrow[MMAX];
#pragma unroll
      for (int m = 0; m < MMAX; ++m) {
        const int mm = min(m, mc - 1);
        xrow[m] = XS ? reinterpret_cast<const uint16_t*>(xs) + (size_t)(xbase + m0 + mm) * p.K
                     : p.xh + (size_t)lst[1 + m0 + mm] * p.x_stride;
      }
      const bool pre = phase == first_phase && pass == 0;
      if (phase == 0)
        stream_rows<0, XS, MMAX>(p, pl, warp, lane, mc, xrow, rowsum, ring, sc_async, pre, pol);
      else
        stream_rows<1, XS, MMAX>(p, pl, warp, lane, mc, xrow, rowsum, ring, sc_async, pre, pol);
      __syncthreads();  // every row sum of this pass is complete
      if constexpr (EPI == EPI_HEAD) {
        Stat stat[MMAX];
#pragma unroll
        for (int m = 0; m < MMAX; ++m) stat[m] = Stat{-INFINITY, 0.0f, 0x7fffffff};
        for (int r = tid; r < nrows; r += kThreads) {
#pragma unroll
          for (int m = 0; m < MMAX; ++m)
            if (m < mc) stat_push(stat[m], rowsum[r * pl.mcap + m], pl.r0 + r);
        }
#pragma unroll
        for (int m = 0; m < MMAX; ++m) {
          if (m < mc) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
              Stat t;
              t.mx = __shfl_xor_sync(0xffffffffu, stat[m].mx, o);
              t.sum = __shfl_xor_sync(0xffffffffu, stat[m].sum, o);
              t.arg = __shfl_xor_sync(0xffffffffu, stat[m].arg, o);
              stat[m] = stat_merge(stat[m], t);
            }
            if (lane == 0) {
              float* hs = hst + (warp * kMM + m) * 3;
              hs[0] = stat[m].mx;
              hs[1] = stat[m].sum;
              hs[2] = __int_as_float(stat[m].arg);
            }
          }
        }
        __syncthreads();
        if (warp == 0 && lane < mc) {
          Stat sm = {-INFINITY, 0.0f, 0x7fffffff};
          for (int w = 0; w < kWarps; ++w) {
            const float* hs = hst + (w * kMM + lane) * 3;
            sm = stat_merge(sm, Stat{hs[0], hs[1], __float_as_int(hs[2])});
          }
          float* dst = p.head_part + ((size_t)blockIdx.x * EE_MAX_BATCH + m0 + lane) * 4;
          dst[0] = sm.mx;
          dst[1] = sm.sum;
          dst[2] = __int_as_float(sm.arg);
        }
      } else {
        int seqs_m[MMAX];
#pragma unroll
        for (int m = 0; m < MMAX; ++m) seqs_m[m] = lst[1 + m0 + min(m, mc - 1)];
        const int npr = nrows >> 1;
        for (int i = tid; i < npr * mc; i += kThreads) {
          const int pr = i / mc, m = i - pr * mc;
          int seq = seqs_m[0];
#pragma unroll
          for (int mm = 1; mm < MMAX; ++mm)
            if (mm == m) seq = seqs_m[mm];
          epi_pair<EPI>(p, seq, pl.r0 + 2 * pr, rowsum[(2 * pr) * pl.mcap + m],
                        rowsum[(2 * pr + 1) * pl.mcap + m]);
        }
      }
      __syncthreads();  // row sums are reused by the next pass
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
    for (int m = warp; m < nrows; m += kWarps) {
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
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(k_linear<EPI, false, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)kSmemMax)) != cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(k_linear<EPI, true, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)kSmemMax)) != cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(k_linear<EPI, false, kMM>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)kSmemMax)) != cudaSuccess)
    return e;
  return cudaFuncSetAttribute(k_linear<EPI, true, kMM>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)kSmemMax);
}

size_t smem_of(const LinearParams& p) {
  return kHeaderBytes + (p.xs_rows > 0 ? (size_t)p.xs_rows * p.K * 2 : 0) +
         ((size_t)p.rows_cap * p.mcap * 4 + 15) / 16 * 16 + (size_t)kWarps * p.nslots * kSlotBytes;
}

template <int EPI>
cudaError_t launch_one(const LinearParams& p, int grid, bool pdl, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem_of(p);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  if (p.mcap == 1) {
    if (p.xs_rows > 0) return cudaLaunchKernelEx(&cfg, k_linear<EPI, true, 1>, p);
    return cudaLaunchKernelEx(&cfg, k_linear<EPI, false, 1>, p);
  }
  if (p.xs_rows > 0) return cudaLaunchKernelEx(&cfg, k_linear<EPI, true, kMM>, p);
  return cudaLaunchKernelEx(&cfg, k_linear<EPI, false, kMM>, p);
}

// Shared-memory plan of one launch: per-row sums for the CTA's rows and the
// activations of the step's rows when they fit.
void plan_smem(LinearParams& p, int grid) {
  const int max_rows = p.max_rows < 1 ? 1 : p.max_rows;
  p.mcap = max_rows < kMM ? max_rows : kMM;
  const int npairs = p.N / 2;
  p.rows_cap = 2 * ((npairs + grid - 1) / grid);
  const size_t xb = (size_t)max_rows * p.K * 2;
  const bool xs = max_rows <= kMM && xb <= kXsMaxBytes;
  p.xs_rows = xs ? max_rows : 0;
  // Three slots (two batches in flight per lane, 64 KB per SM) in a CTA small
  // enough that the next kernel's CTA fits beside it and starts its stream
  // before this one ends; fewer when that does not fit.
  p.nslots = 3;
  while (p.nslots > 2 && smem_of(p) > kSmemPair) --p.nslots;
  if (smem_of(p) > kSmemMax) p.nslots = 2;
}

}  // namespace

size_t linear_smem_bytes() { return kSmemMax; }

cudaError_t linear_prepare() {
  cudaError_t e;
  if ((e = set_smem_attr<EPI_F32>()) != cudaSuccess) return e;
  if ((e = set_smem_attr<EPI_QKV>()) != cudaSuccess) return e;
  if ((e = set_smem_attr<EPI_RESID>()) != cudaSuccess) return e;
  if ((e = set_smem_attr<EPI_SWIGLU>()) != cudaSuccess) return e;
  if ((e = set_smem_attr<EPI_X>()) != cudaSuccess) return e;
  return set_smem_attr<EPI_HEAD>();
}

bool linear_shape_ok(int K) { return K >= 32 && K % 32 == 0; }

int linear_grid(int N, int num_sms) {
  const int pairs = N / 2;
  return pairs < num_sms ? (pairs > 0 ? pairs : 1) : num_sms;
}

cudaError_t launch_linear(const LinearParams& p_in, int grid, bool pdl, cudaStream_t st) {
  LinearParams p = p_in;
  plan_smem(p, grid);
  if (smem_of(p) > kSmemMax) return cudaErrorInvalidConfiguration;
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
