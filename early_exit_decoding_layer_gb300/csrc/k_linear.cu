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
// Data flow: two CTAs of 8 warps per SM each own a balanced, pair-aligned
// range of output rows; warp w owns its CTA's rows w, w+8, ... and walks them
// as one stream of 16-byte vectors, 32 at a time (a warp reads 512 contiguous
// bytes per load instruction), straight into registers.  Two batches per
// lane alternate (8 vectors each for bf16, 4 for int4): the loads of the next
// batch are issued before the current one is consumed, so up to 64 KB per SM
// are in flight -- what HBM3e needs to stream near its peak.  The first batch
// is requested before the grid dependency wait (weights never change), and
// with two CTA slots per SM the next launch's CTAs start that stream in the
// slots this launch's finished CTAs free, while its last CTAs drain.  The
// activations of the step's rows (fp16, a few KB per sequence), written by
// the previous kernel, are copied into shared memory after the wait.  A warp
// finishes each of its rows alone (one warp reduction), so results do not
// depend on timing.  The epilogue (RoPE + KV write, SwiGLU, residual add,
// head statistics) runs once over the CTA's rows.
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
#include "ee_epilogue.cuh"
#include "ee_head.cuh"
#include "ee_kernels.cuh"

namespace ee {

namespace {

constexpr int kWarps = 8;
constexpr int kCtasPerSm = 2;  // two CTAs per SM: one kernel's tail overlaps the next one's start
constexpr int kThreads = kWarps * 32;
constexpr int kBatch = 8;  // 16-byte vectors per lane per batch
constexpr int kMM = 8;     // sequences per pass over the weights

// Shared memory: header (lists, head statistics), the staged activations
// (XS mode), then the per-row sums [rows][mcap].
constexpr size_t kHeaderBytes = 3072;
constexpr size_t kXsMaxBytes = 64 * 1024;
constexpr size_t kSmemMax = 227 * 1024 - 1024;
static_assert(2 * kListLen * 4 + 16 + kWarps * kMM * 3 * 4 <= kHeaderBytes, "header overflow");
// the staging RMSNorm keeps its per-warp sums [kMM][kWarps] in the head-statistics area
static_assert(kMM * kWarps <= kWarps * kMM * 3, "norm scratch");

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

EE_DEV uint16_t ldg_u16(const uint16_t* p) {
  uint16_t v;
  asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}

struct Plan {
  int r0, r1, mcap;
  int passes[2];
};

#ifdef EE_CHECKED
// Debug builds: the staging copies are checked; a bad one is recorded (site
// code in err[0], values in err[1..2]) and skipped.
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

// One warp's share of a phase: its rows r0 + warp + kWarps * i (i < nrw) of
// the bf16 matrix (PH 0) or of the packed int4 matrix (PH 1), nv 16-byte
// vectors each.  When nv % 32 == 0 the rows are walked as one stream of
// steps of 32 vectors (one per lane: a warp reads 512 contiguous bytes per
// step), in batches of kU<PH> steps.  A batch that lies inside one row takes
// the unrolled path; one that crosses a row boundary steps vector by vector.
// Several sequences per pass need more registers per vector: smaller batches.
template <int PH, int MMAX>
constexpr int kU = (PH == 0 ? 8 : 4) / (MMAX == 1 ? 1 : 2);
static_assert(kU<0, 1> <= kBatch && kU<1, 1> <= kBatch, "batch storage");

struct Stream {
  const uint8_t* base;
  size_t rstride;  // bytes per row
  int nv, nrw, row0;
};

template <int PH>
EE_DEV Stream make_stream(const LinearParams& p, const Plan& pl, int warp) {
  Stream s;
  s.base = PH == 0 ? reinterpret_cast<const uint8_t*>(p.w) : p.wq;
  s.rstride = PH == 0 ? (size_t)p.K * 2 : (size_t)p.K / 2;
  s.nv = PH == 0 ? p.K / 8 : p.K / 32;
  const int nrows = pl.r1 - pl.r0;
  s.nrw = nrows > warp ? (nrows - warp + kWarps - 1) / kWarps : 0;
  s.row0 = pl.r0 + warp;
  return s;
}

// Load-side position: row ri of the warp's rows, vector v0 + lane, and this
// lane's weight (and scale) addresses.
struct LoadCursor {
  int ri, v0;
  const uint8_t* wp;
  const uint16_t* sp;
};

template <int PH>
EE_DEV LoadCursor load_start(const LinearParams& p, const Stream& st, int lane) {
  LoadCursor c;
  c.ri = 0;
  c.v0 = 0;
  c.wp = st.base + (size_t)st.row0 * st.rstride + (size_t)lane * 16;
  c.sp = PH == 1 ? p.ws + (size_t)st.row0 * p.sstride + (lane >> 2) : nullptr;
  return c;
}

// Vectors of one batch per lane (and, for int4, their scales, two per word).
struct Batch {
  uint4 w[kBatch];
  uint32_t s[kBatch / 2];
};

template <int PH>
EE_DEV void next_row(const LinearParams& p, const Stream& st, LoadCursor& c) {
  c.v0 = 0;
  ++c.ri;
  c.wp += (size_t)kWarps * st.rstride - (size_t)st.nv * 16;
  if constexpr (PH == 1) c.sp += (size_t)kWarps * p.sstride - st.nv / 4;
}

template <int PH>
EE_DEV void put_scale(Batch& b, int j, uint32_t sv) {
  b.s[j >> 1] = (j & 1) ? (b.s[j >> 1] | (sv << 16)) : sv;
}

template <int PH, int MMAX>
EE_DEV void load_batch(const LinearParams& p, const Stream& st, LoadCursor& c, Batch& b) {
  constexpr int U = kU<PH, MMAX>;
  if (c.ri >= st.nrw) return;
  if (c.v0 + 32 * U <= st.nv) {
#pragma unroll
    for (int j = 0; j < U; ++j) {
      b.w[j] = ldg_stream_v4(c.wp + j * 512);
      if constexpr (PH == 1) put_scale<PH>(b, j, ldg_u16(c.sp + j * 8));
    }
    c.v0 += 32 * U;
    c.wp += 512 * U;
    if constexpr (PH == 1) c.sp += 8 * U;
    if (c.v0 == st.nv) next_row<PH>(p, st, c);
  } else {
#pragma unroll
    for (int j = 0; j < U; ++j) {
      if (c.ri < st.nrw) {
        b.w[j] = ldg_stream_v4(c.wp);
        if constexpr (PH == 1) put_scale<PH>(b, j, ldg_u16(c.sp));
      }
      c.v0 += 32;
      c.wp += 512;
      if constexpr (PH == 1) c.sp += 8;
      if (c.v0 == st.nv) next_row<PH>(p, st, c);
    }
  }
}

// Activations of the pass's sequences: row m starts at xb + xoff[m] (fp16,
// pair order).  int4 rows staged in shared memory (PL) are stored as four
// planes so that the four 16-byte chunks of one vector sit in four planes at
// the lane's index (conflict-free): chunk c at (c % 4) * (K / 32) + c / 4.
template <int PH, bool PL, int MMAX>
EE_DEV void dot_vec(const uint4& wv, uint32_t sbits, const uint16_t* xb, const int32_t* xoff, int v, int nv,
                    int mc, float* acc) {
  if constexpr (PH == 0) {
#pragma unroll
    for (int m = 0; m < MMAX; ++m) {
      if (m < mc) acc[m] = dot8_bf16(wv, *reinterpret_cast<const uint4*>(xb + xoff[m] + v * 8), acc[m]);
    }
  } else {
    const float sc = __uint_as_float(sbits << 16);
#pragma unroll
    for (int m = 0; m < MMAX; ++m) {
      if (m < mc) {
        const uint4* xp = reinterpret_cast<const uint4*>(xb + xoff[m]);
        const int i0 = PL ? v : 4 * v, di = PL ? nv : 1;
        __half2 h = __float2half2_rn(0.0f);
        h = dot8_int4(wv.x, xp[i0], h);
        h = dot8_int4(wv.y, xp[i0 + di], h);
        h = dot8_int4(wv.z, xp[i0 + 2 * di], h);
        h = dot8_int4(wv.w, xp[i0 + 3 * di], h);
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

template <int PH>
EE_DEV uint32_t scale_of(const Batch& b, int j) {
  return PH == 1 ? (b.s[j >> 1] >> (16 * (j & 1))) & 0xFFFFu : 0u;
}

// Consumes one batch; the compute-side cursor (ri, v0) mirrors the load
// side, and each completed row is flushed.
template <int PH, bool PL, int MMAX>
EE_DEV void compute_batch(const Stream& st, int& ri, int& v0, const Batch& b, const uint16_t* xb,
                          const int32_t* xoff, int mc, int mcap, float* acc, float* rowsum, int warp, int lane) {
  constexpr int U = kU<PH, MMAX>;
  if (ri >= st.nrw) return;
  if (v0 + 32 * U <= st.nv) {
#pragma unroll
    for (int j = 0; j < U; ++j)
      dot_vec<PH, PL, MMAX>(b.w[j], scale_of<PH>(b, j), xb, xoff, v0 + 32 * j + lane, st.nv, mc, acc);
    v0 += 32 * U;
    if (v0 == st.nv) {
      flush_row<MMAX>(rowsum, mcap, warp + kWarps * ri, mc, acc, lane);
      v0 = 0;
      ++ri;
    }
  } else {
#pragma unroll
    for (int j = 0; j < U; ++j) {
      if (ri < st.nrw) dot_vec<PH, PL, MMAX>(b.w[j], scale_of<PH>(b, j), xb, xoff, v0 + lane, st.nv, mc, acc);
      v0 += 32;
      if (v0 == st.nv) {
        if (ri < st.nrw) flush_row<MMAX>(rowsum, mcap, warp + kWarps * ri, mc, acc, lane);
        v0 = 0;
        ++ri;
      }
    }
  }
}

// Streams this warp's rows of one phase for the mc sequences of one pass and
// writes each row's sums into rowsum.  Two register batches alternate: the
// next batch's loads are issued before the current one is consumed.  `pre`:
// batch 0 was loaded into `a` (load cursor `lc`) before the dependency wait.
template <int PH, bool PL, int MMAX>
EE_DEV void stream_rows(const LinearParams& p, const Plan& pl, int warp, int lane, int mc, const uint16_t* xb,
                        const int32_t* xoff, float* rowsum, Batch& a, LoadCursor& lc, bool pre) {
  const Stream st = make_stream<PH>(p, pl, warp);
  float acc[MMAX];
#pragma unroll
  for (int m = 0; m < MMAX; ++m) acc[m] = 0.0f;
  if (st.nv % 32 == 0) {
    constexpr int U = kU<PH, MMAX>;
    const int nb = (st.nrw * (st.nv / 32) + U - 1) / U;
    if (!pre) {
      lc = load_start<PH>(p, st, lane);
      load_batch<PH, MMAX>(p, st, lc, a);
    }
    int ri = 0, v0 = 0;
    Batch b;
    for (int i = 0; i < nb; i += 2) {
      if (i + 1 < nb) load_batch<PH, MMAX>(p, st, lc, b);
      compute_batch<PH, PL, MMAX>(st, ri, v0, a, xb, xoff, mc, pl.mcap, acc, rowsum, warp, lane);
      if (i + 2 < nb) load_batch<PH, MMAX>(p, st, lc, a);
      if (i + 1 < nb) compute_batch<PH, PL, MMAX>(st, ri, v0, b, xb, xoff, mc, pl.mcap, acc, rowsum, warp, lane);
    }
  } else {
    // short or odd rows: one row at a time, lanes stride over its vectors
    for (int ri = 0; ri < st.nrw; ++ri) {
      const int row = st.row0 + kWarps * ri;
      for (int v = lane; v < st.nv; v += 32) {
        const uint4 wv = ldg_stream_v4(st.base + (size_t)row * st.rstride + (size_t)v * 16);
        const uint32_t sbits = PH == 1 ? ldg_u16(p.ws + (size_t)row * p.sstride + (v >> 2)) : 0u;
        dot_vec<PH, PL, MMAX>(wv, sbits, xb, xoff, v, st.nv, mc, acc);
      }
      flush_row<MMAX>(rowsum, pl.mcap, warp + kWarps * ri, mc, acc, lane);
    }
  }
}

// Epilogue of one pass: the CTA's row sums for sequences m0 .. m0 + mc - 1
// of list `lst` are complete in rowsum.
template <int MMAX>
EE_DEV void pass_epilogue(const LinearParams& p, const Plan& pl, const int32_t* lst, int m0, int mc,
                          const float* rowsum, float* hst, int nrows, int tid, int warp, int lane) {
  if (p.epi == EPI_HEAD) {
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
      const int ra = pl.r0 + 2 * pr;
      const float ya = rowsum[(2 * pr) * pl.mcap + m], yb = rowsum[(2 * pr + 1) * pl.mcap + m];
      switch (p.epi) {
        case EPI_F32: epi_pair<EPI_F32>(p, seq, ra, ya, yb); break;
        case EPI_QKV: epi_pair<EPI_QKV>(p, seq, ra, ya, yb); break;
        case EPI_RESID: epi_pair<EPI_RESID>(p, seq, ra, ya, yb); break;
        case EPI_SWIGLU: epi_pair<EPI_SWIGLU>(p, seq, ra, ya, yb); break;
        default: epi_pair<EPI_X>(p, seq, ra, ya, yb); break;
      }
    }
  }
}

// Staged position of 16-byte chunk c of an exit (int4) row: four planes.
EE_DEV int x_plane_index(int c, int K) { return (c & 3) * (K / 32) + (c >> 2); }

// Everything up to the first pass: the dependency wait, then the step's
// activations copied into shared memory (XS mode).
template <bool XS>
EE_DEV void wait_and_stage(const LinearParams& p, const int32_t* lf, const int32_t* le, int nf, int nx,
                           uint8_t* xs, float* red, int tid, int warp, int lane) {
  grid_dep_wait();
  grid_dep_launch();
  if (XS && nx > 0 && p.norm_h) {
    // RMSNorm of the step's rows of the residual stream (written by the
    // previous kernel): per-row sum of squares, then the scaled fp16 rows
    const int v8 = p.K / 8;  // runs of 8 columns per row
    for (int m = 0; m < nx; ++m) {
      const int seq = m < nf ? lf[1 + m] : le[1 + m - nf];
      const float4* h = reinterpret_cast<const float4*>(p.norm_h + (size_t)seq * p.norm_stride);
      float ss = 0.0f;
      for (int i = tid; i < v8; i += kThreads) {
        const float4 a = h[2 * i], b = h[2 * i + 1];
        ss = fmaf(a.x, a.x, ss);
        ss = fmaf(a.y, a.y, ss);
        ss = fmaf(a.z, a.z, ss);
        ss = fmaf(a.w, a.w, ss);
        ss = fmaf(b.x, b.x, ss);
        ss = fmaf(b.y, b.y, ss);
        ss = fmaf(b.z, b.z, ss);
        ss = fmaf(b.w, b.w, ss);
      }
      ss = warp_sum(ss);
      if (lane == 0) red[m * kWarps + warp] = ss;
    }
    __syncthreads();
    for (int i = tid; i < nx * v8; i += kThreads) {
      const int m = i / v8, c = i - m * v8;
      const int seq = m < nf ? lf[1 + m] : le[1 + m - nf];
      const int dst = m * v8 + (m < nf ? c : x_plane_index(c, p.K));
      float tot = 0.0f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) tot += red[m * kWarps + w];
      const float r = rsqrtf(tot / (float)p.K + p.norm_eps);
      const float4* h = reinterpret_cast<const float4*>(p.norm_h + (size_t)seq * p.norm_stride) + 2 * c;
      const float4 a = h[0], b = h[1];
      const uint4 gw = *reinterpret_cast<const uint4*>(p.norm_g + (size_t)c * 8);
      uint4 o;  // pair order: (x0,x4) (x1,x5) (x2,x6) (x3,x7)
      o.x = uint32_t(float_to_half_bits(a.x * r * bf16_lo(gw.x))) |
            (uint32_t(float_to_half_bits(b.x * r * bf16_lo(gw.z))) << 16);
      o.y = uint32_t(float_to_half_bits(a.y * r * bf16_hi(gw.x))) |
            (uint32_t(float_to_half_bits(b.y * r * bf16_hi(gw.z))) << 16);
      o.z = uint32_t(float_to_half_bits(a.z * r * bf16_lo(gw.y))) |
            (uint32_t(float_to_half_bits(b.z * r * bf16_lo(gw.w))) << 16);
      o.w = uint32_t(float_to_half_bits(a.w * r * bf16_hi(gw.y))) |
            (uint32_t(float_to_half_bits(b.w * r * bf16_hi(gw.w))) << 16);
      reinterpret_cast<uint4*>(xs)[dst] = o;
    }
  } else if (XS && nx > 0) {
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
      const int dst = m * v16 + (m < nf ? c : x_plane_index(c, p.K));
      reinterpret_cast<uint4*>(xs)[dst] = *reinterpret_cast<const uint4*>(p.xh + (size_t)seq * p.x_stride + c * 8);
    }
  }
  __syncthreads();
}

// All passes of one phase (PH 0: the full list on bf16 weights, PH 1: the
// exit list on int4 weights).
template <bool XS, int MMAX, int PH>
EE_DEV void run_phase(const LinearParams& p, const Plan& pl, const int32_t* lst, int nlist, int xbase,
                      const uint8_t* xs, float* rowsum, float* hst, int nrows, int tid, int warp, int lane,
                      Batch& a, LoadCursor& lc, bool pre) {
  for (int pass = 0; pass < pl.passes[PH]; ++pass) {
    const int m0 = pass * pl.mcap;
    const int mc = min(pl.mcap, nlist - m0);
    const uint16_t* xb = XS ? reinterpret_cast<const uint16_t*>(xs) : p.xh;
    int32_t xoff[MMAX];
#pragma unroll
    for (int m = 0; m < MMAX; ++m) {
      const int mm = min(m, mc - 1);
      xoff[m] = XS ? (xbase + m0 + mm) * p.K : lst[1 + m0 + mm] * p.x_stride;
    }
    stream_rows<PH, XS && PH == 1, MMAX>(p, pl, warp, lane, mc, xb, xoff, rowsum, a, lc, pre && pass == 0);
    __syncthreads();  // every row sum of this pass is complete
    pass_epilogue<MMAX>(p, pl, lst, m0, mc, rowsum, hst, nrows, tid, warp, lane);
    __syncthreads();  // row sums are reused by the next pass
  }
}

// One kernel binary per (staging, sequences per pass) for every projection and
// head: the epilogue is chosen at run time, so consecutive launches of a step
// run the same code and find it warm in the instruction caches.
template <bool XS, int MMAX>
__global__ void __launch_bounds__(kThreads, kCtasPerSm) k_linear(const LinearParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  int32_t* lf = reinterpret_cast<int32_t*>(smem);
  int32_t* le = lf + kListLen;
  float* hst = reinterpret_cast<float*>(smem + 2 * kListLen * 4 + 16);
  uint8_t* xs = smem + kHeaderBytes;
  float* rowsum = reinterpret_cast<float*>(xs + (XS ? (size_t)p.xs_rows * p.K * 2 : 0));
  __shared__ int s_last;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // Lists written at least two launches back (see grid_dep_wait) may be read
  // before this grid's dependency wait; otherwise wait first.
  if (p.lists_after_wait) grid_dep_wait();
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

  // Weights do not depend on the previous kernel: the first batch of this
  // warp's first phase is requested before the dependency wait.
  Batch a;
  LoadCursor lc;
  int pre_phase = -1;
  if (!p.lists_after_wait) {
    if (pl.passes[0] > 0) {
      const Stream st = make_stream<0>(p, pl, warp);
      if (st.nv % 32 == 0) {
        lc = load_start<0>(p, st, lane);
        load_batch<0, MMAX>(p, st, lc, a);
        pre_phase = 0;
      }
    } else if (pl.passes[1] > 0) {
      const Stream st = make_stream<1>(p, pl, warp);
      if (st.nv % 32 == 0) {
        lc = load_start<1>(p, st, lane);
        load_batch<1, MMAX>(p, st, lc, a);
        pre_phase = 1;
      }
    }
  }
  wait_and_stage<XS>(p, lf, le, nf, nx, xs, hst, tid, warp, lane);
  // each phase's code exists once (the kernel stays small in the instruction cache)
#pragma unroll 1
  for (int phase = 0; phase < 2; ++phase) {
    if (phase == 0)
      run_phase<XS, MMAX, 0>(p, pl, lf, nf, 0, xs, rowsum, hst, nrows, tid, warp, lane, a, lc, pre_phase == 0);
    else
      run_phase<XS, MMAX, 1>(p, pl, le, ne, nf, xs, rowsum, hst, nrows, tid, warp, lane, a, lc, pre_phase == 1);
  }

  if (p.epi == EPI_HEAD) {
    // Last CTA to finish merges the per-CTA partials (no spin wait: a counter).
    __syncthreads();
    if (tid == 0) {
      __threadfence();
      const int old = atomicAdd(p.head_counter, 1);
      s_last = (old == (int)gridDim.x - 1);
    }
    __syncthreads();
    if (!s_last) return;
    head_finalize(p, (int)gridDim.x, lf, le, nf, hst);
  }
}

cudaError_t set_smem_attr() {
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(k_linear<false, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemMax)) !=
      cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(k_linear<true, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemMax)) !=
      cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(k_linear<false, kMM>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemMax)) !=
      cudaSuccess)
    return e;
  return cudaFuncSetAttribute(k_linear<true, kMM>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemMax);
}

size_t smem_of(const LinearParams& p) {
  return kHeaderBytes + (p.xs_rows > 0 ? (size_t)p.xs_rows * p.K * 2 : 0) + (size_t)p.rows_cap * p.mcap * 4;
}

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
    if (p.xs_rows > 0) return cudaLaunchKernelEx(&cfg, k_linear<true, 1>, p);
    return cudaLaunchKernelEx(&cfg, k_linear<false, 1>, p);
  }
  if (p.xs_rows > 0) return cudaLaunchKernelEx(&cfg, k_linear<true, kMM>, p);
  return cudaLaunchKernelEx(&cfg, k_linear<false, kMM>, p);
}

// Shared-memory plan of one launch: per-row sums for the CTA's rows and the
// activations of the step's rows when they fit.
void plan_smem(LinearParams& p, int grid) {
  const int max_rows = p.max_rows < 1 ? 1 : p.max_rows;
  p.mcap = max_rows < kMM ? max_rows : kMM;
  const int npairs = p.N / 2;
  p.rows_cap = 2 * ((npairs + grid - 1) / grid);
  p.xs_rows = linear_stages_x(max_rows, p.K) ? max_rows : 0;
}

}  // namespace

size_t linear_smem_bytes() { return kSmemMax; }

cudaError_t linear_prepare() {
  return set_smem_attr();
}

bool linear_shape_ok(int K) { return K >= 32 && K % 32 == 0; }

bool linear_stages_x(int max_rows, int K) {
  const int rows = max_rows < 1 ? 1 : max_rows;
  return rows <= kMM && (size_t)rows * K * 2 <= kXsMaxBytes;
}

int linear_grid(int N, int num_sms) {
  const int pairs = N / 2, ctas = kCtasPerSm * num_sms;
  return pairs < ctas ? (pairs > 0 ? pairs : 1) : ctas;
}

cudaError_t launch_linear(const LinearParams& p_in, int grid, bool pdl, cudaStream_t st) {
  LinearParams p = p_in;
  plan_smem(p, grid);
  if (smem_of(p) > kSmemMax) return cudaErrorInvalidConfiguration;
  if (p.epi < EPI_F32 || p.epi > EPI_HEAD) return cudaErrorInvalidValue;
  return launch_one(p, grid, pdl, st);
}

}  // namespace ee
