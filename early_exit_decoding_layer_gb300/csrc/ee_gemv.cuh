// Device code of the skinny GEMV (see k_linear.cu for the design): the
// per-CTA prologue (lists, row plan, first weight batch) and body (staging,
// streaming, epilogues), included by the GEMV kernel.
#pragma once

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
constexpr size_t kL2PrefetchMax = 64 * 1024;  // int4 slice a CTA prefetches into L2 before its wait

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
// Nibble j holds column j (two's complement).  Masking nibbles (j, j+4) under
// the fp16 exponent of 1024 and flipping their sign bit in the same LOP3
// ((t & m) ^ magic) gives 1024 + q + 8 in the low position or 1024 + 16 (q + 8)
// in the high one; one HADD2 (-1032) or HFMA2 (x 1/16, -72) leaves q exactly.
EE_DEV __half2 dot8_int4(uint32_t t, const uint4& x, __half2 acc) {
  const __half2 m1032 = __half2half2(__ushort_as_half((unsigned short)0xE408));  // -1032
  const __half2 r16 = __half2half2(__ushort_as_half((unsigned short)0x2C00));    // 1/16
  const __half2 m72 = __half2half2(__ushort_as_half((unsigned short)0xD480));    // -72
  const uint32_t t8 = t >> 8;
  const __half2 q04 = __hadd2(u32_as_h2((t & 0x000F000Fu) ^ 0x64086408u), m1032);
  const __half2 q15 = __hfma2(u32_as_h2((t & 0x00F000F0u) ^ 0x64806480u), r16, m72);
  const __half2 q26 = __hadd2(u32_as_h2((t8 & 0x000F000Fu) ^ 0x64086408u), m1032);
  const __half2 q37 = __hfma2(u32_as_h2((t8 & 0x00F000F0u) ^ 0x64806480u), r16, m72);
  acc = __hfma2(q04, u32_as_h2(x.x), acc);
  acc = __hfma2(q15, u32_as_h2(x.y), acc);
  acc = __hfma2(q26, u32_as_h2(x.z), acc);
  acc = __hfma2(q37, u32_as_h2(x.w), acc);
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
// step), in batches of kU<PH> steps.  A batch never crosses a row: where kU
// does not divide a row's steps, the row's last batch holds the remainder.
// One code path for both keeps the streaming loop small.  Several sequences
// per pass need more registers per vector: smaller batches.
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
  const int cnt = min(U, (st.nv - c.v0) >> 5);  // steps left in the row
#pragma unroll
  for (int j = 0; j < U; ++j) {
    if (j < cnt) {
      b.w[j] = ldg_stream_v4(c.wp + j * 512);
      if constexpr (PH == 1) put_scale<PH>(b, j, ldg_u16(c.sp + j * 8));
    }
  }
  c.v0 += 32 * cnt;
  c.wp += 512 * cnt;
  if constexpr (PH == 1) c.sp += 8 * cnt;
  if (c.v0 == st.nv) next_row<PH>(p, st, c);
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
  const int cnt = min(U, (st.nv - v0) >> 5);
#pragma unroll
  for (int j = 0; j < U; ++j)
    if (j < cnt) dot_vec<PH, PL, MMAX>(b.w[j], scale_of<PH>(b, j), xb, xoff, v0 + 32 * j + lane, st.nv, mc, acc);
  v0 += 32 * cnt;
  if (v0 == st.nv) {
    flush_row<MMAX>(rowsum, mcap, warp + kWarps * ri, mc, acc, lane);
    v0 = 0;
    ++ri;
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
    const int nb = st.nrw * ((st.nv / 32 + U - 1) / U);  // batches end at row ends
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
// What a GEMV's prologue hands to its body: the CTA's row plan, the list
// counts, and the first weight batch already requested.
struct LinState {
  Plan pl;
  int nf, ne, nx, nrows, pre_phase;
  Batch a;
  LoadCursor lc;
};

// Prologue of CTA `cta` of `ncta`: reads the sub-batch lists into shared
// memory, plans the CTA's rows and requests the first batch of weights (which
// never change, so this may run before the dependency on the previous kernel
// or phase is met).  The lists must be final when this runs.
template <bool XS, int MMAX>
EE_DEV void linear_prologue(const LinearParams& p, int cta, int ncta, uint8_t* smem, LinState& s) {
  int32_t* lf = reinterpret_cast<int32_t*>(smem);
  int32_t* le = lf + kListLen;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid < kListLen) {
    lf[tid] = p.list_full ? ld_volatile_i32(p.list_full + tid) : (tid == 0 ? p.m_direct_full : tid - 1);
    le[tid] = p.list_exit ? ld_volatile_i32(p.list_exit + tid) : (tid == 0 ? p.m_direct_exit : tid - 1);
  }
  __syncthreads();
  s.nf = p.w ? min(lf[0], EE_MAX_BATCH) : 0;
  s.ne = p.wq ? min(le[0], EE_MAX_BATCH) : 0;
  s.nx = s.nf + s.ne;  // XS mode: rows staged (full rows first, then exit rows)
  const int npairs = p.N >> 1;
  s.pl.r0 = 2 * (int)(((long long)cta * npairs) / ncta);
  s.pl.r1 = 2 * (int)(((long long)(cta + 1) * npairs) / ncta);
  s.pl.mcap = p.mcap;
  s.pl.passes[0] = (s.nf + s.pl.mcap - 1) / s.pl.mcap;
  s.pl.passes[1] = (s.ne + s.pl.mcap - 1) / s.pl.mcap;
  s.nrows = s.pl.r1 - s.pl.r0;
  s.pre_phase = -1;
  // A small int4 slice (the exit copy's QKV and O rows of a CTA) is asked of
  // L2 as a whole before the dependency wait: under programmatic dependent
  // launch the CTA may already be resident while the previous kernel runs.
  if (threadIdx.x == 0 && s.pl.passes[1] > 0 && p.wq) {
    const size_t rb = (size_t)p.K / 2, sb = (size_t)p.sstride * 2;
    const size_t qb = (size_t)s.nrows * rb, qs = (size_t)s.nrows * sb;
    const uint8_t* qa = p.wq + (size_t)s.pl.r0 * rb;
    const uint8_t* sa = reinterpret_cast<const uint8_t*>(p.ws) + (size_t)s.pl.r0 * sb;
    if (qb > 0 && qb <= kL2PrefetchMax && qb % 16 == 0 && ((uintptr_t)qa & 15) == 0)
      asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(qa), "r"((uint32_t)qb) : "memory");
    if (qs > 0 && qs <= kL2PrefetchMax && qs % 16 == 0 && ((uintptr_t)sa & 15) == 0)
      asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(sa), "r"((uint32_t)qs) : "memory");
  }
  if (s.pl.passes[0] > 0) {
    const Stream st = make_stream<0>(p, s.pl, warp);
    if (st.nv % 32 == 0) {
      s.lc = load_start<0>(p, st, lane);
      load_batch<0, MMAX>(p, st, s.lc, s.a);
      s.pre_phase = 0;
    }
  } else if (s.pl.passes[1] > 0) {
    const Stream st = make_stream<1>(p, s.pl, warp);
    if (st.nv % 32 == 0) {
      s.lc = load_start<1>(p, st, lane);
      load_batch<1, MMAX>(p, st, s.lc, s.a);
      s.pre_phase = 1;
    }
  }
}

// Body: the activations (written by the previous kernel or phase) are staged
// after the dependency wait, the rows are streamed and the epilogues run; a
// head launch's last CTA merges the partials.
template <bool XS, int MMAX>
EE_DEV void linear_body(const LinearParams& p, int ncta, uint8_t* smem, LinState& s, int* s_last) {
  int32_t* lf = reinterpret_cast<int32_t*>(smem);
  int32_t* le = lf + kListLen;
  float* hst = reinterpret_cast<float*>(smem + 2 * kListLen * 4 + 16);
  uint8_t* xs = smem + kHeaderBytes;
  float* rowsum = reinterpret_cast<float*>(xs + (XS ? (size_t)p.xs_rows * p.K * 2 : 0));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  wait_and_stage<XS>(p, lf, le, s.nf, s.nx, xs, hst, tid, warp, lane);
  // each phase's code exists once (the kernel stays small in the instruction cache)
#pragma unroll 1
  for (int phase = 0; phase < 2; ++phase) {
    if (phase == 0)
      run_phase<XS, MMAX, 0>(p, s.pl, lf, s.nf, 0, xs, rowsum, hst, s.nrows, tid, warp, lane, s.a, s.lc,
                             s.pre_phase == 0);
    else
      run_phase<XS, MMAX, 1>(p, s.pl, le, s.ne, s.nf, xs, rowsum, hst, s.nrows, tid, warp, lane, s.a, s.lc,
                             s.pre_phase == 1);
  }
  // A head over empty lists (every sequence left at an earlier checkpoint)
  // has nothing to merge or decide: the lists stay as they are.  Every CTA
  // read the same lists, so all of them return here and the counter stays 0.
  if (p.epi == EPI_HEAD && s.nf == 0 && s.ne == 0) return;
  if (p.epi == EPI_HEAD) {
    // Last CTA to finish merges the per-CTA partials (no spin wait: a counter).
    __syncthreads();
    if (tid == 0) {
      __threadfence();
      const int old = atomicAdd(p.head_counter, 1);
      *s_last = (old == ncta - 1);
    }
    __syncthreads();
    if (!*s_last) return;
    head_finalize(p, ncta, lf, le, s.nf, hst);
  }
}

}  // namespace
}  // namespace ee
