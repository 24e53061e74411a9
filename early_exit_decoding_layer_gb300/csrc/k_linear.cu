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
// Data flow per CTA (persistent, one per SM): each CTA owns a contiguous,
// pair-aligned range of output rows, which is one contiguous byte range of the
// row-major weights.  Warp 8's lane 0 streams that range through a ring of
// shared-memory stages, each filled by ONE 16 KB bulk asynchronous copy
// (cp.async.bulk, completion counted on an mbarrier, L2 evict-first; plus one
// 512-byte copy of the stage's int4 scales): the copy engine reaches HBM peak
// only with large requests (1 KB requests stall near 2.5 TB/s on GB300).  The
// weights of the first stages are requested before the grid dependency wait,
// so they stream while the previous kernel finishes; the activations of the
// step's rows (fp16, a few KB per sequence) are bulk-copied into shared memory
// after it.  Warps 0-7 consume: each takes an eighth of a stage, maps every
// 16-byte vector back to (row, column), accumulates per row in registers and
// adds each row's partial into per-row sums in shared memory (one warp
// reduction when the warp's slice lies in one row).  The epilogue (RoPE + KV
// write, SwiGLU, residual add, head statistics) runs once over the CTA's rows.
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

constexpr int kConsumerWarps = 8;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kThreads = kConsumers + 32;
constexpr int kStageW = 16384;  // weight bytes per stage: one bulk copy
constexpr int kStageS = 512;    // int4 scale bytes per stage (16 KB of nibbles = 256 groups)
constexpr int kStageBytes = kStageW + kStageS;
constexpr int kMaxStages = 6;
constexpr int kMM = 8;  // sequences per pass over the weights

// Shared memory: header (barriers, lists, head statistics), the staged
// activations (XS mode), the per-row sums [rows][mcap], then the ring.
constexpr size_t kHeaderBytes = 1536;
constexpr size_t kXsMaxBytes = 48 * 1024;
constexpr size_t kSmemTarget = 112 * 1024;  // two CTAs per SM: the next kernel's CTA can prefetch
constexpr size_t kSmemMax = 160 * 1024;  // attribute; every plan stays below it
static_assert((2 * kMaxStages + 1) * 8 <= 128, "barriers");
static_assert(128 + 2 * kListLen * 4 + 8 + kConsumerWarps * kMM * 3 * 4 <= kHeaderBytes, "header overflow");

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

// Bytes of the per-row sums, rounded up so that the ring behind them starts on
// a 16-byte boundary (bulk copies need it).
__host__ __device__ inline size_t rowsum_bytes(int rows_cap, int mcap) {
  return ((size_t)rows_cap * mcap * 4 + 15) / 16 * 16;
}

// Stage geometry of one phase.  Rows of rb bytes are never split across
// warps: row r of a CTA belongs to consumer warp r % 8.  A stage is either nr
// whole rows (rb <= 16 KB) or one of nparts equal parts of a row (rb > 16 KB).
struct Geo {
  int rb;      // bytes per row
  int S;       // bytes per full stage
  int nr;      // whole rows per stage, or 0 when a stage is part of a row
  int nparts;  // stages per row when nr == 0
};

__host__ __device__ inline Geo make_geo(int rb) {
  Geo g;
  g.rb = rb;
  if (rb <= kStageW) {
    g.nr = kStageW / rb;
    g.nparts = 1;
    g.S = g.nr * rb;
  } else {
    int n = (rb + kStageW - 1) / kStageW;
    while ((rb % n != 0 || (rb / n) % 16 != 0) && n < 64) ++n;
    g.nr = 0;
    g.nparts = n;
    g.S = rb / n;
  }
  return g;
}

__host__ __device__ inline bool geo_ok(const Geo& g) {
  return g.S > 0 && g.S <= kStageW && g.S % 16 == 0 && g.rb % 16 == 0 &&
         (g.nr > 0 || g.S * g.nparts == g.rb);
}

// Per-CTA plan shared by the producer and the consumers.  Phase 0 streams
// the bf16 rows [r0, r1) (K*2 bytes each), phase 1 their int4 copy (K/2
// bytes each); each phase runs one pass per group of at most mcap sequences.
struct Plan {
  int r0, r1, mcap;
  int nst[2], passes[2];
  long long rbytes[2];
  Geo geo[2];
  bool sc_staged;  // int4 scales stream with the weights (one 16-byte-aligned slice per stage)
};

EE_DEV void issue_stage(const LinearParams& p, const Plan& pl, int phase, int s, uint8_t* sbase,
                        uint64_t* bar, uint64_t pol) {
  const long long S = pl.geo[phase].S;
  const long long off = (long long)s * S;
  const uint32_t bytes = (uint32_t)min(S, pl.rbytes[phase] - off);
  if (phase == 0) {
    mbar_arrive_expect_tx(bar, bytes);
    bulk_g2s(sbase, reinterpret_cast<const uint8_t*>(p.w + (size_t)pl.r0 * p.K) + off, bytes, bar, pol);
  } else {
    const uint32_t sb = pl.sc_staged ? bytes / 32 : 0;  // one bf16 scale per 64 bytes of nibbles
    mbar_arrive_expect_tx(bar, bytes + sb);
    bulk_g2s(sbase, p.wq + (size_t)pl.r0 * (p.K / 2) + off, bytes, bar, pol);
    if (sb)
      bulk_g2s(sbase + kStageW, p.ws + (size_t)pl.r0 * p.sstride + (size_t)(off / 64), sb, bar, pol);
  }
}

// Dot products of one stage vector (16 bytes of weights) with the mc
// activation rows at column k, accumulated into acc[m].
template <bool XS>
EE_DEV void vec_dot(int phase, const uint4& wv, float sc, const uint16_t* const* xrow, int k, int mc,
                    float* acc) {
  if (phase == 0) {
#pragma unroll
    for (int m = 0; m < kMM; ++m) {
      if (m < mc) {
        const uint4 xv = XS ? *reinterpret_cast<const uint4*>(xrow[m] + k) : ldg_nc_v4(xrow[m] + k);
        acc[m] = dot8_bf16(wv, xv, acc[m]);
      }
    }
  } else {
#pragma unroll
    for (int m = 0; m < kMM; ++m) {
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
  float* rowsum = reinterpret_cast<float*>(xs + (XS ? (size_t)p.xs_rows * p.K * 2 : 0));
  uint8_t* ring = reinterpret_cast<uint8_t*>(rowsum) + rowsum_bytes(p.rows_cap, p.mcap);
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
    pl.mcap = p.mcap;
    pl.geo[0] = make_geo(p.K * 2);
    pl.geo[1] = make_geo(p.K / 2);
    pl.rbytes[0] = (long long)(pl.r1 - pl.r0) * p.K * 2;
    pl.rbytes[1] = (long long)(pl.r1 - pl.r0) * (p.K / 2);
    pl.nst[0] = (int)((pl.rbytes[0] + pl.geo[0].S - 1) / pl.geo[0].S);
    pl.nst[1] = (int)((pl.rbytes[1] + pl.geo[1].S - 1) / pl.geo[1].S);
    pl.passes[0] = (nf + pl.mcap - 1) / pl.mcap;
    pl.passes[1] = (ne + pl.mcap - 1) / pl.mcap;
    pl.sc_staged = (p.K % 512 == 0) && (p.sstride * EE_QUANT_GROUP == p.K) && (pl.geo[1].S % 512 == 0);
  }

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol = l2_evict_first_policy();
      const uint32_t total =
          (uint32_t)(pl.passes[0] * pl.nst[0] + pl.passes[1] * pl.nst[1]);
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
          for (int s = 0; s < pl.nst[phase]; ++s, ++it) {
            if (!xdone && it == prefill) stage_x();
            const int st = it % nst;
            const uint32_t n = it / nst;
            if (n > 0 && !mbar_wait_bounded(&empty[st], (n - 1) & 1, p.err, DERR_EMPTY_WAIT)) {
              ok = false;
              break;
            }
            issue_stage(p, pl, phase, s, ring + (size_t)st * kStageBytes, &full[st], pol);
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
    const int nrows = pl.r1 - pl.r0;
    uint32_t it = 0;
    for (int phase = 0; phase < 2; ++phase) {
      const int nlist = phase == 0 ? nf : ne;
      const int32_t* lst = phase == 0 ? lf : le;
      const int xbase = phase == 0 ? 0 : nf;  // XS row of the phase's first sequence
      for (int pass = 0; pass < pl.passes[phase]; ++pass) {
        const int m0 = pass * pl.mcap;
        const int mc = min(pl.mcap, nlist - m0);
        int seqs[kMM];
        const uint16_t* xrow[kMM];
#pragma unroll
        for (int m = 0; m < kMM; ++m) {
          const int mm = min(m, mc - 1);
          seqs[m] = lst[1 + m0 + mm];
          xrow[m] = XS ? reinterpret_cast<const uint16_t*>(xs) + (size_t)(xbase + m0 + mm) * p.K
                       : p.xh + (size_t)seqs[m] * p.x_stride;
        }
        const Geo& g = pl.geo[phase];
        const int epb = phase == 0 ? 1 : 4;  // elements per 2 bytes: bf16 1, int4 4
        float acc[kMM];  // carried across the parts of a row longer than a stage
#pragma unroll
        for (int m = 0; m < kMM; ++m) acc[m] = 0.0f;
        for (int s = 0; s < pl.nst[phase]; ++s, ++it) {
          const int st = it % nst;
          // every warp waits for every stage, so that its arrival on the empty
          // barrier below always belongs to this use of the stage
          if (ok) ok = mbar_wait_bounded(&full[st], (it / nst) & 1, p.err, DERR_FULL_WAIT);
          ok = __all_sync(0xffffffffu, ok);
          const uint8_t* sw = ring + (size_t)st * kStageBytes;
          const long long off = (long long)s * g.S;
          const int bytes = (int)min((long long)g.S, pl.rbytes[phase] - off);
          if (ok) {
            if (g.nr > 0) {
              const int row0 = s * g.nr, nrs = bytes / g.rb;
              for (int rr = (warp - row0 % kConsumerWarps + kConsumerWarps) % kConsumerWarps; rr < nrs;
                   rr += kConsumerWarps) {
                const int row = row0 + rr;
                const int rbase = rr * g.rb;
#pragma unroll
                for (int m = 0; m < kMM; ++m) acc[m] = 0.0f;
                for (int v = lane; v < g.rb / 16; v += 32) {
                  const uint4 wv = *reinterpret_cast<const uint4*>(sw + rbase + v * 16);
                  const int k = v * 8 * epb;
                  float sc = 0.0f;
                  if (phase == 1)
                    sc = pl.sc_staged
                             ? bf16_bits_to_float(reinterpret_cast<const uint16_t*>(sw + kStageW)[(rbase + v * 16) >> 6])
                             : bf16_bits_to_float(__ldg(p.ws + (size_t)(pl.r0 + row) * p.sstride + k / EE_QUANT_GROUP));
                  vec_dot<XS>(phase, wv, sc, xrow, k, mc, acc);
                }
#pragma unroll
                for (int m = 0; m < kMM; ++m) {
                  if (m < mc) {
                    const float t = warp_sum(acc[m]);
                    if (lane == 0) rowsum[row * pl.mcap + m] = t;
                  }
                }
              }
            } else {
              const int row = s / g.nparts, part = s % g.nparts;
              if (row % kConsumerWarps == warp) {
                if (part == 0) {
#pragma unroll
                  for (int m = 0; m < kMM; ++m) acc[m] = 0.0f;
                }
                const int kb = part * g.S;  // byte offset of the part within its row
                for (int v = lane; v < bytes / 16; v += 32) {
                  const uint4 wv = *reinterpret_cast<const uint4*>(sw + v * 16);
                  const int k = (kb + v * 16) / 2 * epb;
                  float sc = 0.0f;
                  if (phase == 1)
                    sc = pl.sc_staged
                             ? bf16_bits_to_float(reinterpret_cast<const uint16_t*>(sw + kStageW)[(v * 16) >> 6])
                             : bf16_bits_to_float(__ldg(p.ws + (size_t)(pl.r0 + row) * p.sstride + k / EE_QUANT_GROUP));
                  vec_dot<XS>(phase, wv, sc, xrow, k, mc, acc);
                }
                if (part == g.nparts - 1) {
#pragma unroll
                  for (int m = 0; m < kMM; ++m) {
                    if (m < mc) {
                      const float t = warp_sum(acc[m]);
                      if (lane == 0) rowsum[row * pl.mcap + m] = t;
                    }
                  }
                }
              }
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty[st]);
        }
        consumer_bar();  // every row sum of this pass is complete
        if constexpr (EPI == EPI_HEAD) {
          Stat stat[kMM];
#pragma unroll
          for (int m = 0; m < kMM; ++m) stat[m] = Stat{-INFINITY, 0.0f, 0x7fffffff};
          for (int r = tid; r < nrows; r += kConsumers) {
#pragma unroll
            for (int m = 0; m < kMM; ++m)
              if (m < mc) stat_push(stat[m], rowsum[r * pl.mcap + m], pl.r0 + r);
          }
#pragma unroll
          for (int m = 0; m < kMM; ++m) {
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
          consumer_bar();
          if (warp == 0 && lane < mc) {
            Stat sm = {-INFINITY, 0.0f, 0x7fffffff};
            for (int w = 0; w < kConsumerWarps; ++w) {
              const float* hs = hst + (w * kMM + lane) * 3;
              sm = stat_merge(sm, Stat{hs[0], hs[1], __float_as_int(hs[2])});
            }
            float* dst = p.head_part + ((size_t)blockIdx.x * EE_MAX_BATCH + m0 + lane) * 4;
            dst[0] = sm.mx;
            dst[1] = sm.sum;
            dst[2] = __int_as_float(sm.arg);
          }
        } else {
          const int npr = nrows >> 1;
          for (int i = tid; i < npr * mc; i += kConsumers) {
            const int pr = i / mc, m = i - pr * mc;
            epi_pair<EPI>(p, seqs[m], pl.r0 + 2 * pr, rowsum[(2 * pr) * pl.mcap + m],
                          rowsum[(2 * pr + 1) * pl.mcap + m]);
          }
        }
        consumer_bar();  // row sums are reused by the next pass
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
                         rowsum_bytes(p.rows_cap, p.mcap) + (size_t)p.nstages * kStageBytes;
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

// Shared-memory plan of one launch: per-row sums for the CTA's rows, the
// activations staged when they fit (at most kMM sequences, 48 KB), and as
// many ring stages as keep the CTA within the two-CTAs-per-SM budget.
static void plan_smem(LinearParams& p, int grid) {
  const int max_rows = p.max_rows < 1 ? 1 : p.max_rows;
  p.mcap = max_rows < kMM ? max_rows : kMM;
  const int npairs = p.N / 2;
  p.rows_cap = 2 * ((npairs + grid - 1) / grid);
  const size_t rs = rowsum_bytes(p.rows_cap, p.mcap);
  const size_t xb = (size_t)max_rows * p.K * 2;
  const size_t fixed = kHeaderBytes + rs;
  bool xs = max_rows <= kMM && xb <= kXsMaxBytes;
  int nst = kMaxStages;
  if (xs) {
    const long long room = (long long)kSmemTarget - (long long)(fixed + xb);
    nst = room > 0 ? (int)(room / kStageBytes) : 0;
    if (nst > kMaxStages) nst = kMaxStages;
    if (nst < 4) xs = false;
  }
  if (!xs) {
    const long long room = (long long)kSmemTarget - (long long)fixed;
    nst = room > 0 ? (int)(room / kStageBytes) : 0;
    if (nst > kMaxStages) nst = kMaxStages;
    if (nst < 2) nst = 2;
  }
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

bool linear_shape_ok(int K) {
  if (K < 32 || K % 32) return false;
  return geo_ok(make_geo(K * 2)) && geo_ok(make_geo(K / 2));
}

int linear_grid(int N, int num_sms) {
  const int pairs = N / 2;
  return pairs < num_sms ? (pairs > 0 ? pairs : 1) : num_sms;
}

cudaError_t launch_linear(const LinearParams& p_in, int grid, bool pdl, cudaStream_t st) {
  LinearParams p = p_in;
  plan_smem(p, grid);
  const size_t smem = kHeaderBytes + (p.xs_rows > 0 ? (size_t)p.xs_rows * p.K * 2 : 0) +
                      rowsum_bytes(p.rows_cap, p.mcap) + (size_t)p.nstages * kStageBytes;
  if (smem > kSmemMax) return cudaErrorInvalidConfiguration;
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
