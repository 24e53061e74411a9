// Tensor-core GEMM for steps whose batch is too large for the GEMV to stage:
// Y[m, n] = sum_k X[m, k] W[n, k] for the sequences m of one sub-batch list,
// on the 5th-generation tensor cores (tcgen05.mma, fp32 accumulators in
// tensor memory).
//
// The weights are the MMA's A operand (M = 128 rows of W per tile) and the
// listed sequences' activations its B operand (N columns), both K-major:
//  * full sub-batch (bf16 weights, MODE 0): A tiles come from HBM by TMA with
//    the 128-byte swizzle.  The fp16 activations are split into a bf16 high
//    part and a bf16 remainder (x = hi + lo, 16 significant bits), so the
//    bf16 x bf16 products keep the activations' precision: B has nc hi rows
//    and nc lo rows (N = 2 nc, nc = 32 for lists of up to 32 sequences, else
//    64) and the epilogue adds the two halves of D.  Building B each stage
//    is the producers' work, so the smaller tile halves it.
//  * exit sub-batch (int4 weights, MODE 1): the int4 copy is kept in a
//    layout of its own (k_int4_tc_layout): per 128-row tile and 64-column K
//    step one contiguous block of two halves (columns 0-31, 32-63), each 128
//    rows x 16 bytes of nibbles, then the rows' 128 bf16 scales (4352
//    bytes), which one bulk copy brings into a shared-memory ring.  Producer warps dequantise their row of it to fp16
//    q * s (exact: an 8-bit scale times a 4-bit integer fits fp16's 11
//    bits) and store it into the swizzled A tile; B holds the fp16
//    activations (N = 32 for lists of up to 32 sequences, else 64).  The
//    int4 weights are never written back to HBM.
// Producer warps also gather the listed sequences' activations (fp16, pair
// order) into the B tiles.  One thread issues the MMAs; a stage is released
// by tcgen05.commit when its MMAs have consumed it.
//
// Work unit = (128-row tile, K split).  With several splits per tile each
// CTA writes its fp32 partial tile; the last CTA of the tile (an atomic
// counter, nothing waits) adds them in split order, so results do not depend
// on timing, and runs the epilogue shared with the GEMV (RoPE + K/V write,
// residual, SwiGLU, fp16 output) or the vocabulary-head statistics.
// One launch serves both lists of a projection: the full list's units come
// first in the grid, then (where sequences may have exited) the exit list's,
// each with partials and counters of its own.  A list that is empty returns
// at once, so its CTAs leave room for the other list's in the same launch.
#include <cuda.h>
#include <math.h>

#include "ee_common.cuh"
#include "ee_epilogue.cuh"
#include "ee_head.cuh"
#include "ee_kernels.cuh"

namespace ee {

namespace {

constexpr int kBM = 128;  // weight rows per tile (MMA M)
constexpr int kBK = 64;   // K elements per stage (one 128-byte swizzle row)
constexpr int kMaxStages = 4;
constexpr uint32_t kQ4Block = kBM * 32 + kBM * 2;  // int4 tile-step block: nibbles + scales
constexpr int kRawSlots = 5;  // MODE 1: int4 blocks in flight per CTA (their own ring)
constexpr int kCols = 64;  // sequences per launch at most (EE_MAX_BATCH)
constexpr int kTcThreads = 192;  // warps 0-3 producers + epilogue, 4 TMA, 5 MMA
constexpr uint32_t kABytes = kBM * kBK * 2;
static_assert(kCols == EE_MAX_BATCH, "one launch covers the whole list");

// Stage ring: the A tile and the B tile (N rows) of one K step per stage.
// Two CTAs per SM fit in shared memory with three bf16 stages (N up to 128)
// or four int4 ones (N = 64).  A fourth bf16 stage for N = 64 measured no
// faster: the per-stage B build, not the bytes in flight, sets the pace.
constexpr uint32_t stage_bytes(int n) { return kABytes + (uint32_t)n * kBK * 2; }
// MODE 1 keeps its raw int4 blocks in a ring of their own, refilled as
// soon as the producers have read a block.
constexpr int stage_count(int mode) { return 3; }
template <int MODE>
constexpr size_t kTcSmem = (size_t)stage_count(MODE) * stage_bytes(MODE == 0 ? 2 * kCols : kCols) +
                           (MODE == 1 ? (size_t)kRawSlots * kQ4Block : 0) + 1024;
static_assert(kTcSmem<1> <= kTcSmem<0>, "MODE 1 fits in MODE 0's shared memory");

// Shared memory descriptor of a K-major tile with 128-byte rows and the
// 128-byte swizzle: start address, stride between 8-row groups (1024 B),
// descriptor version 1, swizzle mode 2 (leading offset unused: 1).
EE_DEV uint64_t smem_desc_sw128(uint32_t saddr) {
  uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFF);
  d |= (uint64_t)1 << 16;
  d |= (uint64_t)(1024 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// Instruction descriptor, kind::f16: fp32 accumulators, A and B of type
// `ab` (0 = f16, 1 = bf16), both K-major, N and M given.
constexpr uint32_t instr_desc(uint32_t ab, int n, int m) {
  return (1u << 4) | (ab << 7) | (ab << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

// Byte offset of 16-byte chunk j (8 elements) of row r in a 128B-swizzled tile.
EE_DEV uint32_t sw128(int r, int j) { return (uint32_t)(r * 128 + ((j ^ (r & 7)) << 4)); }

EE_DEV void st_shared_v4(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

EE_DEV void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

EE_DEV void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(map), "r"(x), "r"(y), "r"(smem_addr(bar))
      : "memory");
}

// x = hi + lo for two values: hi their bf16 roundings (one paired
// conversion), lo the remainders, exact in bf16 for fp16 inputs.
EE_DEV void split_bf16x2(float a, float b, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  const __nv_bfloat162 l = __floats2bfloat162_rn(a - __uint_as_float(hi << 16), b - __uint_as_float(hi & 0xFFFF0000u));
  lo = *reinterpret_cast<const uint32_t*>(&l);
}

// 8 fp16 activations stored in pair order (0,4,1,5,2,6,3,7) -> natural order.
EE_DEV void unpair8(const uint4& v, float* x) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
    x[i] = f.x;
    x[i + 4] = f.y;
  }
}

struct TcShared {
  uint64_t full[kMaxStages], empty[kMaxStages], raw[kRawSlots], raw_free[kRawSlots], done;
  uint32_t tmem;
  int32_t lf[kListLen], le[kListLen];
  int last;
  float red[4 * 3 * 16];   // head statistics: [warp][3][column chunk]
  float res[2 * EE_MAX_BATCH];
  EpiSeq col[kCols];       // per-column (sequence) epilogue values
};

template <int MODE>
__device__ __forceinline__ void gemm_tc_body(const TcParams& tp, TcShared& sh, int unit) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* tiles = reinterpret_cast<uint8_t*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const LinearParams& p = tp.lp;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int tile = unit / tp.ksplit, split = unit - tile * tp.ksplit;
  const int units = tp.ntiles * tp.ksplit;  // per list
  const int row0 = tile * kBM;
  const int ks0 = split * tp.nks, ks1 = min(tp.nk, ks0 + tp.nks);  // K steps of this unit
  const int nks = ks1 - ks0;

  if (p.lists_after_wait) grid_dep_wait();
  if (tid < kListLen) {
    sh.lf[tid] = p.list_full ? ld_volatile_i32(p.list_full + tid) : (tid == 0 ? p.m_direct_full : tid - 1);
    sh.le[tid] = p.list_exit ? ld_volatile_i32(p.list_exit + tid) : (tid == 0 ? p.m_direct_exit : tid - 1);
  }
  __syncthreads();
  const int32_t* lst = MODE == 0 ? sh.lf : sh.le;
  const int ncol = min(lst[0], kCols);
  if (ncol == 0 || nks <= 0) {  // uniform over the grid: no unit has work
    grid_dep_wait();
    grid_dep_launch();
    return;
  }
  // B rows: bf16 keeps nc hi rows then nc lo rows; int4 keeps nc fp16 rows
  const int nc = ncol <= kCols / 2 ? kCols / 2 : kCols;  // columns built (bf16: x2 for hi, lo)
  const int N = MODE == 0 ? 2 * nc : nc;
  const int nst = stage_count(MODE);
  const uint32_t stage_b = stage_bytes(N);

  if (tid == 0) {
    for (int s = 0; s < nst; ++s) {
      mbar_init(&sh.full[s], MODE == 0 ? 129 : 128);
      mbar_init(&sh.empty[s], 1);
    }
    for (int s = 0; s < kRawSlots; ++s) {
      mbar_init(&sh.raw[s], 1);
      mbar_init(&sh.raw_free[s], 4);  // one arrival per producer warp
    }
    mbar_init(&sh.done, 1);
    fence_mbar_init();
  }
  if (warp == 5) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(&sh.tmem)),
                 "r"(N)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = sh.tmem;
  const uint32_t tiles_s = smem_addr(tiles);
  uint8_t* raw_ring = tiles + (size_t)nst * stage_b;  // MODE 1: raw int4 blocks

  if (warp == 4) {
    // TMA of the bf16 weight tiles; the first stages go out before the
    // dependency wait (weights never change).
    if (MODE == 0 && lane == 0) {
      const CUtensorMap* map = &tp.amap;
      for (int i = 0, s = 0, n = 0; i < nks; ++i) {  // stage s of ring pass n
        if (i == nst) grid_dep_wait();
        if (n > 0 && !mbar_wait_bounded(&sh.empty[s], (n - 1) & 1, p.err, DERR_EMPTY_WAIT)) break;
        mbar_arrive_expect_tx(&sh.full[s], kABytes);
        tma_load_2d(tiles_s + s * stage_b, map, (ks0 + i) * kBK, row0, &sh.full[s]);
        if (++s == nst) s = 0, ++n;
      }
      if (nks <= nst) grid_dep_wait();
    } else if (MODE == 1 && lane == 0) {
      // the int4 blocks of this unit's K steps, one bulk copy each, into the
      // raw ring; a slot is refilled once every producer warp has read it
      const uint8_t* src = tp.q4t + ((size_t)tile * tp.nk + ks0) * kQ4Block;
      for (int i = 0, s = 0, n = 0; i < nks; ++i) {
        if (i == kRawSlots) grid_dep_wait();
        if (n > 0 && !mbar_wait_bounded(&sh.raw_free[s], (n - 1) & 1, p.err, DERR_EMPTY_WAIT)) break;
        mbar_arrive_expect_tx(&sh.raw[s], kQ4Block);
        bulk_g2s(raw_ring + (size_t)s * kQ4Block, src + (size_t)i * kQ4Block, kQ4Block, &sh.raw[s],
                 l2_evict_first_policy());
        if (++s == kRawSlots) s = 0, ++n;
      }
      if (nks <= kRawSlots) grid_dep_wait();
    } else {
      grid_dep_wait();
    }
    grid_dep_launch();
  } else if (warp == 5) {
    grid_dep_wait();
    grid_dep_launch();
    if (lane == 0) {
      const uint32_t idesc = instr_desc(MODE == 0 ? 1u : 0u, N, kBM);
      for (int i = 0, s = 0, n = 0; i < nks; ++i) {
        if (!mbar_wait_bounded(&sh.full[s], n & 1, p.err, DERR_FULL_WAIT)) break;
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const uint32_t a_s = tiles_s + s * stage_b, b_s = a_s + kABytes;
#pragma unroll
        for (int kk = 0; kk < kBK / 16; ++kk) {
          const uint64_t ad = smem_desc_sw128(a_s + kk * 32), bd = smem_desc_sw128(b_s + kk * 32);
          const uint32_t acc = (i > 0 || kk > 0) ? 1u : 0u;
          asm volatile(
              "{ .reg .pred p; setp.ne.b32 p, %4, 0; tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p; }" ::"r"(tmem),
              "l"(ad), "l"(bd), "r"(idesc), "r"(acc)
              : "memory");
        }
        asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                         smem_addr(&sh.empty[s]))
                     : "memory");
        if (++s == nst) s = 0, ++n;
      }
      asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                       smem_addr(&sh.done))
                   : "memory");
    }
  } else {
    // producers: the B tile (activations of the listed sequences) and, for
    // int4, the dequantised A tile of every stage.  The activations are read
    // ahead of the stores in registers (PD stages, from L2); int4 blocks come
    // through the raw ring.
    grid_dep_wait();
    grid_dep_launch();
    constexpr int PD = 3;  // stages of activation reads in flight per thread
    // B entry e (of nb = 32 or 64) and part of the stage's 8 column chunks:
    // the 128 threads share the nb entries, nch chunks each
    const int nb = nc, nch = nb / 16;
    const int e = tid & (nb - 1), part = tid / nb;
    const bool have = e < ncol;
    const uint16_t* xrow = p.xh + (size_t)(have ? lst[1 + e] : 0) * p.x_stride + 8 * nch * part;
    uint4 xr[PD][4];
    auto fetch = [&](int slot, int i) {
      if (i >= nks) return;
      const int k0 = (ks0 + i) * kBK;
#pragma unroll
      for (int c = 0; c < 4; ++c)
        if (c < nch)
          xr[slot][c] = have ? *reinterpret_cast<const uint4*>(xrow + k0 + 8 * c) : make_uint4(0, 0, 0, 0);
    };
#pragma unroll
    for (int d = 0; d < PD; ++d) fetch(d, d);
    int s = 0, n = 0;  // stage of ring pass n
    for (int i0 = 0; i0 < nks; i0 += PD) {
#pragma unroll
      for (int u = 0; u < PD; ++u) {
        const int i = i0 + u;
        if (i >= nks) break;
        if (n > 0 && !mbar_wait_bounded(&sh.empty[s], (n - 1) & 1, p.err, DERR_EMPTY_WAIT)) {
          i0 = nks;  // give up: the MMA side times out on the stages it misses
          break;
        }
        const uint32_t a_s = tiles_s + s * stage_b, b_s = a_s + kABytes;
        // B: nch chunks of 8 activations of entry e (bf16: rows e and nc + e)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          if (c >= nch) break;
          const uint4 v = xr[u][c];
          const int j = nch * part + c;
          if (MODE == 0) {
            float x[8];
            unpair8(v, x);
            uint32_t hi[4], lo[4];
#pragma unroll
            for (int t = 0; t < 4; ++t) split_bf16x2(x[2 * t], x[2 * t + 1], hi[t], lo[t]);
            st_shared_v4(b_s + sw128(e, j), make_uint4(hi[0], hi[1], hi[2], hi[3]));
            st_shared_v4(b_s + sw128(nc + e, j), make_uint4(lo[0], lo[1], lo[2], lo[3]));
          } else {
            // pair order (x0,x4) (x1,x5) (x2,x6) (x3,x7) -> natural order
            st_shared_v4(b_s + sw128(e, j), make_uint4(__byte_perm(v.x, v.y, 0x5410), __byte_perm(v.z, v.w, 0x5410),
                                                       __byte_perm(v.x, v.y, 0x7632), __byte_perm(v.z, v.w, 0x7632)));
          }
        }
        if constexpr (MODE == 1) {
          // A: row tid of the tile, the stage's 64 columns, from the raw
          // block (row tid's 4 words in each half -- a warp reads 512
          // contiguous bytes per half -- then its scale).  Word j holds columns
          // c = 8j .. c+7 as nibbles (c, c+2, c+4, c+6 | c+1, c+3, c+5, c+7):
          // one masking LOP3 per pair puts (c, c+1) or (c+4, c+5) under the
          // fp16 exponent of 1024 with the sign bits flipped (1024 + q + 8),
          // and (c+2, c+3) or (c+6, c+7) at 16x (1024 + 16 (q + 8)); one
          // HADD2 or HFMA2 leaves q exactly, one HMUL2 applies the scale.
          const int rs = i % kRawSlots, rn = i / kRawSlots;
          if (!mbar_wait_bounded(&sh.raw[rs], rn & 1, p.err, DERR_FULL_WAIT)) {
            i0 = nks;
            break;
          }
          const uint8_t* blk = raw_ring + (size_t)rs * kQ4Block;
          const uint4 w0 = *reinterpret_cast<const uint4*>(blk + tid * 16);
          const uint4 w1 = *reinterpret_cast<const uint4*>(blk + (kBM + tid) * 16);
          const uint16_t sb = *reinterpret_cast<const uint16_t*>(blk + kBM * 32 + tid * 2);
          __syncwarp();
          if (lane == 0) mbar_arrive(&sh.raw_free[rs]);  // this warp is done reading the block
          const __half2 s2 = __float2half2_rn(bf16_bits_to_float(sb));
          const __half2 m1032 = __half2half2(__ushort_as_half((unsigned short)0xE408));  // -1032
          const __half2 r16 = __half2half2(__ushort_as_half((unsigned short)0x2C00));    // 1/16
          const __half2 m72 = __half2half2(__ushort_as_half((unsigned short)0xD480));    // -72
          const uint32_t words[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const uint32_t t = words[j], t8 = t >> 8;
            const uint32_t m0 = (t & 0x000F000Fu) ^ 0x64086408u, m1 = (t & 0x00F000F0u) ^ 0x64806480u;
            const uint32_t m2 = (t8 & 0x000F000Fu) ^ 0x64086408u, m3 = (t8 & 0x00F000F0u) ^ 0x64806480u;
            const __half2 q01 = __hmul2(__hadd2(*reinterpret_cast<const __half2*>(&m0), m1032), s2);
            const __half2 q23 = __hmul2(__hfma2(*reinterpret_cast<const __half2*>(&m1), r16, m72), s2);
            const __half2 q45 = __hmul2(__hadd2(*reinterpret_cast<const __half2*>(&m2), m1032), s2);
            const __half2 q67 = __hmul2(__hfma2(*reinterpret_cast<const __half2*>(&m3), r16, m72), s2);
            st_shared_v4(a_s + sw128(tid, j),
                         make_uint4(*reinterpret_cast<const uint32_t*>(&q01), *reinterpret_cast<const uint32_t*>(&q23),
                                    *reinterpret_cast<const uint32_t*>(&q45), *reinterpret_cast<const uint32_t*>(&q67)));
          }
        }
        fence_proxy_async();
        mbar_arrive(&sh.full[s]);
        fetch(u, i + PD);  // this slot's next stage
        if (++s == nst) s = 0, ++n;
      }
    }
  }

  // ---------------------------------------------------------------- epilogue
  if (warp < 4) {
    const bool ok = mbar_wait_bounded(&sh.done, 0, p.err, DERR_FULL_WAIT);
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const int rl = warp * 32 + lane;  // tile row = TMEM lane
    const uint32_t tl = tmem + ((uint32_t)(warp * 32) << 16);
    float* part = tp.part + ((size_t)MODE * units + unit) * kCols * kBM;
    for (int c0 = 0; c0 < ncol; c0 += 16) {
      uint32_t v[16], w[16];
      asm volatile(
          "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
          : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]),
            "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
          : "r"(tl + c0));
      if (MODE == 0) {
        asm volatile(
            "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
            : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]), "=r"(w[6]), "=r"(w[7]),
              "=r"(w[8]), "=r"(w[9]), "=r"(w[10]), "=r"(w[11]), "=r"(w[12]), "=r"(w[13]), "=r"(w[14]), "=r"(w[15])
            : "r"(tl + nc + c0));
      }
      asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const float y = __uint_as_float(v[j]) + (MODE == 0 ? __uint_as_float(w[j]) : 0.0f);
        if (c0 + j < ncol) part[(size_t)(c0 + j) * kBM + rl] = ok ? y : 0.0f;
      }
    }
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 5) {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(N) : "memory");
  }
  // the last CTA of this tile adds the splits in order and runs the epilogue
  if (tid == 0) {
    __threadfence();
    const int old = tp.ksplit > 1 ? atomicAdd(tp.tile_cnt + MODE * tp.ntiles + tile, 1) : 0;
    sh.last = (old == tp.ksplit - 1);
  }
  __syncthreads();
  if (!sh.last) return;
  __threadfence();
  if (warp >= 4) return;
  const int rl = warp * 32 + lane;
  const int r = row0 + rl;
  const float* parts = tp.part + ((size_t)MODE * units + (size_t)tile * tp.ksplit) * kCols * kBM;
  // per-column values once (one round trip), not per row pair
  if (tid < ncol && p.epi != EPI_HEAD) sh.col[tid] = epi_seq(p, lst[1 + tid]);
  asm volatile("bar.sync 1, 128;" ::: "memory");
  for (int c0 = 0; c0 < ncol; c0 += 16) {
    float y[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) y[j] = 0.0f;
    // splits added in order; the loads of 4 splits x 16 columns are issued
    // together (independent), the sums keep the split order
    int sp = 0;
    for (; sp + 4 <= tp.ksplit; sp += 4) {
      float v[4][16];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float* src = parts + ((size_t)(sp + u) * kCols + c0) * kBM + rl;
#pragma unroll
        for (int j = 0; j < 16; ++j) v[u][j] = c0 + j < ncol ? __ldcg(src + (size_t)j * kBM) : 0.0f;
      }
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int j = 0; j < 16; ++j) y[j] += v[u][j];
    }
    for (; sp < tp.ksplit; ++sp) {
      const float* src = parts + ((size_t)sp * kCols + c0) * kBM + rl;
#pragma unroll
      for (int j = 0; j < 16; ++j)
        if (c0 + j < ncol) y[j] += __ldcg(src + (size_t)j * kBM);
    }
    if (p.epi == EPI_HEAD) {
      // per column (sequence): statistics over this tile's rows
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        Stat st = {-INFINITY, 0.0f, 0x7fffffff};
        if (r < p.N) stat_push(st, y[j], r);
        st = stat_warp_merge(st);
        if (lane == 0) {
          sh.red[(warp * 3 + 0) * 16 + j] = st.mx;
          sh.red[(warp * 3 + 1) * 16 + j] = st.sum;
          sh.red[(warp * 3 + 2) * 16 + j] = __int_as_float(st.arg);
        }
      }
      asm volatile("bar.sync 1, 128;" ::: "memory");
      if (tid < 16 && c0 + tid < ncol) {
        Stat st = {-INFINITY, 0.0f, 0x7fffffff};
        for (int w = 0; w < 4; ++w)
          st = stat_merge(st, Stat{sh.red[(w * 3 + 0) * 16 + tid], sh.red[(w * 3 + 1) * 16 + tid],
                                   __float_as_int(sh.red[(w * 3 + 2) * 16 + tid])});
        float* dst = p.head_part + ((size_t)tile * EE_MAX_BATCH + c0 + tid) * 4;
        dst[0] = st.mx;
        dst[1] = st.sum;
        dst[2] = __int_as_float(st.arg);
      }
      asm volatile("bar.sync 1, 128;" ::: "memory");
    } else {
      float yb[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) yb[j] = __shfl_down_sync(0xffffffffu, y[j], 1);
      if ((rl & 1) == 0 && r < p.N) {
        switch (p.epi) {
#define EE_TC_EPI(E)                                                                       \
  case E:                                                                                  \
    _Pragma("unroll") for (int j = 0; j < 16; ++j) if (c0 + j < ncol)                      \
        epi_pair_at<E>(p, sh.col[c0 + j], r, y[j], yb[j]);                                 \
    break;
          EE_TC_EPI(EPI_F32)
          EE_TC_EPI(EPI_QKV)
          EE_TC_EPI(EPI_RESID)
          EE_TC_EPI(EPI_SWIGLU)
          EE_TC_EPI(EPI_X)
#undef EE_TC_EPI
          default: break;
        }
      }
    }
  }
  if (tid == 0 && tp.ksplit > 1) tp.tile_cnt[MODE * tp.ntiles + tile] = 0;
  if (p.epi == EPI_HEAD) {
    // the last tile to finish merges the vocabulary partials
    if (tid == 0) {
      __threadfence();
      const int old = atomicAdd(p.head_counter, 1);
      sh.last = (old == tp.ntiles - 1);
    }
    asm volatile("bar.sync 1, 128;" ::: "memory");
    if (!sh.last) return;
    head_finalize_group(p, tp.ntiles, sh.lf, sh.le, ncol, sh.res, 128);
  }
}

// Profiled steps pass stamp pointers: thread 0 of every CTA records the
// kernel's first start (atomic min) and last end (atomic max) of
// %globaltimer.  Thread 0 passes every barrier of its CTA and returns from
// the body last, so its end is the CTA's end.
__global__ void __launch_bounds__(kTcThreads, 2) k_gemm_tc(const __grid_constant__ TcParams tp) {
  __shared__ TcShared sh;
  if (tp.lp.stamp_start && threadIdx.x == 0) atomicMin(tp.lp.stamp_start, (unsigned long long)globaltimer());
  const int units = tp.ntiles * tp.ksplit;
  if ((int)blockIdx.x < units)
    gemm_tc_body<0>(tp, sh, blockIdx.x);
  else
    gemm_tc_body<1>(tp, sh, blockIdx.x - units);
  if (tp.lp.stamp_end && threadIdx.x == 0) atomicMax(tp.lp.stamp_end, (unsigned long long)globaltimer());
}

}  // namespace

// Row-layout int4 copy -> the tensor-core GEMM's blocks: thread per word of
// a (tile, K step) block, then per scale.  Word j of row r sits in half
// j / 4 at (j / 4) * 128 * 16 + r * 16 + (j % 4) * 4 and holds columns
// c = 64 ks + 8j .. c+7 of row 128 t + r with nibble i = column c + 2i (i < 4)
// or c + 2(i - 4) + 1: the row layout's word at the same columns with its
// even-column nibbles moved to the low half and its odd ones to the high
// half.  Rows past the matrix are zero.
__global__ void __launch_bounds__(256) k_int4_tc_layout(const uint8_t* __restrict__ q, const uint16_t* __restrict__ s,
                                                        int rows, int cols, int sstride, uint8_t* __restrict__ out) {
  const long long nk = cols / kBK, ntiles = (rows + kBM - 1) / kBM;
  const long long words = ntiles * nk * kBM * 8, scales = ntiles * nk * kBM;
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx < words) {
    const int j = (int)(idx & 7), r = (int)((idx >> 3) % kBM);
    const long long blk = (idx >> 3) / kBM, ks = blk % nk, t = blk / nk;
    const long long row = t * kBM + r;
    uint32_t w = 0;
    if (row < rows) {
      const uint32_t src = *reinterpret_cast<const uint32_t*>(q + (size_t)row * (cols / 2) + (ks * kBK + 8 * j) / 2);
#pragma unroll
      for (int i = 0; i < 8; ++i) {  // source nibble i = column c + i
        const uint32_t v = (src >> (4 * i)) & 0xF;
        const int dst = (i & 1) ? 4 + (i >> 1) : (i >> 1);
        w |= v << (4 * dst);
      }
    }
    *reinterpret_cast<uint32_t*>(out + (size_t)blk * kQ4Block + (size_t)((j >> 2) * kBM + r) * 16 + (j & 3) * 4) = w;
  } else if (idx < words + scales) {
    const long long i = idx - words;
    const int r = (int)(i % kBM);
    const long long blk = i / kBM, ks = blk % nk, t = blk / nk;
    const long long row = t * kBM + r;
    const uint16_t sv = row < rows ? s[(size_t)row * sstride + (ks * kBK) / EE_QUANT_GROUP] : 0;
    *reinterpret_cast<uint16_t*>(out + (size_t)blk * kQ4Block + kBM * 32 + (size_t)r * 2) = sv;
  }
}

TcPlan gemm_tc_plan(int N, int K, int num_sms, int max_units) {
  TcPlan pl;
  pl.ntiles = (N + kBM - 1) / kBM;
  pl.nk = K / kBK;
  // Choose the K split that minimises the estimated time: waves of work units
  // (two CTAs per SM), each paying a fixed cost (set-up, pipeline fill,
  // epilogue, its share of the tile's reduction; about 7 us measured) plus
  // its K steps (about 0.75 us each with every SM streaming).
  constexpr double kFixedUs = 7.0, kStepUs = 0.75;
  const int slots = 2 * num_sms;
  int best = 1;
  double best_t = 1e30;
  for (int s = 1; s <= 32 && s <= pl.nk; ++s) {
    const int nks = (pl.nk + s - 1) / s, splits = (pl.nk + nks - 1) / nks;
    const int units = pl.ntiles * splits;
    if (s > 1 && units > max_units) break;
    const int waves = (units + slots - 1) / slots;
    const double t = waves * (kFixedUs + nks * kStepUs);
    if (t < best_t - 1e-9) {
      best_t = t;
      best = s;
    }
  }
  pl.nks = (pl.nk + best - 1) / best;
  pl.ksplit = (pl.nk + pl.nks - 1) / pl.nks;
  return pl;
}

bool gemm_tc_shape_ok(int K) { return K >= kBK && K % kBK == 0; }

size_t gemm_tc_part_floats(int units) { return (size_t)units * kCols * kBM; }

size_t int4_tc_layout_bytes(int rows, int cols) {
  return (size_t)((rows + kBM - 1) / kBM) * (cols / kBK) * kQ4Block;
}

cudaError_t launch_int4_tc_layout(const uint8_t* packed, const uint16_t* scales, int rows, int cols, int sstride,
                                  uint8_t* out, cudaStream_t st) {
  if (rows < 1 || cols % kBK) return cudaErrorInvalidValue;
  const long long blocks = (long long)((rows + kBM - 1) / kBM) * (cols / kBK);
  const long long n = blocks * kBM * 9;
  k_int4_tc_layout<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(packed, scales, rows, cols, sstride, out);
  return cudaGetLastError();
}

cudaError_t gemm_tc_prepare() {
  return cudaFuncSetAttribute(k_gemm_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kTcSmem<0>);
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

bool encode_weight_map(CUtensorMap* map, const uint16_t* w, int N, int K) {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !f)
      return false;
    fn = reinterpret_cast<EncodeTiledFn>(f);
  }
  if (!w || (uintptr_t)w % 16 || K % kBK || N < 1) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)N};
  const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
  const cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)kBM};
  const cuuint32_t es[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(w), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_gemm_tc(const TcParams& tp, bool pdl, cudaStream_t st) {
  if (tp.modes < 1 || tp.modes > 2 || (tp.modes == 2 && !tp.q4t)) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(tp.ntiles * tp.ksplit * tp.modes);
  cfg.blockDim = dim3(kTcThreads);
  cfg.dynamicSmemBytes = kTcSmem<0>;  // MODE 1's layout fits in MODE 0's
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, k_gemm_tc, tp);
}

}  // namespace ee
