// Small kernels of the decode step (RMSNorm, step start with the embedding
// gather) and the load-time kernels (int4 quantiser, row re-layout,
// transpose, fill).
#include <math.h>

#include "ee_common.cuh"
#include "ee_head.cuh"
#include "ee_kernels.cuh"

namespace ee {

namespace {

// ------------------------------------------------------------------ RMSNorm
// x = h * rsqrt(mean(h^2) + eps) * g for every listed sequence, written in
// fp16 in the GEMV kernels' pair order.
__global__ void __launch_bounds__(256) k_rmsnorm(const NormParams p) {
  __shared__ float red[8];
  grid_dep_wait();
  grid_dep_launch();
  const int count = ld_volatile_i32(p.list);
  const int z = blockIdx.x;
  if (z >= count) return;
  const int seq = p.list[1 + z];
  const float* h = p.h + (size_t)seq * p.h_stride;
  const int tid = threadIdx.x;
  float ss = 0.0f;
  for (int i = tid * 8; i < p.d; i += 256 * 8) {
    const float4 a = *reinterpret_cast<const float4*>(h + i);
    const float4 b = *reinterpret_cast<const float4*>(h + i + 4);
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
  if ((tid & 31) == 0) red[tid >> 5] = ss;
  __syncthreads();
  float tot = 0.0f;
#pragma unroll
  for (int w = 0; w < 8; ++w) tot += red[w];
  const float r = rsqrtf(tot / (float)p.d + p.eps);
  uint16_t* xh = p.xh + (size_t)seq * p.x_stride;
  for (int i = tid * 8; i < p.d; i += 256 * 8) {
    const float4 a = *reinterpret_cast<const float4*>(h + i);
    const float4 b = *reinterpret_cast<const float4*>(h + i + 4);
    const uint4 gw = *reinterpret_cast<const uint4*>(p.g + i);
    const float x[8] = {a.x * r * bf16_lo(gw.x), a.y * r * bf16_hi(gw.x), a.z * r * bf16_lo(gw.y),
                        a.w * r * bf16_hi(gw.y), b.x * r * bf16_lo(gw.z), b.y * r * bf16_hi(gw.z),
                        b.z * r * bf16_lo(gw.w), b.w * r * bf16_hi(gw.w)};
    uint4 o;  // pair order: (x0,x4) (x1,x5) (x2,x6) (x3,x7)
    o.x = uint32_t(float_to_half_bits(x[0])) | (uint32_t(float_to_half_bits(x[4])) << 16);
    o.y = uint32_t(float_to_half_bits(x[1])) | (uint32_t(float_to_half_bits(x[5])) << 16);
    o.z = uint32_t(float_to_half_bits(x[2])) | (uint32_t(float_to_half_bits(x[6])) << 16);
    o.w = uint32_t(float_to_half_bits(x[3])) | (uint32_t(float_to_half_bits(x[7])) << 16);
    *reinterpret_cast<uint4*>(xh + i) = o;
  }
}

// ------------------------------------------------------------------ step start
// CTA z handles the z-th participating sequence: position, new KV block,
// embedding gather h = E[token] (fp32), per-step outputs reset.  CTA 0 also
// sets the lists: full = participants, exit = empty, final-head rows.
__global__ void __launch_bounds__(256) k_step_begin(const BeginParams p) {
  const StepDesc* d = p.desc;
  const int z = blockIdx.x, tid = threadIdx.x;
  const int n = min(d->n_part, EE_MAX_BATCH);
  if (z == 0) {
    if (tid < EE_MAX_BATCH) {
      const int v = tid < n ? d->part[tid] : 0;
      p.lists->part[1 + tid] = v;
      p.lists->full[1 + tid] = v;
      p.lists->exitl[1 + tid] = 0;
      p.lists->fin[1 + tid] = tid < d->n_fin ? d->fin[tid] : 0;
      p.lists->forced[tid] = d->forced_exit[tid];
    }
    if (tid == 0) {
      p.lists->part[0] = n;
      p.lists->full[0] = n;
      p.lists->exitl[0] = 0;
      p.lists->fin[0] = min(d->n_fin, EE_MAX_BATCH);
      p.out->err = 0;
      *p.dbg_flag = d->debug;
    }
  }
  if (z >= n) return;
  const int seq = d->part[z];
  const int pos = d->pos[seq];
  if (tid == 0) {
    p.pos[seq] = pos;
    if (d->new_block[seq] >= 0) p.block_table[(size_t)seq * p.bt_stride + (pos >> 4)] = d->new_block[seq];
    p.out->exit_layer[seq] = p.n_layers - 1;
    p.out->next_token[seq] = -1;
  }
  for (int c = tid; c < EE_MAX_CHECKPOINTS; c += 256)
    p.out->conf[seq * EE_MAX_CHECKPOINTS + c] = __int_as_float(0x7fc00000);
  const uint16_t* e = p.embed + (size_t)d->tokens[seq] * p.d;
  float* h = p.h + (size_t)seq * p.h_stride;
  for (int i = tid * 2; i < p.d; i += 512) {
    const uint32_t w = *reinterpret_cast<const uint32_t*>(e + i);
    *reinterpret_cast<float2*>(h + i) = make_float2(bf16_lo(w), bf16_hi(w));
    if (p.hsave) *reinterpret_cast<float2*>(p.hsave + (size_t)seq * p.h_stride + i) = make_float2(bf16_lo(w), bf16_hi(w));
  }
}

// ------------------------------------------------------------------ similarity exit
// CTA z scores entry z of the full list: cos(h_in, h) = (h_in . h) /
// (max(|h_in|, 1e-12) max(|h|, 1e-12)) in fp32, summed in a fixed order.
// The last CTA to finish (a counter, no spin) takes the decision and
// rebuilds the lists.
__global__ void __launch_bounds__(256) k_sts(const StsParams p) {
  __shared__ float red[3][8];
  __shared__ int32_t lf[kListLen], le[kListLen];
  __shared__ int s_last;
  const int z = blockIdx.x, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  grid_dep_wait();
  grid_dep_launch();
  const int nf = min(ld_volatile_i32(p.lists->full), EE_MAX_BATCH);
  if (z < nf) {
    const int seq = ld_volatile_i32(p.lists->full + 1 + z);
    const float4* a = reinterpret_cast<const float4*>(p.h_in + (size_t)seq * p.h_stride);
    const float4* b = reinterpret_cast<const float4*>(p.h + (size_t)seq * p.h_stride);
    float dot = 0.0f, na = 0.0f, nb = 0.0f;
    for (int i = tid; i < p.d / 4; i += 256) {
      const float4 x = a[i], y = b[i];
      dot = fmaf(x.x, y.x, fmaf(x.y, y.y, fmaf(x.z, y.z, fmaf(x.w, y.w, dot))));
      na = fmaf(x.x, x.x, fmaf(x.y, x.y, fmaf(x.z, x.z, fmaf(x.w, x.w, na))));
      nb = fmaf(y.x, y.x, fmaf(y.y, y.y, fmaf(y.z, y.z, fmaf(y.w, y.w, nb))));
    }
    dot = warp_sum(dot);
    na = warp_sum(na);
    nb = warp_sum(nb);
    if (lane == 0) {
      red[0][warp] = dot;
      red[1][warp] = na;
      red[2][warp] = nb;
    }
    __syncthreads();
    if (tid == 0) {
      float sd = 0.0f, sa = 0.0f, sb = 0.0f;
      for (int w = 0; w < 8; ++w) {
        sd += red[0][w];
        sa += red[1][w];
        sb += red[2][w];
      }
      p.score[z] = sd / (fmaxf(sqrtf(sa), 1e-12f) * fmaxf(sqrtf(sb), 1e-12f));
    }
  }
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    s_last = atomicAdd(p.counter, 1) == (int)gridDim.x - 1;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  if (tid < kListLen) {
    lf[tid] = ld_volatile_i32(p.lists->full + tid);
    le[tid] = ld_volatile_i32(p.lists->exitl + tid);
  }
  __syncthreads();
  if (tid == 0) {
    float sc[EE_MAX_BATCH];
    float low = INFINITY;
    for (int m = 0; m < nf; ++m) {
      sc[m] = __ldcg(p.score + m);
      low = fminf(low, sc[m]);
    }
    if (p.batch_min)  // the batch rule: the sequences on the full path exit together
      for (int m = 0; m < nf; ++m) sc[m] = low;
    checkpoint_decide(p.gamma[p.ckpt_index], p.ckpt_index, p.ckpt_layer, sc, 1, lf, le, nf, p.conf_out,
                      p.exit_layer, p.lists);
    __threadfence();
    *p.counter = 0;
  }
}

// ------------------------------------------------------------------ quantiser
// One warp per (row, group of 128 columns): s = bf16(amax / 7) and
// q = clamp(round_half_even(w / s), -8, 7), both divisions IEEE round to
// nearest in fp32; amax = 0 gives s = 0, q = 0.  Lane l handles columns
// 4l..4l+3 of the group and writes their two packed bytes (column 2j in the
// low nibble).
__global__ void __launch_bounds__(256) k_quantize(const uint16_t* w, int rows, int cols,
                                                  uint8_t* packed, uint16_t* scales, int sstride) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ng = (cols + EE_QUANT_GROUP - 1) / EE_QUANT_GROUP;
  const long long gw = (long long)blockIdx.x * 8 + warp;
  if (gw >= (long long)rows * ng) return;
  const int r = (int)(gw / ng), gi = (int)(gw % ng);
  const int c0 = gi * EE_QUANT_GROUP + lane * 4;
  const bool valid = c0 < cols;
  float v[4] = {0.f, 0.f, 0.f, 0.f};
  if (valid) {
    const uint2 u = *reinterpret_cast<const uint2*>(w + (size_t)r * cols + c0);
    v[0] = bf16_lo(u.x);
    v[1] = bf16_hi(u.x);
    v[2] = bf16_lo(u.y);
    v[3] = bf16_hi(u.y);
  }
  float amax = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
  amax = warp_max(amax);
  const uint16_t sb = float_to_bf16_bits(__fdiv_rn(amax, 7.0f));
  const float s = bf16_bits_to_float(sb);
  int q[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    int qi = 0;
    if (s != 0.0f) {
      qi = __float2int_rn(__fdiv_rn(v[i], s));
      qi = qi < -8 ? -8 : (qi > 7 ? 7 : qi);
    }
    q[i] = qi;
  }
  if (valid) {
    const uint16_t two = (uint16_t)((q[0] & 0xF) | ((q[1] & 0xF) << 4) | ((q[2] & 0xF) << 8) |
                                    ((q[3] & 0xF) << 12));
    *reinterpret_cast<uint16_t*>(packed + (size_t)r * (cols / 2) + c0 / 2) = two;
  }
  if (lane == 0) {
    scales[(size_t)r * sstride + gi] = sb;
    if (gi == ng - 1)
      for (int j = ng; j < sstride; ++j) scales[(size_t)r * sstride + j] = 0;
  }
}

// ------------------------------------------------------------------ re-layout
__device__ __forceinline__ long long map_row(long long r, int map, int param) {
  if (map == MAP_ROPE_PAIRS) {
    const long long head = r / param, i = r % param, half = param / 2;
    return head * param + (i < half ? 2 * i : 2 * (i - half) + 1);
  }
  if (map == MAP_INTERLEAVE) return 2 * r + param;
  return r;
}

__global__ void k_copy_rows16(uint8_t* dst, long long dst_stride, long long dst_row0,
                              const uint8_t* src, long long src_stride, long long row_bytes,
                              long long nrows, int map, int param) {
  const long long per_row = row_bytes / 16;
  const long long total = per_row * nrows;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const long long r = i / per_row, c = i % per_row;
    const long long dr = dst_row0 + map_row(r, map, param);
    *reinterpret_cast<uint4*>(dst + dr * dst_stride + c * 16) =
        *reinterpret_cast<const uint4*>(src + r * src_stride + c * 16);
  }
}

__global__ void k_copy_rows2(uint8_t* dst, long long dst_stride, long long dst_row0,
                             const uint8_t* src, long long src_stride, long long row_bytes,
                             long long nrows, int map, int param) {
  const long long per_row = row_bytes / 2;
  const long long total = per_row * nrows;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const long long r = i / per_row, c = i % per_row;
    const long long dr = dst_row0 + map_row(r, map, param);
    *reinterpret_cast<uint16_t*>(dst + dr * dst_stride + c * 2) =
        *reinterpret_cast<const uint16_t*>(src + r * src_stride + c * 2);
  }
}

__global__ void k_transpose(uint16_t* dst, const uint16_t* src, int n) {
  __shared__ uint16_t tile[32][33];
  const int bx = blockIdx.x * 32, by = blockIdx.y * 32;
  for (int j = threadIdx.y; j < 32; j += 8) {
    const int r = by + j, c = bx + threadIdx.x;
    if (r < n && c < n) tile[j][threadIdx.x] = src[(size_t)r * n + c];
  }
  __syncthreads();
  for (int j = threadIdx.y; j < 32; j += 8) {
    const int r = bx + j, c = by + threadIdx.x;
    if (r < n && c < n) dst[(size_t)r * n + c] = tile[threadIdx.x][j];
  }
}

__global__ void k_fill_u16(uint16_t* p, uint16_t v, long long n) {
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x)
    p[i] = v;
}

cudaLaunchConfig_t make_cfg(dim3 grid, dim3 block, cudaStream_t st, bool pdl, cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.stream = st;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cfg;
}

}  // namespace

cudaError_t launch_rmsnorm(const NormParams& p, int batch_slots, bool pdl, cudaStream_t st) {
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = make_cfg(dim3(batch_slots), dim3(256), st, pdl, attr);
  return cudaLaunchKernelEx(&cfg, k_rmsnorm, p);
}

cudaError_t launch_sts(const StsParams& p, int batch_slots, bool pdl, cudaStream_t st) {
  if (p.d % 4 || p.h_stride % 4) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(batch_slots < 1 ? 1 : batch_slots);
  cfg.blockDim = dim3(256);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, k_sts, p);
}

cudaError_t launch_step_begin(const BeginParams& p, int batch_slots, cudaStream_t st) {
  k_step_begin<<<batch_slots, 256, 0, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_quantize_int4(const uint16_t* w, int rows, int cols, uint8_t* packed,
                                 uint16_t* scales, int sstride, cudaStream_t st) {
  const long long warps = (long long)rows * ((cols + EE_QUANT_GROUP - 1) / EE_QUANT_GROUP);
  const long long blocks = (warps + 7) / 8;
  if (blocks <= 0) return cudaSuccess;
  k_quantize<<<(unsigned)blocks, 256, 0, st>>>(w, rows, cols, packed, scales, sstride);
  return cudaGetLastError();
}

cudaError_t launch_copy_rows(void* dst, int64_t dst_stride_bytes, int64_t dst_row0, const void* src,
                             int64_t src_stride_bytes, int64_t row_bytes, int64_t nrows, int map,
                             int param, cudaStream_t st) {
  if (nrows <= 0 || row_bytes <= 0) return cudaSuccess;
  const bool v16 = (row_bytes % 16 == 0) && (dst_stride_bytes % 16 == 0) &&
                   (src_stride_bytes % 16 == 0) && ((uintptr_t)dst % 16 == 0) &&
                   ((uintptr_t)src % 16 == 0);
  const long long units = v16 ? row_bytes / 16 * nrows : row_bytes / 2 * nrows;
  long long blocks = (units + 255) / 256;
  if (blocks > 65535) blocks = 65535;
  if (v16)
    k_copy_rows16<<<(unsigned)blocks, 256, 0, st>>>((uint8_t*)dst, dst_stride_bytes, dst_row0,
                                                    (const uint8_t*)src, src_stride_bytes, row_bytes,
                                                    nrows, map, param);
  else
    k_copy_rows2<<<(unsigned)blocks, 256, 0, st>>>((uint8_t*)dst, dst_stride_bytes, dst_row0,
                                                   (const uint8_t*)src, src_stride_bytes, row_bytes,
                                                   nrows, map, param);
  return cudaGetLastError();
}

cudaError_t launch_transpose_bf16(uint16_t* dst, const uint16_t* src, int n, cudaStream_t st) {
  dim3 grid((n + 31) / 32, (n + 31) / 32), block(32, 8);
  k_transpose<<<grid, block, 0, st>>>(dst, src, n);
  return cudaGetLastError();
}

cudaError_t launch_fill_u16(uint16_t* p, uint16_t v, int64_t n, cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  long long blocks = (n + 255) / 256;
  if (blocks > 65535) blocks = 65535;
  k_fill_u16<<<(unsigned)blocks, 256, 0, st>>>(p, v, n);
  return cudaGetLastError();
}

}  // namespace ee
