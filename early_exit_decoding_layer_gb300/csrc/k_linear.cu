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
// int4 dequantisation: a packed word holds columns c..c+7 in nibbles 0..7
// (two's complement).  One LOP3 per pair of nibbles (j, j+4) masks them under
// the fp16 exponent of 1024 and flips their sign bits: with mask 0x000F000F
// the half2 is (1024 + q_j + 8, 1024 + q_{j+4} + 8), minus 1032 gives
// (q_j, q_{j+4}); with mask 0x00F000F0 (nibbles 1 and 5, or 3 and 7 after a
// shift by 8) it is 1024 + 16 (q + 8), times 1/16 minus 72.  All exact; 13
// instructions per 8 weights including the 4 HFMA2 of the dot product.
// Products accumulate in fp16 over 32 columns, then in fp32 with the scale.
#include <math.h>

#include "ee_common.cuh"
#include "ee_gemv.cuh"
#include "ee_kernels.cuh"

namespace ee {

namespace {

template <bool XS, int MMAX>
__global__ void __launch_bounds__(kThreads, kCtasPerSm) k_linear(const LinearParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ int s_last;
  // Lists written at least two launches back (see grid_dep_wait) may be read
  // before this grid's dependency wait; otherwise wait first.
  if (p.stamp_start && threadIdx.x == 0) atomicMin(p.stamp_start, (unsigned long long)globaltimer());
  if (p.lists_after_wait) grid_dep_wait();
  LinState s;
  linear_prologue<XS, MMAX>(p, blockIdx.x, gridDim.x, smem, s);
  linear_body<XS, MMAX>(p, gridDim.x, smem, s, &s_last);
  // thread 0 passes every barrier of the CTA, so its end is the CTA's end
  if (p.stamp_end && threadIdx.x == 0) atomicMax(p.stamp_end, (unsigned long long)globaltimer());
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
