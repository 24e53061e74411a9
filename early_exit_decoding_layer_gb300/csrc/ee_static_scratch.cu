// Paged decode attention whose scratch lives in a fixed array compiled into
// the library, for callers that must not allocate device memory.
//
// Some callers cannot call cudaMalloc or hand the library a buffer of their
// own: a host whose caching allocator has already reserved the device's free
// memory (a cudaMalloc from outside it can then fail, and it may synchronise
// the device), or a host that forbids any allocation once it has started up.
// This entry point runs the same attention kernel as ee_op_attention, with its
// partial results and merge counters in g_attn_scratch below.
//
// The array is shared by every call in the process on a given device and keeps
// the previous call's contents; two calls that overlap in time on one device
// (different streams or host threads) race on it and give wrong results.
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/ee.h"

namespace {

static __device__ __align__(256) unsigned char g_attn_scratch[EE_ATTN_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_addr[kMaxDevices] = {};

// Address of g_attn_scratch on the current device, looked up once per device
// (the first call on each device does the lookup).
ee_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return EE_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return EE_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_attn_scratch) != cudaSuccess || !p) return EE_ERR_CUDA;
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return EE_OK;
}

}  // namespace

// The argument checks of ee_op_attention (ee_runtime.cu), run here before the
// array is touched so that a rejected call leaves the device alone.
ee_status ee_attention_args_check(int32_t B, int32_t n_heads, int32_t n_kv_heads, int32_t head_dim,
                                  int32_t max_ctx, const float* q, const uint16_t* kcache,
                                  const uint16_t* vcache, const int32_t* block_table, int32_t bt_stride,
                                  const int32_t* pos, const float* o);

extern "C" ee_status ee_op_attention_noalloc(int32_t B, int32_t n_heads, int32_t n_kv_heads,
                                             int32_t head_dim, int32_t max_ctx, const float* q,
                                             const uint16_t* kcache, const uint16_t* vcache,
                                             const int32_t* block_table, int32_t bt_stride,
                                             const int32_t* pos, float* o, int32_t* err_flag,
                                             void* stream) {
  const ee_status chk = ee_attention_args_check(B, n_heads, n_kv_heads, head_dim, max_ctx, q, kcache, vcache,
                                                block_table, bt_stride, pos, o);
  if (chk != EE_OK) return chk;
  const size_t need = ee_attention_scratch_bytes(B, n_heads, n_kv_heads, head_dim, max_ctx);
  if (need == 0) return EE_ERR_INVALID_ARG;
  if (need > EE_ATTN_STATIC_SCRATCH_BYTES) return EE_ERR_CAPACITY;
  void* scratch = nullptr;
  const ee_status st = scratch_address(&scratch);
  if (st != EE_OK) return st;
  // The merge counters sit at the end of the scratch layout, so their offset
  // moves with the shape: a previous call of another shape may have left
  // partial results there.  Zero them on the caller's stream before the launch.
  const size_t counter_bytes = (size_t)EE_MAX_BATCH * n_kv_heads * 4;
  if (cudaMemsetAsync(static_cast<unsigned char*>(scratch) + (need - counter_bytes), 0, counter_bytes,
                      (cudaStream_t)stream) != cudaSuccess)
    return EE_ERR_CUDA;
  return ee_op_attention(B, n_heads, n_kv_heads, head_dim, max_ctx, q, kcache, vcache, block_table,
                         bt_stride, pos, o, scratch, err_flag, stream);
}
