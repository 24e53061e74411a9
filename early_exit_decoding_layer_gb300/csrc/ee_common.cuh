// Device helpers shared by the kernels: inline PTX for mbarriers, bulk
// copies (global -> shared, completion counted on an mbarrier), programmatic
// dependent launch, L2 policies, and bounded waits that give up with an
// error code instead of spinning forever.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#define EE_DEV __device__ __forceinline__

namespace ee {

// Device error codes written to the context's error word.
enum : int32_t {
  DERR_NONE = 0,
  DERR_FULL_WAIT = 1,    // consumer gave up waiting for a stage to land
  DERR_EMPTY_WAIT = 2,   // producer gave up waiting for a stage to drain
  DERR_DRAIN_WAIT = 3,   // producer gave up draining its copies at exit
};

constexpr uint64_t kWaitTimeoutNs = 2000000000ull;  // 2 s

EE_DEV uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

EE_DEV uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

EE_DEV void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count));
}

EE_DEV void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }

EE_DEV void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

EE_DEV void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

EE_DEV bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for the phase with the given parity to complete.  Gives up after
// kWaitTimeoutNs, records `code` in *err (first writer wins) and returns false.
EE_DEV bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, int32_t* err, int32_t code) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 255u) == 0 && globaltimer() - t0 > kWaitTimeoutNs) {
      if (err) atomicCAS(err, 0, code);
      return false;
    }
  }
}

EE_DEV uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// Bulk copy of `bytes` (multiple of 16, both addresses 16-byte aligned) from
// global memory into this CTA's shared memory; completion is counted in
// bytes on `bar` (whose expected transaction count the caller has raised).
EE_DEV void bulk_g2s(void* dst_smem, const void* src_gmem, uint32_t bytes, uint64_t* bar,
                     uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], "
      "%2, [%3], %4;" ::"r"(smem_addr(dst_smem)),
      "l"(src_gmem), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

// Programmatic dependent launch.  Every kernel of a step follows one rule:
// it reads nothing a kernel before it wrote and writes nothing before
// grid_dep_wait(), except data that the kernel two launches back or earlier
// produced (see the step orchestrator), and it calls grid_dep_launch() only
// after grid_dep_wait().
EE_DEV void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
EE_DEV void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

EE_DEV int32_t ld_volatile_i32(const int32_t* p) {
  int32_t v;
  asm volatile("ld.volatile.global.s32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}

EE_DEV uint4 ldg_nc_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Streaming 16-byte load of data read once per launch (weights): not kept in
// L1, with a 256-byte L2 fetch granule.
EE_DEV uint4 ldg_stream_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

EE_DEV float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
EE_DEV float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
EE_DEV float bf16_bits_to_float(uint16_t b) { return __uint_as_float(uint32_t(b) << 16); }

EE_DEV uint16_t float_to_bf16_bits(float f) {
  __nv_bfloat16 b = __float2bfloat16_rn(f);
  return *reinterpret_cast<uint16_t*>(&b);
}
EE_DEV uint16_t float_to_half_bits(float f) {
  __half h = __float2half_rn(f);
  return *reinterpret_cast<uint16_t*>(&h);
}

EE_DEV float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
EE_DEV float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Position of element k inside the fp16 activation layout used by the int4
// kernels: within each run of 8 elements the order is 0,4,1,5,2,6,3,7, so
// that a 16-byte load yields the half2 pairs (x0,x4) (x1,x5) (x2,x6) (x3,x7)
// that match the nibble pairs one mask-and-or extracts from a packed word.
EE_DEV int xh_slot(int k) { return (k & ~7) | ((k & 3) << 1) | ((k >> 2) & 1); }

}  // namespace ee
