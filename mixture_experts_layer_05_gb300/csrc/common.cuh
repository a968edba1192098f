// Shared device helpers of the GB300 FusedMoE kernels: status word, bounded waits,
// bf16 packing, warp reductions. No routing or expert arithmetic lives here.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/gbmoe.h"

namespace gbmoe {

// A device-side wait gives up after this long (ns of %globaltimer); legitimate waits
// in these kernels last microseconds.
constexpr unsigned long long kWaitTimeoutNs = 1000000000ull;

// Programmatic dependent launch. A kernel launched with programmatic stream serialization
// (launch_kernel below, inside one forward) may start while the kernel before it in the
// stream is still running: pdl_wait() blocks until that kernel has completed and its
// writes are visible (a no-op for an ordinary launch), and pdl_trigger() lets the next
// kernel begin launching. Every kernel calls pdl_wait() before it reads anything an
// earlier kernel of the stream wrote, with one exception: the decode w2 GEMMs read the
// routing's expert blocks before they wait. That is safe because the GEMMs trigger their
// dependents only after their own wait, so a w2 GEMM starts only once everything before
// the w13 GEMM (the routing included) has finished; the small kernels trigger at entry.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void record_status(int* status, int code) {
  if (status) atomicCAS(status, 0, code);
}

__device__ __forceinline__ unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float2 unpack_bf16x2(uint32_t u) {
  __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162*>(&u);
  return __bfloat1622float2(v);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

}  // namespace gbmoe
