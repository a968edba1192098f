// Combine: y[t] = sum over the split-K partial copies and, inside each, over the
// token's slots (routed j ascending, then the shared expert) of the already-weighted
// fp32 expert outputs, accumulated in fp32 in that fixed order and rounded once to
// bf16. The routed outputs arrive weighted by topk_weights (scaled by
// routed_scaling_factor) from the w2 epilogue; the shared-expert slot is unscaled,
// as `DeepseekV2MoE.forward_normal` adds it (sglang `models/deepseek_v2.py` page).
// HBM-bound: 16-byte vector loads and stores, grid-stride over (token, 8 columns).
#include "common.cuh"
#include "kernels.h"

namespace gbmoe {

__global__ void __launch_bounds__(256) combine_kernel(const float4* __restrict__ ytok, int slots,
                                                      int routed_slots, int H8, int T, int splits,
                                                      int splits_last,
                                                      long long split_stride4,
                                                      uint4* __restrict__ y) {
  pdl_trigger();  // the next kernel may start its launch now
  pdl_wait();     // inputs written by the previous kernel are visible
  const size_t total = (size_t)T * H8;
  const int copies = splits > splits_last ? splits : splits_last;
  const int terms = copies * slots;
  for (size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (size_t)gridDim.x * blockDim.x) {
    const size_t t = idx / H8, h = idx % H8;
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
    const float4* row = ytok + (t * slots * H8 + h) * 2;
    // term i = (copy i / slots, slot i % slots), summed in that order; a slot only has the
    // copies of its own problem. Loads of four terms are issued before their adds.
    for (int i = 0; i < terms; i += 4) {
      float4 u[4], v[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int c = (i + j) / slots, sl = (i + j) % slots;
        const bool live = i + j < terms && c < (sl < routed_slots ? splits : splits_last);
        u[j] = v[j] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (live) {
          const float4* src = row + (size_t)c * split_stride4 + (size_t)sl * H8 * 2;
          u[j] = __ldg(src);
          v[j] = __ldg(src + 1);
        }
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        a.x += u[j].x; a.y += u[j].y; a.z += u[j].z; a.w += u[j].w;
        b.x += v[j].x; b.y += v[j].y; b.z += v[j].z; b.w += v[j].w;
      }
    }
    uint4 o;
    o.x = pack_bf16x2(a.x, a.y);
    o.y = pack_bf16x2(a.z, a.w);
    o.z = pack_bf16x2(b.x, b.y);
    o.w = pack_bf16x2(b.z, b.w);
    y[idx] = o;
  }
}

// Small batches: the terms of each (token, 8 columns) are spread over 8 lanes (lane l takes
// terms l, l+8, ...), and the 8 partial sums are added by a fixed xor-butterfly, so the
// result is the same on every run; many more loads are in flight than with one thread.
constexpr int kTermLanes = 8;

__global__ void __launch_bounds__(256) combine_small_kernel(const float4* __restrict__ ytok,
                                                            int slots, int routed_slots, int H8,
                                                            int T, int splits, int splits_last,
                                                            long long split_stride4,
                                                            uint4* __restrict__ y) {
  pdl_trigger();  // the next kernel may start its launch now
  pdl_wait();     // inputs written by the previous kernel are visible
  const size_t groups = (size_t)T * H8;
  const int lane8 = threadIdx.x & (kTermLanes - 1);
  const int copies = splits > splits_last ? splits : splits_last;
  const int terms = copies * slots;
  // The loop runs over each warp's first group, so every lane of a warp takes the same number
  // of trips and reaches the shuffles; lanes past the last group add zeros and store nothing.
  const size_t warp_first = ((size_t)blockIdx.x * blockDim.x + (threadIdx.x & ~31u)) / kTermLanes;
  const size_t stride = (size_t)gridDim.x * blockDim.x / kTermLanes;
  for (size_t g0 = warp_first; g0 < groups; g0 += stride) {
    const size_t g = g0 + (threadIdx.x & 31) / kTermLanes;
    const bool valid = g < groups;
    const size_t t = g / H8, h = g % H8;
    const float4* row = ytok + (t * slots * H8 + h) * 2;
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
    // this lane's terms in increasing order, four loads issued before their adds
    for (int i0 = lane8; valid && i0 < terms; i0 += 4 * kTermLanes) {
      float4 u[4], v[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int i = i0 + q * kTermLanes;
        const int c = i / slots, sl = i % slots;
        u[q] = v[q] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (i < terms && c < (sl < routed_slots ? splits : splits_last)) {
          const float4* src = row + (size_t)c * split_stride4 + (size_t)sl * H8 * 2;
          u[q] = __ldg(src);
          v[q] = __ldg(src + 1);
        }
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        a.x += u[q].x; a.y += u[q].y; a.z += u[q].z; a.w += u[q].w;
        b.x += v[q].x; b.y += v[q].y; b.z += v[q].z; b.w += v[q].w;
      }
    }
#pragma unroll
    for (int o = 1; o < kTermLanes; o <<= 1) {
      a.x += __shfl_xor_sync(0xffffffffu, a.x, o);
      a.y += __shfl_xor_sync(0xffffffffu, a.y, o);
      a.z += __shfl_xor_sync(0xffffffffu, a.z, o);
      a.w += __shfl_xor_sync(0xffffffffu, a.w, o);
      b.x += __shfl_xor_sync(0xffffffffu, b.x, o);
      b.y += __shfl_xor_sync(0xffffffffu, b.y, o);
      b.z += __shfl_xor_sync(0xffffffffu, b.z, o);
      b.w += __shfl_xor_sync(0xffffffffu, b.w, o);
    }
    if (valid && lane8 == 0) {
      uint4 o;
      o.x = pack_bf16x2(a.x, a.y);
      o.y = pack_bf16x2(a.z, a.w);
      o.z = pack_bf16x2(b.x, b.y);
      o.w = pack_bf16x2(b.z, b.w);
      y[g] = o;
    }
  }
}

cudaError_t launch_combine(const void* ytok, int slots, int routed_slots, int H, int T,
                           int splits, int splits_last, long long split_stride, void* y,
                           cudaStream_t stream) {
  const size_t total = (size_t)T * (H / 8);
  if (total * kTermLanes <= (size_t)num_sms() * 1024) {
    const size_t threads_needed = total * kTermLanes;
    size_t blocks = (threads_needed + 255) / 256;
    if (blocks < 1) blocks = 1;
    launch_kernel(combine_small_kernel, dim3((unsigned)blocks), dim3(256), 0, stream,
                  static_cast<const float4*>(ytok), slots, routed_slots, H / 8, T, splits,
                  splits_last, split_stride / 4, static_cast<uint4*>(y));
    return cudaGetLastError();
  }
  const int threads = total < (size_t)num_sms() * 256 ? 64 : 256;  // spread small T over SMs
  size_t blocks = (total + threads - 1) / threads;
  const size_t cap = (size_t)num_sms() * (2048 / threads);
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  launch_kernel(combine_kernel, dim3((unsigned)blocks), dim3(threads), 0, stream,
                static_cast<const float4*>(ytok), slots, routed_slots, H / 8, T, splits,
                splits_last, split_stride / 4, static_cast<uint4*>(y));
  return cudaGetLastError();
}

}  // namespace gbmoe
