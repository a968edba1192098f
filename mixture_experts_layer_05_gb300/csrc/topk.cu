// Stand-alone router top-k: one warp per token (route.cuh), grid-stride over tokens.
#include "kernels.h"
#include "route.cuh"

namespace gbmoe {

template <int EPT>
__global__ void __launch_bounds__(256) topk_kernel(TopkArgs a) {
  pdl_trigger();  // the next kernel may start its launch now
  pdl_wait();     // inputs written by the previous kernel are visible
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < a.zero_count; i += gridDim.x * blockDim.x)
    a.zero[i] = 0;
  const int lane = threadIdx.x & 31;
  const int warps_total = gridDim.x * (blockDim.x >> 5);
  for (int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); t < a.T; t += warps_total)
    route_token_warp<EPT>(a, t, lane);
}

struct TopkLaunch {
  TopkArgs a;
  int blocks;
  cudaStream_t stream;
  template <int EPT>
  void operator()() {
    launch_kernel(topk_kernel<EPT>, dim3(blocks), dim3(256), 0, stream, a);
  }
};

cudaError_t launch_topk(const gbmoe_config_t& c, int T, const float* logits, const float* bias,
                        float* weights, int* ids, int* status, cudaStream_t stream,
                        int logit_splits, long long logit_split_stride, int* zero,
                        int zero_count) {
  const int warps = 256 / 32;
  int blocks = (T + warps - 1) / warps;
  const int cap = num_sms() * 8;
  if (blocks > cap) blocks = cap;
  TopkLaunch L{make_topk_args(c, T, logits, bias, weights, ids, status), blocks, stream};
  L.a.logit_splits = logit_splits;
  L.a.logit_split_stride = logit_split_stride;
  L.a.zero = zero;
  L.a.zero_count = zero_count;
  dispatch_ept(c.num_experts, L);
  return cudaGetLastError();
}

}  // namespace gbmoe
