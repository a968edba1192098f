// moe_align_block_size_no_workspace: the expert align of moe_align_block_size for
// callers that cannot allocate device memory.
//
// Some callers cannot hand this library a workspace: plugins and extensions hosted by
// a framework that owns and pre-plans every device allocation (an inference server
// with a fixed memory pool, a runtime that forbids its extensions from calling
// cudaMalloc) have no buffer to give and may not create one. For them this entry
// point keeps its scratch (the per-chunk expert counts and offsets of the align) in a
// file-scope device array of fixed size instead of a caller workspace, and calls no
// allocating routine of any kind.
//
// Limits and sharing:
//  - the array holds kNoWorkspaceScratchBytes (1 MiB) on every GPU that loads the
//    library, until the process exits;
//  - a request whose scratch, 2 * ceil(T*top_k / 2048) * num_experts * 4 bytes, is larger
//    is rejected with GBMOE_ERR_WORKSPACE (for example E = 256 allows up to 1,048,576
//    flat indices T*top_k: 512 chunks of 2048);
//  - every call on a device shares the one array, and the array keeps the last call's
//    contents. Each call overwrites every byte it reads before reading it (counts, then
//    offsets), so nothing has to start at zero; calls whose kernels overlap on the GPU
//    (different streams without ordering) race on the array and must not be issued;
//  - the first call on a device looks up the array's device address
//    (cudaGetSymbolAddress) with that device current; make that first call before any
//    stream capture;
//  - this variant has no status word: a topk_id outside [0, E) is counted as expert 0
//    but not reported.
#include <mutex>

#include "common.cuh"
#include "kernels.h"

#define GBMOE_API extern "C" __attribute__((visibility("default")))

namespace gbmoe {
namespace {

constexpr size_t kNoWorkspaceScratchBytes = (size_t)1 << 20;

static __device__ __align__(256) unsigned char g_align_scratch[kNoWorkspaceScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_ptr[kMaxDevices] = {nullptr};
std::mutex g_scratch_mutex;

// Device address of g_align_scratch on the current device (set up once per device).
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_align_scratch);
    if (e != cudaSuccess || p == nullptr) return e != cudaSuccess ? e : cudaErrorInvalidSymbol;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace gbmoe

using namespace gbmoe;

GBMOE_API gbmoe_status_t moe_align_block_size_no_workspace(
    const int32_t* topk_ids, int32_t num_tokens, int32_t top_k, int32_t num_experts,
    int32_t block_size, int32_t* sorted_token_ids, int32_t* expert_ids,
    int32_t* num_tokens_post_padded, gbmoe_stream_t stream) {
  if (num_tokens < 0 || num_tokens > (1 << 22) || top_k < 1 || top_k > 32 || num_experts < 1 ||
      num_experts > 1024 || top_k > num_experts || block_size < 1 || block_size > 1024)
    return GBMOE_ERR_INVALID_ARG;
  if (num_tokens == 0) return GBMOE_OK;
  if (!topk_ids || !sorted_token_ids || !expert_ids || !num_tokens_post_padded)
    return GBMOE_ERR_INVALID_ARG;
  const int n = num_tokens * top_k;
  if (align_scratch_bytes(n, num_experts) > kNoWorkspaceScratchBytes) return GBMOE_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return GBMOE_ERR_CUDA;
  const int max_sorted = n + num_experts * (block_size - 1);
  const int max_blocks = max_sorted / block_size + 1;
  PdlChain chain;
  return launch_align(topk_ids, n, num_experts, block_size, sorted_token_ids, expert_ids,
                      max_blocks, num_tokens_post_padded, scratch, nullptr,
                      (cudaStream_t)stream) == cudaSuccess
             ? GBMOE_OK
             : GBMOE_ERR_CUDA;
}
