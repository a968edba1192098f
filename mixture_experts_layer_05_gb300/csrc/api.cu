// C ABI of the FusedMoE forward: host-side validation, workspace layout and the
// launch sequence. Argument checks mirror the raises and asserts of the FusedMoE
// constructor (vLLM `fused_moe/layer` page: grouped routing needs both group
// arguments, non-softmax scoring needs grouped routing) and of `DeepseekV2MLP` /
// `DeepseekV2MoE` (sglang `models/deepseek_v2.py` page: only silu is supported).
#include <climits>
#include <cmath>
#include <cstring>

#include "common.cuh"
#include "kernels.h"

#define GBMOE_API extern "C" __attribute__((visibility("default")))

namespace gbmoe {

int num_sms() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (!cached[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
    cached[dev] = n;
  }
  return cached[dev];
}

namespace {

constexpr int kMaxTokens = 1 << 22;
constexpr size_t kAlign = 256;

size_t up(size_t v, size_t a = kAlign) { return (v + a - 1) / a * a; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

gbmoe_status_t check_routing(const gbmoe_config_t* c) {
  if (!c) return GBMOE_ERR_INVALID_ARG;
  if (c->num_experts < 1 || c->num_experts > 1024) return GBMOE_ERR_INVALID_ARG;
  if (c->top_k < 1 || c->top_k > c->num_experts || c->top_k > 32) return GBMOE_ERR_INVALID_ARG;
  if (c->scoring_func != GBMOE_SCORE_SOFTMAX && c->scoring_func != GBMOE_SCORE_SIGMOID)
    return GBMOE_ERR_INVALID_ARG;
  if (!std::isfinite(c->routed_scaling_factor)) return GBMOE_ERR_INVALID_ARG;
  if (c->use_grouped_topk) {
    const int G = c->num_expert_group, g = c->topk_group;
    if (G < 1 || g < 1) return GBMOE_ERR_INVALID_ARG;
    if (c->num_experts % G != 0 || G > 32 || g > G) return GBMOE_ERR_INVALID_ARG;
    if (c->top_k > g * (c->num_experts / G)) return GBMOE_ERR_INVALID_ARG;
  } else if (c->scoring_func != GBMOE_SCORE_SOFTMAX) {
    return GBMOE_ERR_UNSUPPORTED;
  }
  return GBMOE_OK;
}

gbmoe_status_t check_layer(const gbmoe_config_t* c) {
  gbmoe_status_t s = check_routing(c);
  if (s != GBMOE_OK) return s;
  if (c->hidden_size <= 0 || c->intermediate_size <= 0 || c->shared_intermediate_size < 0)
    return GBMOE_ERR_INVALID_ARG;
  if (c->activation != GBMOE_ACT_SILU || c->is_act_and_mul != 1) return GBMOE_ERR_UNSUPPORTED;
  if (c->hidden_size % 128 || c->intermediate_size % 128 || c->shared_intermediate_size % 128)
    return GBMOE_ERR_UNSUPPORTED;
  if ((long long)c->num_experts * 2 * c->intermediate_size > INT_MAX / 2 ||
      (long long)c->num_experts * c->hidden_size > INT_MAX / 2)
    return GBMOE_ERR_UNSUPPORTED;
  return GBMOE_OK;
}

struct Layout {
  int bs, n, max_sorted, max_blocks, slots;
  size_t status, topk_weights, topk_ids, sorted, expert_ids, npp, scratch, x_perm, act, ytok,
      act_s, total;
};

Layout layout_for(const gbmoe_config_t& c, int T) {
  Layout L;
  const int E = c.num_experts, k = c.top_k, H = c.hidden_size, I = c.intermediate_size;
  const int Is = c.shared_intermediate_size;
  L.bs = kGemmBM;
  L.n = T * k;
  L.max_sorted = L.n + E * (L.bs - 1);
  L.max_blocks = L.max_sorted / L.bs + 1;
  L.slots = k + (Is ? 1 : 0);
  size_t o = 0;
  L.status = o;
  o += kAlign;
  L.topk_weights = o;
  o = up(o + (size_t)L.n * 4);
  L.topk_ids = o;
  o = up(o + (size_t)L.n * 4);
  L.sorted = o;
  o = up(o + (size_t)L.max_sorted * 4);
  L.expert_ids = o;
  o = up(o + (size_t)L.max_blocks * 4);
  L.npp = o;
  o = up(o + 4);
  L.scratch = o;
  o = up(o + align_scratch_bytes(L.n, E));
  L.x_perm = o;
  o = up(o + (size_t)L.max_sorted * H * 2);
  L.act = o;
  o = up(o + (size_t)L.max_sorted * I * 2);
  L.ytok = o;
  o = up(o + (size_t)T * L.slots * H * 4);
  L.act_s = o;
  o = up(o + (size_t)T * Is * 2);
  L.total = o;
  return L;
}

template <typename T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<char*>(ws) + off);
}

gbmoe_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? GBMOE_OK : GBMOE_ERR_CUDA; }

}  // namespace
}  // namespace gbmoe

using namespace gbmoe;

GBMOE_API int32_t gbmoe_version(void) { return (0 << 16) | 1; }

GBMOE_API gbmoe_status_t moe_topk(const gbmoe_config_t* cfg, int32_t num_tokens,
                                  const float* router_logits,
                                  const float* e_score_correction_bias, float* topk_weights,
                                  int32_t* topk_ids, gbmoe_stream_t stream) {
  gbmoe_status_t s = check_routing(cfg);
  if (s != GBMOE_OK) return s;
  if (num_tokens < 0 || num_tokens > kMaxTokens) return GBMOE_ERR_INVALID_ARG;
  if (num_tokens == 0) return GBMOE_OK;
  if (!router_logits || !topk_weights || !topk_ids) return GBMOE_ERR_INVALID_ARG;
  return cuda_status(launch_topk(*cfg, num_tokens, router_logits, e_score_correction_bias,
                                 topk_weights, topk_ids, nullptr, (cudaStream_t)stream));
}

GBMOE_API size_t moe_align_block_size_workspace_size(int32_t num_tokens, int32_t top_k,
                                                     int32_t num_experts) {
  if (num_tokens < 0 || top_k < 1 || num_experts < 1 || num_tokens > kMaxTokens) return 0;
  return kAlign + up(align_scratch_bytes(num_tokens * top_k, num_experts));
}

GBMOE_API gbmoe_status_t moe_align_block_size(const int32_t* topk_ids, int32_t num_tokens,
                                              int32_t top_k, int32_t num_experts,
                                              int32_t block_size, int32_t* sorted_token_ids,
                                              int32_t* expert_ids,
                                              int32_t* num_tokens_post_padded, void* workspace,
                                              size_t workspace_bytes, gbmoe_stream_t stream) {
  if (num_tokens < 0 || num_tokens > kMaxTokens || top_k < 1 || top_k > 32 || num_experts < 1 ||
      num_experts > 1024 || top_k > num_experts || block_size < 1 || block_size > 1024)
    return GBMOE_ERR_INVALID_ARG;
  if (num_tokens == 0) return GBMOE_OK;
  if (!topk_ids || !sorted_token_ids || !expert_ids || !num_tokens_post_padded)
    return GBMOE_ERR_INVALID_ARG;
  const size_t need = moe_align_block_size_workspace_size(num_tokens, top_k, num_experts);
  if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) % kAlign))
    return GBMOE_ERR_WORKSPACE;
  const int n = num_tokens * top_k;
  const int max_sorted = n + num_experts * (block_size - 1);
  const int max_blocks = max_sorted / block_size + 1;
  return cuda_status(launch_align(topk_ids, n, num_experts, block_size, sorted_token_ids,
                                  expert_ids, max_blocks, num_tokens_post_padded,
                                  at<char>(workspace, kAlign), at<int>(workspace, 0),
                                  (cudaStream_t)stream));
}

GBMOE_API size_t moe_forward_workspace_size(const gbmoe_config_t* cfg, int32_t max_num_tokens) {
  if (check_layer(cfg) != GBMOE_OK || max_num_tokens < 0 || max_num_tokens > kMaxTokens) return 0;
  return layout_for(*cfg, max_num_tokens).total;
}

GBMOE_API int32_t moe_forward_block_size(const gbmoe_config_t* cfg, int32_t num_tokens) {
  (void)cfg;
  (void)num_tokens;
  return kGemmBM;
}

GBMOE_API gbmoe_status_t moe_forward_workspace_layout(const gbmoe_config_t* cfg,
                                                      int32_t max_num_tokens,
                                                      gbmoe_workspace_layout_t* out) {
  gbmoe_status_t s = check_layer(cfg);
  if (s != GBMOE_OK) return s;
  if (!out || max_num_tokens < 0 || max_num_tokens > kMaxTokens) return GBMOE_ERR_INVALID_ARG;
  const Layout L = layout_for(*cfg, max_num_tokens);
  out->status = L.status;
  out->topk_weights = L.topk_weights;
  out->topk_ids = L.topk_ids;
  out->sorted_token_ids = L.sorted;
  out->expert_ids = L.expert_ids;
  out->num_tokens_post_padded = L.npp;
  out->act = L.act;
  out->total = L.total;
  return GBMOE_OK;
}

GBMOE_API gbmoe_status_t moe_forward_events(
    const gbmoe_config_t* cfg, int32_t num_tokens, const void* hidden_states,
    const float* router_logits, const float* e_score_correction_bias, const void* w13_weight,
    const void* w2_weight, const void* shared_w13, const void* shared_w2, void* output,
    void* workspace, size_t workspace_bytes, void* const* events, int32_t num_events,
    gbmoe_stream_t stream_) {
  gbmoe_status_t s = check_layer(cfg);
  if (s != GBMOE_OK) return s;
  if (num_tokens < 0 || num_tokens > kMaxTokens) return GBMOE_ERR_INVALID_ARG;
  if (events ? num_events != GBMOE_NUM_STAGE_EVENTS : num_events != 0)
    return GBMOE_ERR_INVALID_ARG;
  const gbmoe_config_t& c = *cfg;
  const int Is = c.shared_intermediate_size;
  if ((shared_w13 != nullptr) != (Is > 0) || (shared_w2 != nullptr) != (Is > 0))
    return GBMOE_ERR_INVALID_ARG;
  if (num_tokens == 0) return GBMOE_OK;
  if (!hidden_states || !router_logits || !w13_weight || !w2_weight || !output)
    return GBMOE_ERR_INVALID_ARG;
  if (!aligned16(hidden_states) || !aligned16(w13_weight) || !aligned16(w2_weight) ||
      !aligned16(output) || (Is && (!aligned16(shared_w13) || !aligned16(shared_w2))))
    return GBMOE_ERR_INVALID_ARG;
  const Layout L = layout_for(c, num_tokens);
  if (!workspace || workspace_bytes < L.total || (reinterpret_cast<uintptr_t>(workspace) % kAlign))
    return GBMOE_ERR_WORKSPACE;

  cudaStream_t stream = (cudaStream_t)stream_;
  const int T = num_tokens, E = c.num_experts, k = c.top_k, H = c.hidden_size,
            I = c.intermediate_size;
  int* status = at<int>(workspace, L.status);
  float* tw = at<float>(workspace, L.topk_weights);
  int* tids = at<int>(workspace, L.topk_ids);
  int* sorted = at<int>(workspace, L.sorted);
  int* eids = at<int>(workspace, L.expert_ids);
  int* npp = at<int>(workspace, L.npp);
  void* x_perm = at<char>(workspace, L.x_perm);
  void* act = at<char>(workspace, L.act);
  void* ytok = at<char>(workspace, L.ytok);
  void* act_s = at<char>(workspace, L.act_s);
  auto rec = [&](int i) -> cudaError_t {
    return events ? cudaEventRecord((cudaEvent_t)events[i], stream) : cudaSuccess;
  };
  const int w2_bn = (H % 256 == 0) ? 256 : 128;
  const int t_pad = (T + kGemmBM - 1) / kGemmBM * kGemmBM;
  cudaError_t e;

#define GBMOE_TRY(x)                   \
  do {                                 \
    e = (x);                           \
    if (e != cudaSuccess) return GBMOE_ERR_CUDA; \
  } while (0)

  GBMOE_TRY(rec(0));
  GBMOE_TRY(launch_topk(c, T, router_logits, e_score_correction_bias, tw, tids, status, stream));
  GBMOE_TRY(launch_align(tids, L.n, E, L.bs, sorted, eids, L.max_blocks, npp,
                         at<char>(workspace, L.scratch), status, stream));
  GBMOE_TRY(launch_gather(hidden_states, H, sorted, npp, L.n, k, L.max_sorted, x_perm, stream));
  GBMOE_TRY(rec(1));

  GemmArgs a;
  std::memset(&a, 0, sizeof(a));
  a.status = status;
  // routed w13 + SiLU*mul
  a.n_tiles = I / kGemmBM;
  a.k_blocks = H / kGemmBK;
  a.m_rows_dev = npp;
  a.max_m_blocks = L.max_sorted / kGemmBM;
  a.expert_ids = eids;
  a.num_experts = E;
  a.b_rows_per_expert = 2 * I;
  a.up_offset = I;
  a.out = act;
  a.ldo = I;
  a.store_rows = L.max_sorted;
  GBMOE_TRY(launch_gemm(kGemmW13, kGemmBM, x_perm, L.max_sorted, H, w13_weight, E * 2 * I, a,
                        stream));
  if (Is) {
    GemmArgs b = a;
    b.n_tiles = Is / kGemmBM;
    b.m_rows_dev = nullptr;
    b.m_rows_host = t_pad;
    b.max_m_blocks = t_pad / kGemmBM;
    b.expert_ids = nullptr;
    b.num_experts = 1;
    b.b_rows_per_expert = 2 * Is;
    b.up_offset = Is;
    b.out = act_s;
    b.ldo = Is;
    b.store_rows = T;
    GBMOE_TRY(launch_gemm(kGemmW13, kGemmBM, hidden_states, T, H, shared_w13, 2 * Is, b, stream));
  }
  GBMOE_TRY(rec(2));

  // routed w2, weighted, scattered to the token's slot
  GemmArgs d;
  std::memset(&d, 0, sizeof(d));
  d.status = status;
  d.n_tiles = H / w2_bn;
  d.k_blocks = I / kGemmBK;
  d.m_rows_dev = npp;
  d.max_m_blocks = L.max_sorted / kGemmBM;
  d.expert_ids = eids;
  d.num_experts = E;
  d.b_rows_per_expert = H;
  d.out = ytok;
  d.ldo = H;
  d.sorted_ids = sorted;
  d.row_weight = tw;
  d.num_flat = L.n;
  d.top_k = k;
  d.slots = L.slots;
  GBMOE_TRY(launch_gemm(kGemmW2, w2_bn, act, L.max_sorted, I, w2_weight, E * H, d, stream));
  if (Is) {
    GemmArgs f = d;
    f.k_blocks = Is / kGemmBK;
    f.m_rows_dev = nullptr;
    f.m_rows_host = t_pad;
    f.max_m_blocks = t_pad / kGemmBM;
    f.expert_ids = nullptr;
    f.num_experts = 1;
    f.sorted_ids = nullptr;
    f.row_weight = nullptr;
    f.store_rows = T;
    f.slot_offset = k;
    GBMOE_TRY(launch_gemm(kGemmW2, w2_bn, act_s, T, Is, shared_w2, H, f, stream));
  }
  GBMOE_TRY(rec(3));
  GBMOE_TRY(launch_combine(ytok, L.slots, H, T, output, stream));
  GBMOE_TRY(rec(4));
#undef GBMOE_TRY
  return GBMOE_OK;
}

GBMOE_API gbmoe_status_t moe_forward(const gbmoe_config_t* cfg, int32_t num_tokens,
                                     const void* hidden_states, const float* router_logits,
                                     const float* e_score_correction_bias, const void* w13_weight,
                                     const void* w2_weight, const void* shared_w13,
                                     const void* shared_w2, void* output, void* workspace,
                                     size_t workspace_bytes, gbmoe_stream_t stream) {
  return moe_forward_events(cfg, num_tokens, hidden_states, router_logits,
                            e_score_correction_bias, w13_weight, w2_weight, shared_w13, shared_w2,
                            output, workspace, workspace_bytes, nullptr, 0, stream);
}

GBMOE_API gbmoe_status_t moe_get_device_status(void* workspace, int32_t* status,
                                               gbmoe_stream_t stream) {
  if (!workspace || !status) return GBMOE_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  int32_t v = 0;
  if (cudaMemcpyAsync(&v, workspace, sizeof(v), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaMemsetAsync(workspace, 0, sizeof(v), s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return GBMOE_ERR_CUDA;
  *status = v;
  return GBMOE_OK;
}
