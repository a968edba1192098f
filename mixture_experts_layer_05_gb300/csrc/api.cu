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

bool& pdl_next() {
  static thread_local bool next = false;
  return next;
}

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
constexpr int kSplitMaxTokens = 64;  // split-K only at decode-sized batches
#ifndef GBMOE_TN_MIN_TOKENS
#define GBMOE_TN_MIN_TOKENS 65
#endif
// bf16 prefill batches of at least this many tokens may run the token-N GEMMs
constexpr int kTnMinTokens = GBMOE_TN_MIN_TOKENS;
#ifndef GBMOE_TN_MIN_ROWS
#define GBMOE_TN_MIN_ROWS 128
#endif
// ... when their experts average at least this many routed rows
constexpr int kTnMinRowsPerExpert = GBMOE_TN_MIN_ROWS;
#ifndef GBMOE_MAX_SPLITS
#define GBMOE_MAX_SPLITS 8
#endif
constexpr size_t kMaxSplits = GBMOE_MAX_SPLITS;  // largest split-K factor
#ifndef GBMOE_UNIT_COST_KB
#define GBMOE_UNIT_COST_KB 4
#endif
// Fixed cost of one unit of a persistent GEMM round (pipeline fill, accumulator hand-off and
// epilogue), in K blocks of streaming. Measured (graph replay): 4 takes DeepSeek-V2 T = 1
// from 95.6 to 93.1 us and T = 16 from 592 to 561 us, and the fp8 DeepSeek-V3 T = 1 from
// 105.5 to 100.7 us; 2 and 8 were no better.
constexpr double kUnitCostKb = GBMOE_UNIT_COST_KB;
constexpr size_t kAlign = 256;
// byte offset, inside the status region, of the fused router's arrival counter
constexpr size_t kGateCounterOffset = 4;
#ifndef GBMOE_GATE_FUSED
#define GBMOE_GATE_FUSED 1
#endif
// small batches given the gate weight compute their router logits inside the routing launch
// (0: with the tensor-core router GEMM first, as larger batches)
constexpr bool kGateFused = GBMOE_GATE_FUSED != 0;

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
  if (c->activation != GBMOE_ACT_SILU) return GBMOE_ERR_UNSUPPORTED;
  if (c->is_act_and_mul != 0 && c->is_act_and_mul != 1) return GBMOE_ERR_INVALID_ARG;
  if (!std::isfinite(c->swiglu_limit) || c->swiglu_limit < 0.f ||
      !std::isfinite(c->gemm1_alpha) || c->gemm1_alpha < 0.f)
    return GBMOE_ERR_INVALID_ARG;
  if (!c->is_act_and_mul &&
      (c->swiglu_limit > 0.f || (c->gemm1_alpha != 0.f && c->gemm1_alpha != 1.f) ||
       c->shared_intermediate_size > 0))
    return GBMOE_ERR_UNSUPPORTED;                  // clamp / alpha / shared need the gated form
  if (c->hidden_size % 128 || c->intermediate_size % 128 || c->shared_intermediate_size % 128)
    return GBMOE_ERR_UNSUPPORTED;
  if (c->weight_quant != GBMOE_QUANT_NONE && c->weight_quant != GBMOE_QUANT_FP8_BLOCK128 &&
      c->weight_quant != GBMOE_QUANT_NVFP4)
    return GBMOE_ERR_INVALID_ARG;
  if (c->weight_quant != GBMOE_QUANT_NONE &&
      (!c->is_act_and_mul || c->swiglu_limit > 0.f ||
       (c->gemm1_alpha != 0.f && c->gemm1_alpha != 1.f) || c->apply_router_weight_on_input ||
       (c->weight_quant == GBMOE_QUANT_FP8_BLOCK128 && c->hidden_size % 256)))
    return GBMOE_ERR_UNSUPPORTED;                  // the quantized layers are the plain gated one
  if ((long long)c->num_experts * 2 * c->intermediate_size > INT_MAX / 2 ||
      (long long)c->num_experts * c->hidden_size > INT_MAX / 2)
    return GBMOE_ERR_UNSUPPORTED;
  return GBMOE_OK;
}

bool use_tn(const gbmoe_config_t& c, int T);

// bf16 prefill whose experts average at least kTnMinRowsPerExpert rows runs the token-N
// GEMMs on CTA pairs: row blocks of 256 rows whose MMA width follows each block's real
// rows, so the padding of the align costs no tensor time. Measured against the tokens-on-M
// GEMMs (graph replay, same box): DeepSeek-V2 T = 4096 (154 rows per expert) 2.13 -> 1.89
// ms, DeepSeek-V3 T = 8192 (256) 6.82 -> 6.66, Mixtral T = 4096 (1024) 2.19 -> 2.12, the
// Zipf-skewed T = 16384 (512) 12.4 -> 11.9; with fewer rows per expert the pair streams
// each weight tile with less in flight per SM and loses (DeepSeek-V3 T = 2048, 64 rows:
// 3.28 -> 3.43).
bool use_tn(const gbmoe_config_t& c, int T) {
  return c.weight_quant == GBMOE_QUANT_NONE && T > kSplitMaxTokens && T >= kTnMinTokens &&
         (long)T * c.top_k >= (long)kTnMinRowsPerExpert * c.num_experts &&
         !route_align_small_ok(T, c.top_k, c.num_experts) &&
         gemm_tn_supported(c.is_act_and_mul ? kGemmW13 : kGemmW1, c.intermediate_size) &&
         gemm_tn_supported(kGemmW2, c.hidden_size);
}

// Split-K factors of a launch with a routed problem (tiles_r tiles of kb_r K blocks) and
// an optional shared problem (tiles_s of kb_s): the persistent grid runs
// ceil(units / SMs) rounds, each as long as the longest unit plus a fixed cost per unit,
// so pick (s_r, s_s) minimising rounds * (max(kb_r / s_r, kb_s / s_s) + kUnitCostKb); a
// split keeps >= 4 K blocks and must beat the best so far by 3 %. Only at decode-sized
// batches.
struct Splits {
  int r, s;
};
Splits choose_splits2(long tiles_r, int kb_r, long tiles_s, int kb_s, int T) {
  Splits best{1, 1};
  if (T > kSplitMaxTokens || tiles_r + tiles_s <= 0) return best;
  const long sms = num_sms();
  auto cost = [&](int sr, int ss) {
    const long units = tiles_r * sr + tiles_s * ss;
    double len = tiles_r ? (double)kb_r / sr : 0.0;
    if (tiles_s && (double)kb_s / ss > len) len = (double)kb_s / ss;
    return (double)((units + sms - 1) / sms) * (len + kUnitCostKb);
  };
  double best_t = cost(1, 1);
  for (int sr = 1; sr <= (int)kMaxSplits && kb_r / sr >= 4; ++sr)
    for (int ss = 1; ss <= (int)kMaxSplits && (tiles_s == 0 ? ss == 1 : kb_s / ss >= 4); ++ss) {
      const double t = cost(sr, ss);
      if (t < best_t * 0.97) {
        best = {sr, ss};
        best_t = t;
      }
    }
  return best;
}
int choose_splits(long tiles, int k_blocks, int T) { return choose_splits2(tiles, k_blocks, 0, 0, T).r; }

long t_blocks_128(int T) { return ((long)T + kGemmBM - 1) / kGemmBM; }

struct Layout {
  int bs, n, max_sorted, max_blocks, slots;
  bool fp8;
  // launch plan of one forward: small-batch routing, fused row copy, token-N GEMMs (tn),
  // split factors
  bool small, fused_copy, tn;
  bool nvfp4;
  int w2_bn, splits13, splits13_shared, splits2, splits2_shared, splits_router, launches;
  size_t status, topk_weights, topk_ids, sorted, expert_ids, npp, block_seg, block_rows, inv,
      scratch,
      x_perm, act, ytok, act_s, part_r, part_s, logits, xq, tile_cnt, tail_part, total;
  int tile_cnt_r, tile_cnt_s;  // counters of the fused split reduce (routed, shared); 0 = none
  int tail_cnt;                // counters of the w2 stream-K tail (after those); 0 = none
  // fp8: byte offsets of the scales inside x_perm / act / act_s / xq
  size_t xs_perm, act_scale, act_s_scale, xs_tok;
};

Layout layout_for(const gbmoe_config_t& c, int T) {
  Layout L;
  const int E = c.num_experts, k = c.top_k, H = c.hidden_size, I = c.intermediate_size;
  const int Is = c.shared_intermediate_size;
  L.tn = use_tn(c, T);
  L.fp8 = c.weight_quant == GBMOE_QUANT_FP8_BLOCK128;
  L.nvfp4 = c.weight_quant == GBMOE_QUANT_NVFP4;
  L.bs = L.tn ? 2 * kGemmBM : (L.nvfp4 ? kFp4BS : kGemmBM);
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
  L.block_seg = o;
  o = up(o + (size_t)L.max_blocks * 8);
  L.block_rows = o;
  o = up(o + (size_t)L.max_blocks * 4);
  L.inv = o;
  o = up(o + (size_t)L.n * 4);
  L.scratch = o;
  o = up(o + align_scratch_bytes(L.n, E));
  L.x_perm = o;
  o = up(o + (size_t)L.max_sorted * H * 2);
  L.act = o;
  o = up(o + (size_t)L.max_sorted * I * 2);
  // split-K copies exist only for T <= kSplitMaxTokens; every region grows with T
  const size_t ts = (size_t)(T < kSplitMaxTokens ? T : kSplitMaxTokens);
  const size_t ytok_rows = (size_t)T > kMaxSplits * ts ? (size_t)T : kMaxSplits * ts;
  L.ytok = o;
  o = up(o + ytok_rows * L.slots * H * 4);
  L.act_s = o;
  {
    const size_t bf16_bytes = (size_t)T * Is * 2;
    const size_t fp8_bytes = Is ? up((size_t)T * Is) + (size_t)(Is / 128) * T * 4 : 0;
    o = up(o + (bf16_bytes > fp8_bytes ? bf16_bytes : fp8_bytes));
  }
  // the NVFP4 first GEMM always writes fp32 partials (its act is quantized by the reduce)
  const size_t part_rows = L.nvfp4 && (size_t)T > kMaxSplits * ts ? (size_t)T : kMaxSplits * ts;
  L.part_r = o;
  o = up(o + part_rows * k * (c.is_act_and_mul ? 2 : 1) * I * 4);
  L.part_s = o;
  o = up(o + part_rows * 2 * Is * 4);
  L.logits = o;                       // router GEMM output (per-split copies at decode)
  o = up(o + ((size_t)T > kMaxSplits * ts ? (size_t)T : kMaxSplits * ts) * E * 4);
  // fp8: e4m3 rows then group-major fp32 scales, inside the bf16-sized regions above (a
  // byte plus 4/128 bytes per element fits in 2 bytes); the token-order input has its own
  L.xq = o;
  if (L.fp8) o = up(o + up((size_t)T * H) + (size_t)(H / kFp8Block) * T * 4);
  if (L.nvfp4 && Is) o = up(o + (size_t)T * H * 2);  // f16 token-order rows (shared expert)
  L.xs_perm = L.fp8 ? up((size_t)L.max_sorted * H) : 0;
  L.act_scale = L.fp8 ? up((size_t)L.max_sorted * I) : 0;
  L.act_s_scale = L.fp8 ? up((size_t)T * Is) : 0;
  L.xs_tok = L.fp8 ? up((size_t)T * H) : 0;
  L.tile_cnt = o;                     // filled in with the launch plan below
  L.total = o;

  // launch plan
  L.small = route_align_small_ok(T, k, E);
  L.fused_copy = L.small && L.n <= kFusedCopyMaxRows && !L.fp8 && !L.nvfp4;
  L.w2_bn = (H % 256 == 0) ? 256 : 128;
  const int kblk = L.fp8 ? kFp8Block : (L.nvfp4 ? kFp4StageK : kGemmBK);  // K per GEMM stage
  const long est_blocks = (long)(L.n < E ? L.n : E) + L.n / kGemmBM;  // >= 1 partial per expert
  const long t_blocks = ((long)T + L.bs - 1) / L.bs;
  if (L.tn) {
    L.splits13 = L.splits13_shared = L.splits2 = L.splits2_shared = 1;
  } else {
    const Splits a = choose_splits2(est_blocks * (I / kGemmBM), H / kblk,
                                    Is ? t_blocks * (Is / kGemmBM) : 0, H / kblk, T);
    L.splits13 = a.r;
    L.splits13_shared = a.s;
    const Splits b = choose_splits2(est_blocks * (H / L.w2_bn), I / kblk,
                                    Is ? t_blocks * (H / L.w2_bn) : 0, Is / kblk, T);
    L.splits2 = b.r;
    L.splits2_shared = b.s;
  }
  // bf16 split-K first GEMMs with two splits finish the activation in their last split
  // (per-tile counters, cleared by the routing kernel). With more splits the units are short
  // and their fence + atomic each cost more than the separate reduce kernel saves (measured:
  // Mixtral T = 1 with 2 splits 175 -> 153 us, DeepSeek-V2 T = 1 with 3 splits 115 -> 120 us),
  // so those, and the fp8 ones, keep the reduce kernel.
  const bool split13 = L.splits13 > 1 || (Is && L.splits13_shared > 1);
  const int max_split13 = L.splits13 > (Is ? L.splits13_shared : 1) ? L.splits13
                                                                     : (Is ? L.splits13_shared : 1);
  const bool fused_reduce = split13 && !L.fp8 && !L.nvfp4 && max_split13 <= 2;
  L.tile_cnt_r = fused_reduce ? (L.max_sorted / L.bs) * (I / kGemmBM) * 4 : 0;
  L.tile_cnt_s = fused_reduce && Is ? (int)t_blocks * (Is / kGemmBM) * 4 : 0;
  // bf16 w2 without split-K: a stream-K tail evens out the last round of tiles (up to one
  // 128 x N-tile fp32 partial per SM)
  const bool tail = T > kSplitMaxTokens && !L.fp8 && !L.nvfp4 && !L.tn;
  L.tail_cnt = tail ? num_sms() * 4 : 0;
  L.tail_part = up(L.tile_cnt + (size_t)(L.tile_cnt_r + L.tile_cnt_s + L.tail_cnt) * 4);
  L.total = up(L.tail_part + (tail ? (size_t)num_sms() * kGemmBM * L.w2_bn * 4 : 0));
  L.launches = (L.small ? (L.fused_copy ? 1 : 2) : 5) + 1 +
               ((split13 && !fused_reduce) || L.nvfp4 ? 1 : 0) + 1 + 1;
  L.splits_router = choose_splits(t_blocks_128(T) * ((E + kGemmBM - 1) / kGemmBM), H / kGemmBK, T);
  return L;
}

template <typename T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<char*>(ws) + off);
}

gbmoe_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? GBMOE_OK : GBMOE_ERR_CUDA; }

// Row blocks walked together: keep a group's A rows (bm x K bf16 each) near 40 MB.
int group_m_for(int K, int bm = kGemmBM) {
  const long per_block = (long)bm * K * 2;
  long g = (40l << 20) / per_block;
  if (g < 1) g = 1;
  if (g > 16) g = 16;
  return (int)g;
}

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
  PdlChain chain;
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
  PdlChain chain;
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
  if (check_layer(cfg) != GBMOE_OK || num_tokens < 0) return kGemmBM;
  return use_tn(*cfg, num_tokens) ? 2 * kGemmBM : kGemmBM;
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
  out->act_scale = L.fp8 ? L.act + L.act_scale : 0;
  out->total = L.total;
  out->act_shared = cfg->shared_intermediate_size ? L.act_s : 0;
  return GBMOE_OK;
}

GBMOE_API gbmoe_status_t moe_forward_ex(const gbmoe_config_t* cfg, int32_t num_tokens,
                                        const gbmoe_forward_args_t* args,
                                        gbmoe_stream_t stream_) {
  if (!args) return GBMOE_ERR_INVALID_ARG;
  const void* hidden_states = args->hidden_states;
  const float* router_logits = args->router_logits;
  const void* gate_weight = args->gate_weight;
  const float* e_score_correction_bias = args->e_score_correction_bias;
  const void* w13_weight = args->w13_weight;
  const void* w2_weight = args->w2_weight;
  const void* shared_w13 = args->shared_w13;
  const void* shared_w2 = args->shared_w2;
  const __nv_bfloat16* w13_bias = static_cast<const __nv_bfloat16*>(args->w13_bias);
  const __nv_bfloat16* w2_bias = static_cast<const __nv_bfloat16*>(args->w2_bias);
  void* output = args->output;
  void* workspace = args->workspace;
  const size_t workspace_bytes = args->workspace_bytes;
  void* const* events = args->events;
  const int32_t num_events = args->num_events;
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
  if (!hidden_states || (!router_logits == !gate_weight) || !w13_weight || !w2_weight ||
      !output || !aligned16(gate_weight))
    return GBMOE_ERR_INVALID_ARG;
  if (!aligned16(hidden_states) || !aligned16(w13_weight) || !aligned16(w2_weight) ||
      !aligned16(output) || (Is && (!aligned16(shared_w13) || !aligned16(shared_w2))) ||
      !aligned16(w13_bias) || !aligned16(w2_bias))
    return GBMOE_ERR_INVALID_ARG;
  const bool fp8 = c.weight_quant == GBMOE_QUANT_FP8_BLOCK128;
  const bool nvfp4 = c.weight_quant == GBMOE_QUANT_NVFP4;
  if ((fp8 || nvfp4) && (w13_bias || w2_bias)) return GBMOE_ERR_UNSUPPORTED;
  if (fp8 ? (!args->w13_scale || !args->w2_scale ||
             (Is && (!args->shared_w13_scale || !args->shared_w2_scale)))
          : (args->w13_scale || args->w2_scale || args->shared_w13_scale || args->shared_w2_scale))
    return GBMOE_ERR_INVALID_ARG;
  auto scale_ok = [](float g) { return std::isfinite(g) && g > 0.f; };
  if (nvfp4 ? (!args->w13_weight_scale_2 || !args->w2_weight_scale_2 ||
               !scale_ok(args->input_scale) || !scale_ok(args->act_scale) ||
               (Is && (!args->shared_weight_scale_2 || !scale_ok(args->shared_input_scale) ||
                       !scale_ok(args->shared_act_scale))))
            : (args->w13_weight_scale_2 || args->w2_weight_scale_2 || args->shared_weight_scale_2))
    return GBMOE_ERR_INVALID_ARG;
  const Layout L = layout_for(c, num_tokens);
  if (!workspace || workspace_bytes < L.total || (reinterpret_cast<uintptr_t>(workspace) % kAlign))
    return GBMOE_ERR_WORKSPACE;

  cudaStream_t stream = (cudaStream_t)stream_;
  const int T = num_tokens, E = c.num_experts, k = c.top_k, H = c.hidden_size,
            I = c.intermediate_size;
  PdlChain chain;  // the forward's kernels overlap their predecessors' tails
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
  // inside a stream capture the records are external, so they become event-record nodes
  // of the graph (a plain record there only marks a capture dependency)
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (events && cudaStreamIsCapturing(stream, &cap) != cudaSuccess) return GBMOE_ERR_CUDA;
  auto rec = [&](int i) -> cudaError_t {
    if (!events || !events[i]) return cudaSuccess;
    pdl_next() = false;  // the kernel after a stage event starts after it
    return cap == cudaStreamCaptureStatusActive
               ? cudaEventRecordWithFlags((cudaEvent_t)events[i], stream, cudaEventRecordExternal)
               : cudaEventRecord((cudaEvent_t)events[i], stream);
  };
  const int w2_bn = L.w2_bn;
  const int t_pad = (T + L.bs - 1) / L.bs * L.bs;
  cudaError_t e;

#define GBMOE_TRY(x)                   \
  do {                                 \
    e = (x);                           \
    if (e != cudaSuccess) return GBMOE_ERR_CUDA; \
  } while (0)

  GBMOE_TRY(rec(0));
  // router GEMM when the caller passes the gate weight instead of logits: inside the routing
  // launch for small batches (GateArgs), else a tensor-core GEMM before it
  int logit_splits = 1;
  long long logit_stride = 0;
  GateArgs gate_args{nullptr, 1, nullptr, nullptr};
  if (!router_logits && L.small && kGateFused) {
    gate_args.gate = gate_weight;
    gate_args.splits = gate_splits(E, H);
    gate_args.part = at<float>(workspace, L.logits);
    gate_args.counter = at<int>(workspace, L.status + kGateCounterOffset);
  } else if (!router_logits) {
    GemmLaunch gr;
    std::memset(&gr, 0, sizeof(gr));
    gr.status = status;
    gr.num_problems = 1;
    gr.splits = L.splits_router;
    GemmProblem& P = gr.p[0];
    const int tp = (T + kGemmBM - 1) / kGemmBM * kGemmBM;
    P.A = hidden_states;
    P.a_rows = T;
    P.B = gate_weight;
    P.b_rows = E;
    P.K = H;
    P.n_tiles = (E + kGemmBM - 1) / kGemmBM;
    P.k_blocks = H / kGemmBK;
    P.m_rows_host = tp;
    P.max_m_blocks = tp / kGemmBM;
    P.group_m = 16;
    P.num_experts = 1;
    P.out = at<float>(workspace, L.logits);
    P.ldo = E;
    P.store_rows = T;
    P.out_split_stride = (long long)T * E;
    GBMOE_TRY(launch_gemm(kGemmRouter, kGemmBM, gr, stream, T));
    router_logits = at<float>(workspace, L.logits);
    logit_splits = gr.splits;
    logit_stride = (long long)T * E;
  }
  int2* bseg = at<int2>(workspace, L.block_seg);
  int* brows = (L.tn || L.nvfp4) ? at<int>(workspace, L.block_rows) : nullptr;
  int* inv = at<int>(workspace, L.inv);
  int* tile_cnt = at<int>(workspace, L.tile_cnt);
  // apply_router_weight_on_input: the gathered rows carry the routing weight instead
  const float* row_scale = c.apply_router_weight_on_input ? tw : nullptr;
  const bool gated = c.is_act_and_mul != 0;
  const float alpha = c.gemm1_alpha == 0.f ? 1.f : c.gemm1_alpha;
  // fp8: the input is quantized once per token while it is gathered (and kept in token
  // order for the shared expert)
  uint8_t* xq_tok = at<uint8_t>(workspace, L.xq);
  float* xs_tok = at<float>(workspace, L.xq + L.xs_tok);
  float* xs_perm = at<float>(workspace, L.x_perm + L.xs_perm);
  void* x_tok16 = at<char>(workspace, L.xq);  // nvfp4: f16 token-order rows (shared expert)
  auto gather = [&]() -> cudaError_t {
    if (nvfp4)
      return launch_quant_gather_fp4(hidden_states, H, inv, L.n, k, T, L.max_sorted,
                                     args->input_scale, x_perm, Is ? x_tok16 : nullptr,
                                     args->shared_input_scale, stream);
    if (fp8)
      return launch_quant_gather_fp8(hidden_states, H, inv, L.n, k, T,
                                     static_cast<uint8_t*>(x_perm), xs_perm, L.max_sorted,
                                     Is ? xq_tok : nullptr, xs_tok, stream);
    return launch_gather(hidden_states, H, inv, L.n, k, L.max_sorted, x_perm, row_scale, stream);
  };
  if (L.small) {
    const bool fused_copy = L.fused_copy;
    GBMOE_TRY(launch_route_align_small(c, T, router_logits, e_score_correction_bias, tw, tids,
                                       L.bs, sorted, eids, L.max_blocks, npp, bseg, inv,
                                       hidden_states, fused_copy ? x_perm : nullptr, row_scale,
                                       status, stream, logit_splits, logit_stride, tile_cnt,
                                       L.tile_cnt_r + L.tile_cnt_s + L.tail_cnt, gate_args));
    if (!fused_copy) GBMOE_TRY(gather());
  } else {
    GBMOE_TRY(launch_topk(c, T, router_logits, e_score_correction_bias, tw, tids, status, stream,
                          logit_splits, logit_stride, tile_cnt,
                          L.tile_cnt_r + L.tile_cnt_s + L.tail_cnt));
    GBMOE_TRY(launch_align(tids, L.n, E, L.bs, sorted, eids, L.max_blocks, npp,
                           at<char>(workspace, L.scratch), status, stream, bseg, inv, brows));
    GBMOE_TRY(gather());
  }
  GBMOE_TRY(rec(1));
  const long long slot_copy = (long long)T * L.slots * H;

  if (nvfp4) {
    // ---- w13 (nvfp4): alpha-scaled fp32 partials of [gate | up], routed and shared
    const int un13 = fp4_unit_rows(2 * I, Is ? 2 * Is : 256);
    const int un2 = fp4_unit_rows(H, H);
    GemmLaunch g1;
    std::memset(&g1, 0, sizeof(g1));
    g1.status = status;
    g1.num_problems = Is ? 2 : 1;
    {
      GemmProblem& P = g1.p[0];
      P.A = x_perm;
      P.a_rows = L.max_sorted;
      P.B = w13_weight;
      P.b_rows = E * 2 * I;
      P.K = H;
      P.n_tiles = 2 * I / un13;
      P.k_blocks = H / kFp4StageK;
      P.m_rows_dev = npp;
      P.max_m_blocks = L.max_sorted / L.bs;
      P.expert_ids = eids;
      P.block_seg = bseg;
      P.block_rows = L.small ? nullptr : brows;
      P.rows_bound = T < kFp4BS ? T : kFp4BS;
      P.group_m = group_m_for(H, L.bs);
      P.num_experts = E;
      P.b_rows_per_expert = 2 * I;
      P.up_offset = I;
      P.out = act;
      P.ldo = I;
      P.store_rows = L.max_sorted;
      P.sorted_ids = sorted;
      P.num_flat = L.n;
      P.flat_row = inv;
      P.part = at<float>(workspace, L.part_r);
      P.part_split_stride = (long long)L.n * 2 * I;
      P.scale2 = args->w13_weight_scale_2;
      P.gscale = args->input_scale;
    }
    if (Is) {
      GemmProblem& P = g1.p[1];
      P.A = x_tok16;
      P.a_rows = T;
      P.B = shared_w13;
      P.b_rows = 2 * Is;
      P.K = H;
      P.n_tiles = 2 * Is / un13;
      P.k_blocks = H / kFp4StageK;
      P.m_rows_host = t_pad;
      P.max_m_blocks = t_pad / L.bs;
      P.group_m = group_m_for(H, L.bs);
      P.num_experts = 1;
      P.b_rows_per_expert = 2 * Is;
      P.up_offset = Is;
      P.out = act_s;
      P.ldo = Is;
      P.store_rows = T;
      P.num_flat = L.n;
      P.part = at<float>(workspace, L.part_s);
      P.part_split_stride = (long long)T * 2 * Is;
      P.scale2 = args->shared_weight_scale_2;
      P.gscale = args->shared_input_scale;
    }
    g1.splits = L.splits13;
    g1.splits_p1 = L.splits13_shared;
    GBMOE_TRY(launch_gemm_fp4(kGemmW13, g1, stream));
    GBMOE_TRY(launch_silu_quant_fp4(g1, npp, L.max_sorted, args->act_scale,
                                    Is ? args->shared_act_scale : 1.f, stream));
    GBMOE_TRY(rec(2));

    // ---- w2 (nvfp4): weighted fp32 slot outputs; the shared expert to slot k
    GemmLaunch g2;
    std::memset(&g2, 0, sizeof(g2));
    g2.status = status;
    g2.num_problems = Is ? 2 : 1;
    {
      GemmProblem& P = g2.p[0];
      P.A = act;
      P.a_rows = L.max_sorted;
      P.B = w2_weight;
      P.b_rows = E * H;
      P.K = I;
      P.n_tiles = H / un2;
      P.k_blocks = I / kFp4StageK;
      P.m_rows_dev = npp;
      P.max_m_blocks = L.max_sorted / L.bs;
      P.expert_ids = eids;
      P.block_seg = bseg;
      P.block_rows = L.small ? nullptr : brows;
      P.rows_bound = T < kFp4BS ? T : kFp4BS;
      P.group_m = group_m_for(I, L.bs);
      P.num_experts = E;
      P.b_rows_per_expert = H;
      P.out = ytok;
      P.ldo = H;
      P.store_rows = L.max_sorted;
      P.sorted_ids = sorted;
      P.row_weight = tw;
      P.num_flat = L.n;
      P.top_k = k;
      P.slots = L.slots;
      P.out_split_stride = slot_copy;
      P.scale2 = args->w2_weight_scale_2;
      P.gscale = args->act_scale;
    }
    if (Is) {
      GemmProblem& P = g2.p[1];
      P.A = act_s;
      P.a_rows = T;
      P.B = shared_w2;
      P.b_rows = H;
      P.K = Is;
      P.n_tiles = H / un2;
      P.k_blocks = Is / kFp4StageK;
      P.m_rows_host = t_pad;
      P.max_m_blocks = t_pad / L.bs;
      P.group_m = group_m_for(Is, L.bs);
      P.num_experts = 1;
      P.b_rows_per_expert = H;
      P.out = ytok;
      P.ldo = H;
      P.store_rows = T;
      P.num_flat = L.n;
      P.top_k = k;
      P.slots = L.slots;
      P.slot_offset = k;
      P.out_split_stride = slot_copy;
      P.scale2 = args->shared_weight_scale_2 + 1;
      P.gscale = args->shared_act_scale;
    }
    g2.splits = L.splits2;
    g2.splits_p1 = L.splits2_shared;
    GBMOE_TRY(launch_gemm_fp4(kGemmW2, g2, stream));
    GBMOE_TRY(rec(3));
    GBMOE_TRY(launch_combine(ytok, L.slots, k, H, T, g2.splits, Is ? g2.splits_p1 : g2.splits,
                             slot_copy, output, stream));
    GBMOE_TRY(rec(4));
    return GBMOE_OK;
  }

  if (fp8) {
    // ---- w13 (fp8): e4m3 act + scales, routed and shared experts in one launch
    GemmLaunch g1;
    std::memset(&g1, 0, sizeof(g1));
    g1.status = status;
    g1.num_problems = Is ? 2 : 1;
    {
      GemmProblem& P = g1.p[0];
      P.A = x_perm;
      P.a_rows = L.max_sorted;
      P.a_scale = xs_perm;
      P.a_scale_ld = L.max_sorted;
      P.B = w13_weight;
      P.b_rows = E * 2 * I;
      P.b_scale = args->w13_scale;
      P.K = H;
      P.n_tiles = I / kFp8Block;
      P.k_blocks = H / kFp8Block;
      P.m_rows_dev = npp;
      P.max_m_blocks = L.max_sorted / L.bs;
      P.expert_ids = eids;
      P.block_seg = bseg;
      P.group_m = group_m_for(H / 2, L.bs);
      P.num_experts = E;
      P.b_rows_per_expert = 2 * I;
      P.up_offset = I;
      P.out = act;
      P.out_scale = at<float>(workspace, L.act + L.act_scale);
      P.out_scale_ld = L.max_sorted;
      P.ldo = I;
      P.store_rows = L.max_sorted;
      P.sorted_ids = sorted;
      P.num_flat = L.n;
      P.part = at<float>(workspace, L.part_r);
      P.part_split_stride = (long long)L.n * 2 * I;
      P.flat_row = inv;
    }
    if (Is) {
      GemmProblem& P = g1.p[1];
      P.A = xq_tok;
      P.a_rows = T;
      P.a_scale = xs_tok;
      P.a_scale_ld = T;
      P.B = shared_w13;
      P.b_rows = 2 * Is;
      P.b_scale = args->shared_w13_scale;
      P.K = H;
      P.n_tiles = Is / kFp8Block;
      P.k_blocks = H / kFp8Block;
      P.m_rows_host = t_pad;
      P.max_m_blocks = t_pad / L.bs;
      P.group_m = group_m_for(H / 2, L.bs);
      P.num_experts = 1;
      P.b_rows_per_expert = 2 * Is;
      P.up_offset = Is;
      P.out = act_s;
      P.out_scale = at<float>(workspace, L.act_s + L.act_s_scale);
      P.out_scale_ld = T;
      P.ldo = Is;
      P.store_rows = T;
      P.num_flat = L.n;
      P.part = at<float>(workspace, L.part_s);
      P.part_split_stride = (long long)T * 2 * Is;
    }
    g1.splits = L.splits13;
    g1.splits_p1 = L.splits13_shared;
    GBMOE_TRY(launch_gemm_fp8(kGemmW13, g1, stream, T));
    if (g1.splits > 1 || (Is && g1.splits_p1 > 1))
      GBMOE_TRY(launch_silu_reduce_fp8(g1, npp, L.max_sorted, stream));
    GBMOE_TRY(rec(2));

    // ---- w2 (fp8): weighted fp32 slot outputs; the shared expert to slot k
    GemmLaunch g2;
    std::memset(&g2, 0, sizeof(g2));
    g2.status = status;
    g2.num_problems = Is ? 2 : 1;
    {
      GemmProblem& P = g2.p[0];
      P.A = act;
      P.a_rows = L.max_sorted;
      P.a_scale = at<float>(workspace, L.act + L.act_scale);
      P.a_scale_ld = L.max_sorted;
      P.B = w2_weight;
      P.b_rows = E * H;
      P.b_scale = args->w2_scale;
      P.K = I;
      P.n_tiles = H / 256;
      P.k_blocks = I / kFp8Block;
      P.m_rows_dev = npp;
      P.max_m_blocks = L.max_sorted / L.bs;
      P.expert_ids = eids;
      P.block_seg = bseg;
      P.group_m = group_m_for(I / 2, L.bs);
      P.num_experts = E;
      P.b_rows_per_expert = H;
      P.out = ytok;
      P.ldo = H;
      P.store_rows = L.max_sorted;
      P.sorted_ids = sorted;
      P.row_weight = tw;
      P.num_flat = L.n;
      P.top_k = k;
      P.slots = L.slots;
      P.out_split_stride = slot_copy;
    }
    if (Is) {
      GemmProblem& P = g2.p[1];
      P.A = act_s;
      P.a_rows = T;
      P.a_scale = at<float>(workspace, L.act_s + L.act_s_scale);
      P.a_scale_ld = T;
      P.B = shared_w2;
      P.b_rows = H;
      P.b_scale = args->shared_w2_scale;
      P.K = Is;
      P.n_tiles = H / 256;
      P.k_blocks = Is / kFp8Block;
      P.m_rows_host = t_pad;
      P.max_m_blocks = t_pad / L.bs;
      P.group_m = group_m_for(Is / 2, L.bs);
      P.num_experts = 1;
      P.b_rows_per_expert = H;
      P.out = ytok;
      P.ldo = H;
      P.store_rows = T;
      P.num_flat = L.n;
      P.top_k = k;
      P.slots = L.slots;
      P.slot_offset = k;
      P.out_split_stride = slot_copy;
    }
    g2.splits = L.splits2;
    g2.splits_p1 = L.splits2_shared;
    GBMOE_TRY(launch_gemm_fp8(kGemmW2, g2, stream, T));
    GBMOE_TRY(rec(3));
    GBMOE_TRY(launch_combine(ytok, L.slots, k, H, T, g2.splits, Is ? g2.splits_p1 : g2.splits,
                             slot_copy, output, stream));
    GBMOE_TRY(rec(4));
    return GBMOE_OK;
  }


  // ---- w13 + SiLU*mul: routed experts and the shared expert in one launch
  GemmLaunch g1;
  std::memset(&g1, 0, sizeof(g1));
  g1.status = status;
  g1.num_problems = Is ? 2 : 1;
  {
    GemmProblem& P = g1.p[0];
    P.A = x_perm;
    P.a_rows = L.max_sorted;
    P.B = w13_weight;
    P.b_rows = E * (gated ? 2 : 1) * I;
    P.K = H;
    P.n_tiles = I / kGemmBM;
    P.bias = w13_bias;
    P.clamp_limit = c.swiglu_limit;
    P.alpha = alpha;
    P.expert_of_flat = tids;
    P.flat_row = inv;
    P.k_blocks = H / kGemmBK;
    P.m_rows_dev = npp;
    P.max_m_blocks = L.max_sorted / L.bs;
    P.expert_ids = eids;
    P.block_seg = bseg;
    P.group_m = group_m_for(H, L.bs);
    P.num_experts = E;
    P.b_rows_per_expert = (gated ? 2 : 1) * I;
    P.up_offset = gated ? I : 0;
    P.out = act;
    P.ldo = I;
    P.store_rows = L.max_sorted;
    P.sorted_ids = sorted;
    P.num_flat = L.n;
    P.part = at<float>(workspace, L.part_r);
    P.part_split_stride = (long long)L.n * (gated ? 2 : 1) * I;
    P.block_rows = brows;
  }
  if (Is) {
    GemmProblem& P = g1.p[1];
    P.A = hidden_states;
    P.a_rows = T;
    P.B = shared_w13;
    P.b_rows = 2 * Is;
    P.K = H;
    P.n_tiles = Is / kGemmBM;
    P.k_blocks = H / kGemmBK;
    P.m_rows_host = t_pad;
    P.max_m_blocks = t_pad / L.bs;
    P.group_m = group_m_for(H, L.bs);
    P.num_experts = 1;
    P.b_rows_per_expert = 2 * Is;
    P.up_offset = Is;
    P.out = act_s;
    P.ldo = Is;
    P.store_rows = T;
    P.num_flat = L.n;
    P.clamp_limit = c.swiglu_limit;              // the shared SwiGLU shares the limit,
    P.alpha = 1.f;                               // not alpha
    P.part = at<float>(workspace, L.part_s);
    P.part_split_stride = (long long)T * 2 * Is;
  }
  g1.splits = L.splits13;
  g1.splits_p1 = L.splits13_shared;
  if (L.tile_cnt_r) {
    g1.p[0].tile_count = tile_cnt;
    if (Is) g1.p[1].tile_count = tile_cnt + L.tile_cnt_r;
  }
  // a row block holds at most T real rows (a token meets an expert once)
  if (L.tn) {
    if (gated) g1.p[0].n_tiles = I / kGemmBM;    // units of 128 features (64 per CTA)
    else g1.p[0].n_tiles = I / 256;              // units of 256 features
    GBMOE_TRY(launch_gemm_tn(gated ? kGemmW13 : kGemmW1, g1, stream));
  } else {
    GBMOE_TRY(launch_gemm(gated ? kGemmW13 : kGemmW1, kGemmBM, g1, stream, T));
  }
  if ((g1.splits > 1 || (Is && g1.splits_p1 > 1)) && !L.tile_cnt_r)
    GBMOE_TRY(launch_silu_reduce(g1, npp, L.max_sorted, gated, stream));
  GBMOE_TRY(rec(2));

  // ---- w2: weighted, scattered to the token's slot; shared expert to slot k
  GemmLaunch g2;
  std::memset(&g2, 0, sizeof(g2));
  g2.status = status;
  g2.num_problems = Is ? 2 : 1;
  {
    GemmProblem& P = g2.p[0];
    P.A = act;
    P.a_rows = L.max_sorted;
    P.B = w2_weight;
    P.b_rows = E * H;
    P.K = I;
    P.n_tiles = H / w2_bn;
    P.k_blocks = I / kGemmBK;
    P.m_rows_dev = npp;
    P.max_m_blocks = L.max_sorted / L.bs;
    P.expert_ids = eids;
    P.block_seg = bseg;
    P.group_m = group_m_for(I, L.bs);
    P.num_experts = E;
    P.b_rows_per_expert = H;
    P.out = ytok;
    P.ldo = H;
    P.store_rows = L.max_sorted;
    P.sorted_ids = sorted;
    P.row_weight = c.apply_router_weight_on_input ? nullptr : tw;
    P.bias = w2_bias;
    P.num_flat = L.n;
    P.top_k = k;
    P.slots = L.slots;
    P.out_split_stride = slot_copy;
    P.block_rows = brows;
  }
  if (Is) {
    GemmProblem& P = g2.p[1];
    P.A = act_s;
    P.a_rows = T;
    P.B = shared_w2;
    P.b_rows = H;
    P.K = Is;
    P.n_tiles = H / w2_bn;
    P.k_blocks = Is / kGemmBK;
    P.m_rows_host = t_pad;
    P.max_m_blocks = t_pad / L.bs;
    P.group_m = group_m_for(Is, L.bs);
    P.num_experts = 1;
    P.b_rows_per_expert = H;
    P.out = ytok;
    P.ldo = H;
    P.store_rows = T;
    P.num_flat = L.n;
    P.top_k = k;
    P.slots = L.slots;
    P.slot_offset = k;
    P.out_split_stride = slot_copy;
  }
  g2.splits = L.splits2;
  g2.splits_p1 = L.splits2_shared;
  if (L.tail_cnt) {
    g2.tail_part = at<float>(workspace, L.tail_part);
    g2.tail_count = tile_cnt + L.tile_cnt_r + L.tile_cnt_s;
    g2.tail_max_splits = 8;
  }
  if (L.tn) {
    g2.p[0].n_tiles = H / 256;                   // units of 256 output rows
    if (Is) g2.p[1].n_tiles = H / 256;
    GBMOE_TRY(launch_gemm_tn(kGemmW2, g2, stream));
  } else {
    GBMOE_TRY(launch_gemm(kGemmW2, w2_bn, g2, stream, T));
  }
  GBMOE_TRY(rec(3));
  GBMOE_TRY(launch_combine(ytok, L.slots, k, H, T, g2.splits, Is ? g2.splits_p1 : g2.splits,
                           slot_copy, output, stream));
  GBMOE_TRY(rec(4));
#undef GBMOE_TRY
  return GBMOE_OK;
}

GBMOE_API gbmoe_status_t moe_forward_events(
    const gbmoe_config_t* cfg, int32_t num_tokens, const void* hidden_states,
    const float* router_logits, const float* e_score_correction_bias, const void* w13_weight,
    const void* w2_weight, const void* shared_w13, const void* shared_w2, void* output,
    void* workspace, size_t workspace_bytes, void* const* events, int32_t num_events,
    gbmoe_stream_t stream) {
  gbmoe_forward_args_t a;
  std::memset(&a, 0, sizeof(a));
  a.hidden_states = hidden_states;
  a.router_logits = router_logits;
  a.e_score_correction_bias = e_score_correction_bias;
  a.w13_weight = w13_weight;
  a.w2_weight = w2_weight;
  a.shared_w13 = shared_w13;
  a.shared_w2 = shared_w2;
  a.output = output;
  a.workspace = workspace;
  a.workspace_bytes = workspace_bytes;
  a.events = events;
  a.num_events = num_events;
  return moe_forward_ex(cfg, num_tokens, &a, stream);
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

GBMOE_API gbmoe_status_t moe_router_logits(int32_t num_tokens, int32_t hidden_size,
                                           int32_t num_experts, const void* hidden_states,
                                           const void* gate_weight, float* router_logits,
                                           gbmoe_stream_t stream) {
  if (num_tokens < 0 || num_tokens > kMaxTokens || hidden_size <= 0 || hidden_size % kGemmBK ||
      num_experts < 1 || num_experts > 1024)
    return GBMOE_ERR_INVALID_ARG;
  if (num_tokens == 0) return GBMOE_OK;
  if (!hidden_states || !gate_weight || !router_logits || !aligned16(hidden_states) ||
      !aligned16(gate_weight) || !aligned16(router_logits))
    return GBMOE_ERR_INVALID_ARG;
  const int T = num_tokens, E = num_experts;
  const int tp = (T + kGemmBM - 1) / kGemmBM * kGemmBM;
  GemmLaunch gr;
  std::memset(&gr, 0, sizeof(gr));
  gr.num_problems = 1;
  gr.splits = 1;
  GemmProblem& P = gr.p[0];
  P.A = hidden_states;
  P.a_rows = T;
  P.B = gate_weight;
  P.b_rows = E;
  P.K = hidden_size;
  P.n_tiles = (E + kGemmBM - 1) / kGemmBM;
  P.k_blocks = hidden_size / kGemmBK;
  P.m_rows_host = tp;
  P.max_m_blocks = tp / kGemmBM;
  P.group_m = 16;
  P.num_experts = 1;
  P.out = router_logits;
  P.ldo = E;
  P.store_rows = T;
  PdlChain chain;
  return cuda_status(launch_gemm(kGemmRouter, kGemmBM, gr, (cudaStream_t)stream, T));
}

GBMOE_API gbmoe_status_t moe_quant_fp8_per_token_group(int32_t num_rows, int32_t hidden_size,
                                                       const void* x, uint8_t* q, float* scale,
                                                       gbmoe_stream_t stream) {
  if (num_rows < 0 || num_rows > kMaxTokens || hidden_size <= 0 || hidden_size % kFp8Block)
    return GBMOE_ERR_INVALID_ARG;
  if (num_rows == 0) return GBMOE_OK;
  if (!x || !q || !scale || !aligned16(x) || !aligned16(q) ||
      (reinterpret_cast<uintptr_t>(scale) & 3u))
    return GBMOE_ERR_INVALID_ARG;
  PdlChain chain;
  return cuda_status(
      launch_quant_fp8(x, num_rows, hidden_size, q, scale, num_rows, (cudaStream_t)stream));
}

GBMOE_API gbmoe_status_t moe_quant_nvfp4(int32_t num_rows, int32_t hidden_size, const void* x,
                                         float global_scale, uint8_t* q, uint8_t* sf,
                                         gbmoe_stream_t stream) {
  if (num_rows < 0 || hidden_size <= 0 || hidden_size % 16 ||
      !std::isfinite(global_scale) || !(global_scale > 0.f))
    return GBMOE_ERR_INVALID_ARG;
  if (num_rows == 0) return GBMOE_OK;
  if (!x || !q || !sf || !aligned16(x) || (reinterpret_cast<uintptr_t>(q) & 7u))
    return GBMOE_ERR_INVALID_ARG;
  PdlChain chain;
  return cuda_status(launch_quant_fp4(x, num_rows, hidden_size, global_scale, q, sf,
                                      (cudaStream_t)stream));
}

GBMOE_API size_t moe_nvfp4_prepared_bytes(int32_t rows, int32_t K) {
  if (rows <= 0 || K <= 0 || rows % 128 || K % 64) return 0;
  return (size_t)rows / 128 * (size_t)(K / 64) * kFp4ChunkBytes;
}

GBMOE_API gbmoe_status_t moe_nvfp4_prepare_weight(int32_t rows, int32_t K, const uint8_t* packed,
                                                  const uint8_t* block_scale, uint8_t* out,
                                                  gbmoe_stream_t stream) {
  if (rows <= 0 || K <= 0 || rows % 128 || K % 64 || !packed || !block_scale || !out ||
      !aligned16(packed) || !aligned16(block_scale) || !aligned16(out))
    return GBMOE_ERR_INVALID_ARG;
  PdlChain chain;
  return cuda_status(launch_prepare_fp4(packed, block_scale, rows, K, out, (cudaStream_t)stream));
}

GBMOE_API int32_t moe_forward_num_launches(const gbmoe_config_t* cfg, int32_t num_tokens) {
  if (check_layer(cfg) != GBMOE_OK || num_tokens < 0 || num_tokens > kMaxTokens) return -1;
  if (num_tokens == 0) return 0;
  return layout_for(*cfg, num_tokens).launches;
}

GBMOE_API int32_t moe_forward_num_launches_ex(const gbmoe_config_t* cfg, int32_t num_tokens,
                                              int32_t from_gate_weight) {
  const int32_t n = moe_forward_num_launches(cfg, num_tokens);
  if (n <= 0 || !from_gate_weight) return n;
  // small batches compute the logits inside the routing launch; others add the router GEMM
  return (layout_for(*cfg, num_tokens).small && kGateFused) ? n : n + 1;
}

GBMOE_API gbmoe_status_t moe_selftest_bounded_wait(void* workspace, int32_t timeout_us,
                                                   gbmoe_stream_t stream) {
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) % kAlign) || timeout_us < 0 ||
      timeout_us > 10000000)
    return GBMOE_ERR_INVALID_ARG;
  return cuda_status(launch_wait_selftest(at<int>(workspace, 0), timeout_us,
                                          (cudaStream_t)stream));
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
