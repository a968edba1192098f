/*
 * gbmoe.h: C ABI of the GB300 (sm_103a) FusedMoE layer forward.
 *
 * The forward is the one the vLLM `fused_moe/layer` page builds around
 * `FusedMoE` (constructor arguments, `select_experts`, `forward_impl`) and the
 * sglang `fused_moe_triton/layer.py` page runs in one call
 * (`FlashInferFusedMoE.forward_impl`: router logits, correction bias, hidden
 * states and both expert weight stacks in, the combined output out), with the
 * DeepSeek shared expert of the sglang `models/deepseek_v2.py` page
 * (`DeepseekV2MoE.forward_normal`) added on top.
 *
 * Conventions for every entry point
 *  - All array pointers are DEVICE pointers owned by the caller. The library
 *    never allocates, frees or keeps them; scratch lives in a caller-provided
 *    workspace whose size the matching *_workspace_size() call returns.
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL = the legacy default
 *    stream) and the call returns without synchronising. Outputs are valid once
 *    the stream reaches that point.
 *  - Arguments are validated on the host before anything is enqueued; a
 *    negative status means nothing was enqueued (except GBMOE_ERR_CUDA, which
 *    reports a failed launch). Kernels never trap: a failed device-side check or a
 *    bounded wait that ran out is recorded in the int32 status word at the start
 *    of the workspace, read (and reset) with moe_get_device_status(). The word
 *    keeps the first error since its last reset, so a new workspace must start
 *    with its first 256 bytes zeroed.
 *  - bf16 tensors are passed as `const void*` (IEEE bfloat16, row-major).
 *  - num_tokens == 0 is a successful no-op (the empty-batch early return of
 *    `DeepseekV2MoE.forward_normal`).
 */
#ifndef GBMOE_H
#define GBMOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* gbmoe_stream_t; /* identical to cudaStream_t */

typedef enum {
  GBMOE_OK = 0,
  GBMOE_ERR_INVALID_ARG = -1,   /* null pointer, bad size, inconsistent flags */
  GBMOE_ERR_UNSUPPORTED = -2,   /* valid for the method, not built here (see each call) */
  GBMOE_ERR_WORKSPACE = -3,     /* workspace null or smaller than *_workspace_size() */
  GBMOE_ERR_CUDA = -4,          /* a CUDA runtime call or launch failed */
  GBMOE_ERR_DEVICE_CHECK = -5,  /* a device-side bounds check failed */
  GBMOE_ERR_TIMEOUT = -6        /* a device-side bounded wait ran out */
} gbmoe_status_t;

typedef enum { GBMOE_SCORE_SOFTMAX = 0, GBMOE_SCORE_SIGMOID = 1 } gbmoe_scoring_t;
typedef enum { GBMOE_ACT_SILU = 0 } gbmoe_act_t;
typedef enum {
  GBMOE_QUANT_NONE = 0,
  GBMOE_QUANT_FP8_BLOCK128 = 1,
  GBMOE_QUANT_NVFP4 = 2
} gbmoe_weight_quant_t;

/*
 * Layer configuration; field names follow the FusedMoE constructor (vLLM
 * `fused_moe/layer` page, `FusedMoE.__init__`) and `DeepseekV2MoE.__init__`
 * (sglang `models/deepseek_v2.py` page) for the shared expert.
 *
 *  num_experts            E, routed experts (1..1024)
 *  top_k                  k, experts per token (1..min(E, 32))
 *  hidden_size            H, a multiple of 128
 *  intermediate_size      I, a multiple of 128
 *  renormalize            !=0: divide the chosen weights by their sum
 *  use_grouped_topk       !=0: group-limited routing (num_expert_group,
 *                         topk_group required; E % num_expert_group == 0,
 *                         num_expert_group <= 32, topk_group <= num_expert_group,
 *                         top_k <= topk_group * E / num_expert_group)
 *  scoring_func           gbmoe_scoring_t; SIGMOID requires use_grouped_topk
 *                         (the constructor rejects non-softmax ungrouped routing)
 *  routed_scaling_factor  multiplies every routed weight (not the shared expert)
 *  activation             must be GBMOE_ACT_SILU (else UNSUPPORTED)
 *  is_act_and_mul         1: gated, w13 [E, 2I, H], act = silu-gate * up;
 *                         0: not gated (`is_gated=False`), w13 [E, I, H], act = silu(z)
 *  shared_intermediate_size  I_s of the dense shared SwiGLU expert; 0 = none;
 *                         else a multiple of 128 (gated routed experts only)
 *  swiglu_limit           > 0: clamp the gate to <= L and the up half to [-L, L]
 *                         before the activation (`swiglu_limit`, `gemm1_clamp_limit`;
 *                         also applied to the shared expert); 0 = no clamp
 *  gemm1_alpha            gated act = g * sigmoid(alpha * g) * u for the routed experts
 *                         (`gemm1_alpha`); 0 means 1
 *  apply_router_weight_on_input  != 0: the routing weight scales the expert's input
 *                         rows instead of its output (FusedMoE constructor argument)
 * The pages name the last three options without their arithmetic; the reading used is
 * the one the NPU clipped-SwiGLU call's arguments (alpha, limit, bias) point to.
 *  weight_quant           gbmoe_weight_quant_t. FP8_BLOCK128: the w8a8 fp8 layer of the
 *                         sglang `models/deepseek_v2.py` page (`DeepseekV2MoE`'s
 *                         quant-once path, `DeepseekV2MLP.forward`'s fp8 down GEMM):
 *                         expert and shared weights are e4m3fn bytes with one fp32 scale
 *                         per 128 x 128 block (w = q * scale[n / 128][k / 128]); the input
 *                         is quantized once per token and group of 128 hidden columns
 *                         (s = max(amax, 1e-10) / 448, q = e4m3(x / s), fp32), feeds the
 *                         routed and the shared experts, and each act is quantized the
 *                         same way before its w2 GEMM. Requires H % 256 == 0, gated SiLU
 *                         without clamp or alpha, no expert biases, no
 *                         apply_router_weight_on_input (else UNSUPPORTED).
 *                         NVFP4: the w4a4 layer of FlashInferFP4MoE (sglang
 *                         `fused_moe_triton/layer.py` page, `trtllm_fp4_block_scale_moe`):
 *                         weights are e2m1 codes with one e4m3 scale per 16 values along K
 *                         and a per-expert fp32 weight_scale_2 (w = q * sf * s2), passed in
 *                         the layout moe_nvfp4_prepare_weight writes; the input is quantized
 *                         per token and block of 16 with the per-tensor input_scale g
 *                         (sf = e4m3(g * amax / 6), q = e2m1(x * g / sf), fp32 steps;
 *                         dequantized q * sf / g), and each act the same way with act_scale
 *                         before its w2 GEMM (moe_quant_nvfp4 is that quantization alone).
 *                         Same restrictions as FP8_BLOCK128 (H % 128 suffices). The pages'
 *                         layer casts e_score_correction_bias to the activations' dtype
 *                         before routing; callers wanting that pass bf16-valued biases.
 */
typedef struct {
  int32_t num_experts;
  int32_t top_k;
  int32_t hidden_size;
  int32_t intermediate_size;
  int32_t renormalize;
  int32_t use_grouped_topk;
  int32_t num_expert_group;
  int32_t topk_group;
  int32_t scoring_func;
  float routed_scaling_factor;
  int32_t activation;
  int32_t is_act_and_mul;
  int32_t shared_intermediate_size;
  float swiglu_limit;
  float gemm1_alpha;
  int32_t apply_router_weight_on_input;
  int32_t weight_quant;
} gbmoe_config_t;

/*
 * moe_topk: router scoring and (grouped) top-k.
 * Defined by `FusedMoE.select_experts` (vLLM `fused_moe/layer` page): the
 * grouped_topk branch (num_expert_group, topk_group, scoring_func,
 * routed_scaling_factor, e_score_correction_bias), the biased fused_topk_bias
 * branch and the plain fused_topk branch.
 *  - score s = softmax(logits row) or sigmoid(logits); key q = s + bias when
 *    `e_score_correction_bias` is non-NULL, else q = s.
 *  - grouped: the topk_group groups (contiguous runs of E/num_expert_group
 *    experts) with the largest group score survive; the group score is the
 *    largest s in the group without a bias and the sum of the two largest q in
 *    the group with one.
 *  - the top_k largest q among surviving experts (ties to the lower index), in
 *    descending q order; weight = s of that expert, divided by the sum of the
 *    chosen s if renormalize, then times routed_scaling_factor.
 * router_logits [T, E] fp32; e_score_correction_bias [E] fp32 or NULL;
 * topk_weights [T, top_k] fp32 (out); topk_ids [T, top_k] int32 (out).
 * Errors: INVALID_ARG (nulls, sizes, group arguments), UNSUPPORTED (sigmoid
 * without grouping).
 */
gbmoe_status_t moe_topk(const gbmoe_config_t* cfg, int32_t num_tokens,
                        const float* router_logits, const float* e_score_correction_bias,
                        float* topk_weights, int32_t* topk_ids, gbmoe_stream_t stream);

/*
 * moe_align_block_size: group the (token, slot) pairs by expert, padded to
 * block_size, for the grouped expert GEMMs of the FusedMoE forward (the
 * Triton fused_moe path behind `UnquantizedFusedMoEMethod` on the vLLM
 * `fused_moe/layer` page).
 *  - flat index f = t*top_k + j of topk_ids [T, top_k] (int32, values in [0, E));
 *  - experts in ascending order, each expert's flat indices ascending (stable),
 *    each run padded with the sentinel T*top_k to a multiple of block_size;
 *  - sorted_token_ids [T*top_k + E*(block_size-1)] int32 (out; entries past
 *    num_tokens_post_padded are unspecified);
 *  - expert_ids [(T*top_k + E*(block_size-1)) / block_size + 1] int32 (out;
 *    one per block; entries past num_tokens_post_padded/block_size are -1);
 *  - num_tokens_post_padded [1] int32 (out) = sum over experts of the padded runs.
 * block_size: 1..1024. Workspace: moe_align_block_size_workspace_size().
 * A topk_id outside [0, E) sets GBMOE_ERR_DEVICE_CHECK in the device status and
 * is counted as expert 0.
 */
size_t moe_align_block_size_workspace_size(int32_t num_tokens, int32_t top_k, int32_t num_experts);
gbmoe_status_t moe_align_block_size(const int32_t* topk_ids, int32_t num_tokens, int32_t top_k,
                                    int32_t num_experts, int32_t block_size,
                                    int32_t* sorted_token_ids, int32_t* expert_ids,
                                    int32_t* num_tokens_post_padded, void* workspace,
                                    size_t workspace_bytes, gbmoe_stream_t stream);

/*
 * moe_align_block_size_no_workspace: moe_align_block_size for callers that cannot
 * allocate device memory. The pages have no counterpart; this entry point exists for
 * the deployment, not the method. Plugins hosted by a framework that owns and
 * pre-plans every device allocation (an inference server with a fixed memory pool, a
 * runtime whose extensions may not call cudaMalloc) have no workspace to pass, so
 * this variant keeps its scratch in a fixed 1 MiB device array inside the library and
 * allocates nothing. Same arguments and outputs as moe_align_block_size, minus the
 * workspace.
 *  - Limit: requests needing more than 1 MiB of scratch
 *    (2 * ceil(T*top_k / 2048) * num_experts * 4 bytes) return GBMOE_ERR_WORKSPACE.
 *  - The array is shared by every call on a device and keeps the last call's
 *    contents; each call overwrites what it reads, so nothing must start at zero.
 *    Calls that overlap on the GPU (unordered streams) race on it: do not issue them.
 *  - The first call on a device looks up the array's device address with that device
 *    current; make that first call before any stream capture.
 *  - No status word: a topk_id outside [0, E) is counted as expert 0, unreported.
 */
gbmoe_status_t moe_align_block_size_no_workspace(const int32_t* topk_ids, int32_t num_tokens,
                                                 int32_t top_k, int32_t num_experts,
                                                 int32_t block_size, int32_t* sorted_token_ids,
                                                 int32_t* expert_ids,
                                                 int32_t* num_tokens_post_padded,
                                                 gbmoe_stream_t stream);

/*
 * moe_forward: the whole layer, from router logits to the combined output.
 *  1. moe_topk (above);
 *  2. align by expert (above) with the block size moe_forward_block_size(),
 *     and gather the hidden rows into expert order;
 *  3. per block: [gate | up] = x_rows @ w13[e]^T, act = silu(gate) * up
 *     (`SiluAndMul` of `DeepseekV2MLP`; w13 rows [0, I) gate, [I, 2I) up as
 *     `FusedMoE._load_w13` lays them out), rounded to bf16;
 *  4. o = act @ w2[e]^T, times the token's routing weight;
 *  5. y[t] = sum over j ascending of the weighted o[t, j], plus the shared expert
 *     silu(x W1s^T) * (x W3s^T) W2s^T unscaled (`DeepseekV2MoE.forward_normal`),
 *     accumulated in fp32 and rounded once to bf16.
 * hidden_states [T, H] bf16; router_logits [T, E] fp32; bias [E] fp32 or NULL;
 * w13_weight [E, 2I, H] bf16; w2_weight [E, H, I] bf16; shared_w13 [2I_s, H] and
 * shared_w2 [H, I_s] bf16 (both NULL iff cfg->shared_intermediate_size == 0);
 * output [T, H] bf16 (out). All bf16 pointers 16-byte aligned.
 * Workspace: moe_forward_workspace_size(cfg, max_tokens) bytes, 256-byte
 * aligned, for any num_tokens <= max_tokens; its layout is reported by
 * moe_forward_workspace_layout().
 */
size_t moe_forward_workspace_size(const gbmoe_config_t* cfg, int32_t max_num_tokens);
int32_t moe_forward_block_size(const gbmoe_config_t* cfg, int32_t num_tokens);
gbmoe_status_t moe_forward(const gbmoe_config_t* cfg, int32_t num_tokens,
                           const void* hidden_states, const float* router_logits,
                           const float* e_score_correction_bias, const void* w13_weight,
                           const void* w2_weight, const void* shared_w13, const void* shared_w2,
                           void* output, void* workspace, size_t workspace_bytes,
                           gbmoe_stream_t stream);

/*
 * moe_forward_events: moe_forward that also records caller-created CUDA events
 * (cudaEvent_t, passed as void*) on `stream` at the stage boundaries:
 * events[0] before routing, [1] after routing + align + gather, [2] after the
 * w13 GEMMs, [3] after the w2 GEMMs, [4] after the combine; a NULL entry is
 * skipped. The records are external (cudaEventRecordExternal): inside a stream
 * capture they become event-record nodes that time each replay. `events` may be
 * NULL (then identical to moe_forward); num_events must then be 0, else 5.
 */
#define GBMOE_NUM_STAGE_EVENTS 5
gbmoe_status_t moe_forward_events(const gbmoe_config_t* cfg, int32_t num_tokens,
                                  const void* hidden_states, const float* router_logits,
                                  const float* e_score_correction_bias, const void* w13_weight,
                                  const void* w2_weight, const void* shared_w13,
                                  const void* shared_w2, void* output, void* workspace,
                                  size_t workspace_bytes, void* const* events, int32_t num_events,
                                  gbmoe_stream_t stream);

/*
 * moe_forward_ex: moe_forward with every tensor in one struct, plus the per-expert
 * biases of the FusedMoE `with_bias` / `has_bias` option (sglang
 * `fused_moe_triton/layer.py` page: `w13_weight_bias`, `w2_weight_bias`):
 *   [gate | up] = x @ w13[e]^T + w13_bias[e]   (w13_bias [E, 2I] bf16; [E, I] not gated)
 *   o = act @ w2[e]^T + w2_bias[e]              (w2_bias [E, H] bf16)
 * Either bias may be NULL; the shared expert has none. events / num_events as in
 * moe_forward_events (NULL / 0 for none).
 */
typedef struct {
  const void* hidden_states;
  const float* router_logits;
  const float* e_score_correction_bias;
  const void* w13_weight;
  const void* w2_weight;
  const void* shared_w13;
  const void* shared_w2;
  const void* w13_bias;
  const void* w2_bias;
  void* output;
  void* workspace;
  size_t workspace_bytes;
  void* const* events;
  int32_t num_events;
  const void* gate_weight;   /* [E, H] bf16: when router_logits is NULL, the logits are
                                computed first as hidden_states @ gate_weight^T with fp32
                                sums (`MoEGate.forward`); exactly one of the two is given.
                                Batches of at most 16 tokens compute them inside the routing
                                launch (no [T, E] logits pass of their own), larger ones with
                                the tensor-core GEMM of moe_router_logits. Uses the int32 at
                                byte 4 of the workspace as an arrival counter (zero between
                                calls, like the status word) */
  /* weight_quant == FP8_BLOCK128 only (else NULL): the weights above are e4m3fn bytes and
     these their fp32 block scales, row-major per matrix:
     w13_scale [E, 2I/128, H/128], w2_scale [E, H/128, I/128],
     shared_w13_scale [2I_s/128, H/128], shared_w2_scale [H/128, I_s/128] */
  const float* w13_scale;
  const float* w2_scale;
  const float* shared_w13_scale;
  const float* shared_w2_scale;
  /* weight_quant == NVFP4 only (else NULL / 0): w13_weight, w2_weight, shared_w13 and
     shared_w2 are prepared NVFP4 weights (moe_nvfp4_prepare_weight of the [E * 2I, H],
     [E * H, I], [2 I_s, H] and [H, I_s] stacks); these their fp32 per-expert scales
     (device): w13_weight_scale_2 [E], w2_weight_scale_2 [E], shared_weight_scale_2 [2]
     (w13, w2); and the per-tensor scales (host values > 0) of the input's and the act's
     quantization, routed and shared */
  const float* w13_weight_scale_2;
  const float* w2_weight_scale_2;
  const float* shared_weight_scale_2;
  float input_scale;
  float act_scale;
  float shared_input_scale;
  float shared_act_scale;
} gbmoe_forward_args_t;
gbmoe_status_t moe_forward_ex(const gbmoe_config_t* cfg, int32_t num_tokens,
                              const gbmoe_forward_args_t* args, gbmoe_stream_t stream);

/*
 * moe_router_logits: the router GEMM in front of the layer, `MoEGate.forward` on the
 * sglang `models/deepseek_v2.py` page: router_logits [T, E] fp32 = hidden_states
 * [T, H] bf16 @ gate_weight [E, H]^T bf16, fp32 accumulation on the tensor cores.
 * H a multiple of 64, 1 <= E <= 1024, pointers 16-byte aligned, T = 0 a no-op.
 */
gbmoe_status_t moe_router_logits(int32_t num_tokens, int32_t hidden_size, int32_t num_experts,
                                 const void* hidden_states, const void* gate_weight,
                                 float* router_logits, gbmoe_stream_t stream);

/*
 * moe_quant_fp8_per_token_group: the per-token-group-128 fp8 quant of bf16 rows that the
 * FP8_BLOCK128 layer applies to its input (sglang `models/deepseek_v2.py` page,
 * `DeepseekV2MoE._maybe_quant_moe_input_once`): for each row r and group g of 128
 * consecutive columns, s = max(max |x|, 1e-10) / 448 and q = e4m3fn(x / s), both one fp32
 * division, the conversion round-to-nearest-even saturating at +-448.
 *   x      [num_rows, hidden_size] bf16, device, 16-byte aligned
 *   q      [num_rows, hidden_size] e4m3fn bytes, device (written)
 *   scale  [hidden_size / 128, num_rows] fp32, device, group-major ("column-major
 *          scales"): scale[g * num_rows + r] (written)
 * hidden_size a positive multiple of 128; num_rows = 0 is a no-op. Asynchronous on
 * `stream`; INVALID_ARG for bad sizes or pointers.
 */
gbmoe_status_t moe_quant_fp8_per_token_group(int32_t num_rows, int32_t hidden_size,
                                             const void* x, uint8_t* q, float* scale,
                                             gbmoe_stream_t stream);

/*
 * moe_quant_nvfp4: fp4_quantize(x, global_scale, 16) as the FlashInferFP4MoE layer applies
 * it to its input (sglang `fused_moe_triton/layer.py` page, `_quantize_hidden_states_fp4`):
 * for each row and block of 16 consecutive columns, amax = max |x|, sf = e4m3(g * (amax /
 * 6)) (round to nearest even, saturating at 448), r = g / sf (0 when sf is 0), q =
 * e2m1(x * r) (round to nearest even, saturating at +-6), every step one fp32 operation.
 *   x      [num_rows, hidden_size] bf16, device, 16-byte aligned
 *   q      [num_rows, hidden_size / 2] bytes, device (written): element 2i in the low
 *          nibble of byte i; codes: bit 3 the sign, magnitudes 0, .5, 1, 1.5, 2, 3, 4, 6
 *   sf     [num_rows, hidden_size / 16] e4m3fn bytes, device (written)
 * hidden_size a positive multiple of 16, global_scale > 0 and finite; num_rows = 0 is a
 * no-op. Asynchronous on `stream`; INVALID_ARG for bad sizes or pointers.
 */
gbmoe_status_t moe_quant_nvfp4(int32_t num_rows, int32_t hidden_size, const void* x,
                               float global_scale, uint8_t* q, uint8_t* sf,
                               gbmoe_stream_t stream);

/*
 * moe_nvfp4_prepare_weight: rewrites one NVFP4 weight stack [rows, K] (the checkpoint
 * layout: packed codes [rows, K / 2], low nibble first, and e4m3 block scales [rows,
 * K / 16]) into the layout the NVFP4 expert GEMMs stream, as the pages' layer shuffles its
 * fp4 weights once at load time: for each tile of 128 rows and stage of 64 K values one
 * 4608-byte chunk, chunk (tile, kb) at byte (tile * K / 64 + kb) * 4608, holding
 *   bytes [h * 2048 + r * 16, +16)  the codes of row tile * 128 + r, values kb * 64 + 32 h
 *                                   .. + 31 (h = 0, 1)
 *   bytes [4096 + r * 4, +4)        that row's four block scales of the stage.
 * A permutation of bytes only. rows a positive multiple of 128, K of 64; packed, scales
 * and out 16-byte aligned device buffers; out holds moe_nvfp4_prepared_bytes(rows, K)
 * bytes (= rows * K * 9 / 16). Asynchronous on `stream`; INVALID_ARG for bad sizes or
 * pointers.
 */
size_t moe_nvfp4_prepared_bytes(int32_t rows, int32_t K);
gbmoe_status_t moe_nvfp4_prepare_weight(int32_t rows, int32_t K, const uint8_t* packed,
                                        const uint8_t* block_scale, uint8_t* out,
                                        gbmoe_stream_t stream);

/*
 * Byte offsets of the intermediate results inside a moe_forward workspace
 * (for inspection and tests). Each is valid after the call completes.
 */
typedef struct {
  size_t status;                 /* int32 device status word (see moe_get_device_status) */
  size_t topk_weights;           /* fp32 [T, top_k] */
  size_t topk_ids;               /* int32 [T, top_k] */
  size_t sorted_token_ids;       /* int32 [T*top_k + E*(bs-1)] */
  size_t expert_ids;             /* int32 [that / bs + 1] */
  size_t num_tokens_post_padded; /* int32 [1] */
  size_t act;                    /* bf16 [rows, I]: silu(gate)*up in expert order
                                    (FP8_BLOCK128: e4m3fn [rows, I], then fp32 scales
                                    [I/128][rows] at act_scale; NVFP4: f16 [rows, I], the
                                    values q * sf of the act's block quantization) */
  size_t act_scale;              /* FP8_BLOCK128 only, else 0 */
  size_t total;                  /* == moe_forward_workspace_size() */
  size_t act_shared;             /* the shared expert's act [T, I_s] in token order (bf16;
                                    NVFP4: f16 values q * sf of the quantized act); 0 when
                                    there is no shared expert */
} gbmoe_workspace_layout_t;
gbmoe_status_t moe_forward_workspace_layout(const gbmoe_config_t* cfg, int32_t max_num_tokens,
                                            gbmoe_workspace_layout_t* layout);

/*
 * moe_get_device_status: wait for `stream`, copy the int32 status word at the
 * start of `workspace` (a moe_forward or moe_align_block_size workspace) to
 * *status (GBMOE_OK or a negative gbmoe_status_t) and reset it to GBMOE_OK.
 * Returns GBMOE_ERR_CUDA if the copy fails.
 */
gbmoe_status_t moe_get_device_status(void* workspace, int32_t* status, gbmoe_stream_t stream);

/*
 * moe_forward_num_launches: number of kernels one moe_forward(cfg, num_tokens, ...)
 * enqueues (it depends on num_tokens: the small-batch routing path, split-K reduces).
 * Returns -1 for an invalid configuration.
 */
int32_t moe_forward_num_launches(const gbmoe_config_t* cfg, int32_t num_tokens);

/*
 * moe_forward_num_launches_ex: moe_forward_num_launches for a moe_forward_ex call that
 * passes the gate weight instead of router logits when from_gate_weight != 0. Batches of
 * at most 16 tokens (when num_tokens * top_k <= 2048) compute the router logits inside
 * their routing launch (the count is unchanged); larger ones add one router GEMM launch.
 * Returns -1 for an invalid configuration.
 */
int32_t moe_forward_num_launches_ex(const gbmoe_config_t* cfg, int32_t num_tokens,
                                    int32_t from_gate_weight);

/*
 * moe_selftest_bounded_wait: failure-detection self test. Enqueues one kernel whose
 * single thread waits on a shared-memory mbarrier that nothing completes, with the
 * same bounded wait the GEMM pipelines use, but giving up after timeout_us
 * (0..10^7) instead of one second; it then records GBMOE_ERR_TIMEOUT in the status
 * word of `workspace` (read it with moe_get_device_status) and exits, leaving the
 * context usable. Has no counterpart on the pages.
 */
gbmoe_status_t moe_selftest_bounded_wait(void* workspace, int32_t timeout_us,
                                         gbmoe_stream_t stream);

/* Library version, (major << 16) | minor. */
int32_t gbmoe_version(void);

#ifdef __cplusplus
}
#endif
#endif /* GBMOE_H */
