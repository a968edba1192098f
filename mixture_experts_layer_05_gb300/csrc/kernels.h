// Internal launch interface between the C ABI (api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/gbmoe.h"

namespace gbmoe {

constexpr int kAlignChunk = 2048;  // flat indices per align chunk (one scatter warp each)
constexpr int kGemmBM = 128;       // token rows per GEMM tile (= align block size)
constexpr int kGemmBK = 64;        // K elements per pipeline stage (one 128-byte swizzle row)

int num_sms();

// Whether the next launch_kernel() of this host thread may overlap the kernel before it in
// the stream (programmatic stream serialization). The forward clears it for its first
// kernel and after each stage event; every launch sets it for the next one.
bool& pdl_next();

// One C-ABI call: its first kernel launches normally, the later ones may overlap their
// predecessor, and nothing carries over to the next call.
struct PdlChain {
  PdlChain() { pdl_next() = false; }
  ~PdlChain() { pdl_next() = false; }
};

// Launch `k` on `stream`; with pdl_next() set, with programmatic stream serialization.
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*k)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  if (pdl_next()) {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  const cudaError_t e = cudaLaunchKernelEx(&cfg, k, static_cast<KArgs>(args)...);
  pdl_next() = true;
  return e;
}

// logits may arrive as logit_splits fp32 copies, logit_split_stride floats apart, whose sum
// is the logit (the split-K router GEMM); 1 = plain logits.
cudaError_t launch_topk(const gbmoe_config_t& c, int T, const float* logits, const float* bias,
                        float* weights, int* ids, int* status, cudaStream_t stream,
                        int logit_splits = 1, long long logit_split_stride = 0,
                        int* zero = nullptr, int zero_count = 0);

size_t align_scratch_bytes(int n, int E);
// block_seg (optional): per block, (first block, block count) of its expert's run.
// inv (optional): per flat index, its position in sorted order.
// block_rows (optional): per block, its real (non-padding) rows.
cudaError_t launch_align(const int* ids, int n, int E, int bs, int* sorted, int* expert_ids,
                         int max_blocks, int* npp, void* scratch, int* status,
                         cudaStream_t stream, int2* block_seg = nullptr, int* inv = nullptr,
                         int* block_rows = nullptr);
// Router logits of a small batch computed inside its routing launch, from the gate weight
// (MoEGate's x @ W_gate^T, bf16 operands, fp32 sums): CTA c takes experts 8 * (c / splits)
// + [0, 8) (a warp each) over K split c % splits, writes fp32 partial logits, and the last
// CTA to finish routes the batch from their split-ordered sum. gate == NULL: logits given.
struct GateArgs {
  const void* gate;   // [E, H] bf16
  int splits;         // K splits; the launch has ceil(E / 8) * splits CTAs
  float* part;        // [splits][T][E] fp32 partial logits (written)
  int* counter;       // CTAs that have finished their slice; zero between forwards
};
constexpr int kGateMaxSplits = 8;
// Gate K splits for a fused small-batch routing launch: about one CTA per SM.
int gate_splits(int E, int H);
// Routing + align of a small batch in one launch (when route_align_small_ok).
bool route_align_small_ok(int T, int k, int E);
cudaError_t launch_route_align_small(const gbmoe_config_t& c, int T, const float* logits,
                                     const float* bias, float* weights, int* ids, int bs,
                                     int* sorted, int* expert_ids, int max_blocks, int* npp,
                                     int2* block_seg, int* inv, const void* x, void* x_perm,
                                     const float* row_scale, int* status, cudaStream_t stream,
                                     int logit_splits = 1, long long logit_split_stride = 0,
                                     int* zero = nullptr, int zero_count = 0,
                                     GateArgs gate = GateArgs{nullptr, 1, nullptr, nullptr});
// x_perm[inv[f]] = x[f / k] (times row_scale[f] when row_scale is not NULL) for f < n
// (x_perm == NULL in the small launch: no copy there).
cudaError_t launch_gather(const void* x, int H, const int* inv, int n, int k, int max_rows,
                          void* x_perm, const float* row_scale, cudaStream_t stream);
constexpr int kFusedCopyMaxRows = 16;  // the small route+align launch copies rows itself

// y[t] = sum over copies c and slots of ytok[c * split_stride + (t * slots + slot) * H + :],
// where the routed slots (< routed_slots) have `splits` copies and the others
// `splits_last` copies (the split-K factors of the two w2 problems).
cudaError_t launch_combine(const void* ytok, int slots, int routed_slots, int H, int T,
                           int splits, int splits_last, long long split_stride, void* y,
                           cudaStream_t stream);

// W1: the non-gated first GEMM; Router: logits = x @ gate^T, fp32 per-split copies
enum GemmKind { kGemmW13 = 0, kGemmW2 = 1, kGemmW1 = 2, kGemmRouter = 3 };

// One grouped GEMM problem. A rows are grouped in blocks of kGemmBM that each belong
// to one expert (expert_ids[block]); B is the expert weight stack flattened to
// [num_experts * b_rows_per_expert, K].
struct GemmProblem {
  const void* A;           // bf16 [a_rows, K] (host side: for the tensor map)
  int a_rows;
  const void* B;           // bf16 [b_rows, K]
  int b_rows;
  int K;
  int n_tiles;             // output tiles along N
  int k_blocks;            // K / kGemmBK
  const int* m_rows_dev;   // device count of A rows (multiple of kGemmBM), or NULL
  int m_rows_host;         // A rows when m_rows_dev is NULL (multiple of kGemmBM)
  int max_m_blocks;        // upper bound on A row blocks
  const int* expert_ids;   // expert per row block, or NULL (all expert 0)
  const int2* block_seg;   // per row block: (first block, block count) of its expert run,
                           // or NULL (one run over all blocks)
  const int* block_rows;   // token-N GEMMs: real rows of each row block (routed problems),
                           // or NULL (identity rows: store_rows bounds them)
  int group_m;             // row blocks walked together across all N tiles (L2 reuse)
  int num_experts;
  int b_rows_per_expert;   // rows of B per expert
  int up_offset;           // w13: row offset of the up half inside an expert
  void* out;               // w13: bf16 act [rows, ldo]; w2: fp32 slot outputs [T*slots, ldo]
  int ldo;                 // output row stride (elements)
  int store_rows;          // identity-row problems: rows >= store_rows are padding
  const int* sorted_ids;   // routed problems: row -> flat index (>= num_flat: padding)
  const float* row_weight; // w2: weight per flat index, or NULL (weight 1)
  int num_flat;            // T * top_k (the sentinel)
  int top_k;               // w2: slots of routed experts per token
  int slots;               // w2: output slots per token
  int slot_offset;         // w2: slot of identity rows
  const __nv_bfloat16* bias;  // per-expert bias (w13: [E][2 ldo] gate | up; w1, w2: [E][ldo]),
                             // routed problem only, or NULL
  float clamp_limit;         // gated first GEMM: > 0 clamps gate <= L and up to [-L, L]
  float alpha;               // gated first GEMM: act = g * sigmoid(alpha g) * u
  const int* expert_of_flat; // split reduce: expert of each flat index (for the bias)
  const int* flat_row;       // split reduce: sorted row of each flat index, or NULL (then
                             // the reduce walks every sorted row)
  float* part;             // first GEMM with splits > 1: fp32 [splits][row][2 ldo] (gate | up;
                           // [row][ldo] non-gated), row = flat index (routed) or token
  long long part_split_stride;
  long long out_split_stride;  // w2: elements between the per-split copies of out
  int* tile_count;         // bf16 first GEMM with splits > 1: per (row block, N tile, TMEM lane
                           // quarter) arrival counters, zero at launch; the last split of each
                           // finishes the activation (no separate reduce). NULL: reduce kernel
  // FP8 (e4m3 w8a8, 128 x 128 weight blocks) problems only: A and B are e4m3 bytes,
  // K blocks are 128 wide, and out (w13) is e4m3 act with fp32 scales.
  const float* a_scale;    // A scales, K-block major: a_scale[kb * a_scale_ld + row]
  int a_scale_ld;          // rows covered by a_scale (rows >= it have no scale)
  const float* b_scale;    // B block scales [b_rows / 128][K / 128], row-major
  float* out_scale;        // w13: act scales, [ldo / 128][out_scale_ld] (group-major)
  int out_scale_ld;
  // NVFP4 problems only: A is f16 (quantized values q * sf), B the prepared fp4 weights,
  // each output scaled by alpha = scale2[expert] / gscale.
  const float* scale2;     // per-expert weight_scale_2 (the shared expert: one value)
  float gscale;            // per-tensor scale of the A rows' quantization
  int rows_bound;          // routed problems: real rows of any block <= it (block_rows, when
                           // given, counts them exactly)
};

// Up to two problems (the routed experts and the shared expert) in one persistent
// launch; every (problem, tile) is cut into `splits` equal K ranges (split-K).
struct GemmLaunch {
  GemmProblem p[2];
  int num_problems;
  int splits;       // split-K factor of problem 0
  int splits_p1;    // split-K factor of problem 1 (0 = same as problem 0)
  int* status;
  // Stream-K tail (bf16 w2): when the tiles leave a last round of at most half the grid, the
  // kernel cuts those tail tiles into up to tail_max_splits K ranges; each range writes an fp32
  // partial tile to tail_part ([range slot][128 rows][N tile]) and the last range to arrive
  // (per tile and TMEM lane quarter, counted in tail_count, zero at launch) sums them in range
  // order and runs the epilogue. tail_max_splits 0: no tail splitting.
  float* tail_part;
  int* tail_count;
  int tail_max_splits;
};

__host__ __device__ inline int splits_of(const GemmLaunch& L, int p) {
  return (p == 0 || L.splits_p1 <= 0) ? L.splits : L.splits_p1;
}

// Tokens-on-M grouped GEMM (128-row blocks, the token rows on the MMA's M side).
// max_rows_per_block: an upper bound on the real rows of any row block (<= 32 lets the
// kernel load 32-row A boxes and run a deeper pipeline).
cudaError_t launch_gemm(int kind, int bn, const GemmLaunch& L, cudaStream_t stream,
                        int max_rows_per_block = kGemmBM);

// Token-N grouped GEMMs on CTA pairs (prefill, no split-K): row blocks of 256 rows, each
// block's tokens on the MMA's N side, N = its real rows (GemmProblem.block_rows, or
// store_rows for identity problems) rounded up to 16. Units: kGemmW13 128 features
// (n_tiles = I / 128), kGemmW1 256 features (I / 256), kGemmW2 256 output rows (H / 256).
// gemm_tn_supported(kind, I or H): whether the sizes tile that way.
bool gemm_tn_supported(int kind, int hidden_or_inter);
cudaError_t launch_gemm_tn(int kind, const GemmLaunch& L, cudaStream_t stream);

// One mbarrier wait that nothing completes; gives up after timeout_us and records
// GBMOE_ERR_TIMEOUT in *status.
cudaError_t launch_wait_selftest(int* status, int timeout_us, cudaStream_t stream);

// act = f(sum_s gate_s + bias, sum_s up_s + bias) for the valid rows of each problem of a
// split first-GEMM launch (routed rows in expert order; identity rows for the shared
// expert, always gated); f = the gated activation with clamp / alpha, or silu (non-gated).
cudaError_t launch_silu_reduce(const GemmLaunch& L, const int* npp, int max_routed_rows,
                               bool gated, cudaStream_t stream);

// ---------------------------------------------------------------- FP8 (w8a8, block 128)
constexpr int kFp8Block = 128;  // quant group / weight block edge, = K elements per GEMM stage

// Per-token-group-128 quant of bf16 rows: q[r][c] = e4m3(x[r][c] / s), s = max(amax, 1e-10)
// / 448 over the row's 128-column group, stored group-major: s_out[g * s_ld + r].
cudaError_t launch_quant_fp8(const void* x, int rows, int H, uint8_t* q, float* s_out, int s_ld,
                             cudaStream_t stream);
// The same quant fused with the gather into expert order: x_perm_q[inv[f]] = q(x[f / k]) and
// its scales at xs_perm[g * perm_ld + inv[f]]; the slot-0 copy (f % k == 0) also writes the
// token-order row to xq_tok / xs_tok[g * T + t] when xq_tok is not NULL.
cudaError_t launch_quant_gather_fp8(const void* x, int H, const int* inv, int n, int k, int T,
                                    uint8_t* x_perm_q, float* xs_perm, int perm_ld,
                                    uint8_t* xq_tok, float* xs_tok, cudaStream_t stream);
// FP8 grouped GEMMs: kind kGemmW13 (bn 128: e4m3 act + scales, or fp32 partials when split)
// or kGemmW2 (bn 256: weighted fp32 slot outputs); K is promoted per 128-wide block.
cudaError_t launch_gemm_fp8(int kind, const GemmLaunch& L, cudaStream_t stream,
                            int max_rows_per_block = kGemmBM);
// Split reduce of an FP8 w13 launch: act = silu(sum gate) * sum up, quantized per group of
// 128 columns into e4m3 act + group-major scales.
cudaError_t launch_silu_reduce_fp8(const GemmLaunch& L, const int* npp, int max_routed_rows,
                                   cudaStream_t stream);

// ---------------------------------------------------------------- NVFP4 (w4a4, block 16)
constexpr int kFp4BS = 128;             // align block size of the NVFP4 forward (max MMA N)
constexpr int kFp4ChunkBytes = 4608;    // prepared weights: 128 rows x 64 K (4096 B of codes
                                        // + 512 B of block scales) per chunk
constexpr int kFp4StageK = 64;          // K per prepared chunk (GemmProblem.k_blocks = K / it;
                                        // the GEMM's stages take two chunks)
// weight rows per NVFP4 GEMM unit (GemmProblem.n_tiles = weight rows / it): 256 when every
// problem of the launch has a multiple of 256 weight rows per expert, else 128
inline int fp4_unit_rows(int rows0, int rows1) {
  return (rows0 % 256 == 0 && rows1 % 256 == 0) ? 256 : 128;
}

// fp4_quantize(x, g, 16) of bf16 rows [rows, H]: packed e2m1 codes q [rows, H / 2] (low
// nibble first) and e4m3 block scales sf [rows, H / 16].
cudaError_t launch_quant_fp4(const void* x, int rows, int H, float g, uint8_t* q, uint8_t* sf,
                             cudaStream_t stream);
// The same quant once per token, its f16 values q * sf written to x_perm row inv[f] for each
// of the token's k slots and, when x_tok is not NULL, to x_tok row t (with scale g_tok).
cudaError_t launch_quant_gather_fp4(const void* x, int H, const int* inv, int n, int k, int T,
                                    int max_rows, float g, void* x_perm, void* x_tok,
                                    float g_tok, cudaStream_t stream);
// NVFP4 grouped GEMMs (256 or 128 weight rows per unit, expanded into tensor memory as the
// MMA's M side; the row block's tokens on N; K a multiple of 128): kGemmW13 writes
// alpha-scaled fp32 partials [split][row][2 ldo] (gate | up), kGemmW2 weighted fp32 slot
// outputs.
cudaError_t launch_gemm_fp4(int kind, const GemmLaunch& L, cudaStream_t stream);
// act = silu(sum gate) * sum up of an NVFP4 first-GEMM launch, block-quantized with g_act
// (routed) / g_act_shared, written as f16 q * sf to out (routed rows through flat_row).
cudaError_t launch_silu_quant_fp4(const GemmLaunch& L, const int* npp, int max_routed_rows,
                                  float g_act, float g_act_shared, cudaStream_t stream);
// The prepared layout of one [rows, K] fp4 weight: see moe_nvfp4_prepare_weight.
cudaError_t launch_prepare_fp4(const uint8_t* packed, const uint8_t* scales, int rows, int K,
                               uint8_t* out, cudaStream_t stream);

}  // namespace gbmoe
