// Internal launch interface between the C ABI (api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/gbmoe.h"

namespace gbmoe {

constexpr int kAlignChunk = 2048;  // flat indices per align chunk (one scatter warp each)
constexpr int kGemmBM = 128;       // token rows per GEMM tile (= align block size)
constexpr int kGemmBK = 64;        // K elements per pipeline stage (one 128-byte swizzle row)

int num_sms();

cudaError_t launch_topk(const gbmoe_config_t& c, int T, const float* logits, const float* bias,
                        float* weights, int* ids, int* status, cudaStream_t stream);

size_t align_scratch_bytes(int n, int E);
cudaError_t launch_align(const int* ids, int n, int E, int bs, int* sorted, int* expert_ids,
                         int max_blocks, int* npp, void* scratch, int* status,
                         cudaStream_t stream);
cudaError_t launch_gather(const void* x, int H, const int* sorted, const int* npp, int n, int k,
                          int max_rows, void* x_perm, cudaStream_t stream);

cudaError_t launch_combine(const void* ytok, int slots, int H, int T, void* y,
                           cudaStream_t stream);

enum GemmKind { kGemmW13 = 0, kGemmW2 = 1 };

// One grouped GEMM launch. A rows are grouped in blocks of kGemmBM that each belong
// to one expert (expert_ids[block]); B is the expert weight stack flattened to
// [num_experts * b_rows_per_expert, K].
struct GemmArgs {
  int n_tiles;             // output tiles along N
  int k_blocks;            // K / kGemmBK
  const int* m_rows_dev;   // device count of A rows (multiple of kGemmBM), or NULL
  int m_rows_host;         // A rows when m_rows_dev is NULL (multiple of kGemmBM)
  int max_m_blocks;        // upper bound on A row blocks
  const int* expert_ids;   // expert per row block, or NULL (all expert 0)
  int num_experts;
  int b_rows_per_expert;   // rows of B per expert
  int up_offset;           // w13: row offset of the up half inside an expert
  void* out;               // w13: bf16 act; w2: fp32 per-slot outputs
  int ldo;                 // output row stride (elements)
  int store_rows;          // w13: rows >= store_rows are not stored; w2 identity rows: valid rows
  const int* sorted_ids;   // w2: row -> flat index, or NULL (row = token, identity)
  const float* row_weight; // w2: weight per flat index, or NULL (weight 1)
  int num_flat;            // w2: T * top_k (the sentinel)
  int top_k;               // w2: slots of routed experts per token
  int slots;               // w2: output slots per token
  int slot_offset;         // w2: slot of identity rows
  int* status;
};

// w13: A [rows, H] (x_perm or x), B = w13 [E*2I, H]; out act [rows, I] bf16
// w2:  A [rows, I] (act),           B = w2  [E*H, I]; out scattered to [T*slots, H] fp32
cudaError_t launch_gemm(int kind, int bn, const void* A, int a_rows_alloc, int K, const void* B,
                        int b_rows_total, const GemmArgs& args, cudaStream_t stream);

}  // namespace gbmoe
