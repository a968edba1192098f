// FP8 (e4m3 w8a8, block 128) activation kernels of the FusedMoE forward:
//
//   quant_fp8_kernel         per-token-group-128 quant of bf16 rows (one warp per row group)
//   quant_gather_fp8_kernel  the same quant, once per token, written to each of the token's
//                            k rows in expert order and (for the shared expert) in token
//                            order: the input is quantized once and feeds both, as
//                            `DeepseekV2MoE._maybe_quant_moe_input_once` does on the sglang
//                            `models/deepseek_v2.py` page
//   silu_reduce_fp8_kernel   split-K reduce of the first GEMM: act = silu(sum gate) * sum up,
//                            then the post-SiLU per-group quant of `DeepseekV2MLP.forward`
//
// Scales are group-major ([group][row]) so that a GEMM epilogue warp reads the scales of
// its 32 rows in one transaction.
#include "fp8.cuh"
#include "kernels.h"

namespace gbmoe {
namespace {

// A warp quantizes one 128-column group of a bf16 row: lane l holds columns 4l .. 4l+3.
struct GroupQ {
  uint32_t q;  // the lane's four e4m3 bytes
  float s;     // the group's scale
};

__device__ __forceinline__ GroupQ quant_group_warp(const __nv_bfloat16* src, int lane) {
  const uint2 v = __ldg(reinterpret_cast<const uint2*>(src) + lane);
  const float2 a = unpack_bf16x2(v.x), b = unpack_bf16x2(v.y);
  const float amax = warp_max(fmaxf(fmaxf(fabsf(a.x), fabsf(a.y)), fmaxf(fabsf(b.x), fabsf(b.y))));
  GroupQ r;
  r.s = fp8_group_scale(amax);
  r.q = e4m3x4(a.x, a.y, b.x, b.y, r.s);
  return r;
}

__global__ void __launch_bounds__(256) quant_fp8_kernel(const __nv_bfloat16* __restrict__ x,
                                                        int rows, int H, uint8_t* __restrict__ q,
                                                        float* __restrict__ s_out, int s_ld) {
  pdl_trigger();  // the next kernel may start its launch now
  pdl_wait();     // inputs written by the previous kernel are visible
  const int lane = threadIdx.x & 31;
  const int groups = H / kFp8Block;
  const long long items = (long long)rows * groups;
  const long long warps = (long long)gridDim.x * (blockDim.x >> 5);
  for (long long it = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); it < items;
       it += warps) {
    const int r = (int)(it / groups), g = (int)(it % groups);
    const size_t off = (size_t)r * H + (size_t)g * kFp8Block;
    const GroupQ v = quant_group_warp(x + off, lane);
    reinterpret_cast<uint32_t*>(q + off)[lane] = v.q;
    if (lane == 0) s_out[(size_t)g * s_ld + r] = v.s;
  }
}

__global__ void __launch_bounds__(256)
    quant_gather_fp8_kernel(const __nv_bfloat16* __restrict__ x, int H,
                            const int* __restrict__ inv, int k, int T, int max_rows,
                            uint8_t* __restrict__ xp, float* __restrict__ xs_perm, int perm_ld,
                            uint8_t* __restrict__ xq_tok, float* __restrict__ xs_tok) {
  pdl_trigger();  // the next kernel may start its launch now
  pdl_wait();     // inputs written by the previous kernel are visible
  const int lane = threadIdx.x & 31;
  const int groups = H / kFp8Block;
  const long long items = (long long)T * groups;
  const long long warps = (long long)gridDim.x * (blockDim.x >> 5);
  for (long long it = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); it < items;
       it += warps) {
    const int t = (int)(it / groups), g = (int)(it % groups);
    const size_t col = (size_t)g * kFp8Block;
    const GroupQ v = quant_group_warp(x + (size_t)t * H + col, lane);
    for (int j = 0; j < k; ++j) {
      const int p = inv[t * k + j];
      if (p < 0 || p >= max_rows) continue;
      reinterpret_cast<uint32_t*>(xp + (size_t)p * H + col)[lane] = v.q;
      if (lane == 0) xs_perm[(size_t)g * perm_ld + p] = v.s;
    }
    if (xq_tok) {
      reinterpret_cast<uint32_t*>(xq_tok + (size_t)t * H + col)[lane] = v.q;
      if (lane == 0) xs_tok[(size_t)g * T + t] = v.s;
    }
  }
}

// One CTA (128 threads) per output row; thread i owns 8 consecutive columns of each
// 1024-column step, so the 16 threads of a half-warp hold one 128-column group and find
// its amax with four xor-shuffles. Every lane runs every step (shuffles stay converged).
__global__ void __launch_bounds__(128) silu_reduce_fp8_kernel(const __grid_constant__ GemmLaunch L,
                                                              const int* npp,
                                                              int max_routed_rows) {
  // Triggering at entry is safe for the decode w2 GEMM that follows (it reads the routing's
  // expert blocks before its wait): this kernel launched only after the w13 GEMM in front of
  // it passed its wait, i.e. after the routing finished.
  pdl_trigger();  // the next kernel may start its launch now
  pdl_wait();     // inputs written by the previous kernel are visible
  const GemmProblem& R = L.p[0];
  int routed_rows = npp ? *npp : R.m_rows_host;
  if (routed_rows > max_routed_rows) routed_rows = max_routed_rows;
  const int shared_rows = L.num_problems > 1 ? L.p[1].store_rows : 0;
  // routed work items: the flat indices (through their sorted rows) or every sorted row
  const int routed_items = R.flat_row ? R.num_flat : max_routed_rows;
  for (int r = blockIdx.x; r < routed_items + shared_rows; r += gridDim.x) {
    const GemmProblem* P;
    int src, dst_row, pi;
    if (r < routed_items) {
      P = &L.p[0];
      pi = 0;
      if (P->flat_row) {
        src = r;
        dst_row = P->flat_row[r];
        if (dst_row < 0 || dst_row >= routed_rows) continue;
      } else {
        if (r >= routed_rows) continue;
        const int f = P->sorted_ids ? P->sorted_ids[r] : r;
        if (f < 0 || f >= P->num_flat) continue;  // padding rows are never read back
        src = f;
        dst_row = r;
      }
    } else {
      P = &L.p[1];
      pi = 1;
      src = dst_row = r - routed_items;
    }
    const int N = P->ldo;
    const int nsp = splits_of(L, pi);
    const float* base = P->part + (size_t)src * 2 * N;
    uint8_t* out = static_cast<uint8_t*>(P->out) + (size_t)dst_row * N;
    for (int j0 = 0; j0 < N; j0 += blockDim.x * 8) {
      const int j = j0 + threadIdx.x * 8;
      const bool valid = j < N;
      float g[8], u[8], a[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) g[i] = u[i] = 0.f;
      for (int s = 0; valid && s < nsp; ++s) {
        const float* q = base + (size_t)s * P->part_split_stride + j;
        const float4 g0 = __ldg(reinterpret_cast<const float4*>(q));
        const float4 g1 = __ldg(reinterpret_cast<const float4*>(q + 4));
        const float4 u0 = __ldg(reinterpret_cast<const float4*>(q + N));
        const float4 u1 = __ldg(reinterpret_cast<const float4*>(q + N + 4));
        g[0] += g0.x; g[1] += g0.y; g[2] += g0.z; g[3] += g0.w;
        g[4] += g1.x; g[5] += g1.y; g[6] += g1.z; g[7] += g1.w;
        u[0] += u0.x; u[1] += u0.y; u[2] += u0.z; u[3] += u0.w;
        u[4] += u1.x; u[5] += u1.y; u[6] += u1.z; u[7] += u1.w;
      }
      float amax = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        a[i] = g[i] / (1.f + __expf(-g[i])) * u[i];
        amax = fmaxf(amax, fabsf(a[i]));
      }
#pragma unroll
      for (int o = 1; o < 16; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
      if (valid) {
        const float sc = fp8_group_scale(amax);
        uint2 w;
        w.x = e4m3x4(a[0], a[1], a[2], a[3], sc);
        w.y = e4m3x4(a[4], a[5], a[6], a[7], sc);
        *reinterpret_cast<uint2*>(out + j) = w;
        if ((threadIdx.x & 15) == 0)
          P->out_scale[(size_t)(j / kFp8Block) * P->out_scale_ld + dst_row] = sc;
      }
    }
  }
}

int grid_for_warps(long long items) {
  long long blocks = (items + 7) / 8;
  const long long cap = (long long)num_sms() * 8;
  if (blocks > cap) blocks = cap;
  return blocks < 1 ? 1 : (int)blocks;
}

}  // namespace

cudaError_t launch_quant_fp8(const void* x, int rows, int H, uint8_t* q, float* s_out, int s_ld,
                             cudaStream_t stream) {
  if (rows <= 0) return cudaSuccess;
  if (H % kFp8Block) return cudaErrorInvalidValue;
  launch_kernel(quant_fp8_kernel, dim3(grid_for_warps((long long)rows * (H / kFp8Block))),
                dim3(256), 0, stream, static_cast<const __nv_bfloat16*>(x), rows, H, q, s_out,
                s_ld);
  return cudaGetLastError();
}

cudaError_t launch_quant_gather_fp8(const void* x, int H, const int* inv, int n, int k, int T,
                                    uint8_t* x_perm_q, float* xs_perm, int perm_ld,
                                    uint8_t* xq_tok, float* xs_tok, cudaStream_t stream) {
  if (T <= 0) return cudaSuccess;
  if (H % kFp8Block || n != T * k) return cudaErrorInvalidValue;
  launch_kernel(quant_gather_fp8_kernel, dim3(grid_for_warps((long long)T * (H / kFp8Block))),
                dim3(256), 0, stream, static_cast<const __nv_bfloat16*>(x), H, inv, k, T, perm_ld,
                x_perm_q, xs_perm, perm_ld, xq_tok, xs_tok);
  return cudaGetLastError();
}

cudaError_t launch_silu_reduce_fp8(const GemmLaunch& L, const int* npp, int max_routed_rows,
                                   cudaStream_t stream) {
  const int rows = (L.p[0].flat_row ? L.p[0].num_flat : max_routed_rows) +
                   (L.num_problems > 1 ? L.p[1].store_rows : 0);
  int grid = num_sms() * 4;
  if (rows < grid) grid = rows;
  if (grid < 1) return cudaSuccess;
  launch_kernel(silu_reduce_fp8_kernel, dim3(grid), dim3(128), 0, stream, L, npp, max_routed_rows);
  return cudaGetLastError();
}

}  // namespace gbmoe
