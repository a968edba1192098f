// NVFP4 activation and weight-layout kernels of the FusedMoE forward:
//
//   quant_fp4_kernel          fp4_quantize(x, g, 16) of bf16 rows into packed e2m1 codes and
//                             e4m3 block scales (the FlashInferFP4MoE input format)
//   quant_gather_fp4_kernel   the same quant, once per token, written as f16 values q * sf
//                             to each of the token's k rows in expert order, and (for the
//                             shared expert) in token order with its own scale
//   silu_quant_fp4_kernel     the first GEMM's split-K sum, act = silu(gate) * up, and the
//                             act's block quant (its own per-tensor scale) as f16 q * sf
//   prepare_fp4_kernel        the weight layout of the GEMMs: per tile of 128 rows and K
//                             stage of 64 values one 4608-byte chunk (a permutation only)
#include "fp4.cuh"
#include "kernels.h"

namespace gbmoe {
namespace {

// 16 bf16 values (32 bytes, 16-byte aligned) as fp32.
__device__ __forceinline__ void load_bf16x16(const __nv_bfloat16* p, float (&x)[16]) {
  const uint4 a = __ldg(reinterpret_cast<const uint4*>(p));
  const uint4 b = __ldg(reinterpret_cast<const uint4*>(p) + 1);
  const uint32_t u[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float2 f = unpack_bf16x2(u[i]);
    x[2 * i] = f.x;
    x[2 * i + 1] = f.y;
  }
}

__device__ __forceinline__ void store32(void* p, const uint32_t (&v)[8]) {
  uint4* d = reinterpret_cast<uint4*>(p);
  d[0] = make_uint4(v[0], v[1], v[2], v[3]);
  d[1] = make_uint4(v[4], v[5], v[6], v[7]);
}

// One thread per (row, block of 16).
__global__ void __launch_bounds__(256) quant_fp4_kernel(const __nv_bfloat16* __restrict__ x,
                                                        int rows, int H, float g,
                                                        uint8_t* __restrict__ q,
                                                        uint8_t* __restrict__ sf) {
  pdl_trigger();  // the next kernel may start its launch now
  pdl_wait();     // inputs written by the previous kernel are visible
  const int nb = H / kFp4Block;
  const long long items = (long long)rows * nb;
  for (long long it = (long long)blockIdx.x * blockDim.x + threadIdx.x; it < items;
       it += (long long)gridDim.x * blockDim.x) {
    const int r = (int)(it / nb), b = (int)(it % nb);
    float v[16];
    load_bf16x16(x + (size_t)r * H + (size_t)b * kFp4Block, v);
    uint32_t codes[2], vals[8];
    uint8_t s;
    fp4_quant_block(v, g, codes, s, vals);
    *reinterpret_cast<uint2*>(q + (size_t)r * (H / 2) + (size_t)b * 8) = make_uint2(codes[0], codes[1]);
    sf[(size_t)r * nb + b] = s;
  }
}

__global__ void __launch_bounds__(256)
    quant_gather_fp4_kernel(const __nv_bfloat16* __restrict__ x, int H,
                            const int* __restrict__ inv, int k, int T, int max_rows, float g,
                            __half* __restrict__ xp, __half* __restrict__ x_tok, float g_tok) {
  pdl_trigger();  // the next kernel may start its launch now
  pdl_wait();     // inputs written by the previous kernel are visible
  const int nb = H / kFp4Block;
  const long long items = (long long)T * nb;
  for (long long it = (long long)blockIdx.x * blockDim.x + threadIdx.x; it < items;
       it += (long long)gridDim.x * blockDim.x) {
    const int t = (int)(it / nb), b = (int)(it % nb);
    const size_t col = (size_t)b * kFp4Block;
    float v[16];
    load_bf16x16(x + (size_t)t * H + col, v);
    uint32_t codes[2], vals[8];
    uint8_t s;
    fp4_quant_block(v, g, codes, s, vals);
    for (int j = 0; j < k; ++j) {
      const int p = inv[t * k + j];
      if (p < 0 || p >= max_rows) continue;
      store32(xp + (size_t)p * H + col, vals);
    }
    if (x_tok) {
      if (g_tok != g) fp4_quant_block(v, g_tok, codes, s, vals);
      store32(x_tok + (size_t)t * H + col, vals);
    }
  }
}

// One CTA (128 threads) per row; thread i takes the 16-column blocks i, i + 128, ...
__global__ void __launch_bounds__(128) silu_quant_fp4_kernel(const __grid_constant__ GemmLaunch L,
                                                             const int* npp, int max_routed_rows,
                                                             float g_act, float g_act_shared) {
  pdl_trigger();  // the next kernel may start its launch now
  pdl_wait();     // inputs written by the previous kernel are visible
  const GemmProblem& R = L.p[0];
  int routed_rows = npp ? *npp : R.m_rows_host;
  if (routed_rows > max_routed_rows) routed_rows = max_routed_rows;
  const int shared_rows = L.num_problems > 1 ? L.p[1].store_rows : 0;
  const int routed_items = R.num_flat;
  for (int r = blockIdx.x; r < routed_items + shared_rows; r += gridDim.x) {
    const GemmProblem* P;
    int src, dst_row, pi;
    if (r < routed_items) {
      P = &L.p[0];
      pi = 0;
      src = r;
      dst_row = P->flat_row[r];
      if (dst_row < 0 || dst_row >= routed_rows) continue;
    } else {
      P = &L.p[1];
      pi = 1;
      src = dst_row = r - routed_items;
    }
    const float g = pi ? g_act_shared : g_act;
    const int N = P->ldo;
    const int nsp = splits_of(L, pi);
    const float* base = P->part + (size_t)src * 2 * N;
    __half* out = static_cast<__half*>(P->out) + (size_t)dst_row * N;
    for (int j = threadIdx.x * kFp4Block; j < N; j += blockDim.x * kFp4Block) {
      float gs[16], us[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) gs[i] = us[i] = 0.f;
      for (int s = 0; s < nsp; ++s) {
        const float4* q = reinterpret_cast<const float4*>(base + (size_t)s * P->part_split_stride + j);
        const float4* qu = reinterpret_cast<const float4*>(base + (size_t)s * P->part_split_stride + N + j);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float4 a = __ldg(q + i), b = __ldg(qu + i);
          gs[4 * i] += a.x; gs[4 * i + 1] += a.y; gs[4 * i + 2] += a.z; gs[4 * i + 3] += a.w;
          us[4 * i] += b.x; us[4 * i + 1] += b.y; us[4 * i + 2] += b.z; us[4 * i + 3] += b.w;
        }
      }
      float act[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) act[i] = gs[i] / (1.f + expf(-gs[i])) * us[i];
      uint32_t codes[2], vals[8];
      uint8_t sfc;
      fp4_quant_block(act, g, codes, sfc, vals);
      store32(out + j, vals);
    }
  }
}

// out[(tile * (K / 64) + kb) * 4608 + h * 2048 + r * 16 + j] = packed[tile * 128 + r][kb * 32 +
// h * 16 + j]; out[... + 4096 + r * 4 + j] = scales[tile * 128 + r][kb * 4 + j].
__global__ void __launch_bounds__(256) prepare_fp4_kernel(const uint8_t* __restrict__ packed,
                                                          const uint8_t* __restrict__ scales,
                                                          int rows, int K,
                                                          uint8_t* __restrict__ out) {
  pdl_trigger();
  pdl_wait();
  const int kbs = K / 64;
  constexpr int kUnits = kFp4ChunkBytes / 16;  // 16-byte pieces of a chunk
  const long long items = (long long)(rows / 128) * kbs * kUnits;
  for (long long it = (long long)blockIdx.x * blockDim.x + threadIdx.x; it < items;
       it += (long long)gridDim.x * blockDim.x) {
    const long long c = it / kUnits;
    const int w = (int)(it % kUnits);
    const long long tile = c / kbs;
    const int kb = (int)(c % kbs);
    uint4 v;
    if (w < 256) {
      const int h = w >> 7, r = w & 127;
      v = __ldg(reinterpret_cast<const uint4*>(packed + (size_t)(tile * 128 + r) * (K / 2) +
                                               (size_t)kb * 32 + h * 16));
    } else {
      const int r0 = 4 * (w - 256);
      uint32_t s[4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
        s[i] = __ldg(reinterpret_cast<const uint32_t*>(
            scales + (size_t)(tile * 128 + r0 + i) * (K / 16) + (size_t)kb * 4));
      v = make_uint4(s[0], s[1], s[2], s[3]);
    }
    reinterpret_cast<uint4*>(out)[it] = v;
  }
}

int grid_for(long long items, int threads) {
  long long g = (items + threads - 1) / threads;
  const long long cap = (long long)num_sms() * 8;
  if (g > cap) g = cap;
  return g < 1 ? 1 : (int)g;
}

}  // namespace

cudaError_t launch_quant_fp4(const void* x, int rows, int H, float g, uint8_t* q, uint8_t* sf,
                             cudaStream_t stream) {
  return launch_kernel(quant_fp4_kernel, dim3(grid_for((long long)rows * (H / kFp4Block), 256)),
                       dim3(256), 0, stream, static_cast<const __nv_bfloat16*>(x), rows, H, g, q,
                       sf);
}

cudaError_t launch_quant_gather_fp4(const void* x, int H, const int* inv, int n, int k, int T,
                                    int max_rows, float g, void* x_perm, void* x_tok,
                                    float g_tok, cudaStream_t stream) {
  (void)n;
  return launch_kernel(quant_gather_fp4_kernel,
                       dim3(grid_for((long long)T * (H / kFp4Block), 256)), dim3(256), 0, stream,
                       static_cast<const __nv_bfloat16*>(x), H, inv, k, T, max_rows, g,
                       static_cast<__half*>(x_perm), static_cast<__half*>(x_tok), g_tok);
}

cudaError_t launch_silu_quant_fp4(const GemmLaunch& L, const int* npp, int max_routed_rows,
                                  float g_act, float g_act_shared, cudaStream_t stream) {
  const int rows = L.p[0].num_flat + (L.num_problems > 1 ? L.p[1].store_rows : 0);
  int grid = rows < num_sms() * 16 ? rows : num_sms() * 16;
  if (grid < 1) grid = 1;
  return launch_kernel(silu_quant_fp4_kernel, dim3(grid), dim3(128), 0, stream, L, npp,
                       max_routed_rows, g_act, g_act_shared);
}

cudaError_t launch_prepare_fp4(const uint8_t* packed, const uint8_t* scales, int rows, int K,
                               uint8_t* out, cudaStream_t stream) {
  const long long items = (long long)(rows / 128) * (K / 64) * (kFp4ChunkBytes / 16);
  return launch_kernel(prepare_fp4_kernel, dim3(grid_for(items, 256)), dim3(256), 0, stream,
                       packed, scales, rows, K, out);
}

}  // namespace gbmoe
