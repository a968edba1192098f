// NVFP4 (w4a4, 16-value blocks with e4m3 scales and a per-tensor fp32 scale) grouped GEMMs
// of the FusedMoE expert MLP, the FlashInferFP4MoE layer of the sglang
// `fused_moe_triton/layer.py` page (`trtllm_fp4_block_scale_moe` with `gemm1_weights` /
// `gemm2_weights` and their block scales):
//
//   w13: z[f][n] = alpha_e * sum_k xq[row][k] w13q[e][n][k]   fp32 partials, n in [0, 2I)
//   w2 : o = alpha_e * sum_k aq[row][k] w2q[e][n][k], times the routing weight, to the
//        token's fp32 slot
//
// with xq / aq the f16 values q * sf of the quantized rows (exact) and w q * sf of the
// weights (exact in f16), alpha_e = weight_scale_2[e] / g (g the rows' per-tensor scale).
//
// The weights arrive prepared (moe_nvfp4_prepare_weight): per tile of 128 rows and K stage
// of 64 values one contiguous 4608-byte chunk, the packed codes of the stage's two K halves
// (16 bytes per row each) then the row's four scale bytes. One bulk copy per stage streams
// the chunk into a 16-deep ring; converter warps expand it to f16 (hardware e2m1x2 and
// e4m3x2 conversions and one packed multiply per pair) in the 128-byte-swizzled K-major
// layout the MMA reads, so HBM carries 0.5625 bytes per weight and the tensor cores see
// ordinary kind::f16 operands. The weights are on the MMA's M side (128 rows per unit), the
// row block's tokens on N (its real rows rounded up to 16, at most 128):
//
//   warp 0       bulk copies of prepared weight chunks into the raw ring (16 x 4.5 KB)
//   warp 1       TMEM (two 128-column accumulators) and the MMAs (M 128, N n, K 16)
//   warp 2       TMA token tiles (boxes of 16 / 32 / 64 / 128 rows) into the stage ring
//   warps 4..11  converters: warp c expands rows 32 (c & 3) .. +31, K half c >> 2
//   warps 12..15 epilogue: TMEM lane quarter warp & 3, one weight row per thread
// Every wait is bounded (kWaitTimeoutNs).
#include "fp4.cuh"
#include "tc.cuh"

namespace gbmoe {
namespace {

constexpr int kF4M = 128;                         // weight rows per unit (MMA M)
constexpr int kF4BK = 64;                         // K values per stage
constexpr uint32_t kF4RawBytes = kFp4ChunkBytes;  // one prepared chunk
constexpr int kF4RawStages = 16;
constexpr int kF4Stages = 4;
constexpr uint32_t kF4WBytes = kF4M * kF4BK * 2;          // f16 weights of a stage: 16 KB
constexpr uint32_t kF4XBytes = kFp4BS * kF4BK * 2;        // up to 128 token rows: 16 KB
constexpr uint32_t kF4StageBytes = kF4WBytes + kF4XBytes;
constexpr int kF4CvtWarps = 8;
constexpr int kF4EpiWarps = 4;
constexpr int kF4Threads = 32 * (4 + kF4CvtWarps + kF4EpiWarps);
constexpr uint32_t kF4TmemCols = 256;             // two 128-column accumulators
constexpr int kF4Boxes = 4;                       // token boxes of 16, 32, 64, 128 rows
constexpr uint32_t kF4BarBytes = 512;
constexpr size_t kF4Smem = 1024 + (size_t)kF4Stages * kF4StageBytes +
                           (size_t)kF4RawStages * kF4RawBytes + kF4BarBytes;
static_assert(kF4Smem <= 232448, "shared memory per CTA exceeded");
static_assert(kF4RawBytes % 16 == 0, "bulk copies move multiples of 16 bytes");

struct F4Maps {
  CUtensorMap x[2][kF4Boxes];  // per problem: f16 token rows, box 64 values x (16 << i) rows
};

// Instruction descriptor of kind::f16 with f16 A and B (format code 0), fp32 D, K-major.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N) {
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Spin (bounded, ignoring the abort flag) until the phase of `bar` with parity `parity`
// has completed: the producers' last copies must land before the CTA exits.
__device__ __noinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  const unsigned long long t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity))
    if (globaltimer_ns() - t0 > 10000000ull) return;
}

struct F4Unit {
  int p, split, mb, nt, kb0, kb1, n, box;
};

// Unit u with its MMA width: the row block's real rows (the align's per-block counts,
// else the launch's bound for routed problems; the identity rows left for the shared one)
// rounded up to 16, and the smallest token box that holds them.
__device__ __forceinline__ F4Unit f4_unit(const GemmLaunch& L, const Schedule& S, int u) {
  const Unit w = S.unit(L, u);
  F4Unit r{w.p, w.split, w.mb, w.nt, w.kb0, w.kb1, 16, 0};
  const GemmProblem& P = L.p[w.p];
  int rows;
  if (P.sorted_ids)
    rows = P.block_rows ? P.block_rows[w.mb] : P.rows_bound;
  else
    rows = P.store_rows - w.mb * kFp4BS;
  rows = rows < 1 ? 1 : (rows > kFp4BS ? kFp4BS : rows);
  r.n = (rows + 15) & ~15;
  r.box = r.n <= 16 ? 0 : (r.n <= 32 ? 1 : (r.n <= 64 ? 2 : 3));
  return r;
}

__device__ __forceinline__ int f4_expert(const GemmProblem& P, int mb, int* status) {
  int e = P.expert_ids ? P.expert_ids[mb] : 0;
  if ((unsigned)e >= (unsigned)P.num_experts) {
    record_status(status, GBMOE_ERR_DEVICE_CHECK);
    e = 0;
  }
  return e;
}

template <int KIND>
__global__ void __launch_bounds__(kF4Threads, 1)
    gemm_fp4_kernel(const __grid_constant__ F4Maps maps, const __grid_constant__ GemmLaunch args) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw0 = smem_addr(smem_raw);
  const uint32_t base = (raw0 + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw0);
  // [stages: f16 weights 16 KB | token rows 16 KB] [raw ring] [barriers]
  const uint32_t raw_base = base + kF4Stages * kF4StageBytes;
  uint8_t* raw_ptr = smem + kF4Stages * kF4StageBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(raw_ptr + kF4RawStages * kF4RawBytes);
  // bars: raw_full[16] raw_empty[16] tok_full[4] cvt_full[4] stage_empty[4] tfull[2] tempty[2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 48);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const uint32_t bar0 = smem_addr(bars);
  auto raw_full = [&](int s) { return bar0 + 8u * s; };
  auto raw_empty = [&](int s) { return bar0 + 8u * (16 + s); };
  auto tok_full = [&](int s) { return bar0 + 8u * (32 + s); };
  auto cvt_full = [&](int s) { return bar0 + 8u * (36 + s); };
  auto stage_empty = [&](int s) { return bar0 + 8u * (40 + s); };
  auto tfull = [&](int b) { return bar0 + 8u * (44 + b); };
  auto tempty = [&](int b) { return bar0 + 8u * (46 + b); };
  auto w_stage = [&](int s) { return base + s * kF4StageBytes; };
  auto x_stage = [&](int s) { return base + s * kF4StageBytes + kF4WBytes; };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kF4RawStages; ++s) {
      mbar_init(raw_full(s), 1);
      mbar_init(raw_empty(s), kF4CvtWarps);
    }
    for (int s = 0; s < kF4Stages; ++s) {
      mbar_init(tok_full(s), 1);
      mbar_init(cvt_full(s), kF4CvtWarps);
      mbar_init(stage_empty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull(b), 1);
      mbar_init(tempty(b), kF4EpiWarps);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 2 && lane == 0) {
    for (int p = 0; p < args.num_problems; ++p)
      for (int i = 0; i < kF4Boxes; ++i) tma_prefetch(&maps.x[p][i]);
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(tmem_slot), kF4TmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_wait();  // the token rows and the routing are earlier kernels' outputs
  if (threadIdx.x == 0) pdl_trigger();

  Schedule sched;
  sched.init(args, kFp4BS);

  if (warp == 0) {
    // ------------------------------------------------------------ prepared weight chunks
    if (lane == 0) {
      const uint64_t policy = l2_evict_first_policy();
      uint32_t it = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < sched.units; u += gridDim.x) {
        const Unit w = sched.unit(args, u);
        const GemmProblem& P = args.p[w.p];
        const int e = f4_expert(P, w.mb, args.status);
        const size_t tile = ((size_t)e * P.b_rows_per_expert + (size_t)w.nt * kF4M) / kF4M;
        const uint8_t* src = static_cast<const uint8_t*>(P.B) +
                             (tile * P.k_blocks + w.kb0) * (size_t)kF4RawBytes;
        for (int kb = w.kb0; kb < w.kb1; ++kb, ++it, src += kF4RawBytes) {
          const int s = it % kF4RawStages;
          const uint32_t ph = (it / kF4RawStages) & 1u;
          if (!wait_fast(raw_empty(s), ph ^ 1u, abort_flag, args.status)) {
            ok = false;
            break;
          }
          mbar_expect_tx(raw_full(s), kF4RawBytes);
          bulk_load(raw_base + s * kF4RawBytes, src, kF4RawBytes, raw_full(s), policy);
        }
      }
      // the last copies of each slot land before the CTA can exit
      for (uint32_t j = it > (uint32_t)kF4RawStages ? it - kF4RawStages : 0; j < it; ++j)
        drain_wait(raw_full(j % kF4RawStages), (j / kF4RawStages) & 1u);
    }
    __syncwarp();
  } else if (warp == 2) {
    // ------------------------------------------------------------ token tiles
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < sched.units; u += gridDim.x) {
        const F4Unit w = f4_unit(args, sched, u);
        const CUtensorMap* map = &maps.x[w.p][w.box];
        const uint32_t bytes = (uint32_t)(16 << w.box) * kF4BK * 2;
        for (int kb = w.kb0; kb < w.kb1; ++kb, ++it) {
          const int s = it % kF4Stages;
          const uint32_t ph = (it / kF4Stages) & 1u;
          if (!wait_fast(stage_empty(s), ph ^ 1u, abort_flag, args.status)) {
            ok = false;
            break;
          }
          mbar_expect_tx(tok_full(s), bytes);
          tma_load_2d(x_stage(s), map, tok_full(s), kb * kF4BK, w.mb * kFp4BS);
        }
      }
      for (uint32_t j = it > (uint32_t)kF4Stages ? it - kF4Stages : 0; j < it; ++j)
        drain_wait(tok_full(j % kF4Stages), (j / kF4Stages) & 1u);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      uint32_t it = 0, uc = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < sched.units; u += gridDim.x, ++uc) {
        const F4Unit w = f4_unit(args, sched, u);
        const uint32_t idesc = idesc_f16(kF4M, w.n);
        const int buf = uc & 1;
        if (!wait_fast(tempty(buf), ((uc >> 1) & 1u) ^ 1u, abort_flag, args.status)) break;
        tc_fence_after();
        const uint32_t d = tmem_base + buf * 128;
        for (int kb = w.kb0; kb < w.kb1; ++kb, ++it) {
          const int s = it % kF4Stages;
          const uint32_t ph = (it / kF4Stages) & 1u;
          if (!wait_fast(tok_full(s), ph, abort_flag, args.status) ||
              !wait_fast(cvt_full(s), ph, abort_flag, args.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < kF4BK / 16; ++kk)
            mma_bf16(d, sdesc_sw128(w_stage(s) + kk * 32), sdesc_sw128(x_stage(s) + kk * 32),
                     idesc, (kb != w.kb0 || kk != 0) ? 1u : 0u);
          mma_commit(stage_empty(s));
        }
        if (ok) mma_commit(tfull(buf));
      }
    }
    __syncwarp();
  } else if (warp >= 4 && warp < 4 + kF4CvtWarps) {
    // ------------------------------------------------------------ fp4 -> f16 expansion
    const int c = warp - 4;
    const int h = c >> 2;                 // K half of the stage: values 32 h .. 32 h + 31
    const int r = 32 * (c & 3) + lane;    // weight row within the tile
    uint32_t it = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < sched.units; u += gridDim.x) {
      const Unit w = sched.unit(args, u);
      for (int kb = w.kb0; kb < w.kb1; ++kb, ++it) {
        const int rs = it % kF4RawStages;
        const int s = it % kF4Stages;
        if (!wait_fast(raw_full(rs), (it / kF4RawStages) & 1u, abort_flag, args.status)) {
          ok = false;
          break;
        }
        const uint8_t* chunk = raw_ptr + rs * kF4RawBytes;
        const uint4 q = *reinterpret_cast<const uint4*>(chunk + h * 2048 + r * 16);
        const uint32_t sc = *reinterpret_cast<const uint16_t*>(chunk + 4096 + r * 4 + 2 * h);
        __syncwarp();
        if (lane == 0) mbar_arrive(raw_empty(rs));
        // the scales of the half's two blocks as f16 pairs (exact)
        __half2_raw s01 = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)sc, __NV_E4M3);
        __half2 sp;
        memcpy(&sp, &s01, 4);
        const __half2 sc0 = __low2half2(sp), sc1 = __high2half2(sp);
        if (!wait_fast(stage_empty(s), ((it / kF4Stages) & 1u) ^ 1u, abort_flag, args.status)) {
          ok = false;
          break;
        }
        const uint32_t words[4] = {q.x, q.y, q.z, q.w};
        const uint32_t row = w_stage(s) + r * 128;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const __half2 scl = i < 2 ? sc0 : sc1;
          uint32_t o[4];
#pragma unroll
          for (int b = 0; b < 4; ++b) {
            const uint32_t hv = e2m1x2_to_f16x2((words[i] >> (8 * b)) & 0xFFu);
            __half2 v;
            memcpy(&v, &hv, 4);
            v = __hmul2(v, scl);
            memcpy(&o[b], &v, 4);
          }
          const uint32_t chunk16 = (uint32_t)((4 * h + i) ^ (r & 7));
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(row + chunk16 * 16),
                       "r"(o[0]), "r"(o[1]), "r"(o[2]), "r"(o[3])
                       : "memory");
        }
        fence_proxy_async_smem();  // the MMA (async proxy) reads what these stores wrote
        __syncwarp();
        if (lane == 0) mbar_arrive(cvt_full(s));
      }
    }
  } else if (warp >= 4 + kF4CvtWarps) {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3;
    const int r = 32 * quarter + lane;   // weight row within the tile
    uint32_t uc = 0;
    for (int u = blockIdx.x; u < sched.units; u += gridDim.x, ++uc) {
      const F4Unit w = f4_unit(args, sched, u);
      const GemmProblem& P = args.p[w.p];
      const int e = f4_expert(P, w.mb, args.status);
      const float alpha = __fdiv_rn(P.scale2 ? P.scale2[P.sorted_ids ? e : 0] : 1.f, P.gscale);
      const int buf = uc & 1;
      if (!wait_fast(tfull(buf), (uc >> 1) & 1u, abort_flag, args.status)) break;
      tc_fence_after();
      const int m0 = w.mb * kFp4BS;
      for (int c0 = 0; c0 < w.n; c0 += 32) {
        uint32_t v[32];
        tmem_ld32(tmem_base + ((uint32_t)(quarter * 32) << 16) + buf * 128 + c0, v);
        tmem_wait_ld(v);
        // this lane's token column c0 + lane: its flat index (routed) or token
        const int m = m0 + c0 + lane;
        int f = -1;
        if (c0 + lane < w.n) {
          if (P.sorted_ids) {
            const int x = P.sorted_ids[m];
            if (x >= 0 && x < P.num_flat) f = x;
          } else if (m < P.store_rows) {
            f = m;
          }
        }
        if (KIND == kGemmW13) {
          float* dst = P.part + (size_t)w.split * P.part_split_stride + (size_t)w.nt * kF4M + r;
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int fj = __shfl_sync(0xffffffffu, f, j);
            if (fj >= 0) dst[(size_t)fj * 2 * P.ldo] = alpha * __uint_as_float(v[j]);
          }
        } else {
          int dest = -1;
          float wt = alpha;
          if (f >= 0) {
            if (P.sorted_ids) {
              dest = (f / P.top_k) * P.slots + (f % P.top_k);
              if (P.row_weight) wt = alpha * P.row_weight[f];
            } else {
              dest = f * P.slots + P.slot_offset;
            }
          }
          float* outp = static_cast<float*>(P.out) + (size_t)w.split * P.out_split_stride +
                        (size_t)w.nt * kF4M + r;
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int dj = __shfl_sync(0xffffffffu, dest, j);
            const float wj = __shfl_sync(0xffffffffu, wt, j);
            if (dj >= 0) outp[(size_t)dj * P.ldo] = wj * __uint_as_float(v[j]);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty(buf));
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kF4TmemCols);
  }
}

template <int KIND>
cudaError_t launch_fp4_typed(const F4Maps& maps, const GemmLaunch& args, int grid,
                             cudaStream_t stream) {
  static int configured_device = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_device != dev) {
    cudaError_t e = cudaFuncSetAttribute(gemm_fp4_kernel<KIND>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kF4Smem);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  return launch_kernel(gemm_fp4_kernel<KIND>, dim3(grid), dim3(kF4Threads), kF4Smem, stream,
                       maps, args);
}

}  // namespace

cudaError_t launch_gemm_fp4(int kind, const GemmLaunch& L, cudaStream_t stream) {
  if (L.num_problems < 1 || L.num_problems > 2 || L.splits < 1) return cudaErrorInvalidValue;
  if (kind != kGemmW13 && kind != kGemmW2) return cudaErrorInvalidValue;
  F4Maps maps;
  long units = 0;
  for (int p = 0; p < 2; ++p) {
    const GemmProblem& P = L.p[L.num_problems > p ? p : 0];
    if (P.K % kF4BK || P.k_blocks != P.K / kF4BK || P.b_rows_per_expert % kF4M ||
        P.n_tiles * kF4M != P.b_rows_per_expert || !P.B || !(P.gscale > 0.f) ||
        (reinterpret_cast<uintptr_t>(P.B) & 15u) || (kind == kGemmW13 ? !P.part : !P.out))
      return cudaErrorInvalidValue;
    for (int i = 0; i < kF4Boxes; ++i)
      if (!make_map_2d(&maps.x[p][i], P.A, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, (uint64_t)P.K,
                       (uint64_t)P.a_rows, (uint32_t)(16 << i)))
        return cudaErrorInvalidValue;
    if (p < L.num_problems) {
      if (splits_of(L, p) < 1 || P.k_blocks < splits_of(L, p)) return cudaErrorInvalidValue;
      units += (long)P.max_m_blocks * P.n_tiles * splits_of(L, p);
    }
  }
  int grid = num_sms();
  if (units < grid) grid = (int)units;
  if (grid < 1) grid = 1;
  return kind == kGemmW13 ? launch_fp4_typed<kGemmW13>(maps, L, grid, stream)
                          : launch_fp4_typed<kGemmW2>(maps, L, grid, stream);
}

}  // namespace gbmoe
