// FP8 (e4m3 w8a8, 128 x 128 weight blocks) grouped GEMMs of the FusedMoE expert MLP on the
// 5th-generation tensor cores, the quantized DeepSeek MoE of the sglang
// `models/deepseek_v2.py` page (`DeepseekV2MoE._compute_moe_quant_once_enabled`: block-128
// fp8 weights with fp32 scales; per-token-group-128 activations):
//
//   w13: [gate | up] = sum_kb sa[row, kb] sb[n / 128, kb] (xq_rows . w13q[e])_kb,
//        act = silu(gate) * up, quantized per 128 columns into e4m3 + fp32 scale
//   w2 : o = sum_kb sa sb (actq_rows . w2q[e])_kb, times the routing weight, scattered to
//        the token's fp32 output slot
//
// One K block (128 e4m3 = 128 bytes) is both one 128-byte swizzle row of a pipeline stage
// and one scale block, so each K block's product is accumulated on its own in TMEM
// (4 x tcgen05.mma kind::f8f6f4, K = 32) and promoted into fp32 registers with its two
// scales by the epilogue, while the next K block's MMAs run into the other TMEM buffer.
//
// Kernel shape (one persistent CTA per SM, 320 threads):
//   warp 0      TMA producer (A box [AROWS x 128 B], B box [256 x 128 B]) into a 4-deep
//               (6-deep with 32-row A boxes) ring of swizzled stages;
//   warp 1      allocates 512 TMEM columns (two 256-column K-block buffers) and issues the
//               MMAs (M = 128, N = 256) of each K block into alternate buffers;
//   warps 2..9  epilogue: the two warps of each TMEM lane quarter split the 256 columns
//               (w13: 64 gate + the matching 64 up columns each; w2: 128 columns each) and
//               keep 128 fp32 running sums per row in registers. With 32-row A boxes only
//               the quarter holding rows 0..31 runs.
// Every wait is bounded (kWaitTimeoutNs), as in the bf16 kernels.
#include "fp8.cuh"
#include "tc.cuh"

namespace gbmoe {
namespace {

constexpr int kF8BK = kFp8Block;  // K elements (= bytes) per stage
constexpr int kF8EpiWarps = 8;
constexpr int kF8Threads = 64 + 32 * kF8EpiWarps;
constexpr uint32_t kF8TmemCols = 512;
constexpr uint32_t kF8BufStride = 256;
constexpr int kF8N = 256;  // MMA N (B rows per stage)

template <int KIND, int AROWS>
struct F8Shape {
  static constexpr int kBN = KIND == kGemmW13 ? 128 : 256;  // output columns per tile
  static constexpr uint32_t kBBytes = kF8N * kF8BK;
  static constexpr uint32_t kARegion = AROWS * kF8BK;
  static constexpr uint32_t kStageBytes = kARegion + kBBytes;
  static constexpr int kNumStages = AROWS == kGemmBM ? 4 : 6;
  static constexpr int kActiveQuarters = AROWS / 32;
  static constexpr int kActiveWarps = 2 * kActiveQuarters;
  // stages, 1024 B of alignment slack, barriers + TMEM slot + abort flag, amax exchange
  static constexpr size_t kSmem = (size_t)kNumStages * kStageBytes + 1024 + 256 + 2 * 2 * 128 * 4;
  static_assert(kSmem <= 232448, "shared memory per CTA exceeded");
};

template <int KIND, int AROWS>
__global__ void __launch_bounds__(kF8Threads, 1)
    gemm_fp8_kernel(const __grid_constant__ CUtensorMap tmA0,
                    const __grid_constant__ CUtensorMap tmB0,
                    const __grid_constant__ CUtensorMap tmA1,
                    const __grid_constant__ CUtensorMap tmB1, const GemmLaunch args) {
  using S = F8Shape<KIND, AROWS>;
  constexpr int kStages = S::kNumStages;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kStages * S::kStageBytes);
  // bars: full[kStages] empty[kStages] tfull[2] tempty[2] pair[4]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kStages + 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* red = reinterpret_cast<float*>(smem + kStages * S::kStageBytes + 256);  // [2][2][128]
  const uint32_t bar0 = smem_addr(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (kStages + s); };
  auto tfull_bar = [&](int b) { return bar0 + 8u * (2 * kStages + b); };
  auto tempty_bar = [&](int b) { return bar0 + 8u * (2 * kStages + 2 + b); };
  auto pair_bar = [&](int q) { return bar0 + 8u * (2 * kStages + 4 + q); };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull_bar(b), 1);
      mbar_init(tempty_bar(b), S::kActiveWarps);
    }
    for (int q = 0; q < 4; ++q) mbar_init(pair_bar(q), 2);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch(&tmA0);
    tma_prefetch(&tmB0);
    if (args.num_problems > 1) {
      tma_prefetch(&tmA1);
      tma_prefetch(&tmB1);
    }
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(tmem_slot), kF8TmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  Schedule sched;
  sched.init(args);

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < sched.units; u += gridDim.x) {
        const Unit w = sched.unit(args, u);
        const GemmProblem& P = args.p[w.p];
        const CUtensorMap* ta = w.p ? &tmA1 : &tmA0;
        const CUtensorMap* tb = w.p ? &tmB1 : &tmB0;
        int e = P.expert_ids ? P.expert_ids[w.mb] : 0;
        if ((unsigned)e >= (unsigned)P.num_experts) {
          record_status(args.status, GBMOE_ERR_DEVICE_CHECK);
          e = 0;
        }
        const int a_row = w.mb * kGemmBM;
        const int b_row = e * P.b_rows_per_expert + w.nt * S::kBN;
        for (int kb = w.kb0; kb < w.kb1; ++kb, ++it) {
          const int s = it % kStages;
          const uint32_t ph = (it / kStages) & 1u;
          if (!wait_bounded(empty_bar(s), ph ^ 1u, abort_flag, args.status)) {
            ok = false;
            break;
          }
          const uint32_t sa = base + s * S::kStageBytes;
          const uint32_t sb = sa + S::kARegion;
          mbar_expect_tx(full_bar(s), S::kStageBytes);
          tma_load_2d(sa, ta, full_bar(s), kb * kF8BK, a_row);
          tma_load_2d(sb, tb, full_bar(s), kb * kF8BK, b_row);
          if (KIND == kGemmW13)
            tma_load_2d(sb + 128 * kF8BK, tb, full_bar(s), kb * kF8BK, b_row + P.up_offset);
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_e4m3(kGemmBM, kF8N);
      uint32_t it = 0, kbc = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < sched.units; u += gridDim.x) {
        const Unit w = sched.unit(args, u);
        for (int kb = w.kb0; kb < w.kb1; ++kb, ++it, ++kbc) {
          const int buf = kbc & 1;
          const uint32_t use = kbc >> 1;
          if (!wait_bounded(tempty_bar(buf), (use & 1u) ^ 1u, abort_flag, args.status)) {
            ok = false;
            break;
          }
          const int s = it % kStages;
          const uint32_t ph = (it / kStages) & 1u;
          if (!wait_bounded(full_bar(s), ph, abort_flag, args.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = base + s * S::kStageBytes;
          const uint32_t sb = sa + S::kARegion;
          const uint32_t d = tmem_base + buf * kF8BufStride;
#pragma unroll
          for (int kk = 0; kk < kF8BK / 32; ++kk)
            mma_e4m3(d, sdesc_sw128(sa + kk * 32), sdesc_sw128(sb + kk * 32), idesc,
                     kk != 0 ? 1u : 0u);
          mma_commit(empty_bar(s));
          mma_commit(tfull_bar(buf));
        }
      }
    }
    __syncwarp();
  } else if ((warp & 3) < S::kActiveQuarters) {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3;             // TMEM lanes [32 quarter, 32 quarter + 32)
    const int half = (warp - 2) >> 2;         // which half of the 256 columns
    const int row = quarter * 32 + lane;
    uint32_t kbc = 0, npair = 0;  // K blocks and amax exchanges done by this warp
    bool ok = true;
    for (int u = blockIdx.x; ok && u < sched.units; u += gridDim.x) {
      const Unit w = sched.unit(args, u);
      const GemmProblem& P = args.p[w.p];
      const int m = w.mb * kGemmBM + row;
      int f = -1;
      if (P.sorted_ids) {
        const int v = P.sorted_ids[m];
        if (v >= 0 && v < P.num_flat) f = v;
      } else if (m < P.store_rows) {
        f = m;
      }
      int e = P.expert_ids ? P.expert_ids[w.mb] : 0;
      if ((unsigned)e >= (unsigned)P.num_experts) e = 0;
      const int KB = P.k_blocks;
      const float* bsc = P.b_scale + (size_t)e * (P.b_rows_per_expert / kFp8Block) * KB;
      // scale rows of this thread's columns: w13 gate block nt and up block (I/128 + nt);
      // w2 the 128-column block of this half
      const float* sb0 = bsc + (size_t)(KIND == kGemmW13 ? w.nt : 2 * w.nt + half) * KB;
      const float* sb1 = bsc + (size_t)(P.up_offset / kFp8Block + w.nt) * KB;
      const bool a_ok = m < P.a_scale_ld;
      float acc[128];
#pragma unroll
      for (int i = 0; i < 128; ++i) acc[i] = 0.f;
      for (int kb = w.kb0; kb < w.kb1; ++kb, ++kbc) {
        const float sa = a_ok ? __ldg(P.a_scale + (size_t)kb * P.a_scale_ld + m) : 0.f;
        const float c0 = sa * __ldg(sb0 + kb);
        const float c1 = KIND == kGemmW13 ? sa * __ldg(sb1 + kb) : c0;
        const int buf = kbc & 1;
        const uint32_t use = kbc >> 1;
        if (!wait_bounded(tfull_bar(buf), use & 1u, abort_flag, args.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t tb = tmem_base + ((uint32_t)(quarter * 32) << 16) + buf * kF8BufStride;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          // w13: chunks 0..3 = gate columns 64 half + [0, 64); chunks 4..7 = the up columns
          const uint32_t col = KIND == kGemmW13
                                   ? (c < 4 ? 64 * half + 16 * c : 128 + 64 * half + 16 * (c - 4))
                                   : 128 * half + 16 * c;
          const float sc = (KIND == kGemmW13 && c >= 4) ? c1 : c0;
          uint32_t v[16];
          tmem_ld16(tb + col, v);
          tmem_wait_ld16(v);
#pragma unroll
          for (int i = 0; i < 16; ++i)
            acc[16 * c + i] = fmaf(sc, __uint_as_float(v[i]), acc[16 * c + i]);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(tempty_bar(buf));
      }
      if (!ok) break;
      const bool split = splits_of(args, w.p) > 1;
      if (KIND == kGemmW13) {
        if (split) {
          // raw fp32 sums of this K range: gate at [0, ldo), up at [ldo, 2 ldo) of the row
          if (f >= 0) {
            float* dst = P.part + (size_t)w.split * P.part_split_stride + (size_t)f * 2 * P.ldo +
                         (size_t)w.nt * 128 + 64 * half;
#pragma unroll
            for (int i = 0; i < 64; i += 4) {
              *reinterpret_cast<float4*>(dst + i) = make_float4(acc[i], acc[i + 1], acc[i + 2], acc[i + 3]);
              *reinterpret_cast<float4*>(dst + P.ldo + i) =
                  make_float4(acc[64 + i], acc[65 + i], acc[66 + i], acc[67 + i]);
            }
          }
        } else {
          float amax = 0.f;
#pragma unroll
          for (int i = 0; i < 64; ++i) {
            acc[i] = acc[i] / (1.f + __expf(-acc[i])) * acc[64 + i];
            amax = fmaxf(amax, fabsf(acc[i]));
          }
          // the 128-column group spans both halves: swap the two halves' amax through shared
          // memory (slot by exchange parity) and a two-warp mbarrier per lane quarter
          float* slot = red + (npair & 1u) * 256;
          slot[half * 128 + row] = amax;
          __syncwarp();
          if (lane == 0) mbar_arrive(pair_bar(quarter));
          if (!wait_bounded(pair_bar(quarter), npair & 1u, abort_flag, args.status)) break;
          ++npair;
          amax = fmaxf(amax, slot[(1 - half) * 128 + row]);
          const float sc = fp8_group_scale(amax);
          const bool store = P.sorted_ids ? true : (m < P.store_rows);
          if (store) {
            uint4* dst = reinterpret_cast<uint4*>(static_cast<uint8_t*>(P.out) + (size_t)m * P.ldo +
                                                  (size_t)w.nt * 128 + 64 * half);
#pragma unroll
            for (int v = 0; v < 4; ++v)
              dst[v] = make_uint4(e4m3x4(acc[16 * v], acc[16 * v + 1], acc[16 * v + 2], acc[16 * v + 3], sc),
                                  e4m3x4(acc[16 * v + 4], acc[16 * v + 5], acc[16 * v + 6], acc[16 * v + 7], sc),
                                  e4m3x4(acc[16 * v + 8], acc[16 * v + 9], acc[16 * v + 10], acc[16 * v + 11], sc),
                                  e4m3x4(acc[16 * v + 12], acc[16 * v + 13], acc[16 * v + 14], acc[16 * v + 15], sc));
            if (half == 0) P.out_scale[(size_t)w.nt * P.out_scale_ld + m] = sc;
          }
        }
      } else {
        int dest = -1;
        float wt = 1.f;
        if (f >= 0) {
          if (P.sorted_ids) {
            dest = (f / P.top_k) * P.slots + (f % P.top_k);
            wt = P.row_weight ? P.row_weight[f] : 1.f;
          } else {
            dest = f * P.slots + P.slot_offset;
          }
        }
        if (dest >= 0) {
          float* dst = static_cast<float*>(P.out) + (size_t)w.split * P.out_split_stride +
                       (size_t)dest * P.ldo + (size_t)w.nt * 256 + 128 * half;
#pragma unroll
          for (int i = 0; i < 128; i += 4)
            *reinterpret_cast<float4*>(dst + i) =
                make_float4(wt * acc[i], wt * acc[i + 1], wt * acc[i + 2], wt * acc[i + 3]);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kF8TmemCols);
  }
}

template <int KIND, int AROWS>
cudaError_t launch_fp8_typed(const CUtensorMap* tm, const GemmLaunch& args, int grid,
                             cudaStream_t stream) {
  using S = F8Shape<KIND, AROWS>;
  static int configured_device = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_device != dev) {
    cudaError_t e = cudaFuncSetAttribute(gemm_fp8_kernel<KIND, AROWS>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)S::kSmem);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  gemm_fp8_kernel<KIND, AROWS>
      <<<grid, kF8Threads, S::kSmem, stream>>>(tm[0], tm[1], tm[2], tm[3], args);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemm_fp8(int kind, const GemmLaunch& L, cudaStream_t stream,
                            int max_rows_per_block) {
  const int arows = max_rows_per_block <= 32 ? 32 : kGemmBM;
  if (L.num_problems < 1 || L.num_problems > 2 || L.splits < 1) return cudaErrorInvalidValue;
  if (kind != kGemmW13 && kind != kGemmW2) return cudaErrorInvalidValue;
  CUtensorMap tm[4];
  long units = 0;
  const uint32_t b_box = kind == kGemmW13 ? 128u : 256u;
  for (int p = 0; p < 2; ++p) {
    const GemmProblem& P = L.p[L.num_problems > p ? p : 0];
    if (P.K % kF8BK || P.k_blocks != P.K / kF8BK || !P.a_scale || !P.b_scale ||
        P.b_rows_per_expert % kFp8Block || (kind == kGemmW13 && !P.part && !P.out_scale))
      return cudaErrorInvalidValue;
    if (!make_map_2d(&tm[2 * p], P.A, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, (uint64_t)P.K,
                     (uint64_t)P.a_rows, (uint32_t)arows) ||
        !make_map_2d(&tm[2 * p + 1], P.B, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, (uint64_t)P.K,
                     (uint64_t)P.b_rows, b_box))
      return cudaErrorInvalidValue;
    if (p < L.num_problems) {
      if (splits_of(L, p) < 1 || P.k_blocks < splits_of(L, p)) return cudaErrorInvalidValue;
      units += (long)P.max_m_blocks * P.n_tiles * splits_of(L, p);
    }
  }
  int grid = num_sms();
  if (units < grid) grid = (int)units;
  if (grid < 1) grid = 1;
  if (kind == kGemmW13)
    return arows == 32 ? launch_fp8_typed<kGemmW13, 32>(tm, L, grid, stream)
                       : launch_fp8_typed<kGemmW13, kGemmBM>(tm, L, grid, stream);
  return arows == 32 ? launch_fp8_typed<kGemmW2, 32>(tm, L, grid, stream)
                     : launch_fp8_typed<kGemmW2, kGemmBM>(tm, L, grid, stream);
}

}  // namespace gbmoe
