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
// Kernel shape (one persistent CTA per SM, 576 threads):
//   warp 0       TMA producer (A box [128 x 128 B], B box [256 x 128 B]) into a 4-deep
//                ring of swizzled stages;
//   warp 1       allocates 512 TMEM columns (two 256-column K-block buffers) and issues the
//                MMAs (M = 128, N = 256) of each K block into alternate buffers;
//   warps 2..17  epilogue: the four warps of each TMEM lane quarter split the 256 columns
//                (w13: 32 gate + the matching 32 up columns each; w2: 64 columns each) and
//                keep 64 fp32 running sums per row in registers; four warps per SM
//                sub-partition hide the TMEM load latency of the per-K-block promotion.
// Row blocks with at most 32 real rows (decode) run gemm_fp8_swap_kernel below instead.
// Every wait is bounded (kWaitTimeoutNs), as in the bf16 kernels.
#include "fp8.cuh"
#include "tc.cuh"

namespace gbmoe {
namespace {

constexpr int kF8BK = kFp8Block;  // K elements (= bytes) per stage
constexpr int kF8Quarters = 4;
constexpr int kF8WarpsPerQuarter = 4;  // epilogue warps sharing a TMEM lane quarter
constexpr int kF8EpiWarps = kF8Quarters * kF8WarpsPerQuarter;
constexpr int kF8Threads = 64 + 32 * kF8EpiWarps;
constexpr uint32_t kF8TmemCols = 512;
constexpr uint32_t kF8BufStride = 256;
constexpr int kF8N = 256;      // MMA N (B rows per stage)
constexpr int kF8Cols = kF8N / kF8WarpsPerQuarter;  // accumulator columns per epilogue thread
constexpr int kF8Stages = 4;
constexpr uint32_t kF8StageBytes = kGemmBM * kF8BK + kF8N * kF8BK;  // 48 KB
// stages, 1024 B of alignment slack, barriers + TMEM slot + abort flag, amax exchange
constexpr size_t kF8Smem = (size_t)kF8Stages * kF8StageBytes + 1024 + 256 +
                           2 * kF8WarpsPerQuarter * 128 * 4;
static_assert(kF8Smem <= 232448, "shared memory per CTA exceeded");

// a0 += s * v0, a1 += s * v1 in one packed fp32 instruction (two IEEE fmas).
__device__ __forceinline__ void fma2(float& a0, float& a1, float s, float v0, float v1) {
  asm("{\n\t.reg .b64 a, v, s;\n\t"
      "mov.b64 a, {%0, %1};\n\t"
      "mov.b64 v, {%2, %3};\n\t"
      "mov.b64 s, {%4, %4};\n\t"
      "fma.rn.f32x2 a, s, v, a;\n\t"
      "mov.b64 {%0, %1}, a;\n\t}"
      : "+f"(a0), "+f"(a1)
      : "f"(v0), "f"(v1), "f"(s));
}

template <int KIND>
__global__ void __launch_bounds__(kF8Threads, 1)
    gemm_fp8_kernel(const __grid_constant__ CUtensorMap tmA0,
                    const __grid_constant__ CUtensorMap tmB0,
                    const __grid_constant__ CUtensorMap tmA1,
                    const __grid_constant__ CUtensorMap tmB1, const GemmLaunch args) {
  constexpr int kStages = kF8Stages;
  constexpr int kBN = KIND == kGemmW13 ? 128 : 256;  // output columns per tile
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kStages * kF8StageBytes);
  // bars: full[kStages] empty[kStages] tfull[2] tempty[2] amax[4 quarters]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kStages + 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  // amax exchange: [2 slots][4 warps of a quarter][128 rows]
  float* red = reinterpret_cast<float*>(smem + kStages * kF8StageBytes + 256);
  const uint32_t bar0 = smem_addr(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (kStages + s); };
  auto tfull_bar = [&](int b) { return bar0 + 8u * (2 * kStages + b); };
  auto tempty_bar = [&](int b) { return bar0 + 8u * (2 * kStages + 2 + b); };
  auto amax_bar = [&](int q) { return bar0 + 8u * (2 * kStages + 4 + q); };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull_bar(b), 1);
      mbar_init(tempty_bar(b), kF8EpiWarps);
    }
    for (int q = 0; q < kF8Quarters; ++q) mbar_init(amax_bar(q), kF8WarpsPerQuarter);
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
  pdl_wait();  // the set-up above overlapped the previous kernel; its outputs are now visible
  // the next kernel may launch once this one's inputs are complete (so that it, too, may
  // rely on everything before this kernel having finished). DEPENDENCE: the decode w2 GEMM
  // reads the routing's expert blocks before its own wait; that is safe only because this
  // trigger comes after this kernel's wait.
  if (threadIdx.x == 0) pdl_trigger();

  Schedule sched;
  sched.init(args);

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t wpolicy = l2_evict_first_policy();
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
        const int b_row = e * P.b_rows_per_expert + w.nt * kBN;
        for (int kb = w.kb0; kb < w.kb1; ++kb, ++it) {
          const int s = it % kStages;
          const uint32_t ph = (it / kStages) & 1u;
          if (!wait_fast(empty_bar(s), ph ^ 1u, abort_flag, args.status)) {
            ok = false;
            break;
          }
          const uint32_t sa = base + s * kF8StageBytes;
          const uint32_t sb = sa + kGemmBM * kF8BK;
          mbar_expect_tx(full_bar(s), kF8StageBytes);
          tma_load_2d(sa, ta, full_bar(s), kb * kF8BK, a_row);
          // weight boxes stream through L2 first-out: their L2 lines then go before the
          // token rows, which every N tile of the row block re-reads. Measured (graph
          // replay): Mixtral T = 4096 2.084 -> 1.977 ms, DeepSeek-V2 T = 4096 2.485 ->
          // 2.368, DeepSeek-V3 T = 2048 2.680 -> 2.438, although DRAM reads of w13 rise
          // (Mixtral T = 4096: 1.79 -> 2.51 GB) as sibling CTAs re-fetch some boxes.
          tma_load_2d_hint(sb, tb, full_bar(s), kb * kF8BK, b_row, wpolicy);
          if (KIND == kGemmW13)
            tma_load_2d_hint(sb + 128 * kF8BK, tb, full_bar(s), kb * kF8BK, b_row + P.up_offset,
                             wpolicy);
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
          if (!wait_fast(tempty_bar(buf), (use & 1u) ^ 1u, abort_flag, args.status)) {
            ok = false;
            break;
          }
          const int s = it % kStages;
          const uint32_t ph = (it / kStages) & 1u;
          if (!wait_fast(full_bar(s), ph, abort_flag, args.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = base + s * kF8StageBytes;
          const uint64_t da = sdesc_sw128(sa), db = sdesc_sw128(sa + kGemmBM * kF8BK);
          const uint32_t d = tmem_base + buf * kF8BufStride;
#pragma unroll
          for (int kk = 0; kk < kF8BK / 32; ++kk)
            mma_e4m3(d, sdesc_advance(da, kk * 32), sdesc_advance(db, kk * 32), idesc,
                     kk != 0 ? 1u : 0u);
          mma_commit(empty_bar(s));
          mma_commit(tfull_bar(buf));
        }
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3;             // TMEM lanes [32 quarter, 32 quarter + 32)
    const int j = (warp - 2) >> 2;            // which of the quarter's 4 column slices
    const int row = quarter * 32 + lane;
    // this thread's 64 accumulator columns: w13 gate [32 j, +32) and up [128 + 32 j, +32);
    // w2 [64 j, +64)
    uint32_t kbc = 0, nex = 0;                // K blocks and amax exchanges done by this warp
    bool ok = true;
    for (int u = blockIdx.x; ok && u < sched.units; u += gridDim.x) {
      const Unit w = sched.unit(args, u);
      const GemmProblem& P = args.p[w.p];
      const int m = w.mb * kGemmBM + row;
      int e = P.expert_ids ? P.expert_ids[w.mb] : 0;
      if ((unsigned)e >= (unsigned)P.num_experts) e = 0;
      const int KB = P.k_blocks;
      const float* bsc = P.b_scale + (size_t)e * (P.b_rows_per_expert / kFp8Block) * KB;
      // scale rows of this thread's columns: w13 gate block nt and up block (I/128 + nt);
      // w2 the 128-column block holding columns [64 j, +64)
      const float* sb0 = bsc + (size_t)(KIND == kGemmW13 ? w.nt : 2 * w.nt + (j >> 1)) * KB;
      const float* sb1 = bsc + (size_t)(P.up_offset / kFp8Block + w.nt) * KB;
      const bool a_ok = m < P.a_scale_ld;
      const float* asc = P.a_scale + m;
      float acc[kF8Cols];
#pragma unroll
      for (int i = 0; i < kF8Cols; ++i) acc[i] = 0.f;
      // the scales of K block kb + 1 load while K block kb is promoted
      float na = a_ok ? __ldg(asc + (size_t)w.kb0 * P.a_scale_ld) : 0.f;
      float nb0 = __ldg(sb0 + w.kb0);
      float nb1 = KIND == kGemmW13 ? __ldg(sb1 + w.kb0) : 0.f;
      for (int kb = w.kb0; kb < w.kb1; ++kb, ++kbc) {
        const float c0 = na * nb0;
        const float c1 = KIND == kGemmW13 ? na * nb1 : c0;
        if (kb + 1 < w.kb1) {
          na = a_ok ? __ldg(asc + (size_t)(kb + 1) * P.a_scale_ld) : 0.f;
          nb0 = __ldg(sb0 + kb + 1);
          if (KIND == kGemmW13) nb1 = __ldg(sb1 + kb + 1);
        }
        const int buf = kbc & 1;
        const uint32_t use = kbc >> 1;
        if (!wait_fast(tfull_bar(buf), use & 1u, abort_flag, args.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t tb = tmem_base + ((uint32_t)(quarter * 32) << 16) + buf * kF8BufStride;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint32_t col = KIND == kGemmW13 ? (c < 2 ? 32 * j + 16 * c : 128 + 32 * j + 16 * (c - 2))
                                                : 64 * j + 16 * c;
          const float sc = (KIND == kGemmW13 && c >= 2) ? c1 : c0;
          uint32_t v[16];
          tmem_ld16(tb + col, v);
          tmem_wait_ld16(v);
#pragma unroll
          for (int i = 0; i < 16; i += 2)
            fma2(acc[16 * c + i], acc[16 * c + i + 1], sc, __uint_as_float(v[i]),
                 __uint_as_float(v[i + 1]));
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(tempty_bar(buf));
      }
      if (!ok) break;
      const bool split = splits_of(args, w.p) > 1;
      // valid row: its flat index (routed) or token (identity rows), else -1
      int f = -1;
      if (P.sorted_ids) {
        const int v = P.sorted_ids[m];
        if (v >= 0 && v < P.num_flat) f = v;
      } else if (m < P.store_rows) {
        f = m;
      }
      if (KIND == kGemmW13) {
        if (split) {
          // raw fp32 sums of this K range: gate at [0, ldo), up at [ldo, 2 ldo) of the row
          if (f >= 0) {
            float* dst = P.part + (size_t)w.split * P.part_split_stride + (size_t)f * 2 * P.ldo +
                         (size_t)w.nt * 128 + 32 * j;
#pragma unroll
            for (int i = 0; i < 32; i += 4) {
              *reinterpret_cast<float4*>(dst + i) = make_float4(acc[i], acc[i + 1], acc[i + 2], acc[i + 3]);
              *reinterpret_cast<float4*>(dst + P.ldo + i) =
                  make_float4(acc[32 + i], acc[33 + i], acc[34 + i], acc[35 + i]);
            }
          }
        } else {
          float amax = 0.f;
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            acc[i] = acc[i] / (1.f + __expf(-acc[i])) * acc[32 + i];
            amax = fmaxf(amax, fabsf(acc[i]));
          }
          // the 128-column group spans the quarter's 4 warps: swap their amax through shared
          // memory (slots alternate by exchange; a warp reaches exchange n + 2 only after all
          // four arrived at n + 1, i.e. after all four read exchange n)
          float* slot = red + (nex & 1u) * (kF8WarpsPerQuarter * 128);
          slot[j * 128 + row] = amax;
          __syncwarp();
          if (lane == 0) mbar_arrive(amax_bar(quarter));
          if (!wait_fast(amax_bar(quarter), nex & 1u, abort_flag, args.status)) break;
          ++nex;
#pragma unroll
          for (int q = 0; q < kF8WarpsPerQuarter; ++q) amax = fmaxf(amax, slot[q * 128 + row]);
          const float sc = fp8_group_scale(amax);
          const bool store = P.sorted_ids ? true : (m < P.store_rows);
          if (store) {
            uint4* dst = reinterpret_cast<uint4*>(static_cast<uint8_t*>(P.out) + (size_t)m * P.ldo +
                                                  (size_t)w.nt * 128 + 32 * j);
#pragma unroll
            for (int v = 0; v < 2; ++v)
              dst[v] = make_uint4(e4m3x4(acc[16 * v], acc[16 * v + 1], acc[16 * v + 2], acc[16 * v + 3], sc),
                                  e4m3x4(acc[16 * v + 4], acc[16 * v + 5], acc[16 * v + 6], acc[16 * v + 7], sc),
                                  e4m3x4(acc[16 * v + 8], acc[16 * v + 9], acc[16 * v + 10], acc[16 * v + 11], sc),
                                  e4m3x4(acc[16 * v + 12], acc[16 * v + 13], acc[16 * v + 14], acc[16 * v + 15], sc));
            if (j == 0) P.out_scale[(size_t)w.nt * P.out_scale_ld + m] = sc;
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
                       (size_t)dest * P.ldo + (size_t)w.nt * 256 + 64 * j;
#pragma unroll
          for (int i = 0; i < kF8Cols; i += 4)
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

// ---------------------------------------------------------------- decode: weights on M
// Row blocks with at most 32 real rows (T <= 32): the MMA runs transposed, D^T = W X^T,
// with 128 weight rows on M and the 32 token rows on N (M = 128, N = 32), two MMAs per
// K block (w13: the gate and the up block of this tile; w2: the tile's two 128-column
// halves). Each K block then leaves only 2 x 32 TMEM columns to promote, read by 4
// epilogue warps (one per TMEM lane quarter): lane = weight row, column = token.
constexpr int kSwN = 32;                       // token rows per row block (MMA N)
constexpr int kSwThreads = 64 + 32 * 4;
constexpr int kSwBufs = 8;                     // K-block buffers of 2 x 32 TMEM columns: the
constexpr uint32_t kSwTmemCols = 64 * kSwBufs;  // MMA runs up to 8 K blocks ahead of the epilogue
constexpr uint32_t kSwStageBytes = 2 * 128 * kF8BK + kSwN * kF8BK;  // 36 KB
constexpr int kSwStages = 6;
constexpr int kSwChunk = 16;                   // K blocks whose scales are staged at once
// per epilogue warp: the token scales [kSwChunk][32] and the two weight scales [2][kSwChunk]
constexpr uint32_t kSwScaleFloats = kSwChunk * 32 + 2 * kSwChunk;
constexpr size_t kSwSmem = (size_t)kSwStages * kSwStageBytes + 1024 + 256 + 2 * 4 * 32 * 4 +
                           4 * kSwScaleFloats * 4;
static_assert(kSwSmem <= 232448, "shared memory per CTA exceeded");

// Lane l ends with max over the warp's lanes of x[l] (a transposing butterfly, 31 shuffles).
__device__ __forceinline__ float warp_transpose_max(float (&x)[32], int lane) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    const bool upper = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < o; ++i) {
      // keep x[i] (lower lanes) or x[i + o] (upper lanes); send the other to lane ^ o
      const float keep = upper ? x[i + o] : x[i];
      const float give = upper ? x[i] : x[i + o];
      x[i] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, give, o));
    }
  }
  return x[0];
}

template <int KIND>
__global__ void __launch_bounds__(kSwThreads, 1)
    gemm_fp8_swap_kernel(const __grid_constant__ CUtensorMap tmA0,
                         const __grid_constant__ CUtensorMap tmB0,
                         const __grid_constant__ CUtensorMap tmA1,
                         const __grid_constant__ CUtensorMap tmB1, const GemmLaunch args) {
  constexpr int kStages = kSwStages;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kStages * kSwStageBytes);
  // bars: full[kStages] empty[kStages] tfull[kSwBufs] tempty[kSwBufs] amax
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kStages + 2 * kSwBufs + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* red = reinterpret_cast<float*>(smem + kStages * kSwStageBytes + 256);  // [2][4][32]
  float* scl = red + 2 * 4 * 32;                                    // [4 warps][kSwScaleFloats]
  const uint32_t bar0 = smem_addr(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (kStages + s); };
  auto tfull_bar = [&](int b) { return bar0 + 8u * (2 * kStages + b); };
  auto tempty_bar = [&](int b) { return bar0 + 8u * (2 * kStages + kSwBufs + b); };
  const uint32_t amax_bar = bar0 + 8u * (2 * kStages + 2 * kSwBufs);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < kSwBufs; ++b) {
      mbar_init(tfull_bar(b), 1);
      mbar_init(tempty_bar(b), 4);
    }
    mbar_init(amax_bar, 4);
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
    tmem_alloc(smem_addr(tmem_slot), kSwTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // w2: the producer sends the weight boxes of its first stages before it waits on the
  // previous kernel. They depend only on the routing's expert blocks, and this kernel is
  // launched only after the previous one got past its own wait, i.e. after the routing
  // finished. Every other thread waits here.
  constexpr bool kEarlyB = KIND == kGemmW2;
  if (!kEarlyB || warp != 0) pdl_wait();  // the set-up above overlapped the previous kernel
  // after the wait: the decode w2 GEMM relies on it (DEPENDENCE note of the prefill kernel)
  if (!kEarlyB && threadIdx.x == 0) pdl_trigger();

  Schedule sched;
  sched.init(args);
  constexpr int kTileCols = KIND == kGemmW13 ? 128 : 256;   // output columns per tile

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t wpolicy = l2_evict_first_policy();
      uint32_t npre = 0;  // leading stages whose weight boxes went out before the wait
      if (kEarlyB) {
        for (int u = blockIdx.x; npre < (uint32_t)kStages && u < sched.units; u += gridDim.x) {
          const Unit w = sched.unit(args, u);
          const GemmProblem& P = args.p[w.p];
          const CUtensorMap* tb = w.p ? &tmB1 : &tmB0;
          int e = P.expert_ids ? P.expert_ids[w.mb] : 0;
          if ((unsigned)e >= (unsigned)P.num_experts) e = 0;  // recorded below
          const int b_row = e * P.b_rows_per_expert + w.nt * kTileCols;
          for (int kb = w.kb0; kb < w.kb1 && npre < (uint32_t)kStages; ++kb, ++npre) {
            // the ring is empty: stage npre takes the npre-th K block
            const uint32_t sw = base + npre * kSwStageBytes;
            mbar_expect_tx(full_bar(npre), kSwStageBytes);
            tma_load_2d_hint(sw, tb, full_bar(npre), kb * kF8BK, b_row, wpolicy);
            tma_load_2d_hint(sw + 128 * kF8BK, tb, full_bar(npre), kb * kF8BK, b_row + 128,
                             wpolicy);
          }
        }
        pdl_wait();  // the token rows are the previous kernel's output
        pdl_trigger();  // after the wait, like every GEMM
      }
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
        const int b_row = e * P.b_rows_per_expert + w.nt * kTileCols;
        const int b_row1 = KIND == kGemmW13 ? b_row + P.up_offset : b_row + 128;
        for (int kb = w.kb0; kb < w.kb1; ++kb, ++it) {
          const int s = it % kStages;
          const uint32_t ph = (it / kStages) & 1u;
          const uint32_t sw = base + s * kSwStageBytes;
          if (it < npre) {  // its weight boxes are on their way already
            tma_load_2d(sw + 256 * kF8BK, ta, full_bar(s), kb * kF8BK, w.mb * kGemmBM);
            continue;
          }
          if (!wait_fast(empty_bar(s), ph ^ 1u, abort_flag, args.status)) {
            ok = false;
            break;
          }
          mbar_expect_tx(full_bar(s), kSwStageBytes);
          // each weight tile has a single reader here: stream it through L2 first-out
          tma_load_2d_hint(sw, tb, full_bar(s), kb * kF8BK, b_row, wpolicy);
          tma_load_2d_hint(sw + 128 * kF8BK, tb, full_bar(s), kb * kF8BK, b_row1, wpolicy);
          tma_load_2d(sw + 256 * kF8BK, ta, full_bar(s), kb * kF8BK, w.mb * kGemmBM);
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_e4m3(128, kSwN);
      uint32_t it = 0, kbc = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < sched.units; u += gridDim.x) {
        const Unit w = sched.unit(args, u);
        for (int kb = w.kb0; kb < w.kb1; ++kb, ++it, ++kbc) {
          const int buf = kbc % kSwBufs;
          const uint32_t use = kbc / kSwBufs;
          if (!wait_fast(tempty_bar(buf), (use & 1u) ^ 1u, abort_flag, args.status)) {
            ok = false;
            break;
          }
          const int s = it % kStages;
          const uint32_t ph = (it / kStages) & 1u;
          if (!wait_fast(full_bar(s), ph, abort_flag, args.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sw = base + s * kSwStageBytes;
          const uint64_t dw = sdesc_sw128(sw), dx = sdesc_sw128(sw + 256 * kF8BK);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint32_t d = tmem_base + buf * 64 + h * kSwN;
#pragma unroll
            for (int kk = 0; kk < kF8BK / 32; ++kk)
              mma_e4m3(d, sdesc_advance(dw, h * 128 * kF8BK + kk * 32),
                       sdesc_advance(dx, kk * 32), idesc, kk != 0 ? 1u : 0u);
          }
          mma_commit(empty_bar(s));
          mma_commit(tfull_bar(buf));
        }
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3;                  // weight rows [32 quarter, +32) of each half
    uint32_t kbc = 0, nex = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < sched.units; u += gridDim.x) {
      const Unit w = sched.unit(args, u);
      const GemmProblem& P = args.p[w.p];
      const int m0 = w.mb * kGemmBM;               // token rows m0 .. m0 + 31
      const int mt = m0 + lane;                    // this lane's token row (for per-token facts)
      int e = P.expert_ids ? P.expert_ids[w.mb] : 0;
      if ((unsigned)e >= (unsigned)P.num_experts) e = 0;
      const int KB = P.k_blocks;
      const float* bsc = P.b_scale + (size_t)e * (P.b_rows_per_expert / kFp8Block) * KB;
      const float* sb0 = bsc + (size_t)(KIND == kGemmW13 ? w.nt : 2 * w.nt) * KB;
      const float* sb1 = KIND == kGemmW13 ? bsc + (size_t)(P.up_offset / kFp8Block + w.nt) * KB
                                          : sb0 + KB;
      const bool a_ok = mt < P.a_scale_ld;
      const float* asc = P.a_scale + mt;
      float* sA = scl + quarter * kSwScaleFloats;  // this warp's staged scales
      float* sB = sA + kSwChunk * 32;
      float acc0[32], acc1[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) acc0[i] = acc1[i] = 0.f;
      for (int kb = w.kb0; kb < w.kb1; ++kb, ++kbc) {
        const int ci = (kb - w.kb0) % kSwChunk;
        if (ci == 0) {
          // stage the next kSwChunk K blocks' scales: independent loads, one latency per chunk
          __syncwarp();
          float ta[kSwChunk];
#pragma unroll
          for (int i = 0; i < kSwChunk; ++i)
            ta[i] = (a_ok && kb + i < w.kb1) ? __ldg(asc + (size_t)(kb + i) * P.a_scale_ld) : 0.f;
          const int kl = kb + (lane & (kSwChunk - 1));
          const float tb = kl < w.kb1 ? __ldg((lane < kSwChunk ? sb0 : sb1) + kl) : 0.f;
#pragma unroll
          for (int i = 0; i < kSwChunk; ++i) sA[i * 32 + lane] = ta[i];
          sB[lane] = tb;                         // [0, 16): sb0, [16, 32): sb1
          __syncwarp();
        }
        const int buf = kbc % kSwBufs;
        const uint32_t use = kbc / kSwBufs;
        if (!wait_fast(tfull_bar(buf), use & 1u, abort_flag, args.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t tb = tmem_base + ((uint32_t)(quarter * 32) << 16) + buf * 64;
        uint32_t v0[32], v1[32];
        tmem_ld32(tb, v0);
        tmem_ld32(tb + kSwN, v1);
        tmem_wait_ld(v0);
        reg_fence(v1);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(tempty_bar(buf));       // the registers hold the block
        const float s0 = sB[ci], s1 = sB[kSwChunk + ci];
        const float4* st4 = reinterpret_cast<const float4*>(sA + ci * 32);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const float4 st = st4[q];                          // the scales of tokens 4q .. 4q+3
          const float sv[4] = {st.x, st.y, st.z, st.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int t = 4 * q + i;
            acc0[t] = fmaf(sv[i] * s0, __uint_as_float(v0[t]), acc0[t]);
            acc1[t] = fmaf(sv[i] * s1, __uint_as_float(v1[t]), acc1[t]);
          }
        }
      }
      if (!ok) break;
      const bool split = splits_of(args, w.p) > 1;
      // per-token facts, computed by the token's lane: flat index (or token) and, for w2,
      // the output slot and routing weight
      int f = -1;
      if (P.sorted_ids) {
        const int v = P.sorted_ids[mt];
        if (v >= 0 && v < P.num_flat) f = v;
      } else if (mt < P.store_rows) {
        f = mt;
      }
      const int r = 32 * quarter + lane;            // weight row within each 128-row half
      if (KIND == kGemmW13) {
        if (split) {
#pragma unroll
          for (int t = 0; t < 32; ++t) {
            const int ft = __shfl_sync(0xffffffffu, f, t);
            if (ft >= 0) {
              float* dst = P.part + (size_t)w.split * P.part_split_stride + (size_t)ft * 2 * P.ldo +
                           (size_t)w.nt * 128 + r;
              dst[0] = acc0[t];
              dst[P.ldo] = acc1[t];
            }
          }
        } else {
          float amax[32];
#pragma unroll
          for (int t = 0; t < 32; ++t) {
            acc0[t] = acc0[t] / (1.f + __expf(-acc0[t])) * acc1[t];   // act of row r, token t
            amax[t] = fabsf(acc0[t]);
          }
          // token t's group (the tile's 128 act columns) spans the 4 warps: reduce within
          // the warp to lane t, then across warps through shared memory
          const float wmax = warp_transpose_max(amax, lane);
          // slots alternate by exchange: a warp can only reach exchange n + 2 after every
          // warp has arrived at n + 1, i.e. after every warp has read exchange n
          float* slot = red + (nex & 1u) * 128;
          slot[quarter * 32 + lane] = wmax;
          __syncwarp();
          if (lane == 0) mbar_arrive(amax_bar);
          if (!wait_fast(amax_bar, nex & 1u, abort_flag, args.status)) break;
          const float tmax = fmaxf(fmaxf(slot[lane], slot[32 + lane]),
                                   fmaxf(slot[64 + lane], slot[96 + lane]));
          ++nex;
          const float sc_l = fp8_group_scale(tmax);  // token (lane)'s act scale
          uint8_t* out = static_cast<uint8_t*>(P.out) + (size_t)w.nt * 128 + r;
          const bool routed = P.sorted_ids != nullptr;
#pragma unroll
          for (int t = 0; t < 32; ++t) {
            const float st = __shfl_sync(0xffffffffu, sc_l, t);
            const int m = m0 + t;
            if (routed || m < P.store_rows) {
              const __nv_fp8_storage_t b =
                  __nv_cvt_float_to_fp8(__fdiv_rn(acc0[t], st), __NV_SATFINITE, __NV_E4M3);
              out[(size_t)m * P.ldo] = b;
            }
          }
          if (quarter == 0 && (routed || mt < P.store_rows))
            P.out_scale[(size_t)w.nt * P.out_scale_ld + mt] = sc_l;
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
        float* outp = static_cast<float*>(P.out) + (size_t)w.split * P.out_split_stride +
                      (size_t)w.nt * 256 + r;
#pragma unroll
        for (int t = 0; t < 32; ++t) {
          const int dt = __shfl_sync(0xffffffffu, dest, t);
          const float wtt = __shfl_sync(0xffffffffu, wt, t);
          if (dt >= 0) {
            outp[(size_t)dt * P.ldo] = wtt * acc0[t];
            outp[(size_t)dt * P.ldo + 128] = wtt * acc1[t];
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kSwTmemCols);
  }
}

template <int KIND>
cudaError_t launch_fp8_swap_typed(const CUtensorMap* tm, const GemmLaunch& args, int grid,
                                  cudaStream_t stream) {
  static int configured_device = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_device != dev) {
    cudaError_t e = cudaFuncSetAttribute(gemm_fp8_swap_kernel<KIND>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kSwSmem);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  return launch_kernel(gemm_fp8_swap_kernel<KIND>, dim3(grid), dim3(kSwThreads), kSwSmem, stream,
                       tm[0], tm[1], tm[2], tm[3], args);
}

template <int KIND>
cudaError_t launch_fp8_typed(const CUtensorMap* tm, const GemmLaunch& args, int grid,
                             cudaStream_t stream) {
  static int configured_device = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_device != dev) {
    cudaError_t e = cudaFuncSetAttribute(gemm_fp8_kernel<KIND>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kF8Smem);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  return launch_kernel(gemm_fp8_kernel<KIND>, dim3(grid), dim3(kF8Threads), kF8Smem, stream,
                       tm[0], tm[1], tm[2], tm[3], args);
}

}  // namespace

cudaError_t launch_gemm_fp8(int kind, const GemmLaunch& L, cudaStream_t stream,
                            int max_rows_per_block) {
  const int arows = max_rows_per_block <= 32 ? 32 : kGemmBM;
  if (L.num_problems < 1 || L.num_problems > 2 || L.splits < 1) return cudaErrorInvalidValue;
  if (kind != kGemmW13 && kind != kGemmW2) return cudaErrorInvalidValue;
  CUtensorMap tm[4];
  long units = 0;
  const bool swap = arows == 32;                   // decode: weights on the MMA's M side
  const uint32_t b_box = (swap || kind == kGemmW13) ? 128u : 256u;
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
  if (swap)
    return kind == kGemmW13 ? launch_fp8_swap_typed<kGemmW13>(tm, L, grid, stream)
                            : launch_fp8_swap_typed<kGemmW2>(tm, L, grid, stream);
  return kind == kGemmW13 ? launch_fp8_typed<kGemmW13>(tm, L, grid, stream)
                          : launch_fp8_typed<kGemmW2>(tm, L, grid, stream);
}

}  // namespace gbmoe
