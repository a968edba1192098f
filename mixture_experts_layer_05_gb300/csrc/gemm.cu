// Grouped bf16 GEMMs of the FusedMoE expert MLP on the 5th-generation tensor cores.
//
//   w13: [gate | up] = x_rows @ w13[e]^T, act = silu(gate) * up  (bf16 out)
//   w2 : o = act_rows @ w2[e]^T, times the row's routing weight, scattered to the
//        token's output slot (fp32 out, so the layer output is rounded to bf16 once)
//
// Layouts follow `FusedMoE._load_w13` / `_load_w2` on the vLLM `fused_moe/layer`
// page: w13 [E, 2I, H] (gate rows [0, I), up rows [I, 2I)), w2 [E, H, I]; both
// operands are K-major, so A and B tiles are plain row slices.
//
// Kernel shape (one persistent CTA per SM, 192 threads, warp-specialised):
//   warp 0      TMA producer: A tile [128 x 64] and B tile [N x 64] per stage into a
//               4-deep ring of 128-byte-swizzled shared-memory stages (mbarrier
//               complete_tx), waiting on the stage's "empty" barrier;
//   warp 1      allocates 512 TMEM columns (two 256-column fp32 accumulators) and,
//               from one lane, issues tcgen05.mma (M=128, N=256, K=16) x4 per stage,
//               tcgen05.commit frees the stage, and a final commit per tile marks
//               the accumulator full;
//   warps 2..5  epilogue: tcgen05.ld of their 32 TMEM lanes, SiLU*mul (bf16 stores) or
//               weighting (fp32 stores); then release the accumulator, so the epilogue of tile i
//               overlaps the MMAs of tile i+1.
// Tiles (row block, N tile) are walked row-block-fastest, so CTAs running at the
// same time share the weight tile of one expert through L2. Every wait is bounded:
// after kWaitTimeoutNs the CTA records GBMOE_ERR_TIMEOUT, stops, and frees its TMEM.
#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.h"

namespace gbmoe {
namespace {

constexpr int kStages = 4;
constexpr int kEpiWarps = 4;
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccStride = 256;
constexpr uint32_t kABytes = kGemmBM * kGemmBK * 2;

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase of `bar` with parity `parity`; false if the CTA is aborting or
// the wait ran past kWaitTimeoutNs (then the CTA is marked aborting).
__device__ __noinline__ bool wait_bounded(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          int* status) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 0u) {
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > kWaitTimeoutNs) {
        *abort_flag = 1;
        record_status(status, GBMOE_ERR_TIMEOUT);
        return false;
      }
    }
  }
}

// ---------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_prefetch(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y)
      : "memory");
}

// ---------------------------------------------------------------- tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// D[tmem] (+)= A[smem] * B[smem]^T, bf16 inputs, fp32 accumulator.
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}
// 32 lanes x 32 consecutive fp32 columns: thread i of the warp gets row (lane base + i).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
               : "r"(taddr));
}
// Wait for outstanding tcgen05.ld; the registers are threaded through so that no use
// of them can be scheduled before the wait.
__device__ __forceinline__ void tmem_wait_ld(uint32_t (&r)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;" : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31]) :: "memory");
}
__device__ __forceinline__ void reg_fence(uint32_t (&r)[32]) {
  asm volatile("" : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31]) :: "memory");
}

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row core groups
// 1024 bytes apart (SBO), leading offset unused for swizzled K-major (1), the
// descriptor version bit of the tcgen05 format, swizzle mode 2 (128 B).
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr) {
  uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)1 << 16;
  d |= (uint64_t)(1024 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// Instruction descriptor of kind::f16: D fp32, A and B bf16, both K-major, N and M.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ float silu_mul(float g, float u) { return g / (1.f + __expf(-g)) * u; }

template <int KIND, int BN>
struct Shape {
  static constexpr int kBRows = KIND == kGemmW13 ? 2 * BN : BN;  // B rows per stage = MMA N
  static constexpr uint32_t kBBytes = kBRows * kGemmBK * 2;
  static constexpr uint32_t kStageBytes = kABytes + kBBytes;
  static constexpr size_t kSmem = (size_t)kStages * kStageBytes + 1024 + 256;
  static_assert(kBRows % 16 == 0 && kBRows <= 256, "MMA N out of range for M=128");
};

template <int KIND, int BN>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const GemmArgs args) {
  using S = Shape<KIND, BN>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;            // 1024-aligned tiles
  uint8_t* smem = smem_raw + (base - raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kStages * S::kStageBytes);
  // bars: full[kStages] empty[kStages] tfull[2] tempty[2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kStages + 4);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const uint32_t bar0 = smem_addr(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (kStages + s); };
  auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * kStages + a); };
  auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * kStages + 2 + a); };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), kEpiWarps);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch(&tmA);
    tma_prefetch(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  int m_rows = args.m_rows_dev ? *args.m_rows_dev : args.m_rows_host;
  if (m_rows < 0 || m_rows % kGemmBM != 0 || m_rows > args.max_m_blocks * kGemmBM) {
    if (threadIdx.x == 0) record_status(args.status, GBMOE_ERR_DEVICE_CHECK);
    m_rows = 0;
  }
  const int m_blocks = m_rows / kGemmBM;
  const int num_tiles = m_blocks * args.n_tiles;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t it = 0;
      for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
        const int mb = tile % m_blocks, nt = tile / m_blocks;
        int e = args.expert_ids ? args.expert_ids[mb] : 0;
        if ((unsigned)e >= (unsigned)args.num_experts) {
          record_status(args.status, GBMOE_ERR_DEVICE_CHECK);
          e = 0;
        }
        const int a_row = mb * kGemmBM;
        const int b_row = e * args.b_rows_per_expert + nt * BN;
        bool ok = true;
        for (int kb = 0; kb < args.k_blocks; ++kb, ++it) {
          const int s = it % kStages;
          const uint32_t ph = (it / kStages) & 1u;
          if (!wait_bounded(empty_bar(s), ph ^ 1u, abort_flag, args.status)) {
            ok = false;
            break;
          }
          const uint32_t sa = base + s * S::kStageBytes;
          const uint32_t sb = sa + kABytes;
          mbar_expect_tx(full_bar(s), S::kStageBytes);
          tma_load_2d(sa, &tmA, full_bar(s), kb * kGemmBK, a_row);
          tma_load_2d(sb, &tmB, full_bar(s), kb * kGemmBK, b_row);
          if (KIND == kGemmW13)
            tma_load_2d(sb + BN * 128, &tmB, full_bar(s), kb * kGemmBK, b_row + args.up_offset);
        }
        if (!ok) break;
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16(kGemmBM, S::kBRows);
      uint32_t it = 0;
      int local = 0;
      for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x, ++local) {
        const int acc = local & 1;
        const uint32_t use = (uint32_t)(local >> 1);
        if (!wait_bounded(tempty_bar(acc), (use & 1u) ^ 1u, abort_flag, args.status)) break;
        tc_fence_after();
        const uint32_t d = tmem_base + acc * kAccStride;
        bool ok = true;
        for (int kb = 0; kb < args.k_blocks; ++kb, ++it) {
          const int s = it % kStages;
          const uint32_t ph = (it / kStages) & 1u;
          if (!wait_bounded(full_bar(s), ph, abort_flag, args.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = base + s * S::kStageBytes;
          const uint32_t sb = sa + kABytes;
#pragma unroll
          for (int kk = 0; kk < kGemmBK / 16; ++kk)
            mma_bf16(d, sdesc_sw128(sa + kk * 32), sdesc_sw128(sb + kk * 32), idesc,
                     (kb | kk) != 0 ? 1u : 0u);
          mma_commit(empty_bar(s));
        }
        if (!ok) break;
        mma_commit(tfull_bar(acc));
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3;            // TMEM lanes [32*quarter, 32*quarter + 32)
    const int row = quarter * 32 + lane;
    int local = 0;
    for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x, ++local) {
      const int acc = local & 1;
      const uint32_t use = (uint32_t)(local >> 1);
      if (!wait_bounded(tfull_bar(acc), use & 1u, abort_flag, args.status)) break;
      tc_fence_after();
      const int mb = tile % m_blocks, nt = tile / m_blocks;
      const int m = mb * kGemmBM + row;
      const uint32_t tbase = tmem_base + ((uint32_t)(quarter * 32) << 16) + acc * kAccStride;
      __nv_bfloat16* out = static_cast<__nv_bfloat16*>(args.out);
      if (KIND == kGemmW13) {
        const bool store = m < args.store_rows;
        uint4* dst = reinterpret_cast<uint4*>(out + (size_t)m * args.ldo + (size_t)nt * BN);
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          uint32_t g[32], u[32];
          tmem_ld32(tbase + c * 32, g);
          tmem_ld32(tbase + BN + c * 32, u);
          tmem_wait_ld(g);
          reg_fence(u);
          uint32_t p[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            p[i] = pack_bf16x2(silu_mul(__uint_as_float(g[2 * i]), __uint_as_float(u[2 * i])),
                               silu_mul(__uint_as_float(g[2 * i + 1]),
                                        __uint_as_float(u[2 * i + 1])));
          if (store) {
#pragma unroll
            for (int v = 0; v < 4; ++v)
              dst[c * 4 + v] = make_uint4(p[4 * v], p[4 * v + 1], p[4 * v + 2], p[4 * v + 3]);
          }
        }
      } else {
        int dest = -1;
        float w = 1.f;
        if (args.sorted_ids) {
          const int f = args.sorted_ids[m];
          if (f >= 0 && f < args.num_flat) {
            dest = (f / args.top_k) * args.slots + (f % args.top_k);
            w = args.row_weight ? args.row_weight[f] : 1.f;
          }
        } else if (m < args.store_rows) {
          dest = m * args.slots + args.slot_offset;
        }
        float4* dst = reinterpret_cast<float4*>(static_cast<float*>(args.out) +
                                                (size_t)(dest < 0 ? 0 : dest) * args.ldo +
                                                (size_t)nt * BN);
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          uint32_t r[32];
          tmem_ld32(tbase + c * 32, r);
          tmem_wait_ld(r);
          if (dest >= 0) {
#pragma unroll
            for (int v = 0; v < 8; ++v)
              dst[c * 8 + v] = make_float4(w * __uint_as_float(r[4 * v]),
                                           w * __uint_as_float(r[4 * v + 1]),
                                           w * __uint_as_float(r[4 * v + 2]),
                                           w * __uint_as_float(r[4 * v + 3]));
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty_bar(acc));
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// 2-D bf16 map over a row-major [rows, inner] tensor, box [box_rows, 64], 128 B swizzle.
bool make_map(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t rows, uint32_t box_rows) {
  auto enc = tensor_map_encoder();
  if (!enc || rows == 0) return false;
  const cuuint64_t dims[2] = {inner, rows};
  const cuuint64_t strides[1] = {inner * 2};
  const cuuint32_t box[2] = {(cuuint32_t)kGemmBK, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int KIND, int BN>
cudaError_t launch_typed(const CUtensorMap& ta, const CUtensorMap& tb, const GemmArgs& args,
                         int grid, cudaStream_t stream) {
  using S = Shape<KIND, BN>;
  static int configured_device = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_device != dev) {
    cudaError_t e = cudaFuncSetAttribute(gemm_kernel<KIND, BN>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)S::kSmem);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  gemm_kernel<KIND, BN><<<grid, kThreads, S::kSmem, stream>>>(ta, tb, args);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemm(int kind, int bn, const void* A, int a_rows_alloc, int K, const void* B,
                        int b_rows_total, const GemmArgs& args, cudaStream_t stream) {
  CUtensorMap ta, tb;
  if (!make_map(&ta, A, (uint64_t)K, (uint64_t)a_rows_alloc, kGemmBM)) return cudaErrorInvalidValue;
  if (!make_map(&tb, B, (uint64_t)K, (uint64_t)b_rows_total, (uint32_t)bn))
    return cudaErrorInvalidValue;
  long tiles = (long)args.max_m_blocks * args.n_tiles;
  int grid = num_sms();
  if (tiles < grid) grid = (int)tiles;
  if (grid < 1) grid = 1;
  if (kind == kGemmW13 && bn == 128) return launch_typed<kGemmW13, 128>(ta, tb, args, grid, stream);
  if (kind == kGemmW2 && bn == 256) return launch_typed<kGemmW2, 256>(ta, tb, args, grid, stream);
  if (kind == kGemmW2 && bn == 128) return launch_typed<kGemmW2, 128>(ta, tb, args, grid, stream);
  return cudaErrorInvalidValue;
}

}  // namespace gbmoe
