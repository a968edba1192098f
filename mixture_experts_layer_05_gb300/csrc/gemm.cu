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
// Tiles (row block, N tile) are walked in expert-aligned groups of row blocks, row
// block fastest (tile_coords), so concurrent CTAs share one expert's weight tile and
// the group's A rows stay resident in L2. Every wait is bounded:
// after kWaitTimeoutNs the CTA records GBMOE_ERR_TIMEOUT, stops, and frees its TMEM.
#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace gbmoe {
namespace {

constexpr int kStages = 4;
constexpr int kEpiWarps = 4;
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccStride = 256;
constexpr uint32_t kABytes = kGemmBM * kGemmBK * 2;

// AROWS: A rows actually loaded per stage (128, or 32 when every row block holds at most
// 32 real rows, T <= 32); the MMA still reads a 128-row A tile, and the rows not loaded
// only feed output rows that are never stored. Smaller stages buy a deeper pipeline.
template <int KIND, int BN, int AROWS = kGemmBM>
struct Shape {
  static constexpr int kBRows = KIND == kGemmW13 ? 2 * BN : BN;  // B rows per stage = MMA N
  // (kGemmW1: the non-gated first GEMM, BN rows of w1 per tile, like kGemmW2)
  static constexpr uint32_t kBBytes = kBRows * kGemmBK * 2;
  // A region of a stage = the rows actually loaded; the MMA's 128-row read of a 32-row
  // region runs on into the stage's own B bytes (inside this CTA's shared memory), which
  // only feeds discarded output rows.
  static constexpr uint32_t kARegion = AROWS * kGemmBK * 2;
  static constexpr uint32_t kStageBytes = kARegion + kBBytes;    // smem footprint per stage
  static constexpr uint32_t kTxBytes = kARegion + kBBytes;       // bytes TMA delivers per stage
  static constexpr int kNumStages = AROWS == kGemmBM ? kStages : 6;
  static constexpr size_t kSmem = (size_t)kNumStages * kStageBytes + 1024 + 256;
  static_assert(kBRows % 16 == 0 && kBRows <= 256, "MMA N out of range for M=128");
  static_assert(kSmem <= 232448, "shared memory per CTA exceeded");
};

__device__ __forceinline__ void store_f32x32(float* dst, const uint32_t (&r)[32], float w) {
  float4* d = reinterpret_cast<float4*>(dst);
#pragma unroll
  for (int v = 0; v < 8; ++v)
    d[v] = make_float4(w * __uint_as_float(r[4 * v]), w * __uint_as_float(r[4 * v + 1]),
                       w * __uint_as_float(r[4 * v + 2]), w * __uint_as_float(r[4 * v + 3]));
}

#ifndef GBMOE_SHARED_PREFETCH
#define GBMOE_SHARED_PREFETCH 1
#endif
constexpr bool kSharedPrefetch = GBMOE_SHARED_PREFETCH != 0;
constexpr int kSharedPrefetchMaxRows = 4;

template <int KIND, int BN, int AROWS>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA0, const __grid_constant__ CUtensorMap tmB0,
                const __grid_constant__ CUtensorMap tmA1, const __grid_constant__ CUtensorMap tmB1,
                const GemmLaunch args) {
  using S = Shape<KIND, BN, AROWS>;
  constexpr int kStages = S::kNumStages;
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
    tma_prefetch(&tmA0);
    tma_prefetch(&tmB0);
    if (args.num_problems > 1) {
      tma_prefetch(&tmA1);
      tma_prefetch(&tmB1);
    }
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // Decode w2: the producer sends the weight boxes of its first stages before it waits on
  // the previous kernel. They depend only on the routing's expert blocks, and this kernel is
  // launched only after the previous one got past its own wait, i.e. after the routing
  // finished. Every other thread waits here.
  constexpr bool kEarlyB = KIND == kGemmW2 && AROWS < kGemmBM;
  // Decode w13 with a shared expert, T <= 4: the shared expert's weights do not depend on
  // the routing, so while the routing runs (this kernel is waiting below) each CTA asks L2
  // for its share of them, kept with an evict_last policy; the routed weights stream
  // evict_first past them, and the shared units at the end of the launch find them in L2.
  // (Measured: DeepSeek-V2 T = 1 82.6 -> 78.5 us, DeepSeek-V3 T = 1 157 -> 152 us; neutral
  // at T = 4, slightly slower from T = 16, where the routing is short next to the GEMM.)
  if (kSharedPrefetch && KIND != kGemmW2 && AROWS < kGemmBM && args.num_problems > 1 &&
      args.p[1].store_rows <= kSharedPrefetchMaxRows && warp == 3 && lane == 0) {
    const GemmProblem& Q = args.p[1];
    const size_t bytes = (size_t)Q.b_rows * Q.K * 2;
    const size_t per = ((bytes + gridDim.x - 1) / gridDim.x + 15) & ~(size_t)15;
    const size_t off = per * blockIdx.x;
    uint64_t keep;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(keep));
    for (size_t o = off; o < off + per && o < bytes; o += 65536) {
      const size_t n = min((size_t)65536, min(off + per, bytes) - o);
      asm volatile("cp.async.bulk.prefetch.L2.global.L2::cache_hint [%0], %1, %2;" ::"l"(
                       reinterpret_cast<uint64_t>(static_cast<const char*>(Q.B) + o)),
                   "r"((uint32_t)(n & ~(size_t)15)), "l"(keep)
                   : "memory");
    }
  }
  if (!kEarlyB || warp != 0) pdl_wait();  // the set-up above overlapped the previous kernel
  // the next kernel may launch once this one's inputs are complete (so that it, too, may
  // rely on everything before this kernel having finished). DEPENDENCE: the decode w2 GEMM
  // (kEarlyB) reads the routing's expert blocks and schedule before its own wait; that is
  // safe only because this trigger comes after this kernel's wait. Moving it earlier (e.g. to
  // kernel entry) lets a w2 GEMM read stale expert ids.
  if (!kEarlyB && threadIdx.x == 0) pdl_trigger();

  Schedule sched;
  sched.init(args);

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t wpolicy = l2_evict_first_policy();
      uint32_t npre = 0;  // leading stages whose weight box went out before the wait
      if (kEarlyB) {
        for (int u = blockIdx.x; npre < (uint32_t)kStages && u < sched.units; u += gridDim.x) {
          const Unit w = sched.unit(args, u);
          const GemmProblem& P = args.p[w.p];
          const CUtensorMap* tb = w.p ? &tmB1 : &tmB0;
          int e = P.expert_ids ? P.expert_ids[w.mb] : 0;
          if ((unsigned)e >= (unsigned)P.num_experts) e = 0;  // recorded below
          const int b_row = e * P.b_rows_per_expert + w.nt * BN;
          for (int kb = w.kb0; kb < w.kb1 && npre < (uint32_t)kStages; ++kb, ++npre) {
            // the ring is empty: stage npre takes the npre-th K block
            const uint32_t sb = base + npre * S::kStageBytes + S::kARegion;
            mbar_expect_tx(full_bar(npre), S::kTxBytes);
            tma_load_2d_hint(sb, tb, full_bar(npre), kb * kGemmBK, b_row, wpolicy);
          }
        }
        pdl_wait();  // the A rows are the previous kernel's output
        pdl_trigger();  // after the wait, like every GEMM (see the DEPENDENCE note above)
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
        const int a_row = w.mb * kGemmBM;
        const int b_row = e * P.b_rows_per_expert + w.nt * BN;
        for (int kb = w.kb0; kb < w.kb1; ++kb, ++it) {
          const int s = it % kStages;
          const uint32_t ph = (it / kStages) & 1u;
          const uint32_t sa = base + s * S::kStageBytes;
          const uint32_t sb = sa + S::kARegion;
          if (it < npre) {  // its weight box is on its way already
            tma_load_2d(sa, ta, full_bar(s), kb * kGemmBK, a_row);
            continue;
          }
          if (!wait_fast(empty_bar(s), ph ^ 1u, abort_flag, args.status)) {
            ok = false;
            break;
          }
          mbar_expect_tx(full_bar(s), S::kTxBytes);
          tma_load_2d(sa, ta, full_bar(s), kb * kGemmBK, a_row);
          if (AROWS < kGemmBM) {
            // decode: each weight tile has a single reader; stream it through L2 first-out
            tma_load_2d_hint(sb, tb, full_bar(s), kb * kGemmBK, b_row, wpolicy);
            if (KIND == kGemmW13)
              tma_load_2d_hint(sb + BN * 128, tb, full_bar(s), kb * kGemmBK, b_row + P.up_offset,
                               wpolicy);
          } else {
            tma_load_2d(sb, tb, full_bar(s), kb * kGemmBK, b_row);
            if (KIND == kGemmW13)
              tma_load_2d(sb + BN * 128, tb, full_bar(s), kb * kGemmBK, b_row + P.up_offset);
          }
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16(kGemmBM, S::kBRows);
      uint32_t it = 0;
      int local = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < sched.units; u += gridDim.x, ++local) {
        const Unit w = sched.unit(args, u);
        const int acc = local & 1;
        const uint32_t use = (uint32_t)(local >> 1);
        if (!wait_fast(tempty_bar(acc), (use & 1u) ^ 1u, abort_flag, args.status)) break;
        tc_fence_after();
        const uint32_t d = tmem_base + acc * kAccStride;
        for (int kb = w.kb0; kb < w.kb1; ++kb, ++it) {
          const int s = it % kStages;
          const uint32_t ph = (it / kStages) & 1u;
          if (!wait_fast(full_bar(s), ph, abort_flag, args.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = base + s * S::kStageBytes;
          const uint64_t da = sdesc_sw128(sa), db = sdesc_sw128(sa + S::kARegion);
#pragma unroll
          for (int kk = 0; kk < kGemmBK / 16; ++kk)
            mma_bf16(d, sdesc_advance(da, kk * 32), sdesc_advance(db, kk * 32), idesc,
                     (kb > w.kb0 || kk != 0) ? 1u : 0u);
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
    for (int u = blockIdx.x; u < sched.units; u += gridDim.x, ++local) {
      const Unit w = sched.unit(args, u);
      const GemmProblem& P = args.p[w.p];
      const int acc = local & 1;
      const uint32_t use = (uint32_t)(local >> 1);
      if (!wait_fast(tfull_bar(acc), use & 1u, abort_flag, args.status)) break;
      tc_fence_after();
      const bool split = splits_of(args, w.p) > 1;
      const int m = w.mb * kGemmBM + row;
      const uint32_t tbase = tmem_base + ((uint32_t)(quarter * 32) << 16) + acc * kAccStride;
      // valid row: its flat index (routed) or token (identity rows), else -1
      int f = -1;
      if (P.sorted_ids) {
        const int v = P.sorted_ids[m];
        if (v >= 0 && v < P.num_flat) f = v;
      } else if (m < P.store_rows) {
        f = m;
      }
      // expert of this tile's rows (its bias), the routed problem only
      int e_tile = 0;
      if (P.bias && P.expert_ids) {
        e_tile = P.expert_ids[w.mb];
        if ((unsigned)e_tile >= (unsigned)P.num_experts) e_tile = 0;
      }
      if (KIND == kGemmW13 || KIND == kGemmW1) {
        constexpr bool kGated = KIND == kGemmW13;
        const int brow = kGated ? 2 * P.ldo : P.ldo;              // bias entries per expert
        const __nv_bfloat16* bg =
            P.bias ? P.bias + (size_t)e_tile * brow + (size_t)w.nt * BN : nullptr;
        if (!split) {
          const bool store = P.sorted_ids ? true : (m < P.store_rows);
          uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(P.out) +
                                                (size_t)m * P.ldo + (size_t)w.nt * BN);
#pragma unroll 1
          for (int c = 0; c < BN / 32; ++c) {
            uint32_t g[32], up[32];
            tmem_ld32(tbase + c * 32, g);
            if (kGated) tmem_ld32(tbase + BN + c * 32, up);
            tmem_wait_ld(g);
            if (kGated) reg_fence(up);
            float gb[32], ub[32];
            load_bias32(bg ? bg + c * 32 : nullptr, gb);
            if (kGated) load_bias32(bg ? bg + P.ldo + c * 32 : nullptr, ub);
            uint32_t p[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              float a0, a1;
              if (kGated) {
                a0 = act_gated(__uint_as_float(g[2 * i]) + gb[2 * i],
                               __uint_as_float(up[2 * i]) + ub[2 * i], P.alpha, P.clamp_limit);
                a1 = act_gated(__uint_as_float(g[2 * i + 1]) + gb[2 * i + 1],
                               __uint_as_float(up[2 * i + 1]) + ub[2 * i + 1], P.alpha,
                               P.clamp_limit);
              } else {
                a0 = silu_f(__uint_as_float(g[2 * i]) + gb[2 * i]);
                a1 = silu_f(__uint_as_float(g[2 * i + 1]) + gb[2 * i + 1]);
              }
              p[i] = pack_bf16x2(a0, a1);
            }
            if (store) {
#pragma unroll
              for (int v = 0; v < 4; ++v)
                dst[c * 4 + v] = make_uint4(p[4 * v], p[4 * v + 1], p[4 * v + 2], p[4 * v + 3]);
            }
          }
        } else {
          // raw K-slice sums; bias and activation follow once every split is in
          const size_t prow = kGated ? 2 * (size_t)P.ldo : (size_t)P.ldo;
          float* dst = P.part + (size_t)w.split * P.part_split_stride +
                       (size_t)(f < 0 ? 0 : f) * prow + (size_t)w.nt * BN;
#pragma unroll 1
          for (int c = 0; c < BN / 32; ++c) {
            uint32_t g[32], up[32];
            tmem_ld32(tbase + c * 32, g);
            if (kGated) tmem_ld32(tbase + BN + c * 32, up);
            tmem_wait_ld(g);
            if (kGated) reg_fence(up);
            if (f >= 0) {
              store_f32x32(dst + c * 32, g, 1.f);
              if (kGated) store_f32x32(dst + P.ldo + c * 32, up, 1.f);
            }
          }
          if (P.tile_count) {
            // the last split to arrive at this (row block, N tile, lane quarter) sums all
            // splits' partials of its 32 rows in split order and finishes the activation
            __threadfence();
            __syncwarp();
            int last = 0;
            if (lane == 0) {
              int* cnt = P.tile_count + ((size_t)w.mb * P.n_tiles + w.nt) * 4 + quarter;
              last = atomicAdd(cnt, 1) == splits_of(args, w.p) - 1;
              if (last) *cnt = 0;                  // every split has arrived: reset for reuse
            }
            last = __shfl_sync(0xffffffffu, last, 0);
            if (last) {
              __threadfence();
              const int nsp = splits_of(args, w.p);
              const float* src0 = P.part + (size_t)(f < 0 ? 0 : f) * prow + (size_t)w.nt * BN;
              __nv_bfloat16* act = static_cast<__nv_bfloat16*>(P.out) + (size_t)m * P.ldo +
                                   (size_t)w.nt * BN;
#pragma unroll 1
              for (int c = 0; c < BN / 32 && f >= 0; ++c) {
                float gs[32], us[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) gs[i] = us[i] = 0.f;
                for (int sp = 0; sp < nsp; ++sp) {
                  const float4* q = reinterpret_cast<const float4*>(
                      src0 + (size_t)sp * P.part_split_stride + c * 32);
#pragma unroll
                  for (int v = 0; v < 8; ++v) {
                    const float4 a4 = __ldcg(q + v);
                    gs[4 * v] += a4.x; gs[4 * v + 1] += a4.y; gs[4 * v + 2] += a4.z; gs[4 * v + 3] += a4.w;
                    if (kGated) {
                      const float4 b4 = __ldcg(q + P.ldo / 4 + v);
                      us[4 * v] += b4.x; us[4 * v + 1] += b4.y; us[4 * v + 2] += b4.z; us[4 * v + 3] += b4.w;
                    }
                  }
                }
                float gb[32], ub[32];
                load_bias32(bg ? bg + c * 32 : nullptr, gb);
                if (kGated) load_bias32(bg ? bg + P.ldo + c * 32 : nullptr, ub);
                uint32_t pk[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                  float a0, a1;
                  if (kGated) {
                    a0 = act_gated(gs[2 * i] + gb[2 * i], us[2 * i] + ub[2 * i], P.alpha, P.clamp_limit);
                    a1 = act_gated(gs[2 * i + 1] + gb[2 * i + 1], us[2 * i + 1] + ub[2 * i + 1], P.alpha,
                                   P.clamp_limit);
                  } else {
                    a0 = silu_f(gs[2 * i] + gb[2 * i]);
                    a1 = silu_f(gs[2 * i + 1] + gb[2 * i + 1]);
                  }
                  pk[i] = pack_bf16x2(a0, a1);
                }
                uint4* o = reinterpret_cast<uint4*>(act + c * 32);
#pragma unroll
                for (int v = 0; v < 4; ++v)
                  o[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
              }
            }
          }
        }
      } else if (KIND == kGemmRouter) {
        // logits[split][m][n] for m < T, n < E (ldo = E); rows/columns past them are the
        // zero fill of out-of-range TMA boxes and are not stored
        float* dst = static_cast<float*>(P.out) + (size_t)w.split * P.out_split_stride +
                     (size_t)m * P.ldo;
        const int col0 = w.nt * BN;
        const bool vec = (P.ldo & 3) == 0;
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          uint32_t r[32];
          tmem_ld32(tbase + c * 32, r);
          tmem_wait_ld(r);
          const int cc = col0 + c * 32;
          if (m < P.store_rows && cc < P.ldo) {
            if (vec && cc + 32 <= P.ldo) {
              store_f32x32(dst + cc, r, 1.f);
            } else {
              for (int i = 0; i < 32 && cc + i < P.ldo; ++i) dst[cc + i] = __uint_as_float(r[i]);
            }
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
        if (w.tail >= 0) {
          // stream-K tail range: the raw partial goes to its scratch slot; the last range of
          // this tile and lane quarter sums the ranges in order and finishes the epilogue
          float* part = args.tail_part +
                        ((size_t)(w.tail * w.tail_splits + w.split) * kGemmBM + row) * BN;
#pragma unroll 1
          for (int c = 0; c < BN / 32; ++c) {
            uint32_t r[32];
            tmem_ld32(tbase + c * 32, r);
            tmem_wait_ld(r);
            store_f32x32(part + c * 32, r, 1.f);
          }
          __threadfence();
          __syncwarp();
          int last = 0;
          if (lane == 0) {
            int* cnt = args.tail_count + (size_t)w.tail * 4 + quarter;
            last = atomicAdd(cnt, 1) == w.tail_splits - 1;
            if (last) *cnt = 0;                      // every range has arrived: reset
          }
          last = __shfl_sync(0xffffffffu, last, 0);
          if (last) {
            __threadfence();
            const __nv_bfloat16* b2 =
                P.bias ? P.bias + (size_t)e_tile * P.ldo + (size_t)w.nt * BN : nullptr;
            float* dst = static_cast<float*>(P.out) + (size_t)(dest < 0 ? 0 : dest) * P.ldo +
                         (size_t)w.nt * BN;
            const float* src0 = args.tail_part +
                                ((size_t)(w.tail * w.tail_splits) * kGemmBM + row) * BN;
#pragma unroll 1
            for (int c = 0; c < BN / 32 && dest >= 0; ++c) {
              float acc[32];
#pragma unroll
              for (int i = 0; i < 32; ++i) acc[i] = 0.f;
              for (int sp = 0; sp < w.tail_splits; ++sp) {
                const float4* q = reinterpret_cast<const float4*>(
                    src0 + (size_t)sp * kGemmBM * BN + c * 32);
#pragma unroll
                for (int v = 0; v < 8; ++v) {
                  const float4 a4 = __ldcg(q + v);
                  acc[4 * v] += a4.x; acc[4 * v + 1] += a4.y; acc[4 * v + 2] += a4.z; acc[4 * v + 3] += a4.w;
                }
              }
              uint32_t r[32];
              float bb[32];
              load_bias32(b2 ? b2 + c * 32 : nullptr, bb);
#pragma unroll
              for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(acc[i] + bb[i]);
              store_f32x32(dst + c * 32, r, wt);
            }
          }
        } else {
          // the expert's output bias enters once (split 0), inside the routing weight
          const __nv_bfloat16* b2 = (P.bias && w.split == 0)
                                        ? P.bias + (size_t)e_tile * P.ldo + (size_t)w.nt * BN
                                        : nullptr;
          float* dst = static_cast<float*>(P.out) + (size_t)w.split * P.out_split_stride +
                       (size_t)(dest < 0 ? 0 : dest) * P.ldo + (size_t)w.nt * BN;
#pragma unroll 1
          for (int c = 0; c < BN / 32; ++c) {
            uint32_t r[32];
            tmem_ld32(tbase + c * 32, r);
            tmem_wait_ld(r);
            if (b2) {
              float bb[32];
              load_bias32(b2 + c * 32, bb);
#pragma unroll
              for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) + bb[i]);
            }
            if (dest >= 0) store_f32x32(dst + c * 32, r, wt);
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

// Self test of the bounded wait: one thread waits on an mbarrier nobody arrives on; the
// wait gives up after timeout_ns and records GBMOE_ERR_TIMEOUT in the status word.
__global__ void wait_selftest_kernel(int* status, unsigned long long timeout_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_addr(&bar), 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) wait_bounded(smem_addr(&bar), 0u, &abort_flag, status, timeout_ns);
}

// act = silu(sum_s gate_s) * sum_s up_s, one CTA per output row, 8 columns per step.
__global__ void __launch_bounds__(128) silu_reduce_kernel(const __grid_constant__ GemmLaunch L,
                                                          const int* npp,
                                                          int max_routed_rows, int gated) {
  // Triggering at entry is safe for the decode w2 GEMM that follows (it reads the routing's
  // expert blocks before its wait): this kernel itself launched only after the w13 GEMM in
  // front of it passed its wait, i.e. after the routing finished.
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
    int src, dst_row, row_gated = gated;
    const __nv_bfloat16* bias = nullptr;
    if (r < routed_items) {
      P = &L.p[0];
      int f;
      if (P->flat_row) {
        f = r;
        dst_row = P->flat_row[r];
        if (dst_row < 0 || dst_row >= routed_rows) continue;
      } else {
        if (r >= routed_rows) continue;
        f = P->sorted_ids ? P->sorted_ids[r] : r;
        if (f < 0 || f >= P->num_flat) continue;        // padding rows are never read back
        dst_row = r;
      }
      src = f;
      if (P->bias && P->expert_of_flat) {
        int e = P->expert_of_flat[f];
        if ((unsigned)e >= (unsigned)P->num_experts) e = 0;
        bias = P->bias + (size_t)e * (row_gated ? 2 * P->ldo : P->ldo);
      }
    } else {
      P = &L.p[1];                                      // the shared expert: always gated
      src = dst_row = r - routed_items;
      row_gated = 1;
    }
    const int N = P->ldo;
    const float* base = P->part + (size_t)src * (row_gated ? 2 * N : N);
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(P->out) + (size_t)dst_row * N;
    for (int j = threadIdx.x * 8; j < N; j += blockDim.x * 8) {
      float g[8], u[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) g[i] = u[i] = 0.f;
      const int nsp = splits_of(L, P == &L.p[0] ? 0 : 1);
#pragma unroll 4
      for (int s = 0; s < nsp; ++s) {
        const float* q = base + (size_t)s * P->part_split_stride + j;
        const float4 g0 = __ldg(reinterpret_cast<const float4*>(q));
        const float4 g1 = __ldg(reinterpret_cast<const float4*>(q + 4));
        g[0] += g0.x; g[1] += g0.y; g[2] += g0.z; g[3] += g0.w;
        g[4] += g1.x; g[5] += g1.y; g[6] += g1.z; g[7] += g1.w;
        if (row_gated) {
          const float4 u0 = __ldg(reinterpret_cast<const float4*>(q + N));
          const float4 u1 = __ldg(reinterpret_cast<const float4*>(q + N + 4));
          u[0] += u0.x; u[1] += u0.y; u[2] += u0.z; u[3] += u0.w;
          u[4] += u1.x; u[5] += u1.y; u[6] += u1.z; u[7] += u1.w;
        }
      }
      if (bias) {
        const uint4 bg = __ldg(reinterpret_cast<const uint4*>(bias + j));
        const uint32_t wg[4] = {bg.x, bg.y, bg.z, bg.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 fb = unpack_bf16x2(wg[i]);
          g[2 * i] += fb.x;
          g[2 * i + 1] += fb.y;
        }
        if (row_gated) {
          const uint4 bu = __ldg(reinterpret_cast<const uint4*>(bias + N + j));
          const uint32_t wu[4] = {bu.x, bu.y, bu.z, bu.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float2 fb = unpack_bf16x2(wu[i]);
            u[2 * i] += fb.x;
            u[2 * i + 1] += fb.y;
          }
        }
      }
      float a[8];
#pragma unroll
      for (int i = 0; i < 8; ++i)
        a[i] = row_gated ? act_gated(g[i], u[i], P->alpha, P->clamp_limit) : silu_f(g[i]);
      uint4 o;
      o.x = pack_bf16x2(a[0], a[1]);
      o.y = pack_bf16x2(a[2], a[3]);
      o.z = pack_bf16x2(a[4], a[5]);
      o.w = pack_bf16x2(a[6], a[7]);
      *reinterpret_cast<uint4*>(out + j) = o;
    }
  }
}

template <int KIND, int BN, int AROWS>
cudaError_t launch_typed(const CUtensorMap* tm, const GemmLaunch& args, int grid,
                         cudaStream_t stream) {
  using S = Shape<KIND, BN, AROWS>;
  static int configured_device = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_device != dev) {
    cudaError_t e = cudaFuncSetAttribute(gemm_kernel<KIND, BN, AROWS>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)S::kSmem);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  return launch_kernel(gemm_kernel<KIND, BN, AROWS>, dim3(grid), dim3(kThreads), S::kSmem, stream,
                       tm[0], tm[1], tm[2], tm[3], args);
}

template <int AROWS>
cudaError_t launch_rows(int kind, int bn, const CUtensorMap* tm, const GemmLaunch& L, int grid,
                        cudaStream_t stream) {
  if (kind == kGemmW13 && bn == 128) return launch_typed<kGemmW13, 128, AROWS>(tm, L, grid, stream);
  if (kind == kGemmW1 && bn == 128) return launch_typed<kGemmW1, 128, AROWS>(tm, L, grid, stream);
  if (kind == kGemmRouter && bn == 128)
    return launch_typed<kGemmRouter, 128, AROWS>(tm, L, grid, stream);
  if (kind == kGemmW2 && bn == 256) return launch_typed<kGemmW2, 256, AROWS>(tm, L, grid, stream);
  if (kind == kGemmW2 && bn == 128) return launch_typed<kGemmW2, 128, AROWS>(tm, L, grid, stream);
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_gemm(int kind, int bn, const GemmLaunch& L, cudaStream_t stream,
                        int max_rows_per_block) {
  const int arows = max_rows_per_block <= 32 ? 32 : kGemmBM;
  if (L.num_problems < 1 || L.num_problems > 2 || L.splits < 1) return cudaErrorInvalidValue;
  CUtensorMap tm[4];
  long units = 0;
  for (int p = 0; p < 2; ++p) {
    const GemmProblem& P = L.p[L.num_problems > p ? p : 0];
    if (!make_map(&tm[2 * p], P.A, (uint64_t)P.K, (uint64_t)P.a_rows, (uint32_t)arows) ||
        !make_map(&tm[2 * p + 1], P.B, (uint64_t)P.K, (uint64_t)P.b_rows, (uint32_t)bn))
      return cudaErrorInvalidValue;
    if (p < L.num_problems) {
      if (splits_of(L, p) < 1 || P.k_blocks < splits_of(L, p)) return cudaErrorInvalidValue;
      units += (long)P.max_m_blocks * P.n_tiles * splits_of(L, p);
    }
  }
  int grid = num_sms();
  if (units < grid) grid = (int)units;
  if (grid < 1) grid = 1;
  return arows == 32 ? launch_rows<32>(kind, bn, tm, L, grid, stream)
                     : launch_rows<kGemmBM>(kind, bn, tm, L, grid, stream);
}

cudaError_t launch_wait_selftest(int* status, int timeout_us, cudaStream_t stream) {
  wait_selftest_kernel<<<1, 32, 0, stream>>>(status, (unsigned long long)timeout_us * 1000ull);
  return cudaGetLastError();
}

cudaError_t launch_silu_reduce(const GemmLaunch& L, const int* npp, int max_routed_rows,
                               bool gated, cudaStream_t stream) {
  const int rows = (L.p[0].flat_row ? L.p[0].num_flat : max_routed_rows) +
                   (L.num_problems > 1 ? L.p[1].store_rows : 0);
  int grid = num_sms() * 4;
  if (rows < grid) grid = rows;
  if (grid < 1) return cudaSuccess;
  return launch_kernel(silu_reduce_kernel, dim3(grid), dim3(128), 0, stream, L, npp,
                       max_routed_rows, gated ? 1 : 0);
}

}  // namespace gbmoe
