// Grouped bf16 GEMMs of the FusedMoE expert MLP with the tokens on the MMA's N side
// ("token-N"), on CTA pairs, for batches whose experts hold many rows (prefill).
//
//   w13: [gate | up] = x_rows @ w13[e]^T, act = silu(gate) * up  (bf16 out)
//   w1 : act = silu(x_rows @ w1[e]^T)                               (not gated)
//   w2 : o = act_rows @ w2[e]^T, times the row's routing weight, scattered to the
//        token's output slot (fp32 out)
//
// Layouts follow `FusedMoE._load_w13` / `_load_w2` on the vLLM `fused_moe/layer` page:
// w13 [E, 2I, H] (gate rows [0, I), up rows [I, 2I)), w2 [E, H, I], both K-major.
//
// Why the tokens go on N: the align pads every expert's rows to whole row blocks, and an
// MMA with the tokens on M spends the same tensor time on a block of 9 real rows as on a
// full one. With the weights on M and the block's tokens on N, the MMA is only as wide as
// the block's real rows rounded up to 16, so padding costs almost nothing.
//
// Why CTA pairs: the tensor cores read both operands from shared memory, and a per-SM
// 128 x 256 tile needs 96 bytes of operands per clock at full rate; measured, such
// kernels level off near two thirds of the MMA rate. A pair of CTAs runs one M = 256 MMA
// (tcgen05.mma.cta_group::2): each CTA stages its own 128 weight rows and half of the
// token rows, 64 bytes per clock per SM, and each stage holds half the bytes, so the ring
// is six stages deep.
//
// Work unit: one row block (256 rows of one expert, or of the tokens for the shared
// expert) times 256 weight rows, 128 in each CTA:
//   w13  CTA r holds up rows f0 + 64 r + [0, 64) and the matching gate rows, so its TMEM
//        lanes 0..63 are up and lanes 64..127 gate of the same 64 features; the warps of
//        lanes 0..63 pass the up values to the warps of lanes 64..127 through shared memory
//        (bounded mbarrier hand-off), which compute silu(gate) * up and store act. (A warp
//        reads the TMEM lanes of its own SM sub-partition, so lanes 64..127 put the
//        activation work on the two sub-partitions that issue neither TMA nor MMAs.)
//   w1   CTA r holds 128 feature rows; w2 CTA r holds output rows h0 + 128 r + [0, 128).
// The block's N tokens are split between the CTAs (rows [0, N/2) in CTA 0, the rest in
// CTA 1), as cta_group::2 takes the N side of its B operand from both CTAs.
//
// Kernel shape (clusters of two CTAs, 320 threads each, warp-specialised):
//   warp 0      TMA producer (both CTAs): weight box(es) and the token box of each stage,
//               counted on the leader's full barrier;
//   warp 1      allocates 512 TMEM columns (two N <= 256 accumulators); in the leader, one
//               lane issues the MMAs (M = 256, N = the block's rows rounded up to 16, K =
//               16) and commits stages and accumulators to the barriers of both CTAs;
//   warps 2..9  epilogue (both CTAs): warp w reads TMEM lane quarter w % 4 and every other
//               32-column chunk, then releases the accumulator on the leader's barrier.
// Units are walked like the tokens-on-M kernel's tiles (expert-aligned row-block groups,
// row block fastest), so concurrent pairs share one weight tile through L2. Every wait is
// bounded: after kWaitTimeoutNs the CTA records GBMOE_ERR_TIMEOUT, stops and frees TMEM.
#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace gbmoe {
namespace {

constexpr int kTnBM = 256;                          // tokens per row block (= align block)
constexpr int kTnStages = 6;
#ifndef GBMOE_TN_GROUP
#define GBMOE_TN_GROUP 2
#endif
// K blocks per barrier round trip: the producer fills kTnGroup consecutive stage buffers
// under one full barrier and the MMA issuer releases them with one commit, so the issuing
// thread's wait + commit (about 150 cycles, which a partial block's short MMAs do not
// cover) is paid once per kTnGroup K blocks.
constexpr int kTnGroup = GBMOE_TN_GROUP;
constexpr int kTnSlots = kTnStages / kTnGroup;     // barrier pairs in use
static_assert(kTnStages % kTnGroup == 0, "stage groups");
constexpr int kTnEpiWarps = 8;
constexpr int kTnThreads = 64 + 32 * kTnEpiWarps;
constexpr uint32_t kTnTmemCols = 512;
constexpr uint32_t kTnAccStride = 256;
constexpr uint32_t kTnWRegion = 128 * kGemmBK * 2;  // 128 weight rows: 16 KB
constexpr uint32_t kTnXRegion = 128 * kGemmBK * 2;  // up to 128 token rows: 16 KB
constexpr uint32_t kTnStageBytes = kTnWRegion + kTnXRegion;
constexpr int kTnBoxes = 4;                          // token boxes of 16, 32, 64, 128 rows
// w13 hand-off of up values to the gate warp of each pair: two buffers (by chunk parity)
// of 32 lanes x 32 floats
constexpr int kTnPairs = 4;
constexpr uint32_t kTnXchgFloats = 32 * 32;
constexpr uint32_t kTnXchgBytes = kTnPairs * 2 * kTnXchgFloats * 4;
#ifndef GBMOE_TN_PREFETCH
#define GBMOE_TN_PREFETCH 0
#endif
#ifndef GBMOE_TN_PREFETCH_MAX_N
#define GBMOE_TN_PREFETCH_MAX_N 128
#endif
// Units whose MMA is at most this wide stream their weights faster than the ring refills:
// the producer also asks L2 for their weight boxes this many K blocks ahead (0: never).
constexpr int kTnPrefetch = GBMOE_TN_PREFETCH;
constexpr int kTnPrefetchMaxN = GBMOE_TN_PREFETCH_MAX_N;
constexpr size_t kTnSmem = (size_t)kTnStages * kTnStageBytes + kTnXchgBytes + 1024 + 512;
static_assert(kTnSmem <= 232448, "shared memory per CTA exceeded");

// Tensor maps of one launch: each problem's weight stack (w13 boxes of 64 rows, else 128)
// and its token rows with boxes of 16, 32, 64 and 128 rows.
struct TnMaps {
  CUtensorMap w[2];
  CUtensorMap x[2][kTnBoxes];
};

__host__ __device__ constexpr int tn_box_rows(int i) { return 16 << i; }

// Real rows of row block mb: from the align's per-block row counts (routed problems) or
// from the identity problem's row count.
__device__ __forceinline__ int tn_rows(const GemmProblem& P, int mb) {
  int n = P.block_rows ? P.block_rows[mb] : P.store_rows - mb * kTnBM;
  return n < 0 ? 0 : (n > kTnBM ? kTnBM : n);
}
// MMA N: the rows rounded up to 16 (at least 16)
__device__ __forceinline__ int tn_n(int rows) { return rows < 16 ? 16 : (rows + 15) & ~15; }
// smallest token box holding half of N
__device__ __forceinline__ int tn_box(int half) {
  return half <= 16 ? 0 : (half <= 32 ? 1 : (half <= 64 ? 2 : 3));
}

// The units of one cluster, walked with their metadata fetched ahead: the row block's
// expert segment (which fixes the rasterised coordinates) two units ahead, and the block's
// expert and real rows one unit ahead, so neither the producer nor the MMA issuer waits on
// global memory at a unit boundary. (This kernel has no split-K and no stream-K tail, so
// units are tiles: problem 0's first.)
struct TnUnit {
  int p, mb, nt, e, rows;
};

struct TnWalk {
  const GemmLaunch* L;
  int tiles0, units, mblk0, mblk1;   // from the launch's Schedule
  int step;
  // pending: the unit after `cur` (segment loaded, coordinates not yet) and the one after
  int p1, t1, p2, t2;
  int2 seg1, seg2;
  bool has1, has2;

  __device__ __forceinline__ void split(int u, int& p, int& t) const {
    p = u < tiles0 ? 0 : 1;
    t = p ? u - tiles0 : u;
  }
  __device__ __forceinline__ int2 load_seg(int p, int t) const {
    const GemmProblem& P = L->p[p];
    const int b = t / P.n_tiles;
    return P.block_seg ? P.block_seg[b] : make_int2(0, p ? mblk1 : mblk0);
  }
  // coordinates of tile t of problem p inside its expert's row-block group (the same walk as
  // tile_coords), then the expert id and real rows of its row block (loads in flight)
  __device__ __forceinline__ TnUnit resolve(int p, int t, int2 sg) const {
    const GemmProblem& P = L->p[p];
    const int b = t / P.n_tiles;
    int s0 = sg.x, sn = sg.y;
    if (sn < 1 || b < s0 || b >= s0 + sn) {
      record_status(L->status, GBMOE_ERR_DEVICE_CHECK);
      s0 = b;
      sn = 1;
    }
    const int gm = P.group_m > 0 ? P.group_m : 1;
    const int g0 = ((b - s0) / gm) * gm;
    const int gs = s0 + g0;
    const int gn = min(gm, sn - g0);
    const int local = t - gs * P.n_tiles;
    TnUnit r;
    r.p = p;
    r.nt = local / gn;
    r.mb = gs + local % gn;
    r.e = P.expert_ids ? P.expert_ids[r.mb] : 0;
    r.rows = tn_rows(P, r.mb);
    return r;
  }
  // first unit of this walk (its loads are waited for)
  __device__ __forceinline__ TnUnit start(int u0, int stride) {
    step = stride;
    TnUnit cur;
    cur.rows = 0;
    int p, t;
    if (u0 < units) {
      split(u0, p, t);
      cur = resolve(p, t, load_seg(p, t));
    }
    has1 = u0 + step < units;
    if (has1) {
      split(u0 + step, p1, t1);
      seg1 = load_seg(p1, t1);
    }
    return cur;
  }
  // begin unit u (whose data `cur` holds): issue the next units' loads; returns the next unit
  __device__ __forceinline__ TnUnit ahead(int u) {
    TnUnit nxt;
    nxt.rows = 0;
    if (has1) nxt = resolve(p1, t1, seg1);
    has2 = u + 2 * step < units;
    if (has2) {
      split(u + 2 * step, p2, t2);
      seg2 = load_seg(p2, t2);
    }
    has1 = has2;
    p1 = p2;
    t1 = t2;
    seg1 = seg2;
    return nxt;
  }
};

template <int KIND>
__global__ void __launch_bounds__(kTnThreads, 1)
    gemm_tn_kernel(const __grid_constant__ TnMaps maps, const __grid_constant__ GemmLaunch args) {
  constexpr bool kGated = KIND == kGemmW13;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;            // 1024-aligned stages
  uint8_t* smem = smem_raw + (base - raw);
  float* xchg = reinterpret_cast<float*>(smem + kTnStages * kTnStageBytes);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kTnStages * kTnStageBytes + kTnXchgBytes);
  // bars: full[S] empty[S] tfull[2] tempty[2] xfull[pairs][2] xempty[pairs][2]
  constexpr int kNumBars = 2 * kTnStages + 4 + 4 * kTnPairs;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const uint32_t bar0 = smem_addr(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (kTnStages + s); };
  auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * kTnStages + a); };
  auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * kTnStages + 2 + a); };
  auto xfull_bar = [&](int p, int b) { return bar0 + 8u * (2 * kTnStages + 4 + 2 * p + b); };
  auto xempty_bar = [&](int p, int b) {
    return bar0 + 8u * (2 * kTnStages + 4 + 2 * kTnPairs + 2 * p + b);
  };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kTnStages; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), 2 * kTnEpiWarps);
    }
    for (int p = 0; p < kTnPairs; ++p)
      for (int b = 0; b < 2; ++b) {
        mbar_init(xfull_bar(p, b), 1);
        mbar_init(xempty_bar(p, b), 1);
      }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    for (int p = 0; p < args.num_problems; ++p) {
      tma_prefetch(&maps.w[p]);
      for (int i = 0; i < kTnBoxes; ++i) tma_prefetch(&maps.x[p][i]);
    }
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_addr(tmem_slot), kTnTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync();             // barriers of both CTAs initialised, TMEM allocated
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const uint32_t leader_full0 = mapa_shared(full_bar(0), 0);
  const uint32_t leader_tempty0 = mapa_shared(tempty_bar(0), 0);
  pdl_wait();  // the set-up above overlapped the previous kernel; its outputs are now visible
  // DEPENDENCE: a decode w2 GEMM after this kernel may read the routing's expert blocks
  // before its own wait; that is safe only because this trigger follows this kernel's wait.
  if (threadIdx.x == 0) pdl_trigger();

  Schedule sched;
  sched.init(args, kTnBM);
  const int cluster_id = blockIdx.x >> 1, num_clusters = gridDim.x >> 1;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer (both CTAs)
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      TnWalk walk{&args, sched.tiles[0], sched.units, sched.mblk[0], sched.mblk[1]};
      TnUnit w = walk.start(cluster_id, num_clusters);
      for (int u = cluster_id; ok && u < sched.units; u += num_clusters) {
        const TnUnit wn = walk.ahead(u);
        const GemmProblem& P = args.p[w.p];
        int e = w.e;
        if ((unsigned)e >= (unsigned)P.num_experts) {
          record_status(args.status, GBMOE_ERR_DEVICE_CHECK);
          e = 0;
        }
        const int half = tn_n(w.rows) / 2;              // token rows per CTA
        const int bi = tn_box(half);
        const CUtensorMap* tw = &maps.w[w.p];
        const CUtensorMap* tx = &maps.x[w.p][bi];
        // both CTAs' bytes land on the leader's full barrier
        const uint32_t tx_bytes = 2u * (kTnWRegion + (uint32_t)tn_box_rows(bi) * (kGemmBK * 2));
        // this CTA's weight rows: w13 gate f0 + 64 r and up f0 + 64 r (64 each; up in the
        // first 64 rows of the stage); w1 / w2 the 128 rows of half r of the unit's 256
        const int row0 = e * P.b_rows_per_expert;
        const int w_row = kGated ? row0 + w.nt * 128 + (int)rank * 64
                                 : row0 + w.nt * 256 + (int)rank * 128;
        const int x_row = w.mb * kTnBM + (int)rank * half;
        const int pf = (kTnPrefetch > 0 && 2 * half <= kTnPrefetchMaxN) ? kTnPrefetch : 0;
        for (int kb = 0; kb < pf && kb < P.k_blocks; ++kb) {
          tma_prefetch_l2_2d(tw, kb * kGemmBK, kGated ? w_row + P.up_offset : w_row);
          if (kGated) tma_prefetch_l2_2d(tw, kb * kGemmBK, w_row);
        }
        for (int kb0 = 0; kb0 < P.k_blocks; kb0 += kTnGroup, ++it) {
          const int q = it % kTnSlots;
          const uint32_t ph = (it / kTnSlots) & 1u;
          if (!wait_bounded_cluster(empty_bar(q), ph ^ 1u, abort_flag, args.status)) {
            ok = false;
            break;
          }
          const int nst = P.k_blocks - kb0 < kTnGroup ? P.k_blocks - kb0 : kTnGroup;
          if (leader) mbar_expect_tx(full_bar(q), (uint32_t)nst * tx_bytes);
          const uint32_t fb = leader_full0 + 8u * q;
          for (int j = 0; j < nst; ++j) {
            const int kb = kb0 + j;
            const uint32_t sw = base + (q * kTnGroup + j) * kTnStageBytes;
            const uint32_t sx = sw + kTnWRegion;
            if (kGated) {
              tma_load_2d_pair(sw, tw, fb, kb * kGemmBK, w_row + P.up_offset);
              tma_load_2d_pair(sw + 64 * 128, tw, fb, kb * kGemmBK, w_row);
            } else {
              tma_load_2d_pair(sw, tw, fb, kb * kGemmBK, w_row);
            }
            tma_load_2d_pair(sx, tx, fb, kb * kGemmBK, x_row);
            if (pf > 0 && kb + pf < P.k_blocks) {
              tma_prefetch_l2_2d(tw, (kb + pf) * kGemmBK, kGated ? w_row + P.up_offset : w_row);
              if (kGated) tma_prefetch_l2_2d(tw, (kb + pf) * kGemmBK, w_row);
            }
          }
        }
        w = wn;
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (leader only)
    if (leader && lane == 0) {
      uint32_t it = 0;
      int local = 0;
      bool ok = true;
      TnWalk walk{&args, sched.tiles[0], sched.units, sched.mblk[0], sched.mblk[1]};
      TnUnit w = walk.start(cluster_id, num_clusters);
      for (int u = cluster_id; ok && u < sched.units; u += num_clusters, ++local) {
        const TnUnit wn = walk.ahead(u);
        const int k_blocks = args.p[w.p].k_blocks;
        const uint32_t idesc = idesc_bf16(2 * 128, tn_n(w.rows));
        const int acc = local & 1;
        const uint32_t use = (uint32_t)(local >> 1);
        if (!wait_bounded_cluster(tempty_bar(acc), (use & 1u) ^ 1u, abort_flag, args.status))
          break;
        tc_fence_after();
        const uint32_t d = tmem_base + acc * kTnAccStride;
        for (int kb0 = 0; kb0 < k_blocks; kb0 += kTnGroup, ++it) {
          const int q = it % kTnSlots;
          const uint32_t ph = (it / kTnSlots) & 1u;
          if (!wait_bounded_cluster(full_bar(q), ph, abort_flag, args.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const int nst = k_blocks - kb0 < kTnGroup ? k_blocks - kb0 : kTnGroup;
          for (int j = 0; j < nst; ++j) {
            const uint32_t sw = base + (q * kTnGroup + j) * kTnStageBytes;
            const uint64_t dw = sdesc_sw128(sw), dx = sdesc_sw128(sw + kTnWRegion);
#pragma unroll
            for (int kk = 0; kk < kGemmBK / 16; ++kk)
              mma_bf16_pair(d, sdesc_advance(dw, kk * 32), sdesc_advance(dx, kk * 32), idesc,
                            (kb0 + j > 0 || kk != 0) ? 1u : 0u);
          }
          mma_commit_pair(empty_bar(q));
        }
        if (!ok) break;
        mma_commit_pair(tfull_bar(acc));
        w = wn;
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue (both CTAs)
    const int ew = warp - 2;
    const int quarter = warp & 3;             // TMEM lanes [32*quarter, 32*quarter + 32)
    const int chalf = ew >> 2;                // this warp takes chunks chalf, chalf + 2, ...
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    // w13 hand-off: the up warp (quarter 0, 1) of each pair writes its up values, the gate
    // warp (quarter 2, 3) reads them and computes the activation. Lane l's 32 floats sit in
    // a row of 32 rotated by l, so the 32 lanes' element j fall in 32 different banks.
    const int pair = (quarter & 1) + 2 * chalf;
    const bool up_warp = quarter < 2;
    float* xbuf = xchg + (size_t)pair * 2 * kTnXchgFloats;
    uint32_t xit = 0;                          // hand-off counter (same in both warps)
    int local = 0;
    TnWalk walk{&args, sched.tiles[0], sched.units, sched.mblk[0], sched.mblk[1]};
    TnUnit w = walk.start(cluster_id, num_clusters);
    for (int u = cluster_id; u < sched.units; u += num_clusters, ++local) {
      const TnUnit wn = walk.ahead(u);
      const GemmProblem& P = args.p[w.p];
      const int acc = local & 1;
      const uint32_t use = (uint32_t)(local >> 1);
      if (!wait_bounded_cluster(tfull_bar(acc), use & 1u, abort_flag, args.status)) break;
      tc_fence_after();
      const int n = w.rows;
      const int nchunks = (n + 31) / 32;
      const uint32_t t0 = tmem_base + lane_base + acc * kTnAccStride;
      int e_tile = 0;
      if (P.bias && P.expert_ids) {
        e_tile = w.e;
        if ((unsigned)e_tile >= (unsigned)P.num_experts) e_tile = 0;
      }
      bool ok = true;
      if (kGated) {
        // feature of this lane: up lanes 0..63 and gate lanes 64..127 share f
        const int f = w.nt * 128 + (int)rank * 64 + (quarter & 1) * 32 + lane;
        float bg = 0.f, bu = 0.f;
        if (P.bias) {
          const __nv_bfloat16* b = P.bias + (size_t)e_tile * 2 * P.ldo;
          bg = __bfloat162float(b[f]);
          bu = __bfloat162float(b[P.ldo + f]);
        }
        __nv_bfloat16* out = static_cast<__nv_bfloat16*>(P.out) + f;
#pragma unroll 1
        for (int c = chalf; c < nchunks; c += 2, ++xit) {
          const int b = xit & 1;
          const uint32_t xph = (xit >> 1) & 1u;
          float* buf = xbuf + b * kTnXchgFloats + lane * 32;
          uint32_t v[32];
          tmem_ld32(t0 + c * 32, v);
          tmem_wait_ld(v);
          if (up_warp) {
            if (!wait_bounded(xempty_bar(pair, b), xph ^ 1u, abort_flag, args.status)) {
              ok = false;
              break;
            }
#pragma unroll
            for (int j = 0; j < 32; ++j) buf[(j + lane) & 31] = __uint_as_float(v[j]);
            __syncwarp();
            if (lane == 0) mbar_arrive(xfull_bar(pair, b));
          } else {
            if (!wait_bounded(xfull_bar(pair, b), xph, abort_flag, args.status)) {
              ok = false;
              break;
            }
            float a[32];
#pragma unroll
            for (int j = 0; j < 32; ++j)
              a[j] = act_gated_fast(__uint_as_float(v[j]) + bg, buf[(j + lane) & 31] + bu,
                                    P.alpha, P.clamp_limit);
            __syncwarp();
            if (lane == 0) mbar_arrive(xempty_bar(pair, b));
            const size_t m0 = (size_t)w.mb * kTnBM + c * 32;
            const int jn = n - c * 32;
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (j < jn) out[(m0 + j) * P.ldo] = __float2bfloat16_rn(a[j]);
          }
        }
      } else if (KIND == kGemmW1) {
        const int f = w.nt * 256 + (int)rank * 128 + quarter * 32 + lane;
        const float bg = P.bias ? __bfloat162float(P.bias[(size_t)e_tile * P.ldo + f]) : 0.f;
        __nv_bfloat16* out = static_cast<__nv_bfloat16*>(P.out) + f;
#pragma unroll 1
        for (int c = chalf; c < nchunks; c += 2) {
          uint32_t v[32];
          tmem_ld32(t0 + c * 32, v);
          tmem_wait_ld(v);
          const size_t m0 = (size_t)w.mb * kTnBM + c * 32;
          const int jn = n - c * 32;
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (j < jn) out[(m0 + j) * P.ldo] = __float2bfloat16_rn(silu_f(__uint_as_float(v[j]) + bg));
        }
      } else {
        // w2: this lane's output row h; TMEM columns are the block's tokens
        const int h = w.nt * 256 + (int)rank * 128 + quarter * 32 + lane;
        const float bh = P.bias ? __bfloat162float(P.bias[(size_t)e_tile * P.ldo + h]) : 0.f;
        float* out = static_cast<float*>(P.out) + h;
#pragma unroll 1
        for (int c = chalf; c < nchunks; c += 2) {
          // lane l finds the output slot and weight of token column c * 32 + l
          const int jj = c * 32 + lane;
          const int m = w.mb * kTnBM + jj;
          int dest = -1;
          float wt = 1.f;
          if (jj < n) {
            if (P.sorted_ids) {
              const int fl = P.sorted_ids[m];
              if (fl >= 0 && fl < P.num_flat) {
                dest = (fl / P.top_k) * P.slots + (fl % P.top_k);
                wt = P.row_weight ? P.row_weight[fl] : 1.f;
              }
            } else if (m < P.store_rows) {
              dest = m * P.slots + P.slot_offset;
            }
          }
          uint32_t v[32];
          tmem_ld32(t0 + c * 32, v);
          tmem_wait_ld(v);
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int dj = __shfl_sync(0xffffffffu, dest, j);
            const float wj = __shfl_sync(0xffffffffu, wt, j);
            if (dj >= 0) out[(size_t)dj * P.ldo] = wj * (__uint_as_float(v[j]) + bh);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(leader_tempty0 + 8u * acc);  // accumulator free
      if (!ok) break;
      w = wn;
    }
  }

  tc_fence_before();
  cluster_sync();             // no CTA leaves while its peer may still signal or read it
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, kTnTmemCols);
  }
}

template <int KIND>
cudaError_t launch_tn_typed(const TnMaps& maps, const GemmLaunch& args, int clusters,
                            cudaStream_t stream) {
  static int configured_device = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_device != dev) {
    cudaError_t e = cudaFuncSetAttribute(gemm_tn_kernel<KIND>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kTnSmem);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * clusters, 1, 1);
  cfg.blockDim = dim3(kTnThreads, 1, 1);
  cfg.dynamicSmemBytes = kTnSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (pdl_next()) {
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.numAttrs = 2;
  }
  const cudaError_t e = cudaLaunchKernelEx(&cfg, gemm_tn_kernel<KIND>, maps, args);
  pdl_next() = true;
  return e;
}

}  // namespace

bool gemm_tn_supported(int kind, int hidden_or_inter) {
  // w13: units of 128 features (I % 128); w1: 256 features; w2: 256 output rows
  if (kind == kGemmW13) return hidden_or_inter % 128 == 0;
  if (kind == kGemmW1 || kind == kGemmW2) return hidden_or_inter % 256 == 0;
  return false;
}

cudaError_t launch_gemm_tn(int kind, const GemmLaunch& L, cudaStream_t stream) {
  if (L.num_problems < 1 || L.num_problems > 2 || L.splits != 1 || splits_of(L, 1) != 1 ||
      L.tail_max_splits > 1 || (kind != kGemmW13 && kind != kGemmW1 && kind != kGemmW2))
    return cudaErrorInvalidValue;
  TnMaps maps;
  long units = 0;
  for (int p = 0; p < 2; ++p) {
    const GemmProblem& P = L.p[L.num_problems > p ? p : 0];
    if (!make_map(&maps.w[p], P.B, (uint64_t)P.K, (uint64_t)P.b_rows,
                  kind == kGemmW13 ? 64u : 128u))
      return cudaErrorInvalidValue;
    for (int i = 0; i < kTnBoxes; ++i)
      if (!make_map(&maps.x[p][i], P.A, (uint64_t)P.K, (uint64_t)P.a_rows,
                    (uint32_t)tn_box_rows(i)))
        return cudaErrorInvalidValue;
    if (p < L.num_problems) units += (long)P.max_m_blocks * P.n_tiles;
  }
  int clusters = num_sms() / 2;
  if (units < clusters) clusters = (int)units;
  if (clusters < 1) clusters = 1;
  if (kind == kGemmW13) return launch_tn_typed<kGemmW13>(maps, L, clusters, stream);
  if (kind == kGemmW1) return launch_tn_typed<kGemmW1>(maps, L, clusters, stream);
  return launch_tn_typed<kGemmW2>(maps, L, clusters, stream);
}

}  // namespace gbmoe
