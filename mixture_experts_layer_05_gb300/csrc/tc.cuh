// Device helpers shared by the grouped GEMM kernels: mbarriers with bounded waits, TMA
// tile loads, tcgen05 (TMEM allocation, MMA issue and commit, TMEM loads), the
// shared-memory and instruction descriptors, the CTA-pair (cluster) forms, the
// activations, and the persistent tile schedule. Included by each GEMM translation
// unit; everything sits in an unnamed namespace, so each unit has its own copy.
#pragma once

#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.h"

namespace gbmoe {
namespace {

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
                                          int* status,
                                          unsigned long long timeout_ns = kWaitTimeoutNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 0u) {
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > timeout_ns) {
        *abort_flag = 1;
        record_status(status, GBMOE_ERR_TIMEOUT);
        return false;
      }
    }
  }
}

// wait_bounded with the first try inline (the common case: the phase has completed).
__device__ __forceinline__ bool wait_fast(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          int* status) {
  if (mbar_try_wait(bar, parity)) return true;
  return wait_bounded(bar, parity, abort_flag, status);
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

// Bring a tile of `map` into L2 without writing shared memory (no completion to wait for).
__device__ __forceinline__ void tma_prefetch_l2_2d(const CUtensorMap* map, int x, int y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y)
               : "memory");
}

// The same load with an L2 eviction policy (createpolicy); streaming operands that no
// other CTA will read again go first, so they do not push everything else out of L2.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ void tma_load_2d_hint(uint32_t dst, const CUtensorMap* map,
                                                 uint32_t bar, int x, int y, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "l"(policy)
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
// 32 lanes x 16 consecutive fp32 columns.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
               : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld16(uint32_t (&r)[16]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;" : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]) :: "memory");
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

// The descriptor of the operand `bytes` further on in shared memory: the start address
// field counts 16-byte units and cannot carry out inside a CTA's shared memory, so the K
// steps of a stage are plain adds (no per-MMA rebuild in the issuing thread's loop).
__device__ __forceinline__ uint64_t sdesc_advance(uint64_t d, uint32_t bytes) {
  return d + (bytes >> 4);
}

// Instruction descriptor of kind::f16: D fp32, A and B bf16, both K-major, N and M.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}

// D[tmem] (+)= A[smem] * B[smem]^T, e4m3 inputs, fp32 accumulator, K = 32 per instruction
// (32 bytes of the 128-byte swizzled row, like kind::f16's 16 bf16 elements).
__device__ __forceinline__ void mma_e4m3(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Instruction descriptor of kind::f8f6f4: D fp32, A and B e4m3 (format code 0), both
// K-major, N and M.
__host__ __device__ constexpr uint32_t idesc_e4m3(int M, int N) {
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// ---------------------------------------------------------------- CTA pair (cluster of 2)
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" :::
                   "memory");
}
// Address of the same shared variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __noinline__ bool wait_bounded_cluster(uint32_t bar, uint32_t parity,
                                                  volatile int* abort_flag, int* status) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const unsigned long long t0 = globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
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
// TMA load into this CTA's shared memory whose completion is counted on an mbarrier
// that may live in the peer CTA of the pair (cluster address).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map,
                                                 uint32_t bar_cluster, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".cta_group::2 [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(x), "r"(y)
      : "memory");
}
__device__ __forceinline__ void tmem_alloc_pair(uint32_t slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
// D[tmem of both CTAs] (+)= A[smem of both CTAs] * B[halves in both CTAs]^T, M = 256.
__device__ __forceinline__ void mma_bf16_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                              uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive on the mbarrier at this offset in both CTAs of the pair once the issued
// MMAs have completed.
__device__ __forceinline__ void mma_commit_pair(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(bar),
      "h"((uint16_t)3)
      : "memory");
}

__device__ __forceinline__ float silu_mul(float g, float u) { return g / (1.f + __expf(-g)) * u; }
__device__ __forceinline__ float silu_f(float g) { return g / (1.f + __expf(-g)); }
// Gated activation with the layer's options: gate' = min(gate, L), up' = clip(up, -L, L)
// when L > 0, act = gate' * sigmoid(alpha * gate') * up'.
__device__ __forceinline__ float act_gated(float g, float u, float alpha, float limit) {
  if (limit > 0.f) {
    g = fminf(g, limit);
    u = fminf(fmaxf(u, -limit), limit);
  }
  return g / (1.f + __expf(-alpha * g)) * u;
}
// act_gated with the fast single-precision division (__fdividef, a couple of ulp): the
// result is rounded to bf16 right after, 2^16 times coarser.
__device__ __forceinline__ float act_gated_fast(float g, float u, float alpha, float limit) {
  if (limit > 0.f) {
    g = fminf(g, limit);
    u = fminf(fmaxf(u, -limit), limit);
  }
  return __fdividef(g, 1.f + __expf(-alpha * g)) * u;
}
// 32 consecutive bf16 biases as fp32 (zeros when b is NULL).
__device__ __forceinline__ void load_bias32(const __nv_bfloat16* b, float (&out)[32]) {
  if (!b) {
#pragma unroll
    for (int i = 0; i < 32; ++i) out[i] = 0.f;
    return;
  }
  const uint4* q = reinterpret_cast<const uint4*>(b);
#pragma unroll
  for (int v = 0; v < 4; ++v) {
    const uint4 x = __ldg(q + v);
    const uint32_t wv[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = unpack_bf16x2(wv[i]);
      out[8 * v + 2 * i] = f.x;
      out[8 * v + 2 * i + 1] = f.y;
    }
  }
}

// Tile t -> (row block, N tile). Row blocks are taken in groups of at most group_m
// consecutive blocks of one expert; a group's tiles run over all N tiles with the
// row block fastest, so the group's A rows stay in L2 while its expert's weight
// tiles stream past, and each weight tile is shared by the group's CTAs.
// The tiles of a group starting at block gs with gn blocks are [gs*NT, (gs+gn)*NT),
// so block t / NT always lies inside the group that owns tile t.
__device__ __forceinline__ void tile_coords(const GemmProblem& a, int m_blocks, int tile,
                                            int* status, int& mb, int& nt) {
  const int b = tile / a.n_tiles;
  int s0 = 0, sn = m_blocks;
  if (a.block_seg) {
    const int2 sg = a.block_seg[b];
    s0 = sg.x;
    sn = sg.y;
    if (sn < 1 || b < s0 || b >= s0 + sn) {
      record_status(status, GBMOE_ERR_DEVICE_CHECK);
      s0 = b;
      sn = 1;
    }
  }
  const int gm = a.group_m > 0 ? a.group_m : 1;
  const int g0 = ((b - s0) / gm) * gm;
  const int gs = s0 + g0;
  const int gn = min(gm, sn - g0);
  const int local = tile - gs * a.n_tiles;
  nt = local / gn;
  mb = gs + local % gn;
}

// Work unit u -> (problem, split, row block, N tile, K-block range).
struct Unit {
  int p, split, mb, nt, kb0, kb1;
  int tail;          // stream-K tail tile index (its K ranges are `split` of tail_splits), or -1
  int tail_splits;
};

struct Schedule {
  int mblk[2], tiles[2], total_tiles, units, units0;
  int dp_units, tail, tail_splits;  // stream-K tail: units [dp_units, units) are tail ranges

  __device__ void init(const GemmLaunch& L, int bm = kGemmBM) {
    total_tiles = 0;
    for (int p = 0; p < 2; ++p) {
      mblk[p] = tiles[p] = 0;
      if (p >= L.num_problems) continue;
      const GemmProblem& P = L.p[p];
      int rows = P.m_rows_dev ? *P.m_rows_dev : P.m_rows_host;
      if (rows < 0 || rows % bm != 0 || rows > P.max_m_blocks * bm) {
        if (threadIdx.x == 0) record_status(L.status, GBMOE_ERR_DEVICE_CHECK);
        rows = 0;
      }
      mblk[p] = rows / bm;
      tiles[p] = mblk[p] * P.n_tiles;
      total_tiles += tiles[p];
    }
    units0 = tiles[0] * splits_of(L, 0);
    units = units0 + tiles[1] * splits_of(L, 1);
    dp_units = units;
    tail = 0;
    tail_splits = 1;
    // stream-K tail: only without split-K, and only when the tail tiles all belong to the
    // last problem
    const int G = gridDim.x;
    const int last = L.num_problems - 1;
    if (L.tail_max_splits > 1 && units == total_tiles && total_tiles >= G) {
      const int tl = total_tiles % G;
      if (tl > 0 && 2 * tl <= G && tl <= tiles[last]) {
        int sp = G / tl;
        if (sp > L.tail_max_splits) sp = L.tail_max_splits;
        if (sp > L.p[last].k_blocks / 4) sp = L.p[last].k_blocks / 4;
        if (sp >= 2) {
          tail = tl;
          tail_splits = sp;
          dp_units = total_tiles - tl;
          units = dp_units + tl * sp;
        }
      }
    }
  }

  // units: problem 0 first, then problem 1; within a problem split-major; then the tail ranges
  // (range-major, so one tile's ranges run on different CTAs of the same round)
  __device__ Unit unit(const GemmLaunch& L, int u) const {
    Unit r;
    r.tail = -1;
    r.tail_splits = 1;
    if (u >= dp_units) {
      const int v = u - dp_units;
      const int j = v % tail, s = v / tail;
      r.p = L.num_problems - 1;
      const int t = dp_units + j - (r.p ? tiles[0] : 0);
      const GemmProblem& P = L.p[r.p];
      tile_coords(P, mblk[r.p], t, L.status, r.mb, r.nt);
      r.split = s;
      r.tail = j;
      r.tail_splits = tail_splits;
      r.kb0 = (s * P.k_blocks) / tail_splits;
      r.kb1 = ((s + 1) * P.k_blocks) / tail_splits;
      return r;
    }
    r.p = u < units0 ? 0 : 1;
    const int local = r.p ? u - units0 : u;
    const int sp = splits_of(L, r.p);
    r.split = local / tiles[r.p];
    const int t = local - r.split * tiles[r.p];
    const GemmProblem& P = L.p[r.p];
    tile_coords(P, mblk[r.p], t, L.status, r.mb, r.nt);
    r.kb0 = (r.split * P.k_blocks) / sp;
    r.kb1 = ((r.split + 1) * P.k_blocks) / sp;
    return r;
  }
};

// ---------------------------------------------------------------- tensor maps (host)
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

// 2-D map over a row-major [rows, inner] tensor of elem_bytes-wide elements, box
// [box_rows, 128 bytes of the row], 128-byte swizzle.
bool make_map_2d(CUtensorMap* m, const void* ptr, CUtensorMapDataType dtype, uint32_t elem_bytes,
                 uint64_t inner, uint64_t rows, uint32_t box_rows) {
  auto enc = tensor_map_encoder();
  if (!enc || rows == 0) return false;
  const cuuint64_t dims[2] = {inner, rows};
  const cuuint64_t strides[1] = {inner * elem_bytes};
  const cuuint32_t box[2] = {128u / elem_bytes, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return enc(m, dtype, 2, const_cast<void*>(ptr), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// bf16 [rows, inner], box [box_rows, 64].
bool make_map(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t rows, uint32_t box_rows) {
  return make_map_2d(m, ptr, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, inner, rows, box_rows);
}

}  // namespace
}  // namespace gbmoe
