// Expert align (stable counting sort of the flat (token, slot) indices by expert,
// runs padded to the block size) and the gather of the real hidden rows into that
// order (padding rows are left unwritten).
//
// The FusedMoE forward (vLLM `fused_moe/layer` page, the Triton fused_moe path
// behind `UnquantizedFusedMoEMethod`) runs its expert GEMMs over tokens grouped by
// expert; sorted_token_ids / expert_ids / num_tokens_post_padded are the outputs of
// that grouping step.
//
// Three launches, no grid-wide waits:
//   count   per chunk of kAlignChunk flat indices, per-expert counts (shared atomics,
//           order-free);
//   scan    one CTA: per-expert totals, padded runs, exclusive scan over experts,
//           per-(chunk, expert) start offsets, sentinel padding, expert_ids, and
//           (for the GEMMs) each block's expert segment (first block, block count) and
//           its real rows;
//   scatter one CTA per chunk; its warps own consecutive slices, count them, take
//           start offsets in slice order, and walk their slices in order, ranking
//           equal experts in each 32-wide step with __match_any_sync: stable order.
#include <climits>

#include "common.cuh"
#include "kernels.h"
#include "route.cuh"

namespace gbmoe {

__global__ void __launch_bounds__(256) align_count_kernel(const int* __restrict__ ids, int n,
                                                          int E, int* __restrict__ counts,
                                                          int* status) {
  pdl_trigger();  // the next kernel may start its launch now
  pdl_wait();     // inputs written by the previous kernel are visible
  extern __shared__ int sc[];
  for (int e = threadIdx.x; e < E; e += blockDim.x) sc[e] = 0;
  __syncthreads();
  const int f0 = blockIdx.x * kAlignChunk;
  const int f1 = min(n, f0 + kAlignChunk);
  for (int f = f0 + threadIdx.x; f < f1; f += blockDim.x) {
    int e = __ldg(ids + f);
    if ((unsigned)e >= (unsigned)E) {
      record_status(status, GBMOE_ERR_DEVICE_CHECK);
      e = 0;
    }
    atomicAdd(&sc[e], 1);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) counts[(size_t)blockIdx.x * E + e] = sc[e];
}

// One CTA of 1024 threads; thread e owns expert e (E <= 1024).
__global__ void __launch_bounds__(1024) align_scan_kernel(const int* __restrict__ counts, int C,
                                                          int E, int bs, int n,
                                                          int* __restrict__ offs,
                                                          int* __restrict__ sorted,
                                                          int* __restrict__ expert_ids,
                                                          int max_blocks, int* __restrict__ npp,
                                                          int2* __restrict__ block_seg,
                                                          int* __restrict__ block_rows) {
  pdl_trigger();  // the next kernel may start its launch now
  pdl_wait();     // inputs written by the previous kernel are visible
  __shared__ int warp_tot[32];
  __shared__ int s_total;
  __shared__ int s_pad0[1024], s_pad1[1024];  // each expert's padding slots [s_pad0, s_pad1)
  const int e = threadIdx.x;
  const int lane = e & 31, wid = e >> 5;
  int tot = 0;
  if (e < E)
    for (int c = 0; c < C; ++c) tot += counts[(size_t)c * E + e];
  const int pad = (tot + bs - 1) / bs * bs;
  // exclusive scan of pad over threads
  int incl = pad;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) warp_tot[wid] = incl;
  __syncthreads();
  if (wid == 0) {
    int w = warp_tot[lane];
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += v;
    }
    warp_tot[lane] = wi - w;  // exclusive prefix of warp totals
    if (lane == 31) s_total = wi;
  }
  __syncthreads();
  const int start = warp_tot[wid] + incl - pad;
  if (e < E) {
    int run = start;
    for (int c = 0; c < C; ++c) {
      offs[(size_t)c * E + e] = run;
      run += counts[(size_t)c * E + e];
    }
    s_pad0[e] = start + tot;
    s_pad1[e] = start + pad;
    for (int b = start / bs; b < (start + pad) / bs; ++b) {
      expert_ids[b] = e;
      if (block_seg) block_seg[b] = make_int2(start / bs, pad / bs);
      if (block_rows) block_rows[b] = min(bs, tot - (b - start / bs) * bs);
    }
  }
  const int total = s_total;
  if (e == 0) *npp = total;
  for (int b = total / bs + e; b < max_blocks; b += blockDim.x) expert_ids[b] = -1;
  // the padding slots get the sentinel n, one expert at a time across the whole CTA
  __syncthreads();
  for (int x = 0; x < E; ++x)
    for (int p = s_pad0[x] + e; p < s_pad1[x]; p += blockDim.x) sorted[p] = n;
}

// One CTA per chunk, kScatterWarps warps, each owning a contiguous slice of the chunk.
// Each warp counts its slice per expert (match_any groups, no atomics), the CTA turns
// the per-warp counts into per-warp start offsets (warps in slice order), then each
// warp walks its slice in order: the order within an expert stays stable.
constexpr int kScatterWarps = 8;
constexpr int kSliceLen = kAlignChunk / kScatterWarps;

__global__ void __launch_bounds__(kScatterWarps * 32)
    align_scatter_kernel(const int* __restrict__ ids, int n, int E, const int* __restrict__ offs,
                         int* __restrict__ sorted, int* __restrict__ inv) {
  pdl_trigger();  // the next kernel may start its launch now
  pdl_wait();     // inputs written by the previous kernel are visible
  extern __shared__ int wcnt[];  // [kScatterWarps][E]
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int* cnt = wcnt + warp * E;
  for (int i = threadIdx.x; i < kScatterWarps * E; i += blockDim.x) wcnt[i] = 0;
  __syncthreads();
  const unsigned lt = (1u << lane) - 1u;
  const int s0 = blockIdx.x * kAlignChunk + warp * kSliceLen;
  const int s1 = min(n, s0 + kSliceLen);
  for (int base = s0; base < s1; base += 32) {
    const int f = base + lane;
    const bool v = f < s1;
    int e = v ? __ldg(ids + f) : -1;
    if (v && (unsigned)e >= (unsigned)E) e = 0;
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    if (v && (peers & lt) == 0u) cnt[e] += __popc(peers);
    __syncwarp();
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int run = offs[(size_t)blockIdx.x * E + e];
    for (int w = 0; w < kScatterWarps; ++w) {
      const int c = wcnt[w * E + e];
      wcnt[w * E + e] = run;
      run += c;
    }
  }
  __syncthreads();
  for (int base = s0; base < s1; base += 32) {
    const int f = base + lane;
    const bool v = f < s1;
    int e = v ? __ldg(ids + f) : -1;
    if (v && (unsigned)e >= (unsigned)E) e = 0;
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    int slot = 0;
    if (v) slot = cnt[e] + __popc(peers & lt);
    __syncwarp();
    if (v) {
      sorted[slot] = f;
      if (inv) inv[f] = slot;
      if ((peers & lt) == 0u) cnt[e] += __popc(peers);
    }
    __syncwarp();
  }
}

__device__ __forceinline__ uint4 scale_bf16x8(uint4 v, float s) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = unpack_bf16x2(w[i]);
    o[i] = pack_bf16x2(f.x * s, f.y * s);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// x_perm[inv[f]] = x[f / k] for every flat index f: only the T*k real rows are written.
// With row_scale (apply_router_weight_on_input) the row is multiplied by row_scale[f]
// in fp32 and rounded once to bf16.
// Padding rows of x_perm are never written: a GEMM output row depends on its own A row
// only, and padding rows are never stored or read back.
__global__ void __launch_bounds__(128) gather_rows_kernel(const uint4* __restrict__ x, int H8,
                                                          const int* __restrict__ inv, int n,
                                                          int k, int max_rows,
                                                          const float* __restrict__ row_scale,
                                                          uint4* __restrict__ xp) {
  pdl_trigger();  // the next kernel may start its launch now
  pdl_wait();     // inputs written by the previous kernel are visible
  for (int f = blockIdx.x; f < n; f += gridDim.x) {
    const int p = inv[f];
    if (p < 0 || p >= max_rows) continue;
    const uint4* src = x + (size_t)(f / k) * H8;
    uint4* dst = xp + (size_t)p * H8;
    if (row_scale) {
      const float sc = row_scale[f];
      for (int i = threadIdx.x; i < H8; i += blockDim.x) dst[i] = scale_bf16x8(__ldg(src + i), sc);
      continue;
    }
    for (int i0 = threadIdx.x; i0 < H8; i0 += 8 * 128) {  // up to eight loads in flight
      uint4 v[8];
#pragma unroll
      for (int q = 0; q < 8; ++q)
        if (i0 + 128 * q < H8) v[q] = __ldg(src + i0 + 128 * q);
#pragma unroll
      for (int q = 0; q < 8; ++q)
        if (i0 + 128 * q < H8) dst[i0 + 128 * q] = v[q];
    }
  }
}

// One warp copies one bf16 row of H8 16-byte vectors (times `scale` when `scaled`), with up
// to eight loads in flight per lane.
__device__ __forceinline__ void copy_row_warp(const uint4* __restrict__ src,
                                              uint4* __restrict__ dst, int H8, int lane,
                                              bool scaled, float scale) {
  if (scaled) {
    for (int j = lane; j < H8; j += 32) dst[j] = scale_bf16x8(__ldg(src + j), scale);
    return;
  }
  int j = lane;
  for (; j + 224 < H8; j += 256) {
    uint4 v[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) v[q] = __ldg(src + j + 32 * q);
#pragma unroll
    for (int q = 0; q < 8; ++q) dst[j + 32 * q] = v[q];
  }
  for (; j + 96 < H8; j += 128) {
    uint4 v[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) v[q] = __ldg(src + j + 32 * q);
#pragma unroll
    for (int q = 0; q < 4; ++q) dst[j + 32 * q] = v[q];
  }
  for (; j < H8; j += 32) dst[j] = __ldg(src + j);
}

// Small batches (T*k <= kAlignChunk): routing and the whole align in one CTA of
// kSmallWarps warps, no global scratch. Warps route tokens (route.cuh) into shared
// memory, count their slices of the flat indices per expert, the CTA scans the padded
// runs (four experts per thread, E <= 1024) and turns the per-warp counts into start
// offsets in slice order, and each warp scatters its slice in order (stable).
constexpr int kSmallWarps = 8;
constexpr int kSmallThreads = kSmallWarps * 32;
// A single token is routed by the whole CTA; from two tokens on a warp per token routes
// them side by side (measured: DeepSeek-V3 T = 4 388 -> 369 us per forward, while T = 1
// stays 2-3 us faster on the CTA-wide path).
constexpr int kBlockRouteMaxTokens = 1;

// The router GEMM of a small batch on CUDA cores (a few tokens against E x H weights is a
// weight stream, not a tensor-core problem): this CTA's warp w takes expert
// 8 * (blockIdx.x / splits) + w over K split blockIdx.x % splits; lane l sums eight
// consecutive products per 256-wide K step for every token, then the warp adds its lanes.
constexpr int kGateMaxTokens = 16;
// TM >= T token rows per pass, U K steps at a time: all loads of a pass (U weight vectors,
// U x TM token vectors) are issued before its FMAs, so a pass costs about one load latency.
// Rows past T re-read row T - 1 (an L1 hit; their sums are not stored); steps past the split
// re-read its last vector and count zero.
template <int TM, int U>
__device__ __forceinline__ void gate_logits_rows(const uint4* __restrict__ wr,
                                                 const uint4* __restrict__ x, int H8, int T,
                                                 int k0, int k1, int lane, float* out) {
  float acc[TM];
#pragma unroll
  for (int t = 0; t < TM; ++t) acc[t] = 0.f;
  for (int kb = k0 + lane; kb < k1; kb += 32 * U) {
    uint4 wv[U], xv[U][TM];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int k = min(kb + 32 * u, k1 - 1);
      wv[u] = __ldg(wr + k);
#pragma unroll
      for (int t = 0; t < TM; ++t) xv[u][t] = __ldg(x + (size_t)min(t, T - 1) * H8 + k);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const bool live = kb + 32 * u < k1;
      const uint32_t wu[4] = {wv[u].x, wv[u].y, wv[u].z, wv[u].w};
      float w[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 f = unpack_bf16x2(wu[i]);
        w[2 * i] = live ? f.x : 0.f;
        w[2 * i + 1] = live ? f.y : 0.f;
      }
#pragma unroll
      for (int t = 0; t < TM; ++t) {
        const uint32_t xu[4] = {xv[u][t].x, xv[u][t].y, xv[u][t].z, xv[u][t].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 f = unpack_bf16x2(xu[i]);
          acc[t] = fmaf(f.x, w[2 * i], acc[t]);
          acc[t] = fmaf(f.y, w[2 * i + 1], acc[t]);
        }
      }
    }
  }
#pragma unroll
  for (int t = 0; t < TM; ++t) out[t] = acc[t];
}

__device__ __forceinline__ void gate_logits_slice(const GateArgs& ga, const uint4* __restrict__ x,
                                                  int H8, int T, int E) {
  const int splits = ga.splits;
  const int grp = blockIdx.x / splits, sp = blockIdx.x % splits;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e = grp * kSmallWarps + warp;
  if (e >= E) return;
  const int kper = (H8 + splits - 1) / splits;
  const int k0 = sp * kper, k1 = min(H8, k0 + kper);
  const uint4* wr = static_cast<const uint4*>(ga.gate) + (size_t)e * H8;
  float acc[kGateMaxTokens];
  if (T <= 1) gate_logits_rows<1, 4>(wr, x, H8, T, k0, k1, lane, acc);
  else if (T <= 2) gate_logits_rows<2, 4>(wr, x, H8, T, k0, k1, lane, acc);
  else if (T <= 4) gate_logits_rows<4, 2>(wr, x, H8, T, k0, k1, lane, acc);
  else if (T <= 8) gate_logits_rows<8, 2>(wr, x, H8, T, k0, k1, lane, acc);
  else gate_logits_rows<kGateMaxTokens, 1>(wr, x, H8, T, k0, k1, lane, acc);
#pragma unroll
  for (int t = 0; t < kGateMaxTokens; ++t) {
    if (t < T) {
      const float v = warp_sum(acc[t]);
      if (lane == 0) ga.part[((size_t)sp * T + t) * E + e] = v;
    }
  }
}

template <int EPT>
__global__ void __launch_bounds__(kSmallThreads, 1)
    route_align_small_kernel(TopkArgs a, int bs, int* __restrict__ sorted,
                             int* __restrict__ expert_ids, int max_blocks, int* __restrict__ npp,
                             int2* __restrict__ block_seg, int* __restrict__ inv,
                             const uint4* __restrict__ x, int H8, uint4* __restrict__ xp,
                             const float* __restrict__ row_scale, GateArgs ga) {
  pdl_trigger();  // the next kernel may start its launch now
  pdl_wait();     // inputs written by the previous kernel are visible
  if (ga.gate) {
    // 0. every CTA computes its slice of the router logits; the last to finish routes
    __shared__ int s_last;
    gate_logits_slice(ga, x, H8, a.T, a.E);
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
      s_last = atomicAdd(ga.counter, 1) == (int)gridDim.x - 1;
      if (s_last) *ga.counter = 0;           // all have arrived: reset for the next forward
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
  }
  extern __shared__ int sm[];
  const int n = a.T * a.k, E = a.E;
  int* s_ids = sm;                                   // [n]
  int* wcnt = sm + ((n + 31) & ~31);                 // [kSmallWarps][E]
  __shared__ int warp_tot[kSmallWarps];
  __shared__ int s_total;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < kSmallWarps * E; i += blockDim.x) wcnt[i] = 0;
  for (int i = threadIdx.x; i < a.zero_count; i += blockDim.x) a.zero[i] = 0;
  // 1. routing: EPT = 0 (a single token) routes it with the whole CTA, in compact code (this
  //    kernel starts each forward, and its code may have to come from HBM after the expert
  //    GEMMs streamed through L2); else a warp per token
  if constexpr (EPT == 0) {
    float* rsm = reinterpret_cast<float*>(wcnt + kSmallWarps * E);
    for (int t = 0; t < a.T; ++t) {
      const int id = route_token_block(a, t, rsm);
      if (threadIdx.x < a.k) s_ids[t * a.k + threadIdx.x] = id;
    }
  } else {
    for (int t = warp; t < a.T; t += kSmallWarps) {
      const int id = route_token_warp<EPT>(a, t, lane);
      if (lane < a.k) s_ids[t * a.k + lane] = id;
    }
  }
  __syncthreads();
  // 1'. at most 32 rows: every active expert holds fewer rows than a block, so each gets
  //     exactly one block, in ascending expert order. One warp ranks the experts and
  //     places the rows (stable: a row's place in its block counts the lower flat indices
  //     of its expert); no pass over all E experts.
  {
    if (n <= 32 && bs >= 32) {
      int* s_slot = wcnt;       // [32] slot of each flat index (the launch sizes the count
      int* s_bcnt = wcnt + 32;  // [32] rows of each block         area to >= 64 ints)
      __shared__ int s_nact;
      if (warp == 0) {
        const int f = lane;
        const bool v = f < n;
        int e = v ? s_ids[f] : INT_MAX;
        if (v && (unsigned)e >= (unsigned)E) e = 0;
        const unsigned lt = (1u << lane) - 1u;
        const unsigned peers = __match_any_sync(0xffffffffu, e);
        const bool first = v && (peers & lt) == 0u;
        const unsigned firsts = __ballot_sync(0xffffffffu, first);
        int rank = 0;  // active experts below e
        for (int i = 0; i < 32; ++i) {
          const int ei = __shfl_sync(0xffffffffu, e, i);
          rank += ((firsts >> i) & 1u) && ei < e;
        }
        if (v) {
          const int slot = rank * bs + __popc(peers & lt);
          s_slot[f] = slot;
          sorted[slot] = f;
          if (inv) inv[f] = slot;
        }
        if (first) {
          expert_ids[rank] = e;
          if (block_seg) block_seg[rank] = make_int2(rank, 1);
          s_bcnt[rank] = __popc(peers);
        }
        if (lane == 0) {
          s_nact = __popc(firsts);
          *npp = __popc(firsts) * bs;
        }
      }
      __syncthreads();
      const int nact = s_nact;
      for (int b = nact + threadIdx.x; b < max_blocks; b += blockDim.x) expert_ids[b] = -1;
      for (int q = threadIdx.x; q < nact * bs; q += blockDim.x)
        if (q % bs >= s_bcnt[q / bs]) sorted[q] = n;  // the padding slots
      if (xp)
        for (int f = warp; f < n; f += kSmallWarps)  // the weights were written above
          copy_row_warp(x + (size_t)(f / a.k) * H8, xp + (size_t)s_slot[f] * H8, H8, lane,
                        row_scale != nullptr, row_scale ? a.weights[f] : 1.f);
      return;
    }
  }
  // 2. per-warp slice counts
  const unsigned lt = (1u << lane) - 1u;
  const int slice = (n + kSmallWarps - 1) / kSmallWarps;
  const int s0 = warp * slice, s1 = min(n, s0 + slice);
  int* cnt = wcnt + warp * E;
  for (int base = s0; base < s1; base += 32) {
    const int f = base + lane;
    const bool v = f < s1;
    int e = v ? s_ids[f] : -1;
    if (v && (unsigned)e >= (unsigned)E) e = 0;
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    if (v && (peers & lt) == 0u) cnt[e] += __popc(peers);
    __syncwarp();
  }
  __syncthreads();
  // 3. padded runs, exclusive scan over experts (thread j owns experts 4j .. 4j+3)
  int tot[4], pad[4], sum = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int e = 4 * threadIdx.x + i;
    tot[i] = 0;
    if (e < E)
      for (int w = 0; w < kSmallWarps; ++w) tot[i] += wcnt[w * E + e];
    pad[i] = (tot[i] + bs - 1) / bs * bs;
    sum += pad[i];
  }
  int incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  if (threadIdx.x == 0) {
    int run = 0;
    for (int w = 0; w < kSmallWarps; ++w) {
      const int v = warp_tot[w];
      warp_tot[w] = run;
      run += v;
    }
    s_total = run;
  }
  __syncthreads();
  int start = warp_tot[warp] + incl - sum;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int e = 4 * threadIdx.x + i;
    if (e < E) {
      int run = start;
      for (int w = 0; w < kSmallWarps; ++w) {
        const int c = wcnt[w * E + e];
        wcnt[w * E + e] = run;
        run += c;
      }
      for (int b = start / bs; b < (start + pad[i]) / bs; ++b) {
        expert_ids[b] = e;
        if (block_seg) block_seg[b] = make_int2(start / bs, pad[i] / bs);
      }
    }
    start += pad[i];
  }
  const int total = s_total;
  if (threadIdx.x == 0) *npp = total;
  for (int b = total / bs + threadIdx.x; b < max_blocks; b += blockDim.x) expert_ids[b] = -1;
  // every slot starts as padding (the sentinel n); the scatter below overwrites the real ones
  // after the barrier, which orders the CTA's writes to the same address
  for (int p = threadIdx.x; p < total; p += blockDim.x) sorted[p] = n;
  __syncthreads();
  // 4. stable scatter of each warp's slice
  for (int base = s0; base < s1; base += 32) {
    const int f = base + lane;
    const bool v = f < s1;
    int e = v ? s_ids[f] : -1;
    if (v && (unsigned)e >= (unsigned)E) e = 0;
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    int slot = 0;
    if (v) slot = cnt[e] + __popc(peers & lt);
    __syncwarp();
    if (v) {
      sorted[slot] = f;
      if (inv) inv[f] = slot;
      if ((peers & lt) == 0u) cnt[e] += __popc(peers);
    }
    __syncwarp();
    // 5. tiny batches: the warp also copies its rows into expert order (the weights were
    //    written by this CTA's routing)
    if (xp) {
      for (int i = 0; i < 32; ++i) {
        const int fi = base + i;
        if (fi >= s1) break;
        const int pi = __shfl_sync(0xffffffffu, slot, i);
        copy_row_warp(x + (size_t)(fi / a.k) * H8, xp + (size_t)pi * H8, H8, lane,
                      row_scale != nullptr, row_scale ? a.weights[fi] : 1.f);
      }
    }
  }
}

struct RouteAlignSmall {
  TopkArgs a;
  int bs;
  int* sorted;
  int* expert_ids;
  int max_blocks;
  int* npp;
  int2* block_seg;
  int* inv;
  const uint4* x;
  int H8;
  uint4* xp;
  const float* row_scale;
  GateArgs ga;
  cudaStream_t stream;
  template <int EPT>
  void operator()() {
    const int n = a.T * a.k;
    // s_ids, the per-warp expert counts, and the CTA-wide routing's scratch (tiny batches)
    const size_t shm = (size_t)(((n + 31) & ~31) + (kSmallWarps * a.E > 64 ? kSmallWarps * a.E : 64) +
                                (a.T <= kBlockRouteMaxTokens ? ((a.E + 3) & ~3) + ((a.E + 15) & ~15) + 128 : 0)) *
                       sizeof(int);
    const int grid = ga.gate ? ((a.E + kSmallWarps - 1) / kSmallWarps) * ga.splits : 1;
    launch_kernel(route_align_small_kernel<EPT>, dim3(grid), dim3(kSmallThreads), shm, stream, a,
                  bs, sorted, expert_ids, max_blocks, npp, block_seg, inv, x, H8, xp, row_scale,
                  ga);
  }
};

// One CTA routes all tokens here (8 warps), so only batches of a few tokens qualify.
bool route_align_small_ok(int T, int k, int E) {
  return T <= kGateMaxTokens && T * k <= kAlignChunk && E <= 1024;
}

int gate_splits(int E, int H) {
  const int groups = (E + kSmallWarps - 1) / kSmallWarps;
  int s = num_sms() / groups;
  const int ksteps = (H / 8 + 31) / 32;           // 256-wide K steps of a warp
  if (s > ksteps) s = ksteps;
  if (s > kGateMaxSplits) s = kGateMaxSplits;
  return s < 1 ? 1 : s;
}

cudaError_t launch_route_align_small(const gbmoe_config_t& c, int T, const float* logits,
                                     const float* bias, float* weights, int* ids, int bs,
                                     int* sorted, int* expert_ids, int max_blocks, int* npp,
                                     int2* block_seg, int* inv, const void* x, void* x_perm,
                                     const float* row_scale, int* status, cudaStream_t stream,
                                     int logit_splits, long long logit_split_stride,
                                     int* zero, int zero_count, GateArgs gate) {
  TopkArgs ta = make_topk_args(c, T, logits, bias, weights, ids, status);
  ta.zero = zero;
  ta.zero_count = zero_count;
  ta.logit_splits = logit_splits;
  ta.logit_split_stride = logit_split_stride;
  if (gate.gate) {                       // the routing reads the launch's own partial logits
    ta.logits = gate.part;
    ta.logit_splits = gate.splits;
    ta.logit_split_stride = (long long)T * c.num_experts;
  }
  RouteAlignSmall L{ta, bs, sorted,
                    expert_ids, max_blocks, npp, block_seg, inv,
                    static_cast<const uint4*>(x), c.hidden_size / 8,
                    static_cast<uint4*>(x_perm), row_scale, gate, stream};
  if (T <= kBlockRouteMaxTokens)
    L.template operator()<0>();
  else
    dispatch_ept(c.num_experts, L);
  return cudaGetLastError();
}

size_t align_scratch_bytes(int n, int E) {
  const size_t C = (size_t)((n + kAlignChunk - 1) / kAlignChunk);
  return 2 * C * (size_t)E * sizeof(int);
}

cudaError_t launch_align(const int* ids, int n, int E, int bs, int* sorted, int* expert_ids,
                         int max_blocks, int* npp, void* scratch, int* status,
                         cudaStream_t stream, int2* block_seg, int* inv, int* block_rows) {
  const int C = (n + kAlignChunk - 1) / kAlignChunk;
  int* counts = static_cast<int*>(scratch);
  int* offs = counts + (size_t)C * E;
  const size_t shm = (size_t)E * sizeof(int);
  if (C > 0) launch_kernel(align_count_kernel, dim3(C), dim3(256), shm, stream, ids, n, E, counts,
                           status);
  launch_kernel(align_scan_kernel, dim3(1), dim3(1024), 0, stream, counts, C, E, bs, n, offs, sorted,
                expert_ids, max_blocks, npp, block_seg, block_rows);
  if (C > 0)
    launch_kernel(align_scatter_kernel, dim3(C), dim3(kScatterWarps * 32), shm * kScatterWarps,
                  stream, ids, n, E, offs, sorted, inv);
  return cudaGetLastError();
}

cudaError_t launch_gather(const void* x, int H, const int* inv, int n, int k, int max_rows,
                          void* x_perm, const float* row_scale, cudaStream_t stream) {
  int blocks = num_sms() * 8;
  if (blocks > n) blocks = n;
  if (blocks < 1) return cudaSuccess;
  launch_kernel(gather_rows_kernel, dim3(blocks), dim3(128), 0, stream,
                static_cast<const uint4*>(x), H / 8, inv, n, k, max_rows, row_scale,
                static_cast<uint4*>(x_perm));
  return cudaGetLastError();
}

}  // namespace gbmoe
