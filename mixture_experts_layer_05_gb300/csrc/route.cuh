// Router scoring and (grouped) top-k of one token by one warp: experts spread over
// lanes (expert e lives in lane e % 32, register slot e / 32), every reduction a
// shuffle. Shared by the stand-alone top-k kernel and the fused small-batch
// routing + align kernel.
//
// Method: `FusedMoE.select_experts` on the vLLM `fused_moe/layer` page (grouped_topk
// with num_expert_group / topk_group / scoring_func / routed_scaling_factor /
// e_score_correction_bias; fused_topk_bias; fused_topk). The group score is the
// largest score in the group without a correction bias and the sum of the two
// largest biased keys with one (the pages name the biased method "noaux_tc" but do
// not spell out its group score; this is the DeepSeek-V3 reading).
#pragma once

#include <climits>
#include <cmath>

#include "common.cuh"

namespace gbmoe {

struct TopkArgs {
  const float* logits;
  const float* bias;
  float* weights;
  int* ids;
  int* status;
  int T, E, k, renorm, grouped, G, g, sigmoid;
  float rsf;
  int logit_splits;              // logits arrive as this many fp32 partial copies (>= 1),
  long long logit_split_stride;  // summed in copy order on load (split-K router GEMM); read
                                 // through L2 (they may come from the same launch)
  int* zero;                     // the forward's split counters, cleared by the routing
  int zero_count;                // kernel (it runs before any GEMM of the forward)
};

// (key, index) pair maximum: larger key wins, equal keys go to the lower index.
__device__ __forceinline__ void warp_argmax(float& key, int& idx) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ok = __shfl_xor_sync(0xffffffffu, key, o);
    const int oi = __shfl_xor_sync(0xffffffffu, idx, o);
    if (ok > key || (ok == key && oi < idx)) {
      key = ok;
      idx = oi;
    }
  }
}

// Float -> unsigned with the same order (sign flipped for positives, all bits for negatives),
// so a warp-wide unsigned max (redux.sync) is a float max.
__device__ __forceinline__ unsigned ordered_bits(float f) {
  const unsigned u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

constexpr int kFastGroups = 8;  // group filters with at most this many groups reduce in parallel

// Routes token t with the calling warp; writes weights[t, :] and ids[t, :] and returns,
// in lane j < k, the j-th chosen expert (-1 in the other lanes).
template <int EPT>
__device__ __forceinline__ int route_token_warp(const TopkArgs& a, int t, int lane) {
  const int gsize = a.grouped ? a.E / a.G : a.E;
  int grp[EPT];
#pragma unroll
  for (int i = 0; i < EPT; ++i) grp[i] = (lane + 32 * i) / gsize;
  const float* row = a.logits + (size_t)t * a.E;
  float s[EPT], q[EPT], bias[EPT];
  float mx = -INFINITY;
  // the logits and the correction bias load together
#pragma unroll
  for (int i = 0; i < EPT; ++i) {
    const int e = lane + 32 * i;
    float l = -INFINITY;
    bias[i] = 0.f;
    if (e < a.E) {
      l = __ldcg(row + e);
      if (a.bias) bias[i] = __ldg(a.bias + e);
      for (int sp = 1; sp < a.logit_splits; ++sp) l += __ldcg(row + sp * a.logit_split_stride + e);
    }
    s[i] = l;
    mx = fmaxf(mx, s[i]);
  }
  // 1. scores
  if (!a.sigmoid) {
    mx = warp_max(mx);
    float sum = 0.f;
#pragma unroll
    for (int i = 0; i < EPT; ++i) {
      const float z = (lane + 32 * i) < a.E ? expf(s[i] - mx) : 0.f;
      s[i] = z;
      sum += z;
    }
    sum = warp_sum(sum);
#pragma unroll
    for (int i = 0; i < EPT; ++i) s[i] = s[i] / sum;
  } else {
#pragma unroll
    for (int i = 0; i < EPT; ++i)
      s[i] = (lane + 32 * i) < a.E ? 1.f / (1.f + expf(-s[i])) : 0.f;
  }
  // 2. selection keys
#pragma unroll
  for (int i = 0; i < EPT; ++i) {
    const int e = lane + 32 * i;
    q[i] = e < a.E ? (a.bias ? s[i] + bias[i] : s[i]) : -INFINITY;
  }
  // 3. group filter: group score = largest score (no bias) or sum of the two largest keys
  uint32_t kept = 0xffffffffu;
  if (a.grouped && a.G <= kFastGroups) {
    // every group's (first, second) best at once: a lane's own candidates, then one
    // butterfly over the warp that merges all groups' pairs per step
    float b1[kFastGroups], b2[kFastGroups];
#pragma unroll
    for (int g = 0; g < kFastGroups; ++g) b1[g] = b2[g] = -INFINITY;
#pragma unroll
    for (int i = 0; i < EPT; ++i) {
      const float v = (lane + 32 * i) < a.E ? (a.bias ? q[i] : s[i]) : -INFINITY;
#pragma unroll
      for (int g = 0; g < kFastGroups; ++g) {
        const float vg = grp[i] == g ? v : -INFINITY;   // branch-free: b1/b2 stay in registers
        b2[g] = fmaxf(b2[g], fminf(b1[g], vg));
        b1[g] = fmaxf(b1[g], vg);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
      for (int g = 0; g < kFastGroups; ++g) {
        const float o1 = __shfl_xor_sync(0xffffffffu, b1[g], o);
        const float o2 = __shfl_xor_sync(0xffffffffu, b2[g], o);
        const float n1 = fmaxf(b1[g], o1);
        b2[g] = fmaxf(fminf(b1[g], o1), fmaxf(b2[g], o2));
        b1[g] = n1;
      }
    }
    // every lane now holds all group scores: pick the kept groups locally (ties to the
    // lower group index)
    float gs[kFastGroups];
#pragma unroll
    for (int g = 0; g < kFastGroups; ++g)
      gs[g] = g < a.G ? (a.bias ? b1[g] + (b2[g] == -INFINITY ? 0.f : b2[g]) : b1[g]) : -INFINITY;
    kept = 0u;
    for (int r = 0; r < a.g; ++r) {
      int bi = -1;
      float bk = -INFINITY;
#pragma unroll
      for (int g = 0; g < kFastGroups; ++g) {
        if (g < a.G && !((kept >> g) & 1u) && (bi < 0 || gs[g] > bk)) {
          bk = gs[g];
          bi = g;
        }
      }
      if (bi < 0) {
        if (lane == 0) record_status(a.status, GBMOE_ERR_DEVICE_CHECK);
        break;
      }
      kept |= 1u << bi;
    }
  } else if (a.grouped) {
    float my_gs = -INFINITY;
    for (int g = 0; g < a.G; ++g) {
      float b1 = -INFINITY, b2 = -INFINITY;
#pragma unroll
      for (int i = 0; i < EPT; ++i) {
        if ((lane + 32 * i) < a.E && grp[i] == g) {
          const float v = a.bias ? q[i] : s[i];
          if (v > b1) {
            b2 = b1;
            b1 = v;
          } else if (v > b2) {
            b2 = v;
          }
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float o1 = __shfl_xor_sync(0xffffffffu, b1, o);
        const float o2 = __shfl_xor_sync(0xffffffffu, b2, o);
        const float n1 = fmaxf(b1, o1);
        const float n2 = fmaxf(fminf(b1, o1), fmaxf(b2, o2));
        b1 = n1;
        b2 = n2;
      }
      const float gs = a.bias ? b1 + (b2 == -INFINITY ? 0.f : b2) : b1;
      if (lane == g) my_gs = gs;
    }
    kept = 0u;
    float key = lane < a.G ? my_gs : -INFINITY;
    for (int r = 0; r < a.g; ++r) {
      float bk = key;
      int bi = lane < a.G ? lane : INT_MAX;
      warp_argmax(bk, bi);
      if (bi == INT_MAX) {
        record_status(a.status, GBMOE_ERR_DEVICE_CHECK);
        break;
      }
      kept |= 1u << bi;
      if (lane == bi) key = -INFINITY;
    }
  }
  // 4. top-k over the surviving experts: per round, the warp's largest key (an unsigned
  //    max over order-preserving bits), then the lowest expert index holding it
  uint32_t taken = 0u;
  float my_w = 0.f;
  int my_id = -1;
  for (int j = 0; j < a.k; ++j) {
    unsigned bk = 0u;                              // below every real key's bits
#pragma unroll
    for (int i = 0; i < EPT; ++i) {
      const int e = lane + 32 * i;
      if (e < a.E && !((taken >> i) & 1u) && ((kept >> grp[i]) & 1u))
        bk = max(bk, ordered_bits(q[i]));
    }
    const unsigned best = __reduce_max_sync(0xffffffffu, bk);
    unsigned mine = 0xffffffffu;                   // lowest expert index of this lane at `best`
#pragma unroll
    for (int i = EPT - 1; i >= 0; --i) {
      const int e = lane + 32 * i;
      if (e < a.E && !((taken >> i) & 1u) && ((kept >> grp[i]) & 1u) &&
          ordered_bits(q[i]) == best)
        mine = (unsigned)e;
    }
    int be = (int)__reduce_min_sync(0xffffffffu, mine);
    float sv = 0.f;
    if (best == 0u || be >= a.E) {
      record_status(a.status, GBMOE_ERR_DEVICE_CHECK);
      be = 0;
    } else if (lane == (be & 31)) {
      const int idx = be >> 5;
#pragma unroll
      for (int i = 0; i < EPT; ++i) {
        if (i == idx) {
          sv = s[i];
          taken |= 1u << i;
        }
      }
    }
    sv = __shfl_sync(0xffffffffu, sv, be & 31);
    if (lane == j) {
      my_w = sv;
      my_id = be;
    }
  }
  // 5. weights
  if (a.renorm) {
    float tot = 0.f;
    for (int j = 0; j < a.k; ++j) tot += __shfl_sync(0xffffffffu, my_w, j);
    my_w = my_w / tot;
  }
  my_w *= a.rsf;
  if (lane < a.k) {
    a.weights[(size_t)t * a.k + lane] = my_w;
    a.ids[(size_t)t * a.k + lane] = my_id;
  }
  return my_id;
}

// Routes token t with the whole CTA (all threads call it together; tiny batches, where
// one warp per token would leave the CTA's other warps idle). Thread i owns experts
// i, i + blockDim.x, ...; softmax by block reductions; thread g < G scores group g; an
// expert's place among the chosen is the number of eligible experts with a larger key
// (ties to the lower index), so the k chosen come out in descending key order, as in
// route_token_warp. smem: 2 E (rounded up to 4) + 128 floats, 16-byte aligned. Returns
// the j-th chosen expert in threads j < k (-1 elsewhere) and writes weights[t, :] and
// ids[t, :].
__device__ __forceinline__ int route_token_block(const TopkArgs& a, int t, float* smem) {
  const int E = a.E, tid = threadIdx.x, nt = blockDim.x;
  const int lane = tid & 31, warp = tid >> 5, nw = nt >> 5;
  const int E4 = (E + 3) & ~3;     // keys start on a 16-byte boundary (read as float4)
  const int E16 = (E + 15) & ~15;  // and run to a multiple of 16 (-inf past E)
  float* sc = smem;                // [E] scores
  float* key = sc + E4;            // [E16] selection keys (-inf once excluded)
  float* gsc = key + E16;          // [G] group scores
  float* ow = gsc + 32;         // [k] chosen weights
  int* oid = reinterpret_cast<int*>(ow + 32);  // [k] chosen experts
  float* red = ow + 64;         // [32] reduction scratch
  const float* row = a.logits + (size_t)t * E;
  if (tid < a.k) oid[tid] = -1;            // set before the first barrier below
  float mx = -INFINITY;
  for (int e = tid; e < E; e += nt) {
    float l = __ldcg(row + e);
    if (a.bias) key[e] = __ldg(a.bias + e);  // the bias is fetched with the logits
    for (int sp = 1; sp < a.logit_splits; ++sp) l += __ldcg(row + sp * a.logit_split_stride + e);
    sc[e] = l;
    mx = fmaxf(mx, l);
  }
  if (!a.sigmoid) {
    mx = warp_max(mx);
    if (lane == 0) red[warp] = mx;
    __syncthreads();
    mx = red[0];
    for (int w = 1; w < nw; ++w) mx = fmaxf(mx, red[w]);
    float sum = 0.f;
    for (int e = tid; e < E; e += nt) {
      const float z = expf(sc[e] - mx);
      sc[e] = z;
      sum += z;
    }
    sum = warp_sum(sum);
    __syncthreads();                       // every thread has read red[] for the max
    if (lane == 0) red[warp] = sum;
    __syncthreads();
    float tot = 0.f;
    for (int w = 0; w < nw; ++w) tot += red[w];
    for (int e = tid; e < E; e += nt) sc[e] = sc[e] / tot;
  } else {
    for (int e = tid; e < E; e += nt) sc[e] = 1.f / (1.f + expf(-sc[e]));
  }
  for (int e = tid; e < E16; e += nt)      // the padded tail never outranks a real key
    key[e] = e >= E ? -INFINITY : (a.bias ? sc[e] + key[e] : sc[e]);
  __syncthreads();
  if (a.grouped) {
    const int gsize = E / a.G;
    if (tid < a.G) {
      // four interleaved (first, second) pairs, merged at the end (max/min are exact)
      const float* src = a.bias ? key : sc;
      float b1[4], b2[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) b1[u] = b2[u] = -INFINITY;
      for (int e0 = tid * gsize; e0 < (tid + 1) * gsize; e0 += 4) {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float v = e0 + u < (tid + 1) * gsize ? src[e0 + u] : -INFINITY;
          b2[u] = fmaxf(b2[u], fminf(b1[u], v));
          b1[u] = fmaxf(b1[u], v);
        }
      }
#pragma unroll
      for (int u = 1; u < 4; ++u) {
        b2[0] = fmaxf(fmaxf(b2[0], b2[u]), fminf(b1[0], b1[u]));
        b1[0] = fmaxf(b1[0], b1[u]);
      }
      gsc[tid] = a.bias ? b1[0] + (b2[0] == -INFINITY ? 0.f : b2[0]) : b1[0];
    }
    __syncthreads();
    for (int e = tid; e < E; e += nt) {
      const int g = e / gsize;
      int rank = 0;
      for (int h = 0; h < a.G; ++h) rank += (gsc[h] > gsc[g] || (gsc[h] == gsc[g] && h < g));
      if (rank >= a.g) key[e] = -INFINITY;   // its group is not among the kept
    }
    __syncthreads();
  }
  for (int e = tid; e < E; e += nt) {
    const float ke = key[e];
    if (ke == -INFINITY) continue;
    int rank = 0;
    // sixteen keys per step, four 16-byte reads in flight; the outer loop stays rolled to
    // keep the code short
#pragma unroll 1
    for (int f0 = 0; f0 < E16 && rank < a.k; f0 += 16) {
      float4 kv[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) kv[q] = *reinterpret_cast<const float4*>(key + f0 + 4 * q);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int f = f0 + 4 * q;
        rank += (kv[q].x > ke || (kv[q].x == ke && f < e)) +
                (kv[q].y > ke || (kv[q].y == ke && f + 1 < e)) +
                (kv[q].z > ke || (kv[q].z == ke && f + 2 < e)) +
                (kv[q].w > ke || (kv[q].w == ke && f + 3 < e));
      }
    }
    if (rank < a.k) {
      oid[rank] = e;
      ow[rank] = sc[e];
    }
  }
  __syncthreads();
  int id = -1;
  if (tid < a.k) {
    float w = ow[tid];
    id = oid[tid];
    if (id < 0 || id >= E) {               // a rank left empty (non-finite logits)
      record_status(a.status, GBMOE_ERR_DEVICE_CHECK);
      id = 0;
      w = 0.f;
    }
    if (a.renorm) {
      float tot = 0.f;
      for (int j = 0; j < a.k; ++j) tot += ow[j];
      w = w / tot;
    }
    a.weights[(size_t)t * a.k + tid] = w * a.rsf;
    a.ids[(size_t)t * a.k + tid] = id;
  }
  __syncthreads();                         // the scratch is reused by the next token
  return id;
}

// Calls f.template operator()<EPT>() with EPT = ceil(E / 32) rounded up to a power of 2.
template <typename F>
__host__ void dispatch_ept(int E, F&& f) {
  if (E <= 32) f.template operator()<1>();
  else if (E <= 64) f.template operator()<2>();
  else if (E <= 128) f.template operator()<4>();
  else if (E <= 256) f.template operator()<8>();
  else if (E <= 512) f.template operator()<16>();
  else f.template operator()<32>();
}

inline TopkArgs make_topk_args(const gbmoe_config_t& c, int T, const float* logits,
                               const float* bias, float* weights, int* ids, int* status) {
  TopkArgs a;
  a.logits = logits;
  a.bias = bias;
  a.weights = weights;
  a.ids = ids;
  a.status = status;
  a.T = T;
  a.E = c.num_experts;
  a.k = c.top_k;
  a.renorm = c.renormalize != 0;
  a.grouped = c.use_grouped_topk != 0;
  a.G = a.grouped ? c.num_expert_group : 1;
  a.g = a.grouped ? c.topk_group : 1;
  a.sigmoid = c.scoring_func == GBMOE_SCORE_SIGMOID;
  a.rsf = c.routed_scaling_factor;
  a.logit_splits = 1;
  a.logit_split_stride = 0;
  a.zero = nullptr;
  a.zero_count = 0;
  return a;
}

}  // namespace gbmoe
