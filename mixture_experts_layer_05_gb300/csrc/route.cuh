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
  long long logit_split_stride;  // summed in copy order on load (split-K router GEMM)
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

// Routes token t with the calling warp; writes weights[t, :] and ids[t, :] and returns,
// in lane j < k, the j-th chosen expert (-1 in the other lanes).
template <int EPT>
__device__ __forceinline__ int route_token_warp(const TopkArgs& a, int t, int lane) {
  const int gsize = a.grouped ? a.E / a.G : a.E;
  int grp[EPT];
#pragma unroll
  for (int i = 0; i < EPT; ++i) grp[i] = (lane + 32 * i) / gsize;
  const float* row = a.logits + (size_t)t * a.E;
  float s[EPT], q[EPT];
  float mx = -INFINITY;
#pragma unroll
  for (int i = 0; i < EPT; ++i) {
    const int e = lane + 32 * i;
    float l = -INFINITY;
    if (e < a.E) {
      l = __ldg(row + e);
      for (int sp = 1; sp < a.logit_splits; ++sp) l += __ldg(row + sp * a.logit_split_stride + e);
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
    q[i] = e < a.E ? (a.bias ? s[i] + __ldg(a.bias + e) : s[i]) : -INFINITY;
  }
  // 3. group filter
  uint32_t kept = 0xffffffffu;
  if (a.grouped) {
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
  // 4. top-k over the surviving experts
  uint32_t taken = 0u;
  float my_w = 0.f;
  int my_id = -1;
  for (int j = 0; j < a.k; ++j) {
    float bq = -INFINITY;
    int be = INT_MAX;
#pragma unroll
    for (int i = 0; i < EPT; ++i) {
      const int e = lane + 32 * i;
      if (e < a.E && !((taken >> i) & 1u) && ((kept >> grp[i]) & 1u)) {
        if (q[i] > bq || (q[i] == bq && e < be)) {
          bq = q[i];
          be = e;
        }
      }
    }
    warp_argmax(bq, be);
    float sv = 0.f;
    if (be == INT_MAX) {
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
  return a;
}

}  // namespace gbmoe
