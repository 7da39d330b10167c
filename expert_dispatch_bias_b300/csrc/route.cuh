// Top-K routing: one warp per token.
//
// Scores, selection keys, group limit, top-K and combine weights as defined in
// the header (moe_route).  Scores are evaluated in float64 so that the float32
// keys are the correctly rounded values of the mathematical ones; the keys then
// decide the selection through exact float32 comparisons and adds only.
#pragma once

#include <math.h>

#include "common.cuh"

namespace moe {

constexpr int kRouteWarps = 8;      // tokens per block
constexpr int kMaxGroupTopn = 8;

struct RouteParams {
  const float* logits;  // [T, E]
  const float* bias;    // [E] or null
  int32_t* ids;         // [T, K]
  float* w;             // [T, K]
  int T, E, K;
  int sigmoid;          // 0 softmax, 1 sigmoid
  int renorm;
  float scale;
  int n_groups, topk_groups, group_topn;
  int key_is_logit;     // softmax without bias and without groups
};

// Total order of candidates: larger key first, then lower expert id.
__device__ __forceinline__ bool beats(float ka, int a, float kb, int b) {
  return ka > kb || (ka == kb && a < b);
}

// PER = experts held by each lane (contiguous: lane l holds l*PER .. l*PER+PER-1).
template <int PER>
__global__ void __launch_bounds__(kRouteWarps * 32) route_kernel(RouteParams p) {
  extern __shared__ float s_keys[];  // [kRouteWarps][E], used with a group limit
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * kRouteWarps + warp;
  if (t >= p.T) return;  // uniform across the warp
  const unsigned full = 0xffffffffu;
  const float* L = p.logits + (size_t)t * p.E;
  constexpr int NONE = 0x7fffffff;

  float lg[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int e = lane * PER + i;
    lg[i] = e < p.E ? L[e] : -INFINITY;
  }

  // ---- scores (float64)
  double s[PER];
  if (!p.sigmoid) {
    float m = -INFINITY;
#pragma unroll
    for (int i = 0; i < PER; ++i) m = fmaxf(m, lg[i]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(full, m, o));
    double z = 0.0;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const int e = lane * PER + i;
      s[i] = e < p.E ? exp((double)lg[i] - (double)m) : 0.0;
      z += s[i];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(full, z, o);
#pragma unroll
    for (int i = 0; i < PER; ++i) s[i] = s[i] / z;
  } else {
#pragma unroll
    for (int i = 0; i < PER; ++i) s[i] = 1.0 / (1.0 + exp(-(double)lg[i]));
  }

  // ---- selection keys
  float key[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int e = lane * PER + i;
    if (p.key_is_logit) {
      key[i] = lg[i];
    } else {
      const double b = (p.bias != nullptr && e < p.E) ? (double)p.bias[e] : 0.0;
      key[i] = (float)(s[i] + b);
    }
  }

  // ---- group limit: bit g of gmask set iff group g is allowed
  uint32_t gmask = full;
  int gsize = p.E;
  if (p.n_groups > 0) {
    float* kk = s_keys + warp * p.E;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const int e = lane * PER + i;
      if (e < p.E) kk[e] = key[i];
    }
    __syncwarp();
    gsize = p.E / p.n_groups;
    float gscore = -INFINITY;
    if (lane < p.n_groups) {
      float top[kMaxGroupTopn];
#pragma unroll
      for (int j = 0; j < kMaxGroupTopn; ++j) top[j] = -INFINITY;
      for (int m = 0; m < gsize; ++m) {  // insertion into a descending list
        float v = kk[lane * gsize + m];
#pragma unroll
        for (int j = 0; j < kMaxGroupTopn; ++j) {
          if (j < p.group_topn && v > top[j]) {
            const float tmp = top[j];
            top[j] = v;
            v = tmp;
          }
        }
      }
      float acc = 0.0f;
#pragma unroll
      for (int j = 0; j < kMaxGroupTopn; ++j)
        if (j < p.group_topn) acc = __fadd_rn(acc, top[j]);
      gscore = acc;
    }
    int rank = 0;
    for (int g = 0; g < p.n_groups; ++g) {
      const float v = __shfl_sync(full, gscore, g);
      if (beats(v, g, gscore, lane)) ++rank;
    }
    gmask = __ballot_sync(full, lane < p.n_groups && rank < p.topk_groups);
  }

  // ---- top-K by repeated warp arg-max
  bool avail[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int e = lane * PER + i;
    avail[i] = e < p.E && ((gmask >> (e / gsize)) & 1u);
  }
  int my_id = 0;
  for (int k = 0; k < p.K; ++k) {
    float bk = -INFINITY;
    int bi = NONE;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const int e = lane * PER + i;
      if (avail[i] && (bi == NONE || beats(key[i], e, bk, bi))) {
        bk = key[i];
        bi = e;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ok = __shfl_xor_sync(full, bk, o);
      const int oi = __shfl_xor_sync(full, bi, o);
      if (oi != NONE && (bi == NONE || beats(ok, oi, bk, bi))) {
        bk = ok;
        bi = oi;
      }
    }
#pragma unroll
    for (int i = 0; i < PER; ++i)
      if (lane * PER + i == bi) avail[i] = false;
    if (lane == k) my_id = bi;
  }

  // ---- weights from the unbiased scores of the chosen experts (float64)
  const int src = lane < p.K ? my_id / PER : 0;
  const int slot = my_id % PER;
  double mys = 0.0;
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const double v = __shfl_sync(full, s[i], src);
    if (i == slot) mys = v;
  }
  if (lane >= p.K) mys = 0.0;
  double tot = mys;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(full, tot, o);
  if (lane < p.K) {
    const double wk = p.renorm ? (mys / tot) : mys;
    p.ids[(size_t)t * p.K + lane] = my_id;
    p.w[(size_t)t * p.K + lane] = (float)(wk * (double)p.scale);
  }
}

}  // namespace moe
