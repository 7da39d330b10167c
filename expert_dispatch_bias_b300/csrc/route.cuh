// Top-K routing: one warp per token selects, then the block's threads share
// the float64 weights of its chosen experts.
//
// Scores, selection keys, group limit, top-K and combine weights as defined in
// the header (moe_route).  Scores are evaluated in float64 so that the float32
// keys are the correctly rounded values of the mathematical ones; the keys then
// decide the selection through exact float32 comparisons and adds only.  The
// float64 pipe is narrow on this GPU, so the weights of a block's tokens are
// evaluated one (token, k) pair per thread rather than by K lanes of each
// token's warp: a quarter of the float64 instructions for K = 8.
#pragma once

#include <math.h>

#include "common.cuh"

namespace moe {

constexpr int kRouteWarps = 8;      // tokens per block
constexpr int kMaxGroupTopn = 8;
constexpr int kRouteMaxK = 16;
constexpr int kRefineMax = 64;      // experts whose keys one refinement step evaluates exactly

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

// Error bounds of the float32 sigmoid keys fl32(1/(1+expf(-x)) + b) against
// the exact keys fl32(sigmoid(x) + b): expf is within 2 ulp, the add and the
// division within half an ulp each, so the score is within 4 ulp of 1 (s <= 1)
// and the key within 4 + 1.2 ulp of 1 (|s + b| <= 1.1); 2^-20 (16 ulp of 1)
// bounds a key, 2n * 2^-20 a group score summed from n keys.
constexpr float kKeyErr = 9.5367431640625e-07f;  // 2^-20

struct RouteSel {
  int my_id;        // lane k < K: the k-th chosen expert
  float min_gap;    // smallest gap between adjacent keys of the K+1 best allowed
  float group_gap;  // gap between the last kept and the first dropped group score
  float kth1;       // key of the (K+1)-th best allowed expert (-inf: fewer allowed)
  uint32_t gmask;   // bit g: group g allowed (all ones without groups)
  int gsize;        // experts per group (E without groups)
};

// Groups that are power-of-two runs of whole lanes (lane l holds experts
// l*PER..) with a top-1 or top-2 group score: the shuffle form of the limit.
template <int PER>
__device__ __forceinline__ bool lane_groups(const RouteParams& p) {
  if (p.n_groups <= 0 || p.group_topn > 2) return false;
  const int gs = p.E / p.n_groups;
  return gs % PER == 0 && ((gs / PER) & (gs / PER - 1)) == 0;
}

// Group limit and top-K on the keys held by this warp (lane l: experts
// l*PER..), with the gaps that decide whether an approximation of the keys
// selects as the exact keys would.  kk: this warp's [E] shared row.
template <int PER>
__device__ __forceinline__ RouteSel route_select(const float* key, const RouteParams& p, float* kk) {
  const unsigned full = 0xffffffffu;
  const int lane = threadIdx.x & 31;
  constexpr int NONE = 0x7fffffff;
  RouteSel r;
  r.group_gap = INFINITY;

  // ---- group limit: bit g of gmask set iff group g is allowed
  uint32_t gmask = full;
  int gsize = p.E;
  if (lane_groups<PER>(p)) {
    // Each group is a power-of-two run of whole lanes: the two largest keys of
    // every lane, merged across the group's lanes by butterfly shuffles.  The
    // group score is the same float32 sum as the general path forms.
    gsize = p.E / p.n_groups;
    const int lanes_per_group = gsize / PER;
    float t1 = -INFINITY, t2 = -INFINITY;  // t1 >= t2
#pragma unroll
    for (int i = 0; i < PER; ++i) {  // NaN keys compare false and are skipped
      const float v = key[i];
      if (v > t2) {
        t2 = v > t1 ? t1 : v;
        t1 = fmaxf(t1, v);
      }
    }
    for (int o = 1; o < lanes_per_group; o <<= 1) {
      const float b1 = __shfl_xor_sync(full, t1, o), b2 = __shfl_xor_sync(full, t2, o);
      t2 = fmaxf(fminf(t1, b1), fmaxf(t2, b2));
      t1 = fmaxf(t1, b1);
    }
    const float mine = p.group_topn == 1 ? t1 : __fadd_rn(t1, t2);
    const float gscore = __shfl_sync(full, mine, (lane % p.n_groups) * lanes_per_group);
    int rank = 0;
    for (int g = 0; g < p.n_groups; ++g) {
      const float v = __shfl_sync(full, gscore, g);
      if (beats(v, g, gscore, lane)) ++rank;
    }
    const bool in = lane < p.n_groups;
    gmask = __ballot_sync(full, in && rank < p.topk_groups);
    if (p.topk_groups < p.n_groups) {
      const int la = __ffs(__ballot_sync(full, in && rank == p.topk_groups - 1)) - 1;
      const int lb = __ffs(__ballot_sync(full, in && rank == p.topk_groups)) - 1;
      r.group_gap = __shfl_sync(full, gscore, la) - __shfl_sync(full, gscore, lb);
    }
  } else if (p.n_groups > 0) {
    __syncwarp();
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
    const bool in = lane < p.n_groups;
    gmask = __ballot_sync(full, in && rank < p.topk_groups);
    if (p.topk_groups < p.n_groups) {
      const int la = __ffs(__ballot_sync(full, in && rank == p.topk_groups - 1)) - 1;
      const int lb = __ffs(__ballot_sync(full, in && rank == p.topk_groups)) - 1;
      r.group_gap = __shfl_sync(full, gscore, la) - __shfl_sync(full, gscore, lb);
    }
  }

  // ---- top-K.  Each lane sorts its allowed keys once (key descending, then
  // lower id); then K+1 rounds of a warp arg-max over the lanes' first keys,
  // the winning lane dropping its first key; the last round measures the gap
  // to the first expert left out.  Sorting once replaces a rescan of all PER
  // keys in every round.
  float sk[PER];
  int si[PER];
  {
    // the experts of a lane are PER consecutive ids: one group per lane when a
    // group holds whole lanes' runs, else a group per expert
    const int g0 = (lane * PER) / gsize;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const int e = lane * PER + i;
      const int g = (gsize % PER == 0) ? g0 : e / gsize;
      const bool ok = e < p.E && ((gmask >> g) & 1u);
      sk[i] = ok ? key[i] : -INFINITY;
      si[i] = ok ? e : NONE;
    }
  }
  // odd-even transposition sort; an allowed entry goes before a disallowed one
#pragma unroll
  for (int round = 0; round < PER; ++round) {
#pragma unroll
    for (int i = round & 1; i + 1 < PER; i += 2) {
      const bool swap = si[i + 1] != NONE && (si[i] == NONE || beats(sk[i + 1], si[i + 1], sk[i], si[i]));
      const float tk = swap ? sk[i + 1] : sk[i];
      const int ti = swap ? si[i + 1] : si[i];
      sk[i + 1] = swap ? sk[i] : sk[i + 1];
      si[i + 1] = swap ? si[i] : si[i + 1];
      sk[i] = tk;
      si[i] = ti;
    }
  }
  r.my_id = 0;
  r.min_gap = INFINITY;
  r.kth1 = -INFINITY;
  r.gmask = gmask;
  r.gsize = gsize;
  float prev = 0.0f;
  for (int k = 0; k <= p.K; ++k) {
    float bk = sk[0];
    int bi = si[0];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ok = __shfl_xor_sync(full, bk, o);
      const int oi = __shfl_xor_sync(full, bi, o);
      if (oi != NONE && (bi == NONE || beats(ok, oi, bk, bi))) {
        bk = ok;
        bi = oi;
      }
    }
    if (bi == NONE) break;  // fewer than K+1 experts allowed
    if (k > 0) r.min_gap = fminf(r.min_gap, prev - bk);
    prev = bk;
    if (k == p.K) {
      r.kth1 = bk;
      break;
    }
    if (si[0] == bi) {  // this lane held the winner: drop it
#pragma unroll
      for (int i = 0; i + 1 < PER; ++i) {
        sk[i] = sk[i + 1];
        si[i] = si[i + 1];
      }
      sk[PER - 1] = -INFINITY;
      si[PER - 1] = NONE;
    }
    if (lane == k) r.my_id = bi;
  }
  return r;
}

// Replaces key[i] by the exact sigmoid key fl32(sigmoid(x) + b), x and the
// sigmoid in float64, for every expert i of this lane with need[i] and not yet
// done[i]: the warp compacts those experts into `eids` and evaluates one per
// lane.  Returns false, changing nothing, when more than kRefineMax would be.
template <int PER>
__device__ __forceinline__ bool refine_keys(float* key, bool* done, const bool* need, const float* L,
                                            const RouteParams& p, int32_t* eids, float* vals) {
  const unsigned full = 0xffffffffu;
  const int lane = threadIdx.x & 31;
  const unsigned below = (1u << lane) - 1u;
  int n = 0;
#pragma unroll
  for (int i = 0; i < PER; ++i) n += __popc(__ballot_sync(full, need[i] && !done[i]));
  if (n > kRefineMax) return false;
  int base = 0;
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const bool f = need[i] && !done[i];
    const unsigned m = __ballot_sync(full, f);
    if (f) eids[base + __popc(m & below)] = lane * PER + i;
    base += __popc(m);
  }
  __syncwarp();
  for (int j = lane; j < n; j += 32) {
    const int e = eids[j];
    const double b = p.bias != nullptr ? (double)p.bias[e] : 0.0;
    vals[j] = (float)(1.0 / (1.0 + exp(-(double)L[e])) + b);
  }
  __syncwarp();
  base = 0;
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const bool f = need[i] && !done[i];
    const unsigned m = __ballot_sync(full, f);
    if (f) {
      key[i] = vals[base + __popc(m & below)];
      done[i] = true;
    }
    base += __popc(m);
  }
  __syncwarp();
  return true;
}

// Selection for token t by the calling warp: writes ids[t, :], the chosen
// logits to xs[0..K), and the softmax max and float64 denominator (when the
// weights need the full one) to *zs, *ms.
template <int PER>
__device__ __forceinline__ void route_token(const RouteParams& p, int t, float* kk, float* xs, double* zs,
                                            float* ms, int32_t* eids, float* vals) {
  const int lane = threadIdx.x & 31;
  const unsigned full = 0xffffffffu;
  const float* L = p.logits + (size_t)t * p.E;

  float lg[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int e = lane * PER + i;
    lg[i] = e < p.E ? L[e] : -INFINITY;
  }
  float m = -INFINITY;  // largest logit (softmax)
#pragma unroll
  for (int i = 0; i < PER; ++i) m = fmaxf(m, lg[i]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(full, m, o));

  // ---- selection keys.  Exact: the logit itself, or fl32(s + b) from
  // float64 scores.  The sigmoid keys are first taken in float32 (within
  // kKeyErr of the exact ones); the selection stands if every gap it depends
  // on exceeds twice the error, else it is redone on the exact keys.
  float key[PER];
  bool exact = true;
  double z = 0.0;  // softmax denominator (float64)
  if (p.key_is_logit) {
#pragma unroll
    for (int i = 0; i < PER; ++i) key[i] = lg[i];
  } else if (p.sigmoid) {
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const int e = lane * PER + i;
      const float b = (p.bias != nullptr && e < p.E) ? p.bias[e] : 0.0f;
      key[i] = e < p.E ? __fadd_rn(1.0f / (1.0f + expf(-lg[i])), b) : -INFINITY;
    }
    exact = false;
  } else {
    double s[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const int e = lane * PER + i;
      s[i] = e < p.E ? exp((double)lg[i] - (double)m) : 0.0;
      z += s[i];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(full, z, o);
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const int e = lane * PER + i;
      const double b = (p.bias != nullptr && e < p.E) ? (double)p.bias[e] : 0.0;
      key[i] = e < p.E ? (float)(s[i] / z + b) : -INFINITY;
    }
  }

  RouteSel sel = route_select<PER>(key, p, kk);
  if (!exact) {
    const float group_tol = 4.0f * (float)p.group_topn * kKeyErr;  // twice 2n * 2^-20
    const bool group_open = p.n_groups > 0 && !(sel.group_gap > group_tol);
    if (!(sel.min_gap > 2.0f * kKeyErr) || group_open) {
      // Refinement: keys within 3 kKeyErr of a threshold are made exact.  An
      // approximate key a (|a - exact| <= kKeyErr) below the n-th largest key
      // tau of its group by more than 2 kKeyErr has an exact key below the n
      // keys at or above tau, so the group score (sum of the n largest) is
      // exact once the keys at or above tau - 2 kKeyErr are; likewise the top
      // K+1 of the allowed experts lie at or above the (K+1)-th key minus
      // 2 kKeyErr.  Comparisons between an exact key and an approximate one
      // more than 2 kKeyErr apart are decided as between the exact keys, so
      // the selection on the refined keys is the selection on the exact keys.
      bool done[PER], need[PER];
#pragma unroll
      for (int i = 0; i < PER; ++i) done[i] = false;
      bool ok = p.n_groups == 0 || lane_groups<PER>(p);
      if (ok && group_open) {
        const int lanes_per_group = p.E / p.n_groups / PER;
        float t1 = -INFINITY, t2 = -INFINITY;  // this group's two largest keys
#pragma unroll
        for (int i = 0; i < PER; ++i) {
          const float v = key[i];
          if (v > t2) {
            t2 = v > t1 ? t1 : v;
            t1 = fmaxf(t1, v);
          }
        }
        for (int o = 1; o < lanes_per_group; o <<= 1) {
          const float b1 = __shfl_xor_sync(full, t1, o), b2 = __shfl_xor_sync(full, t2, o);
          t2 = fmaxf(fminf(t1, b1), fmaxf(t2, b2));
          t1 = fmaxf(t1, b1);
        }
        const float thr = (p.group_topn == 1 ? t1 : t2) - 3.0f * kKeyErr;
#pragma unroll
        for (int i = 0; i < PER; ++i) need[i] = lane * PER + i < p.E && key[i] >= thr;
        ok = refine_keys<PER>(key, done, need, L, p, eids, vals);
        if (ok) sel = route_select<PER>(key, p, kk);  // exact group limit
      }
      if (ok) {
        const float thr = sel.kth1 - 3.0f * kKeyErr;
#pragma unroll
        for (int i = 0; i < PER; ++i) {
          const int e = lane * PER + i;
          need[i] = e < p.E && ((sel.gmask >> (e / sel.gsize)) & 1u) && key[i] >= thr;
        }
        ok = refine_keys<PER>(key, done, need, L, p, eids, vals);
        if (ok) sel = route_select<PER>(key, p, kk);
      }
      if (!ok) {  // too many keys near a threshold: every key exactly
#pragma unroll
        for (int i = 0; i < PER; ++i) {
          const int e = lane * PER + i;
          const double b = (p.bias != nullptr && e < p.E) ? (double)p.bias[e] : 0.0;
          key[i] = e < p.E ? (float)(1.0 / (1.0 + exp(-(double)lg[i])) + b) : -INFINITY;
        }
        sel = route_select<PER>(key, p, kk);
      }
    }
  }

  if (!p.sigmoid && !p.renorm && p.key_is_logit) {  // the weights need the full denominator
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const int e = lane * PER + i;
      z += e < p.E ? exp((double)lg[i] - (double)m) : 0.0;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(full, z, o);
  }
  if (lane < p.K) {
    p.ids[(size_t)t * p.K + lane] = sel.my_id;
    xs[lane] = L[sel.my_id];
  }
  if (lane == 0) {
    *zs = z;
    *ms = m;
  }
}

// PER = experts held by each lane (contiguous: lane l holds l*PER .. l*PER+PER-1).
template <int PER>
__global__ void __launch_bounds__(kRouteWarps * 32, PER <= 8 ? 4 : 1) route_kernel(RouteParams p) {
  pdl_wait();
  extern __shared__ float s_keys[];  // [kRouteWarps][E], used with a group limit
  __shared__ int32_t s_eid[kRouteWarps][kRefineMax];  // experts being refined
  __shared__ float s_eval[kRouteWarps][kRefineMax];   // their exact keys
  __shared__ float s_x[kRouteWarps * kRouteMaxK];    // logits of the chosen experts
  __shared__ double s_s[kRouteWarps * kRouteMaxK];   // their float64 scores
  __shared__ double s_z[kRouteWarps];                // softmax denominators
  __shared__ float s_m[kRouteWarps];                 // largest logits
  const int warp = threadIdx.x >> 5;
  const int t0 = blockIdx.x * kRouteWarps;
  const int nt = min(kRouteWarps, p.T - t0);  // tokens of this block
  if (warp < nt)
    route_token<PER>(p, t0 + warp, s_keys + warp * p.E, s_x + warp * p.K, &s_z[warp], &s_m[warp], s_eid[warp],
                     s_eval[warp]);
  __syncthreads();

  // ---- weights from the unbiased float64 scores of the chosen experts, one
  // (token, k) pair per thread: pair j is token j / K, choice j % K.
  const int pairs = nt * p.K;
  if (p.K == 1 && p.renorm && p.key_is_logit) {
    // renormalised top-1 on the logits: the chosen expert holds the largest
    // logit, so its score is exp(0) = 1 and its weight exactly 1 * scale.  A
    // row whose chosen logit is not finite (NaN, or every logit -inf) gets NaN,
    // as s / s with s = exp(x - max) gives in the general path.
    for (int j = threadIdx.x; j < pairs; j += blockDim.x)
      p.w[(size_t)t0 + j] = isfinite(s_x[j]) ? p.scale : __int_as_float(0x7fffffff);
    return;
  }
  for (int j = threadIdx.x; j < pairs; j += blockDim.x) {
    const double x = (double)s_x[j];
    s_s[j] = p.sigmoid ? 1.0 / (1.0 + exp(-x)) : exp(x - (double)s_m[j / p.K]);
  }
  __syncthreads();
  for (int j = threadIdx.x; j < pairs; j += blockDim.x) {
    const int tl = j / p.K;
    const double* sc = s_s + tl * p.K;
    double tot = 0.0;
    for (int k = 0; k < p.K; ++k) tot += sc[k];
    const double wk = p.renorm ? (s_s[j] / tot) : (p.sigmoid ? s_s[j] : s_s[j] / s_z[tl]);
    p.w[(size_t)t0 * p.K + j] = (float)(wk * (double)p.scale);
  }
}

}  // namespace moe
