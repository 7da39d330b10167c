// Permute (dispatch) and combine.
//
// Permute is a scatter by slot staged through shared memory with the bulk-copy
// (TMA) engine: one thread per block streams its tokens through kPermBufs row
// buffers; each token row is loaded once (cp.async.bulk global->shared,
// completion on an mbarrier) and stored to each of its kept slots
// (cp.async.bulk shared->global).  HBM traffic is the algorithmic minimum: one
// read of every token that has a kept slot, one write per kept assignment.
//
// Narrow rows (a few KB) pay the bulk-copy engine's per-copy cost more than
// its bandwidth, so they are permuted by warps instead (permute_warp_kernel):
// one warp per (token, chunk of kPermChunk 16-byte vectors), each vector read
// once and written to every kept slot.
//
// Combine is a gather: one warp per (token, column chunk of kCombineChunk
// 16-byte vectors), 16-byte vector loads of the K expert-output rows, float32
// accumulation in k order, one vector store.  Chunks rather than whole tokens
// keep the work units small, so a persistent grid ends without a partial wave.
#pragma once

#include "common.cuh"

namespace moe {

constexpr int kPermBufs = 4;  // at most; fewer for very wide rows

struct PermuteParams {
  const uint8_t* x;      // [T, row_bytes]
  const int32_t* slot;   // [T, K]
  uint8_t* xp;           // [R, row_bytes]
  int64_t T;
  int K;
  uint32_t row_bytes;    // h * dtype size, a multiple of 16
  int nbuf;              // row buffers in shared memory, 1..kPermBufs
};

__global__ void __launch_bounds__(32) permute_bulk_kernel(PermuteParams p) {
  pdl_wait();
  extern __shared__ __align__(128) uint8_t sbuf[];  // [nbuf][row_bytes]
  __shared__ __align__(8) uint64_t bar[kPermBufs];
  if (threadIdx.x != 0) return;
  const int nbuf = p.nbuf;
  for (int b = 0; b < nbuf; ++b) mbar_init(&bar[b], 1);
  fence_mbar_init();

  int64_t cursor = blockIdx.x;
  // Next token of this block with at least one kept slot, or -1.
  auto next_token = [&]() -> int64_t {
    while (cursor < p.T) {
      const int64_t t = cursor;
      cursor += gridDim.x;
      for (int k = 0; k < p.K; ++k)
        if (p.slot[t * p.K + k] >= 0) return t;
    }
    return -1;
  };
  auto issue_load = [&](int b, int64_t t) {
    mbar_expect_tx(&bar[b], p.row_bytes);
    bulk_g2s(sbuf + (size_t)b * p.row_bytes, p.x + t * p.row_bytes, p.row_bytes, &bar[b]);
  };

  int64_t tok[kPermBufs];
  uint32_t phase = 0;  // bit b: parity to wait for on buffer b
  for (int b = 0; b < nbuf; ++b) {
    tok[b] = next_token();
    if (tok[b] >= 0) issue_load(b, tok[b]);
  }
  bool ok = true;
  for (int b = 0; tok[b] >= 0; b = (b + 1) % nbuf) {
    if (!mbar_wait(&bar[b], (phase >> b) & 1u)) {
      raise_error(kErrTimeout);
      ok = false;
      break;
    }
    phase ^= 1u << b;
    const uint8_t* src = sbuf + (size_t)b * p.row_bytes;
    const int64_t t = tok[b];
    for (int k = 0; k < p.K; ++k) {
      const int32_t s = p.slot[t * p.K + k];
      if (s >= 0) bulk_s2g(p.xp + (int64_t)s * p.row_bytes, src, p.row_bytes);
    }
    bulk_commit();
    bulk_wait_read<0>();  // the stores have read the buffer: refill it
    tok[b] = next_token();
    if (tok[b] >= 0) issue_load(b, tok[b]);
  }
  if (!ok) {
    // Let loads still in flight land before the block's shared memory is released.
    for (int b = 0; b < nbuf; ++b)
      if (tok[b] >= 0) mbar_wait(&bar[b], (phase >> b) & 1u);
  }
  bulk_wait_all<0>();
}

// Permutation by warps over (token, column chunk) units on a persistent grid:
// row_vecs 16-byte vectors per row; a unit's vectors are read once and stored
// to each of the token's kept slots.
constexpr int kPermChunk = 128;  // 16-byte vectors per work unit (4 per lane)

template <int KMAX>
__global__ void __launch_bounds__(256) permute_warp_kernel(const uint4* x, const int32_t* slot, int64_t T, int K,
                                                           int row_vecs, uint4* xp) {
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  const int chunks = (row_vecs + kPermChunk - 1) / kPermChunk;
  const int64_t units = T * chunks;
  for (int64_t u = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); u < units; u += warps) {
    const int64_t t = u / chunks;
    const int c0 = (int)(u - t * chunks) * kPermChunk;
    const int c1 = min(row_vecs, c0 + kPermChunk);
    const int32_t s_l = lane < K ? slot[t * K + lane] : -1;
    int32_t s[KMAX];
    bool any = false;
#pragma unroll
    for (int k = 0; k < KMAX; ++k) {
      s[k] = __shfl_sync(0xffffffffu, s_l, k);
      any |= k < K && s[k] >= 0;
    }
    if (!any) continue;  // uniform: every assignment of the token was dropped
    const uint4* src = x + t * row_vecs;
    for (int c = c0 + lane; c < c1; c += 32) {
      const uint4 v = __ldg(src + c);
#pragma unroll
      for (int k = 0; k < KMAX; ++k)
        if (k < K && s[k] >= 0) xp[(int64_t)s[k] * row_vecs + c] = v;
    }
  }
}

// Zero the pad rows (row_src == -1) of a padded permuted buffer.
__global__ void zero_pad_rows_kernel(const int32_t* row_src, int64_t R, uint32_t row_vecs, uint4* xp) {
  pdl_wait();
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int64_t n = R * row_vecs;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
    const int64_t r = i / row_vecs;
    if (row_src[r] < 0) xp[i] = make_uint4(0, 0, 0, 0);
  }
}

struct CombineParams {
  const void* yp;        // [R, h]
  const int32_t* slot;   // [T, K]
  const float* w;        // [T, K]
  const void* ys;        // [T, h] per-token term added first (shared expert), or null
  void* y;               // [T, h]
  int64_t T;
  int K, h;
};

template <typename T>
struct Vec;  // 16-byte vector of T
template <>
struct Vec<float> {
  static constexpr int N = 4;
};
template <>
struct Vec<__nv_bfloat16> {
  static constexpr int N = 8;
};

__device__ __forceinline__ void unpack(const uint4& v, float* f, float) {
  f[0] = __uint_as_float(v.x);
  f[1] = __uint_as_float(v.y);
  f[2] = __uint_as_float(v.z);
  f[3] = __uint_as_float(v.w);
}
__device__ __forceinline__ void unpack(const uint4& v, float* f, __nv_bfloat16) {
  const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(u[i] << 16);
    f[2 * i + 1] = __uint_as_float(u[i] & 0xffff0000u);
  }
}
__device__ __forceinline__ uint4 pack(const float* f, float) {
  return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]), __float_as_uint(f[3]));
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}
__device__ __forceinline__ uint4 pack(const float* f, __nv_bfloat16) {
  return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                    pack_bf16x2(f[6], f[7]));
}

constexpr int kCombineChunk = 128;  // 16-byte vectors per work unit (4 per lane)

template <typename T, int KMAX>
__global__ void __launch_bounds__(256) combine_kernel(CombineParams p) {
  pdl_wait();
  constexpr int V = Vec<T>::N;
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  const int vecs = p.h / V;
  const int chunks = (vecs + kCombineChunk - 1) / kCombineChunk;
  const int64_t units = p.T * chunks;
  for (int64_t u = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); u < units; u += warps) {
    const int64_t t = u / chunks;
    const int c0 = (int)(u - t * chunks) * kCombineChunk;
    const int c1 = min(vecs, c0 + kCombineChunk);
    int32_t s_l = -1;
    float w_l = 0.0f;
    if (lane < p.K) {
      s_l = p.slot[t * p.K + lane];
      w_l = p.w[t * p.K + lane];
    }
    int32_t s[KMAX];
    float wk[KMAX];
#pragma unroll
    for (int k = 0; k < KMAX; ++k) {
      s[k] = __shfl_sync(0xffffffffu, s_l, k);
      wk[k] = __shfl_sync(0xffffffffu, w_l, k);
    }
    const uint4* src = static_cast<const uint4*>(p.yp);
    uint4* dst = static_cast<uint4*>(p.y) + t * vecs;
    for (int c = c0 + lane; c < c1; c += 32) {
      uint4 v[KMAX];
#pragma unroll
      for (int k = 0; k < KMAX; ++k)
        if (k < p.K && s[k] >= 0) v[k] = __ldg(src + (int64_t)s[k] * vecs + c);
      float acc[V];
      if (p.ys != nullptr) {
        unpack(__ldg(static_cast<const uint4*>(p.ys) + t * vecs + c), acc, T());
      } else {
#pragma unroll
        for (int i = 0; i < V; ++i) acc[i] = 0.0f;
      }
#pragma unroll
      for (int k = 0; k < KMAX; ++k) {
        if (k < p.K && s[k] >= 0) {
          float f[V];
          unpack(v[k], f, T());
#pragma unroll
          for (int i = 0; i < V; ++i) acc[i] = fmaf(wk[k], f[i], acc[i]);
        }
      }
      dst[c] = pack(acc, T());
    }
  }
}

}  // namespace moe
