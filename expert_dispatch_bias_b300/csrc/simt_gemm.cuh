// CUDA-core (SIMT) GEMMs with float32 accumulation, for the float32 layer (a
// TF32 tensor-core product would miss a 1e-4 relative tolerance) and for the
// router logits.  C[m, n] = sum_k A[m, k] * B[n, k]: both operands K-major.
//
// Rows of A come either from one dense block of M rows or from ragged expert
// segments [offsets[e], offsets[e] + kept[e]); B is expert e's weight matrix.
// Epilogues: plain store, SwiGLU (gate columns n and up columns I + n of the
// same expert, out = silu(gate) * up), or float32 logits plus a per-column
// offset.
#pragma once

#include <math.h>

#include "common.cuh"

namespace moe {

constexpr int kSimtBM = 64, kSimtBN = 64, kSimtBK = 16, kSimtThreads = 256;

enum SimtMode { kSimtPlain = 0, kSimtSwiglu = 1, kSimtLogits = 2 };

struct SimtParams {
  const void* A;
  int64_t lda;              // elements
  const void* B;
  int64_t ldb;              // elements
  int64_t b_expert_rows;    // rows of B per expert (2I for gate/up, h for down)
  int64_t up_rows;          // row offset of the up half (I) for SwiGLU
  void* C;
  int64_t ldc;
  const int32_t* offsets;   // [E+1] or null (dense A of M rows)
  const int32_t* kept;      // [E]
  int E;
  int M, N, K;
  const float* col_bias;    // logits offset [N] or null
  const int32_t* w_map;     // segment -> its B matrix, or null: segment e uses B_e
  int n_w;                  // B matrices available (bounds w_map's entries)
};

// Loads 4 consecutive K-elements of a row as floats (zeros when out of range).
template <typename T>
__device__ __forceinline__ void load4(const T* row, int k, bool valid, float* out);
template <>
__device__ __forceinline__ void load4<float>(const float* row, int k, bool valid, float* out) {
  float4 v = valid ? *reinterpret_cast<const float4*>(row + k) : make_float4(0.f, 0.f, 0.f, 0.f);
  out[0] = v.x;
  out[1] = v.y;
  out[2] = v.z;
  out[3] = v.w;
}
template <>
__device__ __forceinline__ void load4<__nv_bfloat16>(const __nv_bfloat16* row, int k, bool valid, float* out) {
  uint2 v = valid ? *reinterpret_cast<const uint2*>(row + k) : make_uint2(0, 0);
  out[0] = __uint_as_float(v.x << 16);
  out[1] = __uint_as_float(v.x & 0xffff0000u);
  out[2] = __uint_as_float(v.y << 16);
  out[3] = __uint_as_float(v.y & 0xffff0000u);
}

// Finds the expert and first row of m-block `mb` (blocks of kSimtBM rows per
// expert segment).  Returns false if mb is past the last block.
__device__ __forceinline__ bool segment_of_block(const int32_t* offsets, const int32_t* kept, int E, int mb,
                                                 int* e_out, int* row0, int* rows) {
  __shared__ int32_t pre[1025];
  __shared__ int32_t scratch[33];
  for (int e = threadIdx.x; e < E; e += blockDim.x) pre[e] = (kept[e] + kSimtBM - 1) / kSimtBM;
  __syncthreads();
  const int32_t total = block_exclusive_scan(pre, E, scratch);
  if (mb >= total) return false;
  // The block lies in the last expert whose prefix is <= mb: that expert's
  // segment is non-empty because the next prefix is > mb.
  int lo = 0, hi = E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (pre[mid] <= mb) lo = mid; else hi = mid - 1;
  }
  const int e = lo;
  const int j = mb - pre[e];
  *e_out = e;
  *row0 = offsets[e] + j * kSimtBM;
  *rows = min(kSimtBM, kept[e] - j * kSimtBM);
  return true;
}

template <typename T, int MODE>
__global__ void __launch_bounds__(kSimtThreads) simt_gemm_kernel(SimtParams p) {
  pdl_wait();
  constexpr int NB = MODE == kSimtSwiglu ? 2 * kSimtBN : kSimtBN;  // B rows per tile
  __shared__ __align__(16) float As[kSimtBK][kSimtBM];
  __shared__ __align__(16) float Bs[kSimtBK][NB];
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;

  int e = 0, row0, rows;
  if (p.offsets == nullptr) {
    row0 = blockIdx.y * kSimtBM;
    rows = min(kSimtBM, p.M - row0);
    if (rows <= 0) return;
  } else if (!segment_of_block(p.offsets, p.kept, p.E, blockIdx.y, &e, &row0, &rows)) {
    return;
  }
  const int n0 = blockIdx.x * kSimtBN;
  const T* A = static_cast<const T*>(p.A);
  const int we = p.w_map != nullptr ? p.w_map[e] : e;
  if (we < 0 || (p.w_map != nullptr && we >= p.n_w)) {  // uniform across the block
    if (threadIdx.x == 0) raise_error(kErrBadIndex);
    return;
  }
  const T* B = static_cast<const T*>(p.B) + (int64_t)we * p.b_expert_rows * p.ldb;

  float acc[4][4] = {};
  float acc_up[4][4] = {};

  const int lr = tid >> 2, lk = (tid & 3) * 4;  // loader: row, k offset
  for (int k0 = 0; k0 < p.K; k0 += kSimtBK) {
    float v[4];
    load4<T>(A + (int64_t)(row0 + lr) * p.lda, k0 + lk, lr < rows && k0 + lk < p.K, v);
#pragma unroll
    for (int i = 0; i < 4; ++i) As[lk + i][lr] = v[i];
#pragma unroll
    for (int part = 0; part < NB / kSimtBN; ++part) {
      const int n = n0 + lr;
      const int64_t brow = (part == 0 ? 0 : p.up_rows) + n;
      load4<T>(B + brow * p.ldb, k0 + lk, n < p.N && k0 + lk < p.K, v);
#pragma unroll
      for (int i = 0; i < 4; ++i) Bs[lk + i][part * kSimtBN + lr] = v[i];
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < kSimtBK; ++kk) {
      const float4 a = *reinterpret_cast<const float4*>(&As[kk][ty * 4]);
      const float4 b = *reinterpret_cast<const float4*>(&Bs[kk][tx * 4]);
      const float av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
      if (MODE == kSimtSwiglu) {
        const float4 u = *reinterpret_cast<const float4*>(&Bs[kk][kSimtBN + tx * 4]);
        const float uv[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) acc_up[i][j] = fmaf(av[i], uv[j], acc_up[i][j]);
      }
    }
    __syncthreads();
  }

#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = ty * 4 + i;
    if (r >= rows) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tx * 4 + j;
      if (n >= p.N) continue;
      const int64_t off = (int64_t)(row0 + r) * p.ldc + n;
      if (MODE == kSimtLogits) {
        static_cast<float*>(p.C)[off] = acc[i][j] + (p.col_bias ? p.col_bias[n] : 0.0f);
      } else if (MODE == kSimtSwiglu) {
        const float g = acc[i][j];
        const float a = g / (1.0f + expf(-g)) * acc_up[i][j];
        static_cast<T*>(p.C)[off] = from_f32<T>(a);
      } else {
        static_cast<T*>(p.C)[off] = from_f32<T>(acc[i][j]);
      }
    }
  }
}

}  // namespace moe
