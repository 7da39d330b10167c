// FP8 (E4M3) row quantisation for the FP8 experts: one float32 scale per row,
// scale = amax / 448 (1 for an all-zero row), code = E4M3(v / scale) rounded to
// nearest even with saturation; both divisions are IEEE float32 divisions so
// every code is decided exactly as the definition states.
//
//   quant_rows_kernel      rows of a [rows, cols] tensor (weights offline, the
//                          bf16 SwiGLU intermediate before the down projection);
//   quant_permute_kernel   the permutation fused with the quantisation of x:
//                          one warp per token reads its row, quantises it once
//                          and writes the codes and scale to every kept slot.
#pragma once

#include <cuda_fp8.h>

#include "common.cuh"

namespace moe {

constexpr float kE4M3Max = 448.0f;

template <typename T>
__device__ __forceinline__ void load8(const T* p, float* f);
template <>
__device__ __forceinline__ void load8<__nv_bfloat16>(const __nv_bfloat16* p, float* f) {
  const uint4 v = *reinterpret_cast<const uint4*>(p);
  const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(u[i] << 16);
    f[2 * i + 1] = __uint_as_float(u[i] & 0xffff0000u);
  }
}
template <>
__device__ __forceinline__ void load8<float>(const float* p, float* f) {
  const float4 a = *reinterpret_cast<const float4*>(p), b = *reinterpret_cast<const float4*>(p + 4);
  f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
  f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
}

__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d, float scale) {
  const uint32_t q0 = __nv_cvt_float_to_fp8(__fdiv_rn(a, scale), __NV_SATFINITE, __NV_E4M3);
  const uint32_t q1 = __nv_cvt_float_to_fp8(__fdiv_rn(b, scale), __NV_SATFINITE, __NV_E4M3);
  const uint32_t q2 = __nv_cvt_float_to_fp8(__fdiv_rn(c, scale), __NV_SATFINITE, __NV_E4M3);
  const uint32_t q3 = __nv_cvt_float_to_fp8(__fdiv_rn(d, scale), __NV_SATFINITE, __NV_E4M3);
  return q0 | (q1 << 8) | (q2 << 16) | (q3 << 24);
}

// Quantises one row of `cols` values (cols % 16 == 0, 16-byte aligned) held by
// this warp into 16-byte stores of codes; returns the scale.
template <typename T>
__device__ __forceinline__ float quant_row_warp(const T* src, int cols, uint8_t* const* dst, int n_dst) {
  const int lane = threadIdx.x & 31;
  float amax = 0.0f;
  for (int c = lane * 8; c < cols; c += 32 * 8) {
    float f[8];
    load8<T>(src + c, f);
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(f[i]));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const float scale = amax > 0.0f ? __fdiv_rn(amax, kE4M3Max) : 1.0f;
  for (int c = lane * 16; c < cols; c += 32 * 16) {
    float f[16];
    load8<T>(src + c, f);
    load8<T>(src + c + 8, f + 8);
    const uint4 q = make_uint4(e4m3x4(f[0], f[1], f[2], f[3], scale), e4m3x4(f[4], f[5], f[6], f[7], scale),
                               e4m3x4(f[8], f[9], f[10], f[11], scale), e4m3x4(f[12], f[13], f[14], f[15], scale));
    for (int d = 0; d < n_dst; ++d) *reinterpret_cast<uint4*>(dst[d] + c) = q;
  }
  return scale;
}

// One warp per row: codes[r, :] and scales[r] of src[r, :].
template <typename T>
__global__ void __launch_bounds__(256) quant_rows_kernel(const T* src, int64_t rows, int cols, uint8_t* codes,
                                                         float* scales) {
  pdl_wait();
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t r = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < rows; r += warps) {
    uint8_t* dst = codes + r * cols;
    const float s = quant_row_warp<T>(src + r * cols, cols, &dst, 1);
    if ((threadIdx.x & 31) == 0) scales[r] = s;
  }
}

// One warp per token t: quantise x[t] and write its codes and scale to every
// kept permuted row slot[t, k] >= 0 (xq [R, h] codes, sx [R] scales).
template <typename T>
__global__ void __launch_bounds__(256) quant_permute_kernel(const T* x, const int32_t* slot, int64_t T_, int K,
                                                            int h, uint8_t* xq, float* sx) {
  pdl_wait();
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  const int lane = threadIdx.x & 31;
  for (int64_t t = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); t < T_; t += warps) {
    uint8_t* dst[16];
    int n = 0;
    int32_t s_mine = lane < K ? slot[t * K + lane] : -1;
    for (int k = 0; k < K; ++k) {
      const int32_t s = __shfl_sync(0xffffffffu, s_mine, k);
      if (s >= 0) dst[n++] = xq + (int64_t)s * h;
    }
    if (n == 0) continue;  // uniform: every assignment of the token was dropped
    const float scale = quant_row_warp<T>(x + t * h, h, dst, n);
    if (lane < K && s_mine >= 0) sx[s_mine] = scale;
  }
}

}  // namespace moe
