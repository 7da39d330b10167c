// Device side of the seeded input generator (see synth/__init__.py for the
// definition).  Fills whole tensors, or contiguous slices of them, in device
// memory so that multi-gigabyte expert weights never cross the PCIe bus.
// Every operation is exact or a single IEEE-rounded step, so the device values
// equal the host values bit for bit.
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace {

constexpr uint64_t kGamma = 0x9E3779B97F4A7C15ull;
constexpr uint64_t kM1 = 0xBF58476D1CE4E5B9ull;
constexpr uint64_t kM2 = 0x94D049BB133111EBull;
constexpr uint64_t kField = (1ull << 21) - 1;
constexpr int64_t kBias = 6 * (int64_t)kField;

__host__ __device__ __forceinline__ uint64_t mix64(uint64_t z) {
  z ^= z >> 30;
  z *= kM1;
  z ^= z >> 27;
  z *= kM2;
  return z ^ (z >> 31);
}

__device__ __forceinline__ uint64_t word(uint64_t key, int64_t i, int j) {
  return mix64(key + ((uint64_t)i * 4ull + (uint64_t)(j + 1)) * kGamma);
}

__device__ __forceinline__ float normal_f32(uint64_t key, int64_t i, float sigma) {
  int64_t s = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    uint64_t w = word(key, i, j);
    s += (int64_t)(w & kField) + (int64_t)((w >> 21) & kField) + (int64_t)((w >> 42) & kField);
  }
  float n = __fmul_rn((float)(s - kBias), 0x1p-21f);  // both factors exact: product exact
  return __fmul_rn(n, sigma);
}

__global__ void fill_normal_kernel(void* dst, int64_t n, int is_bf16, uint64_t key,
                                   int64_t start, float sigma) {
  int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
    float v = normal_f32(key, start + i, sigma);
    if (is_bf16)
      reinterpret_cast<__nv_bfloat16*>(dst)[i] = __float2bfloat16_rn(v);
    else
      reinterpret_cast<float*>(dst)[i] = v;
  }
}

__global__ void fill_uniform_kernel(float* dst, int64_t n, uint64_t key, double lo, double width) {
  int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
    uint64_t w = word(key, i, 0);
    double t = ((double)(w >> 40) + 0.5) * 0x1p-24;   // exact
    dst[i] = __double2float_rn(__dadd_rn(lo, __dmul_rn(width, t)));
  }
}

uint64_t tensor_key(uint64_t seed, uint64_t tensor_id) { return mix64(seed * kGamma + tensor_id); }

int grid_for(int64_t n) {
  int64_t b = (n + 255) / 256;
  return (int)(b < 148 * 16 ? (b < 1 ? 1 : b) : 148 * 16);
}

}  // namespace

extern "C" {

// Fill dst[0..n) with normal draws of elements start..start+n-1 of tensor
// (seed, tensor_id), scaled by sigma; dtype 0 = float32, 1 = bfloat16.
// Returns 0 or the cudaError_t of the launch.
int synth_fill_normal(void* dst, int64_t n, int dtype, uint64_t seed, uint64_t tensor_id,
                      int64_t start, float sigma, void* stream) {
  if (n <= 0) return 0;
  fill_normal_kernel<<<grid_for(n), 256, 0, (cudaStream_t)stream>>>(
      dst, n, dtype == 1, tensor_key(seed, tensor_id), start, sigma);
  return (int)cudaGetLastError();
}

// Fill dst[0..n) (float32) with uniform draws on [lo, lo + width).
int synth_fill_uniform(float* dst, int64_t n, uint64_t seed, uint64_t tensor_id, double lo,
                       double width, void* stream) {
  if (n <= 0) return 0;
  fill_uniform_kernel<<<grid_for(n), 256, 0, (cudaStream_t)stream>>>(
      dst, n, tensor_key(seed, tensor_id), lo, width);
  return (int)cudaGetLastError();
}

}  // extern "C"
