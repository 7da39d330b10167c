// Shared device helpers: the sticky error word, bounded waits, mbarrier and
// bulk-copy (TMA) wrappers written as inline PTX for sm_103a.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace moe {

enum : uint32_t {
  kErrTimeout = 1u,    // a bounded spin on a flag or mbarrier ran out
  kErrBadIndex = 2u,   // an expert id outside [0, E)
};

// Sticky per-device error word, read and cleared by moe_check().
__device__ uint32_t g_dev_error;

// Upper bound of any device-side wait, in nanoseconds of %globaltimer.
constexpr uint64_t kWaitLimitNs = 1000000000ull;

__device__ __forceinline__ void raise_error(uint32_t bits) { atomicOr(&g_dev_error, bits); }

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint32_t lane_id() { return threadIdx.x & 31u; }

// ------------------------------------------------------------------ programmatic dependent launch
// Every kernel of the library is launched with programmatic stream
// serialisation (launch_k): the stream's next kernel is scheduled as soon as
// this one's CTAs have exited, before the kernel as a whole has completed and
// flushed, which hides the launch latency between the step's kernels.
// pdl_wait() returns once the previous kernel has completed and its writes are
// visible, so each kernel calls it before its first access to global memory:
// the order of memory accesses is the stream order.  No kernel triggers its
// dependents early: with early triggers the next kernel's CTAs wait resident
// on the SMs, and on a power-capped GPU the tensor-heavy layers lost ≈1 %.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ------------------------------------------------------------------ mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// n arrivals at once.
__device__ __forceinline__ void mbar_arrive_n(uint64_t* bar, uint32_t n) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(n) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for the phase of `bar` with the given parity to complete.  Gives up
// after kWaitLimitNs or as soon as *abort becomes non-zero (if given); returns
// false then.  Never spins without bound.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity,
                                          volatile uint32_t* abort = nullptr) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (abort != nullptr && *abort) return false;
    if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
  }
}

// ------------------------------------------------------------------ bulk copies (TMA, non-tensor)
// global -> shared, completion counted on an mbarrier in bytes.  Both addresses
// 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* smem_dst, const void* gsrc, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(smem_dst)),
      "l"(gsrc), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// shared -> global, tracked by the issuing thread's bulk async-groups.
__device__ __forceinline__ void bulk_s2g(void* gdst, const void* smem_src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst),
               "r"(smem_u32(smem_src)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// Wait until at most N bulk groups still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// Wait until at most N bulk groups are incomplete.
template <int N>
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

// ------------------------------------------------------------------ loads/stores
__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_release_u32(uint32_t* p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T>
__device__ __forceinline__ T from_f32(float v);
template <>
__device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) { return __float2bfloat16_rn(v); }

// ------------------------------------------------------------------ block scan
// Exclusive prefix sum of n <= 4 * blockDim.x int32 values in shared memory
// (in place); returns the total.  All threads of the block must call it.
__device__ __forceinline__ int32_t block_exclusive_scan(int32_t* vals, int n, int32_t* scratch /*>= 33 ints*/) {
  const int tid = threadIdx.x;
  const int per = (n + blockDim.x - 1) / blockDim.x;
  const int lo = tid * per;
  int32_t local = 0;
  for (int i = 0; i < per; ++i)
    if (lo + i < n) local += vals[lo + i];
  // warp inclusive scan of local
  int32_t incl = local;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    int32_t o = __shfl_up_sync(0xffffffffu, incl, d);
    if ((int)lane_id() >= d) incl += o;
  }
  const int warp = tid >> 5, nwarps = (blockDim.x + 31) >> 5;
  if (lane_id() == 31) scratch[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int32_t v = (int)lane_id() < nwarps ? scratch[lane_id()] : 0;
    int32_t s = v;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      int32_t o = __shfl_up_sync(0xffffffffu, s, d);
      if ((int)lane_id() >= d) s += o;
    }
    if ((int)lane_id() < nwarps) scratch[lane_id()] = s - v;  // exclusive warp offsets
    if (lane_id() == 31) scratch[32] = s;                      // block total (nwarps <= 32)
  }
  __syncthreads();
  int32_t run = scratch[warp] + incl - local;
  const int32_t total = scratch[32];
  for (int i = 0; i < per; ++i)
    if (lo + i < n) {
      int32_t v = vals[lo + i];
      vals[lo + i] = run;
      run += v;
    }
  __syncthreads();
  return total;
}

}  // namespace moe
