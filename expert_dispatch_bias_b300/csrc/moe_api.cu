// C ABI of the MoE-layer forward pass (declared in include/moe.h).
//
// One translation unit holds every kernel (the headers included below) so that
// the sticky device error word is a single symbol.  Host code here validates
// arguments, carves the caller's workspace, picks launch shapes and enqueues
// kernels on the caller's stream; it never allocates device memory and never
// synchronises except in moe_check.
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <utility>
#include <vector>

#include <cudaTypedefs.h>

#include "moe.h"
#include "common.cuh"
#include "layout.cuh"
#include "permute_combine.cuh"
#include "route.cuh"
#include "simt_gemm.cuh"
#include "tc_gemm.cuh"
#include "ffn_grouped.cuh"
#include "fp8.cuh"

using namespace moe;

// Look-back scratch of moe_dispatch_layout_static: a fixed array, so that the
// call needs no workspace from its caller.  Zero-initialised at module load.
static __device__ __align__(256) unsigned char g_layout_static_scratch[MOE_LAYOUT_STATIC_SCRATCH_BYTES];

namespace {

#define MOE_TRY(expr)                    \
  do {                                   \
    const moe_status st_ = (expr);       \
    if (st_ != MOE_OK) return st_;       \
  } while (0)

// Kernels this library has launched in the process (moe_launch_count).
std::atomic<uint64_t> g_launches{0};

// Called right after every kernel launch: counts it and returns the launch error.
inline cudaError_t launched() {
  g_launches.fetch_add(1, std::memory_order_relaxed);
  return cudaGetLastError();
}

// Launches a kernel of the library on st with programmatic stream
// serialisation: it is scheduled as soon as the stream's previous kernel has
// no CTA left, which hides the launch latency between the kernels of a step
// (Switch-Base step 0.386 -> 0.368 ms, decode T=32 1.791 -> 1.775 ms on B300).
// Every kernel waits for the previous one (pdl_wait, griddepcontrol.wait)
// before its first global memory access, so memory sees plain stream order.
// An error is also left for cudaGetLastError, which launched() reads.
template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, Args&&... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

#define CUDA_TRY(expr)                               \
  do {                                               \
    if ((expr) != cudaSuccess) {                     \
      (void)cudaGetLastError();                      \
      return MOE_ERR_CUDA;                           \
    }                                                \
  } while (0)

inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
inline int ds_of(const moe_config& c) { return c.dtype == MOE_F32 ? 4 : 2; }
// Experts after routing: the E logical experts plus the redundant replicas
// (expert-parallel load balancing); layout, permutation, FFN and combine
// work on these physical experts.
inline int nphys(const moe_config& c) { return c.E + c.n_redundant; }
inline int64_t rows_of(const moe_config& c) {
  return (c.pad && c.capacity > 0) ? (int64_t)nphys(c) * c.capacity : (int64_t)c.T * c.K;
}
inline cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }

moe_status validate(const moe_config* c) {
  if (c == nullptr) return MOE_ERR_INVALID_ARG;
  if (c->T < 0 || c->h <= 0 || c->h % 64 != 0 || c->I <= 0 || c->I % 64 != 0) return MOE_ERR_INVALID_ARG;
  if (c->E < 1 || c->E > 1024 || c->K < 1 || c->K > 16 || c->K > c->E) return MOE_ERR_INVALID_ARG;
  if (c->dtype != MOE_F32 && c->dtype != MOE_BF16) return MOE_ERR_INVALID_ARG;
  if (c->score != MOE_SOFTMAX && c->score != MOE_SIGMOID) return MOE_ERR_INVALID_ARG;
  if (c->renormalize != 0 && c->renormalize != 1) return MOE_ERR_INVALID_ARG;
  if (!isfinite(c->scale)) return MOE_ERR_INVALID_ARG;
  if (c->n_groups < 0) return MOE_ERR_INVALID_ARG;
  if (c->n_groups > 0) {
    if (c->n_groups > 32 || c->E % c->n_groups != 0) return MOE_ERR_INVALID_ARG;
    const int gs = c->E / c->n_groups;
    if (c->topk_groups < 1 || c->topk_groups > c->n_groups) return MOE_ERR_INVALID_ARG;
    if (c->group_topn < 1 || c->group_topn > gs) return MOE_ERR_INVALID_ARG;
    if (c->group_topn > kMaxGroupTopn) return MOE_ERR_UNSUPPORTED;
    if ((int64_t)c->topk_groups * gs < c->K) return MOE_ERR_INVALID_ARG;
  }
  if (c->capacity < 0 || (c->pad != 0 && c->pad != 1)) return MOE_ERR_INVALID_ARG;
  if (c->pad && c->capacity == 0) return MOE_ERR_INVALID_ARG;
  if (c->n_redundant < 0 || (int64_t)c->E + c->n_redundant > 1024) return MOE_ERR_INVALID_ARG;
  if (c->ep_size < 1 || (c->E + c->n_redundant) % c->ep_size != 0) return MOE_ERR_INVALID_ARG;
  if (c->shared_I < 0 || c->shared_I % 64 != 0) return MOE_ERR_INVALID_ARG;
  if ((int64_t)c->T * c->K >= INT32_MAX || rows_of(*c) >= INT32_MAX) return MOE_ERR_INVALID_ARG;
  // one permuted row must fit a shared-memory buffer of the bulk-copy permute
  if ((int64_t)c->h * ds_of(*c) > 200 * 1024) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

moe_status check_dtype_ptr(const void* p) {
  if (p == nullptr) return MOE_ERR_INVALID_ARG;
  return aligned(p, 16) ? MOE_OK : MOE_ERR_ALIGNMENT;
}
moe_status check_ptr(const void* p, size_t a) {
  if (p == nullptr) return MOE_ERR_INVALID_ARG;
  return aligned(p, a) ? MOE_OK : MOE_ERR_ALIGNMENT;
}
moe_status check_opt_ptr(const void* p, size_t a) { return (p == nullptr || aligned(p, a)) ? MOE_OK : MOE_ERR_ALIGNMENT; }

struct DeviceInfo {
  int sms = 0;
};
// SM count per device, looked up once; several host threads may fill an entry
// at the same time (they store the same value), hence the atomics.
DeviceInfo device_info() {
  static std::atomic<int> cache[64];
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) dev = 0;
  DeviceInfo d;
  d.sms = cache[dev].load(std::memory_order_relaxed);
  if (d.sms == 0) {
    cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
    cache[dev].store(d.sms, std::memory_order_relaxed);
  }
  return d;
}

template <typename K>
cudaError_t allow_smem(K kernel, size_t bytes) {
  if (bytes <= 48 * 1024) return cudaSuccess;
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

// ------------------------------------------------------------------ workspace carving
struct Carver {
  char* base;
  size_t off = 0;
  explicit Carver(void* b) : base(static_cast<char*>(b)) {}
  template <typename T>
  T* take(size_t count) {
    T* p = base ? reinterpret_cast<T*>(base + off) : nullptr;
    off += align_up(count * sizeof(T) + 0, 256);
    return p;
  }
};

struct LayerBuffers {
  void* layout_ws;
  size_t layout_ws_bytes;
  float* logits;
  void* logits_ws;     // split sums of the router logits
  int32_t* ids;
  float* w;
  int32_t* counts;
  int32_t* kept;
  int32_t* offsets;
  int32_t* slot;
  int32_t* row_src;
  int64_t* n_ij;
  int64_t* rank_bytes;
  moe_layout_stats* stats;
  void* xp;
  void* yp;
  void* inter;
  void* xdev;
  void* ydev;
  int32_t* phys_ids;   // physical expert of every (t, k) (replicas)
  float* xscale;       // FP8: scale of every permuted row [R]
  void* ys;            // shared expert output [T, h] (block)
  void* shared_ws;     // shared expert intermediate [T, shared_I] (block)
  size_t total;
};

size_t shared_ws_bytes(const moe_config& c) { return align_up((size_t)c.T * c.shared_I * ds_of(c), 256) + 256; }

// Router logits: float32 partial sums of up to kLogitsMaxSplit slices of h.
constexpr int kLogitsMaxSplit = 8;
size_t logits_ws_bytes(const moe_config& c) { return align_up((size_t)kLogitsMaxSplit * c.T * c.E * 4, 256) + 256; }

size_t ffn_fp8_ws_bytes(const moe_config& c);

LayerBuffers carve_layer(const moe_config& c, void* ws, bool host_io, bool block = false, bool fp8 = false) {
  Carver cv(ws);
  LayerBuffers b;
  const int64_t A = (int64_t)c.T * c.K, R = rows_of(c);
  const int N = c.ep_size, ds = ds_of(c);
  b.layout_ws_bytes = layout_scratch_bytes(A, nphys(c));
  b.layout_ws = cv.take<char>(b.layout_ws_bytes);
  b.logits = cv.take<float>((size_t)c.T * c.E);
  b.logits_ws = cv.take<char>(logits_ws_bytes(c));
  b.ids = cv.take<int32_t>(A);
  b.w = cv.take<float>(A);
  b.counts = cv.take<int32_t>(nphys(c));
  b.kept = cv.take<int32_t>(nphys(c));
  b.offsets = cv.take<int32_t>(nphys(c) + 1);
  b.phys_ids = c.n_redundant > 0 ? cv.take<int32_t>(A) : nullptr;
  b.slot = cv.take<int32_t>(A);
  b.row_src = cv.take<int32_t>(R);
  b.n_ij = cv.take<int64_t>((size_t)N * N);
  b.rank_bytes = cv.take<int64_t>(2 * (size_t)N);
  b.stats = cv.take<moe_layout_stats>(1);
  b.xp = cv.take<char>((size_t)R * c.h * ds);
  b.yp = cv.take<char>((size_t)R * c.h * ds);
  b.inter = cv.take<char>(fp8 ? ffn_fp8_ws_bytes(c) : (size_t)R * c.I * ds);
  b.xscale = fp8 ? cv.take<float>(R) : nullptr;
  b.xdev = host_io ? cv.take<char>((size_t)c.T * c.h * ds) : nullptr;
  b.ydev = host_io ? cv.take<char>((size_t)c.T * c.h * ds) : nullptr;
  b.ys = block ? cv.take<char>((size_t)c.T * c.h * ds) : nullptr;
  b.shared_ws = block ? cv.take<char>(shared_ws_bytes(c)) : nullptr;
  b.total = cv.off;
  return b;
}

// Device address of g_layout_static_scratch on the current device, looked up
// once per device, on the first call there (host code cannot use the symbol
// itself as an address).  Concurrent first calls from several host threads
// store the same value; the atomics make that race well defined.  The address
// belongs to the device's current context: after cudaDeviceReset it is stale,
// so a process that resets a device must not call moe_dispatch_layout_static
// on it again.
moe_status static_layout_scratch(void** out) {
  static std::atomic<void*> addr[64];
  int dev = 0;
  CUDA_TRY(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64) return MOE_ERR_UNSUPPORTED;
  void* p = addr[dev].load(std::memory_order_acquire);
  if (p == nullptr) {
    CUDA_TRY(cudaGetSymbolAddress(&p, g_layout_static_scratch));
    if (p == nullptr) return MOE_ERR_CUDA;
    addr[dev].store(p, std::memory_order_release);
  }
  *out = p;
  return MOE_OK;
}

size_t ffn_ws_bytes(const moe_config& c) { return align_up((size_t)rows_of(c) * c.I * ds_of(c), 256) + 256; }
// moe_grouped_ffn_combine: the FFN's workspace, then one arrival counter per
// (token, 32-feature group).
size_t ffn_combine_ws_bytes(const moe_config& c) {
  return ffn_ws_bytes(c) + align_up((size_t)c.T * (c.h / 32) * 4, 256);
}

// ------------------------------------------------------------------ launchers
moe_status launch_logits_simt(const moe_config& c, const void* x, const void* w_r, const float* off, float* logits,
                         cudaStream_t st) {
  if (c.T == 0) return MOE_OK;
  SimtParams p{};
  p.A = x;
  p.lda = c.h;
  p.B = w_r;
  p.ldb = c.h;
  p.b_expert_rows = c.E;
  p.C = logits;
  p.ldc = c.E;
  p.M = c.T;
  p.N = c.E;
  p.K = c.h;
  p.col_bias = off;
  dim3 grid((c.E + kSimtBN - 1) / kSimtBN, (c.T + kSimtBM - 1) / kSimtBM);
  if (c.dtype == MOE_F32)
    (void)launch_k(simt_gemm_kernel<float, kSimtLogits>, grid, kSimtThreads, 0, st, p);
  else
    (void)launch_k(simt_gemm_kernel<__nv_bfloat16, kSimtLogits>, grid, kSimtThreads, 0, st, p);
  CUDA_TRY(launched());
  return MOE_OK;
}

template <int PER>
cudaError_t launch_route_per(const RouteParams& p, cudaStream_t st) {
  const int blocks = (p.T + kRouteWarps - 1) / kRouteWarps;
  const size_t smem = p.n_groups > 0 ? (size_t)kRouteWarps * p.E * sizeof(float) : 0;
  (void)launch_k(route_kernel<PER>, blocks, kRouteWarps * 32, smem, st, p);
  return launched();
}

moe_status launch_route(const moe_config& c, const float* logits, const float* bias, int32_t* ids, float* w,
                        cudaStream_t st) {
  if (c.T == 0) return MOE_OK;
  RouteParams p{};
  p.logits = logits;
  p.bias = bias;
  p.ids = ids;
  p.w = w;
  p.T = c.T;
  p.E = c.E;
  p.K = c.K;
  p.sigmoid = c.score == MOE_SIGMOID;
  p.renorm = c.renormalize;
  p.scale = c.scale;
  p.n_groups = c.n_groups;
  p.topk_groups = c.topk_groups;
  p.group_topn = c.group_topn;
  p.key_is_logit = (c.score == MOE_SOFTMAX && bias == nullptr && c.n_groups == 0) ? 1 : 0;
  const int per = (c.E + 31) / 32;
  cudaError_t e;
  if (per <= 1) e = launch_route_per<1>(p, st);
  else if (per <= 2) e = launch_route_per<2>(p, st);
  else if (per <= 4) e = launch_route_per<4>(p, st);
  else if (per <= 8) e = launch_route_per<8>(p, st);
  else if (per <= 16) e = launch_route_per<16>(p, st);
  else e = launch_route_per<32>(p, st);
  CUDA_TRY(e);
  return MOE_OK;
}

moe_status launch_layout(const moe_config& c, const int32_t* ids, int32_t* counts, int32_t* kept,
                         int32_t* offsets, int32_t* slot, int32_t* row_src, int64_t* n_ij, int64_t* rank_bytes,
                         moe_layout_stats* stats, void* ws, cudaStream_t st) {
  LayoutParams p{};
  p.ids = ids;
  p.A = (int64_t)c.T * c.K;
  p.T = c.T;
  p.K = c.K;
  p.E = nphys(c);
  p.cap = c.capacity;
  p.pad = c.pad;
  p.n_ep = c.ep_size;
  p.ds = ds_of(c);
  p.h = c.h;
  p.R = (int)rows_of(c);
  p.num_tiles = layout_num_tiles(p.A);
  p.counts = counts;
  p.kept = kept;
  p.offsets = offsets;
  p.slot = slot;
  p.row_src = row_src;
  p.n_ij = n_ij;
  p.rank_bytes = rank_bytes;
  p.stats = stats;
  p.ws = layout_scratch_at(ws, p.A, nphys(c));
  if (p.A <= kLayoutSmallMax) {  // one block, one launch
    const size_t smem = layout_small_smem(p.E, p.n_ep);
    CUDA_TRY(allow_smem(layout_small_kernel, smem));
    (void)launch_k(layout_small_kernel, 1, kLayoutSmallThreads, smem, st, p);
    CUDA_TRY(launched());
    return MOE_OK;
  }
  const size_t smem1 = (size_t)(kLayoutWarps + 2) * nphys(c) * sizeof(int32_t);
  CUDA_TRY(allow_smem(layout_rank_kernel, smem1));
  (void)launch_k(layout_rank_kernel, p.num_tiles, kLayoutThreads, smem1, st, p);
  CUDA_TRY(launched());
  const int64_t per_block = kFinalizeThreads * kFinalizeItems;
  const int blocks2 = (int)((p.A + per_block - 1) / per_block) > 0 ? (int)((p.A + per_block - 1) / per_block) : 1;
  (void)launch_k(layout_finalize_kernel, blocks2, kFinalizeThreads, (nphys(c) + 1) * sizeof(int32_t), st, p);
  CUDA_TRY(launched());
  return MOE_OK;
}

// Rows up to this size are permuted by warps (permute_warp_kernel), wider ones
// through shared memory by the bulk-copy engine (permute_bulk_kernel).
constexpr uint32_t kPermWarpMaxRowBytes = 4096;

moe_status launch_permute(const moe_config& c, const void* x, const int32_t* slot, const int32_t* row_src,
                          void* xp, cudaStream_t st) {
  const uint32_t row_bytes = (uint32_t)c.h * ds_of(c);
  if (c.pad && c.capacity > 0) {
    const int64_t R = rows_of(c);
    const uint32_t vecs = row_bytes / 16;
    const int64_t n = R * vecs;
    const int blocks = (int)((n + 255) / 256 < 148 * 8 ? (n + 255) / 256 : 148 * 8);
    if (n > 0) {
      (void)launch_k(zero_pad_rows_kernel, blocks, 256, 0, st, row_src, R, vecs, static_cast<uint4*>(xp));
      CUDA_TRY(launched());
    }
  }
  if (c.T == 0) return MOE_OK;
  if (row_bytes <= kPermWarpMaxRowBytes) {
    auto kern = c.K <= 1 ? permute_warp_kernel<1> : c.K <= 2 ? permute_warp_kernel<2>
              : c.K <= 8 ? permute_warp_kernel<8> : permute_warp_kernel<16>;
    const int row_vecs = (int)(row_bytes / 16);
    const int64_t units = c.T * ((row_vecs + kPermChunk - 1) / kPermChunk);
    int per_sm = 0;
    CUDA_TRY(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 256, 0));
    if (per_sm < 1) per_sm = 1;
    int64_t blocks = (int64_t)device_info().sms * per_sm;
    if (blocks > (units + 7) / 8) blocks = (units + 7) / 8;
    (void)launch_k(kern, (unsigned)blocks, 256, 0, st, static_cast<const uint4*>(x), slot, c.T, c.K, row_vecs,
                                           static_cast<uint4*>(xp));
    CUDA_TRY(launched());
    return MOE_OK;
  }
  PermuteParams p{};
  p.x = static_cast<const uint8_t*>(x);
  p.slot = slot;
  p.xp = static_cast<uint8_t*>(xp);
  p.T = c.T;
  p.K = c.K;
  p.row_bytes = row_bytes;
  int nbuf = (int)((160 * 1024) / row_bytes);
  p.nbuf = nbuf < 1 ? 1 : (nbuf > kPermBufs ? kPermBufs : nbuf);
  const size_t smem = (size_t)p.nbuf * row_bytes;
  CUDA_TRY(allow_smem(permute_bulk_kernel, smem));
  int per_sm = 0;
  CUDA_TRY(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, permute_bulk_kernel, 32, smem));
  if (per_sm < 1) per_sm = 1;
  int64_t blocks = (int64_t)device_info().sms * per_sm;
  if (blocks > c.T) blocks = c.T;
  (void)launch_k(permute_bulk_kernel, (unsigned)blocks, 32, smem, st, p);
  CUDA_TRY(launched());
  return MOE_OK;
}

moe_status launch_combine(const moe_config& c, const void* yp, const int32_t* slot, const float* w, const void* ys,
                          void* y, cudaStream_t st) {
  if (c.T == 0) return MOE_OK;
  CombineParams p{};
  p.yp = yp;
  p.slot = slot;
  p.w = w;
  p.ys = ys;
  p.y = y;
  p.T = c.T;
  p.K = c.K;
  p.h = c.h;
  // Persistent grid: every SM holds as many blocks as fit, each warp strides
  // over (token, chunk) units.
  const bool bf = c.dtype == MOE_BF16;
  auto kern = c.K <= 1   ? (bf ? combine_kernel<__nv_bfloat16, 1> : combine_kernel<float, 1>)
              : c.K <= 2 ? (bf ? combine_kernel<__nv_bfloat16, 2> : combine_kernel<float, 2>)
              : c.K <= 8 ? (bf ? combine_kernel<__nv_bfloat16, 8> : combine_kernel<float, 8>)
                         : (bf ? combine_kernel<__nv_bfloat16, 16> : combine_kernel<float, 16>);
  const int vecs = c.h / (bf ? 8 : 4);
  const int64_t units = c.T * ((vecs + kCombineChunk - 1) / kCombineChunk);
  int per_sm = 0;
  CUDA_TRY(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 256, 0));
  if (per_sm < 1) per_sm = 1;
  int64_t blocks = (int64_t)device_info().sms * per_sm;
  if (blocks > (units + 7) / 8) blocks = (units + 7) / 8;
  (void)launch_k(kern, (unsigned)blocks, 256, 0, st, p);
  CUDA_TRY(launched());
  return MOE_OK;
}

template <typename T>
cudaError_t launch_ffn_simt(const moe_config& c, const void* xp, const int32_t* offsets, const int32_t* kept,
                            const int32_t* w_map, const void* w13, const void* w2, void* yp, void* inter,
                            cudaStream_t st) {
  const int64_t R = rows_of(c);
  const unsigned mblocks = (unsigned)((R + kSimtBM - 1) / kSimtBM + nphys(c));
  SimtParams p{};
  p.A = xp;
  p.lda = c.h;
  p.B = w13;
  p.ldb = c.h;
  p.b_expert_rows = 2LL * c.I;
  p.up_rows = c.I;
  p.C = inter;
  p.ldc = c.I;
  p.offsets = offsets;
  p.kept = kept;
  p.E = nphys(c);
  p.w_map = w_map;
  p.n_w = w_map != nullptr ? c.E : nphys(c);
  p.N = c.I;
  p.K = c.h;
  (void)launch_k(simt_gemm_kernel<T, kSimtSwiglu>, dim3((c.I + kSimtBN - 1) / kSimtBN, mblocks), kSimtThreads, 0, st, p);
  cudaError_t e = launched();
  if (e != cudaSuccess) return e;
  SimtParams q = p;
  q.A = inter;
  q.lda = c.I;
  q.B = w2;
  q.ldb = c.I;
  q.b_expert_rows = c.h;
  q.up_rows = 0;
  q.C = yp;
  q.ldc = c.h;
  q.N = c.h;
  q.K = c.I;
  (void)launch_k(simt_gemm_kernel<T, kSimtPlain>, dim3((c.h + kSimtBN - 1) / kSimtBN, mblocks), kSimtThreads, 0, st, q);
  return launched();
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no -lcuda).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// 2-D bf16 K-major tensor [rows, inner] read in boxes of box_rows x 64 elements
// with the 128-byte swizzle the MMA descriptors expect.
moe_status make_tensor_map(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, uint32_t box_rows,
                           bool bytes = false) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (enc == nullptr) return MOE_ERR_CUDA;
  // bf16 elements, or (bytes) 8-bit codes; either way 128-byte box rows
  const cuuint64_t dims[2] = {inner, rows};
  const cuuint64_t strides[1] = {inner * (bytes ? 1 : 2)};
  const cuuint32_t box[2] = {(cuuint32_t)(bytes ? 128 : kTcBK), box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = enc(map, bytes ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                         const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MOE_OK : MOE_ERR_CUDA;
}

// Experts expected to see more rows than this use token rows as the MMA's M
// operand (tc_gemm.cuh); others use weight rows as M (ffn_grouped.cuh).
#ifndef MOE_FFN_SWAP_MAX_ROWS
#define MOE_FFN_SWAP_MAX_ROWS 160
#endif

// The grouped FFN with token rows as M (128-row m-blocks of an expert's
// segment) and weight rows as N (256 columns: 128 gate + 128 up units, or 256
// output features): the tensor-bound regime of many rows per expert.
constexpr int kFfnBN = 256, kFfnStages = 4;

moe_status launch_ffn_tokens_m_one(const moe_config& c, const void* xp, const int32_t* offsets, const int32_t* kept,
                                   const int32_t* w_map, int n_w, const void* w13, const void* w2, void* yp,
                                   void* inter, cudaStream_t st) {
  using S = TcShape<kFfnBN, kFfnStages>;
  const int64_t R = rows_of(c);
  const int grid = device_info().sms;
  CUtensorMap a1, b1, a2, b2;
  MOE_TRY(make_tensor_map(&a1, xp, c.h, R, kTcBM));
  MOE_TRY(make_tensor_map(&b1, w13, c.h, (uint64_t)n_w * 2 * c.I, kFfnBN / 2));
  MOE_TRY(make_tensor_map(&a2, inter, c.I, R, kTcBM));
  MOE_TRY(make_tensor_map(&b2, w2, c.I, (uint64_t)n_w * c.h, kFfnBN));
  TcParams p1{};
  p1.offsets = offsets;
  p1.kept = kept;
  p1.E = nphys(c);
  p1.w_map = w_map;
  p1.n_tiles = (c.I + kFfnBN / 2 - 1) / (kFfnBN / 2);
  p1.k_blocks = c.h / kTcBK;
  p1.b_rows = 2LL * c.I;
  p1.up_rows = c.I;
  p1.n_valid = c.I;
  p1.out = inter;
  p1.ldo = c.I;
  TcParams p2 = p1;
  p2.n_tiles = (c.h + kFfnBN - 1) / kFfnBN;
  p2.k_blocks = c.I / kTcBK;
  p2.b_rows = c.h;
  p2.up_rows = 0;
  p2.n_valid = c.h;
  p2.out = yp;
  p2.ldo = c.h;
  auto k1 = tc_gemm_kernel<kTcSwiglu, kFfnBN, kFfnStages>;
  auto k2 = tc_gemm_kernel<kTcStore, kFfnBN, kFfnStages>;
  CUDA_TRY(allow_smem(k1, S::kDynSmem));
  CUDA_TRY(allow_smem(k2, S::kDynSmem));
  (void)launch_k(k1, grid, kTcThreads, S::kDynSmem, st, a1, b1, p1);
  CUDA_TRY(launched());
  (void)launch_k(k2, grid, kTcThreads, S::kDynSmem, st, a2, b2, p2);
  CUDA_TRY(launched());
  return MOE_OK;
}

moe_status launch_ffn_tokens_m(const moe_config& c, const void* xp, const int32_t* offsets, const int32_t* kept,
                               const int32_t* w_map, int n_w, const void* w13, const void* w2, void* yp, void* inter,
                               cudaStream_t st) {
  return launch_ffn_tokens_m_one(c, xp, offsets, kept, w_map, n_w, w13, w2, yp, inter, st);
}

// The grouped FFN: gate/up GEMM with the SwiGLU epilogue into the bf16
// intermediate, then the down GEMM into yp, both with the expert weights as
// the MMA's M operand and the expert's token rows as N (ffn_grouped.cuh).
// Token tiles of up to 160 rows; a ring of 4 stages, each a k-block of weights
// (32 KB) and of token rows (20 KB).  Measured at DeepSeek-V3 T=4096 with
// separately sized weight and token rings: 4 + 4 stages 3.94 ms; 5 + 2 (5.20
// ms), 4 + 3 (4.13), 128-row tiles with 5 + 3 (4.30) and 256-row tiles with
// 4 + 2 (5.13) starve the MMA of token k-blocks, whose L2 latency under this
// load needs four in flight.  Equal depths let one barrier pair serve a stage.
constexpr int kFgTileRows = 160, kFgStages = 4;
// The weighted combine fused into the down projection (dropless layers).
struct FusedCombine {
  const int32_t* row_src;
  const int32_t* slot;
  const float* topk_w;
  void* y;
  uint32_t* arrive;   // [T, h/32], zero between calls
};

// row_src non-null: the gate/up GEMM gathers its rows from x = xp through row_src
// (no permuted copy of x); else xp holds the permuted rows.  comb non-null: the
// down projection also writes the combine into comb->y.
template <int BT, int ST>
moe_status launch_ffn_grouped(const moe_config& c, const void* xp, const int32_t* offsets, const int32_t* kept,
                              const int32_t* w_map, int n_w, const void* w13, const void* w2, void* yp, void* inter,
                              cudaStream_t st, const int32_t* row_src = nullptr, const FusedCombine* comb = nullptr) {
  using S = FgShape<BT, ST>;
  const int64_t R = rows_of(c);
  const int grid = device_info().sms;
  CUtensorMap w1m, w2m;
  FgTokenMaps x1, x2;
  MOE_TRY(make_tensor_map(&w1m, w13, c.h, (uint64_t)n_w * 2 * c.I, 128));
  MOE_TRY(make_tensor_map(&w2m, w2, c.I, (uint64_t)n_w * c.h, 128));
  for (int i = 0; i < 4; ++i) {
    // gathered rows are copied from x by the kernel's gather warps: no map of x
    MOE_TRY(make_tensor_map(&x1.m[i], xp, c.h, row_src != nullptr ? (uint64_t)c.T : (uint64_t)R, 128u >> i));
    MOE_TRY(make_tensor_map(&x2.m[i], inter, c.I, R, 128u >> i));
  }
  FgParams p1{};
  p1.offsets = offsets;
  p1.kept = kept;
  p1.E = nphys(c);
  p1.w_map = w_map;
  p1.f_tiles = (c.I + 127) / 128;
  p1.k_blocks = c.h / kTcBK;
  p1.a_rows = 2LL * c.I;
  p1.up_rows = c.I;
  p1.n_valid = c.I;
  p1.out = static_cast<__nv_bfloat16*>(inter);
  p1.ldo = c.I;
  FgParams p2 = p1;
  p2.f_tiles = (c.h + 255) / 256;
  p2.k_blocks = c.I / kTcBK;
  p2.a_rows = c.h;
  p2.up_rows = 0;
  p2.n_valid = c.h;
  p2.out = static_cast<__nv_bfloat16*>(yp);
  p2.ldo = c.h;
  p1.row_src = row_src;
  p1.gather_x = static_cast<const uint8_t*>(xp);
  p1.ldx_bytes = (int64_t)c.h * 2;
  p2.row_src = nullptr;
  if (comb != nullptr) {
    p2.row_src = comb->row_src;
    p2.slot = comb->slot;
    p2.topk_w = comb->topk_w;
    p2.K = c.K;
    p2.groups = c.h / 32;
    p2.y = static_cast<__nv_bfloat16*>(comb->y);
    p2.arrive = comb->arrive;
  }
  const bool gather = row_src != nullptr;
  auto k1 = gather ? ffn_grouped_kernel<kTcSwiglu, BT, ST, false, true> : ffn_grouped_kernel<kTcSwiglu, BT, ST>;
  auto k2 = comb != nullptr ? ffn_grouped_kernel<kTcStore, BT, ST, false, false, true>
                            : ffn_grouped_kernel<kTcStore, BT, ST>;
  CUDA_TRY(allow_smem(k1, S::kDynSmem));
  CUDA_TRY(allow_smem(k2, S::kDynSmem));
  (void)launch_k(k1, grid, gather ? FgThreads<true, ST>::value : kFgThreads, S::kDynSmem, st, w1m, x1, p1);
  CUDA_TRY(launched());
  (void)launch_k(k2, grid, kFgThreads, S::kDynSmem, st, w2m, x2, p2);
  CUDA_TRY(launched());
  return MOE_OK;
}

// Rows an expert is expected to receive: the capacity when there is one, else
// the mean T*K/E.
int64_t expected_rows_per_expert(const moe_config& c) {
  if (c.capacity > 0) return c.capacity < c.T ? c.capacity : c.T;
  return ((int64_t)c.T * c.K + nphys(c) - 1) / nphys(c);
}

// n_w: experts held by w13/w2; w_map: physical expert -> its weights (null:
// the identity, n_w == physical experts).
moe_status launch_ffn_tc(const moe_config& c, const void* xp, const int32_t* offsets, const int32_t* kept,
                         const int32_t* w_map, int n_w, const void* w13, const void* w2, void* yp, void* inter,
                         cudaStream_t st) {
  // TMA row coordinates are 32-bit
  if ((int64_t)n_w * 2 * c.I >= INT32_MAX || (int64_t)n_w * c.h >= INT32_MAX) return MOE_ERR_UNSUPPORTED;
  if (expected_rows_per_expert(c) > MOE_FFN_SWAP_MAX_ROWS)
    return launch_ffn_tokens_m(c, xp, offsets, kept, w_map, n_w, w13, w2, yp, inter, st);
  return launch_ffn_grouped<kFgTileRows, kFgStages>(c, xp, offsets, kept, w_map, n_w, w13, w2, yp, inter, st);
}

// Router logits of a bf16 layer on the tensor cores: one segment of T rows
// times the [E, h] router weight, BN columns per tile with BN chosen so that
// the tiles cover the SMs (BN halves while twice the tiles still fit one wave).
template <int BN, int STAGES>
moe_status launch_logits_tc_bn(const moe_config& c, const void* x, const void* w_r, const float* off,
                               float* logits, int k_split, void* ws, cudaStream_t st) {
  using S = TcShape<BN, STAGES>;
  CUtensorMap a, b;
  MOE_TRY(make_tensor_map(&a, x, c.h, c.T, kTcBM));
  MOE_TRY(make_tensor_map(&b, w_r, c.h, c.E, BN));
  TcParams p{};
  p.offsets = nullptr;
  p.kept = nullptr;
  p.E = 1;
  p.dense_rows = c.T;
  p.n_tiles = (c.E + BN - 1) / BN;
  p.k_blocks = c.h / kTcBK;
  p.b_rows = 0;
  p.n_valid = c.E;
  p.out = logits;
  p.ldo = c.E;
  p.col_bias = off;
  p.k_split = k_split;
  p.partial = static_cast<float*>(ws);
  const int64_t items = (int64_t)((c.T + kTcBM - 1) / kTcBM) * p.n_tiles * k_split;
  const int sms = device_info().sms;
  const int grid = (int)(items < sms ? items : sms);
  auto k = tc_gemm_kernel<kTcLogits, BN, STAGES>;
  CUDA_TRY(allow_smem(k, S::kDynSmem));
  (void)launch_k(k, grid, kTcThreads, S::kDynSmem, st, a, b, p);
  CUDA_TRY(launched());
  if (k_split > 1) {
    const int64_t n = (int64_t)c.T * c.E;
    const int64_t lanes = (c.E % 4 == 0) ? n / 4 : n;
    int64_t blocks = (lanes + 255) / 256;
    if (blocks > (int64_t)sms * 8) blocks = (int64_t)sms * 8;
    (void)launch_k(logits_reduce_kernel, (unsigned)blocks, 256, 0, st, p.partial, k_split, n, c.E, off, logits);
    CUDA_TRY(launched());
  }
  return MOE_OK;
}

// Column-tile width BN and number of slices of the sum over h.  Each work item
// (row tile, column tile, slice) streams its k-blocks through one CTA's TMA
// ring, whose rate is bound by latency, so the choice minimises the bytes the
// busiest SM streams: waves x k-blocks per slice x (16 KB of x + BN rows of w_r),
// with at least 8 k-blocks per slice and at most kLogitsMaxSplit slices; ties
// go to fewer work items.
struct LogitsPlan {
  int bn, k_split;
};
LogitsPlan logits_plan(const moe_config& c, int sms) {
  const int64_t mb = (c.T + kTcBM - 1) / kTcBM;
  const int kb = c.h / kTcBK;
  LogitsPlan best{256, 1};
  int64_t best_cost = -1, best_items = 0;
  for (int bn = 16; bn <= 256; bn *= 2) {
    if (bn > 16 && bn / 2 >= c.E) break;  // a narrower tile already covers E
    for (int ks = 1; ks <= kLogitsMaxSplit; ++ks) {
      if (ks > 1 && kb / ks < 8) break;
      const int64_t items = mb * ((c.E + bn - 1) / bn) * ks;
      const int64_t waves = (items + sms - 1) / sms;
      const int64_t cost = waves * ((kb + ks - 1) / ks) * (int64_t)(kTcBM * 128 + bn * 128);
      if (best_cost < 0 || cost < best_cost || (cost == best_cost && items < best_items)) {
        best = {bn, ks};
        best_cost = cost;
        best_items = items;
      }
    }
  }
  return best;
}

moe_status launch_logits(const moe_config& c, const void* x, const void* w_r, const float* off, float* logits,
                         void* ws, cudaStream_t st) {
  if (c.T == 0) return MOE_OK;
  // float32 layers stay on CUDA cores: a TF32 product would miss their 1e-4 tolerance
  if (c.dtype == MOE_F32) return launch_logits_simt(c, x, w_r, off, logits, st);
  const LogitsPlan lp = logits_plan(c, device_info().sms);
  switch (lp.bn) {
    case 16: return launch_logits_tc_bn<16, 8>(c, x, w_r, off, logits, lp.k_split, ws, st);
    case 32: return launch_logits_tc_bn<32, 8>(c, x, w_r, off, logits, lp.k_split, ws, st);
    case 64: return launch_logits_tc_bn<64, 8>(c, x, w_r, off, logits, lp.k_split, ws, st);
    case 128: return launch_logits_tc_bn<128, 6>(c, x, w_r, off, logits, lp.k_split, ws, st);
    default: return launch_logits_tc_bn<256, 4>(c, x, w_r, off, logits, lp.k_split, ws, st);
  }
}

// FP8 experts: gate/up (E4M3 codes of x rows and w13 rows) with the SwiGLU
// epilogue into the bf16 intermediate, the intermediate re-quantised per row,
// then the down projection into yp.  Weights as M only (experts expected to see
// at most MOE_FFN_SWAP_MAX_ROWS rows).  ws: inter bf16 [R, I], codes [R, I],
// scales [R].
size_t ffn_fp8_ws_bytes(const moe_config& c) {
  const size_t R = (size_t)rows_of(c);
  return align_up(R * c.I * 2, 256) + align_up(R * c.I, 256) + align_up(R * 4, 256) + 256;
}

moe_status launch_ffn_fp8(const moe_config& c, const uint8_t* xq, const float* sx, const int32_t* offsets,
                          const int32_t* kept, const int32_t* w_map, int n_w, const uint8_t* w13q,
                          const float* s13, const uint8_t* w2q, const float* s2, void* yp, void* ws,
                          cudaStream_t st) {
  const int64_t R = rows_of(c);
  if (R == 0) return MOE_OK;
  if (expected_rows_per_expert(c) > MOE_FFN_SWAP_MAX_ROWS) return MOE_ERR_UNSUPPORTED;
  if ((int64_t)n_w * 2 * c.I >= INT32_MAX || (int64_t)n_w * c.h >= INT32_MAX) return MOE_ERR_UNSUPPORTED;
  char* w = static_cast<char*>(ws);
  __nv_bfloat16* inter = reinterpret_cast<__nv_bfloat16*>(w);
  uint8_t* interq = reinterpret_cast<uint8_t*>(w + align_up((size_t)R * c.I * 2, 256));
  float* sinter = reinterpret_cast<float*>(w + align_up((size_t)R * c.I * 2, 256) + align_up((size_t)R * c.I, 256));
  using S = FgShape<kFgTileRows, kFgStages>;
  CUtensorMap w1m, w2m;
  FgTokenMaps x1, x2;
  MOE_TRY(make_tensor_map(&w1m, w13q, c.h, (uint64_t)n_w * 2 * c.I, 128, true));
  MOE_TRY(make_tensor_map(&w2m, w2q, c.I, (uint64_t)n_w * c.h, 128, true));
  for (int i = 0; i < 4; ++i) {
    MOE_TRY(make_tensor_map(&x1.m[i], xq, c.h, R, 128u >> i, true));
    MOE_TRY(make_tensor_map(&x2.m[i], interq, c.I, R, 128u >> i, true));
  }
  FgParams p1{};
  p1.offsets = offsets;
  p1.kept = kept;
  p1.E = nphys(c);
  p1.w_map = w_map;
  p1.f_tiles = (c.I + 127) / 128;
  p1.k_blocks = c.h / 128;
  p1.a_rows = 2LL * c.I;
  p1.up_rows = c.I;
  p1.n_valid = c.I;
  p1.out = inter;
  p1.ldo = c.I;
  p1.w_scale = s13;
  p1.x_scale = sx;
  FgParams p2 = p1;
  p2.f_tiles = (c.h + 255) / 256;
  p2.k_blocks = c.I / 128;
  p2.a_rows = c.h;
  p2.up_rows = 0;
  p2.n_valid = c.h;
  p2.out = static_cast<__nv_bfloat16*>(yp);
  p2.ldo = c.h;
  p2.w_scale = s2;
  p2.x_scale = sinter;
  const int grid = device_info().sms;
  auto k1 = ffn_grouped_kernel<kTcSwiglu, kFgTileRows, kFgStages, true>;
  auto k2 = ffn_grouped_kernel<kTcStore, kFgTileRows, kFgStages, true>;
  CUDA_TRY(allow_smem(k1, S::kDynSmem));
  CUDA_TRY(allow_smem(k2, S::kDynSmem));
  (void)launch_k(k1, grid, kFgThreads, S::kDynSmem, st, w1m, x1, p1);
  CUDA_TRY(launched());
  int64_t qb = (R + 7) / 8;
  if (qb > (int64_t)grid * 16) qb = (int64_t)grid * 16;
  (void)launch_k(quant_rows_kernel<__nv_bfloat16>, (unsigned)qb, 256, 0, st, inter, R, c.I, interq, sinter);
  CUDA_TRY(launched());
  (void)launch_k(k2, grid, kFgThreads, S::kDynSmem, st, w2m, x2, p2);
  CUDA_TRY(launched());
  return MOE_OK;
}

moe_status launch_permute_fp8(const moe_config& c, const void* x, const int32_t* slot, uint8_t* xq, float* sx,
                              cudaStream_t st) {
  if (c.T == 0) return MOE_OK;
  int64_t blocks = (c.T + 7) / 8;
  if (blocks > (int64_t)device_info().sms * 16) blocks = (int64_t)device_info().sms * 16;
  (void)launch_k(quant_permute_kernel<__nv_bfloat16>, (unsigned)blocks, 256, 0, st, static_cast<const __nv_bfloat16*>(x), slot,
                                                                       c.T, c.K, c.h, xq, sx);
  CUDA_TRY(launched());
  return MOE_OK;
}

// The grouped FFN reading its rows straight from x through row_src: bf16,
// weights-as-M layers only (experts expected to see at most
// MOE_FFN_SWAP_MAX_ROWS rows).  Gather warps copy the rows with 16-byte
// cp.async (the four-row TMA gathers tried first cost about as much per
// instruction as a whole box: 1.75x slower at DeepSeek-V3 prefill).  The rows
// are gathered once per feature tile, which at DeepSeek-V3 T=4096 measured a
// few percent slower than the explicit permute + FFN, so the layer calls keep
// the permute.  It saves the permuted copy of x (R x h).
moe_status launch_ffn_gather(const moe_config& c, const void* x, const int32_t* row_src, const int32_t* offsets,
                             const int32_t* kept, const int32_t* w_map, int n_w, const void* w13, const void* w2,
                             void* yp, void* inter, cudaStream_t st) {
  if (rows_of(c) == 0 || c.T == 0) return MOE_OK;
  if (c.dtype != MOE_BF16 || expected_rows_per_expert(c) > MOE_FFN_SWAP_MAX_ROWS) return MOE_ERR_UNSUPPORTED;
  if ((int64_t)n_w * 2 * c.I >= INT32_MAX || (int64_t)n_w * c.h >= INT32_MAX) return MOE_ERR_UNSUPPORTED;
  return launch_ffn_grouped<kFgTileRows, kFgStages>(c, x, offsets, kept, w_map, n_w, w13, w2, yp, inter, st,
                                                    row_src);
}

moe_status launch_ffn(const moe_config& c, const void* xp, const int32_t* offsets, const int32_t* kept,
                      const int32_t* w_map, int n_w, const void* w13, const void* w2, void* yp, void* inter,
                      cudaStream_t st) {
  if (rows_of(c) == 0) return MOE_OK;
  if (c.dtype == MOE_BF16) return launch_ffn_tc(c, xp, offsets, kept, w_map, n_w, w13, w2, yp, inter, st);
  CUDA_TRY(launch_ffn_simt<float>(c, xp, offsets, kept, w_map, w13, w2, yp, inter, st));
  return MOE_OK;
}

// The shared expert: one dense segment of all T tokens through the FFN GEMMs
// (tokens as M on the tensor cores for bf16, CUDA cores for float32); x is read
// in place, no permutation.
moe_status launch_shared_ffn(const moe_config& c, const void* x, const void* w13s, const void* w2s, void* ys,
                             void* inter, cudaStream_t st) {
  if (c.T == 0) return MOE_OK;
  const int Is = c.shared_I;
  if (c.dtype == MOE_F32) {
    SimtParams p{};
    p.A = x;
    p.lda = c.h;
    p.B = w13s;
    p.ldb = c.h;
    p.b_expert_rows = 2LL * Is;
    p.up_rows = Is;
    p.C = inter;
    p.ldc = Is;
    p.E = 1;
    p.M = c.T;
    p.N = Is;
    p.K = c.h;
    const unsigned mblocks = (unsigned)((c.T + kSimtBM - 1) / kSimtBM);
    (void)launch_k(simt_gemm_kernel<float, kSimtSwiglu>, dim3((Is + kSimtBN - 1) / kSimtBN, mblocks), kSimtThreads, 0, st, p);
    CUDA_TRY(launched());
    SimtParams q = p;
    q.A = inter;
    q.lda = Is;
    q.B = w2s;
    q.ldb = Is;
    q.b_expert_rows = c.h;
    q.up_rows = 0;
    q.C = ys;
    q.ldc = c.h;
    q.N = c.h;
    q.K = Is;
    (void)launch_k(simt_gemm_kernel<float, kSimtPlain>, dim3((c.h + kSimtBN - 1) / kSimtBN, mblocks), kSimtThreads, 0, st, q);
    CUDA_TRY(launched());
    return MOE_OK;
  }
  using S = TcShape<kFfnBN, kFfnStages>;
  CUtensorMap a1, b1, a2, b2;
  MOE_TRY(make_tensor_map(&a1, x, c.h, c.T, kTcBM));
  MOE_TRY(make_tensor_map(&b1, w13s, c.h, 2ull * Is, kFfnBN / 2));
  MOE_TRY(make_tensor_map(&a2, inter, Is, c.T, kTcBM));
  MOE_TRY(make_tensor_map(&b2, w2s, Is, c.h, kFfnBN));
  TcParams p1{};
  p1.offsets = nullptr;
  p1.kept = nullptr;
  p1.E = 1;
  p1.dense_rows = c.T;
  p1.n_tiles = (Is + kFfnBN / 2 - 1) / (kFfnBN / 2);
  p1.k_blocks = c.h / kTcBK;
  p1.b_rows = 0;
  p1.up_rows = Is;
  p1.n_valid = Is;
  p1.out = inter;
  p1.ldo = Is;
  TcParams p2 = p1;
  p2.n_tiles = (c.h + kFfnBN - 1) / kFfnBN;
  p2.k_blocks = Is / kTcBK;
  p2.up_rows = 0;
  p2.n_valid = c.h;
  p2.out = ys;
  p2.ldo = c.h;
  const int sms = device_info().sms;
  const int64_t mb = (c.T + kTcBM - 1) / kTcBM;
  const int g1 = (int)(mb * p1.n_tiles < sms ? mb * p1.n_tiles : sms);
  const int g2 = (int)(mb * p2.n_tiles < sms ? mb * p2.n_tiles : sms);
  auto k1 = tc_gemm_kernel<kTcSwiglu, kFfnBN, kFfnStages>;
  auto k2 = tc_gemm_kernel<kTcStore, kFfnBN, kFfnStages>;
  CUDA_TRY(allow_smem(k1, S::kDynSmem));
  CUDA_TRY(allow_smem(k2, S::kDynSmem));
  (void)launch_k(k1, g1, kTcThreads, S::kDynSmem, st, a1, b1, p1);
  CUDA_TRY(launched());
  (void)launch_k(k2, g2, kTcThreads, S::kDynSmem, st, a2, b2, p2);
  CUDA_TRY(launched());
  return MOE_OK;
}

// Device copy of an EPLB plan (moe_eplb_plan's outputs), or all null.
// FP8 expert weights (moe_quantize_fp8 codes and row scales), or all null.
struct Fp8Weights {
  const uint8_t* w13q = nullptr;
  const float* s13 = nullptr;
  const uint8_t* w2q = nullptr;
  const float* s2 = nullptr;
};

struct EplbDev {
  const int32_t* rep_offsets = nullptr;
  const int32_t* rep_phys = nullptr;
  const int32_t* phys_to_log = nullptr;
};

moe_status launch_eplb_map(const moe_config& c, const int32_t* ids, const EplbDev& plan, int32_t* phys,
                           cudaStream_t st) {
  const int64_t A = (int64_t)c.T * c.K;
  if (A == 0) return MOE_OK;
  int64_t blocks = (A + 255) / 256;
  if (blocks > (int64_t)device_info().sms * 8) blocks = (int64_t)device_info().sms * 8;
  (void)launch_k(eplb_map_kernel, (unsigned)blocks, 256, 0, st, ids, A, c.K, c.E, nphys(c), plan.rep_offsets, plan.rep_phys,
                                                      phys);
  CUDA_TRY(launched());
  return MOE_OK;
}

moe_status layer_core(const moe_config& c, const void* x, const void* w_r, const float* logit_offset,
                      const float* sel_bias, const void* w13, const void* w2, const void* w13s, const void* w2s,
                      void* y, const moe_layer_out* out, const LayerBuffers& b, cudaStream_t st,
                      const EplbDev& plan = EplbDev(), const Fp8Weights& q = Fp8Weights()) {
  moe_layer_out o{};
  if (out != nullptr) o = *out;
  float* logits = o.logits ? o.logits : b.logits;
  int32_t* ids = o.topk_ids ? o.topk_ids : b.ids;
  float* w = o.topk_w ? o.topk_w : b.w;
  int32_t* counts = o.counts ? o.counts : b.counts;
  int32_t* kept = o.kept ? o.kept : b.kept;
  int32_t* offsets = o.offsets ? o.offsets : b.offsets;
  int32_t* slot = o.slot ? o.slot : b.slot;
  int32_t* row_src = o.row_src ? o.row_src : b.row_src;
  int64_t* n_ij = o.n_ij ? o.n_ij : b.n_ij;
  int64_t* rank_bytes = o.rank_bytes ? o.rank_bytes : b.rank_bytes;
  moe_layout_stats* stats = o.stats ? o.stats : b.stats;
  // caller's stage events: [0] before the first stage, [s + 1] after stage s
  cudaEvent_t const* ev = reinterpret_cast<cudaEvent_t const*>(o.stage_events);
  auto mark = [&](int i) -> moe_status {
    if (ev != nullptr && ev[i] != nullptr) CUDA_TRY(cudaEventRecord(ev[i], st));
    return MOE_OK;
  };
  MOE_TRY(mark(0));
  MOE_TRY(launch_logits(c, x, w_r, logit_offset, logits, b.logits_ws, st));
  MOE_TRY(mark(MOE_STAGE_LOGITS + 1));
  MOE_TRY(launch_route(c, logits, sel_bias, ids, w, st));
  MOE_TRY(mark(MOE_STAGE_ROUTE + 1));
  const int32_t* lids = ids;  // expert ids the layout sees: physical replicas when the plan has any
  if (c.n_redundant > 0) {
    MOE_TRY(launch_eplb_map(c, ids, plan, b.phys_ids, st));
    lids = b.phys_ids;
  }
  MOE_TRY(mark(MOE_STAGE_EPLB_MAP + 1));
  MOE_TRY(launch_layout(c, lids, counts, kept, offsets, slot, row_src, n_ij, rank_bytes, stats, b.layout_ws, st));
  MOE_TRY(mark(MOE_STAGE_LAYOUT + 1));
  if (q.w13q != nullptr) {  // FP8 experts: quantise x per token while permuting
    MOE_TRY(launch_permute_fp8(c, x, slot, static_cast<uint8_t*>(b.xp), b.xscale, st));
    MOE_TRY(mark(MOE_STAGE_PERMUTE + 1));
    MOE_TRY(launch_ffn_fp8(c, static_cast<const uint8_t*>(b.xp), b.xscale, offsets, kept, plan.phys_to_log,
                           plan.phys_to_log ? c.E : nphys(c), q.w13q, q.s13, q.w2q, q.s2, b.yp, b.inter, st));
  } else {
    MOE_TRY(launch_permute(c, x, slot, row_src, b.xp, st));
    MOE_TRY(mark(MOE_STAGE_PERMUTE + 1));
    MOE_TRY(launch_ffn(c, b.xp, offsets, kept, plan.phys_to_log, plan.phys_to_log ? c.E : nphys(c), w13, w2, b.yp,
                       b.inter, st));
  }
  MOE_TRY(mark(MOE_STAGE_FFN + 1));
  if (b.ys != nullptr)
    MOE_TRY(launch_shared_ffn(c, x, w13s, w2s, b.ys, static_cast<char*>(b.shared_ws) + 256, st));
  MOE_TRY(mark(MOE_STAGE_SHARED + 1));
  MOE_TRY(launch_combine(c, b.yp, slot, w, b.ys, y, st));
  MOE_TRY(mark(MOE_STAGE_COMBINE + 1));
  return MOE_OK;
}

moe_status check_layer_ptrs(const moe_config& c, const void* x, const void* w_r, const float* logit_offset,
                            const float* sel_bias, const void* w13, const void* w2) {
  MOE_TRY(check_dtype_ptr(w_r));
  MOE_TRY(check_dtype_ptr(w13));
  MOE_TRY(check_dtype_ptr(w2));
  MOE_TRY(check_opt_ptr(logit_offset, 4));
  MOE_TRY(check_opt_ptr(sel_bias, 4));
  (void)x;
  (void)c;
  return MOE_OK;
}

}  // namespace

extern "C" {

uint64_t moe_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

const char* moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
    case MOE_ERR_ALIGNMENT: return "MOE_ERR_ALIGNMENT";
    case MOE_ERR_WORKSPACE_TOO_SMALL: return "MOE_ERR_WORKSPACE_TOO_SMALL";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
    case MOE_ERR_DEVICE_TIMEOUT: return "MOE_ERR_DEVICE_TIMEOUT";
    case MOE_ERR_DEVICE_BAD_INDEX: return "MOE_ERR_DEVICE_BAD_INDEX";
  }
  return "MOE_UNKNOWN_STATUS";
}

moe_status moe_validate_config(const moe_config* cfg) { return validate(cfg); }

moe_status moe_rows(const moe_config* cfg, int64_t* rows) {
  MOE_TRY(validate(cfg));
  if (rows == nullptr) return MOE_ERR_INVALID_ARG;
  *rows = rows_of(*cfg);
  return MOE_OK;
}

moe_status moe_workspace_size(const moe_config* cfg, int32_t op, size_t* bytes) {
  MOE_TRY(validate(cfg));
  if (bytes == nullptr) return MOE_ERR_INVALID_ARG;
  switch (op) {
    case MOE_OP_LAYOUT: *bytes = layout_scratch_bytes((int64_t)cfg->T * cfg->K, nphys(*cfg)); return MOE_OK;
    case MOE_OP_FFN: *bytes = ffn_ws_bytes(*cfg); return MOE_OK;
    case MOE_OP_LAYER: *bytes = carve_layer(*cfg, nullptr, false).total; return MOE_OK;
    case MOE_OP_LAYER_HOST: *bytes = carve_layer(*cfg, nullptr, true).total; return MOE_OK;
    case MOE_OP_SHARED: *bytes = shared_ws_bytes(*cfg); return MOE_OK;
    case MOE_OP_BLOCK: *bytes = carve_layer(*cfg, nullptr, false, true).total; return MOE_OK;
    case MOE_OP_BLOCK_HOST: *bytes = carve_layer(*cfg, nullptr, true, true).total; return MOE_OK;
    case MOE_OP_FFN_FP8: *bytes = ffn_fp8_ws_bytes(*cfg); return MOE_OK;
    case MOE_OP_LAYER_FP8: *bytes = carve_layer(*cfg, nullptr, false, false, true).total; return MOE_OK;
    case MOE_OP_LOGITS: *bytes = logits_ws_bytes(*cfg); return MOE_OK;
    case MOE_OP_FFN_COMBINE: *bytes = ffn_combine_ws_bytes(*cfg); return MOE_OK;
  }
  return MOE_ERR_INVALID_ARG;
}

moe_status moe_workspace_init(void* workspace, size_t workspace_bytes, void* stream) {
  if (workspace == nullptr || !aligned(workspace, 256)) return workspace ? MOE_ERR_ALIGNMENT : MOE_ERR_INVALID_ARG;
  CUDA_TRY(cudaMemsetAsync(workspace, 0, workspace_bytes, as_stream(stream)));
  return MOE_OK;
}

moe_status moe_router_logits(const moe_config* cfg, const void* x, const void* w_r, const float* logit_offset,
                             float* logits, void* workspace, size_t workspace_bytes, void* stream) {
  MOE_TRY(validate(cfg));
  if (cfg->T > 0) {
    MOE_TRY(check_dtype_ptr(x));
    MOE_TRY(check_ptr(logits, 4));
    if (cfg->dtype == MOE_BF16) {
      MOE_TRY(check_ptr(workspace, 256));
      if (workspace_bytes < logits_ws_bytes(*cfg)) return MOE_ERR_WORKSPACE_TOO_SMALL;
    }
  }
  MOE_TRY(check_dtype_ptr(w_r));
  MOE_TRY(check_opt_ptr(logit_offset, 4));
  return launch_logits(*cfg, x, w_r, logit_offset, logits, workspace, as_stream(stream));
}

moe_status moe_route(const moe_config* cfg, const float* logits, const float* sel_bias, int32_t* topk_ids,
                     float* topk_w, void* stream) {
  MOE_TRY(validate(cfg));
  if (cfg->T > 0) {
    MOE_TRY(check_ptr(logits, 4));
    MOE_TRY(check_ptr(topk_ids, 4));
    MOE_TRY(check_ptr(topk_w, 4));
  }
  MOE_TRY(check_opt_ptr(sel_bias, 4));
  return launch_route(*cfg, logits, sel_bias, topk_ids, topk_w, as_stream(stream));
}

moe_status moe_dispatch_layout(const moe_config* cfg, const int32_t* topk_ids, int32_t* counts, int32_t* kept,
                               int32_t* offsets, int32_t* slot, int32_t* row_src, int64_t* n_ij,
                               int64_t* rank_bytes, moe_layout_stats* stats, void* workspace,
                               size_t workspace_bytes, void* stream) {
  MOE_TRY(validate(cfg));
  if (cfg->T > 0) {
    MOE_TRY(check_ptr(topk_ids, 4));
    MOE_TRY(check_ptr(slot, 4));
  }
  if (rows_of(*cfg) > 0) MOE_TRY(check_ptr(row_src, 4));
  MOE_TRY(check_ptr(counts, 4));
  MOE_TRY(check_ptr(kept, 4));
  MOE_TRY(check_ptr(offsets, 4));
  MOE_TRY(check_ptr(n_ij, 8));
  MOE_TRY(check_ptr(rank_bytes, 8));
  MOE_TRY(check_ptr(stats, 8));
  MOE_TRY(check_ptr(workspace, 256));
  if (workspace_bytes < layout_scratch_bytes((int64_t)cfg->T * cfg->K, nphys(*cfg))) return MOE_ERR_WORKSPACE_TOO_SMALL;
  return launch_layout(*cfg, topk_ids, counts, kept, offsets, slot, row_src, n_ij, rank_bytes, stats, workspace,
                       as_stream(stream));
}

moe_status moe_dispatch_layout_static(const moe_config* cfg, const int32_t* topk_ids, int32_t* counts,
                                      int32_t* kept, int32_t* offsets, int32_t* slot, int32_t* row_src,
                                      int64_t* n_ij, int64_t* rank_bytes, moe_layout_stats* stats, void* stream) {
  MOE_TRY(validate(cfg));
  if (cfg->T > 0) {
    MOE_TRY(check_ptr(topk_ids, 4));
    MOE_TRY(check_ptr(slot, 4));
  }
  if (rows_of(*cfg) > 0) MOE_TRY(check_ptr(row_src, 4));
  MOE_TRY(check_ptr(counts, 4));
  MOE_TRY(check_ptr(kept, 4));
  MOE_TRY(check_ptr(offsets, 4));
  MOE_TRY(check_ptr(n_ij, 8));
  MOE_TRY(check_ptr(rank_bytes, 8));
  MOE_TRY(check_ptr(stats, 8));
  const int64_t A = (int64_t)cfg->T * cfg->K;
  if (layout_scratch_bytes(A, nphys(*cfg)) > MOE_LAYOUT_STATIC_SCRATCH_BYTES) return MOE_ERR_WORKSPACE_TOO_SMALL;
  void* scratch = nullptr;
  MOE_TRY(static_layout_scratch(&scratch));
  // the counters and tile flags must start at zero (the array keeps the
  // previous call's contents); the per-tile sums are written before they are read
  CUDA_TRY(cudaMemsetAsync(scratch, 0, layout_scratch_zero_bytes(A), as_stream(stream)));
  return launch_layout(*cfg, topk_ids, counts, kept, offsets, slot, row_src, n_ij, rank_bytes, stats, scratch,
                       as_stream(stream));
}

moe_status moe_permute(const moe_config* cfg, const void* x, const int32_t* slot, const int32_t* row_src, void* xp,
                       void* stream) {
  MOE_TRY(validate(cfg));
  if (cfg->T > 0) {
    MOE_TRY(check_dtype_ptr(x));
    MOE_TRY(check_ptr(slot, 4));
  }
  if (rows_of(*cfg) > 0) MOE_TRY(check_dtype_ptr(xp));
  if (cfg->pad && rows_of(*cfg) > 0) MOE_TRY(check_ptr(row_src, 4));
  return launch_permute(*cfg, x, slot, row_src, xp, as_stream(stream));
}

moe_status moe_grouped_ffn(const moe_config* cfg, const void* xp, const int32_t* offsets, const int32_t* kept,
                           const void* w13, const void* w2, void* yp, void* workspace, size_t workspace_bytes,
                           void* stream) {
  MOE_TRY(validate(cfg));
  if (rows_of(*cfg) > 0) {
    MOE_TRY(check_dtype_ptr(xp));
    MOE_TRY(check_dtype_ptr(yp));
  }
  MOE_TRY(check_ptr(offsets, 4));
  MOE_TRY(check_ptr(kept, 4));
  MOE_TRY(check_dtype_ptr(w13));
  MOE_TRY(check_dtype_ptr(w2));
  MOE_TRY(check_ptr(workspace, 256));
  if (workspace_bytes < ffn_ws_bytes(*cfg)) return MOE_ERR_WORKSPACE_TOO_SMALL;
  return launch_ffn(*cfg, xp, offsets, kept, nullptr, nphys(*cfg), w13, w2, yp, static_cast<char*>(workspace) + 256,
                    as_stream(stream));
}

moe_status moe_grouped_ffn_combine(const moe_config* cfg, const void* xp, const int32_t* offsets,
                                   const int32_t* kept, const void* w13, const void* w2, const int32_t* row_src,
                                   const int32_t* slot, const float* topk_w, void* yp, void* y, void* workspace,
                                   size_t workspace_bytes, void* stream) {
  MOE_TRY(validate(cfg));
  if (cfg->dtype != MOE_BF16 || cfg->capacity != 0 || cfg->n_redundant != 0) return MOE_ERR_UNSUPPORTED;
  if (expected_rows_per_expert(*cfg) > MOE_FFN_SWAP_MAX_ROWS) return MOE_ERR_UNSUPPORTED;
  if ((int64_t)cfg->E * 2 * cfg->I >= INT32_MAX || (int64_t)cfg->E * cfg->h >= INT32_MAX) return MOE_ERR_UNSUPPORTED;
  if (cfg->T > 0) {
    MOE_TRY(check_dtype_ptr(xp));
    MOE_TRY(check_dtype_ptr(yp));
    MOE_TRY(check_dtype_ptr(y));
    MOE_TRY(check_ptr(row_src, 4));
    MOE_TRY(check_ptr(slot, 4));
    MOE_TRY(check_ptr(topk_w, 4));
  }
  MOE_TRY(check_ptr(offsets, 4));
  MOE_TRY(check_ptr(kept, 4));
  MOE_TRY(check_dtype_ptr(w13));
  MOE_TRY(check_dtype_ptr(w2));
  MOE_TRY(check_ptr(workspace, 256));
  if (workspace_bytes < ffn_combine_ws_bytes(*cfg)) return MOE_ERR_WORKSPACE_TOO_SMALL;
  if (cfg->T == 0) return MOE_OK;
  FusedCombine fc;
  fc.row_src = row_src;
  fc.slot = slot;
  fc.topk_w = topk_w;
  fc.y = y;
  fc.arrive = reinterpret_cast<uint32_t*>(static_cast<char*>(workspace) + ffn_ws_bytes(*cfg));
  return launch_ffn_grouped<kFgTileRows, kFgStages>(*cfg, xp, offsets, kept, nullptr, cfg->E, w13, w2, yp,
                                                                 static_cast<char*>(workspace) + 256,
                                                                 as_stream(stream), nullptr, &fc);
}

moe_status moe_combine(const moe_config* cfg, const void* yp, const int32_t* slot, const float* topk_w, void* y,
                       void* stream) {
  MOE_TRY(validate(cfg));
  if (cfg->T > 0) {
    MOE_TRY(check_ptr(slot, 4));
    MOE_TRY(check_ptr(topk_w, 4));
    MOE_TRY(check_dtype_ptr(y));
    if (rows_of(*cfg) > 0) MOE_TRY(check_dtype_ptr(yp));
  }
  return launch_combine(*cfg, yp, slot, topk_w, nullptr, y, as_stream(stream));
}

moe_status moe_layer_forward(const moe_config* cfg, const void* x, const void* w_r, const float* logit_offset,
                             const float* sel_bias, const void* w13, const void* w2, void* y,
                             const moe_layer_out* out, void* workspace, size_t workspace_bytes, void* stream) {
  MOE_TRY(validate(cfg));
  if (cfg->T > 0) {
    MOE_TRY(check_dtype_ptr(x));
    MOE_TRY(check_dtype_ptr(y));
  }
  MOE_TRY(check_layer_ptrs(*cfg, x, w_r, logit_offset, sel_bias, w13, w2));
  MOE_TRY(check_ptr(workspace, 256));
  if (cfg->n_redundant > 0) return MOE_ERR_INVALID_ARG;  // replicas need a plan: moe_layer_forward_eplb
  const LayerBuffers b = carve_layer(*cfg, workspace, false);
  if (workspace_bytes < b.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  return layer_core(*cfg, x, w_r, logit_offset, sel_bias, w13, w2, nullptr, nullptr, y, out, b, as_stream(stream));
}

moe_status moe_layer_forward_host(const moe_config* cfg, const void* x_host, const void* w_r,
                                  const float* logit_offset, const float* sel_bias, const void* w13, const void* w2,
                                  void* y_host, void* workspace, size_t workspace_bytes, void* stream) {
  MOE_TRY(validate(cfg));
  if (cfg->T > 0 && (x_host == nullptr || y_host == nullptr)) return MOE_ERR_INVALID_ARG;
  if (cfg->n_redundant > 0) return MOE_ERR_INVALID_ARG;  // replicas need a plan: moe_layer_forward_eplb
  MOE_TRY(check_layer_ptrs(*cfg, x_host, w_r, logit_offset, sel_bias, w13, w2));
  MOE_TRY(check_ptr(workspace, 256));
  const LayerBuffers b = carve_layer(*cfg, workspace, true);
  if (workspace_bytes < b.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  const cudaStream_t st = as_stream(stream);
  const size_t bytes = (size_t)cfg->T * cfg->h * ds_of(*cfg);
  if (bytes > 0) CUDA_TRY(cudaMemcpyAsync(b.xdev, x_host, bytes, cudaMemcpyHostToDevice, st));
  MOE_TRY(layer_core(*cfg, b.xdev, w_r, logit_offset, sel_bias, w13, w2, nullptr, nullptr, b.ydev, nullptr, b, st));
  if (bytes > 0) CUDA_TRY(cudaMemcpyAsync(y_host, b.ydev, bytes, cudaMemcpyDeviceToHost, st));
  return MOE_OK;
}

moe_status moe_shared_ffn(const moe_config* cfg, const void* x, const void* w13s, const void* w2s, void* ys,
                          void* workspace, size_t workspace_bytes, void* stream) {
  MOE_TRY(validate(cfg));
  if (cfg->shared_I <= 0) return MOE_ERR_INVALID_ARG;
  if (cfg->T > 0) {
    MOE_TRY(check_dtype_ptr(x));
    MOE_TRY(check_dtype_ptr(ys));
  }
  MOE_TRY(check_dtype_ptr(w13s));
  MOE_TRY(check_dtype_ptr(w2s));
  MOE_TRY(check_ptr(workspace, 256));
  if (workspace_bytes < shared_ws_bytes(*cfg)) return MOE_ERR_WORKSPACE_TOO_SMALL;
  return launch_shared_ffn(*cfg, x, w13s, w2s, ys, static_cast<char*>(workspace) + 256, as_stream(stream));
}

moe_status moe_combine_add(const moe_config* cfg, const void* yp, const int32_t* slot, const float* topk_w,
                           const void* ys, void* y, void* stream) {
  MOE_TRY(validate(cfg));
  if (cfg->T > 0) {
    MOE_TRY(check_ptr(slot, 4));
    MOE_TRY(check_ptr(topk_w, 4));
    MOE_TRY(check_dtype_ptr(ys));
    MOE_TRY(check_dtype_ptr(y));
    if (rows_of(*cfg) > 0) MOE_TRY(check_dtype_ptr(yp));
  }
  return launch_combine(*cfg, yp, slot, topk_w, ys, y, as_stream(stream));
}

moe_status moe_block_forward(const moe_config* cfg, const void* x, const void* w_r, const float* logit_offset,
                             const float* sel_bias, const void* w13, const void* w2, const void* w13s,
                             const void* w2s, void* y, const moe_layer_out* out, void* workspace,
                             size_t workspace_bytes, void* stream) {
  MOE_TRY(validate(cfg));
  if (cfg->shared_I <= 0 || cfg->n_redundant > 0) return MOE_ERR_INVALID_ARG;
  if (cfg->T > 0) {
    MOE_TRY(check_dtype_ptr(x));
    MOE_TRY(check_dtype_ptr(y));
  }
  MOE_TRY(check_layer_ptrs(*cfg, x, w_r, logit_offset, sel_bias, w13, w2));
  MOE_TRY(check_dtype_ptr(w13s));
  MOE_TRY(check_dtype_ptr(w2s));
  MOE_TRY(check_ptr(workspace, 256));
  const LayerBuffers b = carve_layer(*cfg, workspace, false, true);
  if (workspace_bytes < b.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  return layer_core(*cfg, x, w_r, logit_offset, sel_bias, w13, w2, w13s, w2s, y, out, b, as_stream(stream));
}

moe_status moe_block_forward_host(const moe_config* cfg, const void* x_host, const void* w_r,
                                  const float* logit_offset, const float* sel_bias, const void* w13,
                                  const void* w2, const void* w13s, const void* w2s, void* y_host,
                                  void* workspace, size_t workspace_bytes, void* stream) {
  MOE_TRY(validate(cfg));
  if (cfg->shared_I <= 0 || cfg->n_redundant > 0) return MOE_ERR_INVALID_ARG;
  if (cfg->T > 0 && (x_host == nullptr || y_host == nullptr)) return MOE_ERR_INVALID_ARG;
  MOE_TRY(check_layer_ptrs(*cfg, x_host, w_r, logit_offset, sel_bias, w13, w2));
  MOE_TRY(check_dtype_ptr(w13s));
  MOE_TRY(check_dtype_ptr(w2s));
  MOE_TRY(check_ptr(workspace, 256));
  const LayerBuffers b = carve_layer(*cfg, workspace, true, true);
  if (workspace_bytes < b.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  const cudaStream_t st = as_stream(stream);
  const size_t bytes = (size_t)cfg->T * cfg->h * ds_of(*cfg);
  if (bytes > 0) CUDA_TRY(cudaMemcpyAsync(b.xdev, x_host, bytes, cudaMemcpyHostToDevice, st));
  MOE_TRY(layer_core(*cfg, b.xdev, w_r, logit_offset, sel_bias, w13, w2, w13s, w2s, b.ydev, nullptr, b, st));
  if (bytes > 0) CUDA_TRY(cudaMemcpyAsync(y_host, b.ydev, bytes, cudaMemcpyDeviceToHost, st));
  return MOE_OK;
}

moe_status moe_eplb_plan(int32_t E, int32_t ep_size, int32_t n_redundant, const int64_t* counts,
                         int32_t* rep_offsets, int32_t* rep_phys, int32_t* phys_to_log, int64_t* rank_load) {
  if (E < 1 || ep_size < 1 || n_redundant < 0 || (int64_t)E + n_redundant > 1024) return MOE_ERR_INVALID_ARG;
  if ((E + n_redundant) % ep_size != 0) return MOE_ERR_INVALID_ARG;
  if (counts == nullptr || rep_offsets == nullptr || rep_phys == nullptr || phys_to_log == nullptr)
    return MOE_ERR_INVALID_ARG;
  for (int e = 0; e < E; ++e)
    if (counts[e] < 0 || counts[e] > ((int64_t)1 << 40)) return MOE_ERR_INVALID_ARG;
  const int P = E + n_redundant, slots = P / ep_size;
  // replication: each redundant replica to the largest load per replica
  std::vector<int64_t> n_rep(E, 1);
  for (int i = 0; i < n_redundant; ++i) {
    int best = 0;
    for (int e = 1; e < E; ++e)
      if (counts[e] * n_rep[best] > counts[best] * n_rep[e]) best = e;
    ++n_rep[best];
  }
  // replicas with the even split of their expert's count; heaviest first
  struct Rep {
    int64_t load;
    int e, r;
  };
  std::vector<Rep> reps;
  reps.reserve(P);
  for (int e = 0; e < E; ++e)
    for (int r = 0; r < n_rep[e]; ++r)
      reps.push_back({counts[e] / n_rep[e] + (r < counts[e] % n_rep[e] ? 1 : 0), e, r});
  std::sort(reps.begin(), reps.end(), [](const Rep& a, const Rep& b) {
    if (a.load != b.load) return a.load > b.load;
    if (a.e != b.e) return a.e < b.e;
    return a.r < b.r;
  });
  // placement: least loaded rank with a free slot, ties to the lower rank
  std::vector<int64_t> load(ep_size, 0);
  std::vector<int> fill(ep_size, 0);
  rep_offsets[0] = 0;
  for (int e = 0; e < E; ++e) rep_offsets[e + 1] = rep_offsets[e] + (int32_t)n_rep[e];
  for (const Rep& rp : reps) {
    int best = -1;
    for (int j = 0; j < ep_size; ++j)
      if (fill[j] < slots && (best < 0 || load[j] < load[best])) best = j;
    const int phys = best * slots + fill[best];
    ++fill[best];
    load[best] += rp.load;
    rep_phys[rep_offsets[rp.e] + rp.r] = phys;
    phys_to_log[phys] = rp.e;
  }
  if (rank_load != nullptr)
    for (int j = 0; j < ep_size; ++j) rank_load[j] = load[j];
  return MOE_OK;
}

moe_status moe_eplb_map(const moe_config* cfg, const int32_t* topk_ids, const int32_t* rep_offsets,
                        const int32_t* rep_phys, int32_t* phys_ids, void* stream) {
  MOE_TRY(validate(cfg));
  if (cfg->T > 0) {
    MOE_TRY(check_ptr(topk_ids, 4));
    MOE_TRY(check_ptr(phys_ids, 4));
  }
  MOE_TRY(check_ptr(rep_offsets, 4));
  MOE_TRY(check_ptr(rep_phys, 4));
  EplbDev plan;
  plan.rep_offsets = rep_offsets;
  plan.rep_phys = rep_phys;
  return launch_eplb_map(*cfg, topk_ids, plan, phys_ids, as_stream(stream));
}

moe_status moe_grouped_ffn_mapped(const moe_config* cfg, const void* xp, const int32_t* offsets, const int32_t* kept,
                                  const int32_t* phys_to_log, const void* w13, const void* w2, void* yp,
                                  void* workspace, size_t workspace_bytes, void* stream) {
  MOE_TRY(validate(cfg));
  if (rows_of(*cfg) > 0) {
    MOE_TRY(check_dtype_ptr(xp));
    MOE_TRY(check_dtype_ptr(yp));
  }
  MOE_TRY(check_ptr(offsets, 4));
  MOE_TRY(check_ptr(kept, 4));
  MOE_TRY(check_ptr(phys_to_log, 4));
  MOE_TRY(check_dtype_ptr(w13));
  MOE_TRY(check_dtype_ptr(w2));
  MOE_TRY(check_ptr(workspace, 256));
  if (workspace_bytes < ffn_ws_bytes(*cfg)) return MOE_ERR_WORKSPACE_TOO_SMALL;
  return launch_ffn(*cfg, xp, offsets, kept, phys_to_log, cfg->E, w13, w2, yp, static_cast<char*>(workspace) + 256,
                    as_stream(stream));
}

moe_status moe_layer_forward_eplb(const moe_config* cfg, const void* x, const void* w_r, const float* logit_offset,
                                  const float* sel_bias, const void* w13, const void* w2, const int32_t* rep_offsets,
                                  const int32_t* rep_phys, const int32_t* phys_to_log, void* y,
                                  const moe_layer_out* out, void* workspace, size_t workspace_bytes, void* stream) {
  MOE_TRY(validate(cfg));
  if (cfg->T > 0) {
    MOE_TRY(check_dtype_ptr(x));
    MOE_TRY(check_dtype_ptr(y));
  }
  MOE_TRY(check_layer_ptrs(*cfg, x, w_r, logit_offset, sel_bias, w13, w2));
  MOE_TRY(check_ptr(rep_offsets, 4));
  MOE_TRY(check_ptr(rep_phys, 4));
  MOE_TRY(check_ptr(phys_to_log, 4));
  MOE_TRY(check_ptr(workspace, 256));
  const LayerBuffers b = carve_layer(*cfg, workspace, false);
  if (workspace_bytes < b.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  EplbDev plan;
  plan.rep_offsets = rep_offsets;
  plan.rep_phys = rep_phys;
  plan.phys_to_log = phys_to_log;
  return layer_core(*cfg, x, w_r, logit_offset, sel_bias, w13, w2, nullptr, nullptr, y, out, b, as_stream(stream),
                    plan);
}

moe_status moe_grouped_ffn_gather(const moe_config* cfg, const void* x, const int32_t* row_src,
                                  const int32_t* offsets, const int32_t* kept, const void* w13, const void* w2,
                                  void* yp, void* workspace, size_t workspace_bytes, void* stream) {
  MOE_TRY(validate(cfg));
  if (cfg->T > 0) MOE_TRY(check_dtype_ptr(x));
  if (rows_of(*cfg) > 0) {
    MOE_TRY(check_ptr(row_src, 4));
    MOE_TRY(check_dtype_ptr(yp));
  }
  MOE_TRY(check_ptr(offsets, 4));
  MOE_TRY(check_ptr(kept, 4));
  MOE_TRY(check_dtype_ptr(w13));
  MOE_TRY(check_dtype_ptr(w2));
  MOE_TRY(check_ptr(workspace, 256));
  if (workspace_bytes < ffn_ws_bytes(*cfg)) return MOE_ERR_WORKSPACE_TOO_SMALL;
  return launch_ffn_gather(*cfg, x, row_src, offsets, kept, nullptr, nphys(*cfg), w13, w2, yp,
                           static_cast<char*>(workspace) + 256, as_stream(stream));
}

moe_status fp8_config_ok(const moe_config* cfg) {
  MOE_TRY(validate(cfg));
  if (cfg->dtype != MOE_BF16 || cfg->h % 128 != 0 || cfg->I % 128 != 0) return MOE_ERR_UNSUPPORTED;
  if (cfg->shared_I != 0) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

moe_status moe_quantize_fp8(int64_t rows, int32_t cols, int32_t dtype, const void* src, uint8_t* codes,
                            float* scales, void* stream) {
  if (rows < 0 || cols <= 0 || cols % 16 != 0) return MOE_ERR_INVALID_ARG;
  if (dtype != MOE_F32 && dtype != MOE_BF16) return MOE_ERR_INVALID_ARG;
  if (rows == 0) return MOE_OK;
  MOE_TRY(check_dtype_ptr(src));
  MOE_TRY(check_dtype_ptr(codes));
  MOE_TRY(check_ptr(scales, 4));
  int64_t blocks = (rows + 7) / 8;
  if (blocks > (int64_t)device_info().sms * 16) blocks = (int64_t)device_info().sms * 16;
  if (dtype == MOE_BF16)
    (void)launch_k(quant_rows_kernel<__nv_bfloat16>, (unsigned)blocks, 256, 0, as_stream(stream), 
        static_cast<const __nv_bfloat16*>(src), rows, cols, codes, scales);
  else
    (void)launch_k(quant_rows_kernel<float>, (unsigned)blocks, 256, 0, as_stream(stream), static_cast<const float*>(src), rows,
                                                                              cols, codes, scales);
  CUDA_TRY(launched());
  return MOE_OK;
}

moe_status moe_permute_fp8(const moe_config* cfg, const void* x, const int32_t* slot, uint8_t* xq, float* sx,
                           void* stream) {
  MOE_TRY(fp8_config_ok(cfg));
  if (cfg->T > 0) {
    MOE_TRY(check_dtype_ptr(x));
    MOE_TRY(check_ptr(slot, 4));
  }
  if (rows_of(*cfg) > 0) {
    MOE_TRY(check_dtype_ptr(xq));
    MOE_TRY(check_ptr(sx, 4));
  }
  return launch_permute_fp8(*cfg, x, slot, xq, sx, as_stream(stream));
}

moe_status moe_grouped_ffn_fp8(const moe_config* cfg, const uint8_t* xq, const float* sx, const int32_t* offsets,
                               const int32_t* kept, const uint8_t* w13q, const float* s13, const uint8_t* w2q,
                               const float* s2, void* yp, void* workspace, size_t workspace_bytes, void* stream) {
  MOE_TRY(fp8_config_ok(cfg));
  if (cfg->n_redundant != 0) return MOE_ERR_UNSUPPORTED;
  if (rows_of(*cfg) > 0) {
    MOE_TRY(check_dtype_ptr(xq));
    MOE_TRY(check_ptr(sx, 4));
    MOE_TRY(check_dtype_ptr(yp));
  }
  MOE_TRY(check_ptr(offsets, 4));
  MOE_TRY(check_ptr(kept, 4));
  MOE_TRY(check_dtype_ptr(w13q));
  MOE_TRY(check_dtype_ptr(w2q));
  MOE_TRY(check_ptr(s13, 4));
  MOE_TRY(check_ptr(s2, 4));
  MOE_TRY(check_ptr(workspace, 256));
  if (workspace_bytes < ffn_fp8_ws_bytes(*cfg)) return MOE_ERR_WORKSPACE_TOO_SMALL;
  return launch_ffn_fp8(*cfg, xq, sx, offsets, kept, nullptr, cfg->E, w13q, s13, w2q, s2, yp, workspace,
                        as_stream(stream));
}

moe_status moe_layer_forward_fp8(const moe_config* cfg, const void* x, const void* w_r, const float* logit_offset,
                                 const float* sel_bias, const uint8_t* w13q, const float* s13, const uint8_t* w2q,
                                 const float* s2, void* y, const moe_layer_out* out, void* workspace,
                                 size_t workspace_bytes, void* stream) {
  MOE_TRY(fp8_config_ok(cfg));
  if (cfg->n_redundant != 0) return MOE_ERR_UNSUPPORTED;
  if (cfg->T > 0) {
    MOE_TRY(check_dtype_ptr(x));
    MOE_TRY(check_dtype_ptr(y));
  }
  MOE_TRY(check_dtype_ptr(w_r));
  MOE_TRY(check_opt_ptr(logit_offset, 4));
  MOE_TRY(check_opt_ptr(sel_bias, 4));
  MOE_TRY(check_dtype_ptr(w13q));
  MOE_TRY(check_dtype_ptr(w2q));
  MOE_TRY(check_ptr(s13, 4));
  MOE_TRY(check_ptr(s2, 4));
  MOE_TRY(check_ptr(workspace, 256));
  const LayerBuffers b = carve_layer(*cfg, workspace, false, false, true);
  if (workspace_bytes < b.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  Fp8Weights q;
  q.w13q = w13q;
  q.s13 = s13;
  q.w2q = w2q;
  q.s2 = s2;
  return layer_core(*cfg, x, w_r, logit_offset, sel_bias, nullptr, nullptr, nullptr, nullptr, y, out, b,
                    as_stream(stream), EplbDev(), q);
}

moe_status moe_check(void* stream) {
  if (cudaStreamSynchronize(as_stream(stream)) != cudaSuccess) {
    (void)cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
  uint32_t err = 0;
  CUDA_TRY(cudaMemcpyFromSymbol(&err, g_dev_error, sizeof(err)));
  if (err == 0) return MOE_OK;
  const uint32_t zero = 0;
  CUDA_TRY(cudaMemcpyToSymbol(g_dev_error, &zero, sizeof(zero)));
  return (err & kErrTimeout) ? MOE_ERR_DEVICE_TIMEOUT : MOE_ERR_DEVICE_BAD_INDEX;
}

}  // extern "C"
