// Grouped SwiGLU FFN over ragged expert segments on the tcgen05 tensor cores,
// with the expert's WEIGHT rows as the MMA's M operand and its TOKEN rows as N.
//
// An expert of an MoE layer sees few tokens (DeepSeek-V3 at 4096 tokens: ~128
// rows per expert; decode: 0-32), far fewer than its weight rows.  With tokens
// as M (128-row tiles) an expert of 130 rows costs two full 128-row MMA
// blocks; with tokens as N the MMA width only rounds up to 16.  So a tile is
//   (expert e, feature tile ft, token tile tt)
// and computes, for two 128-row weight sub-tiles A0 and A1,
//   D0[f, r] = sum_k A0[f, k] X[r, k],   D1[f, r] = sum_k A1[f, k] X[r, k]
// over the tile's token rows r:
//   gate/up (SwiGLU epilogue): A0 = gate rows 128ft.., A1 = the matching up
//     rows I+128ft..; out[r, 128ft + f] = bf16(silu(D0) * D1) (the intermediate);
//   down (store epilogue): A0 = rows 256ft.., A1 = rows 256ft+128..;
//     out[r, 256ft + f] = bf16(D0), out[r, 256ft + 128 + f] = bf16(D1).
// A token tile holds up to BT rows (128 <= BT <= 256); both MMAs of a k-step
// take all of them at once (N = rows rounded up to 16).  TMEM holds two
// 256-column slots: a tile of at most 128 rows keeps D0 and D1 in one slot
// (columns 0..127 and 128..255 of it), so such tiles alternate slots and one
// tile's epilogue overlaps the next tile's MMAs; a longer tile keeps D0 in slot
// 0 and D1 in slot 1.  An expert with more than BT rows is split into equal
// token tiles.
//
// Roles (224 threads), one persistent CTA per SM over a static round-robin of
// tiles ordered (expert, feature tile, token tile), so the token tiles sharing
// a weight tile run on neighbouring SMs and the second read hits L2:
//   warp 0      one thread issues the TMA loads of the two 128x64 weight boxes
//               of every k-block into the weight part of an ST-deep ring;
//   warp 6      issues the loads of the tile's token rows (boxes of 128, 64, 32
//               and 16 rows) into the token part of the same stage; when the
//               rows are gathered from x (GATHER), warps 6..6+ST-1 each own one
//               stage and fill its token part with 16-byte cp.async copies of
//               the rows that row_src names;
//   warp 1      allocates 512 TMEM columns; one thread issues tcgen05.mma
//               (M=128, N = the tile's rows rounded up to 16, K=16), two per
//               k-step, once the stage holds the k-block;
//   warps 2..5  drain the accumulators with tcgen05.ld (warp w reads TMEM lanes
//               32*(w%4).. = 32 features), transpose 32 features x 32 tokens
//               through shared memory and store 64-byte row pieces.
// The weights stream from DRAM while the token rows are mostly L2 hits.  A
// stage has one full barrier (the weight producer's arrival with its bytes and
// the token side's) and one empty barrier (one tcgen05.commit), so the issuing
// thread waits once and commits once per k-block.  That thread is the MMA
// pipe's only feeder, and with N <= 160 a k-block's eight MMAs take about 500
// cycles: every cycle it spends elsewhere leaves the pipe idle.  So it tests
// the next stage's barrier while the current MMAs run, keeps the descriptors
// as base + stage offsets, and unrolls its loop over the ring when a tile's
// k-blocks fill whole rounds of it (the launcher's choice of tile and ring and
// the measurements behind it are beside kFgTileRows).
// Rows past a tile's end are computed and masked on store.  Every wait is
// bounded; a wait that runs out raises the sticky error, and the CTA drains its
// copies and MMAs, frees TMEM and exits.
#pragma once

#include "tc_gemm.cuh"

namespace moe {

constexpr int kFgThreads = 224;

// Threads of a grouped-FFN CTA: 7 warps, plus ST - 1 more when the token rows
// are gathered (one gather warp per stage).
template <bool GATHER, int ST>
struct FgThreads {
  static constexpr int value = GATHER ? kFgThreads + 32 * (ST - 1) : kFgThreads;
};
constexpr int kFgXsStride = 40;  // bf16 per row of a warp's 32x32 transpose buffer (80 B: conflict-free 16-B reads)

// A stage holds one k-block: the two weight boxes, then (in a second array)
// the token rows.
template <int BT, int ST>
struct FgShape {
  static_assert(BT % 16 == 0 && BT >= 128 && BT <= 256, "token tiles of 128..256 rows");
  static constexpr uint32_t kWBytes = 128 * kTcBK * 2;            // one 128-row weight box: 16 KB
  static constexpr uint32_t kWStage = 2 * kWBytes;                // both boxes of a k-block
  static constexpr uint32_t kXStage = BT * kTcBK * 2;             // BT token rows of 128 bytes
  static_assert(kXStage % 1024 == 0, "token stages start on 1024-byte swizzle atoms");
  static constexpr size_t kXsBytes = 4 * 32 * kFgXsStride * 2;    // transpose buffers of the 4 epilogue warps
  static constexpr size_t kDynSmem = (size_t)ST * (kWStage + kXStage) + kXsBytes + 1024;
};

struct FgParams {
  const int32_t* offsets;   // [E+1]
  const int32_t* kept;      // [E]
  int E;
  int f_tiles;              // feature tiles per expert: ceil(I/128) (gate/up) or ceil(h/256) (down)
  int k_blocks;             // reduction length / 64
  int64_t a_rows;           // weight rows per expert: 2I (gate/up) or h (down)
  int up_rows;              // gate/up: I
  int n_valid;              // output features: I or h
  __nv_bfloat16* out;       // [R, ldo]
  int64_t ldo;
  const int32_t* w_map;     // expert -> its weight matrices (replicas share a logical expert's), or null
  const float* w_scale;     // FP8: scale of every weight row [experts * a_rows]
  const float* x_scale;     // FP8: scale of every token row [R]
  const int32_t* row_src;   // gather: token of every permuted row [R] (rows are read from x)
  const uint8_t* gather_x;  // gather: x [T, ldx_bytes]
  int64_t ldx_bytes;        // gather: bytes per row of x
  // combine fused into the down epilogue (dropless layers): the token of every
  // row (row_src), each token's K slots and weights, the output y [T, n_valid]
  // and one arrival counter per (token, 32-feature group), zero between calls
  const int32_t* slot;      // [T, K]
  const float* topk_w;      // [T, K]
  int K;
  int groups;               // n_valid / 32
  __nv_bfloat16* y;
  uint32_t* arrive;         // [T, groups]
};

// Tensor maps of the token rows with boxes of 128, 64, 32 and 16 rows.
struct FgTokenMaps {
  CUtensorMap m[4];
};

struct FgTile {
  int e, ft;
  int r0;          // first token row (absolute, in the permuted buffer)
  int n;           // token rows (1..BT)
};

// mbp[e] = token tiles of experts < e, mbp[E] = total.
template <int BT>
__device__ __forceinline__ FgTile fg_decode(int t, const int32_t* mbp, const FgParams& p) {
  int lo = 0, hi = p.E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (mbp[mid] * p.f_tiles <= t) lo = mid; else hi = mid - 1;
  }
  const int e = lo;
  const int local = t - mbp[e] * p.f_tiles;
  const int cnt = mbp[e + 1] - mbp[e];
  const int tt = local % cnt;
  const int kept = p.kept[e];
  const int base = kept / cnt, rem = kept % cnt;   // equal split: rows differ by at most one
  FgTile r;
  r.e = e;
  r.ft = local / cnt;
  r.r0 = p.offsets[e] + tt * base + min(tt, rem);
  r.n = base + (tt < rem ? 1 : 0);
  return r;
}

__device__ __forceinline__ uint32_t round16(int n) { return (uint32_t)((n + 15) & ~15); }

// 16-byte copy global -> shared through the LSU path (L1 bypassed).
__device__ __forceinline__ void cp_async16(uint32_t smem_dst, const void* gsrc) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_dst), "l"(gsrc) : "memory");
}

// Epilogue of one 32-token chunk: v (and u, SwiGLU) hold this warp's 32
// features x 32 tokens; the bf16 results are transposed through the warp's
// shared buffer and each lane stores the 64-byte piece of token row r0 + c + lane.
// The last of a token's K arrivals for one 32-feature group: y[t, feat0..+31]
// = sum over k = 0..K-1 of topk_w[t,k] * yp[slot[t,k], feat0..+31], float32
// fused multiply-adds in k order from 0 (the arithmetic of combine_kernel), the
// staged rows read from L2.
__device__ __forceinline__ void fg_combine_group(int64_t t, int feat0, const FgParams& p) {
  float acc[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) acc[i] = 0.0f;
  for (int k = 0; k < p.K; ++k) {
    const int32_t s = p.slot[t * p.K + k];
    const float w = p.topk_w[t * p.K + k];
    const uint4* src = reinterpret_cast<const uint4*>(p.out + (int64_t)s * p.ldo + feat0);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint4 v = __ldcg(src + q);
      const uint32_t wds[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&wds[i]);
        acc[8 * q + 2 * i] = fmaf(w, __low2float(b), acc[8 * q + 2 * i]);
        acc[8 * q + 2 * i + 1] = fmaf(w, __high2float(b), acc[8 * q + 2 * i + 1]);
      }
    }
  }
  store_bf16_row<32>(p.y + t * (int64_t)p.ldo + feat0, acc);
}

template <int EPI, bool FP8, bool COMB = false>
__device__ __forceinline__ void fg_chunk(const uint32_t* v, const uint32_t* u, int c, int n, int r0, int feat0,
                                         bool feat_ok, const FgParams& p, __nv_bfloat16* xs, float wsg, float wsu) {
  const int lane = threadIdx.x & 31;
  // FP8: token i's scale (lane i loads it; shuffled to every feature lane)
  const float xsc = (FP8 && c + lane < n) ? p.x_scale[r0 + c + lane] : 0.0f;
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    float g = __uint_as_float(v[i]);
    float uu = EPI == kTcSwiglu ? __uint_as_float(u[i]) : 0.0f;
    if (FP8) {
      const float xi = __shfl_sync(0xffffffffu, xsc, i);
      g = g * wsg * xi;
      uu = uu * wsu * xi;
    }
    // silu(g) * u with the fast exponential and division (about 2 ulp of
    // float32, far below the bf16 rounding of the result); the IEEE forms made
    // this loop the slowest part of the tile
    const float a = EPI == kTcSwiglu ? __fdividef(g, 1.0f + __expf(-g)) * uu : g;
    xs[i * kFgXsStride + lane] = __float2bfloat16_rn(a);
  }
  __syncwarp();
  if (feat_ok && c + lane < n) {
    const uint4* src = reinterpret_cast<const uint4*>(xs + lane * kFgXsStride);
    uint4* dst = reinterpret_cast<uint4*>(p.out + (int64_t)(r0 + c + lane) * p.ldo + feat0);
#pragma unroll
    for (int i = 0; i < 4; ++i) dst[i] = src[i];
    if (COMB) {
      // the row's piece is staged; count its arrival, and the K-th arrival
      // for this token and feature group sums the K staged pieces
      const int64_t t = p.row_src[r0 + c + lane];
      uint32_t* ctr = p.arrive + t * p.groups + (feat0 >> 5);
      __threadfence();
      if (atomicAdd(ctr, 1u) == (uint32_t)(p.K - 1)) {
        __threadfence();
        *ctr = 0u;   // every arrival of this call has come: ready for the next call
        fg_combine_group(t, feat0, p);
      }
    }
  }
  __syncwarp();
}

// Drains 32 features (this warp's TMEM lanes) x n tokens of one accumulator
// (columns col0.., and col_up.. for the SwiGLU's up half), two chunks in
// flight: the next chunk's tcgen05.ld runs while this one is transposed and
// stored.
template <int EPI, bool FP8, bool COMB = false>
__device__ __forceinline__ void fg_drain(uint32_t t_lane, uint32_t col0, uint32_t col_up, int n, int r0,
                                         int feat0, bool feat_ok, const FgParams& p, __nv_bfloat16* xs,
                                         float wsg = 1.0f, float wsu = 1.0f) {
  constexpr bool kUp = EPI == kTcSwiglu;
  uint32_t va[32], vb[32], ua[kUp ? 32 : 1], ub[kUp ? 32 : 1];
  tmem_ld<32>(t_lane + col0, va);
  if (kUp) tmem_ld<32>(t_lane + col_up, ua);
#pragma unroll 1
  for (int c = 0; c < n; c += 64) {
    tmem_ld_wait();
    tmem_regs_ready(va);
    if (kUp) tmem_regs_ready(ua);
    if (c + 32 < n) {
      tmem_ld<32>(t_lane + col0 + c + 32, vb);
      if (kUp) tmem_ld<32>(t_lane + col_up + c + 32, ub);
    }
    fg_chunk<EPI, FP8, COMB>(va, ua, c, n, r0, feat0, feat_ok, p, xs, wsg, wsu);
    if (c + 32 >= n) break;
    tmem_ld_wait();
    tmem_regs_ready(vb);
    if (kUp) tmem_regs_ready(ub);
    if (c + 64 < n) {
      tmem_ld<32>(t_lane + col0 + c + 64, va);
      if (kUp) tmem_ld<32>(t_lane + col_up + c + 64, ua);
    }
    fg_chunk<EPI, FP8, COMB>(vb, ub, c + 32, n, r0, feat0, feat_ok, p, xs, wsg, wsu);
  }
}

// The two MMAs of one K=16 step: D0 += A0 X^T and D1 += A1 X^T (k-th step of
// the stage: descriptors advance 32 bytes = 2 units).
template <bool FP8>
__device__ __forceinline__ void fg_mma_step(uint32_t c0, uint32_t c1, uint64_t dw0, uint64_t dw1, uint64_t dx,
                                            uint32_t idesc, uint32_t acc, int k) {
  if (FP8) {
    umma_e4m3(c0, dw0 + 2 * k, dx + 2 * k, idesc, acc);
    umma_e4m3(c1, dw1 + 2 * k, dx + 2 * k, idesc, acc);
  } else {
    umma_bf16(c0, dw0 + 2 * k, dx + 2 * k, idesc, acc);
    umma_bf16(c1, dw1 + 2 * k, dx + 2 * k, idesc, acc);
  }
}

// FP8: E4M3 operands (tcgen05.mma kind::f8f6f4), 128-element k-blocks (the
// same 128-byte rows), results scaled by weight-row and token scales.
// GATHER: the token rows are read straight from x through row_src, so the
// permutation needs no buffer of its own.  Warp 6 + g fills the token part of
// stage g with 16-byte cp.async copies into the 128-byte-swizzled layout the
// MMA expects, waits for its own copies, makes them visible to the tensor
// core's (async proxy) reads with fence.proxy.async, and then arrives on the
// stage's full barrier (all 32 lanes).
// COMBINE (down projection, dropless): the weighted combine fused into the
// epilogue (fg_chunk): expert rows are still staged in out (yp), and the last
// arrival of every (token, 32-feature group) writes y.
// After an abort the producers may have armed a stage's full barrier on one
// side only; once every role has stopped, thread 0 adds the missing side's
// arrivals and waits for the last armed phase of every stage, so no copy is
// still landing when the CTA's shared memory is released.
template <int EPI, int BT, int ST, bool FP8 = false, bool GATHER = false, bool COMBINE = false>
__global__ void __launch_bounds__(FgThreads<GATHER, ST>::value, 1)
    ffn_grouped_kernel(const __grid_constant__ CUtensorMap map_w, const __grid_constant__ FgTokenMaps maps,
                       FgParams p) {
  pdl_wait();
  const CUtensorMap* map_x = maps.m;
  using S = FgShape<BT, ST>;
  constexpr uint32_t kXArrivals = GATHER ? 32u : 1u;   // token-side arrivals per stage fill
  extern __shared__ uint8_t dyn_smem[];
  __shared__ __align__(8) uint64_t full[ST], empty[ST];
  __shared__ __align__(8) uint64_t tmem_full[2], tmem_empty[2], drain_bar;
  __shared__ uint32_t tmem_holder;
  __shared__ volatile uint32_t abort_flag;
  __shared__ volatile uint32_t armed_w[ST], armed_x[ST];   // fills of each stage by each side
  __shared__ int32_t mbp[1025];
  __shared__ int32_t scan_scratch[33];
  __shared__ int32_t src_rows[GATHER ? ST : 1][GATHER ? BT : 1];  // gather: per warp, source token of each row

  uint8_t* ring_w = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dyn_smem) + 1023) & ~uintptr_t(1023));
  uint8_t* ring_x = ring_w + (size_t)ST * S::kWStage;
  __nv_bfloat16* xs_all = reinterpret_cast<__nv_bfloat16*>(ring_x + (size_t)ST * S::kXStage);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // ---- per-expert token-tile prefix (every CTA computes it from kept)
  constexpr int NT = FgThreads<GATHER, ST>::value;
  for (int e = tid; e < p.E; e += NT) mbp[e] = (p.kept[e] + BT - 1) / BT;
  __syncthreads();
  const int32_t total_tt = block_exclusive_scan(mbp, p.E, scan_scratch);
  if (tid == 0) mbp[p.E] = total_tt;
  const int total_tiles = total_tt * p.f_tiles;

  if (tid == 0) {
    for (int s = 0; s < ST; ++s) {
      mbar_init(&full[s], 1 + kXArrivals);
      mbar_init(&empty[s], 1);
      armed_w[s] = 0;
      armed_x[s] = 0;
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tmem_full[a], 1);
      mbar_init(&tmem_empty[a], 128);
    }
    mbar_init(&drain_bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_holder)),
                 "r"(512)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = tmem_holder;

  if (warp == 0) {
    // ------------------------------------------------------------ weight producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      for (int t = blockIdx.x; t < total_tiles && !abort_flag; t += gridDim.x) {
        const FgTile tl = fg_decode<BT>(t, mbp, p);
        // weight rows of the tile's two 128-row boxes
        const int64_t we = p.w_map != nullptr ? p.w_map[tl.e] : tl.e;
        const int64_t a0 = we * p.a_rows + (EPI == kTcSwiglu ? 128 * tl.ft : 256 * tl.ft);
        const int64_t a1 = EPI == kTcSwiglu ? a0 + p.up_rows : a0 + 128;
        for (int kb = 0; kb < p.k_blocks; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, &abort_flag)) {
            abort_flag = 1;
            raise_error(kErrTimeout);
            break;
          }
          uint8_t* sw = ring_w + (size_t)stage * S::kWStage;
          const int kx = kb * (FP8 ? 128 : kTcBK);
          mbar_expect_tx(&full[stage], S::kWStage);
          tma_load_2d(sw, &map_w, kx, (int)a0, &full[stage]);
          tma_load_2d(sw + S::kWBytes, &map_w, kx, (int)a1, &full[stage]);
          armed_w[stage] = armed_w[stage] + 1u;
          if (++stage == ST) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    }
  } else if (!GATHER && warp == 6) {
    // ------------------------------------------------------------ token producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      for (int t = blockIdx.x; t < total_tiles && !abort_flag; t += gridDim.x) {
        const FgTile tl = fg_decode<BT>(t, mbp, p);
        const int n16 = (int)round16(tl.n);
        const uint32_t x_bytes = (uint32_t)n16 * (uint32_t)(kTcBK * 2);
        for (int kb = 0; kb < p.k_blocks; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, &abort_flag)) {
            abort_flag = 1;
            raise_error(kErrTimeout);
            break;
          }
          uint8_t* sx = ring_x + (size_t)stage * S::kXStage;
          const int kx = kb * (FP8 ? 128 : kTcBK);
          mbar_expect_tx(&full[stage], x_bytes);
          // round16(n) rows as boxes of 128 rows, then at most one each of 64, 32 and 16
          int b = 0;
          for (; b + 128 <= n16; b += 128) tma_load_2d(sx + b * (kTcBK * 2), &map_x[0], kx, tl.r0 + b, &full[stage]);
          if ((n16 - b) & 64) { tma_load_2d(sx + b * (kTcBK * 2), &map_x[1], kx, tl.r0 + b, &full[stage]); b += 64; }
          if ((n16 - b) & 32) { tma_load_2d(sx + b * (kTcBK * 2), &map_x[2], kx, tl.r0 + b, &full[stage]); b += 32; }
          if ((n16 - b) & 16) tma_load_2d(sx + b * (kTcBK * 2), &map_x[3], kx, tl.r0 + b, &full[stage]);
          armed_x[stage] = armed_x[stage] + 1u;
          if (++stage == ST) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    }
  } else if (GATHER && warp >= 6 && warp < 6 + ST) {
    // ------------------------------------------------------------ token gather (warp 6 + g fills stage g)
    // k-block j of the CTA's sequence uses stage j % ST, so this warp takes
    // every ST-th k-block.  Its copies are complete (cp.async.wait_group) and
    // fenced before it arrives, so nothing is in flight when it exits.
    const int g = warp - 6;
    int32_t* srow = src_rows[g];
    uint8_t* sx = ring_x + (size_t)g * S::kXStage;
    const uint32_t sx_u32 = smem_u32(sx);
    uint32_t phase = 0;
    int j = 0;   // k-blocks of the sequence before the current one
    bool ok = true;
    for (int t = blockIdx.x; t < total_tiles && ok; t += gridDim.x) {
      if (__shfl_sync(0xffffffffu, abort_flag != 0 ? 1 : 0, 0)) break;
      const FgTile tl = fg_decode<BT>(t, mbp, p);
      const int n16 = (int)round16(tl.n);
      // the first k-block of this tile that is ours
      int kb = ((g - j) % ST + ST) % ST;
      if (kb < p.k_blocks) {
        __syncwarp();
        for (int i = lane; i < n16; i += 32) {
          // rows past the tile's end repeat its first row (computed, masked on store)
          const int32_t src = p.row_src[tl.r0 + (i < tl.n ? i : 0)];
          srow[i] = src >= 0 ? src : 0;
        }
        __syncwarp();
      }
      for (; kb < p.k_blocks; kb += ST) {
        // every lane waits (each of its copies must follow the MMAs' reads of
        // the stage); the warp gives up together if any lane's wait ran out
        const bool w_ok = mbar_wait(&empty[g], phase ^ 1u, &abort_flag);
        if (!__all_sync(0xffffffffu, w_ok)) {
          if (lane == 0) {
            abort_flag = 1;
            raise_error(kErrTimeout);
          }
          ok = false;
          break;
        }
        // pair i = (row i / 8, 16-byte chunk i % 8) of the k-block's 128-byte row pieces
        const uint8_t* xk = p.gather_x + (size_t)kb * (kTcBK * 2);
        for (int i = lane; i < n16 * 8; i += 32) {
          const int r = i >> 3, c = i & 7;
          cp_async16(sx_u32 + (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4)),
                     xk + (size_t)srow[r] * (size_t)p.ldx_bytes + c * 16);
        }
        asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        mbar_arrive(&full[g]);
        __syncwarp();
        if (lane == 0) armed_x[g] = armed_x[g] + 1u;
        phase ^= 1u;
      }
      j += p.k_blocks;
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      // descriptors of stage 0's operands; stage s adds s stage sizes (start
      // addresses stay below 256 KB, so the 14-bit address field never carries)
      const uint64_t dwb = umma_desc_sw128(smem_u32(ring_w)), dxb = umma_desc_sw128(smem_u32(ring_x));
      int st = 0;
      uint32_t ph = 0;
      bool ready = false;        // full[st] already seen complete by the early test
      bool ok = true;
      int slot = 0;              // TMEM slot of the next tile of at most 128 rows
      uint32_t slot_phase = 0;   // bit s: uses of slot s so far, mod 2
      for (int t = blockIdx.x; t < total_tiles && ok && !abort_flag; t += gridDim.x) {
        const FgTile tl = fg_decode<BT>(t, mbp, p);
        const bool big = tl.n > 128;
        const uint32_t idesc = FP8 ? umma_idesc_e4m3(128, (int)round16(tl.n)) : umma_idesc_bf16(128, (int)round16(tl.n));
        // big: D0 = slot 0, D1 = slot 1; else D0, D1 = the two halves of `slot`
        const int s0 = big ? 0 : slot;
        const uint32_t c0 = tmem_base + (uint32_t)(s0 * 256), c1 = big ? tmem_base + 256u : c0 + 128u;
        ok = mbar_wait(&tmem_empty[s0], ((slot_phase >> s0) & 1u) ^ 1u, &abort_flag);
        if (ok && big) ok = mbar_wait(&tmem_empty[1], ((slot_phase >> 1) & 1u) ^ 1u, &abort_flag);
        if (!ok) break;
        tc_fence_after();
        if (st == 0 && p.k_blocks % ST == 0) {
          // whole groups of ST k-blocks starting at stage 0 (every tile when
          // k_blocks is a multiple of ST): unrolled over the stages, so stage
          // indices, descriptors and the next stage to test are constants and
          // the thread spends fewer cycles between k-blocks (MMA path alone:
          // 2.50 -> 2.10 ms at DeepSeek-V3 T=4096)
          for (int kb = 0; kb < p.k_blocks && ok; kb += ST) {
#pragma unroll
            for (int u = 0; u < ST; ++u) {
              if (!ready && !mbar_wait(&full[u], ph, &abort_flag)) {
                ok = false;
                break;
              }
              tc_fence_after();
              const uint64_t dw0 = dwb + (uint64_t)(u * (S::kWStage >> 4));
              const uint64_t dw1 = dw0 + (S::kWBytes >> 4);
              const uint64_t dx = dxb + (uint64_t)(u * (S::kXStage >> 4));
              fg_mma_step<FP8>(c0, c1, dw0, dw1, dx, idesc, (kb + u) != 0 ? 1u : 0u, 0);
              fg_mma_step<FP8>(c0, c1, dw0, dw1, dx, idesc, 1u, 1);
              ready = mbar_try_wait(&full[(u + 1) % ST], u + 1 == ST ? ph ^ 1u : ph);
              fg_mma_step<FP8>(c0, c1, dw0, dw1, dx, idesc, 1u, 2);
              fg_mma_step<FP8>(c0, c1, dw0, dw1, dx, idesc, 1u, 3);
              umma_commit(&empty[u]);
            }
            ph ^= 1u;
          }
        } else
        for (int kb = 0; kb < p.k_blocks; ++kb) {
          if (!ready && !mbar_wait(&full[st], ph, &abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t dw0 = dwb + (uint64_t)((uint32_t)st * (S::kWStage >> 4));
          const uint64_t dw1 = dw0 + (S::kWBytes >> 4);
          const uint64_t dx = dxb + (uint64_t)((uint32_t)st * (S::kXStage >> 4));
          const int nst = st + 1 == ST ? 0 : st + 1;
          const uint32_t nph = st + 1 == ST ? ph ^ 1u : ph;
          static_assert(kTcBK / 16 == 4, "four K=16 steps per k-block");
          fg_mma_step<FP8>(c0, c1, dw0, dw1, dx, idesc, kb != 0 ? 1u : 0u, 0);
          fg_mma_step<FP8>(c0, c1, dw0, dw1, dx, idesc, 1u, 1);
          // test the next stage while these MMAs run: a barrier that has
          // completed stays so until this thread releases the stage
          ready = mbar_try_wait(&full[nst], nph);
          fg_mma_step<FP8>(c0, c1, dw0, dw1, dx, idesc, 1u, 2);
          fg_mma_step<FP8>(c0, c1, dw0, dw1, dx, idesc, 1u, 3);
          umma_commit(&empty[st]);
          st = nst;
          ph = nph;
        }
        if (!ok) break;
        umma_commit(&tmem_full[s0]);
        slot_phase ^= 1u << s0;
        if (big) {
          umma_commit(&tmem_full[1]);
          slot_phase ^= 2u;
        } else {
          slot ^= 1;
        }
      }
      if (!ok) {
        abort_flag = 1;
        raise_error(kErrTimeout);
      }
      umma_commit(&drain_bar);
      mbar_wait(&drain_bar, 0u);
    }
  } else if (warp >= 2 && warp <= 5) {
    // ------------------------------------------------------------ epilogue (warps 2..5)
    const int quarter = warp & 3;
    __nv_bfloat16* xs = xs_all + quarter * 32 * kFgXsStride;
    const uint32_t t_lane = tmem_base + ((uint32_t)(quarter * 32) << 16);
    int slot = 0;
    uint32_t slot_phase = 0;
    for (int t = blockIdx.x; t < total_tiles; t += gridDim.x) {
      const FgTile tl = fg_decode<BT>(t, mbp, p);
      const bool big = tl.n > 128;
      const int s0 = big ? 0 : slot;
      const uint32_t c0 = (uint32_t)(s0 * 256), c1 = big ? 256u : c0 + 128u;
      bool ok = mbar_wait(&tmem_full[s0], (slot_phase >> s0) & 1u, &abort_flag);
      if (ok && big) ok = mbar_wait(&tmem_full[1], (slot_phase >> 1) & 1u, &abort_flag);
      if (!ok) {
        abort_flag = 1;
        raise_error(kErrTimeout);
        break;
      }
      tc_fence_after();
      const int64_t wrow = FP8 ? (int64_t)(p.w_map != nullptr ? p.w_map[tl.e] : tl.e) * p.a_rows : 0;
      if (EPI == kTcSwiglu) {
        const int f0 = 128 * tl.ft + 32 * quarter;
        float wsg = 1.0f, wsu = 1.0f;
        if (FP8 && f0 + 32 <= p.n_valid) {
          wsg = p.w_scale[wrow + f0 + lane];
          wsu = p.w_scale[wrow + p.up_rows + f0 + lane];
        }
        fg_drain<kTcSwiglu, FP8>(t_lane, c0, c1, tl.n, tl.r0, f0, f0 + 32 <= p.n_valid, p, xs, wsg, wsu);
      } else {
        const int f0 = 256 * tl.ft + 32 * quarter;
        const float ws0 = (FP8 && f0 + 32 <= p.n_valid) ? p.w_scale[wrow + f0 + lane] : 1.0f;
        const float ws1 = (FP8 && f0 + 160 <= p.n_valid) ? p.w_scale[wrow + f0 + 128 + lane] : 1.0f;
        fg_drain<kTcStore, FP8, COMBINE>(t_lane, c0, 0, tl.n, tl.r0, f0, f0 + 32 <= p.n_valid, p, xs, ws0);
        if (big) {  // D0 alone fills slot 0: hand it back before draining D1
          tc_fence_before();
          mbar_arrive(&tmem_empty[0]);
        }
        fg_drain<kTcStore, FP8, COMBINE>(t_lane, c1, 0, tl.n, tl.r0, f0 + 128, f0 + 160 <= p.n_valid, p, xs, ws1);
      }
      tc_fence_before();
      if (big) {
        if (EPI == kTcSwiglu) mbar_arrive(&tmem_empty[0]);
        mbar_arrive(&tmem_empty[1]);
        slot_phase ^= 3u;
      } else {
        mbar_arrive(&tmem_empty[s0]);
        slot_phase ^= 1u << s0;
        slot ^= 1;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (abort_flag) {
    // every role has stopped: give each stage's last armed phase the arrival
    // of the side that did not arm it, then wait until its copies have landed
    if (tid == 0) {
      for (int s = 0; s < ST; ++s) {
        const uint32_t w = armed_w[s], x = armed_x[s];
        if (w > x) mbar_arrive_n(&full[s], kXArrivals);
        else if (x > w) mbar_arrive(&full[s]);
        const uint32_t n = w > x ? w : x;
        if (n > 0) mbar_wait(&full[s], (n - 1u) & 1u);
      }
    }
    __syncthreads();
  }
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(512) : "memory");
  }
}

}  // namespace moe
