// Grouped SwiGLU FFN over ragged expert segments on a PAIR of SMs: the
// weights-as-M kernel of ffn_grouped.cuh with the 2-SM form of the tensor-core
// instruction (tcgen05.mma.cta_group::2).
//
// Why a pair.  With weights as the MMA's M operand every k-block a CTA streams
// its two 128-row weight boxes (32 KB) plus the token rows of its tile.  The
// token rows are L2 hits, but they pass through the same TMA ring and the same
// SM ingest as the weights, and an expert with more rows than one token tile
// streams its weights once per tile.  In the 2-SM instruction the two CTAs of
// a cluster share the B operand: each holds HALF of the tile's token rows, and
// one MMA of M = 256 multiplies both CTAs' A rows by all N token rows.  So per
// k-block a CTA loads 32 KB of weights and only N/2 token rows, and a tile can
// hold up to 256 token rows (N = 256), so fewer experts are split into several
// token tiles that each stream the weights again.
//
// A pair tile is (expert e, feature pair fp, token tile tt).  CTA r of the pair
// computes feature tile ft = 2 fp + r exactly as one CTA of ffn_grouped.cuh
// does:
//   gate/up: A0 = gate rows 128 ft.., A1 = up rows I + 128 ft..; SwiGLU epilogue;
//   down:    A0 = rows 256 ft.., A1 = rows 256 ft + 128..; store epilogue.
// Per K=16 step the leader CTA issues two MMAs (M = 256, N = the tile's rows
// rounded up to 32): D0 = [A0 of CTA 0; A0 of CTA 1] x X^T and D1 likewise.
// Each CTA's TMEM receives its own 128 rows of D0 and D1 for all N token
// columns; columns 0..N/2-1 are the token rows CTA 0 loaded, N/2..N-1 those of
// CTA 1.  A feature tile past the end (odd tile counts) loads valid rows and
// masks its stores.
//
// Roles (224 threads per CTA, one CTA per SM, clusters of 2):
//   warp 0      weight producer: the CTA's two 128x64 weight boxes per k-block;
//   warp 6      token producer: the CTA's N/2 token rows per k-block;
//   warp 1      allocates TMEM (both CTAs, collectively); in the leader one
//               thread issues the MMAs once the stage is full in both CTAs and
//               releases it in both with one multicast commit;
//   warps 2..5  epilogue of the CTA's own accumulators (as ffn_grouped.cuh);
//               every epilogue thread of both CTAs reports a drained
//               accumulator on the leader's barrier (mapa address).
// Both CTAs' copies of a stage complete on the LEADER's full barriers (the
// 2-SM form of the bulk tensor copy may signal a barrier of either CTA of the
// pair); the leader arms them with the bytes of both.  So one wait tells the
// MMA issuer that both halves of the operands have landed.  Every wait is
// bounded; a CTA whose wait runs out raises the sticky error and winds down:
// the leader waits (bounded) on its full barriers for the stages it armed,
// which also covers the peer's copies into them, and the pair meets at a
// cluster barrier before TMEM is freed and the CTAs exit.
#pragma once

#include "ffn_grouped.cuh"

namespace moe {

constexpr int kFpThreads = 224;

template <int BT, int S>
struct FpShape {
  static_assert(BT % 32 == 0 && BT >= 64 && BT <= 256, "token tiles of 64..256 rows, N a multiple of 32");
  static constexpr uint32_t kWBytes = 128 * kTcBK * 2;            // one 128-row weight box: 16 KB
  static constexpr uint32_t kWStage = 2 * kWBytes;                // both boxes of a k-block
  static constexpr uint32_t kXStage = (BT / 2) * kTcBK * 2;       // this CTA's half of the token rows
  static_assert(kXStage % 1024 == 0, "token stages start on 1024-byte swizzle atoms");
  static constexpr size_t kXsBytes = 4 * 32 * kFgXsStride * 2;    // transpose buffers of the 4 epilogue warps
  static constexpr size_t kDynSmem = (size_t)S * (kWStage + kXStage) + kXsBytes + 1024;
};

__device__ __forceinline__ uint32_t round32(int n) { return (uint32_t)((n + 31) & ~31); }

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ uint32_t cluster_id_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}

__device__ __forceinline__ uint32_t n_clusters_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}

// Every thread of both CTAs; release/acquire at cluster scope.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Address of the same shared variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t peer_smem(const void* local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(local)), "r"(rank));
  return r;
}

__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

__device__ __forceinline__ void umma2_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                           uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive on the mbarrier at this shared offset in every CTA of `mask` once all
// MMAs this thread issued have completed.
__device__ __forceinline__ void umma2_commit(uint64_t* bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_u32(bar)),
      "h"(mask)
      : "memory");
}

// Bulk tensor copy into this CTA's shared memory whose completion is counted
// on the mbarrier at `bar_cluster` (a shared::cluster address that may name
// the peer CTA's barrier): the 2-SM form of tma_load_2d.
__device__ __forceinline__ void tma_load_2d_pair(void* smem_dst, const CUtensorMap* map, int x, int y,
                                                 uint32_t bar_cluster) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2 [%0], [%1, "
      "{%2, %3}], [%4];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar_cluster)
      : "memory");
}

// mbp[e] = token tiles of experts < e, mbp[E] = total; a pair tile covers
// f_pairs = ceil(f_tiles / 2) feature pairs.
template <int BT>
__device__ __forceinline__ FgTile fp_decode(int t, const int32_t* mbp, const FgParams& p, int f_pairs,
                                            uint32_t rank) {
  int lo = 0, hi = p.E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (mbp[mid] * f_pairs <= t) lo = mid; else hi = mid - 1;
  }
  const int e = lo;
  const int local = t - mbp[e] * f_pairs;
  const int cnt = mbp[e + 1] - mbp[e];
  const int tt = local % cnt;
  const int kept = p.kept[e];
  const int base = kept / cnt, rem = kept % cnt;   // equal split: rows differ by at most one
  FgTile r;
  r.e = e;
  r.ft = 2 * (local / cnt) + (int)rank;
  r.r0 = p.offsets[e] + tt * base + min(tt, rem);
  r.n = base + (tt < rem ? 1 : 0);
  return r;
}

template <int EPI, int BT, int S>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kFpThreads, 1)
    ffn_pair_kernel(const __grid_constant__ CUtensorMap map_w, const __grid_constant__ FgTokenMaps maps,
                    FgParams p) {
  const CUtensorMap* map_x = maps.m;
  using SH = FpShape<BT, S>;
  extern __shared__ uint8_t dyn_smem[];
  __shared__ __align__(8) uint64_t wfull[S], xfull[S], empty[S];   // full: used in the leader only
  __shared__ __align__(8) uint64_t tmem_full[2], tmem_empty[2], drain_bar;
  __shared__ uint32_t tmem_holder;
  __shared__ volatile uint32_t abort_flag;
  __shared__ int32_t mbp[1025];
  __shared__ int32_t scan_scratch[33];

  uint8_t* ring_w = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dyn_smem) + 1023) & ~uintptr_t(1023));
  uint8_t* ring_x = ring_w + (size_t)S * SH::kWStage;
  __nv_bfloat16* xs_all = reinterpret_cast<__nv_bfloat16*>(ring_x + (size_t)S * SH::kXStage);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_rank();
  const bool leader = rank == 0;
  const int pair = (int)cluster_id_x(), n_pairs = (int)n_clusters_x();
  const int f_pairs = (p.f_tiles + 1) >> 1;

  // ---- per-expert token-tile prefix (every CTA computes it from kept)
  for (int e = tid; e < p.E; e += kFpThreads) mbp[e] = (p.kept[e] + BT - 1) / BT;
  __syncthreads();
  const int32_t total_tt = block_exclusive_scan(mbp, p.E, scan_scratch);
  if (tid == 0) mbp[p.E] = total_tt;
  const int total_tiles = total_tt * f_pairs;

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&wfull[s], 1);
      mbar_init(&xfull[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tmem_full[a], 1);
      mbar_init(&tmem_empty[a], 256);   // the 128 epilogue threads of each CTA (the peer's arrive remotely)
    }
    mbar_init(&drain_bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {  // one warp in each CTA of the pair allocates, collectively
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_holder)),
                 "r"(512)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  cluster_sync();   // barriers initialised and TMEM allocated in both CTAs before any remote access
  tc_fence_after();
  const uint32_t tmem_base = tmem_holder;

  if (warp == 0) {
    // ------------------------------------------------------------ weight producer
    if (lane == 0) {
      const uint32_t wfull_l = peer_smem(&wfull[0], 0);   // the leader's barriers
      int stage = 0;
      uint32_t phase = 0, armed = 0, armed_parity = 0;
      for (int t = pair; t < total_tiles && !abort_flag; t += n_pairs) {
        const FgTile tl = fp_decode<BT>(t, mbp, p, f_pairs, rank);
        const int ft = tl.ft < p.f_tiles ? tl.ft : p.f_tiles - 1;   // past the end: valid rows, stores masked
        const int64_t we = p.w_map != nullptr ? p.w_map[tl.e] : tl.e;
        const int64_t a0 = we * p.a_rows + (EPI == kTcSwiglu ? 128 * ft : 256 * ft);
        const int64_t a1 = EPI == kTcSwiglu ? a0 + p.up_rows : a0 + 128;
        for (int kb = 0; kb < p.k_blocks; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, &abort_flag)) {
            abort_flag = 1;
            raise_error(kErrTimeout);
            break;
          }
          uint8_t* sw = ring_w + (size_t)stage * SH::kWStage;
          const int kx = kb * kTcBK;
          const uint32_t bar = wfull_l + (uint32_t)(stage * sizeof(uint64_t));
          if (leader) mbar_expect_tx(&wfull[stage], 2 * SH::kWStage);   // both CTAs' weight boxes
          tma_load_2d_pair(sw, &map_w, kx, (int)a0, bar);
          tma_load_2d_pair(sw + SH::kWBytes, &map_w, kx, (int)a1, bar);
          armed |= 1u << stage;
          armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (abort_flag && leader) {  // every armed stage (both CTAs' copies) lands before shared memory is released
        for (int s = 0; s < S; ++s)
          if ((armed >> s) & 1u) mbar_wait(&wfull[s], (armed_parity >> s) & 1u);
      }
    }
  } else if (warp == 6) {
    // ------------------------------------------------------------ token producer
    if (lane == 0) {
      const uint32_t xfull_l = peer_smem(&xfull[0], 0);   // the leader's barriers
      int stage = 0;
      uint32_t phase = 0, armed = 0, armed_parity = 0;
      for (int t = pair; t < total_tiles && !abort_flag; t += n_pairs) {
        const FgTile tl = fp_decode<BT>(t, mbp, p, f_pairs, rank);
        const int half = (int)round32(tl.n) >> 1;     // rows per CTA: a multiple of 16
        const int row0 = tl.r0 + (int)rank * half;
        const uint32_t x_bytes = 2u * (uint32_t)half * (uint32_t)(kTcBK * 2);   // both CTAs' halves
        for (int kb = 0; kb < p.k_blocks; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, &abort_flag)) {
            abort_flag = 1;
            raise_error(kErrTimeout);
            break;
          }
          uint8_t* sx = ring_x + (size_t)stage * SH::kXStage;
          const int kx = kb * kTcBK;
          const uint32_t bar = xfull_l + (uint32_t)(stage * sizeof(uint64_t));
          if (leader) mbar_expect_tx(&xfull[stage], x_bytes);
          // `half` rows as boxes of 128, then at most one each of 64, 32 and 16
          int b = 0;
          for (; b + 128 <= half; b += 128) tma_load_2d_pair(sx + b * (kTcBK * 2), &map_x[0], kx, row0 + b, bar);
          if ((half - b) & 64) { tma_load_2d_pair(sx + b * (kTcBK * 2), &map_x[1], kx, row0 + b, bar); b += 64; }
          if ((half - b) & 32) { tma_load_2d_pair(sx + b * (kTcBK * 2), &map_x[2], kx, row0 + b, bar); b += 32; }
          if ((half - b) & 16) tma_load_2d_pair(sx + b * (kTcBK * 2), &map_x[3], kx, row0 + b, bar);
          armed |= 1u << stage;
          armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (abort_flag && leader) {
        for (int s = 0; s < S; ++s)
          if ((armed >> s) & 1u) mbar_wait(&xfull[s], (armed_parity >> s) & 1u);
      }
    }
  } else if (warp == 1) {
    if (leader && lane == 0) {
      // ---------------------------------------------------------- MMA issuer (leader)
      int stage = 0;
      uint32_t phase = 0;
      int slot = 0;              // TMEM slot of the next tile of at most 128 token columns
      uint32_t slot_phase = 0;   // bit s: uses of slot s so far, mod 2
      for (int t = pair; t < total_tiles && !abort_flag; t += n_pairs) {
        const FgTile tl = fp_decode<BT>(t, mbp, p, f_pairs, rank);
        const int N = (int)round32(tl.n);
        const bool big = N > 128;
        const uint32_t idesc = umma_idesc_bf16(256, N);
        const int s0 = big ? 0 : slot;
        const uint32_t c0 = tmem_base + (uint32_t)(s0 * 256), c1 = big ? tmem_base + 256u : c0 + 128u;
        bool ok = mbar_wait(&tmem_empty[s0], ((slot_phase >> s0) & 1u) ^ 1u, &abort_flag);
        if (ok && big) ok = mbar_wait(&tmem_empty[1], ((slot_phase >> 1) & 1u) ^ 1u, &abort_flag);
        if (!ok) {
          abort_flag = 1;
          raise_error(kErrTimeout);
          break;
        }
        tc_fence_after();
        for (int kb = 0; kb < p.k_blocks; ++kb) {
          if (!mbar_wait(&wfull[stage], phase, &abort_flag) || !mbar_wait(&xfull[stage], phase, &abort_flag)) {
            abort_flag = 1;
            raise_error(kErrTimeout);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t dw0 = umma_desc_sw128(smem_u32(ring_w + (size_t)stage * SH::kWStage));
          const uint64_t dw1 = dw0 + (SH::kWBytes >> 4);
          const uint64_t dx = umma_desc_sw128(smem_u32(ring_x + (size_t)stage * SH::kXStage));
#pragma unroll
          for (int k = 0; k < kTcBK / 16; ++k) {
            const uint32_t acc = (kb | k) != 0 ? 1u : 0u;
            umma2_bf16(c0, dw0 + 2 * k, dx + 2 * k, idesc, acc);
            umma2_bf16(c1, dw1 + 2 * k, dx + 2 * k, idesc, acc);
          }
          umma2_commit(&empty[stage], 3);   // the stage is free again in both CTAs
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma2_commit(&tmem_full[s0], 3);
        slot_phase ^= 1u << s0;
        if (big) {
          umma2_commit(&tmem_full[1], 3);
          slot_phase ^= 2u;
        } else {
          slot ^= 1;
        }
      }
      umma2_commit(&drain_bar, 1);   // every MMA this thread issued has completed once it fires
      mbar_wait(&drain_bar, 0u);
    }
  } else if (warp >= 2 && warp <= 5) {
    // ------------------------------------------------------------ epilogue (warps 2..5)
    const int quarter = warp & 3;
    __nv_bfloat16* xs = xs_all + quarter * 32 * kFgXsStride;
    const uint32_t t_lane = tmem_base + ((uint32_t)(quarter * 32) << 16);
    // Every epilogue thread of both CTAs arrives on the LEADER's barrier (the
    // peer's remotely): no named barrier among the warps, so a warp that gives
    // up on a wait can never leave the others blocked.
    const uint32_t remote_empty = peer_smem(&tmem_empty[0], 0);
    auto release = [&](int s) {
      tc_fence_before();
      mbar_arrive_remote(remote_empty + (uint32_t)(s * sizeof(uint64_t)));
    };
    int slot = 0;
    uint32_t slot_phase = 0;
    for (int t = pair; t < total_tiles; t += n_pairs) {
      const FgTile tl = fp_decode<BT>(t, mbp, p, f_pairs, rank);
      const int N = (int)round32(tl.n);
      const bool big = N > 128;
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
      const bool tile_ok = tl.ft < p.f_tiles;
      if (EPI == kTcSwiglu) {
        const int f0 = 128 * tl.ft + 32 * quarter;
        fg_drain<kTcSwiglu, false>(t_lane, c0, c1, tl.n, tl.r0, f0, tile_ok && f0 + 32 <= p.n_valid, p, xs);
      } else {
        const int f0 = 256 * tl.ft + 32 * quarter;
        fg_drain<kTcStore, false>(t_lane, c0, 0, tl.n, tl.r0, f0, tile_ok && f0 + 32 <= p.n_valid, p, xs);
        if (big) release(0);   // D0 alone fills slot 0: hand it back before draining D1
        fg_drain<kTcStore, false>(t_lane, c1, 0, tl.n, tl.r0, f0 + 128, tile_ok && f0 + 160 <= p.n_valid, p, xs);
      }
      if (big) {
        if (EPI == kTcSwiglu) release(0);
        release(1);
        slot_phase ^= 3u;
      } else {
        release(s0);
        slot_phase ^= 1u << s0;
        slot ^= 1;
      }
    }
  }

  // both CTAs: every role done, every MMA complete (the leader drained them)
  // and every remote arrive delivered before TMEM is freed and the CTAs exit
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(512) : "memory");
  }
}

}  // namespace moe
