// Grouped GEMM with token rows as M on a PAIR of SMs (tcgen05.mma.cta_group::2):
// the tensor-bound form of the grouped FFN (Mixtral: ~1024 rows per expert)
// and of the shared expert.
//
// C[m, n] = sum_k A[m, k] * B[n, k] over row segments as in tc_gemm.cuh, with
// tiles of 256 token rows x 256 weight rows.  The two CTAs of a cluster share
// one MMA of M = 256, N = 256: CTA r holds the tile's token rows 128 r..
// (its half of A, 16 KB per k-block) and weight rows 128 r.. (its half of B,
// 16 KB), and each CTA's TMEM receives its own 128 token rows x all 256
// columns.  Per k-block a CTA thus loads 32 KB for 128 x 256 x 64 multiply-adds,
// where the one-SM form (tc_gemm.cuh, 128-row tiles) loads 48 KB (16 KB of
// tokens + 32 KB of weights): a third less data into each SM for the same
// tensor work, and stages small enough for a 6-deep ring.
//
// B halves: gate/up (SwiGLU epilogue): CTA 0 the gate rows n0.., CTA 1 the
// matching up rows I + n0.., so columns 0..127 of the accumulator are gate
// units and 128..255 the matching up units, as in tc_gemm.cuh; down (store
// epilogue): rows 256 nt.. and 256 nt + 128.. .  A segment with an odd number
// of 128-row blocks gives its last pair's CTA 1 rows past the segment: they
// are computed and masked on store.
//
// Roles (192 threads per CTA, one CTA per SM, clusters of 2):
//   warp 0      one thread loads the CTA's two boxes of every k-block into a
//               S-deep ring, the copies completing on the LEADER's barrier
//               (the 2-SM form of the bulk tensor copy), which the leader arms
//               with both CTAs' bytes;
//   warp 1      allocates TMEM (both CTAs, collectively); in the leader one
//               thread issues the MMAs (M = 256, N = 256, K = 16) and frees
//               each stage in both CTAs with one multicast commit;
//   warps 2..5  drain the CTA's own accumulator (double-buffered, 2 x 256
//               columns) and report it drained on the leader's barrier.
// Every wait is bounded; a CTA whose wait runs out raises the sticky error and
// winds down (the leader waits, bounded, for the stages it armed), and the pair
// meets at a cluster barrier before TMEM is freed and the CTAs exit.
#pragma once

#include "tc_gemm.cuh"

namespace moe {

constexpr int kTpThreads = 192;

template <int S>
struct TpShape {
  static constexpr uint32_t kABytes = 128 * kTcBK * 2;   // this CTA's 128 token rows
  static constexpr uint32_t kBBytes = 128 * kTcBK * 2;   // this CTA's 128 weight rows
  static constexpr uint32_t kStage = kABytes + kBBytes;
  static constexpr size_t kDynSmem = (size_t)S * kStage + 1024;
};

// ------------------------------------------------------------------ cluster helpers
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
// on the mbarrier at `bar_cluster` (a shared::cluster address, here the
// leader's barrier): the 2-SM form of tma_load_2d.
__device__ __forceinline__ void tma_load_2d_pair(void* smem_dst, const CUtensorMap* map, int x, int y,
                                                 uint32_t bar_cluster) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2 [%0], [%1, "
      "{%2, %3}], [%4];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar_cluster)
      : "memory");
}

// ------------------------------------------------------------------ tile schedule
// mbp[e] = 256-row tiles (pairs of 128-row blocks) of segments < e, mbp[E] =
// total; tiles ordered (segment, column tile, row pair) so that the row pairs
// sharing a weight panel run on neighbouring clusters.  m0 is this CTA's first
// row.
__device__ __forceinline__ TcTile tp_decode(int t, const int32_t* mbp, const TcParams& p, uint32_t rank) {
  int lo = 0, hi = p.E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (mbp[mid] * p.n_tiles <= t) lo = mid; else hi = mid - 1;
  }
  const int e = lo;
  const int local = t - mbp[e] * p.n_tiles;
  const int cnt = mbp[e + 1] - mbp[e];
  TcTile r;
  r.e = e;
  r.nt = local / cnt;
  const int mp = local - r.nt * cnt;
  const int seg0 = p.offsets ? p.offsets[e] : 0;
  r.m0 = seg0 + (2 * mp + (int)rank) * kTcBM;
  r.m_end = seg0 + (p.offsets ? p.kept[e] : p.dense_rows);
  return r;
}

template <int EPI, int S>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kTpThreads, 1)
    tc_pair_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b, TcParams p) {
  static_assert(EPI == kTcSwiglu || EPI == kTcStore, "the pair form serves the FFN GEMMs");
  using SH = TpShape<S>;
  constexpr int BN = 256, CH = 32;
  extern __shared__ uint8_t dyn_smem[];
  __shared__ __align__(8) uint64_t full_bar[S], empty_bar[S];   // full: used in the leader only
  __shared__ __align__(8) uint64_t tmem_full[2], tmem_empty[2], drain_bar;
  __shared__ uint32_t tmem_holder;
  __shared__ volatile uint32_t abort_flag;
  __shared__ int32_t mbp[1025];
  __shared__ int32_t scan_scratch[33];

  uint8_t* tiles = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dyn_smem) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_rank();
  const bool leader = rank == 0;
  const int pair = (int)cluster_id_x(), n_pairs = (int)n_clusters_x();

  // ---- per-segment tile prefix: pairs of 128-row blocks
  for (int e = tid; e < p.E; e += kTpThreads) {
    const int rows = p.offsets ? p.kept[e] : p.dense_rows;
    const int mb = (rows + kTcBM - 1) / kTcBM;
    mbp[e] = (mb + 1) >> 1;
  }
  __syncthreads();
  const int32_t total_mp = block_exclusive_scan(mbp, p.E, scan_scratch);
  if (tid == 0) mbp[p.E] = total_mp;
  const int total_tiles = total_mp * p.n_tiles;

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
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
                 "r"(2 * BN)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  cluster_sync();   // barriers initialised and TMEM allocated in both CTAs before any remote access
  tc_fence_after();
  const uint32_t tmem_base = tmem_holder;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint32_t full_l = peer_smem(&full_bar[0], 0);   // the leader's barriers
      int stage = 0;
      uint32_t phase = 0, armed = 0, armed_parity = 0;
      for (int t = pair; t < total_tiles && !abort_flag; t += n_pairs) {
        const TcTile tl = tp_decode(t, mbp, p, rank);
        const int64_t brow = (int64_t)(p.w_map != nullptr ? p.w_map[tl.e] : tl.e) * p.b_rows;
        const int64_t b0 = EPI == kTcSwiglu ? brow + (rank == 0 ? 0 : p.up_rows) + (int64_t)tl.nt * (BN / 2)
                                            : brow + (int64_t)tl.nt * BN + 128 * (int64_t)rank;
        for (int kb = 0; kb < p.k_blocks; ++kb) {
          if (!mbar_wait(&empty_bar[stage], phase ^ 1u, &abort_flag)) {
            abort_flag = 1;
            raise_error(kErrTimeout);
            break;
          }
          uint8_t* sa = tiles + (size_t)stage * SH::kStage;
          const uint32_t bar = full_l + (uint32_t)(stage * sizeof(uint64_t));
          const int kx = kb * kTcBK;
          if (leader) mbar_expect_tx(&full_bar[stage], 2 * SH::kStage);   // both CTAs' boxes
          tma_load_2d_pair(sa, &map_a, kx, tl.m0, bar);
          tma_load_2d_pair(sa + SH::kABytes, &map_b, kx, (int)b0, bar);
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
          if ((armed >> s) & 1u) mbar_wait(&full_bar[s], (armed_parity >> s) & 1u);
      }
    }
  } else if (warp == 1) {
    if (leader && lane == 0) {
      // ---------------------------------------------------------- MMA issuer (leader)
      constexpr uint32_t idesc = umma_idesc_bf16(256, BN);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      for (int t = pair; t < total_tiles && !abort_flag; t += n_pairs) {
        if (!mbar_wait(&tmem_empty[acc], acc_phase ^ 1u, &abort_flag)) {
          abort_flag = 1;
          raise_error(kErrTimeout);
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
        bool ok = true;
        for (int kb = 0; kb < p.k_blocks; ++kb) {
          if (!mbar_wait(&full_bar[stage], phase, &abort_flag)) {
            abort_flag = 1;
            raise_error(kErrTimeout);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(tiles + (size_t)stage * SH::kStage);
          const uint32_t sb = sa + SH::kABytes;
#pragma unroll
          for (int k = 0; k < kTcBK / 16; ++k)
            umma2_bf16(d_tmem, umma_desc_sw128(sa + k * 32), umma_desc_sw128(sb + k * 32), idesc,
                       (kb != 0 || k != 0) ? 1u : 0u);
          umma2_commit(&empty_bar[stage], 3);   // the stage is free again in both CTAs
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma2_commit(&tmem_full[acc], 3);
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      umma2_commit(&drain_bar, 1);   // every MMA this thread issued has completed once it fires
      mbar_wait(&drain_bar, 0u);
    }
  } else {
    // ------------------------------------------------------------ epilogue (warps 2..5)
    const int quarter = warp & 3;
    const uint32_t remote_empty = peer_smem(&tmem_empty[0], 0);
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int t = pair; t < total_tiles; t += n_pairs) {
      if (!mbar_wait(&tmem_full[acc], acc_phase, &abort_flag)) {
        abort_flag = 1;
        raise_error(kErrTimeout);
        break;
      }
      tc_fence_after();
      const TcTile tl = tp_decode(t, mbp, p, rank);
      const int row = tl.m0 + quarter * 32 + lane;
      const bool valid = row < tl.m_end;
      const uint32_t taddr = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * BN);
      __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(p.out) + (int64_t)row * p.ldo;
      if (EPI == kTcSwiglu) {
        const int n0 = tl.nt * (BN / 2);
#pragma unroll 1
        for (int c = 0; c < BN / 2; c += CH) {
          uint32_t g[CH], u[CH];
          tmem_ld<CH>(taddr + c, g);
          tmem_ld<CH>(taddr + BN / 2 + c, u);
          tmem_ld_wait();
          if (valid && n0 + c + CH <= p.n_valid) {
            float a[CH];
#pragma unroll
            for (int i = 0; i < CH; ++i) {
              const float gi = __uint_as_float(g[i]);
              a[i] = __fdividef(gi, 1.0f + __expf(-gi)) * __uint_as_float(u[i]);  // fast forms, as in tc_gemm.cuh
            }
            store_bf16_row<CH>(orow + n0 + c, a);
          }
        }
      } else {
        const int n0 = tl.nt * BN;
#pragma unroll 1
        for (int c = 0; c < BN; c += CH) {
          uint32_t v[CH];
          tmem_ld<CH>(taddr + c, v);
          tmem_ld_wait();
          if (valid && n0 + c + CH <= p.n_valid) {
            float a[CH];
#pragma unroll
            for (int i = 0; i < CH; ++i) a[i] = __uint_as_float(v[i]);
            store_bf16_row<CH>(orow + n0 + c, a);
          }
        }
      }
      tc_fence_before();
      mbar_arrive_remote(remote_empty + (uint32_t)(acc * sizeof(uint64_t)));
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
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
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(2 * BN) : "memory");
  }
}

}  // namespace moe
