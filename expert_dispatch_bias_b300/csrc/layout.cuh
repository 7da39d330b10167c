// Dispatch layout: stable per-expert rank in token order, capacity drop/pad,
// offsets, slots, row sources and the virtual-EP dispatch matrix n_ij.
//
// Pass 1 (layout_rank_kernel): the T*K assignments, in token order, are cut
// into tiles of kLayoutTile.  Each block takes the next tile id from a counter
// (so every tile it may wait for belongs to a block that is already running),
// ranks its assignments per expert with warp match/popc and per-warp counters,
// publishes its per-expert aggregate, and looks back over earlier tiles
// (decoupled look-back) for the per-expert exclusive prefix.  The last tile's
// inclusive prefix is the histogram.  The look-back spin is bounded.
//
// Pass 2 (layout_finalize_kernel): every block scans kept[] into offsets,
// turns ranks into slots (or -1 when over capacity), fills row_src and counts
// its n_ij entries in shared memory (its tokens fall in a few source chips),
// then adds them to n_ij and to the per-chip sent / received row counts; the
// last block to finish turns those counts into bytes, derives the scalar
// statistics and resets the look-back state for the next call.
#pragma once

#include "common.cuh"
#include "moe.h"

namespace moe {

constexpr int kLayoutThreads = 512;
constexpr int kLayoutWarps = kLayoutThreads / 32;
constexpr int kLayoutItems = 4;                       // per thread
constexpr int kLayoutTile = kLayoutThreads * kLayoutItems;
constexpr int kFinalizeThreads = 256;
constexpr int kFinalizeItems = 4;
constexpr int kFinalizeBins = 4096;  // shared n_ij entries of one block

enum : uint32_t { kTileEmpty = 0u, kTileAggregate = 1u, kTileInclusive = 2u };

// Look-back state kept in the caller's workspace.
struct LayoutScratch {
  uint32_t* header;   // [64]: [0] tile counter, [1] finished-block counter
  uint32_t* flags;    // [num_tiles]
  int32_t* agg;       // [num_tiles][E]
  int32_t* incl;      // [num_tiles][E]
};

__host__ __device__ inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

__host__ __device__ inline int layout_num_tiles(int64_t A) {
  const int64_t n = (A + kLayoutTile - 1) / kLayoutTile;
  return (int)(n < 1 ? 1 : n);
}

inline size_t layout_scratch_bytes(int64_t A, int E) {
  const size_t nt = (size_t)layout_num_tiles(A);
  return 256 + align_up(nt * 4, 256) + 2 * align_up(nt * (size_t)E * 4, 256);
}

inline LayoutScratch layout_scratch_at(void* base, int64_t A, int E) {
  const size_t nt = (size_t)layout_num_tiles(A);
  char* p = static_cast<char*>(base);
  LayoutScratch s;
  s.header = reinterpret_cast<uint32_t*>(p);  // [0] tiles taken, [1] blocks done, [2..3] diagonal rows (u64)
  p += 256;
  s.flags = reinterpret_cast<uint32_t*>(p);
  p += align_up(nt * 4, 256);
  s.agg = reinterpret_cast<int32_t*>(p);
  p += align_up(nt * (size_t)E * 4, 256);
  s.incl = reinterpret_cast<int32_t*>(p);
  return s;
}

struct LayoutParams {
  const int32_t* ids;   // [A] = [T, K]
  int64_t A;
  int T, K, E, cap, pad, n_ep, ds, h, R;
  int num_tiles;
  int32_t* counts;
  int32_t* kept;
  int32_t* offsets;
  int32_t* slot;        // ranks after pass 1, slots after pass 2
  int32_t* row_src;
  int64_t* n_ij;
  int64_t* rank_bytes;
  moe_layout_stats* stats;
  LayoutScratch ws;
};

__global__ void __launch_bounds__(kLayoutThreads) layout_rank_kernel(LayoutParams p) {
  extern __shared__ int32_t sm[];
  int32_t* cnt = sm;                          // [kLayoutWarps][E] per-warp counts, then warp prefixes
  int32_t* tile_agg = sm + kLayoutWarps * p.E;  // [E]
  int32_t* excl = tile_agg + p.E;             // [E]
  __shared__ uint32_t s_tile;
  __shared__ int s_stop;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) s_tile = atomicAdd(&p.ws.header[0], 1u);
  for (int i = tid; i < kLayoutWarps * p.E; i += kLayoutThreads) cnt[i] = 0;

  // Clear what pass 2 accumulates into; fill row_src with -1 (pad/unused rows).
  {
    const int64_t gstride = (int64_t)gridDim.x * kLayoutThreads;
    const int64_t gtid = (int64_t)blockIdx.x * kLayoutThreads + tid;
    for (int64_t r = gtid; r < p.R; r += gstride) p.row_src[r] = -1;
    const int64_t nn = (int64_t)p.n_ep * p.n_ep;
    for (int64_t i = gtid; i < nn; i += gstride) p.n_ij[i] = 0;
    for (int64_t i = gtid; i < 2 * p.n_ep; i += gstride) p.rank_bytes[i] = 0;  // row counts until pass 2 ends
  }
  __syncthreads();
  const int tile = (int)s_tile;
  if (tile >= p.num_tiles) return;  // only when the counter was left dirty

  // ---- stable rank inside the tile: warp w owns a contiguous chunk, in order
  const int64_t base = (int64_t)tile * kLayoutTile + (int64_t)warp * (32 * kLayoutItems);
  int e_of[kLayoutItems];
  int32_t local[kLayoutItems];
#pragma unroll
  for (int r = 0; r < kLayoutItems; ++r) {
    const int64_t a = base + r * 32 + lane;
    int e = a < p.A ? p.ids[a] : -1;
    if (a < p.A && (e < 0 || e >= p.E)) {
      raise_error(kErrBadIndex);
      e = -1;
    }
    const unsigned grp = __match_any_sync(0xffffffffu, e);
    const unsigned lower = grp & ((1u << lane) - 1u);
    const int32_t before = e >= 0 ? cnt[warp * p.E + e] : 0;
    __syncwarp();
    if (e >= 0 && lower == 0) cnt[warp * p.E + e] = before + __popc(grp);
    __syncwarp();
    e_of[r] = e;
    local[r] = before + __popc(lower);
  }
  __syncthreads();
  for (int e = tid; e < p.E; e += kLayoutThreads) {  // exclusive scan over warps
    int32_t run = 0;
    for (int w = 0; w < kLayoutWarps; ++w) {
      const int32_t c = cnt[w * p.E + e];
      cnt[w * p.E + e] = run;
      run += c;
    }
    tile_agg[e] = run;
    if (tile == 0) {
      p.ws.incl[e] = run;
    } else {
      p.ws.agg[(size_t)tile * p.E + e] = run;
    }
  }
  __threadfence();
  __syncthreads();

  // ---- decoupled look-back over earlier tiles
  if (tid == 0) {
    int stop = -1;
    if (tile == 0) {
      st_release_u32(&p.ws.flags[0], kTileInclusive);
    } else {
      st_release_u32(&p.ws.flags[tile], kTileAggregate);
      for (int t = tile - 1; t >= 0; --t) {
        uint32_t f = ld_acquire_u32(&p.ws.flags[t]);
        if (f == kTileEmpty) {
          const uint64_t t0 = globaltimer_ns();
          while ((f = ld_acquire_u32(&p.ws.flags[t])) == kTileEmpty) {
            if (globaltimer_ns() - t0 > kWaitLimitNs) break;
            __nanosleep(64);
          }
        }
        if (f == kTileEmpty) {  // predecessor never published: give up, flag it
          raise_error(kErrTimeout);
          stop = -1;
          break;
        }
        if (f == kTileInclusive) {
          stop = t;
          break;
        }
      }
      // tiles in (stop, tile) contributed their aggregates
    }
    s_stop = stop;
  }
  __syncthreads();
  const int stop = s_stop;
  if (tile > 0) {
    for (int e = tid; e < p.E; e += kLayoutThreads) {
      int32_t v = stop >= 0 ? __ldcg(&p.ws.incl[(size_t)stop * p.E + e]) : 0;
      for (int t = (stop >= 0 ? stop + 1 : 0); t < tile; ++t) v += __ldcg(&p.ws.agg[(size_t)t * p.E + e]);
      excl[e] = v;
      p.ws.incl[(size_t)tile * p.E + e] = v + tile_agg[e];
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) st_release_u32(&p.ws.flags[tile], kTileInclusive);
  } else {
    for (int e = tid; e < p.E; e += kLayoutThreads) excl[e] = 0;
    __syncthreads();
  }

  // ---- ranks, and the histogram from the last tile
#pragma unroll
  for (int r = 0; r < kLayoutItems; ++r) {
    const int64_t a = base + r * 32 + lane;
    const int e = e_of[r];
    if (e >= 0) p.slot[a] = excl[e] + cnt[warp * p.E + e] + local[r];
  }
  if (tile == p.num_tiles - 1) {
    for (int e = tid; e < p.E; e += kLayoutThreads) {
      const int32_t c = excl[e] + tile_agg[e];
      p.counts[e] = c;
      p.kept[e] = p.cap > 0 ? min(c, p.cap) : c;
    }
  }
}

__global__ void __launch_bounds__(kFinalizeThreads) layout_finalize_kernel(LayoutParams p) {
  extern __shared__ int32_t off[];  // [E + 1]
  __shared__ int32_t scratch[33];
  __shared__ bool s_last;
  const int tid = threadIdx.x;
  const bool pad = p.pad && p.cap > 0;
  for (int e = tid; e < p.E; e += kFinalizeThreads) off[e] = pad ? p.cap : p.kept[e];
  __syncthreads();
  const int32_t total = block_exclusive_scan(off, p.E, scratch);
  if (tid == 0) off[p.E] = total;
  __syncthreads();
  if (blockIdx.x == 0)
    for (int e = tid; e <= p.E; e += kFinalizeThreads) p.offsets[e] = off[e];

  const int epr = p.E / p.n_ep;
  const int N = p.n_ep;
  const int64_t a0 = (int64_t)blockIdx.x * (kFinalizeThreads * kFinalizeItems);
  const int64_t a_end = min(p.A, a0 + kFinalizeThreads * kFinalizeItems);
  // Source chips of this block's tokens: [i_lo, i_lo + span).
  const int i_lo = a0 < a_end ? (int)((a0 / p.K) * N / p.T) : 0;
  const int span = a0 < a_end ? (int)(((a_end - 1) / p.K) * N / p.T) - i_lo + 1 : 0;
  const bool local = (int64_t)span * N <= kFinalizeBins;
  __shared__ int32_t bins[kFinalizeBins];
  if (local)
    for (int b = tid; b < span * N; b += kFinalizeThreads) bins[b] = 0;
  __syncthreads();
#pragma unroll
  for (int r = 0; r < kFinalizeItems; ++r) {
    const int64_t a = a0 + r * kFinalizeThreads + tid;
    if (a >= p.A) break;
    const int e = p.ids[a];
    if (e < 0 || e >= p.E) continue;  // already reported by pass 1
    const int32_t rank = p.slot[a];
    // Ranks come from pass 1; if a look-back gave up they may be garbage, so
    // every derived index is bounds-checked before it is used as an address.
    bool keep = p.cap <= 0 || rank < p.cap;
    int32_t s = keep ? off[e] + rank : -1;
    if (rank < 0 || rank >= p.counts[e] || s >= p.R) {
      raise_error(kErrBadIndex);
      keep = false;
      s = -1;
    }
    p.slot[a] = s;
    if (keep) {
      const int64_t t = a / p.K;
      p.row_src[s] = (int32_t)t;
      const int i = (int)((t * N) / p.T), j = e / epr;
      if (local) {
        atomicAdd(&bins[(i - i_lo) * N + j], 1);
      } else {
        atomicAdd(reinterpret_cast<unsigned long long*>(&p.n_ij[(int64_t)i * N + j]), 1ull);
        atomicAdd(reinterpret_cast<unsigned long long*>(&p.rank_bytes[i]), 1ull);
        atomicAdd(reinterpret_cast<unsigned long long*>(&p.rank_bytes[N + j]), 1ull);
        if (i == j) atomicAdd(reinterpret_cast<unsigned long long*>(p.ws.header + 2), 1ull);
      }
    }
  }
  __syncthreads();
  if (local) {
    for (int b = tid; b < span * N; b += kFinalizeThreads) {
      const unsigned long long c = (unsigned long long)bins[b];
      if (c == 0) continue;
      const int i = i_lo + b / N, j = b % N;
      atomicAdd(reinterpret_cast<unsigned long long*>(&p.n_ij[(int64_t)i * N + j]), c);
      atomicAdd(reinterpret_cast<unsigned long long*>(&p.rank_bytes[i]), c);
      atomicAdd(reinterpret_cast<unsigned long long*>(&p.rank_bytes[N + j]), c);
      if (i == j) atomicAdd(reinterpret_cast<unsigned long long*>(p.ws.header + 2), c);
    }
  }

  // ---- the last block derives the per-chip bytes and scalar statistics
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = atomicAdd(&p.ws.header[1], 1u) == gridDim.x - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  __shared__ unsigned long long s_max, s_sum, s_off;
  __shared__ int s_touched;
  __shared__ long long s_kept;
  if (tid == 0) {
    s_max = 0;
    s_sum = 0;
    s_off = 0;
    s_touched = 0;
    s_kept = 0;
  }
  __syncthreads();
  const long long rowbytes = (long long)p.h * p.ds;
  for (int i = tid; i < N; i += kFinalizeThreads) {  // row and column sums of n_ij
    const long long sent = __ldcg(&p.rank_bytes[i]), recv = __ldcg(&p.rank_bytes[N + i]);
    p.rank_bytes[i] = sent * rowbytes;
    p.rank_bytes[N + i] = recv * rowbytes;
    atomicMax(&s_max, (unsigned long long)recv);
    atomicAdd(&s_sum, (unsigned long long)recv);
    atomicAdd(&s_off, (unsigned long long)sent);
  }
  for (int e = tid; e < p.E; e += kFinalizeThreads) {
    const int32_t k = __ldcg(&p.kept[e]);
    if (k > 0) atomicAdd(&s_touched, 1);
    atomicAdd(reinterpret_cast<unsigned long long*>(&s_kept), (unsigned long long)k);
  }
  __syncthreads();
  if (tid == 0) {
    moe_layout_stats st;
    st.kept_total = s_kept;
    st.dropped = p.A - s_kept;
    unsigned long long* diag = reinterpret_cast<unsigned long long*>(p.ws.header + 2);
    st.offdiag_rows = (long long)(s_off - __ldcg(diag));  // all kept rows minus the diagonal
    st.experts_touched = s_touched;
    st.balancedness = s_max == 0 ? 1.0f : (float)((double)s_sum / ((double)N * (double)s_max));
    *p.stats = st;
    // reset the look-back state for the next call on this workspace
    p.ws.header[0] = 0;
    p.ws.header[1] = 0;
    *diag = 0;
  }
  for (int t = tid; t < p.num_tiles; t += kFinalizeThreads) p.ws.flags[t] = kTileEmpty;
}

// Replica map of expert-parallel load balancing: the physical expert of every
// routed (t, k) is replica t mod n_rep(e) of its logical expert e, where the
// replicas of e are rep_phys[rep_offsets[e] .. rep_offsets[e+1]).  An id outside
// [0, E) or a plan entry outside [0, P) raises the bad-index error and writes -1.
__global__ void eplb_map_kernel(const int32_t* ids, int64_t A, int K, int E, int P, const int32_t* rep_offsets,
                                const int32_t* rep_phys, int32_t* out) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < A; i += (int64_t)gridDim.x * blockDim.x) {
    const int e = ids[i];
    int32_t v = -1;
    if (e >= 0 && e < E) {
      const int32_t r0 = rep_offsets[e], n = rep_offsets[e + 1] - r0;
      const int64_t j = n > 0 ? r0 + (i / K) % n : -1;
      if (n > 0 && r0 >= 0 && j < P) v = rep_phys[j];
    }
    if (v < 0 || v >= P) {
      raise_error(kErrBadIndex);
      v = -1;
    }
    out[i] = v;
  }
}

}  // namespace moe
