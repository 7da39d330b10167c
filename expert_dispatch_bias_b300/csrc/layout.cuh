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
//
// Up to kLayoutSmallMax assignments (decode batches) one block does all of it
// in one launch (layout_small_kernel), without the look-back.
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

// Bytes at the start of the scratch that must be zero before a layout call: the
// header (counters) and the tile flags, which layout_scratch_at places first.
// The per-tile sums after them are written before they are read.
inline size_t layout_scratch_zero_bytes(int64_t A) {
  return 256 + align_up((size_t)layout_num_tiles(A) * 4, 256);
}

// Block-wide sum (or max) of one int64 per thread; every thread gets the
// result.  Shuffles within warps, then one warp over the warp results:
// no contended atomics.  All threads of the block must call it.
template <bool MAX>
__device__ __forceinline__ long long block_reduce_ll(long long v, long long* scratch /* >= 33 */) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const long long u = __shfl_xor_sync(0xffffffffu, v, o);
    v = MAX ? (u > v ? u : v) : v + u;
  }
  __syncthreads();  // scratch may still be read by a previous call
  if (lane == 0) scratch[warp] = v;
  __syncthreads();
  if (warp == 0) {
    long long w = lane < nw ? scratch[lane] : 0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const long long u = __shfl_xor_sync(0xffffffffu, w, o);
      w = MAX ? (u > w ? u : w) : w + u;
    }
    if (lane == 0) scratch[32] = w;
  }
  __syncthreads();
  return scratch[32];
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
  pdl_wait();
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
  pdl_wait();
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
  __shared__ long long red[33];
  const long long rowbytes = (long long)p.h * p.ds;
  long long rmax = 0, rsum = 0, ssum = 0, kept_sum = 0, touched = 0;
  for (int i = tid; i < N; i += kFinalizeThreads) {  // row and column sums of n_ij
    const long long sent = __ldcg(&p.rank_bytes[i]), recv = __ldcg(&p.rank_bytes[N + i]);
    p.rank_bytes[i] = sent * rowbytes;
    p.rank_bytes[N + i] = recv * rowbytes;
    rmax = recv > rmax ? recv : rmax;
    rsum += recv;
    ssum += sent;
  }
  for (int e = tid; e < p.E; e += kFinalizeThreads) {
    const int32_t k = __ldcg(&p.kept[e]);
    touched += k > 0;
    kept_sum += k;
  }
  rmax = block_reduce_ll<true>(rmax, red);
  rsum = block_reduce_ll<false>(rsum, red);
  ssum = block_reduce_ll<false>(ssum, red);
  kept_sum = block_reduce_ll<false>(kept_sum, red);
  touched = block_reduce_ll<false>(touched, red);
  if (tid == 0) {
    moe_layout_stats st;
    st.kept_total = kept_sum;
    st.dropped = p.A - kept_sum;
    unsigned long long* diag = reinterpret_cast<unsigned long long*>(p.ws.header + 2);
    st.offdiag_rows = ssum - (long long)__ldcg(diag);  // all kept rows minus the diagonal
    st.experts_touched = (int32_t)touched;
    st.balancedness = rmax == 0 ? 1.0f : (float)((double)rsum / ((double)N * (double)rmax));
    *p.stats = st;
    // reset the look-back state for the next call on this workspace
    p.ws.header[0] = 0;
    p.ws.header[1] = 0;
    *diag = 0;
  }
  for (int t = tid; t < p.num_tiles; t += kFinalizeThreads) p.ws.flags[t] = kTileEmpty;
}

// Small layouts (T*K <= kLayoutSmallMax) in one block of 1024 threads and one
// launch: the same stable per-expert ranks (warp w owns assignments
// [w*256, w*256 + 256) in token order, 8 rounds of 32), the prefix over warps,
// the offsets, slots, row_src, n_ij (in shared memory when N_EP^2 <=
// kFinalizeBins, else global atomics), the per-chip bytes and the statistics;
// no look-back and no cross-block hand-off, so a decode-sized batch costs a few
// global round trips.  The look-back state in the workspace is not touched.
constexpr int kLayoutSmallThreads = 1024;
constexpr int kLayoutSmallItems = 8;
constexpr int kLayoutSmallMax = kLayoutSmallThreads * kLayoutSmallItems;

__host__ __device__ inline size_t layout_small_smem(int E, int n_ep) {
  const size_t bins = (size_t)n_ep * n_ep <= (size_t)kFinalizeBins ? (size_t)n_ep * n_ep : 0;
  return (32 * (size_t)E + (size_t)E + 1 + bins) * sizeof(int32_t);
}

__global__ void __launch_bounds__(kLayoutSmallThreads) layout_small_kernel(LayoutParams p) {
  pdl_wait();
  extern __shared__ int32_t sm[];
  const int E = p.E, N = p.n_ep;
  int32_t* cnt = sm;                 // [32][E]: per-warp counts, then prefixes over warps
  int32_t* off = cnt + 32 * E;       // [E + 1]
  int32_t* bins = off + E + 1;       // [N][N] when local
  const bool local = (int64_t)N * N <= kFinalizeBins;
  __shared__ int32_t scratch[33];
  __shared__ long long red[33];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  for (int i = tid; i < 32 * E; i += kLayoutSmallThreads) cnt[i] = 0;
  if (local)
    for (int i = tid; i < N * N; i += kLayoutSmallThreads) bins[i] = 0;
  for (int64_t r = tid; r < p.R; r += kLayoutSmallThreads) p.row_src[r] = -1;
  if (!local) {
    for (int64_t i = tid; i < (int64_t)N * N; i += kLayoutSmallThreads) p.n_ij[i] = 0;
    for (int i = tid; i < 2 * N; i += kLayoutSmallThreads) p.rank_bytes[i] = 0;
  }
  __syncthreads();

  // ---- stable rank of every assignment among its expert's, per warp
  const int64_t base = (int64_t)warp * (32 * kLayoutSmallItems);
  int e_of[kLayoutSmallItems];
  int32_t local_rank[kLayoutSmallItems];
#pragma unroll
  for (int r = 0; r < kLayoutSmallItems; ++r) {
    const int64_t a = base + r * 32 + lane;
    int e = a < p.A ? p.ids[a] : -1;
    if (a < p.A && (e < 0 || e >= E)) {
      raise_error(kErrBadIndex);
      e = -1;
    }
    const unsigned grp = __match_any_sync(0xffffffffu, e);
    const unsigned lower = grp & ((1u << lane) - 1u);
    const int32_t before = e >= 0 ? cnt[warp * E + e] : 0;
    __syncwarp();
    if (e >= 0 && lower == 0) cnt[warp * E + e] = before + __popc(grp);
    __syncwarp();
    e_of[r] = e;
    local_rank[r] = before + __popc(lower);
  }
  __syncthreads();
  const bool pad = p.pad && p.cap > 0;
  long long kept_sum = 0, touched = 0;
  for (int e = tid; e < E; e += kLayoutSmallThreads) {  // prefix over warps, histogram, kept
    int32_t run = 0;
    for (int w = 0; w < 32; ++w) {
      const int32_t c = cnt[w * E + e];
      cnt[w * E + e] = run;
      run += c;
    }
    const int32_t k = p.cap > 0 ? min(run, p.cap) : run;
    p.counts[e] = run;
    p.kept[e] = k;
    off[e] = pad ? p.cap : k;
    touched += k > 0;
    kept_sum += k;
  }
  kept_sum = block_reduce_ll<false>(kept_sum, red);
  touched = block_reduce_ll<false>(touched, red);
  const int32_t total = block_exclusive_scan(off, E, scratch);
  if (tid == 0) off[E] = total;
  __syncthreads();
  for (int e = tid; e <= E; e += kLayoutSmallThreads) p.offsets[e] = off[e];

  // ---- slots, row sources and the dispatch matrix
  const int epr = E / N;
  long long diag_rows = 0;  // kept rows with i == j, counted here when n_ij is not in shared memory
#pragma unroll
  for (int r = 0; r < kLayoutSmallItems; ++r) {
    const int64_t a = base + r * 32 + lane;
    const int e = e_of[r];
    if (e < 0) continue;
    const int32_t rank = cnt[warp * E + e] + local_rank[r];
    bool keep = p.cap <= 0 || rank < p.cap;
    int32_t s = keep ? off[e] + rank : -1;
    if (s >= p.R) {  // cannot happen for a consistent layout; never used as an address
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
        atomicAdd(&bins[i * N + j], 1);
      } else {
        atomicAdd(reinterpret_cast<unsigned long long*>(&p.n_ij[(int64_t)i * N + j]), 1ull);
        atomicAdd(reinterpret_cast<unsigned long long*>(&p.rank_bytes[i]), 1ull);
        atomicAdd(reinterpret_cast<unsigned long long*>(&p.rank_bytes[N + j]), 1ull);
        diag_rows += i == j;
      }
    }
  }
  __syncthreads();

  // ---- per-chip bytes and statistics: chip i's sent rows (row i of n_ij) and
  // received rows (column i); one warp per chip, lanes over the other index
  const long long rowbytes = (long long)p.h * p.ds;
  long long rmax = 0, rsum = 0, ssum = 0, dsum = 0;
  if (local) {
    for (int i = tid; i < N * N; i += kLayoutSmallThreads) p.n_ij[i] = bins[i];
    for (int i = warp; i < N; i += 32) {
      long long sent = 0, recv = 0;
      for (int j = lane; j < N; j += 32) {
        sent += bins[i * N + j];
        recv += bins[j * N + i];
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        sent += __shfl_xor_sync(0xffffffffu, sent, o);
        recv += __shfl_xor_sync(0xffffffffu, recv, o);
      }
      if (lane == 0) {
        p.rank_bytes[i] = sent * rowbytes;
        p.rank_bytes[N + i] = recv * rowbytes;
        rmax = recv > rmax ? recv : rmax;
        rsum += recv;
        ssum += sent;
        dsum += bins[i * N + i];
      }
    }
  } else {
    for (int i = tid; i < N; i += kLayoutSmallThreads) {
      const long long sent = p.rank_bytes[i], recv = p.rank_bytes[N + i];
      p.rank_bytes[i] = sent * rowbytes;
      p.rank_bytes[N + i] = recv * rowbytes;
      rmax = recv > rmax ? recv : rmax;
      rsum += recv;
      ssum += sent;
    }
    dsum = diag_rows;
  }
  rmax = block_reduce_ll<true>(rmax, red);
  rsum = block_reduce_ll<false>(rsum, red);
  ssum = block_reduce_ll<false>(ssum, red);
  dsum = block_reduce_ll<false>(dsum, red);
  if (tid == 0) {
    moe_layout_stats st;
    st.kept_total = kept_sum;
    st.dropped = p.A - kept_sum;
    st.offdiag_rows = ssum - dsum;
    st.experts_touched = (int32_t)touched;
    st.balancedness = rmax == 0 ? 1.0f : (float)((double)rsum / ((double)N * (double)rmax));
    *p.stats = st;
  }
}

// Replica map of expert-parallel load balancing: the physical expert of every
// routed (t, k) is replica t mod n_rep(e) of its logical expert e, where the
// replicas of e are rep_phys[rep_offsets[e] .. rep_offsets[e+1]).  An id outside
// [0, E) or a plan entry outside [0, P) raises the bad-index error and writes -1.
__global__ void eplb_map_kernel(const int32_t* ids, int64_t A, int K, int E, int P, const int32_t* rep_offsets,
                                const int32_t* rep_phys, int32_t* out) {
  pdl_wait();
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
