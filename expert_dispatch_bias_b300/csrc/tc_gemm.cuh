// Persistent GEMM on the 5th-generation tensor cores (tcgen05, sm_103a) over
// ragged row segments: the grouped SwiGLU FFN of the experts and the router
// logits of the bf16 layer.
//
// C[m, n] = sum_k A[m, k] * B[n, k], both operands bf16 and K-major, float32
// accumulation in TMEM.  Rows of A come in segments: expert e owns rows
// [offsets[e], offsets[e] + kept[e]) of the permuted buffer and multiplies them
// by its own weight matrix B_e; the router is the one-segment case (all T rows,
// one B).  One persistent CTA per SM walks a static round-robin list of output
// tiles of 128 rows by BN accumulator columns, ordered (segment, column tile,
// m-block) so that the m-blocks sharing a weight tile run on neighbouring SMs
// at the same time and the second read of that tile hits L2.
//
// Epilogues:
//   SwiGLU  columns 0..BN/2-1 hold gate units n0.. and columns BN/2..BN-1 the
//           matching up units, so silu(g) * u is formed without leaving the
//           tile and stored in bf16 (the intermediate activation);
//   store   bf16 store of the accumulator (the down projection);
//   logits  float32 store plus an optional per-column offset (the router).
//           With k_split > 1 the sum over K is cut into k_split slices, each
//           its own work item that stores its raw float32 tile to
//           partial[slice]; a separate kernel adds the slices in slice order
//           plus the offset (logits_reduce_kernel).
// Roles (192 threads):
//   warp 0       one thread issues TMA loads (128 A rows and BN B rows of one
//                64-element k-block, 128-byte swizzle) into a STAGES-deep ring;
//   warp 1       allocates two BN-column TMEM accumulators and one thread
//                issues tcgen05.mma (M=128, N=BN, K=16), releasing ring stages
//                with tcgen05.commit;
//   warps 2..5   drain an accumulator with tcgen05.ld (warp w reads TMEM lanes
//                32*(w%4)..+31 = tile rows), apply the epilogue, store the rows
//                inside the segment, and release the accumulator to the tile
//                after next.
// Rows past a segment's end are computed (they belong to the next segment or
// are zero-filled by TMA past the buffer) and masked on store.  Every wait is
// bounded; a wait that runs out raises the sticky error and the CTA drains
// and exits.
#pragma once

#include <cuda.h>

#include "common.cuh"

namespace moe {

constexpr int kTcBM = 128, kTcBK = 64, kTcThreads = 192;

enum TcEpilogue { kTcSwiglu = 0, kTcStore = 1, kTcLogits = 2 };

// Shared-memory and TMEM footprint of a BN-column tile with a STAGES-deep ring.
template <int BN, int STAGES>
struct TcShape {
  static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "tcgen05 M=128 needs N % 16 == 0, 16 <= N <= 256");
  static constexpr uint32_t kABytes = kTcBM * kTcBK * 2;  // 16 KB
  static constexpr uint32_t kBBytes = BN * kTcBK * 2;     // BN rows of 128 bytes
  static constexpr uint32_t kStageBytes = kABytes + kBBytes;
  static constexpr size_t kDynSmem = (size_t)STAGES * kStageBytes + 1024;  // + alignment slack
  static constexpr uint32_t kTmemCols = 2 * BN < 32 ? 32 : 2 * BN;       // power of two >= 32
  static constexpr int kChunk = BN < 32 ? BN : 32;                         // columns per tcgen05.ld
};

struct TcParams {
  const int32_t* offsets;   // [E+1] segment starts, or null: one segment of dense_rows rows at row 0
  const int32_t* kept;      // [E] segment lengths (ignored when offsets is null)
  int E;                    // segments (1 when offsets is null)
  int dense_rows;
  int n_tiles;              // column tiles per segment
  int k_blocks;             // K / 64
  int64_t b_rows;           // rows of B per segment (2I, h or 0 when all segments share B)
  int up_rows;              // SwiGLU: row offset of the up half (I)
  int n_valid;              // output columns (I, h or E)
  void* out;                // [rows, ldo] bf16 (SwiGLU, store) or float32 (logits)
  int64_t ldo;
  const float* col_bias;    // logits: per-column offset [n_valid] or null
  const int32_t* w_map;     // segment -> its B (weight) matrix, or null: segment e uses B_e
  int k_split;              // logits: slices of the K sum (<= 1: none)
  float* partial;           // logits, k_split > 1: [k_split][dense_rows][ldo] float32
};

// K-blocks [kb0, kb1) of slice s of S.
__device__ __forceinline__ void tc_k_range(int s, int S, int k_blocks, int* kb0, int* kb1) {
  *kb0 = (int)((int64_t)s * k_blocks / S);
  *kb1 = (int)((int64_t)(s + 1) * k_blocks / S);
}

// ------------------------------------------------------------------ PTX wrappers
__device__ __forceinline__ void tma_load_2d(void* smem_dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
      "[%4];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, rows of
// 128 bytes in 8-row (1024-byte) atoms.
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);        // start address
  d |= (uint64_t)1u << 16;                        // leading byte offset (unused when swizzled)
  d |= (uint64_t)(1024u >> 4) << 32;              // stride byte offset: 8 rows x 128 B
  d |= (uint64_t)1u << 46;                        // descriptor version
  d |= (uint64_t)2u << 61;                        // 128-byte swizzle
  return d;
}

// Instruction descriptor: kind::f16, A = B = bf16, D = f32, both K-major.
__host__ __device__ constexpr uint32_t umma_idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Instruction descriptor: kind::f8f6f4, A = B = E4M3 (format 0), D = f32, both
// K-major.  One MMA covers K = 32 elements (32 bytes of a 128-byte row).
__host__ __device__ constexpr uint32_t umma_idesc_e4m3(int M, int N) {
  return (1u << 4) | (0u << 7) | (0u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void umma_e4m3(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 32 lanes x N consecutive 32-bit columns: thread i gets row (lane base + i).
template <int N>
__device__ __forceinline__ void tmem_ld(uint32_t taddr, uint32_t* r);

template <>
__device__ __forceinline__ void tmem_ld<32>(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}

template <>
__device__ __forceinline__ void tmem_ld<16>(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Ties 32 registers written by an earlier tmem_ld to a point after a
// tmem_ld_wait, so the compiler cannot read them before the load completed.
__device__ __forceinline__ void tmem_regs_ready(uint32_t* r) {
  asm volatile(""
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                 "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                 "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]),
                 "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]),
                 "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
               :
               : "memory");
}

// Packs 2*n float32 values into n bf16 pairs and stores them as 16-byte vectors.
template <int N>
__device__ __forceinline__ void store_bf16_row(__nv_bfloat16* dst, const float* v) {
  uint32_t packed[N / 2];
#pragma unroll
  for (int i = 0; i < N / 2; ++i) {
    const __nv_bfloat162 b = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
    packed[i] = *reinterpret_cast<const uint32_t*>(&b);
  }
  uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int i = 0; i < N / 8; ++i)
    d[i] = make_uint4(packed[4 * i], packed[4 * i + 1], packed[4 * i + 2], packed[4 * i + 3]);
}

// Stores N float32 columns n0.. of a row, skipping columns >= n_valid.
template <int N>
__device__ __forceinline__ void store_f32_cols(float* row, int n0, int n_valid, bool vec, const float* a) {
  if (vec && n0 + N <= n_valid) {
    float4* d = reinterpret_cast<float4*>(row + n0);
#pragma unroll
    for (int i = 0; i < N / 4; ++i) d[i] = make_float4(a[4 * i], a[4 * i + 1], a[4 * i + 2], a[4 * i + 3]);
  } else {
#pragma unroll
    for (int i = 0; i < N; ++i)
      if (n0 + i < n_valid) row[n0 + i] = a[i];
  }
}

// ------------------------------------------------------------------ tile schedule
struct TcTile {
  int e;        // segment (expert)
  int m0;       // first row (absolute, in A)
  int m_end;    // end of the segment
  int nt;       // column tile
};

// mbp[e] = m-blocks of segments < e (exclusive prefix), mbp[E] = total.
__device__ __forceinline__ TcTile tc_decode(int t, const int32_t* mbp, const TcParams& p) {
  int lo = 0, hi = p.E - 1;  // last segment whose first tile index is <= t
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
  const int mb = local - r.nt * cnt;
  const int seg0 = p.offsets ? p.offsets[e] : 0;
  r.m0 = seg0 + mb * kTcBM;
  r.m_end = seg0 + (p.offsets ? p.kept[e] : p.dense_rows);
  return r;
}

template <int EPI, int BN, int STAGES>
__global__ void __launch_bounds__(kTcThreads, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b, TcParams p) {
  pdl_wait();
  using S = TcShape<BN, STAGES>;
  constexpr int CH = S::kChunk;
  extern __shared__ uint8_t dyn_smem[];
  __shared__ __align__(8) uint64_t full_bar[STAGES], empty_bar[STAGES];
  __shared__ __align__(8) uint64_t tmem_full[2], tmem_empty[2], drain_bar;
  __shared__ uint32_t tmem_holder;
  __shared__ volatile uint32_t abort_flag;
  __shared__ int32_t mbp[1025];
  __shared__ int32_t scan_scratch[33];

  uint8_t* tiles = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dyn_smem) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // ---- per-segment m-block prefix (every CTA computes it from offsets/kept)
  for (int e = tid; e < p.E; e += kTcThreads)
    mbp[e] = ((p.offsets ? p.kept[e] : p.dense_rows) + kTcBM - 1) / kTcBM;
  __syncthreads();
  const int32_t total_mb = block_exclusive_scan(mbp, p.E, scan_scratch);
  if (tid == 0) mbp[p.E] = total_mb;
  const int KS = (EPI == kTcLogits && p.k_split > 1) ? p.k_split : 1;
  const int total_tiles = total_mb * p.n_tiles * KS;  // work items: (tile, K slice)

  if (tid == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
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
                 "r"(S::kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = tmem_holder;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t armed = 0;  // bit s: stage s was ever armed; its last arm had parity (phase bit at the time)
      uint32_t armed_parity = 0;
      for (int t = blockIdx.x; t < total_tiles && !abort_flag; t += gridDim.x) {
        const TcTile tl = tc_decode(t / KS, mbp, p);
        int kb0, kb1;
        tc_k_range(t % KS, KS, p.k_blocks, &kb0, &kb1);
        const int64_t brow = (int64_t)(p.w_map != nullptr ? p.w_map[tl.e] : tl.e) * p.b_rows;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(&empty_bar[stage], phase ^ 1u, &abort_flag)) {
            abort_flag = 1;
            raise_error(kErrTimeout);
            break;
          }
          uint8_t* sa = tiles + (size_t)stage * S::kStageBytes;
          uint8_t* sb = sa + S::kABytes;
          mbar_expect_tx(&full_bar[stage], S::kStageBytes);
          const int kx = kb * kTcBK;
          tma_load_2d(sa, &map_a, kx, tl.m0, &full_bar[stage]);
          if (EPI == kTcSwiglu) {
            const int n0 = tl.nt * (BN / 2);
            tma_load_2d(sb, &map_b, kx, (int)(brow + n0), &full_bar[stage]);
            tma_load_2d(sb + S::kBBytes / 2, &map_b, kx, (int)(brow + p.up_rows + n0), &full_bar[stage]);
          } else {
            const int n0 = tl.nt * BN;
            tma_load_2d(sb, &map_b, kx, (int)(brow + n0), &full_bar[stage]);
          }
          armed |= 1u << stage;
          armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (abort_flag) {
        // let the last load armed on every stage land before the CTA's shared
        // memory is released (bounded like every other wait)
        for (int s = 0; s < STAGES; ++s)
          if ((armed >> s) & 1u) mbar_wait(&full_bar[s], (armed_parity >> s) & 1u);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = umma_idesc_bf16(kTcBM, BN);
      // descriptor of stage 0's A tile; stage s adds s stage sizes (start
      // addresses stay below 256 KB, so the 14-bit address field never carries)
      const uint64_t d0 = umma_desc_sw128(smem_u32(tiles));
      int stage = 0;
      uint32_t phase = 0;
      bool ready = false;   // full_bar[stage] already seen complete by the early test
      int acc = 0;
      uint32_t acc_phase = 0;
      for (int t = blockIdx.x; t < total_tiles && !abort_flag; t += gridDim.x) {
        if (!mbar_wait(&tmem_empty[acc], acc_phase ^ 1u, &abort_flag)) {
          abort_flag = 1;
          raise_error(kErrTimeout);
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
        bool ok = true;
        int kb0, kb1;
        tc_k_range(t % KS, KS, p.k_blocks, &kb0, &kb1);
        if (stage == 0 && (kb1 - kb0) % STAGES == 0) {
          // whole groups of STAGES k-blocks starting at stage 0: unrolled over
          // the stages, so stage indices, descriptors and the next stage to
          // test are constants and the thread spends fewer cycles between
          // k-blocks
          for (int kb = kb0; kb < kb1 && ok; kb += STAGES) {
#pragma unroll
            for (int u = 0; u < STAGES; ++u) {
              if (!ready && !mbar_wait(&full_bar[u], phase, &abort_flag)) {
                abort_flag = 1;
                raise_error(kErrTimeout);
                ok = false;
                break;
              }
              tc_fence_after();
              const uint64_t da = d0 + (uint64_t)(u * (S::kStageBytes >> 4));
              const uint64_t db = da + (S::kABytes >> 4);
              umma_bf16(d_tmem, da, db, idesc, (kb + u) != kb0 ? 1u : 0u);
              umma_bf16(d_tmem, da + 2, db + 2, idesc, 1u);
              ready = mbar_try_wait(&full_bar[(u + 1) % STAGES], u + 1 == STAGES ? phase ^ 1u : phase);
              umma_bf16(d_tmem, da + 4, db + 4, idesc, 1u);
              umma_bf16(d_tmem, da + 6, db + 6, idesc, 1u);
              umma_commit(&empty_bar[u]);
            }
            phase ^= 1u;
          }
        } else
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!ready && !mbar_wait(&full_bar[stage], phase, &abort_flag)) {
            abort_flag = 1;
            raise_error(kErrTimeout);
            ok = false;
            break;
          }
          tc_fence_after();
          // a K=16 step advances 32 bytes (2 descriptor units) in both tiles
          const uint64_t da = d0 + (uint64_t)((uint32_t)stage * (S::kStageBytes >> 4));
          const uint64_t db = da + (S::kABytes >> 4);
          const int next = stage + 1 == STAGES ? 0 : stage + 1;
          const uint32_t next_phase = stage + 1 == STAGES ? phase ^ 1u : phase;
          static_assert(kTcBK / 16 == 4, "four K=16 steps per k-block");
          umma_bf16(d_tmem, da, db, idesc, kb != kb0 ? 1u : 0u);
          umma_bf16(d_tmem, da + 2, db + 2, idesc, 1u);
          // test the next stage while these MMAs run (the single issuing thread
          // is the pipe's only feeder); a completed phase stays complete until
          // this thread releases the stage
          ready = mbar_try_wait(&full_bar[next], next_phase);
          umma_bf16(d_tmem, da + 4, db + 4, idesc, 1u);
          umma_bf16(d_tmem, da + 6, db + 6, idesc, 1u);
          umma_commit(&empty_bar[stage]);
          stage = next;
          phase = next_phase;
        }
        if (!ok) break;
        umma_commit(&tmem_full[acc]);
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      // all MMAs issued by this thread are complete once drain_bar fires
      umma_commit(&drain_bar);
      mbar_wait(&drain_bar, 0u);
    }
  } else {
    // ------------------------------------------------------------ epilogue (warps 2..5)
    const int quarter = warp & 3;
    // float32 rows as float4 when every row start is 16-byte aligned (the
    // partial buffers share the output's row pitch and are 256-byte aligned)
    const bool vec_out = (p.ldo % 4) == 0 && (reinterpret_cast<uintptr_t>(p.out) & 15u) == 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int t = blockIdx.x; t < total_tiles; t += gridDim.x) {
      if (!mbar_wait(&tmem_full[acc], acc_phase, &abort_flag)) {
        abort_flag = 1;
        raise_error(kErrTimeout);
        break;
      }
      tc_fence_after();
      const int slice = t % KS;
      const TcTile tl = tc_decode(t / KS, mbp, p);
      const int row = tl.m0 + quarter * 32 + lane;
      const bool valid = row < tl.m_end;
      const uint32_t taddr = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * BN);
      if (EPI == kTcSwiglu) {
        const int n0 = tl.nt * (BN / 2);
        __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(p.out) + (int64_t)row * p.ldo;
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
              a[i] = __fdividef(gi, 1.0f + __expf(-gi)) * __uint_as_float(u[i]);  // fast forms, as in ffn_grouped.cuh
            }
            store_bf16_row<CH>(orow + n0 + c, a);
          }
        }
      } else if (EPI == kTcStore) {
        const int n0 = tl.nt * BN;
        __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(p.out) + (int64_t)row * p.ldo;
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
      } else {
        const int n0 = tl.nt * BN;
        // a slice stores its raw sum to its partial buffer; the offset is added
        // once, to the sum of the slices
        float* orow = KS > 1 ? p.partial + ((int64_t)slice * p.dense_rows + row) * p.ldo
                             : static_cast<float*>(p.out) + (int64_t)row * p.ldo;
        const bool bias = KS == 1 && p.col_bias != nullptr;
#pragma unroll 1
        for (int c = 0; c < BN; c += CH) {
          uint32_t v[CH];
          tmem_ld<CH>(taddr + c, v);
          tmem_ld_wait();
          if (valid) {
            float a[CH];
#pragma unroll
            for (int i = 0; i < CH; ++i) {
              const int n = n0 + c + i;
              a[i] = __uint_as_float(v[i]) + ((bias && n < p.n_valid) ? p.col_bias[n] : 0.0f);
            }
            store_f32_cols<CH>(orow, n0 + c, p.n_valid, vec_out, a);
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&tmem_empty[acc]);
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(S::kTmemCols)
                 : "memory");
  }
}

// Router logits from k_split partial sums: out[i] = ((P_0[i] + P_1[i]) + ...)
// + offset[i % E], slices added in slice order.  P is [k_split][n] with n = T*E;
// float4 lanes when E % 4 == 0 (every partial starts 256-byte aligned).
__global__ void __launch_bounds__(256) logits_reduce_kernel(const float* P, int k_split, int64_t n, int E,
                                                            const float* off, float* out) {
  pdl_wait();
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  if ((E & 3) == 0) {
    const int64_t n4 = n >> 2;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += stride) {
      float4 a = __ldcg(reinterpret_cast<const float4*>(P) + i);
      for (int s = 1; s < k_split; ++s) {
        const float4 b = __ldcg(reinterpret_cast<const float4*>(P + (int64_t)s * n) + i);
        a.x += b.x;
        a.y += b.y;
        a.z += b.z;
        a.w += b.w;
      }
      if (off != nullptr) {
        const int e = (int)((i << 2) % E);
        a.x += off[e];
        a.y += off[e + 1];
        a.z += off[e + 2];
        a.w += off[e + 3];
      }
      reinterpret_cast<float4*>(out)[i] = a;
    }
  } else {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
      float a = __ldcg(P + i);
      for (int s = 1; s < k_split; ++s) a += __ldcg(P + (int64_t)s * n + i);
      if (off != nullptr) a += off[i % E];
      out[i] = a;
    }
  }
}

}  // namespace moe
