// A warp-specialised tcgen05 GEMM mainloop shared by the dense contractions.
//
// CTA = 2 + E warps: warp 0 issues TMA loads into an S-stage shared-memory
// ring, warp 1 issues tcgen05.mma (one thread) into one of two 128 x BN fp32
// accumulators in TMEM (double-buffered, so the MMAs of the next tile run
// while the epilogue drains this one), and the E = Epi::kEpiWarps (4, 8, 12
// or 16) warps from 2 on drain the accumulator and hand rows to an op-specific
// epilogue: warp w reads the TMEM lane quarter w % 4 it may access, and with
// E > 4 the E / 4 warps of a quarter split the BN columns between them.  The CTA owns
// one BN-column tile (blockIdx.x) and walks row tiles t < epi.tiles(M)
// (strided by gridDim.y, or a contiguous block of them); the epilogue object
// maps a tile to its TMA coordinates.  blockIdx.z selects a chunk of the K
// dimension.
//
// Operands, all bf16 with a 128-byte swizzle:
//   A: NA K-major tiles [128 rows][64 k] (NA = 2: a hi/lo split of an fp32
//      operand, accumulated as A_hi.B + A_lo.B)
//   B: NB tiles, K-major [BN rows][64 k] or MN-major [64 k][BN cols]
//      (NB = 2: hi/lo split, A.B_hi + A.B_lo)
// Every mbarrier wait is bounded (tc::mbar_wait); on a timeout the CTA sets
// the status word, drains its in-flight copies and MMAs, frees TMEM and
// returns.
//
// Cluster reduction (Epi::kClusterReduce): the gridDim.z CTAs that share a
// row tile (chunks of K, or slices of another summed dimension) form one
// thread-block cluster (<= 8 CTAs).  Each CTA leaves its 128 x BN fp32
// result in its own shared memory (over the stage ring, idle by then); after
// a cluster barrier, CTA z finishes rows [128 z / Z, 128 (z+1) / Z) reading
// every rank's rows through distributed shared memory in rank order, so the
// sum is deterministic and no partial goes through global memory.
#pragma once

#include <cstdlib>

#include "tc.cuh"

namespace ps {

struct TcMaps {
  CUtensorMap a[2];
  CUtensorMap b[2];
};

struct TcShape {
  int M;             // rows of A (an upper bound when M_dev is set)
  const int* M_dev;  // device row count, or nullptr
  int KB;            // K / 64
  int kpc;           // 64-wide K blocks per blockIdx.z chunk
  int* status;
  int split_max_rows;  // K is split over blockIdx.z only while M <= this;
                       // above it blockIdx.z == 0 takes the whole K range
  int starve_loads;    // test hook: the producer issues no copies, so the
                       // MMA thread's bounded wait must give up (set only
                       // when PS_TEST_STARVE_TMA is in the environment)
  int a_rows;          // A rows each TMA tile brings (the A maps' box height):
                       // 64 when M <= 64 (the MMA's rows 64..127 then read
                       // stale shared memory into accumulator rows nobody
                       // stores), 0 or 128 otherwise
};

// KS: 64-wide k-blocks per pipeline stage.  Measured on GB300, one SM's TMA
// stream delivers about 1.5x more with 64 KB stages than with 32 KB ones at
// the same bytes in flight (fewer, larger transactions per mbarrier turn),
// so a k-block of 32 KB or less is staged in pairs.
template <int BN, int NA, int NB, bool B_MN>
__host__ __device__ constexpr int tc_ks() {
  return NA * 128 * 64 * 2 + NB * BN * 64 * 2 <= 32768 ? 2 : 1;
}
template <int BN, int NA, int NB, bool B_MN, int KS = tc_ks<BN, NA, NB, B_MN>()>
struct TcCfg {
  static constexpr uint32_t kA = 128 * 64 * 2;
  static constexpr uint32_t kB = BN * 64 * 2;
  static constexpr uint32_t kSub = NA * kA + NB * kB;  // one k-block
  static constexpr uint32_t kStage = KS * kSub;
  static constexpr int kStages = (200 * 1024 / kStage) < 8 ? (200 * 1024 / kStage) : 8;
  static constexpr uint32_t kScratch = 16384;  // epilogue scratch after the barriers
  static constexpr size_t kSmem = 1024 + kStages * kStage + 512 + kScratch;
  static constexpr uint32_t kRedLd = BN + 4;  // row stride (floats) of a cluster result
  static constexpr uint32_t kIdesc = tc::idesc_bf16(128, BN, B_MN);
};

// Epi must provide (device, const unless noted):
//   static constexpr bool kA3D     A maps are 3-D {k, head, row}
//   static constexpr bool kBlocked CTA y takes the contiguous tile range
//                                  [y*ceil(T/gy), ...) instead of striding
//   int tiles(int M)               number of 128-row tiles
//   int arow(int t), ahead(t)      A row (and head, 3-D maps) of tile t
//   int bsel(int t, int n0)        which b map when NB == 1 (else ignored)
//   int bcoord(int t, int n0)      B column (MN-major) or row (K-major)
//   int bkoff(int t)               added to the K coordinate of B
//   struct State                   per-thread epilogue state
//   void consume(int t, int r, int n0, int z, uint32_t taddr, State&)
//        row r (0..127) of tile t; taddr = TMEM address of the row's
//        column 0 (read with tc::tmem_ld32, warp-collective); TMEM is
//        released after it returns
//   void tile_done(int t, int r, int n0, int z, uint8_t* scratch, State&)
//        called by the 128 epilogue threads together after consume; may
//        synchronise with epi_bar_sync(); scratch = 16 KB of shared memory
//   static constexpr int kEpiWarps  4 (default), 8, 12 or 16; above 4 the
//        engine calls consume_part / tile_done_part / consume_red_part, which
//        also take the thread's column part (0 .. kEpiWarps / 4 - 1) and the
//        scratch, and may synchronise the epilogue warps with
//        epi_bar_sync_n<32 * kEpiWarps>()
//   static constexpr bool kZSplitsK  blockIdx.z chunks K (else z is the
//        epilogue's own and every CTA takes the whole K range)
//   bool tile_range(int T, int* begin, int* end, int* step)  optional
//        override of the CTA's tile walk (returns true when it applies)
//   bool active(int t)             optional (not with kClusterReduce): false
//        skips tile t in all three roles -- no copies, no MMAs, no
//        epilogue call; read at the tile from memory that earlier kernels
//        wrote, so every role sees the same answer
//   static constexpr int kAccBufs   accumulators in TMEM (default 2, double
//        buffered: the MMAs of the next tile run under this tile's epilogue;
//        1: the next tile's MMAs wait for the epilogue, for epilogues that
//        need the TMEM columns of the second for themselves)
//   static constexpr int kExtraCols  TMEM columns the epilogue keeps for
//        itself past the two accumulators (default 0); with it, State has a
//        uint32_t `extra` that the engine sets to their address in the
//        thread's lane quarter before the first tile
//   static constexpr bool kAfterTiles, void after_tiles(int t_begin,
//        uint32_t tmem)  optional: with kAfterTiles, every thread of the CTA
//        calls after_tiles once all its tiles are done (after a CTA barrier,
//        with the stage ring idle and TMEM, at address tmem, still
//        allocated; warp w may read TMEM lane quarter w % 4)
//   void prefetch(uint8_t* scratch, int i, int n)  optional: run by the n
//        epilogue threads (index i) before they wait for the first
//        accumulator, to stage data the epilogue reads later into the
//        scratch (with kClusterReduce, read in reduce(), after the CTA and
//        cluster barriers)
// and with kClusterReduce (instead of consume / tile_done):
//   void consume_red(t, r, n0, z, taddr, State&, float* red_row)
//        red_row = this row's slot in the CTA's result (kRedLd floats), or
//        nullptr before the CTA's last tile
//   void reduce(const float* red, int z, int Z, uint8_t* scratch)
//        called by every thread of the CTA after a cluster barrier; must call
//        tc::cluster_arrive() exactly once, uniformly, after its last read
//        of another CTA's shared memory (the CTA waits before leaving)
// TMEM columns a CTA allocates: the two accumulators and the epilogue's
// own, rounded up to a power of two (>= 32, <= 512).
template <int BN, class Epi>
__host__ __device__ constexpr uint32_t tc_tmem_cols() {
  constexpr int need = Epi::kAccBufs * BN + Epi::kExtraCols;
  static_assert(need <= 512, "TMEM holds 512 columns");
  return need <= 32 ? 32 : need <= 64 ? 64 : need <= 128 ? 128 : need <= 256 ? 256 : 512;
}

// The CTA's stage ring: the start of its dynamic shared memory, 1024-byte
// aligned.  Once the accumulator of the CTA's last tile is full, every copy
// into the ring has landed and every MMA that read it has completed, so the
// epilogue may use the ring's Cfg::kStages * Cfg::kStage bytes from then on
// (the last tile's consume / tile_done).
__device__ __forceinline__ uint8_t* tc_ring_base() {
  extern __shared__ uint8_t smem_raw[];
  return reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
}

template <int BN, int NA, int NB, bool B_MN, class Epi>
__device__ __forceinline__ void tc_gemm_body(const TcMaps& maps, const TcShape& sh,
                                             const Epi& epi) {
  // k-blocks go through the ring KS at a time; a chunk with an odd count
  // loads one k-block past its end (out of range, or the next chunk's) into
  // its last stage and issues no MMA for it
  constexpr int KS = tc_ks<BN, NA, NB, B_MN>();
  using Cfg = TcCfg<BN, NA, NB, B_MN, KS>;
  constexpr int S = Cfg::kStages;
  uint8_t* smem = tc_ring_base();
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S * Cfg::kStage);
  uint64_t* empty = full + S;
  uint64_t* acc_full = empty + S;      // [2]
  uint64_t* acc_empty = acc_full + 2;  // [2]
  uint64_t* drain = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  uint8_t* epi_scratch = smem + S * Cfg::kStage + 512;

  // tiles of this CTA first: a CTA without work leaves before any set-up.
  // In a cluster, whose barriers every CTA joins, only whole clusters leave:
  // those whose row-tile slot is empty whatever the K split (a K chunk
  // z > 0 left without tiles because K is not split still joins).
  static_assert(!(Epi::kClusterReduce && Epi::kBlocked), "cluster tiles are strided");
  if (sh.M_dev != nullptr) pdl_prologue();  // the row count is an earlier kernel's output
  const int M = sh.M_dev != nullptr ? min(*sh.M_dev, sh.M) : sh.M;
  const bool ksplit = Epi::kZSplitsK && M <= sh.split_max_rows;
  const int T_all = epi.tiles(M);
  // K not split although the grid has K chunks (the rows outgrew
  // split_max_rows, known only on the device): the gridDim.z CTAs of a
  // column tile take turns on the row tiles instead of idling, z fastest,
  // so the clusters whose first tile lies past the end hold no work at all
  const bool zrows = Epi::kZSplitsK && !ksplit && gridDim.z > 1;
  const int T = T_all;
  int t_begin = zrows ? (int)(blockIdx.y * gridDim.z + blockIdx.z) : (int)blockIdx.y;
  int t_end = T, t_step = zrows ? (int)(gridDim.y * gridDim.z) : (int)gridDim.y;
  if constexpr (Epi::kBlocked) {
    const int per = (T + gridDim.y - 1) / gridDim.y;
    t_begin = blockIdx.y * per;
    t_end = min(T, t_begin + per);
    t_step = 1;
  }
  epi.tile_range(T, &t_begin, &t_end, &t_step);
  if constexpr (Epi::kClusterReduce) {
    int b0 = blockIdx.y, e0 = T_all, s0 = gridDim.y;
    epi.tile_range(T_all, &b0, &e0, &s0);
    if (zrows) b0 = blockIdx.y * gridDim.z;  // the cluster's first tile (z = 0)
    if (b0 >= e0) return;
  } else {
    if (t_begin >= t_end) return;
    // every tile of this CTA skipped (active() false): leave before set-up
    bool any = false;
    for (int t = t_begin; t < t_end && !any; t += t_step) any = epi.active(t);
    if (!any) return;
  }

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      tc::mbar_init(full + s, 1);
      tc::mbar_init(empty + s, 1);
    }
    for (int j = 0; j < 2; ++j) {
      tc::mbar_init(acc_full + j, 1);
      tc::mbar_init(acc_empty + j, Epi::kEpiWarps);
    }
    tc::mbar_init(drain, 1);
    *abort_flag = 0;
    tc::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tc::tma_prefetch(&maps.a[0]);
    tc::tma_prefetch(&maps.b[0]);
  }
  if (warp == 1) tc::tmem_alloc(tmem_slot, tc_tmem_cols<BN, Epi>());
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  pdl_prologue();  // set-up above overlaps the previous grid's tail

  const int n0 = blockIdx.x * BN;
  const int kb0 = ksplit ? blockIdx.z * sh.kpc : 0;
  const int kb1 = ksplit ? min(sh.KB, kb0 + sh.kpc) : sh.KB;

  if (warp == 0) {
    if (lane == 0 && !sh.starve_loads) {
      const uint32_t a_bytes = (sh.a_rows > 0 ? sh.a_rows : 128) * 128u;
      const uint32_t stage_bytes = KS * (NA * a_bytes + NB * Cfg::kB);
      int it = 0;
      bool ok = true;
      for (int t = t_begin; ok && t < t_end; t += t_step) {
        if constexpr (!Epi::kClusterReduce) {
          if (!epi.active(t)) continue;
        }
        const int arow = epi.arow(t);
        const int ahead = epi.ahead(t);
        const int bkoff = epi.bkoff(t);
        const int bsel = epi.bsel(t, n0);
        const int bcol = epi.bcoord(t, n0);
        for (int kb = kb0; kb < kb1; kb += KS) {
          const int s = it % S;
          const uint32_t ph = (it / S) & 1;
          if (!tc::mbar_wait(empty + s, ph ^ 1, sh.status, abort_flag)) { ok = false; break; }
          tc::mbar_expect_tx(full + s, stage_bytes);
#pragma unroll
          for (int sub = 0; sub < KS; ++sub) {
            // a k-block past this chunk (an odd last one) is still loaded,
            // from past the tensor's K extent, so the stage's bytes are whole
            const int kc = kb + sub < kb1 ? (kb + sub) * 64 : sh.KB * 64;
            uint8_t* st = smem + s * Cfg::kStage + sub * Cfg::kSub;
#pragma unroll
            for (int a = 0; a < NA; ++a) {
              if constexpr (Epi::kA3D)
                tc::tma_load_3d(st + a * Cfg::kA, &maps.a[a], full + s, kc, ahead, arow);
              else
                tc::tma_load_2d(st + a * Cfg::kA, &maps.a[a], full + s, kc, arow);
            }
            uint8_t* bs = st + NA * Cfg::kA;
#pragma unroll
            for (int bb = 0; bb < NB; ++bb) {
              const CUtensorMap* bm = &maps.b[NB == 1 ? bsel : bb];
              if constexpr (B_MN) {
#pragma unroll
                for (int q = 0; q < BN / 64; ++q)
                  tc::tma_load_2d(bs + bb * Cfg::kB + q * 8192, bm, full + s, bcol + 64 * q,
                                  kc + bkoff);
              } else {
                tc::tma_load_2d(bs + bb * Cfg::kB, bm, full + s, kc + bkoff, bcol);
              }
            }
          }
          ++it;
        }
      }
      if (!ok) {  // let every copy already issued land before the CTA exits
        for (int j = it > S ? it - S : 0; j < it; ++j) {
          const uint64_t t0 = tc::globaltimer();
          while (!tc::mbar_try_wait(full + j % S, (j / S) & 1) &&
                 tc::globaltimer() - t0 < tc::kWaitLimitNs) {
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      int it = 0, tcount = 0;
      bool ok = true;
      for (int t = t_begin; ok && t < t_end; t += t_step) {
        if constexpr (!Epi::kClusterReduce) {
          if (!epi.active(t)) continue;
        }
        const int buf = tcount % Epi::kAccBufs;
        const uint32_t dacc = tmem + buf * BN;
        if (!tc::mbar_wait(acc_empty + buf, ((tcount / Epi::kAccBufs) & 1) ^ 1, sh.status,
                           abort_flag)) {
          ok = false;
          break;
        }
        tc::fence_after_sync();
        for (int kb = kb0; kb < kb1; kb += KS) {
          const int s = it % S;
          const uint32_t ph = (it / S) & 1;
          if (!tc::mbar_wait(full + s, ph, sh.status, abort_flag)) { ok = false; break; }
          tc::fence_after_sync();
#pragma unroll
          for (int sub = 0; sub < KS; ++sub) {
          if (kb + sub >= kb1) break;  // the zero-filled k-block past the chunk
          const uint32_t a_base = tc::smem_u32(smem + s * Cfg::kStage + sub * Cfg::kSub);
          const uint32_t b_base = a_base + NA * Cfg::kA;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint32_t acc = (kb + sub > kb0 || kk > 0) ? 1u : 0u;
            const uint64_t ad = tc::desc_sw128(a_base + kk * 32, 16, 1024);
            const uint64_t bd = B_MN ? tc::desc_sw128(b_base + kk * 2048, 8192, 1024)
                                     : tc::desc_sw128(b_base + kk * 32, 16, 1024);
            tc::mma_bf16(dacc, ad, bd, Cfg::kIdesc, acc);
            if constexpr (NA == 2)
              tc::mma_bf16(dacc, tc::desc_sw128(a_base + Cfg::kA + kk * 32, 16, 1024), bd,
                           Cfg::kIdesc, 1u);
            if constexpr (NB == 2) {
              const uint64_t bd2 =
                  B_MN ? tc::desc_sw128(b_base + Cfg::kB + kk * 2048, 8192, 1024)
                       : tc::desc_sw128(b_base + Cfg::kB + kk * 32, 16, 1024);
              tc::mma_bf16(dacc, ad, bd2, Cfg::kIdesc, 1u);
            }
          }
          }
          tc::mma_commit(empty + s);
          ++it;
        }
        if (!ok) break;
        tc::mma_commit(acc_full + buf);
        ++tcount;
      }
      if (!ok) {  // wait for the MMAs already issued before TMEM is freed
        tc::mma_commit(drain);
        const uint64_t t0 = tc::globaltimer();
        while (!tc::mbar_try_wait(drain, 0) && tc::globaltimer() - t0 < tc::kWaitLimitNs) {
        }
      }
    }
  } else {
    const int quarter = warp & 3, part = (warp - 2) >> 2;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const int r = quarter * 32 + lane;
    // the epilogue warps stage their per-tile data while the mainloop runs
    epi.prefetch(epi_scratch, threadIdx.x - 64, 32 * Epi::kEpiWarps);
    typename Epi::State est;
    if constexpr (Epi::kExtraCols > 0) est.extra = tmem + Epi::kAccBufs * BN + lane_base;
    int tcount = 0;
    for (int t = t_begin; t < t_end; t += t_step) {
      if constexpr (!Epi::kClusterReduce) {
        if (!epi.active(t)) continue;
      }
      const int buf = tcount % Epi::kAccBufs;
      if (!tc::mbar_wait(acc_full + buf, (tcount / Epi::kAccBufs) & 1, sh.status, abort_flag))
        break;
      tc::fence_after_sync();
      if constexpr (Epi::kClusterReduce) {
        // the stage ring is idle once the CTA's last accumulator is full
        float* red_row = t + t_step >= t_end
                             ? reinterpret_cast<float*>(smem) + r * Cfg::kRedLd
                             : nullptr;
        if constexpr (Epi::kEpiWarps > 4)
          epi.consume_red_part(t, r, part, n0, blockIdx.z, tmem + buf * BN + lane_base,
                               epi_scratch, est, red_row);
        else
          epi.consume_red(t, r, n0, blockIdx.z, tmem + buf * BN + lane_base, est, red_row);
      } else if constexpr (Epi::kEpiWarps > 4) {
        epi.consume_part(t, r, part, n0, blockIdx.z, tmem + buf * BN + lane_base, epi_scratch,
                         est);
      } else {
        epi.consume(t, r, n0, blockIdx.z, tmem + buf * BN + lane_base, est);
      }
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(acc_empty + buf);
      if constexpr (!Epi::kClusterReduce) {
        if constexpr (Epi::kEpiWarps > 4)
          epi.tile_done_part(t, r, part, n0, blockIdx.z, epi_scratch, est);
        else
          epi.tile_done(t, r, n0, blockIdx.z, epi_scratch, est);
      }
      ++tcount;
    }
  }
  // lanes 1..31 of the TMA and MMA warps wait for their lane 0 here, so each
  // warp reaches the CTA barrier converged (the barrier is warp-aligned)
  __syncwarp();
  __syncthreads();
  if constexpr (Epi::kAfterTiles) {
    // skipped after a timed-out wait (the status word is set already)
    if (t_begin < t_end && *abort_flag == 0) epi.after_tiles(t_begin, tmem);
    __syncthreads();
  }
  pdl_trigger();
  if constexpr (Epi::kClusterReduce) {
    static_assert(128 * Cfg::kRedLd * 4 <= Cfg::kStages * Cfg::kStage, "cluster result > ring");
    tc::cluster_sync_all();
    epi.reduce(reinterpret_cast<const float*>(smem), blockIdx.z, gridDim.z, epi_scratch);
  }
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, tc_tmem_cols<BN, Epi>());
  }
  // no CTA leaves while another still reads its result
  if constexpr (Epi::kClusterReduce) tc::cluster_wait();
}

template <int BN, int NA, int NB, bool B_MN, class Epi>
__global__ void __launch_bounds__(64 + 32 * Epi::kEpiWarps, 1)
k_tc_gemm(const __grid_constant__ TcMaps maps, const TcShape sh, const Epi epi) {
  tc_gemm_body<BN, NA, NB, B_MN, Epi>(maps, sh, epi);
}

// Plain epilogue base: 2-D maps, strided tiles, no B offset, one b map.
struct TcEpiBase {
  static constexpr int kEpiWarps = 4;
  static constexpr int kExtraCols = 0;
  static constexpr int kAccBufs = 2;
  static constexpr bool kAfterTiles = false;
  static constexpr bool kA3D = false;
  static constexpr bool kBlocked = false;
  static constexpr bool kClusterReduce = false;
  static constexpr bool kZSplitsK = true;
  __device__ bool tile_range(int, int*, int*, int*) const { return false; }
  __device__ bool active(int) const { return true; }
  __device__ void prefetch(uint8_t*, int, int) const {}
  __device__ void after_tiles(int, uint32_t) const {}
  __device__ int ahead(int) const { return 0; }
  __device__ int bkoff(int) const { return 0; }
  __device__ int bsel(int, int) const { return 0; }
};

__device__ __forceinline__ void epi_bar_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }
// The epilogue warps only (NT = 32 x their number).
template <int NT>
__device__ __forceinline__ void epi_bar_sync_n() {
  asm volatile("bar.sync 1, %0;" ::"n"(NT) : "memory");
}

// Rows [r0, r1) of the cluster's Z (<= ZMAX) results (row stride ld floats,
// at `red` in every CTA's shared memory), summed in rank order four columns
// at a time by all threads of the CTA; each thread issues the loads of a
// batch of items (every rank, LOADS 16-byte loads: 32 where the kernel's
// registers allow) before using any, since a distributed-shared-memory load
// is a round trip of about half a microsecond.  f(r, c, sum) takes columns
// c..c+3 of row r.  ncol: a multiple of 4.
template <int ZMAX, int LOADS = 16, class F>
__device__ __forceinline__ void cluster_rows_sum(const float* red, uint32_t ld, int r0, int r1,
                                                 int ncol, int Z, F&& f) {
  constexpr int kBatch = LOADS / ZMAX > 1 ? LOADS / ZMAX : 1;
  uint32_t base[ZMAX];
  const uint32_t local = tc::smem_u32(red);
#pragma unroll
  for (int q = 0; q < ZMAX; ++q) base[q] = q < Z ? tc::cluster_map(local, q) : 0u;
  const int c4n = ncol / 4, items = (r1 - r0) * c4n, nthr = blockDim.x;
  for (int it0 = threadIdx.x; it0 < items; it0 += kBatch * nthr) {
    float4 x[kBatch][ZMAX];
#pragma unroll
    for (int k = 0; k < kBatch; ++k) {
      const int it = it0 + k * nthr;
      if (it < items) {
        const int r = r0 + it / c4n, c = (it % c4n) * 4;
        const uint32_t off = (uint32_t)(r * ld + c) * 4u;
#pragma unroll
        for (int q = 0; q < ZMAX; ++q)
          if (q < Z) x[k][q] = tc::ld_dsmem_v4(base[q] + off);
      }
    }
#pragma unroll
    for (int k = 0; k < kBatch; ++k) {
      const int it = it0 + k * nthr;
      if (it < items) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int q = 0; q < ZMAX; ++q)
          if (q < Z) {
            acc.x += x[k][q].x;
            acc.y += x[k][q].y;
            acc.z += x[k][q].z;
            acc.w += x[k][q].w;
          }
        f(r0 + it / c4n, (it % c4n) * 4, acc);
      }
    }
  }
}

template <int BN, int NA, int NB, bool B_MN, class Epi>
cudaError_t launch_tc_gemm(const TcMaps& maps, const TcShape& sh, const Epi& epi, dim3 grid,
                           cudaStream_t s) {
  using Cfg = TcCfg<BN, NA, NB, B_MN>;
  auto kern = k_tc_gemm<BN, NA, NB, B_MN, Epi>;
  static bool attr_set = false;  // per instantiation
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(Cfg::kSmem));
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  TcShape shape = sh;
  shape.starve_loads = std::getenv("PS_TEST_STARVE_TMA") != nullptr ? 1 : 0;
  if constexpr (Epi::kClusterReduce) {
    if (grid.z < 1 || grid.z > 8) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(64 + 32 * Epi::kEpiWarps);
    cfg.dynamicSmemBytes = Cfg::kSmem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = kUsePdl ? 1 : 0;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 1;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = grid.z;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return launch_ex(cfg, kern, maps, shape, epi);
  }
  launch_pdl(kern, grid, 64 + 32 * Epi::kEpiWarps, Cfg::kSmem, s, maps, shape, epi);
  return cudaGetLastError();
}

}  // namespace ps
