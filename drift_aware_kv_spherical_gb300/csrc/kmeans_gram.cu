// a1, Gram form: the k-means passes between the first and the last
// assignment, run on the windows' cosine Gram matrices.
//
// [Polestar §2.A, local window & clustering] clusters a window with spherical
// k-means: mu_c = u_c / ||u_c|| with u_c the sum of the member rows' unit
// vectors x_j, and each row joins the centroid of largest cosine.  Since
//   cos(x_i, mu_c) = sum_{j in c} <x_i, x_j> / sqrt(sum_{j,l in c} <x_j, x_l>),
// a pass needs only the Gram matrix K = X X^T and the current labels: no
// centroid is formed and H is not read again.  For a window of N <= 1024 rows
// the whole of K fits in the shared memory of one thread-block cluster, so
// the passes run back to back inside one launch.
//
//   k_tc_gemm<GramClusterEpi>  K = X X^T on the tensor cores (bf16 H, fp32
//        accumulation, upper-triangle tiles, K split over a cluster), each
//        entry scaled by 1/(||h_i|| ||h_j||) and stored as a 24-bit fixed-point
//        integer q = rint(K * 2^20) in two planes (int16 high part, u8 low
//        byte), laid out so that CTA z of the iteration kernel finds the
//        columns of its rows as one contiguous slab.
//   k_km_gram  one cluster of Z (<= 16) CTAs per window; CTA z holds rows
//        [zR, zR + R) of K (its slab, loaded once) and runs every pass:
//        counting-sort the labels, S[i][c] = sum_{j in c} q_ij (exact integer
//        sums), n_c = sum_{i in c} S[i][c] (int64, summed over the cluster
//        through distributed shared memory), cos = S / sqrt(n_c), arg-max,
//        and the new labels pushed to every CTA of the cluster.
//
// Integer sums make every reduction exact, hence independent of order.  The
// fixed-point step (2^-20) bounds a cosine's error by about |c| 2^-21 /
// ||u_c||, a few 1e-7 for the clusters of these windows; ties between
// centroids closer than that may resolve differently from an fp64 Lloyd pass.
// A cluster left empty (or with a zero sum) keeps its centroid, so its column
// of cosines is carried over from the pass that last set it (kept in global
// memory, seeded by the first assignment pass against the given centroids).
#include <climits>
#include <mutex>

#include "ops.h"
#include "tc_gemm.cuh"
#include "vec.cuh"

namespace ps {
namespace {

constexpr int kGramThreads = 512;
constexpr int kGramMaxZ = 16;
constexpr float kGramScale = 1048576.f;  // 2^20 units per unit cosine

// q = 256 hi + lo, sign-extended from 24 bits, assembled by one byte permute:
// bytes (lo, hi.low, hi.high, sign of hi.high) of the pair {l, h}; sel picks
// row k of a four-row group (lo byte k of l, int16 k % 2 of h)
__device__ __forceinline__ int q24(uint32_t l, uint32_t h, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(l), "r"(h), "r"(sel));
  return static_cast<int>(r);
}

// q of rows 2l and 2l + 1 from their packed high parts (two int16) and low bytes
__device__ __forceinline__ int q_lo(uint32_t h, uint32_t l) {
  return static_cast<int>(static_cast<int16_t>(h & 0xffffu)) * 256 + static_cast<int>(l & 0xffu);
}
__device__ __forceinline__ int q_hi(uint32_t h, uint32_t l) {
  return static_cast<int>(static_cast<int16_t>(h >> 16)) * 256 + static_cast<int>((l >> 8) & 0xffu);
}

__device__ __forceinline__ int gram_quant(float k) {
  const int q = __float2int_rn(k * kGramScale);
  return min(max(q, -8388607), 8388607);
}

// Tile t of the Gram GEMM = (window b, u = t mod T): u < T0 is a Gram tile,
// row block mt <= column block nt, the upper triangle of the window's
// 128 x 128 blocks in row-major order; with pass 0 in the launch, u = T0 + mt
// is row block mt against the window's [2C][d] block of centroid hi and lo
// rows (B map 1), whose summed columns are the rows' cosines against the
// given centroids (nt = -1).
struct GramClusterEpi : TcEpiBase {
  static constexpr bool kClusterReduce = true;
  static constexpr uint32_t kLd = 128 + 4;
  int B, N, mtb, T, T0, R, Z, C;
  const float* inv;
  int16_t* qhi;
  uint8_t* qlo;
  float* cos0;  // [B][N][C] pass-0 cosines (centroid tiles)
  struct State {};
  __device__ void tile_of(int t, int& b, int& mt, int& nt) const {
    b = t / T;
    int u = t % T;
    if (u >= T0) {
      mt = u - T0;
      nt = -1;
      return;
    }
    mt = 0;
    while (u >= mtb - mt) {
      u -= mtb - mt;
      ++mt;
    }
    nt = mt + u;
  }
  __device__ int tiles(int) const { return B * T; }
  __device__ int arow(int t) const {
    int b, mt, nt;
    tile_of(t, b, mt, nt);
    return b * N + mt * 128;
  }
  __device__ int bsel(int t, int) const { return t % T >= T0 ? 1 : 0; }
  __device__ int bcoord(int t, int) const {
    int b, mt, nt;
    tile_of(t, b, mt, nt);
    return nt < 0 ? b * 2 * C : b * N + nt * 128;
  }
  __device__ void consume_red(int, int, int, int, uint32_t taddr, State&,
                              float* red_row) const {
    if (red_row == nullptr) return;
#pragma unroll 1
    for (int c0 = 0; c0 < 128; c0 += 32) {
      float v[32];
      tc::tmem_ld32(taddr + c0, v);
#pragma unroll
      for (int j = 0; j < 8; ++j)
        *reinterpret_cast<float4*>(red_row + c0 + 4 * j) =
            make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
    }
  }
  // element (row i, column j) sits at slab offset off(i) + j R, with
  // off(i) = ((b Z + i / R) N) R + i % R; eight consecutive rows from a
  // multiple of 8 (or eight consecutive columns) share one R-row block, since
  // R is a multiple of 16, so their high parts are one 16-byte store and
  // their low bytes one 8-byte store
  __device__ long long slab_off(int b, int i) const {
    return ((long long)b * Z + i / R) * N * R + i % R;
  }
  __device__ void put(long long off, int q) const {
    qhi[off] = static_cast<int16_t>(q >> 8);
    qlo[off] = static_cast<uint8_t>(q & 255);
  }
  __device__ void put8(long long off, const int* q) const {
    uint32_t h[4], l[2] = {0u, 0u};
#pragma unroll
    for (int e = 0; e < 4; ++e)
      h[e] = (static_cast<uint32_t>(q[2 * e] >> 8) & 0xffffu) |
             (static_cast<uint32_t>(q[2 * e + 1] >> 8) << 16);
#pragma unroll
    for (int e = 0; e < 8; ++e) l[e / 4] |= static_cast<uint32_t>(q[e] & 255) << (8 * (e & 3));
    *reinterpret_cast<uint4*>(qhi + off) = make_uint4(h[0], h[1], h[2], h[3]);
    *reinterpret_cast<uint2*>(qlo + off) = make_uint2(l[0], l[1]);
  }
  // scratch: 1/||h|| of the tile's 128 rows and 128 columns, then off() of both
  __device__ void prefetch(uint8_t* scratch, int i, int n) const {
    int b, mt, nt;
    tile_of(blockIdx.y, b, mt, nt);
    float* s_ir = reinterpret_cast<float*>(scratch);
    float* s_ic = s_ir + 128;
    long long* s_ro = reinterpret_cast<long long*>(s_ic + 128);
    long long* s_co = s_ro + 128;
    for (int k = i; k < 128; k += n) {
      const int r = mt * 128 + k, c = nt * 128 + k;
      s_ir[k] = r < N ? inv[(long)b * N + r] : 0.f;
      if (nt < 0) continue;
      s_ic[k] = c < N ? inv[(long)b * N + c] : 0.f;
      s_ro[k] = slab_off(b, r);
      s_co[k] = slab_off(b, c);
    }
  }
  __device__ void reduce(const float* red, int z, int nz, uint8_t* scratch) const {
    const int t = blockIdx.y;
    int b, mt, nt;
    tile_of(t, b, mt, nt);
    // rows [r0, r1) of the tile, cut at multiples of 8 (the 16-byte stores
    // below take eight rows from a multiple of 8); nz <= 8 leaves nr >= 8
    const int r0 = (z * 128 / nz) & ~7, r1 = z + 1 == nz ? 128 : ((z + 1) * 128 / nz) & ~7;
    const int nr = r1 - r0;
    const float* s_ir = reinterpret_cast<const float*>(scratch);  // staged by prefetch
    const float* s_ic = s_ir + 128;
    const long long* s_ro = reinterpret_cast<const long long*>(s_ic + 128);
    const long long* s_co = s_ro + 128;
    if (nt < 0) {  // centroid tile: cos = (<h, mu_hi> + <h, mu_lo>) / ||h||
      float* sums = const_cast<float*>(red);  // this CTA's rows, summed in place
      auto keep = [&](int r, int c, float4 v) {
        *reinterpret_cast<float4*>(sums + r * kLd + c) = v;
      };
      const int ncol = (2 * C + 3) & ~3;
      if (nz <= 4)
        cluster_rows_sum<4, 32>(red, kLd, r0, r1, ncol, nz, keep);
      else
        cluster_rows_sum<8, 32>(red, kLd, r0, r1, ncol, nz, keep);
      tc::cluster_arrive();
      __syncthreads();
      for (int it = threadIdx.x; it < nr * C; it += blockDim.x) {
        const int r = r0 + it / C, c = it % C, i = mt * 128 + r;
        if (i < N)
          cos0[((long)b * N + i) * C + c] = (sums[r * kLd + c] + sums[r * kLd + C + c]) * s_ir[r];
      }
      return;
    }
    // the quantised sums replace this CTA's own rows [r0, r1), which only it reads
    int* own = reinterpret_cast<int*>(const_cast<float*>(red));
    auto quant = [&](int r, int c, float4 v) {
      const float ir = s_ir[r];
      const int4 q = make_int4(gram_quant(v.x * ir * s_ic[c]), gram_quant(v.y * ir * s_ic[c + 1]),
                               gram_quant(v.z * ir * s_ic[c + 2]),
                               gram_quant(v.w * ir * s_ic[c + 3]));
      *reinterpret_cast<int4*>(own + r * kLd + c) = q;
    };
    if (nz <= 4)
      cluster_rows_sum<4, 32>(red, kLd, r0, r1, 128, nz, quant);
    else
      cluster_rows_sum<8, 32>(red, kLd, r0, r1, 128, nz, quant);
    tc::cluster_arrive();
    __syncthreads();
    // K(i, j): eight rows of one column per item
    const int nu = nr / 8;
    for (int it = threadIdx.x; it < 128 * nu; it += blockDim.x) {
      const int c = it / nu, rb = r0 + 8 * (it % nu);
      const int i0 = mt * 128 + rb, j = nt * 128 + c;
      if (j >= N || i0 >= N) continue;
      int q[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) q[e] = own[(rb + e) * kLd + c];
      if (i0 + 8 <= N) {
        put8(s_ro[rb] + (long long)j * R, q);
      } else {
        for (int e = 0; e < 8 && i0 + e < N; ++e) put(s_ro[rb + e] + (long long)j * R, q[e]);
      }
    }
    if (mt != nt) {  // K(j, i) = K(i, j) for the lower triangle: eight columns of one row
      for (int it = threadIdx.x; it < nr * 16; it += blockDim.x) {
        const int r = r0 + it / 16, cb = 8 * (it % 16);
        const int i = mt * 128 + r, j0 = nt * 128 + cb;
        if (i >= N || j0 >= N) continue;
        int q[8];
        const int4 qa = *reinterpret_cast<const int4*>(own + r * kLd + cb);
        const int4 qb = *reinterpret_cast<const int4*>(own + r * kLd + cb + 4);
        q[0] = qa.x; q[1] = qa.y; q[2] = qa.z; q[3] = qa.w;
        q[4] = qb.x; q[5] = qb.y; q[6] = qb.z; q[7] = qb.w;
        if (j0 + 8 <= N) {
          put8(s_co[cb] + (long long)i * R, q);
        } else {
          for (int e = 0; e < 8 && j0 + e < N; ++e) put(s_co[cb + e] + (long long)i * R, q[e]);
        }
      }
    }
  }
};

// Shared-memory layout of k_km_gram (16-byte aligned pieces).
struct GramSmem {
  uint32_t hi, lo, S, slot, npart, lab, prev, perm, chg, nchg, off, cur, hist, invn, keep,
      formed, newlab, best, objp, red, bar, abort, total;
};

__host__ __device__ inline uint32_t al16(uint32_t x) { return (x + 15u) & ~15u; }

__host__ __device__ inline GramSmem gram_smem(int N, int C, int R, int Z) {
  GramSmem o{};
  uint32_t p = 0;
  o.hi = p;     p = al16(p + (uint32_t)N * R * 2);
  o.lo = p;     p = al16(p + (uint32_t)N * R);
  o.S = p;      p = al16(p + (uint32_t)C * (R + 4) * 4);
  o.slot = p;   p = al16(p + (uint32_t)Z * C * 8);
  o.npart = p;  p = al16(p + (uint32_t)C * 8);
  o.lab = p;    p = al16(p + (uint32_t)Z * R);
  o.prev = p;   p = al16(p + (uint32_t)N);
  o.perm = p;   p = al16(p + (uint32_t)N * 2);
  o.chg = p;    p = al16(p + (uint32_t)N * 2);
  o.nchg = p;   p = al16(p + 4);
  o.off = p;    p = al16(p + (uint32_t)(C + 1) * 4);
  o.cur = p;    p = al16(p + (uint32_t)C * 4);
  o.hist = p;   p = al16(p + (uint32_t)C * 4);
  o.invn = p;   p = al16(p + (uint32_t)C * 4);
  o.keep = p;   p = al16(p + (uint32_t)C);
  o.formed = p; p = al16(p + (uint32_t)C);
  o.newlab = p; p = al16(p + (uint32_t)R);
  o.best = p;   p = al16(p + (uint32_t)R * 4);
  o.objp = p;   p = al16(p + (uint32_t)Z * 4);
  o.red = p;    p = al16(p + 32 * 4);
  o.bar = p;    p = al16(p + 8);
  o.abort = p;  p = al16(p + 4);
  o.total = p;
  return o;
}

// mu[b][c] = normalise(sum over rows j with lab[j] == c of h_j / ||h_j||),
// by every thread of the CTA: thread t owns columns 8t.. of each 4096-column
// block (d <= kGramMaxD), members in ascending row order.  Kept as is when
// the sum is zero.
constexpr int kGramMaxD = 4 * kGramThreads * 8;
__device__ void materialise(const __nv_bfloat16* __restrict__ H, int d,
                            const float* __restrict__ inv, float* __restrict__ mu, int b, int N,
                            int C, int c, const uint8_t* lab, float* s_red) {
  constexpr int kChunks = kGramMaxD / (kGramThreads * 8);
  float u[kChunks][8];
#pragma unroll
  for (int q = 0; q < kChunks; ++q)
#pragma unroll
    for (int e = 0; e < 8; ++e) u[q][e] = 0.f;
  for (int j = 0; j < N; ++j) {
    if (lab[j] != c) continue;
    const float sc = inv[(size_t)b * N + j];
    const __nv_bfloat16* h = H + ((size_t)b * N + j) * d;
#pragma unroll
    for (int q = 0; q < kChunks; ++q) {
      const int col = (q * kGramThreads + threadIdx.x) * 8;
      if (col < d) {
        const uint4 raw = *reinterpret_cast<const uint4*>(h + col);
        const __nv_bfloat162* p2 = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = __bfloat1622float2(p2[e]);
          u[q][2 * e] = fmaf(f.x, sc, u[q][2 * e]);
          u[q][2 * e + 1] = fmaf(f.y, sc, u[q][2 * e + 1]);
        }
      }
    }
  }
  float ss = 0.f;
#pragma unroll
  for (int q = 0; q < kChunks; ++q)
#pragma unroll
    for (int e = 0; e < 8; ++e) ss = fmaf(u[q][e], u[q][e], ss);
  ss = block_sum_f32(ss, s_red);
  const float nu = sqrtf(ss);
  if (!(nu > 0.f)) return;
  float* m = mu + ((size_t)b * C + c) * d;
#pragma unroll
  for (int q = 0; q < kChunks; ++q) {
    const int col = (q * kGramThreads + threadIdx.x) * 8;
    if (col < d) {
      reinterpret_cast<float4*>(m + col)[0] =
          make_float4(u[q][0] / nu, u[q][1] / nu, u[q][2] / nu, u[q][3] / nu);
      reinterpret_cast<float4*>(m + col)[1] =
          make_float4(u[q][4] / nu, u[q][5] / nu, u[q][6] / nu, u[q][7] / nu);
    }
  }
}

// One cluster of Z CTAs per window (blockIdx.y); CTA z = blockIdx.x owns rows
// [z R, z R + R).  Passes 1..passes; on entry assign holds the labels of pass
// 0 and L[b][i][c] the cosines against the given centroids; on exit assign
// holds the labels of the last pass, prev those of the pass before, rho the
// last pass's <h_i, mu_{a_i}>, obj[b][0..passes] the objectives (pass 0
// folded from the first assignment's partials objp0), and mu the centroids
// that stopped being formed at some pass (the others are formed afterwards
// from prev, by the last update).
__global__ void __launch_bounds__(kGramThreads, 1)
k_km_gram(const int16_t* __restrict__ qhi, const uint8_t* __restrict__ qlo, int N, int C,
          int R, int passes, const __nv_bfloat16* __restrict__ H, int d,
          const float* __restrict__ inv, float* __restrict__ mu, int32_t* __restrict__ assign,
          int32_t* __restrict__ prev, float* __restrict__ rho, float* __restrict__ L,
          const float* __restrict__ objp0, int ntile0, float* __restrict__ obj, int obj_ld,
          int pass0, int* status) {
  extern __shared__ __align__(16) uint8_t sm[];
  const int Z = gridDim.x, z = blockIdx.x, b = blockIdx.y;
  const GramSmem o = gram_smem(N, C, R, Z);
  const int16_t* s_hi = reinterpret_cast<const int16_t*>(sm + o.hi);
  const uint8_t* s_lo = sm + o.lo;
  int* s_S = reinterpret_cast<int*>(sm + o.S);
  long long* s_slot = reinterpret_cast<long long*>(sm + o.slot);
  long long* s_npart = reinterpret_cast<long long*>(sm + o.npart);
  uint8_t* s_lab = sm + o.lab;
  uint8_t* s_prev = sm + o.prev;
  uint16_t* s_perm = reinterpret_cast<uint16_t*>(sm + o.perm);
  uint16_t* s_chg = reinterpret_cast<uint16_t*>(sm + o.chg);
  int* s_nchg = reinterpret_cast<int*>(sm + o.nchg);
  int* s_off = reinterpret_cast<int*>(sm + o.off);
  int* s_cur = reinterpret_cast<int*>(sm + o.cur);
  int* s_hist = reinterpret_cast<int*>(sm + o.hist);
  float* s_invn = reinterpret_cast<float*>(sm + o.invn);
  uint8_t* s_keep = sm + o.keep;
  uint8_t* s_formed = sm + o.formed;
  uint8_t* s_newlab = sm + o.newlab;
  float* s_best = reinterpret_cast<float*>(sm + o.best);
  float* s_objp = reinterpret_cast<float*>(sm + o.objp);
  float* s_red = reinterpret_cast<float*>(sm + o.red);
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + o.bar);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + o.abort);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nwarps = kGramThreads / 32;
  const int row0 = z * R, nrow = min(R, N - row0);
  // S is [C][R + 4]: the arg-max's eight threads of four rows, and the
  // builds' lanes on consecutive rows, fall on distinct banks (R % 16 == 0)
  const int ldS = R + 4;

  const size_t slab = (size_t)N * R;
  if (tid == 0) {
    *abort_flag = 0;
    tc::mbar_init(bar, 1);
    tc::fence_mbar_init();
  }
  __syncthreads();
  tc::cluster_arrive();  // this CTA has started (awaited before the first remote access)
  if (tid == 0) {
    const uint8_t* gh = reinterpret_cast<const uint8_t*>(qhi + ((size_t)b * Z + z) * slab);
    const uint8_t* gl = qlo + ((size_t)b * Z + z) * slab;
    tc::mbar_expect_tx(bar, static_cast<uint32_t>(slab * 3));
    for (size_t k = 0; k < slab * 2; k += 32768)
      tc::bulk_load(sm + o.hi + k, gh + k, static_cast<uint32_t>(min((size_t)32768, slab * 2 - k)),
                    bar);
    for (size_t k = 0; k < slab; k += 32768)
      tc::bulk_load(sm + o.lo + k, gl + k, static_cast<uint32_t>(min((size_t)32768, slab - k)),
                    bar);
  }
  if (!pass0)
    for (int j = tid; j < N; j += kGramThreads)
      s_lab[j] = static_cast<uint8_t>(assign[(size_t)b * N + j]);
  for (int c = tid; c < C; c += kGramThreads) s_formed[c] = 0;  // pass 0 used the given centroids
  if (!pass0 && obj != nullptr && z == 0) {  // block-uniform: the objective of pass 0
    float so = 0.f;
    for (int t = tid; t < ntile0; t += kGramThreads) so += objp0[(size_t)b * ntile0 + t];
    so = block_sum_f32(so, s_red);
    if (tid == 0) obj[(size_t)b * obj_ld] = so;
  }
  // every thread observes the slab's arrival (a timeout leaves the status set
  // and the passes run on whatever landed; the copies are awaited before exit)
  tc::mbar_wait(bar, 0, status, abort_flag);
  tc::cluster_wait();  // every CTA of the cluster has started

  if (pass0) {
    // pass 0 from L, the cosines against the given centroids: arg-max of
    // this CTA's rows (8 threads per row), then labels and the objective's
    // partial to the cluster as after every pass
    const int r = tid >> 3, sub = tid & 7;
    float bv = -INFINITY;
    int bi = INT_MAX;
    if (r < nrow) {
      const float* Lrow = L + ((size_t)b * N + row0 + r) * C;
      for (int c = sub; c < C; c += 8) {
        const float v = Lrow[c];
        if (v > bv) {
          bv = v;
          bi = c;
        }
      }
    }
#pragma unroll
    for (int d2 = 1; d2 < 8; d2 <<= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, d2);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, d2);
      if (ov > bv || (ov == bv && oi < bi)) {
        bv = ov;
        bi = oi;
      }
    }
    if (sub == 0 && r < R) {
      if (bi == INT_MAX) {
        bi = 0;
        bv = 0.f;
      }
      s_newlab[r] = static_cast<uint8_t>(bi);
      s_best[r] = r < nrow ? bv : 0.f;
    }
    __syncthreads();
    if (obj != nullptr && warp == 0) {
      float so = 0.f;
      for (int q = lane; q < R; q += 32) so += s_best[q];
      so = warp_sum(so);
      if (lane == 0) tc::st_dsmem_f32(tc::cluster_map(tc::smem_u32(s_objp + z), 0), so);
    }
    const int words = R / 4;
    for (int k = tid; k < Z * words; k += kGramThreads) {
      const int q = k / words, w = k % words;
      const uint32_t v = *reinterpret_cast<const uint32_t*>(s_newlab + 4 * w);
      tc::st_dsmem_u32(tc::cluster_map(tc::smem_u32(s_lab + row0 + 4 * w), q), v);
    }
    tc::cluster_sync_all();
    if (obj != nullptr && z == 0 && tid == 0) {
      float so = 0.f;
      for (int q = 0; q < Z; ++q) so += s_objp[q];
      obj[(size_t)b * obj_ld] = so;
    }
  }

  float last_obj = 0.f;  // CTA 0, thread 0: the latest pass objective
  bool relabelled = true;  // the last pass took a new arg-max (cluster-uniform)
  for (int p = 1; p <= passes; ++p) {
    int M = 0;  // labels changed since S was formed (pass 1: all, from scratch)
    if (p == 1) {
      // counting sort of the labels: s_perm lists rows cluster by cluster
      for (int k = tid; k < C * ldS; k += kGramThreads) s_S[k] = 0;
      for (int c = tid; c < C; c += kGramThreads) s_hist[c] = 0;
      __syncthreads();
      for (int j = tid; j < N; j += kGramThreads) atomicAdd(&s_hist[s_lab[j]], 1);
      __syncthreads();
      if (warp == 0) {  // C <= 256: a lane scans 8 consecutive bins
        int v[8], sum = 0;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int c = lane * 8 + k;
          v[k] = c < C ? s_hist[c] : 0;
          sum += v[k];
        }
        int inc = sum;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
          const int x = __shfl_up_sync(0xffffffffu, inc, d);
          if (lane >= d) inc += x;
        }
        int run = inc - sum;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int c = lane * 8 + k;
          if (c < C) {
            s_off[c] = run;
            s_cur[c] = run;
          }
          run += v[k];
        }
        if (lane == 31) s_off[C] = inc;
      }
      __syncthreads();
      for (int j = tid; j < N; j += kGramThreads) {
        const int at = atomicAdd(&s_cur[s_lab[j]], 1);
        s_perm[at] = static_cast<uint16_t>(j);
        s_prev[j] = s_lab[j];
      }
      __syncthreads();

      // S[r][c] = sum over members j of c of q(row0 + r, j).  Warp w takes
      // positions [w N / 16, (w+1) N / 16) of the sorted list; lane l rows
      // 4 (l % 16) .. + 3, the two half-warps alternate positions, and a
      // segment's sums (halves combined) go to S with one atomic per row.
      const int p0 = warp * N / nwarps, p1 = (warp + 1) * N / nwarps;
      const int half = lane >> 4, r4 = 4 * (lane & 15);
      const bool act = r4 < R;
      int pp = p0;
      if (pp < p1) {
        int c = s_lab[s_perm[pp]];
        while (true) {
          const int e = min(s_off[c + 1], p1);
          int a[4] = {0, 0, 0, 0};
          if (act) {
            for (int q = pp + half; q < e; q += 2) {
              const int j = s_perm[q];
              const uint2 h = *reinterpret_cast<const uint2*>(s_hi + j * R + r4);
              const uint32_t l = *reinterpret_cast<const uint32_t*>(s_lo + j * R + r4);
              a[0] += q24(l, h.x, 0xD540u);
              a[1] += q24(l, h.x, 0xF761u);
              a[2] += q24(l, h.y, 0xD542u);
              a[3] += q24(l, h.y, 0xF763u);
            }
          }
          __syncwarp();
#pragma unroll
          for (int k = 0; k < 4; ++k) a[k] += __shfl_xor_sync(0xffffffffu, a[k], 16);
          if (act && half == 0) {
#pragma unroll
            for (int k = 0; k < 4; ++k) atomicAdd(&s_S[c * ldS + r4 + k], a[k]);
          }
          pp = e;
          if (pp >= p1) break;
          c = s_lab[s_perm[pp]];
        }
      }
      M = N;
    } else if (relabelled) {  // else no label can have changed since the last scan
      // rows whose label changed in the last pass move their column of q
      // from the old cluster's sums to the new one's (integer, so S stays
      // equal to the sums formed from scratch)
      if (tid == 0) *s_nchg = 0;
      __syncthreads();
      for (int j = tid; j < N; j += kGramThreads)
        if (s_lab[j] != s_prev[j]) s_chg[atomicAdd(s_nchg, 1)] = static_cast<uint16_t>(j);
      __syncthreads();
      M = *s_nchg;
      if (M > 0) {  // cluster-uniform: every CTA holds the same labels
        const int half = R / 2;
        for (int it = tid; it < M * half; it += kGramThreads) {
          const int k = it / half, r2 = 2 * (it % half);
          const int j = s_chg[k];
          const int co = s_prev[j], cn = s_lab[j];
          const uint32_t h = *reinterpret_cast<const uint32_t*>(s_hi + j * R + r2);
          const uint32_t l = *reinterpret_cast<const uint16_t*>(s_lo + j * R + r2);
          const int v0 = q_lo(h, l), v1 = q_hi(h, l);
          atomicAdd(&s_S[co * ldS + r2], -v0);
          atomicAdd(&s_S[cn * ldS + r2], v0);
          atomicAdd(&s_S[co * ldS + r2 + 1], -v1);
          atomicAdd(&s_S[cn * ldS + r2 + 1], v1);
        }
        for (int k = tid; k < M; k += kGramThreads) {
          const int j = s_chg[k];
          atomicSub(&s_hist[s_prev[j]], 1);
          atomicAdd(&s_hist[s_lab[j]], 1);
        }
        // s_prev keeps the labels of the pass before until the centroids
        // that stop being formed have been materialised below
      }
    }

    if (M > 0) {
      // ||u_c||^2 partial of this CTA's rows, pushed into slot z of every CTA
      for (int c = tid; c < C; c += kGramThreads) s_npart[c] = 0;
      __syncthreads();
      for (int r = tid; r < nrow; r += kGramThreads) {
        const int c = s_lab[row0 + r];
        atomicAdd(reinterpret_cast<unsigned long long*>(&s_npart[c]),
                  static_cast<unsigned long long>(static_cast<long long>(s_S[c * ldS + r])));
      }
      __syncthreads();
      const uint32_t base = tc::smem_u32(s_slot + (size_t)z * C);
      for (int k = tid; k < Z * C; k += kGramThreads) {
        const int q = k / C, c = k % C;
        tc::st_dsmem_u64(tc::cluster_map(base + 8u * c, q),
                         static_cast<unsigned long long>(s_npart[c]));
      }
      tc::cluster_sync_all();
      // 1 / ||u_c|| (2^-10 folds the fixed-point scale of S and of n_c)
      for (int c = tid; c < C; c += kGramThreads) {
        long long n = 0;
        for (int q = 0; q < Z; ++q) n += s_slot[q * C + c];
        const bool keep = s_hist[c] == 0 || n <= 0;
        s_keep[c] = keep ? 1 : 0;
        s_invn[c] = keep ? -1.f : 0.0009765625f / sqrtf(static_cast<float>(n));  // < 0: kept
      }
      __syncthreads();
      // a centroid formed in the last pass but kept from this one stays as
      // it was: normalise(sum of the unit rows labelled c in s_prev), formed
      // here from H (CTA c mod Z) so that the last update can keep it
      for (int c = z; c < C; c += Z) {
        if (!(s_keep[c] && s_formed[c])) continue;  // CTA-uniform
        materialise(H, d, inv, mu, b, N, C, c, s_prev, s_red);
      }
      __syncthreads();
      for (int c = tid; c < C; c += kGramThreads) s_formed[c] = s_keep[c] ? 0 : 1;
      if (p > 1)
        for (int k = tid; k < M; k += kGramThreads) s_prev[s_chg[k]] = s_lab[s_chg[k]];
      __syncthreads();
    }
    // (M == 0: S, the counts and the norms are those of the last pass, so
    // are the cosines, and the last pass's arg-max, labels and objective are
    // this pass's too: they are kept instead of recomputed)

    // cosines and arg-max (first maximum): 8 threads per row, thread `sub`
    // taking clusters sub, sub + 8, ...; a kept cluster's column comes from
    // L, the others refresh it
    if (M > 0) {
      const int r = tid >> 3, sub = tid & 7;
      float bv = -INFINITY;
      int bi = INT_MAX;
      if (r < R) {
        const bool valid = r < nrow;
        float* Lrow = L + ((size_t)b * N + (valid ? row0 + r : 0)) * C;
        for (int c0 = sub; c0 < C; c0 += 64) {  // eight clusters' loads, then their use
          int sv[8];
          float mv[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const int c = c0 + 8 * k;
            sv[k] = c < C ? s_S[c * ldS + r] : 0;
            mv[k] = c < C ? s_invn[c] : -1.f;
          }
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const int c = c0 + 8 * k;
            if (c >= C) break;
            float v;
            if (mv[k] >= 0.f) {
              v = static_cast<float>(sv[k]) * mv[k];
              if (valid && M > 0) Lrow[c] = v;
            } else {
              v = valid ? Lrow[c] : 0.f;
            }
            if (v > bv) {
              bv = v;
              bi = c;
            }
          }
        }
      }
#pragma unroll
      for (int d = 1; d < 8; d <<= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, d);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, d);
        if (ov > bv || (ov == bv && oi < bi)) {
          bv = ov;
          bi = oi;
        }
      }
      if (sub == 0 && r < R) {
        if (bi == INT_MAX) {
          bi = 0;
          bv = 0.f;
        }
        s_newlab[r] = static_cast<uint8_t>(bi);
        s_best[r] = r < nrow ? bv : 0.f;
      }
      __syncthreads();
    }

    relabelled = M > 0;
    if (M > 0) {
      // the pass objective's partial to CTA 0, the new labels to every CTA
      if (obj != nullptr && warp == 0) {
        float so = 0.f;
        for (int r = lane; r < R; r += 32) so += s_best[r];
        so = warp_sum(so);
        if (lane == 0) tc::st_dsmem_f32(tc::cluster_map(tc::smem_u32(s_objp + z), 0), so);
      }
      const int words = R / 4;
      for (int k = tid; k < Z * words; k += kGramThreads) {
        const int q = k / words, w = k % words;
        const uint32_t v = *reinterpret_cast<const uint32_t*>(s_newlab + 4 * w);
        tc::st_dsmem_u32(tc::cluster_map(tc::smem_u32(s_lab + row0 + 4 * w), q), v);
      }
      tc::cluster_sync_all();
      if (obj != nullptr && z == 0 && tid == 0) {
        float so = 0.f;
        for (int q = 0; q < Z; ++q) so += s_objp[q];
        last_obj = so;
      }
    }
    // (M == 0: the same inputs gave the same labels and objective)
    if (obj != nullptr && z == 0 && tid == 0) obj[(size_t)b * obj_ld + p] = last_obj;
  }
  for (int r = tid; r < nrow; r += kGramThreads) {
    const size_t i = (size_t)b * N + row0 + r;
    assign[i] = s_lab[row0 + r];
    prev[i] = s_prev[row0 + r];
    const float iv = inv[i];
    rho[i] = iv > 0.f ? s_best[r] / iv : 0.f;  // <h, mu> = ||h|| cos
  }
  if (tid == 0 && *abort_flag) {  // copies still in flight must land before the CTA leaves
    const uint64_t t0 = tc::globaltimer();
    while (!tc::mbar_try_wait(bar, 0) && tc::globaltimer() - t0 < tc::kWaitLimitNs) {
    }
  }
}

// Clusters of z CTAs of k_km_gram (smem bytes each) the GPU holds at once;
// 0 when the shape cannot launch.  Cached per device and shape.
int gram_capacity(int z, size_t smem) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  static std::mutex mu;
  static int c_dev = -1, c_z = 0;
  static size_t c_smem = 0;
  static int c_val = 0;
  std::lock_guard<std::mutex> lock(mu);
  if (dev == c_dev && z == c_z && smem == c_smem) return c_val;
  int n = 0;
  if (cudaFuncSetAttribute(k_km_gram, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) == cudaSuccess &&
      cudaFuncSetAttribute(k_km_gram, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) ==
          cudaSuccess) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(z, 1, 1);
    cfg.blockDim = dim3(kGramThreads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = z;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, k_km_gram, &cfg) != cudaSuccess) n = 0;
  }
  cudaGetLastError();
  c_dev = dev;
  c_z = z;
  c_smem = smem;
  c_val = n;
  return n;
}

// q of K's element (i, j), kh / kl pointing at row i's base in the slab
__device__ __forceinline__ int kq(const int16_t* kh, const uint8_t* kl, int j, int R) {
  const long long o = (long long)j * R;
  return static_cast<int>(kh[o]) * 256 + static_cast<int>(kl[o]);
}

// k-means++ seeding of a window from its Gram matrix, one CTA of 1024
// threads per window (thread i = row i, N <= 1024).  Round r picks centre r
// as the row-by-row seeding does (row floor(u_0 N) first; then the first row
// whose running weight sum, in row order, exceeds u_r times the total -- the
// count of rows at or below it, the sums being non-decreasing -- or the first
// row not yet chosen when no weight is left) and lowers every
// weight to min(w_i, max(0, 1 - cos(x_i, x_pick))), 0 for chosen rows, with
// the cosine q 2^-20 read from K's column pick (contiguous over the rows of
// a slab).  The weights are then exact multiples of 2^-20, so they are kept
// as integers 2^20 - q (capped at 2^21, |cos| <= 1) and summed exactly in 32
// bits (N 2^21 <= 2^31): the same picks as exact fp64 sums, without the
// fp64 scan.  At the end the seeds mu_r = h_pick / ||h_pick|| are written,
// and pass 0's cosines L[i][r] = K[i][pick_r], which are the rows' cosines
// against the seeds, so that no assignment pass is needed.
__global__ void __launch_bounds__(1024)
k_kpp_gram(const __nv_bfloat16* __restrict__ H, const float* __restrict__ inv_all,
           const double* __restrict__ U, const int16_t* __restrict__ qhi,
           const uint8_t* __restrict__ qlo, int N, int d, int C, int R, int Z,
           float* __restrict__ mu, float* __restrict__ L) {
  __shared__ uint32_t s_scan[32];
  __shared__ int s_min[32];
  __shared__ int s_pick[256];
  __shared__ double s_u[256];
  pdl_prologue();
  const int b = blockIdx.x, i = threadIdx.x;
  const bool live = i < N;
  for (int r = i; r < C; r += blockDim.x) s_u[r] = U[(long)b * C + r];
  __syncthreads();
  // element (i, j) of the window's K at base + j R (the slab layout)
  const long long base = live ? ((long long)b * Z + i / R) * N * R + i % R : 0;
  const int16_t* kh = qhi + base;
  const uint8_t* kl = qlo + base;
  uint32_t wgt = 0u;  // weight in units of 2^-20
  bool chosen = false;
  int pick = min(max((int)floor(s_u[0] * (double)N), 0), N - 1);
  for (int r = 0; r < C; ++r) {
    if (r > 0) {
      const uint32_t wv = live ? wgt : 0u;
      uint32_t total;
      const uint32_t run = block_exclusive_scan<uint32_t>(wv, s_scan, &total) + wv;
      // the running sums do not decrease, so the first row above the target
      // is the number of rows at or below it (N when none is above)
      const double target = s_u[r] * (double)total;
      pick = __syncthreads_count(live && (double)run <= target);
      if (total == 0u || pick >= N) {  // no weight left: first row not yet chosen
        pick = block_min_int(live && !chosen ? i : INT_MAX, s_min);
        if (pick == INT_MAX) pick = 0;
      }
    }
    if (i == pick) chosen = true;
    if (i == 0) s_pick[r] = pick;
    if (r + 1 < C && live) {
      const uint32_t cw =
          chosen ? 0u : static_cast<uint32_t>(min(max((1 << 20) - kq(kh, kl, pick, R), 0), 1 << 21));
      wgt = r == 0 ? cw : min(wgt, cw);
    }
  }
  __syncthreads();
  const __nv_bfloat16* Hb = H + (long)b * N * d;
  const float* inv = inv_all + (long)b * N;
  for (long e = i; e < (long)C * d; e += blockDim.x) {
    const int r = (int)(e / d), k = (int)(e % d), p = s_pick[r];
    mu[((long)b * C + r) * d + k] = to_f32(Hb[(long)p * d + k]) * inv[p];
  }
  if (live) {
    float* Li = L + ((long)b * N + i) * C;
    for (int r = 0; r < C; ++r)
      Li[r] = static_cast<float>(kq(kh, kl, s_pick[r], R)) * (1.f / kGramScale);
  }
}

}  // namespace

GramPlan gram_plan(int dtype, int B, int N, int d, int C) {
  GramPlan g{};
  if (dtype != PS_BF16 || B < 1 || N < 2 || N > 1024 || C < 1 || C > 256 || d < 64 ||
      d > kGramMaxD || d % 8 != 0)
    return g;
  g.R = ceil_div(ceil_div(N, kGramMaxZ), 16) * 16;
  g.Z = ceil_div(N, g.R);
  g.smem = gram_smem(N, C, g.R, g.Z).total;
  if (g.smem > 227 * 1024) return g;
  g.mtb = ceil_div(N, 128);
  g.T0 = g.mtb * (g.mtb + 1) / 2;
  g.fused0 = 2 * C <= 128;  // the centroids' hi and lo rows fit one 128-row B tile
  g.T = g.T0 + (g.fused0 ? g.mtb : 0);
  g.KB = ceil_div(d, 64);
  const int tiles = B * g.T;
  g.nz = 1;
  for (int z = 8; z >= 2; --z)
    if (z <= g.KB && (long)tiles * z <= kSmTarget && tiles <= tc_cluster_capacity(z)) {
      g.nz = z;
      break;
    }
  g.kpc = ceil_div(g.KB, g.nz);
  g.nz = ceil_div(g.KB, g.kpc);
  g.ok = true;
  return g;
}

bool gram_launchable(const GramPlan& g) {
  return g.ok && gram_capacity(g.Z, g.smem) >= 1;
}

cudaError_t gram_build(const GramPlan& g, const __nv_bfloat16* H, const float* inv, int B,
                       int N, int d, int C, const __nv_bfloat16* mu_split, float* cos0,
                       int16_t* qhi, uint8_t* qlo, int* status, cudaStream_t s) {
  TcMaps maps;
  if (!make_tmap_bf16_2d(&maps.a[0], H, d, (uint64_t)B * N, (uint64_t)d * 2, 64, 128))
    return cudaErrorInvalidValue;
  maps.a[1] = maps.a[0];
  maps.b[0] = maps.a[0];
  maps.b[1] = maps.a[0];
  if (mu_split != nullptr &&
      !make_tmap_bf16_2d(&maps.b[1], mu_split, d, (uint64_t)B * 2 * C, (uint64_t)d * 2, 64, 128))
    return cudaErrorInvalidValue;
  const int T = mu_split != nullptr ? g.T : g.T0;
  TcShape sh{B * N, nullptr, g.KB, g.kpc, status, INT_MAX};
  GramClusterEpi epi{{}, B, N, g.mtb, T, g.T0, g.R, g.Z, C, inv, qhi, qlo, cos0};
  return launch_tc_gemm<128, 1, 1, false>(maps, sh, epi, dim3(1, B * T, g.nz), s);
}

cudaError_t gram_iterate(const GramPlan& g, const int16_t* qhi, const uint8_t* qlo, int B, int N,
                         int C, int passes, const __nv_bfloat16* H, int d, const float* inv,
                         float* mu, int32_t* assign, int32_t* prev, float* rho, float* L,
                         const float* objp0, int ntile0, float* obj, int obj_ld, int* status,
                         cudaStream_t s) {
  if (gram_capacity(g.Z, g.smem) < 1) return cudaErrorInvalidConfiguration;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(g.Z, B, 1);
  cfg.blockDim = dim3(kGramThreads);
  cfg.dynamicSmemBytes = g.smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = g.Z;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return launch_ex(cfg, k_km_gram, qhi, qlo, N, C, g.R, passes, H, d, inv, mu, assign, prev, rho,
                   L, objp0, ntile0, obj, obj_ld, objp0 == nullptr ? 1 : 0, status);
}

cudaError_t gram_seed(const GramPlan& g, const __nv_bfloat16* H, const float* inv,
                      const double* U, int B, int N, int d, int C, const int16_t* qhi,
                      const uint8_t* qlo, float* mu, float* L, cudaStream_t s) {
  if (N > 1024 || C > 256) return cudaErrorInvalidValue;
  launch_pdl(k_kpp_gram, dim3(B), 1024, 0, s, H, inv, U, qhi, qlo, N, d, C, g.R, g.Z, mu, L);
  return cudaGetLastError();
}

}  // namespace ps
