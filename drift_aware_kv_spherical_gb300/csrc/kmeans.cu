// a1: spherical k-means of each window's hidden states.
//
// [Polestar §2.A, local window & clustering]: the window's hidden states are
// clustered with spherical k-means.  Per pass: assign every row to the
// centroid of largest cosine (first maximum), then renormalise each cluster's
// sum of unit rows.  Deterministic: every reduction runs in a fixed order.
//
// Kernels (one launch each, all on the caller's stream):
//   k_km_prep       1/||h_i|| (one warp per row) and the bf16 split of mu
//                   for the tensor cores, one launch
//   k_kpp_pick      k-means++ centre r, one CTA per window   (init_mode 1)
//   k_kpp_weights   weights against centre r, warp per row   (C - 1 rounds)
//                   (the Gram form seeds from K instead: k_kpp_gram, one
//                   launch for all rounds; see kmeans_gram.cu)
//   assignment      bf16 windows: tcgen05 tiles of 128 rows x C centroids,
//                   <h, mu_hi> + <h, mu_lo> accumulated in TMEM, split over
//                   d when the windows give too few row tiles.  The d-chunks
//                   of a tile form a thread-block cluster (C <= 128) and sum
//                   their scores in chunk order through distributed shared
//                   memory, a warp per row taking the arg-max; for C > 128
//                   the chunks go through global memory to k_km_argmax.
//                   fp32 windows: k_assign on CUDA cores.
//   k_cluster_scan  per (cluster, window, column slice), the slices of one
//                   cluster forming a thread-block cluster: members in
//                   ascending row order, centroid = normalise(sum of unit
//                   rows) (+ bf16 split), or on the last pass C_hat =
//                   mean(rho) * mu; counts; objective
//
// Large batches (one d-chunk per tile) take the passes in a faster form with
// the same results:
//   * bf16 centroids only.  A pass scores every row against bf16(mu) alone
//     (one MMA instead of the hi + lo pair).  Rounding a centroid to bf16
//     moves every cosine by at most e = max_c ||mu_c - bf16(mu_c)|| (Cauchy-
//     Schwarz), so a row whose best score leads the runner-up by more than
//     ||h|| (2 e + 2^-13) -- the last term for the tensor cores' fp32
//     accumulation over d -- has the same arg-max as exact arithmetic.  Rows
//     within that band are listed with every centroid inside it, and
//     k_km_recheck decides them with fp32 dot products against the fp32
//     centroids.
//   * Early exit.  Once a pass t >= 1 leaves every label of a window as the
//     pass before did, the next update gives back the same centroids bit for
//     bit (the update is a fixed function of H and the labels) and so every
//     later pass the same labels and cosines: those passes and updates are
//     skipped for that window (the CTAs see the window's flags and take no
//     tile), and their objectives repeat the last one computed.  The outputs
//     equal those of computing every pass.
//   * rho exact.  k_km_rho takes rho_i = <h_i, mu_{a_i}> in fp32 after the
//     last pass (the passes' best scores use bf16(mu)).
//   * The last step (C_hat, counts, the last objective) from per-slice
//     cluster statistics (k_km_fin_stats, k_km_fin_chat), no member lists.
#include <algorithm>
#include <climits>
#include <type_traits>

#include "ops.h"
#include "tc_gemm.cuh"
#include "vec.cuh"

namespace ps {
namespace {

constexpr int kTileRows = 64;    // rows per assignment tile
constexpr int kTileC = 128;      // centroids per chunk of an assignment tile
constexpr int kTileK = 32;       // d per shared-memory stage

// Early exit of the passes: changed[b * kMaxPasses + t] = 1 once pass t >= 1
// gave some row of window b another label than pass t - 1.  Pass t of window
// b runs while every pass 1 .. t - 1 changed a label; the update after pass
// t runs while every pass 1 .. t did.  A pass raises its flag only if it ran,
// and it ran only if every pass before it changed a label, so "every pass
// 1 .. t - 1 changed" is the one flag of pass t - 1 (t >= 2).
constexpr int kMaxPasses = 64;
__device__ __forceinline__ bool km_pass_active(const int32_t* changed, int b, int t) {
  return t <= 1 || __ldcg(changed + (long)b * kMaxPasses + t - 1) != 0;
}

// Allowance for the tensor cores' fp32 accumulation of a bf16 score over d
// (relative to ||h||), on top of the centroids' bf16 rounding.
constexpr float kAccAllowance = 1.0f / 8192.0f;

// A row whose bf16-centroid arg-max is not certain: its candidates (every
// centroid whose score lies within the band of the best), in ascending
// order, or n = -1 when there are more than kRcMax of them (then all C).
constexpr int kRcMax = 10;
struct RcEntry {
  int32_t row, n, c[kRcMax];
};


// k-means++ on the sphere, one round r at a time: k_kpp_pick chooses centre
// r (one CTA per window), then k_kpp_weights lowers every row's weight to
// w_i = min(w_i, max(0, 1 - cos(h_i, centre r))) (0 for chosen rows) over the
// whole grid.  Centre 0 is row floor(u_0 N); centre r >= 1 is the first row
// whose running sum of w (fp64, row order) exceeds u_r * sum(w), or the first
// row not yet chosen when every weight is 0.
template <typename T>
__global__ void __launch_bounds__(1024)
k_kpp_pick(const T* __restrict__ H, const float* __restrict__ inv_all,
           const double* __restrict__ U, int N, int d, int C, int r, float* __restrict__ mu,
           const float* __restrict__ w_all, int8_t* __restrict__ chosen_all) {
  __shared__ double s_scan[32];
  __shared__ int s_min[32];
  const int b = blockIdx.x, tid = threadIdx.x;
  const T* Hb = H + (long)b * N * d;
  const float* inv = inv_all + (long)b * N;
  const float* w = w_all + (long)b * N;
  int8_t* chosen = chosen_all + (long)b * N;
  const double* u = U + (long)b * C;
  if (r == 0) {
    for (int i = tid; i < N; i += blockDim.x) chosen[i] = 0;
    __syncthreads();
  }
  int pick;
  if (r == 0) {
    pick = min(max((int)floor(u[0] * (double)N), 0), N - 1);
  } else {
    const int chunk = (N + blockDim.x - 1) / blockDim.x;
    const int lo = tid * chunk, hi = min(N, lo + chunk);
    double sum = 0.0;
    for (int i = lo; i < hi; ++i) sum += (double)w[i];
    double total;
    const double base = block_exclusive_scan<double>(sum, s_scan, &total);
    int cand = INT_MAX;
    if (total > 0.0) {
      const double target = u[r] * total;
      double run = base;
      for (int i = lo; i < hi; ++i) {
        run += (double)w[i];
        if (run > target) { cand = i; break; }
      }
    }
    pick = block_min_int(cand, s_min);
    if (pick == INT_MAX) {  // no weight left: first row not yet chosen
      cand = INT_MAX;
      for (int i = tid; i < N; i += blockDim.x)
        if (!chosen[i]) { cand = i; break; }
      pick = block_min_int(cand, s_min);
      if (pick == INT_MAX) pick = 0;
    }
  }
  __syncthreads();
  if (tid == 0) chosen[pick] = 1;
  const float ip = inv[pick];
  float* mur = mu + ((long)b * C + r) * d;
  for (int k = tid; k < d; k += blockDim.x) mur[k] = to_f32(Hb[(long)pick * d + k]) * ip;
}

// One warp per row: cosine with centre r, weight update.
template <typename T>
__global__ void __launch_bounds__(256)
k_kpp_weights(const T* __restrict__ H, const float* __restrict__ inv, int B, int N, int d,
              int C, int r, const float* __restrict__ mu, float* __restrict__ w,
              const int8_t* __restrict__ chosen) {
  constexpr int V = Vec<T>::n;
  const long row = ((long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (row >= (long)B * N) return;
  const int b = (int)(row / N);
  const T* h = H + row * d;
  const float* m = mu + ((long)b * C + r) * d;
  float dot = 0.f;
  for (int k = lane * V; k < d; k += 32 * V) {
    float hv[V], mv[V];
    load16(h + k, hv);
#pragma unroll
    for (int q = 0; q < V / 4; ++q) load16(m + k + 4 * q, mv + 4 * q);
#pragma unroll
    for (int e = 0; e < V; ++e) dot = fmaf(hv[e], mv[e], dot);
  }
  dot = warp_sum(dot);
  if (lane == 0) {
    const float cw = chosen[row] ? 0.f : fmaxf(0.f, 1.f - dot * inv[row]);
    w[row] = (r == 0) ? cw : fminf(w[row], cw);
  }
}

// One pass of assignments.  CTA = 64 rows of one window; 8 warps x 8 rows;
// lane owns centroids c0 + 4*lane .. +3 of each 128-centroid chunk.
template <typename T>
__global__ void __launch_bounds__(256)
k_assign(const T* __restrict__ H, const float* __restrict__ mu,
         const float* __restrict__ inv, int N, int d, int C,
         int32_t* __restrict__ assign, float* __restrict__ best_dot,
         float* __restrict__ objp) {
  pdl_prologue();
  __shared__ __align__(16) float Hs[kTileK][kTileRows];
  __shared__ __align__(16) float Ms[kTileK][kTileC];
  __shared__ float s_red[8];
  const int b = blockIdx.y, tile = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int row0 = tile * kTileRows;
  const T* Hb = H + (long)b * N * d;
  const float* mub = mu + (long)b * C * d;

  float rv[8];
  int ri[8];
#pragma unroll
  for (int r = 0; r < 8; ++r) { rv[r] = -INFINITY; ri[r] = INT_MAX; }

  for (int c0 = 0; c0 < C; c0 += kTileC) {
    float acc[8][4];
#pragma unroll
    for (int r = 0; r < 8; ++r)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[r][j] = 0.f;

    for (int k0 = 0; k0 < d; k0 += kTileK) {
      {  // H stage: thread -> row tid/4, 8 consecutive k
        const int r = tid >> 2, kq = (tid & 3) * 8;
        const int row = row0 + r;
        float v[8];
        if (row < N && k0 + kq < d) {
          const T* p = Hb + (long)row * d + k0 + kq;
          if constexpr (Vec<T>::n == 8) {
            load16(p, v);
          } else {
            load16(p, v);
            load16(p + 4, v + 4);
          }
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e) v[e] = 0.f;
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) Hs[kq + e][r] = v[e];
      }
      {  // centroid stage: thread -> centroid tid/2, 16 consecutive k
        const int cl = tid >> 1, kq = (tid & 1) * 16;
        const int c = c0 + cl;
        float v[16];
        if (c < C && k0 + kq < d) {
          const float* p = mub + (long)c * d + k0 + kq;
#pragma unroll
          for (int q = 0; q < 4; ++q) load16(p + 4 * q, v + 4 * q);
        } else {
#pragma unroll
          for (int e = 0; e < 16; ++e) v[e] = 0.f;
        }
#pragma unroll
        for (int e = 0; e < 16; ++e) Ms[kq + e][cl] = v[e];
      }
      __syncthreads();
#pragma unroll 8
      for (int kk = 0; kk < kTileK; ++kk) {
        const float4 h0 = *reinterpret_cast<const float4*>(&Hs[kk][warp * 8]);
        const float4 h1 = *reinterpret_cast<const float4*>(&Hs[kk][warp * 8 + 4]);
        const float4 m = *reinterpret_cast<const float4*>(&Ms[kk][lane * 4]);
        const float hv[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
        const float mv[4] = {m.x, m.y, m.z, m.w};
#pragma unroll
        for (int r = 0; r < 8; ++r)
#pragma unroll
          for (int j = 0; j < 4; ++j) acc[r][j] = fmaf(hv[r], mv[j], acc[r][j]);
      }
      __syncthreads();
    }
    // arg-max of this chunk per row, first maximum on ties
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      float bv = -INFINITY;
      int bi = INT_MAX;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int c = c0 + lane * 4 + j;
        if (c < C && (acc[r][j] > bv || (acc[r][j] == bv && c < bi))) {
          bv = acc[r][j];
          bi = c;
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
      }
      if (bv > rv[r] || (bv == rv[r] && bi < ri[r])) { rv[r] = bv; ri[r] = bi; }
    }
  }
  float cs = 0.f;
  if (lane < 8) {
    float v = rv[0];
    int i = ri[0];
#pragma unroll
    for (int r = 1; r < 8; ++r)
      if (lane == r) { v = rv[r]; i = ri[r]; }
    const int row = row0 + warp * 8 + lane;
    if (row < N) {
      if (i == INT_MAX) { i = 0; v = 0.f; }
      assign[(long)b * N + row] = i;
      best_dot[(long)b * N + row] = v;
      cs = v * inv[(long)b * N + row];
    }
  }
  cs = warp_sum(cs);
  if (lane == 0) s_red[warp] = cs;
  __syncthreads();
  if (tid == 0) {
    float s = 0.f;
    for (int w = 0; w < 8; ++w) s += s_red[w];
    objp[(long)b * gridDim.x + tile] = s;
  }
}

// Set-up of a call, in one launch: blocks [0, inv_blocks) take 1/||h_i||
// for 8 rows each (a warp per row, its 16-byte loads unrolled four deep);
// the rest split mu (fp32) into bf16 hi + lo parts (hi = bf16(mu), lo =
// bf16(mu - hi)), four values per thread (a warp per centroid row when emax
// is wanted), into two [B][C][d] arrays or (cd = C d > 0) one [B][2C][d]
// array at hi.  Either part may be empty.  emax (nullable, [B], zeroed by the
// caller): raised to ||mu_c - hi_c|| of every centroid of window b (fp32 bits
// compared as integers, which orders non-negative floats, so the result does
// not depend on the order of the updates).
template <typename T>
__global__ void __launch_bounds__(256)
k_km_prep(const T* __restrict__ H, long rows, int d, float* __restrict__ inv, int inv_blocks,
          const float* __restrict__ mu, long n_mu, __nv_bfloat16* __restrict__ hi,
          __nv_bfloat16* __restrict__ lo, long cd, int C, float* __restrict__ emax) {
  pdl_prologue();
  const int lane = threadIdx.x & 31;
  if ((int)blockIdx.x < inv_blocks) {
    constexpr int V = Vec<T>::n;
    const long row = ((long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (row >= rows) return;
    const T* h = H + row * d;
    float ss = 0.f;
#pragma unroll 4
    for (int k = lane * V; k < d; k += 32 * V) {
      float v[V];
      load16(h + k, v);
#pragma unroll
      for (int e = 0; e < V; ++e) ss = fmaf(v[e], v[e], ss);
    }
    ss = warp_sum(ss);
    if (lane == 0) inv[row] = ss > 0.f ? 1.0f / sqrtf(ss) : 0.f;
    return;
  }
  if (emax == nullptr) {  // no bound wanted: element-wise, four values a thread
    const long n4 = n_mu >> 2;  // n_mu = B * C * d, a multiple of 16
    const long stride = (long)(gridDim.x - inv_blocks) * blockDim.x;
    for (long i = (long)(blockIdx.x - inv_blocks) * blockDim.x + threadIdx.x; i < n4;
         i += stride) {
      const long e = 4 * i;
      const long eh = cd > 0 ? (e / cd) * 2 * cd + e % cd : e;
      const long el = cd > 0 ? eh + cd : e;
      const float4 x = reinterpret_cast<const float4*>(mu)[i];
      const __nv_bfloat162 h0 = __floats2bfloat162_rn(x.x, x.y);
      const __nv_bfloat162 h1 = __floats2bfloat162_rn(x.z, x.w);
      const float2 f0 = __bfloat1622float2(h0), f1 = __bfloat1622float2(h1);
      const __nv_bfloat162 l0 = __floats2bfloat162_rn(x.x - f0.x, x.y - f0.y);
      const __nv_bfloat162 l1 = __floats2bfloat162_rn(x.z - f1.x, x.w - f1.y);
      *reinterpret_cast<uint2*>(hi + eh) = make_uint2(*reinterpret_cast<const uint32_t*>(&h0),
                                                      *reinterpret_cast<const uint32_t*>(&h1));
      *reinterpret_cast<uint2*>(lo + el) = make_uint2(*reinterpret_cast<const uint32_t*>(&l0),
                                                      *reinterpret_cast<const uint32_t*>(&l1));
    }
    return;
  }
  const long nrow = n_mu / d;  // n_mu = B * C * d, d a multiple of 16
  const long nwarps = ((long)(gridDim.x - inv_blocks) * blockDim.x) >> 5;
  for (long r = ((long)(blockIdx.x - inv_blocks) * blockDim.x + threadIdx.x) >> 5; r < nrow;
       r += nwarps) {
    float e2 = 0.f;
    for (int k = lane * 4; k < d; k += 128) {
      // cd > 0: one [2C][d] block per window, the C hi rows then the C lo rows
      const long e = r * d + k;
      const long eh = cd > 0 ? (e / cd) * 2 * cd + e % cd : e;
      const long el = cd > 0 ? eh + cd : e;
      const float4 x = *reinterpret_cast<const float4*>(mu + e);
      const __nv_bfloat162 h0 = __floats2bfloat162_rn(x.x, x.y);
      const __nv_bfloat162 h1 = __floats2bfloat162_rn(x.z, x.w);
      const float2 f0 = __bfloat1622float2(h0), f1 = __bfloat1622float2(h1);
      const __nv_bfloat162 l0 = __floats2bfloat162_rn(x.x - f0.x, x.y - f0.y);
      const __nv_bfloat162 l1 = __floats2bfloat162_rn(x.z - f1.x, x.w - f1.y);
      *reinterpret_cast<uint2*>(hi + eh) = make_uint2(*reinterpret_cast<const uint32_t*>(&h0),
                                                      *reinterpret_cast<const uint32_t*>(&h1));
      if (lo != nullptr)  // the faster passes use the hi part only
        *reinterpret_cast<uint2*>(lo + el) = make_uint2(*reinterpret_cast<const uint32_t*>(&l0),
                                                        *reinterpret_cast<const uint32_t*>(&l1));
      e2 = fmaf(x.x - f0.x, x.x - f0.x, e2);
      e2 = fmaf(x.y - f0.y, x.y - f0.y, e2);
      e2 = fmaf(x.z - f1.x, x.z - f1.x, e2);
      e2 = fmaf(x.w - f1.y, x.w - f1.y, e2);
    }
    if (emax != nullptr) {
      e2 = warp_sum(e2);
      if (lane == 0) atomicMax(reinterpret_cast<int*>(emax) + r / C, __float_as_int(sqrtf(e2)));
    }
  }
}

// Epilogue of the tensor-core assignment.  Tile t = (window b, 128-row block
// mt).  With one d-chunk the arg-max is taken straight from the accumulator
// and the tile's objective partial is folded here; with several, every chunk
// stores its partial scores [z][row][c] and k_km_argmax finishes the rows.
template <int BN>
struct KmAssignEpi : TcEpiBase {
  int B, N, C, mtb, nz;
  float* part;
  const float* inv;
  int32_t* assign;
  float* best;
  float* objp;
  float* scores;  // nullable: [B][N][C] cosines of the pass
  struct State {
    float bv;
    int bi;
  };
  __device__ int tiles(int) const { return B * mtb; }
  __device__ int arow(int t) const { return (t / mtb) * N + (t % mtb) * 128; }
  __device__ int bcoord(int t, int n0) const { return (t / mtb) * C + n0; }
  __device__ void consume(int t, int r, int, int z, uint32_t taddr, State& st) const {
    const int b = t / mtb, i = (t % mtb) * 128 + r;
    st.bv = -INFINITY;
    st.bi = INT_MAX;
    float* dst = part + ((long)z * B * N + (long)b * N + i) * C;
    const bool keep = nz == 1 && scores != nullptr && i < N;
    const float iv = keep ? inv[(long)b * N + i] : 0.f;
#pragma unroll 1
    for (int c0 = 0; c0 < BN; c0 += 32) {
      float v[32];
      tc::tmem_ld32(taddr + c0, v);
      if (nz == 1) {
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (c0 + j < C && v[j] > st.bv) { st.bv = v[j]; st.bi = c0 + j; }
        if (keep) {
          float* so = scores + ((long)b * N + i) * C;
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (c0 + j < C) so[c0 + j] = v[j] * iv;
        }
      } else if (i < N) {
        if (c0 + 32 <= C && (C & 3) == 0) {
#pragma unroll
          for (int j = 0; j < 8; ++j)
            *reinterpret_cast<float4*>(dst + c0 + 4 * j) =
                make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (c0 + j < C) dst[c0 + j] = v[j];
        }
      }
    }
  }
  __device__ void tile_done(int t, int r, int, int, uint8_t* scratch, State& st) const {
    if (nz > 1) return;
    const int b = t / mtb, i = (t % mtb) * 128 + r;
    float* wsum = reinterpret_cast<float*>(scratch + 16);
    float cs = 0.f;
    if (i < N) {
      if (st.bi == INT_MAX) { st.bi = 0; st.bv = 0.f; }
      assign[(long)b * N + i] = st.bi;
      best[(long)b * N + i] = st.bv;
      cs = st.bv * inv[(long)b * N + i];
    }
    cs = warp_sum(cs);
    if ((r & 31) == 0) wsum[r >> 5] = cs;
    epi_bar_sync();
    if (r == 0) objp[t] = ((wsum[0] + wsum[1]) + wsum[2]) + wsum[3];
    epi_bar_sync();
  }
};

// Epilogue of the faster passes (one d-chunk per tile, scores against
// bf16(mu) only; see the file comment).  Per row: the best score (first
// maximum) and the runner-up.  A row whose lead exceeds the band
// ||h|| (2 e_b + kAccAllowance) gets its label and best score here, and
// raises the window's `changed` flag of this pass when the label moved;
// any other row is listed for k_km_recheck with the centroids inside the
// band.  Tiles of windows whose passes have settled are skipped.
template <int BN>
struct KmFastEpi : TcEpiBase {
  int B, N, C, mtb, pass;
  const float* inv;
  const float* emax;   // [B] max_c ||mu_c - bf16(mu_c)||
  int32_t* assign;
  float* best;
  int32_t* changed;    // [B][kMaxPasses]
  int* rc_count;       // entries listed in this pass
  RcEntry* rc_list;    // [B * N]
  struct State {};
  __device__ int tiles(int) const { return B * mtb; }
  __device__ int arow(int t) const { return (t / mtb) * N + (t % mtb) * 128; }
  __device__ int bcoord(int t, int n0) const { return (t / mtb) * C + n0; }
  __device__ bool active(int t) const { return km_pass_active(changed, t / mtb, pass); }
  __device__ void consume(int t, int r, int, int, uint32_t taddr, State&) const {
    const int b = t / mtb, i = (t % mtb) * 128 + r;
    const bool valid = i < N;
    const long row = (long)b * N + i;
    float bv = -INFINITY, sv = -INFINITY;
    int bi = INT_MAX;
#pragma unroll 1
    for (int c0 = 0; c0 < BN; c0 += 32) {
      float v[32];
      tc::tmem_ld32(taddr + c0, v);  // warp-collective
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        if (c0 + j < C) {
          if (v[j] > bv) {
            sv = bv;
            bv = v[j];
            bi = c0 + j;
          } else if (v[j] > sv) {
            sv = v[j];
          }
        }
      }
    }
    float band = 0.f;
    bool certain = true;
    if (valid) {
      const float iv = inv[row];
      band = (iv > 0.f ? 1.0f / iv : 0.f) * (2.0f * emax[b] + kAccAllowance);
      certain = bi == INT_MAX || !(bv - sv <= band);  // ties and near-ties are rechecked
    }
    const bool listed = valid && !certain;
    if (__any_sync(0xffffffffu, listed)) {
      RcEntry en;
      en.row = (int32_t)row;
      en.n = 0;
#pragma unroll 1
      for (int c0 = 0; c0 < BN; c0 += 32) {
        float v[32];
        tc::tmem_ld32(taddr + c0, v);
        if (listed) {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            if (c0 + j < C && v[j] >= bv - band) {
              if (en.n < kRcMax) en.c[en.n] = c0 + j;
              ++en.n;
            }
          }
        }
      }
      if (listed) {
        if (en.n > kRcMax) en.n = -1;
        rc_list[atomicAdd(rc_count, 1)] = en;
      }
    }
    if (valid && certain) {
      if (bi == INT_MAX) { bi = 0; bv = 0.f; }
      if (pass >= 1 && assign[row] != bi) changed[(long)b * kMaxPasses + pass] = 1;
      assign[row] = bi;
      best[row] = bv;
    }
  }
  __device__ void tile_done(int, int, int, int, uint8_t*, State&) const {}
};

// The listed rows of a pass, a warp per row: fp32 dot products of h_i with
// the fp32 centroids of its candidates (lanes over d, summed in a fixed
// order), the first maximum in ascending centroid order; label, best score
// and the window's `changed` flag as in the epilogue.  Runs on a fixed grid
// and reads the number of rows from the device.
__global__ void __launch_bounds__(256)
k_km_recheck(const __nv_bfloat16* __restrict__ H, const float* __restrict__ mu, int N, int d,
             int C, int pass, const int* __restrict__ count, const RcEntry* __restrict__ list,
             int32_t* __restrict__ assign, float* __restrict__ best,
             int32_t* __restrict__ changed) {
  pdl_prologue();
  const int lane = threadIdx.x & 31;
  const int nw = (gridDim.x * blockDim.x) >> 5;
  const int n = *count;
  for (int e = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; e < n; e += nw) {
    const RcEntry en = list[e];
    const long row = en.row;
    const int b = (int)(row / N);
    const __nv_bfloat16* h = H + row * d;
    const int nc = en.n < 0 ? C : en.n;
    float bv = -INFINITY;
    int bi = INT_MAX;
    for (int q = 0; q < nc; ++q) {
      const int c = en.n < 0 ? q : en.c[q];
      const float* m = mu + ((long)b * C + c) * d;
      float dot = 0.f;
#pragma unroll 4
      for (int k = lane * 8; k < d; k += 256) {
        float hv[8];
        load16(h + k, hv);
        const float4 m0 = *reinterpret_cast<const float4*>(m + k);
        const float4 m1 = *reinterpret_cast<const float4*>(m + k + 4);
        dot = fmaf(hv[0], m0.x, dot);
        dot = fmaf(hv[1], m0.y, dot);
        dot = fmaf(hv[2], m0.z, dot);
        dot = fmaf(hv[3], m0.w, dot);
        dot = fmaf(hv[4], m1.x, dot);
        dot = fmaf(hv[5], m1.y, dot);
        dot = fmaf(hv[6], m1.z, dot);
        dot = fmaf(hv[7], m1.w, dot);
      }
      dot = warp_sum(dot);
      if (dot > bv) { bv = dot; bi = c; }  // ascending c: the first maximum
    }
    if (lane == 0) {
      if (bi == INT_MAX) { bi = 0; bv = 0.f; }
      if (pass >= 1 && assign[row] != bi) changed[(long)b * kMaxPasses + pass] = 1;
      assign[row] = bi;
      best[row] = bv;
    }
  }
}

// rho_i = <h_i, mu_{a_i}> in fp32 after the last pass, a warp per row (lanes
// over d, summed in a fixed order): steps of 128 elements, lane j taking
// elements 4j .. 4j+3 of a step, so each warp load of h (8 bytes a lane)
// and of mu (16 bytes a lane) is one contiguous run.
__global__ void __launch_bounds__(256)
k_km_rho(const __nv_bfloat16* __restrict__ H, const float* __restrict__ mu, long rows, int N,
         int d, int C, const int32_t* __restrict__ assign, float* __restrict__ rho) {
  pdl_prologue();
  const int lane = threadIdx.x & 31;
  const long nw = ((long)gridDim.x * blockDim.x) >> 5;
  for (long row = ((long)blockIdx.x * blockDim.x + threadIdx.x) >> 5; row < rows; row += nw) {
    const int b = (int)(row / N);
    const __nv_bfloat16* h = H + row * d;
    // a label is in [0, C) unless a pass gave up (then the status word says
    // so); clamped so that no read leaves the centroids
    const int c = min(max(assign[row], 0), C - 1);
    const float* m = mu + ((long)b * C + c) * d;
    float dot = 0.f;
#pragma unroll 8
    for (int k = lane * 4; k < d; k += 128) {
      const uint2 hw = __ldg(reinterpret_cast<const uint2*>(h + k));
      float hv[4];
      bf16x2_to_f32(hw.x, hv[0], hv[1]);
      bf16x2_to_f32(hw.y, hv[2], hv[3]);
      const float4 m0 = *reinterpret_cast<const float4*>(m + k);
      dot = fmaf(hv[0], m0.x, dot);
      dot = fmaf(hv[1], m0.y, dot);
      dot = fmaf(hv[2], m0.z, dot);
      dot = fmaf(hv[3], m0.w, dot);
    }
    dot = warp_sum(dot);
    if (lane == 0) rho[row] = dot;
  }
}

constexpr int kFinRows = 512;  // rows a CTA of k_km_fin_stats takes

// The faster passes' last step, in two kernels instead of a member list per
// (cluster, window).  k_km_fin_stats, CTA (slice, b): the labels and rho of
// rows [slice kFinRows, ...) of window b staged in shared memory; thread c
// counts the rows labelled c and sums their rho in ascending row order (a
// label outside [0, C) counts for no cluster); the slice's objective terms
// sum rho_i / ||h_i|| in a fixed order.
__global__ void __launch_bounds__(256)
k_km_fin_stats(const int32_t* __restrict__ assign, const float* __restrict__ rho,
               const float* __restrict__ inv, int N, int C, int32_t* __restrict__ cnt_part,
               float* __restrict__ rs_part, float* __restrict__ obj_part) {
  pdl_prologue();
  __shared__ int lab[kFinRows];
  __shared__ float rr[kFinRows];
  __shared__ float s_red[32];
  const int b = blockIdx.y, sl = blockIdx.x, S = gridDim.x, t = threadIdx.x;
  const int r0 = sl * kFinRows, len = min(kFinRows, N - r0);
  const long base = (long)b * N + r0;
  float so = 0.f;
  for (int i = t; i < len; i += blockDim.x) {
    lab[i] = assign[base + i];
    const float rv = rho[base + i];
    rr[i] = rv;
    so = fmaf(rv, inv[base + i], so);
  }
  so = block_sum_f32(so, s_red);  // its barriers also publish lab and rr
  if (t == 0) obj_part[(long)b * S + sl] = so;
  for (int c = t; c < C; c += blockDim.x) {
    int n = 0;
    float rs = 0.f;
    for (int i = 0; i < len; ++i)  // every thread reads the same word: a broadcast
      if (lab[i] == c) {
        rs += rr[i];
        ++n;
      }
    cnt_part[((long)b * S + sl) * C + c] = n;
    rs_part[((long)b * S + sl) * C + c] = rs;
  }
}

// k_km_fin_chat, CTA (c, b): the count and the rho sum of cluster c over the
// slices in slice order; C_hat_c = (sum / n) mu_c, a cluster left empty
// keeping the caller's row; CTA (0, b) writes the pass objective, the
// slices' terms in slice order.
__global__ void __launch_bounds__(256)
k_km_fin_chat(const int32_t* __restrict__ cnt_part, const float* __restrict__ rs_part,
              const float* __restrict__ obj_part, int S, const float* __restrict__ mu, int d,
              int C, int32_t* __restrict__ counts, float* __restrict__ chat,
              float* __restrict__ obj, int obj_ld, int pass) {
  pdl_prologue();
  const int c = blockIdx.x, b = blockIdx.y;
  int n = 0;
  float rs = 0.f;
  for (int sl = 0; sl < S; ++sl) {
    n += cnt_part[((long)b * S + sl) * C + c];
    rs += rs_part[((long)b * S + sl) * C + c];
  }
  if (threadIdx.x == 0) {
    counts[(long)b * C + c] = n;
    if (c == 0 && obj != nullptr) {
      float o = 0.f;
      for (int sl = 0; sl < S; ++sl) o += obj_part[(long)b * S + sl];
      obj[(long)b * obj_ld + pass] = o;
    }
  }
  if (n == 0) return;
  const float mean = rs / (float)n;
  const float4* m4 = reinterpret_cast<const float4*>(mu + ((long)b * C + c) * d);
  float4* o4 = reinterpret_cast<float4*>(chat + ((long)b * C + c) * d);
  for (int k = threadIdx.x; k < d / 4; k += blockDim.x) {
    const float4 v = __ldg(m4 + k);
    o4[k] = make_float4(mean * v.x, mean * v.y, mean * v.z, mean * v.w);
  }
}

// Split assignment inside one thread-block cluster (nz <= 8 d-chunks, C <=
// 128): each CTA leaves its chunk's 128 x C scores in shared memory; CTA z
// then takes rows [128 z / nz, 128 (z+1) / nz) of the tile, one warp per row:
// sums the nz chunks' scores of each centroid in chunk order, takes the first
// arg-max and the cosine, and stores the objective partial of its rows as
// objp[t * nz + z].
template <int BN>
struct KmAssignClusterEpi : TcEpiBase {
  static constexpr bool kClusterReduce = true;
  static constexpr uint32_t kLd = BN + 4;
  int B, N, C, mtb;
  const float* inv;
  int32_t* assign;
  float* best;
  float* objp;
  float* scores;  // nullable: [B][N][C] cosines of the pass
  struct State {};
  __device__ int tiles(int) const { return B * mtb; }
  __device__ int arow(int t) const { return (t / mtb) * N + (t % mtb) * 128; }
  __device__ int bcoord(int t, int n0) const { return (t / mtb) * C + n0; }
  __device__ void consume_red(int, int, int, int, uint32_t taddr, State&,
                              float* red_row) const {
    if (red_row == nullptr) return;
#pragma unroll 1
    for (int c0 = 0; c0 < BN; c0 += 32) {
      float v[32];
      tc::tmem_ld32(taddr + c0, v);
#pragma unroll
      for (int j = 0; j < 8; ++j)
        *reinterpret_cast<float4*>(red_row + c0 + 4 * j) =
            make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
    }
  }
  // scratch: 1/||h|| of this CTA's rows of the tile
  __device__ void prefetch(uint8_t* scratch, int k, int n) const {
    const int t = blockIdx.y, b = t / mtb, mt = t % mtb;
    const int z = blockIdx.z, nz = gridDim.z;
    const int r0 = z * 128 / nz, r1 = (z + 1) * 128 / nz;
    float* s_inv = reinterpret_cast<float*>(scratch);
    for (int j = k; j < r1 - r0; j += n) {
      const int i = mt * 128 + r0 + j;
      s_inv[j] = i < N ? inv[(long)b * N + i] : 0.f;
    }
  }
  __device__ void reduce(const float* red, int z, int nz, uint8_t* scratch) const {
    const int t = blockIdx.y, b = t / mtb, mt = t % mtb;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
    const int r0 = z * 128 / nz, r1 = (z + 1) * 128 / nz;  // <= 64 rows (nz >= 2)
    const float* s_inv = reinterpret_cast<const float*>(scratch);  // [64], staged by prefetch
    float* cosv = reinterpret_cast<float*>(scratch) + 64;          // [64]
    // the summed scores replace this CTA's own rows [r0, r1), which only it reads
    float* own = const_cast<float*>(red);
    cluster_rows_sum<8, 32>(red, kLd, r0, r1, (C + 3) & ~3, nz, [&](int r, int c, float4 v) {
      *reinterpret_cast<float4*>(own + r * kLd + c) = v;
    });
    tc::cluster_arrive();
    __syncthreads();
    for (int r = r0 + warp; r < r1; r += nwarps) {
      const int i = mt * 128 + r;
      float bv = -INFINITY;
      int bi = INT_MAX;
#pragma unroll
      for (int j = 0; j < BN / 32; ++j) {
        const int c = lane + 32 * j;
        const float v = own[r * kLd + c];
        if (c < C && v > bv) { bv = v; bi = c; }
        if (scores != nullptr && c < C && i < N)
          scores[((long)b * N + i) * C + c] = v * s_inv[r - r0];
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
      }
      if (bi == INT_MAX) { bi = 0; bv = 0.f; }
      if (lane == 0) {
        float cs = 0.f;
        if (i < N) {
          const long row = (long)b * N + i;
          assign[row] = bi;
          best[row] = bv;
          cs = bv * s_inv[r - r0];
        }
        cosv[r - r0] = cs;
      }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      float so = 0.f;
      for (int j = 0; j < r1 - r0; ++j) so += cosv[j];
      objp[(long)t * nz + z] = so;
    }
  }
};

// Rows of a split assignment: one warp per row sums the nz partial scores of
// each centroid in chunk order, takes the first arg-max and the cosine;
// block (x, b) covers rows 8x..8x+7 of window b and stores their objective
// partial objp[b][x].
__global__ void __launch_bounds__(256)
k_km_argmax(const float* __restrict__ part, int nz, int B, int N, int C,
            const float* __restrict__ inv, int32_t* __restrict__ assign,
            float* __restrict__ best, float* __restrict__ objp, float* __restrict__ scores) {
  pdl_prologue();
  __shared__ float s_cos[8];
  const int b = blockIdx.y, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int i = blockIdx.x * 8 + warp;
  float cs = 0.f;
  if (i < N) {
    const long row = (long)b * N + i;
    const long zs = (long)B * N * C;
    float bv = -INFINITY;
    int bi = INT_MAX;
    for (int c = lane; c < C; c += 32) {
      float sum = 0.f;
      for (int z = 0; z < nz; ++z) sum += __ldcg(part + z * zs + row * C + c);
      if (sum > bv) { bv = sum; bi = c; }
      if (scores != nullptr) scores[row * C + c] = sum * inv[row];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
    }
    if (bi == INT_MAX) { bi = 0; bv = 0.f; }
    if (lane == 0) {
      assign[row] = bi;
      best[row] = bv;
    }
    cs = bv * inv[row];
  }
  if (lane == 0) s_cos[warp] = cs;
  __syncthreads();
  if (threadIdx.x == 0) {
    float so = 0.f;
    for (int w = 0; w < 8; ++w) so += s_cos[w];
    objp[(long)b * gridDim.x + blockIdx.x] = so;
  }
}

// Per (cluster c, window b, column slice z): members in ascending row order.
// A CTA takes clusters [U x, U x + U) of window y in turn (U from
// scan_units).  The d columns are cut into S slices of W columns (a
// multiple of 16); the S CTAs of one (x, b) form a thread-block cluster along
// z.  Each thread owns V consecutive columns (V = 16 bytes of H) of its
// slice, times G (1 or 2) groups, so a member row costs one 16-byte load per
// thread, and up to 16 (G = 1) or 4 (G = 2) member rows are loaded together.
// Rows are scanned in blocks of 4096: the block's assignments are staged in
// shared memory with 16-byte loads (once for all of the CTA's clusters when
// the window has at most 4096 rows), every thread counts the members in its
// contiguous run of rows, one block scan places them, and the member list
// sits in shared memory (over the staged assignments, which are all read
// before the scan, in a longer window); 1/||h|| of a member is loaded with
// its row.
// Update pass: centroid = normalise(sum_i h_i/||h_i||) (kept when the cluster
// is empty or its sum is zero), plus its bf16 split; the squared norm is the
// sum of the slices' partials, read from each CTA's shared memory across the
// cluster in rank order, so every slice divides by the same number.  Final
// pass: C_hat_c = mean(rho over members) * mu_c (kept when empty).  Slice 0
// writes the cluster size; the CTA of cluster 0 and slice 0 folds the pass
// objective from the tile partials.
constexpr int kScanRows = 4096;
constexpr int kMaxColGroups = 2;
constexpr int kMaxSlices = 8;

template <typename T, bool FINAL, int G, bool FUSED = false>
__global__ void __launch_bounds__(1024)
k_cluster_scan(int U, const T* __restrict__ H, const float* __restrict__ inv,
               const int32_t* __restrict__ assign, const float* __restrict__ rho, int N,
               int d, int C, int W, float* __restrict__ mu, __nv_bfloat16* __restrict__ mu_hi,
               __nv_bfloat16* __restrict__ mu_lo, int32_t* __restrict__ counts,
               float* __restrict__ chat, const float* __restrict__ objp, int ntile,
               float* __restrict__ obj, int obj_ld, int pass,
               const int32_t* __restrict__ assign_fin, const int32_t* __restrict__ changed,
               float* __restrict__ emax) {
  pdl_prologue();
  constexpr int V = Vec<T>::n;
  constexpr int kMemb = G == 1 ? 16 : 4;  // rows loaded together, within 64 registers
  __shared__ __align__(16) int list[kScanRows];  // staged assignments, then members
  // a window of at most kScanRows rows: its assignments staged once for all
  // of this CTA's clusters (the members then go to list)
  __shared__ __align__(16) int lab[kScanRows];
  __shared__ int s_scan[32];
  __shared__ float s_red[32];
  __shared__ float s_ss;
  const int b = blockIdx.y, z = blockIdx.z, S = gridDim.z;
  const int c_lo = blockIdx.x * U, c_hi = min(C, c_lo + U);  // this CTA's clusters
  const int tid = threadIdx.x, nthr = blockDim.x;
  // The pass objective, by the CTA of cluster 0 and slice 0: with `changed`
  // (the faster passes) from the rows' best scores, sum_i best_i / ||h_i|| in a fixed order
  // (rho holds the best scores of the latest pass of this window); else from
  // the assignment tiles' partials.
  auto fold_objective = [&]() {
    if (c_lo != 0 || z != 0 || obj == nullptr) return;  // block-uniform
    float so = 0.f;
    if (changed != nullptr) {
      for (int i = tid; i < N; i += nthr) so = fmaf(rho[(long)b * N + i], inv[(long)b * N + i], so);
    } else {
      for (int t = tid; t < ntile; t += nthr) so += objp[(long)b * ntile + t];
    }
    so = block_sum_f32(so, s_red);
    if (tid == 0) obj[(long)b * obj_ld + pass] = so;
  };
  // a window whose passes have settled keeps its centroids: only the
  // objective of this pass is written (the same as the last one computed)
  if (!FINAL && changed != nullptr && !km_pass_active(changed, b, pass + 1)) {
    fold_objective();
    return;
  }
  const bool whole = N <= kScanRows;
  if (whole) {
    const int32_t* ab = assign + (long)b * N;
    if (((reinterpret_cast<uintptr_t>(ab)) & 15) == 0) {
      const int n4 = N >> 2;
      for (int j = tid; j < n4; j += nthr)
        reinterpret_cast<int4*>(lab)[j] = __ldg(reinterpret_cast<const int4*>(ab) + j);
      for (int j = (n4 << 2) + tid; j < N; j += nthr) lab[j] = __ldg(ab + j);
    } else {
      for (int j = tid; j < N; j += nthr) lab[j] = __ldg(ab + j);
    }
    __syncthreads();
  }
#pragma unroll 1
  for (int c = c_lo; c < c_hi; ++c) {
    {
      const int col0 = z * W, col1 = min(d, col0 + W);
      float u[G][V];
#pragma unroll
      for (int g = 0; g < G; ++g)
#pragma unroll
        for (int e = 0; e < V; ++e) u[g][e] = 0.f;
      float rs = 0.f;
      int n = 0;
      for (int base = 0; base < N; base += kScanRows) {
        const int len = min(kScanRows, N - base);
        const int* src = whole ? lab : list;
        if (!whole) {
          const int32_t* ab = assign + (long)b * N + base;
          if (((reinterpret_cast<uintptr_t>(ab)) & 15) == 0) {
            const int n4 = len >> 2;
            for (int j = tid; j < n4; j += nthr)
              reinterpret_cast<int4*>(list)[j] = __ldg(reinterpret_cast<const int4*>(ab) + j);
            for (int j = (n4 << 2) + tid; j < len; j += nthr) list[j] = __ldg(ab + j);
          } else {
            for (int j = tid; j < len; j += nthr) list[j] = __ldg(ab + j);
          }
          __syncthreads();
        }
        const int R = (len + nthr - 1) / nthr;  // <= 64
        const int q0 = tid * R;
        unsigned long long hit = 0ull;
        int cnt = 0;
        for (int q = 0; q < R; ++q) {
          if (q0 + q < len && src[q0 + q] == c) {
            hit |= 1ull << q;
            ++cnt;
          }
        }
        const int r0 = base + q0;
        int tot;
        int w = block_exclusive_scan<int>(cnt, s_scan, &tot);
        while (hit) {
          const int q = __ffsll(hit) - 1;
          hit &= hit - 1;
          const int i = r0 + q;
          list[w] = i;
          ++w;
        }
        __syncthreads();
        if constexpr (FINAL) {
          for (int m = tid; m < tot; m += nthr) rs += rho[(long)b * N + list[m]];
        } else {
          for (int m = 0; m < tot; m += kMemb) {
            const int cnt_m = min(kMemb, tot - m);
            uint4 raw[kMemb][G];
            float sc[kMemb];
#pragma unroll
            for (int q = 0; q < kMemb; ++q) {
              const long row = (long)b * N + list[m + (q < cnt_m ? q : 0)];
              sc[q] = q < cnt_m ? __ldg(inv + row) : 0.f;
              const T* h = H + row * d;
#pragma unroll
              for (int g = 0; g < G; ++g) {
                const int col = col0 + (g * nthr + tid) * V;
                raw[q][g] = (q < cnt_m && col < col1)
                                ? __ldg(reinterpret_cast<const uint4*>(h + col))
                                : make_uint4(0u, 0u, 0u, 0u);
              }
            }
#pragma unroll
            for (int q = 0; q < kMemb; ++q) {
#pragma unroll
              for (int g = 0; g < G; ++g) {
                float v[V];
                unpack16(raw[q][g], v, T{});
#pragma unroll
                for (int e = 0; e < V; ++e) u[g][e] = fmaf(v[e], sc[q], u[g][e]);
              }
            }
          }
        }
        n += tot;
        __syncthreads();
      }
      if (c == c_lo) fold_objective();
      // fused last update + final pass: the final labels' members give the
      // count and the mean rho of C_hat
      int n_fin = n;
      float rs_fin = 0.f;
      if constexpr (FUSED) {  // assign_fin: the final labels
        int cnt = 0;
        for (int i = tid; i < N; i += nthr)
          if (__ldg(assign_fin + (long)b * N + i) == c) {
            rs_fin += rho[(long)b * N + i];
            ++cnt;
          }
        block_exclusive_scan<int>(cnt, s_scan, &n_fin);
        rs_fin = block_sum_f32(rs_fin, s_red);
      }
      if (z == 0 && tid == 0) counts[(long)b * C + c] = n_fin;
      if constexpr (FINAL) {
        const float tot = block_sum_f32(rs, s_red);
        if (n == 0) goto next_cluster;  // block-uniform
        const float mean = tot / (float)n;
        const float* mc = mu + ((long)b * C + c) * d;
        float* o = chat + ((long)b * C + c) * d;
        for (int k = col0 + tid; k < col1; k += nthr) o[k] = mean * mc[k];
      } else {
        float ss = 0.f;
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
          for (int e = 0; e < V; ++e) ss = fmaf(u[g][e], u[g][e], ss);
        ss = block_sum_f32(ss, s_red);
        if (S > 1) {  // every CTA of the cluster reaches the barrier and the wait below
          if (tid == 0) s_ss = ss;
          tc::cluster_sync_all();
          if (tid == 0) {
            const uint32_t a = tc::smem_u32(&s_ss);
            float part[kMaxSlices];
#pragma unroll
            for (int r = 0; r < kMaxSlices; ++r)
              part[r] = r < S ? tc::ld_dsmem_f32(tc::cluster_map(a, r)) : 0.f;
            float t = 0.f;
#pragma unroll
            for (int r = 0; r < kMaxSlices; ++r)
              if (r < S) t += part[r];
            s_red[0] = t;
          }
          tc::cluster_arrive();
          __syncthreads();
          ss = s_red[0];
        }
        const float nu = sqrtf(ss);
        const bool formed = n > 0 && nu > 0.f;  // else the centroid is kept
        if (!FUSED && !formed) {
          if (S > 1) tc::cluster_wait();
          goto next_cluster;
        }
        const long ro = ((long)b * C + c) * d;
        const float mean = (FUSED && n_fin > 0) ? rs_fin / (float)n_fin : 0.f;
        float e2 = 0.f;  // ||mu_c - bf16(mu_c)||^2 over this slice's columns
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const int col = col0 + (g * nthr + tid) * V;
          if (col < col1) {  // V consecutive columns: 16-byte fp32 stores, 8- or 16-byte bf16
            float x[V];
            if (formed) {
#pragma unroll
              for (int e = 0; e < V; ++e) x[e] = u[g][e] / nu;
              if (emax != nullptr) {
#pragma unroll
                for (int e = 0; e < V; ++e) {
                  const float dv = x[e] - __bfloat162float(__float2bfloat16_rn(x[e]));
                  e2 = fmaf(dv, dv, e2);
                }
              }
              float4* mo = reinterpret_cast<float4*>(mu + ro + col);
#pragma unroll
              for (int e = 0; e < V; e += 4)
                mo[e / 4] = make_float4(x[e], x[e + 1], x[e + 2], x[e + 3]);
              if (mu_hi != nullptr) {
                uint32_t hi[V / 2], lo[V / 2];
#pragma unroll
                for (int e = 0; e < V; e += 2) {
                  const __nv_bfloat162 h = __floats2bfloat162_rn(x[e], x[e + 1]);
                  const float2 hf = __bfloat1622float2(h);
                  const __nv_bfloat162 l = __floats2bfloat162_rn(x[e] - hf.x, x[e + 1] - hf.y);
                  hi[e / 2] = *reinterpret_cast<const uint32_t*>(&h);
                  lo[e / 2] = *reinterpret_cast<const uint32_t*>(&l);
                }
                if constexpr (V == 8) {
                  *reinterpret_cast<uint4*>(mu_hi + ro + col) =
                      make_uint4(hi[0], hi[1], hi[2], hi[3]);
                  if (mu_lo != nullptr)  // the faster passes use the hi part only
                    *reinterpret_cast<uint4*>(mu_lo + ro + col) =
                        make_uint4(lo[0], lo[1], lo[2], lo[3]);
                } else {
                  *reinterpret_cast<uint2*>(mu_hi + ro + col) = make_uint2(hi[0], hi[1]);
                  if (mu_lo != nullptr)
                    *reinterpret_cast<uint2*>(mu_lo + ro + col) = make_uint2(lo[0], lo[1]);
                }
              }
            } else if (FUSED && n_fin > 0) {
              const float4* mi = reinterpret_cast<const float4*>(mu + ro + col);
#pragma unroll
              for (int e = 0; e < V; e += 4) {
                const float4 m4 = mi[e / 4];
                x[e] = m4.x; x[e + 1] = m4.y; x[e + 2] = m4.z; x[e + 3] = m4.w;
              }
            }
            if (FUSED && n_fin > 0) {
              float4* co = reinterpret_cast<float4*>(chat + ro + col);
#pragma unroll
              for (int e = 0; e < V; e += 4)
                co[e / 4] =
                    make_float4(mean * x[e], mean * x[e + 1], mean * x[e + 2], mean * x[e + 3]);
            }
          }
        }
        // the bf16 rounding bound of the window's centroids: this slice's share
        // of ||mu_c - bf16(mu_c)|| times sqrt(S) bounds the whole row's (its
        // square is at most S times the largest slice's)
        if (emax != nullptr && formed) {  // block-uniform
          e2 = block_sum_f32(e2, s_red);
          if (tid == 0) atomicMax(reinterpret_cast<int*>(emax) + b, __float_as_int(sqrtf(e2 * S)));
        }
        // no CTA leaves while another still reads its s_ss
        if (S > 1) tc::cluster_wait();
      }
    }
  next_cluster:
    __syncthreads();  // the shared arrays serve the next cluster
  }
  pdl_trigger();
}

// Column slices of the cluster scan: enough (<= 8, a power of two) that the
// C x B x S CTAs fill the SMs, while a slice keeps >= 2 warps of 16-byte
// vectors.  W = slice width, a multiple of 16 columns.
struct ScanPlan {
  int S, W, threads, G;
};

template <typename T>
ScanPlan scan_plan(int B, int d, int C) {
  constexpr int V = Vec<T>::n;
  ScanPlan p{1, d, 0, 1};
  while (p.S < kMaxSlices && (long)C * B * p.S < kSmTarget && d / (2 * p.S) >= 64 * V) p.S *= 2;
  p.W = ceil_div(ceil_div(d, p.S), 16) * 16;
  const int vecs = ceil_div(p.W, V);
  p.G = vecs <= 1024 ? 1 : kMaxColGroups;
  const int want = ceil_div(vecs, p.G);
  // >= 64 threads keeps each thread's run of rows within a 64-bit mask
  p.threads = std::max(64, std::min(1024, ceil_div(want, 32) * 32));
  return p;
}

// Clusters a scan CTA takes in turn (U): 1 while the C x B x S CTAs are
// about a wave, up to 8 when there are many more, so that a pass whose
// windows have all settled launches few CTAs (each checks its window's flag
// once and leaves) while a working pass keeps several waves of CTAs.
int scan_units(int B, int C, int S) {
  const long ctas = (long)C * B * S;
  return (int)std::max(1L, std::min(8L, ctas / (8L * kSmTarget)));
}

// gated: an update pass of the faster Lloyd form, whose settled windows'
// CTAs leave at once; it and the final scan give a CTA several clusters of
// one window (their labels staged once), the other updates one
template <typename T, bool FINAL, bool FUSED = false, typename... Args>
cudaError_t launch_scan(const ScanPlan& p, int B, int C, bool gated, cudaStream_t s,
                        Args&&... args) {
  const int U = gated || FINAL ? scan_units(B, C, p.S) : 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ceil_div(C, U), B, p.S);
  cfg.blockDim = dim3(p.threads);
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = kUsePdl ? 1 : 0;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = 1;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = p.S;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return p.G == 1
             ? launch_ex(cfg, k_cluster_scan<T, FINAL, 1, FUSED>, U, std::forward<Args>(args)...)
             : launch_ex(cfg, k_cluster_scan<T, FINAL, kMaxColGroups, FUSED>, U,
                         std::forward<Args>(args)...);
}

// PS_KMEANS_LLOYD set in the environment keeps every pass in the Lloyd form
// (centroid update + tensor-core assignment), for comparing the two forms.
bool kmeans_lloyd_forced() {
  static const bool forced = std::getenv("PS_KMEANS_LLOYD") != nullptr;
  return forced;
}

struct KmPlan {
  bool tc;
  bool cluster;  // d-chunks reduced inside a thread-block cluster
  int BN, mtb, nz, kpc, KB;
  int ntile;  // objective partials per window
};

int pow2_at_least(int x) {
  int p = 32;
  while (p < x) p *= 2;
  return p;
}

KmPlan km_plan(int dtype, int B, int N, int d, int C) {
  KmPlan p{};
  p.tc = dtype == PS_BF16 && C <= 256;
  if (p.tc) {
    p.BN = pow2_at_least(C);
    p.mtb = ceil_div(N, 128);
    p.KB = ceil_div(d, 64);
    const int tiles = B * p.mtb;
    int nz = std::min(8, std::max(1, ceil_div(kSmTarget, tiles)));
    nz = std::min(nz, p.KB);
    // the d-chunks of a tile share a cluster: keep the clusters in one wave
    while (nz > 1 && p.BN <= 128 && tiles > tc_cluster_capacity(nz)) --nz;
    p.kpc = ceil_div(p.KB, nz);
    p.nz = ceil_div(p.KB, p.kpc);
    p.cluster = p.nz > 1 && p.BN <= 128;
    p.ntile = p.nz == 1 ? p.mtb : (p.cluster ? p.mtb * p.nz : ceil_div(N, 8));
  } else {
    p.ntile = ceil_div(N, kTileRows);
  }
  return p;
}

struct KmWs {
  float* inv;
  float* objp;
  float* w;
  int8_t* chosen;
  __nv_bfloat16* mu_hi;
  __nv_bfloat16* mu_lo;
  float* part;
  float* L;        // Gram form: [B][N][C] cosines carried for kept centroids
  int32_t* prev;   // Gram form: labels of pass I - 1
  __nv_bfloat16* mu_split;  // Gram form with pass 0 inside: [B][2C][d] hi, lo rows
  int16_t* qhi;    // Gram form: fixed-point Gram matrices, high and low parts
  uint8_t* qlo;
  // faster passes: per-window flags, rounding bound and recheck list; the
  // first three are one contiguous block (zeroed per call)
  int32_t* changed;  // [B][kMaxPasses]
  float* emax;       // [B]
  int* rc_count;     // [kMaxPasses]
  size_t flag_bytes;
  RcEntry* rc_list;  // [B * N]
  // faster passes' last step: per (window, slice) cluster statistics
  int32_t* fin_cnt;  // [B][S][C]
  float* fin_rs;     // [B][S][C]
  float* fin_obj;    // [B][S]
};

inline int fin_slices(int N) { return (N + kFinRows - 1) / kFinRows; }

KmWs km_carve(void* base, const KmPlan& p, const GramPlan& g, int B, int N, int d, int C,
              size_t* bytes) {
  Carver cv(base);
  KmWs w{};
  const long BN_ = (long)B * N;
  w.inv = cv.take<float>(BN_);
  w.objp = cv.take<float>((size_t)B * p.ntile);
  w.w = cv.take<float>(BN_);
  w.chosen = cv.take<int8_t>(BN_);
  if (p.tc) {
    w.mu_hi = cv.take<__nv_bfloat16>((size_t)B * C * d);
    w.mu_lo = cv.take<__nv_bfloat16>((size_t)B * C * d);
    w.part = p.nz > 1 && !p.cluster ? cv.take<float>((size_t)p.nz * C * BN_) : nullptr;
    if (p.nz == 1) {
      const size_t nflag = (size_t)B * kMaxPasses + B + kMaxPasses;
      w.changed = cv.take<int32_t>(nflag);
      w.emax = reinterpret_cast<float*>(w.changed ? w.changed + (size_t)B * kMaxPasses : nullptr);
      w.rc_count = w.changed ? w.changed + (size_t)B * kMaxPasses + B : nullptr;
      w.flag_bytes = nflag * sizeof(int32_t);
      w.rc_list = cv.take<RcEntry>((size_t)BN_);
      const size_t nfs = (size_t)B * fin_slices(N);
      w.fin_cnt = cv.take<int32_t>(nfs * C);
      w.fin_rs = cv.take<float>(nfs * C);
      w.fin_obj = cv.take<float>(nfs);
    }
  }
  if (g.ok) {
    const size_t q = (size_t)B * g.Z * N * g.R;
    w.L = cv.take<float>((size_t)BN_ * C);
    w.prev = cv.take<int32_t>((size_t)BN_);
    if (g.fused0) w.mu_split = cv.take<__nv_bfloat16>((size_t)B * 2 * C * d);
    w.qhi = cv.take<int16_t>(q);
    w.qlo = cv.take<uint8_t>(q);
  }
  if (bytes != nullptr) *bytes = cv.bytes();
  return w;
}

template <int BN>
cudaError_t assign_tc(const KmeansArgs& a, const KmPlan& p, const KmWs& w, float* scores,
                      cudaStream_t s) {
  TcMaps maps;
  const long rows = (long)a.B * a.N;
  if (!make_tmap_bf16_2d(&maps.a[0], a.H, a.d, rows, (uint64_t)a.d * 2, 64, 128) ||
      !make_tmap_bf16_2d(&maps.b[0], w.mu_hi, a.d, (uint64_t)a.B * a.C, (uint64_t)a.d * 2, 64,
                         BN) ||
      !make_tmap_bf16_2d(&maps.b[1], w.mu_lo, a.d, (uint64_t)a.B * a.C, (uint64_t)a.d * 2, 64,
                         BN))
    return cudaErrorInvalidValue;
  maps.a[1] = maps.a[0];
  TcShape sh{(int)rows, nullptr, p.KB, p.kpc, a.status, INT_MAX};
  if constexpr (BN <= 128) {
    if (p.cluster) {
      KmAssignClusterEpi<BN> epi{{}, a.B, a.N, a.C, p.mtb, w.inv, a.assign, a.rho, w.objp,
                                 scores};
      return launch_tc_gemm<BN, 1, 2, false>(maps, sh, epi, dim3(1, a.B * p.mtb, p.nz), s);
    }
  }
  KmAssignEpi<BN> epi{{}, a.B, a.N, a.C, p.mtb, p.nz, w.part, w.inv, a.assign, a.rho,
                      w.objp, scores};
  cudaError_t e =
      launch_tc_gemm<BN, 1, 2, false>(maps, sh, epi, dim3(1, a.B * p.mtb, p.nz), s);
  if (e != cudaSuccess || p.nz == 1) return e;
  launch_pdl(k_km_argmax, dim3(ceil_div(a.N, 8), a.B), 256, 0, s, w.part, p.nz, a.B, a.N, a.C,
                                                          w.inv, a.assign, a.rho, w.objp, scores);
  return cudaGetLastError();
}

// One faster pass (see the file comment): bf16(mu) scores on the tensor
// cores over a persistent grid of at most one CTA per SM walking the row
// tiles, tiles of settled windows skipped; then the recheck of the listed
// rows.
template <int BN>
cudaError_t assign_fast(const KmeansArgs& a, const KmPlan& p, const KmWs& w, int pass,
                        cudaStream_t s) {
  TcMaps maps;
  const long rows = (long)a.B * a.N;
  if (!make_tmap_bf16_2d(&maps.a[0], a.H, a.d, rows, (uint64_t)a.d * 2, 64, 128) ||
      !make_tmap_bf16_2d(&maps.b[0], w.mu_hi, a.d, (uint64_t)a.B * a.C, (uint64_t)a.d * 2, 64,
                         BN))
    return cudaErrorInvalidValue;
  maps.a[1] = maps.a[0];
  maps.b[1] = maps.b[0];
  TcShape sh{(int)rows, nullptr, p.KB, p.KB, a.status, INT_MAX};
  KmFastEpi<BN> epi{{}, a.B, a.N, a.C, p.mtb, pass, w.inv, w.emax, a.assign, a.rho,
                    w.changed, w.rc_count + pass, w.rc_list};
  const int tiles = a.B * p.mtb;
  const int gy = std::min(tiles, a.num_sms > 0 ? a.num_sms : kSmTarget);
  cudaError_t e = launch_tc_gemm<BN, 1, 1, false>(maps, sh, epi, dim3(1, gy, 1), s);
  if (e != cudaSuccess) return e;
  launch_pdl(k_km_recheck, 2 * kSmTarget, 256, 0, s,
             static_cast<const __nv_bfloat16*>(a.H), a.mu, a.N, a.d, a.C, pass,
             w.rc_count + pass, w.rc_list, a.assign, a.rho, w.changed);
  return cudaGetLastError();
}

// PS_KMEANS_SLOW set in the environment keeps the hi + lo passes without
// early exit, for comparing the two.
bool kmeans_fast_disabled() {
  static const bool off = std::getenv("PS_KMEANS_SLOW") != nullptr;
  return off;
}

// Inside a stream capture, pass t >= 2 of the faster passes (with its
// update) becomes the body of a conditional graph node: this kernel, just
// before it, opens the node only if some window still runs pass t, so a
// pass after every window has settled costs one small launch instead of
// three (the assignment, the recheck and the update, all of whose CTAs
// would only find their windows settled).
__global__ void __launch_bounds__(256)
k_km_gate(const int32_t* __restrict__ changed, int B, int t, cudaGraphConditionalHandle h) {
  bool any = false;
  for (int b = threadIdx.x; b < B; b += blockDim.x) any = any || km_pass_active(changed, b, t);
  any = __syncthreads_or(any) != 0;
  if (threadIdx.x == 0) cudaGraphSetConditional(h, any ? 1u : 0u);
}

// The objectives of passes 2 .. I-1 that no window ran (their updates were
// gated off): each repeats the pass before, which is what those updates
// would have written (the fold of the same best scores).  One CTA, passes
// in order.
__global__ void __launch_bounds__(1024)
k_km_obj_carry(const int32_t* __restrict__ changed, int B, int iters, float* __restrict__ obj,
               int obj_ld) {
  for (int t = 2; t < iters; ++t) {
    bool any = false;
    for (int b = threadIdx.x; b < B; b += blockDim.x) any = any || km_pass_active(changed, b, t);
    any = __syncthreads_or(any) != 0;
    if (!any)
      for (int b = threadIdx.x; b < B; b += blockDim.x)
        obj[(long)b * obj_ld + t] = obj[(long)b * obj_ld + t - 1];
    __syncthreads();
  }
}

// While `s` is being captured into a graph: enqueue on `s` the gate for pass
// t and a conditional node whose body `launch_body(stream)` enqueues (on
// the handle's own stream `aux`, captured into the node's body graph).
template <typename F>
cudaError_t gated_pass(cudaStream_t s, cudaStream_t aux, const int32_t* changed, int B, int t,
                       F&& launch_body) {
  cudaStreamCaptureStatus cs;
  cudaGraph_t g;
  const cudaGraphNode_t* deps = nullptr;
  size_t nd = 0;
  cudaError_t e = cudaStreamGetCaptureInfo(s, &cs, nullptr, &g, &deps, nullptr, &nd);
  if (e != cudaSuccess) return e;
  cudaGraphConditionalHandle h;
  e = cudaGraphConditionalHandleCreate(&h, g, 0u, 0u);
  if (e != cudaSuccess) return e;
  k_km_gate<<<1, 256, 0, s>>>(changed, B, t, h);
  e = cudaGetLastError();
  if (e == cudaSuccess) e = cudaStreamGetCaptureInfo(s, &cs, nullptr, &g, &deps, nullptr, &nd);
  if (e != cudaSuccess) return e;
  cudaGraphNodeParams np = {};
  np.type = cudaGraphNodeTypeConditional;
  np.conditional.handle = h;
  np.conditional.type = cudaGraphCondTypeIf;
  np.conditional.size = 1;
  cudaGraphNode_t node;
  e = cudaGraphAddNode(&node, g, deps, nullptr, nd, &np);
  if (e != cudaSuccess) return e;
  e = cudaStreamBeginCaptureToGraph(aux, np.conditional.phGraph_out[0], nullptr, nullptr, 0,
                                    cudaStreamCaptureModeRelaxed);
  if (e != cudaSuccess) return e;
  cudaError_t eb = launch_body(aux);
  cudaGraph_t body;
  e = cudaStreamEndCapture(aux, &body);
  if (eb != cudaSuccess) return eb;
  if (e != cudaSuccess) return e;
  return cudaStreamUpdateCaptureDependencies(s, &node, nullptr, 1,
                                             cudaStreamSetCaptureDependencies);
}

template <typename T>
cudaError_t run_typed(const KmeansArgs& a, cudaStream_t s) {
  const T* H = static_cast<const T*>(a.H);
  const long BN_ = (long)a.B * a.N;
  const KmPlan p = km_plan(a.dtype, a.B, a.N, a.d, a.C);
  const GramPlan g = gram_plan(a.dtype, a.B, a.N, a.d, a.C);
  const KmWs w = km_carve(a.ws, p, g, a.B, a.N, a.d, a.C, nullptr);
  const ScanPlan sp = scan_plan<T>(a.B, a.d, a.C);

  const bool gram = p.tc && g.ok && a.iters >= 2 && !kmeans_lloyd_forced() &&
                    gram_launchable(g);
  const bool fused0 = gram && g.fused0;  // pass 0 inside the Gram GEMM
  __nv_bfloat16* split_hi = fused0 ? w.mu_split : w.mu_hi;
  __nv_bfloat16* split_lo = fused0 ? w.mu_split : w.mu_lo;
  const long cd = fused0 ? (long)a.C * a.d : 0;

  // 1/||h|| and (tensor cores) the split of the given centroids in one
  // launch; with k-means++ seeding the split waits for the seeds
  const int inv_blocks = ceil_div(BN_ * 32, 256);
  const long n_mu = p.tc ? (long)a.B * a.C * a.d : 0;
  const int split_blocks = n_mu > 0 ? std::min(ceil_div(n_mu / 4, 256), 2 * kSmTarget) : 0;
  const bool seeding = a.init_mode == 1;
  // Gram form with k-means++: the seeds come from K itself (gram_seed), one
  // launch instead of 2C - 1, and pass 0's cosines are K's columns
  const bool gram_seeding = gram && seeding;
  // the faster passes (one d-chunk per tile, bf16 windows, no Gram form)
  const bool fast = p.tc && p.nz == 1 && !gram && a.iters + 1 <= kMaxPasses &&
                    !kmeans_fast_disabled() && std::is_same<T, __nv_bfloat16>::value;
  if (fast) {
    cudaError_t e = cudaMemsetAsync(w.changed, 0, w.flag_bytes, s);
    if (e != cudaSuccess) return e;
    split_lo = nullptr;  // the faster passes score against the hi part alone
  }
  float* emax = fast ? w.emax : nullptr;
  launch_pdl(k_km_prep<T>, inv_blocks + (seeding ? 0 : split_blocks), 256, 0, s, H, BN_, a.d,
             w.inv, inv_blocks, a.mu, seeding ? 0L : n_mu, split_hi, split_lo, cd, a.C, emax);
  if (seeding && !gram_seeding) {
    for (int r = 0; r < a.C; ++r) {
      launch_pdl(k_kpp_pick<T>, a.B, 1024, 0, s, H, w.inv, a.init_u, a.N, a.d, a.C, r, a.mu,
                 w.w, w.chosen);
      if (r + 1 < a.C)
        launch_pdl(k_kpp_weights<T>, ceil_div(BN_ * 32, 256), 256, 0, s, H, w.inv, a.B, a.N,
                   a.d, a.C, r, a.mu, w.w, w.chosen);
    }
    if (split_blocks > 0)
      launch_pdl(k_km_prep<T>, split_blocks, 256, 0, s, H, 0L, a.d, w.inv, 0, a.mu, n_mu,
                 split_hi, split_lo, cd, a.C, emax);
  }
  auto assign_pass = [&](float* scores) {
    switch (p.BN) {
      case 32: return assign_tc<32>(a, p, w, scores, s);
      case 64: return assign_tc<64>(a, p, w, scores, s);
      case 128: return assign_tc<128>(a, p, w, scores, s);
      default: return assign_tc<256>(a, p, w, scores, s);
    }
  };
  // Gram form: pass 0's cosines against the given centroids (in the Gram
  // GEMM's launch for C <= 64, else a tensor-core pass) seed the carried
  // columns; passes 0 (arg-max) or 1..I run on the Gram matrices; one scan
  // forms mu^(I) from the labels of pass I - 1 and C_hat from those of pass I
  if (gram) {
    const auto* Hb = static_cast<const __nv_bfloat16*>(a.H);
    const bool pass0_in_l = fused0 || gram_seeding;  // pass 0's cosines arrive in L
    cudaError_t e = pass0_in_l ? cudaSuccess : assign_pass(w.L);
    if (e == cudaSuccess)
      e = gram_build(g, Hb, w.inv, a.B, a.N, a.d, a.C,
                     fused0 && !gram_seeding ? w.mu_split : nullptr, w.L, w.qhi, w.qlo,
                     a.status, s);
    if (e == cudaSuccess && gram_seeding)
      e = gram_seed(g, Hb, w.inv, a.init_u, a.B, a.N, a.d, a.C, w.qhi, w.qlo, a.mu, w.L, s);
    if (e == cudaSuccess)
      e = gram_iterate(g, w.qhi, w.qlo, a.B, a.N, a.C, a.iters, Hb, a.d, w.inv, a.mu, a.assign,
                       w.prev, a.rho, w.L, pass0_in_l ? nullptr : w.objp, p.ntile, a.obj,
                       a.iters + 1, a.status, s);
    if (e == cudaSuccess)
      e = launch_scan<T, false, true>(sp, a.B, a.C, false, s,
                                      H, w.inv, w.prev, a.rho, a.N, a.d, a.C,
                                      sp.W, a.mu, nullptr, nullptr, a.counts, a.chat, w.objp,
                                      p.ntile, nullptr, a.iters + 1, a.iters, a.assign,
                                      static_cast<const int32_t*>(nullptr),
                                      static_cast<float*>(nullptr));
    return e != cudaSuccess ? e : cudaGetLastError();
  }
  if (fast) {
    const auto* Hb = static_cast<const __nv_bfloat16*>(a.H);
    auto pass_fast = [&](int t, cudaStream_t st) {
      switch (p.BN) {
        case 32: return assign_fast<32>(a, p, w, t, st);
        case 64: return assign_fast<64>(a, p, w, t, st);
        case 128: return assign_fast<128>(a, p, w, t, st);
        default: return assign_fast<256>(a, p, w, t, st);
      }
    };
    // inside a capture, passes 2 .. I become conditional nodes (k_km_gate)
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    cudaError_t ec = cudaStreamIsCapturing(s, &cs);
    if (ec != cudaSuccess) return ec;
    const bool gate = cs == cudaStreamCaptureStatusActive && a.aux != nullptr;
    for (int t = 0; t <= a.iters; ++t) {
      auto pass_and_update = [&, t](cudaStream_t st) {
        cudaError_t e = pass_fast(t, st);
        if (e == cudaSuccess && t < a.iters)
          e = launch_scan<T, false>(sp, a.B, a.C, true, st,
                                    H, w.inv, a.assign, a.rho, a.N, a.d, a.C,
                                    sp.W, a.mu, w.mu_hi, static_cast<__nv_bfloat16*>(nullptr),
                                    a.counts, a.chat, w.objp,
                                    p.ntile, a.obj, a.iters + 1, t,
                                    static_cast<const int32_t*>(nullptr),
                                    static_cast<const int32_t*>(w.changed), w.emax);
        return e;
      };
      cudaError_t e = gate && t >= 2
                          ? gated_pass(s, a.aux, w.changed, a.B, t, pass_and_update)
                          : pass_and_update(s);
      if (e != cudaSuccess) return e;
    }
    if (gate && a.obj != nullptr && a.iters > 2) {
      k_km_obj_carry<<<1, 1024, 0, s>>>(w.changed, a.B, a.iters, a.obj, a.iters + 1);
      cudaError_t e = cudaGetLastError();
      if (e != cudaSuccess) return e;
    }
    launch_pdl(k_km_rho, std::min(ceil_div(BN_ * 32, 256), 8 * kSmTarget), 256, 0, s, Hb,
               a.mu, BN_, a.N, a.d, a.C, a.assign, a.rho);
    const int S = fin_slices(a.N);
    launch_pdl(k_km_fin_stats, dim3(S, a.B), 256, 0, s, static_cast<const int32_t*>(a.assign),
               static_cast<const float*>(a.rho), static_cast<const float*>(w.inv), a.N, a.C,
               w.fin_cnt, w.fin_rs, w.fin_obj);
    launch_pdl(k_km_fin_chat, dim3(a.C, a.B), 256, 0, s,
               static_cast<const int32_t*>(w.fin_cnt), static_cast<const float*>(w.fin_rs),
               static_cast<const float*>(w.fin_obj), S, static_cast<const float*>(a.mu), a.d,
               a.C, a.counts, a.chat, a.obj, a.iters + 1, a.iters);
    return cudaGetLastError();
  }
  for (int t = 0; t <= a.iters; ++t) {
    cudaError_t e = cudaSuccess;
    if (p.tc) {
      e = assign_pass(nullptr);
    } else {
      launch_pdl(k_assign<T>, dim3(p.ntile, a.B), 256, 0, s, H, a.mu, w.inv, a.N, a.d, a.C,
                                                     a.assign, a.rho, w.objp);
    }
    if (e != cudaSuccess) return e;
    if (t < a.iters)
      e = launch_scan<T, false>(sp, a.B, a.C, false, s,
                                H, w.inv, a.assign, a.rho, a.N, a.d, a.C,
                                sp.W, a.mu, p.tc ? w.mu_hi : nullptr, w.mu_lo, a.counts,
                                a.chat, w.objp, p.ntile, a.obj, a.iters + 1, t,
                                static_cast<const int32_t*>(nullptr),
                                static_cast<const int32_t*>(nullptr), static_cast<float*>(nullptr));
    if (e != cudaSuccess) return e;
  }
  cudaError_t e = launch_scan<T, true>(sp, a.B, a.C, false, s,
                                       H, w.inv, a.assign, a.rho, a.N, a.d,
                                       a.C, sp.W, a.mu, nullptr, nullptr, a.counts, a.chat,
                                       w.objp, p.ntile, a.obj, a.iters + 1, a.iters,
                                       static_cast<const int32_t*>(nullptr),
                                       static_cast<const int32_t*>(nullptr),
                                       static_cast<float*>(nullptr));
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

size_t kmeans_ws(int B, int N, int d, int C) {
  // dtype-independent: the larger of the tensor-core and CUDA-core plans
  size_t tc = 0, simt = 0;
  km_carve(nullptr, km_plan(PS_BF16, B, N, d, C), gram_plan(PS_BF16, B, N, d, C), B, N, d, C,
           &tc);
  km_carve(nullptr, km_plan(PS_F32, B, N, d, C), GramPlan{}, B, N, d, C, &simt);
  return std::max(tc, simt);
}

cudaError_t kmeans_run(const KmeansArgs& a, cudaStream_t s) {
  return a.dtype == PS_F32 ? run_typed<float>(a, s)
                           : run_typed<__nv_bfloat16>(a, s);
}

}  // namespace ps
