// a1: spherical k-means of each window's hidden states.
//
// [Polestar §2.A, local window & clustering]: the window's hidden states are
// clustered with spherical k-means.  Per pass: assign every row to the
// centroid of largest cosine (first maximum), then renormalise each cluster's
// sum of unit rows.  Deterministic: every reduction runs in a fixed order.
//
// Kernels (one launch each, all on the caller's stream):
//   k_inv_norm   1/||h_i||                                  (one warp per row)
//   k_kpp        k-means++ seeding, one CTA per window      (init_mode 1)
//   k_assign     64-row x 128-centroid dot tiles, arg-max    (per pass)
//   k_sort       stable counting sort of rows by cluster    (per pass)
//   k_update     centroid = normalise(sum of member rows)   (passes < I)
//   k_finalize   C_hat = mean(rho over members) * mu
#include <climits>

#include "ops.h"
#include "vec.cuh"

namespace ps {
namespace {

constexpr int kTileRows = 64;    // rows per assignment tile
constexpr int kTileC = 128;      // centroids per chunk of an assignment tile
constexpr int kTileK = 32;       // d per shared-memory stage
constexpr int kMaxD = 8192;

template <typename T>
__global__ void k_inv_norm(const T* __restrict__ H, long rows, int d,
                           float* __restrict__ inv) {
  constexpr int V = Vec<T>::n;
  const long row = ((long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const T* h = H + row * d;
  float ss = 0.f;
  for (int k = lane * V; k < d; k += 32 * V) {
    float v[V];
    load16(h + k, v);
#pragma unroll
    for (int e = 0; e < V; ++e) ss = fmaf(v[e], v[e], ss);
  }
  ss = warp_sum(ss);
  if (lane == 0) inv[row] = ss > 0.f ? 1.0f / sqrtf(ss) : 0.f;
}

// k-means++ on the sphere: one CTA of 1024 threads per window.  Weights
// w_i = 1 - max cos to the chosen centres (0 for chosen rows); centre r is
// the first row whose running sum of w (fp64) exceeds u_r * sum(w).
template <typename T>
__global__ void __launch_bounds__(1024)
k_kpp(const T* __restrict__ H, const float* __restrict__ inv_all,
      const double* __restrict__ U, int N, int d, int C, float* __restrict__ mu,
      float* __restrict__ w_all, int8_t* __restrict__ chosen_all) {
  extern __shared__ float smu[];  // d floats: the newest centre
  __shared__ double s_scan[32];
  __shared__ int s_min[32];
  const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const T* Hb = H + (long)b * N * d;
  const float* inv = inv_all + (long)b * N;
  float* w = w_all + (long)b * N;
  int8_t* chosen = chosen_all + (long)b * N;
  float* mub = mu + (long)b * C * d;
  const double* u = U + (long)b * C;
  for (int i = tid; i < N; i += blockDim.x) chosen[i] = 0;
  __syncthreads();
  const int chunk = (N + blockDim.x - 1) / blockDim.x;
  for (int r = 0; r < C; ++r) {
    int pick = INT_MAX;
    if (r == 0) {
      pick = min(max((int)floor(u[0] * (double)N), 0), N - 1);
    } else {
      const int lo = tid * chunk, hi = min(N, lo + chunk);
      double s = 0.0;
      for (int i = lo; i < hi; ++i) s += (double)w[i];
      double total;
      double base = block_exclusive_scan<double>(s, s_scan, &total);
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
    for (int k = tid; k < d; k += blockDim.x) {
      const float v = to_f32(Hb[(long)pick * d + k]) * ip;
      smu[k] = v;
      mub[(long)r * d + k] = v;
    }
    __syncthreads();
    for (int row = warp; row < N; row += blockDim.x >> 5) {
      const T* h = Hb + (long)row * d;
      float dot = 0.f;
      for (int k = lane; k < d; k += 32) dot = fmaf(to_f32(h[k]), smu[k], dot);
      dot = warp_sum(dot);
      if (lane == 0) {
        const float cw = chosen[row] ? 0.f : fmaxf(0.f, 1.f - dot * inv[row]);
        w[row] = (r == 0) ? cw : fminf(w[row], cw);
      }
    }
    __syncthreads();
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

// Stable counting sort of one window's rows by cluster: counts, offsets and
// the permutation (ascending row order inside each cluster).  Also folds the
// per-tile objective partials of the pass in tile order.
__global__ void __launch_bounds__(1024)
k_sort(const int32_t* __restrict__ assign, int N, int C,
       int32_t* __restrict__ counts, int32_t* __restrict__ offs,
       int32_t* __restrict__ perm, const float* __restrict__ objp, int ntile,
       float* __restrict__ obj, int obj_ld, int pass) {
  extern __shared__ int sm[];
  int* cnt = sm;            // C
  int* base = sm + C;       // C: next write position of each cluster
  int* wc = sm + 2 * C;     // 32 x C: per-warp counts, then write bases
  __shared__ int s_scan[32];
  const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int32_t* a = assign + (long)b * N;
  for (int c = tid; c < C; c += blockDim.x) cnt[c] = 0;
  __syncthreads();
  for (int i = tid; i < N; i += blockDim.x) {
    const int c = a[i];
    if (c >= 0 && c < C) atomicAdd(&cnt[c], 1);
  }
  __syncthreads();
  const int v = tid < C ? cnt[tid] : 0;
  int total;
  const int ex = block_exclusive_scan<int>(v, s_scan, &total);
  if (tid < C) {
    offs[(long)b * (C + 1) + tid] = ex;
    base[tid] = ex;
    counts[(long)b * C + tid] = v;
  }
  if (tid == 0) offs[(long)b * (C + 1) + C] = total;
  __syncthreads();
  const unsigned lt = (1u << lane) - 1u;
  for (int c0 = 0; c0 < N; c0 += blockDim.x) {
    for (int e = tid; e < 32 * C; e += blockDim.x) wc[e] = 0;
    __syncthreads();
    const int i = c0 + tid;
    int c = i < N ? a[i] : -1;
    if (c >= C) c = -1;
    const unsigned peers = __match_any_sync(0xffffffffu, c);
    const int rank = __popc(peers & lt);
    if (c >= 0 && rank == 0) wc[warp * C + c] = __popc(peers);
    __syncthreads();
    if (tid < C) {
      int run = base[tid];
      for (int w = 0; w < 32; ++w) {
        const int t = wc[w * C + tid];
        wc[w * C + tid] = run;
        run += t;
      }
      base[tid] = run;
    }
    __syncthreads();
    if (c >= 0) perm[(long)b * N + wc[warp * C + c] + rank] = i;
    __syncthreads();
  }
  if (obj != nullptr && tid == 0) {
    float s = 0.f;
    for (int t = 0; t < ntile; ++t) s += objp[(long)b * ntile + t];
    obj[(long)b * obj_ld + pass] = s;
  }
}

// New centroid of cluster (blockIdx.x, window blockIdx.y): the normalised
// sum of its members' unit rows, accumulated in ascending row order.
template <typename T>
__global__ void __launch_bounds__(256)
k_update(const T* __restrict__ H, const float* __restrict__ inv, int N, int d,
         int C, const int32_t* __restrict__ perm, const int32_t* __restrict__ offs,
         const int32_t* __restrict__ counts, float* __restrict__ mu) {
  constexpr int V = Vec<T>::n;
  constexpr int G = kMaxD / (256 * V);
  __shared__ float s_red[8];
  const int c = blockIdx.x, b = blockIdx.y, tid = threadIdx.x;
  const int n = counts[(long)b * C + c];
  if (n == 0) return;
  const int start = offs[(long)b * (C + 1) + c];
  float u[G][V];
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int e = 0; e < V; ++e) u[g][e] = 0.f;
  for (int m = 0; m < n; ++m) {
    const int row = perm[(long)b * N + start + m];
    const float s = inv[(long)b * N + row];
    const T* h = H + ((long)b * N + row) * d;
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const int col = (g * 256 + tid) * V;
      if (col < d) {
        float v[V];
        load16(h + col, v);
#pragma unroll
        for (int e = 0; e < V; ++e) u[g][e] = fmaf(v[e], s, u[g][e]);
      }
    }
  }
  float ss = 0.f;
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int e = 0; e < V; ++e) ss = fmaf(u[g][e], u[g][e], ss);
  ss = block_sum_f32(ss, s_red);
  const float nu = sqrtf(ss);
  if (!(nu > 0.f)) return;
  float* out = mu + ((long)b * C + c) * d;
#pragma unroll
  for (int g = 0; g < G; ++g) {
    const int col = (g * 256 + tid) * V;
    if (col < d) {
#pragma unroll
      for (int e = 0; e < V; ++e) out[col + e] = u[g][e] / nu;
    }
  }
}

__global__ void __launch_bounds__(256)
k_finalize(const float* __restrict__ rho, int N, int d, int C,
           const int32_t* __restrict__ perm, const int32_t* __restrict__ offs,
           const int32_t* __restrict__ counts, const float* __restrict__ mu,
           float* __restrict__ chat) {
  __shared__ float s_red[8];
  const int c = blockIdx.x, b = blockIdx.y, tid = threadIdx.x;
  const int n = counts[(long)b * C + c];
  if (n == 0) return;
  const int start = offs[(long)b * (C + 1) + c];
  float s = 0.f;
  for (int m = tid; m < n; m += blockDim.x)
    s += rho[(long)b * N + perm[(long)b * N + start + m]];
  s = block_sum_f32(s, s_red);
  const float mean = s / (float)n;
  const float* m = mu + ((long)b * C + c) * d;
  float* o = chat + ((long)b * C + c) * d;
  for (int k = tid; k < d; k += blockDim.x) o[k] = mean * m[k];
}

template <typename T>
cudaError_t run_typed(const KmeansArgs& a, cudaStream_t s) {
  const T* H = static_cast<const T*>(a.H);
  const long BN = (long)a.B * a.N;
  const int ntile = ceil_div(a.N, kTileRows);
  Carver cv(a.ws);
  float* inv = cv.take<float>(BN);
  int32_t* perm = cv.take<int32_t>(BN);
  int32_t* offs = cv.take<int32_t>((size_t)a.B * (a.C + 1));
  float* objp = cv.take<float>((size_t)a.B * ntile);
  float* w = cv.take<float>(BN);
  int8_t* chosen = cv.take<int8_t>(BN);

  k_inv_norm<T><<<ceil_div(BN * 32, 256), 256, 0, s>>>(H, BN, a.d, inv);
  if (a.init_mode == 1)
    k_kpp<T><<<a.B, 1024, a.d * sizeof(float), s>>>(H, inv, a.init_u, a.N, a.d,
                                                    a.C, a.mu, w, chosen);
  const size_t sort_smem = (size_t)34 * a.C * sizeof(int);
  for (int t = 0; t <= a.iters; ++t) {
    k_assign<T><<<dim3(ntile, a.B), 256, 0, s>>>(H, a.mu, inv, a.N, a.d, a.C,
                                                 a.assign, a.rho, objp);
    k_sort<<<a.B, 1024, sort_smem, s>>>(a.assign, a.N, a.C, a.counts, offs,
                                        perm, objp, ntile, a.obj, a.iters + 1, t);
    if (t < a.iters)
      k_update<T><<<dim3(a.C, a.B), 256, 0, s>>>(H, inv, a.N, a.d, a.C, perm,
                                                  offs, a.counts, a.mu);
  }
  k_finalize<<<dim3(a.C, a.B), 256, 0, s>>>(a.rho, a.N, a.d, a.C, perm, offs,
                                            a.counts, a.mu, a.chat);
  return cudaGetLastError();
}

}  // namespace

size_t kmeans_ws(int B, int N, int d, int C) {
  (void)d;
  Carver cv(nullptr);
  const long BN = (long)B * N;
  cv.take<float>(BN);
  cv.take<int32_t>(BN);
  cv.take<int32_t>((size_t)B * (C + 1));
  cv.take<float>((size_t)B * ceil_div(N, kTileRows));
  cv.take<float>(BN);
  cv.take<int8_t>(BN);
  return cv.bytes();
}

cudaError_t kmeans_run(const KmeansArgs& a, cudaStream_t s) {
  return a.dtype == PS_F32 ? run_typed<float>(a, s)
                           : run_typed<__nv_bfloat16>(a, s);
}

}  // namespace ps
