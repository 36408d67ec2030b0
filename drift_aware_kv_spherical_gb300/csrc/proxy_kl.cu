// a3+a4: centroid keys, proxy attention and the per-position KL drift.
//
// [Polestar §2.A, sparse updates]: every step computes a proxy attention of
// the window's queries against the cluster centroids.
// [Polestar §2.A, drift measurement]: D_i = KL(A_i^(t) || A_i^(t-1)), with
// A_i the attention distribution of token i.
//
//   k_ckeys         K~ = C_hat . W_k   (64x64 tiles, optional split over d)
//   k_split_reduce  sums the split partials in split order
//   k_proxy         16 window rows x all C centroids per CTA, a slice of the
//                   heads per CTA: scores, per-head softmax, head sum
//   k_proxy_final   sums the head-slice partials, A = sum / Hq, KL
// Every reduction has a fixed order, so identical inputs give identical
// bits and KL(A || A) is exactly 0.
#include <algorithm>
#include <cmath>

#include "gemm_simt.cuh"
#include "ops.h"

namespace ps {
namespace {

constexpr int kRows = 16;   // window rows per proxy CTA
constexpr int kKc = 32;     // head-dim stage of the centroid keys

template <typename TW>
__global__ void __launch_bounds__(256)
k_ckeys(const float* __restrict__ chat, const TW* __restrict__ Wk, int M,
        int nout, int d, int klen, float* __restrict__ out) {
  __shared__ __align__(16) SimtSmem sm;
  __shared__ long arow[kSimtM];
  const int tid = threadIdx.x;
  const int n0 = blockIdx.x * kSimtN, m0 = blockIdx.y * kSimtM;
  const int kb = blockIdx.z * klen, ke = min(d, kb + klen);
  if (tid < kSimtM) arow[tid] = (m0 + tid < M) ? (long)(m0 + tid) : -1L;
  __syncthreads();
  float acc[4][4] = {};
  simt_tile(chat, d, arow, Wk, nout, n0, nout, kb, ke, sm, acc);
  float* o = out + (long)blockIdx.z * M * nout;
  const int ty = tid >> 4, tx = tid & 15;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int m = m0 + ty * 4 + i, n = n0 + tx * 4;
    if (m < M && n < nout)
      *reinterpret_cast<float4*>(o + (long)m * nout + n) =
          make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
  }
}

__global__ void k_split_reduce(const float* __restrict__ part, int nsplit,
                               long count, float* __restrict__ out) {
  for (long i = (long)blockIdx.x * blockDim.x + threadIdx.x; i < count;
       i += (long)gridDim.x * blockDim.x) {
    float s = part[i];
    for (int sp = 1; sp < nsplit; ++sp) s += part[(long)sp * count + i];
    out[i] = s;
  }
}

__device__ __forceinline__ float half_warp_sum(float v) {
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float half_warp_max(float v) {
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// A = Aacc / Hq, KL against A_prev, stores.  Thread (r = tid/16, l = tid%16)
// owns centroids l + 16 j of window row i.
template <int NJ>
__device__ __forceinline__ void proxy_finish(const float* Aacc, int Hq, int b,
                                             int i, int N, int C,
                                             const float* __restrict__ A_prev,
                                             float* __restrict__ A_cur,
                                             float* __restrict__ D) {
  const int l = threadIdx.x & 15;
  const float hq = (float)Hq;
  float kl = 0.f;
#pragma unroll
  for (int j = 0; j < NJ; ++j) {
    const int c = l + 16 * j;
    if (c < C && i < N) {
      const float a = Aacc[j] / hq;
      const long idx = ((long)b * N + i) * C + c;
      A_cur[idx] = a;
      if (A_prev != nullptr && a > 0.f) {
        const float ap = fmaxf(A_prev[idx], 1e-30f);
        kl += a * logf(a / ap);
      }
    }
  }
  kl = half_warp_sum(kl);
  if (l == 0 && i < N) D[(long)b * N + i] = A_prev != nullptr ? fmaxf(kl, 0.f) : 0.f;
}

template <typename T, int NJ>
__global__ void __launch_bounds__(256)
k_proxy(const T* __restrict__ Q, const float* __restrict__ Kt, int N, int C,
        int Hq, int Hkv, int dh, int hps, float scale,
        const float* __restrict__ A_prev, float* __restrict__ A_cur,
        float* __restrict__ D, float* __restrict__ part) {
  extern __shared__ float smem[];
  constexpr int Cp = 16 * NJ;
  constexpr int V = Vec<T>::n;
  const int qld = dh + 1, kld = Cp + 1;
  float* Qs = smem;                  // kRows x (dh + 1)
  float* Ks = smem + kRows * qld;    // kKc x (Cp + 1)
  const int tile = blockIdx.x, b = blockIdx.y, slice = blockIdx.z;
  const int tid = threadIdx.x, r = tid >> 4, l = tid & 15;
  const int i = tile * kRows + r;
  const int G = Hq / Hkv;
  const int h0 = slice * hps, h1 = min(Hq, h0 + hps);
  const long kt_ld = (long)Hkv * dh;
  float Aacc[NJ];
#pragma unroll
  for (int j = 0; j < NJ; ++j) Aacc[j] = 0.f;

  for (int h = h0; h < h1; ++h) {
    const int g = h / G;
    __syncthreads();
    for (int e = tid * V; e < kRows * dh; e += 256 * V) {
      const int rr = e / dh, kk = e % dh, ii = tile * kRows + rr;
      float v[V];
      if (ii < N) {
        load16(Q + (((long)b * N + ii) * Hq + h) * dh + kk, v);
      } else {
#pragma unroll
        for (int q = 0; q < V; ++q) v[q] = 0.f;
      }
#pragma unroll
      for (int q = 0; q < V; ++q) Qs[rr * qld + kk + q] = v[q];
    }
    float s[NJ];
#pragma unroll
    for (int j = 0; j < NJ; ++j) s[j] = 0.f;
    for (int kc = 0; kc < dh; kc += kKc) {
      __syncthreads();
      for (int e = tid; e < Cp * (kKc / 4); e += 256) {
        const int c = e / (kKc / 4), k4 = (e % (kKc / 4)) * 4;
        float v[4] = {0.f, 0.f, 0.f, 0.f};
        if (c < C && kc + k4 < dh)
          load4(Kt + ((long)b * C + c) * kt_ld + (long)g * dh + kc + k4, v);
#pragma unroll
        for (int q = 0; q < 4; ++q) Ks[(k4 + q) * kld + c] = v[q];
      }
      __syncthreads();
      const int klen = min(kKc, dh - kc);
      for (int kk = 0; kk < klen; ++kk) {
        const float q = Qs[r * qld + kc + kk];
#pragma unroll
        for (int j = 0; j < NJ; ++j) s[j] = fmaf(q, Ks[kk * kld + l + 16 * j], s[j]);
      }
    }
    float m = -INFINITY;
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      s[j] = (l + 16 * j < C) ? s[j] * scale : -INFINITY;
      m = fmaxf(m, s[j]);
    }
    m = half_warp_max(m);
    float sum = 0.f;
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      s[j] = (l + 16 * j < C) ? expf(s[j] - m) : 0.f;
      sum += s[j];
    }
    sum = half_warp_sum(sum);
#pragma unroll
    for (int j = 0; j < NJ; ++j) Aacc[j] += s[j] / sum;
  }
  if (part == nullptr) {
    proxy_finish<NJ>(Aacc, Hq, b, i, N, C, A_prev, A_cur, D);
  } else if (i < N) {
    const int B = gridDim.y;
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      const int c = l + 16 * j;
      if (c < C) part[(((long)slice * B + b) * N + i) * C + c] = Aacc[j];
    }
  }
}

template <int NJ>
__global__ void __launch_bounds__(256)
k_proxy_final(const float* __restrict__ part, int nslice, int B, int N, int C,
              int Hq, const float* __restrict__ A_prev, float* __restrict__ A_cur,
              float* __restrict__ D) {
  const int b = blockIdx.y, tid = threadIdx.x, r = tid >> 4, l = tid & 15;
  const int i = blockIdx.x * kRows + r;
  float Aacc[NJ];
#pragma unroll
  for (int j = 0; j < NJ; ++j) {
    const int c = l + 16 * j;
    float s = 0.f;
    if (c < C && i < N)
      for (int sl = 0; sl < nslice; ++sl)
        s += part[(((long)sl * B + b) * N + i) * C + c];
    Aacc[j] = s;
  }
  proxy_finish<NJ>(Aacc, Hq, b, i, N, C, A_prev, A_cur, D);
}

struct Plan {
  int nsplit, klen;   // centroid keys: split of d
  int nslice, hps;    // proxy: head slices
};

Plan make_plan(int B, int N, int d, int C, int Hq, int Hkv, int dh) {
  Plan p;
  const int M = B * C, nout = Hkv * dh;
  const int tiles = ceil_div(M, kSimtM) * ceil_div(nout, kSimtN);
  int ns = std::max(1, ceil_div(2 * kSmTarget, tiles));
  ns = std::min(ns, std::max(1, d / 256));
  p.klen = ceil_div(ceil_div(d, ns), kSimtK) * kSimtK;
  p.nsplit = ceil_div(d, p.klen);
  const int ptiles = ceil_div(N, kRows) * B;
  int sl = std::max(1, ceil_div(2 * kSmTarget, ptiles));
  sl = std::min(sl, Hq);
  p.hps = ceil_div(Hq, sl);
  p.nslice = ceil_div(Hq, p.hps);
  return p;
}

int nj_for(int C) {
  int nj = 1;
  while (16 * nj < C) nj *= 2;
  return nj;
}

size_t proxy_smem(int dh, int NJ) {
  return sizeof(float) * ((size_t)kRows * (dh + 1) + (size_t)kKc * (16 * NJ + 1));
}

template <typename T, int NJ>
cudaError_t launch_proxy(const ProxyArgs& a, const Plan& p, const float* Kt,
                         float* part, cudaStream_t s) {
  const size_t smem = proxy_smem(a.dh, NJ);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(k_proxy<T, NJ>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
  }
  const float scale = (float)(1.0 / std::sqrt((double)a.dh));
  const dim3 grid(ceil_div(a.N, kRows), a.B, p.nslice);
  k_proxy<T, NJ><<<grid, 256, smem, s>>>(
      static_cast<const T*>(a.Q), Kt, a.N, a.C, a.Hq, a.Hkv, a.dh, p.hps, scale,
      a.A_prev, a.A_cur, a.D, p.nslice > 1 ? part : nullptr);
  if (p.nslice > 1)
    k_proxy_final<NJ><<<dim3(ceil_div(a.N, kRows), a.B), 256, 0, s>>>(
        part, p.nslice, a.B, a.N, a.C, a.Hq, a.A_prev, a.A_cur, a.D);
  return cudaGetLastError();
}

template <typename T>
cudaError_t run_typed(const ProxyArgs& a, cudaStream_t s) {
  const Plan p = make_plan(a.B, a.N, a.d, a.C, a.Hq, a.Hkv, a.dh);
  const int M = a.B * a.C, nout = a.Hkv * a.dh;
  Carver cv(a.ws);
  float* Kt = cv.take<float>((size_t)M * nout);
  float* kpart = p.nsplit > 1 ? cv.take<float>((size_t)p.nsplit * M * nout) : nullptr;
  float* apart = p.nslice > 1 ? cv.take<float>((size_t)p.nslice * a.B * a.N * a.C) : nullptr;

  const dim3 g1(ceil_div(nout, kSimtN), ceil_div(M, kSimtM), p.nsplit);
  k_ckeys<T><<<g1, 256, 0, s>>>(a.chat, static_cast<const T*>(a.Wk), M, nout,
                                a.d, p.klen, p.nsplit > 1 ? kpart : Kt);
  if (p.nsplit > 1) {
    const long count = (long)M * nout;
    k_split_reduce<<<std::min(ceil_div(count, 256), 4 * kSmTarget), 256, 0, s>>>(
        kpart, p.nsplit, count, Kt);
  }
  switch (nj_for(a.C)) {
    case 1: return launch_proxy<T, 1>(a, p, Kt, apart, s);
    case 2: return launch_proxy<T, 2>(a, p, Kt, apart, s);
    case 4: return launch_proxy<T, 4>(a, p, Kt, apart, s);
    case 8: return launch_proxy<T, 8>(a, p, Kt, apart, s);
    default: return launch_proxy<T, 16>(a, p, Kt, apart, s);
  }
}

}  // namespace

size_t proxy_ws(int B, int N, int d, int C, int Hq, int Hkv, int dh) {
  const Plan p = make_plan(B, N, d, C, Hq, Hkv, dh);
  const size_t M = (size_t)B * C, nout = (size_t)Hkv * dh;
  Carver cv(nullptr);
  cv.take<float>(M * nout);
  if (p.nsplit > 1) cv.take<float>((size_t)p.nsplit * M * nout);
  if (p.nslice > 1) cv.take<float>((size_t)p.nslice * B * N * C);
  return cv.bytes();
}

cudaError_t proxy_run(const ProxyArgs& a, cudaStream_t s) {
  return a.dtype == PS_F32 ? run_typed<float>(a, s)
                           : run_typed<__nv_bfloat16>(a, s);
}

}  // namespace ps
