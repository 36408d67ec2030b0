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
// bf16 inputs take the tensor-core path instead (C <= 256, dh % 64 == 0):
//   k_split_f32     C_hat -> bf16 hi + lo
//   tcgen05 GEMM    K~ = C_hat_hi W_k + C_hat_lo W_k, W_k streamed through
//                   TMA as MN-major tiles, split over d for small B*C (the
//                   chunks of a tile form a thread-block cluster and sum in
//                   chunk order through distributed shared memory); kept as
//                   K~_hi, K~_lo
//   tcgen05 GEMM    per (window, 128 rows, head slice): S = q K~_hi + q K~_lo
//                   in TMEM, softmax over the C columns in the epilogue (a
//                   row's columns split over 1, 2 or 4 epilogue warps), head
//                   sum in registers; the head slices of a row tile
//                   (<= 8) form a thread-block cluster that sums them in
//                   slice order through distributed shared memory, divides
//                   by Hq and takes KL.  With at least one row tile per SM,
//                   one CTA takes all heads of a row tile and keeps the head
//                   sum in TMEM (ProxyTmemEpi for C <= 128; ProxyHalvesEpi,
//                   a head's scores in two 128-column tiles, for C > 128)
// Every reduction has a fixed order, so identical inputs give identical
// bits and KL(A || A) is exactly 0.
#include <algorithm>
#include <cmath>

#include "gemm_simt.cuh"
#include "ops.h"
#include "tc_gemm.cuh"

namespace ps {
namespace {

constexpr int kRows = 16;   // window rows per proxy CTA
constexpr int kKc = 32;     // head-dim stage of the centroid keys

// 2^x by the special-function unit's approximation (PTX ex2.approx.ftz.f32:
// a relative error of a few ulp, subnormal results flushed to zero, and
// 2^-inf = +0)
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// log2(x) by the special-function unit's approximation (PTX
// lg2.approx.ftz.f32: an absolute error near 2^-22 on [0.5, 2], a relative
// error of a few ulp elsewhere)
__device__ __forceinline__ float lg2_approx(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// 1/x by the special-function unit's approximation (PTX rcp.approx.ftz.f32:
// a relative error of about an ulp)
__device__ __forceinline__ float rcp_approx(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// One KL term a ln(a / p) (a > 0), the ratio as a rcp_approx(p) and the log
// by lg2_approx: their errors, about 2^-22 absolute in the log of a ratio
// near 1, keep a row's KL within about 2^-22 of the exact sum of its terms
// (the terms' weights a sum to 1).  a == p gives exactly 0, so
// KL(A || A) = 0.
__device__ __forceinline__ float kl_term(float a, float p) {
  constexpr float kLn2 = 0.69314718055994531f;
  if (a == p) return 0.f;
  return a * (lg2_approx(a * rcp_approx(fmaxf(p, 1e-30f))) * kLn2);
}

template <typename TW>
__global__ void __launch_bounds__(256)
k_ckeys(const float* __restrict__ chat, const TW* __restrict__ Wk, int M,
        int nout, int d, int klen, float* __restrict__ out) {
  pdl_prologue();
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
  pdl_prologue();
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
  pdl_prologue();
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
  pdl_prologue();
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

int nj_for(int C);

// ------------------------------------------------------------ tensor cores
__global__ void k_split_f32(const float* __restrict__ x, long n, __nv_bfloat16* __restrict__ hi,
                            __nv_bfloat16* __restrict__ lo) {
  pdl_prologue();
  const long stride = (long)gridDim.x * blockDim.x;
  for (long i = (long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
    const float v = x[i];
    const __nv_bfloat16 h = __float2bfloat16_rn(v);
    hi[i] = h;
    lo[i] = __float2bfloat16_rn(v - __bfloat162float(h));
  }
}

__device__ __forceinline__ void split_store(__nv_bfloat16* hi, __nv_bfloat16* lo, float v) {
  const __nv_bfloat16 h = __float2bfloat16_rn(v);
  *hi = h;
  *lo = __float2bfloat16_rn(v - __bfloat162float(h));
}

// K~ tile epilogue: rows of B*C centroids, BN key columns, one d-chunk:
// split and store (several chunks: CkeysClusterEpi).
template <int BN>
struct CkeysEpi : TcEpiBase {
  int M, nkv;
  __nv_bfloat16* khi;
  __nv_bfloat16* klo;
  struct State {};
  __device__ int tiles(int) const { return (M + 127) / 128; }
  __device__ int arow(int t) const { return t * 128; }
  __device__ int bcoord(int, int n0) const { return n0; }
  __device__ void tile_done(int, int, int, int, uint8_t*, State&) const {}
  __device__ void consume(int t, int r, int n0, int, uint32_t taddr, State&) const {
    const int m = t * 128 + r;
#pragma unroll 1
    for (int c0 = 0; c0 < BN; c0 += 32) {
      float v[32];
      tc::tmem_ld32(taddr + c0, v);
      if (m >= M) continue;
      const long o = (long)m * nkv + n0 + c0;  // a multiple of 32 elements
#pragma unroll
      for (int j = 0; j < 32; j += 8) {  // 8 values: one 16-byte store each for hi and lo
        uint32_t h[4], l[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const __nv_bfloat162 hb = __floats2bfloat162_rn(v[j + 2 * q], v[j + 2 * q + 1]);
          const float2 hf = __bfloat1622float2(hb);
          const __nv_bfloat162 lb =
              __floats2bfloat162_rn(v[j + 2 * q] - hf.x, v[j + 2 * q + 1] - hf.y);
          h[q] = *reinterpret_cast<const uint32_t*>(&hb);
          l[q] = *reinterpret_cast<const uint32_t*>(&lb);
        }
        *reinterpret_cast<uint4*>(khi + o + j) = make_uint4(h[0], h[1], h[2], h[3]);
        *reinterpret_cast<uint4*>(klo + o + j) = make_uint4(l[0], l[1], l[2], l[3]);
      }
    }
  }
};

// K~ with its d-chunks in one thread-block cluster: each chunk's 128 x BN
// tile stays in shared memory; CTA z sums rows [128 z / nz, 128 (z+1) / nz)
// over the chunks in chunk order (a warp per row, 4 columns per lane) and
// stores them split into bf16 hi + lo.
template <int BN>
struct CkeysClusterEpi : CkeysEpi<BN> {
  static constexpr bool kClusterReduce = true;
  static constexpr uint32_t kLd = BN + 4;
  using State = typename CkeysEpi<BN>::State;
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
  __device__ void reduce(const float* red, int z, int nz, uint8_t*) const {
    const int t = blockIdx.y, n0 = blockIdx.x * BN;
    const int r0 = z * 128 / nz, r1 = min((z + 1) * 128 / nz, this->M - t * 128);
    cluster_rows_sum<8, 32>(red, kLd, r0, max(r0, r1), BN, nz, [&](int r, int c, float4 v) {
      const long o = (long)(t * 128 + r) * this->nkv + n0 + c;  // a multiple of 4
      const __nv_bfloat162 h0 = __floats2bfloat162_rn(v.x, v.y);
      const __nv_bfloat162 h1 = __floats2bfloat162_rn(v.z, v.w);
      const float2 f0 = __bfloat1622float2(h0), f1 = __bfloat1622float2(h1);
      const __nv_bfloat162 l0 = __floats2bfloat162_rn(v.x - f0.x, v.y - f0.y);
      const __nv_bfloat162 l1 = __floats2bfloat162_rn(v.z - f1.x, v.w - f1.y);
      *reinterpret_cast<uint2*>(this->khi + o) =
          make_uint2(*reinterpret_cast<const uint32_t*>(&h0), *reinterpret_cast<const uint32_t*>(&h1));
      *reinterpret_cast<uint2*>(this->klo + o) =
          make_uint2(*reinterpret_cast<const uint32_t*>(&l0), *reinterpret_cast<const uint32_t*>(&l1));
    });
    tc::cluster_arrive();
  }
};

// Proxy epilogue.  Tiles t = ((b * mtb + mt) * Hq + h), taken in blocks of
// hps heads per CTA.  Per head: softmax of the row's C scores (scaled by
// 1/sqrt(dh)) added to the row's head sum A (registers).  With P > 1 the P
// epilogue warps of a TMEM lane quarter each take W = BN / P columns of the
// row and combine their partial max and sum through shared memory (scratch:
// two head slots of [max | sum][128 rows][P], then KL partials [128][P]).
// The thread-block cluster of a row tile's slices then sums A in slice
// order, divides by Hq and takes KL (ProxyClusterEpi).
template <int BN, int P>
struct ProxyEpi : TcEpiBase {
  static constexpr int kEpiWarps = 4 * P;
  static constexpr int W = BN / P;  // columns per thread
  // scores kept in registers only while they fit next to the head sum A[W]:
  // with more than one epilogue warp per lane quarter (W = 64 columns of
  // scores, exponentials and sums at once would not), TMEM is re-read
  static constexpr bool kReread = W > 64 || P >= 2;
  static constexpr bool kA3D = true;
  static constexpr bool kBlocked = true;
  // two (max, sum) exchange slots of 2 x 128 x P floats
  static_assert(4 * 128 * P * 4 <= (int)TcCfg<BN, 1, 2, false>::kScratch, "scratch");
  int B, N, C, Hq, G, dh, mtb, hps, nslice;
  float scale;
  const float* A_prev;
  float* A_cur;
  float* D;
  struct State {
    float A[W];
  };
  __device__ int tiles(int) const { return B * mtb * Hq; }
  __device__ int arow(int t) const {
    const int bm = t / Hq;
    return (bm / mtb) * N + (bm % mtb) * 128;
  }
  __device__ int ahead(int t) const { return t % Hq; }
  __device__ int bcoord(int t, int) const { return (t / Hq / mtb) * C; }
  __device__ int bkoff(int t) const { return ((t % Hq) / G) * dh; }

  // One head.  Softmax with one reciprocal, in base 2: the scores are scaled
  // by log2(e) / sqrt(dh) once, so each term is one exp2 (a few ulp, far
  // inside the 1e-4 tolerance).  TMEM columns are loaded with one wait; the
  // max and the sum run as four interleaved partials.
  __device__ void head(int t, int r, int part, uint32_t taddr, float* xs, State& st) const {
    const int h = t % Hq;
    if (h % hps == 0) {
#pragma unroll
      for (int c = 0; c < W; ++c) st.A[c] = 0.f;
    }
    constexpr float kLog2e = 1.4426950408889634f;
    const float sl = scale * kLog2e;
    const int c0 = part * W;
    const uint32_t ta = taddr + c0;
    if constexpr (kReread) {  // scores re-read from TMEM in K-column chunks
      // 8 columns a load while the head sum A[W] fills most registers
      constexpr int K = 8;
      auto ld = [&](uint32_t at, uint32_t* raw) {
        if constexpr (K == 8) {
          tc::tmem_ld8_nowait(at, raw);
        } else {
#pragma unroll
          for (int k = 0; k < K; k += 32) tc::tmem_ld32_nowait(at + k, raw + k);
        }
      };
      float m2[2] = {-INFINITY, -INFINITY};
#pragma unroll
      for (int k0 = 0; k0 < W; k0 += K) {
        uint32_t raw[K];
        ld(ta + k0, raw);
        tc::tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < K; ++j)
          if (c0 + k0 + j < C) m2[j & 1] = fmaxf(m2[j & 1], __uint_as_float(raw[j]) * sl);
      }
      float m = fmaxf(m2[0], m2[1]);
      float* mx = xs + (h & 1) * (2 * 128 * P);
      if constexpr (P > 1) {
        mx[r * P + part] = m;
        epi_bar_sync_n<128 * P>();
        m = mx[r * P];
#pragma unroll
        for (int q = 1; q < P; ++q) m = fmaxf(m, mx[r * P + q]);
      }
      // each term's exp2 once: kept in the accumulator's own TMEM columns
      // (this tile's scores are not read again) for the pass below
      float s2[2] = {0.f, 0.f};
#pragma unroll
      for (int k0 = 0; k0 < W; k0 += K) {
        uint32_t raw[K];
        ld(ta + k0, raw);
        tc::tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < K; ++j) {
          const float e =
              c0 + k0 + j < C ? ex2_approx(fmaf(__uint_as_float(raw[j]), sl, -m)) : 0.f;
          s2[j & 1] += e;
          raw[j] = __float_as_uint(e);
        }
        if constexpr (K == 8) {
          tc::tmem_st8(ta + k0, raw);
        } else {
#pragma unroll
          for (int k = 0; k < K; k += 32) tc::tmem_st32(ta + k0 + k, raw + k);
        }
      }
      tc::tmem_wait_st();
      float sum = s2[0] + s2[1];
      if constexpr (P > 1) {
        float* sm = mx + 128 * P;
        sm[r * P + part] = sum;
        epi_bar_sync_n<128 * P>();
        sum = sm[r * P];
#pragma unroll
        for (int q = 1; q < P; ++q) sum += sm[r * P + q];
      }
      const float rs = 1.0f / sum;
#pragma unroll
      for (int k0 = 0; k0 < W; k0 += K) {
        uint32_t raw[K];
        ld(ta + k0, raw);
        tc::tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < K; ++j) st.A[k0 + j] = fmaf(__uint_as_float(raw[j]), rs, st.A[k0 + j]);
      }
    } else {
      uint32_t raw[W];
#pragma unroll
      for (int k0 = 0; k0 < W; k0 += 32) tc::tmem_ld32_nowait(ta + k0, raw + k0);
      tc::tmem_wait_ld();
      float e[W];
      float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int c = 0; c < W; ++c) {
        e[c] = c0 + c < C ? __uint_as_float(raw[c]) * sl : -INFINITY;
        m4[c & 3] = fmaxf(m4[c & 3], e[c]);
      }
      float m = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
      float* mx = xs + (h & 1) * (2 * 128 * P);
      if constexpr (P > 1) {
        mx[r * P + part] = m;
        epi_bar_sync_n<128 * P>();
        m = mx[r * P];
#pragma unroll
        for (int q = 1; q < P; ++q) m = fmaxf(m, mx[r * P + q]);
      }
      float s4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int c = 0; c < W; ++c) {
        e[c] = c0 + c < C ? ex2_approx(e[c] - m) : 0.f;
        s4[c & 3] += e[c];
      }
      float sum = (s4[0] + s4[1]) + (s4[2] + s4[3]);
      if constexpr (P > 1) {
        float* sm = mx + 128 * P;
        sm[r * P + part] = sum;
        epi_bar_sync_n<128 * P>();
        sum = sm[r * P];
#pragma unroll
        for (int q = 1; q < P; ++q) sum += sm[r * P + q];
      }
      const float rs = 1.0f / sum;
#pragma unroll
      for (int c = 0; c < W; ++c) st.A[c] = fmaf(e[c], rs, st.A[c]);
    }
  }
};

// The last step of a row tile whose head sum A / Hq has been staged in
// shared memory, T[r ldT + c] (nrow rows of C <= 32 kJ columns): warp ew of
// E writes rows ew, ew + E, ... to A_cur and takes their KL against A_prev,
// lane j over columns j, j + 32, ... (every warp access one contiguous run
// of a row), then a fixed shuffle tree; D = max(KL, 0), or 0 without a
// previous distribution.  kR rows at a time, all of their A_prev loads
// issued before any is used.
template <int kJ, int kR = 6>
__device__ __forceinline__ void proxy_rows_out(const float* T, int ldT, int nrow, int C,
                                               long row0, int ew, int E,
                                               const float* __restrict__ A_prev,
                                               float* __restrict__ A_cur,
                                               float* __restrict__ D) {
  const int lane = threadIdx.x & 31;
  const bool prev = A_prev != nullptr;
  for (int r = ew; r < nrow; r += kR * E) {
    float pv[kR][kJ];
#pragma unroll
    for (int u = 0; u < kR; ++u)
#pragma unroll
      for (int j = 0; j < kJ; ++j) {
        const int c = lane + 32 * j, ru = r + u * E;
        pv[u][j] = prev && ru < nrow && c < C ? __ldg(A_prev + (row0 + ru) * C + c) : 1.f;
      }
#pragma unroll
    for (int u = 0; u < kR; ++u) {
      const int ru = r + u * E;
      if (ru >= nrow) break;  // warp-uniform
      const long g = (row0 + ru) * C;
      float kl = 0.f;
#pragma unroll
      for (int j = 0; j < kJ; ++j) {
        const int c = lane + 32 * j;
        if (c < C) {
          const float av = T[ru * ldT + c];
          A_cur[g + c] = av;
          if (prev && av > 0.f) kl += kl_term(av, pv[u][j]);
        }
      }
      kl = warp_sum(kl);
      if (lane == 0) D[row0 + ru] = prev ? fmaxf(kl, 0.f) : 0.f;
    }
  }
}

// Row stride (floats) of the staged A: C rounded up to 8, plus 4, so that the
// 16-byte stores of 8 consecutive rows at one column fall in distinct banks.
__host__ __device__ constexpr int proxy_stage_ld(int C) { return ((C + 7) & ~7) + 4; }

// The previous distributions of a row tile (nrow rows of C floats from row
// row0, one contiguous block) into L2 ahead of their use: the 16-byte
// aligned part of the block, by one thread.
__device__ __forceinline__ void proxy_prefetch_prev(const float* A_prev, long row0, int nrow,
                                                    int C) {
  if (A_prev == nullptr || nrow <= 0) return;
  const uintptr_t b0 = reinterpret_cast<uintptr_t>(A_prev + row0 * C);
  const uintptr_t b1 = reinterpret_cast<uintptr_t>(A_prev + (row0 + nrow) * C);
  const uintptr_t a0 = (b0 + 15) & ~static_cast<uintptr_t>(15);
  const uintptr_t a1 = b1 & ~static_cast<uintptr_t>(15);
  if (a1 > a0) tc::bulk_prefetch_l2(reinterpret_cast<const void*>(a0), (uint32_t)(a1 - a0));
}

// A thread's n (a multiple of 4) consecutive head-sum columns from c0 on,
// times inv = RN(1 / Hq) (A / Hq exactly when Hq is a power of two, else
// within an ulp), into row r of the staged tile; columns at or past C are
// left out.
template <int n>
__device__ __forceinline__ void proxy_stage_cols(float* T, int ldT, int r, int c0, int C,
                                                 const uint32_t* a, float inv) {
  static_assert(n % 4 == 0, "whole float4s");
#pragma unroll
  for (int j = 0; j < n; j += 4) {
    const int c = c0 + j;
    const float4 v = make_float4(__uint_as_float(a[j]) * inv, __uint_as_float(a[j + 1]) * inv,
                                 __uint_as_float(a[j + 2]) * inv, __uint_as_float(a[j + 3]) * inv);
    if (c + 4 <= C) {
      *reinterpret_cast<float4*>(T + r * ldT + c) = v;
    } else {
      if (c < C) T[r * ldT + c] = v.x;
      if (c + 1 < C) T[r * ldT + c + 1] = v.y;
      if (c + 2 < C) T[r * ldT + c + 2] = v.z;
    }
  }
}

// Proxy epilogue with the head sum in TMEM, for C <= 128 and one CTA per
// row tile taking all its heads (enough row tiles to fill the GPU): the two
// accumulator buffers (2 BN columns) and the head sum A (BN columns, fp32)
// in TMEM.  Sixteen epilogue warps: the four of a TMEM lane quarter take
// W = BN / 4 columns of their 32 rows and meet through shared memory for a
// row's max and sum (fixed order).  consume(): the scores, the row max m,
// e = 2^(s' - m) kept in registers, the row sum (s' = score / sqrt(dh) in
// base 2).  tile_done(), which the engine calls once the accumulator is
// handed back to the MMA, adds e / sum into A in TMEM, so the next head's
// MMAs run under it; after the row tile's last head (after_tiles, every
// warp of the CTA): A / Hq staged row-major in the idle stage ring, A_cur
// stored and KL taken against A_prev (prefetched into L2 three heads
// before) a row per warp.
template <int BN>
struct ProxyTmemEpi : TcEpiBase {
  static constexpr int kEpiWarps = 16;
  static constexpr int P = 4;            // epilogue warps per lane quarter
  static constexpr int W = BN / P;       // columns a thread takes
  static constexpr int kExtraCols = BN;
  static constexpr bool kAfterTiles = true;
  static constexpr bool kA3D = true;
  static constexpr bool kBlocked = true;
  static_assert(W % 8 == 0 && W <= 32, "part width");
  // a (max, sum) exchange of 2 x 128 x P floats
  static_assert(2 * 128 * P * 4 <= (int)TcCfg<BN, 1, 2, false>::kScratch, "scratch");
  int B, N, C, Hq, G, dh, mtb;
  float scale;
  const float* A_prev;
  float* A_cur;
  float* D;
  struct State {
    float e[W];  // this head's exponentials
    float s;
    uint32_t extra;
  };
  __device__ int tiles(int) const { return B * mtb * Hq; }
  __device__ int arow(int t) const {
    const int bm = t / Hq;
    return (bm / mtb) * N + (bm % mtb) * 128;
  }
  __device__ int ahead(int t) const { return t % Hq; }
  __device__ int bcoord(int t, int) const { return (t / Hq / mtb) * C; }
  __device__ int bkoff(int t) const { return ((t % Hq) / G) * dh; }

  // the row's value from the four warps of a lane quarter (slot: 128 x 4
  // floats of the scratch), combined in warp order
  template <bool MAX>
  __device__ __forceinline__ float row_combine(float v, float* slot, int r, int q) const {
    slot[r * P + q] = v;
    epi_bar_sync_n<32 * kEpiWarps>();
    float x = slot[r * P];
#pragma unroll
    for (int k = 1; k < P; ++k) x = MAX ? fmaxf(x, slot[r * P + k]) : x + slot[r * P + k];
    return x;
  }

  __device__ void consume_part(int, int r, int q, int, int, uint32_t taddr, uint8_t* scratch,
                               State& st) const {
    constexpr float kLog2e = 1.4426950408889634f;
    const float sl = scale * kLog2e;
    const int cq = q * W;  // this thread's first score column
    float* xs = reinterpret_cast<float*>(scratch);
    float m = -INFINITY;
#pragma unroll
    for (int k = 0; k < W; k += 8) {
      uint32_t raw[8];
      tc::tmem_ld8_nowait(taddr + cq + k, raw);
      tc::tmem_wait_ld();
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float v = cq + k + j < C ? __uint_as_float(raw[j]) * sl : -INFINITY;
        st.e[k + j] = v;
        m = fmaxf(m, v);
      }
    }
    m = row_combine<true>(m, xs, r, q);
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < W; ++j) {
      st.e[j] = ex2_approx(st.e[j] - m);
      s += st.e[j];
    }
    st.s = row_combine<false>(s, xs + 128 * P, r, q);
  }

  __device__ void tile_done_part(int t, int r, int q, int, int, uint8_t*, State& st) const {
    const int h = t % Hq;
    if (h == max(Hq - 3, 0) && r == 0 && q == 0) {  // A_prev needed three heads on
      const int bm = t / Hq, i0 = (bm % mtb) * 128;
      proxy_prefetch_prev(A_prev, (long)(bm / mtb) * N + i0, min(128, N - i0), C);
    }
    const float f = 1.0f / st.s;
    const uint32_t at = st.extra + q * W;
#pragma unroll
    for (int k = 0; k < W; k += 8) {
      uint32_t a[8];
      if (h == 0) {
#pragma unroll
        for (int j = 0; j < 8; ++j) a[j] = __float_as_uint(st.e[k + j] * f);
      } else {
        tc::tmem_ld8_nowait(at + k, a);
        tc::tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 8; ++j)
          a[j] = __float_as_uint(fmaf(st.e[k + j], f, __uint_as_float(a[j])));
      }
      tc::tmem_st8(at + k, a);
    }
    tc::tmem_wait_st();
  }

  // After the CTA's tiles, every warp: the epilogue warps stage A / Hq from
  // TMEM in the idle stage ring (row-major), then all warps store it and
  // take the KL a row per warp (proxy_rows_out)
  __device__ void after_tiles(int t_begin, uint32_t tmem) const {
    constexpr int ldT = proxy_stage_ld(BN);
    static_assert(128 * ldT * 4 <= (int)(TcCfg<BN, 1, 2, false>::kStages *
                                          TcCfg<BN, 1, 2, false>::kStage), "staged A > ring");
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int bm = t_begin / Hq, b = bm / mtb, i0 = (bm % mtb) * 128;
    float* T = reinterpret_cast<float*>(tc_ring_base());
    if (warp >= 2) {
      const int quarter = warp & 3, q = (warp - 2) >> 2;
      const uint32_t at =
          tmem + kAccBufs * BN + (static_cast<uint32_t>(quarter * 32) << 16) + q * W;
      tc::fence_after_sync();
      uint32_t raw[W];
      if constexpr (W == 32) {
        tc::tmem_ld32_nowait(at, raw);
      } else if constexpr (W == 16) {
        tc::tmem_ld16_nowait(at, raw);
      } else {
        tc::tmem_ld8_nowait(at, raw);
      }
      tc::tmem_wait_ld();
      proxy_stage_cols<W>(T, proxy_stage_ld(C), quarter * 32 + lane, q * W, C, raw,
                          1.0f / (float)Hq);
    }
    __syncthreads();
    static_assert(BN % 32 == 0, "whole 32-column runs");
    proxy_rows_out<BN / 32>(T, proxy_stage_ld(C), min(128, N - i0), C, (long)b * N + i0, warp,
                            (int)(blockDim.x >> 5), A_prev, A_cur, D);
  }
};

// Proxy epilogue for C in (128, 256] with one CTA per row tile taking all
// its heads, a head's scores in two 128-column parts (two MMA tiles, each in
// its own accumulator, double-buffered) and the head sum A (256 columns,
// fp32) in the rest of TMEM.  Eight epilogue warps, two per TMEM lane
// quarter (so 168 registers a thread), each taking W = 64 columns of each
// part of its 32 rows in two 32-column chunks:
//   consume (either part): per chunk the max m of its scores and
//           e = 2^(s' - m), kept in registers, with their sum s; the part's
//           accumulator goes back to the MMA as soon as it returns, so the
//           next head's MMAs run under the rest of this head's epilogue;
//   tile_done after part 1: the two warps of a row exchange their chunks'
//           (m, s) through shared memory once (fixed order): M = max m,
//           S = sum s 2^(m - M); then A += e 2^(m - M) / S for every chunk
//           (s' = score / sqrt(dh) in base 2).
// After the row tile's last head (after_tiles, every warp of the CTA): A / Hq
// staged row-major in the idle stage ring, then A_cur stored and KL taken
// against A_prev a row per warp, both with contiguous warp accesses; A_prev
// is prefetched into L2 three heads before.  The softmax terms are those of
// one pass over the row up to rounding.
struct ProxyHalvesEpi : TcEpiBase {
  static constexpr int P = 2;          // epilogue warps per lane quarter
  static constexpr int kEpiWarps = 4 * P;
  static constexpr int BN_T = 128;     // columns of a part (one MMA tile)
  static constexpr int W = BN_T / P;   // columns a thread takes of each part
  static constexpr int NCH = W / 32;   // 32-column chunks of a thread's part
  static constexpr int kExtraCols = 2 * BN_T;
  static constexpr bool kAfterTiles = true;
  static constexpr bool kA3D = true;
  static constexpr bool kBlocked = true;
  static_assert(W % 32 == 0, "32-column chunks");
  // two exchange slots of 128 x P threads x NCH float4 (m0, s0, m1, s1)
  static constexpr int kSlot = 128 * P * 4 * NCH;  // floats
  static_assert(2 * kSlot * 4 <= (int)TcCfg<BN_T, 1, 2, false>::kScratch, "scratch");
  int B, N, C, Hq, G, dh, mtb;
  float scale;
  const float* A_prev;
  float* A_cur;
  float* D;
  struct State {
    float e[2][W];  // each part's exponentials, each chunk against its own max
    float m[2][NCH], s[2][NCH];
    uint32_t extra;
  };
  __device__ int tiles(int) const { return B * mtb * Hq * 2; }
  __device__ int arow(int t) const {
    const int bm = t / (Hq * 2);
    return (bm / mtb) * N + (bm % mtb) * 128;
  }
  __device__ int ahead(int t) const { return (t / 2) % Hq; }
  __device__ int bcoord(int t, int) const { return (t / (Hq * 2) / mtb) * C + (t % 2) * BN_T; }
  __device__ int bkoff(int t) const { return (((t / 2) % Hq) / G) * dh; }

  // 32 scores v (raw TMEM words; n < 32: only the first n count, n >= 1):
  // m = sl * max v, e = 2^(v sl - m) in place, their sum
  template <bool kFull>
  __device__ __forceinline__ void exp_chunk(uint32_t* v, int n, float sl, float& m,
                                            float& sum) const {
    if constexpr (!kFull) {
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (j >= n) v[j] = __float_as_uint(-INFINITY);
    }
    float mx[8];
#pragma unroll
    for (int j = 0; j < 8; ++j)
      mx[j] = fmaxf(fmaxf(__uint_as_float(v[j]), __uint_as_float(v[j + 8])),
                    fmaxf(__uint_as_float(v[j + 16]), __uint_as_float(v[j + 24])));
#pragma unroll
    for (int j = 0; j < 4; ++j) mx[j] = fmaxf(mx[j], mx[j + 4]);
    m = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * sl;
    float sp[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const float e = ex2_approx(fmaf(__uint_as_float(v[j]), sl, -m));
      sp[j & 3] += e;
      v[j] = __float_as_uint(e);
    }
    sum = (sp[0] + sp[1]) + (sp[2] + sp[3]);
  }

  __device__ void consume_part(int t, int, int q, int, int, uint32_t taddr, uint8_t*,
                               State& st) const {
    // the part as a constant, so that State stays in registers
    if (t % 2 == 0)
      part<0>(q, taddr, st);
    else
      part<1>(q, taddr, st);
  }

  template <int p>
  __device__ __forceinline__ void part(int q, uint32_t taddr, State& st) const {
    constexpr float kLog2e = 1.4426950408889634f;
    const float sl = scale * kLog2e;
    uint32_t v[W];
#pragma unroll
    for (int k = 0; k < NCH; ++k) tc::tmem_ld32_nowait(taddr + q * W + 32 * k, v + 32 * k);
    tc::tmem_wait_ld();
#pragma unroll
    for (int k = 0; k < NCH; ++k) {
      // columns p 128 + q W + 32 k ..; a chunk past column C is left out
      // (max -inf, sum 0); part 0 is whole (C > 128)
      const int n = p == 0 ? 32 : C - BN_T - q * W - 32 * k;
      st.m[p][k] = -INFINITY;
      st.s[p][k] = 0.f;
      if (n >= 32)
        exp_chunk<true>(v + 32 * k, 32, sl, st.m[p][k], st.s[p][k]);
      else if (n > 0)
        exp_chunk<false>(v + 32 * k, n, sl, st.m[p][k], st.s[p][k]);
    }
#pragma unroll
    for (int j = 0; j < W; ++j) st.e[p][j] = __uint_as_float(v[j]);
  }

  __device__ void tile_done_part(int t, int r, int q, int, int, uint8_t* scratch,
                                 State& st) const {
    if (t % 2 == 0) return;  // tile-uniform: after a head's part 1
    const int h = (t / 2) % Hq;
    if (h == max(Hq - 3, 0) && r == 0 && q == 0) {  // A_prev needed three heads on
      const int bm = t / (Hq * 2), i0 = (bm % mtb) * 128;
      proxy_prefetch_prev(A_prev, (long)(bm / mtb) * N + i0, min(128, N - i0), C);
    }
    // the row's max and sum from the chunks of its P threads, in order
    float4* xs = reinterpret_cast<float4*>(reinterpret_cast<float*>(scratch) + (h & 1) * kSlot);
#pragma unroll
    for (int k = 0; k < NCH; ++k)
      xs[(r * P + q) * NCH + k] = make_float4(st.m[0][k], st.s[0][k], st.m[1][k], st.s[1][k]);
    epi_bar_sync_n<32 * kEpiWarps>();
    float mr = -INFINITY;
#pragma unroll
    for (int k = 0; k < P * NCH; ++k) {
      const float4 x = xs[r * P * NCH + k];
      mr = fmaxf(mr, fmaxf(x.x, x.z));
    }
    float sr = 0.f;
#pragma unroll
    for (int k = 0; k < P * NCH; ++k) {  // a left-out chunk adds 0 x 2^-inf = 0
      const float4 x = xs[r * P * NCH + k];
      sr = fmaf(x.y, ex2_approx(x.x - mr), sr);
      sr = fmaf(x.w, ex2_approx(x.z - mr), sr);
    }
    const float rs = 1.0f / sr;
    const bool first = h == 0;
#pragma unroll
    for (int p = 0; p < 2; ++p) {
#pragma unroll
      for (int k = 0; k < NCH; ++k) {
        // columns at or past C of A are never read: a left-out chunk's
        // weight only has to be finite
        const float f = st.m[p][k] == -INFINITY ? 0.f : ex2_approx(st.m[p][k] - mr) * rs;
#pragma unroll
        for (int hh = 0; hh < 32; hh += 16) {
          const uint32_t at = st.extra + p * BN_T + q * W + 32 * k + hh;
          uint32_t a[16];
          if (first) {
#pragma unroll
            for (int j = 0; j < 16; ++j) a[j] = __float_as_uint(st.e[p][32 * k + hh + j] * f);
          } else {
            tc::tmem_ld16_nowait(at, a);
            tc::tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 16; ++j)
              a[j] = __float_as_uint(fmaf(st.e[p][32 * k + hh + j], f, __uint_as_float(a[j])));
          }
          tc::tmem_st16(at, a);
        }
      }
    }
    tc::tmem_wait_st();
  }

  // After the CTA's tiles, every warp: the epilogue warps stage A / Hq from
  // TMEM in the idle stage ring (row-major), then all warps store it and
  // take the KL a row per warp (proxy_rows_out)
  __device__ void after_tiles(int t_begin, uint32_t tmem) const {
    constexpr int ldT = proxy_stage_ld(2 * BN_T);
    static_assert(128 * ldT * 4 <= (int)(TcCfg<BN_T, 1, 2, false>::kStages *
                                          TcCfg<BN_T, 1, 2, false>::kStage), "staged A > ring");
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int bm = t_begin / (Hq * 2), b = bm / mtb, i0 = (bm % mtb) * 128;
    float* T = reinterpret_cast<float*>(tc_ring_base());
    const int ld = proxy_stage_ld(C);
    if (warp >= 2) {
      const int quarter = warp & 3, q = (warp - 2) >> 2;
      const uint32_t extra = tmem + kAccBufs * BN_T + (static_cast<uint32_t>(quarter * 32) << 16);
      tc::fence_after_sync();
#pragma unroll 1
      for (int k = 0; k < 2 * W; k += 64) {  // 64 columns of one part at a time
        const int c0 = (k / W) * BN_T + q * W + k % W;
        uint32_t a[64];
        tc::tmem_ld32_nowait(extra + c0, a);
        tc::tmem_ld32_nowait(extra + c0 + 32, a + 32);
        tc::tmem_wait_ld();
        proxy_stage_cols<64>(T, ld, quarter * 32 + lane, c0, C, a, 1.0f / (float)Hq);
      }
    }
    __syncthreads();
    proxy_rows_out<2 * BN_T / 32>(T, ld, min(128, N - i0), C, (long)b * N + i0, warp,
                                  (int)(blockDim.x >> 5), A_prev, A_cur, D);
  }
};

// Head slices of one row tile inside one thread-block cluster: CTA z runs
// heads [z hps, (z+1) hps) of row tile blockIdx.y and leaves its head sum in
// shared memory; then CTA z finishes rows [128 z / Z, 128 (z+1) / Z), one
// warp per row: the slices' sums in slice order, A = sum / Hq, KL.
template <int BN, int P>
struct ProxyClusterEpi : ProxyEpi<BN, P> {
  using Base = ProxyEpi<BN, P>;
  static constexpr bool kBlocked = false;
  static constexpr bool kClusterReduce = true;
  static constexpr bool kZSplitsK = false;
  static constexpr uint32_t kLd = BN + 4;
  using State = typename Base::State;
  __device__ bool tile_range(int, int* tb, int* te, int* ts) const {
    *tb = blockIdx.y * this->Hq + blockIdx.z * this->hps;
    *te = *tb + this->hps;
    *ts = 1;
    return true;
  }
  __device__ void stash(int part, const State& st, float* red_row) const {
    if (red_row == nullptr) return;
#pragma unroll
    for (int c = 0; c < Base::W; c += 4)
      *reinterpret_cast<float4*>(red_row + part * Base::W + c) =
          make_float4(st.A[c], st.A[c + 1], st.A[c + 2], st.A[c + 3]);
  }
  __device__ void consume_red(int t, int r, int, int, uint32_t taddr, State& st,
                              float* red_row) const {
    this->head(t, r, 0, taddr, nullptr, st);
    stash(0, st, red_row);
  }
  __device__ void consume_red_part(int t, int r, int part, int, int, uint32_t taddr,
                                   uint8_t* scratch, State& st, float* red_row) const {
    this->head(t, r, part, taddr, reinterpret_cast<float*>(scratch), st);
    stash(part, st, red_row);
  }
  // with one epilogue warp per TMEM quarter (P == 1) the scratch is free:
  // the previous distributions of this CTA's rows are staged there while the
  // mainloop runs, when they fit
  __device__ bool early_prev(int nrow) const {
    return P == 1 && this->A_prev != nullptr && nrow * this->C * 4 <= (int)TcCfg<BN, 1, 2, false>::kScratch;
  }
  __device__ void rows_of(int z, int nz, int mt, int* r0, int* nrow) const {
    const int a = z * 128 / nz, e = (z + 1) * 128 / nz;
    *r0 = a;
    *nrow = max(0, min(e, this->N - mt * 128) - a);
  }
  __device__ void prefetch(uint8_t* scratch, int i, int n) const {
    const int bm = blockIdx.y, b = bm / this->mtb, mt = bm % this->mtb;
    int r0, nrow;
    rows_of(blockIdx.z, gridDim.z, mt, &r0, &nrow);
    if (!early_prev(nrow)) return;
    const float* src = this->A_prev + ((long)b * this->N + mt * 128 + r0) * this->C;
    float* dst = reinterpret_cast<float*>(scratch);
    for (int j = i; j < nrow * this->C; j += n) dst[j] = __ldg(src + j);
  }
  __device__ void reduce(const float* red, int z, int nz, uint8_t* scratch) const {
    const int bm = blockIdx.y, b = bm / this->mtb, mt = bm % this->mtb;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
    int r0, nrow;
    rows_of(z, nz, mt, &r0, &nrow);
    const int C = this->C, N = this->N;
    const int i0 = mt * 128 + r0;
    const long row0 = (long)b * N + i0;
    const float hq = (float)this->Hq;
    // the previous distributions of this CTA's rows (one contiguous block):
    // staged early in the scratch, or here with 16-byte loads past the
    // cluster-read result (this CTA's own shared memory)
    const bool early = early_prev(nrow);
    float* s_prev = early ? reinterpret_cast<float*>(scratch) : const_cast<float*>(red) + 128 * kLd;
    const bool prev = this->A_prev != nullptr;
    using Cfg = TcCfg<BN, 1, 2, false>;
    // staged when it fits in the ring past the result, else read in place
    const bool staged = early || (128 * kLd + nrow * C) * 4 <= Cfg::kStages * Cfg::kStage;
    if (prev && staged && !early) {
      const float* src = this->A_prev + row0 * C;
      const int n = nrow * C;
      if ((reinterpret_cast<uintptr_t>(src) & 15) == 0) {
        const int n4 = n >> 2;
#pragma unroll 4
        for (int j = threadIdx.x; j < n4; j += blockDim.x)
          reinterpret_cast<float4*>(s_prev)[j] = __ldg(reinterpret_cast<const float4*>(src) + j);
        for (int j = (n4 << 2) + threadIdx.x; j < n; j += blockDim.x) s_prev[j] = __ldg(src + j);
      } else {
#pragma unroll 4
        for (int j = threadIdx.x; j < n; j += blockDim.x) s_prev[j] = __ldg(src + j);
      }
    }
    // head-slice sums replace this CTA's own rows, which only it reads
    float* own = const_cast<float*>(red);
    cluster_rows_sum<8>(red, kLd, r0, r0 + nrow, (C + 3) & ~3, nz, [&](int r, int c, float4 v) {
      *reinterpret_cast<float4*>(own + r * kLd + c) = v;
    });
    tc::cluster_arrive();
    __syncthreads();
    for (int r = r0 + warp; r < r0 + nrow; r += nwarps) {
      const long row = row0 + (r - r0);
      float kl = 0.f;
#pragma unroll
      for (int j = 0; j < BN / 32; ++j) {
        const int c = lane + 32 * j;
        if (c < C) {
          const float a = own[r * kLd + c] / hq;
          this->A_cur[row * C + c] = a;
          if (prev && a > 0.f) {
            const float ap = staged ? s_prev[(r - r0) * C + c] : this->A_prev[row * C + c];
            kl += a * logf(a / fmaxf(ap, 1e-30f));
          }
        }
      }
      kl = warp_sum(kl);
      if (lane == 0) this->D[row] = prev ? fmaxf(kl, 0.f) : 0.f;
    }
  }
};

struct TcPlan {
  bool ok;
  int BN, mtb, nslice, hps;             // proxy
  int ck_BN, ck_mt, ck_nt, ck_nz, ck_kpc, KB;  // centroid keys
};

TcPlan tc_plan(int dtype, int B, int N, int d, int C, int Hq, int Hkv, int dh) {
  TcPlan p{};
  const int nkv = Hkv * dh;
  p.ok = dtype == PS_BF16 && C <= 256 && dh % 64 == 0 && nkv % 64 == 0;
  if (!p.ok) return p;
  p.BN = C <= 32 ? 32 : (C <= 64 ? 64 : (C <= 128 ? 128 : 256));
  p.mtb = ceil_div(N, 128);
  // head slices of a row tile share one thread-block cluster: <= 8
  const int want = std::min(8, std::max(1, ceil_div(kSmTarget, B * p.mtb)));
  p.nslice = 1;
  for (int sl = std::min(want, Hq); sl >= 1; --sl)
    if (Hq % sl == 0) { p.nslice = sl; break; }
  p.hps = Hq / p.nslice;
  p.KB = ceil_div(d, 64);
  // centroid keys: column tile BN and d split Z by a simple cost, waves x
  // bytes one CTA streams; a split's Z CTAs form a cluster, and the clusters
  // the GPU holds at once are counted by GPC (tc_cluster_capacity)
  p.ck_mt = ceil_div(B * C, 128);
  double best = 0.0;
  for (int bn : {256, 128, 64}) {
    if (nkv % bn != 0) continue;
    const int nt = nkv / bn, groups = p.ck_mt * nt;
    for (int z = 1; z <= std::min(8, p.KB); ++z) {
      const int kpc = ceil_div(p.KB, z);
      if (ceil_div(p.KB, kpc) != z) continue;  // every chunk non-empty
      const int cap = z == 1 ? kSmTarget : tc_cluster_capacity(z);
      if (cap <= 0) continue;
      const double waves = ceil_div(groups, cap);
      const double arows = B * C <= 64 ? 64.0 : 128.0;
      const double cost = waves * kpc * (2.0 * arows * 64 * 2 + (double)bn * 64 * 2);
      if (best == 0.0 || cost < best) {
        best = cost;
        p.ck_BN = bn;
        p.ck_nt = nt;
        p.ck_kpc = kpc;
        p.ck_nz = z;
      }
    }
  }
  return p;
}

struct TcWs {
  __nv_bfloat16 *chi, *clo, *khi, *klo;
};

TcWs tc_carve(void* base, const TcPlan& p, int B, int N, int d, int C, int nkv, size_t* bytes) {
  Carver cv(base);
  TcWs w{};
  w.chi = cv.take<__nv_bfloat16>((size_t)B * C * d);
  w.clo = cv.take<__nv_bfloat16>((size_t)B * C * d);
  w.khi = cv.take<__nv_bfloat16>((size_t)B * C * nkv);
  w.klo = cv.take<__nv_bfloat16>((size_t)B * C * nkv);
  if (bytes) *bytes = cv.bytes();
  return w;
}

template <int BN>
cudaError_t proxy_tc(const ProxyArgs& a, const TcPlan& p, cudaStream_t s) {
  const int nkv = a.Hkv * a.dh;
  const TcWs w = tc_carve(a.ws, p, a.B, a.N, a.d, a.C, nkv, nullptr);
  const long nc = (long)a.B * a.C * a.d;
  launch_pdl(k_split_f32, std::min(ceil_div(nc, 256), 4 * kSmTarget), 256, 0, s, a.chat, nc, w.chi,
                                                                          w.clo);
  {
    TcMaps maps;
    // with at most 64 centroid rows the tiles bring 64 rows (a quarter less to stream)
    const int a_rows = a.B * a.C <= 64 ? 64 : 128;
    if (!make_tmap_bf16_2d(&maps.a[0], w.chi, a.d, (uint64_t)a.B * a.C, (uint64_t)a.d * 2,
                           64, a_rows) ||
        !make_tmap_bf16_2d(&maps.a[1], w.clo, a.d, (uint64_t)a.B * a.C, (uint64_t)a.d * 2,
                           64, a_rows) ||
        !make_tmap_bf16_2d(&maps.b[0], a.Wk, nkv, a.d, (uint64_t)nkv * 2, 64, 64))
      return cudaErrorInvalidValue;
    maps.b[1] = maps.b[0];
    TcShape sh{a.B * a.C, nullptr, p.KB, p.ck_kpc, a.status, INT_MAX, 0, a_rows};
    // without a d split, at most one CTA per SM walks the row tiles of its
    // column tile (the epilogue of one tile under the MMAs of the next)
    const int gy = p.ck_nz > 1 ? p.ck_mt
                               : std::max(1, std::min(p.ck_mt, (a.num_sms > 0 ? a.num_sms
                                                                               : kSmTarget) /
                                                                   p.ck_nt));
    const dim3 grid(p.ck_nt, gy, p.ck_nz);
    const int M = a.B * a.C;
    cudaError_t e;
    if (p.ck_nz > 1) {  // d-chunks summed inside a thread-block cluster
      switch (p.ck_BN) {
        case 256: e = launch_tc_gemm<256, 2, 1, true>(maps, sh, CkeysClusterEpi<256>{{{}, M, nkv, w.khi, w.klo}}, grid, s); break;
        case 128: e = launch_tc_gemm<128, 2, 1, true>(maps, sh, CkeysClusterEpi<128>{{{}, M, nkv, w.khi, w.klo}}, grid, s); break;
        default: e = launch_tc_gemm<64, 2, 1, true>(maps, sh, CkeysClusterEpi<64>{{{}, M, nkv, w.khi, w.klo}}, grid, s); break;
      }
    } else {
      switch (p.ck_BN) {
        case 256: e = launch_tc_gemm<256, 2, 1, true>(maps, sh, CkeysEpi<256>{{}, M, nkv, w.khi, w.klo}, grid, s); break;
        case 128: e = launch_tc_gemm<128, 2, 1, true>(maps, sh, CkeysEpi<128>{{}, M, nkv, w.khi, w.klo}, grid, s); break;
        default: e = launch_tc_gemm<64, 2, 1, true>(maps, sh, CkeysEpi<64>{{}, M, nkv, w.khi, w.klo}, grid, s); break;
      }
    }
    if (e != cudaSuccess) return e;
  }
  TcMaps maps;
  if (!make_tmap_bf16_3d(&maps.a[0], a.Q, a.dh, a.Hq, (uint64_t)a.B * a.N,
                         (uint64_t)a.dh * 2, (uint64_t)a.Hq * a.dh * 2, 64, 128) ||
      !make_tmap_bf16_2d(&maps.b[0], w.khi, nkv, (uint64_t)a.B * a.C, (uint64_t)nkv * 2, 64,
                         BN) ||
      !make_tmap_bf16_2d(&maps.b[1], w.klo, nkv, (uint64_t)a.B * a.C, (uint64_t)nkv * 2, 64,
                         BN))
    return cudaErrorInvalidValue;
  maps.a[1] = maps.a[0];
  TcShape sh{a.B * a.N, nullptr, a.dh / 64, a.dh / 64, a.status, INT_MAX};
  // columns of a row split over P epilogue warps per lane quarter: two for
  // BN >= 128 (2 + 8 warps: the register file is allotted in 4-warp steps,
  // so 12 warps' worth, 168 registers a thread, room for a 128-column head
  // sum; 16 epilogue warps would get 96 and spill it)
  constexpr int P = BN > 64 ? 2 : 1;
  const float scale = (float)(1.0 / std::sqrt((double)a.dh));
  if (p.nslice == 1) {  // a CTA per row tile, the head sum in TMEM
    if constexpr (BN == 256) {  // two 128-column parts
      TcMaps m2 = maps;
      if (!make_tmap_bf16_2d(&m2.b[0], w.khi, nkv, (uint64_t)a.B * a.C, (uint64_t)nkv * 2, 64,
                             128) ||
          !make_tmap_bf16_2d(&m2.b[1], w.klo, nkv, (uint64_t)a.B * a.C, (uint64_t)nkv * 2, 64,
                             128))
        return cudaErrorInvalidValue;
      ProxyHalvesEpi he{{}, a.B, a.N, a.C, a.Hq, a.Hq / a.Hkv, a.dh, p.mtb, scale, a.A_prev,
                        a.A_cur, a.D};
      return launch_tc_gemm<128, 1, 2, false>(m2, sh, he, dim3(1, a.B * p.mtb, 1), s);
    } else {
      ProxyTmemEpi<BN> te{{}, a.B, a.N, a.C, a.Hq, a.Hq / a.Hkv, a.dh, p.mtb, scale, a.A_prev,
                          a.A_cur, a.D};
      return launch_tc_gemm<BN, 1, 2, false>(maps, sh, te, dim3(1, a.B * p.mtb, 1), s);
    }
  }
  ProxyEpi<BN, P> epi{{}, a.B, a.N, a.C, a.Hq, a.Hq / a.Hkv, a.dh, p.mtb, p.hps, p.nslice,
                      scale, a.A_prev, a.A_cur, a.D};
  ProxyClusterEpi<BN, P> cepi{epi};
  return launch_tc_gemm<BN, 1, 2, false>(maps, sh, cepi, dim3(1, a.B * p.mtb, p.nslice), s);
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
  launch_pdl(k_proxy<T, NJ>, grid, 256, smem, s, 
      static_cast<const T*>(a.Q), Kt, a.N, a.C, a.Hq, a.Hkv, a.dh, p.hps, scale,
      a.A_prev, a.A_cur, a.D, p.nslice > 1 ? part : nullptr);
  if (p.nslice > 1)
    launch_pdl(k_proxy_final<NJ>, dim3(ceil_div(a.N, kRows), a.B), 256, 0, s, 
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
  launch_pdl(k_ckeys<T>, g1, 256, 0, s, a.chat, static_cast<const T*>(a.Wk), M, nout,
                                a.d, p.klen, p.nsplit > 1 ? kpart : Kt);
  if (p.nsplit > 1) {
    const long count = (long)M * nout;
    launch_pdl(k_split_reduce, std::min(ceil_div(count, 256), 4 * kSmTarget), 256, 0, s, 
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
  size_t simt = cv.bytes(), tcb = 0;
  // the tensor-core plan applies to bf16 inputs; size for whichever is larger
  const TcPlan q = tc_plan(PS_BF16, B, N, d, C, Hq, Hkv, dh);
  if (q.ok) tc_carve(nullptr, q, B, N, d, C, Hkv * dh, &tcb);
  return std::max(simt, tcb);
}

cudaError_t proxy_run(const ProxyArgs& a, cudaStream_t s) {
  const TcPlan p = tc_plan(a.dtype, a.B, a.N, a.d, a.C, a.Hq, a.Hkv, a.dh);
  if (p.ok) {
    switch (p.BN) {
      case 32: return proxy_tc<32>(a, p, s);
      case 64: return proxy_tc<64>(a, p, s);
      case 128: return proxy_tc<128>(a, p, s);
      default: return proxy_tc<256>(a, p, s);
    }
  }
  return a.dtype == PS_F32 ? run_typed<float>(a, s)
                           : run_typed<__nv_bfloat16>(a, s);
}

}  // namespace ps
