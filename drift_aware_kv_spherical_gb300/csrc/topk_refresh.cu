// a5: top-k most-drifting clusters with position compaction, and
// a6: sparse K/V refresh of the selected positions.
//
// [Polestar §2.A, sparse updates]: the top-k clusters with the largest drift
// are identified and a sparse forward pass on only their positions refreshes
// the matching KV-cache entries.
#include <algorithm>
#include <climits>

#include "gemm_simt.cuh"
#include "ops.h"
#include "tc_gemm.cuh"

namespace ps {
namespace {

constexpr int kStage = 2048;

// One CTA of 1024 threads per window.  Thread c owns cluster c: its drift
// sum runs in fp64 over members in ascending position order; its rank is the
// number of clusters that beat it (higher mean, or equal mean and lower
// index).  Positions are compacted with a block scan, ascending.
__global__ void __launch_bounds__(1024)
k_topk(const float* __restrict__ D, const int32_t* __restrict__ assign,
       const int32_t* __restrict__ counts, int N, int C, int k,
       int32_t* __restrict__ sel, float* __restrict__ sel_score,
       int32_t* __restrict__ pos, int32_t* __restrict__ npos,
       uint8_t* __restrict__ posmask) {
  __shared__ int s_a[kStage];
  __shared__ float s_d[kStage];
  __shared__ double s_score[1024];
  __shared__ int s_live[1024];
  __shared__ int s_sel[1024];
  __shared__ int s_scan[32];
  const int b = blockIdx.x, tid = threadIdx.x;
  const int32_t* a = assign + (long)b * N;
  const float* Db = D + (long)b * N;
  double sum = 0.0;
  for (int base = 0; base < N; base += kStage) {
    const int lim = min(kStage, N - base);
    __syncthreads();
    for (int e = tid; e < lim; e += blockDim.x) {
      s_a[e] = a[base + e];
      s_d[e] = Db[base + e];
    }
    __syncthreads();
    if (tid < C)
      for (int e = 0; e < lim; ++e)
        if (s_a[e] == tid) sum += (double)s_d[e];
  }
  const int n = tid < C ? counts[(long)b * C + tid] : 0;
  const int live = (tid < C && n > 0) ? 1 : 0;
  s_live[tid] = live;
  s_score[tid] = live ? sum / (double)n : 0.0;
  const int nlive = __syncthreads_count(live);
  int chosen = 0;
  if (live) {
    const double me = s_score[tid];
    int rank = 0;
    for (int c = 0; c < C; ++c)
      if (s_live[c] && (s_score[c] > me || (s_score[c] == me && c < tid))) ++rank;
    if (rank < k) {
      chosen = 1;
      sel[(long)b * k + rank] = tid;
      sel_score[(long)b * k + rank] = (float)me;
    }
  }
  s_sel[tid] = chosen;
  for (int r = nlive + tid; r < k; r += blockDim.x) {
    sel[(long)b * k + r] = -1;
    sel_score[(long)b * k + r] = -INFINITY;
  }
  __syncthreads();
  int run = 0;
  for (int base = 0; base < N; base += blockDim.x) {
    const int i = base + tid;
    const int c = i < N ? a[i] : -1;
    const int m = (c >= 0 && c < C && s_sel[c]) ? 1 : 0;
    if (i < N && posmask != nullptr) posmask[(long)b * N + i] = (uint8_t)m;
    int tot;
    const int ex = block_exclusive_scan<int>(m, s_scan, &tot);
    if (m) pos[(long)b * N + run + ex] = i;
    run += tot;
  }
  if (tid == 0) npos[b] = run;
  for (int j = run + tid; j < N; j += blockDim.x) pos[(long)b * N + j] = -1;
}

// Gathered rows x (W_k | W_v) on CUDA cores; grid.y covers the K column
// tiles then the V column tiles; CTAs stride over the selected rows, whose
// count is read on the device.
template <typename T>
__global__ void __launch_bounds__(256)
k_refresh(const T* __restrict__ H, const int32_t* __restrict__ pos,
          const int32_t* __restrict__ npos, const T* __restrict__ Wk,
          const T* __restrict__ Wv, int N, int d, int nout, T* __restrict__ Kc,
          T* __restrict__ Vc, int Ncache, int off) {
  __shared__ __align__(16) SimtSmem sm;
  __shared__ long arow[kSimtM];
  __shared__ int prow[kSimtM];
  const int b = blockIdx.z, tid = threadIdx.x;
  const int ntn = ceil_div(nout, kSimtN);
  const bool is_v = (int)blockIdx.y >= ntn;
  const int n0 = (blockIdx.y % ntn) * kSimtN;
  const T* W = is_v ? Wv : Wk;
  T* out = is_v ? Vc : Kc;
  const int M = min(max(npos[b], 0), N);
  const int ty = tid >> 4, tx = tid & 15;
  for (int m0 = blockIdx.x * kSimtM; m0 < M; m0 += gridDim.x * kSimtM) {
    __syncthreads();
    if (tid < kSimtM) {
      const int j = m0 + tid;
      int p = j < M ? pos[(long)b * N + j] : -1;
      if (p >= N) p = -1;
      prow[tid] = p;
      arow[tid] = p >= 0 ? (long)b * N + p : -1L;
    }
    __syncthreads();
    float acc[4][4] = {};
    simt_tile(H, d, arow, W, nout, n0, nout, 0, d, sm, acc);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int p = prow[ty * 4 + i];
      if (p < 0) continue;
      T* o = out + ((long)b * Ncache + off + p) * nout;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int n = n0 + tx * 4 + j;
        if (n < nout) Store<T>::put(o + n, acc[i][j]);
      }
    }
  }
}

// ---- tensor-core path (bf16): gather the selected rows of every window into
// one compact matrix X [sum_b npos_b][d] (row m remembers b*N + p), then
// [K | V] = X . [W_k | W_v] on tcgen05 with the weights streamed through TMA
// as MN-major tiles, and a scatter epilogue into the cache rows.

// One warp per selected row; block (x, b) covers rows 8x .. 8x+7 of window b.
__global__ void __launch_bounds__(256)
k_gather_rows(const __nv_bfloat16* __restrict__ H, const int32_t* __restrict__ pos,
              const int32_t* __restrict__ npos, int B, int N, int d,
              __nv_bfloat16* __restrict__ X, int32_t* __restrict__ rowinfo,
              int32_t* __restrict__ M_total) {
  const int b = blockIdx.y, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int off = 0, total = 0;
  for (int bb = 0; bb < B; ++bb) {
    const int n = min(max(npos[bb], 0), N);
    if (bb < b) off += n;
    total += n;
  }
  if (b == 0 && blockIdx.x == 0 && threadIdx.x == 0) *M_total = total;
  const int Mb = min(max(npos[b], 0), N);
  const int j = blockIdx.x * 8 + warp;
  if (j >= Mb) return;
  const int p = pos[(long)b * N + j];
  const bool valid = p >= 0 && p < N;
  const uint4* src = reinterpret_cast<const uint4*>(H + ((long)b * N + (valid ? p : 0)) * d);
  uint4* dst = reinterpret_cast<uint4*>(X + (long)(off + j) * d);
  for (int c = lane; c < d / 8; c += 32)
    dst[c] = valid ? __ldg(src + c) : make_uint4(0u, 0u, 0u, 0u);
  if (lane == 0) rowinfo[off + j] = valid ? b * N + p : -1;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

template <int BN>
struct RefreshEpi : TcEpiBase {
  const int32_t* rowinfo;
  const int32_t* M_total;
  int N, Ncache, off, nkv;
  __nv_bfloat16* Kc;
  __nv_bfloat16* Vc;
  struct State {};
  __device__ int tiles(int M) const { return (M + 127) / 128; }
  __device__ int arow(int t) const { return t * 128; }
  __device__ int bsel(int, int n0) const { return n0 >= nkv ? 1 : 0; }
  __device__ int bcoord(int, int n0) const { return n0 >= nkv ? n0 - nkv : n0; }
  __device__ void tile_done(int, int, int, int, uint8_t*, State&) const {}
  __device__ void consume(int t, int rr, int n0, int, uint32_t taddr, State&) const {
    const int m = t * 128 + rr;
    const int r = m < *M_total ? rowinfo[m] : -1;
    const bool is_v = n0 >= nkv;
    __nv_bfloat16* dst = nullptr;
    if (r >= 0) {
      const int b = r / N, p = r % N;
      dst = (is_v ? Vc : Kc) + ((long)b * Ncache + off + p) * nkv + (is_v ? n0 - nkv : n0);
    }
#pragma unroll 1
    for (int c0 = 0; c0 < BN; c0 += 32) {
      float v[32];
      tc::tmem_ld32(taddr + c0, v);  // warp-collective: every lane loads
      if (dst == nullptr) continue;
#pragma unroll
      for (int c = 0; c < 32; c += 8) {
        uint4 q;
        q.x = pack_bf16x2(v[c + 0], v[c + 1]);
        q.y = pack_bf16x2(v[c + 2], v[c + 3]);
        q.z = pack_bf16x2(v[c + 4], v[c + 5]);
        q.w = pack_bf16x2(v[c + 6], v[c + 7]);
        *reinterpret_cast<uint4*>(dst + c0 + c) = q;
      }
    }
  }
};

template <int BN>
cudaError_t refresh_tc(const RefreshArgs& a, cudaStream_t s) {
  const int nkv = a.Hkv * a.dh;
  const long rows = (long)a.B * a.N;
  Carver cv(a.ws);
  __nv_bfloat16* X = cv.take<__nv_bfloat16>((size_t)rows * a.d);
  int32_t* rowinfo = cv.take<int32_t>((size_t)rows);
  int32_t* M_total = cv.take<int32_t>(4);
  k_gather_rows<<<dim3(ceil_div(a.N, 8), a.B), 256, 0, s>>>(
      static_cast<const __nv_bfloat16*>(a.H), a.pos, a.npos, a.B, a.N, a.d, X, rowinfo,
      M_total);
  TcMaps maps;
  if (!make_tmap_bf16_2d(&maps.a[0], X, a.d, rows, (uint64_t)a.d * 2, 64, 128) ||
      !make_tmap_bf16_2d(&maps.b[0], a.Wk, nkv, a.d, (uint64_t)nkv * 2, 64, 64) ||
      !make_tmap_bf16_2d(&maps.b[1], a.Wv, nkv, a.d, (uint64_t)nkv * 2, 64, 64))
    return cudaErrorInvalidValue;
  maps.a[1] = maps.a[0];
  TcShape sh{(int)rows, M_total, ceil_div(a.d, 64), ceil_div(a.d, 64), a.status};
  const int ntiles = 2 * nkv / BN;
  const int gy = std::max(1, std::min(ceil_div(rows, 128), ceil_div(2 * kSmTarget, ntiles)));
  RefreshEpi<BN> epi{{}, rowinfo, M_total, a.N, a.Ncache, a.cache_off, nkv,
                     static_cast<__nv_bfloat16*>(a.Kc), static_cast<__nv_bfloat16*>(a.Vc)};
  return launch_tc_gemm<BN, 1, 1, true>(maps, sh, epi, dim3(ntiles, gy, 1), s);
}

template <typename T>
cudaError_t refresh_typed(const RefreshArgs& a, cudaStream_t s) {
  const int nout = a.Hkv * a.dh;
  const dim3 grid(std::min(ceil_div(a.N, kSimtM), 8), 2 * ceil_div(nout, kSimtN), a.B);
  k_refresh<T><<<grid, 256, 0, s>>>(
      static_cast<const T*>(a.H), a.pos, a.npos, static_cast<const T*>(a.Wk),
      static_cast<const T*>(a.Wv), a.N, a.d, nout, static_cast<T*>(a.Kc),
      static_cast<T*>(a.Vc), a.Ncache, a.cache_off);
  return cudaGetLastError();
}

}  // namespace

cudaError_t topk_run(const TopkArgs& a, cudaStream_t s) {
  k_topk<<<a.B, 1024, 0, s>>>(a.D, a.assign, a.counts, a.N, a.C, a.k, a.sel,
                              a.sel_score, a.pos, a.npos, a.posmask);
  return cudaGetLastError();
}

bool refresh_tc_ok(int dtype, int Hkv, int dh) {
  return dtype == PS_BF16 && (Hkv * dh) % 64 == 0;
}

size_t refresh_ws(int B, int N, int d) {
  Carver cv(nullptr);
  cv.take<__nv_bfloat16>((size_t)B * N * d);
  cv.take<int32_t>((size_t)B * N);
  cv.take<int32_t>(4);
  return cv.bytes();
}

cudaError_t refresh_run(const RefreshArgs& a, cudaStream_t s) {
  if (refresh_tc_ok(a.dtype, a.Hkv, a.dh) && a.ws != nullptr) return refresh_tc<64>(a, s);
  return a.dtype == PS_F32 ? refresh_typed<float>(a, s)
                           : refresh_typed<__nv_bfloat16>(a, s);
}

}  // namespace ps
