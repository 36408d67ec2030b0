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

// Splits a non-negative finite fp32 x into x = m * 2^e (m < 2^24 an integer,
// e >= -149); returns false for a negative, infinite or NaN x.
__device__ __forceinline__ bool f32_mant_exp(float x, uint32_t* m, int* e) {
  const uint32_t u = __float_as_uint(x) & 0x7fffffffu;  // -0.0 reads as +0.0
  if (x < 0.f || u >= 0x7f800000u) return false;
  const uint32_t ef = u >> 23;
  *m = ef ? ((u & 0x7fffffu) | 0x800000u) : u;
  *e = ef ? (int)ef - 150 : -149;
  return true;
}

// One CTA of 1024 threads per window; C <= 1024.  Thread c owns cluster c.
//
// Drift sum of a cluster: fp64, one member at a time in ascending position
// order.  This sequence is reproduced exactly without per-member fp64 work
// (fp64 issues at a small fraction of the fp32 rate on this part): every
// member value is m * 2^e with m < 2^24, so every partial sum is an integer
// multiple of 2^emin (emin = the smallest member exponent).  When the exact
// integer total S = sum of m << (e - emin) stays below 2^53, every partial
// sum has a 53-bit significand and no fp64 addition rounds, so the
// sequential fp64 sum equals S * 2^emin.  S is order-free, so the members are
// folded with shared-memory integer atomics.  A cluster outside that range
// (a term or the total at or above 2^53, a negative or non-finite value)
// takes the sequential fp64 loop itself, one warp per such cluster.
//
// Rank of a cluster = the number of clusters that beat it (higher mean, or
// equal mean and lower index).  Positions are compacted with a block scan,
// ascending.
__global__ void __launch_bounds__(1024)
k_topk(const float* __restrict__ D, const int32_t* __restrict__ assign,
       const int32_t* __restrict__ counts, int N, int C, int k,
       int32_t* __restrict__ sel, float* __restrict__ sel_score,
       int32_t* __restrict__ pos, int32_t* __restrict__ npos,
       uint8_t* __restrict__ posmask) {
  pdl_prologue();
  __shared__ unsigned long long s_key[1024];  // integer sum, then rank key
  __shared__ int s_emin[1024];
  __shared__ int s_live[1024];  // fallback flag, then liveness
  __shared__ int s_sel[1024];
  __shared__ int s_scan[32];
  __shared__ double s_sum[1024];
  __shared__ int s_nfall;
  __shared__ int s_fall[1024];
  const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int32_t* a = assign + (long)b * N;
  const float* Db = D + (long)b * N;
  s_key[tid] = 0ull;
  s_emin[tid] = INT_MAX;
  s_live[tid] = 0;
  if (tid == 0) s_nfall = 0;
  __syncthreads();
  for (int i = tid; i < N; i += blockDim.x) {  // smallest exponent per cluster
    const int c = a[i];
    uint32_t m;
    int e;
    if (c < 0 || c >= C) continue;
    if (!f32_mant_exp(Db[i], &m, &e)) s_live[c] = 1;
    else if (m != 0u) atomicMin(&s_emin[c], e);
  }
  __syncthreads();
  for (int i = tid; i < N; i += blockDim.x) {  // exact integer totals
    const int c = a[i];
    uint32_t m;
    int e;
    if (c < 0 || c >= C || !f32_mant_exp(Db[i], &m, &e) || m == 0u) continue;
    const int sh = e - s_emin[c];
    if (sh > 29) {  // m << sh could reach 2^53
      s_live[c] = 1;
      continue;
    }
    const unsigned long long t = (unsigned long long)m << sh;
    const unsigned long long old = atomicAdd(&s_key[c], t);
    if (old + t < old) s_live[c] = 1;  // wrapped: the total is far above 2^53
  }
  __syncthreads();
  if (tid < C) {
    const unsigned long long S = s_key[tid];
    if (s_live[tid] || S >= (1ull << 53)) {
      s_fall[atomicAdd(&s_nfall, 1)] = tid;
    } else {
      // S * 2^emin, exact: S < 2^53 converts exactly and 2^emin (emin >=
      // -149) is a normal fp64 power of two, built from its exponent bits
      s_sum[tid] = S == 0ull ? 0.0
                             : (double)S * __longlong_as_double(
                                               (long long)(s_emin[tid] + 1023) << 52);
    }
  }
  __syncthreads();
  for (int f = warp; f < s_nfall; f += 32) {  // the sequential fp64 sum itself
    const int c = s_fall[f];
    double sum = 0.0;
    for (int e0 = 0; e0 < N; e0 += 32) {
      const int e = e0 + lane;
      const bool mine = e < N && a[e] == c;
      const float dv = mine ? Db[e] : 0.f;
      unsigned hit = __ballot_sync(0xffffffffu, mine);
      while (hit) {
        const int j = __ffs(hit) - 1;
        hit &= hit - 1;
        sum += (double)__shfl_sync(0xffffffffu, dv, j);
      }
    }
    if (lane == 0) s_sum[c] = sum;
  }
  __syncthreads();
  const int n = tid < C ? counts[(long)b * C + tid] : 0;
  const int live = (tid < C && n > 0) ? 1 : 0;
  s_live[tid] = live;
  const double me = live ? s_sum[tid] / (double)n : 0.0;
  // D >= 0, so every mean is a non-negative double and its bit pattern
  // orders like its value: rank on integer keys (exact, and cheap here)
  s_key[tid] = live ? (unsigned long long)__double_as_longlong(me) : 0ull;
  const int nlive = __syncthreads_count(live);
  int chosen = 0;
  if (live) {
    const unsigned long long mk = s_key[tid];
    int rank = 0;
    for (int c = 0; c < C; ++c)
      if (s_live[c] && (s_key[c] > mk || (s_key[c] == mk && c < tid))) ++rank;
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
  pdl_prologue();
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

// One warp per selected row; block (x, b) takes rows 8x .. 8x+7 of window b,
// then 8 gridDim.x further on, and so on (the grid is sized to about what
// the GPU holds at once, as the selection's size is known only here).  A
// lane copies 16 bytes of the row per step, eight steps' loads in flight.
__global__ void __launch_bounds__(256, 4)
k_gather_rows(const __nv_bfloat16* __restrict__ H, const int32_t* __restrict__ pos,
              const int32_t* __restrict__ npos, int B, int N, int d,
              __nv_bfloat16* __restrict__ X, int32_t* __restrict__ rowinfo,
              int32_t* __restrict__ M_total) {
  pdl_prologue();
  const int b = blockIdx.y, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int off = 0, total = 0;
  for (int bb = 0; bb < B; ++bb) {
    const int n = min(max(npos[bb], 0), N);
    if (bb < b) off += n;
    total += n;
  }
  if (b == 0 && blockIdx.x == 0 && threadIdx.x == 0) *M_total = total;
  const int Mb = min(max(npos[b], 0), N);
  for (int j = blockIdx.x * 8 + warp; j < Mb; j += gridDim.x * 8) {
    const int p = pos[(long)b * N + j];
    const bool valid = p >= 0 && p < N;
    const uint4* src = reinterpret_cast<const uint4*>(H + ((long)b * N + (valid ? p : 0)) * d);
    uint4* dst = reinterpret_cast<uint4*>(X + (long)(off + j) * d);
#pragma unroll 8
    for (int c = lane; c < d / 8; c += 32)
      dst[c] = valid ? __ldg(src + c) : make_uint4(0u, 0u, 0u, 0u);
    if (lane == 0) rowinfo[off + j] = valid ? b * N + p : -1;
  }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// Column tiles of BN over [K | V]; the epilogue rounds to bf16 and scatters
// each selected row into the K or V cache (a split d: RefreshClusterEpi).
template <int BN>
struct RefreshEpi : TcEpiBase {
  const int32_t* rowinfo;
  const int32_t* M_total;
  int N, Ncache, off, nkv, split_max_rows;
  __nv_bfloat16* Kc;
  __nv_bfloat16* Vc;
  struct State {};
  __device__ int tiles(int M) const { return (M + 127) / 128; }
  __device__ int arow(int t) const { return t * 128; }
  __device__ int bsel(int, int n0) const { return n0 >= nkv ? 1 : 0; }
  __device__ int bcoord(int, int n0) const { return n0 >= nkv ? n0 - nkv : n0; }
  __device__ void tile_done(int, int, int, int, uint8_t*, State&) const {}
  __device__ void consume(int t, int rr, int n0, int, uint32_t taddr, State&) const {
    const int Mt = *M_total;
    const int m = t * 128 + rr;
    const int r = m < Mt ? rowinfo[m] : -1;
    const bool is_v = n0 >= nkv;
    __nv_bfloat16* dst = nullptr;
    if (r >= 0) {
      const int b = r / N, p = r % N;
      dst = (is_v ? Vc : Kc) + ((long)b * Ncache + off + p) * nkv + (is_v ? n0 - nkv : n0);
    }
#pragma unroll 1
    for (int c0 = 0; c0 < BN; c0 += 32) {
      float v[32];
      tc::tmem_ld32(taddr + c0, v);
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

// The d-chunks of a column tile in one thread-block cluster.  While the
// selection is small (split) each chunk's 128 x BN tile stays in shared
// memory and CTA z sums rows [128 z / nz, 128 (z+1) / nz) over the chunks in
// chunk order, a warp per row and 8 columns per lane, rounds to bf16 and
// scatters the row into the K or V cache.  Otherwise chunk 0 takes the whole
// d range and scatters straight from TMEM, the other chunks idle.
template <int BN>
struct RefreshClusterEpi : RefreshEpi<BN> {
  static constexpr bool kClusterReduce = true;
  static constexpr uint32_t kLd = BN + 4;
  using State = typename RefreshEpi<BN>::State;
  __device__ void consume_red(int t, int rr, int n0, int z, uint32_t taddr, State& st,
                              float* red_row) const {
    if (*this->M_total > this->split_max_rows) {
      this->consume(t, rr, n0, z, taddr, st);
      return;
    }
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
  // scratch: destination rows of this CTA's share of the tile (split regime)
  __device__ void prefetch(uint8_t* scratch, int k, int n) const {
    const int Mt = *this->M_total;
    if (Mt > this->split_max_rows) return;
    const int t = blockIdx.y, z = blockIdx.z, nz = gridDim.z;
    const int live = min(128, Mt - t * 128);
    const int r0 = min(z * 128 / nz, live), r1 = min((z + 1) * 128 / nz, live);
    int* s_ri = reinterpret_cast<int*>(scratch);
    for (int j = k; j < r1 - r0; j += n) s_ri[j] = this->rowinfo[t * 128 + r0 + j];
  }
  __device__ void reduce(const float* red, int z, int nz, uint8_t* scratch) const {
    const int Mt = *this->M_total;
    if (Mt <= this->split_max_rows) {
      const int t = blockIdx.y, n0 = blockIdx.x * BN, nkv = this->nkv;
      // rows of this CTA's share that hold selected positions (<= 64, nz >= 2)
      const int live = min(128, Mt - t * 128);
      const int r0 = min(z * 128 / nz, live), r1 = min((z + 1) * 128 / nz, live);
      const bool is_v = n0 >= nkv;
      const int* s_ri = reinterpret_cast<const int*>(scratch);  // [64], staged by prefetch
      __nv_bfloat16* cache = is_v ? this->Vc : this->Kc;
      const int coff = is_v ? n0 - nkv : n0;
      cluster_rows_sum<4, 32>(red, kLd, r0, r1, BN, nz, [&](int r, int c, float4 v) {
        const int ri = s_ri[r - r0];
        if (ri < 0) return;
        const int b = ri / this->N, p = ri % this->N;
        *reinterpret_cast<uint2*>(cache + ((long)b * this->Ncache + this->off + p) * nkv + coff +
                                  c) = make_uint2(pack_bf16x2(v.x, v.y), pack_bf16x2(v.z, v.w));
      });
    }
    tc::cluster_arrive();
  }
};

struct RefreshPlan {
  int BN, ntiles, nz, kpc, KB, split_max_rows;
};

RefreshPlan refresh_plan(int B, int N, int d, int nkv) {
  RefreshPlan p{};
  p.BN = nkv % 256 == 0 ? 256 : (nkv % 128 == 0 ? 128 : 64);
  p.ntiles = 2 * nkv / p.BN;
  p.KB = ceil_div(d, 64);
  p.nz = std::min(4, p.KB);
  p.kpc = ceil_div(p.KB, p.nz);
  p.nz = ceil_div(p.KB, p.kpc);
  // split d only while the selected rows give less than a wave of tiles; the
  // grid's y extent (>= this many row tiles) then gives each CTA one tile
  p.split_max_rows = std::min(B * N, 128 * std::max(1, kSmTarget / p.ntiles));
  if (p.nz == 1) p.split_max_rows = 0;
  return p;
}

template <int BN>
cudaError_t refresh_tc(const RefreshArgs& a, const RefreshPlan& pl, cudaStream_t s) {
  const int nkv = a.Hkv * a.dh;
  const long rows = (long)a.B * a.N;
  Carver cv(a.ws);
  __nv_bfloat16* X = cv.take<__nv_bfloat16>((size_t)rows * a.d);
  int32_t* rowinfo = cv.take<int32_t>((size_t)rows);
  int32_t* M_total = cv.take<int32_t>(4);
  const int gx = std::max(1, std::min(ceil_div(a.N, 8), ceil_div(8 * kSmTarget, a.B)));
  launch_pdl(k_gather_rows, dim3(gx, a.B), 256, 0, s,
      static_cast<const __nv_bfloat16*>(a.H), a.pos, a.npos, a.B, a.N, a.d, X, rowinfo,
      M_total);
  TcMaps maps;
  if (!make_tmap_bf16_2d(&maps.a[0], X, a.d, rows, (uint64_t)a.d * 2, 64, 128) ||
      !make_tmap_bf16_2d(&maps.b[0], a.Wk, nkv, a.d, (uint64_t)nkv * 2, 64, 64) ||
      !make_tmap_bf16_2d(&maps.b[1], a.Wv, nkv, a.d, (uint64_t)nkv * 2, 64, 64))
    return cudaErrorInvalidValue;
  maps.a[1] = maps.a[0];
  TcShape sh{(int)rows, M_total, pl.KB, pl.kpc, a.status, pl.split_max_rows};
  const int gy = std::max(1, std::min(ceil_div(rows, 128), ceil_div(4 * kSmTarget, pl.ntiles)));
  RefreshEpi<BN> epi{{}, rowinfo, M_total, a.N, a.Ncache, a.cache_off, nkv,
                     pl.split_max_rows, static_cast<__nv_bfloat16*>(a.Kc),
                     static_cast<__nv_bfloat16*>(a.Vc)};
  if (pl.nz == 1)
    return launch_tc_gemm<BN, 1, 1, true>(maps, sh, epi, dim3(pl.ntiles, gy, 1), s);
  return launch_tc_gemm<BN, 1, 1, true>(maps, sh, RefreshClusterEpi<BN>{epi},
                                        dim3(pl.ntiles, gy, pl.nz), s);
}

template <typename T>
cudaError_t refresh_typed(const RefreshArgs& a, cudaStream_t s) {
  const int nout = a.Hkv * a.dh;
  const dim3 grid(std::min(ceil_div(a.N, kSimtM), 8), 2 * ceil_div(nout, kSimtN), a.B);
  launch_pdl(k_refresh<T>, grid, 256, 0, s, 
      static_cast<const T*>(a.H), a.pos, a.npos, static_cast<const T*>(a.Wk),
      static_cast<const T*>(a.Wv), a.N, a.d, nout, static_cast<T*>(a.Kc),
      static_cast<T*>(a.Vc), a.Ncache, a.cache_off);
  return cudaGetLastError();
}

}  // namespace

cudaError_t topk_run(const TopkArgs& a, cudaStream_t s) {
  launch_pdl(k_topk, a.B, 1024, 0, s, a.D, a.assign, a.counts, a.N, a.C, a.k, a.sel,
                              a.sel_score, a.pos, a.npos, a.posmask);
  return cudaGetLastError();
}

bool refresh_tc_ok(int dtype, int Hkv, int dh) {
  return dtype == PS_BF16 && (Hkv * dh) % 64 == 0;
}

size_t refresh_ws(int B, int N, int d, int, int) {
  Carver cv(nullptr);
  cv.take<__nv_bfloat16>((size_t)B * N * d);
  cv.take<int32_t>((size_t)B * N);
  cv.take<int32_t>(4);
  return cv.bytes();
}

cudaError_t refresh_run(const RefreshArgs& a, cudaStream_t s) {
  if (refresh_tc_ok(a.dtype, a.Hkv, a.dh) && a.ws != nullptr) {
    const RefreshPlan pl = refresh_plan(a.B, a.N, a.d, a.Hkv * a.dh);
    switch (pl.BN) {
      case 256: return refresh_tc<256>(a, pl, s);
      case 128: return refresh_tc<128>(a, pl, s);
      default: return refresh_tc<64>(a, pl, s);
    }
  }
  return a.dtype == PS_F32 ? refresh_typed<float>(a, s)
                           : refresh_typed<__nv_bfloat16>(a, s);
}

}  // namespace ps
