// 64x64 fp32 tile of C = A . B on CUDA cores, for the f32 path and for
// shapes the tensor-core kernels do not take.  A rows may be gathered
// through an index list; B is row-major [K][ldb].  256 threads, each owning
// a 4x4 block of the tile; 16-deep shared-memory stages.
#pragma once

#include "vec.cuh"

namespace ps {

constexpr int kSimtM = 64, kSimtN = 64, kSimtK = 16;

__device__ __forceinline__ void load4(const float* p, float* o) {
  const float4 v = __ldg(reinterpret_cast<const float4*>(p));
  o[0] = v.x; o[1] = v.y; o[2] = v.z; o[3] = v.w;
}
__device__ __forceinline__ void load4(const __nv_bfloat16* p, float* o) {
  const uint2 v = __ldg(reinterpret_cast<const uint2*>(p));
  bf16x2_to_f32(v.x, o[0], o[1]);
  bf16x2_to_f32(v.y, o[2], o[3]);
}

struct SimtSmem {
  float As[kSimtK][kSimtM];
  float Bs[kSimtK][kSimtN];
};

// acc[i][j] += sum_{k in [k_begin,k_end)} A[row(ty*4+i)][k] * B[k][n0+tx*4+j]
// rows: the tile's m-th row is A + arow[m] * lda (arow[m] < 0: zero row).
// (k_end - k_begin) % 16 == 0, ldb % 4 == 0, lda % 4 == 0, pointers 16-B
// aligned; columns >= n_valid read as zero (n_valid % 4 == 0).
template <typename TA, typename TB>
__device__ __forceinline__ void simt_tile(const TA* __restrict__ A, long lda,
                                          const long* arow,  // [64] in smem
                                          const TB* __restrict__ B, long ldb,
                                          int n0, int n_valid, int k_begin,
                                          int k_end, SimtSmem& sm,
                                          float acc[4][4]) {
  const int tid = threadIdx.x;
  const int ty = tid >> 4, tx = tid & 15;
  const int am = tid >> 2, ak = (tid & 3) * 4;      // A stage: 64 x 16
  const int bk = tid >> 4, bn = (tid & 15) * 4;     // B stage: 16 x 64
  for (int k0 = k_begin; k0 < k_end; k0 += kSimtK) {
    float av[4] = {0.f, 0.f, 0.f, 0.f};
    const long ar = arow[am];
    if (ar >= 0) load4(A + ar * lda + k0 + ak, av);
#pragma unroll
    for (int e = 0; e < 4; ++e) sm.As[ak + e][am] = av[e];
    float bv[4] = {0.f, 0.f, 0.f, 0.f};
    if (n0 + bn < n_valid) load4(B + (long)(k0 + bk) * ldb + n0 + bn, bv);
    *reinterpret_cast<float4*>(&sm.Bs[bk][bn]) = make_float4(bv[0], bv[1], bv[2], bv[3]);
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < kSimtK; ++kk) {
      const float4 a = *reinterpret_cast<const float4*>(&sm.As[kk][ty * 4]);
      const float4 b = *reinterpret_cast<const float4*>(&sm.Bs[kk][tx * 4]);
      const float x[4] = {a.x, a.y, a.z, a.w};
      const float y[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(x[i], y[j], acc[i][j]);
    }
    __syncthreads();
  }
}

}  // namespace ps
