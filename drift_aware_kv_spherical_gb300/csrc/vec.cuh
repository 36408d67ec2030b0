// 16-byte vector loads of f32 / bf16 rows widened to fp32, and block-level
// scans/reductions used by several kernels.
#pragma once

#include "common.cuh"

namespace ps {

template <typename T> struct Vec;
template <> struct Vec<float> { static constexpr int n = 4; };
template <> struct Vec<__nv_bfloat16> { static constexpr int n = 8; };

__device__ __forceinline__ void bf16x2_to_f32(uint32_t w, float& lo, float& hi) {
  lo = __uint_as_float(w << 16);
  hi = __uint_as_float(w & 0xffff0000u);
}

// Loads Vec<T>::n consecutive elements from a 16-byte aligned address.
__device__ __forceinline__ void load16(const float* p, float* out) {
  float4 v = __ldg(reinterpret_cast<const float4*>(p));
  out[0] = v.x; out[1] = v.y; out[2] = v.z; out[3] = v.w;
}
__device__ __forceinline__ void load16(const __nv_bfloat16* p, float* out) {
  uint4 v = __ldg(reinterpret_cast<const uint4*>(p));
  bf16x2_to_f32(v.x, out[0], out[1]);
  bf16x2_to_f32(v.y, out[2], out[3]);
  bf16x2_to_f32(v.z, out[4], out[5]);
  bf16x2_to_f32(v.w, out[6], out[7]);
}

// A 16-byte vector already in registers, widened to fp32.
__device__ __forceinline__ void unpack16(const uint4& r, float* out, float) {
  out[0] = __uint_as_float(r.x); out[1] = __uint_as_float(r.y);
  out[2] = __uint_as_float(r.z); out[3] = __uint_as_float(r.w);
}
__device__ __forceinline__ void unpack16(const uint4& r, float* out, __nv_bfloat16) {
  bf16x2_to_f32(r.x, out[0], out[1]);
  bf16x2_to_f32(r.y, out[2], out[3]);
  bf16x2_to_f32(r.z, out[4], out[5]);
  bf16x2_to_f32(r.w, out[6], out[7]);
}

// Exclusive prefix sum over the threads of a block (blockDim.x % 32 == 0,
// <= 1024).  `scratch` holds 32 values.  Returns the exclusive prefix and
// writes the block total to *total.  Contains __syncthreads().
template <typename V>
__device__ V block_exclusive_scan(V v, V* scratch, V* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nwarps = blockDim.x >> 5;
  V x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    V y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) scratch[warp] = x;
  __syncthreads();
  if (warp == 0) {
    V s = lane < nwarps ? scratch[lane] : V(0);
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      V y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    scratch[lane] = s;  // inclusive prefix of warp totals
  }
  __syncthreads();
  V before = warp > 0 ? scratch[warp - 1] : V(0);
  *total = scratch[nwarps - 1];
  __syncthreads();
  return before + x - v;
}

__device__ __forceinline__ int block_min_int(int v, int* scratch) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = min(v, __shfl_xor_sync(0xffffffffu, v, o));
  if (lane == 0) scratch[warp] = v;
  __syncthreads();
  int r = scratch[0];
  for (int w = 1; w < (int)(blockDim.x >> 5); ++w) r = min(r, scratch[w]);
  __syncthreads();
  return r;
}

// Sum over a block in a fixed order (deterministic).
__device__ __forceinline__ float block_sum_f32(float v, float* scratch) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = warp_sum(v);
  if (lane == 0) scratch[warp] = v;
  __syncthreads();
  float r = 0.f;
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) r += scratch[w];
  __syncthreads();
  return r;
}

}  // namespace ps
