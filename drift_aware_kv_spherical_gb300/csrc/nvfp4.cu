// a2: NVFP4 quantisation of the k-means residuals.
//
// [Polestar §2.A, local window & clustering]: residuals of the clustered
// hidden states are quantised with NVFP4 into compact proxies.  Format:
// E2M1 elements, one E4M3 scale per 16 consecutive elements, one fp32 scale
// per window; round-to-nearest-even with saturation, using Blackwell's
// cvt.rn.satfinite.{e2m1x2,e4m3x2}.f32 conversions.  Every arithmetic step
// is an IEEE fp32 operation with an explicit rounding (no contraction), so
// the outputs are bit-exact functions of the inputs.
//
//   k_fp4_amax   partial max |r| of each unit of a window (r recomputed)
//   k_fp4_quant  tensor scale, block scales and packed codes
// Work units: a window's rows in gx slots of consecutive rows, unit u =
// b gx + slot.  Both kernels run a persistent grid that takes the units in
// order (CTA g: units g, g + G, ...), so the CTAs work on one or two windows
// at a time and those windows' fp32 centroids, read once per element, stay
// in L2.  A warp takes a row: its label, rho and centroid row are looked up
// once.  k_fp4_amax takes the row in steps of 128 elements, lane j taking
// elements 4j .. 4j+3 of a step, so every warp load is one contiguous run
// (256 bytes of bf16 h, 512 of fp32 mu); k_fp4_quant gives lane j the row's
// 16-element blocks j, j + 32, ..., so a block's scale and its eight code
// bytes come from one lane (the quad layout measured slower there: its
// 2-byte code stores and per-quad scale work).
// The quantiser divides r by the block's d = s_blk * S as r * RN(1/d), and
// falls back to the IEEE division where that could change the code: the
// product lies within 3 * 2^-24 relative of RN(r / d) (two roundings and
// the reciprocal's), so when the E2M1 conversion takes the same code at
// q (1 - 2^-20) and q (1 + 2^-20) that is the code of RN(r / d) too.
// The residual r = fl(h - fl(rho * mu_a)) is recomputed in the second kernel
// instead of being stored: re-reading h costs 2 B/element (bf16), storing r
// would cost 8.
#include <algorithm>
#include <cfloat>
#include <mutex>
#include <unordered_map>

#include "ops.h"
#include "vec.cuh"

namespace ps {
namespace {

// 128-thread CTAs, as many as an SM holds (measured 5 % faster than 256:
// 551 against 581 us for both kernels at the stress size).
constexpr int kThreads = 128;

// Eight fp32 values -> eight E2M1 codes, element 2j in the low nibble of
// byte j.  cvt ... e2m1x2 d, a, b puts a in the high nibble, b in the low.
__device__ __forceinline__ uint32_t e2m1x8(const float* v) {
  uint32_t out;
  asm("{\n\t"
      ".reg .b8 q0, q1, q2, q3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q3, %8, %7;\n\t"
      "mov.b32 %0, {q0, q1, q2, q3};\n\t"
      "}"
      : "=r"(out)
      : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]),
        "f"(v[6]), "f"(v[7]));
  return out;
}

// fp32 -> E4M3 code (low byte of the x2 conversion).
__device__ __forceinline__ uint32_t e4m3_code(float x) {
  unsigned short h;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(h) : "f"(0.f), "f"(x));
  return h & 0xFFu;
}

// Exact value of a non-negative E4M3 code (bias 7, subnormal step 2^-9).
__device__ __forceinline__ float e4m3_value(uint32_t c) {
  const uint32_t e = (c >> 3) & 15u, m = c & 7u;
  if (e == 0) return (float)m * 0.001953125f;
  return __uint_as_float(((e + 120u) << 23) | (m << 20));
}

// Four consecutive elements of a row (8- or 16-byte aligned) as fp32.
__device__ __forceinline__ void load4(const float* p, float* out) {
  const float4 v = __ldg(reinterpret_cast<const float4*>(p));
  out[0] = v.x; out[1] = v.y; out[2] = v.z; out[3] = v.w;
}
__device__ __forceinline__ void load4(const __nv_bfloat16* p, float* out) {
  const uint2 v = __ldg(reinterpret_cast<const uint2*>(p));
  bf16x2_to_f32(v.x, out[0], out[1]);
  bf16x2_to_f32(v.y, out[2], out[3]);
}

// r[0..3] = fl(h - fl(rho * mu)) of four elements (m == nullptr: r = h).
template <typename T>
__device__ __forceinline__ void residual4(const T* __restrict__ h, const float* __restrict__ m,
                                          float rh, float* r) {
  load4(h, r);
  if (m != nullptr) {
    float mv[4];
    load4(m, mv);
#pragma unroll
    for (int e = 0; e < 4; ++e) r[e] = __fsub_rn(r[e], __fmul_rn(rh, mv[e]));
  }
}

// The codes of x[0..7] / den (four bytes, element 2j in the low nibble of
// byte j), with rinv = RN(1 / den) finite: the product path where both
// ends of its error band convert alike, else the IEEE division.
__device__ __forceinline__ uint32_t e2m1_div8(const float* x, float den, float rinv) {
  constexpr float kLo = 1.0f - 0x1p-20f, kHi = 1.0f + 0x1p-20f;
  float lo[8], hi[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const float q = __fmul_rn(x[e], rinv);
    lo[e] = __fmul_rn(q, kLo);
    hi[e] = __fmul_rn(q, kHi);
  }
  const uint32_t a = e2m1x8(lo), b = e2m1x8(hi);
  if (a == b) return a;
  float v[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) v[e] = __fdiv_rn(x[e], den);
  return e2m1x8(v);
}

// r[0..15] of the block at h (16 elements of a row) against the matching 16
// centroid values at m (nullptr: r = h) and the row's rho.
template <typename T>
__device__ __forceinline__ void residual16(const T* __restrict__ h, const float* __restrict__ m,
                                           float rh, float* r) {
  constexpr int V = Vec<T>::n;
#pragma unroll
  for (int q = 0; q < 16 / V; ++q) load16(h + q * V, r + q * V);
  if (m != nullptr) {
    float mv[16];
#pragma unroll
    for (int q = 0; q < 4; ++q) load16(m + 4 * q, mv + 4 * q);
#pragma unroll
    for (int e = 0; e < 16; ++e) r[e] = __fsub_rn(r[e], __fmul_rn(rh, mv[e]));
  }
}

// The row's centroid (nullptr when H itself is quantised) and rho.
__device__ __forceinline__ const float* row_centroid(const float* __restrict__ mu,
                                                     const int32_t* __restrict__ assign,
                                                     const float* __restrict__ rho, int b,
                                                     int N, int d, int C, int row, float* rh) {
  if (mu == nullptr) {
    *rh = 0.f;
    return nullptr;
  }
  const long i = (long)b * N + row;
  const int a = min(max(assign[i], 0), C - 1);
  *rh = rho[i];
  return mu + ((long)b * C + a) * d;
}

__device__ __forceinline__ float block_max(float v, float* scratch) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = warp_max(v);
  if (lane == 0) scratch[warp] = v;
  __syncthreads();
  float r = scratch[0];
  for (int w = 1; w < (int)(blockDim.x >> 5); ++w) r = fmaxf(r, scratch[w]);
  __syncthreads();
  return r;
}

// Partials the scratch holds at most (the workspace-free entry point's
// fixed array); a window gets gx <= kMaxParts / B of them.
constexpr int kMaxParts = 16384;

__device__ __forceinline__ void unit_rows(int N, int gx, int slot, int* r0, int* r1) {
  const int per = (N + gx - 1) / gx;
  *r0 = min(N, slot * per);
  *r1 = min(N, *r0 + per);
}

template <typename T>
__global__ void __launch_bounds__(kThreads)
k_fp4_amax(const T* __restrict__ H, const float* __restrict__ mu,
           const int32_t* __restrict__ assign, const float* __restrict__ rho,
           int B, int N, int d, int C, int gx, float* __restrict__ part) {
  pdl_prologue();
  __shared__ float s_red[kThreads / 32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const long units = (long)B * gx;
  for (long u = blockIdx.x; u < units; u += gridDim.x) {  // CTA-uniform
    const int b = (int)(u / gx);
    int r0, r1;
    unit_rows(N, gx, (int)(u % gx), &r0, &r1);
    float m = 0.f;
    for (int row = r0 + warp; row < r1; row += kThreads / 32) {
      float rh;
      const float* mrow = row_centroid(mu, assign, rho, b, N, d, C, row, &rh);
      const T* hrow = H + ((long)b * N + row) * d;
#pragma unroll 8
      for (int c = 4 * lane; c < d; c += 128) {
        float r[4];
        residual4(hrow + c, mrow != nullptr ? mrow + c : nullptr, rh, r);
#pragma unroll
        for (int e = 0; e < 4; ++e) m = fmaxf(m, fabsf(r[e]));
      }
    }
    m = block_max(m, s_red);
    if (threadIdx.x == 0) part[u] = m;
  }
}

// One 16-element block: its E4M3 scale and eight bytes of E2M1 codes.  The
// codes of r / den come from r * RN(1 / den) wherever that cannot change
// them (e2m1_div8), else from the IEEE division.
__device__ __forceinline__ void quant_block(const float* r, float S, float six_s,
                                            uint8_t* __restrict__ codes_at,
                                            uint8_t* __restrict__ scale_at) {
  float bm = 0.f;
#pragma unroll
  for (int e = 0; e < 16; ++e) bm = fmaxf(bm, fabsf(r[e]));
  const uint32_t sc = e4m3_code(__fdiv_rn(bm, six_s));
  const float sb = e4m3_value(sc);
  uint2 q = make_uint2(0u, 0u);
  if (sb != 0.f) {
    const float den = __fmul_rn(sb, S);
    if (den >= FLT_MIN) {
      const float rinv = __frcp_rn(den);
      q.x = e2m1_div8(r, den, rinv);
      q.y = e2m1_div8(r + 8, den, rinv);
    } else {
      float v[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) v[e] = __fdiv_rn(r[e], den);
      q.x = e2m1x8(v);
      q.y = e2m1x8(v + 8);
    }
  }
  *reinterpret_cast<uint2*>(codes_at) = q;
  *scale_at = (uint8_t)sc;
}

template <typename T>
__global__ void __launch_bounds__(kThreads)
k_fp4_quant(const T* __restrict__ H, const float* __restrict__ mu,
            const int32_t* __restrict__ assign, const float* __restrict__ rho,
            int B, int N, int d, int C, int gx, const float* __restrict__ part,
            uint8_t* __restrict__ codes, uint8_t* __restrict__ scales,
            float* __restrict__ S_out) {
  pdl_prologue();
  __shared__ float s_red[kThreads / 32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int bpr = d / 16;
  const long units = (long)B * gx;
  for (long u = blockIdx.x; u < units; u += gridDim.x) {  // CTA-uniform
    const int b = (int)(u / gx), slot = (int)(u % gx);
    float amax = 0.f;
    for (int p = threadIdx.x; p < gx; p += kThreads) amax = fmaxf(amax, part[(long)b * gx + p]);
    amax = block_max(amax, s_red);
    const float S = (amax > 0.f && amax <= FLT_MAX)
                        ? fmaxf(__fdiv_rn(amax, 2688.0f), FLT_MIN) : 1.0f;
    if (slot == 0 && threadIdx.x == 0) S_out[b] = S;
    const float six_s = __fmul_rn(6.0f, S);
    int r0, r1;
    unit_rows(N, gx, slot, &r0, &r1);
    for (int row = r0 + warp; row < r1; row += kThreads / 32) {
      float rh;
      const float* mrow = row_centroid(mu, assign, rho, b, N, d, C, row, &rh);
      const long rowbase = (long)b * N + row;
      const T* hrow = H + rowbase * d;
      for (int k = lane; k < bpr; k += 32) {
        float r[16];
        residual16(hrow + k * 16, mrow != nullptr ? mrow + k * 16 : nullptr, rh, r);
        quant_block(r, S, six_s, codes + rowbase * (d / 2) + k * 8, scales + rowbase * bpr + k);
      }
    }
  }
}

// CTAs of `threads` threads an SM holds at once: the occupancy query, made
// once per kernel type (each kernel here has a type of its own); 1 if it
// fails.
template <typename K>
int resident_ctas(K kern, int threads) {
  static const int n = [&] {
    int v = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, kern, threads, 0) != cudaSuccess) {
      cudaGetLastError();
      v = 1;
    }
    return std::max(1, v);
  }();
  return n;
}

// Slots per window: one row per warp of a CTA, at most kMaxParts / B (so
// B gx partials fit the fixed array for every B <= kMaxParts).
int grid_x(int B, int N, int d) {
  (void)d;
  const int want = ceil_div(N, kThreads / 32);
  const int cap = std::max(1, kMaxParts / std::max(B, 1));
  return std::max(1, std::min(want, cap));
}

template <typename T>
cudaError_t run_typed(const Nvfp4Args& a, cudaStream_t s) {
  const T* H = static_cast<const T*>(a.H);
  const int gx = grid_x(a.B, a.N, a.d);
  float* part = Carver(a.ws).take<float>((size_t)a.B * gx);
  const long units = (long)a.B * gx;
  // persistent grids: as many CTAs as the SMs hold at once, no second wave
  const int sms = a.num_sms > 0 ? a.num_sms : kSmTarget;
  const int g1 = (int)std::min<long>(units, (long)resident_ctas(k_fp4_amax<T>, kThreads) * sms);
  const int g2 = (int)std::min<long>(units, (long)resident_ctas(k_fp4_quant<T>, kThreads) * sms);
  launch_pdl(k_fp4_amax<T>, g1, kThreads, 0, s, H, a.mu, a.assign, a.rho, a.B, a.N, a.d,
             a.C, gx, part);
  launch_pdl(k_fp4_quant<T>, g2, kThreads, 0, s, H, a.mu, a.assign, a.rho, a.B, a.N, a.d,
             a.C, gx, part, a.codes, a.scales, a.S);
  return cudaGetLastError();
}

}  // namespace

size_t nvfp4_ws(int B, int N, int d) {
  Carver cv(nullptr);
  cv.take<float>((size_t)B * grid_x(B, N, d));
  return cv.bytes();
}

cudaError_t nvfp4_run(const Nvfp4Args& a, cudaStream_t s) {
  return a.dtype == PS_F32 ? run_typed<float>(a, s)
                           : run_typed<__nv_bfloat16>(a, s);
}

// ---------------------------------------------------------------------------
// Variant without a caller workspace, for callers that cannot allocate device
// memory (for example a host that hands the library only preallocated input
// and output buffers, or code running where a device allocation is forbidden
// because it could synchronise the device or fail under a fixed memory
// budget).  The per-CTA partial maxima live in a fixed file-scope device
// array instead of the caller's workspace; every GPU that loads the library
// keeps this array until the process exits.
namespace {

constexpr int kStaticParts = kMaxParts;  // floats = 64 KiB; fits B <= 16384
static __device__ __align__(256) float g_nvfp4_static_parts[kStaticParts];

std::mutex g_static_mu;
std::unordered_map<int, float*> g_static_ptr;  // device id -> array address

}  // namespace

bool nvfp4_static_fits(int B, int N, int d) {
  return (long)B * grid_x(B, N, d) <= kStaticParts;
}

// Looks the array's device address up once per device; the caller has made
// `device` current (the entry point checks this).  The first call on a device
// therefore makes a runtime call that must not happen inside a stream
// capture.  The cached address belongs to the device's current context: the
// library must not be used across a reset of that device.
cudaError_t nvfp4_static_scratch(int device, float** out) {
  std::lock_guard<std::mutex> lock(g_static_mu);
  auto it = g_static_ptr.find(device);
  if (it != g_static_ptr.end()) {
    *out = it->second;
    return cudaSuccess;
  }
  float* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(reinterpret_cast<void**>(&p), g_nvfp4_static_parts);
  if (e != cudaSuccess) return e;
  g_static_ptr[device] = p;
  *out = p;
  return cudaSuccess;
}

}  // namespace ps
