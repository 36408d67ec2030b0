// Offload of the quantised clusters to host memory and their fetch back.
//
// [Polestar §2.C, CPU offloading]: the quantised hidden-state clusters live
// in pinned CPU memory, only the centroids stay on the GPU, and the top-k
// clusters are fetched back asynchronously.  On GB300 the GPU reads and
// writes pinned host memory mapped into its address space over NVLink-C2C,
// so the offload and the fetch are kernels: the store of a step is written
// by the GPU itself (no host copy call, no host synchronisation on the
// selection), and the fetch reads only the selected clusters' records.
//
//   k_pack_clusters   per (cluster, window): its rows in ascending position
//                     (block scans), its record range (rows of lower
//                     clusters counted on the way), records copied with
//                     16-byte stores into the store
//   k_fetch_dequant   per selected record: E2M1 codes and E4M3 block scales
//                     read from the store, h~ = fl(fl(rho mu) + fl(v fl(s S)))
//                     in fp32 (no contraction), rounded to bf16 into the row
//
// Record of a row: codes (d/2 bytes) then scales (d/16 bytes), each padded
// to 16 bytes; records grouped by cluster, ascending position inside one.
#include "ops.h"
#include "vec.cuh"

namespace ps {
namespace {

constexpr int kPackThreads = 256;

__host__ __device__ inline int up16(int x) { return (x + 15) & ~15; }

__global__ void __launch_bounds__(kPackThreads)
k_pack_clusters(const uint8_t* __restrict__ codes, const uint8_t* __restrict__ scales,
                const int32_t* __restrict__ assign, int N, int d, int C,
                uint8_t* __restrict__ store, int32_t* __restrict__ order,
                int32_t* __restrict__ cl_off) {
  extern __shared__ int s_members[];  // [N]
  __shared__ int s_scan[32];
  const int c = blockIdx.x, b = blockIdx.y, tid = threadIdx.x;
  const int32_t* a = assign + (long)b * N;
  // the cluster's first record: rows of the clusters before it
  int below = 0;
  for (int i = tid; i < N; i += kPackThreads) {
    const int ai = a[i];
    below += (ai >= 0 && ai < c) ? 1 : 0;
  }
  int start;
  block_exclusive_scan<int>(below, s_scan, &start);
  // members in ascending position, 256 rows a round
  int n = 0;
  for (int base = 0; base < N; base += kPackThreads) {
    const int i = base + tid;
    const int m = (i < N && a[i] == c) ? 1 : 0;
    int tot;
    const int at = block_exclusive_scan<int>(m, s_scan, &tot);
    if (m) s_members[n + at] = i;
    n += tot;
  }
  __syncthreads();
  if (tid == 0) {
    cl_off[(long)b * (C + 1) + c] = start;
    if (c == C - 1) cl_off[(long)b * (C + 1) + C] = start + n;
  }
  const int half = d / 2, q = d / 16, rec = up16(half) + up16(q);
  const int v16 = rec / 16;  // 16-byte vectors per record
  const int code_v = half / 16;  // whole code vectors (d % 32 == 0)
  for (int it = tid; it < n * v16; it += kPackThreads) {
    const int m = it / v16, v = it % v16;
    const int i = s_members[m];
    const int r = start + m;
    if (v == 0) order[(long)b * N + r] = i;
    uint4 w = make_uint4(0u, 0u, 0u, 0u);
    if (v < code_v) {
      w = __ldg(reinterpret_cast<const uint4*>(codes + ((long)b * N + i) * half) + v);
    } else if (v >= up16(half) / 16) {  // scales part: byte by byte (d/16 need not be aligned)
      const int s0 = (v - up16(half) / 16) * 16;
      uint32_t word[4] = {0u, 0u, 0u, 0u};
      const uint8_t* src = scales + ((long)b * N + i) * q;
#pragma unroll
      for (int e = 0; e < 16; ++e)
        if (s0 + e < q) word[e >> 2] |= static_cast<uint32_t>(src[s0 + e]) << (8 * (e & 3));
      w = make_uint4(word[0], word[1], word[2], word[3]);
    }
    reinterpret_cast<uint4*>(store + ((long)b * N + r) * rec)[v] = w;
  }
}

__device__ __forceinline__ float e2m1_value(uint32_t code) {
  // magnitudes of codes 0..7: 0, 0.5, 1, 1.5, 2, 3, 4, 6 (two exponent bits,
  // bias 1, one mantissa bit; exponent 0 is subnormal: m * 0.5)
  const uint32_t e = (code >> 1) & 3u, m = code & 1u;
  const float mag = e == 0u ? 0.5f * (float)m : __uint_as_float((e + 126u) << 23 | m << 22);
  return (code & 8u) ? -mag : mag;
}

__device__ __forceinline__ float e4m3_value(uint32_t code) {
  // non-negative block scales as the quantiser writes them: 4 exponent bits
  // (bias 7), 3 mantissa bits; exponent 0 is subnormal: m * 2^-9
  const uint32_t e = (code >> 3) & 15u, m = code & 7u;
  const float mag =
      e == 0u ? (float)m * 0.001953125f : __uint_as_float((e + 120u) << 23 | m << 20);
  return (code & 0x80u) ? -mag : mag;
}

// grid (N, B): CTA x of window b takes the x-th record of the window's
// selected clusters (in the order of sel), if there is one.
__global__ void __launch_bounds__(256)
k_fetch_dequant(const uint8_t* __restrict__ store, const int32_t* __restrict__ order,
                const int32_t* __restrict__ cl_off, const int32_t* __restrict__ sel, int k,
                const float* __restrict__ mu, const float* __restrict__ rho,
                const float* __restrict__ tensor_scale, int N, int d, int C,
                __nv_bfloat16* __restrict__ Ht) {
  const int x = blockIdx.x, b = blockIdx.y;
  const int32_t* off = cl_off + (long)b * (C + 1);
  int acc = 0, c = -1, r = -1;
  for (int j = 0; j < k; ++j) {
    const int cj = sel[(long)b * k + j];
    if (cj < 0 || cj >= C) continue;
    const int n = off[cj + 1] - off[cj];
    if (x < acc + n) {
      c = cj;
      r = off[cj] + (x - acc);
      break;
    }
    acc += n;
  }
  if (c < 0 || r < 0 || r >= N) return;
  const int i = order[(long)b * N + r];
  if (i < 0 || i >= N) return;
  const int half = d / 2, q = d / 16, rec = up16(half) + up16(q);
  const uint8_t* recp = store + ((long)b * N + r) * rec;
  const float S = tensor_scale[b];
  const float rh = rho[(long)b * N + i];
  const float* mc = mu + ((long)b * C + c) * d;
  __nv_bfloat16* out = Ht + ((long)b * N + i) * d;
  for (int blk = threadIdx.x; blk < q; blk += blockDim.x) {  // 16 elements each
    const uint2 cw = *reinterpret_cast<const uint2*>(recp + blk * 8);
    const float g = __fmul_rn(e4m3_value(recp[up16(half) + blk]), S);
    float mv[16];
#pragma unroll
    for (int e = 0; e < 16; e += 4) {
      const float4 m4 = *reinterpret_cast<const float4*>(mc + blk * 16 + e);
      mv[e] = m4.x; mv[e + 1] = m4.y; mv[e + 2] = m4.z; mv[e + 3] = m4.w;
    }
    uint32_t packed[8];
#pragma unroll
    for (int e = 0; e < 16; e += 2) {
      const uint32_t word = e < 8 ? cw.x : cw.y;
      const uint32_t byte = (word >> (8 * ((e >> 1) & 3))) & 0xffu;
      float h2[2];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const float v = e2m1_value(u == 0 ? (byte & 0xfu) : (byte >> 4));
        h2[u] = __fadd_rn(__fmul_rn(rh, mv[e + u]), __fmul_rn(v, g));
      }
      const __nv_bfloat162 p = __floats2bfloat162_rn(h2[0], h2[1]);
      packed[e >> 1] = *reinterpret_cast<const uint32_t*>(&p);
    }
    uint4* o = reinterpret_cast<uint4*>(out + blk * 16);
    o[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
    o[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
  }
}

}  // namespace

size_t store_record_bytes(int d) { return (size_t)(up16(d / 2) + up16(d / 16)); }

cudaError_t pack_clusters_run(const uint8_t* codes, const uint8_t* scales, const int32_t* assign,
                              int B, int N, int d, int C, uint8_t* store, int32_t* order,
                              int32_t* cl_off, cudaStream_t s) {
  const size_t smem = (size_t)N * sizeof(int);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(k_pack_clusters,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  launch_pdl(k_pack_clusters, dim3(C, B), kPackThreads, smem, s, codes, scales, assign, N, d, C,
             store, order, cl_off);
  return cudaGetLastError();
}

cudaError_t fetch_dequant_run(const uint8_t* store, const int32_t* order, const int32_t* cl_off,
                              const int32_t* sel, int k, const float* mu, const float* rho,
                              const float* tensor_scale, int B, int N, int d, int C,
                              __nv_bfloat16* Ht, cudaStream_t s) {
  launch_pdl(k_fetch_dequant, dim3(N, B), 256, 0, s, store, order, cl_off, sel, k, mu, rho,
             tensor_scale, N, d, C, Ht);
  return cudaGetLastError();
}

}  // namespace ps
