// a7: token confidence and the drift-aware commit rule.
//
// [Polestar §2.B, current block commitment]: a current-block token commits
// when its drift delta exceeds tau_d = alpha (tau_s - c)^2 (or its confidence
// reaches tau_s).  [Polestar §2.B, suffix block commitment]: a suffix token
// whose cluster is among the last layer's top-drift clusters commits only
// with c >= tau_s.
//
//   k_commit_scan  one CTA per 16384-logit chunk of a row: chunk max, first
//                  arg-max, sum exp(l - chunk max) (fp32 pairwise per thread,
//                  fp64 across threads).  Streaming loads of fp32 logits,
//                  or of bf16 ones (exact in fp32; 8 a load where V % 8 == 0,
//                  which groups the per-thread partial sums differently).
//   k_commit_rule  one CTA per sequence: merges the chunks in fp64
//                  (c = 1 / sum), applies the rule, updates the state.
#include <climits>

#include "ops.h"
#include "vec.cuh"

namespace ps {
namespace {

constexpr int kCT = 256;          // threads per scan CTA
constexpr int kPer = 64;          // logits per thread
constexpr int kChunk = kCT * kPer;

// W consecutive logits from W * sizeof(T) aligned bytes (16 bytes, or 8 for
// four bf16 when rows are only 8-byte aligned), streamed past the caches
__device__ __forceinline__ void loadw(const float* p, float* x) {
  const float4 w = __ldcs(reinterpret_cast<const float4*>(p));
  x[0] = w.x; x[1] = w.y; x[2] = w.z; x[3] = w.w;
}
__device__ __forceinline__ void loadw(const __nv_bfloat16* p, float* x, int w_elems) {
  if (w_elems == 8) {
    const uint4 w = __ldcs(reinterpret_cast<const uint4*>(p));
    bf16x2_to_f32(w.x, x[0], x[1]);
    bf16x2_to_f32(w.y, x[2], x[3]);
    bf16x2_to_f32(w.z, x[4], x[5]);
    bf16x2_to_f32(w.w, x[6], x[7]);
  } else {
    const uint2 w = __ldcs(reinterpret_cast<const uint2*>(p));
    bf16x2_to_f32(w.x, x[0], x[1]);
    bf16x2_to_f32(w.y, x[2], x[3]);
  }
}
__device__ __forceinline__ void loadw(const float* p, float* x, int) { loadw(p, x); }

// W logits per load: 4 (fp32; bf16 with V % 8 != 0) or 8 (bf16, V % 8 == 0)
template <typename T, int W>
__global__ void __launch_bounds__(kCT)
k_commit_scan(const T* __restrict__ logits, int V, int nchunk,
              float* __restrict__ pm, int* __restrict__ pidx,
              double* __restrict__ ps) {
  pdl_prologue();
  __shared__ float s_m[kCT / 32];
  __shared__ int s_i[kCT / 32];
  __shared__ double s_s[kCT / 32];
  const long row = blockIdx.y;
  const int chunk = blockIdx.x, tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  const T* L = logits + row * V;
  const int c0 = chunk * kChunk;
  float v[kPer];
#pragma unroll
  for (int it = 0; it < kPer / W; ++it) {
    const int e = c0 + (it * kCT + tid) * W;
#pragma unroll
    for (int q = 0; q < W; ++q) v[it * W + q] = -INFINITY;
    if (e < V) loadw(L + e, v + it * W, W);  // V % W == 0: the group is whole
  }
  // chunk max and its first index (each thread scans its indices in order)
  float m = -INFINITY;
  int mi = INT_MAX;
#pragma unroll
  for (int it = 0; it < kPer / W; ++it)
#pragma unroll
    for (int q = 0; q < W; ++q)
      if (v[it * W + q] > m) { m = v[it * W + q]; mi = c0 + (it * kCT + tid) * W + q; }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float om = __shfl_xor_sync(0xffffffffu, m, o);
    const int oi = __shfl_xor_sync(0xffffffffu, mi, o);
    if (om > m || (om == m && oi < mi)) { m = om; mi = oi; }
  }
  if (lane == 0) { s_m[warp] = m; s_i[warp] = mi; }
  __syncthreads();
  m = s_m[0];
  mi = s_i[0];
  for (int w = 1; w < kCT / 32; ++w)
    if (s_m[w] > m || (s_m[w] == m && s_i[w] < mi)) { m = s_m[w]; mi = s_i[w]; }
  // sum of exp(l - m): pairwise in registers, then fp64 across the block
#pragma unroll
  for (int e = 0; e < kPer; ++e) v[e] = expf(v[e] - m);
#pragma unroll
  for (int w = kPer / 2; w > 0; w >>= 1)
#pragma unroll
    for (int e = 0; e < w; ++e) v[e] += v[e + w];
  double s = warp_sum_f64((double)v[0]);
  if (lane == 0) s_s[warp] = s;
  __syncthreads();
  if (tid == 0) {
    double t = 0.0;
    for (int w = 0; w < kCT / 32; ++w) t += s_s[w];
    pm[row * nchunk + chunk] = m;
    pidx[row * nchunk + chunk] = mi;
    ps[row * nchunk + chunk] = t;
  }
}

__global__ void __launch_bounds__(1024)
k_commit_rule(int P, int nchunk, const float* __restrict__ pm,
              const int* __restrict__ pidx, const double* __restrict__ ps,
              const uint8_t* __restrict__ role, uint8_t* __restrict__ undecided,
              const float* __restrict__ Dblk, int d_ld, float* __restrict__ d_sum,
              int32_t* __restrict__ d_cnt, float* __restrict__ d_prev,
              const uint8_t* __restrict__ suffix_sel, int sel_ld,
              ps_commit_params p, int32_t* __restrict__ token,
              float* __restrict__ conf, uint8_t* __restrict__ commit) {
  pdl_prologue();
  __shared__ double s_c[32];
  __shared__ int s_j[32];
  const int b = blockIdx.x, j = threadIdx.x;
  const int lane = j & 31, warp = j >> 5;
  const bool valid = j < P;
  const long row = (long)b * P + j;
  double c = 0.0;
  int tok = 0;
  if (valid) {
    float M = -INFINITY;
    for (int q = 0; q < nchunk; ++q) M = fmaxf(M, pm[row * nchunk + q]);
    tok = INT_MAX;
    double s = 0.0;
    for (int q = 0; q < nchunk; ++q) {
      const float mq = pm[row * nchunk + q];
      if (mq == M && tok == INT_MAX) tok = pidx[row * nchunk + q];
      // chunk rescale in fp32 (mq <= M; expf is within 2 ulp) -- fp64 exp is
      // a long software sequence here
      s += ps[row * nchunk + q] * (double)expf(mq - M);
    }
    c = 1.0 / s;
  }
  const int rl = valid ? role[j] : 2;
  const int und = valid ? undecided[row] : 0;
  const double tau = (double)p.tau_s;
  int cm = 0;
  if (und && rl == 0) {
    bool ok = c >= tau;
    const int n = d_cnt[row];
    if (n >= 1) {
      const double D = (double)Dblk[(long)b * d_ld + j];
      if (p.mode == 2) {
        ok = ok || D < (double)p.ratio * (double)d_prev[row];
      } else {
        const double mean = (double)d_sum[row] / (double)n;
        const double delta = p.mode == 0 ? mean - D : D - mean;
        const double gap = tau - c;
        ok = ok || delta > (double)p.alpha * (gap * gap);
      }
    }
    cm = ok ? 1 : 0;
  } else if (und && rl == 1) {
    cm = (suffix_sel != nullptr && suffix_sel[(long)b * sel_ld + j] && c >= tau) ? 1 : 0;
  }
  const int cur_und = (und && rl == 0) ? 1 : 0;
  const int any_commit = __syncthreads_or(cur_und && cm);
  const int any_und = __syncthreads_or(cur_und);
  if (p.ensure_progress && any_und && !any_commit) {
    // largest confidence among undecided current tokens, ties to lower j
    double bc = cur_und ? c : -1.0;
    int bj = cur_und ? j : INT_MAX;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const double oc = __shfl_xor_sync(0xffffffffu, bc, o);
      const int oj = __shfl_xor_sync(0xffffffffu, bj, o);
      if (oc > bc || (oc == bc && oj < bj)) { bc = oc; bj = oj; }
    }
    if (lane == 0) { s_c[warp] = bc; s_j[warp] = bj; }
    __syncthreads();
    bc = s_c[0];
    bj = s_j[0];
    for (int w = 1; w < (int)(blockDim.x >> 5); ++w)
      if (s_c[w] > bc || (s_c[w] == bc && s_j[w] < bj)) { bc = s_c[w]; bj = s_j[w]; }
    if (j == bj) cm = 1;
  }
  if (!valid) return;
  if (cur_und) {
    const float D = Dblk[(long)b * d_ld + j];
    d_sum[row] = __fadd_rn(d_sum[row], D);
    d_cnt[row] = d_cnt[row] + 1;
    d_prev[row] = D;
  }
  if (cm) undecided[row] = 0;
  token[row] = tok;
  conf[row] = (float)c;
  commit[row] = (uint8_t)cm;
}

int nchunks(int V) { return ceil_div(V, kChunk); }

// The decode loop's outcome of a step, one CTA: out[0] = the largest number
// of positions any sequence committed, out[1] = 1 when no sequence has an
// undecided current-block position left.  A warp per sequence.
__global__ void __launch_bounds__(256)
k_block_progress(const uint8_t* __restrict__ commit, const uint8_t* __restrict__ undecided,
                 const uint8_t* __restrict__ role, int B, int P, int32_t* __restrict__ out) {
  pdl_prologue();
  __shared__ int s_max, s_open;
  if (threadIdx.x == 0) { s_max = 0; s_open = 0; }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  int open = 0;
  for (int b = warp; b < B; b += nw) {
    int n = 0;
    for (int j = lane; j < P; j += 32) {
      const long row = (long)b * P + j;
      n += commit[row] != 0;
      open |= undecided[row] != 0 && role[j] == 0;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) n += __shfl_xor_sync(0xffffffffu, n, o);
    if (lane == 0) atomicMax(&s_max, n);
  }
  if (__syncthreads_or(open) && threadIdx.x == 0) s_open = 1;
  __syncthreads();
  if (threadIdx.x == 0) {
    out[0] = s_max;
    out[1] = s_open ? 0 : 1;
  }
}

}  // namespace

cudaError_t block_progress_run(const uint8_t* commit, const uint8_t* undecided,
                               const uint8_t* role, int B, int P, int32_t* out,
                               cudaStream_t s) {
  launch_pdl(k_block_progress, 1, 256, 0, s, commit, undecided, role, B, P, out);
  return cudaGetLastError();
}

size_t commit_ws(int B, int P, int V) {
  const size_t rows = (size_t)B * P * nchunks(V);
  Carver cv(nullptr);
  cv.take<float>(rows);
  cv.take<int>(rows);
  cv.take<double>(rows);
  return cv.bytes();
}

cudaError_t commit_run(const CommitArgs& a, cudaStream_t s) {
  const int nc = nchunks(a.V);
  const size_t rows = (size_t)a.B * a.P * nc;
  Carver cv(a.ws);
  float* pm = cv.take<float>(rows);
  int* pidx = cv.take<int>(rows);
  double* ps = cv.take<double>(rows);
  const dim3 grid(nc, a.B * a.P);
  const auto* lb = static_cast<const __nv_bfloat16*>(a.logits);
  if (a.dtype == PS_BF16 && a.V % 8 == 0)
    launch_pdl(k_commit_scan<__nv_bfloat16, 8>, grid, kCT, 0, s, lb, a.V, nc, pm, pidx, ps);
  else if (a.dtype == PS_BF16)
    launch_pdl(k_commit_scan<__nv_bfloat16, 4>, grid, kCT, 0, s, lb, a.V, nc, pm, pidx, ps);
  else
    launch_pdl(k_commit_scan<float, 4>, grid, kCT, 0, s, static_cast<const float*>(a.logits),
               a.V, nc, pm, pidx, ps);
  const int threads = ((a.P + 31) / 32) * 32;
  launch_pdl(k_commit_rule, a.B, threads, 0, s, a.P, nc, pm, pidx, ps, a.role, a.undecided,
                                        a.D, a.d_ld, a.d_sum, a.d_cnt, a.d_prev,
                                        a.suffix_sel, a.sel_ld, a.p, a.token, a.conf,
                                        a.commit);
  return cudaGetLastError();
}

}  // namespace ps
