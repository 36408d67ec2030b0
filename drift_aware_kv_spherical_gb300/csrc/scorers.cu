// Alternative drift signals of the ablation, on the proxy distributions.
//
// [Polestar §2.A, drift measurement] and [Polestar §4, ablation studies]:
// the KL drift is compared against cosine dissimilarity and uncertainty-based
// selection.  The proxy kernels fuse the KL into their epilogue; this pass
// re-reads the distributions they wrote (A_cur [B][N][C], A_prev) and writes
// one signal per position, so the alternatives share the proxy attention
// and the top-k exactly and differ only in the signal:
//   KL       sum_c a ln(a / max(a', 1e-30)) over a > 0, clamped at 0
//   COSINE   1 - <a, a'> / (|a| |a'|), clamped at 0; 0 if a norm is 0
//   ENTROPY  -sum_c a ln a over a > 0 (needs no previous step)
// Without A_prev, KL and COSINE give 0.  One warp per position, lanes stride
// the C entries (coalesced rows), fp32 sums in a fixed shuffle order.
#include "ops.h"

namespace ps {
namespace {

constexpr int kScoreWarps = 8;

__global__ void __launch_bounds__(32 * kScoreWarps)
k_drift_score(const float* __restrict__ A, const float* __restrict__ A_prev, long rows, int C,
              int scorer, float* __restrict__ D) {
  pdl_prologue();
  const long row = (long)blockIdx.x * kScoreWarps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const float* a = A + row * C;
  const float* p = A_prev != nullptr ? A_prev + row * C : nullptr;
  float s0 = 0.f, s1 = 0.f, s2 = 0.f;
  if (scorer == PS_SCORER_ENTROPY) {
    for (int c = lane; c < C; c += 32) {
      const float x = a[c];
      if (x > 0.f) s0 -= x * logf(x);
    }
    s0 = warp_sum(s0);
    if (lane == 0) D[row] = s0;
    return;
  }
  if (p == nullptr) {
    if (lane == 0) D[row] = 0.f;
    return;
  }
  if (scorer == PS_SCORER_KL) {
    for (int c = lane; c < C; c += 32) {
      const float x = a[c];
      if (x > 0.f) s0 += x * logf(x / fmaxf(p[c], 1e-30f));
    }
    s0 = warp_sum(s0);
    if (lane == 0) D[row] = fmaxf(s0, 0.f);
    return;
  }
  for (int c = lane; c < C; c += 32) {  // cosine
    const float x = a[c], y = p[c];
    s0 = fmaf(x, y, s0);
    s1 = fmaf(x, x, s1);
    s2 = fmaf(y, y, s2);
  }
  s0 = warp_sum(s0);
  s1 = warp_sum(s1);
  s2 = warp_sum(s2);
  if (lane == 0)
    D[row] = (s1 > 0.f && s2 > 0.f) ? fmaxf(1.f - s0 / (sqrtf(s1) * sqrtf(s2)), 0.f) : 0.f;
}

}  // namespace

cudaError_t drift_score_run(const float* A_cur, const float* A_prev, int B, int N, int C,
                            int scorer, float* D, cudaStream_t s) {
  const long rows = (long)B * N;
  const unsigned grid = (unsigned)((rows + kScoreWarps - 1) / kScoreWarps);
  launch_pdl(k_drift_score, dim3(grid), 32 * kScoreWarps, 0, s, A_cur, A_prev, rows, C, scorer,
             D);
  return cudaGetLastError();
}

}  // namespace ps
