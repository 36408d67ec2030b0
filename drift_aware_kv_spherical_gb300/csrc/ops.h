// Internal launchers of libpolestar; api.cu validates arguments and calls
// these.  Each returns the first CUDA error of its launches.
#pragma once

#include "common.cuh"

namespace ps {

struct KmeansArgs {
  const void* H; int dtype; int B, N, d, C, iters, init_mode;
  const double* init_u;
  float* mu; int32_t* assign; float* rho; float* chat; int32_t* counts;
  float* obj; void* ws; int* status; int num_sms;
  cudaStream_t aux;  // captures conditional-node bodies (the handle's own stream)
};
size_t kmeans_ws(int B, int N, int d, int C);
cudaError_t kmeans_run(const KmeansArgs& a, cudaStream_t s);

// k-means passes in Gram form (kmeans_gram.cu): bf16 windows of N <= 1024
// rows whose cosine Gram matrix fits one thread-block cluster's shared memory.
struct GramPlan {
  bool ok;
  int R, Z;      // rows per CTA, CTAs per window of the pass kernel
  size_t smem;   // its shared memory per CTA
  int mtb, T0, T;  // 128-row blocks, upper-triangle tiles per window, all tiles
  bool fused0;     // C <= 64: pass 0's cosines are tiles of the Gram GEMM
  int KB, kpc, nz;  // the Gram GEMM's K blocks and split
};
GramPlan gram_plan(int dtype, int B, int N, int d, int C);
bool gram_launchable(const GramPlan& g);
// K = X X^T of every window in 24-bit fixed point (qhi/qlo: B * Z * N * R
// each); with mu_split ([B][2C][d] hi then lo rows of the given centroids)
// also the pass-0 cosines cos0 [B][N][C]
cudaError_t gram_build(const GramPlan& g, const __nv_bfloat16* H, const float* inv, int B,
                       int N, int d, int C, const __nv_bfloat16* mu_split, float* cos0,
                       int16_t* qhi, uint8_t* qlo, int* status, cudaStream_t s);
// k-means++ seeds of every window from its K (after gram_build without
// mu_split): mu [B][C][d] and pass 0's cosines L [B][N][C]; N <= 1024
cudaError_t gram_seed(const GramPlan& g, const __nv_bfloat16* H, const float* inv,
                      const double* U, int B, int N, int d, int C, const int16_t* qhi,
                      const uint8_t* qlo, float* mu, float* L, cudaStream_t s);
// passes 1..passes from the labels in assign and the cosines L of pass 0
// (objp0 == nullptr: pass 0 itself too, from L);
// leaves the last pass's labels in assign, the pass before's in prev, rho,
// the objectives, and in mu the centroids that stopped being formed
cudaError_t gram_iterate(const GramPlan& g, const int16_t* qhi, const uint8_t* qlo, int B, int N,
                         int C, int passes, const __nv_bfloat16* H, int d, const float* inv,
                         float* mu, int32_t* assign, int32_t* prev, float* rho, float* L,
                         const float* objp0, int ntile0, float* obj, int obj_ld, int* status,
                         cudaStream_t s);

// offload of the quantised clusters (offload.cu)
size_t store_record_bytes(int d);
cudaError_t pack_clusters_run(const uint8_t* codes, const uint8_t* scales, const int32_t* assign,
                              int B, int N, int d, int C, uint8_t* store, int32_t* order,
                              int32_t* cl_off, cudaStream_t s);
cudaError_t fetch_dequant_run(const uint8_t* store, const int32_t* order, const int32_t* cl_off,
                              const int32_t* sel, int k, const float* mu, const float* rho,
                              const float* tensor_scale, int B, int N, int d, int C,
                              __nv_bfloat16* Ht, cudaStream_t s);

struct Nvfp4Args {
  const void* H; int dtype; const float* mu; const int32_t* assign;
  const float* rho; int B, N, d, C;
  uint8_t* codes; uint8_t* scales; float* S; void* ws; int num_sms;
};
size_t nvfp4_ws(int B, int N, int d);
cudaError_t nvfp4_run(const Nvfp4Args& a, cudaStream_t s);
// no-workspace variant: a file-scope device array replaces the workspace
bool nvfp4_static_fits(int B, int N, int d);
cudaError_t nvfp4_static_scratch(int device, float** out);

struct ProxyArgs {
  const void* Q; const float* chat; const void* Wk; int dtype;
  int B, N, d, C, Hq, Hkv, dh;
  const float* A_prev; float* A_cur; float* D; void* ws; int num_sms;
  int* status;
};
size_t proxy_ws(int B, int N, int d, int C, int Hq, int Hkv, int dh);
cudaError_t proxy_run(const ProxyArgs& a, cudaStream_t s);

// ablation drift signals over the proxy distributions (PS_SCORER_*)
cudaError_t drift_score_run(const float* A_cur, const float* A_prev, int B, int N, int C,
                            int scorer, float* D, cudaStream_t s);

struct TopkArgs {
  const float* D; const int32_t* assign; const int32_t* counts;
  int B, N, C, k;
  int32_t* sel; float* sel_score; int32_t* pos; int32_t* npos; uint8_t* posmask;
};
cudaError_t topk_run(const TopkArgs& a, cudaStream_t s);

struct RefreshArgs {
  const void* H; int dtype; const int32_t* pos; const int32_t* npos;
  const void* Wk; const void* Wv; int B, N, d, Hkv, dh;
  void* Kc; void* Vc; int Ncache, cache_off; int num_sms;
  void* ws; int* status;
};
bool refresh_tc_ok(int dtype, int Hkv, int dh);
size_t refresh_ws(int B, int N, int d, int Hkv, int dh);
cudaError_t refresh_run(const RefreshArgs& a, cudaStream_t s);

struct CommitArgs {
  const void* logits; int dtype; int B, P, V; const uint8_t* role; uint8_t* undecided;
  const float* D; int d_ld; float* d_sum; int32_t* d_cnt; float* d_prev;
  const uint8_t* suffix_sel; int sel_ld; ps_commit_params p;
  int32_t* token; float* conf; uint8_t* commit; void* ws;
};
size_t commit_ws(int B, int P, int V);
cudaError_t commit_run(const CommitArgs& a, cudaStream_t s);
cudaError_t block_progress_run(const uint8_t* commit, const uint8_t* undecided,
                               const uint8_t* role, int B, int P, int32_t* out,
                               cudaStream_t s);

}  // namespace ps
