// The C ABI of libpolestar: handle management, argument validation,
// workspace sizing and dispatch to the kernels.  Declarations and the
// meaning of every argument are in include/polestar.h.
#include <cstdio>
#include <cstdint>
#include <cstring>
#include <new>
#include <vector>

#include "ops.h"

namespace ps {

struct TraceRec {
  const void* kernel;
  cudaEvent_t a, b;
};
struct TraceSink {
  std::vector<TraceRec> recs;
  cudaEvent_t pending = nullptr;
};

// The calling thread's sink while it runs a ps_* call on a tracing handle.
thread_local TraceSink* g_trace = nullptr;

void trace_begin(cudaStream_t s) {
  if (g_trace == nullptr) return;
  cudaEvent_t a;
  if (cudaEventCreate(&a) != cudaSuccess) return;
  cudaEventRecord(a, s);
  g_trace->pending = a;
}

void trace_end(cudaStream_t s, const void* kernel) {
  if (g_trace == nullptr || g_trace->pending == nullptr) return;
  cudaEvent_t b;
  if (cudaEventCreate(&b) != cudaSuccess) {
    cudaEventDestroy(g_trace->pending);
    g_trace->pending = nullptr;
    return;
  }
  cudaEventRecord(b, s);
  g_trace->recs.push_back({kernel, g_trace->pending, b});
  g_trace->pending = nullptr;
}

}  // namespace ps

using namespace ps;

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

#define PS_REQUIRE(cond) \
  do {                   \
    if (!(cond)) return PS_ERR_ARG; \
  } while (0)

#define PS_PTR(p) PS_REQUIRE((p) != nullptr && aligned16(p))
#define PS_OPT_PTR(p) PS_REQUIRE((p) == nullptr || aligned16(p))
// arrays read or written one element at a time only need to exist
#define PS_NN(p) PS_REQUIRE((p) != nullptr)

thread_local char g_last_cuda_error[192] = "";

ps_status launch_status(cudaError_t e) {
  if (e == cudaSuccess) return PS_OK;
  std::snprintf(g_last_cuda_error, sizeof(g_last_cuda_error), "%s: %s", cudaGetErrorName(e),
                cudaGetErrorString(e));
  return PS_ERR_CUDA;
}

ps_status check_ws(size_t need, const void* ws, size_t ws_bytes) {
  if (need == 0) return PS_OK;
  if (ws == nullptr || ws_bytes < need) return PS_ERR_WORKSPACE;
  if (!aligned16(ws)) return PS_ERR_ARG;
  return PS_OK;
}

bool dtype_ok(int dt) { return dt == PS_F32 || dt == PS_BF16; }

// Sets the calling thread's trace sink for the duration of one ps_* call.
struct TraceScope {
  explicit TraceScope(ps_handle h) { g_trace = h != nullptr ? h->trace : nullptr; }
  ~TraceScope() { g_trace = nullptr; }
};

void trace_clear(TraceSink* t) {
  for (auto& r : t->recs) {
    cudaEventDestroy(r.a);
    cudaEventDestroy(r.b);
  }
  t->recs.clear();
}

constexpr int kMaxC = 256;
constexpr int kMaxD = 8192;
constexpr int kMaxDh = 256;

}  // namespace

extern "C" {

ps_status ps_create(int device, ps_handle* out) {
  if (out == nullptr) return PS_ERR_ARG;
  *out = nullptr;
  int n = 0;
  if (cudaGetDeviceCount(&n) != cudaSuccess || device < 0 || device >= n)
    return PS_ERR_ARG;
  cudaDeviceProp prop;
  cudaError_t e = cudaGetDeviceProperties(&prop, device);
  if (e != cudaSuccess) return launch_status(e);
  if (!(prop.major == 10 && prop.minor == 3)) return PS_ERR_UNSUPPORTED;
  e = cudaSetDevice(device);
  if (e != cudaSuccess) return launch_status(e);
  auto* h = new (std::nothrow) ps_handle_s;
  if (h == nullptr) return PS_ERR_CUDA;
  h->device = device;
  h->num_sms = prop.multiProcessorCount;
  h->status = nullptr;
  h->trace = nullptr;
  h->aux = nullptr;
  e = cudaMalloc(&h->status, 16);
  if (e == cudaSuccess) e = cudaMemset(h->status, 0, 16);
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&h->aux, cudaStreamNonBlocking);
  if (e != cudaSuccess) {
    if (h->status) cudaFree(h->status);
    if (h->aux) cudaStreamDestroy(h->aux);
    delete h;
    return launch_status(e);
  }
  *out = h;
  return PS_OK;
}

ps_status ps_destroy(ps_handle h) {
  if (h == nullptr) return PS_ERR_ARG;
  if (h->trace != nullptr) {
    trace_clear(h->trace);
    delete h->trace;
  }
  cudaFree(h->status);
  if (h->aux) cudaStreamDestroy(h->aux);
  delete h;
  return PS_OK;
}

ps_status ps_check(ps_handle h, void* stream, int synchronize) {
  if (h == nullptr) return PS_ERR_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = synchronize ? cudaStreamSynchronize(s) : cudaSuccess;
  if (e != cudaSuccess) return launch_status(e);
  int word = 0;
  e = cudaMemcpyAsync(&word, h->status, sizeof(int), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return launch_status(e);
  if (word != 0) {
    cudaMemsetAsync(h->status, 0, sizeof(int), s);
    cudaStreamSynchronize(s);
    return word == PS_ERR_TIMEOUT ? PS_ERR_TIMEOUT : PS_ERR_CUDA;
  }
  return PS_OK;
}

const char* ps_status_string(ps_status s) {
  switch (s) {
    case PS_OK: return "ok";
    case PS_ERR_ARG: return "invalid argument";
    case PS_ERR_UNSUPPORTED: return "unsupported device (needs sm_103)";
    case PS_ERR_WORKSPACE: return "workspace too small";
    case PS_ERR_CUDA: return "CUDA error";
    case PS_ERR_TIMEOUT: return "device-side wait timed out";
  }
  return "unknown status";
}

const char* ps_last_cuda_error(void) { return g_last_cuda_error; }

ps_status ps_trace_enable(ps_handle h, int enable) {
  if (h == nullptr) return PS_ERR_ARG;
  if (h->trace != nullptr) {
    trace_clear(h->trace);
    delete h->trace;
    h->trace = nullptr;
  }
  if (enable) {
    h->trace = new (std::nothrow) TraceSink;
    if (h->trace == nullptr) return PS_ERR_CUDA;
  }
  return PS_OK;
}

int ps_trace_count(ps_handle h) {
  return h != nullptr && h->trace != nullptr ? static_cast<int>(h->trace->recs.size()) : 0;
}

ps_status ps_trace_get(ps_handle h, int i, const char** name, float* ms) {
  if (h == nullptr || h->trace == nullptr || name == nullptr || ms == nullptr || i < 0 ||
      i >= static_cast<int>(h->trace->recs.size()))
    return PS_ERR_ARG;
  const TraceRec& r = h->trace->recs[i];
  cudaError_t e = cudaEventSynchronize(r.b);
  if (e == cudaSuccess) e = cudaEventElapsedTime(ms, r.a, r.b);
  if (e == cudaSuccess) e = cudaFuncGetName(name, r.kernel);
  return launch_status(e);
}

size_t ps_workspace_bytes(int op, int B, int N, int d, int C, int Hq, int Hkv,
                          int dh, int k, int P, int V) {
  (void)k;
  if (B <= 0) return 0;
  switch (op) {
    case PS_OP_KMEANS: return (N > 0 && C > 0) ? kmeans_ws(B, N, d, C) : 0;
    case PS_OP_NVFP4: return (N > 0 && d > 0) ? nvfp4_ws(B, N, d) : 0;
    case PS_OP_PROXY_KL:
      return (N > 0 && C > 0 && Hkv > 0 && dh > 0 && Hq > 0)
                 ? proxy_ws(B, N, d, C, Hq, Hkv, dh) : 0;
    case PS_OP_TOPK: return 0;
    case PS_OP_REFRESH:
      return (N > 0 && d > 0 && Hkv > 0 && dh > 0) ? refresh_ws(B, N, d, Hkv, dh) : 0;
    case PS_OP_COMMIT: return (P > 0 && V > 0) ? commit_ws(B, P, V) : 0;
  }
  return 0;
}

ps_status ps_kmeans_spherical(ps_handle h, const void* H, int dtype, int B,
                              int N, int d, int C, int iters, int init_mode,
                              const double* init_u, float* mu, int32_t* assign,
                              float* rho, float* chat, int32_t* counts,
                              float* objective, void* ws, size_t ws_bytes,
                              void* stream) {
  TraceScope trace_scope(h);
  PS_REQUIRE(h != nullptr && dtype_ok(dtype));
  PS_REQUIRE(B >= 0 && iters >= 0 && (init_mode == 0 || init_mode == 1));
  if (B == 0) return PS_OK;
  PS_REQUIRE(d > 0 && d % 16 == 0 && d <= kMaxD);
  PS_REQUIRE(C >= 1 && C <= kMaxC && C <= N);
  PS_REQUIRE((long)B * N <= (long)INT32_MAX / 2);
  PS_PTR(H); PS_PTR(mu); PS_NN(assign); PS_NN(rho); PS_PTR(chat); PS_NN(counts);
  if (init_mode == 1) PS_NN(init_u);
  PS_REQUIRE(B <= 65535);
  ps_status st = check_ws(kmeans_ws(B, N, d, C), ws, ws_bytes);
  if (st != PS_OK) return st;
  KmeansArgs a{H, dtype, B, N, d, C, iters, init_mode, init_u, mu, assign, rho,
               chat, counts, objective, ws, h->status, h->num_sms, h->aux};
  return launch_status(kmeans_run(a, static_cast<cudaStream_t>(stream)));
}

ps_status ps_nvfp4_residual(ps_handle h, const void* H, int dtype,
                            const float* mu, const int32_t* assign,
                            const float* rho, int B, int N, int d, int C,
                            uint8_t* codes, uint8_t* scales,
                            float* tensor_scale, void* ws, size_t ws_bytes,
                            void* stream) {
  TraceScope trace_scope(h);
  PS_REQUIRE(h != nullptr && dtype_ok(dtype));
  PS_REQUIRE(B >= 0);
  if (B == 0) return PS_OK;
  PS_REQUIRE(N >= 1 && d > 0 && d % 16 == 0 && B <= 65535);
  PS_PTR(H); PS_PTR(codes); PS_NN(scales); PS_NN(tensor_scale);
  if (mu != nullptr) {
    PS_PTR(mu); PS_NN(assign); PS_NN(rho);
    PS_REQUIRE(C >= 1);
  } else {
    PS_REQUIRE(dtype == PS_F32 || dtype == PS_BF16);
    C = 1;
  }
  ps_status st = check_ws(nvfp4_ws(B, N, d), ws, ws_bytes);
  if (st != PS_OK) return st;
  Nvfp4Args a{H, dtype, mu, assign, rho, B, N, d, C, codes, scales, tensor_scale,
              ws, h->num_sms};
  return launch_status(nvfp4_run(a, static_cast<cudaStream_t>(stream)));
}

ps_status ps_proxy_attn_kl(ps_handle h, const void* Q, const float* chat,
                           const void* Wk, int dtype, int B, int N, int d,
                           int C, int Hq, int Hkv, int dh, const float* A_prev,
                           float* A_cur, float* D, void* ws, size_t ws_bytes,
                           void* stream) {
  TraceScope trace_scope(h);
  PS_REQUIRE(h != nullptr && dtype_ok(dtype));
  PS_REQUIRE(B >= 0);
  if (B == 0) return PS_OK;
  PS_REQUIRE(N >= 1 && d > 0 && d % 16 == 0 && B <= 65535);
  PS_REQUIRE(C >= 1 && C <= kMaxC);
  PS_REQUIRE(Hkv >= 1 && Hq >= Hkv && Hq % Hkv == 0);
  PS_REQUIRE(dh > 0 && dh % 16 == 0 && dh <= kMaxDh);
  PS_PTR(Q); PS_PTR(chat); PS_PTR(Wk); PS_NN(A_cur); PS_NN(D);
  ps_status st = check_ws(proxy_ws(B, N, d, C, Hq, Hkv, dh), ws, ws_bytes);
  if (st != PS_OK) return st;
  ProxyArgs a{Q, chat, Wk, dtype, B, N, d, C, Hq, Hkv, dh, A_prev, A_cur, D, ws,
              h->num_sms, h->status};
  return launch_status(proxy_run(a, static_cast<cudaStream_t>(stream)));
}

ps_status ps_topk_drift(ps_handle h, const float* D, const int32_t* assign,
                        const int32_t* counts, int B, int N, int C, int k,
                        int32_t* sel, float* sel_score, int32_t* pos,
                        int32_t* npos, uint8_t* posmask, void* ws,
                        size_t ws_bytes, void* stream) {
  TraceScope trace_scope(h);
  (void)ws; (void)ws_bytes;
  PS_REQUIRE(h != nullptr && B >= 0);
  if (B == 0) return PS_OK;
  PS_REQUIRE(N >= 1 && C >= 1 && C <= kMaxC && C <= N && k >= 1 && k <= C);
  PS_REQUIRE(B <= 65535);
  PS_NN(D); PS_NN(assign); PS_NN(counts); PS_NN(sel); PS_NN(sel_score);
  PS_NN(pos); PS_NN(npos);
  TopkArgs a{D, assign, counts, B, N, C, k, sel, sel_score, pos, npos, posmask};
  return launch_status(topk_run(a, static_cast<cudaStream_t>(stream)));
}

ps_status ps_drift_score(ps_handle h, const float* A_cur, const float* A_prev, int B, int N,
                         int C, int scorer, float* D, void* stream) {
  TraceScope trace_scope(h);
  PS_REQUIRE(h != nullptr && B >= 0);
  if (B == 0) return PS_OK;
  PS_REQUIRE(N >= 1 && C >= 1 && C <= 4096 && (long)B * N <= 2147483647L);
  PS_REQUIRE(scorer >= PS_SCORER_KL && scorer <= PS_SCORER_ENTROPY);
  PS_NN(A_cur); PS_NN(D);
  PS_REQUIRE(D != A_cur && D != A_prev);
  return launch_status(drift_score_run(A_cur, A_prev, B, N, C, scorer, D,
                                       static_cast<cudaStream_t>(stream)));
}

ps_status ps_refresh_kv(ps_handle h, const void* H, int dtype,
                        const int32_t* pos, const int32_t* npos,
                        const void* Wk, const void* Wv, int B, int N, int d,
                        int Hkv, int dh, void* Kcache, void* Vcache,
                        int Ncache, int cache_off, void* ws, size_t ws_bytes,
                        void* stream) {
  TraceScope trace_scope(h);
  PS_REQUIRE(h != nullptr && dtype_ok(dtype) && B >= 0);
  if (B == 0) return PS_OK;
  PS_REQUIRE(N >= 1 && d > 0 && d % 16 == 0 && Hkv >= 1 && dh > 0 && dh % 16 == 0);
  PS_REQUIRE(cache_off >= 0 && (long)cache_off + N <= Ncache && B <= 65535);
  PS_REQUIRE(2L * ceil_div((long)Hkv * dh, 64) <= 65535);
  PS_PTR(H); PS_NN(pos); PS_NN(npos); PS_PTR(Wk); PS_PTR(Wv);
  PS_NN(Kcache); PS_NN(Vcache);
  const bool tc = refresh_tc_ok(dtype, Hkv, dh);
  if (tc) {
    PS_PTR(Kcache); PS_PTR(Vcache);
    ps_status st = check_ws(refresh_ws(B, N, d, Hkv, dh), ws, ws_bytes);
    if (st != PS_OK) return st;
  }
  RefreshArgs a{H, dtype, pos, npos, Wk, Wv, B, N, d, Hkv, dh, Kcache, Vcache,
                Ncache, cache_off, h->num_sms, tc ? ws : nullptr, h->status};
  return launch_status(refresh_run(a, static_cast<cudaStream_t>(stream)));
}

ps_status ps_commit(ps_handle h, const void* logits, int dtype, int B, int P, int V,
                    const uint8_t* role, uint8_t* undecided,
                    const float* D_blk, int d_ld, float* d_sum, int32_t* d_cnt,
                    float* d_prev, const uint8_t* suffix_sel, int sel_ld,
                    ps_commit_params params, int32_t* token, float* conf,
                    uint8_t* commit, void* ws, size_t ws_bytes, void* stream) {
  TraceScope trace_scope(h);
  PS_REQUIRE(h != nullptr && dtype_ok(dtype) && B >= 0 && P >= 0);
  if (B == 0 || P == 0) return PS_OK;
  PS_REQUIRE(P <= 1024 && V >= 4 && V % 4 == 0 && (long)B * P <= 65535);
  PS_REQUIRE(d_ld >= P && (suffix_sel == nullptr || sel_ld >= P));
  PS_REQUIRE(params.mode >= 0 && params.mode <= 2);
  PS_REQUIRE(params.ensure_progress == 0 || params.ensure_progress == 1);
  PS_PTR(logits); PS_NN(role); PS_NN(undecided); PS_NN(D_blk); PS_NN(d_sum);
  PS_NN(d_cnt); PS_NN(d_prev); PS_NN(token); PS_NN(conf); PS_NN(commit);
  ps_status st = check_ws(commit_ws(B, P, V), ws, ws_bytes);
  if (st != PS_OK) return st;
  CommitArgs a{logits, dtype, B, P, V, role, undecided, D_blk, d_ld, d_sum, d_cnt, d_prev,
               suffix_sel, sel_ld, params, token, conf, commit, ws};
  return launch_status(commit_run(a, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"

// The same NVFP4 residual quantisation as ps_nvfp4_residual, for callers
// that cannot allocate device memory: no workspace argument, scratch in a
// fixed 64 KiB device array inside the library.  See include/polestar.h.
extern "C" ps_status ps_nvfp4_residual_noalloc(
    ps_handle h, const void* H, int dtype, const float* mu, const int32_t* assign,
    const float* rho, int B, int N, int d, int C, uint8_t* codes, uint8_t* scales,
    float* tensor_scale, void* stream) {
  TraceScope trace_scope(h);
  PS_REQUIRE(h != nullptr && dtype_ok(dtype));
  PS_REQUIRE(B >= 0);
  if (B == 0) return PS_OK;
  PS_REQUIRE(N >= 1 && d > 0 && d % 16 == 0 && B <= 65535);
  PS_PTR(H); PS_PTR(codes); PS_NN(scales); PS_NN(tensor_scale);
  if (mu != nullptr) {
    PS_PTR(mu); PS_NN(assign); PS_NN(rho);
    PS_REQUIRE(C >= 1);
  } else {
    C = 1;
  }
  if (!nvfp4_static_fits(B, N, d)) return PS_ERR_WORKSPACE;
  // the array's address is per device: the kernels must run on the device
  // whose address is used, so the caller's current device must be the
  // handle's
  int cur = -1;
  cudaError_t e = cudaGetDevice(&cur);
  if (e != cudaSuccess) return launch_status(e);
  if (cur != h->device) return PS_ERR_ARG;
  float* scratch = nullptr;
  e = nvfp4_static_scratch(h->device, &scratch);
  if (e != cudaSuccess) return launch_status(e);
  Nvfp4Args a{H, dtype, mu, assign, rho, B, N, d, C, codes, scales, tensor_scale,
              scratch, h->num_sms};
  return launch_status(nvfp4_run(a, static_cast<cudaStream_t>(stream)));
}

// ---- offload of the quantised clusters; see include/polestar.h
namespace {
// device memory, or host memory mapped into this device's address space
bool device_accessible(const void* p) {
  cudaPointerAttributes at{};
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged ||
         (at.type == cudaMemoryTypeHost && at.devicePointer == p);
}
}  // namespace

extern "C" ps_status ps_block_progress(ps_handle h, const uint8_t* commit,
                                       const uint8_t* undecided, const uint8_t* role, int B,
                                       int P, int32_t* out, void* stream) {
  TraceScope trace_scope(h);
  PS_REQUIRE(h != nullptr && B >= 0 && P >= 0);
  PS_NN(out);
  PS_REQUIRE((reinterpret_cast<uintptr_t>(out) & 7u) == 0);
  PS_REQUIRE(device_accessible(out));
  if (B > 0 && P > 0) {
    PS_REQUIRE((long)B * P <= INT32_MAX);
    PS_NN(commit); PS_NN(undecided); PS_NN(role);
  }
  return launch_status(block_progress_run(commit, undecided, role, B, P, out,
                                          static_cast<cudaStream_t>(stream)));
}

extern "C" size_t ps_store_record_bytes(int d) {
  return d > 0 && d % 32 == 0 ? ps::store_record_bytes(d) : 0;
}

extern "C" ps_status ps_host_alloc(size_t bytes, void** ptr) {
  if (ptr == nullptr || bytes == 0) return PS_ERR_ARG;
  *ptr = nullptr;
  void* p = nullptr;
  cudaError_t e = cudaHostAlloc(&p, bytes, cudaHostAllocMapped | cudaHostAllocPortable);
  if (e != cudaSuccess) return launch_status(e);
  void* dp = nullptr;
  e = cudaHostGetDevicePointer(&dp, p, 0);
  if (e != cudaSuccess || dp != p) {  // one address for host and device (unified addressing)
    cudaFreeHost(p);
    return e != cudaSuccess ? launch_status(e) : PS_ERR_CUDA;
  }
  *ptr = p;
  return PS_OK;
}

extern "C" ps_status ps_host_free(void* ptr) {
  if (ptr == nullptr) return PS_OK;
  return launch_status(cudaFreeHost(ptr));
}

extern "C" ps_status ps_nvfp4_pack_clusters(ps_handle h, const uint8_t* codes,
                                            const uint8_t* scales, const int32_t* assign, int B,
                                            int N, int d, int C, void* store, int32_t* order,
                                            int32_t* cl_off, void* stream) {
  TraceScope trace_scope(h);
  PS_REQUIRE(h != nullptr && B >= 0);
  if (B == 0) return PS_OK;
  PS_REQUIRE(N >= 1 && N <= 16384 && d > 0 && d % 32 == 0 && C >= 1 && C <= 65535 &&
             B <= 65535);
  PS_PTR(codes); PS_NN(scales); PS_NN(assign); PS_PTR(store); PS_NN(order); PS_NN(cl_off);
  PS_REQUIRE(device_accessible(store));
  return launch_status(pack_clusters_run(codes, scales, assign, B, N, d, C,
                                         static_cast<uint8_t*>(store), order, cl_off,
                                         static_cast<cudaStream_t>(stream)));
}

extern "C" ps_status ps_nvfp4_fetch_dequant(ps_handle h, const void* store, const int32_t* order,
                                            const int32_t* cl_off, const int32_t* sel, int k,
                                            const float* mu, const float* rho,
                                            const float* tensor_scale, int B, int N, int d, int C,
                                            void* Ht, void* stream) {
  TraceScope trace_scope(h);
  PS_REQUIRE(h != nullptr && B >= 0);
  if (B == 0 || k == 0) return PS_OK;
  PS_REQUIRE(N >= 1 && N <= 65535 && d > 0 && d % 32 == 0 && C >= 1 && k >= 1 && k <= C &&
             B <= 65535);
  PS_PTR(store); PS_NN(order); PS_NN(cl_off); PS_NN(sel); PS_PTR(mu); PS_NN(rho);
  PS_NN(tensor_scale); PS_PTR(Ht);
  PS_REQUIRE(device_accessible(store));
  return launch_status(fetch_dequant_run(static_cast<const uint8_t*>(store), order, cl_off, sel,
                                         k, mu, rho, tensor_scale, B, N, d, C,
                                         static_cast<__nv_bfloat16*>(Ht),
                                         static_cast<cudaStream_t>(stream)));
}
