/*
 * libpolestar -- the per-step drift-scoring and sparse-refresh path of
 * Polestar-Cache / Polestar-Commit on one NVIDIA GB300 (sm_103a).
 *
 * Method source: "Polestar: Drift-Aware Cache Calibration and Token
 * Commitment for Efficient Inference of Diffusion LLMs" (gist.science
 * explainer of arXiv 2607.14107), technical summary, cited below as
 * [Polestar §x, <paragraph>].
 *
 * Conventions shared by every call
 * --------------------------------
 * Memory   Every array argument is a DEVICE pointer to caller-owned memory,
 *          row-major, contiguous, last index fastest, 16-byte aligned.
 *          The library allocates nothing inside an op: scratch comes from the
 *          caller's workspace `ws` of at least ps_workspace_bytes(op, ...)
 *          bytes (NULL is fine when that size is 0).  Outputs must not alias
 *          inputs unless the argument says "in/out".
 * Streams  `stream` is a cudaStream_t passed as void* (NULL = the legacy
 *          default stream).  Calls only enqueue work and return; the results
 *          are valid once the stream reaches that point.
 * Errors   Argument errors are detected on the host before anything is
 *          enqueued and return PS_ERR_ARG (nothing is launched, no output is
 *          touched).  A launch failure returns PS_ERR_CUDA.  A device-side
 *          failure (a bounded wait that gave up) sets the handle's status word;
 *          ps_check() reports it as PS_ERR_TIMEOUT.
 * Sizes    B >= 0 (B == 0 is a no-op), d % 16 == 0, dh % 16 == 0,
 *          Hq % Hkv == 0, 1 <= k <= C <= min(N, 256), d <= 8192,
 *          dh <= 256, V % 4 == 0, P <= 1024, B * P <= 65535.
 * Threads  One handle per concurrently used stream; no C++ exception
 *          crosses this interface.
 * State    Step-to-step state (centroids, previous distributions, drift
 *          history, undecided flags, the KV cache) lives in caller buffers.
 */
#ifndef POLESTAR_H
#define POLESTAR_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  PS_OK = 0,
  PS_ERR_ARG = 1,          /* bad pointer, size, alignment or dtype       */
  PS_ERR_UNSUPPORTED = 2,  /* device is not sm_103                         */
  PS_ERR_WORKSPACE = 3,    /* ws smaller than ps_workspace_bytes()         */
  PS_ERR_CUDA = 4,         /* a CUDA runtime call or launch failed         */
  PS_ERR_TIMEOUT = 5       /* a device-side bounded wait gave up           */
} ps_status;

typedef enum { PS_F32 = 0, PS_BF16 = 1 } ps_dtype;

typedef enum {
  PS_OP_KMEANS = 0, PS_OP_NVFP4 = 1, PS_OP_PROXY_KL = 2,
  PS_OP_TOPK = 3, PS_OP_REFRESH = 4, PS_OP_COMMIT = 5
} ps_op;

typedef struct ps_handle_s* ps_handle;

/* Create a handle on `device` (made current).  Allocates the handle's
 * 16-byte device status word -- the only allocation the library makes.
 * PS_ERR_UNSUPPORTED unless the device has compute capability 10.3. */
ps_status ps_create(int device, ps_handle* out);
ps_status ps_destroy(ps_handle h);

/* Status of device-side work enqueued so far on `stream`: reads the
 * handle's status word after the work on `stream` has finished (the read is
 * ordered on `stream` and waited for; synchronize != 0 additionally
 * synchronises the stream first and reports a failed synchronisation).
 * Clears the word.  Returns PS_OK, PS_ERR_TIMEOUT or PS_ERR_CUDA. */
ps_status ps_check(ps_handle h, void* stream, int synchronize);

const char* ps_status_string(ps_status s);

/* The CUDA runtime error behind the calling thread's most recent
 * PS_ERR_CUDA ("cudaErrorName: description"), or "" if there was none.  The
 * text lives in thread-local storage owned by the library and stays valid
 * until the thread's next call that fails with PS_ERR_CUDA. */
const char* ps_last_cuda_error(void);

/* Kernel trace, for diagnostics (no counterpart in the paper).  While it is
 * enabled on a handle, every kernel a ps_* call on that handle launches is
 * bracketed by two CUDA events on the call's stream, kept in host memory the
 * handle owns.  Enabling (enable != 0) or disabling discards earlier
 * records.  Not for calls made while the stream is captured into a CUDA
 * graph.  PS_ERR_ARG for a NULL handle. */
ps_status ps_trace_enable(ps_handle h, int enable);
/* Number of kernels recorded since tracing was enabled (0 when it is off). */
int ps_trace_count(ps_handle h);
/* Record i (0-based, in launch order): the kernel's name and its duration in
 * milliseconds; waits for the kernel to finish.  The name is owned by the
 * CUDA runtime and stays valid while the library is loaded.  PS_ERR_ARG for
 * an index out of range or NULL outputs, PS_ERR_CUDA if an event query
 * fails. */
ps_status ps_trace_get(ps_handle h, int i, const char** name, float* ms);

/* ---------------------------------------------------------------------------
 * Offload of the quantised clusters.
 * [Polestar §2.C, CPU offloading] -- "quantised hidden-state clusters are
 * offloaded to pinned CPU memory while only the centroids stay on the GPU;
 * the top-k clusters are fetched asynchronously".
 *
 * Store of a window: one record per row, grouped by cluster (ascending id)
 * and by ascending position inside a cluster.  A record holds the row's E2M1
 * codes (d/2 bytes) then its E4M3 block scales (d/16 bytes), each part
 * zero-padded to a multiple of 16 bytes: ps_store_record_bytes(d) bytes
 * (0 unless d is a positive multiple of 32).  Layout [B][N][record].
 *
 * ps_host_alloc: `bytes` of pinned host memory mapped into the device's
 * address space, one pointer valid on host and device (the GPU reaches it
 * over NVLink-C2C or PCIe).  PS_ERR_ARG for ptr == NULL or bytes == 0;
 * PS_ERR_CUDA if the allocation fails.  Release with ps_host_free.
 * ------------------------------------------------------------------------- */
size_t ps_store_record_bytes(int d);
ps_status ps_host_alloc(size_t bytes, void** ptr);
ps_status ps_host_free(void* ptr);

/* Writes the store of every window (the offload: the GPU stores straight
 * into it when it lies in host memory).
 * codes [B][N][d/2] u8, scales [B][N][d/16] u8, assign [B][N] i32 in [0, C)
 * (ps_nvfp4_residual's and ps_kmeans_spherical's outputs)
 * store [B][N][record] u8 out: device memory or ps_host_alloc memory,
 *       16-byte aligned
 * order [B][N] i32 out: position of record r;  cl_off [B][C+1] i32 out:
 *       first record of cluster c (cl_off[C] = rows with a label in [0, C))
 * PS_ERR_ARG for NULL or misaligned pointers, a store the device cannot
 * reach, N > 16384, or d not a multiple of 32. */
ps_status ps_nvfp4_pack_clusters(ps_handle h, const uint8_t* codes,
                                 const uint8_t* scales, const int32_t* assign,
                                 int B, int N, int d, int C, void* store,
                                 int32_t* order, int32_t* cl_off, void* stream);

/* Reads the records of the selected clusters from the store (the fetch) and
 * writes each row's reconstruction into Ht:
 *   g = fl(s_b S), deq = fl(v g), t = fl(rho_i mu_c), h~ = fl(t + deq)
 * (fp32, one rounding each, no fused multiply-add; v the element's E2M1
 * value, s_b its block's E4M3 value, S the window's tensor scale), rounded
 * to bf16 (nearest-even).  Rows of unselected clusters are left untouched,
 * so ps_refresh_kv can take Ht with the same pos / npos.
 * sel [B][k] i32 (ps_topk_drift's; entries < 0 ignored), mu [B][C][d] f32,
 * rho [B][N] f32, tensor_scale [B] f32, Ht [B][N][d] bf16 out.
 * PS_ERR_ARG as for ps_nvfp4_pack_clusters, or k outside [1, C]. */
ps_status ps_nvfp4_fetch_dequant(ps_handle h, const void* store,
                                 const int32_t* order, const int32_t* cl_off,
                                 const int32_t* sel, int k, const float* mu,
                                 const float* rho, const float* tensor_scale,
                                 int B, int N, int d, int C, void* Ht,
                                 void* stream);

/* Workspace bytes `op` needs for these sizes (arguments an op does not use
 * are ignored).  0 means ws may be NULL. */
size_t ps_workspace_bytes(int op, int B, int N, int d, int C, int Hq, int Hkv,
                          int dh, int k, int P, int V);

/* ---------------------------------------------------------------------------
 * a1  Spherical k-means of each window's hidden states.
 * [Polestar §2.A, local window & clustering] -- "clusters the hidden states
 * in the window with spherical k-means".
 *
 * H        [B][N][d]  f32 or bf16 (dtype)      hidden states of the window
 * mu       [B][C][d]  f32, in/out              centroids: input = warm start
 *          (init_mode 0, e.g. the previous step's result) or ignored
 *          (init_mode 1); output = final unit-norm centroids
 * init_u   [B][C]     f64 in [0,1)             k-means++ draws (init_mode 1;
 *          NULL for init_mode 0).  First centre = row floor(u0*N); centre r =
 *          first row whose running sum of w_i = 1 - max cos to the chosen
 *          centres exceeds u_r * sum(w).
 * iters    number of centroid updates I >= 0; I+1 assignment passes run.
 * assign   [B][N] i32 out  final cluster of each row (ties -> lower index)
 * rho      [B][N] f32 out  <h_i, mu_{assign_i}>
 * chat     [B][C][d] f32 in/out  mean(rho of members) * mu_c; clusters left
 *          empty keep the caller's values
 * counts   [B][C] i32 out  cluster sizes
 * objective[B][I+1] f32 out (nullable)  sum_i cos(h_i, mu_{a_i}) per pass;
 *          with the faster passes (bf16 windows, at least one 128-row tile per
 *          SM) the passes before the last sum their bf16-centroid scores, each
 *          within 2^-9 * N of the exact sum; the last pass's is exact up to
 *          fp32 rounding
 * Empty clusters keep their centroid.  Rows of zero norm join cluster 0.
 *
 * Two forms compute the same passes.  bf16 windows of N <= 1024 rows with
 * C <= 256, d <= 16384 and iters >= 2 run them on the window's cosine Gram
 * matrix (24-bit fixed point, exact integer cluster sums) inside one
 * thread-block cluster; a row whose two best cosines lie within about 1e-6
 * may take the other label than an fp64 pass would.  Other shapes, and any
 * call made while PS_KMEANS_LLOYD is set in the environment (read once per
 * process), form every centroid and assign on the tensor cores per pass.
 * ------------------------------------------------------------------------- */
ps_status ps_kmeans_spherical(ps_handle h, const void* H, int dtype, int B,
                              int N, int d, int C, int iters, int init_mode,
                              const double* init_u, float* mu, int32_t* assign,
                              float* rho, float* chat, int32_t* counts,
                              float* objective, void* ws, size_t ws_bytes,
                              void* stream);

/* ---------------------------------------------------------------------------
 * a2  NVFP4 quantisation of the k-means residuals.
 * [Polestar §2.A, local window & clustering] -- "quantises residuals with
 * NVFP4 to create compact proxy representations".
 *
 * r = fl(h - fl(rho_i * mu_{a_i}))  (fp32, two roundings); mu == NULL
 * quantises H itself (then assign/rho are ignored).
 * S_b = max(fl(amax_b / 2688), FLT_MIN) for 0 < amax_b < inf, else 1.
 * Block scale (16 elements along d): E4M3(fl(amax_blk / fl(6 S_b))), RNE,
 * saturating; element: E2M1(fl(r / fl(s_blk * S_b))), RNE, saturating, or
 * 0 when s_blk == 0.  Negative values rounding to zero keep their sign.
 *
 * codes  [B][N][d/2]  u8 out  element 2j in the low nibble of byte j
 * scales [B][N][d/16] u8 out  E4M3 block scales
 * tensor_scale [B]    f32 out S_b
 * Outputs are bit-exact functions of the inputs.
 * ------------------------------------------------------------------------- */
ps_status ps_nvfp4_residual(ps_handle h, const void* H, int dtype,
                            const float* mu, const int32_t* assign,
                            const float* rho, int B, int N, int d, int C,
                            uint8_t* codes, uint8_t* scales,
                            float* tensor_scale, void* ws, size_t ws_bytes,
                            void* stream);

/* ---------------------------------------------------------------------------
 * a3+a4  Proxy attention on centroid keys and the per-position KL drift.
 * [Polestar §2.A, sparse updates] -- proxy attention with cluster centroids;
 * [Polestar §2.A, drift measurement] -- D_i = KL(A_i^(t) || A_i^(t-1)).
 *
 * K~[b][c][g] = chat[b][c] . Wk[:, g*dh:(g+1)*dh]            (fp32)
 * s = q[b][i][h] . K~[b][c][h / (Hq/Hkv)] / sqrt(dh); p = softmax_c(s)
 * A_cur[b][i][c] = mean over the Hq heads of p
 * D[b][i] = max(0, sum_c A_cur (ln A_cur - ln max(A_prev, 1e-30))), terms
 *           with A_cur == 0 skipped; D = 0 when A_prev == NULL.
 *
 * Q      [B][N][Hq][dh]  f32 or bf16 (dtype)
 * chat   [B][C][d]       f32   (from ps_kmeans_spherical)
 * Wk     [d][Hkv*dh]     dtype
 * A_prev [B][N][C] f32 or NULL;  A_cur [B][N][C] f32 out;  D [B][N] f32 out
 * Deterministic: identical inputs give identical bits, so A_prev == A_cur
 * from an identical call gives D == 0 exactly.
 * ------------------------------------------------------------------------- */
ps_status ps_proxy_attn_kl(ps_handle h, const void* Q, const float* chat,
                           const void* Wk, int dtype, int B, int N, int d,
                           int C, int Hq, int Hkv, int dh, const float* A_prev,
                           float* A_cur, float* D, void* ws, size_t ws_bytes,
                           void* stream);

/* ---------------------------------------------------------------------------
 * a5  Top-k most-drifting clusters and the positions they cover.
 * [Polestar §2.A, sparse updates] -- "identifies the top-k drifting
 * clusters and runs a sparse forward pass on only these positions".
 *
 * score_c = (sum of D_i over members, fp64, ascending i) / n_c, for n_c > 0.
 * sel       [B][k] i32 out  clusters by score descending, ties -> lower c,
 *                           padded with -1
 * sel_score [B][k] f32 out  their scores (fp32 of the fp64 mean), pad -inf
 * pos       [B][N] i32 out  ascending positions whose cluster is selected,
 *                           then -1
 * npos      [B]    i32 out  number of such positions (stays on the device)
 * posmask   [B][N] u8  out  (nullable) 1 where the position is selected
 * Bit-exact.
 * ------------------------------------------------------------------------- */
ps_status ps_topk_drift(ps_handle h, const float* D, const int32_t* assign,
                        const int32_t* counts, int B, int N, int C, int k,
                        int32_t* sel, float* sel_score, int32_t* pos,
                        int32_t* npos, uint8_t* posmask, void* ws,
                        size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * a6  Sparse K/V refresh of the selected positions.
 * [Polestar §2.A, sparse updates] -- "a sparse forward pass on only these
 * positions ... refreshes the corresponding KV-cache entries".
 *
 * For j < npos[b], p = pos[b][j]:
 *   Kcache[b][cache_off + p] = round(H[b][p] . Wk), same for V with Wv,
 *   accumulated in fp32, rounded to the cache dtype (bf16 RNE or f32).
 * Rows not listed are untouched.  npos is read on the device.
 * H [B][N][d], Wk/Wv [d][Hkv*dh], Kcache/Vcache [B][Ncache][Hkv][dh], all
 * of `dtype`.  Requires cache_off + N <= Ncache.  bf16 with Hkv*dh a
 * multiple of 64 runs on the tensor cores and needs the workspace
 * (ps_workspace_bytes(PS_OP_REFRESH, ...): the gathered rows, B*N*d bf16
 * at most); the caches must then be 16-byte aligned.
 * ------------------------------------------------------------------------- */
ps_status ps_refresh_kv(ps_handle h, const void* H, int dtype,
                        const int32_t* pos, const int32_t* npos,
                        const void* Wk, const void* Wv, int B, int N, int d,
                        int Hkv, int dh, void* Kcache, void* Vcache,
                        int Ncache, int cache_off, void* ws, size_t ws_bytes,
                        void* stream);

/* ---------------------------------------------------------------------------
 * a7  Confidence and drift-aware commitment of a block.
 * [Polestar §2.B, current block commitment] -- commit when the drift delta
 * exceeds alpha (tau_s - c)^2;  [Polestar §2.B, suffix block commitment] --
 * suffix tokens commit only with c >= tau_s.
 *
 * Per row: token = first arg-max of the logits, conf = 1 / sum exp(l - max).
 * role[j]: 0 current block, 1 suffix block, 2 inactive.
 * Current, undecided j:  commit if conf >= tau_s, or (d_cnt >= 1 and)
 *   mode 0 DELTA_DROP:  d_sum/d_cnt - D > alpha (tau_s - conf)^2
 *   mode 1 DELTA_RISE:  D - d_sum/d_cnt > alpha (tau_s - conf)^2
 *   mode 2 RATIO:       D < ratio * d_prev
 * Suffix, undecided j: commit if suffix_sel[b][j] and conf >= tau_s.
 * ensure_progress: if no current token commits while some are undecided,
 *   the undecided current token with the largest conf commits (ties: lower j).
 * Then every undecided current token sets d_sum = fl32(d_sum + D),
 *   d_cnt += 1, d_prev = D; committed tokens get undecided = 0.
 *
 * logits [B][P][V] of `dtype` (PS_F32, or PS_BF16 as an LM head emits them;
 *   bf16 values are exact in fp32, and the bf16 scan differs from the fp32 one
 *   only in how its fp32 partial sums are grouped, so on the same values the
 *   tokens are equal and the confidences agree to rounding);
 *   role [P] u8; undecided [B][P] u8 in/out;
 * D_blk: element (b, j) at D_blk[b*d_ld + j] (e.g. the last layer's D with
 *   d_ld = N, offset to the block); d_sum/d_prev [B][P] f32 in/out,
 *   d_cnt [B][P] i32 in/out; suffix_sel: element (b, j) at
 *   suffix_sel[b*sel_ld + j] or NULL (no suffix commits);
 * token [B][P] i32, conf [B][P] f32, commit [B][P] u8 out.
 * ------------------------------------------------------------------------- */
typedef struct {
  float tau_s;
  float alpha;
  float ratio;
  int mode;            /* 0 DELTA_DROP, 1 DELTA_RISE, 2 RATIO */
  int ensure_progress; /* 0 or 1 */
} ps_commit_params;

ps_status ps_commit(ps_handle h, const void* logits, int dtype, int B, int P, int V,
                    const uint8_t* role, uint8_t* undecided,
                    const float* D_blk, int d_ld, float* d_sum, int32_t* d_cnt,
                    float* d_prev, const uint8_t* suffix_sel, int sel_ld,
                    ps_commit_params params, int32_t* token, float* conf,
                    uint8_t* commit, void* ws, size_t ws_bytes, void* stream);


/* ---------------------------------------------------------------------------
 * NVFP4 residual quantisation without a workspace.
 * The paper has no counterpart to this call: it exists for callers that
 * cannot allocate device memory -- e.g. a host application that gives the
 * library only preallocated inputs and outputs, or code running where a
 * cudaMalloc is not allowed because it may synchronise the device or break
 * a fixed memory budget.
 *
 * Computes exactly what ps_nvfp4_residual computes (same arguments, same
 * bit-exact outputs) but takes no `ws`: its scratch (per-CTA partial maxima)
 * lives in one fixed 64 KiB file-scope device array inside the library,
 * which every GPU that loads the library keeps until the process exits.
 * It calls no cudaMalloc, cudaFree or allocating library routine.
 *
 * Limit: B <= 16384 (the array holds 16384 partials; a window takes at
 * most 16384 / B of them);
 * larger B returns PS_ERR_WORKSPACE and launches nothing.
 * Device: the handle's device must be the calling thread's current device
 * (PS_ERR_ARG otherwise), since the array's address differs per device.
 * Set-up: the first call on a device looks up the array's device address
 * (cudaGetSymbolAddress) and keeps it; make that first call before any
 * stream capture.  The kept address belongs to the device's context, so the
 * library must not be used across a reset of that device (cudaDeviceReset).
 * A failed look-up returns PS_ERR_CUDA with ps_last_cuda_error() set.
 * Sharing: every call on a device uses the same array and leaves the last
 * call's values in it.  Nothing in it has to start at zero (each call writes
 * every slot it later reads), but calls that overlap on the GPU -- on
 * different streams, or from different threads -- race on it and must be
 * serialised by the caller.
 * ------------------------------------------------------------------------- */
ps_status ps_nvfp4_residual_noalloc(ps_handle h, const void* H, int dtype,
                                    const float* mu, const int32_t* assign,
                                    const float* rho, int B, int N, int d,
                                    int C, uint8_t* codes, uint8_t* scales,
                                    float* tensor_scale, void* stream);

/* ---------------------------------------------------------------------------
 * Alternative drift signals for the ablation.
 * [Polestar §2.A, drift measurement]: KL drift tracks contextual shifts more
 * closely than cosine dissimilarity on subsets; [Polestar §4, ablation
 * studies]: it beats cosine similarity and uncertainty-based selection.
 *
 * One signal per position from the proxy distributions that
 * ps_proxy_attn_kl wrote (call it with A_prev = NULL to skip its fused KL,
 * then this on its A_cur and the previous step's distribution):
 *   PS_SCORER_KL       D = max(0, sum_c a ln(a / max(a', 1e-30))), a > 0
 *   PS_SCORER_COSINE   D = max(0, 1 - <a, a'> / (|a| |a'|)); 0 if a norm is 0
 *   PS_SCORER_ENTROPY  D = -sum_c a ln a over a > 0 (uncertainty of the
 *                      current distribution; A_prev is not read)
 * With A_prev == NULL, KL and COSINE write D = 0.
 *
 * A_cur, A_prev [B][N][C] f32 (rows of any non-negative weights; the proxy
 * writes distributions); D [B][N] f32 out, must not alias either input.
 * Sizes: B >= 0 (0: no-op), N >= 1, 1 <= C <= 4096, B * N <= 2^31 - 1.
 * Errors: a NULL handle, A_cur or D, a bad size or an unknown scorer return
 * PS_ERR_ARG before anything is enqueued.
 * ------------------------------------------------------------------------- */
typedef enum {
  PS_SCORER_KL = 0, PS_SCORER_COSINE = 1, PS_SCORER_ENTROPY = 2
} ps_scorer;

ps_status ps_drift_score(ps_handle h, const float* A_cur, const float* A_prev,
                         int B, int N, int C, int scorer, float* D,
                         void* stream);

/* ---------------------------------------------------------------------------
 * The outcome of a decode step that the refresh schedule below consumes.
 * [Polestar §2.A, schedule]: refreshes are triggered by the number of
 * decoded tokens; the window moves on when the current block is decided.
 *
 * One small kernel writes out[0] = the largest number of positions any of
 * the B sequences committed in this step (commit [B][P] u8, every role) and
 * out[1] = 1 when no sequence has an undecided current-block position left
 * (undecided [B][P] u8, role [P] u8 with 0 = current block), else 0 -- the
 * (committed, block_done) pair of ps_schedule_step, computed where the
 * flags are, so the host reads one 8-byte pair.
 * out: int32[2], 8-byte aligned, in device memory or in ps_host_alloc
 * memory (then readable on the host once the stream has reached it).
 * B == 0 or P == 0 writes (0, 1).  Errors: a NULL handle or out, an
 * unreachable or misaligned out, or NULL flags with B, P > 0 return
 * PS_ERR_ARG before anything is enqueued.
 * ------------------------------------------------------------------------- */
ps_status ps_block_progress(ps_handle h, const uint8_t* commit,
                            const uint8_t* undecided, const uint8_t* role,
                            int B, int P, int32_t* out, void* stream);

/* ---------------------------------------------------------------------------
 * Refresh schedule of the decode loop (host only; no handle, no GPU work).
 * [Polestar §2.A, schedule]: the drift refresh is triggered once the decoded
 * context has moved enough -- after tau_upd tokens were decoded -- and
 * periodic full passes refresh positions outside the top-k clusters too.
 *
 * Called after every decode step with the number of tokens that step
 * committed and whether the current block is now decided; returns the
 * actions of the NEXT step (an OR of the flags below, 0 = reuse the cache):
 *   block_done:        REFRESH | FULL | SLIDE | REINIT -- the window slides
 *                      by block_len, the next step clusters it from scratch
 *                      (k-means++), refreshes every position, and the
 *                      counts restart (since = refreshes = 0);
 *   else since += committed; if since >= tau_upd (tau_upd = 0: every step):
 *                      REFRESH, since = 0, refreshes += 1, and FULL too when
 *                      full_period > 0 and refreshes % full_period == 0.
 * The state is caller-owned; zero it for the first window (whose first step
 * the caller runs as block_done would: clustered and refreshed in full).
 * Errors: NULL pointers, tau_upd < 0, full_period < 0, block_len < 1,
 * committed < 0 or a negative state field return -PS_ERR_ARG and leave the
 * state unchanged.  The token count saturates at INT_MAX.
 * ------------------------------------------------------------------------- */
enum {
  PS_SCHED_REFRESH = 1, /* run the drift path and the top-k refresh         */
  PS_SCHED_FULL = 2,    /* refresh every window position, not only top-k    */
  PS_SCHED_SLIDE = 4,   /* a new block: reset the commit state              */
  PS_SCHED_REINIT = 8   /* re-seed k-means (k-means++), no previous A       */
};

typedef struct {
  int tau_upd;      /* tokens between refreshes, >= 0                        */
  int full_period;  /* every full_period-th refresh is full; 0 = never       */
  int block_len;    /* positions the window slides by, >= 1                  */
} ps_schedule_params;

typedef struct {
  int since;        /* tokens committed since the last refresh              */
  int refreshes;    /* refreshes since the window was built                 */
  int block_start;  /* sequence position of the current block               */
} ps_schedule_state;

int ps_schedule_step(const ps_schedule_params* p, ps_schedule_state* s,
                     int committed, int block_done);

#ifdef __cplusplus
}
#endif

#endif /* POLESTAR_H */
