// Shared device/host helpers of libpolestar (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <utility>

#include "../../include/polestar.h"

namespace ps {
struct TraceSink;
}

struct ps_handle_s {
  int device;
  int num_sms;
  int* status;  // device word: 0 ok, else a PS_ERR_* code set by a kernel
  ps::TraceSink* trace;  // non-null while ps_trace_enable is on
  cudaStream_t aux;      // the library's own stream: captures the bodies of
                         // conditional graph nodes while the caller's stream
                         // is being captured
};

namespace ps {

constexpr int kWarp = 32;
// SM count the grid and workspace heuristics are sized for (GB300: 152).
// Workspace sizes depend only on shapes, never on the device queried.
constexpr int kSmTarget = 152;

// Element loads widened to fp32.
__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) {
  return __bfloat162float(x);
}

template <typename T> struct Store;
template <> struct Store<float> {
  __device__ __forceinline__ static void put(float* p, float v) { *p = v; }
};
template <> struct Store<__nv_bfloat16> {
  __device__ __forceinline__ static void put(__nv_bfloat16* p, float v) {
    *p = __float2bfloat16_rn(v);
  }
};

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ double warp_sum_f64(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Record the first device-side failure of a call in the handle's word.
__device__ __forceinline__ void set_status(int* status, int code) {
  if (status) atomicCAS(status, 0, code);
}

// Kernel launches.  launch_pdl launches through cudaLaunchKernelEx; with
// kUsePdl it asks for programmatic dependent launch.  Every kernel starts
// with pdl_prologue() (griddepcontrol.wait: waits for the previous grid's
// completion and writes when such a dependency exists, a no-op otherwise)
// before its first read of an earlier kernel's output.  The next grid may be
// scheduled once every CTA of this one has called pdl_trigger() or exited;
// the long kernels call it after their main work, so the next grid's
// set-up overlaps only this grid's tail.  Measured in the bench's CUDA-graph
// replay on GB300, programmatic launch made the step slower both with the
// trigger at every kernel's start (0.51 vs 0.43 ms) and with it after the
// main work (0.346 vs 0.341 ms), so it is off.
constexpr bool kUsePdl = false;
__device__ __forceinline__ void pdl_prologue() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Kernel trace (ps_trace_enable): while the calling thread runs a ps_* call
// on a handle with tracing on, every launch below is bracketed by two CUDA
// events on its stream.  Defined in api.cu.
void trace_begin(cudaStream_t s);
void trace_end(cudaStream_t s, const void* kernel);

// Every kernel of the library is launched here.
template <typename... KArgs, typename... Args>
cudaError_t launch_ex(const cudaLaunchConfig_t& cfg, void (*kernel)(KArgs...), Args&&... args) {
  trace_begin(cfg.stream);
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
  trace_end(cfg.stream, reinterpret_cast<const void*>(kernel));
  return e;
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = kUsePdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return launch_ex(cfg, kernel, std::forward<Args>(args)...);
}

__host__ __device__ inline int ceil_div(long a, long b) { return (int)((a + b - 1) / b); }

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Carves a caller workspace into 256-byte aligned pieces.
struct Carver {
  char* base;
  size_t off = 0;
  explicit Carver(void* p) : base((char*)p) {}
  template <typename T> T* take(size_t count) {
    off = align_up(off, 256);
    T* p = base ? (T*)(base + off) : nullptr;
    off += count * sizeof(T);
    return p;
  }
  size_t bytes() const { return align_up(off, 256); }
};

}  // namespace ps
