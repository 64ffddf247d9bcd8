// Shared device/host helpers of libttt (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <cstdio>
#include <string>
#include <utility>

#include "ttt.h"

namespace ttt {

// ---------------------------------------------------------------- errors
void set_error(const std::string& msg);
ttt_status cuda_fail(cudaError_t e, const char* what, const char* file, int line);

#define TTT_CUDA(call)                                                    \
  do {                                                                    \
    cudaError_t e_ = (call);                                              \
    if (e_ != cudaSuccess) return ::ttt::cuda_fail(e_, #call, __FILE__, __LINE__); \
  } while (0)

#define TTT_CHECK_LAUNCH()                                                \
  do {                                                                    \
    cudaError_t e_ = cudaGetLastError();                                  \
    if (e_ != cudaSuccess) return ::ttt::cuda_fail(e_, "kernel launch", __FILE__, __LINE__); \
  } while (0)

#define TTT_TRY(expr)                                                     \
  do {                                                                    \
    ttt_status s_ = (expr);                                               \
    if (s_ != TTT_OK) return s_;                                          \
  } while (0)

// ---------------------------------------------------------------- types
typedef __nv_bfloat16 bf16;

template <typename T> __device__ __forceinline__ float to_f(T v);
template <> __device__ __forceinline__ float to_f<float>(float v) { return v; }
template <> __device__ __forceinline__ float to_f<bf16>(bf16 v) { return __bfloat162float(v); }

template <typename T> __device__ __forceinline__ T from_f(float v);
template <> __device__ __forceinline__ float from_f<float>(float v) { return v; }
template <> __device__ __forceinline__ bf16 from_f<bf16>(float v) { return __float2bfloat16_rn(v); }

// Storage of "operand" tensors (GEMM inputs and the outputs that feed them):
//   float  fp32 values;
//   bf16   bf16 values;
//   Split  fp32-accurate pairs kept as two bf16 planes, hi = bf16(v) at p[i]
//          and lo = bf16(v - hi) at p[lo + i]; a product of two split values is
//          taken as hi*hi + hi*lo + lo*hi (the bf16x3 scheme of Henry, Tang and
//          Heinecke, "Leveraging the bfloat16 Artificial Intelligence Datatype
//          for Higher-Precision Computations", 2019), about 2^-17 relative.
struct Split {};

enum Storage { ST_F32 = 0, ST_BF16 = 1, ST_SPLIT = 2 };

template <typename S> struct OpIO;
template <> struct OpIO<float> {
  __device__ __forceinline__ static float load(const void* p, long long, long long i) {
    return static_cast<const float*>(p)[i];
  }
  __device__ __forceinline__ static void store(void* p, long long, long long i, float v) {
    static_cast<float*>(p)[i] = v;
  }
  __device__ __forceinline__ static void copy(void* d, long long dlo, const void* s, long long slo, long long i) {
    static_cast<float*>(d)[i] = static_cast<const float*>(s)[i];
  }
};
template <> struct OpIO<bf16> {
  __device__ __forceinline__ static float load(const void* p, long long, long long i) {
    return __bfloat162float(static_cast<const bf16*>(p)[i]);
  }
  __device__ __forceinline__ static void store(void* p, long long, long long i, float v) {
    static_cast<bf16*>(p)[i] = __float2bfloat16_rn(v);
  }
  __device__ __forceinline__ static void copy(void* d, long long, const void* s, long long, long long i) {
    static_cast<bf16*>(d)[i] = static_cast<const bf16*>(s)[i];
  }
};
template <> struct OpIO<Split> {
  __device__ __forceinline__ static float load(const void* p, long long lo, long long i) {
    const bf16* q = static_cast<const bf16*>(p);
    return __bfloat162float(q[i]) + __bfloat162float(q[lo + i]);
  }
  __device__ __forceinline__ static void store(void* p, long long lo, long long i, float v) {
    bf16* q = static_cast<bf16*>(p);
    const bf16 h = __float2bfloat16_rn(v);
    q[i] = h;
    q[lo + i] = __float2bfloat16_rn(v - __bfloat162float(h));
  }
  __device__ __forceinline__ static void copy(void* d, long long dlo, const void* s, long long slo, long long i) {
    bf16* dq = static_cast<bf16*>(d);
    const bf16* sq = static_cast<const bf16*>(s);
    dq[i] = sq[i];
    dq[dlo + i] = sq[slo + i];
  }
};

// Element type of the dW output (the GEMM's EPI_DW epilogue): bf16 for bf16 operand storage (the
// clipped update reads it once, and the fp32 master absorbs the step), fp32
// for fp32-accurate storage.  The per-tile sums of squares always come from
// the fp32 accumulators.
template <typename S> struct DwType { using T = float; };
template <> struct DwType<bf16> { using T = bf16; };

// Four consecutive elements from a float4 in operand storage (16 / 8 / 2 x 8
// bytes): the start index must keep the access aligned.
template <typename S> struct QuadIO;
template <> struct QuadIO<float> {
  __device__ __forceinline__ static void store(void* p, long long, long long i, float4 w) {
    *reinterpret_cast<float4*>(static_cast<float*>(p) + i) = w;
  }
};
__device__ __forceinline__ uint2 pack_bf16x4(float a, float b, float c, float d) {
  const __nv_bfloat162 lo = __floats2bfloat162_rn(a, b), hi = __floats2bfloat162_rn(c, d);
  return make_uint2(*reinterpret_cast<const uint32_t*>(&lo), *reinterpret_cast<const uint32_t*>(&hi));
}
// Eight bf16 values in one 16-byte word, and back.
__device__ __forceinline__ uint4 pack_bf16x8(const float* v) {
  uint4 r;
  __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&r);
#pragma unroll
  for (int j = 0; j < 4; ++j) h[j] = __floats2bfloat162_rn(v[2 * j], v[2 * j + 1]);
  return r;
}
__device__ __forceinline__ void unpack_bf16x8(uint4 r, float* v) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&r);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float2 f = __bfloat1622float2(h[j]);
    v[2 * j] = f.x;
    v[2 * j + 1] = f.y;
  }
}
template <> struct QuadIO<bf16> {
  __device__ __forceinline__ static void store(void* p, long long, long long i, float4 w) {
    *reinterpret_cast<uint2*>(static_cast<bf16*>(p) + i) = pack_bf16x4(w.x, w.y, w.z, w.w);
  }
};
template <> struct QuadIO<Split> {
  __device__ __forceinline__ static void store(void* p, long long lo, long long i, float4 w) {
    bf16* q = static_cast<bf16*>(p);
    const uint2 h = pack_bf16x4(w.x, w.y, w.z, w.w);
    const __nv_bfloat162* hb = reinterpret_cast<const __nv_bfloat162*>(&h);
    const float2 h0 = __bfloat1622float2(hb[0]), h1 = __bfloat1622float2(hb[1]);
    *reinterpret_cast<uint2*>(q + i) = h;
    *reinterpret_cast<uint2*>(q + lo + i) = pack_bf16x4(w.x - h0.x, w.y - h0.y, w.z - h1.x, w.w - h1.y);
  }
};


// Two adjacent elements (i, i+1) at once; i even and the base (and, for Split,
// the lo offset) aligned to the pair size.
template <typename S> struct PairIO;
template <> struct PairIO<float> {
  __device__ __forceinline__ static float2 load(const void* p, long long, long long i) {
    return *reinterpret_cast<const float2*>(static_cast<const float*>(p) + i);
  }
  __device__ __forceinline__ static void store(void* p, long long, long long i, float a, float b) {
    *reinterpret_cast<float2*>(static_cast<float*>(p) + i) = make_float2(a, b);
  }
};
template <> struct PairIO<bf16> {
  __device__ __forceinline__ static float2 load(const void* p, long long, long long i) {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(static_cast<const bf16*>(p) + i));
  }
  __device__ __forceinline__ static void store(void* p, long long, long long i, float a, float b) {
    *reinterpret_cast<__nv_bfloat162*>(static_cast<bf16*>(p) + i) = __floats2bfloat162_rn(a, b);
  }
};
template <> struct PairIO<Split> {
  __device__ __forceinline__ static float2 load(const void* p, long long lo, long long i) {
    const bf16* q = static_cast<const bf16*>(p);
    const float2 h = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(q + i));
    const float2 l = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(q + lo + i));
    return make_float2(h.x + l.x, h.y + l.y);
  }
  __device__ __forceinline__ static void store(void* p, long long lo, long long i, float a, float b) {
    bf16* q = static_cast<bf16*>(p);
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    const float2 hf = __bfloat1622float2(h);
    *reinterpret_cast<__nv_bfloat162*>(q + i) = h;
    *reinterpret_cast<__nv_bfloat162*>(q + lo + i) = __floats2bfloat162_rn(a - hf.x, b - hf.y);
  }
};

// Exact (erf) GELU and its derivative, z * Phi(z) and Phi(z) + z phi(z).
__device__ __forceinline__ float gelu_f(float z) {
  return 0.5f * z * (1.0f + erff(z * 0.70710678118654752f));
}
__device__ __forceinline__ float gelu_grad_f(float z) {
  const float cdf = 0.5f * (1.0f + erff(z * 0.70710678118654752f));
  const float pdf = 0.39894228040143268f * expf(-0.5f * z * z);
  return cdf + z * pdf;
}
__device__ __forceinline__ float silu_f(float g) { return g / (1.0f + expf(-g)); }

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

// Block-wide sum; `red` holds >= 32 floats of shared memory.  All threads of
// the block must call it; every thread receives the total.
__device__ __forceinline__ float block_sum(float v, float* red) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int nw = (blockDim.x + 31) >> 5;
  v = warp_sum(v);
  __syncthreads();
  if (lane == 0) red[wid] = v;
  __syncthreads();
  float t = (threadIdx.x < nw) ? red[threadIdx.x] : 0.0f;
  if (wid == 0) {
    t = warp_sum(t);
    if (lane == 0) red[0] = t;
  }
  __syncthreads();
  return red[0];
}

inline int ceil_div(long long a, long long b) { return (int)((a + b - 1) / b); }

// ---------------------------------------------------------------- launches
// Programmatic dependent launch: every libttt kernel starts with pdl_wait()
// (griddepcontrol.wait: block until the previous kernel in the stream has
// completed and its memory is visible) before it touches global memory, then
// pdl_launch() lets the next kernel in the stream start launching.  A kernel
// launched with launch_pdl may thus begin (launch, set-up) while the previous
// kernel drains, but reads and writes nothing of it early.  Without the launch
// attribute both instructions are no-ops.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Whether launches from the calling thread carry the programmatic-serialization
// attribute: on, unless the handle of the API call in progress was created
// with ttt_options.no_pdl (set for the call's duration by PdlScope).
bool pdl_enabled();
class PdlScope {
 public:
  explicit PdlScope(bool on);
  ~PdlScope();
  PdlScope(const PdlScope&) = delete;
  PdlScope& operator=(const PdlScope&) = delete;

 private:
  bool saved_;
};

// ---------------------------------------------------------------- per-context state
// Process-unique id of the CUDA context current on the calling thread (binding
// the current device's primary context if none is), 0 if unknown.  State a
// context owns is cached under this id, so a second device or a context made
// after a device reset starts afresh.
unsigned long long current_context_id();
// Opt `func` into `bytes` of dynamic shared memory in the current context
// (once per kernel, context and size; thread-safe; no-op up to 48 KB).
cudaError_t ensure_dyn_smem(const void* func, size_t bytes);
// Device address of a __device__ variable in the current context (looked up
// with cudaGetSymbolAddress once per context; thread-safe).
cudaError_t symbol_address(const void* symbol, void** out);
// SM count of the current device (cached per context).
int current_sm_count();

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

}  // namespace ttt
