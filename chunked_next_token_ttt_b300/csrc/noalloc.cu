// ttt_clip_sgd_noalloc: the clipped SGD step with its scratch in a file-scope
// device array, for callers that cannot allocate device memory.
//
// Some callers own every byte of device memory themselves (a framework's
// caching allocator, a fixed per-process budget, an embedding host that hands
// out no workspace) or cannot afford the implicit device synchronisation of
// cudaMalloc inside a latency-critical loop.  This entry point lets them run the
// step without cudaMalloc, cudaFree or any allocating library routine: the
// partial sums, per-sequence scales and the status word live in
// g_clip_sgd_scratch below, which every GPU that loads the library holds until
// the process exits.
#include "clip_sgd.h"
#include "ttt_ops.h"

namespace {

// Shared by every call on a device: each call writes every word it later reads
// (partials, scales, the status word) before reading it, so nothing needs to
// start at zero; calls that overlap on the GPU (two streams, or two host
// threads) race on it.
static __device__ __align__(256) float g_clip_sgd_scratch[TTT_CLIP_SGD_NOALLOC_MAX_FLOATS];

// The device address of the scratch array in the current context.  In host
// code the array's name is only a host-side stand-in, so the address is looked
// up with cudaGetSymbolAddress, once per CUDA context (with that context
// current): a second device, or the new context after a device reset, gets its
// own lookup.
ttt_status scratch_for_current_context(float** out) {
  void* p = nullptr;
  const cudaError_t e = ttt::symbol_address((const void*)&g_clip_sgd_scratch, &p);
  if (e != cudaSuccess) return ttt::cuda_fail(e, "cudaGetSymbolAddress", __FILE__, __LINE__);
  *out = static_cast<float*>(p);
  return TTT_OK;
}

}  // namespace

extern "C" ttt_status ttt_clip_sgd_noalloc(int dtype, int nslots, int B, long long n, float* W32, void* Wop,
                                           const float* dW, float eta, float clip, float* norm_out,
                                           float* scale_out, ttt_stream stream) {
  if (nslots < 1 || B < 1 || n < 1 || !W32 || !Wop || !dW || clip < 0.0f ||
      (dtype != TTT_DTYPE_FP32 && dtype != TTT_DTYPE_BF16)) {
    ttt::set_error("bad clip_sgd_noalloc arguments");
    return TTT_ERR_BAD_ARG;
  }
  const size_t need = ttt::clip_sgd_scratch_floats(nslots, B, n);
  if (need > (size_t)TTT_CLIP_SGD_NOALLOC_MAX_FLOATS) {
    ttt::set_error("ttt_clip_sgd_noalloc: nslots * B * ceil(n / 8192) + B + 1 = " + std::to_string(need) +
                   " scratch floats exceed the fixed maximum of " +
                   std::to_string((long long)TTT_CLIP_SGD_NOALLOC_MAX_FLOATS) +
                   "; use ttt_clip_sgd with a caller-provided workspace");
    return TTT_ERR_BAD_SHAPE;
  }
  float* scratch = nullptr;
  TTT_TRY(scratch_for_current_context(&scratch));
  cudaStream_t st = (cudaStream_t)stream;
  TTT_TRY(ttt::launch_clip_sgd(dtype, nslots, B, n, W32, Wop, dW, eta, clip, norm_out, scale_out, scratch, st));
  int flag = 0;
  TTT_CUDA(cudaMemcpyAsync(&flag, scratch + (need - 1), sizeof(int), cudaMemcpyDeviceToHost, st));
  TTT_CUDA(cudaStreamSynchronize(st));
  if (flag) {
    ttt::set_error("non-finite gradient norm: that sequence was not updated");
    return TTT_ERR_NONFINITE;
  }
  return TTT_OK;
}
