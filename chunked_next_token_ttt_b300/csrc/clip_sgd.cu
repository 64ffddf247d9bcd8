// Global-norm clipped SGD step on a fast-weight arena [slot][B][n], computing
// the per-sequence gradient norm directly from dW.
//   1. sum-of-squares partials: one block per 8192-element piece of each
//      (slot, sequence) segment, written to a fixed slot (deterministic order);
//   2. one block reduces every sequence's partials into norm and clip scale;
//   3. the elementwise update W32 -= eta * scale * dW with the operand re-cast.
#include "clip_sgd.h"
#include "kernels.h"

namespace ttt {
namespace {

constexpr int kPiece = 8192;
constexpr int kThreads = 256;

__global__ void sumsq_partials_kernel(long long n, int pieces, const float* __restrict__ dW,
                                      float* __restrict__ partials) {
  pdl_wait();
  pdl_launch();
  __shared__ float red[32];
  const int piece = blockIdx.x, slot = blockIdx.y, s = blockIdx.z;
  const int nslots = gridDim.y, B = gridDim.z;
  const float* src = dW + ((long long)slot * B + s) * n;
  const long long lo = (long long)piece * kPiece;
  const long long hi = lo + kPiece < n ? lo + kPiece : n;
  float acc = 0.0f;
  for (long long i = lo + threadIdx.x; i < hi; i += kThreads) acc += src[i] * src[i];
  acc = block_sum(acc, red);
  if (threadIdx.x == 0) partials[((long long)s * nslots + slot) * pieces + piece] = acc;
}

__global__ void clip_finalize_kernel(int B, int per_seq, const float* __restrict__ partials, float clip,
                                     float* __restrict__ scale, float* __restrict__ norm_out,
                                     float* __restrict__ scale_out, int* __restrict__ flag) {
  pdl_wait();
  pdl_launch();
  __shared__ float red[32];
  int bad = 0;
  for (int s = 0; s < B; ++s) {
    float acc = 0.0f;
    for (int t = threadIdx.x; t < per_seq; t += blockDim.x) acc += partials[(long long)s * per_seq + t];
    acc = block_sum(acc, red);
    if (threadIdx.x == 0) {
      const float nrm = sqrtf(acc);
      float sc = 1.0f;
      if (!isfinite(nrm)) {
        sc = 0.0f;
        bad = 1;
      } else if (clip > 0.0f) {
        sc = fminf(1.0f, clip / (nrm + 1e-6f));
      }
      scale[s] = sc;
      if (norm_out) norm_out[s] = nrm;
      if (scale_out) scale_out[s] = sc;
    }
  }
  if (threadIdx.x == 0) *flag = bad;
}

}  // namespace

int clip_sgd_pieces(long long n) { return (int)((n + kPiece - 1) / kPiece); }

size_t clip_sgd_scratch_floats(int nslots, int B, long long n) {
  return (size_t)nslots * B * clip_sgd_pieces(n) + (size_t)B + 1;
}

ttt_status launch_clip_sgd(int dtype, int nslots, int B, long long n, float* W32, void* Wop, const float* dW,
                           float eta, float clip, float* norm_out, float* scale_out, float* scratch,
                           cudaStream_t st) {
  const int pieces = clip_sgd_pieces(n);
  float* partials = scratch;
  float* scale = scratch + (size_t)nslots * B * pieces;
  int* flag = reinterpret_cast<int*>(scale + B);
  launch_pdl(sumsq_partials_kernel, dim3(pieces, nslots, B), kThreads, 0, st, n, pieces, dW, partials);
  TTT_CHECK_LAUNCH();
  launch_pdl(clip_finalize_kernel, 1, kThreads, 0, st, B, nslots * pieces, partials, clip, scale, norm_out, scale_out,
                                               flag);
  TTT_CHECK_LAUNCH();
  return launch_sgd_update(dtype, nslots, B, n, W32, Wop, 0, dW, scale, eta, st);
}

}  // namespace ttt
