// Sliding-window multi-head attention of the frozen blocks, forward only
// ("End-to-End TTT" review, Method: the sliding-window attention layer of
// window k that lets a chunk remember its own tokens before the update; 3.1:
// attention layers stay frozen during TTT).
//
// One warp per (sequence, head, query position t): the lanes split the head
// dimension; keys t - k + 1 .. t (clipped at position 0) are visited in order
// with an online softmax (running max, running sum, rescaled accumulator), in
// batches of four keys whose dot products are reduced together.  Q, K and V
// come from one fp32 projection buffer [B][rows][3d] (Q | K | V per row);
// the output is written in the operand type for the Wo projection.
#include <cfloat>

#include "kernels.h"

namespace ttt {
namespace {

constexpr int kAttnWarps = 4;       // query positions per block
constexpr int kAttnPerLane = 8;     // head dimension up to 256
constexpr int kAttnKeys = 4;        // keys reduced together

template <typename S>
__global__ void __launch_bounds__(kAttnWarps * 32)
    swa_kernel(int rows, int H, int dh, int window, float scale, const float* __restrict__ qkv, void* out,
               long long out_lo) {
  pdl_wait();
  pdl_launch();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * kAttnWarps + warp;
  if (t >= rows) return;    // whole warps leave; nothing below synchronises the block
  const int head = blockIdx.y;
  const int d = H * dh;
  const long long seq0 = (long long)blockIdx.z * rows;
  const long long ld = 3LL * d;
  const float* qrow = qkv + (seq0 + t) * ld + (long long)head * dh;
  float q[kAttnPerLane], acc[kAttnPerLane];
#pragma unroll
  for (int j = 0; j < kAttnPerLane; ++j) {
    const int e = lane + 32 * j;
    q[j] = e < dh ? qrow[e] * scale : 0.0f;
    acc[j] = 0.0f;
  }
  float m = -FLT_MAX, l = 0.0f;
  const int u0 = t - window + 1 > 0 ? t - window + 1 : 0;
  for (int u = u0; u <= t; u += kAttnKeys) {
    float dot[kAttnKeys];
#pragma unroll
    for (int c = 0; c < kAttnKeys; ++c) {
      dot[c] = 0.0f;
      if (u + c <= t) {
        const float* krow = qkv + (seq0 + u + c) * ld + d + (long long)head * dh;
#pragma unroll
        for (int j = 0; j < kAttnPerLane; ++j) {
          const int e = lane + 32 * j;
          if (e < dh) dot[c] = fmaf(q[j], krow[e], dot[c]);
        }
      }
    }
#pragma unroll
    for (int c = 0; c < kAttnKeys; ++c) dot[c] = warp_sum(dot[c]);
#pragma unroll
    for (int c = 0; c < kAttnKeys; ++c) {
      if (u + c <= t) {
        const float* vrow = qkv + (seq0 + u + c) * ld + 2LL * d + (long long)head * dh;
        const float mn = fmaxf(m, dot[c]);
        const float corr = expf(m - mn);
        const float p = expf(dot[c] - mn);
        l = l * corr + p;
#pragma unroll
        for (int j = 0; j < kAttnPerLane; ++j) {
          const int e = lane + 32 * j;
          if (e < dh) acc[j] = fmaf(p, vrow[e], acc[j] * corr);
        }
        m = mn;
      }
    }
  }
  const float inv = 1.0f / l;
#pragma unroll
  for (int j = 0; j < kAttnPerLane; ++j) {
    const int e = lane + 32 * j;
    if (e < dh) OpIO<S>::store(out, out_lo, (seq0 + t) * d + (long long)head * dh + e, acc[j] * inv);
  }
}

}  // namespace

bool swa_supported(int d, int heads) {
  return heads > 0 && d % heads == 0 && d / heads <= 32 * kAttnPerLane;
}

ttt_status launch_swa(int stg, int B, int rows, int H, int dh, int window, const float* qkv, void* out,
                      long long out_lo, cudaStream_t st) {
  if (B == 0 || rows == 0) return TTT_OK;
  const dim3 grid(ceil_div(rows, kAttnWarps), H, B);
  const float scale = 1.0f / sqrtf((float)dh);
  if (stg == ST_BF16)
    launch_pdl(swa_kernel<bf16>, grid, kAttnWarps * 32, 0, st, rows, H, dh, window, scale, qkv, out, out_lo);
  else if (stg == ST_SPLIT)
    launch_pdl(swa_kernel<Split>, grid, kAttnWarps * 32, 0, st, rows, H, dh, window, scale, qkv, out, out_lo);
  else
    launch_pdl(swa_kernel<float>, grid, kAttnWarps * 32, 0, st, rows, H, dh, window, scale, qkv, out, out_lo);
  TTT_CHECK_LAUNCH();
  return TTT_OK;
}

}  // namespace ttt
