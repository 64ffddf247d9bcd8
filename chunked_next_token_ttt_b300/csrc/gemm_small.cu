// GEMMs with a handful of rows per batch entry (M <= 8): the forward of one
// token per sequence (p_{T+1}, decoding, the b = 1 per-token update) and its
// backward.  Weight-streaming matrix-vector products: every weight element is
// read once, coalesced, and multiplied against the few activation rows.
//   B K-major (B(n,k) = B[n*ldb + k]): one warp per output column n, lanes
//     stride over k, a warp reduction gives the M sums;
//   B N-major (B(n,k) = B[k*ldb + n]): one thread per output column n, the k
//     loop reads consecutive n across the warp.
// A is K-major and small (M * K elements per batch entry); it is read through
// the L1 cache by every warp of the block.
#include "epilogue.cuh"
#include "gemm.h"

namespace ttt {
namespace {

constexpr int kMaxRows = 8;

template <typename S>
__global__ void __launch_bounds__(256) gemm_small_kmajor_kernel(GemmDesc g) {
  pdl_wait();
  pdl_launch();
  using IO = OpIO<S>;
  __shared__ float red[8][kMaxRows];
  const int bz = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long a0 = bz * g.sA, b0 = bz * g.sB;
  float sq = 0.0f;
  for (int n = blockIdx.x * 8 + warp; n < g.N; n += gridDim.x * 8) {
    float acc[kMaxRows];
#pragma unroll
    for (int m = 0; m < kMaxRows; ++m) acc[m] = 0.0f;
    for (int k = lane; k < g.K; k += 32) {
      const float bv = IO::load(g.B, g.loB, b0 + (long long)n * g.ldb + k);
#pragma unroll
      for (int m = 0; m < kMaxRows; ++m)
        if (m < g.M) acc[m] = fmaf(IO::load(g.A, g.loA, a0 + (long long)m * g.lda + k), bv, acc[m]);
    }
#pragma unroll
    for (int m = 0; m < kMaxRows; ++m) acc[m] = warp_sum(acc[m]);
    if (lane == 0)
      for (int m = 0; m < g.M; ++m) sq += epi_value<S>(g, bz, m, n, acc[m]);
  }
  if (g.epi == EPI_DW) {
    sq = warp_sum(sq);
    if (lane == 0) red[warp][0] = sq;
    __syncthreads();
    if (threadIdx.x == 0) {
      float t = 0.0f;
      for (int w = 0; w < 8; ++w) t += red[w][0];
      g.partials[(long long)bz * gridDim.x + blockIdx.x] = t;
    }
  }
}

template <typename S>
__global__ void __launch_bounds__(256) gemm_small_nmajor_kernel(GemmDesc g) {
  pdl_wait();
  pdl_launch();
  using IO = OpIO<S>;
  __shared__ float red[32];
  const int bz = blockIdx.y;
  const long long a0 = bz * g.sA, b0 = bz * g.sB;
  float sq = 0.0f;
  for (int n = blockIdx.x * blockDim.x + threadIdx.x; n < g.N; n += gridDim.x * blockDim.x) {
    float acc[kMaxRows];
#pragma unroll
    for (int m = 0; m < kMaxRows; ++m) acc[m] = 0.0f;
    for (int k = 0; k < g.K; ++k) {
      const float bv = IO::load(g.B, g.loB, b0 + (long long)k * g.ldb + n);
#pragma unroll
      for (int m = 0; m < kMaxRows; ++m)
        if (m < g.M) acc[m] = fmaf(IO::load(g.A, g.loA, a0 + (long long)m * g.lda + k), bv, acc[m]);
    }
    for (int m = 0; m < g.M; ++m) sq += epi_value<S>(g, bz, m, n, acc[m]);
  }
  if (g.epi == EPI_DW) {
    const float t = block_sum(sq, red);
    if (threadIdx.x == 0) g.partials[(long long)bz * gridDim.x + blockIdx.x] = t;
  }
}

int small_grid_x(const GemmDesc& g) {
  const int per_block = g.b_kmajor ? 8 : 256;
  int gx = ceil_div(g.N, per_block);
  // enough blocks to cover the SMs a few times over, at least one column each
  const int target = ceil_div(148 * 4, g.batch);
  return gx < target ? gx : target;
}

}  // namespace

bool gemm_small_supported(const GemmDesc& g) {
  return g.M >= 1 && g.M <= kMaxRows && g.a_kmajor && g.N >= 1 && g.batch >= 1;
}

int gemm_small_partial_tiles(const GemmDesc& g) { return small_grid_x(g); }

ttt_status gemm_small(const GemmDesc& g, cudaStream_t st) {
  dim3 grid(small_grid_x(g), g.batch);
#define TTT_SMALL(KERNEL)                                                                  \
  do {                                                                                     \
    if (g.dtype == ST_BF16) launch_pdl(KERNEL<bf16>, grid, 256, 0, st, g);                         \
    else if (g.dtype == ST_SPLIT) launch_pdl(KERNEL<Split>, grid, 256, 0, st, g);                  \
    else launch_pdl(KERNEL<float>, grid, 256, 0, st, g);                                           \
  } while (0)
  if (g.b_kmajor) TTT_SMALL(gemm_small_kmajor_kernel);
  else TTT_SMALL(gemm_small_nmajor_kernel);
#undef TTT_SMALL
  TTT_CHECK_LAUNCH();
  return TTT_OK;
}

}  // namespace ttt
