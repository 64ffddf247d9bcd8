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

// Eight consecutive elements (16 bytes per plane) as fp32.
template <typename S> struct Vec8;
template <> struct Vec8<bf16> {
  __device__ __forceinline__ static void load(const void* p, long long, long long i, float* v) {
    unpack_bf16x8(*reinterpret_cast<const uint4*>(static_cast<const bf16*>(p) + i), v);
  }
};
template <> struct Vec8<Split> {
  __device__ __forceinline__ static void load(const void* p, long long lo, long long i, float* v) {
    OctIO<Split>::load(p, lo, i, v);
  }
};
template <> struct Vec8<float> {
  __device__ __forceinline__ static void load(const void* p, long long, long long i, float* v) {
    OctIO<float>::load(p, 0, i, v);
  }
};

// B K-major with 16-byte loads: each warp computes CW adjacent output columns
// at once, each lane taking eight consecutive k per step (a warp reads 256
// consecutive k of CW weight rows per step and plane); every 16-byte chunk of
// the M activation rows (through L1) serves all CW columns.  U steps are
// loaded before any of them is used, so a lane keeps U x CW 16-byte weight
// loads in flight.  CW = 4 for wide outputs (N >= kWideN: vocabulary heads,
// wide projections) of one or two rows, 1 otherwise so that narrow outputs
// still spread over enough warps.  U = 4 (2 with four columns), except for
// hi/lo split operands with more than two rows, whose doubled loads would
// spill at that depth (U = 1 measured faster there).  After the warp
// reduction every lane holds
// the sums and lane m applies the epilogue of row m.  Needs K, lda, ldb, the
// batch strides and lo offsets multiples of 8 and 16-byte aligned bases
// (gemm_small_vec_ok).
constexpr int kWideN = 8192;

template <typename S, int kCW, int kU>
__device__ __forceinline__ void kvec_steps(const GemmDesc& g, long long a0, long long b0, int n0, int k,
                                           float (&acc)[kCW][kMaxRows]) {
  float bv[kU][kCW][8];
#pragma unroll
  for (int u = 0; u < kU; ++u)
#pragma unroll
    for (int c = 0; c < kCW; ++c) {
      const int n = n0 + c < g.N ? n0 + c : g.N - 1;   // clamp: the extra columns are not stored
      Vec8<S>::load(g.B, g.loB, b0 + (long long)n * g.ldb + k + 256 * u, bv[u][c]);
    }
#pragma unroll
  for (int u = 0; u < kU; ++u)
#pragma unroll
    for (int m = 0; m < kMaxRows; ++m) {
      if (m < g.M) {
        float av[8];
        Vec8<S>::load(g.A, g.loA, a0 + (long long)m * g.lda + k + 256 * u, av);
#pragma unroll
        for (int c = 0; c < kCW; ++c)
#pragma unroll
          for (int j = 0; j < 8; ++j) acc[c][m] = fmaf(av[j], bv[u][c][j], acc[c][m]);
      }
    }
}

template <typename S, int kCW, int kU>
__global__ void __launch_bounds__(256) gemm_small_kvec_kernel(GemmDesc g) {
  pdl_wait();
  pdl_launch();
  __shared__ float red[8];
  const int bz = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long a0 = bz * g.sA, b0 = bz * g.sB;
  float sq = 0.0f;
  for (int n0 = (blockIdx.x * 8 + warp) * kCW; n0 < g.N; n0 += gridDim.x * 8 * kCW) {
    float acc[kCW][kMaxRows];
#pragma unroll
    for (int c = 0; c < kCW; ++c)
#pragma unroll
      for (int m = 0; m < kMaxRows; ++m) acc[c][m] = 0.0f;
    int k = lane * 8;
    for (; k + 256 * (kU - 1) < g.K; k += 256 * kU) kvec_steps<S, kCW, kU>(g, a0, b0, n0, k, acc);
    for (; k < g.K; k += 256) kvec_steps<S, kCW, 1>(g, a0, b0, n0, k, acc);
#pragma unroll
    for (int c = 0; c < kCW; ++c)
#pragma unroll
      for (int m = 0; m < kMaxRows; ++m)
        if (m < g.M) acc[c][m] = warp_sum(acc[c][m]);
    // lane m takes row m (selected without a dynamic register index)
#pragma unroll
    for (int c = 0; c < kCW; ++c) {
      float v = 0.0f;
#pragma unroll
      for (int m = 0; m < kMaxRows; ++m)
        if (m == lane) v = acc[c][m];
      if (lane < g.M && n0 + c < g.N) sq += epi_value<S>(g, bz, lane, n0 + c, v);
    }
  }
  if (g.epi == EPI_DW) {
    sq = warp_sum(sq);
    if (lane == 0) red[warp] = sq;
    __syncthreads();
    if (threadIdx.x == 0) {
      float t = 0.0f;
      for (int w = 0; w < 8; ++w) t += red[w];
      g.partials[(long long)bz * gridDim.x + blockIdx.x] = t;
    }
  }
}

// Shared-weight products of a few rows with few output columns (the frozen
// blocks and the head of a one-token-per-sequence forward, M = B rows): kw
// warps share one column, each taking every kw-th 256-wide step of K, and the
// block sums their partial dot products in a fixed order before the epilogue
// (lane m takes row m).  This puts kw times more warps in flight than one
// warp per column, for the narrow and long-K shapes where that is too few.
template <typename S>
__global__ void __launch_bounds__(256) gemm_small_ksplit_kernel(GemmDesc g, int kw) {
  pdl_wait();
  pdl_launch();
  __shared__ float part[8][kMaxRows];
  const int bz = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cw = warp / kw, kp = warp % kw;
  const int n = blockIdx.x * (8 / kw) + cw;
  const long long a0 = bz * g.sA, b0 = bz * g.sB;
  float acc[kMaxRows];
#pragma unroll
  for (int m = 0; m < kMaxRows; ++m) acc[m] = 0.0f;
  if (n < g.N) {
    for (int k = (kp * 32 + lane) * 8; k < g.K; k += kw * 256) {
      float bv[8];
      Vec8<S>::load(g.B, g.loB, b0 + (long long)n * g.ldb + k, bv);
#pragma unroll
      for (int m = 0; m < kMaxRows; ++m) {
        if (m < g.M) {
          float av[8];
          Vec8<S>::load(g.A, g.loA, a0 + (long long)m * g.lda + k, av);
#pragma unroll
          for (int j = 0; j < 8; ++j) acc[m] = fmaf(av[j], bv[j], acc[m]);
        }
      }
    }
  }
#pragma unroll
  for (int m = 0; m < kMaxRows; ++m) {
    if (m < g.M) {
      const float v = warp_sum(acc[m]);
      if (lane == 0) part[warp][m] = v;
    }
  }
  __syncthreads();
  if (kp == 0 && n < g.N && lane < g.M) {
    float v = 0.0f;
    for (int q = 0; q < kw; ++q) v += part[cw * kw + q][lane];
    epi_value<S>(g, bz, lane, n, v);
  }
}

bool gemm_small_vec_ok(const GemmDesc& g) {
  auto al = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; };
  const long long m = (long long)g.K | g.lda | g.ldb | g.sA | g.sB | g.loA | g.loB;
  return g.b_kmajor && (m & 7) == 0 && al(g.A) && al(g.B);
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

bool gemm_small_vec_ok(const GemmDesc& g);

// four columns per warp pay for wide outputs with one or two rows; with more
// rows the 4 x M accumulators crowd the registers (measured slower)
int small_cols_per_warp(const GemmDesc& g) { return (g.N >= kWideN && g.M <= 2) ? 4 : 1; }

// warps per output column of the K-split variant (1: not used): a power of
// two up to 8, at most one 256-wide K step each, until the grid holds about 48
// warps per SM; never for dW products (their per-block norm partials follow
// small_grid_x)
int small_ksplit(const GemmDesc& g) {
  if (!gemm_small_vec_ok(g) || g.M <= 2 || g.epi == EPI_DW) return 1;
  const long long cols = (long long)g.N * g.batch;
  int kmax = ceil_div(g.K, 256);
  if (kmax > 8) kmax = 8;
  int kw = 1;
  while (kw * 2 <= kmax && cols * kw < 148LL * 48) kw *= 2;
  return kw;
}

// the deeply unrolled weight-streaming variant (U = 4) suits this product
bool small_deep_unroll(const GemmDesc& g) { return g.dtype != ST_SPLIT || g.M <= 2; }

int small_grid_x(const GemmDesc& g) {
  const int per_block = gemm_small_vec_ok(g) ? 8 * small_cols_per_warp(g) : (g.b_kmajor ? 8 : 256);
  int gx = ceil_div(g.N, per_block);
  // enough blocks to cover the SMs several times over (more for the
  // latency-bound one- and two-row products), at least one column each
  const int target = ceil_div(148 * (small_deep_unroll(g) ? 8 : 4), g.batch);
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
#define TTT_KVEC(CW, U)                                                                        \
  do {                                                                                         \
    if (g.dtype == ST_BF16) launch_pdl(gemm_small_kvec_kernel<bf16, CW, U>, grid, 256, 0, st, g);        \
    else if (g.dtype == ST_SPLIT) launch_pdl(gemm_small_kvec_kernel<Split, CW, U>, grid, 256, 0, st, g); \
    else launch_pdl(gemm_small_kvec_kernel<float, CW, U>, grid, 256, 0, st, g);                          \
  } while (0)
  const int kw = small_ksplit(g);
  if (kw > 1) {
    const dim3 kgrid(ceil_div(g.N, 8 / kw), g.batch);
    if (g.dtype == ST_BF16) launch_pdl(gemm_small_ksplit_kernel<bf16>, kgrid, 256, 0, st, g, kw);
    else if (g.dtype == ST_SPLIT) launch_pdl(gemm_small_ksplit_kernel<Split>, kgrid, 256, 0, st, g, kw);
    else launch_pdl(gemm_small_ksplit_kernel<float>, kgrid, 256, 0, st, g, kw);
  } else if (gemm_small_vec_ok(g) && small_cols_per_warp(g) == 4) TTT_KVEC(4, 2);
  else if (gemm_small_vec_ok(g) && small_deep_unroll(g)) TTT_KVEC(1, 4);
  else if (gemm_small_vec_ok(g)) TTT_KVEC(1, 1);
#undef TTT_KVEC
  else if (g.b_kmajor) TTT_SMALL(gemm_small_kmajor_kernel);
  else TTT_SMALL(gemm_small_nmajor_kernel);
#undef TTT_SMALL
  TTT_CHECK_LAUNCH();
  return TTT_OK;
}

}  // namespace ttt
