// Plain SIMT GEMM with the TTT epilogues (fp32 FMA, fp32 accumulation).
//
// Serves shapes the tensor-core kernel does not take (per-sequence row counts
// that are not a multiple of 128: the b = 1 toy, decoding, p_{T+1}) and is the
// fp32 reference path.  64x64 output tile, 16-deep k slices, 256 threads,
// 4x4 outputs per thread.
#include "epilogue.cuh"
#include "gemm.h"

namespace ttt {
namespace {

constexpr int TM = 64, TN = 64, TK = 16;

template <typename S, bool AK, bool BK>
__global__ void __launch_bounds__(256) gemm_simt_kernel(GemmDesc g) {
  pdl_wait();
  pdl_launch();
  using IO = OpIO<S>;
  __shared__ float As[TK][TM + 4];
  __shared__ float Bs[TK][TN + 4];
  __shared__ float red[32];
  const int bz = blockIdx.z;
  const long long a0 = bz * g.sA, b0 = bz * g.sB;
  const int m0 = blockIdx.y * TM, n0 = blockIdx.x * TN;
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.0f;

  for (int k0 = 0; k0 < g.K; k0 += TK) {
    for (int i = tid; i < TM * TK; i += 256) {
      int mm, kk;
      if (AK) { mm = i / TK; kk = i % TK; } else { kk = i / TM; mm = i % TM; }
      const int gm = m0 + mm, gk = k0 + kk;
      float v = 0.0f;
      if (gm < g.M && gk < g.K)
        v = IO::load(g.A, g.loA, a0 + (AK ? (long long)gm * g.lda + gk : (long long)gk * g.lda + gm));
      As[kk][mm] = v;
    }
    for (int i = tid; i < TN * TK; i += 256) {
      int nn, kk;
      if (BK) { nn = i / TK; kk = i % TK; } else { kk = i / TN; nn = i % TN; }
      const int gn = n0 + nn, gk = k0 + kk;
      float v = 0.0f;
      if (gn < g.N && gk < g.K)
        v = IO::load(g.B, g.loB, b0 + (BK ? (long long)gn * g.ldb + gk : (long long)gk * g.ldb + gn));
      Bs[kk][nn] = v;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < TK; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }

  float sq = 0.0f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int m = m0 + ty * 4 + i;
    if (m >= g.M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tx * 4 + j;
      if (n < g.N) sq += epi_value<S>(g, bz, m, n, acc[i][j]);
    }
  }
  if (g.epi == EPI_DW) {
    const float tot = block_sum(sq, red);
    if (tid == 0)
      g.partials[(long long)bz * gridDim.x * gridDim.y + blockIdx.y * gridDim.x + blockIdx.x] = tot;
  }
}

template <typename S>
void launch(const GemmDesc& g, dim3 grid, cudaStream_t st) {
  if (g.a_kmajor && g.b_kmajor) launch_pdl(gemm_simt_kernel<S, true, true>, grid, 256, 0, st, g);
  else if (g.a_kmajor) launch_pdl(gemm_simt_kernel<S, true, false>, grid, 256, 0, st, g);
  else if (g.b_kmajor) launch_pdl(gemm_simt_kernel<S, false, true>, grid, 256, 0, st, g);
  else launch_pdl(gemm_simt_kernel<S, false, false>, grid, 256, 0, st, g);
}

}  // namespace

int gemm_simt_partial_tiles(const GemmDesc& g) { return ceil_div(g.M, TM) * ceil_div(g.N, TN); }

ttt_status gemm_simt(const GemmDesc& g, cudaStream_t st) {
  if (g.M <= 0 || g.N <= 0 || g.batch <= 0) return TTT_OK;
  dim3 grid(ceil_div(g.N, TN), ceil_div(g.M, TM), g.batch);
  if (g.dtype == ST_BF16) launch<bf16>(g, grid, st);
  else if (g.dtype == ST_SPLIT) launch<Split>(g, grid, st);
  else launch<float>(g, grid, st);
  TTT_CHECK_LAUNCH();
  return TTT_OK;
}

}  // namespace ttt
