// Per-element GEMM epilogues shared by the SIMT and tensor-core kernels.
#pragma once

#include "gemm.h"

namespace ttt {

// Applies epilogue g.epi to accumulator `acc` of element (bz, m, n) and
// returns acc^2 for EPI_DW (the per-tile sum of squares feeding the
// per-sequence gradient norm), 0 otherwise.  S is the operand storage.
template <typename S>
__device__ __forceinline__ float epi_value(const GemmDesc& g, int bz, int m, int n, float acc) {
  using IO = OpIO<S>;
  switch (g.epi) {
    case EPI_STORE:
      IO::store(g.out, g.loO, bz * g.sO + (long long)m * g.ldo + n, acc);
      break;
    case EPI_STORE_F32:
      static_cast<float*>(g.out)[bz * g.sO + (long long)m * g.ldo + n] = acc;
      break;
    case EPI_GELU:
      if (g.out) IO::store(g.out, g.loO, bz * g.sO + (long long)m * g.ldo + n, acc);
      IO::store(g.out2, g.loO2, bz * g.sO2 + (long long)m * g.ldo2 + n, gelu_f(acc));
      break;
    case EPI_RESID: {
      const float r = static_cast<const float*>(g.aux)[bz * g.sX + (long long)m * g.ldx + n];
      const float v = r + acc;
      static_cast<float*>(g.out)[bz * g.sO + (long long)m * g.ldo + n] = v;
      if (g.out2) IO::store(g.out2, g.loO2, bz * g.sO2 + (long long)m * g.ldo2 + n, v);
      break;
    }
    case EPI_SWIGLU: {
      const float gt = static_cast<const float*>(g.aux)[bz * g.sX + (long long)m * g.ldx + n];
      IO::store(g.out, g.loO, bz * g.sO + (long long)m * g.ldo + n, silu_f(gt) * acc);
      break;
    }
    case EPI_DGELU: {
      const float z = IO::load(g.aux, g.loX, bz * g.sX + (long long)m * g.ldx + n);
      IO::store(g.out, g.loO, bz * g.sO + (long long)m * g.ldo + n, acc * gelu_grad_f(z));
      break;
    }
    case EPI_DW:
      static_cast<float*>(g.out)[bz * g.sO + (long long)m * g.ldo + n] = acc;
      return acc * acc;
  }
  return 0.0f;
}

// Epilogue kind as a compile-time value; EK_ANY reads g.epi at run time.
constexpr int EK_ANY = -1;

// Pair version of epi_value for elements (m, n) and (m, n + 1), both inside
// the output (n even; every leading dim, batch stride and lo offset even).
// With EK fixed the compiler drops every other branch.
template <typename S, int EK>
__device__ __forceinline__ float epi_pair(const GemmDesc& g, int bz, int m, int n, float a0, float a1) {
  using P = PairIO<S>;
  const int ek = EK == EK_ANY ? (int)g.epi : EK;
  if (ek == EPI_STORE) {
    P::store(g.out, g.loO, bz * g.sO + (long long)m * g.ldo + n, a0, a1);
  } else if (ek == EPI_STORE_F32) {
    PairIO<float>::store(g.out, 0, bz * g.sO + (long long)m * g.ldo + n, a0, a1);
  } else if (ek == EPI_GELU) {
    if (g.out) P::store(g.out, g.loO, bz * g.sO + (long long)m * g.ldo + n, a0, a1);
    P::store(g.out2, g.loO2, bz * g.sO2 + (long long)m * g.ldo2 + n, gelu_f(a0), gelu_f(a1));
  } else if (ek == EPI_RESID) {
    const float2 r = PairIO<float>::load(g.aux, 0, bz * g.sX + (long long)m * g.ldx + n);
    const float v0 = r.x + a0, v1 = r.y + a1;
    PairIO<float>::store(g.out, 0, bz * g.sO + (long long)m * g.ldo + n, v0, v1);
    if (g.out2) P::store(g.out2, g.loO2, bz * g.sO2 + (long long)m * g.ldo2 + n, v0, v1);
  } else if (ek == EPI_SWIGLU) {
    const float2 gt = PairIO<float>::load(g.aux, 0, bz * g.sX + (long long)m * g.ldx + n);
    P::store(g.out, g.loO, bz * g.sO + (long long)m * g.ldo + n, silu_f(gt.x) * a0, silu_f(gt.y) * a1);
  } else if (ek == EPI_DGELU) {
    const float2 z = P::load(g.aux, g.loX, bz * g.sX + (long long)m * g.ldx + n);
    P::store(g.out, g.loO, bz * g.sO + (long long)m * g.ldo + n, a0 * gelu_grad_f(z.x), a1 * gelu_grad_f(z.y));
  } else if (ek == EPI_DW) {
    PairIO<float>::store(g.out, 0, bz * g.sO + (long long)m * g.ldo + n, a0, a1);
    return a0 * a0 + a1 * a1;
  }
  return 0.0f;
}

}  // namespace ttt
