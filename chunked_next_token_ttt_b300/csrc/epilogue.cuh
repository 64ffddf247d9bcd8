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

}  // namespace ttt
