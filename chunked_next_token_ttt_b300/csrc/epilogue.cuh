// Per-element GEMM epilogues shared by the SIMT and tensor-core kernels.
#pragma once

#include "gemm.h"

namespace ttt {

// Applies epilogue g.epi to accumulator `acc` of element (bz, m, n) and
// returns acc^2 for EPI_DW (the per-tile sum of squares feeding the
// per-sequence gradient norm), 0 otherwise.
template <typename OpT>
__device__ __forceinline__ float epi_value(const GemmDesc& g, int bz, int m, int n, float acc) {
  switch (g.epi) {
    case EPI_STORE:
      static_cast<OpT*>(g.out)[bz * g.sO + (long long)m * g.ldo + n] = from_f<OpT>(acc);
      break;
    case EPI_STORE_F32:
      static_cast<float*>(g.out)[bz * g.sO + (long long)m * g.ldo + n] = acc;
      break;
    case EPI_GELU:
      if (g.out) static_cast<OpT*>(g.out)[bz * g.sO + (long long)m * g.ldo + n] = from_f<OpT>(acc);
      static_cast<OpT*>(g.out2)[bz * g.sO2 + (long long)m * g.ldo2 + n] = from_f<OpT>(gelu_f(acc));
      break;
    case EPI_RESID: {
      const float r = static_cast<const float*>(g.aux)[bz * g.sX + (long long)m * g.ldx + n];
      const float v = r + acc;
      static_cast<float*>(g.out)[bz * g.sO + (long long)m * g.ldo + n] = v;
      if (g.out2) static_cast<OpT*>(g.out2)[bz * g.sO2 + (long long)m * g.ldo2 + n] = from_f<OpT>(v);
      break;
    }
    case EPI_SWIGLU: {
      const float gt = static_cast<const float*>(g.aux)[bz * g.sX + (long long)m * g.ldx + n];
      static_cast<OpT*>(g.out)[bz * g.sO + (long long)m * g.ldo + n] = from_f<OpT>(silu_f(gt) * acc);
      break;
    }
    case EPI_DGELU: {
      const float z = to_f(static_cast<const OpT*>(g.aux)[bz * g.sX + (long long)m * g.ldx + n]);
      static_cast<OpT*>(g.out)[bz * g.sO + (long long)m * g.ldo + n] = from_f<OpT>(acc * gelu_grad_f(z));
      break;
    }
    case EPI_DW:
      static_cast<float*>(g.out)[bz * g.sO + (long long)m * g.ldo + n] = acc;
      return acc * acc;
  }
  return 0.0f;
}

}  // namespace ttt
