// GEMM dispatch: the tcgen05 tensor-core kernel where the operand type, shape
// and alignment allow it, the SIMT kernel otherwise (or when forced by impl).
#include "gemm.h"

namespace ttt {

static bool use_tc(const GemmDesc& g) {
  if (g.impl == 1) return false;
  if (g.impl == 2) return true;
  return gemm_tc_supported(g);
}

int gemm_partial_tiles(const GemmDesc& g) {
  return use_tc(g) ? gemm_tc_partial_tiles(g) : gemm_simt_partial_tiles(g);
}

ttt_status gemm(const GemmDesc& g, cudaStream_t st) { return use_tc(g) ? gemm_tc(g, st) : gemm_simt(g, st); }

}  // namespace ttt
