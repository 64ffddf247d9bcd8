// GEMM dispatch: the weight-streaming small-M kernel for a few rows per batch
// entry, the tcgen05 tensor-core kernel where the operand storage, shape and
// alignment allow it, the SIMT kernel otherwise (or when forced by impl).
#include "gemm.h"

namespace ttt {

enum Route { ROUTE_SIMT, ROUTE_TC, ROUTE_SMALL };

static Route route(const GemmDesc& g) {
  if (g.B2) return ROUTE_TC;
  if (g.impl == 1) return ROUTE_SIMT;
  if (g.impl == 2 || g.epi == EPI_LOGITS) return ROUTE_TC;
  if (gemm_small_supported(g)) return ROUTE_SMALL;
  if (gemm_tc_supported(g)) return ROUTE_TC;
  return ROUTE_SIMT;
}

int gemm_partial_tiles(const GemmDesc& g) {
  switch (route(g)) {
    case ROUTE_TC: return gemm_tc_partial_tiles(g);
    case ROUTE_SMALL: return gemm_small_partial_tiles(g);
    default: return gemm_simt_partial_tiles(g);
  }
}

int gemm_launches(const GemmDesc&) { return 1; }

ttt_status gemm(const GemmDesc& g, cudaStream_t st) {
  if (g.B2 && !gemm_tc_supported(g)) {
    set_error("a two-plane B operand runs on the tensor-core GEMM only");
    return TTT_ERR_UNSUPPORTED;
  }
  if (g.epi == EPI_LOGITS && route(g) != ROUTE_TC) {
    set_error("the fused logits epilogue runs on the tensor-core GEMM only");
    return TTT_ERR_UNSUPPORTED;
  }
  switch (route(g)) {
    case ROUTE_TC: return gemm_tc(g, st);
    case ROUTE_SMALL: return gemm_small(g, st);
    default: return gemm_simt(g, st);
  }
}

}  // namespace ttt
