// tcgen05 GEMM instantiations: A MN-major, B MN-major (dW products).
#include "gemm_tc_kernel.cuh"

namespace ttt {
namespace tc {

template <bool SPLIT>
static ttt_status dispatch_mm(const GemmDesc& g, const CUtensorMap* maps, int nkb, int splitk, cudaStream_t st) {
  switch (g.epi) {
    case EPI_DW: return launch_kernel<true, true, SPLIT, EPI_DW>(g, maps, nkb, splitk, st);
    default: return launch_kernel<true, true, SPLIT, EK_ANY>(g, maps, nkb, splitk, st);
  }
}

ttt_status launch_mm(const GemmDesc& g, const CUtensorMap* maps, int nkb, int splitk, cudaStream_t st) {
  return g.dtype == ST_SPLIT ? dispatch_mm<true>(g, maps, nkb, splitk, st)
                             : dispatch_mm<false>(g, maps, nkb, splitk, st);
}

}  // namespace tc
}  // namespace ttt
