// tcgen05 GEMM instantiations: A MN-major, B K-major.
#include "gemm_tc_kernel.cuh"

namespace ttt {
namespace tc {

template <bool SPLIT>
static ttt_status dispatch_mk(const GemmDesc& g, const CUtensorMap* maps, int nkb, int splitk, cudaStream_t st) {
  return launch_kernel<true, false, SPLIT, EK_ANY>(g, maps, nkb, splitk, st);
}

ttt_status launch_mk(const GemmDesc& g, const CUtensorMap* maps, int nkb, int splitk, cudaStream_t st) {
  return g.dtype == ST_SPLIT ? dispatch_mk<true>(g, maps, nkb, splitk, st)
                             : dispatch_mk<false>(g, maps, nkb, splitk, st);
}

}  // namespace tc
}  // namespace ttt
