// tcgen05 GEMM instantiations: A K-major, B MN-major (dX and head-backward products).
#include "gemm_tc_kernel.cuh"

namespace ttt {
namespace tc {

template <bool SPLIT>
static ttt_status dispatch_km(const GemmDesc& g, const CUtensorMap* maps, int nkb, int splitk, cudaStream_t st) {
  switch (g.epi) {
    case EPI_STORE_F32: return launch_kernel<false, true, SPLIT, EPI_STORE_F32>(g, maps, nkb, splitk, st);
    case EPI_DGELU: return launch_kernel<false, true, SPLIT, EPI_DGELU>(g, maps, nkb, splitk, st);
    case EPI_RESID: return launch_kernel<false, true, SPLIT, EPI_RESID>(g, maps, nkb, splitk, st);
    default: return launch_kernel<false, true, SPLIT, EK_ANY>(g, maps, nkb, splitk, st);
  }
}

ttt_status launch_km(const GemmDesc& g, const CUtensorMap* maps, int nkb, int splitk, cudaStream_t st) {
  return g.dtype == ST_SPLIT ? dispatch_km<true>(g, maps, nkb, splitk, st)
                             : dispatch_km<false>(g, maps, nkb, splitk, st);
}

}  // namespace tc
}  // namespace ttt
