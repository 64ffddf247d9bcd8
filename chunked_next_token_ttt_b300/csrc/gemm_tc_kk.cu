// tcgen05 GEMM instantiations: A K-major, B K-major (forward products).
#include "gemm_tc_kernel.cuh"

namespace ttt {
namespace tc {

template <bool SPLIT>
static ttt_status dispatch_kk(const GemmDesc& g, const CUtensorMap* maps, int nkb, int splitk, cudaStream_t st) {
  switch (g.epi) {
    case EPI_STORE: return launch_kernel<false, false, SPLIT, EPI_STORE>(g, maps, nkb, splitk, st);
    case EPI_STORE_F32: return launch_kernel<false, false, SPLIT, EPI_STORE_F32>(g, maps, nkb, splitk, st);
    case EPI_GELU: return launch_kernel<false, false, SPLIT, EPI_GELU>(g, maps, nkb, splitk, st);
    case EPI_RESID: return launch_kernel<false, false, SPLIT, EPI_RESID>(g, maps, nkb, splitk, st);
    case EPI_SWIGLU: return launch_kernel<false, false, SPLIT, EPI_SWIGLU>(g, maps, nkb, splitk, st);
    case EPI_DGELU: return launch_kernel<false, false, SPLIT, EPI_DGELU>(g, maps, nkb, splitk, st);
    case EPI_DW: return launch_kernel<false, false, SPLIT, EPI_DW>(g, maps, nkb, splitk, st);
    case EPI_LOGITS:
      if constexpr (!SPLIT) return launch_kernel<false, false, false, EPI_LOGITS>(g, maps, nkb, splitk, st);
      set_error("the fused logits epilogue takes bf16 operands");
      return TTT_ERR_UNSUPPORTED;
    default: return launch_kernel<false, false, SPLIT, EK_ANY>(g, maps, nkb, splitk, st);
  }
}

ttt_status launch_kk_b2(const GemmDesc& g, const CUtensorMap* maps, int nkb, int splitk, cudaStream_t st) {
  switch (g.epi) {
    case EPI_GELU: return launch_bn<kBN, false, false, PL_B2, EPI_GELU>(g, maps, nkb, splitk, st);
    case EPI_RESID: return launch_bn<kBN, false, false, PL_B2, EPI_RESID>(g, maps, nkb, splitk, st);
    default:
      set_error("a two-plane B operand runs with the GELU or residual epilogue");
      return TTT_ERR_UNSUPPORTED;
  }
}

ttt_status launch_kk(const GemmDesc& g, const CUtensorMap* maps, int nkb, int splitk, cudaStream_t st) {
  return g.dtype == ST_SPLIT ? dispatch_kk<true>(g, maps, nkb, splitk, st)
                             : dispatch_kk<false>(g, maps, nkb, splitk, st);
}

}  // namespace tc
}  // namespace ttt
