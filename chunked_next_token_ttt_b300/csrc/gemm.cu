// GEMM dispatch: the tcgen05 tensor-core kernel where the shape allows it,
// the SIMT kernel otherwise.
#include "gemm.h"

namespace ttt {

int gemm_partial_tiles(const GemmDesc& g) { return gemm_simt_partial_tiles(g); }

ttt_status gemm(const GemmDesc& g, cudaStream_t st) { return gemm_simt(g, st); }

}  // namespace ttt
