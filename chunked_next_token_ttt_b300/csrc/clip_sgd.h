// Clipped SGD step computed from dW (used by the single-operation entry points).
#pragma once

#include "common.cuh"

namespace ttt {

int clip_sgd_pieces(long long n);
// Floats of scratch one call needs: partial sums, per-sequence scales, a flag word.
size_t clip_sgd_scratch_floats(int nslots, int B, long long n);
// Three launches on `st`; *scratch need not be initialised.  The flag word (the
// last float of the scratch, as int) ends up 1 if some sequence's norm was not
// finite, else 0.
ttt_status launch_clip_sgd(int dtype, int nslots, int B, long long n, float* W32, void* Wop, const float* dW,
                           float eta, float clip, float* norm_out, float* scale_out, float* scratch,
                           cudaStream_t st);

}  // namespace ttt
