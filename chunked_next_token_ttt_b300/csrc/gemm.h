// Internal GEMM interface of libttt: C[M, N] = sum_k A(m, k) B(n, k), batched,
// with the fused epilogues the TTT chunk step needs.
#pragma once

#include "common.cuh"

namespace ttt {

enum EpiKind {
  EPI_STORE = 0,   // out(op type) = acc
  EPI_STORE_F32,   // out(float) = acc
  EPI_GELU,        // out(op) = z = acc (stash), out2(op) = GELU(z)
  EPI_RESID,       // out(float) = aux(float) + acc; out2(op) = same, if non-null
  EPI_SWIGLU,      // out(op) = silu(aux(float)) * acc
  EPI_DGELU,       // out(op) = acc * GELU'(aux(op))
  EPI_DW,          // out = acc (bf16 for bf16 storage, float otherwise);
                   // partials += per-tile sum of acc^2 (fp32 accumulators)
  EPI_LOGITS,      // tensor-core path only, batch 1: out(bf16) = acc when out is
                   // non-null; lse_part[m][tile] = (max, sum exp(acc - max)) over the
                   // tile's columns
};

struct GemmDesc {
  int M = 0, N = 0, K = 0, batch = 1;
  int dtype = ST_F32;              // operand storage of A, B and op-typed outputs (Storage)
  bool a_kmajor = true;            // A(m,k) at A[m*lda + k] (else A[k*lda + m])
  bool b_kmajor = true;            // B(n,k) at B[n*ldb + k] (else B[k*ldb + n])
  const void* A = nullptr; long long lda = 0, sA = 0;   // strides in elements
  const void* B = nullptr; long long ldb = 0, sB = 0;
  // bf16 storage only: B is the sum of two bf16 planes, B and B2 (same leading
  // dim and batch stride), taken as two tensor-core products
  const void* B2 = nullptr;
  EpiKind epi = EPI_STORE;
  void* out = nullptr; long long ldo = 0, sO = 0;
  void* out2 = nullptr; long long ldo2 = 0, sO2 = 0;
  const void* aux = nullptr; long long ldx = 0, sX = 0;
  float* partials = nullptr;       // EPI_DW: [batch][gemm_partial_tiles()]
  // ST_SPLIT only: element offset of each op-typed pointer's lo plane
  long long loA = 0, loB = 0, loO = 0, loO2 = 0, loX = 0;
  float2* lse_part = nullptr;      // EPI_LOGITS: [M][lse_ld] online-softmax states
  long long lse_ld = 0;
  int* err = nullptr;              // device status word for bounded-wait timeouts
  int impl = 0;                    // 0 auto, 1 SIMT, 2 tensor cores
  // optional fp32 workspace; the tensor-core path uses it to split K when a
  // GEMM has too few output tiles to fill the GPU
  float* ws = nullptr;
  long long ws_elems = 0;
  // split-K arrival counters, one per output tile, zero between launches; GEMMs
  // that share them must run in stream order (null: K is never split)
  int* cnt = nullptr;
  // cap on the tensor-core kernel's persistent grid (0: one CTA per SM)
  int max_ctas = 0;
  // set by the tensor-core host code: every epilogue pointer, leading dim,
  // batch stride and lo offset is a multiple of 16 elements with 32-byte aligned
  // pointers (2: 32-byte accesses), else of 8 elements with 16-byte aligned
  // pointers (1: 16-byte accesses), else 0 (element by element)
  int vec = 0;
  int bn = 128;                    // output tile width chosen by the tensor-core host code
};

// Status bits the tensor-core kernel raises in *err when a bounded wait gives up.
constexpr int kErrGemmTimeout = 8 | 16 | 32;

// Which implementation ran a GEMM (for launch accounting and tests).
enum GemmImpl { GEMM_IMPL_SIMT = 0, GEMM_IMPL_TC = 1 };

// Number of per-batch partial slots an EPI_DW launch writes.
int gemm_partial_tiles(const GemmDesc& g);
ttt_status gemm(const GemmDesc& g, cudaStream_t st);
// Kernels one gemm() call launches.
int gemm_launches(const GemmDesc& g);
int gemm_tc_splitk(const GemmDesc& g);
ttt_status gemm_simt(const GemmDesc& g, cudaStream_t st);
int gemm_simt_partial_tiles(const GemmDesc& g);
bool gemm_small_supported(const GemmDesc& g);
int gemm_small_partial_tiles(const GemmDesc& g);
ttt_status gemm_small(const GemmDesc& g, cudaStream_t st);
bool gemm_tc_supported(const GemmDesc& g);
// Output-tile width the tensor-core kernel uses for g (the column tiles of
// EPI_LOGITS, the per-tile partials of EPI_DW).
int gemm_tc_tile_n(const GemmDesc& g);
// Capacity of a split-K arrival-counter array, in output tiles.
int gemm_tc_max_split_tiles();
// The library's status word for tensor-core GEMMs launched without one.
ttt_status gemm_tc_status_word(int** err);
int gemm_tc_partial_tiles(const GemmDesc& g);
ttt_status gemm_tc(const GemmDesc& g, cudaStream_t st);

}  // namespace ttt
