/*
 * libttt single-operation entry points.
 *
 * Each call runs one stage of the TTT chunk step on device buffers the caller
 * owns, in stream order on `stream`; none allocates device memory, and only
 * the clipped SGD step synchronises (to read its status).  They exist for
 * per-kernel tests and measurements and for callers that assemble their own
 * loop; ttt.h's ttt_prefill runs the same stages.  All pointers are device
 * pointers.  Errors are returned as ttt_status (ttt.h); nothing aborts.
 */
#ifndef TTT_OPS_H_
#define TTT_OPS_H_

#include "ttt.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Epilogues of ttt_op_gemm (acc = sum_k A(m,k) B(n,k) in fp32). */
enum {
  TTT_EPI_STORE = 0,     /* out(operand type) = acc                              */
  TTT_EPI_STORE_F32 = 1, /* out(float) = acc                                     */
  TTT_EPI_GELU = 2,      /* out(op) = acc (may be NULL), out2(op) = GELU(acc)    */
  TTT_EPI_RESID = 3,     /* out(float) = aux(float) + acc; out2(op) = same or NULL */
  TTT_EPI_SWIGLU = 4,    /* out(op) = silu(aux(float)) * acc                     */
  TTT_EPI_DGELU = 5,     /* out(op) = acc * GELU'(aux(op))                       */
  TTT_EPI_DW = 6         /* out = acc (bf16 when dtype is TTT_DTYPE_BF16, float
                            otherwise); partials[b * tiles + t] = per-tile sum of
                            acc^2 of the fp32 accumulators (tiles =
                            ttt_op_gemm_partial_tiles)                           */
};
enum { TTT_GEMM_AUTO = 0, TTT_GEMM_SIMT = 1, TTT_GEMM_TENSOR = 2 };
/* Operand storage code accepted by ttt_op_gemm besides TTT_DTYPE_FP32/BF16:
 * fp32-accurate values kept as two bf16 planes, hi = bf16(v) at p[i] and
 * lo = bf16(v - hi) at p[lo + i] (lo offsets in ttt_gemm_args.lo*); products
 * are taken as hi*hi + hi*lo + lo*hi with fp32 accumulation. */
enum { TTT_STORAGE_BF16X3 = 2 };

/* A batched GEMM C[b][m][n] = epilogue(sum_k A[b](m,k) B[b](n,k)).
 * A(m,k) = A[m*lda + k] when a_kmajor, else A[k*lda + m]; likewise B(n,k) with
 * b_kmajor.  s* are per-batch strides; all strides are in elements.  dtype is
 * the operand storage of A, B and every "op"-typed output (TTT_DTYPE_FP32,
 * TTT_DTYPE_BF16 or TTT_STORAGE_BF16X3).  impl selects the kernel:
 * TTT_GEMM_TENSOR (tcgen05; bf16 or bf16x3 storage, leading dims, batch
 * strides and lo offsets multiples of 8, 16-byte aligned bases) returns
 * TTT_ERR_UNSUPPORTED when the shape does not qualify. */
typedef struct {
  int M, N, K, batch;
  int dtype, a_kmajor, b_kmajor, epi, impl;
  const void* A; long long lda, sA;
  const void* B; long long ldb, sB;
  void* out; long long ldo, sO;
  void* out2; long long ldo2, sO2;
  const void* aux; long long ldx, sX;
  float* partials;
  long long loA, loB, loO, loO2, loX;   /* lo-plane offsets (TTT_STORAGE_BF16X3 only) */
  float* workspace;                     /* optional fp32 device buffer (more than 4096
                                           elements): lets the tensor-core path split K
                                           when the output has few tiles.  Its last 4096
                                           words hold the split-K arrival counters, which
                                           the call clears in stream order; calls that
                                           share a workspace must run in stream order */
  long long workspace_elems;
} ttt_gemm_args;

ttt_status ttt_op_gemm(const ttt_gemm_args* args, ttt_stream stream);
/* Number of partial sums per batch entry an TTT_EPI_DW call writes. */
int ttt_op_gemm_partial_tiles(const ttt_gemm_args* args);

/* Sliding-window multi-head attention, forward ("End-to-End TTT" review,
 * Method: the sliding-window attention fix of the bigram defect), as the fused
 * tensor-core kernel the prefill runs: bf16 storage, head width 64 or 128.
 *   qkv  [B][L][3d] bf16 rows Q | K | V (d = heads * head_dim); position p of
 *        sequence s is row pad + p, p < rows; L >= pad + ceil(rows / 128) * 128;
 *        rows of other positions must hold finite values (they are read, then
 *        masked).
 *   out  [B][L][d] bf16: row pad + p gets, for every head h, softmax over keys
 *        p - window < q <= p (q >= 0) of (Q_p . K_q) / sqrt(head_dim), times V.
 * Errors: BAD_ARG, UNSUPPORTED (dtype, head width, alignment), TIMEOUT (read
 * by synchronising `stream`), CUDA. */
ttt_status ttt_op_sliding_window_attention(int dtype, int B, int rows, int heads, int head_dim, int window,
                                           const void* qkv, int pad, long long L, void* out, ttt_stream stream);

/* Softmax cross-entropy of each row of logits [M, V] (operand type) against
 * targets [M] (int32 in [0, V)): losses[m] = logsumexp(row) - row[target]
 * ("End-to-End TTT" review, eq. (1)).  When grad != 0 the row is overwritten
 * in place by dlogits = (softmax(row) - onehot(target)) * scale (eq. (5) uses
 * scale = 1/b).  A target outside [0, V) is read as 0 (no out-of-range access). */
ttt_status ttt_op_cross_entropy(int dtype, int M, int V, void* logits, const int32_t* targets,
                                float scale, int grad, float* losses, ttt_stream stream);

/* RMSNorm with unit gain: y = x * rstd, rstd = 1/sqrt(mean(x^2) + eps).
 * x [M, d] float; y [M, d] operand type; rstd [M] float. */
ttt_status ttt_op_rmsnorm_forward(int dtype, int M, int d, const float* x, float eps, void* y,
                                  float* rstd, ttt_stream stream);

/* dx = rstd * (dy - xhat * mean(xhat * dy)), xhat = x * rstd.  dx [M, d] float;
 * dx_op [M, d] operand type or NULL. */
ttt_status ttt_op_rmsnorm_backward(int dtype, int M, int d, const float* x, const float* rstd,
                                   const float* dy, float* dx, void* dx_op, ttt_stream stream);

/* Global-norm clipped SGD step on a fast-weight arena ("Self-Generated Feedback
 * Destabilizes TTT" summary: one clipped gradient step per chunk; "End-to-End
 * TTT" review eq. (5): W <- W - eta * g).
 *   W32  [nslots][B][n] float, updated in place.
 *   Wop  [nslots][B][n] operand-type copy of the result (non-NULL).
 *   dW   [nslots][B][n] float gradients.
 * For each sequence s, norm_s = ||dW[:, s, :]||_2 over all its slots,
 * scale_s = min(1, clip / (norm_s + 1e-6)) (1 when clip == 0; 0 and status
 * TTT_ERR_NONFINITE when norm_s is not finite, which leaves that sequence's
 * weights unchanged), then W32 -= eta * scale_s * dW.
 * norm_out, scale_out [B] float or NULL.  workspace: device buffer of at least
 * ttt_clip_sgd_workspace_size(nslots, B, n) bytes, caller-owned; its contents
 * need no initialisation.  The call synchronises `stream` to read the status. */
ttt_status ttt_clip_sgd(int dtype, int nslots, int B, long long n, float* W32, void* Wop,
                        const float* dW, float eta, float clip, float* norm_out, float* scale_out,
                        void* workspace, size_t workspace_bytes, ttt_stream stream);
size_t ttt_clip_sgd_workspace_size(int nslots, int B, long long n);

/* ttt_clip_sgd without a workspace, for callers that cannot allocate device
 * memory: their device memory is owned by their own allocator or budget and
 * they have no buffer to hand over, or they cannot accept cudaMalloc's
 * implicit synchronisation in their loop.  The pages have no counterpart: this
 * is a property of the library, not of the method.
 * Same arguments, results and status codes as ttt_clip_sgd.  The scratch is a
 * fixed device array of TTT_CLIP_SGD_NOALLOC_MAX_FLOATS floats (4 MiB) inside
 * the library, held by every GPU that loads it until the process exits; the
 * call allocates nothing (no cudaMalloc, cudaFree or allocating routine).
 * Sizes needing more than the maximum, i.e. nslots * B * ceil(n / 8192) + B + 1
 * floats, return TTT_ERR_BAD_SHAPE with a message naming the limit.
 * The first call in a CUDA context (per device, and again after a device
 * reset) looks up the array's device address there (cudaGetSymbolAddress);
 * make that first call before any stream capture.  Like ttt_clip_sgd, every
 * call copies the status word to the host and synchronises `stream` before it
 * returns.  All calls share the one array: calls that overlap on the GPU (on
 * different streams or from different host threads) race and must be
 * serialised by the caller.  Nothing in the array needs to start at zero:
 * each call writes every word before it reads it. */
#define TTT_CLIP_SGD_NOALLOC_MAX_FLOATS (1 << 20)
ttt_status ttt_clip_sgd_noalloc(int dtype, int nslots, int B, long long n, float* W32, void* Wop,
                                const float* dW, float eta, float clip, float* norm_out,
                                float* scale_out, ttt_stream stream);

#ifdef __cplusplus
}
#endif
#endif /* TTT_OPS_H_ */
