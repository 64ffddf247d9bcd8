// Single-operation C entry points (include/ttt_ops.h).
#include "clip_sgd.h"
#include "gemm.h"
#include "kernels.h"
#include "ttt_ops.h"

using namespace ttt;

// Status word of the single-operation cross-entropy (token ids outside [0, V)
// are recorded here): file-scope device memory, so no call allocates.
static __device__ int g_ce_status;
// Status word of the single-operation attention (bounded-wait timeouts).
static __device__ int g_attn_status;

static ttt_status bad(ttt_status s, const char* msg) {
  set_error(msg);
  return s;
}

static bool to_desc(const ttt_gemm_args* a, GemmDesc* g) {
  if (!a || a->M < 0 || a->N < 0 || a->K < 0 || a->batch < 1 || a->epi < 0 || a->epi > TTT_EPI_DW) return false;
  if (a->dtype != ST_F32 && a->dtype != ST_BF16 && a->dtype != ST_SPLIT) return false;
  if (!a->A || !a->B || !a->out) return false;
  g->M = a->M; g->N = a->N; g->K = a->K; g->batch = a->batch; g->dtype = a->dtype;
  g->a_kmajor = a->a_kmajor != 0; g->b_kmajor = a->b_kmajor != 0;
  g->A = a->A; g->lda = a->lda; g->sA = a->sA;
  g->B = a->B; g->ldb = a->ldb; g->sB = a->sB;
  g->epi = static_cast<EpiKind>(a->epi);
  g->out = a->out; g->ldo = a->ldo; g->sO = a->sO;
  g->out2 = a->out2; g->ldo2 = a->ldo2; g->sO2 = a->sO2;
  g->aux = a->aux; g->ldx = a->ldx; g->sX = a->sX;
  g->partials = a->partials;
  g->impl = a->impl;
  g->loA = a->loA; g->loB = a->loB; g->loO = a->loO; g->loO2 = a->loO2; g->loX = a->loX;
  // the workspace's last gemm_tc_max_split_tiles() words hold the split-K
  // arrival counters; the rest takes the partial tiles
  const long long ncnt = gemm_tc_max_split_tiles();
  if (a->workspace && a->workspace_elems > ncnt) {
    g->ws = a->workspace;
    g->ws_elems = a->workspace_elems - ncnt;
    g->cnt = reinterpret_cast<int*>(a->workspace + g->ws_elems);
  }
  return true;
}

extern "C" {

ttt_status ttt_op_gemm(const ttt_gemm_args* args, ttt_stream stream) {
  GemmDesc g;
  if (!to_desc(args, &g)) return bad(TTT_ERR_BAD_ARG, "bad ttt_gemm_args");
  if ((g.epi == EPI_GELU && !g.out2) || ((g.epi == EPI_RESID || g.epi == EPI_SWIGLU || g.epi == EPI_DGELU) && !g.aux) ||
      (g.epi == EPI_DW && !g.partials))
    return bad(TTT_ERR_BAD_ARG, "epilogue operand missing");
  if (g.impl == TTT_GEMM_TENSOR && !gemm_tc_supported(g))
    return bad(TTT_ERR_UNSUPPORTED, "shape/alignment not supported by the tensor-core GEMM");
  if (g.cnt)   // this call's counters start at zero, in stream order
    TTT_CUDA(cudaMemsetAsync(g.cnt, 0, (size_t)gemm_tc_max_split_tiles() * sizeof(int), (cudaStream_t)stream));
  return gemm(g, (cudaStream_t)stream);
}

int ttt_op_gemm_partial_tiles(const ttt_gemm_args* args) {
  GemmDesc g;
  if (!to_desc(args, &g)) return -1;
  return gemm_partial_tiles(g);
}

ttt_status ttt_op_cross_entropy(int dtype, int M, int V, void* logits, const int32_t* targets, float scale,
                                int grad, float* losses, ttt_stream stream) {
  if (M < 0 || V < 1 || !logits || !targets || (dtype != TTT_DTYPE_FP32 && dtype != TTT_DTYPE_BF16))
    return bad(TTT_ERR_BAD_ARG, "bad cross-entropy arguments");
  if (M == 0) return TTT_OK;
  // One "sequence" of M rows whose target of row j is targets[j]: the kernel
  // reads tok[tok_off + j + 1], so tok_off = -1.
  TokView tv;
  tv.tok = targets;
  tv.tok_ld = 0;
  tv.tok_off = -1;
  tv.rows = M;
  tv.n_valid = M;
  tv.vocab = V;
  void* err = nullptr;
  TTT_CUDA(symbol_address((const void*)&g_ce_status, &err));
  tv.err = static_cast<int*>(err);
  return launch_ce(dtype, 1, tv, V, logits, V, scale, nullptr, grad != 0, losses, 0, 0, nullptr,
                   (cudaStream_t)stream);
}

ttt_status ttt_op_rmsnorm_forward(int dtype, int M, int d, const float* x, float eps, void* y, float* rstd,
                                  ttt_stream stream) {
  if (M < 0 || d < 1 || !x || !y || !rstd) return bad(TTT_ERR_BAD_ARG, "bad rmsnorm arguments");
  return launch_rmsnorm_fwd(dtype, M, d, x, eps, y, 0, rstd, nullptr, nullptr, (cudaStream_t)stream);
}

ttt_status ttt_op_rmsnorm_backward(int dtype, int M, int d, const float* x, const float* rstd, const float* dy,
                                   float* dx, void* dx_op, ttt_stream stream) {
  if (M < 0 || d < 1 || !x || !rstd || !dy || !dx) return bad(TTT_ERR_BAD_ARG, "bad rmsnorm arguments");
  return launch_rmsnorm_bwd(dtype, M, d, x, rstd, dy, dx, dx_op, 0, (cudaStream_t)stream);
}

ttt_status ttt_op_sliding_window_attention(int dtype, int B, int rows, int heads, int head_dim, int window,
                                           const void* qkv, int pad, long long L, void* out, ttt_stream stream) {
  if (B < 0 || rows < 0 || heads < 1 || head_dim < 1 || window < 1 || pad < 0 || !qkv || !out)
    return bad(TTT_ERR_BAD_ARG, "bad sliding-window attention arguments");
  if (dtype != TTT_DTYPE_BF16 || !swa_fused_supported(ST_BF16, heads * head_dim, heads))
    return bad(TTT_ERR_UNSUPPORTED, "the fused attention runs bf16 with head width 64 or 128");
  if (L < (long long)pad + ceil_div(rows, 128) * 128LL) return bad(TTT_ERR_BAD_SHAPE, "L too small for pad + rows");
  void* err = nullptr;
  TTT_CUDA(symbol_address((const void*)&g_attn_status, &err));
  cudaStream_t st = (cudaStream_t)stream;
  TTT_CUDA(cudaMemsetAsync(err, 0, sizeof(int), st));
  TTT_TRY(launch_swa_fused(B, rows, heads, head_dim, window, qkv, pad, L, out, static_cast<int*>(err), st));
  int flag = 0;
  TTT_CUDA(cudaMemcpyAsync(&flag, err, sizeof(int), cudaMemcpyDeviceToHost, st));
  TTT_CUDA(cudaStreamSynchronize(st));
  if (flag) return bad(TTT_ERR_TIMEOUT, "a fused attention wait timed out");
  return TTT_OK;
}

size_t ttt_clip_sgd_workspace_size(int nslots, int B, long long n) {
  if (nslots < 1 || B < 1 || n < 1) return 0;
  return clip_sgd_scratch_floats(nslots, B, n) * sizeof(float);
}

ttt_status ttt_clip_sgd(int dtype, int nslots, int B, long long n, float* W32, void* Wop, const float* dW, float eta,
                        float clip, float* norm_out, float* scale_out, void* workspace, size_t workspace_bytes,
                        ttt_stream stream) {
  if (nslots < 1 || B < 1 || n < 1 || !W32 || !Wop || !dW || !workspace || clip < 0.0f ||
      (dtype != TTT_DTYPE_FP32 && dtype != TTT_DTYPE_BF16))
    return bad(TTT_ERR_BAD_ARG, "bad clip_sgd arguments");
  if (workspace_bytes < ttt_clip_sgd_workspace_size(nslots, B, n))
    return bad(TTT_ERR_BAD_SHAPE, "workspace smaller than ttt_clip_sgd_workspace_size()");
  cudaStream_t st = (cudaStream_t)stream;
  float* scratch = static_cast<float*>(workspace);
  TTT_TRY(launch_clip_sgd(dtype, nslots, B, n, W32, Wop, dW, eta, clip, norm_out, scale_out, scratch, st));
  int flag = 0;
  const size_t flag_off = clip_sgd_scratch_floats(nslots, B, n) - 1;
  TTT_CUDA(cudaMemcpyAsync(&flag, scratch + flag_off, 4, cudaMemcpyDeviceToHost, st));
  TTT_CUDA(cudaStreamSynchronize(st));
  if (flag) return bad(TTT_ERR_NONFINITE, "non-finite gradient norm: that sequence was not updated");
  return TTT_OK;
}

}  // extern "C"
