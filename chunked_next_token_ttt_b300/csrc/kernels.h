// Internal launchers of the non-GEMM kernels of libttt.
#pragma once

#include "common.cuh"

namespace ttt {

// Row m = s * rows + j of a per-sequence row block reads token
// tok[s * tok_ld + tok_off + j]; its target is the next token of the same
// sequence, tok[s * tok_ld + tok_off + j + 1], for j < n_valid, and none after.
struct TokView {
  const int32_t* tok = nullptr;
  long long tok_ld = 0;
  long long tok_off = 0;
  int rows = 0;
  int n_valid = 0;
  int vocab = 0;          // tokens outside [0, vocab) are replaced by 0 and
  int* err = nullptr;     // raise bit 2 of *err (no out-of-range access)
};

// Storage codes (Storage in common.cuh): ST_F32, ST_BF16, ST_SPLIT.  `lo` is
// the element offset of an op-typed pointer's lo plane (ST_SPLIT only).

// h32[m, :] = E[x_m, :] (float), hop[m, :] = same in the operand storage.  E is
// bf16 for ST_BF16 and float otherwise.
ttt_status launch_embed(int stg, int B, const TokView& tv, const void* E, int d, float* h32,
                        void* hop, long long hop_lo, cudaStream_t st);

// y = x * rstd (operand type), rstd = 1/sqrt(mean(x^2) + eps).  With tv
// non-null it also writes tgt[m], the target token of row m (-1 past n_valid).
ttt_status launch_rmsnorm_fwd(int stg, int M, int d, const float* x, float eps, void* y, long long y_lo,
                              float* rstd, const TokView* tv, int32_t* tgt, cudaStream_t st);

// dx = rstd * (dy - xhat * mean(xhat * dy)), xhat = x * rstd; dx32 and its
// operand-type copy dxop (may be null).
ttt_status launch_rmsnorm_bwd(int stg, int M, int d, const float* x, const float* rstd,
                              const float* dy, float* dx32, void* dxop, long long dx_lo, cudaStream_t st);

// Row-wise cross-entropy of logits [B*rows, V] (leading dim ldl elements).
// For valid rows: loss -> losses[s * loss_ld + loss_off + j] (if losses != null)
// and row_loss[m] (if != null); when `grad` the row is overwritten in place by
// dlogits = (softmax - onehot(target)) * scale (rscale[m] per row when rscale
// is non-null).  Invalid rows get dlogits 0.
// ST_F32 / ST_BF16: logits and dlogits in that type.  ST_SPLIT: logits are
// float (ldl floats per row); dlogits are written inside each row's own bytes
// as a split pair, hi plane at bf16 offset 0 and lo plane at bf16 offset V of
// the row (a bf16 matrix with leading dim 2*ldl and lo offset V); V must fit
// the kernel's shared-memory row buffer (ce_split_max_vocab()).
ttt_status launch_ce(int stg, int B, const TokView& tv, int V, void* logits, long long ldl,
                     float scale, const float* rscale, bool grad, float* losses, long long loss_ld,
                     long long loss_off, float* row_loss, cudaStream_t st);
int ce_split_max_vocab();

// Fused cross-entropy after the EPI_LOGITS head GEMM (bf16 operands):
// lse[m] from the nt per-column-tile states part[m * ld + t]; the target logit
// y[m] . U[tgt[m]] (y [M, d], U [V, d] bf16); for valid rows the loss lse - logit
// goes to losses / row_loss as in launch_ce.
ttt_status launch_lse_combine(int B, const TokView& tv, const float2* part, long long ld, int nt, const void* y,
                              const void* U, int d, const int32_t* tgt, float* lse, float* losses,
                              long long loss_ld, long long loss_off, float* row_loss, cudaStream_t st);
// In place over bf16 logits [M, V] (leading dim V, V % 8 == 0, 16-byte aligned):
// dlogits = (exp(x - lse[m]) - [v == tgt[m]]) * scale; rows with tgt[m] < 0 get 0.
ttt_status launch_dlogits(int M, int V, void* logits, const float* lse, const int32_t* tgt, float scale,
                          const float* rscale, cudaStream_t st);
// Source Masking: per-row loss scales of one chunk, rscale[s * rows + j] =
// m / max(1, count of set mask entries of sequence s in the chunk), m =
// (mask[s * mask_ld + off + j] != 0).
ttt_status launch_chunk_row_scale(int B, int rows, const uint8_t* mask, long long mask_ld, long long off,
                                  float* rscale, cudaStream_t st);

// Where the dW GEMMs left their per-tile sums of squares: for GEMM k, the
// partials of sequence s are partials[off[k] + s * tiles[k] + t], t < tiles[k].
struct PartialSlots {
  int n = 0;
  long long off[16];
  int tiles[16];
};
// W32 -= eta * scale[s] * dW over the arena [slot][B][n]; Wop = cast(W32).
ttt_status launch_sgd_update(int stg, int nslots, int B, long long n, float* W32, void* Wop, long long wop_lo,
                             const float* dW, const float* scale, float eta, cudaStream_t st);

// Per sequence s: norm = sqrt(sum of its dW partials), the clip scale
// s_s = min(1, clip/(norm+1e-6)) (1 when clip == 0), then W32 -= eta * s_s * dW over the arena
// [slot][B][n] and Wop = cast(W32), in one launch.  scale_out / norm_out [B]
// (may be null) receive s_s and the norm; a non-finite norm skips that
// sequence's update and raises bit 1 of *flag.
ttt_status launch_clip_sgd_update(int stg, int nslots, int B, long long n, float* W32, void* Wop, long long wop_lo,
                                  const void* dW, const PartialSlots& ps, const float* partials, float clip,
                                  float eta, float* scale_out, float* norm_out, int* flag, cudaStream_t st);

// W32[slot][s] = W0[slot] for every s; Wop = cast.
ttt_status launch_broadcast_w0(int stg, int nslots, int B, long long n, const float* W0,
                               float* W32, void* Wop, long long wop_lo, cudaStream_t st);

// out[i] = cast(in[i]) for n floats.
ttt_status launch_cast(int stg, long long n, const float* in, void* out, long long out_lo, cudaStream_t st);

// mean over the n_valid valid rows of each sequence's row_loss block.
ttt_status launch_seq_mean(int B, int rows, int n_valid, const float* row_loss, float* mean,
                           cudaStream_t st);

// A = Lc - Lw; accept = (A >= 0).  Then per sequence: accept ? Wc <- W : W <- Wc
// over fp32 masters and operand copies.
// D = bf16(W32 - Wc32) over the fast-weight arena [nslots][B][n] (bf16 out).
ttt_status launch_delta_plane(int nslots, int B, long long n, const float* W32, const float* Wc32, void* D,
                              cudaStream_t st);
ttt_status launch_settle_apply(int stg, int nslots, int B, long long n, const float* Lc,
                               const float* Lw, float* A, uint8_t* accept, float* W32, void* Wop,
                               float* Wc32, void* Wcop, long long op_lo, cudaStream_t st);

// p[m, :] = softmax(logits32[m, :]); lse[m] = logsumexp of the row (lse may be null).
// p = softmax(logits32) row by row and lse = its logsumexp, in two launches;
// part holds M * kSoftmaxMaxSlices slice states.
constexpr int kSoftmaxMaxSlices = 32;
ttt_status launch_softmax(int M, int V, const float* logits32, float* p, float* lse, float2* part, cudaStream_t st);
// loss[s] = lse[s] - logits32[s * V + x_s] with x_s = tok[s * tok_ld + off]
// (ids outside [0, V) read as 0 and raise bit 2 of *err).
ttt_status launch_next_token_loss(int B, int V, const float* logits32, const float* lse, const int32_t* tok,
                                  long long tok_ld, long long off, float* loss, int* err, cudaStream_t st);

// Per-token TTT (b = 1) for a network without frozen prefix and one GELU block
// whose matrices W1 (slot_w1) and W2 (slot_w2) are fast, fp32 storage: one CTA
// per sequence keeps W1, W2 and U in shared memory and runs tokens 0 .. T-1 of
// tok[s * tok_ld + .] (forward, loss, backward, clipped step; with mask non-null
// a token whose mask[s * mask_ld + t] is 0 is scored without a step), writing
// losses[s * loss_ld + t] and, at the end, the fp32 masters and their copy.
bool token_steps_supported(int d, int f, int V);
ttt_status launch_token_steps(int B, const int32_t* tok, long long tok_ld, int T, const uint8_t* mask,
                              long long mask_ld, const float* E, const float* U,
                              float* W32, float* Wop, int slot_w1, int slot_w2, float* losses, long long loss_ld,
                              int d, int f, int V, float eps, float eta, float clip, int* err, cudaStream_t st);

// Decoding's next-token forward as one persistent cooperative kernel
// (decode_persist.cu): bf16 storage, GELU or SwiGLU blocks, no attention or
// extra frozen MLPs, B <= 8.  Weight pointers are bf16 [N][K] row-major (the
// GEMM's K-major B operand); the per-sequence fast weights of sequence s sit
// at the given pointer + s * n.
constexpr int kDecodeMaxBlocks = 48;
struct DecodeNet {
  int B = 0, d = 0, f = 0, V = 0, swiglu = 0, n_pre = 0, n_fast = 0;
  float eps = 0.0f;
  const int32_t* tok = nullptr;               // [B] the new inputs
  const void* E = nullptr;                     // [V][d]
  const void* pre[kDecodeMaxBlocks][3] = {};   // frozen prefix blocks: up (gate), up (SwiGLU), down
  const void* ffrozen[kDecodeMaxBlocks][2] = {};   // SwiGLU fast blocks: frozen gate and up
  const void* fup[kDecodeMaxBlocks] = {};      // GELU fast blocks: W1 of sequence 0
  const void* fdown[kDecodeMaxBlocks] = {};    // fast down projection of sequence 0
  long long n = 0;                             // per-sequence stride of the fast weights
  const void* U = nullptr;                     // [V][d]
  float* x32 = nullptr;                        // [2][B][d] residual stream, by block parity
  float* px = nullptr;                         // [2][8][B][d] down-projection partial sums over K segments
  void* act = nullptr;                         // [B][f] bf16 activations
  float* logits = nullptr;                     // [B][V] out
  float* p = nullptr;                          // [B][V] out: softmax
  float* lse = nullptr;                        // [B] out
  float2* part = nullptr;                      // [grid][B] per-CTA softmax states
  unsigned* bar = nullptr;                     // [4] grid barrier state (zeroed before each launch)
  int* err = nullptr;
};
// The grid the launch uses (one CTA per SM) and whether this GPU can hold it;
// 0 when the shapes or the GPU do not allow the persistent kernel.
int decode_persist_grid(int B, int d, int f);
// bar_clear: the barrier state (net.bar, 4 words) is still to be zeroed; false
// when the caller already did in stream order.
ttt_status launch_decode_persist(const DecodeNet& net, int grid, bool bar_clear, cudaStream_t st);

// Sliding-window attention of the frozen blocks (attention.cu): for B
// sequences of `rows` positions, qkv [B][rows][3d] fp32 (Q | K | V of each
// row, d = H * dh), out [B][rows][d] in operand type: per head,
// softmax(Q K^T / sqrt(dh)) V over keys t - window < s <= t.
bool swa_supported(int d, int heads);
// The tensor-core path of the same attention materialises, per head, the
// scores of query blocks of kSwaTcRows rows against their nw-key windows
// (two batched GEMMs around this masked row softmax); see the engine's
// prefix pass for the padded row layout.
constexpr int kSwaTcRows = 128;
// Fused sliding-window attention on the tensor cores (bf16 storage, head width
// 64 or 128): per (128-query block, head, sequence) one CTA reads Q, K and V
// from the padded projection rows qkvp [B][L][3d] (position p of a sequence
// at row pad + p) and writes the heads' output into out [B][L][d] at the
// same rows; scores and probabilities stay on chip.  Bounded-wait timeouts
// set bits of *err.
bool swa_fused_supported(int stg, int d, int heads);
ttt_status launch_swa_fused(int B, int rows, int H, int dh, int window, const void* qkvp, int pad, long long L,
                            void* out, int* err, cudaStream_t st);
ttt_status launch_band_softmax(int stg, long long nbatch, int nw, int nqb, int j0, int pad, int rows, int window,
                               float scale, const float* Sc, void* P, long long p_lo, cudaStream_t st);
ttt_status launch_swa(int stg, int B, int rows, int H, int dh, int window, const float* qkv, void* out,
                      long long out_lo, cudaStream_t st);

// Decoding with attention (attention.cu).  kv_fill: the K and V rows of the
// last min(R, window) positions of a whole-sequence pass (src rows
// s * seq_rows + row0 + pos, 3d wide, operand type of stg) into the fp32 cache
// ck / cv [B][window][d] at slot pos % window.  swa_decode: for the position
// *pos of every sequence, appends the K | V of qkv [B][3d] (fp32) to the
// cache and writes the heads' output [B][d] in operand type; needs
// dh <= 128 (its shared memory, swa_decode_smem_bytes, does not grow with
// the window).
ttt_status launch_kv_fill(int stg, int B, int R, int window, int d, const void* src, long long src_lo,
                          long long seq_rows, long long row0, float* ck, float* cv, cudaStream_t st);
size_t swa_decode_smem_bytes(int window, int dh);
// The decoded position on the device: *p = v, and *p += 1 (one thread each).
ttt_status launch_pos_set(int* p, int v, cudaStream_t st);
ttt_status launch_pos_add(int* p, cudaStream_t st);
// work: swa_decode_work_floats(B, H) floats; cnt: B * H ints, zero before the
// first launch (every launch leaves them at zero).
ttt_status launch_swa_decode(int stg, int B, int H, int dh, int window, const int* pos, const float* qkv, float* ck,
                             float* cv, float* work, int* cnt, void* out, long long out_lo, cudaStream_t st);
size_t swa_decode_work_floats(int B, int H);

// Shift the pending decode buffer: tok[s][0] = tok[s][b].
ttt_status launch_pending_shift(int B, int b, int32_t* pend, cudaStream_t st);
// A decoding step's inputs: *flag = 0, bar[0..3] = 0 when bar is not null,
// pend[s * ld + col] = x_dev[s] = x_new[s] (device x_new), and when loss is
// not null loss[s] = lse[s] - logits32[s][x_new[s]] (a token outside [0, V)
// sets bit 2 of *flag and scores token 0).  One block: B at most a few hundred.
ttt_status launch_decode_inputs(int B, int ld, int col, const int32_t* x_new, int32_t* pend, int32_t* x_dev,
                                int* flag, unsigned* bar, int V, const float* logits32, const float* lse,
                                float* loss, cudaStream_t st);

}  // namespace ttt
