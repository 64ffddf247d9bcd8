/*
 * libttt — chunked next-token test-time training (TTT) on one B300 (sm_103a).
 *
 * The library runs the TTT prefill inner loop: for each chunk of b tokens it
 * runs the fast-weight MLP blocks forward, then the final RMSNorm and the LM
 * head, takes the next-token cross-entropy, backpropagates to the fast weights
 * only, and applies one clipped SGD step to fp32 master fast weights.  It
 * returns the prequential per-token losses, the final fast weights W_T and
 * p_{T+1}; optionally it gates the updates with the Settlement rule.
 *
 * Definitions this API follows:
 *  - "End-to-End Test-Time Training for Long Context" (paper review page):
 *    Method 1, eq. (1) per-token loss l_t(W) = CE(f(x_{t-1}; W), x_t) and
 *    eq. (2) online update; Method 2, eq. (3) prequential loss; Method 3,
 *    eq. (5) mini-batch update W_i = W_{i-1} - eta (1/b) sum grad l_t(W_{i-1})
 *    and eq. (6); output p_{T+1} = f(x_T; W_{T/b}); 3.1 "TTT only the MLP
 *    layers" / "only the last blocks"; 3.2 "Decoding Multiple Tokens".
 *  - "In-Place Test-Time Training" (review page), Key Terms: the MLP final
 *    projection (down_proj) as the only fast weight.
 *  - "Self-Generated Feedback Destabilizes Test-Time Training" (summary page):
 *    one clipped gradient step per chunk on the last FFN modules; Settlement,
 *    A(delta; W, q) = L(q, W) - L(q, W + delta), commit only when A >= 0.
 *
 * Conventions (all arrays row-major, C order):
 *  - Tokens are int32 in [0, vocab).  Sequence s of a [B, T+1] token array is
 *    x_0 .. x_T with x_0 the BOS token.  Chunk i (1-based) uses inputs
 *    x_{(i-1)b} .. x_{ib-1} and targets x_{(i-1)b+1} .. x_{ib}.
 *  - Every sequence owns its fast weights (all start from the shared W_0).
 *  - Linear maps are stored [out, in]: GELU block W1 [d_ff, d], W2 [d, d_ff];
 *    SwiGLU block Wg [d_ff, d], Wu [d_ff, d], Wd [d, d_ff].  Embedding
 *    E [V, d]; LM head U [V, d] with logits = y U^T.
 *  - Block: h <- h + GELU(h W1^T) W2^T (exact erf GELU), or
 *    h <- h + (silu(h Wg^T) * (h Wu^T)) Wd^T.  No per-block norm, no bias.
 *    Final RMSNorm y = x / sqrt(mean(x^2) + rms_eps) with unit frozen gain.
 *  - Clip: s = min(1, clip / (||g||_2 + 1e-6)) with g all fast-matrix
 *    gradients of one sequence; clip = 0 disables it.  W <- W - eta * s * g.
 *
 * Memory: pointer arguments may be host or device memory unless a parameter
 * says otherwise; the library detects which (cudaPointerGetAttributes).
 * Device pointers are used in stream order on `stream`; host buffers are
 * copied inside the call, which then synchronises `stream` before it returns.
 * The library owns its copies of the weights, the fp32 masters, the committed
 * Settlement copy and all workspace; the caller owns every array it passes.
 * Nothing is freed across the boundary.
 *
 * Errors: every call returns a ttt_status; nothing aborts or throws.  A CUDA
 * error is reported as TTT_ERR_CUDA and its text is kept for
 * ttt_last_error().  Sticky CUDA errors are reported, not cleared.
 */
#ifndef TTT_H_
#define TTT_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
/* The same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st* ttt_stream;

typedef enum {
  TTT_OK = 0,
  TTT_ERR_BAD_ARG = 1,      /* NULL handle/pointer, negative size, bad enum */
  TTT_ERR_BAD_SHAPE = 2,    /* sizes inconsistent with the handle's dims    */
  TTT_ERR_OOM = 3,          /* device allocation failed                     */
  TTT_ERR_CUDA = 4,         /* a CUDA runtime/driver call failed            */
  TTT_ERR_NONFINITE = 5,    /* a non-finite gradient norm: that update was
                               skipped for that sequence, the rest ran      */
  TTT_ERR_TIMEOUT = 6,      /* a bounded device-side wait gave up; that
                               call's outputs are undefined, and the handle
                               clears its split-K counters before returning,
                               so later calls run normally                  */
  TTT_ERR_UNSUPPORTED = 7,  /* a valid request the library does not run    */
  TTT_ERR_STATE = 8         /* call out of order (e.g. decode before prefill) */
} ttt_status;

enum { TTT_BLOCK_GELU = 0, TTT_BLOCK_SWIGLU = 1 };
enum { TTT_DTYPE_FP32 = 0, TTT_DTYPE_BF16 = 1 };
/* fast_mask bits.  GELU: bit0 = W1, bit1 = W2.  SwiGLU: bit0 = Wg, bit1 = Wd,
 * bit2 = Wu.  The library runs GELU with mask 3 and SwiGLU with mask 2 (the
 * In-Place down projection); other masks return TTT_ERR_UNSUPPORTED. */
enum { TTT_FAST_W1 = 1, TTT_FAST_W2 = 2, TTT_FAST_WG = 1, TTT_FAST_WD = 2, TTT_FAST_WU = 4 };

typedef struct {
  int d;            /* model width                                            */
  int d_ff;         /* MLP hidden width                                       */
  int vocab;        /* V                                                      */
  int n_prefix;     /* frozen MLP blocks after the embedding (>= 0)           */
  int n_fast;       /* trailing blocks holding fast weights (>= 1)            */
  int block_kind;   /* TTT_BLOCK_GELU or TTT_BLOCK_SWIGLU                     */
  int fast_mask;    /* which matrices of a fast block are fast                */
  int dtype;        /* TTT_DTYPE_FP32: fp32-accurate arithmetic throughout;
                       TTT_DTYPE_BF16: bf16 weights/activations, fp32
                       accumulation and fp32 master fast weights             */
  float rms_eps;    /* RMSNorm epsilon inside the square root (1e-6)          */
  int static_mlp;   /* 1: every fast block also holds a frozen MLP of the same
                       kind and widths that runs before its fast MLP
                       ("End-to-End TTT" review, 3.1, Two MLP layers per
                       block): h += MLP_s(h); h += MLP_f(h).  GELU blocks
                       only; 0 = off                                          */
  int attn_heads;   /* > 0: every frozen prefix block runs sliding-window
                       multi-head attention before its MLP ("End-to-End TTT"
                       review, Method: the sliding-window attention fix of
                       the bigram defect): h += Attn(h), keys t-k < s <= t,
                       scale 1/sqrt(d/attn_heads), no positional encoding.
                       Needs n_prefix >= 1, d % attn_heads == 0,
                       d/attn_heads <= 128.  Prefill runs the prefix of
                       x_0..x_T as one pass; decoding continues the
                       positions through a K/V cache of the last
                       attn_window inputs (needs a prefill after create,
                       ttt_reset or ttt_set_state: STATE otherwise; windows
                       above ~57K positions return UNSUPPORTED there);
                       Settlement returns UNSUPPORTED.  0 = no attention     */
  int attn_window;  /* k >= 1 when attn_heads > 0                             */
} ttt_dims;

typedef struct {
  float eta;          /* SGD step size                                        */
  float clip;         /* global-norm clip per sequence; 0 = off               */
  int chunk;          /* b, tokens per TTT mini-batch (>= 1)                  */
  int settle_every;   /* chunks between Settlement events in prefill; 0 = off */
  int max_batch;      /* B, sequences; fixed for the handle's life             */
  int settle_len;     /* Lq, tokens per held-out chunk (0 when unused)        */
  int reset_every;    /* periodic reset ("Self-Generated Feedback Destabilizes
                         TTT" summary, limits paragraph: the 8-chunk reset):
                         after every reset_every-th chunk update, prefill and
                         decoding counted together, the fast weights of every
                         sequence return to W_0.  0 = off; > 0 requires
                         settle_every == 0 (the two are alternatives)         */
} ttt_hparams;

/* Initial weights, float32 values (host or device).  The library copies them
 * and rounds to the storage type (exact when the values are representable).
 * prefix: n_prefix * n_mats pointers, blocks in order, matrices in the order
 * (W1, W2) or (Wg, Wu, Wd).  fast: n_fast * n_mats pointers, the same order,
 * giving W_0 of every matrix of the fast blocks (frozen ones included). */
typedef struct {
  const float* E;
  const float* U;
  const float* const* prefix;
  const float* const* fast;
  const float* const* statics;   /* static_mlp: n_fast * n_mats pointers, the
                                    frozen MLP of each fast block (NULL otherwise) */
  const float* const* attn;      /* attn_heads > 0: n_prefix * 4 pointers, (Wq, Wk,
                                    Wv, Wo) of each prefix block, each [d, d]
                                    stored [out, in] (NULL otherwise)         */
} ttt_weights;

typedef struct ttt_handle ttt_handle;

/* Execution options of a handle.  A zero-filled struct (or NULL) selects the
 * library's defaults, which are what ttt_create uses; nothing outside this
 * struct (no environment variable, no global) changes how a handle runs.  The
 * non-default settings exist for tests and measurements: each selects another
 * path to the same results, or limits the GPU the handle uses. */
typedef struct {
  int no_pdl;          /* 1: launch kernels without programmatic dependent launch */
  int no_decode_graph; /* 1: ttt_decode_step launches its next-token forward kernel
                          by kernel instead of replaying one captured CUDA graph */
  int fp32_simt;       /* 1: TTT_DTYPE_FP32 handles keep plain fp32 operands and
                          SIMT GEMMs instead of bf16x3 tensor-core products   */
  int hoist_chunks;    /* > 0: at most this many chunks share one pass of the
                          frozen prefix (0: as many as a 4 GiB buffer holds, up
                          to 64)                                              */
  int no_token_kernel; /* 1: chunk = 1 runs the general chunk step instead of the
                          persistent per-token kernel                          */
  int max_ctas;        /* > 0: at most this many CTAs in a tensor-core GEMM's
                          persistent grid (0: one per SM)                      */
  int no_dw_stream;    /* 1: the weight-gradient GEMMs run in stream order with
                          the input-gradient chain instead of on the handle's
                          second stream beside it                             */
  int attn_unfused;    /* 1: bf16 sliding-window attention runs as score GEMM,
                          windowed softmax and P V GEMM per head instead of the
                          fused kernel that keeps scores on chip             */
  int no_decode_persist; /* 1: ttt_decode_step's next-token forward never runs as
                          the one persistent cooperative kernel (bf16 storage,
                          no attention or extra frozen MLPs, B <= 8), but as
                          the captured graph (or launch by launch)           */
} ttt_options;

/* Validate dims/hparams, allocate every device buffer the handle needs for
 * B = max_batch sequences and upload the weights.  On success *out owns all
 * of it until ttt_destroy.  Errors: BAD_ARG, UNSUPPORTED, OOM, CUDA. */
ttt_status ttt_create(const ttt_dims* dims, const ttt_hparams* hp,
                      const ttt_weights* w, ttt_handle** out);
/* ttt_create with execution options (NULL = defaults).  Errors: as ttt_create,
 * and BAD_ARG for a negative option. */
ttt_status ttt_create_ex(const ttt_dims* dims, const ttt_hparams* hp,
                         const ttt_weights* w, const ttt_options* opt, ttt_handle** out);

/* Free everything the handle owns.  NULL is accepted. */
ttt_status ttt_destroy(ttt_handle* h);

/* Prefill ("End-to-End TTT" review, Method 3, eqs. (5)-(6)).  Resets the fast
 * weights of every sequence to W_0, then for i = 1 .. T/b runs one chunk step
 * for all B sequences and writes losses[s, (i-1)b + j] = l_t(W_{i-1}).
 *   tokens   [B, T+1] int32 (host or device).
 *   losses   [B, T] float32 out (host or device).
 *   p_next   [B, V] float32 out or NULL: softmax(f(x_T; W_final)).
 *   settle_q [E, B, Lq] int32 or NULL, E = (T/b) / settle_every held-out
 *            chunks, one per Settlement event (required when settle_every>0).
 *   accept   [E, B] uint8 out or NULL; A [E, B] float32 out or NULL.
 * If b does not divide T the trailing T mod b losses are scored with the last
 * weights and those tokens wait in the pending buffer for decoding.
 * Errors: BAD_ARG, BAD_SHAPE (B != max_batch, T < 1, Lq != settle_len),
 * NONFINITE (some update skipped), CUDA. */
ttt_status ttt_prefill(ttt_handle* h, const int32_t* tokens, int B, int T,
                       float* losses, float* p_next,
                       const int32_t* settle_q, int Lq,
                       uint8_t* accept, float* A, ttt_stream stream);

/* ttt_prefill with Source Masking ("Self-Generated Feedback Destabilizes TTT"
 * summary, Settlement paragraph: Source Masking, which keeps the tokens a
 * source label marks as generated out of the update).  loss_mask [B, T] uint8
 * (host or device; NULL = all ones): target x_{t+1} of sequence s enters the
 * update iff loss_mask[s, t] != 0.  Every token is still scored into losses;
 * a chunk's TTT loss is the mean over its unmasked targets (1/n sum, n =
 * their count), and a chunk without any leaves the weights unchanged.  The
 * trailing T mod b targets and decoded tokens are not masked.  Other
 * arguments, results and errors as ttt_prefill. */
ttt_status ttt_prefill_masked(ttt_handle* h, const int32_t* tokens, const uint8_t* loss_mask, int B, int T,
                              float* losses, float* p_next, const int32_t* settle_q, int Lq, uint8_t* accept,
                              float* A, ttt_stream stream);

/* One decoded token per sequence ("End-to-End TTT" review, 3.2).  Appends the
 * pair (x_prev, x_new); when b pairs are pending it takes one clipped step on
 * them with the weights that scored them.
 *   x_new    [B] int32 (host or device).
 *   p_next   [B, V] float32 out: softmax(f(x_new; W)) after any step.
 *   loss     [B] float32 out or NULL: l of (x_prev -> x_new) before the step.
 * Errors: STATE (no prefill yet), BAD_ARG, NONFINITE, CUDA. */
ttt_status ttt_decode_step(ttt_handle* h, const int32_t* x_new, float* p_next,
                           float* loss, ttt_stream stream);

/* Settlement ("Self-Generated Feedback Destabilizes TTT", Settlement rule):
 * per sequence, A = L(q, W_c) - L(q, W) with W_c the committed weights and W
 * = W_c + delta the current ones; A >= 0 commits (W_c <- W), otherwise W
 * reverts to W_c bit-exactly.  L is the mean next-token CE over q.
 *   q [B, Lq] int32 (Lq == settle_len); accept [B] uint8 out; A [B] float out.
 * Errors: BAD_ARG, BAD_SHAPE, STATE, CUDA. */
ttt_status ttt_settle(ttt_handle* h, const int32_t* q, int Lq, uint8_t* accept,
                      float* A, ttt_stream stream);

/* Copy the fp32 master of one fast matrix of sequence `seq` into dst
 * ([out, in] float32, host or device).  block in [0, n_fast); mat indexes
 * the block's matrices in the order (W1, W2) or (Wg, Wu, Wd).
 * Errors: BAD_ARG, CUDA. */
ttt_status ttt_get_fast_weights(ttt_handle* h, int seq, int block, int mat, float* dst,
                                ttt_stream stream);

/* Restore W_0 for every sequence, clear the committed copy and the pending
 * decode buffer.  Errors: BAD_ARG, CUDA. */
ttt_status ttt_reset(ttt_handle* h, ttt_stream stream);

/* Checkpoint / resume: the fp32 fast weights, the committed Settlement copy,
 * the pending decode tokens and the step counters, as one opaque byte blob
 * (host memory).  ttt_state_size gives its size; ttt_get_state fills it;
 * ttt_set_state restores a blob taken from a handle with the same dims and
 * hparams.  Errors: BAD_ARG, BAD_SHAPE (size or dims mismatch), CUDA. */
ttt_status ttt_state_size(ttt_handle* h, size_t* bytes);
ttt_status ttt_get_state(ttt_handle* h, void* dst, size_t bytes, ttt_stream stream);
ttt_status ttt_set_state(ttt_handle* h, const void* src, size_t bytes, ttt_stream stream);

/* Per-kernel timing of prefill, for roofline accounting.  While enabled,
 * every launch of the named kernel class inside ttt_prefill is bracketed by
 * CUDA events on the launching stream; ttt_profile_read returns the number of
 * launches and their summed device time in ms, then clears the record.
 * Kernel classes: see ttt_kernel_class_name.  Errors: BAD_ARG, CUDA. */
ttt_status ttt_profile_enable(ttt_handle* h, int kernel_class);
ttt_status ttt_profile_read(ttt_handle* h, int* launches, double* total_ms);
const char* ttt_kernel_class_name(int kernel_class);
int ttt_kernel_class_count(void);

/* The arithmetic the handle's GEMMs use, fixed at create: 0 = plain fp32
 * (SIMT), 1 = bf16 operands, 2 = bf16x3 (fp32 values as bf16 hi/lo pairs,
 * three tensor-core products per product), or -1 for a null handle. */
int ttt_operand_storage(ttt_handle* h);

/* Number of kernels the last ttt_prefill launched on the GPU. */
ttt_status ttt_last_launch_count(ttt_handle* h, long long* launches);

/* Launch-class log, for matching a profiler's launch list to kernel classes.
 * While enabled (on != 0; enabling clears it), every kernel the handle
 * launches appends its class (ttt_kernel_class_name) in launch order, one
 * entry per kernel, on the host.  ttt_launch_log_read copies up to cap entries
 * into out (host memory) and returns the number of entries logged (which may
 * exceed cap), or -1 for a null handle. */
ttt_status ttt_launch_log_enable(ttt_handle* h, int on);
int ttt_launch_log_read(ttt_handle* h, int8_t* out, int cap);

/* Static text for a status code, and the last error message of this thread. */
const char* ttt_status_string(ttt_status s);
const char* ttt_last_error(void);

#ifdef __cplusplus
}
#endif
#endif /* TTT_H_ */
