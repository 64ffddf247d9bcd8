// The libttt handle and the chunk-step sequencer (host side).
#pragma once

#include <vector>

#include "common.cuh"
#include "gemm.h"
#include "kernels.h"

// Kernel classes for launch accounting and per-class timing.
enum KClass {
  K_EMBED = 0, K_GEMM_PREFIX, K_GEMM_FAST_FWD, K_RMSNORM_FWD, K_GEMM_HEAD, K_CE, K_GEMM_HEAD_BWD,
  K_RMSNORM_BWD, K_GEMM_BWD_DX, K_GEMM_DW, K_NORM, K_SGD, K_SETTLE, K_OTHER, K_TOKEN, K_ATTN, K_COUNT
};

// An operand-storage buffer: its pointer and, for ST_SPLIT, the element
// offset of its lo plane (0 otherwise).
struct OpBuf {
  void* p = nullptr;
  long long lo = 0;
};

struct ttt_handle {
  ttt_dims dm{};
  ttt_hparams hp{};
  ttt_options opt{};      // execution options fixed at create (zero = defaults)
  int B = 0, b = 0, d = 0, f = 0, V = 0;
  int nm = 0;             // matrices per block (2 GELU, 3 SwiGLU)
  int nslots = 0;         // fast matrices in total (arena slots)
  long long n = 0;        // elements of one matrix (d * d_ff)
  int dtype = 0;          // TTT_DTYPE_* requested at create
  int stg = 0;            // operand storage (ST_F32, ST_BF16, ST_SPLIT)
  size_t esz = 4;         // bytes per element of one operand plane
  std::vector<int> slot_of;   // [n_fast * nm] -> arena slot or -1

  // frozen weights
  void* E = nullptr;                 // bf16 for ST_BF16, float otherwise
  OpBuf U;
  std::vector<OpBuf> prefix;         // [n_pre * nm]: the frozen blocks, then (static_mlp) fast block 0's static MLP
  int n_pre = 0;                     // frozen blocks the prefix pass runs
  std::vector<OpBuf> statics;        // [n_fast * nm] static MLP of fast block l >= 1 (static_mlp)
  // sliding-window attention of the frozen prefix blocks (attn_heads > 0)
  std::vector<OpBuf> attn_qkv;       // [n_prefix] (Wq | Wk | Wv) as one [3d, d] operand
  std::vector<OpBuf> attn_o;         // [n_prefix] Wo [d, d]
  // whole-sequence prefix pass of an attention prefill, B * (T + 1) rows, grown on demand
  size_t arows_cap = 0;
  float* ax32 = nullptr;
  OpBuf ax_op, ax_xop, ax_tmp_a, ax_a, att_o;
  float* ax_tmp_g = nullptr;
  float* qkv32 = nullptr;            // fp32 storage: Q | K | V rows for the tiled attention kernel
  // tensor-core attention (bf16 and split storage): padded Q | K | V rows, one
  // head's score blocks and probabilities, the heads' output in padded rows
  OpBuf qkvp, Pp, att_p;
  float* Sc = nullptr;
  size_t qkvp_cap = 0, sc_cap = 0, attp_cap = 0;
  // decoding with attention: the frozen blocks' K/V cache, the newest input's
  // position, the one-row prefix pass of the next-token forward, and the
  // prefix rows of the pending inputs (row j = input pend[j])
  float* kv = nullptr;               // [n_prefix][2][B][attn_window][d] fp32
  int* dec_pos = nullptr;
  bool attn_ctx = false;             // a prefill filled the cache and the pending rows
  float* dec_x32 = nullptr;
  float* dec_qkv = nullptr;          // [B][3d]
  float* dec_work = nullptr;         // decoding attention: per-split partial states
  int* dec_cnt = nullptr;            // and their arrival counts [B][heads] (zero between launches)
  float* dec_tmp_g = nullptr;
  OpBuf dec_op, dec_xop, dec_tmp_a, dec_a, dec_att;
  float* prow32 = nullptr;           // [B][b + 1][d]
  OpBuf prow_op, prow_a;
  std::vector<OpBuf> fastfrozen;     // [n_fast * nm], empty where fast

  // fast weights: arenas [slot][B][n]
  float* W0 = nullptr;     // [slot][n]
  float* W32 = nullptr;
  OpBuf Wop;
  float* Wc32 = nullptr;
  OpBuf Wcop;
  // bf16 storage with Settlement: bf16(W32 - Wc32), the candidate's offset from
  // the committed copy (Settlement scores W as Wcop + Wdel)
  OpBuf Wdel;
  void* dW = nullptr;      // [slot][B][n] gradients: bf16 for ST_BF16, fp32 otherwise
  size_t dw_esz = 4;       // bytes per dW element

  // chunk workspace for up to Mmax rows
  int Mmax = 0;
  float* x32 = nullptr;
  OpBuf xop;
  std::vector<OpBuf> hlvl, zst, ast;
  std::vector<OpBuf> szst, shin;     // static MLP of fast block l >= 1: its z stash and its output (fast MLP input)
  OpBuf tmp_a;
  float* tmp_g = nullptr;
  // hoisted prefix of a group of up to hoist_chunks chunks, rows [B][g * b]
  int hoist_chunks = 1;
  float* hx32 = nullptr;             // residual stream after the frozen prefix
  OpBuf hx_op;                       // its operand copy (input of fast block 0)
  OpBuf hx_xop, hx_tmp_a;            // prefix ping-pong and hidden-width temporaries
  float* hx_tmp_g = nullptr;         // SwiGLU gate temporary
  OpBuf ha;                          // SwiGLU fast block 0: silu(gate h) * (up h)
  // prefix output of a Settlement chunk q [B][Lq][.] (shared by its two forwards)
  float* qx32 = nullptr;
  OpBuf qx_op, qa;
  // inputs of fast block 0 in the last forward (backward reads them)
  OpBuf hin0, a0;
  long long hin0_s = 0, a0_s = 0;
  OpBuf y;
  float* rstd = nullptr;
  void* logits = nullptr;            // [Mmax, V]: float for ST_SPLIT, operand type otherwise
  float* row_loss = nullptr;
  float* rscale = nullptr;           // [Mmax] Source Masking: per-row loss scales of a chunk
  bool rscale_on = false;            // set only while a masked chunk step runs its forward
  uint8_t* mask_dev = nullptr; size_t mask_cap = 0;   // staging for a host mask
  float2* lse_part = nullptr;        // [Mmax][lse_ld] head-tile softmax states
  long long lse_ld = 0;
  float* lse = nullptr;              // [Mmax]
  int32_t* tgt = nullptr;            // [Mmax] target token per row, -1 = none
  float* dy32 = nullptr;
  float* dh32 = nullptr;
  OpBuf dhop;
  // weight gradients beside the input-gradient chain (GELU blocks without
  // static MLPs): the second stream, its fork/join events and the second
  // operand-copy buffer of dh
  cudaStream_t bstream = nullptr;
  std::vector<cudaEvent_t> bev;
  OpBuf dhop2;
  float* gemm_ws = nullptr;          // split-K partial products
  long long gemm_ws_elems = 0;
  int* split_cnt = nullptr;          // split-K arrival counters (zero between GEMMs)
  float* partials = nullptr;
  long long partial_cap = 0;
  ttt::PartialSlots pslots{};
  float* scale = nullptr;
  float* gnorm = nullptr;
  int* flag = nullptr;
  int* flag_host = nullptr;
  float* logits32 = nullptr;
  float* p_dev = nullptr;
  float* lse_next = nullptr;         // [B] logsumexp of logits32 (next-token softmax)
  float2* soft_part = nullptr;       // [B][kSoftmaxMaxSlices] slice states of that softmax
  bool next_valid = false;           // logits32 / lse_next score the next decoded token
  // decoding's next-token forward, captured once as a CUDA graph
  cudaStream_t gstream = nullptr;
  cudaEvent_t gev[2] = {nullptr, nullptr};
  cudaGraphExec_t dec_exec = nullptr;
  long long dec_kernels = 0;
  // or as one persistent cooperative kernel (dp_grid: -1 not yet decided, 0 not used)
  int dp_grid = -1;
  ttt::DecodeNet dp_net;
  float* dp_x32 = nullptr;
  float* dp_px = nullptr;
  void* dp_act = nullptr;
  float2* dp_part = nullptr;
  unsigned* dp_bar = nullptr;
  float* Lc = nullptr;
  float* Lw = nullptr;

  // staging for host-side inputs and outputs
  int32_t* tok_dev = nullptr; size_t tok_cap = 0;
  float* loss_dev = nullptr; size_t loss_cap = 0;
  int32_t* q_dev = nullptr; size_t q_cap = 0;
  float* A_dev = nullptr; size_t A_cap = 0;
  uint8_t* acc_dev = nullptr; size_t acc_cap = 0;
  int32_t* x_dev = nullptr;

  // decoding
  int32_t* pend = nullptr;     // [B][b+1]
  int pend_count = 0;
  bool has_context = false;
  long long chunks_done = 0;

  // accounting
  long long launches = 0;
  int prof_class = -1;
  std::vector<cudaEvent_t> ev;
  int ev_used = 0;
  int prof_launches = 0;
  bool log_on = false;
  std::vector<int8_t> launch_log;   // kernel class of every launch, in order

  std::vector<void*> allocs;
};
