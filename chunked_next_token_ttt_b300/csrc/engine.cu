// libttt C ABI: handle life cycle and the stream-ordered chunk sequencer.
//
// One chunk step ("End-to-End Test-Time Training for Long Context" review,
// Method 3, eq. (5)) for all B sequences at once:
//   embed + frozen prefix -> fast blocks forward (stash z, a, h) -> RMSNorm
//   -> LM head -> fused CE (losses, dlogits in place) -> dy = dlogits U
//   -> RMSNorm backward -> fast blocks backward (dW per sequence, dh)
//   -> per-sequence global norm -> clip + SGD on the fp32 masters.
// Every step runs in stream order on the caller's stream; the host only
// synchronises at the end of a call that returns host data or a status flag.
#include <cstring>
#include <mutex>
#include <string>

#include "engine.h"

namespace ttt {

static thread_local std::string g_last_error;

void set_error(const std::string& msg) { g_last_error = msg; }

ttt_status cuda_fail(cudaError_t e, const char* what, const char* file, int line) {
  char buf[512];
  snprintf(buf, sizeof buf, "%s: %s (%s:%d)", what, cudaGetErrorString(e), file, line);
  set_error(buf);
  return e == cudaErrorMemoryAllocation ? TTT_ERR_OOM : TTT_ERR_CUDA;
}

static ttt_status fail(ttt_status s, const std::string& msg) {
  set_error(msg);
  return s;
}

static bool is_device_ptr(const void* p) {
  if (!p) return false;
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged;
}

template <typename T>
static ttt_status dalloc(ttt_handle* h, T** p, size_t bytes) {
  *p = nullptr;
  if (bytes == 0) return TTT_OK;
  void* q = nullptr;
  cudaError_t e = cudaMalloc(&q, bytes);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(TTT_ERR_OOM, "cudaMalloc of " + std::to_string(bytes) + " bytes failed");
  }
  h->allocs.push_back(q);
  *p = static_cast<T*>(q);
  return TTT_OK;
}

// Runs one launcher as kernel class `cls`, bracketing it with events when that
// class is being profiled.
template <class F>
static ttt_status run(ttt_handle* h, int cls, cudaStream_t st, int nkernels, F&& f) {
  const bool prof = h->prof_class == cls;
  if (prof && h->ev_used + 2 > (int)h->ev.size()) {
    // grow the event pool: every profiled launch of a long call keeps its pair
    const size_t old = h->ev.size();
    h->ev.resize(old + 4096);
    for (size_t i = old; i < h->ev.size(); ++i) TTT_CUDA(cudaEventCreate(&h->ev[i]));
  }
  if (prof) TTT_CUDA(cudaEventRecord(h->ev[h->ev_used], st));
  TTT_TRY(f());
  if (prof) {
    TTT_CUDA(cudaEventRecord(h->ev[h->ev_used + 1], st));
    h->ev_used += 2;
    h->prof_launches += 1;
  }
  h->launches += nkernels;
  if (h->log_on)
    for (int k = 0; k < nkernels; ++k) h->launch_log.push_back((int8_t)cls);
  return TTT_OK;
}

// Slice of an operand buffer starting `elems` elements in (same lo plane offset).
static OpBuf op_at(const ttt_handle* h, const OpBuf& b, long long elems) {
  OpBuf r;
  r.p = static_cast<char*>(b.p) + elems * (long long)h->esz;
  r.lo = b.lo;
  return r;
}

static int gemm_count(const GemmDesc& g) { return gemm_launches(g); }

static ttt_status rungemm(ttt_handle* h, int cls, const GemmDesc& g_in, cudaStream_t st) {
  GemmDesc g = g_in;
  g.err = h->flag;
  g.dtype = h->stg;
  g.ws = h->gemm_ws;
  g.ws_elems = h->gemm_ws_elems;
  g.cnt = h->split_cnt;
  g.max_ctas = h->opt.max_ctas;
  return run(h, cls, st, gemm_count(g), [&] { return gemm(g, st); });
}

// Operand setters for a GemmDesc from OpBufs.
static void setA(GemmDesc& g, const OpBuf& b, long long ld, long long s = 0) { g.A = b.p; g.loA = b.lo; g.lda = ld; g.sA = s; }
static void setB(GemmDesc& g, const OpBuf& b, long long ld, long long s = 0) { g.B = b.p; g.loB = b.lo; g.ldb = ld; g.sB = s; }
static void setOut(GemmDesc& g, const OpBuf& b, long long ld, long long s = 0) { g.out = b.p; g.loO = b.lo; g.ldo = ld; g.sO = s; }
static void setOut2(GemmDesc& g, const OpBuf& b, long long ld, long long s = 0) { g.out2 = b.p; g.loO2 = b.lo; g.ldo2 = ld; g.sO2 = s; }

// ---------------------------------------------------------------- forward
// Buffers of one pass of the embedding and the frozen prefix over B * rows rows
// (row s * rows + j): the fp32 residual stream, an operand-type ping-pong
// buffer, the operand copy of the prefix output, the hidden-width temporaries,
// and, for a SwiGLU fast block whose gate and up projections are frozen, the
// activation silu(gate h) * (up h) it feeds to its (fast) down projection.
struct PrefixBufs {
  float* x32 = nullptr;
  OpBuf xop, hout, tmp_a;
  float* tmp_g = nullptr;
  OpBuf swiglu_a;        // p == nullptr: not computed here
  bool attn = false;     // attention buffers present (whole-sequence passes only)
  bool attn_dec = false; // one decoded row per sequence against the K/V cache
};

// Row layout of the tensor-core attention of one whole-sequence pass of R
// positions per sequence with window k: query blocks of Bq rows; each
// block's window holds nw >= k + Bq - 1 keys ending at its last row; every
// sequence's rows start after `pad` zero rows (so every window starts inside
// the buffer) and fill L = nqb * Bq padded rows; the score GEMMs run over the
// nb = B * nqb - j0 blocks from the first real one (j0 = pad / Bq) on.
struct SwaGeom {
  long long Bq, nw, pad, L, nqb, j0, nb;
};

static long long round_up(long long a, long long m) { return (a + m - 1) / m * m; }

static SwaGeom swa_geom(int B, long long R, int k) {
  SwaGeom g;
  g.Bq = kSwaTcRows;
  g.nw = round_up(k + g.Bq - 1, 16);
  g.pad = round_up(g.nw > g.Bq ? g.nw - g.Bq : 0, g.Bq);
  g.L = g.pad + round_up(R, g.Bq);
  g.nqb = g.L / g.Bq;
  g.j0 = g.pad / g.Bq;
  g.nb = (long long)B * g.nqb - g.j0;
  return g;
}

// The decoding K/V cache of frozen block p: [B][attn_window][d] each.
static float* kv_k(ttt_handle* h, int p) {
  return h->kv + (size_t)(2 * p) * h->B * h->dm.attn_window * h->d;
}
static float* kv_v(ttt_handle* h, int p) { return kv_k(h, p) + (size_t)h->B * h->dm.attn_window * h->d; }

// h += Attn(h) for prefix block p of one decoded row per sequence (position
// *dec_pos): the Q | K | V projection, the cached-window attention (which
// appends this row's K and V to the cache), Wo with the residual.
static ttt_status attention_decode(ttt_handle* h, int p, float* x32, const OpBuf& cur, cudaStream_t st) {
  const int B = h->B, d = h->d, H = h->dm.attn_heads, dh = d / H, k = h->dm.attn_window, stg = h->stg;
  GemmDesc gq;
  gq.M = B; gq.N = 3 * d; gq.K = d;
  setA(gq, cur, d); setB(gq, h->attn_qkv[p], d);
  gq.epi = EPI_STORE_F32; gq.out = h->dec_qkv; gq.ldo = 3 * d;
  TTT_TRY(rungemm(h, K_GEMM_PREFIX, gq, st));
  TTT_TRY(run(h, K_ATTN, st, 1, [&] {
    return launch_swa_decode(stg, B, H, dh, k, h->dec_pos, h->dec_qkv, kv_k(h, p), kv_v(h, p), h->dec_work,
                             h->dec_cnt, h->dec_att.p, h->dec_att.lo, st);
  }));
  GemmDesc gw;
  gw.M = B; gw.N = d; gw.K = d;
  setA(gw, h->dec_att, d); setB(gw, h->attn_o[p], d);
  gw.epi = EPI_RESID; gw.aux = x32; gw.ldx = d; gw.out = x32; gw.ldo = d;
  setOut2(gw, cur, d);
  return rungemm(h, K_GEMM_PREFIX, gw, st);
}

// Whether the attention of the frozen blocks runs as the one fused kernel.
static bool attn_fused(const ttt_handle* h) {
  return !h->opt.attn_unfused && swa_fused_supported(h->stg, h->d, h->dm.attn_heads);
}

// h += Attn(h) for prefix block p over B sequences of `rows` positions from 0:
// x32 is the fp32 residual stream and cur its operand copy (both [B][rows][d]),
// updated in place.  One GEMM projects to Q | K | V; fp32 storage then runs
// the tiled attention kernel, bf16 and split storage the tensor-core form
// (per head: batched score GEMM over the query blocks' windows, masked row
// softmax, batched P V GEMM); Wo adds the heads' output to the residual.
static ttt_status attention_sublayer(ttt_handle* h, int p, int rows, float* x32, const OpBuf& cur, cudaStream_t st) {
  const int B = h->B, d = h->d, H = h->dm.attn_heads, dh = d / H, k = h->dm.attn_window, stg = h->stg;
  const long long M = (long long)B * rows;
  GemmDesc gw;
  gw.N = d; gw.K = d;
  setB(gw, h->attn_o[p], d);
  gw.epi = EPI_RESID;
  if (stg == ST_F32) {
    GemmDesc gq;
    gq.M = M; gq.N = 3 * d; gq.K = d;
    setA(gq, cur, d); setB(gq, h->attn_qkv[p], d);
    gq.epi = EPI_STORE_F32; gq.out = h->qkv32; gq.ldo = 3 * d;
    TTT_TRY(rungemm(h, K_GEMM_PREFIX, gq, st));
    TTT_TRY(run(h, K_ATTN, st, 1, [&] {
      return launch_kv_fill(stg, B, rows, k, d, h->qkv32, 0, rows, 0, kv_k(h, p), kv_v(h, p), st);
    }));
    TTT_TRY(run(h, K_ATTN, st, 1, [&] {
      return launch_swa(stg, B, rows, H, dh, k, h->qkv32, h->att_o.p, h->att_o.lo, st);
    }));
    gw.M = M;
    setA(gw, h->att_o, d);
    gw.aux = x32; gw.ldx = d; gw.out = x32; gw.ldo = d;
    setOut2(gw, cur, d);
    return rungemm(h, K_GEMM_PREFIX, gw, st);
  }
  const SwaGeom g = swa_geom(B, rows, k);
  const long long ld = 3LL * d;
  // the projections take one GEMM per sequence (the weights are shared, and the
  // padded rows of sequence s start at s * L + pad)
  for (int s = 0; s < B; ++s) {
    GemmDesc gq;
    gq.M = rows; gq.N = 3 * d; gq.K = d;
    setA(gq, op_at(h, cur, (long long)s * rows * d), d); setB(gq, h->attn_qkv[p], d);
    gq.epi = EPI_STORE;
    setOut(gq, op_at(h, h->qkvp, ((long long)s * g.L + g.pad) * ld), ld);
    TTT_TRY(rungemm(h, K_GEMM_PREFIX, gq, st));
  }
  TTT_TRY(run(h, K_ATTN, st, 1, [&] {
    return launch_kv_fill(stg, B, rows, k, d, h->qkvp.p, h->qkvp.lo, g.L, g.pad, kv_k(h, p), kv_v(h, p), st);
  }));
  const long long q_row = g.j0 * g.Bq, k_row = g.j0 * g.Bq + g.Bq - g.nw;   // first block's query / window row
  if (attn_fused(h)) {
    // every head in one launch; scores and probabilities stay on chip
    TTT_TRY(run(h, K_ATTN, st, 1, [&] {
      return launch_swa_fused(B, rows, H, dh, k, h->qkvp.p, (int)g.pad, g.L, h->att_p.p, h->flag, st);
    }));
  }
  for (int hh = 0; hh < H && !attn_fused(h); ++hh) {
    GemmDesc gs;
    gs.M = g.Bq; gs.N = g.nw; gs.K = dh; gs.batch = (int)g.nb;
    setA(gs, op_at(h, h->qkvp, q_row * ld + (long long)hh * dh), ld, g.Bq * ld);
    setB(gs, op_at(h, h->qkvp, k_row * ld + d + (long long)hh * dh), ld, g.Bq * ld);
    gs.epi = EPI_STORE_F32; gs.out = h->Sc; gs.ldo = g.nw; gs.sO = g.Bq * g.nw;
    TTT_TRY(rungemm(h, K_ATTN, gs, st));
    TTT_TRY(run(h, K_ATTN, st, 1, [&] {
      return launch_band_softmax(stg, g.nb, (int)g.nw, (int)g.nqb, (int)g.j0, (int)g.pad, rows, k,
                                 1.0f / sqrtf((float)dh), h->Sc, h->Pp.p, h->Pp.lo, st);
    }));
    GemmDesc go;
    go.M = g.Bq; go.N = dh; go.K = g.nw; go.batch = (int)g.nb;
    setA(go, h->Pp, g.nw, g.Bq * g.nw);
    go.b_kmajor = false;
    setB(go, op_at(h, h->qkvp, k_row * ld + 2LL * d + (long long)hh * dh), ld, g.Bq * ld);
    go.epi = EPI_STORE;
    setOut(go, op_at(h, h->att_p, q_row * d + (long long)hh * dh), d, g.Bq * d);
    TTT_TRY(rungemm(h, K_ATTN, go, st));
  }
  for (int s = 0; s < B; ++s) {
    GemmDesc gs = gw;
    gs.M = rows;
    setA(gs, op_at(h, h->att_p, ((long long)s * g.L + g.pad) * d), d);
    float* xs = x32 + (long long)s * rows * d;
    gs.aux = xs; gs.ldx = d; gs.out = xs; gs.ldo = d;
    setOut2(gs, op_at(h, cur, (long long)s * rows * d), d);
    TTT_TRY(rungemm(h, K_GEMM_PREFIX, gs, st));
  }
  return TTT_OK;
}

// Embedding + frozen prefix (and the frozen SwiGLU front of fast block 0 when
// pb.swiglu_a is set) for the tokens of tv: W-independent work.
static ttt_status prefix_pass(ttt_handle* h, const TokView& tv, const PrefixBufs& pb, cudaStream_t st) {
  const int B = h->B, M = B * tv.rows, d = h->d, f = h->f, stg = h->stg;
  OpBuf cur = h->n_pre > 0 ? pb.xop : pb.hout;
  TTT_TRY(run(h, K_EMBED, st, 1, [&] { return launch_embed(stg, B, tv, h->E, d, pb.x32, cur.p, cur.lo, st); }));
  for (int p = 0; p < h->n_pre; ++p) {
    if (p < h->dm.n_prefix && h->dm.attn_heads > 0) {
      if (pb.attn_dec) {
        TTT_TRY(attention_decode(h, p, pb.x32, cur, st));
      } else {
        if (!pb.attn || tv.tok_off != 0)
          return fail(TTT_ERR_UNSUPPORTED, "attention runs in whole-sequence or decoding prefix passes only");
        TTT_TRY(attention_sublayer(h, p, tv.rows, pb.x32, cur, st));
      }
    }
    const OpBuf* W = &h->prefix[(size_t)p * h->nm];
    const OpBuf next = (p == h->n_pre - 1) ? pb.hout : pb.xop;
    if (h->dm.block_kind == TTT_BLOCK_GELU) {
      GemmDesc g;
      g.M = M; g.N = f; g.K = d;
      setA(g, cur, d); setB(g, W[0], d);
      g.epi = EPI_GELU; g.out = nullptr; setOut2(g, pb.tmp_a, f);
      TTT_TRY(rungemm(h, K_GEMM_PREFIX, g, st));
    } else {
      GemmDesc g;
      g.M = M; g.N = f; g.K = d;
      setA(g, cur, d); setB(g, W[0], d);
      g.epi = EPI_STORE_F32; g.out = pb.tmp_g; g.ldo = f;
      TTT_TRY(rungemm(h, K_GEMM_PREFIX, g, st));
      setB(g, W[1], d); g.epi = EPI_SWIGLU; g.aux = pb.tmp_g; g.ldx = f; setOut(g, pb.tmp_a, f);
      TTT_TRY(rungemm(h, K_GEMM_PREFIX, g, st));
    }
    GemmDesc g2;
    g2.M = M; g2.N = d; g2.K = f;
    setA(g2, pb.tmp_a, f); setB(g2, W[h->nm - 1], f);
    g2.epi = EPI_RESID; g2.aux = pb.x32; g2.ldx = d; g2.out = pb.x32; g2.ldo = d;
    setOut2(g2, next, d);
    TTT_TRY(rungemm(h, K_GEMM_PREFIX, g2, st));
    cur = next;
  }
  if (pb.swiglu_a.p) {
    const OpBuf* W = &h->fastfrozen[0];
    GemmDesc g;
    g.M = M; g.N = f; g.K = d;
    setA(g, pb.hout, d); setB(g, W[0], d);
    g.epi = EPI_STORE_F32; g.out = pb.tmp_g; g.ldo = f;
    TTT_TRY(rungemm(h, K_GEMM_FAST_FWD, g, st));
    setB(g, W[1], d); g.epi = EPI_SWIGLU; g.aux = pb.tmp_g; g.ldx = f; setOut(g, pb.swiglu_a, f);
    TTT_TRY(rungemm(h, K_GEMM_FAST_FWD, g, st));
  }
  return TTT_OK;
}

// Rows taken from a hoisted prefix pass (over a group of chunks, or over a
// Settlement chunk q): per sequence the pass holds `rows_total` rows and these
// rows start at row0; x32 / op / a are the pass's fp32 residual, its operand
// copy and (SwiGLU) the block-0 activation.
struct Hoisted {
  bool on = false;
  long long row0 = 0, rows_total = 0;
  const float* x32 = nullptr;
  OpBuf op, a;
};

// Forward over B * tv.rows rows with the current (or committed) fast weights.
// train: keep the stash for backward and turn logits into dlogits in place.
// head_f32: write fp32 logits into logits32 (rows must be 1) instead of the CE.
// hz.on: the prefix output (and SwiGLU activation) of these rows is already in
// the hoisted buffers; otherwise the embedding and the prefix run here.
// delta: the current weights as the committed bf16 copy plus the bf16 offset
// Wdel (two tensor-core products per fast-weight GEMM), for Settlement's score.
static ttt_status forward(ttt_handle* h, const TokView& tv_in, bool committed, bool train,
                          float* losses, long long loss_ld, long long loss_off, bool head_f32,
                          cudaStream_t st, const Hoisted& hz = Hoisted(), bool delta = false) {
  TokView tv = tv_in;
  tv.vocab = h->V;
  tv.err = h->flag;
  const int B = h->B, rows = tv.rows, M = B * rows, d = h->d, f = h->f, V = h->V;
  const int stg = h->stg;
  const OpBuf& Wop = (committed || delta) ? h->Wcop : h->Wop;
  // the second plane of a fast weight's operand when scoring with the offset
  auto wdel = [&](int slot) -> const void* { return delta ? op_at(h, h->Wdel, (long long)slot * B * h->n).p : nullptr; };
  // inputs of fast block 0: its operand rows, their batch stride, the fp32 residual
  OpBuf hin0 = h->hlvl[0];
  long long hin0_s = (long long)rows * d;
  const float* x0 = h->x32;
  OpBuf a0;          // SwiGLU activation of block 0 when hoisted
  long long a0_s = 0;
  if (hz.on) {
    hin0 = op_at(h, hz.op, hz.row0 * d);
    hin0_s = hz.rows_total * d;
    x0 = hz.x32 + hz.row0 * d;
    if (hz.a.p) {
      a0 = op_at(h, hz.a, hz.row0 * f);
      a0_s = hz.rows_total * f;
    }
  } else {
    PrefixBufs pb;
    pb.x32 = h->x32; pb.xop = h->xop; pb.hout = h->hlvl[0]; pb.tmp_a = h->tmp_a; pb.tmp_g = h->tmp_g;
    TTT_TRY(prefix_pass(h, tv, pb, st));
  }
  h->hin0 = hin0;
  h->hin0_s = hin0_s;
  h->a0 = a0;
  h->a0_s = a0_s;

  for (int l = 0; l < h->dm.n_fast; ++l) {
    if (l > 0 && h->dm.static_mlp) {
      // the block's frozen MLP (shared weights: one GEMM over all B * rows rows)
      const OpBuf* W = &h->statics[(size_t)l * h->nm];
      GemmDesc g;
      g.M = M; g.N = f; g.K = d;
      setA(g, h->hlvl[l], d); setB(g, W[0], d);
      g.epi = EPI_GELU;
      if (train) setOut(g, h->szst[l], f);
      else g.out = nullptr;
      setOut2(g, h->tmp_a, f);
      TTT_TRY(rungemm(h, K_GEMM_FAST_FWD, g, st));
      GemmDesc g2;
      g2.M = M; g2.N = d; g2.K = f;
      setA(g2, h->tmp_a, f); setB(g2, W[1], f);
      g2.epi = EPI_RESID; g2.aux = h->x32; g2.ldx = d; g2.out = h->x32; g2.ldo = d;
      setOut2(g2, h->shin[l], d);
      TTT_TRY(rungemm(h, K_GEMM_FAST_FWD, g2, st));
    }
    const OpBuf hin = l == 0 ? hin0 : (h->dm.static_mlp ? h->shin[l] : h->hlvl[l]);
    const long long hin_s = l == 0 ? hin0_s : (long long)rows * d;
    OpBuf a_out = train ? h->ast[l] : h->tmp_a;
    long long a_s = (long long)rows * f;
    const bool has_next = l + 1 < h->dm.n_fast;
    const int s_down = h->slot_of[(size_t)l * h->nm + (h->nm - 1)];
    if (h->dm.block_kind == TTT_BLOCK_GELU) {
      const int s_up = h->slot_of[(size_t)l * h->nm + 0];
      GemmDesc g;
      g.M = rows; g.N = f; g.K = d; g.batch = B;
      setA(g, hin, d, hin_s);
      setB(g, op_at(h, Wop, (long long)s_up * B * h->n), d, h->n);
      g.B2 = wdel(s_up);
      g.epi = EPI_GELU;
      if (train) setOut(g, h->zst[l], f, (long long)rows * f);
      else g.out = nullptr;
      setOut2(g, a_out, f, a_s);
      TTT_TRY(rungemm(h, K_GEMM_FAST_FWD, g, st));
    } else if (l == 0 && a0.p) {
      a_out = a0;
      a_s = a0_s;
    } else {
      // the frozen gate and up projections (rows contiguous across sequences here)
      const OpBuf* W = &h->fastfrozen[(size_t)l * h->nm];
      GemmDesc g;
      g.M = M; g.N = f; g.K = d;
      setA(g, hin, d); setB(g, W[0], d);
      g.epi = EPI_STORE_F32; g.out = h->tmp_g; g.ldo = f;
      TTT_TRY(rungemm(h, K_GEMM_FAST_FWD, g, st));
      setB(g, W[1], d); g.epi = EPI_SWIGLU; g.aux = h->tmp_g; g.ldx = f; setOut(g, a_out, f);
      TTT_TRY(rungemm(h, K_GEMM_FAST_FWD, g, st));
    }
    if (l == 0 && h->dm.block_kind != TTT_BLOCK_GELU) {
      h->a0 = a_out;
      h->a0_s = a_s;
    }
    GemmDesc g2;
    g2.M = rows; g2.N = d; g2.K = f; g2.batch = B;
    setA(g2, a_out, f, a_s);
    setB(g2, op_at(h, Wop, (long long)s_down * B * h->n), f, h->n);
    g2.B2 = wdel(s_down);
    g2.epi = EPI_RESID;
    g2.aux = l == 0 ? x0 : h->x32; g2.ldx = d; g2.sX = l == 0 ? (hz.on ? hz.rows_total * d : (long long)rows * d)
                                                               : (long long)rows * d;
    g2.out = h->x32; g2.ldo = d; g2.sO = (long long)rows * d;
    if (has_next) setOut2(g2, h->hlvl[l + 1], d, (long long)rows * d);
    TTT_TRY(rungemm(h, K_GEMM_FAST_FWD, g2, st));
  }

  GemmDesc gh;
  gh.M = M; gh.N = V; gh.K = d;
  setA(gh, h->y, d); setB(gh, h->U, d);
  // bf16 workloads fold the softmax statistics into the head GEMM's epilogue
  // when it runs on the tensor cores (the per-row cross-entropy kernel otherwise)
  GemmDesc gl = gh;
  gl.dtype = stg;
  gl.epi = EPI_LOGITS; gl.out = train ? h->logits : nullptr; gl.ldo = V;
  gl.lse_part = h->lse_part; gl.lse_ld = h->lse_ld;
  const bool fused = !head_f32 && stg == ST_BF16 && V % 8 == 0 && gemm_tc_supported(gl);

  TTT_TRY(run(h, K_RMSNORM_FWD, st, 1, [&] {
    return launch_rmsnorm_fwd(stg, M, d, h->x32, h->dm.rms_eps, h->y.p, h->y.lo, h->rstd, fused ? &tv : nullptr,
                              h->tgt, st);
  }));

  const float scale = tv.n_valid > 0 ? 1.0f / (float)tv.n_valid : 0.0f;
  // Source Masking: per-row scales of this chunk (set by chunk_step) replace 1/b
  const float* rscale = train && h->rscale_on ? h->rscale : nullptr;
  if (fused) {
    TTT_TRY(rungemm(h, K_GEMM_HEAD, gl, st));
    const int nt = ceil_div(V, gemm_tc_tile_n(gl));
    TTT_TRY(run(h, K_CE, st, 1, [&] {
      return launch_lse_combine(B, tv, h->lse_part, h->lse_ld, nt, h->y.p, h->U.p, d, h->tgt, h->lse, losses,
                                loss_ld, loss_off, h->row_loss, st);
    }));
    if (!train) return TTT_OK;
    return run(h, K_CE, st, 1, [&] { return launch_dlogits(M, V, h->logits, h->lse, h->tgt, scale, rscale, st); });
  }
  if (head_f32) {
    gh.epi = EPI_STORE_F32; gh.out = h->logits32; gh.ldo = V;
    return rungemm(h, K_GEMM_HEAD, gh, st);
  }
  if (stg == ST_SPLIT) {
    gh.epi = EPI_STORE_F32; gh.out = h->logits; gh.ldo = V;
  } else {
    gh.epi = EPI_STORE; gh.out = h->logits; gh.ldo = V;
  }
  TTT_TRY(rungemm(h, K_GEMM_HEAD, gh, st));
  return run(h, K_CE, st, 1, [&] {
    return launch_ce(stg, B, tv, V, h->logits, V, scale, rscale, train, losses, loss_ld, loss_off, h->row_loss, st);
  });
}

// ---------------------------------------------------------------- backward + update
static ttt_status backward_update(ttt_handle* h, int rows, cudaStream_t st) {
  const int B = h->B, M = B * rows, d = h->d, f = h->f, V = h->V, stg = h->stg;
  GemmDesc gy;
  gy.M = M; gy.N = d; gy.K = V;
  if (stg == ST_SPLIT) {
    // dlogits were written inside each fp32 row as [hi: V bf16 | lo: V bf16]
    gy.A = h->logits; gy.lda = 2LL * V; gy.loA = V;
  } else {
    gy.A = h->logits; gy.lda = V;
  }
  setB(gy, h->U, d); gy.b_kmajor = false;
  gy.epi = EPI_STORE_F32; gy.out = h->dy32; gy.ldo = d;
  TTT_TRY(rungemm(h, K_GEMM_HEAD_BWD, gy, st));
  TTT_TRY(run(h, K_RMSNORM_BWD, st, 1, [&] {
    return launch_rmsnorm_bwd(stg, M, d, h->x32, h->rstd, h->dy32, h->dh32, h->dhop.p, h->dhop.lo, st);
  }));

  PartialSlots ps{};
  long long poff = 0;
  // GELU blocks without static MLPs run each weight gradient on the handle's
  // second stream beside the input-gradient chain (dW2 of block l needs only
  // dh and the a stash, dW1 only dz and the block input), so each dW GEMM fills
  // the tail waves of its dX partner.  The operand copy of dh alternates between
  // two buffers, so the chain never rewrites a dh that a dW still reads.
  // (profiled steps keep the dW GEMMs in stream order: each class's events then
  // bracket its own kernels only)
  const bool side = h->bstream != nullptr && h->prof_class < 0;
  cudaStream_t ws = side ? h->bstream : st;   // stream of the dW GEMMs
  const int nf = h->dm.n_fast;
  auto dh_buf = [&](int l) -> const OpBuf& { return side && (nf - 1 - l) % 2 ? h->dhop2 : h->dhop; };
  auto dw_gemm = [&](GemmDesc& g, int slot) -> ttt_status {
    g.epi = EPI_DW;
    g.dtype = h->stg;
    g.partials = h->partials + poff;
    const int tiles = gemm_partial_tiles(g);
    if (ps.n >= 16 || poff + (long long)tiles * B > h->partial_cap)
      return fail(TTT_ERR_UNSUPPORTED, "too many gradient-norm partial slots");
    g.out = static_cast<char*>(h->dW) + (long long)slot * B * h->n * (long long)h->dw_esz; g.sO = h->n;
    ps.off[ps.n] = poff;
    ps.tiles[ps.n] = tiles;
    ps.n++;
    poff += (long long)tiles * B;
    return rungemm(h, K_GEMM_DW, g, ws);
  };
  // events of the second stream: [0, nf) dh of block l ready, [nf, 2 nf) dz of
  // block l ready, [2 nf, 3 nf) dW2 of block l done, 3 nf: every dW done
  auto ev = [&](int kind, int l) { return h->bev[(size_t)kind * nf + l]; };

  for (int l = nf - 1; l >= 0; --l) {
    if (h->dm.block_kind == TTT_BLOCK_GELU) {
      const int s1 = h->slot_of[(size_t)l * 2 + 0], s2 = h->slot_of[(size_t)l * 2 + 1];
      const OpBuf& dh = dh_buf(l);
      if (side) {
        TTT_CUDA(cudaEventRecord(ev(0, l), st));
        TTT_CUDA(cudaStreamWaitEvent(ws, ev(0, l), 0));
      }
      // dW2 = dh^T a   [d, f], K = rows
      GemmDesc g;
      g.M = d; g.N = f; g.K = rows; g.batch = B;
      g.a_kmajor = false; setA(g, dh, d, (long long)rows * d);
      g.b_kmajor = false; setB(g, h->ast[l], f, (long long)rows * f);
      g.ldo = f;
      TTT_TRY(dw_gemm(g, s2));
      if (side) TTT_CUDA(cudaEventRecord(ev(2, l), ws));
      // dz = (dh W2) * GELU'(z), in place over the z stash
      GemmDesc gz;
      gz.M = rows; gz.N = f; gz.K = d; gz.batch = B;
      setA(gz, dh, d, (long long)rows * d);
      gz.b_kmajor = false; setB(gz, op_at(h, h->Wop, (long long)s2 * B * h->n), f, h->n);
      gz.epi = EPI_DGELU; gz.aux = h->zst[l].p; gz.loX = h->zst[l].lo; gz.ldx = f; gz.sX = (long long)rows * f;
      setOut(gz, h->zst[l], f, (long long)rows * f);
      TTT_TRY(rungemm(h, K_GEMM_BWD_DX, gz, st));
      if (side) {
        TTT_CUDA(cudaEventRecord(ev(1, l), st));
        TTT_CUDA(cudaStreamWaitEvent(ws, ev(1, l), 0));
      }
      // dW1 = dz^T h_in   [f, d]
      GemmDesc g1;
      g1.M = f; g1.N = d; g1.K = rows; g1.batch = B;
      g1.a_kmajor = false; setA(g1, h->zst[l], f, (long long)rows * f);
      if (l == 0) { g1.b_kmajor = false; setB(g1, h->hin0, d, h->hin0_s); }
      else { g1.b_kmajor = false; setB(g1, h->dm.static_mlp ? h->shin[l] : h->hlvl[l], d, (long long)rows * d); }
      g1.ldo = d;
      TTT_TRY(dw_gemm(g1, s1));
      if (l > 0) {
        // dh_below = dh + dz W1, its operand copy into the other dh buffer,
        // which dW2 of block l + 1 (two levels up) read last
        if (side && l + 1 < nf) TTT_CUDA(cudaStreamWaitEvent(st, ev(2, l + 1), 0));
        GemmDesc gb;
        gb.M = rows; gb.N = d; gb.K = f; gb.batch = B;
        setA(gb, h->zst[l], f, (long long)rows * f);
        gb.b_kmajor = false; setB(gb, op_at(h, h->Wop, (long long)s1 * B * h->n), d, h->n);
        gb.epi = EPI_RESID; gb.aux = h->dh32; gb.ldx = d; gb.sX = (long long)rows * d;
        gb.out = h->dh32; gb.ldo = d; gb.sO = (long long)rows * d;
        setOut2(gb, dh_buf(l - 1), d, (long long)rows * d);
        TTT_TRY(rungemm(h, K_GEMM_BWD_DX, gb, st));
        if (h->dm.static_mlp) {
          // through the block's frozen MLP: dz_s = (dh W2s) * GELU'(z_s); dh += dz_s W1s
          const OpBuf* W = &h->statics[(size_t)l * 2];
          GemmDesc sz;
          sz.M = M; sz.N = f; sz.K = d;
          setA(sz, h->dhop, d);
          sz.b_kmajor = false; setB(sz, W[1], f);
          sz.epi = EPI_DGELU; sz.aux = h->szst[l].p; sz.loX = h->szst[l].lo; sz.ldx = f;
          setOut(sz, h->szst[l], f);
          TTT_TRY(rungemm(h, K_GEMM_BWD_DX, sz, st));
          GemmDesc sb;
          sb.M = M; sb.N = d; sb.K = f;
          setA(sb, h->szst[l], f);
          sb.b_kmajor = false; setB(sb, W[0], d);
          sb.epi = EPI_RESID; sb.aux = h->dh32; sb.ldx = d; sb.out = h->dh32; sb.ldo = d;
          setOut2(sb, h->dhop, d);
          TTT_TRY(rungemm(h, K_GEMM_BWD_DX, sb, st));
        }
      }
    } else {
      const int sd = h->slot_of[(size_t)l * 3 + 2];
      GemmDesc g;
      g.M = d; g.N = f; g.K = rows; g.batch = B;
      g.a_kmajor = false; setA(g, h->dhop, d, (long long)rows * d);
      if (l == 0) { g.b_kmajor = false; setB(g, h->a0, f, h->a0_s); }
      else { g.b_kmajor = false; setB(g, h->ast[l], f, (long long)rows * f); }
      g.ldo = f;
      TTT_TRY(dw_gemm(g, sd));
    }
  }
  if (side) {
    // the update reads every dW: join the second stream
    TTT_CUDA(cudaEventRecord(h->bev[(size_t)3 * nf], ws));
    TTT_CUDA(cudaStreamWaitEvent(st, h->bev[(size_t)3 * nf], 0));
  }
  // the per-sequence norm is reduced inside the update kernel (grad_norm has no launch of its own)
  TTT_TRY(run(h, K_SGD, st, 1, [&] {
    return launch_clip_sgd_update(stg, h->nslots, B, h->n, h->W32, h->Wop.p, h->Wop.lo, h->dW, ps, h->partials,
                                  h->hp.clip, h->hp.eta, h->scale, h->gnorm, h->flag, st);
  }));
  h->chunks_done++;
  if (h->hp.reset_every > 0 && h->chunks_done % h->hp.reset_every == 0)
    TTT_TRY(run(h, K_OTHER, st, 1, [&] {
      return launch_broadcast_w0(stg, h->nslots, B, h->n, h->W0, h->W32, h->Wop.p, h->Wop.lo, st);
    }));
  return TTT_OK;
}

// One chunk step; with `mask` (Source Masking, [B][mask_ld], the chunk's
// targets at offset tv.tok_off) the chunk's loss is the mean over its unmasked
// targets instead of all b.
static ttt_status chunk_step(ttt_handle* h, const TokView& tv, float* losses, long long loss_ld,
                             long long loss_off, cudaStream_t st, const Hoisted& hz = Hoisted(),
                             const uint8_t* mask = nullptr, long long mask_ld = 0) {
  if (mask)
    TTT_TRY(run(h, K_OTHER, st, 1, [&] {
      return launch_chunk_row_scale(h->B, tv.rows, mask, mask_ld, tv.tok_off, h->rscale, st);
    }));
  h->rscale_on = mask != nullptr;
  const ttt_status fs = forward(h, tv, false, true, losses, loss_ld, loss_off, false, st, hz);
  h->rscale_on = false;
  TTT_TRY(fs);
  return backward_update(h, tv.rows, st);
}

// The embedding and frozen prefix of chunks i0 .. i0+g-1 of every sequence in
// one pass over B * g * b rows (they do not depend on the fast weights), into
// the hoisted buffers laid out [B][g * b][.].
static ttt_status hoisted_prefix(ttt_handle* h, const int32_t* tok, long long tok_ld, int i0, int g,
                                 cudaStream_t st) {
  TokView tv;
  tv.tok = tok; tv.tok_ld = tok_ld; tv.tok_off = (long long)i0 * h->b; tv.rows = g * h->b; tv.n_valid = g * h->b;
  tv.vocab = h->V;
  tv.err = h->flag;
  PrefixBufs pb;
  pb.x32 = h->hx32; pb.xop = h->hx_xop; pb.hout = h->hx_op; pb.tmp_a = h->hx_tmp_a; pb.tmp_g = h->hx_tmp_g;
  pb.swiglu_a = h->ha;
  return prefix_pass(h, tv, pb, st);
}

// Settlement on held-out q [B, Lq] (device): writes A[B], accept[B].
static ttt_status settle_event(ttt_handle* h, const int32_t* q, int Lq, float* A, uint8_t* acc,
                               cudaStream_t st) {
  TokView tv;
  tv.tok = q; tv.tok_ld = Lq; tv.tok_off = 0; tv.rows = Lq; tv.n_valid = Lq - 1;
  tv.vocab = h->V;
  tv.err = h->flag;
  // q's frozen prefix does not depend on the fast weights: one pass serves the
  // committed and the current forward
  Hoisted hz;
  if (h->qx32) {
    PrefixBufs pb;
    pb.x32 = h->qx32; pb.xop = h->xop; pb.hout = h->qx_op; pb.tmp_a = h->tmp_a; pb.tmp_g = h->tmp_g;
    pb.swiglu_a = h->qa;
    TTT_TRY(prefix_pass(h, tv, pb, st));
    hz.on = true; hz.row0 = 0; hz.rows_total = Lq;
    hz.x32 = h->qx32; hz.op = h->qx_op; hz.a = h->qa;
  }
  TTT_TRY(forward(h, tv, true, false, nullptr, 0, 0, false, st, hz));
  TTT_TRY(run(h, K_SETTLE, st, 1, [&] { return launch_seq_mean(h->B, Lq, Lq - 1, h->row_loss, h->Lc, st); }));
  // bf16 storage scores the candidate as the committed bf16 copy plus its
  // offset in bf16: both losses then round the weights alike, so A sees the
  // whole update (a bf16 copy of W alone would round most of an update below
  // half an ulp away, and W_0 starts on the bf16 grid)
  const bool delta = h->Wdel.p != nullptr;
  if (delta)
    TTT_TRY(run(h, K_SETTLE, st, 1, [&] {
      return launch_delta_plane(h->nslots, h->B, h->n, h->W32, h->Wc32, h->Wdel.p, st);
    }));
  TTT_TRY(forward(h, tv, false, false, nullptr, 0, 0, false, st, hz, delta));
  TTT_TRY(run(h, K_SETTLE, st, 1, [&] { return launch_seq_mean(h->B, Lq, Lq - 1, h->row_loss, h->Lw, st); }));
  return run(h, K_SETTLE, st, 2, [&] {
    return launch_settle_apply(h->stg, h->nslots, h->B, h->n, h->Lc, h->Lw, A, acc, h->W32, h->Wop.p,
                               h->Wc32, h->Wcop.p, h->Wop.lo, st);
  });
}

// Next-token forward of one decoded row per sequence with attention: the
// one-row prefix pass against the K/V cache into the decoding buffers, then
// the fast blocks and the head from those rows (fp32 logits).
static ttt_status attn_next_forward(ttt_handle* h, const TokView& tv_in, cudaStream_t st) {
  TokView tv = tv_in;      // the embedding checks ids against V and reports through the status word
  tv.vocab = h->V;
  tv.err = h->flag;
  PrefixBufs pb;
  pb.x32 = h->dec_x32; pb.xop = h->dec_xop; pb.hout = h->dec_op; pb.tmp_a = h->dec_tmp_a; pb.tmp_g = h->dec_tmp_g;
  pb.swiglu_a = h->dec_a;
  pb.attn_dec = true;
  TTT_TRY(prefix_pass(h, tv, pb, st));
  Hoisted hz;
  hz.on = true; hz.row0 = 0; hz.rows_total = 1;
  hz.x32 = h->dec_x32; hz.op = h->dec_op; hz.a = h->dec_a;
  return forward(h, tv, false, false, nullptr, 0, 0, true, st, hz);
}

static ttt_status p_next_from_pending(ttt_handle* h, float* p_out, cudaStream_t st,
                                      const Hoisted& hz = Hoisted()) {
  TokView tv;
  tv.tok = h->pend; tv.tok_ld = h->b + 1; tv.tok_off = h->pend_count; tv.rows = 1; tv.n_valid = 0;
  if (h->dm.attn_heads > 0 && !hz.on) TTT_TRY(attn_next_forward(h, tv, st));
  else TTT_TRY(forward(h, tv, false, false, nullptr, 0, 0, true, st, hz));
  TTT_TRY(run(h, K_OTHER, st, 2, [&] {
    return launch_softmax(h->B, h->V, h->logits32, p_out, h->lse_next, h->soft_part, st);
  }));
  // logits32 / lse_next now hold the next-token distribution under the current
  // weights: the next decode step scores its token from them
  h->next_valid = true;
  return TTT_OK;
}

// Decoding's next-token forward as the one persistent cooperative kernel when
// the network and the GPU allow it (bf16 storage, GELU or SwiGLU blocks, no
// attention or extra frozen MLPs, B <= 8): token from the fixed slot x_dev,
// writes logits32, p_dev and lse_next like the graph below.  Returns false
// (nothing launched) when it does not apply.
static bool decode_persist_applies(ttt_handle* h) {
  if (h->dp_grid < 0) {
    h->dp_grid = 0;
    if (!h->opt.no_decode_persist && h->stg == ST_BF16 && h->dm.attn_heads == 0 && !h->dm.static_mlp &&
        h->B <= 8 && h->n_pre + h->dm.n_fast <= kDecodeMaxBlocks)
      h->dp_grid = decode_persist_grid(h->B, h->d, h->f);
  }
  return h->dp_grid > 0;
}

// The persistent forward's buffers and parameter block, on first use.
static ttt_status decode_persist_setup(ttt_handle* h) {
  DecodeNet& n = h->dp_net;
  if (!h->dp_x32) {
    TTT_TRY(dalloc(h, &h->dp_x32, (size_t)2 * h->B * h->d * 4));
    TTT_TRY(dalloc(h, &h->dp_px, (size_t)2 * 8 * h->B * h->d * 4));
    TTT_TRY(dalloc(h, &h->dp_act, (size_t)h->B * h->f * 2));
    TTT_TRY(dalloc(h, &h->dp_part, (size_t)h->dp_grid * h->B * sizeof(float2)));
    TTT_TRY(dalloc(h, &h->dp_bar, 4 * sizeof(unsigned)));
    const int B = h->B, nm = h->nm;
    n.B = B; n.d = h->d; n.f = h->f; n.V = h->V;
    n.swiglu = h->dm.block_kind == TTT_BLOCK_GELU ? 0 : 1;
    n.n_pre = h->n_pre; n.n_fast = h->dm.n_fast;
    n.eps = h->dm.rms_eps;
    n.tok = h->x_dev;
    n.E = h->E;
    for (int p = 0; p < h->n_pre; ++p)
      for (int k = 0; k < nm; ++k) n.pre[p][k] = h->prefix[(size_t)p * nm + k].p;
    for (int l = 0; l < h->dm.n_fast; ++l) {
      if (n.swiglu) {
        n.ffrozen[l][0] = h->fastfrozen[(size_t)l * nm + 0].p;
        n.ffrozen[l][1] = h->fastfrozen[(size_t)l * nm + 1].p;
      } else {
        n.fup[l] = op_at(h, h->Wop, (long long)h->slot_of[(size_t)l * nm + 0] * B * h->n).p;
      }
      n.fdown[l] = op_at(h, h->Wop, (long long)h->slot_of[(size_t)l * nm + (nm - 1)] * B * h->n).p;
    }
    n.n = h->n;
    n.U = h->U.p;
    n.x32 = h->dp_x32; n.px = h->dp_px; n.act = h->dp_act;
    n.logits = h->logits32; n.p = h->p_dev; n.lse = h->lse_next;
    n.part = h->dp_part; n.bar = h->dp_bar; n.err = h->flag;
  }
  return TTT_OK;
}

// The persistent forward, its softmax into p_out (device); bar_clear as
// launch_decode_persist.
static ttt_status decode_persist(ttt_handle* h, float* p_out, bool bar_clear, cudaStream_t st) {
  TTT_TRY(decode_persist_setup(h));
  DecodeNet n = h->dp_net;
  n.p = p_out;
  TTT_TRY(run(h, K_OTHER, st, 1, [&] { return launch_decode_persist(n, h->dp_grid, bar_clear, st); }));
  h->next_valid = true;
  return TTT_OK;
}

// Decoding's next-token forward (embedding -> blocks -> head -> softmax of one
// row per sequence, token from the fixed slot x_dev) as a CUDA graph: captured
// on first use on the handle's own stream, then replayed after the caller's
// stream (event edges both ways).  Every pointer it reads is the handle's, so
// one capture serves every later step.  Writes p_dev, logits32 and lse_next.
static ttt_status decode_forward_graph(ttt_handle* h, cudaStream_t st) {
  if (!h->dec_exec) {
    if (!h->gstream) {
      TTT_CUDA(cudaStreamCreateWithFlags(&h->gstream, cudaStreamNonBlocking));
      TTT_CUDA(cudaEventCreateWithFlags(&h->gev[0], cudaEventDisableTiming));
      TTT_CUDA(cudaEventCreateWithFlags(&h->gev[1], cudaEventDisableTiming));
    }
    const int saved_prof = h->prof_class;   // no profiling events inside the graph
    const bool saved_log = h->log_on;
    h->prof_class = -1;
    h->log_on = false;
    const long long l0 = h->launches;
    TTT_CUDA(cudaStreamBeginCapture(h->gstream, cudaStreamCaptureModeThreadLocal));
    TokView tv;
    tv.tok = h->x_dev; tv.tok_ld = 1; tv.tok_off = 0; tv.rows = 1; tv.n_valid = 0;
    ttt_status s = h->dm.attn_heads > 0 ? attn_next_forward(h, tv, h->gstream)
                                        : forward(h, tv, false, false, nullptr, 0, 0, true, h->gstream);
    if (s == TTT_OK)
      s = run(h, K_OTHER, h->gstream, 2, [&] {
        return launch_softmax(h->B, h->V, h->logits32, h->p_dev, h->lse_next, h->soft_part, h->gstream);
      });
    cudaGraph_t graph = nullptr;
    const cudaError_t e = cudaStreamEndCapture(h->gstream, &graph);
    h->prof_class = saved_prof;
    h->log_on = saved_log;
    h->dec_kernels = h->launches - l0;
    h->launches = l0;
    if (s != TTT_OK) {
      if (graph) cudaGraphDestroy(graph);
      return s;
    }
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamEndCapture", __FILE__, __LINE__);
    const cudaError_t ei = cudaGraphInstantiate(&h->dec_exec, graph, 0);
    cudaGraphDestroy(graph);
    if (ei != cudaSuccess) {
      h->dec_exec = nullptr;
      return cuda_fail(ei, "cudaGraphInstantiate", __FILE__, __LINE__);
    }
  }
  TTT_CUDA(cudaEventRecord(h->gev[0], st));
  TTT_CUDA(cudaStreamWaitEvent(h->gstream, h->gev[0], 0));
  TTT_CUDA(cudaGraphLaunch(h->dec_exec, h->gstream));
  TTT_CUDA(cudaEventRecord(h->gev[1], h->gstream));
  TTT_CUDA(cudaStreamWaitEvent(st, h->gev[1], 0));
  h->launches += h->dec_kernels;
  h->next_valid = true;
  return TTT_OK;
}

static ttt_status reset_weights(ttt_handle* h, cudaStream_t st) {
  TTT_TRY(run(h, K_OTHER, st, 1, [&] {
    return launch_broadcast_w0(h->stg, h->nslots, h->B, h->n, h->W0, h->W32, h->Wop.p, h->Wop.lo, st);
  }));
  if (h->Wc32) {
    TTT_TRY(run(h, K_OTHER, st, 1, [&] {
      return launch_broadcast_w0(h->stg, h->nslots, h->B, h->n, h->W0, h->Wc32, h->Wcop.p, h->Wcop.lo, st);
    }));
  }
  h->pend_count = 0;
  h->chunks_done = 0;
  return TTT_OK;
}

// Wait for the stream and turn the device status word into a status code.
static ttt_status finish(ttt_handle* h, cudaStream_t st) {
  TTT_CUDA(cudaMemcpyAsync(h->flag_host, h->flag, 4, cudaMemcpyDeviceToHost, st));
  TTT_CUDA(cudaStreamSynchronize(st));
  if (*h->flag_host & kErrGemmTimeout) {
    // a split-K CTA that gave up left its tile's arrival counter non-zero:
    // clear every counter so the next call counts from zero
    TTT_CUDA(cudaMemsetAsync(h->split_cnt, 0, (size_t)gemm_tc_max_split_tiles() * sizeof(int), st));
    TTT_CUDA(cudaStreamSynchronize(st));
    return fail(TTT_ERR_TIMEOUT, "a GEMM pipeline wait timed out");
  }
  if (*h->flag_host & 2) return fail(TTT_ERR_BAD_ARG, "token id outside [0, vocab)");
  if (*h->flag_host & 1) return fail(TTT_ERR_NONFINITE, "non-finite gradient norm: update skipped");
  return TTT_OK;
}

static ttt_status ensure_staging(ttt_handle* h, void** p, size_t* cap, size_t bytes) {
  if (*cap >= bytes) return TTT_OK;
  if (*p) {
    for (auto& a : h->allocs)
      if (a == *p) a = nullptr;
    cudaFree(*p);
    *p = nullptr;
    *cap = 0;
  }
  void* q = nullptr;
  TTT_TRY(dalloc(h, &q, bytes));
  *p = q;
  *cap = bytes;
  return TTT_OK;
}

static void dfree(ttt_handle* h, void* p) {
  if (!p) return;
  for (auto& a : h->allocs)
    if (a == p) a = nullptr;
  cudaFree(p);
}

// Buffers of the whole-sequence prefix pass of an attention prefill: `rows`
// = B * (T + 1) rows, reallocated only when a longer prefill arrives.
static ttt_status ensure_op_elems(ttt_handle* h, OpBuf* b, size_t* cap, size_t count, bool zero) {
  if (count <= *cap) return TTT_OK;
  dfree(h, b->p);
  *b = OpBuf();
  *cap = 0;
  const size_t planes = h->stg == ST_SPLIT ? 2 : 1;
  TTT_TRY(dalloc(h, &b->p, count * h->esz * planes));
  b->lo = planes == 2 ? (long long)count : 0;
  if (zero) TTT_CUDA(cudaMemset(b->p, 0, count * h->esz * planes));
  *cap = count;
  return TTT_OK;
}

// Buffers of the tensor-core attention for sequences of T + 1 positions.
static ttt_status ensure_attn_tc(ttt_handle* h, long long R) {
  const SwaGeom g = swa_geom(h->B, R, h->dm.attn_window);
  const size_t d = h->d;
  // zero once: rows the projections never write (the padding) must hold finite values
  TTT_TRY(ensure_op_elems(h, &h->qkvp, &h->qkvp_cap, (size_t)h->B * g.L * 3 * d, true));
  TTT_TRY(ensure_op_elems(h, &h->att_p, &h->attp_cap, (size_t)h->B * g.L * d, false));
  if (attn_fused(h)) return TTT_OK;    // scores and probabilities stay on chip
  const size_t blk = (size_t)g.nb * g.Bq * g.nw;
  size_t pp_cap = h->sc_cap;
  if (blk > h->sc_cap) {
    dfree(h, h->Sc);
    h->Sc = nullptr;
    h->sc_cap = 0;
    TTT_TRY(dalloc(h, &h->Sc, blk * 4));
    h->sc_cap = blk;
  }
  return ensure_op_elems(h, &h->Pp, &pp_cap, blk, false);
}

static ttt_status ensure_attn_rows(ttt_handle* h, size_t rows) {
  if (rows <= h->arows_cap) return TTT_OK;
  const size_t planes = h->stg == ST_SPLIT ? 2 : 1;
  OpBuf* ops[] = {&h->ax_op, &h->ax_xop, &h->ax_tmp_a, &h->ax_a, &h->att_o};
  for (OpBuf* b : ops) {
    dfree(h, b->p);
    *b = OpBuf();
  }
  dfree(h, h->ax32); h->ax32 = nullptr;
  dfree(h, h->ax_tmp_g); h->ax_tmp_g = nullptr;
  dfree(h, h->qkv32); h->qkv32 = nullptr;
  h->arows_cap = 0;
  const size_t d = h->d, f = h->f;
  auto op = [&](OpBuf* b, size_t count) -> ttt_status {
    TTT_TRY(dalloc(h, &b->p, count * h->esz * planes));
    b->lo = planes == 2 ? (long long)count : 0;
    return TTT_OK;
  };
  TTT_TRY(dalloc(h, &h->ax32, rows * d * 4));
  TTT_TRY(op(&h->ax_op, rows * d));
  TTT_TRY(op(&h->ax_xop, rows * d));
  TTT_TRY(op(&h->ax_tmp_a, rows * f));
  if (h->stg == ST_F32) {
    TTT_TRY(op(&h->att_o, rows * d));
    TTT_TRY(dalloc(h, &h->qkv32, rows * 3 * d * 4));
  }
  if (h->dm.block_kind == TTT_BLOCK_SWIGLU) {
    TTT_TRY(dalloc(h, &h->ax_tmp_g, rows * f * 4));
    TTT_TRY(op(&h->ax_a, rows * f));
  }
  h->arows_cap = rows;
  return TTT_OK;
}

// One operand buffer's rows: nrows rows per sequence from src (src_rows per
// sequence, starting at src_row0) to dst (dst_rows per sequence, at dst_row0),
// width elements each, every plane.
static ttt_status copy_op_rows(ttt_handle* h, const OpBuf& dst, long long dst_rows, long long dst_row0, const OpBuf& src,
                               long long src_rows, long long src_row0, long long nrows, long long width,
                               cudaStream_t st) {
  const size_t es = h->esz;
  const int planes = h->stg == ST_SPLIT ? 2 : 1;
  for (int q = 0; q < planes; ++q) {
    char* d0 = static_cast<char*>(dst.p) + ((q ? dst.lo : 0) + dst_row0 * width) * es;
    const char* s0 = static_cast<const char*>(src.p) + ((q ? src.lo : 0) + src_row0 * width) * es;
    TTT_CUDA(cudaMemcpy2DAsync(d0, (size_t)(dst_rows * width * es), s0, (size_t)(src_rows * width * es),
                               (size_t)(nrows * width * es), h->B, cudaMemcpyDeviceToDevice, st));
  }
  return TTT_OK;
}

// Prefix rows (fp32 residual, operand copy, SwiGLU activation) into the
// pending-row buffers of decoding with attention, rows dst_row0 ...
static ttt_status save_pending_rows(ttt_handle* h, const float* x32, const OpBuf& op, const OpBuf& a, long long src_rows,
                                    long long src_row0, long long dst_row0, long long nrows, cudaStream_t st) {
  const long long pr = h->b + 1, d = h->d;
  TTT_CUDA(cudaMemcpy2DAsync(h->prow32 + dst_row0 * d, (size_t)(pr * d * 4), x32 + src_row0 * d,
                             (size_t)(src_rows * d * 4), (size_t)(nrows * d * 4), h->B, cudaMemcpyDeviceToDevice, st));
  TTT_TRY(copy_op_rows(h, h->prow_op, pr, dst_row0, op, src_rows, src_row0, nrows, d, st));
  if (h->prow_a.p && a.p) TTT_TRY(copy_op_rows(h, h->prow_a, pr, dst_row0, a, src_rows, src_row0, nrows, h->f, st));
  return TTT_OK;
}

static ttt_status copy_in(ttt_handle* h, const void* src, void** stage, size_t* cap, size_t bytes,
                          const void** dev, cudaStream_t st) {
  if (is_device_ptr(src)) {
    *dev = src;
    return TTT_OK;
  }
  TTT_TRY(ensure_staging(h, stage, cap, bytes));
  TTT_CUDA(cudaMemcpyAsync(*stage, src, bytes, cudaMemcpyHostToDevice, st));
  *dev = *stage;
  return TTT_OK;
}

}  // namespace ttt

using namespace ttt;

// ====================================================================== C ABI
extern "C" {

const char* ttt_status_string(ttt_status s) {
  switch (s) {
    case TTT_OK: return "ok";
    case TTT_ERR_BAD_ARG: return "bad argument";
    case TTT_ERR_BAD_SHAPE: return "bad shape";
    case TTT_ERR_OOM: return "out of device memory";
    case TTT_ERR_CUDA: return "CUDA error";
    case TTT_ERR_NONFINITE: return "non-finite gradient norm (update skipped)";
    case TTT_ERR_TIMEOUT: return "device wait timed out";
    case TTT_ERR_UNSUPPORTED: return "unsupported configuration";
    case TTT_ERR_STATE: return "call out of order";
  }
  return "unknown status";
}

const char* ttt_last_error(void) { return g_last_error.c_str(); }

static const char* kKClassNames[K_COUNT] = {
    "embed", "gemm_prefix", "gemm_fast_fwd", "rmsnorm_fwd", "gemm_head", "ce_fused",
    "gemm_head_bwd", "rmsnorm_bwd", "gemm_bwd_dx", "gemm_dw", "grad_norm", "clip_sgd_update",
    "settle", "other", "token_step", "attention"};

const char* ttt_kernel_class_name(int c) { return (c >= 0 && c < K_COUNT) ? kKClassNames[c] : ""; }
int ttt_kernel_class_count(void) { return K_COUNT; }

ttt_status ttt_destroy(ttt_handle* h) {
  if (!h) return TTT_OK;
  for (void* p : h->allocs)
    if (p) cudaFree(p);
  for (auto e : h->ev) cudaEventDestroy(e);
  if (h->dec_exec) cudaGraphExecDestroy(h->dec_exec);
  for (auto e : h->gev)
    if (e) cudaEventDestroy(e);
  if (h->gstream) cudaStreamDestroy(h->gstream);
  for (auto e : h->bev)
    if (e) cudaEventDestroy(e);
  if (h->bstream) cudaStreamDestroy(h->bstream);
  if (h->flag_host) cudaFreeHost(h->flag_host);
  delete h;
  return TTT_OK;
}

ttt_status ttt_create(const ttt_dims* dims, const ttt_hparams* hp, const ttt_weights* w, ttt_handle** out) {
  return ttt_create_ex(dims, hp, w, nullptr, out);
}

ttt_status ttt_create_ex(const ttt_dims* dims, const ttt_hparams* hp, const ttt_weights* w, const ttt_options* opt,
                         ttt_handle** out) {
  if (!dims || !hp || !w || !out) return fail(TTT_ERR_BAD_ARG, "null argument to ttt_create");
  *out = nullptr;
  const ttt_options O = opt ? *opt : ttt_options{};
  if (O.no_pdl < 0 || O.no_decode_graph < 0 || O.fp32_simt < 0 || O.hoist_chunks < 0 || O.no_token_kernel < 0 ||
      O.max_ctas < 0 || O.no_dw_stream < 0 || O.attn_unfused < 0 || O.no_decode_persist < 0)
    return fail(TTT_ERR_BAD_ARG, "negative ttt_options field");
  PdlScope pdl(!O.no_pdl);
  const ttt_dims& D = *dims;
  if (D.d <= 0 || D.d_ff <= 0 || D.vocab <= 0 || D.n_prefix < 0 || D.n_fast < 1 || D.rms_eps < 0.0f)
    return fail(TTT_ERR_BAD_ARG, "bad dims");
  if (D.block_kind != TTT_BLOCK_GELU && D.block_kind != TTT_BLOCK_SWIGLU)
    return fail(TTT_ERR_BAD_ARG, "bad block_kind");
  if (D.dtype != TTT_DTYPE_FP32 && D.dtype != TTT_DTYPE_BF16) return fail(TTT_ERR_BAD_ARG, "bad dtype");
  if (hp->chunk < 1 || hp->max_batch < 1 || hp->settle_every < 0 || hp->settle_len < 0 || hp->clip < 0.0f)
    return fail(TTT_ERR_BAD_ARG, "bad hparams");
  if (hp->reset_every < 0 || (hp->reset_every > 0 && hp->settle_every > 0))
    return fail(TTT_ERR_BAD_ARG, "reset_every must be >= 0 and is not combined with settle_every");
  if (hp->settle_every > 0 && hp->settle_len < 2)
    return fail(TTT_ERR_BAD_ARG, "settle_len must be >= 2 when settle_every > 0");
  if (D.block_kind == TTT_BLOCK_GELU && D.fast_mask != (TTT_FAST_W1 | TTT_FAST_W2))
    return fail(TTT_ERR_UNSUPPORTED, "GELU blocks run with both W1 and W2 fast (fast_mask 3)");
  if (D.block_kind == TTT_BLOCK_SWIGLU && (D.fast_mask != TTT_FAST_WD || D.n_fast != 1))
    return fail(TTT_ERR_UNSUPPORTED, "SwiGLU runs with one fast block whose down projection is fast");
  if (D.static_mlp != 0 && D.static_mlp != 1) return fail(TTT_ERR_BAD_ARG, "static_mlp must be 0 or 1");
  if (D.attn_heads < 0 || D.attn_window < 0 || (D.attn_heads > 0 && (D.n_prefix < 1 || D.attn_window < 1)))
    return fail(TTT_ERR_BAD_ARG, "attention needs n_prefix >= 1 and attn_window >= 1");
  if (D.attn_heads > 0 && !swa_supported(D.d, D.attn_heads))
    return fail(TTT_ERR_UNSUPPORTED, "attention needs d % attn_heads == 0 and d / attn_heads <= 128");
  if (D.attn_heads > 0 && hp->settle_every > 0)
    return fail(TTT_ERR_UNSUPPORTED, "Settlement with attention is not built");
  if (D.attn_heads > 0 && !w->attn) return fail(TTT_ERR_BAD_ARG, "null attention weight pointer");
  if (D.static_mlp && D.block_kind != TTT_BLOCK_GELU)
    return fail(TTT_ERR_UNSUPPORTED, "static MLPs run in GELU fast blocks");
  if (!w->E || !w->U || (D.n_prefix > 0 && !w->prefix) || !w->fast || (D.static_mlp && !w->statics))
    return fail(TTT_ERR_BAD_ARG, "null weight pointer");

  ttt_handle* h = new ttt_handle();
  h->dm = D;
  h->hp = *hp;
  h->opt = O;
  h->B = hp->max_batch; h->b = hp->chunk; h->d = D.d; h->f = D.d_ff; h->V = D.vocab;
  h->nm = D.block_kind == TTT_BLOCK_GELU ? 2 : 3;
  h->n = (long long)D.d * D.d_ff;
  h->dtype = D.dtype;
  // fp32-accurate workloads run their GEMMs on the tensor cores as bf16 hi/lo
  // pairs when every leading dimension suits TMA and the chunk fills a tile
  // row block; otherwise they stay in plain fp32 (SIMT GEMMs).
  const bool force_f32 = O.fp32_simt != 0;
  if (D.dtype == TTT_DTYPE_BF16)
    h->stg = ST_BF16;
  else if (!force_f32 && hp->chunk >= 64 && D.d % 8 == 0 && D.d_ff % 8 == 0 && D.vocab % 8 == 0 &&
           D.vocab <= ce_split_max_vocab())
    h->stg = ST_SPLIT;
  else
    h->stg = ST_F32;
  h->esz = h->stg == ST_F32 ? 4 : 2;
  h->slot_of.assign((size_t)D.n_fast * h->nm, -1);
  for (int l = 0; l < D.n_fast; ++l)
    for (int m = 0; m < h->nm; ++m) {
      const int bit = (D.block_kind == TTT_BLOCK_GELU) ? (1 << m) : (m == 0 ? 1 : (m == 1 ? 4 : 2));
      if (D.fast_mask & bit) h->slot_of[(size_t)l * h->nm + m] = h->nslots++;
    }

  auto bail = [&](ttt_status s) { ttt_destroy(h); return s; };
  const int B = h->B, d = h->d, f = h->f, V = h->V;
  const size_t es = h->esz;
  const bool split = h->stg == ST_SPLIT;
  cudaStream_t st = 0;
  // an operand buffer of `count` elements (two planes for ST_SPLIT)
  auto op_alloc = [&](OpBuf* b, size_t count) -> ttt_status {
    TTT_TRY(dalloc(h, &b->p, count * es * (split ? 2 : 1)));
    b->lo = split ? (long long)count : 0;
    return TTT_OK;
  };

  // ---- weights
  float* stage = nullptr;
  size_t big = (size_t)V * d > (size_t)h->n ? (size_t)V * d : (size_t)h->n;
  if ((size_t)d * d > big) big = (size_t)d * d;     // attention projections
  ttt_status s;
  if ((s = dalloc(h, &stage, big * 4)) != TTT_OK) return bail(s);
  auto upload = [&](const float* src, size_t count, const OpBuf& dst, int stg) -> ttt_status {
    if (!src) return fail(TTT_ERR_BAD_ARG, "null weight matrix");
    TTT_CUDA(cudaMemcpy(stage, src, count * 4, cudaMemcpyDefault));
    TTT_TRY(launch_cast(stg, (long long)count, stage, dst.p, dst.lo, st));
    TTT_CUDA(cudaStreamSynchronize(st));
    return TTT_OK;
  };
  {
    // E feeds only the embedding gather: bf16 for bf16 workloads, fp32 otherwise
    const int e_stg = h->stg == ST_BF16 ? ST_BF16 : ST_F32;
    OpBuf eb;
    if ((s = dalloc(h, &eb.p, (size_t)V * d * (e_stg == ST_BF16 ? 2 : 4))) != TTT_OK) return bail(s);
    if ((s = upload(w->E, (size_t)V * d, eb, e_stg)) != TTT_OK) return bail(s);
    h->E = eb.p;
  }
  if ((s = op_alloc(&h->U, (size_t)V * d)) != TTT_OK) return bail(s);
  if ((s = upload(w->U, (size_t)V * d, h->U, h->stg)) != TTT_OK) return bail(s);
  // fast block 0's static MLP depends on no fast weight: it runs as one more prefix block
  h->n_pre = D.n_prefix + (D.static_mlp ? 1 : 0);
  h->prefix.assign((size_t)h->n_pre * h->nm, OpBuf());
  for (size_t i = 0; i < h->prefix.size(); ++i) {
    const float* src = i < (size_t)D.n_prefix * h->nm ? w->prefix[i] : w->statics[i - (size_t)D.n_prefix * h->nm];
    if ((s = op_alloc(&h->prefix[i], (size_t)h->n)) != TTT_OK) return bail(s);
    if ((s = upload(src, (size_t)h->n, h->prefix[i], h->stg)) != TTT_OK) return bail(s);
  }
  if (D.attn_heads > 0) {
    const size_t dd = (size_t)d * d;
    h->attn_qkv.assign(D.n_prefix, OpBuf());
    h->attn_o.assign(D.n_prefix, OpBuf());
    for (int p = 0; p < D.n_prefix; ++p) {
      if ((s = op_alloc(&h->attn_qkv[p], 3 * dd)) != TTT_OK) return bail(s);
      for (int j = 0; j < 3; ++j)
        if ((s = upload(w->attn[(size_t)p * 4 + j], dd, op_at(h, h->attn_qkv[p], (long long)(j * dd)), h->stg)) !=
            TTT_OK)
          return bail(s);
      if ((s = op_alloc(&h->attn_o[p], dd)) != TTT_OK) return bail(s);
      if ((s = upload(w->attn[(size_t)p * 4 + 3], dd, h->attn_o[p], h->stg)) != TTT_OK) return bail(s);
    }
  }
  if (D.static_mlp) {
    h->statics.assign((size_t)D.n_fast * h->nm, OpBuf());
    for (size_t i = (size_t)h->nm; i < h->statics.size(); ++i) {
      if ((s = op_alloc(&h->statics[i], (size_t)h->n)) != TTT_OK) return bail(s);
      if ((s = upload(w->statics[i], (size_t)h->n, h->statics[i], h->stg)) != TTT_OK) return bail(s);
    }
  }
  h->fastfrozen.assign((size_t)D.n_fast * h->nm, OpBuf());
  if ((s = dalloc(h, &h->W0, (size_t)h->nslots * h->n * 4)) != TTT_OK) return bail(s);
  for (size_t i = 0; i < h->fastfrozen.size(); ++i) {
    const int slot = h->slot_of[i];
    if (slot >= 0) {
      if (!w->fast[i]) return bail(fail(TTT_ERR_BAD_ARG, "null fast weight matrix"));
      cudaError_t e = cudaMemcpy(h->W0 + (size_t)slot * h->n, w->fast[i], (size_t)h->n * 4, cudaMemcpyDefault);
      if (e != cudaSuccess) return bail(cuda_fail(e, "upload W0", __FILE__, __LINE__));
    } else {
      if ((s = op_alloc(&h->fastfrozen[i], (size_t)h->n)) != TTT_OK) return bail(s);
      if ((s = upload(w->fast[i], (size_t)h->n, h->fastfrozen[i], h->stg)) != TTT_OK) return bail(s);
    }
  }
  const size_t arena = (size_t)h->nslots * B * h->n;
  if ((s = dalloc(h, &h->W32, arena * 4)) != TTT_OK) return bail(s);
  if ((s = op_alloc(&h->Wop, arena)) != TTT_OK) return bail(s);
  h->dw_esz = h->stg == ST_BF16 ? 2 : 4;
  if ((s = dalloc(h, &h->dW, arena * h->dw_esz)) != TTT_OK) return bail(s);
  // the committed copy serves Settlement (prefill events and ttt_settle)
  if ((s = dalloc(h, &h->Wc32, arena * 4)) != TTT_OK) return bail(s);
  if ((s = op_alloc(&h->Wcop, arena)) != TTT_OK) return bail(s);
  // the candidate's bf16 offset for Settlement's score, when its fast-weight
  // GEMMs fit the tensor-core kernel (every row block and width >= 64, widths
  // multiples of 8); otherwise the candidate is scored from its own bf16 copy
  if (h->stg == ST_BF16 && hp->settle_len >= 64 && D.d >= 64 && D.d_ff >= 64 && D.d % 8 == 0 && D.d_ff % 8 == 0)
    if ((s = op_alloc(&h->Wdel, arena)) != TTT_OK) return bail(s);

  // ---- workspace
  int rows_max = h->b;
  if (hp->settle_len > rows_max) rows_max = hp->settle_len;
  if (rows_max < 2) rows_max = 2;
  h->Mmax = B * rows_max;
  const size_t Mm = (size_t)h->Mmax;
  if ((s = dalloc(h, &h->x32, Mm * d * 4)) != TTT_OK) return bail(s);
  if ((s = op_alloc(&h->xop, Mm * d)) != TTT_OK) return bail(s);
  h->hlvl.assign(D.n_fast, OpBuf());
  h->zst.assign(D.n_fast, OpBuf());
  h->ast.assign(D.n_fast, OpBuf());
  for (int l = 0; l < D.n_fast; ++l) {
    if ((s = op_alloc(&h->hlvl[l], Mm * d)) != TTT_OK) return bail(s);
    if (D.block_kind == TTT_BLOCK_GELU)
      if ((s = op_alloc(&h->zst[l], Mm * f)) != TTT_OK) return bail(s);
    if ((s = op_alloc(&h->ast[l], Mm * f)) != TTT_OK) return bail(s);
  }
  h->szst.assign(D.n_fast, OpBuf());
  h->shin.assign(D.n_fast, OpBuf());
  for (int l = 1; l < D.n_fast && D.static_mlp; ++l) {
    if ((s = op_alloc(&h->szst[l], Mm * f)) != TTT_OK) return bail(s);
    if ((s = op_alloc(&h->shin[l], Mm * d)) != TTT_OK) return bail(s);
  }
  if ((s = op_alloc(&h->tmp_a, Mm * f)) != TTT_OK) return bail(s);
  // Settlement chunk q: its prefix output, shared by the event's two forwards
  if (hp->settle_len > 0) {
    const size_t Mq = (size_t)B * hp->settle_len;
    if ((s = dalloc(h, &h->qx32, Mq * d * 4)) != TTT_OK) return bail(s);
    if ((s = op_alloc(&h->qx_op, Mq * d)) != TTT_OK) return bail(s);
    if (D.block_kind == TTT_BLOCK_SWIGLU)
      if ((s = op_alloc(&h->qa, Mq * f)) != TTT_OK) return bail(s);
  }
  // hoisted prefix: groups of up to hoist_chunks chunks, within a 4 GiB budget
  {
    const size_t P = split ? 2 : 1;
    size_t per_row = (size_t)d * 4 + (size_t)d * es * P + (h->n_pre > 0 ? (size_t)d * es * P : 0) +
                     (size_t)f * es * P;
    if (D.block_kind == TTT_BLOCK_SWIGLU) per_row += (size_t)f * 4 + (size_t)f * es * P;
    const size_t per_chunk = per_row * (size_t)B * h->b;
    long long gmax = (long long)((4ull << 30) / per_chunk);
    if (gmax > 64) gmax = 64;
    // the option caps the group (tests use it to cross group boundaries)
    if (O.hoist_chunks > 0 && O.hoist_chunks < gmax) gmax = O.hoist_chunks;
    if (gmax < 1) gmax = 1;
    h->hoist_chunks = (int)gmax;
    const size_t Mh = (size_t)B * h->b * gmax;
    if ((s = dalloc(h, &h->hx32, Mh * d * 4)) != TTT_OK) return bail(s);
    if ((s = op_alloc(&h->hx_op, Mh * d)) != TTT_OK) return bail(s);
    if (h->n_pre > 0)
      if ((s = op_alloc(&h->hx_xop, Mh * d)) != TTT_OK) return bail(s);
    if ((s = op_alloc(&h->hx_tmp_a, Mh * f)) != TTT_OK) return bail(s);
    if (D.block_kind == TTT_BLOCK_SWIGLU) {
      if ((s = dalloc(h, &h->hx_tmp_g, Mh * f * 4)) != TTT_OK) return bail(s);
      if ((s = op_alloc(&h->ha, Mh * f)) != TTT_OK) return bail(s);
    }
  }
  if (D.block_kind == TTT_BLOCK_SWIGLU)
    if ((s = dalloc(h, &h->tmp_g, Mm * f * 4)) != TTT_OK) return bail(s);
  if ((s = op_alloc(&h->y, Mm * d)) != TTT_OK) return bail(s);
  if ((s = dalloc(h, &h->rstd, Mm * 4)) != TTT_OK) return bail(s);
  if ((s = dalloc(h, &h->logits, Mm * V * (split ? 4 : es))) != TTT_OK) return bail(s);
  if ((s = dalloc(h, &h->row_loss, Mm * 4)) != TTT_OK) return bail(s);
  if ((s = dalloc(h, &h->rscale, Mm * 4)) != TTT_OK) return bail(s);
  // fused cross-entropy state: one online-softmax pair per row and head column tile
  h->lse_ld = ceil_div(V, 128);  // the narrowest tensor-core tile
  if ((s = dalloc(h, &h->lse_part, Mm * (size_t)h->lse_ld * sizeof(float2))) != TTT_OK) return bail(s);
  if ((s = dalloc(h, &h->lse, Mm * 4)) != TTT_OK) return bail(s);
  if ((s = dalloc(h, &h->tgt, Mm * 4)) != TTT_OK) return bail(s);
  if ((s = dalloc(h, &h->dy32, Mm * d * 4)) != TTT_OK) return bail(s);
  if ((s = dalloc(h, &h->dh32, Mm * d * 4)) != TTT_OK) return bail(s);
  if ((s = op_alloc(&h->dhop, Mm * d)) != TTT_OK) return bail(s);
  if (D.block_kind == TTT_BLOCK_GELU && !D.static_mlp && !O.no_dw_stream) {
    if ((s = op_alloc(&h->dhop2, Mm * d)) != TTT_OK) return bail(s);
    cudaError_t ce = cudaStreamCreateWithFlags(&h->bstream, cudaStreamNonBlocking);
    if (ce != cudaSuccess) {
      h->bstream = nullptr;
      return bail(cuda_fail(ce, "cudaStreamCreateWithFlags", __FILE__, __LINE__));
    }
    h->bev.assign((size_t)3 * D.n_fast + 1, nullptr);
    for (auto& e : h->bev)
      if ((ce = cudaEventCreateWithFlags(&e, cudaEventDisableTiming)) != cudaSuccess) {
        e = nullptr;
        return bail(cuda_fail(ce, "cudaEventCreateWithFlags", __FILE__, __LINE__));
      }
  }
  // split-K workspace: up to 8 fp32 partial slices of a [Mmax, d] output, at most 64 MB
  // split-K partial tiles (fp32): the planner splits only while they fit (256 MB)
  h->gemm_ws_elems = 64LL << 20;
  if ((s = dalloc(h, &h->gemm_ws, (size_t)h->gemm_ws_elems * 4)) != TTT_OK) return bail(s);
  if ((s = dalloc(h, &h->split_cnt, (size_t)gemm_tc_max_split_tiles() * 4)) != TTT_OK) return bail(s);
  if (cudaMemset(h->split_cnt, 0, (size_t)gemm_tc_max_split_tiles() * 4) != cudaSuccess)
    return bail(fail(TTT_ERR_CUDA, "cudaMemset of the split-K counters failed"));
  // partial sums of squares: at most one per 64x64 output tile per matrix and sequence
  h->partial_cap = (long long)h->nslots * B * ceil_div(d, 64) * ceil_div(f, 64);
  if ((s = dalloc(h, &h->partials, (size_t)h->partial_cap * 4)) != TTT_OK) return bail(s);
  if ((s = dalloc(h, &h->scale, (size_t)B * 4)) != TTT_OK) return bail(s);
  if ((s = dalloc(h, &h->gnorm, (size_t)B * 4)) != TTT_OK) return bail(s);
  if ((s = dalloc(h, &h->flag, 4)) != TTT_OK) return bail(s);
  if (cudaMallocHost(&h->flag_host, 4) != cudaSuccess) {
    cudaGetLastError();
    return bail(fail(TTT_ERR_OOM, "cudaMallocHost"));
  }
  if ((s = dalloc(h, &h->logits32, (size_t)B * V * 4)) != TTT_OK) return bail(s);
  if ((s = dalloc(h, &h->p_dev, (size_t)B * V * 4)) != TTT_OK) return bail(s);
  if ((s = dalloc(h, &h->lse_next, (size_t)B * 4)) != TTT_OK) return bail(s);
  if ((s = dalloc(h, &h->soft_part, (size_t)B * kSoftmaxMaxSlices * sizeof(float2))) != TTT_OK) return bail(s);
  if ((s = dalloc(h, &h->Lc, (size_t)B * 4)) != TTT_OK) return bail(s);
  if ((s = dalloc(h, &h->Lw, (size_t)B * 4)) != TTT_OK) return bail(s);
  if ((s = dalloc(h, &h->pend, (size_t)B * (h->b + 1) * 4)) != TTT_OK) return bail(s);
  if ((s = dalloc(h, &h->x_dev, (size_t)B * 4)) != TTT_OK) return bail(s);
  if (D.attn_heads > 0) {
    // decoding with attention: the K/V cache of every frozen block, the one-row
    // prefix pass and the pending inputs' prefix rows
    const size_t kw = (size_t)D.attn_window;
    if ((s = dalloc(h, &h->kv, (size_t)D.n_prefix * 2 * B * kw * d * 4)) != TTT_OK) return bail(s);
    if ((s = dalloc(h, &h->dec_pos, 4)) != TTT_OK) return bail(s);
    if ((s = dalloc(h, &h->dec_x32, (size_t)B * d * 4)) != TTT_OK) return bail(s);
    if ((s = dalloc(h, &h->dec_qkv, (size_t)B * 3 * d * 4)) != TTT_OK) return bail(s);
    if ((s = dalloc(h, &h->dec_work, swa_decode_work_floats(B, D.attn_heads) * 4)) != TTT_OK) return bail(s);
    if ((s = dalloc(h, &h->dec_cnt, (size_t)B * D.attn_heads * 4)) != TTT_OK) return bail(s);
    if (cudaMemset(h->dec_cnt, 0, (size_t)B * D.attn_heads * 4) != cudaSuccess) {
      cudaGetLastError();
      return bail(fail(TTT_ERR_CUDA, "cudaMemset of the decoding attention counters failed"));
    }
    if ((s = op_alloc(&h->dec_op, (size_t)B * d)) != TTT_OK) return bail(s);
    if ((s = op_alloc(&h->dec_xop, (size_t)B * d)) != TTT_OK) return bail(s);
    if ((s = op_alloc(&h->dec_att, (size_t)B * d)) != TTT_OK) return bail(s);
    if ((s = op_alloc(&h->dec_tmp_a, (size_t)B * f)) != TTT_OK) return bail(s);
    const size_t pr = (size_t)B * (h->b + 1);
    if ((s = dalloc(h, &h->prow32, pr * d * 4)) != TTT_OK) return bail(s);
    if ((s = op_alloc(&h->prow_op, pr * d)) != TTT_OK) return bail(s);
    if (D.block_kind == TTT_BLOCK_SWIGLU) {
      if ((s = dalloc(h, &h->dec_tmp_g, (size_t)B * f * 4)) != TTT_OK) return bail(s);
      if ((s = op_alloc(&h->dec_a, (size_t)B * f)) != TTT_OK) return bail(s);
      if ((s = op_alloc(&h->prow_a, pr * f)) != TTT_OK) return bail(s);
    }
  }
  if ((s = reset_weights(h, st)) != TTT_OK) return bail(s);
  cudaError_t e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return bail(cuda_fail(e, "create sync", __FILE__, __LINE__));
  // the weight staging buffer is no longer needed
  for (auto& a : h->allocs)
    if (a == stage) a = nullptr;
  cudaFree(stage);
  h->launches = 0;
  *out = h;
  return TTT_OK;
}

ttt_status ttt_prefill(ttt_handle* h, const int32_t* tokens, int B, int T, float* losses, float* p_next,
                       const int32_t* settle_q, int Lq, uint8_t* accept, float* A, ttt_stream stream) {
  return ttt_prefill_masked(h, tokens, nullptr, B, T, losses, p_next, settle_q, Lq, accept, A, stream);
}

ttt_status ttt_prefill_masked(ttt_handle* h, const int32_t* tokens, const uint8_t* loss_mask, int B, int T,
                              float* losses, float* p_next, const int32_t* settle_q, int Lq, uint8_t* accept,
                              float* A, ttt_stream stream) {
  if (!h || !tokens || !losses) return fail(TTT_ERR_BAD_ARG, "null argument to ttt_prefill");
  if (B != h->B || T < 1) return fail(TTT_ERR_BAD_SHAPE, "B must equal max_batch and T >= 1");
  PdlScope pdl(!h->opt.no_pdl);
  cudaStream_t st = (cudaStream_t)stream;
  const int b = h->b, n_full = T / b, rem = T % b;
  const int n_events = h->hp.settle_every > 0 ? n_full / h->hp.settle_every : 0;
  if (n_events > 0) {
    if (!settle_q) return fail(TTT_ERR_BAD_ARG, "settle_q is required when Settlement events occur");
    if (Lq != h->hp.settle_len) return fail(TTT_ERR_BAD_SHAPE, "Lq must equal settle_len");
  }
  h->launches = 0;

  const int32_t* tok = nullptr;
  TTT_TRY(copy_in(h, tokens, (void**)&h->tok_dev, &h->tok_cap, (size_t)B * (T + 1) * 4, (const void**)&tok, st));
  const uint8_t* mask = nullptr;
  if (loss_mask)
    TTT_TRY(copy_in(h, loss_mask, (void**)&h->mask_dev, &h->mask_cap, (size_t)B * T, (const void**)&mask, st));
  const int32_t* q = nullptr;
  if (n_events > 0)
    TTT_TRY(copy_in(h, settle_q, (void**)&h->q_dev, &h->q_cap, (size_t)n_events * B * Lq * 4,
                    (const void**)&q, st));
  const bool loss_host = !is_device_ptr(losses);
  float* loss_d = losses;
  if (loss_host) {
    TTT_TRY(ensure_staging(h, (void**)&h->loss_dev, &h->loss_cap, (size_t)B * T * 4));
    loss_d = h->loss_dev;
  }
  if (n_events > 0) {
    TTT_TRY(ensure_staging(h, (void**)&h->A_dev, &h->A_cap, (size_t)n_events * B * 4));
    TTT_TRY(ensure_staging(h, (void**)&h->acc_dev, &h->acc_cap, (size_t)n_events * B));
  }

  TTT_TRY(reset_weights(h, st));
  h->next_valid = false;
  TTT_CUDA(cudaMemsetAsync(h->flag, 0, 4, st));
  // b = 1 on a network whose fast block and head fit in shared memory: one
  // persistent CTA per sequence steps through every token
  const bool token_path = b == 1 && h->n_pre == 0 && h->dm.n_fast == 1 &&
                          h->dm.block_kind == TTT_BLOCK_GELU && h->stg == ST_F32 && h->hp.settle_every == 0 &&
                          h->hp.reset_every == 0 &&
                          token_steps_supported(h->d, h->f, h->V) && !h->opt.no_token_kernel;
  const bool attn = h->dm.attn_heads > 0;
  Hoisted hz_all;     // attention: the prefix of x_0 .. x_T of every sequence, one pass
  if (attn) {
    const long long R = (long long)T + 1;
    TTT_TRY(ensure_attn_rows(h, (size_t)B * R));
    if (h->stg != ST_F32) TTT_TRY(ensure_attn_tc(h, R));
    TokView tv;
    tv.tok = tok; tv.tok_ld = T + 1; tv.tok_off = 0; tv.rows = (int)R; tv.n_valid = (int)R;
    tv.vocab = h->V;
    tv.err = h->flag;
    PrefixBufs pb;
    pb.x32 = h->ax32; pb.xop = h->ax_xop; pb.hout = h->ax_op; pb.tmp_a = h->ax_tmp_a; pb.tmp_g = h->ax_tmp_g;
    pb.swiglu_a = h->ax_a;
    pb.attn = true;
    TTT_TRY(prefix_pass(h, tv, pb, st));
    hz_all.on = true; hz_all.rows_total = R;
    hz_all.x32 = h->ax32; hz_all.op = h->ax_op; hz_all.a = h->ax_a;
    for (int i = 0; i < n_full; ++i) {
      TokView tc;
      tc.tok = tok; tc.tok_ld = T + 1; tc.tok_off = (long long)i * b; tc.rows = b; tc.n_valid = b;
      Hoisted hz = hz_all;
      hz.row0 = (long long)i * b;
      TTT_TRY(chunk_step(h, tc, loss_d, T, (long long)i * b, st, hz, mask, T));
    }
  }
  if (token_path && n_full > 0 && !attn) {
    TTT_TRY(run(h, K_TOKEN, st, 1, [&] {
      return launch_token_steps(B, tok, T + 1, n_full, mask, T, static_cast<const float*>(h->E),
                                static_cast<const float*>(h->U.p), h->W32, static_cast<float*>(h->Wop.p),
                                h->slot_of[0], h->slot_of[1], loss_d, T, h->d, h->f, h->V, h->dm.rms_eps,
                                h->hp.eta, h->hp.clip, h->flag, st);
    }));
    h->chunks_done += n_full;
  }
  // chunks in groups whose frozen prefix runs as one pass before the group's TTT steps
  const int G = h->hoist_chunks;

  for (int i0 = (token_path || attn) ? n_full : 0; i0 < n_full; i0 += G) {
    const int g = n_full - i0 < G ? n_full - i0 : G;
    TTT_TRY(hoisted_prefix(h, tok, T + 1, i0, g, st));
    for (int i = i0; i < i0 + g; ++i) {
      TokView tv;
      tv.tok = tok; tv.tok_ld = T + 1; tv.tok_off = (long long)i * b; tv.rows = b; tv.n_valid = b;
      Hoisted hz;
      hz.on = true; hz.row0 = (long long)(i - i0) * b; hz.rows_total = (long long)g * b;
      hz.x32 = h->hx32; hz.op = h->hx_op; hz.a = h->ha;
      TTT_TRY(chunk_step(h, tv, loss_d, T, (long long)i * b, st, hz, mask, T));
      if (h->hp.settle_every > 0 && (i + 1) % h->hp.settle_every == 0) {
        const int e = (i + 1) / h->hp.settle_every - 1;
        TTT_TRY(settle_event(h, q + (size_t)e * B * Lq, Lq, h->A_dev + (size_t)e * B, h->acc_dev + (size_t)e * B,
                             st));
      }
    }
  }
  if (rem > 0) {   // the tail is scored only (and, as decoding, never masked)
    TokView tv;
    tv.tok = tok; tv.tok_ld = T + 1; tv.tok_off = (long long)n_full * b; tv.rows = rem; tv.n_valid = rem;
    Hoisted hz = hz_all;
    hz.row0 = (long long)n_full * b;
    TTT_TRY(forward(h, tv, false, false, loss_d, T, (long long)n_full * b, false, st, hz));
  }
  // pending decode buffer: tokens x_{n_full b} .. x_T
  TTT_CUDA(cudaMemcpy2DAsync(h->pend, (size_t)(b + 1) * 4, tok + (size_t)n_full * b, (size_t)(T + 1) * 4,
                             (size_t)(rem + 1) * 4, B, cudaMemcpyDeviceToDevice, st));
  if (attn) {
    // decoding goes on from here: the prefix rows of x_{n_full b} .. x_T, and x_T's position
    TTT_TRY(save_pending_rows(h, h->ax32, h->ax_op, h->ax_a, (long long)T + 1, (long long)n_full * b, 0, rem + 1, st));
    TTT_TRY(run(h, K_OTHER, st, 1, [&] { return launch_pos_set(h->dec_pos, T, st); }));
    h->attn_ctx = true;
  }
  h->pend_count = rem;
  h->has_context = true;
  if (p_next) {
    const bool dev = is_device_ptr(p_next);
    Hoisted hz = hz_all;       // attention: x_T's prefix row from the whole-sequence pass
    hz.row0 = T;
    TTT_TRY(p_next_from_pending(h, dev ? p_next : h->p_dev, st, hz));
    if (!dev) TTT_CUDA(cudaMemcpyAsync(p_next, h->p_dev, (size_t)B * h->V * 4, cudaMemcpyDeviceToHost, st));
  }
  if (loss_host) TTT_CUDA(cudaMemcpyAsync(losses, loss_d, (size_t)B * T * 4, cudaMemcpyDeviceToHost, st));
  if (n_events > 0 && A) TTT_CUDA(cudaMemcpyAsync(A, h->A_dev, (size_t)n_events * B * 4, cudaMemcpyDefault, st));
  if (n_events > 0 && accept)
    TTT_CUDA(cudaMemcpyAsync(accept, h->acc_dev, (size_t)n_events * B, cudaMemcpyDefault, st));
  return finish(h, st);
}

ttt_status ttt_decode_step(ttt_handle* h, const int32_t* x_new, float* p_next, float* loss, ttt_stream stream) {
  if (!h || !x_new || !p_next) return fail(TTT_ERR_BAD_ARG, "null argument to ttt_decode_step");
  if (!h->has_context) return fail(TTT_ERR_STATE, "decode before prefill");
  PdlScope pdl(!h->opt.no_pdl);
  const bool attn = h->dm.attn_heads > 0;
  if (attn && !h->attn_ctx) return fail(TTT_ERR_STATE, "decoding with attention needs a prefill first");
  if (attn && swa_decode_smem_bytes(h->dm.attn_window, h->d / h->dm.attn_heads) > 227 * 1024)
    return fail(TTT_ERR_UNSUPPORTED, "attention window too long for decoding");
  cudaStream_t st = (cudaStream_t)stream;
  const int B = h->B, b = h->b;
  // attention: the pending inputs' prefix rows (row j = input pend[j])
  Hoisted hp;
  if (attn) {
    hp.on = true; hp.rows_total = b + 1;
    hp.x32 = h->prow32; hp.op = h->prow_op; hp.a = h->prow_a;
  }
  h->launches = 0;
  // x_new -> pend[s][pend_count + 1] (and, for the persistent forward, its
  // token slot), the status word cleared
  const bool x_dev_ptr = is_device_ptr(x_new);
  const bool persist = decode_persist_applies(h);
  const bool one_launch_in = x_dev_ptr;   // the inputs (and the loss) in one kernel
  // the loss of (x_prev -> x_new) from the cached distribution, in the same launch
  const bool loss_dev = loss && is_device_ptr(loss);
  float* loss_dst = loss ? (loss_dev ? loss : h->Lc) : nullptr;
  const bool loss_in = one_launch_in && loss && h->next_valid;
  if (one_launch_in) {
    if (persist) TTT_TRY(decode_persist_setup(h));
    TTT_TRY(run(h, K_OTHER, st, 1, [&] {
      return launch_decode_inputs(B, b + 1, h->pend_count + 1, x_new, h->pend, h->x_dev, h->flag,
                                  persist ? h->dp_bar : nullptr, h->V, h->logits32, h->lse_next,
                                  loss_in ? loss_dst : nullptr, st);
    }));
  } else {
    TTT_CUDA(cudaMemcpy2DAsync(h->pend + h->pend_count + 1, (size_t)(b + 1) * 4, x_new, 4, 4, B,
                               x_dev_ptr ? cudaMemcpyDeviceToDevice : cudaMemcpyHostToDevice, st));
    TTT_CUDA(cudaMemsetAsync(h->flag, 0, 4, st));
  }
  // loss of (x_prev -> x_new) with the weights that score it: the previous
  // step's (or the prefill's) next-token softmax already holds them
  if (loss) {
    const bool dev = loss_dev;
    float* dst = loss_dst;
    if (loss_in) {
      // scored by the inputs kernel above
    } else if (h->next_valid) {
      TTT_TRY(run(h, K_OTHER, st, 1, [&] {
        return launch_next_token_loss(B, h->V, h->logits32, h->lse_next, h->pend, b + 1, h->pend_count + 1, dst,
                                      h->flag, st);
      }));
    } else {
      TokView tv;
      tv.tok = h->pend; tv.tok_ld = b + 1; tv.tok_off = h->pend_count; tv.rows = 1; tv.n_valid = 1;
      Hoisted hz = hp;
      hz.row0 = h->pend_count;
      TTT_TRY(forward(h, tv, false, false, dst, 1, 0, false, st, hz));
    }
    if (!dev) TTT_CUDA(cudaMemcpyAsync(loss, dst, (size_t)B * 4, cudaMemcpyDeviceToHost, st));
  }
  h->pend_count++;
  if (h->pend_count == b) {
    TokView tv;
    tv.tok = h->pend; tv.tok_ld = b + 1; tv.tok_off = 0; tv.rows = b; tv.n_valid = b;
    Hoisted hz = hp;
    hz.row0 = 0;
    TTT_TRY(chunk_step(h, tv, nullptr, 0, 0, st, hz));
    TTT_TRY(run(h, K_OTHER, st, 1, [&] { return launch_pending_shift(B, b, h->pend, st); }));
    h->pend_count = 0;
  }
  // attention: x_new's position (the decoding attention appends its K and V there)
  if (attn) TTT_TRY(run(h, K_OTHER, st, 1, [&] { return launch_pos_add(h->dec_pos, st); }));
  const bool dev = is_device_ptr(p_next);
  if (persist) {
    if (!one_launch_in)
      TTT_CUDA(cudaMemcpyAsync(h->x_dev, x_new, (size_t)B * 4, cudaMemcpyHostToDevice, st));
    TTT_TRY(decode_persist(h, dev ? p_next : h->p_dev, !one_launch_in, st));
    if (!dev) TTT_CUDA(cudaMemcpyAsync(p_next, h->p_dev, (size_t)B * h->V * 4, cudaMemcpyDeviceToHost, st));
  } else if (!h->opt.no_decode_graph) {
    // the newest token into the fixed slot the captured forward reads (the
    // inputs kernel put it there already for a device x_new)
    if (!one_launch_in) TTT_CUDA(cudaMemcpyAsync(h->x_dev, x_new, (size_t)B * 4, cudaMemcpyHostToDevice, st));
    TTT_TRY(decode_forward_graph(h, st));
    TTT_CUDA(cudaMemcpyAsync(p_next, h->p_dev, (size_t)B * h->V * 4,
                             dev ? cudaMemcpyDeviceToDevice : cudaMemcpyDeviceToHost, st));
  } else {
    TTT_TRY(p_next_from_pending(h, dev ? p_next : h->p_dev, st));
    if (!dev) TTT_CUDA(cudaMemcpyAsync(p_next, h->p_dev, (size_t)B * h->V * 4, cudaMemcpyDeviceToHost, st));
  }
  // attention: x_new's prefix row is the pending row of input pend[pend_count]
  if (attn) TTT_TRY(save_pending_rows(h, h->dec_x32, h->dec_op, h->dec_a, 1, 0, h->pend_count, 1, st));
  return finish(h, st);
}

ttt_status ttt_settle(ttt_handle* h, const int32_t* q, int Lq, uint8_t* accept, float* A, ttt_stream stream) {
  if (!h || !q || !accept || !A) return fail(TTT_ERR_BAD_ARG, "null argument to ttt_settle");
  if (Lq != h->hp.settle_len || Lq < 2) return fail(TTT_ERR_BAD_SHAPE, "Lq must equal settle_len (>= 2)");
  if (h->dm.attn_heads > 0) return fail(TTT_ERR_UNSUPPORTED, "Settlement with attention is not built");
  PdlScope pdl(!h->opt.no_pdl);
  cudaStream_t st = (cudaStream_t)stream;
  const int B = h->B;
  h->launches = 0;
  const int32_t* qd = nullptr;
  TTT_TRY(copy_in(h, q, (void**)&h->q_dev, &h->q_cap, (size_t)B * Lq * 4, (const void**)&qd, st));
  h->next_valid = false;   // a revert changes the weights that scored the cached softmax
  TTT_TRY(ensure_staging(h, (void**)&h->A_dev, &h->A_cap, (size_t)B * 4));
  TTT_TRY(ensure_staging(h, (void**)&h->acc_dev, &h->acc_cap, (size_t)B));
  TTT_CUDA(cudaMemsetAsync(h->flag, 0, 4, st));
  TTT_TRY(settle_event(h, qd, Lq, h->A_dev, h->acc_dev, st));
  TTT_CUDA(cudaMemcpyAsync(A, h->A_dev, (size_t)B * 4, cudaMemcpyDefault, st));
  TTT_CUDA(cudaMemcpyAsync(accept, h->acc_dev, (size_t)B, cudaMemcpyDefault, st));
  return finish(h, st);
}

ttt_status ttt_get_fast_weights(ttt_handle* h, int seq, int block, int mat, float* dst, ttt_stream stream) {
  if (!h || !dst) return fail(TTT_ERR_BAD_ARG, "null argument");
  if (seq < 0 || seq >= h->B || block < 0 || block >= h->dm.n_fast || mat < 0 || mat >= h->nm)
    return fail(TTT_ERR_BAD_ARG, "index out of range");
  const int slot = h->slot_of[(size_t)block * h->nm + mat];
  if (slot < 0) return fail(TTT_ERR_BAD_ARG, "that matrix is not a fast weight");
  cudaStream_t st = (cudaStream_t)stream;
  TTT_CUDA(cudaMemcpyAsync(dst, h->W32 + ((size_t)slot * h->B + seq) * h->n, (size_t)h->n * 4,
                           cudaMemcpyDefault, st));
  TTT_CUDA(cudaStreamSynchronize(st));
  return TTT_OK;
}

ttt_status ttt_reset(ttt_handle* h, ttt_stream stream) {
  if (!h) return fail(TTT_ERR_BAD_ARG, "null handle");
  h->next_valid = false;
  PdlScope pdl(!h->opt.no_pdl);
  cudaStream_t st = (cudaStream_t)stream;
  TTT_TRY(reset_weights(h, st));
  h->has_context = false;
  h->attn_ctx = false;
  TTT_CUDA(cudaStreamSynchronize(st));
  return TTT_OK;
}

// ---- checkpoint blob: header, W32, Wc32, pending tokens
struct StateHeader {
  uint64_t magic;
  int32_t d, d_ff, vocab, n_fast, block_kind, fast_mask, dtype, B, b, nslots;
  int32_t pend_count, has_context;
  int64_t chunks_done;
};
static const uint64_t kStateMagic = 0x7474745354415445ULL;  // "tttSTATE"

ttt_status ttt_state_size(ttt_handle* h, size_t* bytes) {
  if (!h || !bytes) return fail(TTT_ERR_BAD_ARG, "null argument");
  const size_t arena = (size_t)h->nslots * h->B * h->n * 4;
  *bytes = sizeof(StateHeader) + 2 * arena + (size_t)h->B * (h->b + 1) * 4;
  return TTT_OK;
}

ttt_status ttt_get_state(ttt_handle* h, void* dst, size_t bytes, ttt_stream stream) {
  size_t need = 0;
  TTT_TRY(ttt_state_size(h, &need));
  if (!dst) return fail(TTT_ERR_BAD_ARG, "null dst");
  if (bytes != need) return fail(TTT_ERR_BAD_SHAPE, "state size mismatch");
  cudaStream_t st = (cudaStream_t)stream;
  StateHeader hd{kStateMagic, h->d, h->f, h->V, h->dm.n_fast, h->dm.block_kind, h->dm.fast_mask, h->dtype,
                 h->B, h->b, h->nslots, h->pend_count, h->has_context ? 1 : 0, h->chunks_done};
  char* p = static_cast<char*>(dst);
  memcpy(p, &hd, sizeof hd);
  p += sizeof hd;
  const size_t arena = (size_t)h->nslots * h->B * h->n * 4;
  TTT_CUDA(cudaMemcpyAsync(p, h->W32, arena, cudaMemcpyDefault, st));
  TTT_CUDA(cudaMemcpyAsync(p + arena, h->Wc32, arena, cudaMemcpyDefault, st));
  TTT_CUDA(cudaMemcpyAsync(p + 2 * arena, h->pend, (size_t)h->B * (h->b + 1) * 4, cudaMemcpyDefault, st));
  TTT_CUDA(cudaStreamSynchronize(st));
  return TTT_OK;
}

ttt_status ttt_set_state(ttt_handle* h, const void* src, size_t bytes, ttt_stream stream) {
  size_t need = 0;
  TTT_TRY(ttt_state_size(h, &need));
  if (!src) return fail(TTT_ERR_BAD_ARG, "null src");
  if (bytes != need) return fail(TTT_ERR_BAD_SHAPE, "state size mismatch");
  StateHeader hd;
  memcpy(&hd, src, sizeof hd);
  if (hd.magic != kStateMagic || hd.d != h->d || hd.d_ff != h->f || hd.vocab != h->V ||
      hd.n_fast != h->dm.n_fast || hd.block_kind != h->dm.block_kind || hd.fast_mask != h->dm.fast_mask ||
      hd.dtype != h->dtype || hd.B != h->B || hd.b != h->b || hd.nslots != h->nslots ||
      hd.pend_count < 0 || hd.pend_count >= h->b)
    return fail(TTT_ERR_BAD_SHAPE, "state blob does not match this handle");
  PdlScope pdl(!h->opt.no_pdl);
  cudaStream_t st = (cudaStream_t)stream;
  h->next_valid = false;
  const char* p = static_cast<const char*>(src) + sizeof hd;
  const size_t arena = (size_t)h->nslots * h->B * h->n * 4;
  TTT_CUDA(cudaMemcpyAsync(h->W32, p, arena, cudaMemcpyDefault, st));
  TTT_CUDA(cudaMemcpyAsync(h->Wc32, p + arena, arena, cudaMemcpyDefault, st));
  TTT_CUDA(cudaMemcpyAsync(h->pend, p + 2 * arena, (size_t)h->B * (h->b + 1) * 4, cudaMemcpyDefault, st));
  const long long total = (long long)h->nslots * h->B * h->n;
  TTT_TRY(launch_cast(h->stg, total, h->W32, h->Wop.p, h->Wop.lo, st));
  TTT_TRY(launch_cast(h->stg, total, h->Wc32, h->Wcop.p, h->Wcop.lo, st));
  TTT_CUDA(cudaStreamSynchronize(st));
  h->pend_count = hd.pend_count;
  h->has_context = hd.has_context != 0;
  h->attn_ctx = false;     // the attention context (K/V cache, pending rows) is not part of the blob
  h->chunks_done = hd.chunks_done;
  return TTT_OK;
}

ttt_status ttt_profile_enable(ttt_handle* h, int kernel_class) {
  if (!h || kernel_class < -1 || kernel_class >= K_COUNT) return fail(TTT_ERR_BAD_ARG, "bad kernel class");
  h->prof_class = kernel_class;
  if (kernel_class >= 0 && h->ev.empty()) {
    h->ev.resize(8192);
    for (auto& e : h->ev) TTT_CUDA(cudaEventCreate(&e));
  }
  h->ev_used = 0;
  h->prof_launches = 0;
  return TTT_OK;
}

ttt_status ttt_profile_read(ttt_handle* h, int* launches, double* total_ms) {
  if (!h || !launches || !total_ms) return fail(TTT_ERR_BAD_ARG, "null argument");
  double tot = 0.0;
  for (int i = 0; i + 1 < h->ev_used; i += 2) {
    TTT_CUDA(cudaEventSynchronize(h->ev[i + 1]));
    float ms = 0.0f;
    TTT_CUDA(cudaEventElapsedTime(&ms, h->ev[i], h->ev[i + 1]));
    tot += ms;
  }
  *launches = h->prof_launches;
  *total_ms = tot;
  h->ev_used = 0;
  h->prof_launches = 0;
  return TTT_OK;
}

ttt_status ttt_launch_log_enable(ttt_handle* h, int on) {
  if (!h) return fail(TTT_ERR_BAD_ARG, "null handle");
  h->log_on = on != 0;
  h->launch_log.clear();
  return TTT_OK;
}

int ttt_launch_log_read(ttt_handle* h, int8_t* out, int cap) {
  if (!h) return -1;
  const int n = (int)h->launch_log.size();
  for (int i = 0; i < n && i < cap && out; ++i) out[i] = h->launch_log[(size_t)i];
  return n;
}

int ttt_operand_storage(ttt_handle* h) { return h ? h->stg : -1; }

ttt_status ttt_last_launch_count(ttt_handle* h, long long* launches) {
  if (!h || !launches) return fail(TTT_ERR_BAD_ARG, "null argument");
  *launches = h->launches;
  return TTT_OK;
}

}  // extern "C"
