// Per-token TTT (chunk b = 1) in one persistent CTA per sequence, for networks
// small enough that the fast block and the LM head live in one SM's shared
// memory for the whole stream.
//
// "End-to-End Test-Time Training for Long Context" review, eq. (2): for every
// token t, l_t(W_{t-1}) is scored, then W_t = W_{t-1} - eta * grad l_t(W_{t-1});
// with b = 1 each step is eq. (5) for a one-token chunk.  Network (no frozen
// prefix, one residual GELU block with both matrices fast, final RMSNorm with a
// unit gain, LM head U):
//   h = E[x];  z = W1 h;  a = GELU(z);  h2 = h + W2 a;  y = h2 / rms(h2);
//   logits = U y;  l = logsumexp(logits) - logits[target].
// Backward for one token: dlogits = softmax - onehot;  dy = U^T dlogits;
// dh2 = rstd (dy - y mean(y dy));  dW2 = dh2 a^T;  da = W2^T dh2;
// dz = da GELU'(z);  dW1 = dz h^T.  Both gradients are outer products, so the
// global norm is exact in closed form, ||dW2||^2 + ||dW1||^2 =
// |dh2|^2 |a|^2 + |dz|^2 |h|^2, and the clipped step s = min(1, c / (norm +
// 1e-6)) ("Self-Generated Feedback Destabilizes TTT" summary: one clipped step
// per chunk) is applied to the shared-memory copies without forming dW.
//
// With a loss mask, a masked token is scored but takes no step (Source
// Masking: its chunk of one target has no unmasked target).
//
// Shared memory (fp32): W1 [f][d+1], W2 [d][f+1], U [V][d+1] (the +1 pads keep
// row-wise and column-wise walks free of most bank conflicts) and the token's
// vectors.  The fp32 masters are read from the arena at the start and written
// back (masters and operand copy) at the end.
#include <cfloat>

#include "kernels.h"

namespace ttt {
namespace {

constexpr int kTokThreads = 512;
// reduction scratch: 32 floats for block sums, then the column partials of
// coldot (up to blockDim floats) or four floats per warp for tok_sum4
constexpr int kRed = 32 + kTokThreads;

struct TokenArgs {
  const int32_t* tok;
  long long tok_ld;
  int T;
  const uint8_t* mask;  // [B][mask_ld] or null: target t+1 enters the update iff mask[t]
  long long mask_ld;
  const float* E;       // [V][d]
  const float* U;       // [V][d]
  float* W32;           // arena [slot][B][d*f]
  float* Wop;           // operand copy (fp32), same layout
  int slot_w1, slot_w2, B;
  float* losses;
  long long loss_ld;
  int d, f, V;
  float eps, eta, clip;
  int* err;
};

// out(r, sum_c M[r*S + c] x[c]) for r < R: G threads per row (power of two
// <= 32), reduced with shuffles inside the group.
template <class Out>
__device__ __forceinline__ void rowdot(const float* M, int S, int R, int L, const float* x, Out out) {
  const int nt = blockDim.x;
  int G = 1;
  while (G < 32 && G * 2 * R <= nt) G *= 2;
  const int g = threadIdx.x % G;
  for (int r0 = 0; r0 < R; r0 += nt / G) {
    const int r = r0 + threadIdx.x / G;
    float acc = 0.0f;
    if (r < R) {
      const float* row = M + (long long)r * S;
      for (int c = g; c < L; c += G) acc = fmaf(row[c], x[c], acc);
    }
    for (int o = G / 2; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (g == 0 && r < R) out(r, acc);
  }
}

// out[c] = sum_r M[r*S + c] x[r] for c < C: P = blockDim / C row parts per
// column (partials in red[P][C], summed in part order).
__device__ __forceinline__ void coldot(const float* M, int S, int R, int C, const float* x, float* out, float* red) {
  const int nt = blockDim.x;
  const int P = nt / C >= 1 ? nt / C : 1;
  for (int c0 = 0; c0 < C; c0 += nt) {
    const int c = c0 + threadIdx.x % (P > 1 ? C : nt);
    const int p = P > 1 ? threadIdx.x / C : 0;
    float acc = 0.0f;
    if (c < C && p < P)
      for (int r = p; r < R; r += P) acc = fmaf(M[(long long)r * S + c], x[r], acc);
    if (P > 1) {
      if (p < P) red[p * C + c] = acc;
    } else if (c < C) {
      out[c] = acc;
    }
  }
  if (P > 1) {
    __syncthreads();
    for (int c = threadIdx.x; c < C; c += nt) {
      float s = 0.0f;
      for (int p = 0; p < P; ++p) s += red[p * C + c];
      out[c] = s;
    }
  }
}

// Block-wide sum of four values at once (one barrier round); red: >= 128 floats.
__device__ __forceinline__ float4 tok_sum4(float4 v, float* red) {
  v.x = warp_sum(v.x); v.y = warp_sum(v.y); v.z = warp_sum(v.z); v.w = warp_sum(v.w);
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  __syncthreads();
  if (lane == 0) reinterpret_cast<float4*>(red)[wid] = v;
  __syncthreads();
  float4 t = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  for (int w = 0; w < nw; ++w) {
    const float4 q = reinterpret_cast<const float4*>(red)[w];
    t.x += q.x; t.y += q.y; t.z += q.z; t.w += q.w;
  }
  return t;
}

// Block-wide sum and max; every thread receives the result.  red: >= 32 floats.
__device__ __forceinline__ float tok_sum(float v, float* red) { return block_sum(v, red); }
__device__ __forceinline__ float tok_max(float v, float* red) {
  v = warp_max(v);
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  __syncthreads();
  if (lane == 0) red[wid] = v;
  __syncthreads();
  float m = -FLT_MAX;
  for (int w = 0; w < nw; ++w) m = fmaxf(m, red[w]);
  return m;
}

__global__ void __launch_bounds__(kTokThreads) token_steps_kernel(TokenArgs a) {
  pdl_wait();
  pdl_launch();
  extern __shared__ __align__(16) float sm[];
  const int d = a.d, f = a.f, V = a.V, s = blockIdx.x;
  const int S1 = d + 1, S2 = f + 1, SU = d + 1;
  float* red = sm;                      // [kRed]: reductions first (16-byte aligned)
  float* W1 = red + kRed;               // [f][d+1]
  float* W2 = W1 + f * S1;              // [d][f+1]
  float* U = W2 + d * S2;               // [V][d+1]
  float* h = U + V * SU;                // [d]
  float* h2 = h + d;                    // [d]
  float* y = h2 + d;                    // [d]
  float* dy = y + d;                    // [d]
  float* dh = dy + d;                   // [d]
  float* z = dh + d;                    // [f]
  float* av = z + f;                    // [f]
  float* da = av + f;                   // [f]
  float* lg = da + f;                   // [V]
  const int nt = blockDim.x, tid = threadIdx.x;
  const long long n = (long long)d * f;
  const float* w1g = a.W32 + ((long long)a.slot_w1 * a.B + s) * n;
  const float* w2g = a.W32 + ((long long)a.slot_w2 * a.B + s) * n;
  for (long long e = tid; e < n; e += nt) {
    const int r1 = (int)(e / d), c1 = (int)(e % d);
    W1[r1 * S1 + c1] = w1g[e];
    const int r2 = (int)(e / f), c2 = (int)(e % f);
    W2[r2 * S2 + c2] = w2g[e];
  }
  for (long long e = tid; e < (long long)V * d; e += nt) U[(e / d) * SU + e % d] = a.U[e];
  __syncthreads();

  const int32_t* tk = a.tok + (long long)s * a.tok_ld;
  for (int t = 0; t < a.T; ++t) {
    int x = tk[t], tgt = tk[t + 1];
    if ((unsigned)x >= (unsigned)V || (unsigned)tgt >= (unsigned)V) {
      if (tid == 0) atomicOr(a.err, 2);
      if ((unsigned)x >= (unsigned)V) x = 0;
      if ((unsigned)tgt >= (unsigned)V) tgt = 0;
    }
    // ---- forward
    for (int k = tid; k < d; k += nt) h[k] = a.E[(long long)x * d + k];
    __syncthreads();
    rowdot(W1, S1, f, d, h, [&](int j, float v) {
      z[j] = v;
      av[j] = gelu_f(v);
    });
    __syncthreads();
    rowdot(W2, S2, d, f, av, [&](int i, float v) { h2[i] = h[i] + v; });
    __syncthreads();
    float ss = 0.0f;
    for (int i = tid; i < d; i += nt) ss += h2[i] * h2[i];
    const float rstd = rsqrtf(tok_sum(ss, red) / d + a.eps);
    for (int i = tid; i < d; i += nt) y[i] = h2[i] * rstd;
    __syncthreads();
    rowdot(U, SU, V, d, y, [&](int v, float l) { lg[v] = l; });
    __syncthreads();
    float mx = -FLT_MAX;
    for (int v = tid; v < V; v += nt) mx = fmaxf(mx, lg[v]);
    mx = tok_max(mx, red);
    float se = 0.0f;
    for (int v = tid; v < V; v += nt) se += expf(lg[v] - mx);
    se = tok_sum(se, red);
    const float lse = mx + logf(se);
    if (tid == 0) a.losses[(long long)s * a.loss_ld + t] = lse - lg[tgt];
    __syncthreads();
    // Source Masking: a masked target is scored but takes no step (uniform per block)
    if (a.mask && !a.mask[(long long)s * a.mask_ld + t]) continue;
    // ---- backward (the mean over a one-token chunk is the token itself)
    for (int v = tid; v < V; v += nt) lg[v] = expf(lg[v] - lse) - (v == tgt ? 1.0f : 0.0f);
    __syncthreads();
    coldot(U, SU, V, d, lg, dy, red + 32);
    __syncthreads();
    float yd = 0.0f;
    for (int i = tid; i < d; i += nt) yd += y[i] * dy[i];
    const float myd = tok_sum(yd, red) / d;
    for (int i = tid; i < d; i += nt) dh[i] = rstd * (dy[i] - y[i] * myd);
    __syncthreads();
    coldot(W2, S2, d, f, dh, da, red + 32);
    __syncthreads();
    for (int j = tid; j < f; j += nt) da[j] *= gelu_grad_f(z[j]);   // dz
    __syncthreads();
    // ---- clipped step on the outer products
    float4 q = make_float4(0.0f, 0.0f, 0.0f, 0.0f);   // |dh|^2, |h|^2, |a|^2, |dz|^2
    for (int i = tid; i < d; i += nt) {
      q.x += dh[i] * dh[i];
      q.y += h[i] * h[i];
    }
    for (int j = tid; j < f; j += nt) {
      q.z += av[j] * av[j];
      q.w += da[j] * da[j];
    }
    q = tok_sum4(q, red + 32);
    const float norm = sqrtf(q.x * q.z + q.w * q.y);
    float sc = 1.0f;
    if (!isfinite(norm)) {
      sc = 0.0f;
      if (tid == 0) atomicOr(a.err, 1);
    } else if (a.clip > 0.0f) {
      sc = fminf(1.0f, a.clip / (norm + 1e-6f));
    }
    const float step = a.eta * sc;
    if (step != 0.0f) {
      // one warp per row, lanes along the row
      const int warp = tid >> 5, lane = tid & 31, nw = nt >> 5;
      for (int i = warp; i < d; i += nw) {
        const float gi = step * dh[i];
        float* row = W2 + i * S2;
        for (int j = lane; j < f; j += 32) row[j] -= gi * av[j];
      }
      for (int j = warp; j < f; j += nw) {
        const float gj = step * da[j];
        float* row = W1 + j * S1;
        for (int k = lane; k < d; k += 32) row[k] -= gj * h[k];
      }
    }
    __syncthreads();
  }

  float* w1o = a.W32 + ((long long)a.slot_w1 * a.B + s) * n;
  float* w2o = a.W32 + ((long long)a.slot_w2 * a.B + s) * n;
  float* w1p = a.Wop + ((long long)a.slot_w1 * a.B + s) * n;
  float* w2p = a.Wop + ((long long)a.slot_w2 * a.B + s) * n;
  for (long long e = tid; e < n; e += nt) {
    const float v1 = W1[(e / d) * S1 + e % d];
    const float v2 = W2[(e / f) * S2 + e % f];
    w1o[e] = v1;
    w1p[e] = v1;
    w2o[e] = v2;
    w2p[e] = v2;
  }
}

size_t token_smem_bytes(int d, int f, int V) {
  const size_t fl = (size_t)kRed + (size_t)f * (d + 1) + (size_t)d * (f + 1) + (size_t)V * (d + 1) + 5 * (size_t)d +
                    3 * (size_t)f + (size_t)V;
  return fl * sizeof(float);
}

}  // namespace

bool token_steps_supported(int d, int f, int V) {
  return d >= 1 && f >= 1 && V >= 1 && token_smem_bytes(d, f, V) <= 227 * 1024;
}

ttt_status launch_token_steps(int B, const int32_t* tok, long long tok_ld, int T, const uint8_t* mask,
                              long long mask_ld, const float* E, const float* U,
                              float* W32, float* Wop, int slot_w1, int slot_w2, float* losses, long long loss_ld,
                              int d, int f, int V, float eps, float eta, float clip, int* err, cudaStream_t st) {
  if (!token_steps_supported(d, f, V)) {
    set_error("per-token kernel: weights do not fit in shared memory");
    return TTT_ERR_UNSUPPORTED;
  }
  if (B == 0 || T == 0) return TTT_OK;
  const size_t smem = token_smem_bytes(d, f, V);
  TTT_CUDA(ensure_dyn_smem((const void*)token_steps_kernel, smem));
  TokenArgs a{tok, tok_ld, T, mask, mask_ld, E, U, W32, Wop, slot_w1, slot_w2, B, losses, loss_ld, d, f, V, eps, eta,
              clip, err};
  launch_pdl(token_steps_kernel, B, kTokThreads, smem, st, a);
  TTT_CHECK_LAUNCH();
  return TTT_OK;
}

}  // namespace ttt
