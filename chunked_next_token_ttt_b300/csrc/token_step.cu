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

// ---------------------------------------------------------------------------
// Register-resident form for the width-64, hidden-256, vocabulary-256 network:
// W1 and W2 stay in registers for the whole stream (32 + 32 per thread), U in
// shared memory.  Thread (warp w, lane l) owns rows i = 4 (l % 16) .. + 3 of
// the width and columns j = 8 g .. + 7 of the hidden (and vocabulary)
// dimension, g = 2 w + l / 16, of W1^T, W2 and U^T.  Products that reduce over
// i (z = W1 h, logits = U y, da = W2^T dh) reduce over the 16 lanes of a
// half-warp with a shuffle reduce-scatter that leaves one j per lane pair;
// products that reduce over j (W2 a, U^T dlogits) reduce the lane halves by
// one shuffle step and the 16 warps through shared memory, where warp 0 folds
// the 64 results (with the RMSNorm and its backward).  Six block barriers per
// token; both rank-one updates are applied in registers.
constexpr int kRD = 64, kRF = 256, kRV = 256;
constexpr int kRThreads = 512;
constexpr unsigned kFull = 0xffffffffu;

// Sum of v[0..7] over the 16 lanes of the half-warp, scattered: the lane
// returns the total of element ((l >> 3) & 1) * 4 + ((l >> 2) & 1) * 2 +
// ((l >> 1) & 1); lanes l and l ^ 1 return the same element.
__device__ __forceinline__ float half_reduce_scatter8(const float (&v)[8], int lane) {
  float a[4], b[2];
  const bool u8 = lane & 8, u4 = lane & 4, u2 = lane & 2;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float send = u8 ? v[q] : v[q + 4], keep = u8 ? v[q + 4] : v[q];
    a[q] = keep + __shfl_xor_sync(kFull, send, 8);
  }
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const float send = u4 ? a[q] : a[q + 2], keep = u4 ? a[q + 2] : a[q];
    b[q] = keep + __shfl_xor_sync(kFull, send, 4);
  }
  const float send = u2 ? b[0] : b[1], keep = u2 ? b[1] : b[0];
  float c = keep + __shfl_xor_sync(kFull, send, 2);
  return c + __shfl_xor_sync(kFull, c, 1);
}

// The inverse: every lane of the half-warp receives the 8 elements that
// half_reduce_scatter8 spread over it, in order.
__device__ __forceinline__ void half_all_gather8(float c, float (&v)[8], int lane) {
  const bool u8 = lane & 8, u4 = lane & 4, u2 = lane & 2;
  const float o = __shfl_xor_sync(kFull, c, 2);
  const float b0 = u2 ? o : c, b1 = u2 ? c : o;
  const float o0 = __shfl_xor_sync(kFull, b0, 4), o1 = __shfl_xor_sync(kFull, b1, 4);
  const float a[4] = {u4 ? o0 : b0, u4 ? o1 : b1, u4 ? b0 : o0, u4 ? b1 : o1};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float p = __shfl_xor_sync(kFull, a[q], 8);
    v[q] = u8 ? p : a[q];
    v[q + 4] = u8 ? a[q] : p;
  }
}

struct RegSmem {
  float U[kRV * kRD];     // [v][i]
  float part[16 * kRD];   // per-warp partial sums over j of a width-64 vector
  float y[kRD];
  float dh[kRD];
  float2 stat[16];        // per-warp (max, sum of exp) of the logits, then (|a|^2, |dz|^2)
  float2 stat2[16];
  float scal[4];          // rstd, |h|^2, |dh|^2
};

__global__ void __launch_bounds__(kRThreads, 1) token_steps_reg_kernel(TokenArgs a) {
  pdl_wait();
  pdl_launch();
  extern __shared__ __align__(16) float sm_raw[];
  RegSmem& S = *reinterpret_cast<RegSmem*>(sm_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, s = blockIdx.x;
  const int li = lane & 15, hb = lane >> 4, g = warp * 2 + hb;
  const int i0 = 4 * li, j0 = 8 * g;
  const int qs = ((lane >> 3) & 1) * 4 + ((lane >> 2) & 1) * 2 + ((lane >> 1) & 1);
  const int js = j0 + qs;                      // the element this lane holds after a reduce-scatter
  const bool uniq = (lane & 1) == 0;           // one lane of each pair counts it in block sums
  const long long n = (long long)kRD * kRF;
  const float* w1g = a.W32 + ((long long)a.slot_w1 * a.B + s) * n;   // W1 [F][D]
  const float* w2g = a.W32 + ((long long)a.slot_w2 * a.B + s) * n;   // W2 [D][F]
  float w1[4][8], w2[4][8];                    // w1[p][q] = W1[j0+q][i0+p], w2[p][q] = W2[i0+p][j0+q]
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const float4 r = *reinterpret_cast<const float4*>(w1g + (long long)(j0 + q) * kRD + i0);
    w1[0][q] = r.x; w1[1][q] = r.y; w1[2][q] = r.z; w1[3][q] = r.w;
  }
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    const float4 r0 = *reinterpret_cast<const float4*>(w2g + (long long)(i0 + p) * kRF + j0);
    const float4 r1 = *reinterpret_cast<const float4*>(w2g + (long long)(i0 + p) * kRF + j0 + 4);
    w2[p][0] = r0.x; w2[p][1] = r0.y; w2[p][2] = r0.z; w2[p][3] = r0.w;
    w2[p][4] = r1.x; w2[p][5] = r1.y; w2[p][6] = r1.z; w2[p][7] = r1.w;
  }
  for (int e = tid; e < kRV * kRD / 4; e += kRThreads)
    reinterpret_cast<float4*>(S.U)[e] = reinterpret_cast<const float4*>(a.U)[e];

  const int32_t* tk = a.tok + (long long)s * a.tok_ld;
  auto valid = [&](int x) {
    if ((unsigned)x < (unsigned)kRV) return x;
    if (tid == 0) atomicOr(a.err, 2);
    return 0;
  };
  // token t's input row (four elements per thread; two more for warp 0's fold)
  int x = a.T > 0 ? valid(tk[0]) : 0;
  float4 hrow = *reinterpret_cast<const float4*>(a.E + (long long)x * kRD + i0);
  float hw0 = 0.0f, hw1 = 0.0f;
  if (warp == 0) {
    hw0 = a.E[(long long)x * kRD + lane];
    hw1 = a.E[(long long)x * kRD + 32 + lane];
  }
  __syncthreads();

  for (int t = 0; t < a.T; ++t) {
    const int tgt = valid(tk[t + 1]);
    const bool take = !a.mask || a.mask[(long long)s * a.mask_ld + t];
    const float h[4] = {hrow.x, hrow.y, hrow.z, hrow.w};
    const float h0 = hw0, h1 = hw1;
    // the next token's input row, loaded while this one runs
    if (t + 1 < a.T) {
      hrow = *reinterpret_cast<const float4*>(a.E + (long long)tgt * kRD + i0);
      if (warp == 0) {
        hw0 = a.E[(long long)tgt * kRD + lane];
        hw1 = a.E[(long long)tgt * kRD + 32 + lane];
      }
    }
    // ---- z = W1 h, a = GELU(z)
    float zp[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) zp[q] = fmaf(w1[3][q], h[3], fmaf(w1[2][q], h[2], fmaf(w1[1][q], h[1], w1[0][q] * h[0])));
    const float zs = half_reduce_scatter8(zp, lane);
    const float as = gelu_f(zs), gs = gelu_grad_f(zs);
    float av[8];
    half_all_gather8(as, av, lane);
    // ---- h2 = h + W2 a: partial sums over this thread's j, then the lane halves
    float hp[4];
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      float acc = 0.0f;
#pragma unroll
      for (int q = 0; q < 8; ++q) acc = fmaf(w2[p][q], av[q], acc);
      hp[p] = acc;
    }
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const float send = hb ? hp[k] : hp[k + 2], keep = hb ? hp[k + 2] : hp[k];
      S.part[warp * kRD + i0 + 2 * hb + k] = keep + __shfl_xor_sync(kFull, send, 16);
    }
    __syncthreads();                                             // 1
    if (warp == 0) {
      float v0 = h0, v1 = h1;
#pragma unroll
      for (int w = 0; w < 16; ++w) {
        v0 += S.part[w * kRD + lane];
        v1 += S.part[w * kRD + 32 + lane];
      }
      const float rstd = rsqrtf(warp_sum(v0 * v0 + v1 * v1) / kRD + a.eps);
      S.y[lane] = v0 * rstd;
      S.y[32 + lane] = v1 * rstd;
      const float hh = warp_sum(h0 * h0 + h1 * h1);
      if (lane == 0) {
        S.scal[0] = rstd;
        S.scal[1] = hh;
      }
    }
    __syncthreads();                                             // 2
    // ---- logits = U y (y = h2 rstd), scattered one per lane pair
    const float4 y4 = *reinterpret_cast<const float4*>(S.y + i0);
    float lp[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const float4 u = *reinterpret_cast<const float4*>(S.U + (j0 + q) * kRD + i0);
      lp[q] = fmaf(u.w, y4.w, fmaf(u.z, y4.z, fmaf(u.y, y4.y, u.x * y4.x)));
    }
    const float ls = half_reduce_scatter8(lp, lane);
    {
      const float mw = warp_max(ls);
      const float sw = warp_sum(uniq ? expf(ls - mw) : 0.0f);
      if (lane == 0) S.stat[warp] = make_float2(mw, sw);
    }
    __syncthreads();                                             // 3
    float lse;
    {
      const float2 st = lane < 16 ? S.stat[lane] : make_float2(-FLT_MAX, 0.0f);
      const float M = warp_max(st.x);
      lse = M + logf(warp_sum(lane < 16 ? st.y * expf(st.x - M) : 0.0f));
    }
    if (uniq && js == tgt) a.losses[(long long)s * a.loss_ld + t] = lse - ls;
    // Source Masking: a masked target is scored but takes no step (uniform per block)
    if (!take) continue;
    // ---- dy = U^T dlogits (dlogits = softmax - onehot)
    float dl[8];
    half_all_gather8(expf(ls - lse) - (js == tgt ? 1.0f : 0.0f), dl, lane);
    float dp[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const float4 u = *reinterpret_cast<const float4*>(S.U + (j0 + q) * kRD + i0);
      dp[0] = fmaf(u.x, dl[q], dp[0]);
      dp[1] = fmaf(u.y, dl[q], dp[1]);
      dp[2] = fmaf(u.z, dl[q], dp[2]);
      dp[3] = fmaf(u.w, dl[q], dp[3]);
    }
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const float send = hb ? dp[k] : dp[k + 2], keep = hb ? dp[k + 2] : dp[k];
      S.part[warp * kRD + i0 + 2 * hb + k] = keep + __shfl_xor_sync(kFull, send, 16);
    }
    __syncthreads();                                             // 4
    if (warp == 0) {
      float d0 = 0.0f, d1 = 0.0f;
#pragma unroll
      for (int w = 0; w < 16; ++w) {
        d0 += S.part[w * kRD + lane];
        d1 += S.part[w * kRD + 32 + lane];
      }
      const float rstd = S.scal[0];
      const float y0 = S.y[lane], y1 = S.y[32 + lane];
      const float myd = warp_sum(y0 * d0 + y1 * d1) / kRD;
      const float e0 = rstd * (d0 - y0 * myd), e1 = rstd * (d1 - y1 * myd);
      S.dh[lane] = e0;
      S.dh[32 + lane] = e1;
      const float dd = warp_sum(e0 * e0 + e1 * e1);
      if (lane == 0) S.scal[2] = dd;
    }
    __syncthreads();                                             // 5
    // ---- da = W2^T dh, dz = da GELU'(z); norms of the two outer products
    const float4 dh4 = *reinterpret_cast<const float4*>(S.dh + i0);
    float dap[8];
#pragma unroll
    for (int q = 0; q < 8; ++q)
      dap[q] = fmaf(w2[3][q], dh4.w, fmaf(w2[2][q], dh4.z, fmaf(w2[1][q], dh4.y, w2[0][q] * dh4.x)));
    const float dzs = half_reduce_scatter8(dap, lane) * gs;
    {
      const float aa = warp_sum(uniq ? as * as : 0.0f), zz = warp_sum(uniq ? dzs * dzs : 0.0f);
      if (lane == 0) S.stat2[warp] = make_float2(aa, zz);
    }
    __syncthreads();                                             // 6
    float aa, zz;
    {
      const float2 st = lane < 16 ? S.stat2[lane] : make_float2(0.0f, 0.0f);
      aa = warp_sum(st.x);
      zz = warp_sum(st.y);
    }
    // ||dW2||^2 + ||dW1||^2 = |dh|^2 |a|^2 + |dz|^2 |h|^2
    const float norm = sqrtf(S.scal[2] * aa + zz * S.scal[1]);
    float sc = 1.0f;
    if (!isfinite(norm)) {
      sc = 0.0f;
      if (tid == 0) atomicOr(a.err, 1);
    } else if (a.clip > 0.0f) {
      sc = fminf(1.0f, a.clip / (norm + 1e-6f));
    }
    const float step = a.eta * sc;
    float dz[8];
    half_all_gather8(dzs, dz, lane);
    const float sdh[4] = {step * dh4.x, step * dh4.y, step * dh4.z, step * dh4.w};
#pragma unroll
    for (int p = 0; p < 4; ++p) {
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        w1[p][q] = fmaf(-step * dz[q], h[p], w1[p][q]);
        w2[p][q] = fmaf(-sdh[p], av[q], w2[p][q]);
      }
    }
  }

  float* w1o = a.W32 + ((long long)a.slot_w1 * a.B + s) * n;
  float* w2o = a.W32 + ((long long)a.slot_w2 * a.B + s) * n;
  float* w1p = a.Wop + ((long long)a.slot_w1 * a.B + s) * n;
  float* w2p = a.Wop + ((long long)a.slot_w2 * a.B + s) * n;
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const float4 r = make_float4(w1[0][q], w1[1][q], w1[2][q], w1[3][q]);
    *reinterpret_cast<float4*>(w1o + (long long)(j0 + q) * kRD + i0) = r;
    *reinterpret_cast<float4*>(w1p + (long long)(j0 + q) * kRD + i0) = r;
  }
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    const float4 r0 = make_float4(w2[p][0], w2[p][1], w2[p][2], w2[p][3]);
    const float4 r1 = make_float4(w2[p][4], w2[p][5], w2[p][6], w2[p][7]);
    *reinterpret_cast<float4*>(w2o + (long long)(i0 + p) * kRF + j0) = r0;
    *reinterpret_cast<float4*>(w2o + (long long)(i0 + p) * kRF + j0 + 4) = r1;
    *reinterpret_cast<float4*>(w2p + (long long)(i0 + p) * kRF + j0) = r0;
    *reinterpret_cast<float4*>(w2p + (long long)(i0 + p) * kRF + j0 + 4) = r1;
  }
}

bool token_steps_reg_shape(int d, int f, int V) { return d == kRD && f == kRF && V == kRV; }

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
  TokenArgs a{tok, tok_ld, T, mask, mask_ld, E, U, W32, Wop, slot_w1, slot_w2, B, losses, loss_ld, d, f, V, eps, eta,
              clip, err};
  const bool aligned = ((reinterpret_cast<uintptr_t>(E) | reinterpret_cast<uintptr_t>(U) |
                         reinterpret_cast<uintptr_t>(W32) | reinterpret_cast<uintptr_t>(Wop)) & 15) == 0;
  if (token_steps_reg_shape(d, f, V) && aligned) {
    TTT_CUDA(ensure_dyn_smem((const void*)token_steps_reg_kernel, sizeof(RegSmem)));
    launch_pdl(token_steps_reg_kernel, B, kRThreads, sizeof(RegSmem), st, a);
  } else {
    const size_t smem = token_smem_bytes(d, f, V);
    TTT_CUDA(ensure_dyn_smem((const void*)token_steps_kernel, smem));
    launch_pdl(token_steps_kernel, B, kTokThreads, smem, st, a);
  }
  TTT_CHECK_LAUNCH();
  return TTT_OK;
}

}  // namespace ttt
