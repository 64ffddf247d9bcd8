// Decoding's next-token forward as one persistent kernel (bf16 storage, GELU
// or SwiGLU blocks without attention or extra frozen MLPs): embedding, every
// block's up and down projection, the final RMSNorm, the LM head and the
// softmax of one new row per sequence ("End-to-End TTT" review, 3.2: each
// decoded token is scored by the current weights and the next-token
// distribution is formed from them; eq. (1) for the loss that reads it).
//
// At one row per sequence every product is a weight-streaming GEMV, so the
// step is bound by reading each weight once (prefix and head weights shared by
// the sequences, fast weights per sequence).  One cooperative launch of one CTA
// per SM replaces the ~30 launches of the launch-by-launch forward: each phase
// spreads the output rows of one projection over all warps of the grid (a warp
// keeps several rows' 16-byte weight loads in flight), and a grid-wide barrier
// separates the phases (2 per block, 2 around the head).  A down projection
// with fewer rows than the grid has warps splits its K into segments whose
// partial sums the next phase folds into the residual stream (in segment
// order, identically in every CTA), so no element is read, modified and
// written across CTAs.  Each barrier's wait is bounded: on a timeout the kernel records a
// code in the status word, raises an abort flag that the other CTAs see, and
// every CTA returns.
//
// Numerics follow the launch-by-launch path: the GEMV inputs are the bf16
// operand copies of the fp32 residual stream and of the activations; products
// accumulate in fp32; the residual stream stays fp32.
#include <cfloat>

#include "kernels.h"

namespace ttt {
namespace dp {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kSeq = 8;                 // sequences a warp accumulates at once
constexpr long long kTimeoutNs = 1000000000LL;

__device__ __forceinline__ unsigned long long now_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Grid-wide barrier of a cooperative launch: bar[0] counts arrivals over the
// whole launch (barrier g is complete at g * gridDim.x), bar[1] is the
// generation the last arrival publishes, bar[2] an abort flag.  The arrival
// is a release (it orders the CTA's writes, made visible to thread 0 by the
// block barrier before it) and the wait an acquire, so no separate fences are
// needed.  Returns false (in every thread of the CTA) when the wait timed out
// or another CTA aborted.
__device__ bool grid_sync(unsigned* bar, unsigned& gen, int* err) {
  __syncthreads();
  int ok = 1;
  if (threadIdx.x == 0) {
    const unsigned next = gen + 1;
    unsigned old;
    asm volatile("atom.add.release.gpu.global.u32 %0, [%1], 1;" : "=r"(old) : "l"(bar) : "memory");
    if (old == next * gridDim.x - 1) {
      asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(bar + 1), "r"(next) : "memory");
    } else {
      const unsigned long long t0 = now_ns();
      while (ld_acquire(&bar[1]) != next) {
        if (ld_acquire(&bar[2]) != 0u) {
          ok = 0;
          break;
        }
        if (now_ns() - t0 > (unsigned long long)kTimeoutNs) {
          atomicOr(err, 4);
          atomicExch(&bar[2], 1u);
          ok = 0;
          break;
        }
      }
    }
  }
  gen += 1;
  return __syncthreads_and(ok) != 0;
}

// 8 bf16 (16 bytes) as floats.
__device__ __forceinline__ void bf8(const uint4& u, float (&f)[8]) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 t = __bfloat1622float2(h[i]);
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}

__device__ __forceinline__ float warp_total(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Pairs of floats for the two-wide FMA pipe instructions (f32x2): even and odd
// elements of a piece accumulate in the two halves.
typedef unsigned long long f2;
__device__ __forceinline__ f2 f2make(float x, float y) {
  f2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(x), "f"(y));
  return r;
}
__device__ __forceinline__ float f2sum(f2 v) {
  float x, y;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(x), "=f"(y) : "l"(v));
  return x + y;
}
__device__ __forceinline__ f2 f2fma(f2 a, f2 b, f2 c) {
  f2 r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
// 8 bf16 as four pairs of floats
__device__ __forceinline__ void bf8x2(const uint4& u, f2 (&p)[4]) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 t = __bfloat1622float2(h[i]);
    p[i] = f2make(t.x, t.y);
  }
}


// Sum over the 32 lanes of v[0..7], scattered: the lane receives the total of
// element ((l >> 4) & 1) * 4 + ((l >> 3) & 1) * 2 + ((l >> 2) & 1); the four
// lanes that share bits 4..2 receive the same element.
__device__ __forceinline__ int scatter_index(int lane) {
  return ((lane >> 4) & 1) * 4 + ((lane >> 3) & 1) * 2 + ((lane >> 2) & 1);
}
__device__ __forceinline__ float reduce_scatter8(const float (&v)[8], int lane) {
  float a[4], b[2];
  const bool u16 = lane & 16, u8 = lane & 8, u4 = lane & 4;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float send = u16 ? v[q] : v[q + 4], keep = u16 ? v[q + 4] : v[q];
    a[q] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
  }
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const float send = u8 ? a[q] : a[q + 2], keep = u8 ? a[q + 2] : a[q];
    b[q] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
  }
  const float send = u4 ? b[0] : b[1], keep = u4 ? b[1] : b[0];
  float c = keep + __shfl_xor_sync(0xffffffffu, send, 4);
  c += __shfl_xor_sync(0xffffffffu, c, 2);
  return c + __shfl_xor_sync(0xffffffffu, c, 1);
}

// The warp total of sequence m's value (S = 8: scattered, m = scatter_index;
// S = 1: every lane, m = 0).
template <int S>
__device__ __forceinline__ float reduce_seq(const float (&v)[S], int lane) {
  if constexpr (S == 1) {
    return warp_total(v[0]);
  } else {
    return reduce_scatter8(v, lane);
  }
}

// acc[i][q][s] += W_q(row i) . xs[s] over K for R rows of NW weight matrices
// shared by the sequences (a null row contributes nothing) and nb sequences of
// fp32 operand rows in shared memory in the split layout of stage_fold (piece
// c of sequence s: elements 0..3 at xs[s * ld8 + c], 4..7 at xs[half + ...],
// so that lanes reading consecutive pieces hit distinct banks).  Lanes take 8-element
// pieces; every weight piece of a batch of CB pieces per lane is loaded before
// any is used (R * NW * CB 16-byte loads in flight per lane), and each piece is
// unpacked once for all sequences.
template <int R, int NW, int CB, int S>
__device__ __forceinline__ void dots_shared(const bf16* const (&w)[R][NW], const float4* xs, int half, int K, int ld8,
                                            int nb, float (&acc)[R][NW][S], int lane) {
  const int K8 = K / 8;
  f2 acc2[R][NW][S];
#pragma unroll
  for (int i = 0; i < R; ++i)
#pragma unroll
    for (int q = 0; q < NW; ++q)
#pragma unroll
      for (int s = 0; s < S; ++s) acc2[i][q][s] = 0ull;
  for (int c0 = lane; c0 < K8; c0 += 32 * CB) {
    uint4 wv[CB][R][NW];
#pragma unroll
    for (int b = 0; b < CB; ++b)
#pragma unroll
      for (int i = 0; i < R; ++i)
#pragma unroll
        for (int q = 0; q < NW; ++q)
          wv[b][i][q] = (c0 + 32 * b < K8 && w[i][q]) ? __ldg(reinterpret_cast<const uint4*>(w[i][q]) + c0 + 32 * b)
                                                      : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int b = 0; b < CB; ++b) {
      const int c = c0 + 32 * b;
      if (c >= K8) break;
      f2 wf[R][NW][4];
#pragma unroll
      for (int i = 0; i < R; ++i)
#pragma unroll
        for (int q = 0; q < NW; ++q) bf8x2(wv[b][i][q], wf[i][q]);
#pragma unroll
      for (int s = 0; s < S; ++s) {
        if (s < nb) {
          const ulonglong2 x0 = *reinterpret_cast<const ulonglong2*>(xs + s * ld8 + c);
          const ulonglong2 x1 = *reinterpret_cast<const ulonglong2*>(xs + half + s * ld8 + c);
          const f2 xf[4] = {x0.x, x0.y, x1.x, x1.y};
#pragma unroll
          for (int i = 0; i < R; ++i)
#pragma unroll
            for (int q = 0; q < NW; ++q) {
              f2 t = acc2[i][q][s];
#pragma unroll
              for (int e = 0; e < 4; ++e) t = f2fma(wf[i][q][e], xf[e], t);
              acc2[i][q][s] = t;
            }
        }
      }
    }
  }
#pragma unroll
  for (int i = 0; i < R; ++i)
#pragma unroll
    for (int q = 0; q < NW; ++q)
#pragma unroll
      for (int s = 0; s < S; ++s) acc[i][q][s] += f2sum(acc2[i][q][s]);
}

// acc[s] += W_s(row) . xs[s] over K where sequence s has its own weight row at
// w0 + s * wseq (the fast weights), nb <= NS sequences; loads batched as above.
template <int S, int NS, int CB>
__device__ __forceinline__ void dots_per_seq(const bf16* w0, long long wseq, const float4* xs, int half, int K,
                                             int ld8, int nb, float (&acc)[S], int lane) {
  const int K8 = K / 8;
  for (int c0 = lane; c0 < K8; c0 += 32 * CB) {
    uint4 wv[CB][NS];
#pragma unroll
    for (int b = 0; b < CB; ++b)
#pragma unroll
      for (int s = 0; s < NS; ++s)
        wv[b][s] = (c0 + 32 * b < K8 && s < nb) ? __ldg(reinterpret_cast<const uint4*>(w0 + s * wseq) + c0 + 32 * b)
                                                : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int b = 0; b < CB; ++b) {
      const int c = c0 + 32 * b;
      if (c >= K8) break;
#pragma unroll
      for (int s = 0; s < NS; ++s) {
        if (s < nb) {
          const float4 x0 = xs[s * ld8 + c], x1 = xs[half + s * ld8 + c];
          const float xf[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
          float wf[8];
          bf8(wv[b][s], wf);
          float t = acc[s];
#pragma unroll
          for (int e = 0; e < 8; ++e) t = fmaf(wf[e], xf[e], t);
          acc[s] = t;
        }
      }
    }
  }
}

// The residual stream entering a block into shared memory: x = xin + the
// nseg partial sums of the previous down projection (summed in segment order,
// the same in every CTA), as fp32 and, when `round`, rounded to bf16 like the
// operand copies of the launch-by-launch path.  When xout is given, this CTA
// also stores its share of x there (16-byte groups g with g % gridDim.x ==
// blockIdx.x), so that every element is written once.
// Element e of the split layout (piece e / 8, half (e / 4) % 2, lane e % 4).
__device__ __forceinline__ float& xs_at(float4* xs, int half, int e) {
  return reinterpret_cast<float*>(xs + (e >> 3) + ((e >> 2) & 1) * half)[e & 3];
}

__device__ __forceinline__ void stage_fold(const float* xin, const float* ps, int nseg, long long pstride,
                                           float* xout, float4* xs, int half, int count, bool round) {
  const float4* x4 = reinterpret_cast<const float4*>(xin);
  const int n4 = count / 4;
  for (int idx = threadIdx.x; idx < n4; idx += kThreads) {
    float4 q[9];
    q[0] = __ldcg(x4 + idx);
#pragma unroll
    for (int k = 0; k < 8; ++k)
      q[k + 1] = k < nseg ? __ldcg(reinterpret_cast<const float4*>(ps + k * pstride) + idx)
                          : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    float4 v = q[0];
#pragma unroll
    for (int k = 0; k < 8; ++k)
      if (k < nseg) {
        v.x += q[k + 1].x;
        v.y += q[k + 1].y;
        v.z += q[k + 1].z;
        v.w += q[k + 1].w;
      }
    if (xout && idx % (int)gridDim.x == (int)blockIdx.x) reinterpret_cast<float4*>(xout)[idx] = v;
    if (round) {
      v.x = __bfloat162float(__float2bfloat16_rn(v.x));
      v.y = __bfloat162float(__float2bfloat16_rn(v.y));
      v.z = __bfloat162float(__float2bfloat16_rn(v.z));
      v.w = __bfloat162float(__float2bfloat16_rn(v.w));
    }
    xs[(idx >> 1) + (idx & 1) * half] = v;
  }
}
__device__ __forceinline__ void stage_bf16(const bf16* src, float4* dst, int half, int count) {
  const uint4* s4 = reinterpret_cast<const uint4*>(src);
  const int n8 = count / 8;
  for (int base = threadIdx.x; base < n8; base += 4 * kThreads) {
    uint4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int idx = base + u * kThreads;
      v[u] = idx < n8 ? __ldcg(s4 + idx) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int idx = base + u * kThreads;
      if (idx < n8) {
        float f8[8];
        bf8(v[u], f8);
        dst[idx] = make_float4(f8[0], f8[1], f8[2], f8[3]);
        dst[half + idx] = make_float4(f8[4], f8[5], f8[6], f8[7]);
      }
    }
  }
}

__device__ __forceinline__ void soft_fold(float& m, float& s, float x) {
  if (x > m) {
    s = s * expf(m - x) + 1.0f;
    m = x;
  } else {
    s += expf(x - m);
  }
}
__device__ __forceinline__ void soft_join(float& m, float& s, float m2, float s2) {
  if (s2 == 0.0f) return;
  if (s == 0.0f) {
    m = m2;
    s = s2;
    return;
  }
  const float n = fmaxf(m, m2);
  s = s * expf(m - n) + s2 * expf(m2 - n);
  m = n;
}

constexpr int kRows = 2;       // rows a warp takes at once in the block projections
constexpr int kHeadRows = 2;   // and in the LM head

// S: the sequences a warp accumulates at once (8, or 1 for a single
// sequence, which frees registers for deeper load batches: CB pieces per lane)
template <int S>
__global__ void __launch_bounds__(kThreads, 1) decode_persist_kernel(const __grid_constant__ DecodeNet a) {
  constexpr int CB = S == 1 ? 8 : 4;
  constexpr int NS = S == 1 ? 1 : 4;           // sequences of a per-sequence-weight unit
  extern __shared__ __align__(16) uint8_t smraw[];
  float* red = reinterpret_cast<float*>(smraw);                        // [kWarps][kSeq][2] reductions
  float4* xs = reinterpret_cast<float4*>(smraw + kWarps * kSeq * 2 * 4);  // fp32 operand rows of the phase
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gw = blockIdx.x * kWarps + warp, GW = gridDim.x * kWarps;
  const int B = a.B, d = a.d, f = a.f, V = a.V;
  // after a reduction this lane holds sequence m's total; one lane of those that hold it writes it
  const int m = S == 1 ? 0 : scatter_index(lane);
  const bool writer = S == 1 ? lane == 0 : ((lane & 3) == 0 && m < B);
  const bool lead = S == 1 ? lane == 0 : (lane & 3) == 0;
  // the down projections split K = f into nseg segments when d rows alone
  // would leave warps idle; their partial sums are folded in by the next stage
  int nseg = 1;
  for (int c = 8; c > 1; --c)
    if ((long long)d * c <= GW && f % (8 * c) == 0) {
      nseg = c;
      break;
    }
  // per-sequence weights: a unit takes half of the sequences when there are more than four
  const int nh = B > 4 ? 2 : 1, hb = (B + nh - 1) / nh;    // hb <= NS for B <= 8
  const int sl = f / nseg;
  const long long BD = (long long)B * d;
  const int half = B * (d > f ? d : f) / 8;     // pieces of the operand buffer; split layout
  const int d8 = d / 8, f8 = f / 8;
  const int L = a.n_pre + a.n_fast;
  unsigned gen = 0;
  pdl_wait();

  // ---- embedding of the new inputs into the fp32 residual stream
  for (long long e = (long long)blockIdx.x * kThreads + tid; e < (long long)B * d; e += (long long)gridDim.x * kThreads) {
    const int s = (int)(e / d), c = (int)(e % d);
    int x = a.tok[s];
    if ((unsigned)x >= (unsigned)V) {
      if (c == 0) atomicOr(a.err, 2);
      x = 0;
    }
    a.x32[e] = __bfloat162float(static_cast<const bf16*>(a.E)[(long long)x * d + c]);
  }
  if (!grid_sync(a.bar, gen, a.err)) return;

  bf16* act = static_cast<bf16*>(a.act);
  for (int l = 0; l < a.n_pre + a.n_fast; ++l) {
    const bool fastb = l >= a.n_pre;
    const int lf = l - a.n_pre;
    // ---- the block's input x_l = x_{l-1} + the previous block's partial sums
    // (kept in x32[l & 1]); up projection: act[s][j] = GELU(W1 x) or
    // silu(Wg x) (Wu x), rows j over the grid's warps
    if (l == 0)
      stage_fold(a.x32, nullptr, 0, 0, nullptr, xs, half, B * d, true);
    else
      stage_fold(a.x32 + ((l - 1) & 1) * BD, a.px + ((l - 1) & 1) * 8 * BD, nseg, BD, a.x32 + (l & 1) * BD, xs,
                 half, B * d, true);
    __syncthreads();
    if (fastb && !a.swiglu) {
      // the fast W1 of each sequence
      const bf16* w1 = static_cast<const bf16*>(a.fup[lf]);
      for (int u = gw; u < f * nh; u += GW) {
        const int j = u / nh, s0 = (u % nh) * hb, nb = min(hb, B - s0);
        float acc[S] = {};
        dots_per_seq<S, NS, CB>(w1 + s0 * a.n + (long long)j * d, a.n, xs + s0 * d8, half, d, d8, nb, acc, lane);
        const float z = reduce_seq<S>(acc, lane);
        if (lead && m < nb) act[(long long)(s0 + m) * f + j] = __float2bfloat16_rn(gelu_f(z));
      }
    } else if (a.swiglu) {
      const bf16* wg = static_cast<const bf16*>(fastb ? a.ffrozen[lf][0] : a.pre[l][0]);
      const bf16* wu = static_cast<const bf16*>(fastb ? a.ffrozen[lf][1] : a.pre[l][1]);
      for (int j = gw; j < f; j += GW) {
        const bf16* w[1][2] = {{wg + (long long)j * d, wu + (long long)j * d}};
        float acc[1][2][S] = {};
        dots_shared<1, 2, CB, S>(w, xs, half, d, d8, B, acc, lane);
        const float g = reduce_seq<S>(acc[0][0], lane), u = reduce_seq<S>(acc[0][1], lane);
        if (writer) act[(long long)m * f + j] = __float2bfloat16_rn(silu_f(g) * u);
      }
    } else {
      const bf16* w1 = static_cast<const bf16*>(a.pre[l][0]);
      for (int j0 = gw; j0 < f; j0 += kRows * GW) {
        const bf16* w[kRows][1];
#pragma unroll
        for (int i = 0; i < kRows; ++i) w[i][0] = j0 + i * GW < f ? w1 + (long long)(j0 + i * GW) * d : nullptr;
        float acc[kRows][1][S] = {};
        dots_shared<kRows, 1, CB, S>(w, xs, half, d, d8, B, acc, lane);
#pragma unroll
        for (int i = 0; i < kRows; ++i) {
          const float z = reduce_seq<S>(acc[i][0], lane);
          const int j = j0 + i * GW;
          if (writer && j < f) act[(long long)m * f + j] = __float2bfloat16_rn(gelu_f(z));
        }
      }
    }
    if (!grid_sync(a.bar, gen, a.err)) return;
    // ---- down projection: partial sums px[l & 1][k][s][i] = W2[i, segment k] . act[s, segment k]
    // over units (i, k), i < d, k < nseg, spread over the grid's warps
    stage_bf16(act, xs, half, B * f);
    __syncthreads();
    float* pout = a.px + (l & 1) * 8 * BD;
    const bf16* w2 = static_cast<const bf16*>(fastb ? a.fdown[lf] : a.pre[l][a.swiglu ? 2 : 1]);
    const int nhu = fastb ? nh : 1;      // sequence groups per unit
    for (int u = gw; u < d * nseg * nhu; u += GW) {
      const int i = u / (nseg * nhu), k = (u / nhu) % nseg;
      const int s0 = (u % nhu) * hb, nb = fastb ? min(hb, B - s0) : B;
      const bf16* wrow = w2 + (long long)i * f + (long long)k * sl;
      float y;
      if (fastb) {
        float acc[S] = {};
        dots_per_seq<S, NS, CB>(wrow + s0 * a.n, a.n, xs + s0 * f8 + k * (sl / 8), half, sl, f8, nb, acc, lane);
        y = reduce_seq<S>(acc, lane);
      } else {
        const bf16* w[1][1] = {{wrow}};
        float acc[1][1][S] = {};
        dots_shared<1, 1, CB, S>(w, xs + k * (sl / 8), half, sl, f8, B, acc, lane);
        y = reduce_seq<S>(acc[0][0], lane);
      }
      if (lead && m < nb) pout[(long long)k * BD + (long long)(s0 + m) * d + i] = y;
    }
    if (!grid_sync(a.bar, gen, a.err)) return;
  }

  // ---- the final residual stream (fold of the last block's partial sums),
  // RMSNorm (unit gain; every CTA for itself), then the LM head:
  // logits[s][v] = U[v] . y[s], rows v over the grid's warps
  stage_fold(a.x32 + ((L - 1) & 1) * BD, a.px + ((L - 1) & 1) * 8 * BD, nseg, BD, nullptr, xs, half, B * d, false);
  __syncthreads();
  for (int s = warp; s < B; s += kWarps) {
    float sq = 0.0f;
    for (int c = lane; c < d; c += 32) {
      const float v = xs_at(xs, half, s * d + c);
      sq = fmaf(v, v, sq);
    }
    sq = warp_total(sq);
    if (lane == 0) red[s] = rsqrtf(sq / d + a.eps);
  }
  __syncthreads();
  for (int e = tid; e < B * d; e += kThreads) {
    float& x = xs_at(xs, half, e);
    x = __bfloat162float(__float2bfloat16_rn(x * red[e / d]));
  }
  __syncthreads();
  float mx = -FLT_MAX, se = 0.0f;      // writer lanes: softmax state of sequence m over this warp's rows
  const bf16* U = static_cast<const bf16*>(a.U);
  for (int v0 = gw; v0 < V; v0 += kHeadRows * GW) {
    const bf16* w[kHeadRows][1];
#pragma unroll
    for (int i = 0; i < kHeadRows; ++i) w[i][0] = v0 + i * GW < V ? U + (long long)(v0 + i * GW) * d : nullptr;
    float acc[kHeadRows][1][S] = {};
    dots_shared<kHeadRows, 1, CB, S>(w, xs, half, d, d8, B, acc, lane);
#pragma unroll
    for (int i = 0; i < kHeadRows; ++i) {
      const float x = reduce_seq<S>(acc[i][0], lane);
      const int v = v0 + i * GW;
      if (writer && v < V) {
        a.logits[(long long)m * V + v] = x;
        soft_fold(mx, se, x);
      }
    }
  }
  if (writer) {
    red[(warp * kSeq + m) * 2] = mx;
    red[(warp * kSeq + m) * 2 + 1] = se;
  }
  __syncthreads();
  if (tid < B) {
    float mm = -FLT_MAX, ss = 0.0f;
    for (int w = 0; w < kWarps; ++w) soft_join(mm, ss, red[(w * kSeq + tid) * 2], red[(w * kSeq + tid) * 2 + 1]);
    a.part[(long long)blockIdx.x * B + tid] = make_float2(mm, ss);
  }
  if (!grid_sync(a.bar, gen, a.err)) return;
  // ---- logsumexp of every sequence (each CTA in the same fixed order), p = exp(logits - lse)
  for (int s = warp; s < B; s += kWarps) {
    float mm = -FLT_MAX, ss = 0.0f;
    for (int g = lane; g < (int)gridDim.x; g += 32) {
      const float2 q = __ldcg(a.part + (long long)g * B + s);
      soft_join(mm, ss, q.x, q.y);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float m2 = __shfl_xor_sync(0xffffffffu, mm, o), s2 = __shfl_xor_sync(0xffffffffu, ss, o);
      soft_join(mm, ss, m2, s2);
    }
    if (lane == 0) {
      const float lse = mm + logf(ss);
      red[s] = lse;
      if (blockIdx.x == 0) a.lse[s] = lse;
    }
  }
  __syncthreads();
  for (int v0 = gw; v0 < V; v0 += kHeadRows * GW)
#pragma unroll
    for (int i = 0; i < kHeadRows; ++i) {
      const int v = v0 + i * GW;
      if (writer && v < V) {
        const long long o = (long long)m * V + v;
        a.p[o] = expf(a.logits[o] - red[m]);
      }
    }
}

size_t smem_bytes(int B, int d, int f) {
  return (size_t)kWarps * kSeq * 2 * 4 + (size_t)B * (d > f ? d : f) * 4;
}

}  // namespace dp

int decode_persist_grid(int B, int d, int f) {
  if (B < 1 || B > dp::kSeq || d % 8 || f % 8) return 0;
  const size_t smem = dp::smem_bytes(B, d, f);
  if (smem > 227 * 1024) return 0;
  const void* kern = B == 1 ? (const void*)dp::decode_persist_kernel<1> : (const void*)dp::decode_persist_kernel<8>;
  if (ensure_dyn_smem(kern, smem) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  int dev = 0, coop = 0, per_sm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) != cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, dp::kThreads, smem) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  if (!coop || per_sm < 1) return 0;
  return current_sm_count();
}

ttt_status launch_decode_persist(const DecodeNet& net, int grid, bool bar_clear, cudaStream_t st) {
  if (grid < 1 || net.B < 1 || net.B > dp::kSeq || net.n_pre + net.n_fast > kDecodeMaxBlocks || !net.bar ||
      !net.err) {
    set_error("persistent decode: bad configuration");
    return TTT_ERR_BAD_ARG;
  }
  if (bar_clear) TTT_CUDA(cudaMemsetAsync(net.bar, 0, 4 * sizeof(unsigned), st));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(dp::kThreads);
  cfg.dynamicSmemBytes = dp::smem_bytes(net.B, net.d, net.f);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (net.B == 1)
    TTT_CUDA(cudaLaunchKernelEx(&cfg, dp::decode_persist_kernel<1>, net));
  else
    TTT_CUDA(cudaLaunchKernelEx(&cfg, dp::decode_persist_kernel<8>, net));
  return TTT_OK;
}

}  // namespace ttt
