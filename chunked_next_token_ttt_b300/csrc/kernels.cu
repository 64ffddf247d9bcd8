// Non-GEMM kernels of the TTT chunk step: embedding gather, RMSNorm forward
// and backward, the fused softmax cross-entropy (loss + dlogits in place),
// the per-sequence global-norm reduction, clip+SGD on the fp32 masters, and
// the Settlement helpers.  All are HBM-bound row or elementwise kernels.
#include <cfloat>

#include <type_traits>

#include "kernels.h"

namespace ttt {
namespace {

template <typename ET, typename S>
__global__ void embed_kernel(TokView tv, const ET* __restrict__ E, int d, float* __restrict__ h32, void* hop,
                             long long hop_lo) {
  pdl_wait();
  pdl_launch();
  const int m = blockIdx.x;
  const int s = m / tv.rows, j = m % tv.rows;
  int x = tv.tok[s * tv.tok_ld + tv.tok_off + j];
  if ((unsigned)x >= (unsigned)tv.vocab) {
    if (threadIdx.x == 0) atomicOr(tv.err, 2);
    x = 0;
  }
  const ET* src = E + (long long)x * d;
  for (int c = threadIdx.x; c < d; c += blockDim.x) {
    const float v = to_f(src[c]);
    h32[(long long)m * d + c] = v;
    if (hop) OpIO<S>::store(hop, hop_lo, (long long)m * d + c, v);
  }
}

__device__ __forceinline__ int target_of(const TokView& tv, int s, int j, int V);

template <typename S>
__global__ void rmsnorm_fwd_kernel(int d, const float* __restrict__ x, float eps, void* y, long long y_lo,
                                   float* __restrict__ rstd, TokView tv, int32_t* __restrict__ tgt) {
  pdl_wait();
  pdl_launch();
  __shared__ float red[32];
  const long long m = blockIdx.x;
  if (tgt && threadIdx.x == 0) {
    // the target column of this row for the fused logits epilogue (-1: no target)
    const int s = (int)(m / tv.rows), j = (int)(m % tv.rows);
    tgt[m] = j < tv.n_valid ? target_of(tv, s, j, tv.vocab) : -1;
  }
  const float* xr = x + m * d;
  float sq = 0.0f;
  for (int c = threadIdx.x; c < d; c += blockDim.x) sq += xr[c] * xr[c];
  sq = block_sum(sq, red);
  const float r = rsqrtf(sq / d + eps);
  if (threadIdx.x == 0) rstd[m] = r;
  for (int c = threadIdx.x; c < d; c += blockDim.x) OpIO<S>::store(y, y_lo, m * d + c, xr[c] * r);
}

template <typename S>
__global__ void rmsnorm_bwd_kernel(int d, const float* __restrict__ x, const float* __restrict__ rstd,
                                   const float* __restrict__ dy, float* __restrict__ dx32, void* dxop,
                                   long long dx_lo) {
  pdl_wait();
  pdl_launch();
  __shared__ float red[32];
  const long long m = blockIdx.x;
  const float r = rstd[m];
  const float* xr = x + m * d;
  const float* dyr = dy + m * d;
  float dot = 0.0f;
  for (int c = threadIdx.x; c < d; c += blockDim.x) dot += xr[c] * r * dyr[c];
  dot = block_sum(dot, red) / d;
  for (int c = threadIdx.x; c < d; c += blockDim.x) {
    const float v = r * (dyr[c] - xr[c] * r * dot);
    dx32[m * d + c] = v;
    if (dxop) OpIO<S>::store(dxop, dx_lo, m * d + c, v);
  }
}

// The same two operations with one warp per row (8 rows per 256-thread block)
// and 16-byte loads, for rows whose width is a multiple of 4: no block barrier,
// every load of a lane in flight at once.
template <typename S>
__global__ void rmsnorm_fwd_warp_kernel(int M, int d, const float* __restrict__ x, float eps, void* y, long long y_lo,
                                        float* __restrict__ rstd, TokView tv, int32_t* __restrict__ tgt) {
  pdl_wait();
  pdl_launch();
  const int lane = threadIdx.x & 31;
  const long long m = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (m >= M) return;
  if (tgt && lane == 0) {
    const int s = (int)(m / tv.rows), j = (int)(m % tv.rows);
    tgt[m] = j < tv.n_valid ? target_of(tv, s, j, tv.vocab) : -1;
  }
  const float4* xr = reinterpret_cast<const float4*>(x + m * d);
  float sq = 0.0f;
  for (int c = lane; c < d / 4; c += 32) {
    const float4 v = xr[c];
    sq = fmaf(v.x, v.x, fmaf(v.y, v.y, fmaf(v.z, v.z, fmaf(v.w, v.w, sq))));
  }
  sq = warp_sum(sq);
  const float r = rsqrtf(sq / d + eps);
  if (lane == 0) rstd[m] = r;
  for (int c = lane; c < d / 4; c += 32) {
    const float4 v = xr[c];
    const long long i = m * d + 4LL * c;
    OpIO<S>::store(y, y_lo, i, v.x * r);
    OpIO<S>::store(y, y_lo, i + 1, v.y * r);
    OpIO<S>::store(y, y_lo, i + 2, v.z * r);
    OpIO<S>::store(y, y_lo, i + 3, v.w * r);
  }
}

template <typename S>
__global__ void rmsnorm_bwd_warp_kernel(int M, int d, const float* __restrict__ x, const float* __restrict__ rstd,
                                        const float* __restrict__ dy, float* __restrict__ dx32, void* dxop,
                                        long long dx_lo) {
  pdl_wait();
  pdl_launch();
  const int lane = threadIdx.x & 31;
  const long long m = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (m >= M) return;
  const float r = rstd[m];
  const float4* xr = reinterpret_cast<const float4*>(x + m * d);
  const float4* dyr = reinterpret_cast<const float4*>(dy + m * d);
  float dot = 0.0f;
  for (int c = lane; c < d / 4; c += 32) {
    const float4 a = xr[c], g = dyr[c];
    dot = fmaf(a.x * r, g.x, fmaf(a.y * r, g.y, fmaf(a.z * r, g.z, fmaf(a.w * r, g.w, dot))));
  }
  dot = warp_sum(dot) / d;
  for (int c = lane; c < d / 4; c += 32) {
    const float4 a = xr[c], g = dyr[c];
    const float4 v = make_float4(r * (g.x - a.x * r * dot), r * (g.y - a.y * r * dot), r * (g.z - a.z * r * dot),
                                 r * (g.w - a.w * r * dot));
    reinterpret_cast<float4*>(dx32 + m * d)[c] = v;
    if (dxop) {
      const long long i = m * d + 4LL * c;
      OpIO<S>::store(dxop, dx_lo, i, v.x);
      OpIO<S>::store(dxop, dx_lo, i + 1, v.y);
      OpIO<S>::store(dxop, dx_lo, i + 2, v.z);
      OpIO<S>::store(dxop, dx_lo, i + 3, v.w);
    }
  }
}

// Combine two online-softmax partial states (max, sum of exp(x - max)).
__device__ __forceinline__ void lse_combine(float& m, float& s, float m2, float s2) {
  if (m2 > m) {
    s = s * __expf(m - m2) + s2;
    m = m2;
  } else if (m2 > -FLT_MAX) {
    s += s2 * __expf(m2 - m);
  }
}

// Block-wide (max, sum-exp) reduction of per-thread online states; returns lse.
__device__ __forceinline__ float block_lse(float mx, float se, float* sm_m, float* sm_s) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, mx, o);
    const float s2 = __shfl_xor_sync(0xffffffffu, se, o);
    lse_combine(mx, se, m2, s2);
  }
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  if (lane == 0) { sm_m[wid] = mx; sm_s[wid] = se; }
  __syncthreads();
  if (wid == 0) {
    mx = lane < nw ? sm_m[lane] : -FLT_MAX;
    se = lane < nw ? sm_s[lane] : 0.0f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float m2 = __shfl_xor_sync(0xffffffffu, mx, o);
      const float s2 = __shfl_xor_sync(0xffffffffu, se, o);
      lse_combine(mx, se, m2, s2);
    }
    if (lane == 0) { sm_m[0] = mx; sm_s[0] = se; }
  }
  __syncthreads();
  return sm_m[0] + logf(sm_s[0]);
}

__device__ __forceinline__ void online_push(float x, float& mx, float& se) {
  if (x > mx) {
    se = se * __expf(mx - x) + 1.0f;
    mx = x;
  } else {
    se += __expf(x - mx);
  }
}

__device__ __forceinline__ int target_of(const TokView& tv, int s, int j, int V) {
  int tgt = tv.tok[s * tv.tok_ld + tv.tok_off + j + 1];
  if ((unsigned)tgt >= (unsigned)V) {
    if (threadIdx.x == 0) atomicOr(tv.err, 2);
    tgt = 0;
  }
  return tgt;
}

template <typename OpT>
__global__ void ce_kernel(TokView tv, int V, OpT* __restrict__ logits, long long ldl, float scale,
                          const float* __restrict__ rscale, bool grad, float* __restrict__ losses,
                          long long loss_ld, long long loss_off, float* __restrict__ row_loss) {
  pdl_wait();
  pdl_launch();
  __shared__ float sm_m[32], sm_s[32];
  const int m = blockIdx.x;
  const int s = m / tv.rows, j = m % tv.rows;
  OpT* row = logits + (long long)m * ldl;
  if (j >= tv.n_valid) {
    if (grad)
      for (int v = threadIdx.x; v < V; v += blockDim.x) row[v] = from_f<OpT>(0.0f);
    return;
  }
  const int tgt = target_of(tv, s, j, V);
  float mx = -FLT_MAX, se = 0.0f;
  for (int v = threadIdx.x; v < V; v += blockDim.x) online_push(to_f(row[v]), mx, se);
  const float lse = block_lse(mx, se, sm_m, sm_s);
  if (threadIdx.x == 0) {
    const float loss = lse - to_f(row[tgt]);
    if (losses) losses[s * loss_ld + loss_off + j] = loss;
    if (row_loss) row_loss[m] = loss;
  }
  if (!grad) return;
  const float sc = rscale ? rscale[m] : scale;
  __syncthreads();   // the target logit is read above before being overwritten
  for (int v = threadIdx.x; v < V; v += blockDim.x) {
    const float p = __expf(to_f(row[v]) - lse);
    row[v] = from_f<OpT>((p - (v == tgt ? 1.0f : 0.0f)) * sc);
  }
}

// fp32 logits in, split dlogits written into the row's own bytes: the row is
// staged in shared memory first, so no thread overwrites a value another
// thread has yet to read.
constexpr int kCeSplitMaxV = 32768;

__global__ void ce_split_kernel(TokView tv, int V, float* __restrict__ logits, long long ldl, float scale,
                                const float* __restrict__ rscale, bool grad, float* __restrict__ losses,
                                long long loss_ld, long long loss_off, float* __restrict__ row_loss) {
  pdl_wait();
  pdl_launch();
  extern __shared__ float srow[];
  __shared__ float sm_m[32], sm_s[32];
  const int m = blockIdx.x;
  const int s = m / tv.rows, j = m % tv.rows;
  float* row = logits + (long long)m * ldl;
  bf16* out = reinterpret_cast<bf16*>(row);
  if (j >= tv.n_valid) {
    if (grad)
      for (int v = threadIdx.x; v < V; v += blockDim.x) {
        out[v] = __float2bfloat16_rn(0.0f);
        out[V + v] = __float2bfloat16_rn(0.0f);
      }
    return;
  }
  const int tgt = target_of(tv, s, j, V);
  float mx = -FLT_MAX, se = 0.0f;
  for (int v = threadIdx.x; v < V; v += blockDim.x) {
    const float x = row[v];
    srow[v] = x;
    online_push(x, mx, se);
  }
  const float lse = block_lse(mx, se, sm_m, sm_s);   // contains __syncthreads
  if (threadIdx.x == 0) {
    const float loss = lse - srow[tgt];
    if (losses) losses[s * loss_ld + loss_off + j] = loss;
    if (row_loss) row_loss[m] = loss;
  }
  if (!grad) return;
  const float sc = rscale ? rscale[m] : scale;
  for (int v = threadIdx.x; v < V; v += blockDim.x) {
    const float g = (__expf(srow[v] - lse) - (v == tgt ? 1.0f : 0.0f)) * sc;
    const bf16 h = __float2bfloat16_rn(g);
    out[v] = h;
    out[V + v] = __float2bfloat16_rn(g - __bfloat162float(h));
  }
}

// ce_split_kernel for rows of at most 512 * EPT logits (V a multiple of 8,
// 16-byte aligned rows): each thread keeps its EPT logits in registers, loaded
// with 16-byte reads all in flight, and writes its hi and lo bf16 pieces with
// 16-byte stores; the row's values are all read before the block reduction,
// so the in-place writes after it cannot overtake a read.
template <int EPT>
__global__ void __launch_bounds__(512) ce_split_reg_kernel(TokView tv, int V, float* __restrict__ logits, long long ldl,
                                                           float scale, const float* __restrict__ rscale, bool grad,
                                                           float* __restrict__ losses, long long loss_ld,
                                                           long long loss_off, float* __restrict__ row_loss) {
  pdl_wait();
  pdl_launch();
  __shared__ float sm_m[32], sm_s[32];
  const int m = blockIdx.x;
  const int s = m / tv.rows, j = m % tv.rows;
  float* row = logits + (long long)m * ldl;
  bf16* out = reinterpret_cast<bf16*>(row);
  const int base = threadIdx.x * EPT;
  const bool mine = base < V;          // V is a multiple of 8 and EPT of 8: whole pieces
  if (j >= tv.n_valid) {
    if (grad && mine)
#pragma unroll
      for (int e = 0; e < EPT; e += 8) {
        reinterpret_cast<uint4*>(out + base + e)[0] = make_uint4(0, 0, 0, 0);
        reinterpret_cast<uint4*>(out + V + base + e)[0] = make_uint4(0, 0, 0, 0);
      }
    return;
  }
  const int tgt = target_of(tv, s, j, V);
  float x[EPT];
  float mx = -FLT_MAX, se = 0.0f;
  if (mine) {
#pragma unroll
    for (int e = 0; e < EPT; e += 4) {
      const float4 q = reinterpret_cast<const float4*>(row + base + e)[0];
      x[e] = q.x; x[e + 1] = q.y; x[e + 2] = q.z; x[e + 3] = q.w;
    }
#pragma unroll
    for (int e = 0; e < EPT; ++e) mx = fmaxf(mx, x[e]);
#pragma unroll
    for (int e = 0; e < EPT; ++e) se += __expf(x[e] - mx);
  }
  const float lse = block_lse(mx, se, sm_m, sm_s);   // contains __syncthreads
  if (mine && tgt >= base && tgt < base + EPT) {
    float xt = x[0];
#pragma unroll
    for (int e = 1; e < EPT; ++e)
      if (tgt == base + e) xt = x[e];
    const float loss = lse - xt;
    if (losses) losses[s * loss_ld + loss_off + j] = loss;
    if (row_loss) row_loss[m] = loss;
  }
  if (!grad || !mine) return;
  const float sc = rscale ? rscale[m] : scale;
#pragma unroll
  for (int e = 0; e < EPT; e += 8) {
    float g[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) g[q] = (__expf(x[e + q] - lse) - (base + e + q == tgt ? 1.0f : 0.0f)) * sc;
    float lo[8];
    const uint4 hi = pack_bf16x8(g);
    float hf[8];
    unpack_bf16x8(hi, hf);
#pragma unroll
    for (int q = 0; q < 8; ++q) lo[q] = g[q] - hf[q];
    reinterpret_cast<uint4*>(out + base + e)[0] = hi;
    reinterpret_cast<uint4*>(out + V + base + e)[0] = pack_bf16x8(lo);
  }
}

// One warp per row: the row's logsumexp from the per-column-tile online
// softmax states the head GEMM left, the target's logit y[m] . U[target] (fp32
// sum of the same bf16 products the GEMM takes), then the loss lse - logit.
__global__ void lse_combine_kernel(TokView tv, int M, const float2* __restrict__ part, long long ld, int nt,
                                   const bf16* __restrict__ y, const bf16* __restrict__ U, int d,
                                   const int32_t* __restrict__ tgt, float* __restrict__ lse,
                                   float* __restrict__ losses, long long loss_ld, long long loss_off,
                                   float* __restrict__ row_loss) {
  pdl_wait();
  pdl_launch();
  const int lane = threadIdx.x & 31;
  const int m = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (m >= M) return;
  const int t = tgt[m];
  float dot = 0.0f;
  if (t >= 0) {
    const bf16* yr = y + (long long)m * d;
    const bf16* ur = U + (long long)t * d;
    if ((d & 7) == 0) {
      // eight products per lane per step from 16-byte loads (rows are 16-byte aligned when d % 8 == 0)
      for (int k = lane * 8; k < d; k += 256) {
        float a[8], b[8];
        unpack_bf16x8(*reinterpret_cast<const uint4*>(yr + k), a);
        unpack_bf16x8(*reinterpret_cast<const uint4*>(ur + k), b);
#pragma unroll
        for (int j = 0; j < 8; ++j) dot = fmaf(a[j], b[j], dot);
      }
    } else {
      for (int k = lane; k < d; k += 32) dot = fmaf(__bfloat162float(yr[k]), __bfloat162float(ur[k]), dot);
    }
    dot = warp_sum(dot);
  }
  float mx = -FLT_MAX, se = 0.0f;
  for (int t = lane; t < nt; t += 32) {
    const float2 p = part[(long long)m * ld + t];
    lse_combine(mx, se, p.x, p.y);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, mx, o);
    const float s2 = __shfl_xor_sync(0xffffffffu, se, o);
    lse_combine(mx, se, m2, s2);
  }
  if (lane == 0) {
    const float l = mx + logf(se);
    lse[m] = l;
    const int s = m / tv.rows, j = m % tv.rows;
    if (j < tv.n_valid) {
      const float loss = l - dot;
      if (losses) losses[s * loss_ld + loss_off + j] = loss;
      if (row_loss) row_loss[m] = loss;
    }
  }
}

// Source Masking: rscale[s * rows + j] = mask_j / max(1, sum of the mask over
// the chunk's rows of sequence s), mask_j = mask[s * mask_ld + off + j] != 0.
__global__ void chunk_row_scale_kernel(int rows, const uint8_t* __restrict__ mask, long long mask_ld, long long off,
                                       float* __restrict__ rscale) {
  pdl_wait();
  pdl_launch();
  __shared__ float red[32];
  const int s = blockIdx.x;
  const uint8_t* mr = mask + s * mask_ld + off;
  float cnt = 0.0f;
  for (int j = threadIdx.x; j < rows; j += blockDim.x) cnt += mr[j] ? 1.0f : 0.0f;
  cnt = block_sum(cnt, red);
  const float inv = 1.0f / fmaxf(cnt, 1.0f);
  for (int j = threadIdx.x; j < rows; j += blockDim.x) rscale[(long long)s * rows + j] = mr[j] ? inv : 0.0f;
}

// dlogits = (softmax - onehot(target)) * scale over bf16 logits [M, V] in place,
// eight elements (16 bytes) per access; rows without a target get 0.  The
// scale is folded into the exponent, exp(x - (lse - ln scale)), and the one
// target element of a row is corrected on its own.  Grid: x over the row's
// 16-byte vectors, y over rows.
constexpr int kDlVec = 4;   // 16-byte vectors per thread, all loaded before any is rewritten

__global__ void dlogits_kernel(int M, int V, bf16* __restrict__ logits, const float* __restrict__ lse,
                               const int32_t* __restrict__ tgt, float scale, const float* __restrict__ rscale) {
  pdl_wait();
  pdl_launch();
  const int nv = V / 8;
  for (int m = blockIdx.y; m < M; m += gridDim.y) {
    uint4* row = reinterpret_cast<uint4*>(logits + (long long)m * V);
    const float sc = rscale ? rscale[m] : scale;
    const int t = sc > 0.0f ? tgt[m] : -1;   // a zero scale (masked row) writes zeros
    const float l = lse[m] - logf(sc > 0.0f ? sc : 1.0f);
    const int i0 = blockIdx.x * blockDim.x * kDlVec + threadIdx.x;
    uint4 buf[kDlVec];
#pragma unroll
    for (int u = 0; u < kDlVec; ++u) {
      const int i = i0 + u * blockDim.x;
      if (t >= 0 && i < nv) buf[u] = row[i];
    }
#pragma unroll
    for (int u = 0; u < kDlVec; ++u) {
      const int i = i0 + u * blockDim.x;
      if (i >= nv) continue;
      if (t < 0) {
        row[i] = make_uint4(0u, 0u, 0u, 0u);
        continue;
      }
      uint4 raw = buf[u];
      __nv_bfloat162* h2 = reinterpret_cast<__nv_bfloat162*>(&raw);
      const int c = i * 8;
      float tx = 0.0f;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float2 x = __bfloat1622float2(h2[q]);
        if ((unsigned)(t - c - 2 * q) < 2u) tx = (t - c - 2 * q) ? x.y : x.x;
        h2[q] = __floats2bfloat162_rn(__expf(x.x - l), __expf(x.y - l));
      }
      if ((unsigned)(t - c) < 8u) {
        bf16* e = reinterpret_cast<bf16*>(&raw) + (t - c);
        *e = __float2bfloat16_rn(__expf(tx - l) - sc);
      }
      row[i] = raw;
    }
  }
}

// One (slot, sequence) segment of n elements per blockIdx.y: W32 -= eta *
// scale[s] * dW, operand copy re-cast; float4 accesses when n is a multiple of 4.
template <typename S>
__global__ void sgd_scale_kernel(int B, long long n, float* __restrict__ W32, void* Wop, long long wop_lo,
                                 const float* __restrict__ dW, const float* __restrict__ scale, float eta) {
  pdl_wait();
  pdl_launch();
  const int s = blockIdx.y % B;
  const float sc = scale[s];
  if (sc == 0.0f) return;  // skipped update (non-finite norm): W stays as it is
  const float step = eta * sc;
  const long long base = (long long)blockIdx.y * n;
  const long long stride = (long long)gridDim.x * blockDim.x;
  if ((n & 3) == 0) {
    float4* w4 = reinterpret_cast<float4*>(W32 + base);
    const float4* g4 = reinterpret_cast<const float4*>(dW + base);
    for (long long q = (long long)blockIdx.x * blockDim.x + threadIdx.x; q < n / 4; q += stride) {
      float4 w = w4[q];
      const float4 gr = g4[q];
      w.x -= step * gr.x; w.y -= step * gr.y; w.z -= step * gr.z; w.w -= step * gr.w;
      w4[q] = w;
      const long long i = base + 4 * q;
      OpIO<S>::store(Wop, wop_lo, i, w.x);
      OpIO<S>::store(Wop, wop_lo, i + 1, w.y);
      OpIO<S>::store(Wop, wop_lo, i + 2, w.z);
      OpIO<S>::store(Wop, wop_lo, i + 3, w.w);
    }
  } else {
    for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < n; e += stride) {
      const float w = W32[base + e] - step * dW[base + e];
      W32[base + e] = w;
      OpIO<S>::store(Wop, wop_lo, base + e, w);
    }
  }
}

// Four consecutive elements i .. i+3 of an operand buffer in one store per
// plane (i a multiple of 4; base and lo offset 4-element aligned).
// Per-sequence clip scale from the dW GEMMs' per-tile sums of squares:
// s = min(1, clip / (norm + 1e-6)) (1 when clip == 0), 0 when the norm is not
// finite.  Every thread of the block receives it; red: >= 32 floats.
__device__ __forceinline__ float seq_clip_scale(const PartialSlots& ps, const float* __restrict__ partials, int s,
                                                float clip, float* red, float* norm_out) {
  float acc = 0.0f;
  for (int k = 0; k < ps.n; ++k) {
    const float* p = partials + ps.off[k] + (long long)s * ps.tiles[k];
    for (int t = threadIdx.x; t < ps.tiles[k]; t += blockDim.x) acc += p[t];
  }
  acc = block_sum(acc, red);
  const float n = sqrtf(acc);
  if (norm_out) *norm_out = n;
  if (!isfinite(n)) return 0.0f;
  return clip > 0.0f ? fminf(1.0f, clip / (n + 1e-6f)) : 1.0f;
}

// One (slot, sequence) segment of n elements per blockIdx.y; every block first
// reduces its sequence's gradient norm from the per-tile partials (a few
// hundred to a few thousand floats, from L2), then W32 -= eta * s * dW and the
// operand copy is re-cast.  float4 accesses when n is a multiple of 4 (every
// fast matrix: n = d * d_ff).
// Four dW values from 16-byte-aligned fp32 or 8-byte-aligned bf16 storage.
__device__ __forceinline__ float4 load_dw4(const float* p, long long i) {
  return *reinterpret_cast<const float4*>(p + i);
}
__device__ __forceinline__ float4 load_dw4(const bf16* p, long long i) {
  const uint2 r = *reinterpret_cast<const uint2*>(p + i);
  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&r.x));
  const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&r.y));
  return make_float4(a.x, a.y, b.x, b.y);
}

template <typename S>
__global__ void sgd_update_kernel(int B, long long n, float* __restrict__ W32, void* Wop, long long wop_lo,
                                  const void* dW_raw, PartialSlots ps, const float* __restrict__ partials,
                                  float clip, float eta, float* __restrict__ scale_out, float* __restrict__ norm_out,
                                  int* __restrict__ flag) {
  pdl_wait();
  pdl_launch();
  __shared__ float red[32];
  const int s = blockIdx.y % B;
  const bool first = blockIdx.x == 0 && blockIdx.y == s;   // slot 0, first block of the sequence
  float nrm = 0.0f;
  const float sc = seq_clip_scale(ps, partials, s, clip, red, &nrm);
  if (first && threadIdx.x == 0) {
    if (scale_out) scale_out[s] = sc;
    if (norm_out) norm_out[s] = nrm;
    if (sc == 0.0f && !isfinite(nrm)) atomicOr(flag, 1);
  }
  if (sc == 0.0f) return;  // skipped update (non-finite norm): W stays as it is
  const float step = eta * sc;
  const long long base = (long long)blockIdx.y * n;
  const long long stride = (long long)gridDim.x * blockDim.x;
  // dW in the epilogue's storage (bf16 for bf16 operands, fp32 otherwise)
  using DT = typename DwType<S>::T;
  const DT* dW = static_cast<const DT*>(dW_raw);
  if ((n & 3) == 0 && (wop_lo & 3) == 0) {
    float4* w4 = reinterpret_cast<float4*>(W32 + base);
    for (long long q = (long long)blockIdx.x * blockDim.x + threadIdx.x; q < n / 4; q += stride) {
      float4 w = w4[q];
      const float4 gr = load_dw4(dW, base + 4 * q);
      w.x -= step * gr.x; w.y -= step * gr.y; w.z -= step * gr.z; w.w -= step * gr.w;
      w4[q] = w;
      QuadIO<S>::store(Wop, wop_lo, base + 4 * q, w);
    }
  } else {
    for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < n; e += stride) {
      const float w = W32[base + e] - step * OpIO<DT>::load(dW, 0, base + e);
      W32[base + e] = w;
      OpIO<S>::store(Wop, wop_lo, base + e, w);
    }
  }
}

// W32[slot][s] = W0[slot] and its operand copy; blockIdx.y = slot * B + s.
template <typename S>
__global__ void broadcast_w0_kernel(int B, long long n, const float* __restrict__ W0, float* __restrict__ W32,
                                    void* Wop, long long wop_lo) {
  pdl_wait();
  pdl_launch();
  const float* src = W0 + (long long)(blockIdx.y / B) * n;
  const long long base = (long long)blockIdx.y * n;
  const long long stride = (long long)gridDim.x * blockDim.x;
  const long long t0 = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if ((n & 3) == 0 && (wop_lo & 3) == 0) {
    for (long long q = t0; q < n / 4; q += stride) {
      const float4 w = reinterpret_cast<const float4*>(src)[q];
      reinterpret_cast<float4*>(W32 + base)[q] = w;
      QuadIO<S>::store(Wop, wop_lo, base + 4 * q, w);
    }
  } else {
    for (long long e = t0; e < n; e += stride) {
      const float w = src[e];
      W32[base + e] = w;
      OpIO<S>::store(Wop, wop_lo, base + e, w);
    }
  }
}

template <typename S>
__global__ void cast_kernel(long long n, const float* __restrict__ in, void* out, long long out_lo) {
  pdl_wait();
  pdl_launch();
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride)
    OpIO<S>::store(out, out_lo, i, in[i]);
}

__global__ void seq_mean_kernel(int rows, int n_valid, const float* __restrict__ row_loss, float* __restrict__ mean) {
  pdl_wait();
  pdl_launch();
  __shared__ float red[32];
  const int s = blockIdx.x;
  float acc = 0.0f;
  for (int j = threadIdx.x; j < n_valid; j += blockDim.x) acc += row_loss[(long long)s * rows + j];
  acc = block_sum(acc, red);
  if (threadIdx.x == 0) mean[s] = acc / n_valid;
}

__global__ void settle_decide_kernel(int B, const float* __restrict__ Lc, const float* __restrict__ Lw,
                                     float* __restrict__ A, uint8_t* __restrict__ accept) {
  pdl_wait();
  pdl_launch();
  const int s = blockIdx.x * blockDim.x + threadIdx.x;
  if (s >= B) return;
  const float a = Lc[s] - Lw[s];
  A[s] = a;
  accept[s] = a >= 0.0f ? 1 : 0;
}

// Settlement's candidate as an offset from the committed weights, in bf16:
// D = bf16(W32 - Wc32); blockIdx.y is one (slot, sequence) segment of n.
__global__ void delta_plane_kernel(long long n, const float* __restrict__ W32, const float* __restrict__ Wc32,
                                   bf16* __restrict__ D) {
  pdl_wait();
  pdl_launch();
  const long long base = (long long)blockIdx.y * n;
  const long long stride = (long long)gridDim.x * blockDim.x;
  const long long t0 = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if ((n & 3) == 0) {
    for (long long q = t0; q < n / 4; q += stride) {
      const float4 w = reinterpret_cast<const float4*>(W32 + base)[q];
      const float4 c = reinterpret_cast<const float4*>(Wc32 + base)[q];
      *reinterpret_cast<uint2*>(D + base + 4 * q) = pack_bf16x4(w.x - c.x, w.y - c.y, w.z - c.z, w.w - c.w);
    }
  } else {
    for (long long e = t0; e < n; e += stride) D[base + e] = __float2bfloat16_rn(W32[base + e] - Wc32[base + e]);
  }
}

// Eight consecutive operand-storage elements copied between two arrays with
// the same lo-plane offset (index a multiple of 8, bases 16-byte aligned).
template <typename S>
__device__ __forceinline__ void copy_op8(void* dst, const void* src, long long lo, long long i) {
  if constexpr (std::is_same<S, float>::value) {
    const float4* s4 = reinterpret_cast<const float4*>(static_cast<const float*>(src) + i);
    float4* d4 = reinterpret_cast<float4*>(static_cast<float*>(dst) + i);
    d4[0] = s4[0];
    d4[1] = s4[1];
  } else {
    const bf16* sb = static_cast<const bf16*>(src);
    bf16* db = static_cast<bf16*>(dst);
    *reinterpret_cast<uint4*>(db + i) = *reinterpret_cast<const uint4*>(sb + i);
    if constexpr (std::is_same<S, Split>::value)
      *reinterpret_cast<uint4*>(db + lo + i) = *reinterpret_cast<const uint4*>(sb + lo + i);
  }
}

// Settlement's commit or revert, per sequence: blockIdx.y is one fast matrix
// of one sequence (slot * B + s), so the decision is uniform over the block;
// a commit copies the current weights (fp32 master and operand copy) into the
// committed ones, a revert copies them back.
template <typename S>
__global__ void settle_apply_kernel(int B, long long n, const uint8_t* __restrict__ accept, float* W32, void* Wop,
                                    float* Wc32, void* Wcop, long long lo) {
  pdl_wait();
  pdl_launch();
  const bool acc = accept[blockIdx.y % B] != 0;
  float* dst32 = acc ? Wc32 : W32;
  const float* src32 = acc ? W32 : Wc32;
  void* dop = acc ? Wcop : Wop;
  const void* sop = acc ? Wop : Wcop;
  const long long base = (long long)blockIdx.y * n;
  const long long stride = (long long)gridDim.x * blockDim.x;
  const long long t0 = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if ((n & 7) == 0 && (lo & 7) == 0) {
    for (long long q = t0; q < n / 8; q += stride) {
      const float4* s4 = reinterpret_cast<const float4*>(src32 + base) + 2 * q;
      float4* d4 = reinterpret_cast<float4*>(dst32 + base) + 2 * q;
      const float4 a = s4[0], b = s4[1];
      d4[0] = a;
      d4[1] = b;
      copy_op8<S>(dop, sop, lo, base + 8 * q);
    }
  } else {
    for (long long e = t0; e < n; e += stride) {
      dst32[base + e] = src32[base + e];
      OpIO<S>::copy(dop, lo, sop, lo, base + e);
    }
  }
}

// Softmax of M rows of V fp32 logits in two launches over S slices per row
// (S * M blocks each, so a few rows still fill the GPU): the first writes
// each slice's (max, sum of exp) state, the second merges the row's S states
// into the logsumexp and writes p = exp(logit - lse) over its slice.
// (max, sum of exp) merge of two softmax states
__device__ __forceinline__ void soft_merge(float& m, float& s, float m2, float s2) {
  const float n = fmaxf(m, m2);
  s = s * expf(m - n) + s2 * expf(m2 - n);
  m = n;
}

constexpr int kSoftBatch = 8;    // logits a thread loads before using any of them

__global__ void softmax_part_kernel(int V, int L, const float* __restrict__ logits, float2* __restrict__ part) {
  pdl_wait();
  pdl_launch();
  __shared__ float2 wstate[32];
  const long long m = blockIdx.y;
  const int v0 = blockIdx.x * L, v1 = min(V, v0 + L);
  const float* row = logits + m * V;
  float mx = -FLT_MAX, se = 0.0f;
  for (int base = v0 + threadIdx.x; base < v1; base += blockDim.x * kSoftBatch) {
    float x[kSoftBatch];
#pragma unroll
    for (int j = 0; j < kSoftBatch; ++j) {
      const int v = base + j * blockDim.x;
      x[j] = v < v1 ? row[v] : -FLT_MAX;
    }
    float bm = x[0];
#pragma unroll
    for (int j = 1; j < kSoftBatch; ++j) bm = fmaxf(bm, x[j]);
    float bs = 0.0f;
#pragma unroll
    for (int j = 0; j < kSoftBatch; ++j)
      if (base + j * (int)blockDim.x < v1) bs += expf(x[j] - bm);
    soft_merge(mx, se, bm, bs);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, mx, o), s2 = __shfl_xor_sync(0xffffffffu, se, o);
    soft_merge(mx, se, m2, s2);
  }
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  if (lane == 0) wstate[wid] = make_float2(mx, se);
  __syncthreads();
  if (threadIdx.x == 0) {
    float m2 = wstate[0].x, s2 = wstate[0].y;
    for (int k = 1; k < nw; ++k) soft_merge(m2, s2, wstate[k].x, wstate[k].y);
    part[m * gridDim.x + blockIdx.x] = make_float2(m2, s2);
  }
}

__global__ void softmax_write_kernel(int V, int L, const float* __restrict__ logits,
                                     const float2* __restrict__ part, float* __restrict__ p,
                                     float* __restrict__ lse_out) {
  pdl_wait();
  pdl_launch();
  const long long m = blockIdx.y;
  const int S = gridDim.x;
  // every thread merges the row's S states in the same order (no shared memory)
  float mx = part[m * S].x, se = part[m * S].y;
  for (int k = 1; k < S; ++k) soft_merge(mx, se, part[m * S + k].x, part[m * S + k].y);
  const float lse = mx + logf(se);
  if (lse_out && blockIdx.x == 0 && threadIdx.x == 0) lse_out[m] = lse;
  const int v0 = blockIdx.x * L, v1 = min(V, v0 + L);
  const float* row = logits + m * V;
  float* prow = p + m * V;
  for (int base = v0 + threadIdx.x; base < v1; base += blockDim.x * kSoftBatch) {
    float x[kSoftBatch];
#pragma unroll
    for (int j = 0; j < kSoftBatch; ++j) {
      const int v = base + j * blockDim.x;
      x[j] = v < v1 ? row[v] : 0.0f;
    }
#pragma unroll
    for (int j = 0; j < kSoftBatch; ++j) {
      const int v = base + j * blockDim.x;
      if (v < v1) prow[v] = expf(x[j] - lse);
    }
  }
}

// loss[s] = lse[s] - logits[s][x]: the next-token loss of x from a softmax
// already taken (the row's logits and logsumexp), x = tok[s * tok_ld + off].
__global__ void next_token_loss_kernel(int B, int V, const float* __restrict__ logits, const float* __restrict__ lse,
                                       const int32_t* __restrict__ tok, long long tok_ld, long long off,
                                       float* __restrict__ loss, int* __restrict__ err) {
  pdl_wait();
  pdl_launch();
  const int s = blockIdx.x * blockDim.x + threadIdx.x;
  if (s >= B) return;
  int x = tok[s * tok_ld + off];
  if ((unsigned)x >= (unsigned)V) {
    atomicOr(err, 2);
    x = 0;
  }
  loss[s] = lse[s] - logits[(long long)s * V + x];
}

__global__ void pending_shift_kernel(int B, int b, int32_t* pend) {
  pdl_wait();
  pdl_launch();
  const int s = blockIdx.x * blockDim.x + threadIdx.x;
  if (s < B) pend[(long long)s * (b + 1)] = pend[(long long)s * (b + 1) + b];
}

// A decoding step's inputs in one launch (one block, B <= its threads): the
// call's status word and (when given) a 4-word grid-barrier state cleared,
// then x_new[s] into column col of the pending buffer (row stride ld) and into
// the forward's token slot x_dev, and, when loss is given, the loss of x_new
// under the cached next-token distribution (as next_token_loss_kernel).
__global__ void decode_inputs_kernel(int B, int ld, int col, const int32_t* x_new, int32_t* pend, int32_t* x_dev,
                                     int* flag, unsigned* bar, int V, const float* logits, const float* lse,
                                     float* loss) {
  pdl_wait();
  pdl_launch();
  if (threadIdx.x == 0) *flag = 0;
  if (bar && threadIdx.x < 4) bar[threadIdx.x] = 0u;
  __syncthreads();   // the cleared status word before any report below
  for (int s = threadIdx.x; s < B; s += blockDim.x) {
    int32_t x = x_new[s];
    pend[(long long)s * ld + col] = x;
    x_dev[s] = x;
    if (loss) {
      if ((unsigned)x >= (unsigned)V) {
        atomicOr(flag, 2);
        x = 0;
      }
      loss[s] = lse[s] - logits[(long long)s * V + x];
    }
  }
}

int grid_for(long long n, int threads) {
  long long g = (n + threads - 1) / threads;
  const long long cap = 148LL * 16;
  return (int)(g < 1 ? 1 : (g > cap ? cap : g));
}

}  // namespace

// Instantiates KERNEL<S> for the storage code and launches it.
#define LAUNCH_BY_STORAGE(stg, KERNEL, GRID, BLOCK, SMEM, STREAM, ...)                      \
  do {                                                                                      \
    if ((stg) == ST_BF16) launch_pdl(KERNEL<bf16>, GRID, BLOCK, SMEM, STREAM, __VA_ARGS__);         \
    else if ((stg) == ST_SPLIT) launch_pdl(KERNEL<Split>, GRID, BLOCK, SMEM, STREAM, __VA_ARGS__);  \
    else launch_pdl(KERNEL<float>, GRID, BLOCK, SMEM, STREAM, __VA_ARGS__);                         \
  } while (0)

// A token view must carry the vocabulary and the status word its kernels
// report out-of-range ids through; a view without them is refused here.
static ttt_status check_view(const TokView& tv) {
  if (!tv.err || tv.vocab <= 0 || !tv.tok) {
    set_error("token view without vocabulary, status word or tokens");
    return TTT_ERR_BAD_ARG;
  }
  return TTT_OK;
}

ttt_status launch_embed(int stg, int B, const TokView& tv, const void* E, int d, float* h32, void* hop,
                        long long hop_lo, cudaStream_t st) {
  const int M = B * tv.rows;
  if (M == 0) return TTT_OK;
  TTT_TRY(check_view(tv));
  if (stg == ST_BF16)
    launch_pdl(embed_kernel<bf16, bf16>, M, 256, 0, st, tv, static_cast<const bf16*>(E), d, h32, hop, hop_lo);
  else if (stg == ST_SPLIT)
    launch_pdl(embed_kernel<float, Split>, M, 256, 0, st, tv, static_cast<const float*>(E), d, h32, hop, hop_lo);
  else
    launch_pdl(embed_kernel<float, float>, M, 256, 0, st, tv, static_cast<const float*>(E), d, h32, hop, hop_lo);
  TTT_CHECK_LAUNCH();
  return TTT_OK;
}

ttt_status launch_rmsnorm_fwd(int stg, int M, int d, const float* x, float eps, void* y, long long y_lo, float* rstd,
                              const TokView* tv, int32_t* tgt, cudaStream_t st) {
  if (M == 0) return TTT_OK;
  if (tv) TTT_TRY(check_view(*tv));
  const TokView tvv = tv ? *tv : TokView();
  // a warp per row pays off once there are enough rows to fill the SMs with warps
  if (M >= 4096 && d % 4 == 0 && (reinterpret_cast<uintptr_t>(x) & 15) == 0)
    LAUNCH_BY_STORAGE(stg, rmsnorm_fwd_warp_kernel, ceil_div(M, 8), 256, 0, st, M, d, x, eps, y, y_lo, rstd, tvv,
                      tv ? tgt : nullptr);
  else
    LAUNCH_BY_STORAGE(stg, rmsnorm_fwd_kernel, M, 256, 0, st, d, x, eps, y, y_lo, rstd, tvv, tv ? tgt : nullptr);
  TTT_CHECK_LAUNCH();
  return TTT_OK;
}

ttt_status launch_rmsnorm_bwd(int stg, int M, int d, const float* x, const float* rstd, const float* dy, float* dx32,
                              void* dxop, long long dx_lo, cudaStream_t st) {
  if (M == 0) return TTT_OK;
  const bool a16 = ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(dy) |
                     reinterpret_cast<uintptr_t>(dx32)) & 15) == 0;
  if (M >= 4096 && d % 4 == 0 && a16)
    LAUNCH_BY_STORAGE(stg, rmsnorm_bwd_warp_kernel, ceil_div(M, 8), 256, 0, st, M, d, x, rstd, dy, dx32, dxop, dx_lo);
  else
    LAUNCH_BY_STORAGE(stg, rmsnorm_bwd_kernel, M, 256, 0, st, d, x, rstd, dy, dx32, dxop, dx_lo);
  TTT_CHECK_LAUNCH();
  return TTT_OK;
}

int ce_split_max_vocab() { return kCeSplitMaxV; }

ttt_status launch_ce(int stg, int B, const TokView& tv, int V, void* logits, long long ldl, float scale,
                     const float* rscale, bool grad, float* losses, long long loss_ld, long long loss_off,
                     float* row_loss, cudaStream_t st) {
  const int M = B * tv.rows;
  if (M == 0) return TTT_OK;
  TTT_TRY(check_view(tv));
  if (stg == ST_SPLIT) {
    if (V > kCeSplitMaxV) {
      set_error("vocabulary too large for the split cross-entropy kernel");
      return TTT_ERR_UNSUPPORTED;
    }
    const bool reg = V % 8 == 0 && ldl % 4 == 0 && (reinterpret_cast<uintptr_t>(logits) & 15) == 0;
    if (reg && V <= 512 * 8) {
      launch_pdl(ce_split_reg_kernel<8>, M, 512, 0, st, tv, V, static_cast<float*>(logits), ldl, scale, rscale, grad,
                 losses, loss_ld, loss_off, row_loss);
    } else if (reg && V <= 512 * 16) {
      launch_pdl(ce_split_reg_kernel<16>, M, 512, 0, st, tv, V, static_cast<float*>(logits), ldl, scale, rscale, grad,
                 losses, loss_ld, loss_off, row_loss);
    } else {
      const size_t smem = (size_t)V * sizeof(float);
      TTT_CUDA(ensure_dyn_smem((const void*)ce_split_kernel, smem));
      launch_pdl(ce_split_kernel, M, 512, smem, st, tv, V, static_cast<float*>(logits), ldl, scale, rscale, grad,
                 losses, loss_ld, loss_off, row_loss);
    }
  } else if (stg == ST_BF16) {
    launch_pdl(ce_kernel<bf16>, M, 512, 0, st, tv, V, static_cast<bf16*>(logits), ldl, scale, rscale, grad, losses, loss_ld,
                                       loss_off, row_loss);
  } else {
    launch_pdl(ce_kernel<float>, M, 512, 0, st, tv, V, static_cast<float*>(logits), ldl, scale, rscale, grad, losses, loss_ld,
                                        loss_off, row_loss);
  }
  TTT_CHECK_LAUNCH();
  return TTT_OK;
}

ttt_status launch_lse_combine(int B, const TokView& tv, const float2* part, long long ld, int nt, const void* y,
                              const void* U, int d, const int32_t* tgt, float* lse, float* losses, long long loss_ld,
                              long long loss_off, float* row_loss, cudaStream_t st) {
  const int M = B * tv.rows;
  if (M == 0) return TTT_OK;
  TTT_TRY(check_view(tv));
  launch_pdl(lse_combine_kernel, ceil_div(M, 8), 256, 0, st, tv, M, part, ld, nt, static_cast<const bf16*>(y),
                                                    static_cast<const bf16*>(U), d, tgt, lse, losses, loss_ld,
                                                    loss_off, row_loss);
  TTT_CHECK_LAUNCH();
  return TTT_OK;
}

ttt_status launch_chunk_row_scale(int B, int rows, const uint8_t* mask, long long mask_ld, long long off,
                                  float* rscale, cudaStream_t st) {
  if (B == 0 || rows == 0) return TTT_OK;
  launch_pdl(chunk_row_scale_kernel, B, 256, 0, st, rows, mask, mask_ld, off, rscale);
  TTT_CHECK_LAUNCH();
  return TTT_OK;
}

ttt_status launch_dlogits(int M, int V, void* logits, const float* lse, const int32_t* tgt, float scale,
                          const float* rscale, cudaStream_t st) {
  if (M == 0) return TTT_OK;
  if (V % 8 || (reinterpret_cast<uintptr_t>(logits) & 15)) {
    set_error("dlogits: V must be a multiple of 8 and the logits 16-byte aligned");
    return TTT_ERR_UNSUPPORTED;
  }
  // 256-thread blocks each cover 256 * kDlVec 16-byte vectors of a row; rows fill the rest of the grid
  const int bx = ceil_div(V / 8, 256 * kDlVec);
  const int by = M < 65535 ? M : 65535;
  launch_pdl(dlogits_kernel, dim3(bx, by), 256, 0, st, M, V, static_cast<bf16*>(logits), lse, tgt, scale, rscale);
  TTT_CHECK_LAUNCH();
  return TTT_OK;
}

static dim3 update_grid(int nslots, int B, long long n) {
  // blocks per segment: enough for ~16 blocks per SM over all segments
  const int segs = nslots * B;
  long long per = ((n + 3) / 4 + 255) / 256;
  const long long cap = (148LL * 16 + segs - 1) / segs;
  if (per > cap) per = cap;
  if (per < 1) per = 1;
  return dim3((unsigned)per, (unsigned)segs);
}

ttt_status launch_sgd_update(int stg, int nslots, int B, long long n, float* W32, void* Wop, long long wop_lo,
                             const float* dW, const float* scale, float eta, cudaStream_t st) {
  const dim3 grid = update_grid(nslots, B, n);
  LAUNCH_BY_STORAGE(stg, sgd_scale_kernel, grid, 256, 0, st, B, n, W32, Wop, wop_lo, dW, scale, eta);
  TTT_CHECK_LAUNCH();
  return TTT_OK;
}

ttt_status launch_clip_sgd_update(int stg, int nslots, int B, long long n, float* W32, void* Wop, long long wop_lo,
                                  const void* dW, const PartialSlots& ps, const float* partials, float clip,
                                  float eta, float* scale_out, float* norm_out, int* flag, cudaStream_t st) {
  const dim3 grid = update_grid(nslots, B, n);
  LAUNCH_BY_STORAGE(stg, sgd_update_kernel, grid, 256, 0, st, B, n, W32, Wop, wop_lo, dW, ps, partials, clip, eta,
                    scale_out, norm_out, flag);
  TTT_CHECK_LAUNCH();
  return TTT_OK;
}

ttt_status launch_broadcast_w0(int stg, int nslots, int B, long long n, const float* W0, float* W32, void* Wop,
                               long long wop_lo, cudaStream_t st) {
  const dim3 g = update_grid(nslots, B, n);
  LAUNCH_BY_STORAGE(stg, broadcast_w0_kernel, g, 256, 0, st, B, n, W0, W32, Wop, wop_lo);
  TTT_CHECK_LAUNCH();
  return TTT_OK;
}

ttt_status launch_cast(int stg, long long n, const float* in, void* out, long long out_lo, cudaStream_t st) {
  const int g = grid_for(n, 256);
  LAUNCH_BY_STORAGE(stg, cast_kernel, g, 256, 0, st, n, in, out, out_lo);
  TTT_CHECK_LAUNCH();
  return TTT_OK;
}

ttt_status launch_seq_mean(int B, int rows, int n_valid, const float* row_loss, float* mean, cudaStream_t st) {
  launch_pdl(seq_mean_kernel, B, 256, 0, st, rows, n_valid, row_loss, mean);
  TTT_CHECK_LAUNCH();
  return TTT_OK;
}

ttt_status launch_settle_apply(int stg, int nslots, int B, long long n, const float* Lc, const float* Lw, float* A,
                               uint8_t* accept, float* W32, void* Wop, float* Wc32, void* Wcop, long long op_lo,
                               cudaStream_t st) {
  launch_pdl(settle_decide_kernel, ceil_div(B, 128), 128, 0, st, B, Lc, Lw, A, accept);
  TTT_CHECK_LAUNCH();
  const dim3 g = update_grid(nslots, B, n);
  LAUNCH_BY_STORAGE(stg, settle_apply_kernel, g, 256, 0, st, B, n, accept, W32, Wop, Wc32, Wcop, op_lo);
  TTT_CHECK_LAUNCH();
  return TTT_OK;
}

ttt_status launch_delta_plane(int nslots, int B, long long n, const float* W32, const float* Wc32, void* D,
                              cudaStream_t st) {
  const dim3 g = update_grid(nslots, B, n);
  launch_pdl(delta_plane_kernel, g, 256, 0, st, n, W32, Wc32, static_cast<bf16*>(D));
  TTT_CHECK_LAUNCH();
  return TTT_OK;
}

ttt_status launch_next_token_loss(int B, int V, const float* logits32, const float* lse, const int32_t* tok,
                                  long long tok_ld, long long off, float* loss, int* err, cudaStream_t st) {
  launch_pdl(next_token_loss_kernel, ceil_div(B, 128), 128, 0, st, B, V, logits32, lse, tok, tok_ld, off, loss, err);
  TTT_CHECK_LAUNCH();
  return TTT_OK;
}

int softmax_slices(int M, int V) {
  int S = ceil_div(148 * 4, M > 0 ? M : 1);
  if (S > kSoftmaxMaxSlices) S = kSoftmaxMaxSlices;
  const int by_len = ceil_div(V, 256);       // at least 256 logits per slice
  if (S > by_len) S = by_len;
  return S < 1 ? 1 : S;
}

ttt_status launch_softmax(int M, int V, const float* logits32, float* p, float* lse, float2* part, cudaStream_t st) {
  if (M == 0) return TTT_OK;
  const int S = softmax_slices(M, V), L = ceil_div(V, S);
  launch_pdl(softmax_part_kernel, dim3(S, M), 256, 0, st, V, L, logits32, part);
  TTT_CHECK_LAUNCH();
  launch_pdl(softmax_write_kernel, dim3(S, M), 256, 0, st, V, L, logits32, (const float2*)part, p, lse);
  TTT_CHECK_LAUNCH();
  return TTT_OK;
}

ttt_status launch_decode_inputs(int B, int ld, int col, const int32_t* x_new, int32_t* pend, int32_t* x_dev,
                                int* flag, unsigned* bar, int V, const float* logits32, const float* lse,
                                float* loss, cudaStream_t st) {
  launch_pdl(decode_inputs_kernel, 1, 256, 0, st, B, ld, col, x_new, pend, x_dev, flag, bar, V, logits32, lse, loss);
  TTT_CHECK_LAUNCH();
  return TTT_OK;
}

ttt_status launch_pending_shift(int B, int b, int32_t* pend, cudaStream_t st) {
  launch_pdl(pending_shift_kernel, ceil_div(B, 128), 128, 0, st, B, b, pend);
  TTT_CHECK_LAUNCH();
  return TTT_OK;
}

}  // namespace ttt
