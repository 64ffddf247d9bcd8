// Sliding-window multi-head attention of the frozen blocks, forward only
// ("End-to-End TTT" review, Method: the sliding-window attention layer of
// window k that lets a chunk remember its own tokens before the update; 3.1:
// attention layers stay frozen during TTT).
//
// One block per (sequence, head, tile of 64 query positions): the tile's
// queries stay in shared memory while the key/value tiles of 64 positions
// that the window reaches (t - k + 1 .. t, clipped at 0) stream through it.
// 256 threads as 16 x 16: thread (ty, tx) owns query rows ty + 16 i and, for
// the scores, key columns tx + 16 j (i, j < 4); each row's 16 owners sit in
// one half-warp and keep its online-softmax state (running max, running
// sum) with shuffles.  Probabilities go through shared memory to the P V
// product, where the same thread owns output columns tx + 16 c.  Rows are
// padded by one float so that the strided column reads hit distinct banks.
// Q, K and V come from one fp32 projection buffer [B][rows][3d] (Q | K | V
// per row); the output is written in the operand type for the Wo projection.
#include <cfloat>

#include "kernels.h"

namespace ttt {
namespace {

constexpr int kTile = 64;            // query and key positions per tile
constexpr int kMaxDh = 128;          // head dimension limit
constexpr int kOutCols = kMaxDh / 16;
constexpr int kTc = kSwaTcRows;      // query rows per score block of the tensor-core path

size_t swa_smem_bytes(int dh) { return (size_t)(3 * kTile * (dh + 1) + kTile * (kTile + 1)) * sizeof(float); }

template <typename S>
__global__ void __launch_bounds__(256)
    swa_tile_kernel(int rows, int H, int dh, int window, float scale, const float* __restrict__ qkv, void* out,
                    long long out_lo) {
  pdl_wait();
  pdl_launch();
  extern __shared__ float sm[];
  const int dp = dh + 1;
  float* Qs = sm;                    // [kTile][dp]
  float* Ks = Qs + kTile * dp;       // [kTile][dp]
  float* Vs = Ks + kTile * dp;       // [kTile][dp]
  float* Ps = Vs + kTile * dp;       // [kTile][kTile + 1]
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  const int head = blockIdx.y;
  const int d = H * dh;
  const long long ld = 3LL * d;
  const long long seq0 = (long long)blockIdx.z * rows;
  const int q0 = blockIdx.x * kTile;

  // the query tile, pre-scaled by 1/sqrt(dh); rows past the sequence read 0
  for (int i = tid; i < kTile * dh; i += 256) {
    const int r = i / dh, e = i % dh;
    Qs[r * dp + e] = q0 + r < rows ? qkv[(seq0 + q0 + r) * ld + (long long)head * dh + e] * scale : 0.0f;
  }
  float m[4], l[4], acc[4][kOutCols];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    m[i] = -FLT_MAX;
    l[i] = 0.0f;
#pragma unroll
    for (int c = 0; c < kOutCols; ++c) acc[i][c] = 0.0f;
  }
  const int lo = q0 - window + 1 > 0 ? q0 - window + 1 : 0;
  const int hi = q0 + kTile - 1 < rows - 1 ? q0 + kTile - 1 : rows - 1;
  for (int k0 = (lo / kTile) * kTile; k0 <= hi; k0 += kTile) {
    __syncthreads();   // the previous tile's P V reads are done (and the Q tile is stored)
    for (int i = tid; i < kTile * dh; i += 256) {
      const int r = i / dh, e = i % dh;
      const bool in = k0 + r < rows;
      const long long row = (seq0 + k0 + r) * ld + (long long)head * dh + e;
      Ks[r * dp + e] = in ? qkv[row + d] : 0.0f;
      Vs[r * dp + e] = in ? qkv[row + 2LL * d] : 0.0f;
    }
    __syncthreads();
    float sc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) sc[i][j] = 0.0f;
    for (int e = 0; e < dh; ++e) {
      float qv[4], kv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) qv[i] = Qs[(ty + 16 * i) * dp + e];
#pragma unroll
      for (int j = 0; j < 4; ++j) kv[j] = Ks[(tx + 16 * j) * dp + e];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) sc[i][j] = fmaf(qv[i], kv[j], sc[i][j]);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int qp = q0 + ty + 16 * i;
      bool ok[4];
      float rmax = -FLT_MAX;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int kp = k0 + tx + 16 * j;
        ok[j] = kp <= qp && kp > qp - window && kp < rows;
        if (ok[j]) rmax = fmaxf(rmax, sc[i][j]);
      }
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) rmax = fmaxf(rmax, __shfl_xor_sync(0xffffffffu, rmax, o));
      const float mn = fmaxf(m[i], rmax);
      const float corr = expf(m[i] - mn);
      float rsum = 0.0f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float p = ok[j] ? expf(sc[i][j] - mn) : 0.0f;
        rsum += p;
        Ps[(ty + 16 * i) * (kTile + 1) + tx + 16 * j] = p;
      }
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) rsum += __shfl_xor_sync(0xffffffffu, rsum, o);
      l[i] = l[i] * corr + rsum;
      m[i] = mn;
#pragma unroll
      for (int c = 0; c < kOutCols; ++c) acc[i][c] *= corr;
    }
    __syncthreads();
    for (int key = 0; key < kTile; ++key) {
      float pv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) pv[i] = Ps[(ty + 16 * i) * (kTile + 1) + key];
#pragma unroll
      for (int c = 0; c < kOutCols; ++c) {
        const int col = tx + 16 * c;
        if (col < dh) {
          const float v = Vs[key * dp + col];
#pragma unroll
          for (int i = 0; i < 4; ++i) acc[i][c] = fmaf(pv[i], v, acc[i][c]);
        }
      }
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int qp = q0 + ty + 16 * i;
    if (qp >= rows) continue;
    const float inv = 1.0f / l[i];
#pragma unroll
    for (int c = 0; c < kOutCols; ++c) {
      const int col = tx + 16 * c;
      if (col < dh) OpIO<S>::store(out, out_lo, (seq0 + qp) * d + (long long)head * dh + col, acc[i][c] * inv);
    }
  }
}

template <typename S>
ttt_status launch_swa_typed(int B, int rows, int H, int dh, int window, const float* qkv, void* out,
                            long long out_lo, cudaStream_t st) {
  const size_t smem = swa_smem_bytes(dh);
  TTT_CUDA(ensure_dyn_smem((const void*)swa_tile_kernel<S>, smem));
  const dim3 grid(ceil_div(rows, kTile), H, B);
  launch_pdl(swa_tile_kernel<S>, grid, 256, smem, st, rows, H, dh, window, 1.0f / sqrtf((float)dh), qkv, out,
             out_lo);
  TTT_CHECK_LAUNCH();
  return TTT_OK;
}

// Masked row softmax of the score blocks of the tensor-core path.  Block j of
// a sequence holds query rows j*kTc .. j*kTc + kTc - 1 of the padded row space
// (position = row - pad) and nw window keys starting at padded row
// j*kTc + kTc - nw; batch entry e is block j0 + e of the flattened (sequence,
// block) space.  One warp per row: the valid keys (t - k < s <= t, s >= 0,
// t < rows) form one contiguous range of n; P = exp(S - max) / sum there and
// 0 elsewhere, written in the operand type (rows of no real query are all 0).
// 16-byte score loads (nw is a multiple of 16), 4-element stores; a row
// (nw fp32) stays in L1 across its three passes.  The exponentials use the
// fast __expf (relative error about 1e-6 over the clipped range of
// max-subtracted scores).
template <typename S>
__global__ void __launch_bounds__(256)
    band_softmax_kernel(long long nrows, int nw, int nqb, int j0, int pad, int rows, int window, float scale,
                        const float* __restrict__ Sc, void* P, long long p_lo) {
  pdl_wait();
  pdl_launch();
  const long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= nrows) return;          // whole warps leave; no block synchronisation below
  const long long e = row / kTc;
  const int r = (int)(row % kTc);
  const long long J = e + j0;
  const int j = (int)(J % nqb);
  const int qpos = j * kTc + r - pad;
  const int ws = j * kTc + kTc - nw;             // padded row of window key 0
  int n_lo = 0, n_hi = -1;                        // valid keys n_lo .. n_hi
  if (qpos >= 0 && qpos < rows) {
    n_hi = qpos + pad - ws;                       // key position == qpos
    n_lo = n_hi - window + 1;
    if (pad - ws > n_lo) n_lo = pad - ws;         // key position >= 0
    if (n_lo < 0) n_lo = 0;
  }
  const float4* s4 = reinterpret_cast<const float4*>(Sc + row * nw);
  const int q_lo = n_lo >> 2, q_hi = n_hi >= 0 ? n_hi >> 2 : -1;
  float mx = -FLT_MAX;
  for (int q = q_lo + lane; q <= q_hi; q += 32) {
    const float4 v = s4[q];
    const float x[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int c = 0; c < 4; ++c)
      if (4 * q + c >= n_lo && 4 * q + c <= n_hi) mx = fmaxf(mx, x[c] * scale);
  }
  mx = warp_max(mx);
  float se = 0.0f;
  for (int q = q_lo + lane; q <= q_hi; q += 32) {
    const float4 v = s4[q];
    const float x[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int c = 0; c < 4; ++c)
      if (4 * q + c >= n_lo && 4 * q + c <= n_hi) se += __expf(x[c] * scale - mx);
  }
  se = warp_sum(se);
  const float inv = n_hi >= n_lo ? 1.0f / se : 0.0f;
  for (int q = lane; q < nw / 4; q += 32) {
    float o[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    if (q >= q_lo && q <= q_hi) {
      const float4 v = s4[q];
      const float x[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int c = 0; c < 4; ++c)
        if (4 * q + c >= n_lo && 4 * q + c <= n_hi) o[c] = __expf(x[c] * scale - mx) * inv;
    }
    QuadIO<S>::store(P, p_lo, row * nw + 4LL * q, make_float4(o[0], o[1], o[2], o[3]));
  }
}

// Key/value cache of decoding: per frozen block, the K and V rows of the last
// `window` positions of every sequence, fp32, slot = position % window
// ([B][window][d] each).  Filled from a whole-sequence pass's projections
// (rows row0 + pos of a per-sequence stride of seq_rows rows, 3d wide: Q | K | V).
template <typename S>
__global__ void kv_fill_kernel(int R, int window, int d, const void* __restrict__ src, long long src_lo,
                               long long seq_rows, long long row0, float* __restrict__ ck, float* __restrict__ cv) {
  pdl_wait();
  pdl_launch();
  const long long s = blockIdx.y;
  const int n = R < window ? R : window;
  const int p0 = R - n;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < (long long)n * d;
       i += (long long)gridDim.x * blockDim.x) {
    const int pos = p0 + (int)(i / d), e = (int)(i % d);
    const long long r = (s * seq_rows + row0 + pos) * 3LL * d;
    const long long c = (s * window + pos % window) * d + e;
    ck[c] = OpIO<S>::load(src, src_lo, r + d + e);
    cv[c] = OpIO<S>::load(src, src_lo, r + 2LL * d + e);
  }
}

// One decoded position per sequence (`*pos_ptr`, the same for every
// sequence), the keys of the window being positions pos - j, j = 0 .. n - 1,
// n = min(pos + 1, window).  Split-window online softmax: the window is cut
// into nsplit ranges of j, one block of kDecThreads per (head, sequence,
// range); in a block each half-warp takes four keys at a time (its 16 lanes
// read 16 consecutive elements of each key's K and V rows, so a warp's loads
// are contiguous row pieces, and all eight rows' loads are in flight before
// any is used), folds the scores into a running (max, sum, output) state, and
// the block merges its 16 states.  NE: row elements per lane, dh / 16 rounded
// up.  Split 0 appends the new
// row's K and V to the cache; every split reads key 0 from the Q | K | V row
// itself.  With more than one split, each block stores its state and the last
// block of a (head, sequence) to finish (an arrival count it resets to zero)
// merges them into the output.
constexpr int kDecThreads = 256;
constexpr int kDecHalves = kDecThreads / 16;
constexpr int kDecSplitMax = 8;
constexpr int kDecU = 4;              // keys a half-warp loads at once

__device__ __forceinline__ float half_sum(float v) {
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

template <typename S, int NE>
__global__ void __launch_bounds__(kDecThreads)
    swa_decode_kernel(int H, int dh, int window, int nsplit, float scale, const int* __restrict__ pos_ptr,
                      const float* __restrict__ qkv, float* __restrict__ ck, float* __restrict__ cv,
                      float* __restrict__ part, int* __restrict__ cnt, void* out, long long out_lo) {
  pdl_wait();
  pdl_launch();
  __shared__ float hm[kDecHalves], hs[kDecHalves], ho[kDecHalves][kMaxDh];
  __shared__ int last;
  const int head = blockIdx.x, sp = blockIdx.z, tid = threadIdx.x;
  const long long s = blockIdx.y;
  const int d = H * dh;
  const int pos = *pos_ptr;
  const int slot = pos % window;
  const float* row = qkv + s * 3LL * d;
  float* kc = ck + s * (long long)window * d + (long long)head * dh;
  float* vc = cv + s * (long long)window * d + (long long)head * dh;
  if (sp == 0)
    for (int e = tid; e < dh; e += kDecThreads) {
      kc[(long long)slot * d + e] = row[d + head * dh + e];
      vc[(long long)slot * d + e] = row[2 * d + head * dh + e];
    }
  const int n = pos + 1 < window ? pos + 1 : window;
  const int per = (n + nsplit - 1) / nsplit;
  const int j0 = sp * per, j1 = min(n, j0 + per);
  const int hw = tid >> 4, hl = tid & 15;
  float q[NE], o[NE];
#pragma unroll
  for (int c = 0; c < NE; ++c) {
    const int e = hl + 16 * c;
    q[c] = e < dh ? row[head * dh + e] * scale : 0.0f;
    o[c] = 0.0f;
  }
  float m = -INFINITY, l = 0.0f;
  // Both half-warps of a warp take the same steps (the trip count follows the
  // warp's first half-warp; keys past j1 are masked), so the full-warp
  // shuffles of half_sum always find all 32 lanes.
  for (int jw = j0 + (hw & ~1); jw < j1; jw += kDecU * kDecHalves) {
    const int jb = jw + (hw & 1);   // this half-warp's first key of the step
    float kv[kDecU][NE], vv[kDecU][NE];
#pragma unroll
    for (int u = 0; u < kDecU; ++u) {
      const int j = jb + u * kDecHalves;
      const bool in = j < j1;
      const long long r = in && j > 0 ? (long long)((pos - j) % window) * d : 0;
      const float* kr = j == 0 ? row + d + head * dh : kc + r;
      const float* vr = j == 0 ? row + 2 * d + head * dh : vc + r;
#pragma unroll
      for (int c = 0; c < NE; ++c) {
        const int e = hl + 16 * c;
        kv[u][c] = in && e < dh ? kr[e] : 0.0f;
        vv[u][c] = in && e < dh ? vr[e] : 0.0f;
      }
    }
    float a[kDecU];
#pragma unroll
    for (int u = 0; u < kDecU; ++u) {
      float t = 0.0f;
#pragma unroll
      for (int c = 0; c < NE; ++c) t = fmaf(q[c], kv[u][c], t);
      a[u] = t;
    }
#pragma unroll
    for (int u = 0; u < kDecU; ++u) a[u] = half_sum(a[u]);
#pragma unroll
    for (int u = 0; u < kDecU; ++u) {
      if (jb + u * kDecHalves >= j1) break;
      if (a[u] > m) {
        const float al = expf(m - a[u]);   // 0 for the first key
        l *= al;
#pragma unroll
        for (int c = 0; c < NE; ++c) o[c] *= al;
        m = a[u];
      }
      const float pj = expf(a[u] - m);
      l += pj;
#pragma unroll
      for (int c = 0; c < NE; ++c) o[c] = fmaf(pj, vv[u][c], o[c]);
    }
  }
  if (hl == 0) {
    hm[hw] = m;
    hs[hw] = l;
  }
#pragma unroll
  for (int c = 0; c < NE; ++c) {
    const int e = hl + 16 * c;
    if (e < dh) ho[hw][e] = o[c];
  }
  __syncthreads();
  // the block's state: M = max over half-warps, L and O rescaled to it (a
  // half-warp without keys has l = 0 and contributes nothing)
  float M = -INFINITY;
  for (int w = 0; w < kDecHalves; ++w)
    if (hs[w] > 0.0f) M = fmaxf(M, hm[w]);
  float L = 0.0f, O = 0.0f;
  if (tid < dh) {
    for (int w = 0; w < kDecHalves; ++w)
      if (hs[w] > 0.0f) {
        const float f = expf(hm[w] - M);
        L = fmaf(hs[w], f, L);
        O = fmaf(ho[w][tid], f, O);
      }
  }
  const long long o_at = s * d + (long long)head * dh + tid;
  if (nsplit == 1) {
    if (tid < dh) OpIO<S>::store(out, out_lo, o_at, O / L);
    return;
  }
  const long long hsq = s * H + head;
  float* mine = part + (hsq * nsplit + sp) * (kMaxDh + 2);
  if (tid < dh) mine[2 + tid] = O;
  if (tid == 0) {
    mine[0] = M;
    mine[1] = L;
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const int prev = atomicAdd(&cnt[hsq], 1);
    last = prev == nsplit - 1;
    if (last) {
      cnt[hsq] = 0;   // ready for the next step, in stream order
      __threadfence();
    }
  }
  __syncthreads();
  if (!last || tid >= dh) return;
  const float* all = part + hsq * nsplit * (kMaxDh + 2);
  float MM = -INFINITY;
  for (int r = 0; r < nsplit; ++r)
    if (__ldcg(all + r * (kMaxDh + 2) + 1) > 0.0f) MM = fmaxf(MM, __ldcg(all + r * (kMaxDh + 2)));
  float LL = 0.0f, OO = 0.0f;
  for (int r = 0; r < nsplit; ++r) {
    const float lr = __ldcg(all + r * (kMaxDh + 2) + 1);
    if (lr > 0.0f) {
      const float f = expf(__ldcg(all + r * (kMaxDh + 2)) - MM);
      LL = fmaf(lr, f, LL);
      OO = fmaf(__ldcg(all + r * (kMaxDh + 2) + 2 + tid), f, OO);
    }
  }
  OpIO<S>::store(out, out_lo, o_at, OO / LL);
}

__global__ void pos_set_kernel(int* p, int v) {
  pdl_wait();
  pdl_launch();
  *p = v;
}

__global__ void pos_add_kernel(int* p) {
  pdl_wait();
  pdl_launch();
  *p += 1;
}

}  // namespace

ttt_status launch_pos_set(int* p, int v, cudaStream_t st) {
  launch_pdl(pos_set_kernel, 1, 1, 0, st, p, v);
  TTT_CHECK_LAUNCH();
  return TTT_OK;
}

ttt_status launch_pos_add(int* p, cudaStream_t st) {
  launch_pdl(pos_add_kernel, 1, 1, 0, st, p);
  TTT_CHECK_LAUNCH();
  return TTT_OK;
}

ttt_status launch_kv_fill(int stg, int B, int R, int window, int d, const void* src, long long src_lo,
                          long long seq_rows, long long row0, float* ck, float* cv, cudaStream_t st) {
  if (B == 0 || R == 0) return TTT_OK;
  const long long n = (long long)(R < window ? R : window) * d;
  const int gx = (int)((n + 255) / 256 < 1024 ? (n + 255) / 256 : 1024);
  if (stg == ST_BF16)
    launch_pdl(kv_fill_kernel<bf16>, dim3(gx, B), 256, 0, st, R, window, d, src, src_lo, seq_rows, row0, ck, cv);
  else if (stg == ST_SPLIT)
    launch_pdl(kv_fill_kernel<Split>, dim3(gx, B), 256, 0, st, R, window, d, src, src_lo, seq_rows, row0, ck, cv);
  else
    launch_pdl(kv_fill_kernel<float>, dim3(gx, B), 256, 0, st, R, window, d, src, src_lo, seq_rows, row0, ck, cv);
  TTT_CHECK_LAUNCH();
  return TTT_OK;
}

size_t swa_decode_smem_bytes(int window, int dh) {
  (void)window;
  (void)dh;
  return sizeof(float) * (2 * kDecHalves + kDecHalves * kMaxDh) + sizeof(int);
}

int swa_decode_splits(int window) {
  const int sp = (window + 255) / 256;
  return sp < 1 ? 1 : (sp > kDecSplitMax ? kDecSplitMax : sp);
}

size_t swa_decode_work_floats(int B, int H) { return (size_t)B * H * kDecSplitMax * (kMaxDh + 2); }

template <typename S>
static ttt_status launch_swa_decode_typed(int B, int H, int dh, int window, const int* pos, const float* qkv,
                                          float* ck, float* cv, float* work, int* cnt, void* out, long long out_lo,
                                          cudaStream_t st) {
  const int nsplit = swa_decode_splits(window);
  const dim3 grid(H, B, nsplit);
  const float scale = 1.0f / sqrtf((float)dh);
  switch ((dh + 15) / 16) {
#define TTT_DEC_CASE(ne)                                                                                        \
  case ne:                                                                                                      \
    launch_pdl(swa_decode_kernel<S, ne>, grid, kDecThreads, 0, st, H, dh, window, nsplit, scale, pos, qkv, ck, \
               cv, work, cnt, out, out_lo);                                                                     \
    break;
    TTT_DEC_CASE(1)
    TTT_DEC_CASE(2)
    TTT_DEC_CASE(3)
    TTT_DEC_CASE(4)
    TTT_DEC_CASE(5)
    TTT_DEC_CASE(6)
    TTT_DEC_CASE(7)
    TTT_DEC_CASE(8)
#undef TTT_DEC_CASE
    default:
      set_error("decoding attention: head width above 128");
      return TTT_ERR_UNSUPPORTED;
  }
  TTT_CHECK_LAUNCH();
  return TTT_OK;
}

ttt_status launch_swa_decode(int stg, int B, int H, int dh, int window, const int* pos, const float* qkv, float* ck,
                             float* cv, float* work, int* cnt, void* out, long long out_lo, cudaStream_t st) {
  if (B == 0) return TTT_OK;
  if (dh < 1 || dh > kMaxDh || window < 1 || !work || !cnt) {
    set_error("decoding attention: head width 1..128, a window, a workspace and arrival counters");
    return TTT_ERR_UNSUPPORTED;
  }
  if (stg == ST_BF16)
    return launch_swa_decode_typed<bf16>(B, H, dh, window, pos, qkv, ck, cv, work, cnt, out, out_lo, st);
  if (stg == ST_SPLIT)
    return launch_swa_decode_typed<Split>(B, H, dh, window, pos, qkv, ck, cv, work, cnt, out, out_lo, st);
  return launch_swa_decode_typed<float>(B, H, dh, window, pos, qkv, ck, cv, work, cnt, out, out_lo, st);
}

ttt_status launch_band_softmax(int stg, long long nbatch, int nw, int nqb, int j0, int pad, int rows, int window,
                               float scale, const float* Sc, void* P, long long p_lo, cudaStream_t st) {
  const long long nrows = nbatch * kTc;
  if (nrows == 0) return TTT_OK;
  const int grid = (int)((nrows + 7) / 8);
  if (stg == ST_BF16)
    launch_pdl(band_softmax_kernel<bf16>, grid, 256, 0, st, nrows, nw, nqb, j0, pad, rows, window, scale, Sc, P,
               p_lo);
  else if (stg == ST_SPLIT)
    launch_pdl(band_softmax_kernel<Split>, grid, 256, 0, st, nrows, nw, nqb, j0, pad, rows, window, scale, Sc, P,
               p_lo);
  else
    launch_pdl(band_softmax_kernel<float>, grid, 256, 0, st, nrows, nw, nqb, j0, pad, rows, window, scale, Sc, P,
               p_lo);
  TTT_CHECK_LAUNCH();
  return TTT_OK;
}

bool swa_supported(int d, int heads) { return heads > 0 && d % heads == 0 && d / heads <= kMaxDh; }

ttt_status launch_swa(int stg, int B, int rows, int H, int dh, int window, const float* qkv, void* out,
                      long long out_lo, cudaStream_t st) {
  if (B == 0 || rows == 0) return TTT_OK;
  if (stg == ST_BF16) return launch_swa_typed<bf16>(B, rows, H, dh, window, qkv, out, out_lo, st);
  if (stg == ST_SPLIT) return launch_swa_typed<Split>(B, rows, H, dh, window, qkv, out, out_lo, st);
  return launch_swa_typed<float>(B, rows, H, dh, window, qkv, out, out_lo, st);
}

}  // namespace ttt
