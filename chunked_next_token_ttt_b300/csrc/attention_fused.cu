// Fused sliding-window attention on the tensor cores (bf16 operands) for the
// frozen blocks ("End-to-End TTT" review, Method: sliding-window attention of
// window k keeps the current chunk's tokens visible before the update; 3.1:
// attention stays frozen during TTT).  One CTA per (128-query block, head,
// sequence); no score or probability block ever reaches global memory.
//
// Two passes over the key blocks (128 keys each) the query block's window
// reaches:
//   pass 1  S = Q K^T into TMEM; the softmax warps read S and keep each query
//           row's running maximum m and sum l of exp(S - m) over its window;
//   pass 2  S = Q K^T again; P = exp(S - m) (unnormalised, in [0, 1]) goes to
//           shared memory as bf16 in the tensor core's K-major 128B-swizzled
//           layout, and O += P V accumulates in TMEM;
// then out = O / l.  With m and l final before any P is formed, O is never
// rescaled (the price is a second Q K^T per key block).
//
// Warps: 0 TMA producer (Q once; K, then K and V, per key block through a
// two-slot ring), 1 TMEM allocator and MMA issuer (S double-buffered in TMEM,
// so the next S is computed while the softmax works on the current one),
// 2..9 softmax and output: the warps of TMEM lane quadrant q (w % 4 == q) own
// query rows 32 q .. 32 q + 31, one thread per row in each of two column
// halves (64 keys of a block, half of the head's output columns); the halves
// combine their running maximum and sum once, after pass 1.
// Every mbarrier wait is bounded (tc::mbar_wait); a timeout records a code in
// the status word and the CTA unwinds.
#include "gemm_tc_kernel.cuh"
#include "kernels.h"

namespace ttt {
namespace fa {

using namespace tc;

constexpr int BQ = 128;                  // query rows per CTA (UMMA M)
constexpr int BKV = 128;                 // keys per block (UMMA N of S, K of P V)
constexpr int KST = 2;                   // K/V ring slots
constexpr int NSW = 8;                   // softmax warps (two per TMEM lane quadrant)
constexpr int NTHREADS = 64 + 32 * NSW;  // producer, MMA, softmax
constexpr int HALF = BKV / 2;            // keys of a block per softmax thread
constexpr int PANEL_BYTES = 128 * 128;   // 128 rows x 64 bf16: one 128B-swizzle panel

template <int DH>
struct Layout {
  static constexpr int NP = DH / 64;                       // 64-wide panels of a head
  static constexpr int TILE = NP * PANEL_BYTES;            // a Q, K or V tile of 128 rows
  static constexpr int Q_OFF = 0;
  static constexpr int K_OFF = Q_OFF + TILE;               // [KST] K tiles
  static constexpr int V_OFF = K_OFF + KST * TILE;         // [KST] V tiles
  static constexpr int P_OFF = V_OFF + KST * TILE;         // P: 2 panels (128 keys)
  static constexpr int ML_OFF = P_OFF + 2 * PANEL_BYTES;   // [2 halves][128 rows] (m, l) exchange
  static constexpr int BAR_OFF = ML_OFF + 2 * BQ * 8;
  // q_full, kv_full[KST], kv_empty[KST], s_full[2], s_empty[2], p_full, p_empty, o_full; the TMEM slot
  static constexpr int NBAR = 1 + 2 * KST + 4 + 3;
  static constexpr int TOTAL = BAR_OFF + NBAR * 8 + 16;
  static constexpr int ALLOC = TOTAL + 1024;               // room to align the base to 1024 bytes
  static constexpr uint32_t TMEM_COLS = 512;               // S0: 0..127, S1: 128..255, O: 256..256+DH
};

struct Args {
  int rows;          // real positions per sequence
  int pad;           // zero rows before position 0 of every sequence
  int L;             // padded rows per sequence
  int window;        // k
  int d;             // model width (Q | K | V rows are 3d wide)
  float c;           // (1 / sqrt(dh)) * log2(e): scores as base-2 exponents
  bf16* out;         // [B][L][d], padded rows
  int* err;
};

// Barrier among the softmax warps only (id 1) that returns the AND of `ok`
// over all of them, so that they all take the same branch after it.
__device__ __forceinline__ bool softmax_all(bool ok) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, 1, %2, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}\n"
      : "=r"(r)
      : "r"((uint32_t)ok), "n"(32 * NSW)
      : "memory");
  return r != 0;
}

// A bounded mbarrier wait whose verdict is the same for every lane of the warp.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, int* err, int code) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, err, code));
}

template <int DH>
__global__ void __launch_bounds__(NTHREADS, 1)
    swa_fused_kernel(const __grid_constant__ CUtensorMap tm, const Args a, int nkb) {
  using L = Layout<DH>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::BAR_OFF);
  uint64_t* q_full = bars;
  uint64_t* kv_full = bars + 1;
  uint64_t* kv_empty = kv_full + KST;
  uint64_t* s_full = kv_empty + KST;       // [2]
  uint64_t* s_empty = s_full + 2;          // [2]
  uint64_t* p_full = s_empty + 2;
  uint64_t* p_empty = p_full + 1;
  uint64_t* o_full = p_empty + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + L::NBAR);
  float2* ml = reinterpret_cast<float2*>(smem + L::ML_OFF);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int q0 = blockIdx.x * BQ;             // first query position of the block
  const int hc = blockIdx.y * DH;             // the head's first column of Q (K at + d, V at + 2d)
  const int seq = blockIdx.z;
  // key block j holds positions kb0 + 128 j ..; block nkb - 1 ends at q0 + 127.
  // Blocks before j_lo hold no position >= max(0, q0 - k + 1).
  const int kb0 = q0 + BQ - nkb * BKV;
  const int j_lo = (max(0, q0 - a.window + 1) - kb0) / BKV;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < KST; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&s_full[b], 1);
      mbar_init(&s_empty[b], NSW);
    }
    mbar_init(p_full, NSW);
    mbar_init(p_empty, 1);
    mbar_init(o_full, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(L::TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tO = tmem + 2 * BKV;
  // Q | K | V were written by the projection GEMM before this kernel
  pdl_wait();
  pdl_launch();

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------ TMA producer
    mbar_expect_tx(q_full, L::TILE);
    for (int p = 0; p < L::NP; ++p)
      tma_load_3d(smem + L::Q_OFF + p * PANEL_BYTES, &tm, q_full, hc + 64 * p, a.pad + q0, seq);
    uint32_t u = 0;
    bool ok = true;
    for (int pass = 0; pass < 2 && ok; ++pass) {
      for (int j = j_lo; j < nkb; ++j, ++u) {
        const int s = u % KST;
        if (u >= (uint32_t)KST && !mbar_wait(&kv_empty[s], ((u / KST) & 1) ^ 1, a.err, 8)) {
          ok = false;
          break;
        }
        const int ky = a.pad + kb0 + j * BKV;    // may be negative: TMA fills zeros there
        mbar_expect_tx(&kv_full[s], pass ? 2 * L::TILE : L::TILE);
        for (int p = 0; p < L::NP; ++p)
          tma_load_3d(smem + L::K_OFF + s * L::TILE + p * PANEL_BYTES, &tm, &kv_full[s], hc + a.d + 64 * p, ky,
                      seq);
        if (pass)
          for (int p = 0; p < L::NP; ++p)
            tma_load_3d(smem + L::V_OFF + s * L::TILE + p * PANEL_BYTES, &tm, &kv_full[s], hc + 2 * a.d + 64 * p,
                        ky, seq);
      }
    }
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------ MMA issuer
    constexpr uint32_t idS = umma_idesc(BQ, BKV, false, false);   // S = Q K^T: both operands K-major
    constexpr uint32_t idO = umma_idesc(BQ, DH, false, true);     // O += P V: V MN-major
    const uint32_t sq = smem_u32(smem + L::Q_OFF), sp = smem_u32(smem + L::P_OFF);
    // S = Q K^T of ring slot s into TMEM buffer b (DH / 16 steps of 16)
    auto issue_s = [&](int s, int b) {
      const uint32_t sk = smem_u32(smem + L::K_OFF + s * L::TILE);
#pragma unroll
      for (int kk = 0; kk < DH / 16; ++kk) {
        const uint32_t off = (kk / 4) * PANEL_BYTES + (kk % 4) * 32;
        umma_bf16(tmem + b * BKV, umma_desc(sq + off, 16, 1024), umma_desc(sk + off, 16, 1024), idS,
                  kk > 0 ? 1u : 0u);
      }
    };
    // O += P V of ring slot s (8 steps of 16 keys); the first block starts O
    auto issue_pv = [&](int s, bool first) {
      const uint32_t sv = smem_u32(smem + L::V_OFF + s * L::TILE);
#pragma unroll
      for (int kk = 0; kk < BKV / 16; ++kk) {
        const uint64_t ad = umma_desc(sp + (kk / 4) * PANEL_BYTES + (kk % 4) * 32, 16, 1024);
        const uint64_t bd = umma_desc(sv + kk * 2048, PANEL_BYTES, 1024);
        umma_bf16(tO, ad, bd, idO, (!first || kk > 0) ? 1u : 0u);
      }
    };
    bool ok = mbar_wait(q_full, 0, a.err, 16);
    uint32_t u = 0, t = 0;       // ring uses; S products issued
    int prev = -1;               // ring slot of the pass-2 block whose P V is still to issue
    int npv = 0;                 // P V products issued
    for (int pass = 0; pass < 2 && ok; ++pass) {
      for (int j = j_lo; j < nkb && ok; ++j, ++u, ++t) {
        const int s = u % KST, b = t & 1;
        if (!mbar_wait(&kv_full[s], (u / KST) & 1, a.err, 16)) { ok = false; break; }
        // the softmax warps have read the S that last used TMEM buffer b
        if (t >= 2 && !mbar_wait(&s_empty[b], ((t >> 1) - 1) & 1, a.err, 16)) { ok = false; break; }
        tc_fence_after();
        issue_s(s, b);
        umma_commit(&s_full[b]);
        if (pass == 0) {
          umma_commit(&kv_empty[s]);     // pass 1 reads only K
          continue;
        }
        if (prev >= 0) {
          // the previous block's P is in shared memory: O += P V, then free its slot and P
          if (!mbar_wait(p_full, npv & 1, a.err, 16)) { ok = false; break; }
          tc_fence_after();
          issue_pv(prev, npv == 0);
          ++npv;
          umma_commit(&kv_empty[prev]);
          umma_commit(p_empty);
        }
        prev = s;
      }
    }
    if (ok && prev >= 0 && mbar_wait(p_full, npv & 1, a.err, 16)) {
      tc_fence_after();
      issue_pv(prev, npv == 0);
      umma_commit(&kv_empty[prev]);
      umma_commit(p_empty);
      umma_commit(o_full);
    }
  } else if (warp >= 2) {
    // ------------------------------------------------ softmax and output
    const int quad = warp & 3;
    const int half = (warp - 2) >> 2;          // which 64 keys of a block (and half of the output)
    const int r = quad * 32 + lane;            // query row of the block
    const int qi = q0 + r;                     // its position in the sequence
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const int col0 = half * HALF;
    float m = -FLT_MAX, l = 0.0f;              // base-2 running maximum and sum of this half
    uint32_t t = 0;
    int np = 0;                                // P blocks written
    bool ok = true;
    uint8_t* prow = smem + L::P_OFF + half * PANEL_BYTES + r * 128;
    for (int pass = 0; pass < 2; ++pass) {
      if (pass == 1) {
        // combine the two halves' (m, l) of every row: both threads of a row take
        // the total (every softmax warp reaches this vote once, timed out or not)
        ml[half * BQ + r] = make_float2(m, l);
        if (!softmax_all(ok)) {
          ok = false;
          break;
        }
        const float2 o = ml[(half ^ 1) * BQ + r];
        const float nm = fmaxf(m, o.x);
        l = (m > -FLT_MAX ? l * exp2f(m - nm) : 0.0f) + (o.x > -FLT_MAX ? o.y * exp2f(o.x - nm) : 0.0f);
        m = nm;
      }
      for (int j = j_lo; j < nkb; ++j, ++t) {
        const int b = t & 1;
        if (!warp_wait(&s_full[b], (t >> 1) & 1, a.err, 32)) { ok = false; break; }
        tc_fence_after();
        float v[HALF];
#pragma unroll
        for (int c = 0; c < HALF / 32; ++c)
          tmem_ld32(tmem + b * BKV + col0 + c * 32 + lane_off, *reinterpret_cast<float(*)[32]>(v + 32 * c));
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s_empty[b]);
        // the row's valid keys among this thread's columns: lo .. hi
        const int kp = kb0 + j * BKV + col0;
        const int lo = max(max(0, qi - a.window + 1), kp) - kp;
        const int hi = min(qi, kp + HALF - 1) - kp;
        const bool all = lo <= 0 && hi >= HALF - 1;
        if (pass == 0) {
          if (hi < lo) continue;
          float bm[4] = {-FLT_MAX, -FLT_MAX, -FLT_MAX, -FLT_MAX};
#pragma unroll
          for (int c = 0; c < HALF; ++c) {
            v[c] *= a.c;
            if (all || (c >= lo && c <= hi)) bm[c & 3] = fmaxf(bm[c & 3], v[c]);
          }
          const float nm = fmaxf(m, fmaxf(fmaxf(bm[0], bm[1]), fmaxf(bm[2], bm[3])));
          float se[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
          for (int c = 0; c < HALF; ++c)
            if (all || (c >= lo && c <= hi)) se[c & 3] += exp2f(v[c] - nm);
          l = (m > -FLT_MAX ? l * exp2f(m - nm) : 0.0f) + ((se[0] + se[1]) + (se[2] + se[3]));
          m = nm;
          continue;
        }
        // pass 2: this block's P once the previous P V has read the buffer
        if (np >= 1 && !warp_wait(p_empty, (np - 1) & 1, a.err, 32)) { ok = false; break; }
#pragma unroll
        for (int c8 = 0; c8 < HALF / 8; ++c8) {
          float p8[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int c = c8 * 8 + e;
            p8[e] = (all || (c >= lo && c <= hi)) ? exp2f(v[c] * a.c - m) : 0.0f;
          }
          // 16-byte chunk c8 of the row's 128-byte line in this half's panel, swizzled by the row
          *reinterpret_cast<uint4*>(prow + ((c8 ^ (r & 7)) * 16)) = pack_bf16x8(p8);
        }
        // the generic-proxy stores must be visible to the tensor core's reads
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) mbar_arrive(p_full);
        ++np;
      }
    }
    // out = O / l for the block's real rows: each half writes half of the head's columns
    if (ok && warp_wait(o_full, 0, a.err, 32)) {
      tc_fence_after();
      constexpr int OC = DH / 2;
      float o[OC];
#pragma unroll
      for (int c = 0; c < OC / 32; ++c)
        tmem_ld32(tO + half * OC + c * 32 + lane_off, *reinterpret_cast<float(*)[32]>(o + 32 * c));
      if (qi < a.rows) {
        const float inv = l > 0.0f ? 1.0f / l : 0.0f;
#pragma unroll
        for (int e = 0; e < OC; ++e) o[e] *= inv;
        bf16* dst = a.out + ((long long)seq * a.L + a.pad + qi) * a.d + hc + half * OC;
#pragma unroll
        for (int c8 = 0; c8 < OC / 8; ++c8) *reinterpret_cast<uint4*>(dst + 8 * c8) = pack_bf16x8(o + 8 * c8);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(L::TMEM_COLS) : "memory");
  }
}

template <int DH>
ttt_status launch_dh(const CUtensorMap& tm, const Args& a, int nqb, int H, int B, int nkb, cudaStream_t st) {
  using L = Layout<DH>;
  auto kern = swa_fused_kernel<DH>;
  TTT_CUDA(ensure_dyn_smem((const void*)kern, L::ALLOC));
  launch_pdl(kern, dim3(nqb, H, B), NTHREADS, L::ALLOC, st, tm, a, nkb);
  TTT_CHECK_LAUNCH();
  return TTT_OK;
}

}  // namespace fa

bool swa_fused_supported(int stg, int d, int heads) {
  if (stg != ST_BF16 || heads <= 0 || d % heads) return false;
  const int dh = d / heads;
  return dh == 64 || dh == 128;
}

ttt_status launch_swa_fused(int B, int rows, int H, int dh, int window, const void* qkvp, int pad, long long L,
                            void* out, int* err, cudaStream_t st) {
  if (B == 0 || rows == 0) return TTT_OK;
  const int d = H * dh;
  if (!swa_fused_supported(ST_BF16, d, H) || window < 1 || !err || L < rows + pad || L > (1LL << 30) ||
      (reinterpret_cast<uintptr_t>(qkvp) & 15) || (reinterpret_cast<uintptr_t>(out) & 15)) {
    set_error("fused attention: bf16, head width 64 or 128, 16-byte aligned buffers, a status word");
    return TTT_ERR_UNSUPPORTED;
  }
  TTT_TRY(tc::init_driver());
  // one map over the padded Q | K | V rows [B][L][3d]; a box is 64 columns x 128 rows
  CUtensorMap tm;
  TTT_TRY(tc::make_map(&tm, qkvp, 3LL * d, L, B, 3LL * d, L * 3LL * d, 64, fa::BQ));
  fa::Args a;
  a.rows = rows; a.pad = pad; a.L = (int)L; a.window = window; a.d = d;
  a.c = 1.4426950408889634f / sqrtf((float)dh);
  a.out = static_cast<bf16*>(out);
  a.err = err;
  const int nqb = ceil_div(rows, fa::BQ);
  const int nkb = ceil_div((long long)window + fa::BQ - 1, fa::BKV);
  if (dh == 64) return fa::launch_dh<64>(tm, a, nqb, H, B, nkb, st);
  return fa::launch_dh<128>(tm, a, nqb, H, B, nkb, st);
}

}  // namespace ttt
