#pragma once
// tcgen05 tensor-core GEMM kernel for sm_103a (template; instantiated per
// operand-major combination in gemm_tc_{kk,km,mk,mm}.cu): bf16 operands (or bf16 hi/lo pairs
// for fp32-accurate products), fp32 accumulation in TMEM, operands staged by
// TMA into 128B-swizzled shared memory, with the TTT epilogues applied on the
// way out of TMEM.
//
// Persistent: one CTA per SM walks the work units (output tile x K split) of
// the GEMM in a static round robin.
//   warp 0 (one lane)  TMA producer: a STAGES-deep ring of k-slices of 64
//                      elements; a slot holds the A and B tiles (A_hi, A_lo,
//                      B_hi, B_lo for split products), guarded by full/empty
//                      mbarriers
//   warp 1             allocates 2 x BN TMEM columns (two accumulators); one
//                      lane issues tcgen05.mma (M=128, N=BN, K=16) into the
//                      accumulator of the current unit, releases ring slots
//                      with tcgen05.commit and hands the accumulator to the
//                      epilogue with another commit
//   warps 2..9         epilogue: warp w reads TMEM lane quadrant w % 4 (the
//                      hardware's rule) and one 64-column half of the tile, so
//                      each thread holds 64 consecutive accumulators of one row
//                      (two tcgen05.ld.32x32b.x32); it hands the accumulator back
//                      to the MMA warp at once and applies the epilogue straight
//                      from registers with 16-byte loads and stores (whole
//                      sectors of a row per thread).  Unit i's epilogue
//                      overlaps unit i+1's MMAs.  The epilogue kind is a
//                      template argument (EK).
// Split K: with splitk > 1 each unit is one K range of an output tile; its
// epilogue writes the fp32 partial tile to the workspace, and the CTA that
// completes a tile's last partial (a per-tile arrival counter) sums the
// partials in split order and applies the epilogue, so the result does not
// depend on which CTA finished last.
// Operands may be K-major or MN-major (the backward's transposed products);
// TMA loads MN-major operands as 64-element-wide column panels and the UMMA
// descriptor's leading/stride byte offsets walk them.
//
// Every mbarrier wait is bounded (about 2 s of %globaltimer); on timeout the
// waiting thread records a code in the error word and the CTA unwinds: the
// producer waits (bounded) for its copies in flight, the MMA issuer for its
// MMAs, and TMEM is freed.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cfloat>
#include <type_traits>

#include "epilogue.cuh"
#include "gemm.h"

namespace ttt {
namespace tc {

constexpr int BM = 128;        // UMMA M (one CTA, TMEM lanes 0..127 = rows)
constexpr int BK = 64;         // k-slice: 64 bf16 = 128 bytes = one swizzle span
constexpr int PANEL = 64;      // MN-major panel width (elements)
constexpr int NUM_EPI_WARPS = 8;   // two per 32-lane TMEM quadrant, splitting the columns
constexpr int NUM_THREADS = 64 + 32 * NUM_EPI_WARPS;
constexpr int kBN = 128;           // output tile width
constexpr int kCols = 64;          // accumulator columns per epilogue thread
constexpr int kMaxSplitTiles = 4096;  // output tiles of a split-K GEMM (arrival counters)
constexpr long long kTimeoutNs = 2000000000LL;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// The polling loop of a wait whose first test failed: bounded, false (and
// *err |= code) after the timeout.  Out of line: it is the rare path.
static __device__ __noinline__ bool mbar_wait_slow(uint64_t* bar, uint32_t parity, int* err, int code) {
  const uint64_t t0 = globaltimer();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 256; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (globaltimer() - t0 > (uint64_t)kTimeoutNs) {
      atomicOr(err, code);
      return false;
    }
  }
}

// Bounded wait on phase `parity`; false (and *err |= code) after the timeout.
// The first test is inline: a thread that issues tcgen05.mma stalls the tensor
// pipe for as long as it spends between two MMAs, and a call costs hundreds of
// clocks even when the phase is already complete.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int* err, int code) {
  return mbar_try_wait(bar, parity) || mbar_wait_slow(bar, parity, err, code);
}

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* tm, uint64_t* bar, int c0, int c1,
                                            int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

// UMMA shared-memory descriptor, 128-byte swizzle.
__device__ __forceinline__ uint64_t umma_desc(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;  // descriptor version for tcgen05
  d |= (uint64_t)2 << 61;  // SWIZZLE_128B
  return d;
}

// Instruction descriptor, kind::f16 with bf16 A/B and fp32 D.
__host__ __device__ constexpr uint32_t umma_idesc(int M, int N, bool a_mn, bool b_mn) {
  return (1u << 4)                       // D = F32
         | (1u << 7)                     // A = BF16
         | (1u << 10)                    // B = BF16
         | ((a_mn ? 1u : 0u) << 15)      // A major: 0 = K, 1 = MN
         | ((b_mn ? 1u : 0u) << 16)      // B major
         | ((uint32_t)(N >> 3) << 17)    // N / 8
         | ((uint32_t)(M >> 4) << 24);   // M / 16
}

__device__ __forceinline__ void umma_bf16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
      "%14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// Barrier among the epilogue warps only (id 1; id 0 is __syncthreads).
__device__ __forceinline__ void epi_bar() {
  asm volatile("bar.sync 1, %0;" ::"n"(32 * NUM_EPI_WARPS) : "memory");
}

// Barrier among the epilogue warps that returns the AND of `ok` over all of
// them, so that every epilogue warp takes the same exit after a bounded wait
// and none is left waiting at a later barrier.
__device__ __forceinline__ bool epi_all(bool ok) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, 1, %2, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}\n"
      : "=r"(r)
      : "r"((uint32_t)ok), "n"(32 * NUM_EPI_WARPS)
      : "memory");
  return r != 0;
}

// Operand planes of a GEMM: PL_ONE bf16 A and B (one product); PL_SPLIT
// fp32-accurate A and B as bf16 hi/lo pairs (three products: hi*hi, hi*lo,
// lo*hi); PL_B2 bf16 A and a B given as the sum of two bf16 planes (two
// products, A*B0 + A*B1).
constexpr int PL_ONE = 0, PL_SPLIT = 1, PL_B2 = 2;

template <int BN, int PL>
struct Smem {
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_BYTES = BN * BK * 2;
  static constexpr int NA = PL == PL_SPLIT ? 2 : 1;          // planes of A
  static constexpr int NB = PL == PL_ONE ? 1 : 2;            // planes of B
  static constexpr int STAGE_BYTES = NA * A_BYTES + NB * B_BYTES;
  static constexpr int STAGING = 2 * (NUM_EPI_WARPS / 4) * BM * 4;  // per-row softmax states of EPI_LOGITS
  static constexpr int MAX_DYN = 232448;                     // per-block opt-in limit
  static constexpr int OVERHEAD = 1024 + 512;                // base alignment + barriers
  static constexpr int STAGES = (MAX_DYN - OVERHEAD - STAGING) / STAGE_BYTES;
  static constexpr int RING = STAGES * STAGE_BYTES;
  static constexpr int BAR_OFF = RING + STAGING;
  static constexpr int TOTAL = BAR_OFF + (2 * STAGES + 5) * 8 + 16 + NUM_EPI_WARPS * 4;
  static constexpr int ALLOC = TOTAL + 1024;
  static_assert(STAGES >= 2, "ring too shallow");
  static_assert(ALLOC <= MAX_DYN, "shared memory over the per-block limit");
};

// Work unit u: the output dimension with fewer tiles fastest (so the CTAs that
// run at the same time share the larger operand's tiles through L2: an LM head
// with a few row tiles streams each vocabulary tile of U from DRAM once), then
// the other, then batch entry, then K split.
struct Unit {
  int m0, n0, bz, ks, mt, nt;
};
__device__ __forceinline__ Unit decode_unit(int u, int mtiles, int ntiles, int batch, int BN) {
  Unit w;
  if (mtiles < ntiles) {
    w.mt = u % mtiles;
    w.nt = (u / mtiles) % ntiles;
  } else {
    w.nt = u % ntiles;
    w.mt = (u / ntiles) % mtiles;
  }
  const int z = u / (ntiles * mtiles);
  w.bz = z % batch;
  w.ks = z / batch;
  w.m0 = w.mt * BM;
  w.n0 = w.nt * BN;
  return w;
}

template <int BN, bool A_MN, bool B_MN, int PL, int EK>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmA2, const __grid_constant__ CUtensorMap tmB2,
                   const GemmDesc g, int nkb, int splitk, int mtiles, int ntiles, int* err) {
  using L = Smem<BN, PL>;
  constexpr int STAGES = L::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* stage = reinterpret_cast<float*>(smem + L::RING);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::BAR_OFF);
  uint64_t* empty = full + STAGES;
  uint64_t* accf = empty + STAGES;     // [2] accumulator ready (MMA -> epilogue)
  uint64_t* acce = accf + 2;           // [2] accumulator free (epilogue -> MMA)
  uint64_t* drain = acce + 2;          // the MMA issuer's wait for its own MMAs when it stops early
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  float* red = reinterpret_cast<float*>(tmem_slot + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int units = splitk * g.batch * mtiles * ntiles;
  const int kper = (nkb + splitk - 1) / splitk;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&accf[b], 1);
      mbar_init(&acce[b], NUM_EPI_WARPS);
    }
    mbar_init(drain, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(2 * BN)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // everything above touches only this CTA's shared memory and TMEM; global
  // memory (operands, outputs, counters) waits for the previous kernel
  pdl_wait();
  pdl_launch();

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------ TMA producer
    uint32_t kit = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
      const Unit w = decode_unit(u, mtiles, ntiles, g.batch, BN);
      const int kb_lo = w.ks * kper;
      const int nk = min(nkb, kb_lo + kper) - kb_lo;
      for (int kb = 0; kb < nk; ++kb, ++kit) {
        const int s = kit % STAGES;
        if (kit >= (uint32_t)STAGES && !mbar_wait(&empty[s], ((kit / STAGES) & 1) ^ 1, err, 8)) {
          ok = false;
          break;
        }
        uint8_t* sa = smem + s * L::STAGE_BYTES;
        uint8_t* sb = sa + L::NA * L::A_BYTES;
        mbar_expect_tx(&full[s], L::STAGE_BYTES);
        const int k0 = (kb_lo + kb) * BK;
#pragma unroll
        for (int p = 0; p < L::NA; ++p) {
          const CUtensorMap* ma = p ? &tmA2 : &tmA;
          uint8_t* da = sa + p * L::A_BYTES;
          if (!A_MN) {
            tma_load_3d(da, ma, &full[s], k0, w.m0, w.bz);
          } else {
#pragma unroll
            for (int j = 0; j < BM / PANEL; ++j) tma_load_3d(da + j * PANEL * BK * 2, ma, &full[s], w.m0 + j * PANEL, k0, w.bz);
          }
        }
#pragma unroll
        for (int p = 0; p < L::NB; ++p) {
          const CUtensorMap* mb = p ? &tmB2 : &tmB;
          uint8_t* db = sb + p * L::B_BYTES;
          if (!B_MN) {
            tma_load_3d(db, mb, &full[s], k0, w.n0, w.bz);
          } else {
#pragma unroll
            for (int j = 0; j < BN / PANEL; ++j) tma_load_3d(db + j * PANEL * BK * 2, mb, &full[s], w.n0 + j * PANEL, k0, w.bz);
          }
        }
      }
    }
    // no copy may still be landing in shared memory when the CTA exits (the
    // MMA issuer may have stopped early): wait, bounded, for each stage's last load
    for (uint32_t q = kit > (uint32_t)STAGES ? kit - STAGES : 0; q < kit; ++q)
      if (!mbar_wait(&full[q % STAGES], (q / STAGES) & 1, err, 8)) break;
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------ MMA issuer
    constexpr uint32_t idesc = umma_idesc(BM, BN, A_MN, B_MN);
    uint32_t kit = 0;
    uint32_t polled = ~0u;   // the k-slice whose stage was tested ahead, and the verdict
    bool ready = false;
    bool ok = true;
    int i = 0;
    for (int u = blockIdx.x; u < units && ok; u += gridDim.x, ++i) {
      const Unit w = decode_unit(u, mtiles, ntiles, g.batch, BN);
      const int kb_lo = w.ks * kper;
      const int nk = min(nkb, kb_lo + kper) - kb_lo;
      const int ab = i & 1, use = i >> 1;
      if (use >= 1 && !mbar_wait(&acce[ab], (use - 1) & 1, err, 16)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t d_tmem = tmem + (uint32_t)(ab * BN);
      for (int kb = 0; kb < nk; ++kb, ++kit) {
        const int s = kit % STAGES;
        if (!(polled == kit && ready) && !mbar_wait(&full[s], (kit / STAGES) & 1, err, 16)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sa = smem_u32(smem + s * L::STAGE_BYTES);
        const uint32_t sb = sa + L::NA * L::A_BYTES;
        constexpr int NPROD = PL == PL_SPLIT ? 3 : (PL == PL_B2 ? 2 : 1);
#pragma unroll
        for (int t = 0; t < NPROD; ++t) {
          // split products: hi*hi, hi*lo, lo*hi; two-plane B: A*B0, A*B1
          const uint32_t pa = sa + (t == 2 ? L::A_BYTES : 0);
          const uint32_t pb = sb + (t == 1 ? L::B_BYTES : 0);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k) {
            // K-major: the 16-element k-step is 32 bytes inside the swizzle span.
            // MN-major: 16 k-rows of 128 bytes; panels of 64 MN-elements are BK*128 bytes apart.
            const uint64_t ad = A_MN ? umma_desc(pa + k * 2048, PANEL * BK * 2, 1024) : umma_desc(pa + k * 32, 16, 1024);
            const uint64_t bd = B_MN ? umma_desc(pb + k * 2048, PANEL * BK * 2, 1024) : umma_desc(pb + k * 32, 16, 1024);
            umma_bf16(d_tmem, ad, bd, idesc, (kb > 0 || t > 0 || k > 0) ? 1u : 0u);
          }
        }
        umma_commit(&empty[s]);
        // test the next k-slice's stage now, while this one's MMAs run: its
        // latency is then off the issue path
        polled = kit + 1;
        ready = mbar_try_wait(&full[polled % STAGES], (polled / STAGES) & 1);
      }
      umma_commit(&accf[ab]);
    }
    if (!ok) {
      // stopped early: the MMAs already issued finish before TMEM is freed
      umma_commit(drain);
      mbar_wait(drain, 0, err, 16);
    }
  } else if (warp >= 2) {
    // ------------------------------------------------ epilogue
    using S = typename std::conditional<PL == PL_SPLIT, Split, bf16>::type;
    constexpr int HALVES = NUM_EPI_WARPS / 4;   // warps per TMEM lane quadrant
    constexpr int GPW = BN / kCols / HALVES;    // 64-column groups per thread
    static_assert(GPW >= 1 && GPW * kCols * HALVES == BN, "tile width not covered by the epilogue warps");
    const int ew = warp - 2;                    // 0..7
    const int quad = warp & 3;                  // TMEM lanes this warp may read
    const int half = ew >> 2;                   // which half of the tile's columns
    const int r = quad * 32 + lane;             // tile row of this thread
    float* lse_m = stage;                       // EPI_LOGITS: [HALVES][BM] row maxima
    float* lse_s = stage + HALVES * BM;         //             [HALVES][BM] row sums of exp
    const long long tiles = (long long)g.batch * mtiles * ntiles;
    int i = 0;
    constexpr bool AUX = epi_reads_aux<EK>();
    for (int u = blockIdx.x; u < units; u += gridDim.x, ++i) {
      const Unit w = decode_unit(u, mtiles, ntiles, g.batch, BN);
      const int ab = i & 1, use = i >> 1;
      const int row = w.m0 + r;
      // the aux input of a 64-column group (written by earlier kernels, not by
      // this GEMM): its loads for the first group are issued before waiting for
      // the accumulator, so they overlap the MMAs
      float xa[AUX ? kCols : 1];
      auto load_x = [&](int c) {
        const int n = w.n0 + c * kCols;
        if (splitk == 1 && g.vec == 2 && n + kCols <= g.N && row < g.M) {
#pragma unroll
          for (int j = 0; j < kCols; j += 16) load_aux16<S, EK>(g, w.bz, row, n + j, xa + j);
        }
      };
      if constexpr (AUX) load_x(half * GPW);
      if (!epi_all(mbar_wait(&accf[ab], use & 1, err, 32))) break;
      tc_fence_after();
      const long long tix = ((long long)w.bz * mtiles + w.mt) * ntiles + w.nt;
      float sq = 0.0f;
      float rmax = -FLT_MAX, rsum = 0.0f;       // EPI_LOGITS: this row over this thread's columns
#pragma unroll 1
      for (int gi = 0; gi < GPW; ++gi) {
        const int c = half * GPW + gi;          // column group of the tile
        if constexpr (AUX) {
          if (gi > 0) load_x(c);
        }
        float v[kCols];
        {
          const uint32_t ta = tmem + (uint32_t)(ab * BN + c * kCols) + ((uint32_t)(quad * 32) << 16);
          float (&v0)[32] = *reinterpret_cast<float(*)[32]>(v);
          float (&v1)[32] = *reinterpret_cast<float(*)[32]>(v + 32);
          tmem_ld32(ta, v0);
          tmem_ld32(ta + 32, v1);
        }
        if (gi == GPW - 1) {
          // every TMEM read of this accumulator is done: hand it back to the MMA warp
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&acce[ab]);
        }
        const int n = w.n0 + c * kCols;
        const bool full_vec = g.vec && n + kCols <= g.N;
        const bool wide = g.vec == 2 && n + kCols <= g.N;
        if (splitk > 1) {
          // fp32 partial tile of this K range in the workspace, column-major inside
          // the tile (column j holds the tile's BM rows), so that for every column
          // a warp's 32 rows are one 128-byte line
          float* dst = g.ws + ((long long)w.ks * tiles + tix) * (BM * BN) + (long long)(c * kCols) * BM + r;
#pragma unroll
          for (int j = 0; j < kCols; ++j) dst[j * BM] = v[j];
        } else if constexpr (EK == EPI_LOGITS) {
          // bf16 logits out (when kept); online-softmax state of these values,
          // folded into the row's running state
          float mx = -FLT_MAX, se = 0.0f;
          if (n + kCols <= g.N) {
#pragma unroll
            for (int j = 0; j < kCols; ++j) mx = fmaxf(mx, v[j]);
#pragma unroll
            for (int j = 0; j < kCols; ++j) se += __expf(v[j] - mx);
          } else {
#pragma unroll
            for (int j = 0; j < kCols; ++j)
              if (n + j < g.N) mx = fmaxf(mx, v[j]);
#pragma unroll
            for (int j = 0; j < kCols; ++j)
              if (n + j < g.N) se += __expf(v[j] - mx);
          }
          if (mx > -FLT_MAX) {
            const float mm = fmaxf(rmax, mx);
            rsum = (rmax > -FLT_MAX ? rsum * __expf(rmax - mm) : 0.0f) + se * __expf(mx - mm);
            rmax = mm;
          }
          if (row < g.M) {
            if (g.out) {
              if (wide) {
#pragma unroll
                for (int j = 0; j < kCols; j += 16)
                  HexIO<bf16>::store(g.out, 0, (long long)row * g.ldo + n + j, v + j);
              } else if (full_vec) {
#pragma unroll
                for (int j = 0; j < kCols; j += 8)
                  OctIO<bf16>::store(g.out, 0, (long long)row * g.ldo + n + j, v + j);
              } else {
                bf16* dst = static_cast<bf16*>(g.out) + (long long)row * g.ldo + n;
#pragma unroll
                for (int j = 0; j < kCols; ++j)
                  if (n + j < g.N) dst[j] = __float2bfloat16_rn(v[j]);
              }
            }
          }
        } else if (row < g.M) {
          if (wide) {
            if constexpr (AUX) {
#pragma unroll
              for (int j = 0; j < kCols; j += 16) epi_hex_x<S, EK>(g, w.bz, row, n + j, v + j, xa + j);
            } else {
#pragma unroll
              for (int j = 0; j < kCols; j += 16) sq += epi_hex<S, EK>(g, w.bz, row, n + j, v + j);
            }
          } else if (full_vec) {
#pragma unroll
            for (int j = 0; j < kCols; j += 8) sq += epi_oct<S, EK>(g, w.bz, row, n + j, v + j);
          } else {
#pragma unroll
            for (int j = 0; j < kCols; ++j)
              if (n + j < g.N) sq += epi_value<S>(g, w.bz, row, n + j, v[j]);
          }
        }
      }
      if (splitk > 1) {
        // Publish the partial; the CTA completing the tile's last partial reduces
        // them.  The barrier orders every epilogue thread's partial stores before
        // one thread's GPU-scope release fence and arrival (fences are
        // cumulative); the last arrival's acquire fence and the barrier after it
        // order the other CTAs' partials before this CTA's loads.
        epi_bar();
        if (ew == 0 && lane == 0) {
          asm volatile("fence.acq_rel.gpu;" ::: "memory");
          const int last = atomicAdd(&g.cnt[tix], 1) == splitk - 1;
          if (last) {
            g.cnt[tix] = 0;  // ready for the next split-K GEMM in stream order
            asm volatile("fence.acq_rel.gpu;" ::: "memory");
          }
          tmem_slot[1] = (uint32_t)last;
        }
        epi_bar();
        if (tmem_slot[1] && row < g.M) {
          // sum the partials in split order; one split's loads are all in flight at once
#pragma unroll 1
          for (int gi = 0; gi < GPW; ++gi) {
            const int c = half * GPW + gi;
            const int n = w.n0 + c * kCols;
            const float* src = g.ws + tix * (BM * BN) + (long long)(c * kCols) * BM + r;
            float v[kCols];
#pragma unroll
            for (int j = 0; j < kCols; ++j) v[j] = 0.0f;
#pragma unroll 1
            for (int q = 0; q < splitk; ++q) {
              const float* sl = src + q * tiles * (BM * BN);
#pragma unroll
              for (int j = 0; j < kCols; ++j) v[j] += __ldcg(sl + j * BM);
            }
            if (g.vec == 2 && n + kCols <= g.N) {
#pragma unroll
              for (int j = 0; j < kCols; j += 16) epi_hex<S, EK>(g, w.bz, row, n + j, v + j);
            } else if (g.vec && n + kCols <= g.N) {
#pragma unroll
              for (int j = 0; j < kCols; j += 8) epi_oct<S, EK>(g, w.bz, row, n + j, v + j);
            } else {
#pragma unroll
              for (int j = 0; j < kCols; ++j)
                if (n + j < g.N) epi_value<S>(g, w.bz, row, n + j, v[j]);
            }
          }
        }
        epi_bar();
      }
      if constexpr (EK == EPI_LOGITS) {
        // combine the row's state over the tile's column halves
        lse_m[half * BM + r] = rmax;
        lse_s[half * BM + r] = rsum;
        epi_bar();
        if (half == 0 && row < g.M) {
          float m0 = -FLT_MAX, s0 = 0.0f;
#pragma unroll
          for (int c = 0; c < HALVES; ++c) {
            const float m2 = lse_m[c * BM + r], s2 = lse_s[c * BM + r];
            if (m2 > -FLT_MAX) {
              const float mm = fmaxf(m0, m2);
              s0 = (m0 > -FLT_MAX ? s0 * __expf(m0 - mm) : 0.0f) + s2 * __expf(m2 - mm);
              m0 = mm;
            }
          }
          g.lse_part[(long long)row * g.lse_ld + w.nt] = make_float2(m0, s0);
        }
        epi_bar();
      }
      if (EK == EPI_DW || (EK == EK_ANY && g.epi == EPI_DW)) {
        sq = warp_sum(sq);
        if (lane == 0) red[ew] = sq;
        epi_bar();
        if (ew == 0 && lane == 0) {
          float t = 0.0f;
          for (int q = 0; q < NUM_EPI_WARPS; ++q) t += red[q];
          g.partials[(long long)w.bz * mtiles * ntiles + w.mt * ntiles + w.nt] = t;
        }
        epi_bar();
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(2 * BN) : "memory");
  }
}

// Host helpers (gemm_tc.cu): the driver's tensor-map encoder, and a 3-D bf16
// tensor map over X[batch][outer][inner] (leading dim ld, batch stride sz, in
// elements) with 128B swizzle and a box of box_inner x box_outer elements.
ttt_status init_driver();
ttt_status make_map(CUtensorMap* m, const void* base, long long inner, long long outer, int batch, long long ld,
                    long long sz, int box_inner, int box_outer);

// Launch one instantiation (persistent grid, one CTA per SM at most).
template <int BN, bool A_MN, bool B_MN, int PL, int EK>
ttt_status launch_bn(const GemmDesc& g, const CUtensorMap* maps, int nkb, int splitk, cudaStream_t st) {
  using L = Smem<BN, PL>;
  auto kern = gemm_tc_kernel<BN, A_MN, B_MN, PL, EK>;
  TTT_CUDA(ensure_dyn_smem((const void*)kern, L::ALLOC));
  const int mtiles = ceil_div(g.M, BM), ntiles = ceil_div(g.N, BN);
  const long long units = (long long)mtiles * ntiles * g.batch * splitk;
  int ctas = current_sm_count();
  if (g.max_ctas > 0 && g.max_ctas < ctas) ctas = g.max_ctas;
  const int grid = (int)(units < ctas ? units : ctas);
  launch_pdl(kern, grid, NUM_THREADS, L::ALLOC, st, maps[0], maps[1], maps[2], maps[3], g, nkb, splitk, mtiles, ntiles, g.err);
  TTT_CHECK_LAUNCH();
  return TTT_OK;
}

// bf16 GEMMs with many output tiles use 128 x 256 tiles (g.bn == 256): a third
// less shared-memory operand traffic per FLOP than 128 x 128.  bf16x3 products
// keep 128 x 128 (their ring stages are twice as large).
template <bool A_MN, bool B_MN, bool SPLIT, int EK>
ttt_status launch_kernel(const GemmDesc& g, const CUtensorMap* maps, int nkb, int splitk, cudaStream_t st) {
  if constexpr (!SPLIT) {
    if (g.bn == 256) return launch_bn<256, A_MN, B_MN, PL_ONE, EK>(g, maps, nkb, splitk, st);
  }
  return launch_bn<kBN, A_MN, B_MN, SPLIT ? PL_SPLIT : PL_ONE, EK>(g, maps, nkb, splitk, st);
}

// Two-plane B (GemmDesc::B2), K-major operands, 128-wide tiles: the fast-block
// forward products that score Settlement's candidate weights.
ttt_status launch_kk_b2(const GemmDesc& g, const CUtensorMap* maps, int nkb, int splitk, cudaStream_t st);

// Per operand-major combination: picks the instantiation for (storage, epilogue).
ttt_status launch_kk(const GemmDesc& g, const CUtensorMap* maps, int nkb, int splitk, cudaStream_t st);
ttt_status launch_km(const GemmDesc& g, const CUtensorMap* maps, int nkb, int splitk, cudaStream_t st);
ttt_status launch_mk(const GemmDesc& g, const CUtensorMap* maps, int nkb, int splitk, cudaStream_t st);
ttt_status launch_mm(const GemmDesc& g, const CUtensorMap* maps, int nkb, int splitk, cudaStream_t st);

}  // namespace tc
}  // namespace ttt
