// Fused sliding-window attention on the tensor cores (bf16 operands) for the
// frozen blocks ("End-to-End TTT" review, Method: sliding-window attention of
// window k keeps the current chunk's tokens visible before the update; 3.1:
// attention stays frozen during TTT).  No score or probability block ever
// reaches global memory.
//
// One pass over the key blocks (128 keys each) a query tile's window reaches,
// online softmax: per block, S = Q K^T into TMEM; the softmax threads take the
// block's row maximum; the row's running maximum m is raised only when the
// block's exceeds it by more than TAU (base 2), and then the row's partial
// output O in TMEM and its sum l are rescaled by 2^(m_old - m_new) before the
// block's P V is issued; P = 2^(S c - m) (at most 2^TAU) goes to TMEM as
// packed bf16 pairs, and O += P V accumulates in TMEM with P as the MMA's A
// operand read from TMEM (P never touches shared memory, whose bandwidth the
// K/V copies and the operand reads already share).  out = O / l.
//
// Head width 64 (two::swa_fused2_kernel): two 128-query tiles per CTA that
// share the K/V blocks; each 128-key block is taken as two 64-key sub-blocks,
// with S and P double-buffered per tile in TMEM (S 2 x 64, P 2 x 32, O 64
// columns: 256 per tile), so S of the next sub-block is computed while the
// softmax works on this one and P V of the last one runs meanwhile.  Four
// softmax warps per tile, one thread per query row, hold the sub-block's whole
// score row in registers (S is released right after the load).  One
// MMA-issuing warp per tile: a thread issuing back-to-back MMAs of these
// shapes reaches about half the tensor pipe's rate, and every instruction it
// runs between two MMAs idles the pipe.
//
// Head width 128 (swa_fused_kernel<128>): one 128-query tile per CTA; S and P
// double-buffered in TMEM; two softmax warps per TMEM lane quadrant, one
// thread per row in each of two column halves (64 keys of a block, half of the
// output columns), which exchange their block maxima once per block at a
// barrier of the quadrant's warps that also carries their wait verdicts, so
// they rescale alike and leave together.
//
// Warps: 0 TMA producer (Q once; K and V per key block through a ring),
// 1 TMEM allocator and MMA issuer, 2..9 softmax and output (head width 64: a
// second MMA issuer, warp 10).  Every mbarrier
// wait is bounded (tc::mbar_wait); a timeout records a code in the status word
// and the CTA unwinds: the producer waits (bounded) for its copies in flight,
// the MMA issuer for its MMAs, and TMEM is freed.
#include "gemm_tc_kernel.cuh"
#include "kernels.h"

namespace ttt {
namespace fa {

using namespace tc;

constexpr int BQ = 128;                  // query rows per CTA (UMMA M)
constexpr int BKV = 128;                 // keys per block (UMMA N of S, K of P V)
constexpr int NPART = 2;                 // softmax warps per TMEM lane quadrant
constexpr int NSW = 4 * NPART;           // softmax warps
constexpr int NTHREADS = 64 + 32 * NSW;  // producer, MMA, softmax
constexpr int QK = BKV / NPART;          // keys of a block per softmax thread
// pairs of every 8 consecutive P values computed by the polynomial 2^x on the
// FMA pipe instead of the MUFU unit (which does 32 exponentials per clock per
// SM here); every split measured slower, so none is
constexpr int EMU_PAIRS = 0;
constexpr int PANEL_BYTES = 128 * 128;   // 128 rows x 64 bf16: one 128B-swizzle panel
constexpr float TAU = 8.0f;              // raise the running maximum only beyond this (P <= 2^TAU)

template <int DH>
struct Layout {
  static constexpr int NP = DH / 64;                       // 64-wide panels of a head
  static constexpr int NSB = 2;                            // S buffers (in TMEM)
  static constexpr int NPB = 2;                            // P buffers (in TMEM)
  static constexpr int KST = DH == 64 ? 3 : 2;             // K/V ring slots
  static constexpr int TILE = NP * PANEL_BYTES;            // a Q, K or V tile of 128 rows
  static constexpr int Q_OFF = 0;
  static constexpr int K_OFF = Q_OFF + TILE;               // [KST] K tiles
  static constexpr int V_OFF = K_OFF + KST * TILE;         // [KST] V tiles
  // exchange between a row's NPART threads: [2 block parities][NPART][128 rows]
  // block maxima, then [NPART][128 rows] sums
  static constexpr int X_OFF = V_OFF + KST * TILE;
  static constexpr int BAR_OFF = X_OFF + 3 * NPART * BQ * 4;
  // q_full, kv_full[KST], kv_empty[KST], s_full[NSB], s_empty[NSB], p_full[NPB],
  // p_empty[NPB], o_full, drain; the TMEM slot
  static constexpr int NBAR = 1 + 2 * KST + 2 * NSB + 2 * NPB + 2;
  static constexpr int TOTAL = BAR_OFF + NBAR * 8 + 16;
  static constexpr int ALLOC = TOTAL + 1024;               // room to align the base to 1024 bytes
  // TMEM columns: NSB S buffers of 128 (fp32), O of DH (fp32), then NPB P
  // buffers of 64 (128 bf16 keys per row, two per column)
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t T_O = NSB * BKV;
  static constexpr uint32_t T_P = T_O + DH;
  static_assert(T_P + NPB * BKV / 2 <= TMEM_COLS, "TMEM columns");
  static_assert(ALLOC <= 232448, "shared memory over the per-block limit");
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

// Barrier of the NPART softmax warps of TMEM lane quadrant q (id 2 + q) that
// returns the AND of `ok` over them, so that they take the same branch.
__device__ __forceinline__ bool quad_all(int quad, bool ok) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}\n"
      : "=r"(r)
      : "r"((uint32_t)ok), "r"(2 + quad), "n"(32 * NPART)
      : "memory");
  return r != 0;
}

// 2^x by the hardware's approximate base-2 exponential (PTX ex2.approx.ftz:
// about 2 ulp; 2^-inf = 0, which masks out-of-window scores).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Packed pairs of floats for the two-wide FMA pipe instructions (f32x2).
typedef unsigned long long f2;
__device__ __forceinline__ f2 f2make(float x, float y) {
  f2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(x), "f"(y));
  return r;
}
__device__ __forceinline__ void f2split(f2 v, float& x, float& y) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(x), "=f"(y) : "l"(v));
}
__device__ __forceinline__ f2 f2fma(f2 a, f2 b, f2 c) {
  f2 r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ f2 f2add(f2 a, f2 b) {
  f2 r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ f2 f2sub(f2 a, f2 b) {
  f2 r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}

// 2^x for a pair on the FMA pipe.  x is clamped to >= -126 (2^-126 and below
// contribute nothing a bf16 P can carry); x = n + f with n = round(x), taken
// by adding 1.5 * 2^23 (which leaves n in the low mantissa bits) and f in
// [-1/2, 1/2]; 2^f by a cubic in Horner form whose coefficients are a
// relative-error-weighted least-squares fit of 2^f on [-1/2, 1/2] (largest
// relative error 7.5e-5, below bf16's 2^-9); 2^n enters by adding n to the
// exponent field (p lies in [0.70, 1.42], so the field stays in 0 .. 135).
__device__ __forceinline__ void ex2_poly2(float& x0, float& x1) {
  const f2 kRound = f2make(12582912.0f, 12582912.0f);
  const f2 x = f2make(fmaxf(x0, -126.0f), fmaxf(x1, -126.0f));
  const f2 j = f2add(x, kRound);
  const f2 f = f2sub(x, f2sub(j, kRound));
  f2 p = f2fma(f2make(0.05517115443944931f, 0.05517115443944931f), f,
               f2make(0.2426101416349411f, 0.2426101416349411f));
  p = f2fma(p, f, f2make(0.6932609677314758f, 0.6932609677314758f));
  p = f2fma(p, f, f2make(0.9999281167984009f, 0.9999281167984009f));
  float p0, p1, j0, j1;
  f2split(p, p0, p1);
  f2split(j, j0, j1);
  x0 = __int_as_float(__float_as_int(p0) + (__float_as_int(j0) << 23));
  x1 = __int_as_float(__float_as_int(p1) + (__float_as_int(j1) << 23));
}

// max(x, y, z) in one three-input instruction.
__device__ __forceinline__ float max3(float x, float y, float z) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(x), "f"(y), "f"(z));
  return r;
}

// A bounded mbarrier wait whose verdict is the same for every lane of the warp.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, int* err, int code) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, err, code));
}

// 16 consecutive TMEM columns of the warp's 32 lanes to and from registers.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])),
      "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])),
      "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])), "r"(__float_as_uint(v[15]))
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// 32 consecutive TMEM columns of the warp's 32 lanes from registers.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])),
      "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])),
      "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])), "r"(__float_as_uint(v[15])),
      "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])), "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])),
      "r"(__float_as_uint(v[20])), "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
      "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])), "r"(__float_as_uint(v[27])),
      "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])), "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Start loading 32 consecutive TMEM columns of the warp's 32 lanes; the values
// may be read only after tmem_ld_wait on the same registers.
__device__ __forceinline__ void tmem_ld32_start(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
      "%14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}

// Wait for every TMEM load the thread has started.  The registers pass
// through the wait, so the compiler schedules no use of them before it.
__device__ __forceinline__ void tmem_ld_wait(uint32_t (&r)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                 "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                 "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]),
                 "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]),
                 "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
               :
               : "memory");
}

// 16 consecutive TMEM columns of the warp's 32 lanes from registers, without
// waiting for the write (tcgen05.wait::st before the columns are published).
__device__ __forceinline__ void tmem_st16_nowait(uint32_t taddr, const float (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])),
      "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])),
      "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])), "r"(__float_as_uint(v[15]))
      : "memory");
}

// D (+)= A B with A (M = 128 rows, 16 bf16 of K packed in 8 columns) read
// from TMEM and B from shared memory.
__device__ __forceinline__ void umma_bf16_tmem_a(uint32_t tmem_d, uint32_t tmem_a, uint64_t bdesc, uint32_t idesc,
                                                 uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}\n" ::"r"(tmem_d),
      "r"(tmem_a), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// N consecutive TMEM columns (16 or a multiple of 32) of the warp's lanes.
template <int N>
__device__ __forceinline__ void tmem_ldn(uint32_t taddr, float (&v)[N]) {
  if constexpr (N == 16) {
    tmem_ld16(taddr, v);
  } else {
#pragma unroll
    for (int c = 0; c < N / 32; ++c) tmem_ld32(taddr + 32 * c, *reinterpret_cast<float(*)[32]>(v + 32 * c));
  }
}
template <int N>
__device__ __forceinline__ void tmem_stn(uint32_t taddr, const float (&v)[N]) {
  if constexpr (N == 16) {
    tmem_st16(taddr, v);
  } else {
#pragma unroll
    for (int c = 0; c < N / 32; ++c)
      tmem_st32(taddr + 32 * c, *reinterpret_cast<const float(*)[32]>(v + 32 * c));
  }
}

template <int DH>
__global__ void __launch_bounds__(NTHREADS, 1)
    swa_fused_kernel(const __grid_constant__ CUtensorMap tm, const Args a, int nkb) {
  using L = Layout<DH>;
  constexpr int KST = L::KST, NPB = L::NPB, NSB = L::NSB;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::BAR_OFF);
  uint64_t* q_full = bars;
  uint64_t* kv_full = bars + 1;
  uint64_t* kv_empty = kv_full + KST;
  uint64_t* s_full = kv_empty + KST;       // [NSB]
  uint64_t* s_empty = s_full + NSB;        // [NSB]
  uint64_t* p_full = s_empty + NSB;        // [NPB]
  uint64_t* p_empty = p_full + NPB;        // [NPB]
  uint64_t* o_full = p_empty + NPB;
  uint64_t* drain = o_full + 1;            // the MMA issuer's wait for its own MMAs when it stops early
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + L::NBAR);
  float* xch = reinterpret_cast<float*>(smem + L::X_OFF);

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
    for (int b = 0; b < NSB; ++b) {
      mbar_init(&s_full[b], 1);
      mbar_init(&s_empty[b], NSW);
    }
    for (int b = 0; b < NPB; ++b) {
      mbar_init(&p_full[b], NSW);
      mbar_init(&p_empty[b], 1);
    }
    mbar_init(o_full, 1);
    mbar_init(drain, 1);
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
  const uint32_t tO = tmem + L::T_O;
  // Q | K | V were written by the projection GEMM before this kernel
  pdl_wait();
  pdl_launch();

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------ TMA producer
    mbar_expect_tx(q_full, L::TILE);
    for (int p = 0; p < L::NP; ++p)
      tma_load_3d(smem + L::Q_OFF + p * PANEL_BYTES, &tm, q_full, hc + 64 * p, a.pad + q0, seq);
    uint32_t u = 0;
    for (int j = j_lo; j < nkb; ++j, ++u) {
      const int s = u % KST;
      if (u >= (uint32_t)KST && !mbar_wait(&kv_empty[s], ((u / KST) & 1) ^ 1, a.err, 8)) break;
      const int ky = a.pad + kb0 + j * BKV;    // may be negative: TMA fills zeros there
      mbar_expect_tx(&kv_full[s], 2 * L::TILE);
      for (int p = 0; p < L::NP; ++p) {
        tma_load_3d(smem + L::K_OFF + s * L::TILE + p * PANEL_BYTES, &tm, &kv_full[s], hc + a.d + 64 * p, ky, seq);
        tma_load_3d(smem + L::V_OFF + s * L::TILE + p * PANEL_BYTES, &tm, &kv_full[s], hc + 2 * a.d + 64 * p, ky,
                    seq);
      }
    }
    // no copy may still be landing in shared memory when the CTA exits (the
    // MMA issuer may have stopped early): wait, bounded, for Q and each slot's last load
    bool landed = mbar_wait(q_full, 0, a.err, 8);
    for (uint32_t q = u > (uint32_t)KST ? u - KST : 0; q < u && landed; ++q)
      landed = mbar_wait(&kv_full[q % KST], (q / KST) & 1, a.err, 8);
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------ MMA issuer
    constexpr uint32_t idS = umma_idesc(BQ, BKV, false, false);   // S = Q K^T: both operands K-major
    constexpr uint32_t idO = umma_idesc(BQ, DH, false, true);     // O += P V: V MN-major
    const uint32_t sq = smem_u32(smem + L::Q_OFF);
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
    // O += P V of ring slot s and TMEM P buffer pb (8 steps of 16 keys, 8
    // columns of packed pairs each); the first block starts O
    auto issue_pv = [&](int s, int pb, bool first) {
      const uint32_t sv = smem_u32(smem + L::V_OFF + s * L::TILE);
      const uint32_t tp = tmem + L::T_P + pb * (BKV / 2);
#pragma unroll
      for (int kk = 0; kk < BKV / 16; ++kk) {
        const uint64_t bd = umma_desc(sv + kk * 2048, PANEL_BYTES, 1024);
        umma_bf16_tmem_a(tO, tp + kk * 8, bd, idO, (!first || kk > 0) ? 1u : 0u);
      }
    };
    bool ok = mbar_wait(q_full, 0, a.err, 16);
    uint32_t t = 0;               // blocks whose S is issued (ring use t, TMEM buffer t & 1)
    int prev = -1;                // ring slot of the block whose P V is still to issue
    for (int j = j_lo; j < nkb && ok; ++j, ++t) {
      const int s = t % KST, b = t % NSB;
      if (!mbar_wait(&kv_full[s], (t / KST) & 1, a.err, 16)) { ok = false; break; }
      // the softmax warps have read the S that last used TMEM buffer b
      if (t >= (uint32_t)NSB && !mbar_wait(&s_empty[b], ((t / NSB) - 1) & 1, a.err, 16)) { ok = false; break; }
      tc_fence_after();
      issue_s(s, b);
      umma_commit(&s_full[b]);
      if (prev >= 0) {
        // the previous block's P is in shared memory (and O rescaled): O += P V
        const int pb = (t - 1) % NPB;
        if (!mbar_wait(&p_full[pb], ((t - 1) / NPB) & 1, a.err, 16)) { ok = false; break; }
        tc_fence_after();
        issue_pv(prev, pb, t == 1);
        umma_commit(&kv_empty[prev]);
        umma_commit(&p_empty[pb]);
      }
      prev = s;
    }
    if (ok && prev >= 0) {
      const int pb = (t - 1) % NPB;
      if (mbar_wait(&p_full[pb], ((t - 1) / NPB) & 1, a.err, 16)) {
        tc_fence_after();
        issue_pv(prev, pb, t == 1);
        umma_commit(&kv_empty[prev]);
        umma_commit(&p_empty[pb]);
        umma_commit(o_full);
      } else {
        ok = false;
      }
    }
    if (!ok) {
      // stopped early: the MMAs already issued finish before TMEM is freed
      umma_commit(drain);
      mbar_wait(drain, 0, a.err, 16);
    }
  } else if (warp >= 2) {
    // ------------------------------------------------ softmax and output
    const int quad = warp & 3;
    const int part = (warp - 2) >> 2;          // which QK keys of a block (and which OC output columns)
    const int r = quad * 32 + lane;            // query row of the block
    const int qi = q0 + r;                     // its position in the sequence
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const int col0 = part * QK;
    constexpr int OC = DH / NPART;             // output columns of this thread
    static_assert(OC == 16 || OC == 32 || OC == 64, "output columns per thread");
    float m = -INFINITY;                       // the row's running maximum (base 2), shared by its NPART threads
    float l = 0.0f;                            // this thread's part of the row's sum of P
    uint32_t t = 0;
    // ok: every wait of this warp so far ended in time (warp-uniform); a
    // failure is voted at the next quadrant barrier, where all NPART warps leave
    bool ok = true;
    for (int j = j_lo; j < nkb; ++j, ++t) {
      const int b = t % NSB, pb = t % NPB, xb = t & 1;
      ok = ok && warp_wait(&s_full[b], (t / NSB) & 1, a.err, 32);
      float v[QK];
      if (ok) {
        tc_fence_after();
        tmem_ldn<QK>(tmem + b * BKV + col0 + lane_off, v);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s_empty[b]);
      }
      // the row's valid keys among this thread's columns: lo .. hi; scores
      // outside them become -inf (2^-inf = 0), only in the window's edge blocks
      // (every lane takes the same path below: the warp-wide waits and TMEM
      // accesses need the warp converged)
      const int kp = kb0 + j * BKV + col0;
      const int lo = max(max(0, qi - a.window + 1), kp) - kp;
      const int hi = min(qi, kp + QK - 1) - kp;
      if (hi < lo) {
#pragma unroll
        for (int c = 0; c < QK; ++c) v[c] = -INFINITY;
      } else if (lo > 0 || hi < QK - 1) {
#pragma unroll
        for (int c = 0; c < QK; ++c)
          if (c < lo || c > hi) v[c] = -INFINITY;
      }
      float bm4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int c = 0; c < QK; c += 8) {
        bm4[0] = max3(bm4[0], v[c], v[c + 1]);
        bm4[1] = max3(bm4[1], v[c + 2], v[c + 3]);
        bm4[2] = max3(bm4[2], v[c + 4], v[c + 5]);
        bm4[3] = max3(bm4[3], v[c + 6], v[c + 7]);
      }
      // this part's block maximum (base 2) to the row's other threads; the P
      // buffer this block writes must have been read by the P V of block t - NPB
      xch[(xb * NPART + part) * BQ + r] = max3(bm4[0], bm4[1], fmaxf(bm4[2], bm4[3])) * a.c;
      if (ok && t >= (uint32_t)NPB) ok = warp_wait(&p_empty[pb], ((t / NPB) - 1) & 1, a.err, 32);
      if (!quad_all(quad, ok)) {
        ok = false;
        break;
      }
      const float* xr = xch + xb * NPART * BQ + r;
      float bm = xr[0];
#pragma unroll
      for (int q = 1; q < NPART; ++q) bm = fmaxf(bm, xr[q * BQ]);
      // raise the running maximum only by more than TAU: rescale l and O (the
      // partial output this thread owns) by 2^(m_old - m_new); all threads of
      // a row decide alike
      const bool raise = bm > m + TAU;
      const bool rescale = raise && m > -INFINITY;
      const float alpha = rescale ? ex2(m - bm) : 1.0f;
      if (raise) {
        l *= alpha;
        m = bm;
      }
      if (t >= 1 && __any_sync(0xffffffffu, rescale)) {
        // O must hold block t - 1's P V first (with one P buffer the wait
        // above has already covered it)
        if (NPB > 1) ok = warp_wait(&p_empty[(t - 1) % NPB], ((t - 1) / NPB) & 1, a.err, 32);
        if (ok) {
          tc_fence_after();
          float o[OC];
          tmem_ldn<OC>(tO + part * OC + lane_off, o);
#pragma unroll
          for (int e = 0; e < OC; ++e) o[e] *= alpha;
          tmem_stn<OC>(tO + part * OC + lane_off, o);
          tc_fence_before();
        }
      }
      // P = 2^(S c - m): scale and sum in pairs on the FMA pipe; EMU_PAIRS of
      // every four pairs through the polynomial, the rest through the MUFU unit
      const f2 c2 = f2make(a.c, a.c);
      const float nmv = m > -INFINITY ? -m : 0.0f;   // no valid key yet: every P is 2^-inf = 0
      const f2 nm2 = f2make(nmv, nmv);
      f2 se2[2] = {f2make(0.0f, 0.0f), f2make(0.0f, 0.0f)};
      float pw[QK / 2];                          // packed bf16 pairs (even key in the low half), as raw bits
#pragma unroll
      for (int c8 = 0; c8 < QK / 8; ++c8) {
#pragma unroll
        for (int e = 0; e < 8; e += 2) {
          f2 x = f2fma(f2make(v[c8 * 8 + e], v[c8 * 8 + e + 1]), c2, nm2);
          float x0, x1;
          f2split(x, x0, x1);
          if (e / 2 < EMU_PAIRS) {
            ex2_poly2(x0, x1);
          } else {
            x0 = ex2(x0);
            x1 = ex2(x1);
          }
          se2[(e >> 1) & 1] = f2add(se2[(e >> 1) & 1], f2make(x0, x1));
          const __nv_bfloat162 pr = __floats2bfloat162_rn(x0, x1);
          pw[c8 * 4 + e / 2] = *reinterpret_cast<const float*>(&pr);
        }
      }
      // this thread's keys part * QK .. + QK - 1 are P columns part * QK / 2 ..
      tmem_stn<QK / 2>(tmem + L::T_P + pb * (BKV / 2) + part * (QK / 2) + lane_off, pw);
      {
        float s0, s1, s2, s3;
        f2split(se2[0], s0, s1);
        f2split(se2[1], s2, s3);
        l += (s0 + s1) + (s2 + s3);
      }
      // the TMEM stores are complete (tcgen05.wait::st) before the MMA issuer
      // learns of them
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[pb]);
    }
    // out = O / (l over the row's NPART threads) for the block's real rows
    float* lx = xch + 2 * NPART * BQ;
    lx[part * BQ + r] = l;
    const bool fin = quad_all(quad, ok && warp_wait(o_full, 0, a.err, 32));
    if (fin) {
      float lt = lx[r];
#pragma unroll
      for (int q = 1; q < NPART; ++q) lt += lx[q * BQ + r];
      tc_fence_after();
      float o[OC];
      tmem_ldn<OC>(tO + part * OC + lane_off, o);
      if (qi < a.rows) {
        const float inv = lt > 0.0f ? 1.0f / lt : 0.0f;
#pragma unroll
        for (int e = 0; e < OC; ++e) o[e] *= inv;
        bf16* dst = a.out + ((long long)seq * a.L + a.pad + qi) * a.d + hc + part * OC;
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

// ---------------------------------------------------------------------------
// Head width 64: two 128-query tiles per CTA (queries q0 .. q0 + 255), each
// with its own four softmax warps (one thread per query row, all 128 keys of a
// block) and its own S, P and O in TMEM (128 + 64 + 64 columns per tile, 512
// in all).  The tiles share the K/V blocks: tile 1's window is tile 0's moved
// on by one block, so every block but the two ends serves both.  The tensor
// core alternates between the tiles, computing one tile's S or P V while the
// other's softmax runs, and no softmax warp waits for another.
namespace two {

constexpr int NT = 2;                          // query tiles per CTA
constexpr int NSW2 = 4 * NT;                   // softmax warps
// warp 0: TMA producer; warp 1 and warp 2 + NSW2: the MMA issuers of tile 0
// and tile 1 (a thread issuing tcgen05.mma feeds the tensor pipe at a limited
// rate, so each tile has its own); warps 2 .. 1 + NSW2: softmax
constexpr int NTHREADS2 = 96 + 32 * NSW2;
constexpr int KST2 = 4;                        // K/V ring slots (128 keys each)
constexpr int DH2 = 64;
constexpr int SUB = 64;                        // keys of a sub-block: one S and one P V
constexpr int SUB_BYTES = SUB * 128;           // a sub-block's rows of a K or V tile
constexpr int TILE2 = PANEL_BYTES;             // 128 rows x 64 bf16
constexpr int Q_OFF2 = 0;                      // [NT] Q tiles
constexpr int K_OFF2 = Q_OFF2 + NT * TILE2;    // [KST2] K tiles
constexpr int V_OFF2 = K_OFF2 + KST2 * TILE2;  // [KST2] V tiles
constexpr int BAR_OFF2 = V_OFF2 + KST2 * TILE2;
// q_full, kv_full[KST2], kv_empty[KST2], then per tile s_full[2], s_free[2],
// p_full[2], p_free[2], o_full, drain; the TMEM slot
constexpr int NBAR2 = 1 + 2 * KST2 + 10 * NT;
constexpr int ALLOC2 = BAR_OFF2 + NBAR2 * 8 + 16 + 1024;
static_assert(ALLOC2 <= 232448, "shared memory over the per-block limit");
// TMEM columns of tile t, from 256 t: S buffers (fp32, 64 keys) at 0 and 64,
// P buffers (bf16 pairs, 64 keys) at 128 and 160, O (fp32) at 192
constexpr uint32_t TMEM_COLS2 = 512;
constexpr uint32_t S_COL = 0, P_COL = 128, O_COL = 192;

__global__ void __launch_bounds__(NTHREADS2, 1)
    swa_fused2_kernel(const __grid_constant__ CUtensorMap tm, const Args a, int nkb) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + BAR_OFF2);
  uint64_t* q_full = bars;
  uint64_t* kv_full = bars + 1;
  uint64_t* kv_empty = kv_full + KST2;
  uint64_t* tile_bars = kv_empty + KST2;   // 10 per tile
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tile_bars + 10 * NT);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int q0 = blockIdx.x * (NT * BQ);
  const int hc = blockIdx.y * DH2;
  const int seq = blockIdx.z;
  // union key block u (128 keys) holds positions kb0 + 128 u ..; tile t reads
  // blocks ulo[t] .. nkb - 1 + t, the last ending at its last query
  // q0 + 128 t + 127, each as two 64-key sub-blocks
  const int kb0 = q0 + BQ - nkb * BKV;
  const int ulo0 = (max(0, q0 - a.window + 1) - kb0) / BKV;
  const int ulo1 = (max(0, q0 + BQ - a.window + 1) - kb0) / BKV;
  const int nu = nkb + 1 - ulo0;           // union blocks the CTA reads, from ulo0

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < KST2; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], NT);             // released by both issuers
    }
    for (int t = 0; t < NT; ++t) {
      uint64_t* tbar = tile_bars + 10 * t;
      for (int b = 0; b < 2; ++b) {
        mbar_init(&tbar[b], 1);                // s_full[b]: S of the buffer's sub-block is in TMEM
        mbar_init(&tbar[2 + b], 4);            // s_free[b]: the tile's four softmax warps have read it
        mbar_init(&tbar[4 + b], 4);            // p_full[b]: its P is in TMEM
        mbar_init(&tbar[6 + b], 1);            // p_free[b]: its P V is done (P free, O holds it)
      }
      mbar_init(&tbar[8], 1);                  // o_full: the tile's last P V is done
      mbar_init(&tbar[9], 1);                  // drain
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(TMEM_COLS2)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // Q | K | V were written by the projection GEMM before this kernel
  pdl_wait();
  pdl_launch();

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------ TMA producer
    mbar_expect_tx(q_full, NT * TILE2);
    for (int t = 0; t < NT; ++t)
      tma_load_3d(smem + Q_OFF2 + t * TILE2, &tm, q_full, hc, a.pad + q0 + BQ * t, seq);
    uint32_t i = 0;
    for (; i < (uint32_t)nu; ++i) {
      const int s = i % KST2;
      if (i >= (uint32_t)KST2 && !mbar_wait(&kv_empty[s], ((i / KST2) & 1) ^ 1, a.err, 8)) break;
      const int ky = a.pad + kb0 + (ulo0 + (int)i) * BKV;   // may be negative: TMA fills zeros there
      mbar_expect_tx(&kv_full[s], 2 * TILE2);
      tma_load_3d(smem + K_OFF2 + s * TILE2, &tm, &kv_full[s], hc + a.d, ky, seq);
      tma_load_3d(smem + V_OFF2 + s * TILE2, &tm, &kv_full[s], hc + 2 * a.d, ky, seq);
    }
    // no copy may still be landing in shared memory when the CTA exits
    bool landed = mbar_wait(q_full, 0, a.err, 8);
    for (uint32_t q = i > (uint32_t)KST2 ? i - KST2 : 0; q < i && landed; ++q)
      landed = mbar_wait(&kv_full[q % KST2], (q / KST2) & 1, a.err, 8);
  } else if ((warp == 1 || warp == 2 + NSW2) && lane == 0) {
    // ------------------------------------------------ MMA issuer of tile t
    // Every union block passes through both issuers in order: each waits for
    // it to land and releases its ring slot (kv_empty counts both), whether or
    // not its tile reads it, so a slot is refilled only after both are done.
    // Sub-block j of the tile uses S and P buffer j & 1: S(j) is computed while
    // the softmax works on sub-block j - 1, and P V(j - 1) once its P is in.
    const int t = warp == 1 ? 0 : 1;
    uint64_t* tbar = tile_bars + 10 * t;
    uint64_t *s_full = tbar, *s_free = tbar + 2, *p_full = tbar + 4, *p_free = tbar + 6;
    constexpr uint32_t idS = umma_idesc(BQ, SUB, false, false);   // S = Q K^T: both operands K-major
    constexpr uint32_t idO = umma_idesc(BQ, DH2, false, true);    // O += P V: P from TMEM, V MN-major
    const int off = (t ? ulo1 : ulo0) - ulo0;   // union index of the tile's first block
    const int nb = nkb + t - (t ? ulo1 : ulo0); // union blocks the tile reads
    const int nj = 2 * nb;                      // its sub-blocks
    const uint32_t sq = smem_u32(smem + Q_OFF2 + t * TILE2);
    const uint32_t tt = tmem + 256u * t;
    bool ok = mbar_wait(q_full, 0, a.err, 16);
    // union step i: for each half h, the tile's S of sub-block 2 n + h (n the
    // tile's index of union block i), then its P V of the sub-block before
    for (int i = 0; i <= nu && ok; ++i) {
      const int n = i - off;
      if (i < nu && !mbar_wait(&kv_full[i % KST2], (i / KST2) & 1, a.err, 16)) {
        ok = false;
        break;
      }
      for (int h = 0; h < 2; ++h) {
        const int j = 2 * n + h;
        if (i < nu && n >= 0 && n < nb) {
          const int b = j & 1;
          // the softmax has read S(j - 2) from this buffer
          if (j >= 2 && !mbar_wait(&s_free[b], ((j >> 1) - 1) & 1, a.err, 16)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sk = smem_u32(smem + K_OFF2 + (i % KST2) * TILE2 + h * SUB_BYTES);
#pragma unroll
          for (int kk = 0; kk < DH2 / 16; ++kk)
            umma_bf16(tt + S_COL + SUB * b, umma_desc(sq + kk * 32, 16, 1024), umma_desc(sk + kk * 32, 16, 1024),
                      idS, kk > 0 ? 1u : 0u);
          umma_commit(&s_full[b]);
        }
        const int jp = j - 1;
        if (jp >= 0 && jp < nj) {
          const int bp = jp & 1;
          if (!mbar_wait(&p_full[bp], (jp >> 1) & 1, a.err, 16)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const int ip = (jp >> 1) + off;       // union block of sub-block jp
          const uint32_t sv = smem_u32(smem + V_OFF2 + (ip % KST2) * TILE2 + (jp & 1) * SUB_BYTES);
#pragma unroll
          for (int kk = 0; kk < SUB / 16; ++kk)
            umma_bf16_tmem_a(tt + O_COL, tt + P_COL + (SUB / 2) * bp + kk * 8,
                             umma_desc(sv + kk * 2048, PANEL_BYTES, 1024), idO, (jp > 0 || kk > 0) ? 1u : 0u);
          umma_commit(&p_free[bp]);
          if (jp == nj - 1) umma_commit(&tbar[8]);
        }
        // union block i - 1 is done with: its last P V was just issued
        if (h == 0 && i >= 1) umma_commit(&kv_empty[(i - 1) % KST2]);
      }
    }
    if (!ok) {
      // stopped early: the MMAs already issued finish before TMEM is freed
      umma_commit(&tbar[9]);
      mbar_wait(&tbar[9], 0, a.err, 16);
    }
  } else if (warp >= 2 && warp < 2 + NSW2) {
    // ------------------------------------------------ softmax and output
    const int t = (warp - 2) >> 2;             // query tile
    uint64_t* tbar = tile_bars + 10 * t;
    uint64_t *s_full = tbar, *s_free = tbar + 2, *p_full = tbar + 4, *p_free = tbar + 6;
    const int quad = warp & 3;                 // TMEM lanes 32 quad .. + 31
    const int r = quad * 32 + lane;            // query row of the tile
    const int qi = q0 + BQ * t + r;            // its position in the sequence
    const uint32_t tt = tmem + 256u * t + ((uint32_t)(quad * 32) << 16);
    const int u_lo = t ? ulo1 : ulo0;
    const int nj = 2 * (nkb + t - u_lo);       // the tile's 64-key sub-blocks
    const f2 c2 = f2make(a.c, a.c);
    float m = -INFINITY;                       // the row's running maximum (base 2)
    float l = 0.0f;                            // the row's sum of P
    bool ok = true;
    for (int j = 0; j < nj; ++j) {
      const int b = j & 1;
      ok = warp_wait(&s_full[b], (j >> 1) & 1, a.err, 32);
      if (!ok) break;
      // the whole row of the sub-block's scores into registers; S is then free
      tc_fence_after();
      uint32_t ra[32], rb[32];
      tmem_ld32_start(tt + S_COL + SUB * b, ra);
      tmem_ld32_start(tt + S_COL + SUB * b + 32, rb);
      tmem_ld_wait(ra);
      tmem_ld_wait(rb);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_free[b]);
      // the row's valid keys lo .. hi of the sub-block; the rest become -inf
      // (2^-inf = 0), only in the window's edge sub-blocks
      const int kp = kb0 + (u_lo + (j >> 1)) * BKV + (j & 1) * SUB;
      const int lo = max(max(0, qi - a.window + 1), kp) - kp;
      const int hi = min(qi, kp + SUB - 1) - kp;
      float v[SUB];
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        v[e] = __uint_as_float(ra[e]);
        v[32 + e] = __uint_as_float(rb[e]);
      }
      if (lo > 0 || hi < SUB - 1) {
#pragma unroll
        for (int e = 0; e < SUB; ++e)
          if (e < lo || e > hi) v[e] = -INFINITY;
      }
      float bm4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int e = 0; e < SUB; e += 8) {
        bm4[0] = max3(bm4[0], v[e], v[e + 1]);
        bm4[1] = max3(bm4[1], v[e + 2], v[e + 3]);
        bm4[2] = max3(bm4[2], v[e + 4], v[e + 5]);
        bm4[3] = max3(bm4[3], v[e + 6], v[e + 7]);
      }
      const float bm = max3(bm4[0], bm4[1], fmaxf(bm4[2], bm4[3])) * a.c;
      // raise the running maximum only by more than TAU; then l and O are
      // rescaled by 2^(m_old - m_new)
      const bool raise = bm > m + TAU;
      const bool rescale = raise && m > -INFINITY;
      const float alpha = rescale ? ex2(m - bm) : 1.0f;
      if (raise) {
        l *= alpha;
        m = bm;
      }
      // P buffer b is free once P V(j - 2) is done
      if (j >= 2) {
        ok = warp_wait(&p_free[b], ((j >> 1) - 1) & 1, a.err, 32);
        if (!ok) break;
      }
      // a rescale needs O current: P V(j - 1) done (the P Vs complete in order)
      if (__any_sync(0xffffffffu, rescale)) {
        ok = warp_wait(&p_free[b ^ 1], ((j - 1) >> 1) & 1, a.err, 32);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < DH2 / 32; ++c) {
          float o[32];
          tmem_ld32(tt + O_COL + 32 * c, o);
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] *= alpha;
          tmem_st32(tt + O_COL + 32 * c, o);
        }
      }
      // P = 2^(S c - m), scale and sums in pairs on the FMA pipe; packed bf16
      // pairs (even key in the low half) to P buffer b
      const float nmv = m > -INFINITY ? -m : 0.0f;   // no valid key yet: every P is 2^-inf = 0
      const f2 nm2 = f2make(nmv, nmv);
      f2 se2[2] = {f2make(0.0f, 0.0f), f2make(0.0f, 0.0f)};
#pragma unroll
      for (int c = 0; c < SUB / 32; ++c) {
        float pw[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const f2 x = f2fma(f2make(v[32 * c + e], v[32 * c + e + 1]), c2, nm2);
          float x0, x1;
          f2split(x, x0, x1);
          if ((e / 2) % 4 < EMU_PAIRS) {
            ex2_poly2(x0, x1);
          } else {
            x0 = ex2(x0);
            x1 = ex2(x1);
          }
          se2[(e >> 1) & 1] = f2add(se2[(e >> 1) & 1], f2make(x0, x1));
          const __nv_bfloat162 pr = __floats2bfloat162_rn(x0, x1);
          pw[e / 2] = *reinterpret_cast<const float*>(&pr);
        }
        tmem_st16_nowait(tt + P_COL + (SUB / 2) * b + 16 * c, pw);
      }
      asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      {
        float s0, s1, s2, s3;
        f2split(se2[0], s0, s1);
        f2split(se2[1], s2, s3);
        l += (s0 + s1) + (s2 + s3);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[b]);
    }
    // out = O / l for the tile's real rows
    if (ok && warp_wait(&tbar[8], 0, a.err, 32)) {
      tc_fence_after();
      const float inv = l > 0.0f ? 1.0f / l : 0.0f;
      bf16* dst = a.out + ((long long)seq * a.L + a.pad + qi) * a.d + hc;
#pragma unroll
      for (int c = 0; c < DH2 / 32; ++c) {
        float o[32];
        tmem_ld32(tt + O_COL + 32 * c, o);
        if (qi < a.rows) {
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] *= inv;
#pragma unroll
          for (int c8 = 0; c8 < 4; ++c8) *reinterpret_cast<uint4*>(dst + 32 * c + 8 * c8) = pack_bf16x8(o + 8 * c8);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS2) : "memory");
  }
}

ttt_status launch(const CUtensorMap& tm, const Args& a, int rows, int H, int B, int nkb, cudaStream_t st) {
  TTT_CUDA(ensure_dyn_smem((const void*)swa_fused2_kernel, ALLOC2));
  launch_pdl(swa_fused2_kernel, dim3(ceil_div(rows, NT * BQ), H, B), NTHREADS2, ALLOC2, st, tm, a, nkb);
  TTT_CHECK_LAUNCH();
  return TTT_OK;
}

}  // namespace two

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
  if (dh == 64) return fa::two::launch(tm, a, rows, H, B, nkb, st);
  return fa::launch_dh<128>(tm, a, nqb, H, B, nkb, st);
}

}  // namespace ttt
