// tcgen05 tensor-core GEMM for sm_103a: bf16 operands, fp32 accumulation in
// TMEM, operands staged by TMA into 128B-swizzled shared memory, with the TTT
// epilogues applied on the way out of TMEM.
//
// One CTA computes one 128 x BN output tile of one batch entry:
//   warp 0 (one lane)  TMA producer: a STAGES-deep ring of (A, B) k-slices of
//                      64 elements, each slot guarded by a full/empty mbarrier
//   warp 1             allocates BN TMEM columns; one lane issues
//                      tcgen05.mma (M=128, N=BN, K=16) x 4 per slice and
//                      releases the slot with tcgen05.commit
//   warps 2..9         epilogue: tcgen05.ld of their 32-lane TMEM quadrant
//                      (two warps per quadrant, splitting the columns), staged
//                      through shared memory so that each warp then stores
//                      whole row segments (coalesced), per-element epilogue
// Operands may be K-major or MN-major (the backward's transposed products);
// TMA loads MN-major operands as 64-element-wide column panels and the UMMA
// descriptor's leading/stride byte offsets walk them.
//
// Every mbarrier wait is bounded (about 2 s of %globaltimer); on timeout the
// waiting thread records a code in the error word and the CTA unwinds.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "epilogue.cuh"
#include "gemm.h"

namespace ttt {
namespace tc {

constexpr int BM = 128;        // UMMA M (one CTA, TMEM lanes 0..127 = rows)
constexpr int BK = 64;         // k-slice: 64 bf16 = 128 bytes = one swizzle span
constexpr int PANEL = 64;      // MN-major panel width (elements)
constexpr int NUM_EPI_WARPS = 8;  // two per 32-lane TMEM quadrant, splitting the columns
constexpr int NUM_THREADS = 64 + 32 * NUM_EPI_WARPS;
constexpr int STAGE_LD = 65;      // staging row stride in floats (64 columns + 1 against bank conflicts)
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

// Bounded wait on phase `parity`; false (and *err |= code) after the timeout.
__device__ __noinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int* err, int code) {
  if (mbar_try_wait(bar, parity)) return true;
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

template <int BN, int STAGES>
struct Smem {
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_BYTES = BN * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int BAR_OFF = STAGES * STAGE_BYTES;
  static constexpr int TOTAL = BAR_OFF + (2 * STAGES + 1) * 8 + 16 + NUM_EPI_WARPS * 4;
  static_assert(BM * STAGE_LD * 4 <= BAR_OFF, "epilogue staging must fit in the operand ring");
  static constexpr int ALLOC = TOTAL + 1024;  // slack to align the base to 1024 bytes
};

// SPLIT: operands are bf16 hi/lo plane pairs; the k loop runs three times
// (hi*hi, hi*lo, lo*hi) into the same TMEM accumulator.  tmA2/tmB2 map the lo
// planes (unused otherwise).
template <int BN, int STAGES, bool A_MN, bool B_MN, bool SPLIT>
__global__ void __launch_bounds__(NUM_THREADS, 2)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmA2, const __grid_constant__ CUtensorMap tmB2,
                   const GemmDesc g, int nkb, int splitk, int* err) {
  // K range of this CTA (split-K: blockIdx.z = ks * batch + bz)
  const int ks = blockIdx.z / g.batch;
  const int kper = (nkb + splitk - 1) / splitk;
  const int kb_lo = ks * kper;
  const int nk_local = min(nkb, kb_lo + kper) - kb_lo;
  const int num_kb = SPLIT ? 3 * nk_local : nk_local;
  using L = Smem<BN, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::BAR_OFF);
  uint64_t* empty = full + STAGES;
  uint64_t* accb = empty + STAGES;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accb + 1);
  float* red = reinterpret_cast<float*>(tmem_slot + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN, bz = blockIdx.z % g.batch;
  // split-K partials go to slice ks * batch + bz of the fp32 workspace
  const int bz_out = blockIdx.z;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(accb, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(BN)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (threadIdx.x < NUM_EPI_WARPS) red[threadIdx.x] = 0.0f;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------ TMA producer
    for (int kb = 0; kb < num_kb; ++kb) {
      const int s = kb % STAGES;
      if (kb >= STAGES && !mbar_wait(&empty[s], ((kb / STAGES) & 1) ^ 1, err, 8)) break;
      uint8_t* sa = smem + s * L::STAGE_BYTES;
      uint8_t* sb = sa + L::A_BYTES;
      mbar_expect_tx(&full[s], L::STAGE_BYTES);
      const int term = SPLIT ? kb / nk_local : 0;
      const int k0 = (kb_lo + (SPLIT ? kb - term * nk_local : kb)) * BK;
      const CUtensorMap* ma = (SPLIT && term == 2) ? &tmA2 : &tmA;
      const CUtensorMap* mb = (SPLIT && term == 1) ? &tmB2 : &tmB;
      if (!A_MN) {
        tma_load_3d(sa, ma, &full[s], k0, m0, bz);
      } else {
#pragma unroll
        for (int j = 0; j < BM / PANEL; ++j) tma_load_3d(sa + j * PANEL * BK * 2, ma, &full[s], m0 + j * PANEL, k0, bz);
      }
      if (!B_MN) {
        tma_load_3d(sb, mb, &full[s], k0, n0, bz);
      } else {
#pragma unroll
        for (int j = 0; j < BN / PANEL; ++j) tma_load_3d(sb + j * PANEL * BK * 2, mb, &full[s], n0 + j * PANEL, k0, bz);
      }
    }
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------ MMA issuer
    constexpr uint32_t idesc = umma_idesc(BM, BN, A_MN, B_MN);
    bool ok = true;
    for (int kb = 0; kb < num_kb && ok; ++kb) {
      const int s = kb % STAGES;
      ok = mbar_wait(&full[s], (kb / STAGES) & 1, err, 16);
      if (!ok) break;
      tc_fence_after();
      const uint32_t sa = smem_u32(smem + s * L::STAGE_BYTES);
      const uint32_t sb = sa + L::A_BYTES;
#pragma unroll
      for (int k = 0; k < BK / 16; ++k) {
        // K-major: the 16-element k-step is 32 bytes inside the swizzle span.
        // MN-major: 16 k-rows of 128 bytes; panels of 64 MN-elements are BK*128 bytes apart.
        const uint64_t ad = A_MN ? umma_desc(sa + k * 2048, PANEL * BK * 2, 1024) : umma_desc(sa + k * 32, 16, 1024);
        const uint64_t bd = B_MN ? umma_desc(sb + k * 2048, PANEL * BK * 2, 1024) : umma_desc(sb + k * 32, 16, 1024);
        umma_bf16(tmem, ad, bd, idesc, (kb > 0 || k > 0) ? 1u : 0u);
      }
      umma_commit(&empty[s]);
    }
    umma_commit(accb);
  } else if (warp >= 2) {
    // ------------------------------------------------ epilogue
    // TMEM -> shared staging (the operand ring is idle once the accumulator
    // is complete) -> row-contiguous, coalesced global stores.
    bool ok = mbar_wait(accb, 0, err, 32);
    ok = __all_sync(0xffffffffu, ok);
    tc_fence_after();
    if (ok) {
      const int quad = warp & 3;              // TMEM lanes this warp may read
      const int half = (warp - 2) >> 2;       // which 32 of each 64 columns it reads
      const int ew = warp - 2;                // rows it stores: ew*16 .. ew*16+15
      float* stage = reinterpret_cast<float*>(smem);
      float sq = 0.0f;
#pragma unroll 1
      for (int c0 = 0; c0 < BN; c0 += 64) {
        float v[32];
        tmem_ld32(tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)(c0 + 32 * half), v);
        float* srow = stage + (quad * 32 + lane) * STAGE_LD + 32 * half;
#pragma unroll
        for (int i = 0; i < 32; ++i) srow[i] = v[i];
        epi_bar();
#pragma unroll 1
        for (int k = 0; k < BM / NUM_EPI_WARPS; ++k) {
          const int r = ew * (BM / NUM_EPI_WARPS) + k;
          const int row = m0 + r;
          if (row < g.M) {
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
              const int n = n0 + c0 + cc * 32 + lane;
              const float a = stage[r * STAGE_LD + cc * 32 + lane];
              if (n < g.N) {
                if (splitk > 1) static_cast<float*>(g.out)[(long long)bz_out * g.sO + (long long)row * g.ldo + n] = a;
                else sq += SPLIT ? epi_value<Split>(g, bz, row, n, a) : epi_value<bf16>(g, bz, row, n, a);
              }
            }
          }
        }
        epi_bar();
      }
      if (g.epi == EPI_DW) {
        sq = warp_sum(sq);
        if (lane == 0) red[ew] = sq;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (g.epi == EPI_DW && threadIdx.x == 0) {
    float t = 0.0f;
    for (int w = 0; w < NUM_EPI_WARPS; ++w) t += red[w];
    g.partials[(long long)bz * gridDim.x * gridDim.y + blockIdx.y * gridDim.x + blockIdx.x] = t;
  }
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(BN) : "memory");
  }
}

// ---------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;
int* g_err = nullptr;

ttt_status init_driver() {
  std::call_once(g_encode_once, [] {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    else
      cudaGetLastError();
  });
  if (!g_encode) {
    set_error("cuTensorMapEncodeTiled is not available");
    return TTT_ERR_CUDA;
  }
  return TTT_OK;
}

// 3-D bf16 tensor map over X[batch][outer][inner] (leading dim ld, batch stride sz, in elements).
ttt_status make_map(CUtensorMap* m, const void* base, long long inner, long long outer, int batch, long long ld,
                    long long sz, int box_inner, int box_outer) {
  cuuint64_t dims[3] = {(cuuint64_t)inner, (cuuint64_t)outer, (cuuint64_t)batch};
  const long long bstride = batch > 1 ? sz : ld * outer;
  cuuint64_t strides[2] = {(cuuint64_t)ld * 2, (cuuint64_t)bstride * 2};
  cuuint32_t box[3] = {(cuuint32_t)box_inner, (cuuint32_t)box_outer, 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    set_error("cuTensorMapEncodeTiled failed with code " + std::to_string((int)r));
    return TTT_ERR_CUDA;
  }
  return TTT_OK;
}

constexpr int kBN = 128;
constexpr int kStages = 3;

// acc = sum over the split-K partial slices (fixed order); then the epilogue.
template <typename S>
__global__ void splitk_reduce_kernel(const GemmDesc g, const float* __restrict__ ws, int splitk) {
  const int bz = blockIdx.y / g.M, m = blockIdx.y % g.M;
  const long long slice = (long long)g.M * g.N;
  for (int n = blockIdx.x * blockDim.x + threadIdx.x; n < g.N; n += gridDim.x * blockDim.x) {
    const long long off = (long long)m * g.N + n;
    float acc = 0.0f;
    for (int k = 0; k < splitk; ++k) acc += ws[((long long)k * g.batch + bz) * slice + off];
    epi_value<S>(g, bz, m, n, acc);
  }
}

template <bool A_MN, bool B_MN, bool SPLIT>
ttt_status launch_variant(const GemmDesc& g, const CUtensorMap* maps, int nkb, int splitk, cudaStream_t st) {
  using L = Smem<kBN, kStages>;
  auto kern = gemm_tc_kernel<kBN, kStages, A_MN, B_MN, SPLIT>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::ALLOC);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute", __FILE__, __LINE__);
    attr_set = true;
  }
  dim3 grid(ceil_div(g.N, kBN), ceil_div(g.M, BM), g.batch * splitk);
  if (splitk == 1) {
    kern<<<grid, NUM_THREADS, L::ALLOC, st>>>(maps[0], maps[1], maps[2], maps[3], g, nkb, 1, g.err);
    TTT_CHECK_LAUNCH();
    return TTT_OK;
  }
  GemmDesc gp = g;   // partial products into the workspace, fp32, one slice per (split, batch)
  gp.out = g.ws;
  gp.ldo = g.N;
  gp.sO = (long long)g.M * g.N;
  kern<<<grid, NUM_THREADS, L::ALLOC, st>>>(maps[0], maps[1], maps[2], maps[3], gp, nkb, splitk, g.err);
  TTT_CHECK_LAUNCH();
  dim3 rgrid(ceil_div(g.N, 256), g.batch * g.M);
  if (SPLIT) splitk_reduce_kernel<Split><<<rgrid, 256, 0, st>>>(g, g.ws, splitk);
  else splitk_reduce_kernel<bf16><<<rgrid, 256, 0, st>>>(g, g.ws, splitk);
  TTT_CHECK_LAUNCH();
  return TTT_OK;
}

}  // namespace tc

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

bool gemm_tc_supported(const GemmDesc& g) {
  if (g.dtype != ST_BF16 && g.dtype != ST_SPLIT) return false;
  if (g.dtype == ST_SPLIT && (g.loA % 8 || g.loB % 8 || g.loA <= 0 || g.loB <= 0)) return false;
  if (g.M < 64 || g.N < 64 || g.K < 16 || g.batch < 1) return false;
  if (!aligned16(g.A) || !aligned16(g.B)) return false;
  if (g.lda % 8 || g.ldb % 8) return false;
  if (g.batch > 1 && (g.sA % 8 || g.sB % 8 || g.sA <= 0 || g.sB <= 0)) return false;
  if (g.epi == EPI_DW && !g.partials) return false;
  return true;
}

// Split K when the output has too few 128x128 tiles to cover the SMs twice:
// every split keeps at least 4 k-slices, the partial slices must fit the
// workspace, and the dW epilogue (per-tile norm partials) never splits.
int gemm_tc_splitk(const GemmDesc& g) {
  if (!g.ws || g.epi == EPI_DW) return 1;
  const long long tiles = (long long)ceil_div(g.N, tc::kBN) * ceil_div(g.M, tc::BM) * g.batch;
  const int nkb = ceil_div(g.K, tc::BK);
  if (tiles >= 148 || nkb < 8) return 1;
  int want = (int)((2 * 148 + tiles - 1) / tiles);
  if (want > nkb / 4) want = nkb / 4;
  const long long slice = (long long)g.M * g.N * g.batch;
  while (want > 1 && slice * want > g.ws_elems) --want;
  if (want <= 1) return 1;
  const int kper = ceil_div(nkb, want);
  return ceil_div(nkb, kper);
}

int gemm_tc_partial_tiles(const GemmDesc& g) { return ceil_div(g.N, tc::kBN) * ceil_div(g.M, tc::BM); }

ttt_status gemm_tc_error_word(int** err) {
  if (!tc::g_err) {
    cudaError_t e = cudaMalloc(&tc::g_err, 4);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMalloc", __FILE__, __LINE__);
    e = cudaMemset(tc::g_err, 0, 4);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemset", __FILE__, __LINE__);
  }
  *err = tc::g_err;
  return TTT_OK;
}

ttt_status gemm_tc(const GemmDesc& g, cudaStream_t st) {
  if (!gemm_tc_supported(g)) {
    set_error("shape/alignment not supported by the tensor-core GEMM");
    return TTT_ERR_UNSUPPORTED;
  }
  TTT_TRY(tc::init_driver());
  GemmDesc gd = g;
  if (!gd.err) TTT_TRY(gemm_tc_error_word(&gd.err));
  const bool a_mn = !g.a_kmajor, b_mn = !g.b_kmajor;
  const bool split = g.dtype == ST_SPLIT;
  // maps: A hi, B hi, A lo, B lo.  A: K-major [batch][M][K] boxes {64, 128};
  // MN-major [batch][K][M] panels {64, 64}.  Likewise B with BN rows.
  CUtensorMap maps[4];
  const bf16* planesA[2] = {static_cast<const bf16*>(g.A), static_cast<const bf16*>(g.A) + (split ? g.loA : 0)};
  const bf16* planesB[2] = {static_cast<const bf16*>(g.B), static_cast<const bf16*>(g.B) + (split ? g.loB : 0)};
  for (int p = 0; p < 2; ++p) {
    if (!a_mn) TTT_TRY(tc::make_map(&maps[2 * p], planesA[p], g.K, g.M, g.batch, g.lda, g.sA, tc::BK, tc::BM));
    else TTT_TRY(tc::make_map(&maps[2 * p], planesA[p], g.M, g.K, g.batch, g.lda, g.sA, tc::PANEL, tc::BK));
    if (!b_mn) TTT_TRY(tc::make_map(&maps[2 * p + 1], planesB[p], g.K, g.N, g.batch, g.ldb, g.sB, tc::BK, tc::kBN));
    else TTT_TRY(tc::make_map(&maps[2 * p + 1], planesB[p], g.N, g.K, g.batch, g.ldb, g.sB, tc::PANEL, tc::BK));
  }
  const int nkb = ceil_div(g.K, tc::BK);
  const int splitk = gemm_tc_splitk(g);
#define TTT_TC_LAUNCH(AMN, BMN)                                                              \
  return split ? tc::launch_variant<AMN, BMN, true>(gd, maps, nkb, splitk, st)              \
               : tc::launch_variant<AMN, BMN, false>(gd, maps, nkb, splitk, st)
  if (!a_mn && !b_mn) TTT_TC_LAUNCH(false, false);
  if (!a_mn && b_mn) TTT_TC_LAUNCH(false, true);
  if (a_mn && !b_mn) TTT_TC_LAUNCH(true, false);
  TTT_TC_LAUNCH(true, true);
#undef TTT_TC_LAUNCH
}

}  // namespace ttt
