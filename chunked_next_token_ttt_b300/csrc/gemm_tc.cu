// Host side of the tcgen05 GEMM: tensor maps, shape checks, the split-K choice
// and the dispatch to the per-major instantiations.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "gemm_tc_kernel.cuh"

namespace ttt {
namespace tc {

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

// Status word for GEMMs launched without one (the single-operation API): a
// bounded wait that gives up records its code here.  File-scope device
// memory, so no call allocates; every GPU that loads the library holds it.
__device__ int g_tc_status;

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

}  // namespace tc

struct TcPlan {
  int bn = 128;      // output tile width
  int splitk = 1;    // K ranges
};
static TcPlan plan(const GemmDesc& g);
static int choose_bn(const GemmDesc& g) { return plan(g).bn; }

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

bool gemm_tc_supported(const GemmDesc& g) {
  if (g.dtype != ST_BF16 && g.dtype != ST_SPLIT) return false;
  if (g.dtype == ST_SPLIT && (g.loA % 8 || g.loB % 8 || g.loA <= 0 || g.loB <= 0)) return false;
  if (g.M < 64 || g.N < 64 || g.K < 16 || g.batch < 1) return false;
  if (!aligned16(g.A) || !aligned16(g.B)) return false;
  if (g.lda % 8 || g.ldb % 8) return false;
  if (g.batch > 1 && (g.sA % 8 || g.sB % 8 || g.sA <= 0 || g.sB <= 0)) return false;
  if (g.epi == EPI_DW && !g.partials) return false;
  if (g.B2 && (g.dtype != ST_BF16 || !aligned16(g.B2) || !g.a_kmajor || !g.b_kmajor ||
               (g.epi != EPI_GELU && g.epi != EPI_RESID)))
    return false;
  if (g.epi == EPI_LOGITS &&
      (g.dtype != ST_BF16 || g.batch != 1 || !g.a_kmajor || !g.b_kmajor || !g.lse_part ||
       g.lse_ld < ceil_div(g.N, choose_bn(g))))
    return false;
  // the epilogue stores column pairs: even leading dims, batch strides and lo offsets
  if ((g.ldo | g.sO | g.ldo2 | g.sO2 | g.ldx | g.sX | g.loO | g.loO2 | g.loX) & 1) return false;
  return true;
}

// Tile width and split of K, chosen together by a cost in units of one
// 128-wide k-slice's time: waves(units) x k-slices per unit x (1.21 for a
// 256-wide k-slice: twice the work at the measured 1.65x throughput), plus, when
// K is split, the partial tiles written and read back by each tile's last CTA
// (2 + 3 per partial, twice that for 256-wide tiles).  Measured on the TTT
// shapes: splitting pays for GEMMs with fewer tiles than SMs, and for larger
// ones only with long K ranges, so a GEMM that already fills a wave splits only
// if every range keeps at least 64 k-slices.  256-wide tiles are bf16 only;
// every K range keeps at least 4 k-slices; split partial tiles must fit the
// workspace and the arrival counters; the dW and logits epilogues (per-tile
// partial sums) never split.
static constexpr int kMaxSplitK = 32;

static TcPlan plan(const GemmDesc& g) {
  TcPlan best;
  double best_cost = 1e300;
  const int nkb = ceil_div(g.K, tc::BK);
  const bool can_split = g.ws && g.cnt && g.epi != EPI_DW && g.epi != EPI_LOGITS && !(g.N & 1) && nkb >= 8;
  for (int bn : {256, 128}) {
    if (bn == 256 && (g.dtype != ST_BF16 || g.B2)) continue;
    const long long tiles = (long long)ceil_div(g.N, bn) * ceil_div(g.M, tc::BM) * g.batch;
    const double kslice = bn == 256 ? 1.21 : 1.0;
    const double fix = bn == 256 ? 2.0 : 1.0;
    for (int sk = 1; sk <= kMaxSplitK; ++sk) {
      if (sk > 1 && (!can_split || sk > nkb / 4 || tiles > tc::kMaxSplitTiles ||
                     tiles * tc::BM * bn * sk > g.ws_elems))
        break;
      const int kper = ceil_div(nkb, sk);
      const int ranges = ceil_div(nkb, kper);
      if (sk > 1 && ranges != sk) continue;
      if (sk > 1 && tiles >= 148 && kper < 64) continue;
      const long long units = tiles * ranges;
      const long long waves = (units + 147) / 148;
      const double cost = (double)waves * kper * kslice + (ranges > 1 ? fix * (2.0 + 3.0 * ranges) : 0.0);
      if (cost < best_cost - 1e-9) {
        best_cost = cost;
        best.bn = bn;
        best.splitk = ranges;
      }
    }
  }
  return best;
}

int gemm_tc_splitk(const GemmDesc& g) { return plan(g).splitk; }

int gemm_tc_tile_n(const GemmDesc& g) { return choose_bn(g); }

int gemm_tc_partial_tiles(const GemmDesc& g) { return ceil_div(g.N, choose_bn(g)) * ceil_div(g.M, tc::BM); }

ttt_status gemm_tc_status_word(int** err) {
  void* p = nullptr;
  TTT_CUDA(symbol_address((const void*)&tc::g_tc_status, &p));
  *err = static_cast<int*>(p);
  return TTT_OK;
}

int gemm_tc_max_split_tiles() { return tc::kMaxSplitTiles; }

ttt_status gemm_tc(const GemmDesc& g, cudaStream_t st) {
  if (!gemm_tc_supported(g)) {
    set_error("shape/alignment not supported by the tensor-core GEMM");
    return TTT_ERR_UNSUPPORTED;
  }
  TTT_TRY(tc::init_driver());
  GemmDesc gd = g;
  if (!gd.err) TTT_TRY(gemm_tc_status_word(&gd.err));
  const bool a_mn = !g.a_kmajor, b_mn = !g.b_kmajor;
  const bool split = g.dtype == ST_SPLIT;
  const TcPlan pl = plan(g);
  gd.bn = pl.bn;
  // maps: A hi, B hi, A lo, B lo.  A: K-major [batch][M][K] boxes {64, 128};
  // MN-major [batch][K][M] panels {64, 64}.  Likewise B with BN rows.
  CUtensorMap maps[4];
  const bf16* planesA[2] = {static_cast<const bf16*>(g.A), static_cast<const bf16*>(g.A) + (split ? g.loA : 0)};
  const bf16* planesB[2] = {static_cast<const bf16*>(g.B),
                            g.B2 ? static_cast<const bf16*>(g.B2) : static_cast<const bf16*>(g.B) + (split ? g.loB : 0)};
  for (int p = 0; p < 2; ++p) {
    if (!a_mn) TTT_TRY(tc::make_map(&maps[2 * p], planesA[p], g.K, g.M, g.batch, g.lda, g.sA, tc::BK, tc::BM));
    else TTT_TRY(tc::make_map(&maps[2 * p], planesA[p], g.M, g.K, g.batch, g.lda, g.sA, tc::PANEL, tc::BK));
    if (!b_mn) TTT_TRY(tc::make_map(&maps[2 * p + 1], planesB[p], g.K, g.N, g.batch, g.ldb, g.sB, tc::BK, gd.bn));
    else TTT_TRY(tc::make_map(&maps[2 * p + 1], planesB[p], g.N, g.K, g.batch, g.ldb, g.sB, tc::PANEL, tc::BK));
  }
  const int nkb = ceil_div(g.K, tc::BK);
  const int splitk = pl.splitk;
  // 16-byte epilogue accesses need every epilogue address, leading dim, batch
  // stride and lo offset on an 8-element boundary
  {
    auto al = [](const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; };
    const long long m = g.ldo | g.sO | g.ldo2 | g.sO2 | g.ldx | g.sX | g.loO | g.loO2 | g.loX;
    if ((m & 15) == 0 && al(g.out, 32) && al(g.out2, 32) && al(g.aux, 32)) gd.vec = 2;
    else if ((m & 7) == 0 && al(g.out, 16) && al(g.out2, 16) && al(g.aux, 16)) gd.vec = 1;
    else gd.vec = 0;
  }
  if (splitk > 1) {
    // partial tiles go to the workspace; the caller's per-tile arrival counters
    // start at zero and every split-K launch that completes leaves them at zero
    const long long tiles = (long long)ceil_div(g.M, tc::BM) * ceil_div(g.N, gd.bn) * g.batch;
    if (tiles > tc::kMaxSplitTiles || !gd.cnt) {
      set_error("split-K GEMM with too many output tiles or without arrival counters");
      return TTT_ERR_UNSUPPORTED;
    }
  }
  if (g.B2) return tc::launch_kk_b2(gd, maps, nkb, splitk, st);
  if (!a_mn && !b_mn) return tc::launch_kk(gd, maps, nkb, splitk, st);
  if (!a_mn) return tc::launch_km(gd, maps, nkb, splitk, st);
  if (!b_mn) return tc::launch_mk(gd, maps, nkb, splitk, st);
  return tc::launch_mm(gd, maps, nkb, splitk, st);
}

}  // namespace ttt
